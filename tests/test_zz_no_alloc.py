"""kvq_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some users of this library run where cudaMalloc is off limits (inside an
allocator or memory-pool callback, in a plugin host that forbids device
allocations after start-up, in a loop that must never reach the driver's
allocator).  kvq_decode_attn_noalloc serves them: it keeps the split-KV
partials in a fixed scratch array inside the library instead of a caller
workspace.  This test calls it through the C ABI and checks, on two calls in a
row, that its output matches kvq_decode_attn's (which uses a caller-allocated
workspace) within the attention tolerance the other tests use.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one; the test also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from kvq_helpers import attn_tolerance

pytestmark = pytest.mark.gpu


def _noalloc(kvq):
    f = kvq.lib.kvq_decode_attn_noalloc
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_float, ctypes.c_void_p]
    return f


@pytest.mark.parametrize("shape", [
    # (batch, kv heads, query heads, head_dim, tokens, K format, V format)
    (1, 8, 24, 128, 8192, ("affine_token", 4, 64), ("affine_token", 4, 64)),
    (4, 8, 32, 128, 4096, ("q4_0", 4, 32), ("affine_token", 8, 128)),
])
def test_noalloc_matches_workspace_decode_twice(shape):
    import bit_kv_cache_quant_gb300 as kvq

    B, Hkv, Hq, D, T, kf, vf = shape
    f = _noalloc(kvq)
    lib = kvq.lib
    lib.kvq_noalloc_scratch_bytes.restype = ctypes.c_size_t
    g = torch.Generator().manual_seed(T + Hq)
    cache = kvq.KVCache(B, Hkv, D, T + 8, *kf, *vf)
    k = torch.randn(B, Hkv, T, D, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, Hkv, T, D, generator=g).to(torch.bfloat16).cuda()
    cache.append(k, v)
    need = kvq.kvq_decode_workspace_bytes(cache.handle, Hq)
    assert 0 < need <= lib.kvq_noalloc_scratch_bytes()    # the call really runs split-KV through its scratch
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16).cuda()
        ref = cache.decode_attn(q)
        out = torch.full_like(q, float("nan"))
        st = f(cache.handle, q.data_ptr(), out.data_ptr(), Hq, kvq.DTYPES[q.dtype], 0.0, stream)
        assert st == 0, lib.kvq_last_error().decode()
        torch.cuda.synchronize()
        r = ref.float().cpu().numpy().astype(np.float64)
        o = out.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(o)), f"call {call}: output not fully written"
        assert np.all(np.abs(o - r) <= attn_tolerance(r, q.dtype)), f"call {call}: max diff {np.abs(o - r).max()}"
