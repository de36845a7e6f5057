"""GPU parity: the KIVI residual buffer (full-precision tail, per-channel K in closed blocks).

bf16 decodes run the tensor-core kernel (fragments folded with each block's
channel scales, one CTA for the tail); fp32 decodes the CUDA-core kernel.

MLX memo, section 3: the newest tokens are kept unquantised; when the buffer is
full, its keys are quantised per channel as one closed block; attention reads the
quantised bulk and then the unquantised tail.  Codes, block scales, value planes
and the fp32 tail are compared bit-exactly with the oracle; attention within
the decode tolerance of the io dtype.
"""
import numpy as np
import pytest
import torch

from kvq_helpers import assert_attention_close, assert_cache_equal, host, oracle_spec
from oracle import attention as oatt
from oracle.cache import OracleCache

pytestmark = pytest.mark.gpu

SIDES = [
    # (k_bits, R, v_bits, v_group)
    (4, 64, 4, 32),
    (4, 128, 4, 32),
    (8, 64, 8, 128),
]


@pytest.fixture(scope="module")
def kvq():
    import bit_kv_cache_quant_gb300 as m

    assert torch.cuda.is_available()
    return m


def _inputs(shape, seed, dtype, offset_sigma=2.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g)
    x = x + torch.randn(shape[1], shape[3], generator=g)[None, :, None, :] * offset_sigma
    return x.to(dtype)


def _pair(kvq, B, H, D, cap, side):
    kb, R, vb, vg = side
    vg = min(vg, D)
    cache = kvq.KVCache(B, H, D, cap, "kivi_block", kb, R, "affine_token", vb, vg)
    return cache, OracleCache(oracle_spec(cache))


@pytest.mark.parametrize("side", SIDES, ids=lambda s: f"k{s[0]}R{s[1]}-v{s[2]}g{s[3]}")
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16])
def test_prefill_then_chunks_bit_exact(kvq, side, D, dtype):
    B, H = 2, 3
    cache, oc = _pair(kvq, B, H, D, 600, side)
    R = side[1]
    seed = 10 * D + side[0]
    # a prefill that closes blocks and leaves a tail, then chunks that cross block boundaries
    for i, n in enumerate((R * 2 + 37, 1, R - 40, 5, R + 3, 1)):
        k = _inputs((B, H, n, D), seed + 2 * i, dtype)
        v = _inputs((B, H, n, D), seed + 2 * i + 1, dtype, 0.0)
        cache.append(k.cuda(), v.cuda())
        oc.append(host(k), host(v))
        assert_cache_equal(cache, oc, f"after chunk {i} (n={n})")
    st = cache.stats()
    assert st.stored == oc.stored and st.tail == oc.n_tail and st.pos == oc.pos


@pytest.mark.parametrize("side", SIDES[:2], ids=lambda s: f"k{s[0]}R{s[1]}")
def test_single_tokens_across_flushes(kvq, side):
    # decode-style appends: the tail fills to R and empties into a closed block, twice
    B, H, D = 1, 2, 128
    cache, oc = _pair(kvq, B, H, D, 512, side)
    R = side[1]
    for t in range(2 * R + 3):
        k = _inputs((B, H, 1, D), 500 + t, torch.bfloat16)
        v = _inputs((B, H, 1, D), 900 + t, torch.bfloat16, 0.0)
        cache.append(k.cuda(), v.cuda())
        oc.append(host(k), host(v))
        if t in (R - 2, R - 1, R, 2 * R - 1, 2 * R + 2):
            assert_cache_equal(cache, oc, f"token {t}")


@pytest.mark.parametrize("side", SIDES, ids=lambda s: f"k{s[0]}R{s[1]}-v{s[2]}g{s[3]}")
@pytest.mark.parametrize("n", [40, 128, 300, 700])
@pytest.mark.parametrize("G", [1, 3, 4])
def test_decode_matches_oracle(kvq, side, n, G):
    # tail only (n < R), whole blocks and no tail (n = 128 = 2 R or R), blocks plus a tail
    B, H, D = 2, 2, 128
    cache, oc = _pair(kvq, B, H, D, 800, side)
    k = _inputs((B, H, n, D), n + G, torch.bfloat16)
    v = _inputs((B, H, n, D), n + G + 1, torch.bfloat16, 0.0)
    cache.append(k.cuda(), v.cuda())
    oc.append(host(k), host(v))
    kh, vh = oc.dequant()
    for dtype in (torch.bfloat16, torch.float32):
        q = _inputs((B, H * G, D)[:2] + (1, D), 7 * n + G, dtype, 0.0).reshape(B, H * G, D)
        out = cache.decode_attn(q.cuda())
        ref = oatt.decode_attention(host(q), kh, vh)
        assert_attention_close(out, ref, f"n={n} G={G} {dtype}")


def test_decode_many_splits_and_an_empty_cache(kvq):
    # a long bulk (several splits plus the tail CTA) and a cache with no token at all
    B, H, D, G = 1, 2, 64, 2
    cache, oc = _pair(kvq, B, H, D, 9000, (4, 128, 4, 32))
    empty = cache.decode_attn(torch.ones((B, H * G, D), dtype=torch.float32).cuda())
    assert torch.count_nonzero(empty) == 0
    k = _inputs((B, H, 8300, D), 3, torch.bfloat16)
    v = _inputs((B, H, 8300, D), 4, torch.bfloat16, 0.0)
    cache.append(k.cuda(), v.cuda())
    oc.append(host(k), host(v))
    assert oc.n_tail == 8300 % 128
    kh, vh = oc.dequant()
    q = _inputs((B, H * G, 1, D), 5, torch.float32, 0.0).reshape(B, H * G, D)
    out = cache.decode_attn(q.cuda())
    assert_attention_close(out, oatt.decode_attention(host(q), kh, vh), "8300 tokens")
    assert torch.equal(out, cache.decode_attn(q.cuda()))   # split counters reset


def test_overflow_and_unsupported_calls(kvq):
    B, H, D = 1, 1, 64
    cache, oc = _pair(kvq, B, H, D, 128, (4, 64, 4, 32))   # a bulk of two blocks
    for n, seed in ((120, 1), (20, 2)):                      # one block + 56, then two blocks + 12
        k = _inputs((B, H, n, D), seed, torch.bfloat16)
        cache.append(k.cuda(), k.cuda())
        oc.append(host(k), host(k))
    assert_cache_equal(cache, oc, "two blocks and a tail")
    # 60 more would close a third block: refused on the device, nothing written
    k = _inputs((B, H, 60, D), 3, torch.bfloat16)
    cache.append(k.cuda(), k.cuda())
    assert cache.stats().device_status == kvq.DEV_OVERFLOW
    kvq.kvq_clear_status(cache.handle)
    assert cache.stats().device_status == 0
    assert_cache_equal(cache, oc, "after the refused append")
    with pytest.raises(kvq.KvqError):
        cache.evict_keepset(torch.zeros((B, H, 4), dtype=torch.int32).cuda())
    with pytest.raises(kvq.KvqError):
        cache.append(k.cuda(), k.cuda(), calibrate_k=True)
    with pytest.raises(kvq.KvqError):   # over four heads per kv head: tensor-core path only (16-bit io)
        cache.decode_attn(torch.zeros((B, 5 * H, D), dtype=torch.float32).cuda())


@pytest.mark.parametrize("G", [5, 8])
@pytest.mark.parametrize("n", [100, 400])
def test_decode_up_to_eight_heads_per_kv_head(kvq, G, n):
    B, H, D = 1, 2, 128
    cache, oc = _pair(kvq, B, H, D, 512, (4, 64, 4, 32))
    k = _inputs((B, H, n, D), 3 * n + G, torch.bfloat16)
    v = _inputs((B, H, n, D), 3 * n + G + 1, torch.bfloat16, 0.0)
    cache.append(k.cuda(), v.cuda())
    oc.append(host(k), host(v))
    kh, vh = oc.dequant()
    q = _inputs((B, H * G, 1, D), 11 * n + G, torch.bfloat16, 0.0).reshape(B, H * G, D)
    assert_attention_close(cache.decode_attn(q.cuda()), oatt.decode_attention(host(q), kh, vh), f"G={G} n={n}")
