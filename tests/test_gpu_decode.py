"""GPU parity: fused decode attention against float64 attention on the oracle's
dequantised cache (same stored bytes)."""
import numpy as np
import pytest
import torch

from kvq_helpers import assert_attention_close, host, oracle_spec
from oracle import attention as oatt
from oracle.cache import OracleCache

pytestmark = pytest.mark.gpu

PAIRS = [
    ("fp16", 16, 0, "fp16", 16, 0),
    ("kivi_chan", 8, 0, "affine_token", 8, 128),
    ("kivi_chan", 4, 0, "affine_token", 4, 32),
    ("affine_token", 8, 64, "affine_token", 8, 64),
    ("affine_token", 4, 64, "affine_token", 4, 64),
    ("q4_0", 4, 32, "affine_token", 8, 128),
    ("q4_0", 4, 32, "affine_token", 4, 32),
]


@pytest.fixture(scope="module")
def kvq():
    import bit_kv_cache_quant_gb300 as m

    return m


def _rand(shape, seed, dtype, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(dtype)


def _build(kvq, pair, B, H, D, T, dtype, seed, cap=None, bias=False):
    kf, kb, kg, vf, vb, vg = pair
    kg, vg = (min(kg, D) if kg else 0), (min(vg, D) if vg else 0)
    kbias = _rand((H, D), seed + 7, torch.float32, 1.5) if bias else None
    cache = kvq.KVCache(B, H, D, cap or T, kf, kb, kg, vf, vb, vg,
                        k_bias=None if kbias is None else kbias.cuda())
    oc = OracleCache(oracle_spec(cache, None if kbias is None else kbias.numpy()))
    k = _rand((B, H, T, D), seed, dtype, 1.0)
    if kbias is not None:
        k = (k.float() + kbias[None, :, None, :]).to(dtype)
    v = _rand((B, H, T, D), seed + 1, dtype)
    cache.append(k.cuda(), v.cuda(), calibrate_k=(kf == "kivi_chan"))
    if kf == "kivi_chan":
        oc.calibrate_k(host(k))
    oc.append(host(k), host(v))
    return cache, oc


def _check(kvq, cache, oc, G, dtype, seed, what):
    B, H, D = cache.batch, cache.n_kv_heads, cache.head_dim
    q = _rand((B, H * G, D), seed + 2, dtype, 1.0)
    out = cache.decode_attn(q.cuda())
    kh, vh = oc.dequant()
    ref = oatt.decode_attention(host(q), kh, vh)
    return assert_attention_close(out, ref, what)


@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}{p[1]}-{p[3]}{p[4]}")
@pytest.mark.parametrize("G", [1, 2, 3, 4])
@pytest.mark.parametrize("D,T", [(128, 1000), (64, 333), (32, 65)])
def test_decode_matches_oracle(kvq, pair, G, D, T):
    cache, oc = _build(kvq, pair, 2, 2, D, T, torch.bfloat16, seed=D + T, bias=pair[0] == "q4_0")
    _check(kvq, cache, oc, G, torch.bfloat16, seed=G, what=f"G={G} D={D} T={T}")


@pytest.mark.parametrize("T", [1, 2, 15, 31, 33, 64, 255, 257, 1023, 4099])
def test_decode_ragged_lengths(kvq, T):
    pair = ("affine_token", 4, 64, "affine_token", 4, 64)
    cache, oc = _build(kvq, pair, 1, 2, 128, T, torch.bfloat16, seed=T)
    _check(kvq, cache, oc, 3, torch.bfloat16, seed=T, what=f"T={T}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_decode_io_dtypes(kvq, dtype):
    pair = ("kivi_chan", 8, 0, "affine_token", 8, 32)
    cache, oc = _build(kvq, pair, 1, 8, 32, 260, dtype, seed=5)
    _check(kvq, cache, oc, 1, dtype, seed=6, what=str(dtype))


def test_single_token_returns_value(kvq):
    pair = ("affine_token", 8, 64, "affine_token", 8, 64)
    cache, oc = _build(kvq, pair, 1, 2, 64, 1, torch.float32, seed=9)
    q = _rand((1, 4, 64), 3, torch.float32, 5.0)
    out = cache.decode_attn(q.cuda()).cpu().numpy()
    _, vh = oc.dequant()
    for h in range(4):
        np.testing.assert_allclose(out[0, h], vh[0, h // 2, 0], rtol=0, atol=1e-6)


def test_empty_cache_gives_zeros(kvq):
    cache = kvq.KVCache(1, 2, 128, 64, "affine_token", 4, 64, "affine_token", 4, 64)
    out = cache.decode_attn(torch.randn(1, 6, 128, device="cuda", dtype=torch.bfloat16))
    assert torch.all(out == 0)


def test_peaked_attention_and_custom_scale(kvq):
    # large logits (scale 1.0, keys with offsets) exercise the online-softmax rescaling
    pair = ("q4_0", 4, 32, "affine_token", 8, 128)
    cache, oc = _build(kvq, pair, 1, 2, 128, 3000, torch.bfloat16, seed=11, bias=True)
    q = _rand((1, 8, 128), 12, torch.bfloat16, 2.0)
    out = cache.decode_attn(q.cuda(), softmax_scale=0.5)
    kh, vh = oc.dequant()
    ref = oatt.decode_attention(host(q), kh, vh, scale=0.5)
    assert_attention_close(out, ref, "scale 0.5")


@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}{p[1]}-{p[3]}{p[4]}")
@pytest.mark.parametrize("G", [5, 6, 7, 8])
def test_decode_up_to_eight_heads_per_kv_head(kvq, pair, G):
    # bf16 io and head_dim 128 take the tensor-core kernel, which carries up to 8 heads
    cache, oc = _build(kvq, pair, 1, 2, 128, 700, torch.bfloat16, seed=G, bias=pair[0] == "q4_0")
    _check(kvq, cache, oc, G, torch.bfloat16, seed=G + 1, what=f"G={G}")


@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}{p[1]}-{p[3]}{p[4]}")
def test_decode_fp32_io_head_dim_128(kvq, pair):
    # fp32 io keeps the exact CUDA-core kernel (1e-5 tolerance) at head_dim 128 too
    cache, oc = _build(kvq, pair, 2, 2, 128, 600, torch.float32, seed=77, bias=pair[0] == "q4_0")
    _check(kvq, cache, oc, 4, torch.float32, seed=78, what="fp32 io")


def test_repeated_calls_are_identical(kvq):
    # split merge counters reset themselves: the same call twice gives the same bytes
    pair = ("affine_token", 4, 64, "affine_token", 4, 64)
    cache, _ = _build(kvq, pair, 1, 8, 128, 8192, torch.bfloat16, seed=13)
    q = _rand((1, 24, 128), 14, torch.bfloat16).cuda()
    a = cache.decode_attn(q).clone()
    b = cache.decode_attn(q)
    assert torch.equal(a, b)
    assert kvq.kvq_decode_workspace_bytes(cache.handle, 24) > 0


# The tensor-core decode picks its launch shape from the number of (batch row,
# kv head) pairs and the cache length.  On a 152-SM GB300 these cases land on
# each shape: one sixteen-warp CTA per SM (few pairs, long caches: 19 or 9
# splits per pair); eight-warp CTAs, two per SM, when the grid fits one wave
# otherwise, with one or many splits; four-warp CTAs (larger grids).  Over
# four query heads per kv head (G = 8 here) every CTA carries a second head
# group of warps over the same tiles, and the one-wave shape holds one CTA
# per SM.  Whatever the shape, the result must match the oracle.
LAUNCH_SHAPES = [
    ("sixteen_warps_19_splits", 1, 8, 8192 + 37, None),
    ("sixteen_warps_9_splits", 1, 16, 3000, None),
    ("eight_warps_4_splits", 2, 4, 300, None),
    ("eight_warps_2_splits", 13, 8, 150, 150),
    ("four_warps", 16, 8, 2000, None),
]


@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}{p[1]}-{p[3]}{p[4]}")
@pytest.mark.parametrize("name,B,H,T,cap", LAUNCH_SHAPES, ids=[s[0] for s in LAUNCH_SHAPES])
def test_decode_launch_shapes(kvq, pair, name, B, H, T, cap):
    cache, oc = _build(kvq, pair, B, H, 128, T, torch.bfloat16, seed=T + B, cap=cap, bias=pair[0] == "q4_0")
    for G in (3, 8):
        _check(kvq, cache, oc, G, torch.bfloat16, seed=G + 11, what=f"{name} G={G}")


def test_tile_wait_timeout_reports_and_recovers(kvq):
    # A tile that never completes (the test hook arms each CTA's first tile
    # barrier for more bytes than arrive): its bounded wait runs out, the
    # launch reports KVQ_DEV_TIMEOUT, the CTAs that stopped still arrive on
    # their split's merge counter (which the last arrival resets), and after
    # kvq_clear_status the same cache decodes exactly as before.
    pair = ("affine_token", 4, 64, "affine_token", 4, 64)
    cache, _ = _build(kvq, pair, 2, 8, 128, 4096, torch.bfloat16, seed=31)
    q = _rand((2, 24, 128), 32, torch.bfloat16).cuda()
    ref = cache.decode_attn(q).clone()
    torch.cuda.synchronize()
    assert cache.stats().device_status == 0
    kvq.kvq_test_stall_decode_tiles(True)
    try:
        cache.decode_attn(q)
        torch.cuda.synchronize()
    finally:
        kvq.kvq_test_stall_decode_tiles(False)
    assert cache.stats().device_status == kvq.DEV_TIMEOUT
    lay = cache.layout
    sem = cache.buf[lay.split_sem: lay.split_sem + 4 * 16].view(torch.int32)
    assert torch.all(sem == 0), "a merge counter was left short of its reset"
    kvq.kvq_clear_status(cache.handle)
    assert cache.stats().device_status == 0
    assert torch.equal(cache.decode_attn(q), ref)
