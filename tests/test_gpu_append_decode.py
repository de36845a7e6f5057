"""GPU parity of the one-call decode step (kvq_append_decode): its cache bytes
must equal those of the separate calls (append, eviction, decode) bit for bit,
and its attention must match float64 attention over the oracle's dequantised
cache after the same appends and evictions."""
import numpy as np
import pytest
import torch

from kvq_helpers import assert_attention_close, assert_cache_equal, host, oracle_spec
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


def _rand(shape, g, dtype, scale=1.0, offset=None):
    x = torch.randn(shape, generator=g) * scale
    if offset is not None:
        x = x + offset
    return x.to(dtype)


def _pair_caches(kvq, pair, B, H, D, cap, layout, sink, window, bias):
    kf, kb, kg, vf, vb, vg = pair
    kg, vg = (min(kg, D) if kg else 0), (min(vg, D) if vg else 0)
    kw = dict(layout=layout, sink=sink, window=window, k_bias=None if bias is None else bias.cuda())
    a = kvq.KVCache(B, H, D, cap, kf, kb, kg, vf, vb, vg, **kw)
    b = kvq.KVCache(B, H, D, cap, kf, kb, kg, vf, vb, vg, **kw)
    oc = OracleCache(oracle_spec(a, None if bias is None else bias.numpy()))
    return a, b, oc


def _run(kvq, pair, B, H, D, G, cap, T0, steps, layout="linear", sink=0, window=0, dtype=torch.bfloat16, seed=0):
    """T0 tokens by a bulk append, then `steps` decode steps, fused on one cache and separate on another."""
    g = torch.Generator().manual_seed(seed)
    kf = pair[0]
    bias = _rand((H, D), g, torch.float32, 1.5) if kf == "q4_0" else None
    off = (bias[None, :, None, :] if bias is not None else _rand((1, H, 1, D), g, torch.float32, 2.0))
    a, b, oc = _pair_caches(kvq, pair, B, H, D, cap, layout, sink, window, bias)
    calib = kf == "kivi_chan"
    if T0 or calib:
        n0 = max(T0, 1)
        k0 = _rand((B, H, n0, D), g, dtype, 1.0, off)
        v0 = _rand((B, H, n0, D), g, dtype)
        for c in (a, b):
            c.append(k0.cuda(), v0.cuda(), calibrate_k=calib)
            if layout != "linear":
                c.evict_middle()
        if calib:
            oc.calibrate_k(host(k0))
        oc.append(host(k0), host(v0))
        if layout != "linear":
            oc.evict_middle()
    worst = 0.0
    for t in range(steps):
        k1 = _rand((B, H, 1, D), g, dtype, 1.0, off)
        v1 = _rand((B, H, 1, D), g, dtype)
        q = _rand((B, H * G, D), g, dtype)
        out_a = a.append_decode(k1.cuda(), v1.cuda(), q.cuda())
        b.append(k1.cuda(), v1.cuda())
        if layout != "linear":
            b.evict_middle()
        out_b = b.decode_attn(q.cuda())
        oc.append(host(k1), host(v1))
        if layout != "linear":
            oc.evict_middle()
        kh, vh = oc.dequant()
        ref = oatt.decode_attention(host(q), kh, vh)
        worst = max(worst, assert_attention_close(out_a, ref, f"fused step {t}"))
        assert_attention_close(out_b, ref, f"separate step {t}")
    torch.cuda.synchronize()
    sa, sb = a.stats(), b.stats()
    assert (sa.pos, sa.stored, sa.device_status) == (sb.pos, sb.stored, sb.device_status)
    assert (sa.pos, sa.stored) == (oc.pos, oc.stored)
    assert_cache_equal(a, oc, "fused cache")
    assert_cache_equal(b, oc, "separate-call cache")
    return worst


@pytest.mark.parametrize("pair", PAIRS, ids=lambda p: f"{p[0]}{p[1]}-{p[3]}{p[4]}")
@pytest.mark.parametrize("G", [3, 8])
def test_linear_steps(kvq, pair, G):
    _run(kvq, pair, 2, 2, 128, G, cap=400, T0=300, steps=4, seed=G)


@pytest.mark.parametrize("pair", [PAIRS[0], PAIRS[2], PAIRS[4], PAIRS[5]], ids=["fp16", "kivi4", "aff4", "q40v8"])
def test_head_dim_64_and_fp16_io(kvq, pair):
    _run(kvq, pair, 1, 4, 64, 2, cap=200, T0=129, steps=3, dtype=torch.float16, seed=5)


@pytest.mark.parametrize("pair", [PAIRS[2], PAIRS[4], PAIRS[6]], ids=["kivi4", "aff4", "q40v4"])
def test_ring_filling_then_wrapping(kvq, pair):
    # sink 4 + window 128: the ring fills during the steps, then every step
    # overwrites the oldest window slot (which the attention must leave out)
    _run(kvq, pair, 1, 2, 128, 4, cap=132, T0=100, steps=70, layout="ring", sink=4, window=128, seed=9)


def test_ring_full_many_wraps(kvq):
    pair = ("kivi_chan", 4, 0, "affine_token", 4, 32)
    _run(kvq, pair, 2, 1, 128, 3, cap=68, T0=68, steps=150, layout="ring", sink=4, window=64, seed=11)


def test_compact_layout_runs_the_separate_steps(kvq):
    pair = ("kivi_chan", 8, 0, "affine_token", 8, 128)
    _run(kvq, pair, 1, 2, 128, 2, cap=133, T0=130, steps=6, layout="compact", sink=4, window=128, seed=13)


def test_fp32_io_runs_the_separate_steps(kvq):
    pair = ("kivi_chan", 8, 0, "affine_token", 8, 32)
    _run(kvq, pair, 1, 8, 32, 1, cap=300, T0=260, steps=3, dtype=torch.float32, seed=15)


@pytest.mark.parametrize("pair", [PAIRS[4], PAIRS[5]], ids=["aff4", "q40v8"])
def test_empty_cache_first_step(kvq, pair):
    # the first token only: the output is that token's dequantised value
    _run(kvq, pair, 1, 2, 128, 3, cap=64, T0=0, steps=2, seed=17)


def test_long_cache_one_wave_shape(kvq):
    # the 8K mlx layer's launch shape (8 kv heads, sixteen-warp CTAs)
    pair = ("affine_token", 4, 64, "affine_token", 4, 64)
    _run(kvq, pair, 1, 8, 128, 3, cap=8192 + 64, T0=8192 + 30, steps=3, seed=19)


def test_full_linear_cache_reports_overflow(kvq):
    pair = ("affine_token", 4, 64, "affine_token", 4, 64)
    a, b, oc = _pair_caches(kvq, pair, 1, 2, 128, 64, "linear", 0, 0, None)
    g = torch.Generator().manual_seed(21)
    k0 = _rand((1, 2, 64, 128), g, torch.bfloat16)
    a.append(k0.cuda(), k0.cuda())
    oc.append(host(k0), host(k0))
    before = a.buf.clone()
    q = _rand((1, 6, 128), g, torch.bfloat16)
    k1 = _rand((1, 2, 1, 128), g, torch.bfloat16)
    out = a.append_decode(k1.cuda(), k1.cuda(), q.cuda())
    st = a.stats()
    assert st.device_status == kvq.DEV_OVERFLOW and st.stored == 64 and st.pos == 64
    lay = a.layout
    assert torch.equal(a.buf[lay.k_codes:], before[lay.k_codes:]), "an overflowing step wrote the cache"
    kh, vh = oc.dequant()
    assert_attention_close(out, oatt.decode_attention(host(q), kh, vh), "overflow: the stored rows only")


@pytest.mark.parametrize("pair", [PAIRS[4], PAIRS[5], PAIRS[2]], ids=["aff4", "q40v8", "kivi4"])
def test_layers_in_turn_with_early_read(kvq, pair):
    # Two layers' caches stepped in turn with KVQ_STEP_EARLY_READ (the kernel
    # before each call is the other layer's step, which never writes this
    # cache): the counters and stored rows are read before the dependency
    # wait, and every step must still match the oracle.
    B, H, D, G, T0, steps = 1, 8, 128, 3, 1500, 5
    g = torch.Generator().manual_seed(23)
    layers = []
    for li in range(2):
        bias = _rand((H, D), g, torch.float32, 1.5) if pair[0] == "q4_0" else None
        off = bias[None, :, None, :] if bias is not None else _rand((1, H, 1, D), g, torch.float32, 2.0)
        a, _, oc = _pair_caches(kvq, pair, B, H, D, 2048, "linear", 0, 0, bias)
        k0 = _rand((B, H, T0, D), g, torch.bfloat16, 1.0, off)
        v0 = _rand((B, H, T0, D), g, torch.bfloat16)
        calib = pair[0] == "kivi_chan"
        a.append(k0.cuda(), v0.cuda(), calibrate_k=calib)
        if calib:
            oc.calibrate_k(host(k0))
        oc.append(host(k0), host(v0))
        layers.append((a, oc, off))
    for t in range(steps):
        for a, oc, off in layers:
            k1 = _rand((B, H, 1, D), g, torch.bfloat16, 1.0, off)
            v1 = _rand((B, H, 1, D), g, torch.bfloat16)
            q = _rand((B, H * G, D), g, torch.bfloat16)
            out = a.append_decode(k1.cuda(), v1.cuda(), q.cuda(), early_read=True)
            oc.append(host(k1), host(v1))
            kh, vh = oc.dequant()
            assert_attention_close(out, oatt.decode_attention(host(q), kh, vh), f"early-read step {t}")
    for a, oc, _ in layers:
        assert_cache_equal(a, oc, "early-read cache")


@pytest.mark.parametrize("pair", [PAIRS[4], PAIRS[6]], ids=["aff4", "q40v4"])
def test_layer_step_one_call_matches_per_layer_calls(kvq, pair):
    # kvq_append_decode_layers over four layers: the same outputs and cache
    # bytes as four kvq_append_decode calls, and the oracle's attention.
    B, H, D, G, T0, L, steps = 1, 8, 128, 3, 700, 4, 3
    g = torch.Generator().manual_seed(31)
    one, per, ocs, offs = [], [], [], []
    for _ in range(L):
        bias = _rand((H, D), g, torch.float32, 1.5) if pair[0] == "q4_0" else None
        off = bias[None, :, None, :] if bias is not None else _rand((1, H, 1, D), g, torch.float32, 2.0)
        a, b, oc = _pair_caches(kvq, pair, B, H, D, 1024, "linear", 0, 0, bias)
        k0 = _rand((B, H, T0, D), g, torch.bfloat16, 1.0, off)
        v0 = _rand((B, H, T0, D), g, torch.bfloat16)
        for c in (a, b):
            c.append(k0.cuda(), v0.cuda())
        oc.append(host(k0), host(v0))
        one.append(a), per.append(b), ocs.append(oc), offs.append(off)
    ks = [torch.empty(B, H, 1, D, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    vs = [torch.empty_like(k) for k in ks]
    qs = [torch.empty(B, H * G, D, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    outs = [torch.empty_like(q) for q in qs]
    step = kvq.LayerStep(one, ks, vs, qs, outs)
    for t in range(steps):
        inputs = []
        for li in range(L):
            k1 = _rand((B, H, 1, D), g, torch.bfloat16, 1.0, offs[li])
            v1 = _rand((B, H, 1, D), g, torch.bfloat16)
            q = _rand((B, H * G, D), g, torch.bfloat16)
            ks[li].copy_(k1), vs[li].copy_(v1), qs[li].copy_(q)
            inputs.append((k1, v1, q))
        step.run()
        assert step.launches == L
        for li, (k1, v1, q) in enumerate(inputs):
            ref_out = per[li].append_decode(k1.cuda(), v1.cuda(), q.cuda())
            assert torch.equal(outs[li], ref_out), f"layer {li} step {t}: one call differs from per-layer calls"
            ocs[li].append(host(k1), host(v1))
            kh, vh = ocs[li].dequant()
            assert_attention_close(outs[li], oatt.decode_attention(host(q), kh, vh), f"layer {li} step {t}")
    for a, b, oc in zip(one, per, ocs):
        assert_cache_equal(a, oc, "one-call cache")
        assert_cache_equal(b, oc, "per-layer cache")


def test_layer_step_rejects_a_shared_cache(kvq):
    c = kvq.KVCache(1, 2, 64, 64, "affine_token", 4, 64, "affine_token", 4, 64)
    k = torch.zeros(1, 2, 1, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(1, 2, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(kvq.KvqError, match="share one cache"):
        kvq.kvq_append_decode_layers([c.handle, c.handle], [k, k], [k, k], kvq.DTYPES[k.dtype], [q, q], [out, out],
                                     2, kvq.DTYPES[q.dtype])
    assert c.stats().pos == 0
    step = kvq.LayerStep([c], [k], [k], [q], [out])
    c.reset()
    with pytest.raises(ValueError, match="reset or released"):
        step.run()
