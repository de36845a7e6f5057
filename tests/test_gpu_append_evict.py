"""GPU parity: quantise-on-append and eviction, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from kvq_helpers import assert_cache_equal, gpu_planes, host, oracle_spec
from oracle.cache import OracleCache

pytestmark = pytest.mark.gpu

FORMATS = [
    # (k_format, k_bits, k_group, v_format, v_bits, v_group)
    ("fp16", 16, 0, "fp16", 16, 0),
    ("kivi_chan", 8, 0, "affine_token", 8, 128),
    ("kivi_chan", 4, 0, "affine_token", 4, 32),
    ("affine_token", 8, 64, "affine_token", 8, 64),
    ("affine_token", 4, 64, "affine_token", 4, 64),
    ("affine_token", 4, 16, "affine_token", 8, 32),
    ("q4_0", 4, 32, "affine_token", 8, 128),
    ("q4_0", 4, 32, "affine_token", 4, 32),
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


def _clip(D, group):
    return min(group, D) if group else group


@pytest.mark.parametrize("fmt", FORMATS, ids=lambda f: f"{f[0]}{f[1]}-{f[3]}{f[4]}g{f[5]}")
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16])
def test_append_bit_exact(kvq, fmt, D, dtype):
    kf, kb, kg, vf, vb, vg = fmt
    kg, vg = _clip(D, kg), _clip(D, vg)
    B, H, cap = 2, 3, 90
    bias = None
    if kf == "q4_0":
        bias = (torch.randn(H, D, generator=torch.Generator().manual_seed(D)) * 1.5).float()
    cache = kvq.KVCache(B, H, D, cap, kf, kb, kg, vf, vb, vg, k_bias=None if bias is None else bias.cuda())
    oc = OracleCache(oracle_spec(cache, None if bias is None else bias.numpy()))
    k = _inputs((B, H, 67, D), 1, dtype)
    v = _inputs((B, H, 67, D), 2, dtype, 0.0)
    calibrate = kf == "kivi_chan"
    cache.append(k.cuda(), v.cuda(), calibrate_k=calibrate)
    if calibrate:
        oc.calibrate_k(host(k))
    oc.append(host(k), host(v))
    assert_cache_equal(cache, oc, "bulk append")
    for step, n in enumerate((1, 1, 5, 16)):
        k2 = _inputs((B, H, n, D), 10 + step, dtype) * 1.5     # frozen K scales clamp some of these
        v2 = _inputs((B, H, n, D), 20 + step, dtype, 0.0)
        cache.append(k2.cuda(), v2.cuda())
        oc.append(host(k2), host(v2))
    assert_cache_equal(cache, oc, "decode appends")


def test_zero_bias_is_byte_identical_to_no_bias(kvq):
    # disabled centering is a no-op: no bias and an all-zero bias give the same bytes
    B, H, D = 1, 2, 128
    k = _inputs((B, H, 40, D), 3, torch.bfloat16)
    a = kvq.KVCache(B, H, D, 64, "q4_0", 4, 32, "affine_token", 8, 128)
    b = kvq.KVCache(B, H, D, 64, "q4_0", 4, 32, "affine_token", 8, 128, k_bias=torch.zeros(H, D, device="cuda"))
    a.append(k.cuda(), k.cuda())
    b.append(k.cuda(), k.cuda())
    pa, pb = gpu_planes(a), gpu_planes(b)
    # rows past the 40 stored ones were never written and hold whatever the buffer held
    np.testing.assert_array_equal(pa["k_rows"][:, :, :40], pb["k_rows"][:, :, :40])
    np.testing.assert_array_equal(pa["k_tok_scale"][:, :, :40].view(np.uint16),
                                  pb["k_tok_scale"][:, :, :40].view(np.uint16))


def test_constant_and_zero_rows(kvq):
    B, H, D = 1, 1, 64
    k = torch.zeros(B, H, 8, D)
    k[0, 0, 3] = 0.25
    k[0, 0, 5, :32] = 1.0
    for kf, kb, kg in (("affine_token", 4, 64), ("q4_0", 4, 32)):
        cache = kvq.KVCache(B, H, D, 16, kf, kb, kg, "affine_token", 8, 64)
        oc = OracleCache(oracle_spec(cache))
        cache.append(k.cuda(), k.cuda())
        oc.append(k.numpy(), k.numpy())
        assert_cache_equal(cache, oc, kf)


def test_overflow_sets_status_and_writes_nothing(kvq):
    cache = kvq.KVCache(1, 2, 64, 10, "affine_token", 8, 64, "affine_token", 8, 64)
    k = _inputs((1, 2, 8, 64), 4, torch.bfloat16)
    cache.append(k.cuda(), k.cuda())
    before = gpu_planes(cache)
    k2 = _inputs((1, 2, 3, 64), 5, torch.bfloat16)
    cache.append(k2.cuda(), k2.cuda())
    after = gpu_planes(cache)
    assert after["status"] == kvq.DEV_OVERFLOW
    assert after["stored"] == 8 and after["pos"] == 8
    np.testing.assert_array_equal(before["k_rows"], after["k_rows"])
    st = cache.stats()
    assert st.device_status == kvq.DEV_OVERFLOW
    kvq.kvq_clear_status(cache.handle)
    assert cache.stats().device_status == 0


@pytest.mark.parametrize("fmt", [FORMATS[2], FORMATS[4], FORMATS[6]], ids=["kivi4", "aff4", "q40-int8"])
def test_bulk_append_many_chunks_per_cta(kvq, fmt):
    """A prefill long enough that every CTA of the staged bulk append cycles its
    shared-memory stages several times, with a ragged last chunk per (b, kv head)."""
    kf, kb, kg, vf, vb, vg = fmt
    B, H, D, n = 4, 8, 128, 4096 + 17
    bias = None
    if kf == "q4_0":
        bias = (torch.randn(H, D, generator=torch.Generator().manual_seed(41)) * 1.5).float()
    cache = kvq.KVCache(B, H, D, n + 8, kf, kb, kg, vf, vb, vg, k_bias=None if bias is None else bias.cuda())
    oc = OracleCache(oracle_spec(cache, None if bias is None else bias.numpy()))
    k = _inputs((B, H, n, D), 42, torch.bfloat16)
    v = _inputs((B, H, n, D), 43, torch.bfloat16, 0.0)
    calibrate = kf == "kivi_chan"
    cache.append(k.cuda(), v.cuda(), calibrate_k=calibrate)
    if calibrate:
        oc.calibrate_k(host(k))
    oc.append(host(k), host(v))
    assert_cache_equal(cache, oc, "bulk append, many chunks per CTA")


@pytest.mark.parametrize("fmt", [FORMATS[2], FORMATS[6]], ids=["kivi4", "q40-int8"])
def test_misaligned_input_takes_the_per_row_kernel_with_the_same_bytes(kvq, fmt):
    """Inputs that do not start on a 16-byte boundary cannot be staged by bulk copies or
    read as 16-byte vectors; the append (and the KIVI calibration) read them element by
    element instead, to the same bytes."""
    kf, kb, kg, vf, vb, vg = fmt
    B, H, D, n = 2, 4, 128, 300
    k = _inputs((B, H, n, D), 44, torch.bfloat16).cuda()
    v = _inputs((B, H, n, D), 45, torch.bfloat16, 0.0).cuda()
    shifted = []
    for x in (k, v):
        flat = torch.empty(x.numel() + 4, dtype=x.dtype, device="cuda")
        y = flat[4:].view(x.shape)
        y.copy_(x)
        assert y.data_ptr() % 16 == 8
        shifted.append(y)
    bias = None
    if kf == "q4_0":
        bias = (torch.randn(H, D, generator=torch.Generator().manual_seed(46)) * 1.5).float().cuda()
    a = kvq.KVCache(B, H, D, n + 8, kf, kb, kg, vf, vb, vg, k_bias=bias)
    b = kvq.KVCache(B, H, D, n + 8, kf, kb, kg, vf, vb, vg, k_bias=bias)
    calibrate = kf == "kivi_chan"
    a.append(k, v, calibrate_k=calibrate)
    b.append(*shifted, calibrate_k=calibrate)
    pa, pb = gpu_planes(a), gpu_planes(b)
    assert pa["stored"] == pb["stored"] == n
    for name in ("k_rows", "v_rows"):
        np.testing.assert_array_equal(pa[name][:, :, :n], pb[name][:, :, :n])
    for name in ("k_tok_scale", "v_tok_scale", "v_tok_zero"):
        if name in pa:
            np.testing.assert_array_equal(pa[name][:, :, :n].view(np.uint16), pb[name][:, :, :n].view(np.uint16))
    for name in ("k_ch_scale32", "k_ch_zero32"):
        if name in pa:
            np.testing.assert_array_equal(pa[name], pb[name])


def test_bulk_append_overflow_writes_nothing(kvq):
    cache = kvq.KVCache(1, 2, 128, 40, "affine_token", 4, 64, "affine_token", 4, 64)
    k = _inputs((1, 2, 8, 128), 47, torch.bfloat16)
    cache.append(k.cuda(), k.cuda())
    before = gpu_planes(cache)
    big = _inputs((1, 2, 33, 128), 48, torch.bfloat16)    # a whole bulk chunk and more, past the capacity
    cache.append(big.cuda(), big.cuda())
    after = gpu_planes(cache)
    assert after["status"] == kvq.DEV_OVERFLOW
    assert after["stored"] == 8 and after["pos"] == 8
    np.testing.assert_array_equal(before["k_rows"], after["k_rows"])
    np.testing.assert_array_equal(before["v_rows"], after["v_rows"])
    kvq.kvq_clear_status(cache.handle)


def test_uncalibrated_kivi_append_rejected(kvq):
    cache = kvq.KVCache(1, 1, 32, 16, "kivi_chan", 8, 0, "affine_token", 8, 32)
    k = torch.randn(1, 1, 2, 32, device="cuda")
    with pytest.raises(kvq.KvqError):
        cache.append(k, k)


@pytest.mark.parametrize("layout,n_steps", [("compact", 1), ("compact", 195), ("compact", 197), ("compact", 236),
                                            ("ring", 197), ("ring", 636)])
def test_streaming_decode_matches_oracle(kvq, layout, n_steps):
    # KIVI int8, sink 4 + window 256: the per-channel K scales calibrated over
    # a 64-token fill (so later keys code to interior levels, not only to the
    # clamps), then one append + one evict per step; 64 + n_steps tokens in all
    # cover the cache before, at and past sink + window = 260
    sink, window, D, B, H, n0 = 4, 256, 32, 1, 2, 64
    cap = sink + window + (1 if layout == "compact" else 0)
    cache = kvq.KVCache(B, H, D, cap, "kivi_chan", 8, 0, "affine_token", 8, 32, layout=layout, sink=sink,
                        window=window)
    oc = OracleCache(oracle_spec(cache))
    fill = _inputs((B, H, n0, D), 7, torch.float32)
    cache.append(fill.cuda(), fill.cuda(), calibrate_k=True)
    cache.evict_middle()
    oc.calibrate_k(host(fill))
    oc.append(host(fill), host(fill))
    oc.evict_middle()
    g = torch.Generator().manual_seed(8)
    # later keys from the fill's distribution (its channel offsets), so most codes are interior
    off = fill.float().mean(dim=2, keepdim=True)
    ks = torch.randn(n_steps, B, H, 1, D, generator=g) + off
    vs = torch.randn(n_steps, B, H, 1, D, generator=g)
    ksd, vsd = ks.cuda(), vs.cuda()
    for t in range(n_steps):
        cache.append(ksd[t], vsd[t])
        cache.evict_middle()
        oc.append(ks[t].numpy(), vs[t].numpy())
        oc.evict_middle()
    assert_cache_equal(cache, oc, f"{layout} after {n0 + n_steps} tokens")
    assert oc.stored == min(n0 + n_steps, sink + window)
    u = oc.k.codes(oc.stored).astype(np.int64)
    assert ((u > 0) & (u < 255)).mean() > 0.9, "most key codes should be interior levels"


def test_ring_forty_thousand_steps(kvq):
    # The long streaming run of the ring workload on a reduced instance (B 1,
    # 2 kv heads, sink 4 + window 256): a 260-token calibrated fill, then
    # 40 000 single-token appends (graph replays of 1 000 each).  The final
    # cache equals the oracle's, whose state after any number of steps is a
    # function of the surviving tokens and their positions (the ring appends
    # of one call and of many give the same cache): 260 rows, positions 0..3
    # and the last 256.
    sink, window, D, B, H, n0, N = 4, 256, 128, 1, 2, 260, 40000
    chunk = 1000
    cache = kvq.KVCache(B, H, D, sink + window, "kivi_chan", 4, 0, "affine_token", 4, 32, layout="ring", sink=sink,
                        window=window)
    oc = OracleCache(oracle_spec(cache))
    fill_k = _inputs((B, H, n0, D), 41, torch.bfloat16)
    fill_v = _inputs((B, H, n0, D), 42, torch.bfloat16, 0.0)
    cache.append(fill_k.cuda(), fill_v.cuda(), calibrate_k=True)
    oc.calibrate_k(host(fill_k))
    oc.append(host(fill_k), host(fill_v))
    g = torch.Generator().manual_seed(43)
    off = fill_k.float().mean(dim=2, keepdim=True)
    ks = (torch.randn(B, H, N, D, generator=g) + off).to(torch.bfloat16)
    vs = torch.randn(B, H, N, D, generator=g).to(torch.bfloat16)
    ksd, vsd = ks.cuda(), vs.cuda()
    stage_k = torch.empty(chunk, B, H, 1, D, dtype=torch.bfloat16, device="cuda")
    stage_v = torch.empty_like(stage_k)
    cache.append(stage_k[0].zero_(), stage_v[0].zero_())   # loads the kernel before capture
    cache.reset()
    cache.append(fill_k.cuda(), fill_v.cuda(), calibrate_k=True)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(chunk):
            cache.append(stage_k[i], stage_v[i])
            cache.evict_middle()
    for c0 in range(0, N, chunk):
        stage_k.copy_(ksd[:, :, c0:c0 + chunk].permute(2, 0, 1, 3).unsqueeze(3))
        stage_v.copy_(vsd[:, :, c0:c0 + chunk].permute(2, 0, 1, 3).unsqueeze(3))
        graph.replay()
    torch.cuda.synchronize()
    st = cache.stats()
    assert (st.pos, st.stored, st.device_status) == (n0 + N, sink + window, 0)
    oc.append(host(ks), host(vs))
    assert_cache_equal(cache, oc, "ring after 40 000 steps")
    q = torch.randn(B, 3 * H, D, generator=g).to(torch.bfloat16)
    kh, vh = oc.dequant()
    from oracle import attention as oatt
    from kvq_helpers import assert_attention_close
    assert_attention_close(cache.decode_attn(q.cuda()), oatt.decode_attention(host(q), kh, vh), "after 40 000 steps")


def test_ring_bulk_append_longer_than_window(kvq):
    sink, window, D = 4, 64, 128
    cache = kvq.KVCache(2, 2, D, sink + window, "kivi_chan", 4, 0, "affine_token", 4, 32, layout="ring", sink=sink,
                        window=window)
    oc = OracleCache(oracle_spec(cache))
    k = _inputs((2, 2, 200, D), 9, torch.bfloat16)
    v = _inputs((2, 2, 200, D), 10, torch.bfloat16, 0.0)
    cache.append(k.cuda(), v.cuda(), calibrate_k=True)
    oc.calibrate_k(host(k))
    oc.append(host(k), host(v))
    assert_cache_equal(cache, oc, "ring bulk")


@pytest.mark.parametrize("fmt", [FORMATS[0], FORMATS[4], FORMATS[6]], ids=["fp16", "aff4", "q40"])
def test_keepset_gather(kvq, fmt):
    kf, kb, kg, vf, vb, vg = fmt
    B, H, D, S, n_keep = 2, 3, 128, 700, 130
    cache = kvq.KVCache(B, H, D, S + 8, kf, kb, kg, vf, vb, vg)
    oc = OracleCache(oracle_spec(cache))
    k = _inputs((B, H, S, D), 11, torch.float16)
    v = _inputs((B, H, S, D), 12, torch.float16, 0.0)
    cache.append(k.cuda(), v.cuda())
    oc.append(host(k), host(v))
    rng = np.random.default_rng(3)
    idx = np.stack([np.stack([np.sort(rng.choice(S, n_keep, replace=False)) for _ in range(H)]) for _ in range(B)])
    idx[0, 0, :4] = np.arange(4)
    idx = idx.astype(np.int32)
    cache.evict_keepset(torch.from_numpy(idx).cuda())
    oc.evict_keepset(idx)
    assert_cache_equal(cache, oc, "keep-set")
    t = _inputs((B, H, 1, D), 13, torch.float16)
    cache.append(t.cuda(), t.cuda())
    oc.append(host(t), host(t))
    assert_cache_equal(cache, oc, "append after keep-set")
    assert cache.stats().pos == S + 1


def test_bad_keepset_sets_status(kvq):
    cache = kvq.KVCache(1, 1, 64, 40, "fp16", 16, 0, "fp16", 16, 0)
    k = torch.randn(1, 1, 20, 64, dtype=torch.float16, device="cuda")
    cache.append(k, k)
    idx = torch.tensor([[[0, 5, 5, 9]]], dtype=torch.int32, device="cuda")     # not strictly ascending
    cache.evict_keepset(idx)
    assert gpu_planes(cache)["status"] == kvq.DEV_BAD_KEEPSET


@pytest.mark.parametrize("fmt", FORMATS, ids=lambda f: f"{f[0]}{f[1]}-{f[3]}{f[4]}g{f[5]}")
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_convert_from_dense_cache(kvq, fmt, dtype):
    """kvq_convert codes the first T tokens of a dense [B, Hkv, C, D] cache exactly as an
    append of those tokens would; rows past T (huge values here) are never read."""
    kf, kb, kg, vf, vb, vg = fmt
    D, B, H, C, T = 128, 2, 3, 300, 233
    kg, vg = _clip(D, kg), _clip(D, vg)
    bias = None
    if kf == "q4_0":
        bias = (torch.randn(H, D, generator=torch.Generator().manual_seed(5)) * 1.5).float()
    k = _inputs((B, H, C, D), 31, dtype)
    v = _inputs((B, H, C, D), 32, dtype, 0.0)
    k[:, :, T:] = 3.0e4
    v[:, :, T:] = -3.0e4
    cache = kvq.KVCache(B, H, D, T + 8, kf, kb, kg, vf, vb, vg, k_bias=None if bias is None else bias.cuda())
    oc = OracleCache(oracle_spec(cache, None if bias is None else bias.numpy()))
    calibrate = kf == "kivi_chan"
    cache.convert(k.cuda(), v.cuda(), T, calibrate_k=calibrate)
    kt, vt = k[:, :, :T].contiguous(), v[:, :, :T].contiguous()
    if calibrate:
        oc.calibrate_k(host(kt))
    oc.append(host(kt), host(vt))
    assert_cache_equal(cache, oc, "convert")
    # the converted cache keeps appending like any other
    k2, v2 = _inputs((B, H, 3, D), 33, dtype), _inputs((B, H, 3, D), 34, dtype, 0.0)
    cache.append(k2.cuda(), v2.cuda())
    oc.append(host(k2), host(v2))
    assert_cache_equal(cache, oc, "append after convert")


def test_convert_rejects_short_stride(kvq):
    cache = kvq.KVCache(1, 2, 64, 32, "affine_token", 8, 64, "affine_token", 8, 64)
    k = torch.zeros((1, 2, 10, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KvqError):
        kvq.kvq_convert(cache.handle, k, k, 8, 10, kvq.DTYPES[torch.float16])


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("layout", ["linear", "compact"])
@pytest.mark.parametrize("D", [64, 128])
def test_recompute_k_on_append_bit_exact(kvq, bits, layout, D):
    """KVQ_APPEND_RECOMPUTE_K: every append recomputes the per-channel K range over the stored
    (dequantised) and new keys and codes the whole block again; bit-exact against the oracle,
    through evictions, and decode attention over the result matches."""
    from kvq_helpers import assert_attention_close
    from oracle import attention as oatt

    B, H = 2, 2
    sink, window = (4, 48) if layout == "compact" else (0, 0)
    cap = 120 if layout == "linear" else sink + window + 8
    cache = kvq.KVCache(B, H, D, cap, "kivi_chan", bits, 0, "affine_token", bits, D, layout=layout, sink=sink,
                        window=window)
    oc = OracleCache(oracle_spec(cache, None))
    steps = [20, 1, 3, 1, 8, 1, 1] if layout == "linear" else [30, 8, 8, 8, 5, 1, 7]
    for i, n in enumerate(steps):
        k = _inputs((B, H, n, D), 70 + i, torch.bfloat16) * (1.0 + 0.4 * i)   # later tokens widen the range
        v = _inputs((B, H, n, D), 90 + i, torch.bfloat16, 0.0)
        cache.append(k.cuda(), v.cuda(), recompute_k=True)
        oc.append_recompute_k(host(k), host(v))
        if layout == "compact":
            cache.evict_middle()
            oc.evict_middle()
        assert_cache_equal(cache, oc, f"step {i}")
    q = torch.randn((B, 3 * H, D), generator=torch.Generator().manual_seed(99)).to(torch.bfloat16)
    out = cache.decode_attn(q.cuda())
    kh, vh = oc.dequant()
    assert_attention_close(out, oatt.decode_attention(host(q), kh, vh), "decode after recompute appends")


def test_recompute_k_flag_gates(kvq):
    x = torch.zeros((1, 1, 2, 64), dtype=torch.bfloat16, device="cuda")
    ring = kvq.KVCache(1, 1, 64, 36, "kivi_chan", 8, 0, "affine_token", 8, 64, layout="ring", sink=4, window=32)
    with pytest.raises(kvq.KvqError):
        ring.append(x, x, recompute_k=True)
    aff = kvq.KVCache(1, 1, 64, 36, "affine_token", 8, 64, "affine_token", 8, 64)
    with pytest.raises(kvq.KvqError):
        aff.append(x, x, recompute_k=True)
    kiv = kvq.KVCache(1, 1, 64, 36, "kivi_chan", 8, 0, "affine_token", 8, 64)
    with pytest.raises(kvq.KvqError):
        kiv.append(x, x, calibrate_k=True, recompute_k=True)
