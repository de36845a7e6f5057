"""Pins of the oracle's cache model: StreamingLLM cap, ring vs compact, keep-set, gates, bytes."""
import numpy as np
import pytest

from oracle import accounting as acc
from oracle import attention as att
from oracle import quantize as qz
from oracle.cache import CacheSpec, OracleCache, ring_slot, streaming_survivors


def _pos_tokens(positions, D=32):
    """fp32 K/V rows [1,1,n,D] that carry their own absolute position exactly in fp16."""
    p = np.asarray(positions, np.float32)
    x = np.zeros((1, 1, len(p), D), np.float32)
    x[0, 0, :, 0] = np.floor(p / 1024)
    x[0, 0, :, 1] = p % 1024
    return x


def _positions_of(cache):
    kh, _ = cache.dequant()
    return (kh[0, 0, :, 0] * 1024 + kh[0, 0, :, 1]).astype(np.int64)


def _streaming_cache(layout, sink, window):
    cap = sink + window + (1 if layout == "compact" else 0)
    return OracleCache(CacheSpec(batch=1, n_kv_heads=1, head_dim=32, capacity=cap, layout=layout,
                                 sink=sink, window=window))


def _decode(cache, n_steps, start=0):
    for p in range(start, start + n_steps):
        t = _pos_tokens([p])
        cache.append(t, t)
        cache.evict_middle()


@pytest.mark.parametrize("n", [1, 259, 260, 261, 500])
def test_streaming_cap_page_example(golden, n):
    g = golden("streaming_kivi_page.json")["streaming_cap"]
    sink, window = g["sink"], g["window"]
    for layout in ("compact", "ring"):
        c = _streaming_cache(layout, sink, window)
        _decode(c, n)
        assert c.stored == min(n, g["stored"])
        assert c.pos == n
        got = sorted(_positions_of(c).tolist())
        assert got == streaming_survivors(n, sink, window)
    if n == g["tokens_generated"]:
        assert c.stored == g["stored"]


def test_streaming_closed_form_survivors():
    assert streaming_survivors(3, 4, 256) == [0, 1, 2]
    s = streaming_survivors(40000, 4, 256)
    assert s[:4] == [0, 1, 2, 3] and s[4:] == list(range(40000 - 256, 40000)) and len(s) == 260


def test_compact_keeps_logical_order_and_ring_keeps_slots():
    c = _streaming_cache("compact", 4, 16)
    r = _streaming_cache("ring", 4, 16)
    _decode(c, 100)
    _decode(r, 100)
    # compact: concatenation in logical order
    assert _positions_of(c).tolist() == streaming_survivors(100, 4, 16)
    # ring: each survivor sits in its closed-form slot
    got = _positions_of(r)
    for slot, p in enumerate(got.tolist()):
        assert ring_slot(p, 4, 16) == slot


@pytest.mark.slow
def test_long_run_simulation_equals_closed_form():
    # 40 000 single-token steps with one eviction each (reduced instance).
    r = _streaming_cache("ring", 4, 4096)
    _decode(r, 40000)
    assert sorted(_positions_of(r).tolist()) == streaming_survivors(40000, 4, 4096)
    c = _streaming_cache("compact", 4, 256)
    _decode(c, 40000)
    assert _positions_of(c).tolist() == streaming_survivors(40000, 4, 256)


def test_ring_bulk_append_equals_sequential():
    a = _streaming_cache("ring", 4, 16)
    b = _streaming_cache("ring", 4, 16)
    t = _pos_tokens(range(0, 57))
    a.append(t, t)
    _decode(b, 57)
    np.testing.assert_array_equal(a.k.rows[:, :, :a.stored], b.k.rows[:, :, :b.stored])
    assert a.stored == b.stored == 20 and a.pos == b.pos == 57


def test_evict_moves_per_token_metadata_not_channel_scales():
    rng = np.random.default_rng(4)
    spec = CacheSpec(batch=2, n_kv_heads=2, head_dim=32, capacity=4 + 8 + 1, layout="compact", sink=4, window=8,
                     k_format="kivi_chan", k_bits=8, v_format="affine_token", v_bits=8, v_group=32)
    c = OracleCache(spec)
    fill_k = rng.standard_normal((2, 2, 12, 32)).astype(np.float32)
    fill_v = rng.standard_normal((2, 2, 12, 32)).astype(np.float32)
    c.calibrate_k(fill_k)
    c.append(fill_k, fill_v)
    ch_s, ch_z = c.k.ch_scale.copy(), c.k.ch_zero.copy()
    vs_before = c.v.tok_scale[:, :, :12].copy()
    k_new = rng.standard_normal((2, 2, 1, 32)).astype(np.float32)
    c.append(k_new, k_new)
    c.evict_middle()
    assert c.stored == 12
    np.testing.assert_array_equal(c.k.ch_scale, ch_s)
    np.testing.assert_array_equal(c.k.ch_zero, ch_z)
    # rows [0,4) unchanged, rows [4,11) were rows [5,12), row 11 is the new token
    np.testing.assert_array_equal(c.v.tok_scale[:, :, :4], vs_before[:, :, :4])
    np.testing.assert_array_equal(c.v.tok_scale[:, :, 4:11], vs_before[:, :, 5:12])


def test_keepset_gather_and_true_offset():
    rng = np.random.default_rng(8)
    S = 40
    spec = CacheSpec(batch=1, n_kv_heads=2, head_dim=32, capacity=S + 5)
    c = OracleCache(spec)
    k = rng.standard_normal((1, 2, S, 32)).astype(np.float16).astype(np.float32)
    c.append(k, k)
    idx = np.stack([np.sort(rng.choice(S, 10, replace=False)) for _ in range(2)])[None].astype(np.int32)
    before = c.k.rows[:, :, :S].copy()
    c.evict_keepset(idx)
    assert c.stored == 10 and c.pos == S
    for h in range(2):
        np.testing.assert_array_equal(c.k.rows[0, h, :10], before[0, h, idx[0, h]])
    # decode after the keep-set appends at the true position and never evicts
    t = rng.standard_normal((1, 2, 1, 32)).astype(np.float32)
    c.append(t, t)
    assert c.stored == 11 and c.pos == S + 1


def test_bias_gate_and_disabled_centering_is_a_no_op():
    rng = np.random.default_rng(12)
    with pytest.raises(ValueError):
        OracleCache(CacheSpec(batch=1, n_kv_heads=2, head_dim=32, capacity=4, k_format="affine_token",
                              k_bits=4, k_group=32, k_bias=np.zeros((2, 32), np.float32)))
    k = (rng.standard_normal((1, 2, 6, 64)) * 3).astype(np.float32)
    base = dict(batch=1, n_kv_heads=2, head_dim=64, capacity=8, k_format="q4_0", k_bits=4, k_group=32)
    a = OracleCache(CacheSpec(**base))
    b = OracleCache(CacheSpec(**base, k_bias=np.zeros((2, 64), np.float32)))
    a.append(k, k)
    b.append(k, k)
    np.testing.assert_array_equal(a.k.rows, b.k.rows)
    np.testing.assert_array_equal(a.k.tok_scale.view(np.uint16), b.k.tok_scale.view(np.uint16))
    u, d = qz.q4_0_quantize(k)
    np.testing.assert_array_equal(a.k.rows[:, :, :6], qz.pack_nibbles(u))


def test_mean_centering_softmax_invariance(golden):
    # "kv-cache ... mean-centering for Q4_0", "Why this is safe": subtracting
    # the same kbar from every key adds q . kbar to every logit of a row; the
    # softmax does not see it.  Checked on an unquantised fp32 K cache.
    bound = golden("mean_center_page.json")["invariance"]["nmse_bound_used"]
    rng = np.random.default_rng(13)
    B, Hkv, G, T, D = 2, 4, 3, 300, 64
    k = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    kbar = (rng.standard_normal((Hkv, D)) * 1.5).astype(np.float32)
    k = k + kbar[None, :, None, :]
    v = rng.standard_normal((B, Hkv, T, D))
    q = rng.standard_normal((B, Hkv * G, D))
    o_ref = att.decode_attention(q, k, v)
    o_c = att.decode_attention(q, qz.mean_center(k, kbar), v)
    nmse = np.sum((o_c - o_ref) ** 2) / np.sum(o_ref ** 2)
    assert nmse <= bound
    # negative control: a bias that varies by token is not invisible
    o_bad = att.decode_attention(q, k - rng.standard_normal((1, 1, T, 1)) * kbar[None, :, None, :], v)
    assert np.sum((o_bad - o_ref) ** 2) / np.sum(o_ref ** 2) > 1e-4


def test_page_byte_accounting(golden):
    g = golden("streaming_kivi_page.json")
    f = g["flagship_huge_bytes"]
    L, H, D, T = f["layers"], f["heads"], f["head_dim"], f["T"]
    assert round(acc.dense_cache_bytes(L, H, T, D, 2) / 1e6, 1) == f["bf16_total_bytes_MB"]
    assert acc.side_fixed_bytes("kivi_chan", D) * L * H // 2 == f["kScales_bytes_each_KB"] * 1024
    assert L * H * T * 2 == f["vScales_bytes_each_KB"] * 1000
    assert round(acc.kivi_cache_bytes(L, H, T, D, 8) / 1e6, 1) == f["int8_kivi_total_MB"]
    s = g["smoke_100_tokens"]
    assert round(acc.kivi_cache_bytes(s["layers"], s["heads"], s["T"], s["head_dim"], 8) / 1e3) == s["int8_kivi_KB"]
    assert round(acc.dense_cache_bytes(s["layers"], s["heads"], s["T"], s["head_dim"], 4) / 1e6, 1) == s["unquantised_MB"]


def test_bits_per_element(golden):
    g = golden("mlx_memo_page.json")
    assert acc.bits_per_element(4, 64) == g["bits_per_element"]["g64_4bit"]
    assert acc.bits_per_element(4, 32) == g["bits_per_element"]["g32_4bit"]
    extra = acc.bits_per_element(4, 32) / acc.bits_per_element(4, 64) - 1
    assert round(extra, 2) == g["bits_per_element"]["extra_fraction_g32_vs_g64"]
    assert round(16 / acc.bits_per_element(4, 64), 1) == g["reduction_vs_fp16"]["g64_4bit"]
    assert round(16 / acc.bits_per_element(3, 64), 1) == g["reduction_vs_fp16"]["g64_3bit"]
    # the per-format byte counts agree with the bits-per-element rule
    assert acc.side_bytes_per_token("affine_token", 4, 64, 128) * 8 / 128 == acc.bits_per_element(4, 64)
    assert acc.side_bytes_per_token("affine_token", 4, 32, 128) * 8 / 128 == acc.bits_per_element(4, 32)


def test_decode_read_bytes_of_the_workloads():
    # codes + metadata + Q + O of one decode-attention call, per layer
    assert acc.decode_read_bytes(1, 8, 8, 32, 260, "kivi_chan", 8, 0, "affine_token", 8, 32, 4) == 144512
    assert acc.decode_read_bytes(1, 8, 24, 128, 8192, "affine_token", 4, 64, "affine_token", 4, 64, 2) == 9449472
    assert acc.decode_read_bytes(8, 8, 32, 128, 32768, "q4_0", 4, 32, "affine_token", 8, 128, 2) == 427950080
    assert acc.decode_read_bytes(64, 8, 32, 128, 4100, "kivi_chan", 4, 0, "affine_token", 4, 32, 2) == 303595520


# ---- recompute-on-append K scales ("KIVI", "Caveats") ------------------------

def _kivi_cache(bits, cap=200, layout="linear", D=16, H=2):
    return OracleCache(CacheSpec(batch=1, n_kv_heads=H, head_dim=D, capacity=cap, layout=layout,
                                 sink=4 if layout == "compact" else 0, window=64 if layout == "compact" else 0,
                                 k_format="kivi_chan", k_bits=bits, k_group=0,
                                 v_format="affine_token", v_bits=bits, v_group=D))


@pytest.mark.parametrize("bits", [8, 4])
def test_recompute_first_append_equals_calibrated_append(bits):
    rng = np.random.default_rng(40 + bits)
    k = (rng.standard_normal((1, 2, 30, 16)) * 2).astype(np.float32)
    v = rng.standard_normal((1, 2, 30, 16)).astype(np.float32)
    a, b = _kivi_cache(bits), _kivi_cache(bits)
    a.append_recompute_k(k, v)
    b.calibrate_k(k)
    b.append(k, v)
    np.testing.assert_array_equal(a.k.rows, b.k.rows)
    np.testing.assert_array_equal(a.k.ch_scale, b.k.ch_scale)
    np.testing.assert_array_equal(a.k.ch_zero, b.k.ch_zero)


@pytest.mark.parametrize("bits", [8, 4])
def test_recompute_recodes_to_nearest_level_without_clamping(bits):
    rng = np.random.default_rng(50 + bits)
    c = _kivi_cache(bits)
    L = qz.levels(bits)
    c.append_recompute_k((rng.standard_normal((1, 2, 20, 16))).astype(np.float32),
                         rng.standard_normal((1, 2, 20, 16)).astype(np.float32))
    for step in range(4):
        # the new tokens widen some channels' range (x3), so the stored keys must move
        u_prev = c.k.codes(c.stored).astype(np.float32)
        x_prev = (u_prev * c.k.ch_scale.astype(np.float32)[:, :, None, :]).astype(np.float32) \
            + c.k.ch_zero.astype(np.float32)[:, :, None, :]
        k_new = (rng.standard_normal((1, 2, 3, 16)) * (1 + step)).astype(np.float32)
        n_prev = c.stored
        c.append_recompute_k(k_new, rng.standard_normal((1, 2, 3, 16)).astype(np.float32))
        s = c.k.ch_scale32.astype(np.float64)[:, :, None, :]
        z = c.k.ch_zero32.astype(np.float64)[:, :, None, :]
        vals = np.concatenate([x_prev, k_new], axis=2).astype(np.float64)
        # the new range brackets every value: nothing is clamped
        assert np.all(vals >= z - 1e-6 * np.abs(z)) and np.all(vals <= z + L * s + 1e-5 * (np.abs(z) + L * s))
        # every stored code is the nearest of the L + 1 levels (float64 brute force), ties excepted
        u = c.k.codes(c.stored).astype(np.float64)
        lv = np.arange(L + 1, dtype=np.float64)
        dist = np.abs(vals[..., None] - (lv * s[..., None] + z[..., None]))
        best = dist.min(axis=-1)
        mine = np.take_along_axis(dist, u[..., None].astype(np.int64), axis=-1)[..., 0]
        assert np.all(mine <= best + 1e-6 * s), f"step {step}: a code is not the nearest level"
        assert c.stored == n_prev + 3


@pytest.mark.parametrize("bits", [8, 4])
def test_recompute_inside_range_moves_zero_by_one_fp16_rounding_at_most(bits):
    rng = np.random.default_rng(60 + bits)
    c = _kivi_cache(bits)
    k0 = (rng.standard_normal((1, 2, 40, 16)) * 3).astype(np.float32)
    c.append_recompute_k(k0, k0)
    z32, z16 = c.k.ch_zero32.copy(), c.k.ch_zero.astype(np.float32)
    # a new key strictly inside every channel's range
    mid = ((k0.min(axis=2) + k0.max(axis=2)) / 2)[:, :, None, :].astype(np.float32)
    c.append_recompute_k(mid, mid)
    # the smallest stored key dequantises to the fp16 zero, so the new zero is that value
    np.testing.assert_array_equal(c.k.ch_zero32, z16)
    assert np.all(np.abs(c.k.ch_zero32 - z32) <= np.abs(z32) * 2.0 ** -11 + 1e-12)


def test_recompute_gate():
    c = OracleCache(CacheSpec(batch=1, n_kv_heads=1, head_dim=16, capacity=20, layout="linear", sink=0, window=0,
                              k_format="affine_token", k_bits=8, k_group=16,
                              v_format="affine_token", v_bits=8, v_group=16))
    x = np.zeros((1, 1, 2, 16), np.float32)
    with pytest.raises(ValueError):
        c.append_recompute_k(x, x)


# ------------------------------------------------------------ KIVI residual buffer
# MLX memo, section 3: the newest tokens are kept unquantised; a full buffer's
# keys are quantised per channel as one closed block; attention reads the
# quantised bulk and then the unquantised tail.

def _residual_spec(R=64, bits=4, D=64, cap=512):
    return CacheSpec(batch=2, n_kv_heads=2, head_dim=D, capacity=cap, k_format="kivi_block", k_bits=bits,
                     k_group=R, v_format="affine_token", v_bits=4, v_group=32)


def _kv(n, seed, D=64, offsets=True):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((2, 2, n, D)).astype(np.float32)
    if offsets:
        k += rng.normal(0, 2, (2, 2, 1, D)).astype(np.float32)   # per-channel K offsets
    v = rng.standard_normal((2, 2, n, D)).astype(np.float32)
    return k, v


def _live(c):
    return (c.stored, c.n_tail, c.k.rows[:, :, : c.stored].copy(), c.k.blk_scale[:, :, : c.stored // c.spec.k_group].copy(),
            c.k.blk_zero[:, :, : c.stored // c.spec.k_group].copy(), c.v.rows[:, :, : c.stored].copy(),
            c.v.tok_scale[:, :, : c.stored].copy(), c.tail_k[:, :, : c.n_tail].copy(), c.tail_v[:, :, : c.n_tail].copy())


@pytest.mark.parametrize("n", [1, 63, 64, 65, 200, 448])
def test_residual_counts(n):
    c = OracleCache(_residual_spec())
    k, v = _kv(n, n)
    c.append(k, v)
    assert (c.stored, c.n_tail, c.pos) == ((n // 64) * 64, n % 64, n)


def test_residual_call_boundaries_do_not_matter():
    k, v = _kv(300, 1)
    one = OracleCache(_residual_spec())
    one.append(k, v)
    rng = np.random.default_rng(5)
    cuts = np.sort(rng.choice(np.arange(1, 300), 17, replace=False))
    chunked = OracleCache(_residual_spec())
    for a, b in zip(np.r_[0, cuts], np.r_[cuts, 300]):
        chunked.append(k[:, :, a:b], v[:, :, a:b])
    steps = OracleCache(_residual_spec())
    for i in range(300):
        steps.append(k[:, :, i:i + 1], v[:, :, i:i + 1])
    for other in (chunked, steps):
        for x, y in zip(_live(one), _live(other)):
            assert np.array_equal(x, y)


def test_residual_tail_is_exact_and_attention_without_a_block_is_exact():
    k, v = _kv(50, 2)
    c = OracleCache(_residual_spec())
    c.append(k, v)
    kh, vh = c.dequant()
    assert c.stored == 0 and np.array_equal(kh, k.astype(np.float64)) and np.array_equal(vh, v.astype(np.float64))
    q = np.random.default_rng(3).standard_normal((2, 6, 64))
    assert np.array_equal(att.decode_attention(q, kh, vh), att.decode_attention(q, k.astype(np.float64), v.astype(np.float64)))
    k2, v2 = _kv(100, 4)
    c.append(k2, v2)   # 150 tokens: two closed blocks, 22 in the tail
    kh, vh = c.dequant()
    allk = np.concatenate([k, k2], axis=2)
    assert c.stored == 128 and np.array_equal(kh[:, :, 128:], allk[:, :, 128:].astype(np.float64))


def test_residual_blocks_are_closed():
    k, v = _kv(200, 6)
    base = OracleCache(_residual_spec())
    base.append(k, v)
    for lo, hi in ((64, 128), (128, 192), (192, 200)):   # a later block, the last block, the tail
        k2 = k.copy()
        k2[:, :, lo:hi] *= 3.0
        other = OracleCache(_residual_spec())
        other.append(k2, v)
        # every block before the perturbed one keeps its codes and scales
        nb = lo // 64
        assert np.array_equal(base.k.rows[:, :, : nb * 64], other.k.rows[:, :, : nb * 64])
        assert np.array_equal(base.k.blk_scale[:, :, :nb], other.k.blk_scale[:, :, :nb])
        if hi <= 192:
            assert not np.array_equal(base.k.blk_scale[:, :, nb], other.k.blk_scale[:, :, nb])


@pytest.mark.parametrize("bits", [4, 8])
def test_residual_block_range_ends_and_error_bound(bits):
    k, v = _kv(256, 7 + bits)
    c = OracleCache(_residual_spec(bits=bits))
    c.append(k, v)
    L = qz.levels(bits)
    u = c.k.codes(256).astype(np.int64)
    kh, _ = c.dequant()
    for j in range(4):
        blk = k[:, :, 64 * j:64 * (j + 1)]
        ub = u[:, :, 64 * j:64 * (j + 1)]
        # each channel's smallest key of the block sits on code 0, its largest on code L
        amin = blk.argmin(axis=2)[:, :, None, :]
        amax = blk.argmax(axis=2)[:, :, None, :]
        assert np.all(np.take_along_axis(ub, amin, 2) == 0)
        assert np.all(np.take_along_axis(ub, amax, 2) == L)
        # reconstruction within half a step of the block's own range, plus the fp16 rounding of
        # the stored scale and zero
        step = (blk.max(axis=2) - blk.min(axis=2)).astype(np.float64) / L
        s16 = c.k.blk_scale[:, :, j].astype(np.float64)
        z16 = c.k.blk_zero[:, :, j].astype(np.float64)
        tol = step / 2 * (1 + 1e-6) + L * np.abs(s16 - step) + np.abs(z16 - blk.min(axis=2))
        err = np.abs(kh[:, :, 64 * j:64 * (j + 1)] - blk)
        assert np.all(err <= tol[:, :, None, :] + 1e-7)


def test_residual_needs_linear_layout_and_affine_values():
    with pytest.raises(ValueError):
        OracleCache(CacheSpec(1, 1, 64, 256, layout="compact", sink=4, window=128, k_format="kivi_block",
                              k_bits=4, k_group=64, v_format="affine_token", v_bits=4, v_group=32))
    with pytest.raises(ValueError):
        OracleCache(CacheSpec(1, 1, 64, 256, k_format="kivi_block", k_bits=4, k_group=64))


def test_keepset_moves_per_token_scales_with_their_codes():
    # "SnapKV", "How it works", step 4 on a quantised cache: each kept row
    # carries its own per-token scales, so the dequantised cache after the
    # keep-set is the dequantised cache before it, read at the kept rows.
    rng = np.random.default_rng(18)
    S, D = 48, 64
    spec = CacheSpec(batch=2, n_kv_heads=2, head_dim=D, capacity=S, k_format="q4_0", k_bits=4, k_group=32,
                     v_format="affine_token", v_bits=4, v_group=32)
    c = OracleCache(spec)
    k = (rng.standard_normal((2, 2, S, D)) * rng.uniform(0.1, 9, size=(2, 2, S, 1))).astype(np.float32)
    v = (rng.standard_normal((2, 2, S, D)) * rng.uniform(0.1, 9, size=(2, 2, S, 1))).astype(np.float32)
    c.append(k, v)
    kh0, vh0 = c.dequant()
    idx = np.stack([np.stack([np.sort(rng.choice(S, 12, replace=False)) for _ in range(2)])
                    for _ in range(2)]).astype(np.int32)
    c.evict_keepset(idx)
    kh1, vh1 = c.dequant()
    for b in range(2):
        for h in range(2):
            np.testing.assert_array_equal(kh1[b, h], kh0[b, h, idx[b, h]])
            np.testing.assert_array_equal(vh1[b, h], vh0[b, h, idx[b, h]])


def test_cache_planes_are_the_page_layout():
    # "StreamingLLM + KIVI", "Storage layout" and "Cache-bytes table": int8
    # codes, fp16 per-channel K scale and zero, fp16 per-token V scale and
    # zero.  The oracle's planes hold exactly the bytes the page's accounting
    # counts (pinned above to the page's printed totals), in fp16.
    B, H, T, D = 1, 8, 100, 32
    spec = CacheSpec(batch=B, n_kv_heads=H, head_dim=D, capacity=T, k_format="kivi_chan", k_bits=8,
                     v_format="affine_token", v_bits=8, v_group=D)
    c = OracleCache(spec)
    rng = np.random.default_rng(19)
    x = rng.standard_normal((B, H, T, D)).astype(np.float32)
    c.calibrate_k(x)
    c.append(x, x)
    planes = [c.k.rows, c.k.ch_scale, c.k.ch_zero, c.v.rows, c.v.tok_scale, c.v.tok_zero]
    assert all(p.dtype == np.float16 for p in planes[1:3] + planes[4:])
    assert sum(p.nbytes for p in planes) == acc.kivi_cache_bytes(1, H, T, D, 8, batch=B)


@pytest.mark.parametrize("k_fmt,k_bits,k_group,v_bits,v_group", [
    ("affine_token", 4, 64, 4, 64), ("affine_token", 8, 32, 8, 128), ("q4_0", 4, 32, 8, 128),
    ("q4_0", 4, 32, 4, 32), ("kivi_chan", 4, 0, 4, 32), ("kivi_chan", 8, 0, 8, 64)])
def test_cache_round_trip_within_the_per_group_bound(k_fmt, k_bits, k_group, v_bits, v_group):
    # "StreamingLLM + KIVI", "Affine quantisation formula" (and Q4_0's
    # symmetric blocks): every stored element reads back within half a step
    # of its own group's true range, plus the fp16 rounding of the stored
    # scale (up to L steps) and zero.  The bound is computed here from the
    # inputs alone, per group, independently of the oracle's planes.
    rng = np.random.default_rng(23)
    B, H, T, D = 2, 2, 40, 128
    k = (rng.standard_normal((B, H, T, D)) * rng.uniform(0.2, 6, size=(B, H, T, 1))
         + rng.standard_normal((B, H, 1, D))).astype(np.float32)
    v = (rng.standard_normal((B, H, T, D)) * rng.uniform(0.2, 6, size=(B, H, T, 1))).astype(np.float32)
    c = OracleCache(CacheSpec(batch=B, n_kv_heads=H, head_dim=D, capacity=T, k_format=k_fmt, k_bits=k_bits,
                              k_group=k_group, v_format="affine_token", v_bits=v_bits, v_group=v_group))
    if k_fmt == "kivi_chan":
        c.calibrate_k(k)
    c.append(k, v)
    kh, vh = c.dequant()
    u16 = 2.0 ** -11

    def affine_bound(x, bits, axis_groups):
        L = (1 << bits) - 1
        g = axis_groups(x)
        lo, hi = g.min(axis=-1, keepdims=True), g.max(axis=-1, keepdims=True)
        s = np.maximum(1e-5, (hi - lo) / L)
        b = 0.5 * s + L * s * u16 + np.abs(lo) * u16 + 2.0 ** -20 * (np.abs(g) + L * s)
        return np.broadcast_to(b, g.shape)

    # values: per token, groups of v_group channels
    vb = affine_bound(v.astype(np.float64), v_bits, lambda x: x.reshape(B, H, T, D // v_group, v_group))
    assert np.all(np.abs(vh - v).reshape(vb.shape) <= vb)
    if k_fmt == "affine_token":
        kb = affine_bound(k.astype(np.float64), k_bits, lambda x: x.reshape(B, H, T, D // k_group, k_group))
        assert np.all(np.abs(kh - k).reshape(kb.shape) <= kb)
    elif k_fmt == "kivi_chan":
        # per channel over the tokens: move the token axis last
        kt = np.swapaxes(k.astype(np.float64), 2, 3)
        kb = affine_bound(kt, k_bits, lambda x: x)
        assert np.all(np.abs(np.swapaxes(kh, 2, 3) - kt) <= kb)
    else:
        blk = k.astype(np.float64).reshape(B, H, T, D // 32, 32)
        d = np.abs(blk).max(axis=-1, keepdims=True) / 7
        kb = 0.5 * d * (1 + 1e-6) + 7 * d * u16
        assert np.all(np.abs(kh.reshape(blk.shape) - blk) <= kb)
