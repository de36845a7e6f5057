"""Pins of the oracle's quantisers against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the page's
printed constants, the round-trip bound |x - deq(q(x))| <= scale/2, brute
force over every level, the degenerate constant-channel case, symmetry.
"""
import numpy as np
import pytest

from oracle import quantize as qz


def _rng(seed):
    return np.random.default_rng(seed)


def _fp32_slack(x, z, s, L):
    # two fp32 roundings in t = fl(fl(x - z) / s) move the unrounded level by
    # at most ~2 ulp of t; in value that is <= 2^-22 * (|x - z| + L * s).
    return 2.0 ** -22 * (np.abs(x - z) + L * s)


def test_page_constants(golden):
    g = golden("streaming_kivi_page.json")["affine_formula"]
    assert qz.EPS == np.float32(g["eps"])
    assert qz.QRANGE[8] == tuple(g["int8_qmin_qmax"])
    assert qz.QRANGE[4] == tuple(g["int4_qmin_qmax"])
    assert qz.levels(8) == 255 and qz.levels(4) == 15


def test_hand_worked_example():
    # x = 0, 1, 2, 3 at int4: xmin 0, xmax 3, scale = 3/15 = 0.2, zero 0,
    # levels u = 0, 5, 10, 15, i.e. q = -8, -3, 2, 7, dequantised back to x.
    x = np.array([[[[0.0, 1.0, 2.0, 3.0]]]], np.float32)
    u, s, z = qz.affine_token_quantize(x, 4, 4)
    assert s[0, 0, 0, 0] == np.float32(3.0) / np.float32(15.0)
    assert z[0, 0, 0, 0] == 0.0
    assert u.ravel().tolist() == [0, 5, 10, 15]
    assert (u.astype(int) + qz.QRANGE[4][0]).ravel().tolist() == [-8, -3, 2, 7]
    xh = u.astype(np.float64) * np.float64(s[0, 0, 0, 0])
    np.testing.assert_allclose(xh.ravel(), [0, 1, 2, 3], rtol=1e-6)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("group", [32, 64, 128])
def test_affine_token_roundtrip_bound(bits, group):
    rng = _rng(bits * 1000 + group)
    x = (rng.standard_normal((2, 3, 17, 128)) * rng.uniform(0.01, 30, size=(2, 3, 17, 1))
         + rng.standard_normal((2, 3, 17, 1)) * 5).astype(np.float32)
    u, s, z = qz.affine_token_quantize(x, bits, group)
    L = qz.levels(bits)
    assert u.dtype == np.uint8 and u.min() >= 0 and u.max() <= L
    B, H, T, D = x.shape
    ng = D // group
    sg = np.repeat(s.astype(np.float64), group, axis=-1).reshape(B, H, T, D)
    zg = np.repeat(z.astype(np.float64), group, axis=-1).reshape(B, H, T, D)
    xh = u.astype(np.float64) * sg + zg
    err = np.abs(x.astype(np.float64) - xh)
    assert np.all(err <= 0.5 * sg + _fp32_slack(x.astype(np.float64), zg, sg, L))
    # every group reaches both ends of its range
    ug = u.reshape(B, H, T, ng, group)
    assert np.all(ug.min(axis=-1) == 0)
    assert np.all(ug.max(axis=-1) == L)


@pytest.mark.parametrize("bits", [8, 4])
def test_affine_brute_force_nearest_level(bits):
    rng = _rng(7 + bits)
    x = (rng.standard_normal((1, 2, 40, 64)) * 3).astype(np.float32)
    u, s, z = qz.affine_token_quantize(x, bits, 64)
    L = qz.levels(bits)
    s64 = s.astype(np.float64)[..., None]
    z64 = z.astype(np.float64)[..., None]
    cand = np.arange(L + 1, dtype=np.float64)
    # distance of each element to every level u' * s + z, float64
    xg = x.astype(np.float64).reshape(1, 2, 40, 1, 64)
    lv = cand[None, None, None, None, :] * s64[..., None] + z64[..., None]   # [1,2,40,1,1,L+1]
    dist = np.abs(xg[..., None] - lv)
    best = dist.argmin(axis=-1)
    srt = np.sort(dist, axis=-1)
    tie = (srt[..., 1] - srt[..., 0]) < 1e-6 * s64
    mism = (best.reshape(u.shape) != u) & ~tie.reshape(u.shape)
    assert not mism.any()
    assert tie.mean() < 1e-3


def test_constant_channel_uses_eps():
    # "StreamingLLM + KIVI", failure mode 1: a constant channel has zero range;
    # the scale falls back to eps, every code is the lowest level, and the
    # dequantised value is exactly the zero point.
    x = np.full((1, 1, 9, 32), 0.375, np.float32)
    s, z = qz.kivi_channel_calibrate(x, 8)
    assert np.all(s == qz.EPS) and np.all(z == np.float32(0.375))
    u = qz.kivi_channel_codes(x, s, z, 8)
    assert np.all(u == 0)
    xh = qz.dequant_affine(u, qz.to_fp16(s)[:, :, None, :], qz.to_fp16(z)[:, :, None, :])
    assert np.all(xh == np.float64(np.float16(0.375)))
    # all-zero per-token group: same fallback, no NaN
    u2, s2, z2 = qz.affine_token_quantize(np.zeros((1, 1, 2, 64), np.float32), 4, 64)
    assert np.all(s2 == qz.EPS) and np.all(z2 == 0) and np.all(u2 == 0)


@pytest.mark.parametrize("bits", [8, 4])
def test_kivi_channel_frozen_scales_and_clamp(bits):
    rng = _rng(31 + bits)
    fill = (rng.standard_normal((2, 2, 50, 32)) + rng.standard_normal((2, 2, 1, 32)) * 2).astype(np.float32)
    s, z = qz.kivi_channel_calibrate(fill, bits)
    np.testing.assert_array_equal(z, fill.min(axis=2))
    L = qz.levels(bits)
    u = qz.kivi_channel_codes(fill, s, z, bits)
    # the fill reaches both ends of every channel's range
    assert np.all(u.min(axis=2) == 0) and np.all(u.max(axis=2) == L)
    # later tokens beyond the frozen range clamp to the end levels
    lo = (z - 3 * s * L)[:, :, None, :]
    hi = (z + 3 * s * L)[:, :, None, :]
    assert np.all(qz.kivi_channel_codes(lo.astype(np.float32), s, z, bits) == 0)
    assert np.all(qz.kivi_channel_codes(hi.astype(np.float32), s, z, bits) == L)
    # round trip for in-range values
    zz = z.astype(np.float64)[:, :, None, :]
    ss = s.astype(np.float64)[:, :, None, :]
    xh = u.astype(np.float64) * ss + zz
    assert np.all(np.abs(fill - xh) <= 0.5 * ss + _fp32_slack(fill.astype(np.float64), zz, ss, L))


def test_stored_metadata_bound():
    # dequantising with fp16-stored scale and zero moves x_hat by at most
    # |dz| + u * |ds| beyond the fp32-metadata bound.
    rng = _rng(5)
    x = (rng.standard_normal((1, 4, 64, 128)) * 2).astype(np.float32)
    for bits, group in ((4, 64), (8, 128), (4, 32)):
        u, s, z = qz.affine_token_quantize(x, bits, group)
        s16, z16 = qz.to_fp16(s), qz.to_fp16(z)
        ds = np.abs(s16.astype(np.float64) - s.astype(np.float64))
        dz = np.abs(z16.astype(np.float64) - z.astype(np.float64))
        assert np.all(ds <= 2.0 ** -11 * s) and np.all(dz <= 2.0 ** -11 * np.abs(z) + 2.0 ** -25)
        B, H, T, D = x.shape
        rep = lambda a: np.repeat(a.astype(np.float64), group, axis=-1).reshape(B, H, T, D)
        xh16 = u.astype(np.float64) * rep(s16) + rep(z16)
        L = qz.levels(bits)
        bound = 0.5 * rep(s) + rep(dz) + L * rep(ds) + _fp32_slack(x.astype(np.float64), rep(z), rep(s), L)
        assert np.all(np.abs(x - xh16) <= bound)


def test_q4_0_bound_brute_force_and_symmetry(golden):
    g = golden("mean_center_page.json")["q4_0_block"]
    assert qz.Q4_0_BLOCK == g["block"]
    rng = _rng(11)
    x = (rng.standard_normal((2, 2, 33, 128)) * rng.uniform(0.1, 10, size=(2, 2, 33, 1))).astype(np.float32)
    u, d = qz.q4_0_quantize(x)
    assert u.max() <= 15 and d.dtype == np.float32
    blk = x.reshape(2, 2, 33, 4, 32).astype(np.float64)
    np.testing.assert_array_equal(d, (np.abs(x.reshape(2, 2, 33, 4, 32)).max(-1) / np.float32(7)))
    q = u.reshape(2, 2, 33, 4, 32).astype(np.float64) - 8
    d64 = d.astype(np.float64)[..., None]
    err = np.abs(blk - q * d64)
    assert np.all(err <= 0.5 * d64 * (1 + 1e-6))
    # brute force over the 16 levels
    lv = np.arange(-8, 8, dtype=np.float64)
    dist = np.abs(blk[..., None] - lv * d64[..., None])
    best = lv[dist.argmin(-1)]
    srt = np.sort(dist, -1)
    tie = (srt[..., 1] - srt[..., 0]) < 1e-6 * d64
    assert np.all((best == q) | tie)
    # symmetric: negating the block negates every level
    un, dn = qz.q4_0_quantize(-x)
    np.testing.assert_array_equal(dn, d)
    np.testing.assert_array_equal(un.astype(int) - 8, -(u.astype(int) - 8))
    # the block's extreme element lands on +-7; level -8 is never used
    assert np.all(np.abs(q).max(-1) == 7) and q.min() >= -7


def test_q4_0_zero_block():
    x = np.zeros((1, 1, 2, 64), np.float32)
    x[0, 0, 1, 40] = 3.5
    u, d = qz.q4_0_quantize(x)
    assert d[0, 0, 0, 0] == 0 and d[0, 0, 0, 1] == 0 and d[0, 0, 1, 0] == 0
    assert np.all(u[0, 0, 0] == 8) and np.all(u[0, 0, 1, :32] == 8)
    assert d[0, 0, 1, 1] == np.float32(0.5) and u[0, 0, 1, 40] == 15


def test_nibble_order():
    # channel 2j in the low nibble of byte j: eight consecutive codes read as
    # one little-endian 32-bit word 0x76543210.
    u = np.arange(8, dtype=np.uint8)[None]
    b = qz.pack_nibbles(u)
    assert b.tolist() == [[0x10, 0x32, 0x54, 0x76]]
    assert int(b.view("<u4")[0, 0]) == 0x76543210
    rng = _rng(3)
    u = rng.integers(0, 16, size=(3, 64), dtype=np.uint8)
    np.testing.assert_array_equal(qz.unpack_nibbles(qz.pack_nibbles(u)), u)


def test_int8_storage_is_signed_level():
    u = np.array([0, 1, 127, 128, 255], np.uint8)
    q = qz.stored_int8(u)
    assert q.tolist() == [-128, -127, -1, 0, 127]
    np.testing.assert_array_equal(qz.int8_to_codes(q), u)


def test_mean_center_subtracts_per_head_channel():
    rng = _rng(9)
    k = rng.standard_normal((2, 3, 5, 32)).astype(np.float32)
    kbar = rng.standard_normal((3, 32)).astype(np.float32)
    kc = qz.mean_center(k, kbar)
    for b in range(2):
        for h in range(3):
            for t in range(5):
                np.testing.assert_array_equal(kc[b, h, t], k[b, h, t] - kbar[h])


def test_centering_reduces_q4_0_error_on_biased_channels():
    # the motivation the mean-centering page gives: a symmetric quantiser
    # wastes range on a consistent channel bias; removing it shrinks error.
    rng = _rng(21)
    kbar = (rng.standard_normal((4, 128)) * 1.5).astype(np.float32)
    k = (rng.standard_normal((1, 4, 256, 128)) + kbar[None, :, None, :]).astype(np.float32)
    u0, d0 = qz.q4_0_quantize(k)
    err0 = np.abs(qz.dequant_q4_0(u0, qz.to_fp16(d0)) - k).mean()
    kc = qz.mean_center(k, kbar)
    u1, d1 = qz.q4_0_quantize(kc)
    err1 = np.abs(qz.dequant_q4_0(u1, qz.to_fp16(d1)) + kbar[None, :, None, :] - k).mean()
    assert err1 < 0.8 * err0


def test_exact_ties_round_to_even():
    # Reading of "round" in the affine formula and in Q4_0: IEEE round to
    # nearest, ties to even (the fp32 hardware rounding).  With a group
    # spanning exactly 0..L the scale is exactly 1 and zero is 0, so every
    # x + 0.5 sits on a tie that half-away rounding would send up.
    x4 = np.array([[[[0, 15, 0.5, 1.5, 2.5, 3.5, 13.5, 14.5]]]], np.float32)
    u4, s4, z4 = qz.affine_token_quantize(x4, 4, 8)
    assert s4.ravel()[0] == 1.0 and z4.ravel()[0] == 0.0
    assert u4.ravel().tolist() == [0, 15, 0, 2, 2, 4, 14, 14]
    x8 = np.array([[[[0, 255, 0.5, 1.5, 126.5, 127.5, 253.5, 254.5]]]], np.float32)
    u8, s8, _ = qz.affine_token_quantize(x8, 8, 8)
    assert s8.ravel()[0] == 1.0
    assert u8.ravel().tolist() == [0, 255, 0, 2, 126, 128, 254, 254]
    # Q4_0: max|x| = 7 gives d = 1; signed ties go to the even level
    xq = np.zeros((1, 1, 1, 32), np.float32)
    xq[0, 0, 0, :7] = [7, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5]
    uq, dq = qz.q4_0_quantize(xq)
    assert dq.ravel()[0] == 1.0
    assert (uq.ravel()[:7].astype(int) - 8).tolist() == [7, 0, 2, 2, 0, -2, -2]


def test_q4_0_blocks_are_per_token_runs_of_32_channels():
    # "32-element blocks with one fp16 scale" along the head vector: a token's
    # codes and scales do not depend on the other tokens, and a spike in one
    # channel moves only the scale of its own 32-channel block of that token.
    rng = _rng(31)
    x = rng.standard_normal((1, 2, 32, 128)).astype(np.float32)
    u, d = qz.q4_0_quantize(x)
    for t in (0, 7, 31):
        ut, dt = qz.q4_0_quantize(x[:, :, t:t + 1])
        np.testing.assert_array_equal(ut[:, :, 0], u[:, :, t])
        np.testing.assert_array_equal(dt[:, :, 0], d[:, :, t])
    y = x.copy()
    y[0, 1, 5, 70] = 50.0
    uy, dy = qz.q4_0_quantize(y)
    changed = np.argwhere(dy != d)
    assert changed.tolist() == [[0, 1, 5, 2]]
    assert dy[0, 1, 5, 2] == np.float32(50.0) / np.float32(7.0)
    same = np.ones(u.shape, bool)
    same[0, 1, 5, 64:96] = False
    np.testing.assert_array_equal(uy[same], u[same])


def test_q4_0_stored_roundtrip():
    # the stored path: nibbles and the fp16 scale, dequantised by the oracle's
    # own routine, land within half a step of x plus the fp16 rounding of the
    # scale times the largest level (7); an all-zero block reads back as zeros.
    rng = _rng(33)
    x = (rng.standard_normal((2, 2, 9, 64)) * rng.uniform(0.05, 20, size=(2, 2, 9, 1))).astype(np.float32)
    x[1, 1, 3, 32:] = 0.0
    u, d = qz.q4_0_quantize(x)
    d16 = qz.to_fp16(d)
    xh = qz.dequant_q4_0(u, d16)
    rep = lambda a: np.repeat(a.astype(np.float64), 32, axis=-1)
    bound = 0.5 * rep(d) * (1 + 1e-6) + 7 * np.abs(rep(d16) - rep(d))
    assert np.all(np.abs(x.astype(np.float64) - xh) <= bound)
    assert np.all(xh[1, 1, 3, 32:] == 0.0)
    # the extreme element of every nonzero block comes back as +-7 d16
    blk = xh.reshape(2, 2, 9, 2, 32)
    amax = np.abs(blk).max(-1)
    nz = d > 0
    np.testing.assert_array_equal(amax[nz], 7 * d16.astype(np.float64)[nz])
