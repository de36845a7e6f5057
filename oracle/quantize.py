"""Quantisers of the compressed KV cache, written out in numpy.

All decisions that produce an integer code are taken in IEEE fp32 with
round-to-nearest-even (numpy float32 ufuncs), so that a kernel computing
the same formula in fp32 lands on the same code.  Stored metadata (scales,
zeros) is rounded to fp16; dequantisation upcasts the stored fp16 values.
"""
from __future__ import annotations

import numpy as np

# "StreamingLLM + KIVI" page, section "Affine quantisation formula":
# the scale never falls below eps = 1e-5; the level range is -128..127 at
# 8 bits and -8..7 at 4 bits (the "clamped to +-7" remark under "Storage
# layout" is read as this same 4-bit range).
EPS = np.float32(1e-5)
QRANGE = {8: (-128, 127), 4: (-8, 7)}

# Symmetric Q4_0: the page ("kv-cache: optional per-channel K-cache
# mean-centering for Q4_0", section "The idea") calls it a symmetric block
# quantiser without a zero point, and gives neither block size nor
# arithmetic.  The layout used is that of the Q4_0 K-cache workload, blocks of
# 32 elements with one fp16 scale; the reading is d = max|x| / 7 and
# q = clamp(rint(x / d), -8, 7), stored as the nibble q + 8.
Q4_0_BLOCK = 32
Q4_0_QMAX = np.float32(7.0)


def levels(bits: int) -> int:
    """qMax - qMin: 255 for int8, 15 for int4."""
    qmin, qmax = QRANGE[bits]
    return qmax - qmin


def affine_scale_zero(xmin: np.ndarray, xmax: np.ndarray, bits: int):
    """scale = max(eps, (xMax - xMin) / (qMax - qMin)), zero = xMin, in fp32.

    "StreamingLLM + KIVI" page, "Affine quantisation formula".
    """
    xmin = np.asarray(xmin, dtype=np.float32)
    xmax = np.asarray(xmax, dtype=np.float32)
    rng = xmax - xmin                                   # fp32 subtract
    scale = np.maximum(EPS, rng / np.float32(levels(bits)))  # fp32 divide
    zero = xmin.copy()
    return scale.astype(np.float32), zero


def affine_codes(x: np.ndarray, scale: np.ndarray, zero: np.ndarray, bits: int) -> np.ndarray:
    """u = clamp(rint((x - zero) / scale), 0, qMax - qMin), as uint8.

    The page writes q = round((x - zero)/scale + qMin); the integer qMin is
    added after rounding here (identical in exact arithmetic, one fp32
    rounding fewer).  The level is q = u + qMin; the dequantised value is
    (q - qMin) * scale + zero = u * scale + zero.  Values beyond the
    calibrated range (frozen per-channel K scales) clamp to 0 or qMax - qMin.
    """
    x = np.asarray(x, dtype=np.float32)
    t = (x - zero) / scale                              # two fp32 roundings
    u = np.clip(np.rint(t), np.float32(0), np.float32(levels(bits)))
    return u.astype(np.uint8)


def kivi_channel_calibrate(k: np.ndarray, bits: int):
    """Per-(b, kv-head, channel) scale and zero over the token axis of k [B,H,T,D].

    KIVI codes keys channel by channel: every stored token of a (batch row,
    head) uses that channel's single (scale, zero) ("StreamingLLM + KIVI", "KIVI --
    int8/int4 KV cache").  Here the scales are computed once from the tokens
    given and then frozen (the group-boundary freezing the page's caveats
    attribute to the KIVI paper); returns fp32 [B,H,D] scale and zero.
    """
    k = np.asarray(k, dtype=np.float32)
    return affine_scale_zero(k.min(axis=2), k.max(axis=2), bits)


def kivi_channel_codes(k: np.ndarray, scale: np.ndarray, zero: np.ndarray, bits: int) -> np.ndarray:
    """Codes u [B,H,T,D] of k against the frozen per-channel fp32 scale/zero [B,H,D]."""
    return affine_codes(k, scale[:, :, None, :], zero[:, :, None, :], bits)


def affine_token_quantize(x: np.ndarray, bits: int, group: int):
    """Per-token, per-channel-group asymmetric quantisation of x [B,H,T,D].

    Each token's head vector is cut into D / group contiguous groups; each
    group gets its own (scale, zero) from its min and max.  With group = D
    this is KIVI's per-token V ("StreamingLLM + KIVI", "KIVI"); with
    group = 64 it is mlx-lm's QuantizedKVCache scheme ("Low-bit KV caches on
    MLX", section 1).  Returns codes u [B,H,T,D] and fp32 scale, zero
    [B,H,T,D/group].
    """
    x = np.asarray(x, dtype=np.float32)
    B, H, T, D = x.shape
    assert D % group == 0
    g = x.reshape(B, H, T, D // group, group)
    scale, zero = affine_scale_zero(g.min(axis=-1), g.max(axis=-1), bits)
    u = affine_codes(g, scale[..., None], zero[..., None], bits)
    return u.reshape(B, H, T, D), scale, zero


def q4_0_quantize(x: np.ndarray):
    """Symmetric 32-block quantisation of x [B,H,T,D] (D a multiple of 32).

    Per block: a = max|x|, d = a / 7 (fp32).  If d == 0 the block stores
    d = 0 and every code is 8 (the level 0).  Otherwise
    q = clamp(rint(x / d), -8, 7) and the stored nibble is q + 8.
    Dequantisation is (nibble - 8) * d.  Returns codes u [B,H,T,D] and fp32
    d [B,H,T,D/32].
    """
    x = np.asarray(x, dtype=np.float32)
    B, H, T, D = x.shape
    assert D % Q4_0_BLOCK == 0
    blk = x.reshape(B, H, T, D // Q4_0_BLOCK, Q4_0_BLOCK)
    a = np.abs(blk).max(axis=-1)
    d = (a / Q4_0_QMAX).astype(np.float32)
    zero_block = d == np.float32(0)
    safe_d = np.where(zero_block, np.float32(1), d)
    q = np.clip(np.rint(blk / safe_d[..., None]), np.float32(-8), np.float32(7))
    q = np.where(zero_block[..., None], np.float32(0), q)
    u = (q + np.float32(8)).astype(np.uint8)
    return u.reshape(B, H, T, D), d


def mean_center(k: np.ndarray, kbar: np.ndarray) -> np.ndarray:
    """k - kbar[kv-head, channel] in fp32, the subtraction made right before K is quantised.

    "kv-cache: optional per-channel K-cache mean-centering for Q4_0",
    sections "Summary" and "Why this is safe": one precomputed value per
    (kv head, channel) comes off K as it is written to the cache, and decode
    adds nothing back.
    """
    k = np.asarray(k, dtype=np.float32)
    kbar = np.asarray(kbar, dtype=np.float32)
    return k - kbar[None, :, None, :]


# ---------------------------------------------------------------- storage --

def to_fp16(x: np.ndarray) -> np.ndarray:
    """Round fp32 metadata to fp16 (nearest, ties to even)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16)


def stored_int8(u: np.ndarray) -> np.ndarray:
    """8-bit levels are stored as the signed q = u + qMin = u - 128 (KIVI keysQ/valuesQ int8)."""
    return (u.astype(np.int16) - 128).astype(np.int8)


def int8_to_codes(q: np.ndarray) -> np.ndarray:
    return (q.astype(np.int16) + 128).astype(np.uint8)


def pack_nibbles(u: np.ndarray) -> np.ndarray:
    """4-bit codes [..., D] -> bytes [..., D/2]: element 2j in the low nibble of byte j.

    Two codes per byte, low nibble first, so that a little-endian 32-bit
    word holds eight consecutive channels ("packed nibbles in uint32 rows").
    """
    u = np.asarray(u, dtype=np.uint8)
    assert u.shape[-1] % 2 == 0 and int(u.max(initial=0)) < 16
    return (u[..., 0::2] | (u[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (b.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    return out


def dequant_affine(u: np.ndarray, scale16: np.ndarray, zero16: np.ndarray) -> np.ndarray:
    """x_dq = (q - qMin) * scale + zero = u * scale + zero, in float64 from fp16 metadata."""
    return u.astype(np.float64) * scale16.astype(np.float64) + zero16.astype(np.float64)


def dequant_q4_0(u: np.ndarray, d16: np.ndarray) -> np.ndarray:
    """(nibble - 8) * d, float64, with d broadcast over its 32-element block."""
    B, H, T, D = u.shape
    blk = u.reshape(B, H, T, D // Q4_0_BLOCK, Q4_0_BLOCK).astype(np.float64) - 8.0
    return (blk * d16.astype(np.float64)[..., None]).reshape(B, H, T, D)
