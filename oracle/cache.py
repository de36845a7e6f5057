"""The compressed KV cache as plain numpy planes: append, evict, dequantise.

Physical layout (the same one the CUDA library documents for its device
buffer, written here independently from that description):

* code rows   ``[B, Hkv, cap, row_bytes]`` uint8.  fp16 rows hold the raw
  fp16 bytes; 8-bit rows hold the signed level q = u - 128; 4-bit rows hold
  nibbles, channel 2j in the low nibble of byte j.
* per-token metadata (affine groups, Q4_0 blocks) ``[B, Hkv, cap, n_groups]``
  fp16 scale (and zero for affine formats).
* per-channel metadata (KIVI keys) ``[B, Hkv, D]`` fp16 scale and zero, plus
  the fp32 values the codes were computed from.

KIVI residual buffer (MLX memo, section 3, "What KIVI and KVQuant found";
k_format "kivi_block", k_group = R): the most recent tokens stay at full
precision in a tail of fewer than R rows (fp32, the values the caller gave);
whenever the tail reaches R tokens its keys are quantised per channel over
exactly those R tokens (a closed block: its own KIVI scale and zero per
channel, fp16 planes [B, Hkv, cap / R, D]) and its values per token, the
codes go to the next R rows of the quantised bulk and the tail empties.
Attention runs over the dequantised bulk followed by the exact tail.

Eviction, from "StreamingLLM + KIVI" ("Implementation"): when the stored
length exceeds sink + window, logical positions [sink, len - window) are
dropped and the rest is concatenated in order; K's per-channel scales are
untouched, per-token metadata moves with its token.  It runs after each
append.  The ring layout keeps the same survivors without moving data: the
token at absolute position p >= sink lives in slot sink + (p - sink) mod
window.  SnapKV ("SnapKV", "How it works", step 4) keeps only a chosen,
ascending set of rows.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from . import quantize as qz


@dataclasses.dataclass
class CacheSpec:
    batch: int
    n_kv_heads: int
    head_dim: int
    capacity: int
    layout: str = "linear"          # "linear" | "compact" | "ring"
    sink: int = 0
    window: int = 0
    k_format: str = "fp16"          # "fp16" | "kivi_chan" | "affine_token" | "q4_0" | "kivi_block"
    k_bits: int = 16
    k_group: int = 0
    v_format: str = "fp16"          # "fp16" | "affine_token"
    v_bits: int = 16
    v_group: int = 0
    k_bias: Optional[np.ndarray] = None   # fp32 [Hkv, D]; legal only with q4_0 keys


def row_bytes(fmt: str, bits: int, D: int) -> int:
    if fmt == "fp16":
        return 2 * D
    return D * bits // 8


def n_token_groups(fmt: str, group: int, D: int) -> int:
    if fmt == "affine_token":
        return D // group
    if fmt == "q4_0":
        return D // qz.Q4_0_BLOCK
    return 0


def ring_slot(p: int, sink: int, window: int) -> int:
    """Slot of absolute position p in the sink + window ring."""
    return p if p < sink else sink + (p - sink) % window


def streaming_survivors(n_seen: int, sink: int, window: int) -> list:
    """Logical positions held after n_seen appends with evict-after-append: closed form."""
    if n_seen <= sink + window:
        return list(range(n_seen))
    return list(range(sink)) + list(range(n_seen - window, n_seen))


class _Side:
    """The planes of one of K or V."""

    def __init__(self, spec: CacheSpec, fmt: str, bits: int, group: int):
        B, H, D, cap = spec.batch, spec.n_kv_heads, spec.head_dim, spec.capacity
        self.fmt, self.bits, self.group, self.D = fmt, bits, group, D
        self.rows = np.zeros((B, H, cap, row_bytes(fmt, bits, D)), np.uint8)
        ng = n_token_groups(fmt, group, D)
        self.tok_scale = np.zeros((B, H, cap, ng), np.float16) if ng else None
        self.tok_zero = np.zeros((B, H, cap, ng), np.float16) if fmt == "affine_token" else None
        self.ch_scale = np.zeros((B, H, D), np.float16) if fmt == "kivi_chan" else None
        self.ch_zero = np.zeros((B, H, D), np.float16) if fmt == "kivi_chan" else None
        self.ch_scale32 = None
        self.ch_zero32 = None
        # closed-block per-channel metadata (kivi_block keys; group = block length R)
        nblk = cap // group if fmt == "kivi_block" else 0
        self.blk_scale = np.zeros((B, H, nblk, D), np.float16) if nblk else None
        self.blk_zero = np.zeros((B, H, nblk, D), np.float16) if nblk else None

    # per-token planes move with their token on eviction
    def token_planes(self):
        return [p for p in (self.rows, self.tok_scale, self.tok_zero) if p is not None]

    def calibrate(self, x: np.ndarray):
        s, z = qz.kivi_channel_calibrate(x, self.bits)
        self.ch_scale32, self.ch_zero32 = s, z
        self.ch_scale, self.ch_zero = qz.to_fp16(s), qz.to_fp16(z)

    def encode(self, x: np.ndarray, bias: Optional[np.ndarray]):
        """x fp32 [B,H,n,D] -> (rows [B,H,n,row_bytes], token scale, token zero)."""
        fmt, bits = self.fmt, self.bits
        if fmt == "fp16":
            return qz.to_fp16(x).view(np.uint8).reshape(x.shape[:3] + (-1,)), None, None
        if fmt == "kivi_chan":
            if self.ch_scale32 is None:
                raise RuntimeError("per-channel K scales were never calibrated")
            u = qz.kivi_channel_codes(x, self.ch_scale32, self.ch_zero32, bits)
            return self._pack(u), None, None
        if fmt == "affine_token":
            u, s, z = qz.affine_token_quantize(x, bits, self.group)
            return self._pack(u), qz.to_fp16(s), qz.to_fp16(z)
        if fmt == "q4_0":
            if bias is not None:
                x = qz.mean_center(x, bias)
            u, d = qz.q4_0_quantize(x)
            return qz.pack_nibbles(u), qz.to_fp16(d), None
        raise ValueError(fmt)

    def _pack(self, u):
        if self.bits == 8:
            return qz.stored_int8(u).view(np.uint8)
        return qz.pack_nibbles(u)

    def codes(self, n: int) -> np.ndarray:
        """Unsigned codes u [B,H,n,D] of physical rows [0, n)."""
        r = self.rows[:, :, :n]
        if self.bits == 8:
            return qz.int8_to_codes(r.view(np.int8))
        return qz.unpack_nibbles(r)

    def dequant(self, n: int) -> np.ndarray:
        """float64 [B,H,n,D] values of physical rows [0, n) from the stored bytes."""
        B, H, _, _ = self.rows.shape
        D = self.D
        if self.fmt == "fp16":
            return self.rows[:, :, :n].copy().view(np.float16).astype(np.float64).reshape(B, H, n, D)
        u = self.codes(n)
        if self.fmt == "kivi_chan":
            return qz.dequant_affine(u, self.ch_scale[:, :, None, :], self.ch_zero[:, :, None, :])
        if self.fmt == "kivi_block":
            blk = np.arange(n) // self.group
            return qz.dequant_affine(u, self.blk_scale[:, :, blk, :], self.blk_zero[:, :, blk, :])
        if self.fmt == "affine_token":
            g = self.group
            ug = u.reshape(B, H, n, D // g, g)
            x = qz.dequant_affine(ug, self.tok_scale[:, :, :n, :, None], self.tok_zero[:, :, :n, :, None])
            return x.reshape(B, H, n, D)
        if self.fmt == "q4_0":
            return qz.dequant_q4_0(u, self.tok_scale[:, :, :n])
        raise ValueError(self.fmt)


class OracleCache:
    """One layer's compressed KV cache with its counters (absolute position, stored rows)."""

    def __init__(self, spec: CacheSpec):
        if spec.k_bias is not None and spec.k_format != "q4_0":
            # "kv-cache ... mean-centering for Q4_0", "What's included": the
            # bias is gated to Q4_0 K caches, a mismatch is a hard error.
            raise ValueError("a K mean-centering bias requires q4_0 keys")
        if spec.layout == "ring":
            assert spec.capacity >= spec.sink + spec.window
        self.spec = spec
        self.k = _Side(spec, spec.k_format, spec.k_bits, spec.k_group)
        self.v = _Side(spec, spec.v_format, spec.v_bits, spec.v_group)
        self.pos = 0        # absolute position of the next token (tokens seen)
        self.stored = 0     # physical rows holding live tokens (the quantised bulk)
        if spec.k_format == "kivi_block":
            if spec.layout != "linear" or spec.k_group < 1 or spec.v_format != "affine_token":
                raise ValueError("kivi_block keys need a linear layout, k_group >= 1 and affine_token values")
            B, H, D, R = spec.batch, spec.n_kv_heads, spec.head_dim, spec.k_group
            self.tail_k = np.zeros((B, H, R, D), np.float32)   # full-precision recent tokens
            self.tail_v = np.zeros((B, H, R, D), np.float32)
            self.n_tail = 0

    def calibrate_k(self, k: np.ndarray):
        """Freeze per-channel K scales from k [B,H,n,D] (fp32 values of the io dtype)."""
        self.k.calibrate(np.asarray(k, np.float32))

    def append(self, k: np.ndarray, v: np.ndarray):
        """Quantise and store n new tokens k, v [B,H,n,D] (fp32 values of the io dtype)."""
        spec = self.spec
        k = np.asarray(k, np.float32)
        v = np.asarray(v, np.float32)
        n = k.shape[2]
        if spec.k_format == "kivi_block":
            self._append_residual(k, v)
            return
        kr, ks, kz = self.k.encode(k, spec.k_bias)
        vr, vs, vz = self.v.encode(v, None)
        if spec.layout == "ring":
            dst = []
            for i in range(n):
                p = self.pos + i
                if p < spec.sink or p >= self.pos + n - spec.window:
                    dst.append((i, ring_slot(p, spec.sink, spec.window)))
            self.stored = min(self.pos + n, spec.sink + spec.window)
        else:
            if self.stored + n > spec.capacity:
                raise OverflowError("append beyond capacity")
            dst = [(i, self.stored + i) for i in range(n)]
            self.stored += n
        for i, slot in dst:
            for side, rows, sc, zr in ((self.k, kr, ks, kz), (self.v, vr, vs, vz)):
                side.rows[:, :, slot] = rows[:, :, i]
                if sc is not None:
                    side.tok_scale[:, :, slot] = sc[:, :, i]
                if zr is not None:
                    side.tok_zero[:, :, slot] = zr[:, :, i]
        self.pos += n

    def _append_residual(self, k: np.ndarray, v: np.ndarray):
        """KIVI residual buffer: the tail followed by the new tokens, taken in order; every
        run of R tokens that completes is a closed block, quantised and moved to the bulk;
        the rest stays in the tail.  Call boundaries do not matter."""
        spec = self.spec
        R = spec.k_group
        n = k.shape[2]
        seq_k = np.concatenate([self.tail_k[:, :, : self.n_tail], k], axis=2)
        seq_v = np.concatenate([self.tail_v[:, :, : self.n_tail], v], axis=2)
        nb = seq_k.shape[2] // R
        if self.stored + nb * R > spec.capacity:
            raise OverflowError("append beyond capacity")
        for j in range(nb):
            bk = seq_k[:, :, j * R:(j + 1) * R]
            bv = seq_v[:, :, j * R:(j + 1) * R]
            s32, z32 = qz.kivi_channel_calibrate(bk, spec.k_bits)
            u = qz.kivi_channel_codes(bk, s32, z32, spec.k_bits)
            r0 = self.stored
            self.k.rows[:, :, r0:r0 + R] = self.k._pack(u)
            self.k.blk_scale[:, :, r0 // R] = qz.to_fp16(s32)
            self.k.blk_zero[:, :, r0 // R] = qz.to_fp16(z32)
            vr, vs, vz = self.v.encode(bv, None)
            self.v.rows[:, :, r0:r0 + R] = vr
            self.v.tok_scale[:, :, r0:r0 + R] = vs
            self.v.tok_zero[:, :, r0:r0 + R] = vz
            self.stored += R
        rest = seq_k.shape[2] - nb * R
        self.tail_k[:, :, :rest] = seq_k[:, :, nb * R:]
        self.tail_v[:, :, :rest] = seq_v[:, :, nb * R:]
        self.n_tail = rest
        self.pos += n

    def append_recompute_k(self, k: np.ndarray, v: np.ndarray):
        """Append with the per-channel K range recomputed ("StreamingLLM + KIVI", "KIVI" and
        "Caveats": the range may shift with every new token, so the whole K block is coded
        again; O(T D) per append).  Reading: the stored keys are dequantised in fp32 from the
        stored fp16 scale and zero (the page casts them to fp32 before dequantising), u * s
        then + z, each rounded once; the range is taken over those values and the new keys;
        every stored key is coded again against the new fp32 scale and zero, and the new
        tokens are appended with them.  KIVI per-channel keys, linear or compact layouts."""
        spec = self.spec
        if spec.k_format != "kivi_chan" or spec.layout == "ring":
            raise ValueError("recompute-on-append needs kivi_chan keys and a linear or compact layout")
        k = np.asarray(k, np.float32)
        n_old = self.stored
        if n_old + k.shape[2] > spec.capacity:
            raise OverflowError("append beyond capacity")
        if n_old > 0:
            u = self.k.codes(n_old).astype(np.float32)
            s16 = self.k.ch_scale.astype(np.float32)[:, :, None, :]
            z16 = self.k.ch_zero.astype(np.float32)[:, :, None, :]
            x_old = (u * s16).astype(np.float32) + z16            # two fp32 roundings
            allx = np.concatenate([x_old, k], axis=2)
        else:
            x_old, allx = None, k
        self.k.calibrate(allx)
        if n_old > 0:
            self.k.rows[:, :, :n_old] = self.k._pack(
                qz.kivi_channel_codes(x_old, self.k.ch_scale32, self.k.ch_zero32, self.k.bits))
        self.append(k, v)

    def evict_middle(self):
        """StreamingLLM: drop logical [sink, len - window) when len > sink + window."""
        spec = self.spec
        if spec.layout == "ring":
            return  # the ring already holds exactly the survivors
        if spec.layout != "compact":
            raise ValueError("evict_middle needs a streaming layout")
        L = self.stored
        if L <= spec.sink + spec.window:
            return
        keep = list(range(spec.sink)) + list(range(L - spec.window, L))
        for side in (self.k, self.v):
            for plane in side.token_planes():
                plane[:, :, : len(keep)] = plane[:, :, keep].copy()
        self.stored = len(keep)

    def evict_keepset(self, idx: np.ndarray):
        """SnapKV: keep rows idx [B,H,n_keep] (ascending per head), compacted to rows [0, n_keep)."""
        idx = np.asarray(idx)
        B, H, n_keep = idx.shape
        for b in range(B):
            for h in range(H):
                sel = idx[b, h]
                assert np.all(np.diff(sel) > 0) and sel[-1] < self.stored
                for side in (self.k, self.v):
                    for plane in side.token_planes():
                        plane[b, h, :n_keep] = plane[b, h, sel].copy()
        self.stored = n_keep

    def dequant(self):
        """float64 K-hat, V-hat [B,H,stored,D] of the live rows (kivi_block keys: the bulk,
        then the exact tail, [B,H,stored + n_tail,D])."""
        kh, vh = self.k.dequant(self.stored), self.v.dequant(self.stored)
        if self.spec.k_format == "kivi_block":
            kh = np.concatenate([kh, self.tail_k[:, :, : self.n_tail].astype(np.float64)], axis=2)
            vh = np.concatenate([vh, self.tail_v[:, :, : self.n_tail].astype(np.float64)], axis=2)
        return kh, vh
