"""The oracle's pins catch plausible mistakes in the oracle.

Each case below plants one plausible slip in an oracle function on the CPU (a
dropped term, a wrong sign, an off-by-one, a wrong axis or index, a swapped
operand), runs the pin tests of the oracle's area in-process against the
mutated function, and requires at least one pin to fail.  The mutants only
replace attributes for the duration of one case (pytest's monkeypatch), so
the oracle itself is left as it is.  Equivalent rewrites (say, a softmax
without the max shift) are left out: no pin could or should catch them.
"""
from __future__ import annotations

import importlib.util
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import accounting as acc
from oracle import attention as att
from oracle import cache as oc
from oracle import quantize as qz
from oracle import snapkv as sk

HERE = os.path.dirname(os.path.abspath(__file__))
PIN_FILES = {
    "quantize": "test_oracle_quantize.py",
    "cache": "test_oracle_cache.py",
    "attention": "test_oracle_attention_snapkv.py",
}


def _load(area):
    path = os.path.join(HERE, PIN_FILES[area])
    spec = importlib.util.spec_from_file_location(f"_pins_{area}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _golden(name):
    with open(os.path.join(HERE, "golden", name)) as f:
        return json.load(f)


def _cases(fn):
    """Every argument set of a pin test, expanded from its parametrize marks."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    combos = [{}]
    for m in marks:
        names = m.args[0]
        names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
        grown = []
        for c, vals in itertools.product(combos, m.args[1]):
            vals = tuple(vals) if len(names) > 1 else (vals,)
            grown.append({**c, **dict(zip(names, vals))})
        combos = grown
    return combos


def _pins(mod):
    for name in sorted(dir(mod)):
        fn = getattr(mod, name)
        if not (name.startswith("test_") and callable(fn)):
            continue
        if any(m.name in ("slow", "gpu") for m in getattr(fn, "pytestmark", [])):
            continue
        for kw in _cases(fn):
            if "golden" in fn.__code__.co_varnames[: fn.__code__.co_argcount]:
                kw = {**kw, "golden": _golden}
            yield name, fn, kw


def _first_failing_pin(areas):
    """Run the pins of the given areas; return the first that fails, or None."""
    for area in areas:
        mod = _load(area)
        for name, fn, kw in _pins(mod):
            try:
                fn(**kw)
            except Exception as e:  # a failed assertion or a crash both reject the mutant
                return f"{PIN_FILES[area]}::{name}{kw if kw else ''}: {type(e).__name__}"
    return None


def test_unmutated_oracle_passes_every_pin():
    assert _first_failing_pin(["quantize", "cache", "attention"]) is None


# ------------------------------------------------------------------ mutants --
# name -> (areas whose pins must catch it, [(module, attribute, replacement), ...])

MUTANTS = {}


def mutant(name, areas):
    def reg(build):
        MUTANTS[name] = (areas, build)
        return build
    return reg


# quantisers ------------------------------------------------------------------

@mutant("affine scale divides by qMax - qMin + 1", ["quantize"])
def _m():
    def f(xmin, xmax, bits):
        xmin = np.asarray(xmin, np.float32)
        xmax = np.asarray(xmax, np.float32)
        s = np.maximum(qz.EPS, (xmax - xmin) / np.float32(qz.levels(bits) + 1))
        return s.astype(np.float32), xmin.copy()
    return [(qz, "affine_scale_zero", f)]


@mutant("affine zero taken at the maximum", ["quantize"])
def _m():
    orig = qz.affine_scale_zero

    def f(xmin, xmax, bits):
        s, _ = orig(xmin, xmax, bits)
        return s, np.asarray(xmax, np.float32).copy()
    return [(qz, "affine_scale_zero", f)]


@mutant("affine scale without the eps guard", ["quantize"])
def _m():
    def f(xmin, xmax, bits):
        xmin = np.asarray(xmin, np.float32)
        xmax = np.asarray(xmax, np.float32)
        with np.errstate(all="ignore"):
            s = (xmax - xmin) / np.float32(qz.levels(bits))
        return s.astype(np.float32), xmin.copy()
    return [(qz, "affine_scale_zero", f)]


@mutant("affine eps added to the scale instead of bounding it", ["quantize"])
def _m():
    def f(xmin, xmax, bits):
        xmin = np.asarray(xmin, np.float32)
        xmax = np.asarray(xmax, np.float32)
        s = (xmax - xmin) / np.float32(qz.levels(bits)) + qz.EPS
        return s.astype(np.float32), xmin.copy()
    return [(qz, "affine_scale_zero", f)]


@mutant("affine codes truncated instead of rounded", ["quantize"])
def _m():
    def f(x, scale, zero, bits):
        t = (np.asarray(x, np.float32) - zero) / scale
        return np.clip(np.floor(t), 0, qz.levels(bits)).astype(np.uint8)
    return [(qz, "affine_codes", f)]


@mutant("affine codes round half away from zero", ["quantize"])
def _m():
    def f(x, scale, zero, bits):
        t = (np.asarray(x, np.float32) - zero) / scale
        return np.clip(np.floor(t + np.float32(0.5)), 0, qz.levels(bits)).astype(np.uint8)
    return [(qz, "affine_codes", f)]


@mutant("affine codes not clamped", ["quantize"])
def _m():
    def f(x, scale, zero, bits):
        t = (np.asarray(x, np.float32) - zero) / scale
        return np.rint(t).astype(np.int64).astype(np.uint8)
    return [(qz, "affine_codes", f)]


@mutant("affine codes keep qMin added (signed level stored as the code)", ["quantize"])
def _m():
    orig = qz.affine_codes

    def f(x, scale, zero, bits):
        u = orig(x, scale, zero, bits).astype(np.int64)
        return (u + qz.QRANGE[bits][0]).astype(np.uint8)
    return [(qz, "affine_codes", f)]


@mutant("per-channel K range taken over channels instead of tokens", ["quantize"])
def _m():
    def f(k, bits):
        k = np.asarray(k, np.float32)
        return qz.affine_scale_zero(k.min(axis=3), k.max(axis=3), bits)
    return [(qz, "kivi_channel_calibrate", f)]


@mutant("per-token groups cut across tokens (transposed reshape)", ["quantize"])
def _m():
    def f(x, bits, group):
        x = np.asarray(x, np.float32)
        B, H, T, D = x.shape
        g = np.swapaxes(x, 2, 3).reshape(B, H, T, D // group, group)
        s, z = qz.affine_scale_zero(g.min(axis=-1), g.max(axis=-1), bits)
        u = qz.affine_codes(g, s[..., None], z[..., None], bits)
        return np.swapaxes(u.reshape(B, H, D, T), 2, 3).reshape(B, H, T, D), s, z
    return [(qz, "affine_token_quantize", f)]


@mutant("Q4_0 scale max|x| / 8", ["quantize"])
def _m():
    def f(x):
        x = np.asarray(x, np.float32)
        B, H, T, D = x.shape
        blk = x.reshape(B, H, T, D // 32, 32)
        d = (np.abs(blk).max(axis=-1) / np.float32(8)).astype(np.float32)
        sd = np.where(d == 0, np.float32(1), d)
        q = np.clip(np.rint(blk / sd[..., None]), -8, 7)
        q = np.where((d == 0)[..., None], 0, q)
        return (q + 8).astype(np.uint8).reshape(B, H, T, D), d
    return [(qz, "q4_0_quantize", f)]


@mutant("Q4_0 scale from the signed maximum, not max|x|", ["quantize"])
def _m():
    def f(x):
        x = np.asarray(x, np.float32)
        B, H, T, D = x.shape
        blk = x.reshape(B, H, T, D // 32, 32)
        d = (blk.max(axis=-1) / np.float32(7)).astype(np.float32)
        sd = np.where(d == 0, np.float32(1), d)
        q = np.clip(np.rint(blk / sd[..., None]), -8, 7)
        q = np.where((d == 0)[..., None], 0, q)
        return (q + 8).astype(np.uint8).reshape(B, H, T, D), d
    return [(qz, "q4_0_quantize", f)]


@mutant("Q4_0 nibble offset 7 instead of 8", ["quantize"])
def _m():
    orig = qz.q4_0_quantize

    def f(x):
        u, d = orig(x)
        return (u.astype(np.int16) - 1).clip(0, 15).astype(np.uint8), d
    return [(qz, "q4_0_quantize", f)]


@mutant("Q4_0 all-zero block stores the placeholder divisor as its scale", ["quantize"])
def _m():
    def f(x):
        x = np.asarray(x, np.float32)
        B, H, T, D = x.shape
        blk = x.reshape(B, H, T, D // 32, 32)
        d = (np.abs(blk).max(axis=-1) / np.float32(7)).astype(np.float32)
        d = np.where(d == 0, np.float32(1), d)
        q = np.clip(np.rint(blk / d[..., None]), -8, 7)
        return (q + 8).astype(np.uint8).reshape(B, H, T, D), d
    return [(qz, "q4_0_quantize", f)]


@mutant("Q4_0 blocks taken over the token axis", ["quantize"])
def _m():
    orig = qz.q4_0_quantize

    def f(x):
        x = np.asarray(x, np.float32)
        if x.shape[2] % 32:
            return orig(x)
        u, d = orig(np.swapaxes(x, 2, 3))
        return np.swapaxes(u, 2, 3), np.swapaxes(d, 2, 3).reshape(x.shape[:3] + (-1,))
    return [(qz, "q4_0_quantize", f)]


@mutant("mean-centering adds the bias", ["quantize", "cache"])
def _m():
    def f(k, kbar):
        return np.asarray(k, np.float32) + np.asarray(kbar, np.float32)[None, :, None, :]
    return [(qz, "mean_center", f)]


@mutant("mean-centering bias indexed with channels reversed", ["quantize", "cache"])
def _m():
    def f(k, kbar):
        return np.asarray(k, np.float32) - np.asarray(kbar, np.float32)[None, :, None, ::-1]
    return [(qz, "mean_center", f)]


@mutant("nibbles packed high nibble first", ["quantize"])
def _m():
    def f(u):
        u = np.asarray(u, np.uint8)
        return (u[..., 1::2] | (u[..., 0::2] << 4)).astype(np.uint8)
    return [(qz, "pack_nibbles", f)]


@mutant("8-bit rows store the unsigned code", ["quantize", "cache"])
def _m():
    def f(u):
        return np.asarray(u, np.uint8).view(np.int8)
    return [(qz, "stored_int8", f)]


@mutant("affine dequantisation subtracts the zero", ["quantize", "cache"])
def _m():
    def f(u, s16, z16):
        return u.astype(np.float64) * s16.astype(np.float64) - z16.astype(np.float64)
    return [(qz, "dequant_affine", f)]


@mutant("Q4_0 dequantisation offset 7", ["quantize", "cache"])
def _m():
    def f(u, d16):
        B, H, T, D = u.shape
        blk = u.reshape(B, H, T, D // 32, 32).astype(np.float64) - 7.0
        return (blk * d16.astype(np.float64)[..., None]).reshape(B, H, T, D)
    return [(qz, "dequant_q4_0", f)]


@mutant("fp16 metadata truncated toward zero", ["quantize"])
def _m():
    def f(x):
        x = np.asarray(x, np.float32)
        r = x.astype(np.float16)
        over = np.abs(r.astype(np.float32)) > np.abs(x)
        return np.where(over, np.nextafter(r, np.float16(0)), r).astype(np.float16)
    return [(qz, "to_fp16", f)]


@mutant("nibbles unpacked high nibble first", ["quantize", "cache"])
def _m():
    def f(b):
        b = np.asarray(b, np.uint8)
        out = np.empty(b.shape[:-1] + (b.shape[-1] * 2,), dtype=np.uint8)
        out[..., 0::2] = b >> 4
        out[..., 1::2] = b & 0x0F
        return out
    return [(qz, "unpack_nibbles", f)]


@mutant("signed 8-bit level read back with offset 127", ["quantize", "cache"])
def _m():
    return [(qz, "int8_to_codes", lambda q: (np.asarray(q).astype(np.int16) + 127).astype(np.uint8))]


@mutant("new keys coded against the scale and zero of the previous channel", ["quantize", "cache"])
def _m():
    orig = qz.affine_codes

    def f(k, scale, zero, bits):
        return orig(k, np.roll(scale, 1, axis=-1)[:, :, None, :], np.roll(zero, 1, axis=-1)[:, :, None, :], bits)
    return [(qz, "kivi_channel_codes", f)]


# attention -------------------------------------------------------------------

def _attention_variant(kv_head=None, scale_of=None, normalise=True, values_from_keys=False):
    def f(q, khat, vhat, scale=None):
        q = np.asarray(q, np.float64)
        khat = np.asarray(khat, np.float64)
        vhat = np.asarray(vhat, np.float64)
        B, Hq, D = q.shape
        Hkv = khat.shape[1]
        G = Hq // Hkv
        sc = (scale_of(D) if scale_of else 1.0 / math.sqrt(D)) if scale is None else scale
        out = np.empty((B, Hq, D))
        for b in range(B):
            for h in range(Hq):
                kv = kv_head(h, G, Hkv) if kv_head else h // G
                s = khat[b, kv] @ q[b, h] * sc
                p = np.exp(s - s.max())
                if normalise:
                    p /= p.sum()
                out[b, h] = p @ (khat if values_from_keys else vhat)[b, kv]
        return out
    return f


@mutant("attention scale 1/D", ["attention", "cache"])
def _m():
    return [(att, "decode_attention", _attention_variant(scale_of=lambda D: 1.0 / D))]


@mutant("GQA maps query head h to kv head h mod Hkv", ["attention"])
def _m():
    return [(att, "decode_attention", _attention_variant(kv_head=lambda h, G, Hkv: h % Hkv))]


@mutant("softmax weights not normalised", ["attention", "cache"])
def _m():
    return [(att, "decode_attention", _attention_variant(normalise=False))]


@mutant("attention weights the keys instead of the values", ["attention", "cache"])
def _m():
    return [(att, "decode_attention", _attention_variant(values_from_keys=True))]


@mutant("attention ignores a caller-given softmax scale", ["attention"])
def _m():
    orig = att.decode_attention
    return [(att, "decode_attention", lambda q, khat, vhat, scale=None: orig(q, khat, vhat))]


@mutant("split merge sums the l terms without rescaling them", ["attention"])
def _m():
    def f(parts):
        live = [(m, l, a) for m, l, a in parts if m != -math.inf]
        ms = max(m for m, _, _ in live)
        return sum(a * math.exp(m - ms) for m, _, a in live) / sum(l for _, l, _ in live)
    return [(att, "merge_partials", f)]


@mutant("split merge rescales by exp(m* - m_i)", ["attention"])
def _m():
    def f(parts):
        live = [(m, l, a) for m, l, a in parts if m != -math.inf]
        ms = max(m for m, _, _ in live)
        return (sum(a * math.exp(ms - m) for m, _, a in live)
                / sum(l * math.exp(ms - m) for m, l, _ in live))
    return [(att, "merge_partials", f)]


@mutant("split merge averages the splits' outputs", ["attention"])
def _m():
    def f(parts):
        live = [(m, l, a) for m, l, a in parts if m != -math.inf]
        return sum(a / l for _, l, a in live) / len(live)
    return [(att, "merge_partials", f)]


# SnapKV ----------------------------------------------------------------------

def _scores_variant(rows="last", axis=1, reduce="mean", scale_of=None):
    def f(k, obs_window):
        k = np.asarray(k, np.float64)
        S, D = k.shape
        w = min(obs_window, S)
        qrows = k[S - w:] if rows == "last" else k[:w]
        lg = qrows @ k.T * (scale_of(D) if scale_of else 1.0 / math.sqrt(D))
        lg = lg - lg.max(axis=axis, keepdims=True)
        p = np.exp(lg)
        p /= p.sum(axis=axis, keepdims=True)
        return p.mean(axis=0) if reduce == "mean" else p.sum(axis=0)
    return f


@mutant("observation window taken from the first rows", ["attention"])
def _m():
    return [(sk, "obs_window_scores", _scores_variant(rows="first"))]


@mutant("observation softmax over the window axis", ["attention"])
def _m():
    return [(sk, "obs_window_scores", _scores_variant(axis=0))]


@mutant("observation scores summed instead of averaged", ["attention"])
def _m():
    return [(sk, "obs_window_scores", _scores_variant(reduce="sum"))]


@mutant("observation logits scaled by 1/D", ["attention"])
def _m():
    return [(sk, "obs_window_scores", _scores_variant(scale_of=lambda D: 1.0 / D))]


def _select_variant(ties="low", sinks=True, sort=True, n_rest=lambda budget, ns: budget - ns):
    def f(scores, budget, n_sink):
        scores = np.asarray(scores)
        S = scores.shape[0]
        if n_sink > budget:
            raise ValueError("n_sink must not exceed budget")
        if budget >= S:
            return np.arange(S, dtype=np.int32)
        ns = min(n_sink, S) if sinks else 0
        rest = np.arange(ns, S)
        tie_key = rest if ties == "low" else -rest
        order = np.lexsort((tie_key, -scores[rest].astype(np.float64)))
        chosen = rest[order[: n_rest(budget, ns)]]
        out = np.concatenate([np.arange(ns), chosen])
        return (np.sort(out) if sort else out).astype(np.int32)
    return f


@mutant("equal scores keep the higher position", ["attention"])
def _m():
    return [(sk, "select_indices", _select_variant(ties="high"))]


@mutant("sinks not forced", ["attention"])
def _m():
    return [(sk, "select_indices", _select_variant(sinks=False))]


@mutant("kept positions left in score order", ["attention"])
def _m():
    return [(sk, "select_indices", _select_variant(sort=False))]


@mutant("top-budget taken after the sinks (keeps budget + sinks)", ["attention"])
def _m():
    return [(sk, "select_indices", _select_variant(n_rest=lambda budget, ns: budget))]


@mutant("max-pool radius one too small", ["attention"])
def _m():
    def f(scores, kernel_size):
        scores = np.asarray(scores)
        S = scores.shape[-1]
        r = max(kernel_size // 2 - 1, 0)
        out = np.empty_like(scores)
        for j in range(S):
            out[..., j] = scores[..., max(0, j - r): min(S, j + r + 1)].max(axis=-1)
        return out
    return [(sk, "max_pool", f)]


@mutant("keep-set gather reads the rows in reverse", ["attention"])
def _m():
    orig = sk.keepset_gather

    def f(rows, idx):
        return orig(rows, np.asarray(idx)[..., ::-1])
    return [(sk, "keepset_gather", f)]


@mutant("coverage divides by the kept count", ["attention"])
def _m():
    def f(scores, idx):
        scores = np.asarray(scores, np.float64)
        return float(scores[np.asarray(idx)].sum() / len(idx))
    return [(sk, "coverage", f)]


@mutant("random-coverage baseline leaves out the forced sinks", ["attention"])
def _m():
    def f(scores, budget, n_sink):
        scores = np.asarray(scores, np.float64)
        S = scores.shape[0]
        if budget >= S:
            return 1.0
        ns = min(n_sink, S)
        return float(((budget - ns) / (S - ns) * scores[ns:].sum()) / scores.sum())
    return [(sk, "random_coverage", f)]


# cache model -----------------------------------------------------------------

@mutant("ring slot without the sink offset removed", ["cache"])
def _m():
    return [(oc, "ring_slot", lambda p, sink, window: p if p < sink else sink + p % window)]


@mutant("ring wraps over the sinks too", ["cache"])
def _m():
    return [(oc, "ring_slot", lambda p, sink, window: p % (sink + window))]


@mutant("closed-form survivors keep window + 1 recent tokens", ["cache"])
def _m():
    def f(n_seen, sink, window):
        if n_seen <= sink + window:
            return list(range(n_seen))
        return list(range(sink)) + list(range(n_seen - window - 1, n_seen))
    return [(oc, "streaming_survivors", f)]


def _evict_variant(extra_recent=0, move_metadata=True):
    def f(self):
        spec = self.spec
        if spec.layout == "ring":
            return
        if spec.layout != "compact":
            raise ValueError("evict_middle needs a streaming layout")
        L = self.stored
        if L <= spec.sink + spec.window + extra_recent:
            return
        keep = list(range(spec.sink)) + list(range(L - spec.window - extra_recent, L))
        for side in (self.k, self.v):
            planes = side.token_planes() if move_metadata else [side.rows]
            for plane in planes:
                plane[:, :, : len(keep)] = plane[:, :, keep].copy()
        self.stored = len(keep)
    return f


@mutant("eviction keeps one token too many", ["cache"])
def _m():
    return [(oc.OracleCache, "evict_middle", _evict_variant(extra_recent=1))]


@mutant("eviction moves the codes but not their per-token scales", ["cache"])
def _m():
    return [(oc.OracleCache, "evict_middle", _evict_variant(move_metadata=False))]


@mutant("keep-set eviction leaves per-token scales in place", ["cache"])
def _m():
    def f(self, idx):
        idx = np.asarray(idx)
        B, H, n_keep = idx.shape
        for b in range(B):
            for h in range(H):
                for side in (self.k, self.v):
                    side.rows[b, h, :n_keep] = side.rows[b, h, idx[b, h]].copy()
        self.stored = n_keep
    return [(oc.OracleCache, "evict_keepset", f)]


@mutant("per-channel K scales kept in fp32 instead of stored as fp16", ["cache", "quantize"])
def _m():
    def f(self, x):
        s, z = qz.kivi_channel_calibrate(x, self.bits)
        self.ch_scale32, self.ch_zero32 = s, z
        self.ch_scale, self.ch_zero = s.copy(), z.copy()
    return [(oc._Side, "calibrate", f)]


@mutant("residual blocks share one range over every block of the call", ["cache"])
def _m():
    orig = oc.OracleCache._append_residual
    cal = qz.kivi_channel_calibrate

    def f(self, k, v):
        R = self.spec.k_group
        seq_k = np.concatenate([self.tail_k[:, :, : self.n_tail], np.asarray(k, np.float32)], axis=2)
        nb = seq_k.shape[2] // R
        if nb == 0:
            return orig(self, k, v)
        s_all, z_all = cal(seq_k[:, :, : nb * R], self.spec.k_bits)
        qz.kivi_channel_calibrate = lambda bk, bits: (s_all, z_all)
        try:
            return orig(self, k, v)
        finally:
            qz.kivi_channel_calibrate = cal
    return [(oc.OracleCache, "_append_residual", f)]


@mutant("residual tail dropped at each append", ["cache"])
def _m():
    orig = oc.OracleCache._append_residual

    def f(self, k, v):
        orig(self, k, v)
        self.n_tail = 0
    return [(oc.OracleCache, "_append_residual", f)]


@mutant("recompute dequantises the old keys from the fp32 range, not the stored fp16", ["cache"])
def _m():
    def f(self, k, v):
        spec = self.spec
        if spec.k_format != "kivi_chan" or spec.layout == "ring":
            raise ValueError("recompute-on-append needs kivi_chan keys and a linear or compact layout")
        k = np.asarray(k, np.float32)
        n_old = self.stored
        if n_old > 0:
            u = self.k.codes(n_old).astype(np.float32)
            x_old = (u * self.k.ch_scale32[:, :, None, :]).astype(np.float32) + self.k.ch_zero32[:, :, None, :]
            allx = np.concatenate([x_old, k], axis=2)
        else:
            x_old, allx = None, k
        self.k.calibrate(allx)
        if n_old > 0:
            self.k.rows[:, :, :n_old] = self.k._pack(
                qz.kivi_channel_codes(x_old, self.k.ch_scale32, self.k.ch_zero32, self.k.bits))
        self.append(k, v)
    return [(oc.OracleCache, "append_recompute_k", f)]


@mutant("ring bulk append lets an earlier token win a shared slot", ["cache"])
def _m():
    orig_slot = oc.ring_slot
    orig = oc.OracleCache.append

    def f(self, k, v):
        spec = self.spec
        if spec.layout != "ring" or spec.k_format == "kivi_block":
            return orig(self, k, v)
        k = np.asarray(k, np.float32)
        v = np.asarray(v, np.float32)
        n = k.shape[2]
        kr, ks, kz = self.k.encode(k, spec.k_bias)
        vr, vs, vz = self.v.encode(v, None)
        dst = [(i, orig_slot(self.pos + i, spec.sink, spec.window)) for i in reversed(range(n))]
        self.stored = min(self.pos + n, spec.sink + spec.window)
        for i, slot in dst:
            for side, rows, sc, zr in ((self.k, kr, ks, kz), (self.v, vr, vs, vz)):
                side.rows[:, :, slot] = rows[:, :, i]
                if sc is not None:
                    side.tok_scale[:, :, slot] = sc[:, :, i]
                if zr is not None:
                    side.tok_zero[:, :, slot] = zr[:, :, i]
        self.pos += n
    return [(oc.OracleCache, "append", f)]


@mutant("per-token group scales indexed by channel modulo the group count", ["cache", "quantize"])
def _m():
    orig = oc._Side.dequant

    def f(self, n):
        if self.fmt != "affine_token" or self.D // self.group == 1:
            return orig(self, n)
        B, H = self.rows.shape[:2]
        D, g = self.D, self.group
        ng = D // g
        u = self.codes(n).astype(np.float64)
        gi = np.arange(D) % ng                      # should be channel // g
        s = self.tok_scale[:, :, :n][..., gi].astype(np.float64)
        z = self.tok_zero[:, :, :n][..., gi].astype(np.float64)
        return u * s + z
    return [(oc._Side, "dequant", f)]


@mutant("residual bulk read with the first block's scales for every block", ["cache"])
def _m():
    orig = oc._Side.dequant

    def f(self, n):
        if self.fmt != "kivi_block":
            return orig(self, n)
        u = self.codes(n)
        return qz.dequant_affine(u, self.blk_scale[:, :, :1, :], self.blk_zero[:, :, :1, :])
    return [(oc._Side, "dequant", f)]


@mutant("recompute takes the range over the new keys only", ["cache"])
def _m():
    def f(self, k, v):
        spec = self.spec
        if spec.k_format != "kivi_chan" or spec.layout == "ring":
            raise ValueError("recompute-on-append needs kivi_chan keys and a linear or compact layout")
        k = np.asarray(k, np.float32)
        n_old = self.stored
        if n_old > 0:
            u = self.k.codes(n_old).astype(np.float32)
            s16 = self.k.ch_scale.astype(np.float32)[:, :, None, :]
            z16 = self.k.ch_zero.astype(np.float32)[:, :, None, :]
            x_old = (u * s16).astype(np.float32) + z16
        self.k.calibrate(k)
        if n_old > 0:
            self.k.rows[:, :, :n_old] = self.k._pack(
                qz.kivi_channel_codes(x_old, self.k.ch_scale32, self.k.ch_zero32, self.k.bits))
        self.append(k, v)
    return [(oc.OracleCache, "append_recompute_k", f)]


@mutant("compact eviction drops [sink, len - window] one past the end", ["cache"])
def _m():
    def f(self):
        spec = self.spec
        if spec.layout == "ring":
            return
        if spec.layout != "compact":
            raise ValueError("evict_middle needs a streaming layout")
        L = self.stored
        if L <= spec.sink + spec.window:
            return
        keep = list(range(spec.sink)) + list(range(L - spec.window + 1, L))
        for side in (self.k, self.v):
            for plane in side.token_planes():
                plane[:, :, : len(keep)] = plane[:, :, keep].copy()
        self.stored = len(keep)
    return [(oc.OracleCache, "evict_middle", f)]


# byte accounting ---------------------------------------------------------------

@mutant("bits per element count one fp16 word per group", ["cache"])
def _m():
    return [(acc, "bits_per_element", lambda bits, group, meta_bits=16, meta_per_group=1:
             bits + meta_per_group * meta_bits / group)]


@mutant("KIVI cache bytes without the per-channel K scales", ["cache"])
def _m():
    def f(layers, heads, T, D, code_bits, batch=1):
        return 2 * layers * batch * heads * T * D * code_bits // 8 + 2 * layers * batch * heads * T * 2
    return [(acc, "kivi_cache_bytes", f)]


@mutant("Q4_0 blocks counted with a zero point", ["cache"])
def _m():
    orig = acc.side_bytes_per_token

    def f(fmt, bits, group, D):
        return orig(fmt, bits, group, D) + (2 * (D // 32) if fmt == "q4_0" else 0)
    return [(acc, "side_bytes_per_token", f)]


@mutant("decode bytes leave out Q and O", ["cache"])
def _m():
    orig = acc.decode_read_bytes

    def f(w_batch, hkv, hq, D, T, *rest):
        io = rest[-1]
        return orig(w_batch, hkv, hq, D, T, *rest) - 2 * w_batch * hq * D * io
    return [(acc, "decode_read_bytes", f)]


# ------------------------------------------------------------------- runner --

@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    areas, build = MUTANTS[name]
    for owner, attr, repl in build():
        monkeypatch.setattr(owner, attr, repl)
    caught = _first_failing_pin(areas)
    assert caught is not None, f"no pin of {areas} fails when the oracle has: {name}"
