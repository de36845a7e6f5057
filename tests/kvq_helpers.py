"""Shared helpers of the GPU parity tests: read the library's device planes as
the oracle's arrays, build matching oracle caches, apply the tolerances."""
from __future__ import annotations

import numpy as np
import torch

from oracle.cache import CacheSpec, OracleCache

# Attention tolerances (max-abs): fp32 outputs 1e-5; bf16 / fp16 outputs
# 2e-3 or one output ulp of the float64 reference, whichever is larger.
TOL_F32 = 1e-5
TOL_LOW = 2e-3


def ulp(ref: np.ndarray, dtype) -> np.ndarray:
    mant = {torch.bfloat16: 7, torch.float16: 10, torch.float32: 23}[dtype]
    a = np.maximum(np.abs(ref), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - mant)


def attn_tolerance(ref: np.ndarray, dtype) -> np.ndarray:
    if dtype == torch.float32:
        return np.full(ref.shape, TOL_F32)
    return np.maximum(TOL_LOW, ulp(ref, dtype))


def assert_attention_close(got: torch.Tensor, ref: np.ndarray, what: str = "") -> float:
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    tol = attn_tolerance(ref, got.dtype)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} outputs out of tolerance, max err {err.max():.3e} "
                           f"(at ref {ref.ravel()[err.argmax()]:.4f})")
    return float(err.max())


def oracle_spec(cache, bias: np.ndarray | None = None) -> CacheSpec:
    """The oracle CacheSpec of a KVCache (from its kvq_config)."""
    c = cache.cfg
    inv_fmt = {0: "fp16", 1: "kivi_chan", 2: "affine_token", 3: "q4_0", 4: "kivi_block"}
    inv_lay = {0: "linear", 1: "compact", 2: "ring"}
    return CacheSpec(batch=c.batch, n_kv_heads=c.n_kv_heads, head_dim=c.head_dim, capacity=c.capacity,
                     layout=inv_lay[c.layout], sink=c.sink, window=c.window,
                     k_format=inv_fmt[c.k_format], k_bits=c.k_bits, k_group=c.k_group,
                     v_format=inv_fmt[c.v_format], v_bits=c.v_bits, v_group=c.v_group, k_bias=bias)


def host(t: torch.Tensor) -> np.ndarray:
    """fp32 numpy copy of a tensor of any io dtype (exact for bf16 / fp16)."""
    return t.detach().float().cpu().numpy()


def _plane(buf: np.ndarray, off: int, nbytes: int) -> np.ndarray:
    return buf[off: off + nbytes]


def gpu_planes(cache) -> dict:
    """The cache's device planes as numpy arrays shaped like the oracle's (all cap_alloc rows)."""
    c, L = cache.cfg, cache.layout
    buf = cache.buf.cpu().numpy()
    B, H, D, ca = c.batch, c.n_kv_heads, c.head_dim, L.cap_alloc
    out = {}
    for side, rb, ng in (("k", L.k_row_bytes, L.k_n_groups), ("v", L.v_row_bytes, L.v_n_groups)):
        off = getattr(L, f"{side}_codes")
        out[f"{side}_rows"] = _plane(buf, off, B * H * ca * rb).reshape(B, H, ca, rb)
        for name in ("tok_scale", "tok_zero"):
            off = getattr(L, f"{side}_{name}")
            if off:
                out[f"{side}_{name}"] = _plane(buf, off, B * H * ca * ng * 2).view(np.float16).reshape(B, H, ca, ng)
    for name, dt, sz in (("ch_scale", np.float16, 2), ("ch_zero", np.float16, 2),
                         ("ch_scale32", np.float32, 4), ("ch_zero32", np.float32, 4)):
        off = getattr(L, f"k_{name}")
        if off:
            out[f"k_{name}"] = _plane(buf, off, B * H * D * sz).view(dt).reshape(B, H, D)
    if L.k_blk_scale:   # KIVI residual buffer: per-block channel metadata and the fp32 tails
        R = c.k_group
        for name in ("blk_scale", "blk_zero"):
            out[f"k_{name}"] = _plane(buf, getattr(L, f"k_{name}"), B * H * (ca // R) * D * 2).view(
                np.float16).reshape(B, H, ca // R, D)
        for side in ("k", "v"):
            out[f"{side}_tail"] = _plane(buf, getattr(L, f"{side}_tail"), B * H * R * D * 4).view(
                np.float32).reshape(B, H, R, D)
    st = _plane(buf, L.state, 32)
    out["pos"] = int(st[:8].view(np.int64)[0])
    out["stored"] = int(st[8:12].view(np.int32)[0])
    out["status"] = int(st[12:16].view(np.int32)[0])
    out["tail"] = int(st[28:32].view(np.int32)[0])
    return out


def _bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype == np.float16 else a.view(np.uint32) if a.dtype == np.float32 else a


def assert_cache_equal(cache, oc: OracleCache, what: str = "", sel=None, planes=None) -> None:
    """Counters and every live row of every plane bit-exact against the oracle cache.

    sel = (b, h) compares only that (batch, kv head) slice of the device cache
    with an oracle cache built for batch 1, one kv head.
    """
    g = dict(planes) if planes is not None else gpu_planes(cache)
    if sel is not None:
        b, h = sel
        for key, val in list(g.items()):
            if isinstance(val, np.ndarray):
                g[key] = val[b:b + 1, h:h + 1]
    assert g["status"] == 0, f"{what}: device status {g['status']}"
    assert g["pos"] == oc.pos and g["stored"] == oc.stored, (
        f"{what}: counters pos {g['pos']} stored {g['stored']} vs oracle {oc.pos} {oc.stored}")
    n = oc.stored
    for side in ("k", "v"):
        o = getattr(oc, side)
        np.testing.assert_array_equal(g[f"{side}_rows"][:, :, :n], o.rows[:, :, :n], err_msg=f"{what}: {side} codes")
        if o.tok_scale is not None:
            np.testing.assert_array_equal(_bits(g[f"{side}_tok_scale"][:, :, :n]), _bits(o.tok_scale[:, :, :n]),
                                          err_msg=f"{what}: {side} token scales")
        if o.tok_zero is not None:
            np.testing.assert_array_equal(_bits(g[f"{side}_tok_zero"][:, :, :n]), _bits(o.tok_zero[:, :, :n]),
                                          err_msg=f"{what}: {side} token zeros")
    if oc.spec.k_format == "kivi_block":
        R, nb, nt = oc.spec.k_group, oc.stored // oc.spec.k_group, oc.n_tail
        assert g["tail"] == nt, f"{what}: tail {g['tail']} vs oracle {nt}"
        for name in ("blk_scale", "blk_zero"):
            np.testing.assert_array_equal(_bits(g[f"k_{name}"][:, :, :nb]), _bits(getattr(oc.k, name)[:, :, :nb]),
                                          err_msg=f"{what}: k {name}")
        np.testing.assert_array_equal(_bits(g["k_tail"][:, :, :nt]), _bits(oc.tail_k[:, :, :nt]),
                                      err_msg=f"{what}: k tail")
        np.testing.assert_array_equal(_bits(g["v_tail"][:, :, :nt]), _bits(oc.tail_v[:, :, :nt]),
                                      err_msg=f"{what}: v tail")
    if oc.k.ch_scale32 is not None:
        for name, arr in (("ch_scale", oc.k.ch_scale), ("ch_zero", oc.k.ch_zero),
                          ("ch_scale32", oc.k.ch_scale32), ("ch_zero32", oc.k.ch_zero32)):
            np.testing.assert_array_equal(_bits(g[f"k_{name}"]), _bits(arr), err_msg=f"{what}: k {name}")
