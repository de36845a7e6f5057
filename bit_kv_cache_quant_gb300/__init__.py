"""GB300 compressed KV cache for single-token LLM decode: Python binding.

A thin ctypes layer over ``libkvq.so`` (the C ABI declared in
``include/kvq.h``).  It only marshals arguments: torch tensors become raw
device pointers, the current torch stream becomes the ``cudaStream_t``, and
every step of the path runs in the library's CUDA kernels.  Importing this
package fails loudly when the library has not been built; there is no
fallback of any kind.

The functions named ``kvq_*`` / ``snapkv_*`` mirror the C entry points one
to one; :class:`KVCache` bundles a cache buffer, its handle and a decode
workspace for convenience.
"""
from __future__ import annotations

import ctypes
import os
import re
from ctypes import POINTER, Structure, byref, c_char_p, c_float, c_int32, c_int64, c_size_t, c_void_p
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "kvq.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libkvq.so is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
        "(or bit_kv_cache_quant_gb300/build.py) first")

lib = ctypes.CDLL(LIB_PATH)

# ------------------------------------------------------------------ enums --
KVQ_OK = 0
STATUS_NAMES = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_CAPACITY",
                4: "KVQ_ERR_DEVICE", 5: "KVQ_ERR_CUDA"}
FORMATS = {"fp16": 0, "kivi_chan": 1, "affine_token": 2, "q4_0": 3, "kivi_block": 4}
LAYOUTS = {"linear": 0, "compact": 1, "ring": 2}
DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
EVICT_MIDDLE = 0
EVICT_KEEPSET = 1
APPEND_CALIBRATE_K = 1
APPEND_RECOMPUTE_K = 2
STEP_EARLY_READ = 1
DEV_OK, DEV_OVERFLOW, DEV_BAD_KEEPSET, DEV_TIMEOUT = 0, 1, 2, 3


class kvq_config(Structure):
    _fields_ = [("batch", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32), ("capacity", c_int32),
                ("layout", c_int32), ("sink", c_int32), ("window", c_int32),
                ("k_format", c_int32), ("k_bits", c_int32), ("k_group", c_int32),
                ("v_format", c_int32), ("v_bits", c_int32), ("v_group", c_int32),
                ("k_bias", c_void_p)]


class kvq_cache_layout(Structure):
    _fields_ = [("total_bytes", c_size_t), ("cap_alloc", c_int32), ("k_row_bytes", c_int32),
                ("v_row_bytes", c_int32), ("k_n_groups", c_int32), ("v_n_groups", c_int32),
                ("state", c_size_t), ("split_sem", c_size_t),
                ("k_codes", c_size_t), ("k_tok_scale", c_size_t), ("k_tok_zero", c_size_t),
                ("k_ch_scale", c_size_t), ("k_ch_zero", c_size_t), ("k_ch_scale32", c_size_t),
                ("k_ch_zero32", c_size_t), ("k_bias", c_size_t),
                ("v_codes", c_size_t), ("v_tok_scale", c_size_t), ("v_tok_zero", c_size_t),
                ("k_blk_scale", c_size_t), ("k_blk_zero", c_size_t), ("k_tail", c_size_t), ("v_tail", c_size_t)]


class kvq_stats(Structure):
    _fields_ = [("pos", c_int64), ("stored", c_int32), ("capacity", c_int32), ("device_status", c_int32),
                ("k_calibrated", c_int32), ("cache_bytes", c_size_t), ("live_bytes", c_size_t),
                ("tail", c_int32)]


def _proto(name, res, *args):
    f = getattr(lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_proto("kvq_cache_layout_query", c_int32, POINTER(kvq_config), POINTER(kvq_cache_layout))
_proto("kvq_cache_init", c_int32, POINTER(kvq_config), c_void_p, c_size_t, c_void_p, POINTER(c_void_p))
_proto("kvq_cache_release", None, c_void_p)
_proto("kvq_append", c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p)
_proto("kvq_convert", c_int32, c_void_p, c_void_p, c_void_p, c_int64, c_int32, c_int32, c_int32, c_void_p)
_proto("kvq_evict", c_int32, c_void_p, c_int32, c_void_p, c_int32, c_void_p)
_proto("kvq_decode_workspace_bytes", c_size_t, c_void_p, c_int32)
_proto("kvq_decode_plan_query", c_int32, POINTER(kvq_config), c_int32, c_int32, POINTER(c_int32), POINTER(c_int32),
       POINTER(c_int32))
_proto("kvq_decode_attn", c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_float, c_void_p, c_size_t,
       c_void_p)
_proto("kvq_append_decode", c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_int32,
       c_float, c_void_p, c_size_t, c_int32, c_void_p)
_proto("kvq_append_decode_layers", c_int32, c_int32, POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p), c_int32,
       POINTER(c_void_p), POINTER(c_void_p), c_int32, c_int32, c_float, POINTER(c_void_p), POINTER(c_size_t), c_int32,
       c_void_p)
_proto("kvq_test_stall_decode_tiles", None, c_int32)
_proto("snapkv_workspace_bytes", c_size_t, c_int32, c_int32, c_int32, c_int32, c_int32)
_proto("snapkv_pool", c_int32, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p)
_proto("snapkv_select", c_int32, c_void_p, c_int64, c_int32, c_int32, c_int32, c_int32, c_int32, c_int32, c_int32,
       c_void_p, c_void_p, c_void_p, c_size_t, c_void_p)
_proto("snapkv_topk", c_int32, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p)
_proto("kvq_stats_read", c_int32, c_void_p, POINTER(kvq_stats))
_proto("kvq_clear_status", c_int32, c_void_p, c_void_p)
_proto("kvq_last_launch_count", c_int32)
_proto("kvq_last_error", c_char_p)
_proto("kvq_abi_version", c_int32)


class KvqError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _check(status: int) -> None:
    if status != KVQ_OK:
        raise KvqError(status, (lib.kvq_last_error() or b"").decode())


def declared_functions() -> list:
    """Names of the functions include/kvq.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:kvq_status|size_t|void|int32_t|const char\*)\s+(\w+)\s*\(", text, re.M)))


def _stream(stream=None) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev_ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def make_config(batch, n_kv_heads, head_dim, capacity, k_format, k_bits, k_group, v_format, v_bits, v_group,
                layout="linear", sink=0, window=0, k_bias: Optional[torch.Tensor] = None) -> kvq_config:
    return kvq_config(batch, n_kv_heads, head_dim, capacity, LAYOUTS[layout], sink, window,
                      FORMATS[k_format], k_bits, k_group, FORMATS[v_format], v_bits, v_group,
                      None if k_bias is None else _dev_ptr(k_bias))


# ------------------------------------------------------- C entry points --

def kvq_cache_layout_query(cfg: kvq_config) -> kvq_cache_layout:
    lay = kvq_cache_layout()
    _check(lib.kvq_cache_layout_query(byref(cfg), byref(lay)))
    return lay


def kvq_cache_init(cfg: kvq_config, buf: torch.Tensor, stream=None) -> c_void_p:
    h = c_void_p()
    _check(lib.kvq_cache_init(byref(cfg), _dev_ptr(buf), buf.numel() * buf.element_size(), _stream(stream),
                              byref(h)))
    return h


def kvq_append(cache, k: torch.Tensor, v: torch.Tensor, n_tokens: int, in_dtype: int, flags: int = 0,
               stream=None) -> None:
    _check(lib.kvq_append(cache, _dev_ptr(k), _dev_ptr(v), n_tokens, in_dtype, flags, _stream(stream)))


def kvq_convert(cache, k: torch.Tensor, v: torch.Tensor, head_stride: int, n_tokens: int, in_dtype: int,
                flags: int = 0, stream=None) -> None:
    _check(lib.kvq_convert(cache, _dev_ptr(k), _dev_ptr(v), head_stride, n_tokens, in_dtype, flags,
                           _stream(stream)))


def kvq_evict(cache, mode: int, keep_idx: Optional[torch.Tensor] = None, n_keep: int = 0, stream=None) -> None:
    _check(lib.kvq_evict(cache, mode, _dev_ptr(keep_idx), n_keep, _stream(stream)))


def kvq_decode_workspace_bytes(cache, n_q_heads: int) -> int:
    return lib.kvq_decode_workspace_bytes(cache, n_q_heads)


def kvq_decode_plan_query(cfg: kvq_config, n_q_heads: int, sms: int):
    """(splits, tensor-core splits, wide) of the decode launch for this configuration and SM count."""
    ns, ntc, wide = c_int32(), c_int32(), c_int32()
    _check(lib.kvq_decode_plan_query(byref(cfg), n_q_heads, sms, byref(ns), byref(ntc), byref(wide)))
    return ns.value, ntc.value, wide.value


def kvq_decode_attn(cache, q: torch.Tensor, out: torch.Tensor, n_q_heads: int, io_dtype: int,
                    softmax_scale: float = 0.0, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.kvq_decode_attn(cache, _dev_ptr(q), _dev_ptr(out), n_q_heads, io_dtype, softmax_scale,
                               _dev_ptr(workspace), ws_bytes, _stream(stream)))


def kvq_append_decode(cache, k: torch.Tensor, v: torch.Tensor, in_dtype: int, q: torch.Tensor, out: torch.Tensor,
                      n_q_heads: int, io_dtype: int, softmax_scale: float = 0.0,
                      workspace: Optional[torch.Tensor] = None, flags: int = 0, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.kvq_append_decode(cache, _dev_ptr(k), _dev_ptr(v), in_dtype, _dev_ptr(q), _dev_ptr(out), n_q_heads,
                                 io_dtype, softmax_scale, _dev_ptr(workspace), ws_bytes, flags, _stream(stream)))


def kvq_append_decode_layers(caches: list, ks: list, vs: list, in_dtype: int, qs: list, outs: list, n_q_heads: int,
                             io_dtype: int, softmax_scale: float = 0.0, workspaces: Optional[list] = None,
                             flags: int = 0, stream=None) -> None:
    n = len(caches)
    arr = lambda xs: (c_void_p * n)(*xs)
    ws = wsb = None
    if workspaces is not None:
        ws = arr([_dev_ptr(w) for w in workspaces])
        wsb = (c_size_t * n)(*[0 if w is None else w.numel() * w.element_size() for w in workspaces])
    _check(lib.kvq_append_decode_layers(n, arr([c.value for c in caches]), arr([_dev_ptr(t) for t in ks]),
                                        arr([_dev_ptr(t) for t in vs]), in_dtype, arr([_dev_ptr(t) for t in qs]),
                                        arr([_dev_ptr(t) for t in outs]), n_q_heads, io_dtype, softmax_scale, ws, wsb,
                                        flags, _stream(stream)))


class LayerStep:
    """One decode step over a stack of layer caches as one call (kvq_append_decode_layers):
    layer l appends ks[l], vs[l] [B, Hkv, 1, D] to caches[l], evicts, and attends with
    qs[l] [B, Hq, D] into outs[l].  The per-layer pointer arrays are built once here, so the
    tensors must stay alive and in place while the step is in use."""

    def __init__(self, caches: list, ks: list, vs: list, qs: list, outs: list, softmax_scale: float = 0.0):
        n = len(caches)
        if not n or not all(len(x) == n for x in (ks, vs, qs, outs)):
            raise ValueError("one k, v, q and out per cache")
        for c, k, v, q, o in zip(caches, ks, vs, qs, outs):
            c._check_rows(k, v)
            if k.shape[2] != 1:
                raise ValueError("a step takes one token per (batch row, kv head)")
            if q.dim() != 3 or q.shape[0] != c.batch or q.shape[2] != c.head_dim or q.dtype not in DTYPES:
                raise ValueError(f"q must be [{c.batch}, Hq, {c.head_dim}] fp32 / bf16 / fp16")
            if o.shape != q.shape or o.dtype != q.dtype:
                raise ValueError("out must have q's shape and dtype")
        self.n = n
        self.hq = qs[0].shape[1]
        self.in_dtype, self.io_dtype = DTYPES[ks[0].dtype], DTYPES[qs[0].dtype]
        self.softmax_scale = softmax_scale
        ws = [c.workspace(self.hq) for c in caches]
        arr = lambda xs: (c_void_p * n)(*xs)
        self._args = (arr([c.handle.value for c in caches]), arr([_dev_ptr(t) for t in ks]),
                      arr([_dev_ptr(t) for t in vs]), arr([_dev_ptr(t) for t in qs]),
                      arr([_dev_ptr(t) for t in outs]), arr([_dev_ptr(w) for w in ws]),
                      (c_size_t * n)(*[0 if w is None else w.numel() * w.element_size() for w in ws]))
        self._keep = (list(caches), list(ks), list(vs), list(qs), list(outs), ws)
        self._handles = tuple(c.handle for c in caches)   # the handle objects: reset() makes new ones
        self.launches = 0

    def run(self, early_read: bool = False, stream=None) -> None:
        """early_read: the kernel just before this call on the stream writes none of the caches."""
        if any(c.handle is not h for c, h in zip(self._keep[0], self._handles)):
            raise ValueError("a cache of this step was reset or released; build a new LayerStep")
        h, k, v, q, o, ws, wsb = self._args
        _check(lib.kvq_append_decode_layers(self.n, h, k, v, self.in_dtype, q, o, self.hq, self.io_dtype,
                                            self.softmax_scale, ws, wsb, STEP_EARLY_READ if early_read else 0,
                                            _stream(stream)))
        self.launches = kvq_last_launch_count()


def kvq_test_stall_decode_tiles(on: bool) -> None:
    lib.kvq_test_stall_decode_tiles(1 if on else 0)


def snapkv_workspace_bytes(batch, n_kv_heads, S, head_dim, obs_window) -> int:
    return lib.snapkv_workspace_bytes(batch, n_kv_heads, S, head_dim, obs_window)


def snapkv_select(k: torch.Tensor, head_stride: int, batch: int, n_kv_heads: int, S: int, head_dim: int,
                  obs_window: int, budget: int, n_sink: int, scores_out: Optional[torch.Tensor],
                  idx_out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    _check(lib.snapkv_select(_dev_ptr(k), head_stride, batch, n_kv_heads, S, head_dim, obs_window, budget, n_sink,
                             _dev_ptr(scores_out), _dev_ptr(idx_out), _dev_ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)))


def snapkv_pool(scores: torch.Tensor, pooled: torch.Tensor, kernel_size: int, stream=None) -> torch.Tensor:
    """Max-pool smoothing of scores [B, Hkv, S] (fp32, device) into pooled (same shape)."""
    B, H, S = scores.shape
    _check(lib.snapkv_pool(_dev_ptr(scores), _dev_ptr(pooled), B, H, S, kernel_size, _stream(stream)))
    return pooled


def snapkv_topk(scores: torch.Tensor, batch: int, n_kv_heads: int, S: int, budget: int, n_sink: int,
                idx_out: torch.Tensor, stream=None) -> None:
    _check(lib.snapkv_topk(_dev_ptr(scores), batch, n_kv_heads, S, budget, n_sink, _dev_ptr(idx_out),
                           _stream(stream)))


def kvq_stats_read(cache) -> kvq_stats:
    st = kvq_stats()
    status = lib.kvq_stats_read(cache, byref(st))
    if status not in (KVQ_OK, 4):      # KVQ_ERR_DEVICE still fills the counters
        _check(status)
    return st


def kvq_clear_status(cache, stream=None) -> None:
    _check(lib.kvq_clear_status(cache, _stream(stream)))


def kvq_last_launch_count() -> int:
    return lib.kvq_last_launch_count()


# ------------------------------------------------------------ convenience --

class KVCache:
    """One layer's compressed cache: a device buffer, its handle and a decode workspace."""

    def __init__(self, batch, n_kv_heads, head_dim, capacity, k_format="fp16", k_bits=16, k_group=0,
                 v_format="fp16", v_bits=16, v_group=0, layout="linear", sink=0, window=0,
                 k_bias: Optional[torch.Tensor] = None, device="cuda", stream=None):
        self.cfg = make_config(batch, n_kv_heads, head_dim, capacity, k_format, k_bits, k_group, v_format, v_bits,
                               v_group, layout, sink, window, k_bias)
        self.layout = kvq_cache_layout_query(self.cfg)
        self._bias = k_bias      # kept alive until the stream-ordered copy in kvq_cache_init has run
        self.buf = torch.empty(self.layout.total_bytes, dtype=torch.uint8, device=device)
        self.handle = kvq_cache_init(self.cfg, self.buf, stream)
        self.batch, self.n_kv_heads, self.head_dim = batch, n_kv_heads, head_dim
        self._ws = {}
        self.launches = 0

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            lib.kvq_cache_release(h)
            self.handle = None

    def reset(self, stream=None) -> None:
        """Empties the cache (counters to zero) on the same device buffer."""
        lib.kvq_cache_release(self.handle)
        self.handle = None
        self.handle = kvq_cache_init(self.cfg, self.buf, stream)

    def _check_rows(self, k: torch.Tensor, v: torch.Tensor) -> None:
        """k, v: one shape [B, Hkv, n, D] of this cache and one dtype: the C call gets raw pointers and
        reads both with k's dtype.  One short-circuit test on the common path (eager decode calls it
        once per layer)."""
        s = k.shape
        if (s != v.shape or k.dtype is not v.dtype or len(s) != 4 or s[0] != self.batch
                or s[1] != self.n_kv_heads or s[3] != self.head_dim):
            if s != v.shape or k.dtype is not v.dtype:
                raise ValueError(f"k {tuple(s)} {k.dtype} and v {tuple(v.shape)} {v.dtype} must match")
            raise ValueError(f"k and v must be [{self.batch}, {self.n_kv_heads}, n, {self.head_dim}], "
                             f"got {tuple(s)}")
        if k.dtype not in DTYPES:
            raise ValueError(f"unsupported input dtype {k.dtype}")

    def append(self, k: torch.Tensor, v: torch.Tensor, calibrate_k: bool = False, recompute_k: bool = False,
               stream=None) -> None:
        self._check_rows(k, v)
        n = k.shape[2]
        flags = (APPEND_CALIBRATE_K if calibrate_k else 0) | (APPEND_RECOMPUTE_K if recompute_k else 0)
        kvq_append(self.handle, k, v, n, DTYPES[k.dtype], flags, stream)
        self.launches += kvq_last_launch_count()

    def convert(self, k: torch.Tensor, v: torch.Tensor, n_tokens: int, calibrate_k: bool = False,
                stream=None) -> None:
        """Quantises the first n_tokens tokens of a dense cache k, v [B, Hkv, C, D] (C >= n_tokens,
        rows contiguous) into this cache."""
        if k.shape != v.shape or k.dim() != 4 or not k.is_contiguous() or not v.is_contiguous():
            raise ValueError("k and v must be contiguous [B, Hkv, C, D] tensors of one shape")
        self._check_rows(k, v)
        if not 1 <= n_tokens <= k.shape[2]:
            raise ValueError(f"n_tokens must be in 1..{k.shape[2]}")
        kvq_convert(self.handle, k, v, k.shape[2], n_tokens, DTYPES[k.dtype],
                    APPEND_CALIBRATE_K if calibrate_k else 0, stream)
        self.launches += kvq_last_launch_count()

    def evict_middle(self, stream=None) -> None:
        kvq_evict(self.handle, EVICT_MIDDLE, None, 0, stream)
        self.launches += kvq_last_launch_count()

    def evict_keepset(self, idx: torch.Tensor, stream=None) -> None:
        kvq_evict(self.handle, EVICT_KEEPSET, idx, idx.shape[-1], stream)
        self.launches += kvq_last_launch_count()

    def workspace(self, n_q_heads: int) -> Optional[torch.Tensor]:
        if n_q_heads not in self._ws:
            nb = kvq_decode_workspace_bytes(self.handle, n_q_heads)
            self._ws[n_q_heads] = torch.empty(nb, dtype=torch.uint8, device=self.buf.device) if nb else None
        return self._ws[n_q_heads]

    def decode_attn(self, q: torch.Tensor, out: Optional[torch.Tensor] = None, softmax_scale: float = 0.0,
                    stream=None) -> torch.Tensor:
        s = q.shape
        if len(s) != 3 or s[0] != self.batch or s[2] != self.head_dim or q.dtype not in DTYPES:
            raise ValueError(f"q must be [{self.batch}, Hq, {self.head_dim}] fp32 / bf16 / fp16, "
                             f"got {tuple(q.shape)} {q.dtype}")
        if out is None:
            out = torch.empty_like(q)
        elif out.shape != q.shape or out.dtype != q.dtype:
            raise ValueError("out must have q's shape and dtype")
        hq = q.shape[1]
        kvq_decode_attn(self.handle, q, out, hq, DTYPES[q.dtype], softmax_scale, self.workspace(hq), stream)
        self.launches += kvq_last_launch_count()
        return out

    def append_decode(self, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor, out: Optional[torch.Tensor] = None,
                      softmax_scale: float = 0.0, early_read: bool = False, stream=None) -> torch.Tensor:
        """One decode step: append the token k, v [B, Hkv, 1, D], evict (streaming layouts) and attend
        with q [B, Hq, D] over the cache including that token.  early_read: the kernel just before
        this call on the stream writes neither this cache nor its counters (KVQ_STEP_EARLY_READ)."""
        self._check_rows(k, v)
        if k.shape[2] != 1:
            raise ValueError("append_decode takes one token per (batch row, kv head)")
        s = q.shape
        if len(s) != 3 or s[0] != self.batch or s[2] != self.head_dim or q.dtype not in DTYPES:
            raise ValueError(f"q must be [{self.batch}, Hq, {self.head_dim}] fp32 / bf16 / fp16, "
                             f"got {tuple(q.shape)} {q.dtype}")
        if out is None:
            out = torch.empty_like(q)
        elif out.shape != q.shape or out.dtype != q.dtype:
            raise ValueError("out must have q's shape and dtype")
        hq = q.shape[1]
        kvq_append_decode(self.handle, k, v, DTYPES[k.dtype], q, out, hq, DTYPES[q.dtype], softmax_scale,
                          self.workspace(hq), STEP_EARLY_READ if early_read else 0, stream)
        self.launches += kvq_last_launch_count()
        return out

    def stats(self) -> kvq_stats:
        return kvq_stats_read(self.handle)

    def plane(self, name: str, nbytes: int) -> torch.Tensor:
        """uint8 view of `nbytes` bytes of plane `name` (a kvq_cache_layout field)."""
        off = getattr(self.layout, name)
        return self.buf[off: off + nbytes]


def snapkv(k: torch.Tensor, obs_window: int, budget: int, n_sink: int, want_scores: bool = True, stream=None):
    """Scores and kept indices of fp16 keys k [B, Hkv, S, D]."""
    B, H, S, D = k.shape
    ws = torch.empty(snapkv_workspace_bytes(B, H, S, D, obs_window), dtype=torch.uint8, device=k.device)
    scores = torch.empty((B, H, S), dtype=torch.float32, device=k.device) if want_scores else None
    idx = torch.empty((B, H, min(budget, S)), dtype=torch.int32, device=k.device)
    snapkv_select(k, S, B, H, S, D, obs_window, budget, n_sink, scores, idx, ws, stream)
    return scores, idx
