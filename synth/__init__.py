"""Seeded synthetic inputs for the compressed KV-cache workloads.

This module is shared by the CUDA path's tests/bench and by the CPU oracle.
It holds shapes, seeds and value distributions only: no quantisation,
eviction, selection or attention arithmetic lives here.  Every tensor is
drawn from a ``torch.Generator`` seeded from (workload seed, layer, stream
name), so the same call returns the same bits on the same machine whether
it runs on the host (small cases) or on the device (full-size cases).  The
oracle always receives the very tensor the device received (copied to the
host), never a regenerated one.

Workloads follow the five shapes the pages discuss:

* a tinygpt-sized StreamingLLM + KIVI int8 cache (sink 4 + window 256),
* an mlx-lm-style per-token group-64 affine 4-bit cache on a Llama-3.2-3B
  attention shape at 8K context,
* a llama.cpp-style symmetric Q4_0 K cache with per-(kv-head, channel)
  mean-centering bias and int8 per-token V at 32K context, batch 8,
* a SnapKV prefill eviction (16K prompt to a 512-token budget) followed by
  fp16 decode appends,
* a long streaming decode with KIVI int4 and a 4 + 4096 ring,
* a KIVI residual buffer (full-precision tail, int4 keys per channel in
  closed blocks of 128 tokens) on the Llama-3.2-3B attention shape at 8K.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "get_workload",
    "normal",
    "layer_inputs",
    "decode_token_inputs",
    "snapkv_prefill",
    "k_bias",
    "rope_rotate",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    context: int                 # tokens held by the cache when decode starts
    k_format: str                # "fp16" | "kivi_chan" | "affine_token" | "q4_0" | "kivi_block"
    k_bits: int
    k_group: int
    v_format: str                # "fp16" | "affine_token"
    v_bits: int
    v_group: int
    io_dtype: str                # dtype of K/V/Q inputs and of the attention output
    layout: str = "linear"       # "linear" | "compact" | "ring"
    sink: int = 0
    window: int = 0
    seed: int = 1000
    # value-distribution knobs
    k_channel_offset_sigma: float = 0.0   # K += offset[kvh, d] ~ N(0, sigma)
    k_outlier_fraction: float = 0.0       # fraction of (kvh, d) K channels scaled
    k_outlier_scale: float = 1.0
    k_bias_sigma: float = 0.0             # K = N(0,1) + kbar[kvh, d], kbar ~ N(0, sigma)
    use_k_bias: bool = False              # the cache subtracts kbar before quantising
    sink_rows: int = 0                    # rows [0, sink_rows) of K scaled by sink_row_scale
    sink_row_scale: float = 1.0
    rope_theta: float = 0.0               # > 0: RoPE baked into K (and Q) at absolute positions
    # SnapKV prefill
    prompt_len: int = 0
    obs_window: int = 0
    budget: int = 0
    n_sink: int = 0
    decode_steps: int = 0
    # long streaming decode
    generated_steps: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        # tinygpt-shaped single decode step, KIVI int8, sink 4 + window 256.
        Workload(
            name="tinygpt_kivi8_sink4_win256",
            batch=1, layers=1, n_q_heads=8, n_kv_heads=8, head_dim=32,
            context=260,
            k_format="kivi_chan", k_bits=8, k_group=0,
            v_format="affine_token", v_bits=8, v_group=32,
            io_dtype="float32", layout="compact", sink=4, window=256,
            seed=1001, k_channel_offset_sigma=2.0,
        ),
        # mlx-lm style per-token group-64 affine 4-bit, Llama-3.2-3B attention.
        Workload(
            name="llama3b_mlx_affine4_g64_ctx8k",
            batch=1, layers=28, n_q_heads=24, n_kv_heads=8, head_dim=128,
            context=8192,
            k_format="affine_token", k_bits=4, k_group=64,
            v_format="affine_token", v_bits=4, v_group=64,
            io_dtype="bfloat16", seed=1002,
            k_outlier_fraction=0.01, k_outlier_scale=10.0,
        ),
        # llama.cpp-style Q4_0 K with mean-centering bias, int8 per-token V.
        Workload(
            name="q4_0_centered_k_int8_v_ctx32k_b8",
            batch=8, layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
            context=32768,
            k_format="q4_0", k_bits=4, k_group=32,
            v_format="affine_token", v_bits=8, v_group=128,
            io_dtype="bfloat16", seed=1003,
            k_bias_sigma=1.5, use_k_bias=True,
        ),
        # SnapKV prefill eviction (16K prompt -> 512 budget), then fp16 decode.
        Workload(
            name="snapkv_s16k_budget512_fp16",
            batch=1, layers=1, n_q_heads=24, n_kv_heads=8, head_dim=128,
            context=512,
            k_format="fp16", k_bits=16, k_group=0,
            v_format="fp16", v_bits=16, v_group=0,
            io_dtype="float16", seed=1004,
            sink_rows=4, sink_row_scale=8.0,
            prompt_len=16384, obs_window=32, budget=512, n_sink=4,
            decode_steps=256,
        ),
        # Long streaming decode: KIVI int4 (frozen per-channel K, V g32), ring 4 + 4096.
        Workload(
            name="kivi4_ring_sink4_win4096_b64",
            batch=64, layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
            context=4100,
            k_format="kivi_chan", k_bits=4, k_group=0,
            v_format="affine_token", v_bits=4, v_group=32,
            io_dtype="bfloat16", layout="ring", sink=4, window=4096,
            seed=1005, k_channel_offset_sigma=2.0, rope_theta=10000.0,
            generated_steps=40000,
        ),
        # KIVI residual buffer: fp32 tail, int4 K per channel in closed blocks of 128, V g32.
        Workload(
            name="kivi4_residual_r128_ctx8k",
            batch=1, layers=28, n_q_heads=24, n_kv_heads=8, head_dim=128,
            context=8192 + 100,
            k_format="kivi_block", k_bits=4, k_group=128,
            v_format="affine_token", v_bits=4, v_group=32,
            io_dtype="bfloat16", seed=1006, k_channel_offset_sigma=2.0,
        ),
    ]
}

# Short aliases used on command lines.
ALIASES = {
    "tinygpt": "tinygpt_kivi8_sink4_win256",
    "mlx8k": "llama3b_mlx_affine4_g64_ctx8k",
    "q4_0_32k": "q4_0_centered_k_int8_v_ctx32k_b8",
    "snapkv": "snapkv_s16k_budget512_fp16",
    "ring": "kivi4_ring_sink4_win4096_b64",
    "residual": "kivi4_residual_r128_ctx8k",
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[ALIASES.get(name, name)]


_DTYPES = {"float32": torch.float32, "bfloat16": torch.bfloat16, "float16": torch.float16}


def torch_dtype(name: str) -> torch.dtype:
    return _DTYPES[name]


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def normal(shape, *seed_parts, device="cpu") -> torch.Tensor:
    """fp32 N(0, 1) tensor of `shape`, reproducible from `seed_parts`."""
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*seed_parts))
    return torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)


def _channel_offsets(w: Workload, layer: int, device) -> Optional[torch.Tensor]:
    if w.k_channel_offset_sigma == 0.0:
        return None
    off = normal((w.n_kv_heads, w.head_dim), w.seed, layer, "k_channel_offset", device=device)
    return off * w.k_channel_offset_sigma


def k_bias(w: Workload, layer: int, device="cpu") -> Optional[torch.Tensor]:
    """The per-(kv-head, channel) K mean kbar carried by the synthetic keys, fp32 [Hkv, D]."""
    if w.k_bias_sigma == 0.0:
        return None
    return normal((w.n_kv_heads, w.head_dim), w.seed, layer, "k_bias", device=device) * w.k_bias_sigma


def _outlier_mask(w: Workload, layer: int, device) -> Optional[torch.Tensor]:
    if w.k_outlier_fraction == 0.0:
        return None
    n = w.n_kv_heads * w.head_dim
    k = max(1, int(round(w.k_outlier_fraction * n)))
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed(w.seed, layer, "k_outliers"))
    idx = torch.randperm(n, generator=g)[:k]
    scale = torch.ones(n, dtype=torch.float32)
    scale[idx] = w.k_outlier_scale
    return scale.view(w.n_kv_heads, w.head_dim).to(device)


def rope_rotate(x: torch.Tensor, positions: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotate-half rotary embedding of fp32 x [..., T, D] at absolute `positions` [T].

    Input preparation only: the cache stores keys that already carry their
    rotation, exactly as a model hands them over after its RoPE step.
    """
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-torch.arange(0, half, device=x.device, dtype=torch.float64) / half)
    ang = positions.to(torch.float64)[:, None] * inv[None, :]
    cos = torch.cos(ang).to(torch.float32)
    sin = torch.sin(ang).to(torch.float32)
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def _finish_k(w: Workload, layer: int, k: torch.Tensor, positions: torch.Tensor) -> torch.Tensor:
    dev = k.device
    off = _channel_offsets(w, layer, dev)
    if off is not None:
        k = k + off[None, :, None, :]
    mask = _outlier_mask(w, layer, dev)
    if mask is not None:
        k = k * mask[None, :, None, :]
    kb = k_bias(w, layer, dev)
    if kb is not None:
        k = k + kb[None, :, None, :]
    if w.sink_rows > 0:
        sel = positions < w.sink_rows
        if bool(sel.any()):
            k = k.clone()
            k[:, :, sel, :] *= w.sink_row_scale
    if w.rope_theta > 0.0:
        k = rope_rotate(k, positions, w.rope_theta)
    return k


def layer_inputs(w: Workload, layer: int, start: int, n: int, device="cpu", batch: Optional[int] = None):
    """K, V for absolute positions [start, start + n) of one layer: [B, Hkv, n, D] in io dtype.

    Tokens are generated per (layer, position block) so that any window of
    positions can be produced without producing the ones before it.
    """
    B = w.batch if batch is None else batch
    dt = torch_dtype(w.io_dtype)
    positions = torch.arange(start, start + n, device=device)
    k = normal((B, w.n_kv_heads, n, w.head_dim), w.seed, layer, "k", start, n, B, device=device)
    v = normal((B, w.n_kv_heads, n, w.head_dim), w.seed, layer, "v", start, n, B, device=device)
    k = _finish_k(w, layer, k, positions)
    return k.to(dt).contiguous(), v.to(dt).contiguous()


def decode_token_inputs(w: Workload, layer: int, step: int, position: int, device="cpu", batch: Optional[int] = None):
    """Q [B, Hq, D] and one new K/V token [B, Hkv, 1, D] for a decode step at `position`."""
    B = w.batch if batch is None else batch
    dt = torch_dtype(w.io_dtype)
    q = normal((B, w.n_q_heads, w.head_dim), w.seed, layer, "q", step, B, device=device)
    if w.rope_theta > 0.0:
        q = rope_rotate(q[:, :, None, :], torch.tensor([position], device=device), w.rope_theta)[:, :, 0, :]
    k = normal((B, w.n_kv_heads, 1, w.head_dim), w.seed, layer, "k_step", step, B, device=device)
    v = normal((B, w.n_kv_heads, 1, w.head_dim), w.seed, layer, "v_step", step, B, device=device)
    k = _finish_k(w, layer, k, torch.tensor([position], device=device))
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()


def snapkv_prefill(w: Workload, layer: int = 0, device="cpu", prompt_len: Optional[int] = None,
                   batch: Optional[int] = None):
    """Prompt K, V [B, Hkv, S, D] fp16 for a SnapKV prefill (rows [0, sink_rows) scaled)."""
    S = w.prompt_len if prompt_len is None else prompt_len
    return layer_inputs(w, layer, 0, S, device=device, batch=batch)


def planted_top_scores(S: int, n_sink: int, planted, seed: int) -> torch.Tensor:
    """fp32 scores in [0, 1): small noise everywhere, large values at `planted` positions."""
    s = (normal((S,), seed, "planted").abs() * 1e-4).clamp_(max=1e-3)
    s[list(planted)] = 0.5 + 0.01 * torch.arange(len(planted), dtype=torch.float32)
    return s
