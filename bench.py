"""Decode-step benchmark of the GB300 compressed KV cache.

One step = the whole hot path of one decode step over every layer of the
workload: quantise-on-append of the new token, StreamingLLM eviction (for
streaming layouts) and fused decode attention.  Prints one JSON line.

  python bench.py [--gpus N --steps K --warmup W] [--workload mlx8k|q4_0_32k|ring|tinygpt|snapkv]
  python bench.py --impl reference ...    # the CPU oracle on a bounded sample of the same workload

Inputs are seeded synthetic tensors (synth), resident in HBM before the timed
region.  L2 is flushed (a 256 MiB write) between timed steps, outside the
per-step events.  Timing: CUDA events on the launching stream, barrier +
synchronize around the timed region, max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

# the CPU legs time the oracle single-threaded; say so by pinning BLAS threads
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
import synth  # noqa: E402

METRIC = "decode-attn KV-cache GB/s (% of GB300 HBM peak) and decode steps/s per config"
DEFAULT_WORKLOAD = "mlx8k"
L2_FLUSH_BYTES = 256 << 20


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget")
    p.add_argument("--layers", type=int, default=0,
                   help="override the workload's layer count (profiling small footprints; not a bench line)")
    p.add_argument("--floor", action="store_true",
                   help="measure the per-launch floor of a chain of dependent launches that only read the "
                        "default workload's per-layer decode bytes (probe/floor_probe.cu) and print it")
    p.add_argument("--separate-step", action="store_true",
                   help="run each layer's append, eviction and decode as separate launches even where the "
                        "library fuses them (kvq_append_decode), to compare the two")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the other workloads' summary that a one-GPU run of the default workload adds")
    a = p.parse_args(argv)
    a.warmup = max(a.warmup, 3)
    return a


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------ byte model --

def side_token_bytes(fmt, bits, group, D):
    if fmt == "fp16":
        return 2 * D
    codes = D * bits // 8
    if fmt == "affine_token":
        return codes + 4 * (D // group)
    if fmt == "q4_0":
        return codes + 2 * (D // 32)
    return codes


def decode_bytes(w, T):
    """Algorithmic bytes of one decode-attention launch (one layer): codes + metadata + Q + O.
    A residual buffer (kivi_block keys) holding T tokens reads its closed blocks as codes plus one
    fp16 scale and zero per (block, channel), and its T mod R tail rows as fp32 K and V."""
    io = torch.empty((), dtype=synth.torch_dtype(w.io_dtype)).element_size()
    tail = 0
    if w.k_format == "kivi_block":
        tail = T % w.k_group
        T -= tail
    per_head = T * (side_token_bytes(w.k_format, w.k_bits, w.k_group, w.head_dim)
                    + side_token_bytes(w.v_format, w.v_bits, w.v_group, w.head_dim))
    if w.k_format == "kivi_chan":
        per_head += 4 * w.head_dim
    if w.k_format == "kivi_block":
        per_head += (T // w.k_group) * 4 * w.head_dim + tail * 8 * w.head_dim
    return w.batch * w.n_kv_heads * per_head + 2 * w.batch * w.n_q_heads * w.head_dim * io


def append_bytes(w, n):
    """Bytes of one append of n tokens (one layer): inputs read, codes + metadata written."""
    io = torch.empty((), dtype=synth.torch_dtype(w.io_dtype)).element_size()
    rows = w.batch * w.n_kv_heads * n
    wr = (side_token_bytes(w.k_format, w.k_bits, w.k_group, w.head_dim)
          + side_token_bytes(w.v_format, w.v_bits, w.v_group, w.head_dim))
    if w.k_format == "kivi_block":
        # the token enters the fp32 tail; each closed block reads its tail rows back once and
        # writes codes plus the block's per-channel scale and zero (per token, amortised)
        wr += 8 * w.head_dim + 8 * w.head_dim + 4 * w.head_dim // w.k_group
    return rows * (2 * w.head_dim * io + wr)


def stored_after(w, t_seen):
    if w.layout == "linear":
        return t_seen
    return min(t_seen, w.sink + w.window)


# ------------------------------------------------------ decode workloads --

def fused_step(kvq, w, cfg, sms):
    """Whether kvq_append_decode runs this workload's decode step (append, eviction, attention) as
    one launch per layer: LINEAR and RING caches on the tensor-core decode with head_dim 128 (16-bit
    io), not KIVI_BLOCK keys, whose decode grid is one wave (the plan's `wide` >= 1).  Otherwise the
    step runs as separate launches, and the bench groups every layer's append before every layer's
    decode."""
    if not (w.layout in ("linear", "ring") and w.k_format != "kivi_block" and w.io_dtype != "float32"
            and w.head_dim == 128):
        return False
    return kvq.kvq_decode_plan_query(cfg, w.n_q_heads, sms)[2] >= 1


class DecodeStep:
    """All layers of one workload: caches filled to the context, per-layer step
    inputs and outputs resident in HBM, and captured CUDA graphs: one launch
    per layer (kvq_append_decode) where the library fuses the step, else every
    layer's append + eviction, then every layer's decode attention."""

    def __init__(self, kvq, w, extra_rows, device, separate=False):
        self.kvq, self.w, self.device = kvq, w, device
        dt = synth.torch_dtype(w.io_dtype)
        if w.layout == "linear":
            cap = w.context + extra_rows
        else:
            cap = w.sink + w.window + (1 if w.layout == "compact" else 0)
        self.caches = []
        for layer in range(w.layers):
            bias = synth.k_bias(w, layer, device=device) if w.use_k_bias else None
            c = kvq.KVCache(w.batch, w.n_kv_heads, w.head_dim, cap, w.k_format, w.k_bits, w.k_group,
                            w.v_format, w.v_bits, w.v_group, layout=w.layout, sink=w.sink, window=w.window,
                            k_bias=bias, device=device)
            k, v = synth.layer_inputs(w, layer, 0, w.context, device=device)
            c.append(k, v, calibrate_k=(w.k_format == "kivi_chan"))
            del k, v
            self.caches.append(c)
        torch.cuda.synchronize()
        self.t_seen = w.context
        # step inputs (Q, new K, new V per layer) packed in one buffer so that an
        # end-to-end step is one host-to-device copy; outputs likewise
        L, B, Hq, Hkv, D = w.layers, w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
        per = B * Hq * D + 2 * B * Hkv * D
        self.stage = torch.empty(L * per, dtype=dt, device=device)
        self.outbuf = torch.empty(L * B * Hq * D, dtype=dt, device=device)
        self.q, self.k1, self.v1, self.out = [], [], [], []
        for layer in range(L):
            q, k1, v1 = synth.decode_token_inputs(w, layer, 0, w.context, device=device)
            base = layer * per
            qv = self.stage[base: base + q.numel()].view(q.shape)
            kv_ = self.stage[base + q.numel(): base + q.numel() + k1.numel()].view(k1.shape)
            vv = self.stage[base + q.numel() + k1.numel(): base + per].view(v1.shape)
            qv.copy_(q), kv_.copy_(k1), vv.copy_(v1)
            self.q.append(qv), self.k1.append(kv_), self.v1.append(vv)
            self.out.append(self.outbuf[layer * B * Hq * D: (layer + 1) * B * Hq * D].view(B, Hq, D))
        for c in self.caches:                      # workspaces allocated before capture
            c.workspace(Hq)
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.fused = not separate and fused_step(kvq, w, self.caches[0].cfg, sms)
        self.launches_append = 0
        self.launches_decode = 0
        self.layer_step = None

    def eager_step(self):
        """One step through the public API; returns the library's launch count."""
        if not self.fused:
            return self.eager_append() + self.eager_decode()
        # one call for all layers; layer 0 follows the previous step's last layer (or the input
        # copy), so with more than one layer the kernel before it never writes its cache
        if self.layer_step is None:
            self.layer_step = self.kvq.LayerStep(self.caches, self.k1, self.v1, self.q, self.out)
        self.layer_step.run(early_read=len(self.caches) > 1)
        self.t_seen += 1
        return self.layer_step.launches

    def eager_append(self):
        n = 0
        for layer, c in enumerate(self.caches):
            c.launches = 0
            c.append(self.k1[layer], self.v1[layer])
            if self.w.layout != "linear":
                c.evict_middle()
            n += c.launches
        self.t_seen += 1
        return n

    def eager_decode(self):
        n = 0
        for layer, c in enumerate(self.caches):
            c.launches = 0
            c.decode_attn(self.q[layer], out=self.out[layer])
            n += c.launches
        return n

    def capture(self):
        # one eager pass first: every kernel is loaded before capture
        if self.fused:
            self.eager_step()
            torch.cuda.synchronize()
            self.g_step = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.g_step):
                self.launches_decode = self.eager_step()
            self.t_seen -= 1      # capture records the launches without running them
            torch.cuda.synchronize()
            return
        self.eager_append()
        self.eager_decode()
        torch.cuda.synchronize()
        self.g_append = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_append):
            self.launches_append = self.eager_append()
        self.t_seen -= 1      # capture records the launches without running them
        self.g_decode = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_decode):
            self.launches_decode = self.eager_decode()
        torch.cuda.synchronize()

    def replay(self):
        if self.fused:
            self.g_step.replay()
        else:
            self.g_append.replay()
            self.g_decode.replay()
        self.t_seen += 1

    def replay_timed(self, e0, e1, e2):
        """One step with events before, between (appends | decodes) and after; a fused step records
        its one graph between e0 and e2 (e1 right after e0)."""
        e0.record()
        if self.fused:
            e1.record()
            self.g_step.replay()
        else:
            self.g_append.replay()
            e1.record()
            self.g_decode.replay()
        e2.record()
        self.t_seen += 1

    def stored(self):
        return stored_after(self.w, self.t_seen)

    def step_bytes(self):
        """(append + eviction + attention bytes of the next step, bytes per launch of the step's
        dominant kernel: the fused append + decode, else the decode attention)."""
        w = self.w
        T = stored_after(w, self.t_seen + 1)
        dec = decode_bytes(w, T)
        app = append_bytes(w, 1)
        ev = 0
        if w.layout == "compact" and self.t_seen + 1 > w.sink + w.window:
            ev = 2 * w.batch * w.n_kv_heads * w.window * (
                side_token_bytes(w.k_format, w.k_bits, w.k_group, w.head_dim)
                + side_token_bytes(w.v_format, w.v_bits, w.v_group, w.head_dim))
        return w.layers * (dec + app + ev), dec + (app if self.fused else 0)


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) while the GPU works."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.lines = []

    def start(self):
        ident = []
        try:
            ident = [f"--id=GPU-{torch.cuda.get_device_properties(torch.cuda.current_device()).uuid}"]
        except Exception:
            ident = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *ident, f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(1.0)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarize(out)

    @staticmethod
    def summarize(out):
        """Median SM clock under load, max clock and the throttle reasons seen, from the sampler's CSV."""
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 7]
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[0]) for r in rows]
        mx = max(num(r[1]) for r in rows)
        busy = [s for s, r in zip(sm, rows) if num(r[2]) > 0.3 * max(num(q[2]) for q in rows)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ timed runs --

def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world):
    """Largest x over the ranks (the slowest rank's time); NCCL reduces a device tensor, gloo a host one."""
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def timed_decode(ds, steps, warmup, world):
    """K timed steps (graph replays), L2 flushed between them outside the events."""
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=ds.device)
    for _ in range(warmup):
        flush.zero_()
        ds.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    total_bytes = 0
    dec_bytes = []
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        b, d = ds.step_bytes()
        total_bytes += b
        dec_bytes.append(d)
        flush.zero_()
        ds.replay_timed(*ev[i])
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    return total_bytes, step_ms, dec_ms, dec_bytes


def e2e_decode(ds, steps, world):
    """Through the public Python API, eager calls, inputs from pinned host memory, result read back."""
    host_in = torch.empty(ds.stage.shape, dtype=ds.stage.dtype, pin_memory=True)
    host_in.copy_(ds.stage)
    host_out = torch.empty(ds.outbuf.shape, dtype=ds.outbuf.dtype, pin_memory=True)
    for _ in range(2):
        ds.stage.copy_(host_in, non_blocking=True)
        ds.eager_step()
        host_out.copy_(ds.outbuf, non_blocking=True)
        torch.cuda.synchronize()
    total = 0
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        total += ds.step_bytes()[0]
        ds.stage.copy_(host_in, non_blocking=True)
        ds.eager_step()
        host_out.copy_(ds.outbuf, non_blocking=True)
        torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    dt = max_over_ranks(t1 - t0, world)
    return total, dt, host_in.numel() * host_in.element_size(), host_out.numel() * host_out.element_size()


# ---------------------------------------------------- the oracle on the CPU --

class OracleSample:
    """The oracle's decode step on one (batch 0, kv head 0) slice of layer 0 of the
    workload: quantise-on-append of one token, eviction, float64 attention over
    the dequantised cache for the kv head's query heads."""

    def __init__(self, w):
        from oracle import attention as oatt
        from oracle.cache import CacheSpec, OracleCache

        self.oatt = oatt
        self.w = w
        G = w.group
        k, v = synth.layer_inputs(w, 0, 0, w.context, batch=1)
        k, v = k[:, :1].float().numpy(), v[:, :1].float().numpy()
        bias = synth.k_bias(w, 0)[:1].numpy() if w.use_k_bias else None
        if w.layout == "linear":
            cap = w.context + 8192
        else:
            cap = w.sink + w.window + (1 if w.layout == "compact" else 0)
        self.oc = OracleCache(CacheSpec(batch=1, n_kv_heads=1, head_dim=w.head_dim, capacity=cap, layout=w.layout,
                                        sink=w.sink, window=w.window, k_format=w.k_format, k_bits=w.k_bits,
                                        k_group=w.k_group, v_format=w.v_format, v_bits=w.v_bits, v_group=w.v_group,
                                        k_bias=bias))
        if w.k_format == "kivi_chan":
            self.oc.calibrate_k(k)
        self.oc.append(k, v)
        q, k1, v1 = synth.decode_token_inputs(w, 0, 0, w.context, batch=1)
        self.q = q[:, :G].float().numpy()
        self.k1 = k1[:, :1].float().numpy()
        self.v1 = v1[:, :1].float().numpy()
        self.slice_w = w.with_(batch=1, n_kv_heads=1, n_q_heads=G, layers=1)
        self.cap = cap

    def step(self):
        """Runs one step; returns its algorithmic bytes."""
        if self.w.layout == "linear" and self.oc.stored + 1 > self.cap:
            raise RuntimeError("oracle sample cache full")
        self.oc.append(self.k1, self.v1)
        if self.w.layout != "linear":
            self.oc.evict_middle()
        kh, vh = self.oc.dequant()
        self.oatt.decode_attention(self.q, kh, vh)
        return decode_bytes(self.slice_w, self.oc.stored + getattr(self.oc, "n_tail", 0)) + append_bytes(self.slice_w, 1)

    def describe(self):
        w = self.w
        held = self.oc.stored + getattr(self.oc, "n_tail", 0)
        return (f"layer 0, batch row 0, kv head 0 of {w.name} ({w.group} query heads, "
                f"{held} stored tokens): append + evict + float64 attention per step")


class SnapKVOracleSample:
    """The oracle's SnapKV episode on one (batch 0, kv head 0) slice: observation
    window scores and sink-forced top-k over the prompt's keys, keep-set
    gather, then the decode steps (fp16 append + float64 attention)."""

    def __init__(self, w):
        from oracle import attention as oatt
        from oracle import snapkv as osnap
        from oracle.cache import CacheSpec

        self.oatt, self.osnap, self.w = oatt, osnap, w
        self.G = w.group
        k, v = synth.snapkv_prefill(w, batch=1)
        self.k = k[:, :1].float().numpy()
        self.v = v[:, :1].float().numpy()
        self.spec = CacheSpec(batch=1, n_kv_heads=1, head_dim=w.head_dim, capacity=w.prompt_len + w.decode_steps,
                              layout="linear", sink=0, window=0, k_format="fp16", k_bits=16, k_group=0,
                              v_format="fp16", v_bits=16, v_group=0, k_bias=None)
        self.steps = []
        for t in range(w.decode_steps):
            q, k1, v1 = synth.decode_token_inputs(w, 0, t, w.prompt_len + t, batch=1)
            self.steps.append((q[:, :self.G].float().numpy(), k1[:, :1].float().numpy(), v1[:, :1].float().numpy()))
        sel, gat, dec = snapkv_episode_bytes(w, 1, 1)
        self.bytes = sel + gat + dec

    def step(self):
        """One episode; returns its algorithmic bytes."""
        from oracle.cache import OracleCache

        w = self.w
        oc = OracleCache(self.spec)
        oc.append(self.k, self.v)
        _, idx = self.osnap.snapkv_select(self.k, w.obs_window, w.budget, w.n_sink)
        oc.evict_keepset(idx)
        for q, k1, v1 in self.steps:
            oc.append(k1, v1)
            kh, vh = oc.dequant()
            self.oatt.decode_attention(q, kh, vh)
        return self.bytes

    def describe(self):
        w = self.w
        return (f"batch row 0, kv head 0 of {w.name} ({self.G} query heads): prompt of {w.prompt_len} keys, "
                f"scores + top-{w.budget} + keep-set gather, then {w.decode_steps} fp16 append + float64 "
                f"attention steps, per episode")


def oracle_sample(w):
    return SnapKVOracleSample(w) if w.prompt_len else OracleSample(w)


def _oracle_run(name, seconds):
    """Builds one oracle sample of workload `name` and steps it for about `seconds`:
    (bytes, steps, wall time, description)."""
    s = oracle_sample(synth.get_workload(name))
    s.step()
    nbytes, n, t0 = 0, 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        nbytes += s.step()
        n += 1
    return nbytes, n, time.perf_counter() - t0, s.describe()


def _oracle_worker(args):
    return _oracle_run(*args)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    import platform

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(w, seconds, all_cores=True, nproc=None):
    """The oracle on the host: one thread, then (all_cores) one spawned process per core (nproc of
    them if given), each stepping its own copy of the same one-slice sample (the slices of a step are
    independent), the rate summed over the processes."""
    nbytes, n, dt, desc = _oracle_run(w.name, seconds)
    nproc = nproc or os.cpu_count() or 1
    line = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} steps of {desc}; {dt:.1f} s single-threaded numpy",
            "nproc": nproc, "cpu_model": cpu_model()}
    if all_cores and nproc > 1:
        import multiprocessing as mp

        # spawned, not forked: this process already holds a CUDA context
        with mp.get_context("spawn").Pool(nproc) as pool:
            res = pool.map(_oracle_worker, [(w.name, seconds)] * nproc)
        total, steps, wall = sum(r[0] for r in res), sum(r[1] for r in res), max(r[2] for r in res)
        line["all_cores"] = {"value": total / wall / 1e9, "unit": "GB/s", "cores": nproc,
                             "sample": f"{nproc} processes x one copy each of the same sample, {steps} steps "
                                       f"in {wall:.1f} s (one thread per process)"}
    return line


def run_reference(a, rank, world):
    if world > 1 and rank != 0:
        return
    w = synth.get_workload(a.workload)
    s = oracle_sample(w)
    for _ in range(a.warmup):
        s.step()
    nbytes, t0 = 0, time.perf_counter()
    for _ in range(a.steps):
        nbytes += s.step()
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": dt * 1e3 / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": "one (batch, kv head) slice of one layer per step"
                                                     if not w.prompt_len else "one (batch, kv head) slice per episode"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{a.steps} steps of {s.describe()}"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


DECODE_SOURCES = ("kvq_internal.cuh", "async_copy.cuh", "decode_impl.cuh", "decode_tc_frag.cuh", "decode_tc.cuh",
                  "quantize_row.cuh")
SNAPKV_SOURCES = ("kvq_internal.cuh", "snapkv.cu")
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "dram_traffic.json")


def sources_sha(kvq_dir, names):
    """sha256 over kernel sources (in order): a committed ncu figure holds only for these bytes."""
    import hashlib

    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(kvq_dir, "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def decode_source_sha(kvq_dir):
    return sources_sha(kvq_dir, DECODE_SOURCES)


def decode_kernel_name(w):
    """The decode kernel the library launches for this workload (tensor-core path for 16-bit io, D 64/128)."""
    tc = w.io_dtype != "float32" and w.head_dim in (64, 128)
    return "decode_tc_kernel" if tc else "decode_kernel"


def profile_traffic(name, kvq_dir):
    """DRAM bytes per launch of the dominant kernel of workload `name` from the committed ncu summary
    (profiles/dram_traffic.json), if it was taken on the current sources of that kernel; else None."""
    if not os.path.exists(TRAFFIC_JSON):
        return None
    with open(TRAFFIC_JSON) as f:
        d = json.load(f)
    entry = d.get(name)
    if not entry:
        return None
    names = tuple(entry.get("sources", DECODE_SOURCES))
    if entry.get("sources_sha256") != sources_sha(kvq_dir, names):
        return None
    return entry.get("dram_bytes_per_launch")


def decode_traffic(w, kvq_dir):
    return profile_traffic(w.name, kvq_dir)


def run_floor(a):
    """Builds and runs probe/floor_probe.cu for the default workload's layer count and decode bytes
    per layer; prints its JSON lines and one summary line."""
    import importlib.util

    pkg = os.path.join(ROOT, "bit_kv_cache_quant_gb300")
    src = os.path.join(pkg, "probe", "floor_probe.cu")
    exe = os.path.join(pkg, "_build", "floor_probe")
    os.makedirs(os.path.dirname(exe), exist_ok=True)
    if not os.path.exists(exe) or os.path.getmtime(exe) < os.path.getmtime(src):
        spec = importlib.util.spec_from_file_location("kvq_build", os.path.join(pkg, "build.py"))
        build = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(build)
        subprocess.run([build._nvcc(), *build.ARCH, "-O3", "-std=c++17", src, "-o", exe], check=True)
    w = synth.get_workload(DEFAULT_WORKLOAD)
    nbytes = decode_bytes(w, w.context)
    out = subprocess.run([exe, str(w.layers), str(nbytes)], capture_output=True, text=True, check=True).stdout
    rows = [json.loads(x) for x in out.splitlines() if x.startswith("{")]
    for r in rows:
        print(json.dumps(r))
    best = {m: min((r for r in rows if r["mode"] == m), key=lambda r: r["us_per_launch"])
            for m in {r["mode"] for r in rows}}
    print(json.dumps({"floor": w.name, "layers": w.layers, "bytes_per_launch": nbytes,
                      "best_us_per_launch": {str(m): best[m]["us_per_launch"] for m in sorted(best)}}))


# -------------------------------------------------------------------- main --

def bench_decode(a, kvq, w, rank, world):
    device = torch.device("cuda", torch.cuda.current_device())
    extra = 2 * (a.steps + a.warmup) + 64
    ds = DecodeStep(kvq, w, extra, device, separate=a.separate_step)
    ds.capture()
    clocks = ClockSampler()
    clocks.start()
    total_bytes, step_ms, dec_ms, dec_bytes = timed_decode(ds, a.steps, a.warmup, world)
    clk = clocks.stop()
    t_step = sum(step_ms) / 1e3
    t_max = max_over_ranks(t_step, world)
    value = world * total_bytes / t_max / 1e9
    avg_dec_launch_s = sum(dec_ms) / 1e3 / (a.steps * w.layers)
    dec_bytes_launch = sum(dec_bytes) / len(dec_bytes)
    peak, peak_kind = read_peaks()
    achieved = dec_bytes_launch / avg_dec_launch_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": t_max * 1e3 / a.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u4/u8 codes, f32 math" if w.k_format != "fp16" else "f16 codes, f32 math",
        "data": "synthetic",
        "config": {"workload": w.name, "layers": w.layers, "batch": w.batch, "n_q_heads": w.n_q_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "context": w.context,
                   "k_format": f"{w.k_format}{w.k_bits}" + (f"g{w.k_group}" if w.k_group else ""),
                   "v_format": f"{w.v_format}{w.v_bits}" + (f"g{w.v_group}" if w.v_group else ""),
                   "layout": w.layout,
                   "step": ("per layer: append 1 token, evict, decode attention"
                            + (" (one fused launch per layer)" if ds.fused else " (separate launches)")),
                   "l2": "flushed (256 MiB write) between timed steps, outside the events",
                   "parallelism": f"replicas x{world}"},
        "decode_steps_per_s": world * a.steps / t_max,
        "tokens_appended_per_s": world * a.steps * w.batch / t_max,
        "decode_attn_gbs": world * sum(dec_bytes) * w.layers / max_over_ranks(sum(dec_ms) / 1e3, world) / 1e9,
        "gpu_launches": (ds.launches_append + ds.launches_decode) * a.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": decode_traffic(w, os.path.dirname(kvq.__file__)),
                     "kernel": decode_kernel_name(w), "bytes_per_launch": dec_bytes_launch,
                     "avg_launch_us": avg_dec_launch_s * 1e6, "peak_kind": f"{peak_kind} copy bandwidth"},
        "clocks": clk,
    }
    if w.layout == "linear":
        line["convert"] = bench_convert(kvq, w, device, a.warmup)
    if w.k_format == "kivi_chan" and w.layout != "ring":
        line["recompute_k_append"] = bench_recompute(kvq, w, device, a.warmup)
    if not a.no_e2e:
        e_bytes, e_dt, h2d, d2h = e2e_decode(ds, max(3, min(a.steps, 200)), world)
        line["e2e"] = {"value": world * e_bytes / e_dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h,
                       "how": ("public Python API, " + ("one LayerStep call (kvq_append_decode_layers) per step"
                                                          if ds.fused else "eager calls per layer")
                               + ", pinned host inputs copied in and outputs read back every step (wall clock)")}
    return line


def snapkv_episode_bytes(w, batch, n_kv_heads):
    """Algorithmic bytes of one SnapKV episode: (select, keep-set gather, decode steps).

    select: the prompt's K read, scores written and read back by the top-k,
    indices written; gather: every kept K and V row read and written; decode:
    each step's single-token append plus attention over the kept rows and the
    tokens appended so far."""
    S, D, budget = w.prompt_len, w.head_dim, w.budget
    bh = batch * n_kv_heads
    sel = bh * (S * D * 2 + 2 * S * 4 + budget * 4)
    gather = 2 * bh * budget * 2 * D * 2
    w1 = w.with_(batch=batch, n_kv_heads=n_kv_heads, n_q_heads=n_kv_heads * w.group)
    dec = sum(decode_bytes(w1, budget + t + 1) + append_bytes(w1, 1) for t in range(w.decode_steps))
    return sel, gather, dec


class SnapKVEpisode:
    """SnapKV prefill eviction and the decode that follows, on the device: the
    prompt's K/V in an fp16 cache, observation-window scoring + top-k, keep-set
    gather into the cache, then `decode_steps` decode steps (each one launch:
    the single-token append and the attention over the cache including it).
    The episode (everything after the prompt fill) is one CUDA graph; each
    replay starts from a freshly filled cache."""

    def __init__(self, kvq, w, device):
        self.kvq, self.w = kvq, w
        self.k, self.v = synth.snapkv_prefill(w, device=device)
        B, H, S, D = self.k.shape
        self.B, self.H, self.S, self.D = B, H, S, D
        Hq, steps = w.n_q_heads, w.decode_steps
        self.cache = kvq.KVCache(B, H, D, S + steps, "fp16", 16, 0, "fp16", 16, 0, device=device)
        self.ws = torch.empty(kvq.snapkv_workspace_bytes(B, H, S, D, w.obs_window), dtype=torch.uint8, device=device)
        self.scores = torch.empty((B, H, S), dtype=torch.float32, device=device)
        self.idx = torch.empty((B, H, w.budget), dtype=torch.int32, device=device)
        per = B * Hq * D + 2 * B * H * D
        self.stage = torch.empty(steps * per, dtype=torch.float16, device=device)
        self.q, self.k1, self.v1 = [], [], []
        for t in range(steps):
            q, k1, v1 = synth.decode_token_inputs(w, 0, t, S + t, device=device, batch=B)
            base = t * per
            views = []
            for x, off in ((q, 0), (k1, q.numel()), (v1, q.numel() + k1.numel())):
                vw = self.stage[base + off: base + off + x.numel()].view(x.shape)
                vw.copy_(x)
                views.append(vw)
            self.q.append(views[0]), self.k1.append(views[1]), self.v1.append(views[2])
        self.out = torch.empty((steps, B, Hq, D), dtype=torch.float16, device=device)
        self.cache.workspace(Hq)
        self.launches = 0

    def fill(self):
        self.cache.reset()
        self.cache.append(self.k, self.v)

    def episode(self):
        kvq, w, c = self.kvq, self.w, self.cache
        n = 0
        kvq.snapkv_select(self.k, self.S, self.B, self.H, self.S, self.D, w.obs_window, w.budget, w.n_sink,
                          self.scores, self.idx, self.ws)
        n += kvq.kvq_last_launch_count()
        c.launches = 0
        c.evict_keepset(self.idx)
        for t in range(w.decode_steps):
            # one launch: the token is coded into the fp16 cache and attended over
            c.append_decode(self.k1[t], self.v1[t], self.q[t], out=self.out[t])
        return n + c.launches

    def capture(self):
        self.fill()
        self.episode()
        self.fill()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.launches = self.episode()
        torch.cuda.synchronize()


def bench_convert(kvq, w, device, warmup):
    """Bulk quantise-on-convert of one layer: the context's tokens of a dense cache
    (the workload's io dtype) into a fresh quantised cache, timed alone."""
    k, v = synth.layer_inputs(w, 0, 0, w.context, device=device)
    bias = synth.k_bias(w, 0, device=device) if w.use_k_bias else None
    cache = kvq.KVCache(w.batch, w.n_kv_heads, w.head_dim, w.context, w.k_format, w.k_bits, w.k_group,
                        w.v_format, w.v_bits, w.v_group, k_bias=bias, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    cal = w.k_format == "kivi_chan"
    reps = 5
    times = []
    for i in range(warmup + reps):
        cache.reset()
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        cache.convert(k, v, w.context, calibrate_k=cal)
        e1.record()
        torch.cuda.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
    t = statistics.median(times)
    nbytes = append_bytes(w, w.context)
    if cal:
        nbytes += w.batch * w.n_kv_heads * w.context * w.head_dim * k.element_size()   # calibration pass over K
    return {"tokens_per_s": w.batch * w.context / t, "gbs": nbytes / t / 1e9, "us": t * 1e6,
            "tokens": w.context, "what": "one layer's dense cache, every (batch row, kv head), into a fresh cache"}


def bench_recompute(kvq, w, device, warmup):
    """One single-token append with the per-channel K range recomputed over the whole
    stored block (KVQ_APPEND_RECOMPUTE_K), on one layer filled to the context."""
    cap = w.sink + w.window + 1 if w.layout == "compact" else w.context + 64
    cache = kvq.KVCache(w.batch, w.n_kv_heads, w.head_dim, cap, w.k_format, w.k_bits, w.k_group, w.v_format,
                        w.v_bits, w.v_group, layout=w.layout, sink=w.sink, window=w.window, device=device)
    k, v = synth.layer_inputs(w, 0, 0, w.context, device=device)
    cache.append(k, v, recompute_k=True)
    _, k1, v1 = synth.decode_token_inputs(w, 0, 0, w.context, device=device)
    reps = 20
    times = []
    for i in range(warmup + reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        cache.append(k1, v1, recompute_k=True)
        e1.record()
        if w.layout == "compact":
            cache.evict_middle()
        torch.cuda.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
    t = statistics.median(times)
    stored = cache.stats().stored
    return {"us": t * 1e6, "stored_tokens": stored, "appends_per_s": 1.0 / t,
            "what": "append of one token per (batch row, kv head) recoding every stored key"}


def coverage_stats(scores, idx, budget, n_sink):
    """Mean over (batch row, kv head) of the kept rows' share of the score mass, and of the
    expected share of the sinks plus (budget - n_sink) uniformly random other rows.
    scores [B, H, S] and idx [B, H, n] tensors on any device; float64 sums."""
    sc = scores.double()
    tot = sc.sum(-1)
    kept = torch.gather(sc, 2, idx.long()).sum(-1) / tot
    S = sc.shape[-1]
    if budget >= S:
        rnd = torch.ones_like(tot)
    else:
        ns = min(n_sink, S)
        rnd = (sc[..., :ns].sum(-1) + (budget - ns) / (S - ns) * sc[..., ns:].sum(-1)) / tot
    return float(kept.mean()), float(rnd.mean())


def bench_snapkv(a, kvq, w, rank, world):
    device = torch.device("cuda", torch.cuda.current_device())
    ep = SnapKVEpisode(kvq, w, device)
    ep.capture()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    sel_b, gat_b, dec_b = snapkv_episode_bytes(w, ep.B, ep.H)
    total_b = sel_b + gat_b + dec_b
    for _ in range(a.warmup):
        ep.fill()
        ep.graph.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    clocks = ClockSampler()
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    for i in range(a.steps):
        ep.fill()
        flush.zero_()
        ev[i][0].record()
        ep.graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    t = max_over_ranks(sum(s_.elapsed_time(e_) for s_, e_ in ev) / 1e3, world)
    # the select alone, for the roofline of its two scoring passes + top-k
    sel_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    for i in range(a.steps):
        flush.zero_()
        sel_ev[i][0].record()
        kvq.snapkv_select(ep.k, ep.S, ep.B, ep.H, ep.S, ep.D, w.obs_window, w.budget, w.n_sink, ep.scores, ep.idx,
                          ep.ws)
        sel_ev[i][1].record()
    torch.cuda.synchronize()
    t_sel = sum(s_.elapsed_time(e_) for s_, e_ in sel_ev) / 1e3 / a.steps
    peak, peak_kind = read_peaks()
    achieved = sel_b / t_sel / 1e9
    cov_kept, cov_rnd = coverage_stats(ep.scores, ep.idx, w.budget, w.n_sink)
    line = {"metric": METRIC, "value": world * total_b * a.steps / t / 1e9, "unit": "GB/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": t * 1e3 / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16 in, f32 accumulate", "data": "synthetic",
            "config": {"workload": w.name, "prompt": ep.S, "n_kv_heads": ep.H, "n_q_heads": w.n_q_heads,
                       "head_dim": ep.D, "obs_window": w.obs_window, "budget": w.budget, "n_sink": w.n_sink,
                       "decode_steps": w.decode_steps,
                       "step": "one episode: snapkv_select (scores + top-k), keep-set gather into the cache, "
                               "then per decode step an fp16 append and decode attention (one CUDA graph)",
                       "l2": "flushed (256 MiB write) after the prompt fill, before each timed episode",
                       "parallelism": f"replicas x{world}"},
            "snapkv_select_us": t_sel * 1e6,
            "coverage": {"kept": cov_kept, "random_same_size": cov_rnd,
                         "what": "share of the observation-window score mass held by the kept rows, mean over "
                                 "heads, against sinks plus a uniformly random set of the same size"},
            "decode_steps_per_s": world * w.decode_steps * a.steps / t,
            "gpu_launches": ep.launches * a.steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": profile_traffic(w.name, os.path.dirname(kvq.__file__)),
                         "kernel": "snapkv_select (one-pass scoring + top-k)",
                         "bytes_per_launch": sel_b, "avg_launch_us": t_sel * 1e6,
                         "peak_kind": f"{peak_kind} copy bandwidth"},
            "clocks": clk}
    if not a.no_e2e:
        line["e2e"] = e2e_snapkv(ep, max(3, min(a.steps, 20)), world, total_b)
    return line


def e2e_snapkv(ep, episodes, world, total_b):
    """Public API, eager calls: the decode steps' inputs copied in from pinned host
    memory, the selected indices and every step's output read back."""
    host_in = torch.empty(ep.stage.shape, dtype=ep.stage.dtype, pin_memory=True)
    host_in.copy_(ep.stage)
    host_out = torch.empty(ep.out.shape, dtype=ep.out.dtype, pin_memory=True)
    host_idx = torch.empty(ep.idx.shape, dtype=ep.idx.dtype, pin_memory=True)

    def once():
        ep.fill()
        ep.stage.copy_(host_in, non_blocking=True)
        ep.episode()
        host_idx.copy_(ep.idx, non_blocking=True)
        host_out.copy_(ep.out, non_blocking=True)

    once()
    torch.cuda.synchronize()
    dt = 0.0
    barrier(world)
    for _ in range(episodes):
        ep.fill()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ep.stage.copy_(host_in, non_blocking=True)
        ep.episode()
        host_idx.copy_(ep.idx, non_blocking=True)
        host_out.copy_(ep.out, non_blocking=True)
        torch.cuda.synchronize()
        dt += time.perf_counter() - t0
    barrier(world)
    dt = max_over_ranks(dt, world)
    return {"value": world * total_b * episodes / dt / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": host_in.numel() * host_in.element_size(),
            "d2h_bytes_per_step": host_out.numel() * host_out.element_size() + host_idx.numel() * 4,
            "how": "public Python API, eager calls per episode (prompt fill outside the timing), pinned host "
                   "inputs copied in and outputs read back every episode (wall clock)"}


def per_config(a, kvq):
    """The other workloads measured in the same run (one GPU, device time only):
    the metric is quoted per config.  Each entry holds that workload's bench
    line essentials; a failure is recorded, not raised."""
    out = {}
    for name in ("tinygpt", "q4_0_32k", "snapkv", "ring", "residual"):
        w = synth.get_workload(name)
        sub = argparse.Namespace(**vars(a))
        sub.steps, sub.warmup, sub.no_e2e = (20, 3, True) if w.batch > 1 or w.prompt_len else (50, 5, True)
        try:
            ln = bench_snapkv(sub, kvq, w, 0, 1) if w.prompt_len else bench_decode(sub, kvq, w, 0, 1)
            r = ln["roofline"]
            out[w.name] = {"value": ln["value"], "unit": ln["unit"], "ms_per_step": ln["ms_per_step"],
                           "steps": sub.steps, "decode_steps_per_s": ln.get("decode_steps_per_s"),
                           "roofline_kernel": r.get("kernel"), "kernel_us": r.get("avg_launch_us"),
                           "bytes_per_launch": r.get("bytes_per_launch"), "frac": r["frac"],
                           "traffic": r.get("traffic"), "clocks": ln.get("clocks")}
            for key in ("snapkv_select_us", "convert", "recompute_k_append"):
                if key in ln:
                    out[w.name][key] = ln[key]
        except Exception as e:  # noqa: BLE001 - the primary line must still print
            out[w.name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def main(argv=None):
    a = parse_args(argv)
    if a.floor:
        run_floor(a)
        return
    rank, world, local = dist_env()
    if a.impl == "reference":
        run_reference(a, rank, world)
        return
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    import bit_kv_cache_quant_gb300 as kvq

    w = synth.get_workload(a.workload)
    if a.layers > 0:
        w = w.with_(layers=a.layers)
    line = bench_snapkv(a, kvq, w, rank, world) if w.prompt_len else bench_decode(a, kvq, w, rank, world)
    if rank == 0 and not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, a.cpu_seconds)
    if world == 1 and not a.no_per_config and a.workload == DEFAULT_WORKLOAD and a.layers == 0:
        line["per_config"] = per_config(a, kvq)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
