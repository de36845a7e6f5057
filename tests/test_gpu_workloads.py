"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.  Where the oracle would take minutes over every (batch, kv
head), it checks sampled slices: every (b, kv head) is coded and attended
independently, so a slice's codes, metadata and outputs are exactly those
of a batch-1, one-head cache fed that slice."""
import numpy as np
import pytest
import torch

import synth
from kvq_helpers import assert_attention_close, assert_cache_equal, gpu_planes, host, oracle_spec
from oracle import attention as oatt
from oracle import snapkv as osk
from oracle.cache import CacheSpec, OracleCache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import bit_kv_cache_quant_gb300 as m

    return m


def _cache_for(kvq, w, capacity=None, bias=None):
    cap = capacity or (w.sink + w.window + (1 if w.layout == "compact" else 0) if w.layout != "linear" else w.context)
    return kvq.KVCache(w.batch, w.n_kv_heads, w.head_dim, cap, w.k_format, w.k_bits, w.k_group, w.v_format, w.v_bits,
                       w.v_group, layout=w.layout, sink=w.sink, window=w.window, k_bias=bias)


def _slice_spec(cache, bias_row=None):
    s = oracle_spec(cache, bias_row)
    s.batch, s.n_kv_heads = 1, 1
    return s


def test_tinygpt_kivi8_streaming_full(kvq):
    w = synth.get_workload("tinygpt")
    cache = _cache_for(kvq, w)
    oc = OracleCache(oracle_spec(cache))
    k, v = synth.layer_inputs(w, 0, 0, w.context)
    cache.append(k.cuda(), v.cuda(), calibrate_k=True)
    cache.evict_middle()
    oc.calibrate_k(host(k))
    oc.append(host(k), host(v))
    oc.evict_middle()
    for step in range(3):     # decode steps past the cap: append, evict, attend
        q, k1, v1 = synth.decode_token_inputs(w, 0, step, w.context + step)
        cache.append(k1.cuda(), v1.cuda())
        cache.evict_middle()
        out = cache.decode_attn(q.cuda())
        oc.append(host(k1), host(v1))
        oc.evict_middle()
        assert_cache_equal(cache, oc, f"step {step}")
        kh, vh = oc.dequant()
        assert_attention_close(out, oatt.decode_attention(host(q), kh, vh), f"step {step}")
    assert cache.stats().stored == 260


def test_mlx_affine4_ctx8k_one_layer_full(kvq):
    w = synth.get_workload("mlx8k")
    cache = _cache_for(kvq, w, capacity=w.context + 8)
    oc = OracleCache(oracle_spec(cache))
    k, v = synth.layer_inputs(w, 3, 0, w.context, device="cuda")
    cache.append(k, v)
    oc.append(host(k), host(v))
    q, k1, v1 = synth.decode_token_inputs(w, 3, 0, w.context, device="cuda")
    cache.append(k1, v1)
    oc.append(host(k1), host(v1))
    out = cache.decode_attn(q)
    assert_cache_equal(cache, oc, "mlx g64 layer")
    kh, vh = oc.dequant()
    assert_attention_close(out, oatt.decode_attention(host(q), kh, vh), "mlx g64 layer")


def test_residual_buffer_ctx8k_one_layer_full(kvq):
    # the residual workload at full context (64 closed blocks of 128 and a 100-token tail), then
    # 30 decode-step appends: the 28th closes a block mid-decode
    w = synth.get_workload("residual")
    cache = _cache_for(kvq, w, capacity=w.context + 64)
    oc = OracleCache(oracle_spec(cache))
    k, v = synth.layer_inputs(w, 1, 0, w.context, device="cuda")
    cache.append(k, v)
    oc.append(host(k), host(v))
    assert (oc.stored, oc.n_tail) == (8192, 100)
    for step in range(30):
        q, k1, v1 = synth.decode_token_inputs(w, 1, step, w.context + step, device="cuda")
        cache.append(k1, v1)
        oc.append(host(k1), host(v1))
    out = cache.decode_attn(q)
    assert (oc.stored, oc.n_tail) == (8320, 2)
    assert_cache_equal(cache, oc, "residual layer")
    kh, vh = oc.dequant()
    assert_attention_close(out, oatt.decode_attention(host(q), kh, vh), "residual layer")


@pytest.mark.parametrize("name,samples", [("q4_0_32k", [(0, 0), (3, 5), (7, 7)]),
                                          ("ring", [(0, 0), (17, 3), (63, 7)])])
def test_large_batch_workloads_sampled(kvq, name, samples):
    w = synth.get_workload(name)
    bias = synth.k_bias(w, 0, device="cuda") if w.use_k_bias else None
    cache = _cache_for(kvq, w, capacity=w.context + 4 if w.layout == "linear" else None, bias=bias)
    k, v = synth.layer_inputs(w, 0, 0, w.context, device="cuda")
    calibrate = w.k_format == "kivi_chan"
    cache.append(k, v, calibrate_k=calibrate)
    steps = []
    for step in range(3):
        q, k1, v1 = synth.decode_token_inputs(w, 0, step, w.context + step, device="cuda")
        cache.append(k1, v1)
        cache.evict_middle() if w.layout == "ring" else None
        steps.append((q, k1, v1))
    out = cache.decode_attn(steps[-1][0])
    planes = gpu_planes(cache)
    G = w.group
    for b, h in samples:
        brow = None if bias is None else host(bias)[h:h + 1]
        oc = OracleCache(_slice_spec(cache, brow))
        kk = host(k[b:b + 1, h:h + 1])
        if calibrate:
            oc.calibrate_k(kk)
        oc.append(kk, host(v[b:b + 1, h:h + 1]))
        for q, k1, v1 in steps:
            oc.append(host(k1[b:b + 1, h:h + 1]), host(v1[b:b + 1, h:h + 1]))
            oc.evict_middle() if w.layout == "ring" else None
        assert_cache_equal(cache, oc, f"{name} slice {(b, h)}", sel=(b, h), planes=planes)
        kh, vh = oc.dequant()
        qs = host(steps[-1][0][b:b + 1, h * G:(h + 1) * G])
        ref = oatt.decode_attention(qs, kh, vh)
        assert_attention_close(out[b:b + 1, h * G:(h + 1) * G], ref, f"{name} slice {(b, h)}")


def test_snapkv_prefill_then_decode_full(kvq):
    w = synth.get_workload("snapkv")
    S = w.prompt_len
    k, v = synth.snapkv_prefill(w, device="cuda")
    cache = kvq.KVCache(1, w.n_kv_heads, w.head_dim, S + w.decode_steps, "fp16", 16, 0, "fp16", 16, 0)
    cache.append(k, v)
    _, idx = kvq.snapkv(k, w.obs_window, w.budget, w.n_sink, want_scores=False)
    cache.evict_keepset(idx)
    oc = OracleCache(oracle_spec(cache))
    oc.append(host(k), host(v))
    oc.evict_keepset(idx.cpu().numpy())
    # the kept set is the oracle's own selection where the cutoff is well conditioned
    kn = host(k)
    ig = idx.cpu().numpy()
    for h in range(w.n_kv_heads):
        ref = osk.obs_window_scores(kn[0, h], w.obs_window)
        rest = np.sort(ref[w.n_sink:])[::-1]
        gap = rest[w.budget - w.n_sink - 1] - rest[w.budget - w.n_sink]
        eps = 1e-5 * ref.max()
        if gap > eps:
            np.testing.assert_array_equal(ig[0, h], osk.select_indices(ref, w.budget, w.n_sink))
        else:
            # an ill-conditioned cutoff: the device set must still be a valid
            # top-k under the oracle's scores within eps (sinks kept, sorted,
            # budget rows, no unselected row clearly above a selected one)
            sel = ig[0, h]
            assert len(sel) == w.budget and np.all(np.diff(sel) > 0)
            assert np.array_equal(sel[:w.n_sink], np.arange(w.n_sink))
            kth = rest[w.budget - w.n_sink - 1]
            mask = np.zeros(S, bool)
            mask[sel] = True
            others = np.flatnonzero(~mask)
            assert ref[sel[w.n_sink:]].min() >= kth - eps
            assert others.size == 0 or ref[others].max() <= kth + eps
    outs = []
    for step in range(w.decode_steps):
        q, k1, v1 = synth.decode_token_inputs(w, 0, step, S + step, device="cuda")
        cache.append(k1, v1)
        oc.append(host(k1), host(v1))
        outs.append((q, cache.decode_attn(q)))
    st = cache.stats()
    assert st.stored == w.budget + w.decode_steps and st.pos == S + w.decode_steps
    assert_cache_equal(cache, oc, "snapkv after decode")
    q, out = outs[-1]
    kh, vh = oc.dequant()
    assert_attention_close(out, oatt.decode_attention(host(q), kh, vh), "snapkv decode")
