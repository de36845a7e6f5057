"""GPU parity: SnapKV scoring (fp32 vs the float64 oracle) and selection.

Selection on identical fp32 scores (snapkv_topk) must equal the oracle's
bit-exactly.  For the fused call the indices must equal the oracle's exactly
whenever the oracle's gap at the top-k cutoff exceeds twice the measured
score error; otherwise the GPU set must still be a valid top-k under the
oracle scores widened by that error.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import snapkv as osk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import bit_kv_cache_quant_gb300 as m

    return m


def _keys(B, H, S, D, seed, sink_rows=4, sink_scale=8.0):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(B, H, S, D, generator=g)
    k[:, :, :sink_rows] *= sink_scale
    return k.half()


def _topk_gpu(kvq, scores: np.ndarray, budget, n_sink):
    B, H, S = scores.shape
    idx = torch.empty((B, H, min(budget, S)), dtype=torch.int32, device="cuda")
    kvq.snapkv_topk(torch.from_numpy(scores).cuda(), B, H, S, budget, n_sink, idx)
    return idx.cpu().numpy()


@pytest.mark.parametrize("S,budget,n_sink", [(5000, 512, 4), (100, 512, 4), (1024, 1023, 0), (3000, 4, 4),
                                             (17, 9, 3), (70000, 2048, 16), (1, 1, 1), (600, 600, 4)])
def test_topk_bit_exact_on_identical_scores(kvq, S, budget, n_sink):
    rng = np.random.default_rng(S + budget)
    scores = rng.random((2, 3, S)).astype(np.float32) * 1e-3
    # exact ties across the cutoff, zeros and negative zeros
    scores[:, :, rng.integers(0, S, size=min(S, 50))] = scores[0, 0, S // 2]
    scores[0, 1, : S // 3] = 0.0
    scores[1, 2, : S // 4] = -0.0
    got = _topk_gpu(kvq, scores, budget, n_sink)
    for b in range(2):
        for h in range(3):
            ref = osk.select_indices(scores[b, h], budget, n_sink)
            np.testing.assert_array_equal(got[b, h], ref, err_msg=f"b{b} h{h}")


# Prompts of 4096 positions and more run the selection on a cluster of CTAs per
# head (each a contiguous slice of the positions): ties and kept positions
# cross the slice boundaries.
@pytest.mark.parametrize("S,budget,n_sink", [(16384, 512, 4), (65536, 4096, 0), (8192, 4, 4), (4096, 4095, 1),
                                             (4097, 2000, 7)])
def test_topk_cluster_sizes(kvq, S, budget, n_sink):
    rng = np.random.default_rng(S + 3 * budget)
    scores = (rng.random((1, 2, S)).astype(np.float32) * 1e-3)
    scores[0, 0, rng.integers(0, S, size=200)] = scores[0, 0, S // 3]   # ties around the cutoff
    got = _topk_gpu(kvq, scores, budget, n_sink)
    for h in range(2):
        np.testing.assert_array_equal(got[0, h], osk.select_indices(scores[0, h], budget, n_sink), err_msg=f"h{h}")


def test_topk_cluster_all_equal(kvq):
    # every score equal: the lowest positions are kept, across all slices
    S, budget, n_sink = 20000, 9000, 4
    scores = np.full((1, 1, S), 0.25, np.float32)
    got = _topk_gpu(kvq, scores, budget, n_sink)
    assert got[0, 0].tolist() == list(range(budget)) == osk.select_indices(scores[0, 0], budget, n_sink).tolist()


def test_topk_negative_scores_order(kvq):
    scores = np.array([[[-3.0, -1.0, -2.0, 5.0, -0.5, 0.0]]], np.float32)
    got = _topk_gpu(kvq, scores, 3, 1)
    assert got[0, 0].tolist() == osk.select_indices(scores[0, 0], 3, 1).tolist() == [0, 3, 5]


def _check_select(kvq, k, w, budget, n_sink):
    B, H, S, D = k.shape
    scores, idx = kvq.snapkv(k.cuda(), w, budget, n_sink)
    sg = scores.cpu().numpy().astype(np.float64)
    ig = idx.cpu().numpy()
    kn = k.float().numpy()
    worst_gap_ratio = np.inf
    for b in range(B):
        for h in range(H):
            ref = osk.obs_window_scores(kn[b, h], w)
            eps = np.abs(sg[b, h] - ref).max()
            assert eps <= 1e-5 * ref.max() + 1e-9, f"score error {eps:.3e}"
            np.testing.assert_allclose(sg[b, h].sum(), 1.0, rtol=1e-4)
            ref_idx = osk.select_indices(ref, budget, n_sink)
            if budget >= S:
                np.testing.assert_array_equal(ig[b, h], np.arange(S))
                continue
            ns = min(n_sink, S)
            rest = np.sort(ref[ns:])[::-1]
            kk = budget - ns
            gap = rest[kk - 1] - rest[kk] if kk > 0 else np.inf
            worst_gap_ratio = min(worst_gap_ratio, gap / max(eps, 1e-30))
            if gap > 2 * eps:
                np.testing.assert_array_equal(ig[b, h], ref_idx)
            else:
                sel = set(ig[b, h].tolist())
                assert set(range(ns)) <= sel and len(sel) == budget
                cut = rest[kk - 1]
                for j in range(ns, S):
                    if ref[j] > cut + 2 * eps:
                        assert j in sel
                    if ref[j] < cut - 2 * eps:
                        assert j not in sel
            assert np.all(np.diff(ig[b, h]) > 0)
    return worst_gap_ratio


@pytest.mark.parametrize("S,D,w", [(700, 128, 32), (513, 64, 16), (2000, 32, 64), (40, 128, 32), (9, 64, 5)])
def test_select_small(kvq, S, D, w):
    k = _keys(1, 2, S, D, seed=S + w)
    _check_select(kvq, k, w, 64, 4)


def test_select_budget_covers_everything(kvq):
    k = _keys(1, 1, 300, 128, seed=3)
    _check_select(kvq, k, 32, 512, 4)


def test_select_full_size_prompt(kvq):
    # the 16K-token prompt, 8 kv heads, w = 32, budget 512 with 4 sinks
    w = synth.get_workload("snapkv")
    k, _ = synth.snapkv_prefill(w)
    ratio = _check_select(kvq, k, w.obs_window, w.budget, w.n_sink)
    print(f"smallest cutoff gap / score error over heads: {ratio:.1f}")


def test_select_on_cache_rows_with_head_stride(kvq):
    # keys read in place from a cache's fp16 K plane (row stride = cap_alloc)
    B, H, S, D = 1, 2, 600, 128
    cache = kvq.KVCache(B, H, D, S, "fp16", 16, 0, "fp16", 16, 0)
    k = _keys(B, H, S, D, seed=21)
    cache.append(k.cuda(), k.cuda())
    ws = torch.empty(kvq.snapkv_workspace_bytes(B, H, S, D, 32), dtype=torch.uint8, device="cuda")
    idx = torch.empty((B, H, 100), dtype=torch.int32, device="cuda")
    kplane = cache.plane("k_codes", B * H * cache.layout.cap_alloc * 2 * D).view(torch.float16)
    kvq.snapkv_select(kplane, cache.layout.cap_alloc, B, H, S, D, 32, 100, 4, None, idx, ws)
    _, ref = kvq.snapkv(k.cuda(), 32, 100, 4)
    assert torch.equal(idx, ref)


# ---- variants: max-pool smoothing, chunked prefill ---------------------------

@pytest.mark.parametrize("S,ksize", [(1, 1), (17, 3), (300, 5), (1000, 7), (5000, 63), (257, 9)])
def test_pool_matches_oracle(kvq, S, ksize):
    rng = np.random.default_rng(S + ksize)
    scores = (rng.random((2, 3, S)) * 1e-3).astype(np.float32)
    scores[:, :, rng.integers(0, S, size=min(S, 9))] = 0.5
    got = torch.empty((2, 3, S), dtype=torch.float32, device="cuda")
    kvq.snapkv_pool(torch.from_numpy(scores).cuda(), got, ksize)
    np.testing.assert_array_equal(got.cpu().numpy(), osk.max_pool(scores, ksize))


def test_pool_rejects_even_kernel_and_overlap(kvq):
    s = torch.zeros((1, 1, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KvqError):
        kvq.snapkv_pool(s, torch.empty_like(s), 4)
    with pytest.raises(kvq.KvqError):
        kvq.snapkv_pool(s, s, 3)


def test_select_on_pooled_scores(kvq):
    # snapkv_select -> snapkv_pool -> snapkv_topk equals the oracle's selection on the pooled fp32 scores
    B, H, S, D, w, budget, ns = 1, 4, 3000, 128, 32, 256, 4
    k = _keys(B, H, S, D, seed=77)
    scores, _ = kvq.snapkv(k.cuda(), w, budget, ns)
    pooled = torch.empty_like(scores)
    kvq.snapkv_pool(scores, pooled, 7)
    idx = torch.empty((B, H, budget), dtype=torch.int32, device="cuda")
    kvq.snapkv_topk(pooled, B, H, S, budget, ns, idx)
    p = pooled.cpu().numpy()
    np.testing.assert_array_equal(p, osk.max_pool(scores.cpu().numpy(), 7))
    for h in range(H):
        np.testing.assert_array_equal(idx.cpu().numpy()[0, h], osk.select_indices(p[0, h], budget, ns))


def _assert_valid_topk(ig, ref, eps, budget, n_sink):
    """ig is the exact top-k of ref when the cutoff gap exceeds 2 eps, else a valid one within eps."""
    S = len(ref)
    ns = min(n_sink, S)
    rest = np.sort(ref[ns:])[::-1]
    kk = budget - ns
    gap = rest[kk - 1] - rest[kk] if 0 < kk < len(rest) else np.inf
    if gap > 2 * eps:
        np.testing.assert_array_equal(ig, osk.select_indices(ref, budget, n_sink))
        return
    sel = set(ig.tolist())
    assert set(range(ns)) <= sel and len(sel) == budget
    cut = rest[kk - 1]
    for j in range(ns, S):
        if ref[j] > cut + 2 * eps:
            assert j in sel
        if ref[j] < cut - 2 * eps:
            assert j not in sel


def test_chunked_prefill_reenforces_budget(kvq):
    """Prefill in chunks: each chunk is appended to the kept rows, and when the cache holds more
    than the budget it is scored (the chunk's last w keys as proxies, read in place from the
    cache's fp16 K plane) and gathered back down to the budget.  Stored rows stay capped at the
    budget while the absolute position counts every prompt token."""
    from kvq_helpers import assert_cache_equal, host, oracle_spec
    from oracle.cache import OracleCache

    B, H, D, w, budget, ns = 1, 2, 64, 8, 48, 4
    chunks = [40, 30, 25, 50, 7, 64]
    cap = budget + max(chunks)
    cache = kvq.KVCache(B, H, D, cap, "fp16", 16, 0, "fp16", 16, 0)
    oc = OracleCache(oracle_spec(cache, None))
    ca = cache.layout.cap_alloc
    ws = torch.empty(kvq.snapkv_workspace_bytes(B, H, cap, D, w), dtype=torch.uint8, device="cuda")
    kplane = cache.plane("k_codes", B * H * ca * 2 * D).view(torch.float16)
    pos = 0
    for i, n in enumerate(chunks):
        k = _keys(B, H, n, D, seed=100 + i, sink_rows=4 if i == 0 else 0)
        v = _keys(B, H, n, D, seed=200 + i, sink_rows=0)
        cache.append(k.cuda(), v.cuda())
        oc.append(host(k), host(v))
        pos += n
        stored = oc.stored
        if stored > budget:
            idx = torch.empty((B, H, budget), dtype=torch.int32, device="cuda")
            scores = torch.empty((B, H, stored), dtype=torch.float32, device="cuda")
            kvq.snapkv_select(kplane, ca, B, H, stored, D, w, budget, ns, scores, idx, ws)
            kh, _ = oc.dequant()
            ig, sg = idx.cpu().numpy(), scores.cpu().numpy().astype(np.float64)
            for h in range(H):
                ref = osk.obs_window_scores(kh[0, h], w)
                eps = np.abs(sg[0, h] - ref).max()
                assert eps <= 1e-5 * ref.max() + 1e-9
                _assert_valid_topk(ig[0, h], ref, eps, budget, ns)
            cache.evict_keepset(idx)
            oc.evict_keepset(ig)    # the validated GPU choice, so both caches stay identical
        st = cache.stats()
        assert st.stored == oc.stored == min(stored, budget)
        assert st.pos == pos
        assert_cache_equal(cache, oc, f"chunk {i}")


def test_one_pass_and_two_pass_scores_are_the_same_bits(kvq):
    # 8 heads of a 16K prompt fit on the device at once: the scores come from
    # the one-pass cooperative launch.  The same keys as batch row 0 of an
    # 8-row batch (4096 scoring CTAs, more than the device holds at once) take
    # the two-pass path.  Both compute every logit and statistic in the same
    # order, so row 0's scores and indices must agree bit for bit.
    k = _keys(1, 8, 16384, 128, 51)
    kd = k.cuda()
    s1, i1 = kvq.snapkv(kd, 32, 512, 4)
    kb = torch.cat([kd] + [_keys(1, 8, 16384, 128, 52 + j).cuda() for j in range(7)], dim=0)
    s8, i8 = kvq.snapkv(kb, 32, 512, 4)
    assert torch.equal(s1[0], s8[0]) and torch.equal(i1[0], i8[0])
