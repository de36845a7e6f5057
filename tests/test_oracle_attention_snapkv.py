"""Pins of the oracle's decode attention and SnapKV scoring/selection."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as att
from oracle import snapkv as sk


# ------------------------------------------------------------- attention --

def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((2, 6, 32))
    k = rng.standard_normal((2, 3, 1, 32))
    v = rng.standard_normal((2, 3, 1, 32))
    o = att.decode_attention(q, k, v)
    for h in range(6):
        np.testing.assert_array_equal(o[:, h], v[:, h // 2, 0])


def test_equal_keys_give_mean_value():
    rng = np.random.default_rng(2)
    k = np.repeat(rng.standard_normal((1, 2, 1, 16)), 50, axis=2)
    v = rng.standard_normal((1, 2, 50, 16))
    q = rng.standard_normal((1, 2, 16)) * 10
    o = att.decode_attention(q, k, v)
    np.testing.assert_allclose(o, v.mean(axis=2), rtol=1e-12, atol=1e-14)


def test_gqa_equals_mha_on_repeated_heads():
    rng = np.random.default_rng(3)
    B, Hkv, G, T, D = 2, 2, 4, 33, 32
    q = rng.standard_normal((B, Hkv * G, D))
    k = rng.standard_normal((B, Hkv, T, D))
    v = rng.standard_normal((B, Hkv, T, D))
    o_gqa = att.decode_attention(q, k, v)
    o_mha = att.decode_attention(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1))
    np.testing.assert_allclose(o_gqa, o_mha, rtol=0, atol=1e-14)


def test_matches_torch_sdpa_float64():
    rng = np.random.default_rng(4)
    B, Hkv, G, T, D = 3, 2, 3, 45, 64
    q = rng.standard_normal((B, Hkv * G, D))
    k = rng.standard_normal((B, Hkv, T, D)) * 2
    v = rng.standard_normal((B, Hkv, T, D))
    o = att.decode_attention(q, k, v)
    tq = torch.from_numpy(q)[:, :, None, :]
    tk = torch.from_numpy(np.repeat(k, G, axis=1))
    tv = torch.from_numpy(np.repeat(v, G, axis=1))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[:, :, 0, :].numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


def test_row_permutation_invariance():
    # the ring layout stores the same tokens in another order
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 4, 32))
    k = rng.standard_normal((1, 2, 60, 32))
    v = rng.standard_normal((1, 2, 60, 32))
    perm = rng.permutation(60)
    np.testing.assert_allclose(att.decode_attention(q, k, v), att.decode_attention(q, k[:, :, perm], v[:, :, perm]),
                               rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- SnapKV --

def _scores_by_loops(k, w):
    """Brute force: each logit, each exponential and each normaliser written out."""
    S, D = k.shape
    w = min(w, S)
    out = [0.0] * S
    for r in range(S - w, S):
        logits = [sum(float(k[r, d]) * float(k[j, d]) for d in range(D)) / math.sqrt(D) for j in range(S)]
        m = max(logits)
        e = [math.exp(x - m) for x in logits]
        z = sum(e)
        for j in range(S):
            out[j] += e[j] / z / w
    return np.array(out)


def test_scores_brute_force_and_properties():
    rng = np.random.default_rng(6)
    k = rng.standard_normal((23, 8)) * 1.5
    s = sk.obs_window_scores(k, 5)
    np.testing.assert_allclose(s, _scores_by_loops(k, 5), rtol=1e-12, atol=1e-15)
    assert s.shape == (23,)
    assert np.all((s >= 0) & (s <= 1))
    assert abs(s.sum() - 1.0) < 1e-12


def test_single_row_window_is_one_softmax_row():
    rng = np.random.default_rng(7)
    k = rng.standard_normal((50, 16))
    s = sk.obs_window_scores(k, 1)
    ref = torch.softmax(torch.from_numpy(k[-1] @ k.T / 4.0), dim=0).numpy()
    np.testing.assert_allclose(s, ref, rtol=1e-12, atol=1e-15)


def test_window_clamped_to_sequence():
    rng = np.random.default_rng(8)
    k = rng.standard_normal((6, 8))
    np.testing.assert_array_equal(sk.obs_window_scores(k, 32), sk.obs_window_scores(k, 6))


def _brute_select(scores, budget, n_sink):
    S = len(scores)
    if budget >= S:
        return list(range(S))
    ns = min(n_sink, S)
    rest = sorted(range(ns, S), key=lambda j: (-float(scores[j]), j))
    return sorted(list(range(ns)) + rest[: budget - ns])


@pytest.mark.parametrize("S,budget,n_sink", [(50, 10, 4), (50, 50, 4), (50, 60, 4), (7, 3, 3), (100, 31, 0), (64, 8, 1)])
def test_selection_brute_force(S, budget, n_sink):
    rng = np.random.default_rng(S * 7 + budget)
    scores = rng.random(S).astype(np.float32)
    scores[rng.integers(0, S, 5)] = scores[3]          # a few exact ties
    idx = sk.select_indices(scores, budget, n_sink)
    assert idx.tolist() == _brute_select(scores, budget, n_sink)
    assert len(idx) == min(budget, S)
    assert np.all(np.diff(idx) > 0)


def test_sinks_win_with_zero_scores(golden):
    d = golden("snapkv_page.json")["defaults"]
    scores = np.zeros(1000, np.float32)
    scores[600:] = 0.5
    idx = sk.select_indices(scores, d["snap_budget"], d["snap_n_sink"])
    assert idx[: d["snap_n_sink"]].tolist() == list(range(d["snap_n_sink"]))
    assert len(idx) == d["snap_budget"]


def test_planted_top_rows_are_selected():
    rng = np.random.default_rng(9)
    S = 4096
    scores = (rng.random(S) * 1e-4).astype(np.float32)
    planted = rng.choice(np.arange(4, S), 60, replace=False)
    scores[planted] = 0.5
    idx = sk.select_indices(scores, 64, 4)
    assert set(idx.tolist()) == set(range(4)) | set(planted.tolist())


def test_equal_scores_keep_lower_positions():
    idx = sk.select_indices(np.ones(20, np.float32), 8, 2)
    assert idx.tolist() == list(range(8))


def test_sink_budget_validation():
    with pytest.raises(ValueError):
        sk.select_indices(np.ones(10, np.float32), 3, 4)


def test_end_to_end_keeps_planted_key_rows():
    # proxy queries that align with a few planted keys pull those rows in
    rng = np.random.default_rng(10)
    S, D, w = 300, 32, 8
    k = rng.standard_normal((1, 1, S, D)) * 0.3
    direction = rng.standard_normal(D)
    planted = [50, 120, 200]
    for p in planted:
        k[0, 0, p] = direction * 3
    k[0, 0, S - w:] += direction
    scores, idx = sk.snapkv_select(k, w, 16, 4)
    assert set(planted) <= set(idx[0, 0].tolist())
    assert idx.shape == (1, 1, 16)
    np.testing.assert_allclose(scores.sum(-1), 1.0, rtol=1e-12)


def test_keepset_gather_order():
    rows = np.arange(2 * 3 * 10).reshape(2, 3, 10)
    idx = np.array([[[0, 4, 9]] * 3] * 2)
    out = sk.keepset_gather(rows, idx)
    np.testing.assert_array_equal(out[1, 2], rows[1, 2, [0, 4, 9]])


# ---- variants: max-pool smoothing, coverage --------------------------------

@pytest.mark.parametrize("k", [1, 3, 5, 7])
def test_max_pool_matches_torch_max_pool1d(k):
    rng = np.random.default_rng(20 + k)
    s = rng.random((2, 3, 41))
    ref = torch.nn.functional.max_pool1d(torch.from_numpy(s).reshape(6, 1, 41), k, stride=1, padding=k // 2)
    np.testing.assert_array_equal(sk.max_pool(s, k), ref.reshape(2, 3, 41).numpy())


def test_max_pool_identity_spike_and_bounds():
    rng = np.random.default_rng(21)
    s = rng.random(30) * 1e-3
    np.testing.assert_array_equal(sk.max_pool(s, 1), s)
    s[10] = 1.0
    p = sk.max_pool(s, 5)
    assert np.all(p >= s)
    assert np.all(p[8:13] == 1.0) and p[7] < 1.0 and p[13] < 1.0
    with pytest.raises(ValueError):
        sk.max_pool(s, 4)


def test_coverage_and_random_baseline():
    s = np.array([0.4, 0.1, 0.1, 0.1, 0.1, 0.1, 0.1])
    assert sk.coverage(s, [0, 1, 2]) == pytest.approx(0.6)
    # sinks {0} plus 2 of the 6 others drawn uniformly: 0.4 + 2/6 * 0.6
    assert sk.random_coverage(s, 3, 1) == pytest.approx(0.6)
    assert sk.random_coverage(s, 7, 1) == 1.0
    # planted scores: the top-k keeps more mass than a random set of the same size
    rng = np.random.default_rng(22)
    sc = rng.random(500) * 1e-4
    sc[[50, 90, 300]] = 0.3
    idx = sk.select_indices(sc, 20, 4)
    assert sk.coverage(sc, idx) > sk.random_coverage(sc, 20, 4) + 0.5


@pytest.mark.parametrize("scale", [0.5, 0.02, 1.7])
def test_explicit_softmax_scale(scale):
    # a caller-given scale replaces 1/sqrt(D): equal to torch SDPA (float64)
    # with that scale, and to the default-scale result for q * scale * sqrt(D)
    rng = np.random.default_rng(41)
    B, Hkv, G, T, D = 2, 2, 2, 33, 64
    q = rng.standard_normal((B, Hkv * G, D))
    k = rng.standard_normal((B, Hkv, T, D))
    v = rng.standard_normal((B, Hkv, T, D))
    o = att.decode_attention(q, k, v, scale)
    tq = torch.from_numpy(q)[:, :, None, :]
    tk = torch.from_numpy(np.repeat(k, G, axis=1))
    tv = torch.from_numpy(np.repeat(v, G, axis=1))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[:, :, 0, :].numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o, att.decode_attention(q * scale * math.sqrt(D), k, v), rtol=1e-12, atol=1e-13)
    assert not np.allclose(o, att.decode_attention(q, k, v), atol=1e-3)


def _random_bounds(rng, T, n):
    cuts = np.sort(rng.integers(0, T + 1, size=n - 1))
    edges = [0, *cuts.tolist(), T]
    return [(edges[i], edges[i + 1]) for i in range(n)]


@pytest.mark.parametrize("T,n", [(1, 1), (7, 3), (64, 1), (300, 5), (300, 32), (1000, 128)])
def test_split_merge_equals_unsplit_attention(T, n):
    # the split-KV merge rule: any partition of the rows into splits, empty ones
    # included and in any order, merges to the same output as one softmax over all rows
    rng = np.random.default_rng(T * 131 + n)
    D = 64
    q = rng.standard_normal(D) * 2
    k = rng.standard_normal((T, D)) * 1.5
    v = rng.standard_normal((T, D))
    ref = att.decode_attention(q[None, None], k[None, None], v[None, None])[0, 0]
    bounds = _random_bounds(rng, T, n)
    parts = att.split_partials(q, k, v, bounds)
    np.testing.assert_allclose(att.merge_partials(parts), ref, rtol=1e-12, atol=1e-13)
    order = rng.permutation(len(parts))
    np.testing.assert_allclose(att.merge_partials([parts[i] for i in order]), ref, rtol=1e-12, atol=1e-13)
    # one split per row: each split's l is 1 and acc its own value row
    singles = att.split_partials(q, k, v, [(t, t + 1) for t in range(T)])
    assert all(l == 1.0 for _, l, _ in singles)
    np.testing.assert_allclose(att.merge_partials(singles), ref, rtol=1e-12, atol=1e-13)


def test_split_merge_with_far_apart_maxima():
    # splits whose maxima differ by hundreds: exp(m_i - m*) underflows to 0 for
    # the low split without producing NaN, and the high split decides the output
    D = 16
    q = np.ones(D)
    k = np.zeros((4, D))
    k[2:] = 100.0
    v = np.arange(4 * D, dtype=np.float64).reshape(4, D)
    parts = att.split_partials(q, k, v, [(0, 2), (2, 4)], scale=1.0)
    out = att.merge_partials(parts)
    np.testing.assert_allclose(out, v[2:].mean(axis=0), rtol=1e-12)
    assert np.all(np.isfinite(out))


def test_softmax_shift_invariance():
    # adding one vector c_h to every key of kv head h adds q . c_h to every score
    # of each query on that head, the same constant across its row: the output
    # must not move (a per-token shift, by contrast, must)
    rng = np.random.default_rng(43)
    B, Hkv, G, T, D = 2, 3, 2, 50, 32
    q = rng.standard_normal((B, Hkv * G, D))
    k = rng.standard_normal((B, Hkv, T, D))
    v = rng.standard_normal((B, Hkv, T, D))
    c = rng.standard_normal((B, Hkv, 1, D)) * 5
    o = att.decode_attention(q, k, v)
    np.testing.assert_allclose(att.decode_attention(q, k + c, v), o, rtol=1e-10, atol=1e-12)
    per_token = rng.standard_normal((B, Hkv, T, 1)) * c
    assert not np.allclose(att.decode_attention(q, k + per_token, v), o, atol=1e-3)
