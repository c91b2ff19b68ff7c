"""Pins for the oracle's routing and weighted combine around the expert GEMM.

Source: "Where the engine is going: HRX and the NPU", section "4-bit
activations reach the MoE experts" (the route covers the expert matmuls of a
mixture-of-experts model).  The pages do not spell out the router; the
readings pinned here: top k experts by logit with ties to the lower id, listed
by decreasing logit; weights = softmax over the k chosen logits (the full
softmax's top-k probabilities renormalised); rows grouped by expert, then by
token; the combine adds a token's k rows in choice order with fp32 fma from
+0.  Each check compares the oracle with an independent computation or a
closed form."""
import numpy as np

import oracle
from hadamard_rotated_bit_gb300 import workloads as wl


def _logits_with_ties(T, E, seed):
    r = np.random.default_rng(seed)
    l = r.standard_normal((T, E)).astype(np.float32)
    # copy some values across columns of the same row: equal logits
    for t in range(0, T, 3):
        a, b = r.integers(0, E, 2)
        l[t, b] = l[t, a]
    l[5, :] = 0.25          # a row of equal logits
    return l


def _topk_lexsort(l, k):
    ids = np.arange(l.shape[1])
    return np.stack([np.lexsort((ids, -row.astype(np.float64)))[:k] for row in l]).astype(np.int32)


def test_topk_matches_an_independent_sort():
    for T, E, k in ((200, 37, 5), (64, 128, 8), (9, 4, 4), (30, 1, 1)):
        l = _logits_with_ties(T, E, T + E)
        ids, w, off, ridx, row_of = oracle.moe_route(l, k)
        assert np.array_equal(ids, _topk_lexsort(l, k))


def test_ties_and_weights_closed_form():
    l = np.array([[0.5, 0.9, 0.9, 0.1, 0.9]], np.float32)
    ids, w, off, ridx, row_of = oracle.moe_route(l, 3)
    assert ids.tolist() == [[1, 2, 4]]
    # three equal chosen logits: exp(0) = 1 each, sum 3, weight fl(1/3)
    assert np.array_equal(w, np.full((1, 3), np.float32(1) / np.float32(3)))
    ids1, w1, _, _, _ = oracle.moe_route(l, 1)
    assert ids1.tolist() == [[1]] and w1.tolist() == [[1.0]]
    # the row of equal logits takes the lowest ids
    ids5, _, _, _, _ = oracle.moe_route(_logits_with_ties(8, 6, 0), 2)
    assert ids5[5].tolist() == [0, 1]


def test_weights_are_the_renormalised_softmax():
    l = _logits_with_ties(300, 64, 3) * np.float32(3)
    k = 6
    ids, w, _, _, _ = oracle.moe_route(l, k)
    l64 = l.astype(np.float64)
    # softmax over the chosen logits
    ch = np.take_along_axis(l64, ids.astype(np.int64), axis=1)
    e = np.exp(ch - ch[:, :1])
    ref = e / e.sum(axis=1, keepdims=True)
    assert np.max(np.abs(w - ref) / ref) <= 1e-6
    # the same from the full softmax (a different formula)
    p = np.exp(l64 - l64.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ps = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    assert np.max(np.abs(w - ps / ps.sum(axis=1, keepdims=True)) / ref) <= 1e-6
    assert np.all(np.diff(w.astype(np.float64), axis=1) <= 0)   # decreasing logits
    assert np.max(np.abs(w.astype(np.float64).sum(axis=1) - 1)) <= k * 2.0 ** -23


def test_grouping_is_by_expert_then_token():
    T, E, k = 150, 21, 4
    l = _logits_with_ties(T, E, 9)
    ids, w, off, ridx, row_of = oracle.moe_route(l, k)
    cnt = np.bincount(ids.reshape(-1), minlength=E)
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(cnt)]))
    tok = np.repeat(np.arange(T), k)
    exp = ids.reshape(-1).astype(np.int64)
    order = np.lexsort((tok, exp))
    assert np.array_equal(ridx, tok[order])
    # row_of is the inverse: the grouped row of choice (t, j) holds token t in group ids[t, j]
    assert np.array_equal(np.sort(row_of.reshape(-1)), np.arange(T * k))
    assert np.array_equal(ridx[row_of], np.repeat(np.arange(T)[:, None], k, axis=1))
    grp = np.searchsorted(off, row_of, side="right") - 1
    assert np.array_equal(grp, ids)


def test_route_matches_the_workload_grouping():
    cfg = wl.MOE
    ridx_ref, off_ref, exp_ref = wl.moe_routing(cfg)
    ids, w, off, ridx, row_of = oracle.moe_route(wl.moe_logits(cfg), cfg.top_k)
    assert np.array_equal(off, off_ref) and np.array_equal(ridx, ridx_ref)
    assert np.array_equal(np.repeat(np.arange(cfg.E), np.diff(off)), exp_ref)


def test_combine_one_hot_and_order():
    y = np.array([[1e8, 2.0], [-1e8, 3.0], [1.0, 5.0]], np.float32)
    row_of = np.array([[0, 1, 2], [2, 1, 0]], np.int32)
    w = np.ones((2, 3), np.float32)
    out = oracle.moe_combine(y, row_of, w)
    # choice order: 1e8, then 0, then 1 -> 1;  the other order loses the 1
    assert out[0, 0] == 1.0 and out[1, 0] == 0.0
    assert out[0, 1] == 10.0
    oh = np.array([[0, 1, 0], [0, 0, 1]], np.float32)
    assert np.array_equal(oracle.moe_combine(y, row_of, oh), np.stack([y[1], y[0]]))


def test_combine_within_the_fp32_bound():
    r = np.random.default_rng(4)
    T, k, H = 40, 8, 96
    R = T * k
    y = r.standard_normal((R, H)).astype(np.float32)
    row_of = r.permutation(R).reshape(T, k).astype(np.int32)
    w = r.random((T, k)).astype(np.float32)
    out = oracle.moe_combine(y, row_of, w).astype(np.float64)
    terms = w.astype(np.float64)[:, :, None] * y.astype(np.float64)[row_of]
    ref = terms.sum(axis=1)
    bound = (k + 1) * 2.0 ** -24 * np.abs(terms).sum(axis=1)
    assert np.all(np.abs(out - ref) <= bound)


def test_non_finite_logits_closed_forms():
    """Masked (-inf), infinite and NaN logits follow the limits of the rule: a
    NaN ranks below every number (-inf included); weights are the softmax over
    the finite chosen logits (0 for a chosen -inf or NaN), shared equally by
    the +inf choices when the largest is +inf, and equal when every chosen
    logit is -inf or NaN."""
    ninf, nan, inf = -np.inf, np.nan, np.inf
    l = np.array([[1.0, ninf, 2.0, ninf, nan, 0.5]], np.float32)
    ids, w, _, _, _ = oracle.moe_route(l, 4)
    assert ids.tolist() == [[2, 0, 5, 1]]
    e = np.exp(np.array([0.0, -1.0, -1.5], np.float64))
    assert np.allclose(w[0, :3], e / e.sum(), rtol=1e-6, atol=0)
    assert w[0, 3] == 0.0
    ids, w, _, _, _ = oracle.moe_route(l, 6)
    assert ids.tolist() == [[2, 0, 5, 1, 3, 4]] and w[0, 3:].tolist() == [0.0, 0.0, 0.0]
    third = np.float32(1) / np.float32(3)
    for row in ([ninf] * 5, [nan] * 5, [nan, ninf, ninf, nan, nan]):
        ids, w, _, _, _ = oracle.moe_route(np.array([row], np.float32), 3)
        assert np.array_equal(w, np.full((1, 3), third))
    ids, _, _, _, _ = oracle.moe_route(np.array([[nan, ninf, ninf, nan, nan]], np.float32), 3)
    assert ids.tolist() == [[1, 2, 0]]
    ids, w, _, _, _ = oracle.moe_route(np.array([[0.0, inf, 3.0, inf]], np.float32), 3)
    assert ids.tolist() == [[1, 3, 2]] and w.tolist() == [[0.5, 0.5, 0.0]]
    # masked experts are never grouped ahead of a finite choice of the same token
    l = np.array([[ninf, 0.0, ninf, 1.0], [2.0, ninf, ninf, ninf]], np.float32)
    ids, w, off, ridx, row_of = oracle.moe_route(l, 2)
    assert ids.tolist() == [[3, 1], [0, 1]]
    assert w[1].tolist() == [1.0, 0.0]
