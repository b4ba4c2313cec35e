"""Pins for the oracle's relevance scoring, top-k and weight softmax.

The GCA retrieval step (rebuttal "Cmt 1": r_t^k = l_t^T l_k / sqrt(d) for
G=1; official README "Model Architecture": the landmark of chunk c-1 selects
the past chunks used by chunk c; rebuttal Q4: Eq. 3 is the softmax off by
one) is checked here against things other than the oracle itself: a
hand-worked example, a brute-force Gram matrix with a stable Python sort, and
closed forms of the two softmax variants.
"""
import math

import numpy as np
import pytest

import oracle
from retrieval_sparse_attention_gb300 import inputs


def brute_topk(lm, topk, include_self, off_by_one, scale):
    B, nC, D = lm.shape
    idx = -np.ones((B, nC, topk), dtype=np.int32)
    r = np.zeros((B, nC, topk))
    w = np.zeros((B, nC, topk))
    for b in range(B):
        G = lm[b] @ lm[b].T                      # every chunk pair, exact for integers
        for c in range(1, nC):
            t = c - 1
            cand = list(range(t + 1 if include_self else t))
            cand.sort(key=lambda kap: (-G[t, kap], kap))
            sel = cand[:topk]
            for j, kap in enumerate(sel):
                idx[b, c, j] = kap
                r[b, c, j] = G[t, kap] * scale
            if sel:
                x = r[b, c, :len(sel)]
                if off_by_one:
                    e = np.exp(x)
                    w[b, c, :len(sel)] = e / (1.0 + e.sum())
                else:
                    e = np.exp(x - x.max())
                    w[b, c, :len(sel)] = e / e.sum()
    return idx, r, w


def test_hand_worked_example():
    # D = 1, landmarks 1, 2, 2, 0, 5 (strict causal set, scale 1, k = 2).
    lm = np.array([1, 2, 2, 0, 5], dtype=np.float64).reshape(1, 5, 1)
    idx, r, w = oracle.score_topk(lm, 2, include_self=False, off_by_one=False, score_scale=1.0)
    # c=0, c=1: no earlier chunk than c-1 -> empty.
    assert (idx[0, 0] == -1).all() and (idx[0, 1] == -1).all()
    assert (w[0, 0] == 0).all() and (w[0, 1] == 0).all()
    # c=2: landmark 1 (value 2) vs chunk 0 (value 1): one candidate, s = 2.
    assert list(idx[0, 2]) == [0, -1] and r[0, 2, 0] == 2.0 and w[0, 2, 0] == 1.0
    # c=3: landmark 2 (value 2) vs chunks 0, 1: s = 2, 4 -> order 1, 0.
    assert list(idx[0, 3]) == [1, 0]
    assert list(r[0, 3]) == [4.0, 2.0]
    e2 = math.exp(2.0)
    assert np.allclose(w[0, 3], [e2 / (1 + e2), 1 / (1 + e2)], rtol=1e-15)
    # c=4: landmark 3 (value 0): all three scores tie at 0 -> lower index first.
    assert list(idx[0, 4]) == [0, 1]
    assert np.allclose(w[0, 4], [0.5, 0.5], rtol=1e-15)
    # include_self: chunk c-1 joins the candidates.
    idx2, r2, _ = oracle.score_topk(lm, 2, include_self=True, off_by_one=False, score_scale=1.0)
    assert list(idx2[0, 1]) == [0, -1] and r2[0, 1, 0] == 1.0     # l0 . l0
    assert list(idx2[0, 3]) == [1, 2]                             # 4 == 4: tie -> lower index


def test_signed_zero_scores_tie_toward_lower_index():
    # Every score is zero, some computed from negative zeros (-0 * x, -0 + -0):
    # -0 and +0 are the same score, so every slot goes to the lowest indices, in
    # order, and the vanilla weights are uniform.
    lm = np.zeros((1, 9, 4))
    lm[0, 1::2] = -0.0
    lm[0, 2, 0] = 3.0                 # chunk 2 is orthogonal to every other landmark
    lm[0, 4, :] = np.array([-0.0, 0.0, -0.0, 0.0])
    assert np.signbit(lm[0, 1]).all()
    idx, r, w = oracle.score_topk(lm, 3, include_self=False, off_by_one=False, score_scale=1.0)
    for c in range(4, 9):
        assert list(idx[0, c]) == [0, 1, 2], c
        assert (r[0, c] == 0).all()
        assert np.allclose(w[0, c], 1.0 / 3.0, rtol=1e-15)
    di, dr, dw = oracle.decode_retrieve(lm[0], -lm[0, 1], 4)
    assert list(di) == [0, 1, 2, 3]
    assert np.allclose(dw, 0.25, rtol=1e-15)


@pytest.mark.parametrize("include_self", [False, True])
@pytest.mark.parametrize("off_by_one", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 4, 1), (1, 2, 3, 2), (2, 5, 8, 3), (3, 17, 130, 5),
                                   (2, 40, 7, 8), (1, 33, 2, 16)])
def test_topk_matches_bruteforce(shape, include_self, off_by_one):
    B, nC, D, k = shape
    rng = np.random.default_rng(1000 + nC * 7 + D)
    lm = rng.integers(-2, 3, size=(B, nC, D)).astype(np.float64)   # small range: many ties
    scale = 1.0 / math.sqrt(D)
    got = oracle.score_topk(lm, k, include_self, off_by_one, scale)
    want = brute_topk(lm, k, include_self, off_by_one, scale)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_allclose(got[1], want[1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[2], want[2], rtol=1e-12, atol=1e-15)


def test_tiny_workload_topk():
    wl = inputs.WORKLOADS["tiny_fp32"]
    x = inputs.make(wl)
    lm = x["lm"].double().numpy()
    got = oracle.score_topk(lm, wl.topk, False, wl.off_by_one)
    want = brute_topk(lm, wl.topk, False, wl.off_by_one, 1.0 / math.sqrt(wl.D))
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_allclose(got[2], want[2], rtol=1e-12)
    # strict causal set: chunk c sees c-1 candidates, so min(k, c-1) valid slots
    valid = (got[0][0] >= 0).sum(-1)
    assert list(valid) == [max(0, min(wl.topk, c - 1)) for c in range(wl.nC)]


@pytest.mark.parametrize("m", [1, 2, 5, 8])
def test_weights_closed_forms(m):
    rng = np.random.default_rng(m)
    r = rng.normal(size=m) * 3
    w = oracle.weights_from_scores(r, off_by_one=False)
    assert abs(w.sum() - 1.0) < 1e-14
    # shift invariance of the vanilla softmax
    np.testing.assert_allclose(oracle.weights_from_scores(r + 17.0, False), w, rtol=1e-12)
    # equal scores -> uniform
    np.testing.assert_allclose(oracle.weights_from_scores(np.full(m, 0.3), False), np.full(m, 1.0 / m))
    # off by one: w_j = e^{r_j} / (1 + sum e^{r_i}); the missing mass is 1 / (1 + sum e^r)
    w1 = oracle.weights_from_scores(r, off_by_one=True)
    den = 1.0 + np.exp(r).sum()
    assert abs((1.0 - w1.sum()) - 1.0 / den) < 1e-14
    assert w1.sum() < 1.0
    # ratios between slots are the same as in the vanilla softmax
    np.testing.assert_allclose(w1 / w1.sum(), w, rtol=1e-12)


def test_weights_special_values():
    # one slot: vanilla gives 1, off-by-one gives the logistic sigmoid
    for x in (-30.0, -1.0, 0.0, 2.5, 40.0):
        assert oracle.weights_from_scores([x], False)[0] == 1.0
        assert abs(oracle.weights_from_scores([x], True)[0] - 1.0 / (1.0 + math.exp(-x))) < 1e-15
    # very large scores stay finite in both modes
    for ob in (False, True):
        w = oracle.weights_from_scores([900.0, 899.0, -900.0], ob)
        assert np.isfinite(w).all()
        np.testing.assert_allclose(w[:2] / w[:2].sum(), [1 / (1 + math.exp(-1)), 1 / (1 + math.e)])


@pytest.mark.parametrize("N,D,k", [(1, 3, 1), (5, 2, 8), (1000, 16, 8), (4097, 33, 16), (300, 1, 32)])
@pytest.mark.parametrize("off_by_one", [False, True])
def test_decode_matches_bruteforce(N, D, k, off_by_one):
    rng = np.random.default_rng(N + D)
    lm = rng.integers(-2, 3, size=(N, D)).astype(np.float64)
    ql = rng.integers(-2, 3, size=D).astype(np.float64)
    scale = 1.0 / math.sqrt(D)
    idx, r, w = oracle.decode_retrieve(lm, ql, k, off_by_one, scale)
    s = lm @ ql
    order = np.lexsort((np.arange(N), -s))[:k]          # score desc, index asc
    m = len(order)
    np.testing.assert_array_equal(idx[:m], order)
    assert (idx[m:] == -1).all() and (w[m:] == 0).all()
    np.testing.assert_allclose(r[:m], s[order] * scale, atol=1e-12)
    x = s[order] * scale
    if off_by_one:
        want = np.exp(x) / (1.0 + np.exp(x).sum())
    else:
        want = np.exp(x - x.max()) / np.exp(x - x.max()).sum()
    np.testing.assert_allclose(w[:m], want, rtol=1e-12)


def test_decode_agrees_with_causal_scoring():
    # The last query chunk of a training row with include_self scores the
    # landmark of chunk nC-2 against chunks 0..nC-2: the decode retrieval over
    # those nC-1 landmarks with that query must give the same slots.
    rng = np.random.default_rng(7)
    lm = rng.integers(-4, 5, size=(1, 50, 24)).astype(np.float64)
    idx, r, w = oracle.score_topk(lm, 8, include_self=True, off_by_one=True)
    di, dr, dw = oracle.decode_retrieve(lm[0, :49], lm[0, 48], 8, off_by_one=True)
    np.testing.assert_array_equal(idx[0, 49], di)
    np.testing.assert_allclose(w[0, 49], dw, rtol=1e-14)
