"""Pins for the oracle's landmark gradient (section 1 and 3: the retriever
learns from the next-token loss through the relevance scores; rebuttal
"Cmt 1": r = sigma l_{c-1}.l_kappa) and its Gumbel-perturbed top-k (section
3.2: noise is added to the relevance scores before the top-k selection)."""
import math

import numpy as np
import pytest

import oracle


def selected_score_sum(lm, idx_ref, g, include_self):
    idx, r, _ = oracle.score_topk(lm, idx_ref.shape[-1], include_self, False)
    assert np.array_equal(idx, idx_ref), "the perturbation changed the selection"
    return float((g * np.where(idx >= 0, r, 0.0)).sum())


@pytest.mark.parametrize("include_self", [False, True])
def test_landmark_grad_matches_finite_differences(include_self):
    rng = np.random.default_rng(11)
    B, nC, D, k = 2, 9, 5, 3
    lm = rng.normal(size=(B, nC, D))            # continuous values: no ties
    idx, r, w = oracle.score_topk(lm, k, include_self, False)
    g = rng.normal(size=idx.shape) * (idx >= 0)
    dl = oracle.landmark_bwd(lm, idx, g)
    h = 1e-6
    fd = np.zeros_like(lm)
    for i in np.ndindex(*lm.shape):
        lp = lm.copy(); lp[i] += h
        lmn = lm.copy(); lmn[i] -= h
        fd[i] = (selected_score_sum(lp, idx, g, include_self) -
                 selected_score_sum(lmn, idx, g, include_self)) / (2 * h)
    np.testing.assert_allclose(dl, fd, rtol=1e-6, atol=1e-8)


def test_landmark_grad_hand_worked():
    # D = 1, three chunks, strict set, k = 1: only chunk 2 has a slot (chunk 0),
    # r = sigma * l1 * l0 with sigma = 1.
    lm = np.array([[[3.0], [5.0], [7.0]]])
    idx, r, w = oracle.score_topk(lm, 1, False, False, score_scale=1.0)
    assert idx[0, 2, 0] == 0 and r[0, 2, 0] == 15.0
    g = np.zeros((1, 3, 1)); g[0, 2, 0] = 2.0
    dl = oracle.landmark_bwd(lm, idx, g, score_scale=1.0)
    assert dl[0, 0, 0] == 2.0 * 5.0      # d/dl0 of g * l1 * l0
    assert dl[0, 1, 0] == 2.0 * 3.0      # d/dl1
    assert dl[0, 2, 0] == 0.0


def test_noisy_topk_without_noise_is_plain_topk():
    rng = np.random.default_rng(3)
    lm = rng.integers(-3, 4, size=(2, 30, 12)).astype(np.float64)
    for inc in (False, True):
        for ob in (False, True):
            a = oracle.score_topk(lm, 4, inc, ob)
            b = oracle.score_topk_noisy(lm, np.zeros((2, 30, 30), np.float32), 4, inc, ob)
            for x, y in zip(a, b):
                np.testing.assert_array_equal(x, y)


def test_noisy_topk_matches_float32_bruteforce():
    rng = np.random.default_rng(5)
    B, nC, D, k = 2, 25, 16, 5
    lm = rng.integers(-2, 3, size=(B, nC, D)).astype(np.float64)
    noise = rng.gumbel(size=(B, nC, nC)).astype(np.float32)
    sig = 1.0 / math.sqrt(D)
    idx, r, w = oracle.score_topk_noisy(lm, noise, k)
    for b in range(B):
        G = lm[b] @ lm[b].T
        for c in range(1, nC):
            cand = np.arange(c - 1)
            if cand.size == 0:
                assert (idx[b, c] == -1).all()
                continue
            key = (G[c - 1, cand].astype(np.float32) * np.float32(sig)).astype(np.float32) + noise[b, c, cand]
            order = cand[np.lexsort((cand, -key.astype(np.float64)))][:k]
            np.testing.assert_array_equal(idx[b, c, :order.size], order)
            np.testing.assert_allclose(r[b, c, :order.size], G[c - 1, order] * sig, rtol=1e-15)
            x = G[c - 1, order] * sig
            np.testing.assert_allclose(w[b, c, :order.size], np.exp(x - x.max()) / np.exp(x - x.max()).sum(),
                                       rtol=1e-12)


def test_noise_can_override_the_score_order():
    lm = np.array([[[1.0], [1.0], [2.0], [0.0], [1.0]]])       # D = 1
    noise = np.zeros((1, 5, 5), np.float32)
    noise[0, 4, 0] = 100.0                                      # chunk 4 prefers chunk 0
    idx, r, w = oracle.score_topk_noisy(lm, noise, 1, score_scale=1.0)
    assert idx[0, 4, 0] == 0
    assert r[0, 4, 0] == 0.0          # clean score l3 . l0 = 0, not the noisy key
    plain, _, _ = oracle.score_topk(lm, 1, score_scale=1.0)
    assert plain[0, 4, 0] == 0        # all clean scores tie at 0 here; lowest index anyway
    noise[0, 4, 2] = 200.0
    idx, _, _ = oracle.score_topk_noisy(lm, noise, 1, score_scale=1.0)
    assert idx[0, 4, 0] == 2
