"""Pins for the oracle's GCA forward (stage 1 per-chunk attention, stage 2
weighted fusion; official README "Model Architecture", Figure 1/2, Eq. 2 as
the batch form of Figure 2 per the rebuttal answer to W2) and its
log-sum-exp output (App. B: the forward returns O and the log-sum-exp).

Checked against: a brute force that materialises every per-slot output
O_t^j, PyTorch's scaled_dot_product_attention for the k = 1 reduction, the
closed form for a chunk whose keys are all equal, SciPy's logsumexp, and the
empty-slot special cases.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle


def make_case(seed, B, nC, S, H, d, k, include_self=True, off_by_one=False, lm_range=3):
    rng = np.random.default_rng(seed)
    lm = rng.integers(-lm_range, lm_range + 1, size=(B, nC, 3 * H)).astype(np.float64)
    idx, r, w = oracle.score_topk(lm, k, include_self, off_by_one)
    q = rng.normal(size=(B, nC * S, H, d))
    kk = rng.normal(size=(B, nC * S, H, d))
    v = rng.normal(size=(B, nC * S, H, d))
    return q, kk, v, idx, r, w


def brute_fwd(q, k, v, idx, w, S, scale):
    """Materialise O_t^j for every (b, c, t, h, j), then fuse."""
    B, L, H, d = q.shape
    nQ, topk = idx.shape[1], idx.shape[2]
    Oj = np.zeros((B, L, H, topk, d))
    lse = np.full((B, L, H, topk), -np.inf)
    for b in range(B):
        for c in range(nQ):
            for j in range(topk):
                kap = idx[b, c, j]
                if kap < 0:
                    continue
                Kc = k[b, kap * S:(kap + 1) * S]            # [S, H, d]
                Vc = v[b, kap * S:(kap + 1) * S]
                Qc = q[b, c * S:(c + 1) * S]                # [S, H, d]
                a = np.einsum("thd,shd->hts", Qc, Kc) * scale
                lse[b, c * S:(c + 1) * S, :, j] = logsumexp(a, axis=-1).T
                p = softmax(a, axis=-1)
                Oj[b, c * S:(c + 1) * S, :, j] = np.einsum("hts,shd->thd", p, Vc)
    wt = np.repeat(w, S, axis=1)                            # [B, L, k]
    O = np.einsum("blhjd,blj->blhd", Oj, wt)
    return O, lse, Oj


@pytest.mark.parametrize("case", [
    dict(seed=1, B=1, nC=4, S=2, H=1, d=1, k=1),
    dict(seed=2, B=2, nC=6, S=4, H=2, d=3, k=3),
    dict(seed=3, B=1, nC=9, S=5, H=3, d=4, k=4, include_self=False),
    dict(seed=4, B=2, nC=7, S=8, H=2, d=8, k=2, off_by_one=True),
])
def test_fwd_matches_bruteforce(case):
    S = case["S"]
    q, k, v, idx, r, w = make_case(**case)
    scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = oracle.fwd(q, k, v, idx, w, S)
    bo, blse, _ = brute_fwd(q, k, v, idx, w, S, scale)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-13)
    fin = np.isfinite(blse)
    assert (np.isfinite(lse) == fin).all()
    np.testing.assert_allclose(lse[fin], blse[fin], rtol=1e-13)


@pytest.mark.parametrize("off_by_one", [False, True])
def test_k1_reduces_to_plain_attention(off_by_one):
    # With one slot, stage 2 multiplies a single attention output by w:
    # w = 1 (vanilla) or sigmoid(r) (off by one).  Compare with PyTorch SDPA
    # over the retrieved chunk.
    B, nC, S, H, d = 2, 6, 8, 3, 4
    q, k, v, idx, r, w = make_case(11, B, nC, S, H, d, 1, include_self=True, off_by_one=off_by_one)
    o, _ = oracle.fwd(q, k, v, idx, w, S)
    for b in range(B):
        for c in range(nC):
            kap = idx[b, c, 0]
            got = o[b, c * S:(c + 1) * S]
            if kap < 0:
                assert (got == 0).all()
                continue
            Q = torch.from_numpy(q[b, c * S:(c + 1) * S]).permute(1, 0, 2)   # [H, S, d]
            K = torch.from_numpy(k[b, kap * S:(kap + 1) * S]).permute(1, 0, 2)
            V = torch.from_numpy(v[b, kap * S:(kap + 1) * S]).permute(1, 0, 2)
            ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V).permute(1, 0, 2).numpy()
            gain = 1.0 / (1.0 + math.exp(-r[b, c, 0])) if off_by_one else 1.0
            np.testing.assert_allclose(got, gain * ref, rtol=1e-11, atol=1e-13)


def test_equal_keys_give_mean_of_values():
    # If every key of a chunk is the same vector, attention over it is uniform
    # and O^j is the mean of that chunk's values, for any query.
    B, nC, S, H, d = 1, 7, 6, 2, 5
    q, k, v, idx, r, w = make_case(5, B, nC, S, H, d, 3)
    for kap in range(nC):
        k[0, kap * S:(kap + 1) * S] = k[0, kap * S]
    o, lse = oracle.fwd(q, k, v, idx, w, S)
    for c in range(nC):
        want = np.zeros((H, d))
        for j in range(3):
            kap = idx[0, c, j]
            if kap >= 0:
                want += w[0, c, j] * v[0, kap * S:(kap + 1) * S].mean(axis=0)
                # lse = a + ln S for S equal logits a
                a = np.einsum("thd,hd->th", q[0, c * S:(c + 1) * S], k[0, kap * S]) / math.sqrt(d)
                np.testing.assert_allclose(lse[0, c * S:(c + 1) * S, :, j], a + math.log(S), rtol=1e-13)
        np.testing.assert_allclose(o[0, c * S:(c + 1) * S], np.broadcast_to(want, (S, H, d)), atol=1e-13)


def test_empty_slots_and_chunks():
    B, nC, S, H, d = 1, 5, 4, 2, 3
    q, k, v, idx, r, w = make_case(6, B, nC, S, H, d, 4, include_self=False)
    o, lse = oracle.fwd(q, k, v, idx, w, S)
    # chunks 0 and 1 have no candidates under the strict causal set
    assert (o[0, :2 * S] == 0).all()
    assert np.isneginf(lse[0, :2 * S]).all()
    # chunk 3 has two candidates (0, 1): slots 2, 3 are empty
    assert list(idx[0, 3]) [2:] == [-1, -1]
    assert np.isneginf(lse[0, 3 * S:4 * S, :, 2:]).all()
    assert np.isfinite(lse[0, 3 * S:4 * S, :, :2]).all()


def test_qmask_subset_equals_full():
    q, k, v, idx, r, w = make_case(8, 2, 6, 4, 2, 3, 3)
    o, lse = oracle.fwd(q, k, v, idx, w, 4)
    mask = np.zeros((2, 6), dtype=bool)
    mask[0, 3] = mask[1, 5] = True
    om, lm = oracle.fwd(q, k, v, idx, w, 4, qmask=mask)
    np.testing.assert_array_equal(om[0, 12:16], o[0, 12:16])
    np.testing.assert_array_equal(om[1, 20:24], o[1, 20:24])
    assert (om[0, :12] == 0).all()


def test_decode_shape_fwd():
    # Decode: one query chunk over a pool of chunks (idx rows index the pool).
    rng = np.random.default_rng(9)
    S, H, d, nP = 4, 2, 3, 10
    q = rng.normal(size=(1, S, H, d))
    k = rng.normal(size=(1, nP * S, H, d))
    v = rng.normal(size=(1, nP * S, H, d))
    idx = np.array([[[7, 2, 9]]], dtype=np.int32)
    w = np.array([[[0.5, 0.3, 0.2]]])
    o, lse = oracle.fwd(q, k, v, idx, w, S)
    bo, blse, _ = brute_fwd(q, k, v, idx, w, S, 1.0 / math.sqrt(d))
    np.testing.assert_allclose(o, bo, rtol=1e-12)
