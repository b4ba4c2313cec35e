"""Pins for the oracle's GCA backward (App. B backward: gradients for Q, K, V
and the weights; section 3 and the official README: the relevance scores get
gradients from the next-token loss through the fusion weights).

Checked against central finite differences of the oracle's own forward (a
different computation from the hand-written chain rule), against PyTorch
autograd through an independent fp64 PyTorch forward, and against the
softmax-Jacobian invariant sum_j dr_j = 0 for the vanilla softmax.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def make_case(seed, B, nC, S, H, d, k, include_self=True, off_by_one=False):
    rng = np.random.default_rng(seed)
    lm = rng.integers(-3, 4, size=(B, nC, 2 * H + 1)).astype(np.float64)
    idx, r, w = oracle.score_topk(lm, k, include_self, off_by_one)
    q = rng.normal(size=(B, nC * S, H, d))
    kk = rng.normal(size=(B, nC * S, H, d))
    v = rng.normal(size=(B, nC * S, H, d))
    g = rng.normal(size=(B, nC * S, H, d))
    return q, kk, v, idx, r, w, g


def weights_of(idx, r, off_by_one):
    w = np.zeros_like(r)
    B, nQ, k = r.shape
    for b in range(B):
        for c in range(nQ):
            m = int((idx[b, c] >= 0).sum())
            if m:
                w[b, c, :m] = oracle.weights_from_scores(r[b, c, :m], off_by_one)
    return w


@pytest.mark.parametrize("off_by_one", [False, True])
def test_grads_match_finite_differences(off_by_one):
    S = 3
    q, k, v, idx, r, w, g = make_case(3, 1, 5, S, 2, 2, 2, off_by_one=off_by_one)
    dq, dk, dv, ds = oracle.bwd(q, k, v, idx, w, g, S)

    def loss(q_, k_, v_, r_):
        o, _ = oracle.fwd(q_, k_, v_, idx, weights_of(idx, r_, off_by_one), S)
        return float((o * g).sum())

    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp = x.copy(); xp[i] += h
            xm = x.copy(); xm[i] -= h
            args_p = [q, k, v, r]
            args_m = [q, k, v, r]
            pos = "qkv".index(name)
            args_p[pos], args_m[pos] = xp, xm
            fd[i] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=name)
    fd = np.zeros_like(r)
    for i in np.ndindex(*r.shape):
        if idx[i] < 0:
            continue
        rp = r.copy(); rp[i] += h
        rm = r.copy(); rm[i] -= h
        fd[i] = (loss(q, k, v, rp) - loss(q, k, v, rm)) / (2 * h)
    np.testing.assert_allclose(ds, fd, rtol=1e-6, atol=1e-8, err_msg="dscore")
    assert (ds[idx < 0] == 0).all()


def torch_gca(q, k, v, idx, r, S, off_by_one):
    """Independent fp64 PyTorch forward used only for autograd."""
    B, L, H, d = q.shape
    nQ, topk = idx.shape[1], idx.shape[2]
    outs = []
    for b in range(B):
        rows = []
        for c in range(nQ):
            valid = [j for j in range(topk) if idx[b, c, j] >= 0]
            Qc = q[b, c * S:(c + 1) * S].transpose(0, 1)            # [H, S, d]
            if not valid:
                rows.append(torch.zeros_like(q[b, c * S:(c + 1) * S]))
                continue
            rv = r[b, c, valid]
            if off_by_one:
                wv = torch.exp(rv) / (1 + torch.exp(rv).sum())
            else:
                wv = torch.softmax(rv, 0)
            acc = 0
            for n, j in enumerate(valid):
                kap = int(idx[b, c, j])
                K = k[b, kap * S:(kap + 1) * S].transpose(0, 1)
                V = v[b, kap * S:(kap + 1) * S].transpose(0, 1)
                P = torch.softmax(Qc @ K.transpose(1, 2) / math.sqrt(d), -1)
                acc = acc + wv[n] * (P @ V)
            rows.append(acc.transpose(0, 1))
        outs.append(torch.cat(rows, 0))
    return torch.stack(outs, 0)


@pytest.mark.parametrize("off_by_one", [False, True])
def test_grads_match_autograd(off_by_one):
    S = 8
    q, k, v, idx, r, w, g = make_case(5, 2, 7, S, 2, 4, 3, include_self=False, off_by_one=off_by_one)
    dq, dk, dv, ds = oracle.bwd(q, k, v, idx, w, g, S)
    tq, tk, tv, tr = (torch.tensor(x, requires_grad=True) for x in (q, k, v, r))
    o = torch_gca(tq, tk, tv, idx, tr, S, off_by_one)
    (o * torch.from_numpy(g)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ds, tr.grad.numpy(), rtol=1e-10, atol=1e-12)
    # chunks nobody retrieved get exactly zero dK / dV
    retrieved = set(int(x) for x in idx[idx >= 0].ravel())
    for kap in range(7):
        if all(int(x) != kap for x in idx[0].ravel()):
            assert (dk[0, kap * S:(kap + 1) * S] == 0).all()


def test_vanilla_score_grads_sum_to_zero():
    q, k, v, idx, r, w, g = make_case(6, 2, 9, 4, 3, 3, 4)
    _, _, _, ds = oracle.bwd(q, k, v, idx, w, g, 4)
    np.testing.assert_allclose(ds.sum(-1), 0.0, atol=1e-12)


def test_masked_bwd_equals_full():
    S = 4
    q, k, v, idx, r, w, g = make_case(7, 2, 6, S, 2, 3, 3)
    full = oracle.bwd(q, k, v, idx, w, g, S)
    qm = np.zeros((2, 6), bool); qm[1, 4] = True
    km = np.zeros((2, 6), bool); km[0, 2] = True; km[1, 0] = True
    part = oracle.bwd(q, k, v, idx, w, g, S, qmask=qm, kmask=km)
    np.testing.assert_array_equal(part[0][1, 16:20], full[0][1, 16:20])
    np.testing.assert_array_equal(part[3][1, 4], full[3][1, 4])
    np.testing.assert_array_equal(part[1][0, 8:12], full[1][0, 8:12])
    np.testing.assert_array_equal(part[2][1, 0:4], full[2][1, 0:4])
    assert (part[0][0] == 0).all()
