"""Pins of the sliding-window self-attention oracle (the 512-token window that
a DRT layer runs before its GCA module; paper summary sections 1 and 4.1.2).
Reading: token t attends to keys max(0, t - W + 1) .. t.  The oracle is
checked against PyTorch's scaled_dot_product_attention with an explicit
window mask, closed forms (W = 1), the causal special case, a probability
invariant, central finite differences and fp64 autograd."""
import numpy as np
import pytest
import torch

import oracle


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def sdpa(q, k, v, W, scale):
    """Library routine: torch SDPA on [B, H, L, d] with a boolean window mask."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))) for x in (q, k, v))
    L = q.shape[1]
    t = torch.arange(L)
    mask = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - W)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    return o.numpy().transpose(0, 2, 1, 3)


@pytest.mark.parametrize("B,L,H,d,W", [(2, 37, 3, 8, 5), (1, 64, 2, 16, 16), (1, 50, 1, 4, 64)])
def test_matches_sdpa_with_window_mask(B, L, H, d, W):
    q, k, v = rnd((B, L, H, d), 1), rnd((B, L, H, d), 2), rnd((B, L, H, d), 3)
    scale = 1.0 / np.sqrt(d)
    o, lse = oracle.swa_fwd(q, k, v, W)
    np.testing.assert_allclose(o, sdpa(q, k, v, W, scale), rtol=1e-12, atol=1e-12)


def test_window_covering_the_sequence_is_causal_attention():
    q, k, v = rnd((1, 30, 2, 8), 4), rnd((1, 30, 2, 8), 5), rnd((1, 30, 2, 8), 6)
    o, _ = oracle.swa_fwd(q, k, v, 30)
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True).numpy()
    np.testing.assert_allclose(o, ref.transpose(0, 2, 1, 3), rtol=1e-12, atol=1e-12)
    o2, _ = oracle.swa_fwd(q, k, v, 1000)
    np.testing.assert_array_equal(o, o2)


def test_window_of_one_returns_v():
    q, k, v = rnd((2, 9, 2, 4), 7), rnd((2, 9, 2, 4), 8), rnd((2, 9, 2, 4), 9)
    o, lse = oracle.swa_fwd(q, k, v, 1, attn_scale=0.3)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, 0.3 * np.einsum("blhe,blhe->blh", q, k), rtol=1e-13)
    dq, dk, dv = oracle.swa_bwd(q, k, v, rnd((2, 9, 2, 4), 10), 1)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


def test_lse_normalises_the_window_and_early_rows_are_causal():
    q, k, v = rnd((1, 40, 2, 8), 11), rnd((1, 40, 2, 8), 12), rnd((1, 40, 2, 8), 13)
    W = 7
    o, lse = oracle.swa_fwd(q, k, v, W)
    a = np.einsum("bthe,bshe->bhts", q, k) / np.sqrt(8)
    for t in range(40):
        s0 = max(0, t - W + 1)
        tot = np.exp(a[0, :, t, s0:t + 1] - lse[0, t, :, None]).sum(-1)
        np.testing.assert_allclose(tot, 1.0, rtol=1e-12)
    oc, lc = oracle.swa_fwd(q, k, v, 40)
    np.testing.assert_allclose(o[:, :W], oc[:, :W], rtol=1e-13, atol=1e-15)
    assert not np.allclose(o[:, W:], oc[:, W:])


def test_gradients_match_finite_differences():
    B, L, H, d, W = 1, 11, 2, 3, 4
    q, k, v, g = (rnd((B, L, H, d), s) for s in (20, 21, 22, 23))
    dq, dk, dv = oracle.swa_bwd(q, k, v, g, W)
    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[i] += h
            xm[i] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fp = (oracle.swa_fwd(args_p["q"], args_p["k"], args_p["v"], W)[0] * g).sum()
            fm = (oracle.swa_fwd(args_m["q"], args_m["k"], args_m["v"], W)[0] * g).sum()
            num[i] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8, err_msg=name)


def test_gradients_match_autograd_through_sdpa():
    B, L, H, d, W = 2, 45, 3, 8, 9
    q, k, v, g = (rnd((B, L, H, d), s) for s in (30, 31, 32, 33))
    dq, dk, dv = oracle.swa_bwd(q, k, v, g, W)
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))).requires_grad_()
                  for x in (q, k, v))
    t = torch.arange(L)
    mask = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - W)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    (o * torch.from_numpy(np.ascontiguousarray(g.transpose(0, 2, 1, 3)))).sum().backward()
    for got, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(got, ref.numpy().transpose(0, 2, 1, 3), rtol=1e-10, atol=1e-12)
