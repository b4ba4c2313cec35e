"""GPU parity of the sliding-window self-attention (gca_swa_fwd) against the
fp64 oracle: element by element on small problems that span several query and
key tiles with ragged tails, on windows below, at and above the 128-token
tile, on inputs that force the kernel's rescaling of its running maximum, and
on sampled rows of the full-size workload (B=8, L=16384, H=12, W=512)."""
import numpy as np
import pytest
import torch

import oracle
from retrieval_sparse_attention_gb300 import api
from retrieval_sparse_attention_gb300._lib import GcaError

from gpu_helpers import BF16_ATOL, BF16_RTOL, assert_close, f64

pytestmark = pytest.mark.gpu


def qkv(B, L, H, d, seed, std=0.125):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn(B, L, H, d, generator=g) * std).to(torch.bfloat16) for _ in range(3)]


def check(q, k, v, W):
    o, lse = api.swa_fwd(q.cuda(), k.cuda(), v.cuda(), window=W)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    oo, ol = oracle.swa_fwd(f64(q), f64(k), f64(v), W)
    assert_close("o", f64(o), oo, BF16_ATOL, BF16_RTOL)
    assert_close("lse", f64(lse), ol, 1e-3, 0.0)
    return o, lse


@pytest.mark.parametrize("B,L,H,W", [(2, 384, 2, 512), (1, 1000, 3, 200), (2, 640, 2, 64),
                                     (1, 256, 1, 1), (1, 517, 2, 128), (1, 700, 2, 129),
                                     (1, 1536, 4, 512), (3, 100, 1, 5000)])
def test_every_element(B, L, H, W):
    q, k, v = qkv(B, L, H, 64, seed=B * 1000 + L + W)
    check(q, k, v, W)


def test_running_max_rescales():
    # score(t, s) ~ s / 16: each 128-key tile raises the row maximum by ~8 nats
    # (11.5 in log2 units), past the kernel's rescaling threshold of 2^8
    B, L, H, d, W = 1, 768, 2, 64, 512
    g = torch.Generator().manual_seed(7)
    q = torch.full((B, L, H, d), 0.5)
    pos = torch.arange(L, dtype=torch.float32).view(1, L, 1, 1)
    k = pos / 64.0 * torch.ones(B, L, H, d) + 0.01 * torch.randn(B, L, H, d, generator=g)
    v = torch.randn(B, L, H, d, generator=g) * 0.125
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    s = (f64(q)[0, -1, 0] * f64(k)[0, :, 0]).sum(-1) / 8.0
    assert s[-1] - s[-129] > 5.6                      # the premise: growth per tile > 8 log2 units
    check(q, k, v, W)


def test_full_size_sampled_rows():
    B, L, H, d, W = 8, 16384, 12, 64, 512
    q, k, v = qkv(B, L, H, d, seed=11)
    o, lse = api.swa_fwd(q.cuda(), k.cuda(), v.cuda(), window=W)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    o, lse = f64(o), f64(lse)
    rng = np.random.default_rng(3)
    picks = [(b, t) for b, t in zip(rng.integers(0, B, 24), rng.integers(0, L, 24))]
    picks += [(0, 0), (7, L - 1), (3, 511), (3, 512), (5, 127), (5, 128)]
    for b, t in picks:
        # token t's output depends only on the window ending at t: run the
        # oracle on that slice and take its last row
        s0 = max(0, t - W + 1)
        oo, ol = oracle.swa_fwd(f64(q[b:b + 1, s0:t + 1]), f64(k[b:b + 1, s0:t + 1]),
                                f64(v[b:b + 1, s0:t + 1]), W)
        assert_close("o[%d,%d]" % (b, t), o[b, t], oo[0, -1], BF16_ATOL, BF16_RTOL)
        assert_close("lse[%d,%d]" % (b, t), lse[b, t], ol[0, -1], 1e-3, 0.0)


def test_deterministic():
    q, k, v = (x.cuda() for x in qkv(2, 1024, 3, 64, seed=5))
    a = api.swa_fwd(q, k, v, window=512)
    b = api.swa_fwd(q, k, v, window=512)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_unsupported_and_invalid():
    q, k, v = (x.cuda() for x in qkv(1, 128, 1, 64, seed=1))
    with pytest.raises(GcaError) as e:
        api.swa_fwd(q.float(), k.float(), v.float(), window=64)
    assert e.value.code == 2
    q32 = torch.zeros(1, 128, 1, 32, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(GcaError) as e:
        api.swa_fwd(q32, q32, q32, window=64)
    assert e.value.code == 2
    with pytest.raises(GcaError) as e:
        api.swa_fwd(q, k, v, window=0)
    assert e.value.code == 1


def check_bwd(q, k, v, g, W):
    qc, kc, vc, gc = (x.cuda() for x in (q, k, v, g))
    o, lse = api.swa_fwd(qc, kc, vc, window=W)
    dq, dk, dv = api.swa_bwd(qc, kc, vc, o, lse, gc, window=W)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    rq, rk, rv = oracle.swa_bwd(f64(q), f64(k), f64(v), f64(g), W)
    assert_close("dq", f64(dq), rq, BF16_ATOL, BF16_RTOL)
    assert_close("dk", f64(dk), rk, BF16_ATOL, BF16_RTOL)
    assert_close("dv", f64(dv), rv, BF16_ATOL, BF16_RTOL)
    return dq, dk, dv


def dout_like(q, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(q.shape, generator=g).to(torch.bfloat16)


# (1, 3000, 1, 1000): a window so wide that consecutive query tiles cannot keep
# their shared key tiles resident, so every tile loads its whole window
@pytest.mark.parametrize("B,L,H,W", [(2, 384, 2, 512), (1, 1000, 3, 200), (2, 640, 2, 64),
                                     (1, 256, 1, 1), (1, 517, 2, 128), (1, 700, 2, 129),
                                     (1, 1536, 4, 512), (3, 100, 1, 5000), (1, 3000, 1, 1000),
                                     (2, 2304, 3, 512)])
def test_bwd_every_element(B, L, H, W):
    q, k, v = qkv(B, L, H, 64, seed=B * 1000 + L + W)
    check_bwd(q, k, v, dout_like(q, 99), W)


def test_bwd_full_size_sampled():
    # dq of token t and dk/dv of key s depend only on the W-token neighbourhood:
    # run the oracle on a slice that contains it and compare the row
    B, L, H, d, W = 8, 16384, 12, 64, 512
    q, k, v = qkv(B, L, H, d, seed=11)
    g = dout_like(q, 12)
    qc, kc, vc, gc = (x.cuda() for x in (q, k, v, g))
    o, lse = api.swa_fwd(qc, kc, vc, window=W)
    dq, dk, dv = api.swa_bwd(qc, kc, vc, o, lse, gc, window=W)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    dq, dk, dv = f64(dq), f64(dk), f64(dv)
    rng = np.random.default_rng(4)
    picks = [(int(b), int(t)) for b, t in zip(rng.integers(0, B, 10), rng.integers(0, L, 10))]
    picks += [(0, 0), (7, L - 1), (2, 511), (2, 512), (6, L - 512)]
    for b, t in picks:
        # dq_t needs tokens t-W+1 .. t; dk_t and dv_t need the queries t .. t+W-1
        # and their windows: tokens t-W+1 .. t+W-1 (one more window of margin)
        lo, s1 = max(0, t - 2 * W + 2), min(L, t + W)
        sl = slice(lo, s1)
        rq, rk, rv = oracle.swa_bwd(f64(q[b:b + 1, sl]), f64(k[b:b + 1, sl]), f64(v[b:b + 1, sl]),
                                    f64(g[b:b + 1, sl]), W)
        i = t - lo
        assert_close("dq[%d,%d]" % (b, t), dq[b, t], rq[0, i], BF16_ATOL, BF16_RTOL)
        assert_close("dk[%d,%d]" % (b, t), dk[b, t], rk[0, i], BF16_ATOL, BF16_RTOL)
        assert_close("dv[%d,%d]" % (b, t), dv[b, t], rv[0, i], BF16_ATOL, BF16_RTOL)


def test_bwd_deterministic():
    q, k, v = (x.cuda() for x in qkv(2, 1024, 3, 64, seed=5))
    g = dout_like(q, 6).cuda()
    o, lse = api.swa_fwd(q, k, v, window=512)
    a = api.swa_bwd(q, k, v, o, lse, g, window=512)
    b = api.swa_bwd(q, k, v, o, lse, g, window=512)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
