"""GPU parity of the rows beyond the core path: the Gumbel-perturbed top-k
(section 3.2) and the landmark gradients (sections 1 and 3), against the fp64
oracle.  Noise and upstream gradients are seeded inputs fed to both sides."""
import numpy as np
import pytest
import torch

import oracle
from retrieval_sparse_attention_gb300 import api, inputs

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_fp32", "gpt2s_fwd_b4", "long64k_S128_k8"])
@pytest.mark.parametrize("include_self", [False, True])
def test_noisy_topk(name, include_self):
    wl = inputs.WORKLOADS[name]
    lm = inputs.make(wl, with_dout=False)["lm"]
    B, nC = lm.shape[0], lm.shape[1]
    g = torch.Generator().manual_seed(123)
    u = torch.rand(B, nC, nC, generator=g, dtype=torch.float64).clamp_(1e-12, 1 - 1e-12)
    noise = (-torch.log(-torch.log(u))).to(torch.float32)          # Gumbel(0, 1)
    idx, r, w = api.score_topk_noisy(lm.cuda(), noise.cuda(), S=wl.S, H=wl.H, d=wl.d, topk=wl.topk,
                                     off_by_one=wl.off_by_one, include_self=include_self)
    torch.cuda.synchronize()
    oi, orr, ow = oracle.score_topk_noisy(f64(lm), noise.numpy(), wl.topk, include_self, wl.off_by_one)
    np.testing.assert_array_equal(idx.cpu().numpy(), oi)
    assert_close("score", f64(r), orr, 1e-5, 1e-6)
    assert_close("weight", f64(w), ow, 1e-6, 1e-5)
    # the noise must actually change some selections
    pi, _, _ = oracle.score_topk(f64(lm), wl.topk, include_self, wl.off_by_one)
    assert (pi != oi).any()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(1, 16, 128, 2), (2, 64, 768, 8), (1, 300, 96, 16), (1, 40, 100, 4)])
def test_landmark_grad_seeded_dscore(dtype, shape):
    B, nC, D, k = shape
    gen = torch.Generator().manual_seed(nC)
    lm = torch.randint(-4, 5, (B, nC, D), generator=gen).to(dtype)
    idx, _, _ = oracle.score_topk(f64(lm), k)
    dr = torch.randn(B, nC, k, generator=gen, dtype=torch.float64) * torch.from_numpy(idx >= 0)
    got = api.landmark_bwd(lm.cuda(), torch.from_numpy(idx).cuda(), dr.float().cuda(), S=64, H=1, d=D)
    torch.cuda.synchronize()
    want = oracle.landmark_bwd(f64(lm), idx, dr.float().double().numpy())
    if dtype == torch.float32:
        assert_close("dlandmarks", f64(got), want, 1e-4, 1e-5)
    else:
        assert_close("dlandmarks", f64(got), want, 2e-2, 2e-2)


def test_landmark_grad_long_inverse_list():
    # chunk 0 outscores every other landmark, so every query chunk that may retrieve it
    # does: its list of terms is longer than one staging pass of the kernel (1024 terms)
    B, nC, D, k = 1, 1100, 64, 4
    gen = torch.Generator().manual_seed(5)
    lm = torch.randint(0, 3, (B, nC, D), generator=gen).to(torch.float32)
    lm[:, 0, :] = 8
    idx, _, _ = oracle.score_topk(f64(lm), k)
    assert (idx == 0).sum() > 1024
    dr = torch.randn(B, nC, k, generator=gen, dtype=torch.float64) * torch.from_numpy(idx >= 0)
    got = api.landmark_bwd(lm.cuda(), torch.from_numpy(idx).cuda(), dr.float().cuda(), S=64, H=1, d=D)
    torch.cuda.synchronize()
    want = oracle.landmark_bwd(f64(lm), idx, dr.float().double().numpy())
    assert_close("dlandmarks", f64(got), want, 1e-4, 1e-5)


def test_landmark_grad_after_backward_pipeline():
    # the full training chain: scores -> forward -> backward -> landmark gradient
    wl = inputs.WORKLOADS["gpt2s_fwdbwd_b8"]
    x = inputs.make(wl, B=1, L=2048)
    dev = "cuda"
    lm, q, k, v, g = (x[n].to(dev) for n in ("lm", "q", "k", "v", "dout"))
    idx, r, w = api.score_topk(lm, S=wl.S, H=wl.H, d=wl.d, topk=wl.topk)
    o, lse = api.fwd(q, k, v, idx, w, S=wl.S)
    _, _, _, ds = api.bwd(q, k, v, idx, w, lse, g, S=wl.S)
    dl = api.landmark_bwd(lm, idx, ds, S=wl.S, H=wl.H, d=wl.d)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    oi, orr, ow = oracle.score_topk(f64(x["lm"]), wl.topk)
    _, _, _, ods = oracle.bwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), oi, ow, f64(x["dout"]), wl.S)
    want = oracle.landmark_bwd(f64(x["lm"]), oi, ods)
    assert_close("dscore", f64(ds), ods, 2e-2, 2e-2)
    # the landmark kernel itself, fed the GPU's own d(score): fp32 accumulation,
    # then one rounding to bf16 (relative error at most 2^-9)
    assert_close("dlandmarks | gpu dscore", f64(dl), oracle.landmark_bwd(f64(x["lm"]), oi, f64(ds)),
                 1e-4, 4e-3)
    # and the whole chain against the oracle, at the bf16 bound
    assert_close("dlandmarks", f64(dl), want, 2e-2, 2e-2)
