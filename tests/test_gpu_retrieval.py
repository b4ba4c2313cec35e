"""GPU parity of the retrieval steps against the fp64 oracle: causal scoring +
top-k + softmax (gca_score_topk) and decode-time retrieval
(gca_decode_retrieve).  Indices are compared bit-exactly and in order; the
scores and weights within fp32 rounding."""
import numpy as np
import pytest
import torch

import oracle
from retrieval_sparse_attention_gb300 import api, inputs

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu


def run_score(lm_cpu, S, H, d, topk, off_by_one, include_self):
    lm = lm_cpu.cuda()
    idx, r, w = api.score_topk(lm, S=S, H=H, d=d, topk=topk, off_by_one=off_by_one,
                               include_self=include_self)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    oi, orr, ow = oracle.score_topk(f64(lm_cpu), topk, include_self, off_by_one)
    np.testing.assert_array_equal(idx.cpu().numpy(), oi)
    assert_close("score", f64(r), orr, 1e-5, 1e-6)
    assert_close("weight", f64(w), ow, 1e-6, 1e-5)
    return oi, ow


@pytest.mark.parametrize("name", ["tiny_fp32", "gpt2s_fwd_b4", "gpt2s_fwdbwd_b8",
                                  "long64k_S64_k16", "long64k_S128_k4"])
@pytest.mark.parametrize("include_self", [False, True])
@pytest.mark.parametrize("off_by_one", [False, True])
def test_score_topk_workloads(name, include_self, off_by_one):
    wl = inputs.WORKLOADS[name]
    lm = inputs.make(wl, with_dout=False)["lm"]
    run_score(lm, wl.S, wl.H, wl.d, wl.topk, off_by_one, include_self)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(3, 37, 8, 5), (1, 2, 16, 4), (2, 70, 24, 32), (1, 600, 16, 1)])
def test_score_topk_ties_and_ragged(dtype, shape):
    B, nC, D, k = shape
    g = torch.Generator().manual_seed(nC)
    lm = torch.randint(-1, 2, (B, nC, D), generator=g).to(dtype)   # values in {-1,0,1}: many ties
    run_score(lm, 64, 1, D, k, False, False)
    run_score(lm, 64, 1, D, k, True, True)


def test_score_topk_all_equal():
    # every score ties: slots must be chunks 0, 1, 2, ... in order
    lm = torch.ones(1, 20, 16, dtype=torch.bfloat16)
    oi, ow = run_score(lm, 64, 1, 16, 4, False, False)
    assert list(oi[0, 19]) == [0, 1, 2, 3]
    assert np.allclose(ow[0, 19], 0.25)


# ---------------------------------------------------------------------------------------
def run_decode(lm_cpu, ql_cpu, topk, off_by_one):
    idx, r, w = api.decode_retrieve(lm_cpu.cuda(), ql_cpu.cuda(), topk=topk, off_by_one=off_by_one)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    oi, orr, ow = oracle.decode_retrieve(f64(lm_cpu), f64(ql_cpu), topk, off_by_one)
    np.testing.assert_array_equal(idx.cpu().numpy(), oi)
    assert_close("score", f64(r), orr, 1e-5, 1e-6)
    assert_close("weight", f64(w), ow, 1e-6, 1e-5)
    return idx


@pytest.mark.parametrize("N,D,k", [(1, 8, 4), (7, 16, 8), (1000, 768, 8), (4099, 64, 16),
                                   (65536, 768, 32), (300000, 8, 1)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("off_by_one", [False, True])
def test_decode_small(N, D, k, dtype, off_by_one):
    g = torch.Generator().manual_seed(N + D)
    lm = torch.randint(-2, 3, (N, D), generator=g).to(dtype)
    ql = torch.randint(-2, 3, (D,), generator=g).to(dtype)
    run_decode(lm, ql, k, off_by_one)


def test_decode_full_16m_context():
    x = inputs.decode_inputs()
    p = inputs.DECODE
    for _ in range(2):              # a second call reuses the workspace (ticket reset)
        run_decode(x["lm"], x["ql"], p["topk"], p["off_by_one"])


def test_decode_ties_across_blocks():
    # identical rows everywhere: the top-k must be rows 0..k-1, across CTA boundaries
    lm = torch.ones(100000, 32, dtype=torch.bfloat16)
    lm[77777] = 2
    idx = run_decode(lm, torch.ones(32, dtype=torch.bfloat16), 8, False)
    assert idx.cpu().tolist() == [77777, 0, 1, 2, 3, 4, 5, 6]


def test_decode_all_equal_full_table():
    # every score ties at full size: the bound filter keeps every CTA's whole
    # list, and the top-k must still be rows 0..k-1 in order
    lm = torch.ones(262144, 8, dtype=torch.bfloat16)
    idx = run_decode(lm, torch.ones(8, dtype=torch.bfloat16), 32, False)
    assert idx.cpu().tolist() == list(range(32))


def test_synth_fill_matches_host_generator():
    S, H, d = 64, 12, 64
    n = 5 * S * H * d
    buf = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    api.gca_synth_fill_hash(buf, 4, 1, first_elem=3 * S * H * d)
    torch.cuda.synchronize()
    got = f64(buf).reshape(5, S, H, d)
    for i in range(5):
        want = inputs.decode_cache_chunk_np(4, 1, 3 + i, S, H, d)
        np.testing.assert_array_equal(got[i], want)


def test_signed_zero_scores_tie_toward_lower_index():
    # all scores are zero, some from negative zeros: -0 and +0 are one score,
    # so the slots go to the lowest indices in order (scoring and decode)
    lm = torch.zeros(1, 40, 16)
    lm[0, 1::2] = -0.0
    lm[0, 6, 3] = 2.0                 # orthogonal to every other landmark
    oi, ow = run_score(lm, 64, 1, 16, 8, False, False)
    assert list(oi[0, 39]) == list(range(8))
    tab = torch.zeros(70000, 16)
    tab[1::3] = -0.0
    tab[5, 0] = 1.0
    q = torch.zeros(16)
    q[1:] = -0.0
    idx = run_decode(tab, q, 8, False)
    assert idx.cpu().tolist() == list(range(8))


@pytest.mark.parametrize("B,nC,D,k", [(16, 200, 64, 8), (8, 256, 768, 16), (4, 520, 128, 5)])
@pytest.mark.parametrize("include_self", [False, True])
@pytest.mark.parametrize("off_by_one", [False, True])
def test_score_topk_tensor_core_path(B, nC, D, k, include_self, off_by_one):
    # shapes with at least 16 row tiles of 128 landmarks (bf16, D a multiple of 64,
    # k <= 16) take the tensor-core scorer; values in {-1, 0, 1} make many ties
    g = torch.Generator().manual_seed(B * nC + D)
    lm = torch.randint(-1, 2, (B, nC, D), generator=g).to(torch.bfloat16)
    run_score(lm, 64, 1, D, k, off_by_one, include_self)


@pytest.mark.parametrize("include_self", [False, True])
def test_noisy_topk_tensor_core_path(include_self):
    B, nC, D, k = 16, 256, 128, 8
    g = torch.Generator().manual_seed(7)
    lm = torch.randint(-2, 3, (B, nC, D), generator=g).to(torch.bfloat16)
    u = torch.rand(B, nC, nC, generator=g, dtype=torch.float64).clamp_(1e-12, 1 - 1e-12)
    noise = (-torch.log(-torch.log(u))).to(torch.float32)
    idx, r, w = api.score_topk_noisy(lm.cuda(), noise.cuda(), S=64, H=1, d=D, topk=k,
                                     include_self=include_self)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    oi, orr, ow = oracle.score_topk_noisy(f64(lm), noise.numpy(), k, include_self, False)
    np.testing.assert_array_equal(idx.cpu().numpy(), oi)
    assert_close("score", f64(r), orr, 1e-5, 1e-6)
    assert_close("weight", f64(w), ow, 1e-6, 1e-5)
