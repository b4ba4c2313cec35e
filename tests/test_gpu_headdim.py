"""GPU parity of the tensor-core path at head dimensions 32 and 128 (bf16),
forward and backward.

The workloads' model uses 64-dimensional heads; these cases keep the 64K
sweep's recipe (integer landmarks in [-4, 4], Q/K/V ~ N(0, 1/d) rounded to
bf16, dO ~ N(0, 1)) and change the head dimension, at both chunk sizes and
several ragged lengths, every element against the fp64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from retrieval_sparse_attention_gb300 import inputs

from gpu_helpers import assert_close, assert_lse, f64, tol_for
from test_gpu_attention import gpu_pipeline

pytestmark = pytest.mark.gpu


def workload(S, d, k, H):
    base = inputs.WORKLOADS["long64k_S%d_k8" % S]
    return dataclasses.replace(base, name="d%d_S%d_k%d" % (d, S, k), d=d, H=H, topk=k,
                               qkv_std=float(d) ** -0.5)


FWD = [(64, 32, 8, 12, 1, 2048, False, False), (64, 32, 4, 6, 2, 1472, True, True),
       (64, 128, 8, 12, 1, 2048, False, False), (64, 128, 16, 4, 2, 1344, True, True),
       (128, 32, 8, 12, 1, 3072, False, False), (128, 32, 4, 5, 1, 1920, True, False),
       (128, 128, 8, 12, 1, 3072, False, False), (128, 128, 16, 3, 2, 2176, False, True)]


@pytest.mark.parametrize("S,d,k,H,B,L,off_by_one,include_self", FWD)
def test_fwd_head_dims_every_element(S, d, k, H, B, L, off_by_one, include_self):
    wl = workload(S, d, k, H)
    x = inputs.make(wl, B=B, L=L)
    got = gpu_pipeline(x, wl, off_by_one, include_self, backward=False)
    lm, q, kk, v = (f64(x[n]) for n in ("lm", "q", "k", "v"))
    oi, orr, ow = oracle.score_topk(lm, wl.topk, include_self, off_by_one)
    np.testing.assert_array_equal(got["idx"].cpu().numpy(), oi)
    atol, rtol = tol_for(x["q"].dtype)
    oo, olse = oracle.fwd(q, kk, v, oi, ow, wl.S)
    assert_close("o", f64(got["o"]), oo, atol, rtol)
    assert_lse(f64(got["lse"]), olse, 1e-3)


BWD = [(64, 32, 8, 12, 1, 2048, False, False), (64, 32, 16, 4, 2, 1600, False, True),
       (64, 128, 8, 12, 1, 2048, False, False), (64, 128, 4, 6, 2, 1472, True, False),
       (128, 32, 8, 12, 1, 3072, False, False), (128, 32, 16, 5, 1, 2304, True, True),
       (128, 128, 8, 12, 1, 3072, False, False), (128, 128, 4, 3, 2, 1664, False, True)]


@pytest.mark.parametrize("S,d,k,H,B,L,off_by_one,include_self", BWD)
def test_fwd_bwd_head_dims_every_element(S, d, k, H, B, L, off_by_one, include_self):
    wl = workload(S, d, k, H)
    x = inputs.make(wl, B=B, L=L)
    got = gpu_pipeline(x, wl, off_by_one, include_self)
    lm, q, kk, v, g = (f64(x[n]) for n in ("lm", "q", "k", "v", "dout"))
    oi, orr, ow = oracle.score_topk(lm, wl.topk, include_self, off_by_one)
    np.testing.assert_array_equal(got["idx"].cpu().numpy(), oi)
    atol, rtol = tol_for(x["q"].dtype)
    oo, olse = oracle.fwd(q, kk, v, oi, ow, wl.S)
    assert_close("o", f64(got["o"]), oo, atol, rtol)
    dq, dk, dv, ds = oracle.bwd(q, kk, v, oi, ow, g, wl.S)
    assert_close("dq", f64(got["dq"]), dq, atol, rtol)
    assert_close("dk", f64(got["dk"]), dk, atol, rtol)
    assert_close("dv", f64(got["dv"]), dv, atol, rtol)
    assert_close("dscore", f64(got["ds"]), ds, atol, rtol)


@pytest.mark.parametrize("S,d", [(64, 32), (64, 128), (128, 32), (128, 128)])
def test_bwd_head_dims_deterministic(S, d):
    wl = workload(S, d, 8, 12)
    x = inputs.make(wl, B=1, L=32 * S)
    a = gpu_pipeline(x, wl, False, False)
    b = gpu_pipeline(x, wl, False, False)
    for n in ("o", "lse", "dq", "dk", "dv", "ds"):
        assert torch.equal(a[n], b[n]), n
