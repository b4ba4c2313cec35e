"""The allocation-free decode entry point (gca_decode_retrieve_noalloc).

Some callers are handed only input and output buffers and may not allocate
device memory themselves (engine plugins, runtimes that plan all device memory
up front, latency-critical loops).  For them the library offers a decode
retrieval that uses a fixed device array inside the library instead of a
caller-provided workspace.  This test checks, through the C ABI, that it
returns what the workspace entry point returns, on consecutive calls that
reuse the shared array, and that requests larger than the array are refused.
It lives in a file of its own that pytest collects last.
"""
import numpy as np
import pytest
import torch

from retrieval_sparse_attention_gb300 import api, inputs
from retrieval_sparse_attention_gb300._lib import GcaError

pytestmark = pytest.mark.gpu


def noalloc(lm, ql, topk, off_by_one):
    N, D = lm.shape
    idx = torch.full((topk,), -7, dtype=torch.int32, device=lm.device)
    r = torch.full((topk,), float("nan"), device=lm.device)
    w = torch.full((topk,), float("nan"), device=lm.device)
    api.gca_decode_retrieve_noalloc(lm, ql, N, D, topk, lm.dtype, off_by_one, 0.0, idx, r, w)
    return idx, r, w


def check_same(got, ref):
    np.testing.assert_array_equal(got[0].cpu().numpy(), ref[0].cpu().numpy())
    np.testing.assert_allclose(got[1].cpu().numpy(), ref[1].cpu().numpy(), atol=1e-5, rtol=1e-6)
    np.testing.assert_allclose(got[2].cpu().numpy(), ref[2].cpu().numpy(), atol=1e-6, rtol=1e-5)


def test_noalloc_matches_workspace_entry_point():
    x = inputs.decode_inputs()                        # 262144 landmarks x 768, bf16
    lm, ql = x["lm"].cuda(), x["ql"].cuda()
    ref = api.decode_retrieve(lm, ql, topk=8)
    first = noalloc(lm, ql, 8, False)
    assert api.gca_last_launch_count() == 1
    second = noalloc(lm, ql, 8, False)                # the array keeps the first call's contents
    torch.cuda.synchronize()
    check_same(first, ref)
    check_same(second, ref)

    # a smaller, different problem right after, then the large one again
    g = torch.Generator().manual_seed(3)
    lm2 = torch.randint(-2, 3, (5000, 64), generator=g).to(torch.float32).cuda()
    ql2 = torch.randint(-2, 3, (64,), generator=g).to(torch.float32).cuda()
    check_same(noalloc(lm2, ql2, 16, True), api.decode_retrieve(lm2, ql2, topk=16, off_by_one=True))
    check_same(noalloc(lm, ql, 8, False), ref)
    assert api.gca_get_status() == 0


def test_noalloc_refuses_requests_beyond_its_array():
    lm = torch.zeros(262144, 32, dtype=torch.bfloat16, device="cuda")
    ql = torch.zeros(32, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(GcaError) as e:
        noalloc(lm, ql, 32, False)                    # 2048 CTAs x 32 ranks > the array
    assert e.value.code == 3                          # GCA_ERR_WORKSPACE


def test_noalloc_reports_device_errors_through_the_status_word():
    # a bounded wait that runs out inside this entry point is recorded in the
    # same per-device status word as every other entry's (test-only stall
    # switch), and the next call is normal again
    x = inputs.decode_inputs(N=65536)
    lm, ql = x["lm"].cuda(), x["ql"].cuda()
    ref = api.decode_retrieve(lm, ql, topk=8)
    assert api.gca_get_status() == 0
    api.gca_debug_stall_next_decode(200_000)
    noalloc(lm, ql, 8, False)
    assert api.gca_last_launch_count() == 1
    assert api.gca_get_status() == 5                  # GCA_ERR_TIMEOUT
    check_same(noalloc(lm, ql, 8, False), ref)
    assert api.gca_get_status() == 0
