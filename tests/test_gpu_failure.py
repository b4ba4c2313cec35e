"""The device-side failure path, exercised without a real hang or fault.

Every wait in the library's kernels is bounded.  A test-only switch
(gca_debug_stall_next_decode) makes one CTA of the next decode retrieval
withhold a stage of its landmark stream and shortens the bound to a few
hundred microseconds: the waiting warps give up, record GCA_ERR_TIMEOUT,
wait for the copies they did issue, and return.  The context must stay
usable: the next call, made normally, must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from retrieval_sparse_attention_gb300 import api, inputs

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu

GCA_ERR_TIMEOUT = 5


def check_decode(lm, ql, topk, got):
    oi, orr, ow = oracle.decode_retrieve(f64(lm), f64(ql), topk)
    np.testing.assert_array_equal(got[0].cpu().numpy(), oi)
    assert_close("score", f64(got[1]), orr, 1e-5, 1e-6)
    assert_close("weight", f64(got[2]), ow, 1e-6, 1e-5)


@pytest.mark.parametrize("N,D,topk", [(65536, 768, 8), (3000, 64, 16)])
def test_decode_wait_timeout_is_reported_and_recovers(N, D, topk):
    x = inputs.decode_inputs(N=N) if D == 768 else None
    if x is None:
        g = torch.Generator().manual_seed(N)
        lm = torch.randint(-3, 4, (N, D), generator=g).to(torch.bfloat16)
        ql = torch.randint(-3, 4, (D,), generator=g).to(torch.bfloat16)
    else:
        lm, ql = x["lm"], x["ql"]
    dl, dq = lm.cuda(), ql.cuda()
    assert api.gca_get_status() == 0
    api.gca_debug_stall_next_decode(200_000)                  # 200 us bound, one stage withheld
    api.decode_retrieve(dl, dq, topk=topk)
    assert api.gca_get_status() == GCA_ERR_TIMEOUT
    assert api.gca_get_status() == 0                          # reading clears it
    # the switch was consumed: the next call runs normally on the same context
    got = api.decode_retrieve(dl, dq, topk=topk)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    check_decode(lm, ql, topk, got)


def test_stall_switch_rejects_out_of_range_bounds():
    from retrieval_sparse_attention_gb300._lib import GcaError
    for bad in (0, 999, 2_000_000_000):
        with pytest.raises(GcaError):
            api.gca_debug_stall_next_decode(bad)
