"""Decode with the K/V cache offloaded to page-locked host memory (section 3.2:
past chunks live in CPU memory and are reloaded when retrieved): retrieval on
the device, gca_gather_chunks reads the retrieved chunks over the CPU-GPU link
into a compact device pool, gca_fwd runs on it.  The result must equal the
forward over the device-resident cache bit for bit, and the oracle."""
import numpy as np
import pytest
import torch

import oracle
from retrieval_sparse_attention_gb300 import api, inputs

from gpu_helpers import assert_close, assert_lse, f64

pytestmark = pytest.mark.gpu


def make_cache(N, S, H, d, seed):
    ck = torch.empty(N, S, H, d, dtype=torch.bfloat16, device="cuda")
    cv = torch.empty_like(ck)
    api.gca_synth_fill_hash(ck, seed, 0)
    api.gca_synth_fill_hash(cv, seed, 1)
    torch.cuda.synchronize()
    return ck, cv


@pytest.mark.parametrize("N,topk", [(512, 8), (37, 16), (5, 8)])
def test_offloaded_decode_matches_device_resident(N, topk):
    p = inputs.DECODE
    S, H, d, seed = p["S"], p["H"], p["d"], p["seed"]
    x = inputs.decode_inputs(N=N)
    lm, ql, q = x["lm"].cuda(), x["ql"].cuda(), x["q"].cuda().view(1, S, H, d)
    ck, cv = make_cache(N, S, H, d, seed)
    hk = ck.cpu().pin_memory()
    hv = cv.cpu().pin_memory()
    idx, r, w = api.decode_retrieve(lm, ql, topk=topk)
    # device-resident pool
    o_dev, lse_dev = api.fwd(q, ck.view(1, N * S, H, d), cv.view(1, N * S, H, d), idx.view(1, 1, topk),
                             w.view(1, 1, topk), S=S)
    # offloaded pool: gather from pinned host memory, then the same forward
    pk, pv, pidx = api.gather_chunks(hk, hv, idx)
    o_off, lse_off = api.fwd(q, pk, pv, pidx, w.view(1, 1, topk), S=S)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    assert torch.equal(o_dev, o_off)
    assert torch.equal(lse_dev, lse_off)
    # and the oracle, from the host generator's chunks
    gi = idx.cpu().numpy()
    oi, _, ow = oracle.decode_retrieve(f64(x["lm"]), f64(x["ql"]), topk)
    np.testing.assert_array_equal(gi, oi)
    valid = [int(c) for c in oi if c >= 0]
    kk = np.concatenate([inputs.decode_cache_chunk_np(seed, 0, c, S, H, d) for c in valid])[None]
    vv = np.concatenate([inputs.decode_cache_chunk_np(seed, 1, c, S, H, d) for c in valid])[None]
    ridx = np.array([[[j if j < len(valid) else -1 for j in range(topk)]]], dtype=np.int32)
    oo, olse = oracle.fwd(f64(x["q"]).reshape(1, S, H, d), kk, vv, ridx, ow.reshape(1, 1, topk), S)
    assert_close("o", f64(o_off), oo, 2e-2, 2e-2)
    assert_lse(f64(lse_off), olse, 1e-3)


def test_gather_reports_out_of_range_and_zero_fills():
    S, H, d = 64, 2, 64
    ck = torch.ones(4, S, H, d, dtype=torch.bfloat16).pin_memory()
    cv = torch.ones(4, S, H, d, dtype=torch.bfloat16).pin_memory()
    idx = torch.tensor([2, 9, -1], dtype=torch.int32, device="cuda")
    pk, pv, pidx = api.gather_chunks(ck, cv, idx)
    assert api.gca_get_status() == 6                  # GCA_ERR_DEVICE_INDEX
    assert pidx.view(-1).tolist() == [0, -1, -1]
    assert (pk[0, :S] == 1).all() and (pk[0, S:] == 0).all()
