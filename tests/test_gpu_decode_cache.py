"""The decode workload end to end at full size: a 16M-token context (262144
chunk landmarks x 768, section 4.3 / Table 3: retrieval once per 64 generated
tokens), one 64-token query chunk scores every landmark, takes the top 8
(gca_decode_retrieve), and attends to the retrieved chunks of the per-chunk
K/V cache held in HBM (gca_fwd over [262144 * 64, 12, 64] K and V, 51.5 GB).

The cache is filled on the device by the counter-based generator, and the
host regenerates exactly the retrieved chunks for the oracle, so the forward
is checked element by element at row offsets tens of GB into the tensors."""
import numpy as np
import pytest
import torch

import oracle
from retrieval_sparse_attention_gb300 import api, inputs

from gpu_helpers import assert_close, assert_lse, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("off_by_one", [False, True])
def test_decode_retrieve_then_fwd_over_full_cache(off_by_one):
    p = inputs.DECODE
    N, D, S, H, d, topk, seed = p["N"], p["D"], p["S"], p["H"], p["d"], p["topk"], p["seed"]
    x = inputs.decode_inputs()
    lm, ql, q = x["lm"].cuda(), x["ql"].cuda(), x["q"].cuda().view(1, S, H, d)
    free, _ = torch.cuda.mem_get_info()
    need = 2 * N * S * H * d * 2
    if free < need + (4 << 30):
        pytest.skip("the 51.5 GB cache does not fit on this device")
    ck = torch.empty(1, N * S, H, d, dtype=torch.bfloat16, device="cuda")
    cv = torch.empty_like(ck)
    try:
        api.gca_synth_fill_hash(ck, seed, 0)
        api.gca_synth_fill_hash(cv, seed, 1)
        idx, r, w = api.decode_retrieve(lm, ql, topk=topk, off_by_one=off_by_one)
        o, lse = api.fwd(q, ck, cv, idx.view(1, 1, topk), w.view(1, 1, topk), S=S)
        torch.cuda.synchronize()
        assert api.gca_get_status() == 0
        gi = idx.cpu().numpy()
    finally:
        del ck, cv
        torch.cuda.empty_cache()
    oi, orr, ow = oracle.decode_retrieve(f64(x["lm"]), f64(x["ql"]), topk, off_by_one)
    np.testing.assert_array_equal(gi, oi)
    assert_close("weight", f64(w), ow, 1e-6, 1e-5)
    # the retrieved chunks lie far into the cache: offsets beyond 2^31 bytes
    assert int(oi.max()) * S * H * d * 2 > (1 << 31)
    kk = np.concatenate([inputs.decode_cache_chunk_np(seed, 0, int(c), S, H, d) for c in oi])[None]
    vv = np.concatenate([inputs.decode_cache_chunk_np(seed, 1, int(c), S, H, d) for c in oi])[None]
    ridx = np.arange(topk, dtype=np.int32).reshape(1, 1, topk)
    oo, olse = oracle.fwd(f64(x["q"]).reshape(1, S, H, d), kk, vv, ridx, ow.reshape(1, 1, topk), S)
    assert_close("o", f64(o), oo, 2e-2, 2e-2)
    assert_lse(f64(lse), olse, 1e-3)
