"""GPU parity of the GCA forward (gca_fwd) and backward (gca_bwd) against the
fp64 oracle.  The GPU runs its own pipeline (gca_score_topk -> gca_fwd ->
gca_bwd); the oracle runs its own from the same seeded inputs.  Small cases
are compared on every element; the full-size workloads on sampled chunks
whose oracle results are computed one by one."""
import numpy as np
import pytest
import torch

import oracle
from retrieval_sparse_attention_gb300 import api, inputs

from gpu_helpers import assert_close, assert_lse, f64, mini_problem, take_chunks, tol_for

pytestmark = pytest.mark.gpu


def gpu_pipeline(x, wl, off_by_one, include_self, backward=True):
    dev = "cuda"
    lm, q, k, v = (x[n].to(dev) for n in ("lm", "q", "k", "v"))
    idx, r, w = api.score_topk(lm, S=wl.S, H=wl.H, d=wl.d, topk=wl.topk, off_by_one=off_by_one,
                               include_self=include_self)
    o, lse = api.fwd(q, k, v, idx, w, S=wl.S)
    out = {"idx": idx, "w": w, "o": o, "lse": lse}
    if backward:
        g = x["dout"].to(dev)
        dq, dk, dv, ds = api.bwd(q, k, v, idx, w, lse, g, S=wl.S)
        out.update(dq=dq, dk=dk, dv=dv, ds=ds)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    return out


SMALL = [
    ("tiny_fp32", None, None, False, False),
    ("tiny_fp32", None, None, True, True),
    ("gpt2s_fwdbwd_b8", 2, 2048, False, False),
    ("gpt2s_fwdbwd_b8", 1, 1600, True, False),
    ("gpt2s_fwdbwd_b8", 1, 1536, False, True),
    ("long64k_S128_k8", 1, 4096, False, False),
    ("long64k_S128_k4", 2, 1664, True, True),
    ("long64k_S64_k16", 1, 2304, False, False),
    ("long64k_S128_k16", 1, 3328, False, False),
    ("long64k_S128_k16", 1, 2560, True, True),
    ("long64k_S64_k4", 1, 1984, False, True),
]


@pytest.mark.parametrize("name,B,L,off_by_one,include_self", SMALL)
def test_fwd_bwd_every_element(name, B, L, off_by_one, include_self):
    wl = inputs.WORKLOADS[name]
    x = inputs.make(wl, B=B, L=L)
    got = gpu_pipeline(x, wl, off_by_one, include_self)
    lm, q, k, v, g = (f64(x[n]) for n in ("lm", "q", "k", "v", "dout"))
    oi, orr, ow = oracle.score_topk(lm, wl.topk, include_self, off_by_one)
    np.testing.assert_array_equal(got["idx"].cpu().numpy(), oi)
    atol, rtol = tol_for(x["q"].dtype)
    oo, olse = oracle.fwd(q, k, v, oi, ow, wl.S)
    assert_close("o", f64(got["o"]), oo, atol, rtol)
    assert_lse(f64(got["lse"]), olse, 1e-3 if atol > 1e-3 else 1e-4)
    dq, dk, dv, ds = oracle.bwd(q, k, v, oi, ow, g, wl.S)
    assert_close("dq", f64(got["dq"]), dq, atol, rtol)
    assert_close("dk", f64(got["dk"]), dk, atol, rtol)
    assert_close("dv", f64(got["dv"]), dv, atol, rtol)
    assert_close("dscore", f64(got["ds"]), ds, atol, rtol)


FULL = [("gpt2s_fwd_b4", True, False), ("gpt2s_fwdbwd_b8", False, True)] + \
    [("long64k_S%d_k%d" % (S, k), False, True) for S in (64, 128) for k in (4, 8, 16)]


@pytest.mark.parametrize("name,off_by_one,backward", FULL)
def test_full_size_sampled(name, off_by_one, backward):
    wl = inputs.WORKLOADS[name]
    x = inputs.make(wl, with_dout=backward)
    got = gpu_pipeline(x, wl, off_by_one, False, backward=backward)
    S, nC = wl.S, wl.nC
    oi, orr, ow = oracle.score_topk(f64(x["lm"]), wl.topk, False, off_by_one)
    gi = got["idx"].cpu().numpy()
    np.testing.assert_array_equal(gi, oi)
    atol, rtol = tol_for(x["q"].dtype)
    rng = np.random.default_rng(17)
    for b in range(wl.B):
        # query side: a few chunks (first with slots, last, random)
        cs = sorted(set([2, 3, nC - 1] + list(rng.integers(0, nC, 3))))
        pool, rows = mini_problem(oi[b], cs, S)
        q_ = take_chunks(x["q"], b, cs, S)
        k_ = take_chunks(x["k"], b, pool, S)
        v_ = take_chunks(x["v"], b, pool, S)
        w_ = ow[b, cs][None]
        oo, olse = oracle.fwd(q_, k_, v_, rows[None], w_, S)
        go = take_chunks(got["o"], b, cs, S)
        assert_close("o[b=%d]" % b, go, oo, atol, rtol)
        gl = take_chunks(got["lse"], b, cs, S)
        assert_lse(gl, olse, 1e-3)
        if not backward:
            continue
        g_ = take_chunks(x["dout"], b, cs, S)
        dq, _, _, ds = oracle.bwd(q_, k_, v_, rows[None], w_, g_, S,
                                  kmask=np.zeros((1, len(pool)), bool))
        gdq = take_chunks(got["dq"], b, cs, S)
        assert_close("dq[b=%d]" % b, gdq, dq, atol, rtol)
        assert_close("dscore[b=%d]" % b, f64(got["ds"][b, cs])[None], ds, atol, rtol)
        # key side: the most retrieved chunk, an unretrieved one and a random one
        counts = np.bincount(oi[b][oi[b] >= 0].ravel(), minlength=nC)
        for kap in (int(np.argmax(counts)), nC - 1, int(rng.integers(0, nC))):
            users = [c for c in range(nC) if (oi[b, c] == kap).any()]
            rows_k = np.where(oi[b, users] == kap, 0, -1).astype(np.int32)
            q_ = take_chunks(x["q"], b, users, S)
            g_ = take_chunks(x["dout"], b, users, S)
            k_ = take_chunks(x["k"], b, [kap], S)
            v_ = take_chunks(x["v"], b, [kap], S)
            if not users:
                want_k = np.zeros_like(k_)
                want_v = np.zeros_like(v_)
            else:
                _, want_k, want_v, _ = oracle.bwd(q_, k_, v_, rows_k[None], ow[b, users][None], g_, S,
                                                  qmask=np.zeros((1, len(users)), bool))
            assert_close("dk[b=%d,chunk=%d]" % (b, kap), f64(got["dk"][b, kap * S:(kap + 1) * S])[None],
                         want_k, atol, rtol)
            assert_close("dv[b=%d,chunk=%d]" % (b, kap), f64(got["dv"][b, kap * S:(kap + 1) * S])[None],
                         want_v, atol, rtol)


def test_bwd_is_deterministic():
    wl = inputs.WORKLOADS["gpt2s_fwdbwd_b8"]
    x = inputs.make(wl, B=2, L=4096)
    a = gpu_pipeline(x, wl, False, False)
    b = gpu_pipeline(x, wl, False, False)
    for n in ("o", "lse", "dq", "dk", "dv", "ds"):
        assert torch.equal(a[n], b[n]), n


def test_no_slots_anywhere():
    # two chunks under the strict causal set: no query chunk has a candidate
    wl = inputs.WORKLOADS["gpt2s_fwdbwd_b8"]
    x = inputs.make(wl, B=1, L=128)
    got = gpu_pipeline(x, wl, False, False)
    assert (got["idx"] == -1).all()
    for n in ("o", "dq", "dk", "dv", "ds"):
        assert (got[n] == 0).all(), n
    assert torch.isneginf(got["lse"]).all()


def test_single_pool_chunk_decode_shape():
    # one query chunk against a pool of one chunk, fed explicit idx/weights
    dev = "cuda"
    g = torch.Generator().manual_seed(5)
    q = (torch.randn(1, 64, 12, 64, generator=g) / 8).to(torch.bfloat16)
    k = (torch.randn(1, 64, 12, 64, generator=g) / 8).to(torch.bfloat16)
    v = (torch.randn(1, 64, 12, 64, generator=g) / 8).to(torch.bfloat16)
    idx = torch.tensor([[[0, -1, -1]]], dtype=torch.int32)
    w = torch.tensor([[[0.7, 0.0, 0.0]]], dtype=torch.float32)
    o, lse = api.fwd(q.to(dev), k.to(dev), v.to(dev), idx.to(dev), w.to(dev), S=64)
    torch.cuda.synchronize()
    oo, olse = oracle.fwd(f64(q), f64(k), f64(v), idx.numpy(), f64(w), 64)
    assert_close("o", f64(o), oo, 2e-2, 2e-2)
    assert_lse(f64(lse), olse, 1e-3)


def test_out_of_range_index_sets_status():
    # an index past the pool is caught by the kernel's own bounds check:
    # the slot is skipped and the status word reports it; nothing faults.
    dev = "cuda"
    q = torch.zeros(1, 64, 12, 64, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 128, 12, 64, dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    idx = torch.tensor([[[5, 0]]], dtype=torch.int32, device=dev)
    w = torch.tensor([[[0.5, 0.5]]], dtype=torch.float32, device=dev)
    api.fwd(q, k, v, idx, w, S=64)
    assert api.gca_get_status() == 6      # GCA_ERR_DEVICE_INDEX
    assert api.gca_get_status() == 0      # reading clears it


def test_long_row_inverse_index_fallback():
    # 4096 chunks x k = 8 in one batch row: the row's inverse index (count, offset
    # and entry arrays, ~400 KB) does not fit one CTA's shared memory, so the
    # backward builds it in three passes.  Caller-supplied retrieval: each query
    # chunk c >= 1 takes k distinct random earlier chunks, weights a softmax.
    S, nC, H, d, k = 64, 4096, 1, 64, 8
    L = nC * S
    g = torch.Generator().manual_seed(21)
    q, kk, v, dout = [(torch.randn(1, L, H, d, generator=g) * s).to(torch.bfloat16)
                      for s in (0.125, 0.125, 0.125, 1.0)]
    rng = np.random.default_rng(22)
    idx = np.full((1, nC, k), -1, np.int32)
    for c in range(1, nC):
        m = min(k, c)
        idx[0, c, :m] = np.sort(rng.choice(c, m, replace=False))
    raw = rng.standard_normal((1, nC, k))
    w = np.where(idx >= 0, np.exp(raw), 0.0)
    w = (w / np.maximum(w.sum(-1, keepdims=True), 1e-30)).astype(np.float32)
    dev = "cuda"
    ti, tw = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)
    qc, kc, vc, gc = (x.to(dev) for x in (q, kk, v, dout))
    o, lse = api.fwd(qc, kc, vc, ti, tw, S=S)
    dq, dk, dv, ds = api.bwd(qc, kc, vc, ti, tw, lse, gc, S=S)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0
    atol, rtol = tol_for(torch.bfloat16)
    w64 = w.astype(np.float64)
    # key side: the most retrieved chunk, the last (never retrieved) and random ones
    counts = np.bincount(idx[0][idx[0] >= 0].ravel(), minlength=nC)
    for kap in [int(np.argmax(counts)), nC - 1] + [int(x) for x in rng.integers(0, nC - 1, 3)]:
        users = [c for c in range(nC) if (idx[0, c] == kap).any()]
        k_ = take_chunks(kk, 0, [kap], S)
        v_ = take_chunks(v, 0, [kap], S)
        if not users:
            want_k, want_v = np.zeros_like(k_), np.zeros_like(v_)
        else:
            rows_k = np.where(idx[0, users] == kap, 0, -1).astype(np.int32)
            _, want_k, want_v, _ = oracle.bwd(take_chunks(q, 0, users, S), k_, v_, rows_k[None],
                                              w64[0, users][None], take_chunks(dout, 0, users, S), S,
                                              qmask=np.zeros((1, len(users)), bool))
        assert_close("dk[chunk=%d]" % kap, f64(dk[0, kap * S:(kap + 1) * S])[None], want_k, atol, rtol)
        assert_close("dv[chunk=%d]" % kap, f64(dv[0, kap * S:(kap + 1) * S])[None], want_v, atol, rtol)
    # query side: a few chunks
    cs = sorted(set([1, 2, nC - 1] + [int(x) for x in rng.integers(1, nC, 3)]))
    pool, rows = mini_problem(idx[0], cs, S)
    q_ = take_chunks(q, 0, cs, S)
    k_ = take_chunks(kk, 0, pool, S)
    v_ = take_chunks(v, 0, pool, S)
    g_ = take_chunks(dout, 0, cs, S)
    want_dq, _, _, want_ds = oracle.bwd(q_, k_, v_, rows[None], w64[0, cs][None], g_, S,
                                        kmask=np.zeros((1, len(pool)), bool))
    assert_close("dq", take_chunks(dq, 0, cs, S), want_dq, atol, rtol)
    assert_close("dscore", f64(ds[0, cs])[None], want_ds, atol, rtol)
