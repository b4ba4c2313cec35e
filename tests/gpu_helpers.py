"""Helpers shared by the GPU parity tests (plumbing only, no GCA arithmetic)."""
import numpy as np
import torch

BF16_ATOL = 2e-2
BF16_RTOL = 2e-2
F32_TOL = 1e-4


def f64(t):
    return t.detach().double().cpu().numpy()


def tol_for(dtype):
    return (BF16_ATOL, BF16_RTOL) if dtype == torch.bfloat16 else (F32_TOL, 0.0)


def assert_close(name, got, want, atol, rtol):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.isfinite(got).all(), "%s has non-finite values" % name
    excess = np.abs(got - want) - (atol + rtol * np.abs(want))
    if (excess > 0).any():
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError("%s: %d elements outside |err| <= %g + %g|ref|; worst at %s: got %r want %r"
                             % (name, int((excess > 0).sum()), atol, rtol, i, got[i], want[i]))


def assert_lse(got, want, atol):
    got = np.asarray(got, dtype=np.float64)
    inf_w = np.isneginf(want)
    assert (np.isneginf(got) == inf_w).all(), "empty-slot lse must be -inf exactly where the oracle's is"
    assert_close("lse", got[~inf_w], want[~inf_w], atol, 0.0)


def mini_problem(idx, c_list, S):
    """Compact the query chunks `c_list` of one batch row and the chunks they
    retrieve into a small problem: returns (pool chunk ids, remapped idx rows)."""
    rows = idx[c_list]                                   # [n, k]
    pool = sorted(set(int(x) for x in rows.ravel() if x >= 0))
    remap = {p: i for i, p in enumerate(pool)}
    new = np.vectorize(lambda x: remap.get(int(x), -1))(rows).astype(np.int32) if rows.size else rows
    return pool, new


def take_chunks(x, b, chunks, S):
    """x [B, L, H, d] (torch, any device) -> [1, len(chunks)*S, H, d] host fp64 for
    the chunks `chunks` of row b (only those slices are converted)."""
    if len(chunks) == 0:
        return np.zeros((1, 0) + tuple(x.shape[2:]))
    parts = [f64(x[b, c * S:(c + 1) * S]) for c in chunks]
    return np.concatenate(parts, axis=0)[None]


def cuda_inputs(x, dev="cuda"):
    return {k: v.to(dev) for k, v in x.items()}
