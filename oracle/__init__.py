"""fp64 CPU oracle for Grouped Cross Attention (GCA) -- test infrastructure.

This package wraps ``gca_oracle.c`` (plain double-precision loops that state
what the GCA hot path computes) through ctypes on NumPy arrays.  Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The product path (the CUDA library and its binding) never does; it
fails loudly when the CUDA library is missing instead of falling back here.

Method source: "Efficient Length-Generalizable Attention via Causal Retrieval
for Long-Context Language Modeling" (ICML 2025, arXiv 2410.01651): the
rebuttal comment "Cmt 1" (G=1 form of Eq. 1, r = l_t^T l_k / sqrt(d)), the
answers to W2 (Eq. 2 is the batch form of Figure 2) and Q4 (Eq. 3, softmax
off by one), the official README's "Model Architecture" (two-stage
attention, weighted fusion), and sections 1 and 4.1.2 of the paper summary
for the 512-token sliding-window self-attention that precedes GCA in a layer.  Every function below is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gca_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgca_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gca_oracle.c into libgca_oracle.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i32, f64 = ctypes.c_int, ctypes.c_double
        vp = ctypes.c_void_p
        lib.oracle_weights_from_scores.argtypes = [i32, vp, i32, vp]
        lib.oracle_score_topk.argtypes = [i32, i32, i32, i32, i32, i32, f64, vp, vp, vp, vp]
        lib.oracle_score_topk.restype = i32
        lib.oracle_decode_retrieve.argtypes = [i32, i32, i32, i32, f64, vp, vp, vp, vp, vp]
        lib.oracle_decode_retrieve.restype = i32
        lib.oracle_fwd.argtypes = [i32] * 7 + [f64] + [vp] * 8
        lib.oracle_bwd.argtypes = [i32] * 7 + [f64] + [vp] * 12
        lib.oracle_num_threads.restype = i32
        lib.oracle_landmark_bwd.argtypes = [i32, i32, i32, i32, f64, vp, vp, vp, vp]
        lib.oracle_score_topk_noisy.argtypes = [i32, i32, i32, i32, i32, i32, f64, vp, vp, vp, vp, vp]
        lib.oracle_score_topk_noisy.restype = i32
        lib.oracle_swa_fwd.argtypes = [i32] * 5 + [f64] + [vp] * 5
        lib.oracle_swa_bwd.argtypes = [i32] * 5 + [f64] + [vp] * 7
        _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().oracle_num_threads())


def weights_from_scores(r, off_by_one: bool):
    """Softmax (or softmax-off-by-one) of a 1-D array of valid scores."""
    r = _f64(r)
    w = np.zeros_like(r)
    _load().oracle_weights_from_scores(r.size, _ptr(r), int(off_by_one), _ptr(w))
    return w


def score_topk(lm, topk: int, include_self: bool = False, off_by_one: bool = False,
               score_scale: float | None = None):
    """Causal scoring + top-k + softmax.  lm: [B, nC, D].  Returns idx, r, w [B, nC, topk]."""
    lm = _f64(lm)
    B, nC, D = lm.shape
    if score_scale is None:
        score_scale = 1.0 / np.sqrt(D)
    idx = np.empty((B, nC, topk), dtype=np.int32)
    r = np.empty((B, nC, topk))
    w = np.empty((B, nC, topk))
    rc = _load().oracle_score_topk(B, nC, D, topk, int(include_self), int(off_by_one),
                                   float(score_scale), _ptr(lm), _ptr(idx), _ptr(r), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_score_topk: topk must be in [1, 64]")
    return idx, r, w


def decode_retrieve(lm, ql, topk: int, off_by_one: bool = False, score_scale: float | None = None):
    """Decode retrieval over every landmark.  lm: [N, D], ql: [D].  Returns idx, r, w [topk]."""
    lm = _f64(lm)
    ql = _f64(ql)
    N, D = lm.shape
    if score_scale is None:
        score_scale = 1.0 / np.sqrt(D)
    idx = np.empty(topk, dtype=np.int32)
    r = np.empty(topk)
    w = np.empty(topk)
    rc = _load().oracle_decode_retrieve(N, D, topk, int(off_by_one), float(score_scale),
                                        _ptr(lm), _ptr(ql), _ptr(idx), _ptr(r), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_decode_retrieve: topk must be in [1, 64]")
    return idx, r, w


def _mask(m, shape):
    if m is None:
        return None
    return np.ascontiguousarray(np.asarray(m, dtype=np.uint8).reshape(shape))


def fwd(q, k, v, idx, w, S: int, attn_scale: float | None = None, qmask=None):
    """GCA forward.  q [B, Lq, H, d]; k, v [B, Lp, H, d]; idx, w [B, Lq/S, topk].

    Returns (o [B, Lq, H, d], lse [B, Lq, H, topk]).  With ``qmask`` [B, nQ]
    only the selected query chunks are computed (the rest stays 0)."""
    q, k, v, w = _f64(q), _f64(k), _f64(v), _f64(w)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    B, Lq, H, d = q.shape
    Lp = k.shape[1]
    nQ, nP, topk = Lq // S, Lp // S, idx.shape[-1]
    assert idx.shape == (B, nQ, topk) and w.shape == (B, nQ, topk)
    if attn_scale is None:
        attn_scale = 1.0 / np.sqrt(d)
    o = np.zeros_like(q)
    lse = np.zeros((B, Lq, H, topk))
    qm = _mask(qmask, (B, nQ))
    _load().oracle_fwd(B, nQ, nP, S, H, d, topk, float(attn_scale), _ptr(q), _ptr(k), _ptr(v),
                       _ptr(idx), _ptr(w), _ptr(o), _ptr(lse), _ptr(qm))
    return o, lse


def bwd(q, k, v, idx, w, dout, S: int, attn_scale: float | None = None, qmask=None, kmask=None):
    """GCA backward.  Returns (dq, dk, dv, dscore); dscore = dLoss/dr [B, nQ, topk]."""
    q, k, v, w, dout = _f64(q), _f64(k), _f64(v), _f64(w), _f64(dout)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    B, Lq, H, d = q.shape
    Lp = k.shape[1]
    nQ, nP, topk = Lq // S, Lp // S, idx.shape[-1]
    if attn_scale is None:
        attn_scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    ds = np.zeros((B, nQ, topk))
    qm = _mask(qmask, (B, nQ))
    km = _mask(kmask, (B, nP))
    _load().oracle_bwd(B, nQ, nP, S, H, d, topk, float(attn_scale), _ptr(q), _ptr(k), _ptr(v),
                       _ptr(idx), _ptr(w), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ds),
                       _ptr(qm), _ptr(km))
    return dq, dk, dv, ds


def landmark_bwd(lm, idx, dscore, score_scale: float | None = None):
    """Gradient of the loss w.r.t. the landmarks given dLoss/dr.  lm [B, nC, D]."""
    lm = _f64(lm)
    dscore = _f64(dscore)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    B, nC, D = lm.shape
    topk = idx.shape[-1]
    if score_scale is None:
        score_scale = 1.0 / np.sqrt(D)
    dl = np.zeros_like(lm)
    _load().oracle_landmark_bwd(B, nC, D, topk, float(score_scale), _ptr(lm), _ptr(idx),
                                _ptr(dscore), _ptr(dl))
    return dl


def score_topk_noisy(lm, noise, topk: int, include_self: bool = False, off_by_one: bool = False,
                     score_scale: float | None = None):
    """Top-k selected by r + noise (fp32 key), softmax over the clean r.
    noise [B, nC, nC] float32."""
    lm = _f64(lm)
    noise = np.ascontiguousarray(noise, dtype=np.float32)
    B, nC, D = lm.shape
    assert noise.shape == (B, nC, nC)
    if score_scale is None:
        score_scale = 1.0 / np.sqrt(D)
    idx = np.empty((B, nC, topk), dtype=np.int32)
    r = np.empty((B, nC, topk))
    w = np.empty((B, nC, topk))
    rc = _load().oracle_score_topk_noisy(B, nC, D, topk, int(include_self), int(off_by_one),
                                         float(score_scale), _ptr(lm), _ptr(noise), _ptr(idx),
                                         _ptr(r), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_score_topk_noisy: topk must be in [1, 64]")
    return idx, r, w


def swa_fwd(q, k, v, window: int, attn_scale: float | None = None):
    """Sliding-window causal self-attention.  q, k, v [B, L, H, d]; token t
    attends to keys max(0, t-window+1) .. t.  Returns (o [B,L,H,d], lse [B,L,H])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, L, H, d = q.shape
    if attn_scale is None:
        attn_scale = 1.0 / np.sqrt(d)
    o = np.zeros_like(q)
    lse = np.zeros((B, L, H))
    _load().oracle_swa_fwd(B, L, H, d, int(window), float(attn_scale), _ptr(q), _ptr(k), _ptr(v),
                           _ptr(o), _ptr(lse))
    return o, lse


def swa_bwd(q, k, v, dout, window: int, attn_scale: float | None = None):
    """Gradients of sum(dout * swa_fwd(q, k, v).o): returns (dq, dk, dv)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, L, H, d = q.shape
    if attn_scale is None:
        attn_scale = 1.0 / np.sqrt(d)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    _load().oracle_swa_bwd(B, L, H, d, int(window), float(attn_scale), _ptr(q), _ptr(k), _ptr(v),
                           _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv
