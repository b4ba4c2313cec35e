"""Thin PyTorch binding of the GCA C ABI (argument marshalling only).

Each ``gca_*`` function has the name and argument order of its C entry point
and passes ``data_ptr()`` of CUDA tensors plus the current CUDA stream; every
step of the computation runs in libgca.so.  The convenience functions
``score_topk``, ``fwd``, ``bwd`` and ``decode_retrieve`` only allocate the
outputs (and workspace) with PyTorch, then call the same entry points.

GCA itself ("Efficient Length-Generalizable Attention via Causal Retrieval
for Long-Context Language Modeling", ICML 2025) is documented in
include/gca.h next to each entry point.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import GCA_BF16, GCA_F32, GcaError, GcaParams, GcaSwaParams

_DT = {torch.bfloat16: GCA_BF16, torch.float32: GCA_F32}


def dtype_code(t: torch.dtype) -> int:
    if t not in _DT:
        raise TypeError("GCA supports bfloat16 and float32 tensors, got %s" % t)
    return _DT[t]


def make_params(*, B, Lq, S, H, d, topk, n_pool_chunks=None, landmark_dim=0, dtype=torch.bfloat16,
                off_by_one=False, include_self=False, score_scale=0.0, attn_scale=0.0) -> GcaParams:
    return GcaParams(B=B, Lq=Lq, S=S, H=H, d=d, topk=topk,
                     n_pool_chunks=(Lq // S if n_pool_chunks is None else n_pool_chunks),
                     landmark_dim=landmark_dim, dtype=dtype_code(dtype),
                     softmax_off_by_one=int(bool(off_by_one)), include_self=int(bool(include_self)),
                     score_scale=float(score_scale), attn_scale=float(attn_scale))


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("GCA entry points take CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("GCA entry points take contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, code):
    if code != 0:
        raise GcaError(fn, code)


# --- the C entry points, same names --------------------------------------------------
def gca_score_topk(params: GcaParams, landmarks, idx, score, weight, stream=None):
    _check("gca_score_topk", _lib.load().gca_score_topk(ctypes.byref(params), _p(landmarks), _p(idx),
                                                        _p(score), _p(weight), _stream(stream)))


def gca_score_topk_noisy(params: GcaParams, landmarks, noise, idx, score, weight, stream=None):
    _check("gca_score_topk_noisy", _lib.load().gca_score_topk_noisy(
        ctypes.byref(params), _p(landmarks), _p(noise), _p(idx), _p(score), _p(weight),
        _stream(stream)))


def gca_landmark_bwd_workspace_size(params: GcaParams) -> int:
    return int(_lib.load().gca_landmark_bwd_workspace_size(ctypes.byref(params)))


def gca_landmark_bwd(params: GcaParams, landmarks, idx, dscore, dlandmarks, workspace, stream=None):
    _check("gca_landmark_bwd", _lib.load().gca_landmark_bwd(
        ctypes.byref(params), _p(landmarks), _p(idx), _p(dscore), _p(dlandmarks), _p(workspace),
        workspace.numel(), _stream(stream)))


def gca_fwd(params: GcaParams, q, k, v, idx, weight, o, lse=None, stream=None):
    _check("gca_fwd", _lib.load().gca_fwd(ctypes.byref(params), _p(q), _p(k), _p(v), _p(idx),
                                          _p(weight), _p(o), _p(lse), _stream(stream)))


def gca_bwd_workspace_size(params: GcaParams) -> int:
    return int(_lib.load().gca_bwd_workspace_size(ctypes.byref(params)))


def gca_bwd(params: GcaParams, q, k, v, idx, weight, lse, dout, dq, dk, dv, dscore, workspace,
            stream=None):
    _check("gca_bwd", _lib.load().gca_bwd(ctypes.byref(params), _p(q), _p(k), _p(v), _p(idx),
                                          _p(weight), _p(lse), _p(dout), _p(dq), _p(dk), _p(dv),
                                          _p(dscore), _p(workspace), workspace.numel(),
                                          _stream(stream)))


def gca_decode_workspace_size(n_landmarks: int, D: int, topk: int) -> int:
    return int(_lib.load().gca_decode_workspace_size(n_landmarks, D, topk))


def gca_decode_retrieve(landmarks, query_landmark, N, D, topk, dtype, off_by_one, score_scale,
                        idx, score, weight, workspace, stream=None):
    _check("gca_decode_retrieve", _lib.load().gca_decode_retrieve(
        _p(landmarks), _p(query_landmark), N, D, topk, dtype_code(dtype), int(bool(off_by_one)),
        float(score_scale), _p(idx), _p(score), _p(weight), _p(workspace), workspace.numel(),
        _stream(stream)))


def gca_decode_retrieve_noalloc(landmarks, query_landmark, N, D, topk, dtype, off_by_one,
                                score_scale, idx, score, weight, stream=None):
    """Decode retrieval without a workspace argument, for callers that may not
    allocate device memory (the library's own fixed device array is used)."""
    _check("gca_decode_retrieve_noalloc", _lib.load().gca_decode_retrieve_noalloc(
        _p(landmarks), _p(query_landmark), N, D, topk, dtype_code(dtype), int(bool(off_by_one)),
        float(score_scale), _p(idx), _p(score), _p(weight), _stream(stream)))


def _pa(t):
    """Pointer of a CUDA tensor, or of a pinned host tensor (device-addressable)."""
    if t.is_cuda:
        return _p(t)
    if not t.is_pinned():
        raise ValueError("offloaded caches must be in page-locked (pinned) host memory")
    if not t.is_contiguous():
        raise ValueError("GCA entry points take contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def gca_gather_chunks(src_k, src_v, n_src, chunk_bytes, idx, topk, dst_k, dst_v, dst_idx,
                      stream=None):
    _check("gca_gather_chunks", _lib.load().gca_gather_chunks(
        _pa(src_k), _pa(src_v), n_src, chunk_bytes, _p(idx), topk, _p(dst_k), _p(dst_v),
        _p(dst_idx), _stream(stream)))


def make_swa_params(*, B, L, H, d, window, dtype=torch.bfloat16, attn_scale=0.0) -> GcaSwaParams:
    return GcaSwaParams(B=B, L=L, H=H, d=d, window=window, dtype=dtype_code(dtype),
                        attn_scale=float(attn_scale))


def gca_swa_fwd(params: GcaSwaParams, q, k, v, o, lse, stream=None):
    _check("gca_swa_fwd", _lib.load().gca_swa_fwd(ctypes.byref(params), _p(q), _p(k), _p(v), _p(o),
                                                  _p(lse), _stream(stream)))


def swa_fwd(q, k, v, *, window, attn_scale=0.0, with_lse=True):
    """Sliding-window self-attention: q, k, v [B, L, H, d] -> (o, lse [B, L, H])."""
    B, L, H, d = q.shape
    p = make_swa_params(B=B, L=L, H=H, d=d, window=window, dtype=q.dtype, attn_scale=attn_scale)
    o = torch.empty_like(q)
    lse = torch.empty(B, L, H, dtype=torch.float32, device=q.device) if with_lse else None
    gca_swa_fwd(p, q, k, v, o, lse)
    return o, lse


def gca_swa_bwd_workspace_size(params: GcaSwaParams) -> int:
    return int(_lib.load().gca_swa_bwd_workspace_size(ctypes.byref(params)))


def gca_swa_bwd(params: GcaSwaParams, q, k, v, o, lse, dout, dq, dk, dv, workspace, stream=None):
    _check("gca_swa_bwd", _lib.load().gca_swa_bwd(
        ctypes.byref(params), _p(q), _p(k), _p(v), _p(o), _p(lse), _p(dout), _p(dq), _p(dk), _p(dv),
        _p(workspace), workspace.numel(), _stream(stream)))


def swa_bwd(q, k, v, o, lse, dout, *, window, attn_scale=0.0, workspace=None):
    """Gradients of the sliding-window self-attention: returns (dq, dk, dv)."""
    B, L, H, d = q.shape
    p = make_swa_params(B=B, L=L, H=H, d=d, window=window, dtype=q.dtype, attn_scale=attn_scale)
    if workspace is None:
        workspace = torch.empty(gca_swa_bwd_workspace_size(p), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    gca_swa_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, workspace)
    return dq, dk, dv


def gather_chunks(cache_k, cache_v, idx):
    """cache_k/v [n_chunks, S, H, d] (device or pinned host) -> compact
    pools [1, topk*S, H, d] on the device and the remapped idx [1, 1, topk]."""
    n, S, H, d = cache_k.shape
    topk = idx.numel()
    dev = idx.device
    dk = torch.empty(topk * S, H, d, dtype=cache_k.dtype, device=dev)
    dv = torch.empty_like(dk)
    di = torch.empty(topk, dtype=torch.int32, device=dev)
    chunk_bytes = S * H * d * cache_k.element_size()
    gca_gather_chunks(cache_k, cache_v, n, chunk_bytes, idx, topk, dk, dv, di)
    return dk.view(1, topk * S, H, d), dv.view(1, topk * S, H, d), di.view(1, 1, topk)


def gca_get_status(stream=None) -> int:
    return int(_lib.load().gca_get_status(_stream(stream)))


def gca_debug_stall_next_decode(wait_ns: int):
    """Test-only: the next decode launch on this thread withholds one stage and
    bounds its waits by ``wait_ns`` (include/gca_debug.h)."""
    _check("gca_debug_stall_next_decode", _lib.load().gca_debug_stall_next_decode(int(wait_ns)))


def gca_last_launch_count() -> int:
    return int(_lib.load().gca_last_launch_count())


def gca_synth_fill_hash(dst, seed: int, tensor_id: int, first_elem: int = 0, stream=None):
    _check("gca_synth_fill_hash", _lib.load().gca_synth_fill_hash(
        _p(dst), dst.numel(), dtype_code(dst.dtype), seed, tensor_id, first_elem, _stream(stream)))


# --- allocating helpers ----------------------------------------------------------------
def score_topk(landmarks, *, S, H, d, topk, off_by_one=False, include_self=False, score_scale=0.0):
    """landmarks [B, nC, D] -> idx int32, score fp32, weight fp32, each [B, nC, topk]."""
    B, nC, D = landmarks.shape
    p = make_params(B=B, Lq=nC * S, S=S, H=H, d=d, topk=topk, landmark_dim=D,
                    dtype=landmarks.dtype, off_by_one=off_by_one, include_self=include_self,
                    score_scale=score_scale)
    dev = landmarks.device
    idx = torch.empty(B, nC, topk, dtype=torch.int32, device=dev)
    score = torch.empty(B, nC, topk, dtype=torch.float32, device=dev)
    weight = torch.empty(B, nC, topk, dtype=torch.float32, device=dev)
    gca_score_topk(p, landmarks, idx, score, weight)
    return idx, score, weight


def score_topk_noisy(landmarks, noise, *, S, H, d, topk, off_by_one=False, include_self=False,
                     score_scale=0.0):
    """Like score_topk, selecting by score + noise (noise [B, nC, nC] fp32)."""
    B, nC, D = landmarks.shape
    p = make_params(B=B, Lq=nC * S, S=S, H=H, d=d, topk=topk, landmark_dim=D,
                    dtype=landmarks.dtype, off_by_one=off_by_one, include_self=include_self,
                    score_scale=score_scale)
    dev = landmarks.device
    idx = torch.empty(B, nC, topk, dtype=torch.int32, device=dev)
    score = torch.empty(B, nC, topk, dtype=torch.float32, device=dev)
    weight = torch.empty(B, nC, topk, dtype=torch.float32, device=dev)
    gca_score_topk_noisy(p, landmarks, noise, idx, score, weight)
    return idx, score, weight


def landmark_bwd(landmarks, idx, dscore, *, S, H, d, score_scale=0.0):
    """dLoss/dlandmarks [B, nC, D] from dLoss/dr."""
    B, nC, D = landmarks.shape
    p = make_params(B=B, Lq=nC * S, S=S, H=H, d=d, topk=idx.shape[-1], landmark_dim=D,
                    dtype=landmarks.dtype, score_scale=score_scale)
    ws = torch.empty(gca_landmark_bwd_workspace_size(p), dtype=torch.uint8, device=landmarks.device)
    dl = torch.empty_like(landmarks)
    gca_landmark_bwd(p, landmarks, idx, dscore, dl, ws)
    return dl


def fwd(q, k, v, idx, weight, *, S, attn_scale=0.0, with_lse=True):
    """q [B, Lq, H, d]; k, v [B, nP*S, H, d]; idx, weight [B, Lq/S, topk] -> (o, lse)."""
    B, Lq, H, d = q.shape
    topk = idx.shape[-1]
    p = make_params(B=B, Lq=Lq, S=S, H=H, d=d, topk=topk, n_pool_chunks=k.shape[1] // S,
                    dtype=q.dtype, attn_scale=attn_scale)
    o = torch.empty_like(q)
    lse = torch.empty(B, Lq, H, topk, dtype=torch.float32, device=q.device) if with_lse else None
    gca_fwd(p, q, k, v, idx, weight, o, lse)
    return o, lse


def bwd(q, k, v, idx, weight, lse, dout, *, S, attn_scale=0.0, workspace=None):
    """Returns (dq, dk, dv, dscore)."""
    B, Lq, H, d = q.shape
    topk = idx.shape[-1]
    p = make_params(B=B, Lq=Lq, S=S, H=H, d=d, topk=topk, n_pool_chunks=k.shape[1] // S,
                    dtype=q.dtype, attn_scale=attn_scale)
    need = gca_bwd_workspace_size(p)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dscore = torch.empty(B, Lq // S, topk, dtype=torch.float32, device=q.device)
    gca_bwd(p, q, k, v, idx, weight, lse, dout, dq, dk, dv, dscore, workspace)
    return dq, dk, dv, dscore


def decode_retrieve(landmarks, query_landmark, *, topk, off_by_one=False, score_scale=0.0,
                    workspace=None):
    """landmarks [N, D], query_landmark [D] -> idx, score, weight [topk]."""
    N, D = landmarks.shape
    need = gca_decode_workspace_size(N, D, topk)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=landmarks.device)
    dev = landmarks.device
    idx = torch.empty(topk, dtype=torch.int32, device=dev)
    score = torch.empty(topk, dtype=torch.float32, device=dev)
    weight = torch.empty(topk, dtype=torch.float32, device=dev)
    gca_decode_retrieve(landmarks, query_landmark, N, D, topk, landmarks.dtype, off_by_one,
                        score_scale, idx, score, weight, workspace)
    return idx, score, weight
