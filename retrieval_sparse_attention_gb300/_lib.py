"""ctypes view of the C ABI in include/gca.h (libgca.so, built in-tree).

Loading never falls back to anything: if the library is missing or cannot be
loaded, every call raises.  Build it with ``python -c "import __graft_entry__
as g; g.build()"`` or ``python retrieval_sparse_attention_gb300/build.py``.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgca.so")

GCA_BF16 = 0
GCA_F32 = 1

STATUS_NAMES = {0: "GCA_OK", 1: "GCA_ERR_INVALID_ARG", 2: "GCA_ERR_UNSUPPORTED",
                3: "GCA_ERR_WORKSPACE", 4: "GCA_ERR_CUDA", 5: "GCA_ERR_TIMEOUT",
                6: "GCA_ERR_DEVICE_INDEX"}

#: every symbol the headers under include/ declare
EXPORTED = ("gca_score_topk", "gca_fwd", "gca_bwd_workspace_size", "gca_bwd",
            "gca_decode_workspace_size", "gca_decode_retrieve", "gca_get_status",
            "gca_status_string", "gca_last_launch_count", "gca_synth_fill_hash",
            "gca_prof_enable", "gca_prof_read", "gca_decode_retrieve_noalloc",
            "gca_score_topk_noisy", "gca_landmark_bwd_workspace_size", "gca_landmark_bwd",
            "gca_gather_chunks", "gca_swa_fwd", "gca_swa_bwd_workspace_size", "gca_swa_bwd",
            "gca_debug_stall_next_decode")


class GcaParams(ctypes.Structure):
    """Mirror of gca_params_t."""
    _fields_ = [("B", ctypes.c_int), ("Lq", ctypes.c_int), ("S", ctypes.c_int),
                ("H", ctypes.c_int), ("d", ctypes.c_int), ("topk", ctypes.c_int),
                ("n_pool_chunks", ctypes.c_int), ("landmark_dim", ctypes.c_int),
                ("dtype", ctypes.c_int), ("softmax_off_by_one", ctypes.c_int),
                ("include_self", ctypes.c_int), ("score_scale", ctypes.c_float),
                ("attn_scale", ctypes.c_float)]


class GcaSwaParams(ctypes.Structure):
    """Mirror of gca_swa_params_t."""
    _fields_ = [("B", ctypes.c_int), ("L", ctypes.c_int), ("H", ctypes.c_int), ("d", ctypes.c_int),
                ("window", ctypes.c_int), ("dtype", ctypes.c_int), ("attn_scale", ctypes.c_float)]


class GcaError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s returned %s (%d)" % (fn, STATUS_NAMES.get(code, "?"), code))
        self.code = code


_lib = None


def load() -> ctypes.CDLL:
    """Load libgca.so (raises OSError if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError("GCA CUDA library not built: %s is missing" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        P = ctypes.POINTER(GcaParams)
        sig = {
            "gca_score_topk": ([P, vp, vp, vp, vp, vp], i32),
            "gca_fwd": ([P, vp, vp, vp, vp, vp, vp, vp, vp], i32),
            "gca_score_topk_noisy": ([P, vp, vp, vp, vp, vp, vp], i32),
            "gca_landmark_bwd_workspace_size": ([P], sz),
            "gca_landmark_bwd": ([P, vp, vp, vp, vp, vp, sz, vp], i32),
            "gca_bwd_workspace_size": ([P], sz),
            "gca_bwd": ([P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
            "gca_decode_workspace_size": ([i32, i32, i32], sz),
            "gca_decode_retrieve": ([vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, sz, vp],
                                    i32),
            "gca_decode_retrieve_noalloc": ([vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp],
                                            i32),
            "gca_gather_chunks": ([vp, vp, i32, sz, vp, i32, vp, vp, vp, vp], i32),
            "gca_swa_fwd": ([ctypes.POINTER(GcaSwaParams), vp, vp, vp, vp, vp, vp], i32),
            "gca_swa_bwd_workspace_size": ([ctypes.POINTER(GcaSwaParams)], sz),
            "gca_swa_bwd": ([ctypes.POINTER(GcaSwaParams)] + [vp] * 10 + [sz, vp], i32),
            "gca_get_status": ([vp], i32),
            "gca_status_string": ([i32], ctypes.c_char_p),
            "gca_last_launch_count": ([], i32),
            "gca_debug_stall_next_decode": ([ctypes.c_uint64], i32),
            "gca_synth_fill_hash": ([vp, sz, i32, ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_uint64, vp], i32),
            "gca_prof_enable": ([i32], None),
            "gca_prof_read": ([i32, vp, vp, vp], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib
