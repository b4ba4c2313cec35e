"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol the headers declare, and rejects bad arguments with the
documented status codes before touching the device."""
import ctypes
import glob
import os
import re

import pytest

from retrieval_sparse_attention_gb300 import _lib
from retrieval_sparse_attention_gb300._lib import GcaParams

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    from retrieval_sparse_attention_gb300 import build
    build.build()
    return _lib.load()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(gca_[a-z0-9_]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert {"gca_score_topk", "gca_fwd", "gca_bwd", "gca_decode_retrieve"} <= names
    for n in names:
        assert hasattr(lib, n), "libgca.so does not export %s" % n
    assert names <= set(_lib.EXPORTED) | set(names)


def params(**kw):
    base = dict(B=2, Lq=1024, S=64, H=12, d=64, topk=8, n_pool_chunks=16, landmark_dim=0,
                dtype=0, softmax_off_by_one=0, include_self=0, score_scale=0.0, attn_scale=0.0)
    base.update(kw)
    return GcaParams(**base)


FAKE = ctypes.c_void_p(0x10000)      # aligned, never dereferenced: validation fails first


def fwd(lib, p, q=FAKE, o=FAKE):
    return lib.gca_fwd(ctypes.byref(p) if p is not None else None, q, FAKE, FAKE, FAKE, FAKE, o,
                       None, None)


def test_fwd_validation(lib):
    assert fwd(lib, None) == INVALID
    assert fwd(lib, params(), q=None) == INVALID                     # null tensor
    assert fwd(lib, params(), o=ctypes.c_void_p(0x10008)) == INVALID  # misaligned
    assert fwd(lib, params(Lq=1000)) == INVALID                      # not a multiple of S
    assert fwd(lib, params(n_pool_chunks=0)) == INVALID
    assert fwd(lib, params(topk=0)) == INVALID
    assert fwd(lib, params(dtype=7)) == INVALID
    assert fwd(lib, params(score_scale=-1.0)) == INVALID
    assert fwd(lib, params(topk=33)) == UNSUPPORTED
    assert fwd(lib, params(d=48)) == UNSUPPORTED                     # bf16 path: d in {32, 64, 128}
    assert fwd(lib, params(d=16)) == UNSUPPORTED
    assert fwd(lib, params(d=256)) == UNSUPPORTED
    assert fwd(lib, params(S=32)) == UNSUPPORTED
    assert fwd(lib, params(dtype=1, d=128, S=64)) == UNSUPPORTED


def test_bwd_workspace_and_validation(lib):
    p = params()
    n = lib.gca_bwd_workspace_size(ctypes.byref(p))
    # delta [B,Lq,H,k] + dw partials [B,nQ,H,k] fp32 + the inverse index
    assert n >= 4 * (2 * 1024 * 12 * 8 + 2 * 16 * 12 * 8) + 4 * (2 * 16 + 2 * 17 + 2 * 16 * 8)
    assert n % 256 == 0
    assert lib.gca_bwd_workspace_size(None) == 0
    args = [FAKE] * 11
    rc = lib.gca_bwd(ctypes.byref(p), *args, None, n, None)
    assert rc == WORKSPACE
    rc = lib.gca_bwd(ctypes.byref(p), *args, ctypes.c_void_p(0x10000), n - 256, None)
    assert rc == WORKSPACE
    rc = lib.gca_bwd(ctypes.byref(p), *args, ctypes.c_void_p(0x10080), n, None)   # not 256-aligned
    assert rc == WORKSPACE


def test_decode_validation(lib):
    n = lib.gca_decode_workspace_size(262144, 768, 8)
    assert 0 < n <= 256 + 2048 * 8 * 8
    assert lib.gca_decode_workspace_size(0, 768, 8) == 0
    assert lib.gca_decode_workspace_size(10, 768, 33) == 0

    def call(N=1000, D=768, k=8, dt=0, ws=FAKE, nbytes=1 << 20):
        return lib.gca_decode_retrieve(FAKE, FAKE, N, D, k, dt, 0, 0.0, FAKE, FAKE, FAKE, ws,
                                       nbytes, None)
    assert call(N=0) == INVALID
    assert call(dt=3) == INVALID
    assert call(k=40) == UNSUPPORTED
    assert call(D=13) == UNSUPPORTED          # rows must be whole 16-byte vectors
    assert call(ws=None) == WORKSPACE
    assert call(nbytes=16) == WORKSPACE


def test_score_topk_validation(lib):
    p = params()
    assert lib.gca_score_topk(ctypes.byref(p), None, FAKE, FAKE, FAKE, None) == INVALID
    assert lib.gca_score_topk(ctypes.byref(params(landmark_dim=9000)), FAKE, FAKE, FAKE, FAKE,
                              None) == UNSUPPORTED


def test_debug_stall_validation(lib):
    assert lib.gca_debug_stall_next_decode(0) == INVALID
    assert lib.gca_debug_stall_next_decode(999) == INVALID
    assert lib.gca_debug_stall_next_decode(2_000_000_000) == INVALID


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.gca_status_string(code).decode() == name


def test_product_path_has_no_cpu_fallback():
    # The binding must not import the oracle or fall back to any CPU path.
    import retrieval_sparse_attention_gb300.api as api_mod
    src = open(api_mod.__file__).read() + open(_lib.__file__).read()
    assert "oracle" not in src.replace("no fallback", "")


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libgca.so"))
    with pytest.raises(OSError):
        _lib.load()
