"""Seeded synthetic inputs for the GCA workloads.

This module generates inputs only: it holds none of the method's arithmetic,
so both the CUDA path and the fp64 oracle can be fed from it.  The shapes and
value distributions follow the DRT setup of "Efficient Length-Generalizable
Attention via Causal Retrieval for Long-Context Language Modeling" (App. A:
12 heads, 768-dim; section 4.1.2: 64-token chunks, 8 retrieved chunks) and the
five named workloads below.  Landmark vectors are small integers so that
every relevance score is exact in fp32 and fp64 and the retrieved indices are
uniquely defined.

Generation order inside one seed: landmarks, Q, K, V (``torch.Generator`` on
the CPU, fixed seed), then dO from the separate upstream-gradient seed.
bf16 tensors are rounded from fp32 with round-to-nearest-even by torch.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int            # query tokens per batch row (also the K/V pool length in training)
    S: int            # chunk size
    H: int
    d: int
    topk: int
    off_by_one: bool
    dtype: str        # "f32" or "bf16"
    lm_range: int     # landmarks uniform integers in [-lm_range, lm_range]
    qkv_std: float    # Q/K/V ~ N(0, qkv_std^2)
    seed: int
    dout_seed: int    # seed of the upstream gradient dO (-1: forward-only workload)
    include_self: bool = False

    @property
    def nC(self) -> int:
        return self.L // self.S

    @property
    def D(self) -> int:
        return self.H * self.d


def _wl(name, **kw):
    return Workload(name=name, **kw)


#: The named workloads.  ``tiny_fp32`` is the small case the oracle finishes in
#: seconds; ``gpt2s_fwd_b4`` / ``gpt2s_fwdbwd_b8`` are the GPT-2-small-shaped
#: 16K-context cases; ``long64k_*`` is the chunk-size / top-k sweep at 64K.
WORKLOADS = {
    "tiny_fp32": _wl("tiny_fp32", B=1, L=1024, S=64, H=4, d=32, topk=2, off_by_one=False,
                     dtype="f32", lm_range=8, qkv_std=1.0, seed=0, dout_seed=0),
    "gpt2s_fwd_b4": _wl("gpt2s_fwd_b4", B=4, L=16384, S=64, H=12, d=64, topk=8, off_by_one=True,
                        dtype="bf16", lm_range=4, qkv_std=1.0 / 8.0, seed=1, dout_seed=-1),
    "gpt2s_fwdbwd_b8": _wl("gpt2s_fwdbwd_b8", B=8, L=16384, S=64, H=12, d=64, topk=8,
                           off_by_one=False, dtype="bf16", lm_range=4, qkv_std=1.0 / 8.0,
                           seed=1, dout_seed=2),
}
for _S in (64, 128):
    for _k in (4, 8, 16):
        _n = "long64k_S%d_k%d" % (_S, _k)
        WORKLOADS[_n] = _wl(_n, B=1, L=65536, S=_S, H=12, d=64, topk=_k, off_by_one=False,
                            dtype="bf16", lm_range=4, qkv_std=1.0 / 8.0, seed=3, dout_seed=3)


def make(wl: Workload, *, B: int | None = None, L: int | None = None, with_dout: bool = True):
    """Generate the inputs of ``wl`` on the CPU.

    ``B`` / ``L`` may shrink the batch or the context (same seed, same
    distributions) for parity cases that the oracle finishes quickly.
    Returns a dict of CPU tensors: lm [B, nC, D], q/k/v [B, L, H, d] and,
    when the workload has an upstream gradient, dout [B, L, H, d].
    """
    B = wl.B if B is None else B
    L = wl.L if L is None else L
    assert L % wl.S == 0
    nC, H, d, D = L // wl.S, wl.H, wl.d, wl.H * wl.d
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(wl.seed)
    lm = torch.randint(-wl.lm_range, wl.lm_range + 1, (B, nC, D), generator=g).to(dt)
    q = (torch.randn(B, L, H, d, generator=g) * wl.qkv_std).to(dt)
    k = (torch.randn(B, L, H, d, generator=g) * wl.qkv_std).to(dt)
    v = (torch.randn(B, L, H, d, generator=g) * wl.qkv_std).to(dt)
    out = {"lm": lm, "q": q, "k": k, "v": v}
    if with_dout and wl.dout_seed >= 0:
        g2 = torch.Generator().manual_seed(wl.dout_seed)
        if wl.dout_seed == wl.seed:
            g2 = g  # same stream, continued after V
        out["dout"] = torch.randn(B, L, H, d, generator=g2).to(dt)
    return out


def random_case(seed: int, *, B, nC, S, H, d, topk, lm_range=3, dtype="f32", qkv_std=1.0):
    """A small random case (for edge-case and ragged-shape tests)."""
    wl = Workload(name="random", B=B, L=nC * S, S=S, H=H, d=d, topk=topk, off_by_one=False,
                  dtype=dtype, lm_range=lm_range, qkv_std=qkv_std, seed=seed, dout_seed=seed)
    return make(wl)


# --------------------------------------------------------------------------
# Decode workload: 262144 landmarks (a 16M-token context at 64-token chunks)
# plus a per-chunk K/V cache [N, S, H, d] that is too large to generate on the
# host.  Its values come from a stateless counter-based generator, SplitMix64
# (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
# OOPSLA 2014), so the device can fill the cache and the host can regenerate
# any chunk of it bit-for-bit.
# --------------------------------------------------------------------------
DECODE = dict(N=262144, D=768, S=64, H=12, d=64, topk=8, off_by_one=False, lm_range=4, seed=4)
_M64 = (1 << 64) - 1


def splitmix64_np(x: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser applied to each uint64 counter value."""
    with np.errstate(over="ignore"):
        z = (x.astype(np.uint64) + np.uint64(0x9E3779B97F4A7C15))
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def hash_values_np(seed: int, tensor_id: int, elem: np.ndarray) -> np.ndarray:
    """Cache value of each element index: (u0+u1+u2+u3 - 14) / 32, where the u_i
    are the four low 3-bit fields of SplitMix64((seed << 56) ^ (tensor_id << 48) ^ elem).
    Values are multiples of 1/32 in [-14/32, 14/32]; every one is exact in bf16."""
    ctr = (np.uint64(seed) << np.uint64(56)) ^ (np.uint64(tensor_id) << np.uint64(48)) \
        ^ elem.astype(np.uint64)
    h = splitmix64_np(ctr)
    s = np.zeros(h.shape, dtype=np.int64)
    for i in range(4):
        s += ((h >> np.uint64(3 * i)) & np.uint64(7)).astype(np.int64)
    return (s - 14).astype(np.float64) / 32.0


def decode_inputs(N: int | None = None, seed: int | None = None):
    """Host part of the decode workload: landmarks [N, D] and the query landmark [D]
    (bf16 holding integers in [-4, 4]), and the 64-token query chunk q [S, H, d]."""
    p = dict(DECODE)
    N = p["N"] if N is None else N
    seed = p["seed"] if seed is None else seed
    g = torch.Generator().manual_seed(seed)
    r = p["lm_range"]
    lm = torch.randint(-r, r + 1, (N, p["D"]), generator=g).to(torch.bfloat16)
    ql = torch.randint(-r, r + 1, (p["D"],), generator=g).to(torch.bfloat16)
    q = (torch.randn(p["S"], p["H"], p["d"], generator=g) * 0.125).to(torch.bfloat16)
    return {"lm": lm, "ql": ql, "q": q}


def decode_cache_chunk_np(seed: int, tensor_id: int, chunk: int, S: int, H: int, d: int):
    """Regenerate one chunk [S, H, d] of the device-filled cache (tensor_id 0 = K, 1 = V)."""
    per = S * H * d
    elem = np.arange(chunk * per, (chunk + 1) * per, dtype=np.uint64)
    return hash_values_np(seed, tensor_id, elem).reshape(S, H, d)

