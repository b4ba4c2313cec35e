#!/usr/bin/env python
"""Benchmark of the GCA hot path on GB300.

One step = the whole hot path on one batch of the GPT-2-small-shaped 16K
workload (B=8, L=16384, S=64, H=12, d=64, top-k=8, bf16, vanilla softmax):
gca_score_topk -> gca_fwd -> gca_bwd.  The metric is query tokens per second
(B*L per step, summed over ranks).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 it is launched under torch.distributed.run, one rank per GPU; the
batch rows of different ranks are independent (weak scaling, no collective
on the data path).  ``--impl reference`` times the fp64 CPU oracle on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "gpt2s_fwdbwd_b8"
METRIC = "GCA fwd+bwd query-tokens/s at 16K ctx; % of HBM/tensor roofline (1 GB300)"
UNIT = "query-tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the forward-only and decode lines")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--case", default=None, choices=sorted(CASES),
                    help="profiling mode: run only this path (warm-up + steps), print timings")
    return ap.parse_args()


#: small cases for profiler captures: (workload, batch rows, with backward)
CASES = {"fwd_b4": ("gpt2s_fwd_b4", 4, False), "fwdbwd_b4": ("gpt2s_fwdbwd_b8", 4, True),
         "fwdbwd_b8": ("gpt2s_fwdbwd_b8", 8, True), "long_s64_k16": ("long64k_S64_k16", 1, True),
         "long_s128_k8": ("long64k_S128_k8", 1, True), "decode": (None, 1, False),
         "swa": ("swa", 8, False), "swa_bwd": ("swa", 8, True),
         "swa_b2": ("swa", 2, False), "swa_bwd_b2": ("swa", 2, True)}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 100 ms.

    Sampling starts before the timed region (the first sample is awaited, up to
    3 s, so the sampler is live when the region starts) and stops 150 ms after
    it.  Each sample is stamped on arrival; ``mark_start`` / ``mark_end`` bracket
    the timed region.  The median SM clock is taken over the samples that arrived
    inside the region when there are any, else over all of them; the throttle
    reasons are those active in any sample.
    """

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, first_wait_s: float = 3.0):
        self.idx = gpu_index
        self.proc = None
        self.lines = []          # (arrival time, line)
        self.first_wait_s = first_wait_s
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.idx)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        deadline = time.monotonic() + self.first_wait_s
        while (self.proc is not None and not self.lines and self.proc.poll() is None
               and time.monotonic() < deadline):
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        samples, reasons = [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in list(self.lines):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                samples.append((ts, float(f[1]), float(f[2])))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        inside = [x for x in samples
                  if self.t0 is not None and self.t1 is not None and self.t0 <= x[0] <= self.t1]
        use = inside or samples
        return {"sm_mhz": statistics.median(x[1] for x in use) if use else None,
                "sm_max_mhz": max(x[2] for x in samples) if samples else None,
                "reasons": sorted(reasons), "samples": len(samples),
                "samples_in_region": len(inside)}


# --------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms: float, device=None) -> float:
    """Largest per-rank time (the job finishes when its slowest rank does)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank_step: int, steps: int, world: int, ms_max: float) -> float:
    """Whole-job query tokens per second: every rank processes its own batch."""
    return world * tokens_per_rank_step * steps / (ms_max / 1e3)


def read_prof(lib):
    import ctypes
    n = 32
    names = ctypes.create_string_buffer(64 * n)
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int * n)()
    k = lib.gca_prof_read(n, names, ms, cnt)
    out = {}
    for i in range(max(k, 0)):
        nm = names.raw[64 * i:64 * (i + 1)].split(b"\0")[0].decode()
        out[nm] = (float(ms[i]), int(cnt[i]))
    return out


def traffic_table():
    """Per-launch DRAM bytes from the committed ncu summary (kernel -> bytes)."""
    p = os.path.join(ROOT, "profiles", "ncu_dram_traffic.txt")
    t = {}
    if os.path.exists(p):
        for ln in open(p):
            f = ln.split()
            if len(f) >= 3 and not ln.startswith("#"):
                t[(f[0], f[1])] = float(f[2])
    return t


def alg_bytes(wl, U, H, D, k):
    """Algorithmic bytes per launch of each kernel (bf16 tensors, fp32 lse/delta).

    U = valid (batch row, query chunk, slot) units.  Each unit gathers one
    retrieved chunk: 2 tiles of S x D (K and V, or Q and dO) of 2 bytes."""
    B, L, S = wl.B, wl.L, wl.S
    tok = B * L * D * 2                       # one [B, L, H, d] bf16 tensor
    lse = B * L * H * k * 4
    gather = U * 2 * S * D * 2
    return {
        "fwd": gather + 2 * tok + lse,                              # K/V gather, Q in, O out, lse out
        "bwd_q": gather + 3 * tok + 2 * lse,                        # K/V gather, Q, dO in, dQ out; lse in, delta out
        "bwd_kv": gather + U * 2 * S * H * 4 + 4 * tok,             # Q/dO gather + lse/delta rows; K, V in; dK, dV out
    }


# --------------------------------------------------------------------------- ours
def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from retrieval_sparse_attention_gb300 import _lib, api, inputs

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = _lib.load()
    wl = inputs.WORKLOADS[WORKLOAD]
    B, L, S, H, d, k = wl.B, wl.L, wl.S, wl.H, wl.d, wl.topk
    D = H * d
    x = inputs.make(wl)
    host = {n: t.pin_memory() for n, t in x.items()}
    g = {n: t.to(dev) for n, t in x.items()}
    p = api.make_params(B=B, Lq=L, S=S, H=H, d=d, topk=k, dtype=torch.bfloat16,
                        off_by_one=wl.off_by_one)
    idx = torch.empty(B, wl.nC, k, dtype=torch.int32, device=dev)
    r = torch.empty(B, wl.nC, k, dtype=torch.float32, device=dev)
    w = torch.empty_like(r)
    o = torch.empty_like(g["q"])
    lse = torch.empty(B, L, H, k, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(o), torch.empty_like(o), torch.empty_like(o)
    ds = torch.empty_like(r)
    wsb = torch.empty(api.gca_bwd_workspace_size(p), dtype=torch.uint8, device=dev)
    launches = [0]

    def step(t):
        api.gca_score_topk(p, t["lm"], idx, r, w)
        n = api.gca_last_launch_count()
        api.gca_fwd(p, t["q"], t["k"], t["v"], idx, w, o, lse)
        n += api.gca_last_launch_count()
        api.gca_bwd(p, t["q"], t["k"], t["v"], idx, w, lse, t["dout"], dq, dk, dv, ds, wsb)
        n += api.gca_last_launch_count()
        launches[0] += n

    for _ in range(args.warmup):
        step(g)
    torch.cuda.synchronize()
    assert api.gca_get_status() == 0, "device-side error during warm-up"
    U = int((idx >= 0).sum().item())

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- timed region: K steps, device events on the launching stream
    launches[0] = 0
    lib.gca_prof_read(0, None, None, None)
    lib.gca_prof_enable(1)
    barrier()
    with ClockSampler(local) as clk:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        clk.mark_start()
        e0.record()
        for _ in range(args.steps):
            step(g)
        e1.record()
        barrier()
        clk.mark_end()
    lib.gca_prof_enable(0)
    ms = e0.elapsed_time(e1)
    prof = read_prof(lib)
    n_launch = launches[0]
    assert api.gca_get_status() == 0, "device-side error in the timed region"
    ms_max = max_over_ranks(ms, dev)
    value = job_throughput(B * L, args.steps, ws, ms_max)

    # ---- end to end through the public API with host buffers: every step copies
    # its inputs in from pinned host memory and its results (O, dQ, dK, dV,
    # d-score) back out.  Two device buffer sets and separate copy streams let
    # step i+1's inputs arrive while step i computes and step i-1 drains.
    names_out = ("o", "dq", "dk", "dv", "ds")
    out_host = [{n: torch.empty(t.shape, dtype=t.dtype).pin_memory()
                 for n, t in zip(names_out, (o, dq, dk, dv, ds))} for _ in range(2)]
    dbuf = [{n: torch.empty_like(t) for n, t in g.items()} for _ in range(2)]
    dout_buf = [{n: torch.empty_like(t) for n, t in zip(names_out, (o, dq, dk, dv, ds))}
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host[0].values())
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n_steps):
        for i in range(n_steps):
            k = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[k])          # step i-2 has finished with dbuf[k]
                for n in dbuf[k]:
                    dbuf[k][n].copy_(host[n], non_blocking=True)
                ev_in[k].record(s_in)
            comp.wait_event(ev_in[k])
            if i >= 2:
                comp.wait_event(ev_out[k])               # step i-2's results have left dout_buf[k]
            ob = dout_buf[k]
            api.gca_score_topk(p, dbuf[k]["lm"], idx, r, w)
            api.gca_fwd(p, dbuf[k]["q"], dbuf[k]["k"], dbuf[k]["v"], idx, w, ob["o"], lse)
            api.gca_bwd(p, dbuf[k]["q"], dbuf[k]["k"], dbuf[k]["v"], idx, w, lse, dbuf[k]["dout"],
                        ob["dq"], ob["dk"], ob["dv"], ob["ds"], wsb)
            ev_done[k].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[k])
                for n in names_out:
                    out_host[k][n].copy_(ob[n], non_blocking=True)
                ev_out[k].record(s_out)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    t_start = time.perf_counter()
    e2e_run(args.e2e_steps)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t_start) * 1e3, dev)
    e2e_value = job_throughput(B * L, args.e2e_steps, ws, e2e_ms)
    # the last step's results arrived in host memory
    assert torch.isfinite(out_host[(args.e2e_steps - 1) & 1]["ds"]).all()

    # ---- roofline of the dominant kernel
    hbm, tflops, src = peaks()
    ab = alg_bytes(wl, U, H, D, k)
    total = sum(v[0] for v in prof.values()) or 1.0
    dom = max(prof.items(), key=lambda kv: kv[1][0])
    dom_name, (dom_ms, dom_n) = dom
    fam = "bwd_kv" if "kv" in dom_name else ("bwd_q" if "bwd_q" in dom_name else
                                             ("fwd" if "fwd" in dom_name else None))
    avg_s = dom_ms / dom_n / 1e3
    roof = None
    if fam is not None:
        achieved = ab[fam] / avg_s / 1e9
        tr = traffic_table().get((dom_name, WORKLOAD))
        roof = {"kernel": dom_name, "bound": "hbm", "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % src if src == "measured" else src,
                "traffic": tr, "alg_bytes_per_launch": ab[fam],
                "avg_launch_ms": round(dom_ms / dom_n, 4)}
    kernels = {n: {"ms_total": round(v[0], 3), "launches": v[1], "share": round(v[0] / total, 4),
                   "ms_per_launch": round(v[0] / v[1], 4)} for n, v in sorted(prof.items())}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; integer landmarks in [-4,4], Q/K/V ~ N(0,1/64), dO ~ N(0,1))",
        "config": {"workload": WORKLOAD, "B": B, "L": L, "S": S, "H": H, "d": d, "topk": k,
                   "softmax": "vanilla", "step": "gca_score_topk + gca_fwd + gca_bwd",
                   "valid_units": U, "parallelism": "replicas" if ws == 1 else "dp%d" % ws,
                   "l2": "inputs %.2f GB > 129 MB L2; no flush" % (
                       sum(t.numel() * t.element_size() for t in g.values()) / 1e9)},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "timing": "host wall clock around K pipelined steps (copy-in, compute, copy-out "
                          "on three streams), synchronised on both sides"},
        "gpu_launches": n_launch,
        "roofline": roof,
        "kernels": kernels,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_extra:
        line["extra"] = extra_workloads(lib, api, inputs, dev, hbm, tflops)
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def extra_workloads(lib, api, inputs, dev, hbm, tflops):
    """gca_fwd alone on the B=4 off-by-one workload, and decode retrieval over
    262144 landmarks followed by gca_fwd on the 51.5 GB K/V cache."""
    import torch
    out = {}
    wl = inputs.WORKLOADS["gpt2s_fwd_b4"]
    x = {n: t.to(dev) for n, t in inputs.make(wl, with_dout=False).items()}
    idx, r, w = api.score_topk(x["lm"], S=wl.S, H=wl.H, d=wl.d, topk=wl.topk, off_by_one=True)
    o, lse = api.fwd(x["q"], x["k"], x["v"], idx, w, S=wl.S)
    torch.cuda.synchronize()
    U = int((idx >= 0).sum().item())
    n = 20
    for _ in range(3):
        api.fwd(x["q"], x["k"], x["v"], idx, w, S=wl.S)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        api.fwd(x["q"], x["k"], x["v"], idx, w, S=wl.S)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    D = wl.H * wl.d
    ab = alg_bytes(wl, U, wl.H, D, wl.topk)["fwd"]
    out["gpt2s_fwd_b4"] = {"kernel": "gca_fwd", "query_tokens_per_s": round(wl.B * wl.L / (ms / 1e3), 1),
                           "ms": round(ms, 4), "valid_units": U,
                           "roofline": {"bound": "hbm", "achieved": round(ab / ms / 1e6, 1), "peak": hbm,
                                        "unit": "GB/s", "frac": round(ab / ms / 1e6 / hbm, 4)}}
    del x, o, lse
    # decode: 16M-token context
    p = inputs.DECODE
    hx = inputs.decode_inputs()
    lm, ql, q = hx["lm"].to(dev), hx["ql"].to(dev), hx["q"].to(dev)
    N, Dd, kk = p["N"], p["D"], p["topk"]
    wsb = torch.empty(api.gca_decode_workspace_size(N, Dd, kk), dtype=torch.uint8, device=dev)
    for _ in range(3):
        api.decode_retrieve(lm, ql, topk=kk, workspace=wsb)
    e0.record()
    for _ in range(n):
        api.decode_retrieve(lm, ql, topk=kk, workspace=wsb)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    byts = N * Dd * 2 + Dd * 2
    dec = {"kernel": "gca_decode_retrieve", "N": N, "D": Dd, "topk": kk, "us": round(ms * 1e3, 2),
           "roofline": {"bound": "hbm", "achieved": round(byts / ms / 1e6, 1), "peak": hbm, "unit": "GB/s",
                        "frac": round(byts / ms / 1e6 / hbm, 4)}}
    # decode + forward over the HBM-resident cache
    try:
        cache_k = torch.empty(N * p["S"], p["H"], p["d"], dtype=torch.bfloat16, device=dev)
        cache_v = torch.empty_like(cache_k)
        api.gca_synth_fill_hash(cache_k, p["seed"], 0)
        api.gca_synth_fill_hash(cache_v, p["seed"], 1)
        qq = q.view(1, p["S"], p["H"], p["d"])
        kc, vc = cache_k.view(1, N * p["S"], p["H"], p["d"]), cache_v.view(1, N * p["S"], p["H"], p["d"])

        def dstep():
            di, dr, dw = api.decode_retrieve(lm, ql, topk=kk, workspace=wsb)
            api.fwd(qq, kc, vc, di.view(1, 1, kk), dw.view(1, 1, kk), S=p["S"])
        for _ in range(3):
            dstep()
        e0.record()
        for _ in range(n):
            dstep()
        e1.record()
        torch.cuda.synchronize()
        dec["retrieve_plus_fwd_us"] = round(e0.elapsed_time(e1) / n * 1e3, 2)
        dec["cache_gb"] = round(2 * cache_k.numel() * 2 / 1e9, 2)
        del cache_k, cache_v
    except RuntimeError as exc:           # out of device memory on a smaller part
        dec["retrieve_plus_fwd_us"] = None
        dec["cache_error"] = str(exc)[:120]
    out["decode_16m"] = dec
    out.update(sweep_rows(lib, api, inputs, dev, hbm))
    out.update(next_rows(api, inputs, dev, hbm))
    x = swa_inputs(dev)
    us = _event_us(lambda i=0: api.swa_fwd(x[0], x[1], x[2], window=SWA_WINDOW), n=20)
    out["swa_fwd_b8_16k"] = {"kernel": "gca_swa_fwd", "B": 8, "L": 16384, "H": 12, "d": 64,
                             "window": SWA_WINDOW, "us": round(us, 2),
                             "query_tokens_per_s": round(8 * 16384 / (us / 1e6), 1),
                             "roofline": swa_roofline(8, 16384, 12, 64, SWA_WINDOW, us / 1e3, hbm, tflops)}
    o, lse = api.swa_fwd(x[0], x[1], x[2], window=SWA_WINDOW)
    g = swa_inputs(dev, seed=12)[0] * 8
    us = _event_us(lambda i=0: api.swa_bwd(x[0], x[1], x[2], o, lse, g, window=SWA_WINDOW), n=10)
    out["swa_bwd_b8_16k"] = {"kernel": "gca_swa_bwd", "B": 8, "L": 16384, "H": 12, "d": 64,
                             "window": SWA_WINDOW, "us": round(us, 2),
                             "roofline": swa_roofline(8, 16384, 12, 64, SWA_WINDOW, us / 1e3, hbm, tflops,
                                                      backward=True)}
    del x, o, lse, g
    return out


def sweep_rows(lib, api, inputs, dev, hbm, steps=10, warm=3):
    """The chunk-size / top-k sweep at long context: B=1, L=65536, H=12, d=64,
    S in {64, 128}, top-k in {4, 8, 16}, vanilla softmax, one fwd+bwd step
    (gca_score_topk + gca_fwd + gca_bwd) per point.  Each row gives query
    tokens/s, the step against its gathered-bytes roofline (three gathers of
    2 S D bf16 per valid unit: K/V in the forward, K/V and Q/dO in the
    backward) and every kernel against its own algorithmic bytes."""
    import torch
    out = {}
    for S in (64, 128):
        base = inputs.WORKLOADS["long64k_S%d_k4" % S]
        x = {n: t.to(dev) for n, t in inputs.make(base).items()}
        B, L, H, d = base.B, base.L, base.H, base.d
        D, nC = H * d, L // S
        for k in (4, 8, 16):
            wl = inputs.WORKLOADS["long64k_S%d_k%d" % (S, k)]
            p = api.make_params(B=B, Lq=L, S=S, H=H, d=d, topk=k, dtype=torch.bfloat16)
            idx = torch.empty(B, nC, k, dtype=torch.int32, device=dev)
            r, w, ds = (torch.empty(B, nC, k, dtype=torch.float32, device=dev) for _ in range(3))
            o, dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(4))
            lse = torch.empty(B, L, H, k, dtype=torch.float32, device=dev)
            wsb = torch.empty(api.gca_bwd_workspace_size(p), dtype=torch.uint8, device=dev)

            def step():
                api.gca_score_topk(p, x["lm"], idx, r, w)
                api.gca_fwd(p, x["q"], x["k"], x["v"], idx, w, o, lse)
                api.gca_bwd(p, x["q"], x["k"], x["v"], idx, w, lse, x["dout"], dq, dk, dv, ds, wsb)
            for _ in range(warm):
                step()
            torch.cuda.synchronize()
            lib.gca_prof_read(0, None, None, None)
            lib.gca_prof_enable(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                step()
            e1.record()
            torch.cuda.synchronize()
            lib.gca_prof_enable(0)
            prof = read_prof(lib)
            assert api.gca_get_status() == 0, "device-side error in the sweep"
            ms = e0.elapsed_time(e1) / steps
            U = int((idx >= 0).sum().item())
            ab = alg_bytes(wl, U, H, D, k)
            gathered = 3 * U * 2 * S * D * 2
            kern = {}
            for n, (t, c) in sorted(prof.items()):
                fam = "bwd_kv" if "kv" in n else ("bwd_q" if "bwd_q" in n else ("fwd" if "fwd" in n else None))
                row = {"ms": round(t / c, 4)}
                if fam is not None:
                    row["frac"] = round(ab[fam] / (t / c / 1e3) / 1e9 / hbm, 4)
                kern[n] = row
            out["sweep_64k_S%d_k%d" % (S, k)] = {
                "step": "gca_score_topk + gca_fwd + gca_bwd", "B": B, "L": L, "S": S, "topk": k,
                "valid_units": U, "ms": round(ms, 4), "query_tokens_per_s": round(B * L / (ms / 1e3), 1),
                "roofline": {"bound": "hbm", "gathered_bytes": gathered,
                             "achieved": round(gathered / ms / 1e6, 1), "peak": hbm, "unit": "GB/s",
                             "frac": round(gathered / ms / 1e6 / hbm, 4)},
                "kernels": kern}
            del idx, r, w, ds, o, dq, dk, dv, lse, wsb
        del x
        torch.cuda.empty_cache()
    return out


SWA_WINDOW = 512


def swa_inputs(dev, B=8, L=16384, H=12, d=64, seed=11):
    """Q, K, V [B, L, H, d] ~ N(0, 1/64) in bf16 (the GCA workloads' recipe)."""
    import torch
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn(B, L, H, d, generator=g) * 0.125).to(torch.bfloat16).to(dev) for _ in range(3)]


def swa_roofline(B, L, H, d, W, ms, hbm, tflops, backward=False):
    """Slower of algorithmic bytes at HBM bandwidth and algorithmic FLOPs at
    tensor peak.  Forward bytes: Q, K, V read and O written once (bf16), lse
    (fp32); FLOPs: 4 d per (token, head, visible key), token t seeing
    min(t + 1, W) keys.  Backward: Q, K, V, O, dO read and dQ, dK, dV written
    once plus lse; 10 d FLOPs per (token, head, visible key)."""
    byts = (8 if backward else 4) * B * L * H * d * 2 + B * L * H * 4
    keys = W * (W + 1) // 2 + (L - W) * W if L >= W else L * (L + 1) // 2
    flops = (10.0 if backward else 4.0) * d * B * H * keys
    t_hbm, t_tc = byts / (hbm * 1e9), flops / (tflops * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    if bound == "hbm":
        ach, peak, unit = byts / (ms / 1e3) / 1e9, hbm, "GB/s"
    else:
        ach, peak, unit = flops / (ms / 1e3) / 1e12, tflops, "TFLOP/s"
    return {"bound": bound, "achieved": round(ach, 1), "peak": peak, "unit": unit,
            "frac": round(max(t_hbm, t_tc) / (ms / 1e3), 4), "alg_bytes": byts, "alg_flops": flops}


def _event_us(fn, n=50, warm=3):
    import torch
    for _ in range(warm):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n * 1e3


def next_rows(api, inputs, dev, hbm):
    """The widened rows: noisy (Gumbel) top-k, landmark gradients, and the
    reload of retrieved chunks from a K/V cache offloaded to page-locked host
    memory, each timed alone with CUDA events on the current stream."""
    import torch
    out = {}
    wl = inputs.WORKLOADS[WORKLOAD]
    x = inputs.make(wl, with_dout=False)
    lm = x["lm"].to(dev)
    B, nC, D = lm.shape
    g = torch.Generator(device="cpu").manual_seed(5)
    u = torch.rand(B, nC, nC, generator=g).clamp_(1e-12, 1 - 1e-7)
    noise = (-torch.log(-torch.log(u))).float().to(dev)           # Gumbel(0, 1)
    kw = dict(S=wl.S, H=wl.H, d=wl.d, topk=wl.topk)
    clean_us = _event_us(lambda i=0: api.score_topk(lm, **kw))
    noisy_us = _event_us(lambda i=0: api.score_topk_noisy(lm, noise, **kw))
    cand = B * nC * (nC - 1) // 2
    out["noisy_topk_b8"] = {"kernel": "gca_score_topk_noisy", "us": round(noisy_us, 2),
                            "clean_us": round(clean_us, 2),
                            "roofline": {"bound": "hbm", "achieved": round((lm.numel() * 2 + cand * 4) / noisy_us / 1e3, 1),
                                         "peak": hbm, "unit": "GB/s",
                                         "frac": round((lm.numel() * 2 + cand * 4) / noisy_us / 1e3 / hbm, 4),
                                         "note": "latency-bound: the tensor-core scorer with the noisy selection key; per-row top-k selection and the cross-CTA merge dominate"}}
    idx, r, w = api.score_topk(lm, **kw)
    dr = (torch.randn(B, nC, wl.topk, generator=g) * 0.1).float().to(dev) * (idx >= 0)
    U = int((idx >= 0).sum().item())
    lbw_us = _event_us(lambda i=0: api.landmark_bwd(lm, idx, dr, S=wl.S, H=wl.H, d=wl.d))
    lb_bytes = 2 * lm.numel() * 2 + 2 * U * D * 2                 # rows in and out, two row reads per unit
    out["landmark_bwd_b8"] = {"kernel": "gca_landmark_bwd", "us": round(lbw_us, 2), "valid_units": U,
                              "roofline": {"bound": "hbm", "achieved": round(lb_bytes / lbw_us / 1e3, 1),
                                           "peak": hbm, "unit": "GB/s",
                                           "frac": round(lb_bytes / lbw_us / 1e3 / hbm, 4)}}
    del x, lm, noise
    # offloaded cache: 2048 chunks of K and of V (2 x 201 MB) in page-locked host memory
    p = inputs.DECODE
    S, H, d, k = p["S"], p["H"], p["d"], p["topk"]
    n_src = 2048
    ck = torch.empty(n_src, S, H, d, dtype=torch.bfloat16, device=dev)
    cv = torch.empty_like(ck)
    api.gca_synth_fill_hash(ck, p["seed"], 0)
    api.gca_synth_fill_hash(cv, p["seed"], 1)
    hk = torch.empty(ck.shape, dtype=ck.dtype, pin_memory=True)
    hv = torch.empty(cv.shape, dtype=cv.dtype, pin_memory=True)
    hk.copy_(ck)
    hv.copy_(cv)
    del ck, cv
    n_it = 50
    sets = torch.stack([torch.randperm(n_src, generator=g)[:k] for _ in range(n_it + 3)]).int().to(dev)
    chunk = S * H * d * 2
    dk = torch.empty(k * S, H, d, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    di = torch.empty(k, dtype=torch.int32, device=dev)
    gat = lambda i=0: api.gca_gather_chunks(hk, hv, n_src, chunk, sets[i], k, dk, dv, di)
    gat_us = _event_us(gat, n=n_it)
    big_h = torch.empty(64 << 20, dtype=torch.float32, pin_memory=True)
    big_d = torch.empty_like(big_h, device=dev)
    copy_us = _event_us(lambda i=0: big_d.copy_(big_h, non_blocking=True), n=5, warm=1)
    link = big_h.numel() * 4 / copy_us / 1e3
    gb = 2 * k * chunk
    out["offload_gather"] = {"kernel": "gca_gather_chunks", "us": round(gat_us, 2), "bytes": gb,
                             "chunks": k, "source": "page-locked host memory (2 x 2048 chunks)",
                             "roofline": {"bound": "host link", "achieved": round(gb / gat_us / 1e3, 1),
                                          "peak": round(link, 1), "unit": "GB/s",
                                          "frac": round(gb / gat_us / 1e3 / link, 4),
                                          "peak_source": "cudaMemcpyAsync of 256 MB page-locked host -> device, same process"}}
    return out


# --------------------------------------------------------------------------- oracle
def oracle_step(L_sample, B_sample=1):
    """One oracle pass (score + fwd + bwd) on the first B_sample batch rows of
    the workload truncated to L_sample tokens.  Returns seconds."""
    import numpy as np

    import oracle
    from retrieval_sparse_attention_gb300 import inputs
    wl = inputs.WORKLOADS[WORKLOAD]
    x = inputs.make(wl, B=B_sample, L=L_sample)
    f = {n: t.double().numpy() for n, t in x.items()}
    t0 = time.perf_counter()
    idx, r, w = oracle.score_topk(f["lm"], wl.topk, False, wl.off_by_one)
    oracle.fwd(f["q"], f["k"], f["v"], idx, w, wl.S)
    oracle.bwd(f["q"], f["k"], f["v"], idx, w, f["dout"], wl.S)
    return time.perf_counter() - t0


def cpu_baseline(L_sample=16384, B_sample=4):
    import oracle
    oracle.build()
    t = oracle_step(L_sample, B_sample)
    return {"value": round(B_sample * L_sample / t, 2), "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "sample": "fp64 oracle score+fwd+bwd on batch rows 0-%d (of 8), all %d "
            "tokens each, of the workload; %.2f s" % (B_sample - 1, L_sample, t)}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    # size the per-step sample so that warm-up + steps end within about two minutes
    t1 = oracle_step(1024)
    L = 1024
    while L < 16384 and (t1 * (2 * L / 1024)) * (args.steps + args.warmup) < 120.0:
        L *= 2
    for _ in range(args.warmup):
        oracle_step(L)
    ts = [oracle_step(L) for _ in range(args.steps)]
    tot = sum(ts)
    value = L * args.steps / tot
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_tokens": L, "B": 1},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": "score+fwd+bwd on batch row 0, first %d tokens per step" % L},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_case(args):
    """Profiling mode: only the named path, W warm-up + K timed steps."""
    import torch

    from retrieval_sparse_attention_gb300 import api, inputs
    name, B, backward = CASES[args.case]
    dev = torch.device("cuda", 0)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if name == "swa":
        x = swa_inputs(dev, B=B)
        if backward:
            o, lse = api.swa_fwd(x[0], x[1], x[2], window=SWA_WINDOW)
            g = swa_inputs(dev, B=B, seed=12)[0] * 8
            step = lambda: api.swa_bwd(x[0], x[1], x[2], o, lse, g, window=SWA_WINDOW)
        else:
            step = lambda: api.swa_fwd(x[0], x[1], x[2], window=SWA_WINDOW)
    elif name is None:
        hx = inputs.decode_inputs()
        lm, ql = hx["lm"].to(dev), hx["ql"].to(dev)
        p = inputs.DECODE
        ws = torch.empty(api.gca_decode_workspace_size(p["N"], p["D"], p["topk"]), dtype=torch.uint8,
                         device=dev)
        step = lambda: api.decode_retrieve(lm, ql, topk=p["topk"], workspace=ws)
    else:
        wl = inputs.WORKLOADS[name]
        x = {n: t.to(dev) for n, t in inputs.make(wl, B=B, with_dout=backward).items()}
        ob = wl.off_by_one

        def step():
            idx, r, w = api.score_topk(x["lm"], S=wl.S, H=wl.H, d=wl.d, topk=wl.topk, off_by_one=ob)
            o, lse = api.fwd(x["q"], x["k"], x["v"], idx, w, S=wl.S)
            if backward:
                api.bwd(x["q"], x["k"], x["v"], idx, w, lse, x["dout"], S=wl.S)
    from retrieval_sparse_attention_gb300 import _lib
    lib = _lib.load()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    lib.gca_prof_read(0, None, None, None)
    lib.gca_prof_enable(1)
    ev0.record()
    for _ in range(args.steps):
        step()
    ev1.record()
    torch.cuda.synchronize()
    lib.gca_prof_enable(0)
    prof = read_prof(lib)
    assert api.gca_get_status() == 0
    print(json.dumps({"case": args.case, "ms_per_step": ev0.elapsed_time(ev1) / args.steps,
                      "kernel_ms": {k: round(v[0] / v[1], 4) for k, v in sorted(prof.items())}}))


if __name__ == "__main__":
    a = parse()
    if a.case is not None:
        run_case(a)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
