"""Host-side parts of bench.py: the roofline's algorithmic bytes of each GCA
kernel (gathered tiles plus the resident tensors it reads and writes once)
worked out by hand for a small case, the committed DRAM-traffic table it reads
per kernel and workload, and the clock sampler (driven by a stand-in
nvidia-smi that prints fixed samples)."""
import os
import stat
import time
import types

import bench


def test_alg_bytes_hand_worked_case():
    # B=1, L=128 tokens, S=64, H=2 heads of d=64 (D = 128), k=2, U=3 valid units.
    wl = types.SimpleNamespace(B=1, L=128, S=64)
    got = bench.alg_bytes(wl, U=3, H=2, D=128, k=2)
    tensor = 128 * 128 * 2            # one [B, L, H, d] bf16 tensor: 32768 bytes
    lse = 128 * 2 * 2 * 4             # [B, L, H, k] fp32: 2048 bytes
    gather = 3 * 2 * 64 * 128 * 2     # 3 units x (two 64 x 128 bf16 tiles): 98304 bytes
    rows = 3 * 2 * 64 * 2 * 4         # per unit: lse and delta rows of S per head: 3072 bytes
    assert got["fwd"] == gather + 2 * tensor + lse == 165888
    assert got["bwd_q"] == gather + 3 * tensor + 2 * lse == 200704
    assert got["bwd_kv"] == gather + rows + 4 * tensor == 232448


def test_traffic_table_reads_only_data_lines():
    t = bench.traffic_table()
    assert t, "profiles/ncu_dram_traffic.txt missing or empty"
    for (kernel, workload), nbytes in t.items():
        assert not kernel.startswith("#")
        assert nbytes > 0 and nbytes == int(nbytes)
    assert ("fwd_tc", "gpt2s_fwdbwd_b8") in t
    assert ("decode_retrieve", "decode_262144x768") in t


def _fake_smi(tmp_path, lines):
    """An executable named nvidia-smi that prints `lines` in a loop, 20 ms apart."""
    body = "".join("echo '%s'; sleep 0.02; " % ln for ln in lines)
    p = tmp_path / "nvidia-smi"
    p.write_text("#!/bin/sh\nwhile true; do %sdone\n" % body)
    p.chmod(p.stat().st_mode | stat.S_IXUSR | stat.S_IXGRP | stat.S_IXOTH)
    return str(tmp_path)


def test_clock_sampler_counts_samples_inside_the_region(tmp_path, monkeypatch):
    d = _fake_smi(tmp_path, ["0, 2070, 2070, 900.5, Not Active, Not Active, Not Active, Active",
                             "0, 2055, 2070, 910.0, Not Active, Not Active, Not Active, Not Active",
                             "garbage line"])
    monkeypatch.setenv("PATH", d + os.pathsep + os.environ.get("PATH", ""))
    with bench.ClockSampler(0) as clk:
        assert clk.lines, "the first sample is awaited before the region starts"
        clk.mark_start()
        time.sleep(0.3)
        clk.mark_end()
    s = clk.summary()
    assert s["samples_in_region"] >= 3
    assert s["samples"] >= s["samples_in_region"]
    assert 2055.0 <= s["sm_mhz"] <= 2070.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))          # nothing executable there
    with bench.ClockSampler(0, first_wait_s=0.2) as clk:
        clk.mark_start()
        clk.mark_end()
    assert clk.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                             "samples": 0, "samples_in_region": 0}
