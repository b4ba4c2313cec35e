"""Host-side arithmetic of bench.py's roofline: the algorithmic bytes of each
GCA kernel (gathered tiles plus the resident tensors it reads and writes once)
worked out by hand for a small case, and the committed DRAM-traffic table it
reads per kernel and workload."""
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
