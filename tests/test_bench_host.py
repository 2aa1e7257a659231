"""Host-side counting in bench.py: algorithmic flops and bytes against brute force."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_attn_flops_matches_a_per_row_count():
    rng = np.random.default_rng(0)
    L = rng.integers(1, 300, size=20)
    ql = np.array([rng.integers(0, l + 1) for l in L])
    Hq, D = 6, 64
    brute = 0
    for l, q in zip(L, ql):
        for j in range(q):
            brute += (l - q + j + 1) * Hq * 4 * D  # positions 0 .. L - ql + j
    assert bench.attn_flops(L, ql, Hq, D) == brute


def test_attn_bytes_counts_each_kv_element_once_per_kv_head():
    # one sequence, L = 33 tokens, page 16: 3 block-table entries
    got = bench.attn_bytes([33], [2], Hq=8, Hkv=2, D=64, P=16, elem=2)
    kv = 33 * 2 * 64 * 2 * 2
    qo = 2 * 8 * 64 * 2 * 2
    assert got == kv + qo + 3 * 4 + 2 * 8 * 4


def test_attn_bytes_of_a_quantised_pool():
    # 1-byte codes for K and V plus one fp32 scale per token and KV head for each; q and
    # out stay bf16
    got = bench.attn_bytes([33], [2], Hq=8, Hkv=2, D=64, P=16, elem=2, kv_elem=1)
    kv = 33 * 2 * (64 * 2 * 1 + 2 * 4)
    qo = 2 * 8 * 64 * 2 * 2
    assert got == kv + qo + 3 * 4 + 2 * 8 * 4
    from verify_attention_spec_gb300 import workloads as wl
    assert bench.elem_sizes(wl.FP8) == (2, 1) and bench.elem_sizes(wl.BF16) == (2, 2)


def test_unique_kv_bytes_counts_shared_pages_once():
    # two sequences sharing pages 5 and 6 (32 tokens) and each with a page of its own
    bt = np.array([[5, 6, 1], [5, 6, 2]])
    got = bench.unique_kv_bytes(bt, [40, 35], Hkv=2, D=8, P=16, kv_elem=2)
    tokens = 16 + 16 + 8 + 3
    assert got == tokens * 2 * 8 * 2 * 2
    # without sharing it equals the per-sequence count
    bt2 = np.array([[5, 6, 1], [7, 8, 2]])
    assert bench.unique_kv_bytes(bt2, [40, 35], 2, 8, 16, 2) == (40 + 35) * 2 * 8 * 2 * 2


def test_acceptance_stats_counts_tests_run_and_sum_of_minima():
    # Sequences accepting 0, 4 and 2 of k = 4 drafts ran 1, 4 and 3 ratio tests.
    acc = np.array([0, 4, 2])
    p = np.zeros((3, 5, 4))
    q = np.zeros((3, 4, 4))
    p[:, :, :2] = 0.5                 # p = (1/2, 1/2, 0, 0) at every position
    q[:] = 0.25                       # q uniform: sum_x min(p, q) = 1/2
    q[2, 3] = [0.5, 0.5, 0.0, 0.0]    # one position with q = p: sum of minima 1
    st = bench.acceptance_stats(acc, 4, p, q)
    assert st["mean_accepted"] == 2.0
    assert st["per_token_acceptance"] == 6 / 8
    assert np.isclose(st["alpha_sum_min_pq"], (0.5 + 0.5 + (0.5 * 3 + 1.0) / 4) / 3)
    assert "alpha_sum_min_pq" not in bench.acceptance_stats(acc, 4)


def test_verify_bytes_reads_two_rows_after_a_rejection_and_one_after_full_acceptance():
    k, V = 4, 10
    scalars = k * 4 + k * 8 + (k + 1) * 4 + 4  # drafts, p and q at them, outputs, length
    assert bench.verify_bytes([0, 4], k, V) == (2 + 1) * V * 4 + 2 * scalars
    assert bench.verify_bytes([4, 4, 4], k, V) == 3 * V * 4 + 3 * scalars


def test_tree_verify_bytes_by_where_the_walk_ends():
    # Node 0 is the root; drafts 1..3 with parents 0, 1, 0 (draft i is node i).
    parents = np.array([[0, 1, 0], [0, 1, 0]])
    path = np.array([[1, 2, 0], [1, 0, 0]])
    V, n = 16, 3
    per_seq = n * 4 * 3 + n * 8 + (n + 1) * 4 + 4
    # Sequence 0 accepted the chain 1 -> 2 (node 2 is a leaf: its p row alone); sequence 1
    # accepted node 1, which has a child (p and q rows).
    assert bench.tree_verify_bytes([2, 1], path, parents, V) == (1 + 2) * V * 4 + 2 * per_seq


def test_ncu_traffic_is_dropped_when_the_kernel_source_changed(tmp_path, monkeypatch):
    csrc = tmp_path / "verify_attention_spec_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["paged_attn"]:
        (csrc / f).write_text("// kernel " + f + "\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("paged_attn")
    prof = tmp_path / "profiles" / "paged_attn_w_ncu.md"
    prof.write_text(f"kernel_source_sha256_16: {h}\ndram_bytes_per_full_launch: 12345\n")
    assert bench.ncu_traffic("w") == 12345.0
    assert bench.ncu_traffic("other") is None
    (csrc / bench.KERNEL_SOURCES["paged_attn"][0]).write_text("// changed\n")
    assert bench.ncu_traffic("w") is None


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores (no GPU needed) and
    prints one JSON line with the contract's keys; under a launcher only rank 0 prints."""
    import json
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload",
           "tiny", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, RANK="0")
    out = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600, check=True)
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["value"] == d["value"] and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    other = subprocess.run(cmd, capture_output=True, text=True, env=dict(os.environ, RANK="1"),
                           timeout=600, check=True)
    assert other.stdout.strip() == ""


def test_clock_sampler_reads_clocks_and_throttle_reasons(tmp_path, monkeypatch):
    """The sampler takes the median SM clock, the highest maximum clock and every
    throttle reason seen Active, from nvidia-smi's CSV (a stand-in script here)."""
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "echo '2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "echo '1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "echo '2010, 2070, 1200.5, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "echo '[N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench.ClockSampler(0)
    s.start()
    import time
    time.sleep(0.5)
    got = s.stop()
    assert got == {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}
    monkeypatch.setenv("PATH", str(tmp_path / "empty"))
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop()["reasons"] == ["unavailable"]


def test_kv_bytes_match_the_pages_worked_example():
    """The bench's KV byte count for one layer, times the layers, gives the per-token and
    per-context cache sizes the pages work out (tests/golden/kv_cache_bytes_per_token.txt)."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "kv_cache_bytes_per_token.txt")
    g = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (x.strip() for x in line.split("="))
            g[k] = float(v)
    layers, H, D = int(g["layers"]), int(g["kv_heads"]), int(g["head_dim"])
    e, ctx = int(g["bytes_per_element"]), int(g["context_tokens"])
    P = 16
    # one layer, one sequence of ctx tokens with no query rows: KV plus the block table
    one_layer = bench.attn_bytes([ctx], [0], Hq=H, Hkv=H, D=D, P=P, elem=e)
    kv_layer = one_layer - (ctx + P - 1) // P * 4
    per_token = kv_layer // ctx * layers
    assert per_token == 2 * layers * H * D * e == 2_621_440
    assert abs(per_token / 1e6 - g["per_token_mb_printed"]) < 0.05
    per_context = per_token * ctx
    assert abs(per_context / 1e9 - g["per_context_gb_printed"]) < 0.8  # 10.7 GB: "about 10"
