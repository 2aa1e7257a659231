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
