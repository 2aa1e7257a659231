"""GPU parity of paged decode/verify attention against the float64 oracle, through the
C ABI (include/vas.h: paged_attn_fwd)."""
import numpy as np
import pytest
import torch

import oracle
from verify_attention_spec_gb300 import workloads as wl

from gpu_common import (compare_attention, oracle_attention, query_slice_inputs,
                        run_gpu_attention, to_device)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "decode64", "verify32", "mixed272"])
def test_workload_full_parity(vas_lib, name):
    a = wl.workload_attention(name)
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, a.kv_dtype)
    assert vas_lib.vas_last_device_error() == 0


def test_stress70b_full_size(vas_lib):
    """The full 70B-shape batch (512 sequences, 64/8 heads, page 32, ~8 GB of KV) in the
    bench's launch configuration, every row against the oracle: every work-order
    position, split count and merge of the headline launch."""
    a = to_device(wl.workload_attention("stress70b", pool_device="cuda"))
    out, lse = run_gpu_attention(vas_lib, a)
    assert vas_lib.vas_last_device_error() == 0
    ref_o, ref_l = oracle_attention(a)
    compare_attention(out, lse, ref_o, ref_l, a.kv_dtype)


def _case(lens, qlens, Hq=8, Hkv=2, D=128, P=16, dtype=wl.BF16, seed=3, pool_pages=None):
    return wl.attention_inputs(lens, qlens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                               page_size=P, kv_dtype=dtype, seed=seed, pool_pages=pool_pages)


@pytest.mark.parametrize("D,P,Hq,Hkv", [(128, 16, 8, 2), (128, 32, 64, 8), (64, 16, 4, 4),
                                        (64, 32, 16, 2), (128, 16, 4, 2), (128, 32, 64, 2),
                                        (128, 16, 8, 8)])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_shapes_and_ragged_edges(vas_lib, D, P, Hq, Hkv, dtype):
    """Page boundaries (L = P, P+1), a single token, a window covering the whole context
    (ql = L), long sequences spanning many stages, ragged tails, and an empty query."""
    lens = [1, P, P + 1, 5, 3 * P - 1, 700, 1500, 64, 2 * P + 7]
    qlens = [1, 1, 2, 5, 4, 1, 8, 0, 3]
    a = _case(lens, qlens, Hq, Hkv, D, P, dtype, seed=D + P)
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, dtype)
    assert vas_lib.vas_last_device_error() == 0


@pytest.mark.parametrize("dtype", [wl.BF16, wl.FP8])
def test_idle_slots(vas_lib, dtype):
    """Batch slots with no context and no query (L = 0, ql = 0) between live sequences,
    at the front and at the end: they get no work and leave their neighbours' rows alone."""
    lens = [0, 37, 0, 0, 200, 16, 0, 1200, 0]
    qlens = [0, 1, 0, 0, 5, 16, 0, 1, 0]
    a = _case(lens, qlens, Hq=32, Hkv=8, D=128, P=16, dtype=dtype, seed=61)
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, dtype)
    assert vas_lib.vas_last_device_error() == 0


def test_row_blocks_beyond_64_rows(vas_lib):
    """GQA group 8 x 9 query tokens = 72 rows: two row blocks per KV head."""
    a = _case([300, 90, 1000], [9, 9, 1], Hq=64, Hkv=8, D=128, P=32, seed=11)
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, wl.BF16)


def test_split_invariance(vas_lib):
    """The minimum workspace forbids splitting; the recommended one splits long
    sequences.  Both match the oracle and each other within fp32 merge error."""
    a = _case([9000, 30, 4100, 17], [1, 5, 5, 1], Hq=32, Hkv=8, seed=5)
    ref_o, ref_l = oracle_attention(a)
    ad = to_device(a)
    dims = vas_lib.attn_dims(ad.q, ad.k_pages, ad.block_table, ad.seq_lens)
    o1, l1 = run_gpu_attention(vas_lib, ad, workspace_bytes=vas_lib.paged_attn_workspace_min(dims))
    o2, l2 = run_gpu_attention(vas_lib, ad)
    compare_attention(o1, l1, ref_o, ref_l, wl.BF16)
    compare_attention(o2, l2, ref_o, ref_l, wl.BF16)
    assert (o1.float() - o2.float()).abs().max().item() <= 2 ** -7
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_many_splits(vas_lib):
    """Contexts of 70000 tokens split into more pieces than a warp has lanes: a decode
    sequence (narrow units) and a k=4 verify sequence (wide units), 35 and 38 splits on a
    152-SM part, each merged by the CTA that finishes its last split.  Against the
    oracle, and against the unsplit result."""
    a = _case([70000, 70000, 40], [1, 5, 1], Hq=32, Hkv=8, D=128, P=16, seed=31)
    ref_o, ref_l = oracle_attention(a)
    ad = to_device(a)
    out, lse = run_gpu_attention(vas_lib, ad)
    compare_attention(out, lse, ref_o, ref_l, wl.BF16)
    dims = vas_lib.attn_dims(ad.q, ad.k_pages, ad.block_table, ad.seq_lens)
    o1, l1 = run_gpu_attention(vas_lib, ad, workspace_bytes=vas_lib.paged_attn_workspace_min(dims))
    compare_attention(o1, l1, ref_o, ref_l, wl.BF16)
    assert (o1.float() - out.float()).abs().max().item() <= 2 ** -7
    assert (l1 - lse).abs().max().item() <= 1e-4
    assert vas_lib.vas_last_device_error() == 0


def test_more_sequences_than_the_plan_caches(vas_lib):
    """4500 sequences, more than the plan keeps in shared memory (4096): it reads the
    lengths from global memory.  Decode and short verify windows, against the oracle."""
    rng = np.random.default_rng(45)
    lens = rng.integers(1, 90, size=4500)
    qlens = np.where(rng.random(4500) < 0.1, np.minimum(lens, 3), 1)
    a = _case(lens, qlens, Hq=4, Hkv=1, D=64, P=16, seed=45)
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, wl.BF16)
    assert vas_lib.vas_last_device_error() == 0


@pytest.mark.parametrize("name", ["decode64", "verify32", "mixed272"])
def test_deterministic_reruns(vas_lib, name):
    """Same inputs, same bits, whichever SM and CTA ends up with which work unit."""
    a = to_device(wl.workload_attention(name))
    o1, l1 = run_gpu_attention(vas_lib, a)
    for _ in range(3):
        o2, l2 = run_gpu_attention(vas_lib, a)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_poisoned_pool_slots_and_outputs(vas_lib):
    """NaN in every pool slot no sequence owns (including the tails of last pages) must not
    leak into the result, and NaN-prefilled outputs must be fully overwritten."""
    lens, qlens = [37, 100, 5, 250], [1, 4, 5, 1]
    a = _case(lens, qlens, Hq=8, Hkv=2, seed=8, pool_pages=40)
    bt = a.block_table.numpy()
    k, v = a.k_pages.clone(), a.v_pages.clone()
    owned = np.zeros((a.num_pages, a.page_size), dtype=bool)
    for i, L in enumerate(lens):
        for t in range(L):
            owned[bt[i, t // a.page_size], t % a.page_size] = True
    mask = torch.from_numpy(~owned)
    k[mask] = float("nan")
    v[mask] = float("nan")
    a_nan = wl.AttentionInputs(a.q, k, v, a.block_table, a.seq_lens, a.query_lens, 8, 2, 128, 16,
                               wl.BF16)
    ref_o, ref_l = oracle_attention(a)  # oracle never reads unowned slots
    ad = to_device(a_nan)
    out = torch.full_like(ad.q, float("nan"))
    lse = torch.full((ad.q.shape[0], 8), float("nan"), device="cuda")
    out, lse = run_gpu_attention(vas_lib, ad, out=out, lse=lse)
    compare_attention(out, lse, ref_o, ref_l, wl.BF16)


def test_bad_page_id_poisons_only_its_sequence(vas_lib):
    a = _case([40, 70, 33], [1, 3, 1], seed=9)
    ref_o, ref_l = oracle_attention(a)
    ad = to_device(a)
    bt = ad.block_table.clone()
    bt[1, 2] = a.num_pages + 5
    ad = wl.AttentionInputs(ad.q, ad.k_pages, ad.v_pages, bt, ad.seq_lens, ad.query_lens, 8, 2, 128,
                            16, wl.BF16)
    vas_lib.vas_last_device_error()
    out, lse = run_gpu_attention(vas_lib, ad)
    bits = vas_lib.vas_last_device_error()
    assert bits & vas_lib.VAS_DEV_BAD_PAGE
    rows_bad = np.arange(1, 4)
    rows_ok = np.array([0, 4])
    assert torch.isnan(out[rows_bad].float()).all() and torch.isnan(lse[rows_bad]).all()
    compare_attention(out, lse, ref_o[rows_ok], ref_l[rows_ok], wl.BF16, rows=rows_ok)


def test_inconsistent_lengths_are_reported(vas_lib):
    a = _case([40, 70, 33], [1, 3, 1], seed=10)
    ad = to_device(a)
    ql = ad.query_lens.clone()
    sl = ad.seq_lens.clone()
    sl[2] = 0                       # query_len 1 > seq_len 0
    ad = wl.AttentionInputs(ad.q, ad.k_pages, ad.v_pages, ad.block_table, sl, ql, 8, 2, 128, 16,
                            wl.BF16)
    vas_lib.vas_last_device_error()
    out, lse = run_gpu_attention(vas_lib, ad)
    assert vas_lib.vas_last_device_error() & vas_lib.VAS_DEV_BAD_LENGTHS
    assert torch.isnan(out[4].float()).all() and torch.isnan(lse[4]).all()
    ref_o, ref_l = oracle_attention(a)
    compare_attention(out, lse, ref_o[:4], ref_l[:4], wl.BF16, rows=np.arange(4))


def test_query_rows_mismatch_total(vas_lib):
    """sum(query_lens) smaller than total_q_tokens: the uncovered rows are NaN."""
    a = _case([40, 70], [1, 3], seed=12)
    ad = to_device(a)
    q = torch.cat([ad.q, ad.q[:2]])  # two extra rows no sequence owns
    ad2 = wl.AttentionInputs(q, ad.k_pages, ad.v_pages, ad.block_table, ad.seq_lens, ad.query_lens,
                             8, 2, 128, 16, wl.BF16)
    vas_lib.vas_last_device_error()
    out, lse = run_gpu_attention(vas_lib, ad2)
    assert vas_lib.vas_last_device_error() & vas_lib.VAS_DEV_BAD_LENGTHS
    assert torch.isnan(out[4:].float()).all()
    ref_o, ref_l = oracle_attention(a)
    compare_attention(out, lse, ref_o, ref_l, wl.BF16, rows=np.arange(4))


def test_chunked_prefill_queries(vas_lib):
    """Prompt chunks as queries: a 256-token chunk on 2048 of context, a whole 700-token
    prompt (query length = context) and a 1024-token chunk, causal within each chunk;
    GQA group 4, so up to 64 row blocks per KV head."""
    a = _case([2048, 700, 1500], [256, 700, 1024], Hq=32, Hkv=8, D=128, P=16, seed=21)
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, wl.BF16)
    assert vas_lib.vas_last_device_error() == 0


def test_prefill8_sampled(vas_lib):
    """The chunked-prefill workload (8 x 1024-token chunks on 4096 of context, 70B
    shape) in full on the GPU; the oracle checks slices of it at their own positions:
    the first and the last 64 query tokens of one chunk and 64 from the middle of
    another."""
    a = to_device(wl.workload_attention("prefill8", pool_device="cuda"))
    out, lse = run_gpu_attention(vas_lib, a)
    for seq, j0 in [(0, 0), (0, 960), (5, 500)]:
        sub, rows = query_slice_inputs(a, seq, j0, 64)
        ref_o, ref_l = oracle_attention(sub)
        compare_attention(out, lse, ref_o, ref_l, wl.BF16, rows=rows)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    assert vas_lib.vas_last_device_error() == 0


def test_shared_prefix_pages(vas_lib):
    """Block tables that alias a prefix: groups of 3 sequences share their first 4 pages
    (a 64-token prompt), in decode, verify and chunk form, against the oracle."""
    lens = np.array([70, 64 + 33, 64 + 200, 64 + 5, 64 + 1000, 90, 64 + 17])
    qlens = np.array([1, 5, 33, 1, 9, 1, 2])
    a = wl.attention_inputs(lens, qlens, num_q_heads=32, num_kv_heads=8, head_dim=128,
                            page_size=16, kv_dtype=wl.BF16, seed=23, prefix_pages=4,
                            prefix_group=3)
    bt = a.block_table.numpy()
    assert (bt[0, :4] == bt[2, :4]).all() and (bt[3, :4] == bt[5, :4]).all()
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, wl.BF16)
    assert vas_lib.vas_last_device_error() == 0
