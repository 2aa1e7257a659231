"""GPU parity of attention over quantised KV pages (include/vas.h: paged_attn_fwd_quant)
against the float64 oracle, which decodes the same FP8 E4M3 / INT8 codes and scales
exactly ("llm-inference-optimization-batching", tempatgunting.com, section
"Quantization and Precision Choices for KV")."""
import numpy as np
import pytest
import torch

from verify_attention_spec_gb300 import workloads as wl

from gpu_common import (ancestor_masks, compare_attention, oracle_attention, run_gpu_attention,
                        to_device)

pytestmark = pytest.mark.gpu


def _case(lens, qlens, Hq, Hkv, D, P, kv, seed):
    return wl.attention_inputs(lens, qlens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                               page_size=P, kv_dtype=kv, seed=seed)


# Decode rows, verify rows in 16-row and wide units, a 72-row and a 128-row block,
# sequences shorter than 64 (the precise path), page boundaries, a long context that
# splits, and an empty query.
LENS = [1, 16, 33, 5, 70, 300, 1500, 64, 9000, 130, 2100, 95]
QLENS = [1, 1, 2, 5, 9, 1, 8, 0, 5, 17, 33, 64]


@pytest.mark.parametrize("D,P,Hq,Hkv", [(128, 32, 64, 8), (128, 16, 32, 8), (64, 16, 4, 4),
                                        (64, 32, 16, 2)])
@pytest.mark.parametrize("kv", [wl.FP8, wl.INT8])
def test_shapes(vas_lib, D, P, Hq, Hkv, kv):
    a = _case(LENS, QLENS, Hq, Hkv, D, P, kv, seed=D + P + Hq)
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, kv)
    assert vas_lib.vas_last_device_error() == 0


@pytest.mark.parametrize("kv", [wl.FP8, wl.INT8])
def test_trees_on_quantised_pages(vas_lib, kv):
    lens, qlens = [40, 3000, 64, 700], [2, 9, 64, 33]
    a = _case(lens, qlens, 64, 8, 128, 32, kv, seed=29)
    parents = wl.draft_tree_parents(qlens, seed=29, extra_roots=0.1)
    ref_o, ref_l = oracle_attention(a, parents=parents)
    out, lse = run_gpu_attention(vas_lib, to_device(a), tree_masks=ancestor_masks(parents, qlens))
    compare_attention(out, lse, ref_o, ref_l, kv)


@pytest.mark.parametrize("kv", [wl.FP8, wl.INT8])
def test_split_invariance(vas_lib, kv):
    a = _case([9000, 30, 4100, 17], [1, 5, 5, 1], 32, 8, 128, 16, kv, seed=5)
    ref_o, ref_l = oracle_attention(a)
    ad = to_device(a)
    dims = vas_lib.attn_dims(ad.q, ad.k_pages, ad.block_table, ad.seq_lens, quant=kv)
    o1, l1 = run_gpu_attention(vas_lib, ad, workspace_bytes=vas_lib.paged_attn_workspace_min(dims))
    o2, l2 = run_gpu_attention(vas_lib, ad)
    compare_attention(o1, l1, ref_o, ref_l, kv)
    compare_attention(o2, l2, ref_o, ref_l, kv)


def test_q_beyond_the_f16_range(vas_lib):
    """|q| near 2^18 (beyond f16's 65504), with the softmax scale divided by the same
    2^16: the unit's Q is scaled into f16 range by a power of two and the scores scaled
    back, so the result matches the oracle's."""
    import oracle
    a = _case([200, 50, 3000], [1, 5, 9], 32, 8, 128, 16, wl.FP8, seed=7)
    a.q = (a.q.float() * 65536.0).to(torch.bfloat16)  # exact: a power of two
    scale = 1.0 / (65536.0 * np.sqrt(128))
    ref_o, ref_l = oracle.paged_attn_quant(
        wl.bf16_bits(a.q), a.k_pages.numpy(), a.v_pages.numpy(), a.k_scale.numpy(),
        a.v_scale.numpy(), a.block_table.numpy(), a.seq_lens.numpy(), a.query_lens.numpy(),
        fmt=oracle.Q_E4M3, scale=scale)
    ad = to_device(a)
    dims = vas_lib.attn_dims(ad.q, ad.k_pages, ad.block_table, ad.seq_lens, scale=scale, quant=wl.FP8)
    out = torch.empty_like(ad.q)
    lse = torch.empty(ad.q.shape[0], ad.q.shape[1], dtype=torch.float32, device="cuda")
    ws = vas_lib.alloc_workspace(dims)
    vas_lib.paged_attn_fwd_quant(ad.q, ad.k_pages, ad.v_pages, ad.k_scale, ad.v_scale,
                                 ad.block_table, ad.seq_lens, ad.query_lens, out, lse, ws,
                                 quant=wl.FP8, dims=dims)
    torch.cuda.synchronize()
    compare_attention(out, lse, ref_o, ref_l, wl.FP8)


def test_poisoned_unowned_slots(vas_lib):
    """Codes and scales of slots past each sequence's end are NaN: nothing leaks."""
    a = _case([17, 40, 33], [1, 4, 2], 8, 2, 128, 16, wl.FP8, seed=3)
    lens = a.seq_lens.numpy()
    bt = a.block_table.numpy()
    for i, L in enumerate(lens):
        last = bt[i, (L - 1) // 16]
        for t in range(L % 16 or 16, 16):
            a.k_pages[last, t] = 0x7F  # E4M3 NaN
            a.v_pages[last, t] = 0x7F
            a.k_scale[last, :, t] = float("nan")
            a.v_scale[last, :, t] = float("nan")
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, wl.FP8)


@pytest.mark.parametrize("name", ["decode64_fp8", "decode64_int8"])
def test_workload_full_parity(vas_lib, name):
    a = wl.workload_attention(name)
    ref_o, ref_l = oracle_attention(a)
    out, lse = run_gpu_attention(vas_lib, to_device(a))
    compare_attention(out, lse, ref_o, ref_l, a.kv_dtype)
    assert vas_lib.vas_last_device_error() == 0


@pytest.mark.parametrize("name", ["stress70b_fp8", "stress70b_int8"])
def test_stress70b_quant_full_size(vas_lib, name):
    """The 70B batch with FP8 / INT8 pages at full size, in the bench's launch
    configuration, every row against the oracle's exact decode of the same codes."""
    a = to_device(wl.workload_attention(name, pool_device="cuda"))
    out, lse = run_gpu_attention(vas_lib, a)
    assert vas_lib.vas_last_device_error() == 0
    ref_o, ref_l = oracle_attention(a)
    compare_attention(out, lse, ref_o, ref_l, a.kv_dtype)
