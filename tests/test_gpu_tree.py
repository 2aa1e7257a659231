"""GPU parity of draft-tree attention (include/vas.h: paged_attn_fwd_tree) against the
float64 oracle given the same trees as parent pointers.  The tree is the one of
"Continuous Batching & Speculative Decoding" (neuralmasteryai.com), section "4. Tree
Attention & Medusa Heads": every draft token sees the context, its ancestors and
itself."""
import numpy as np
import pytest
import torch

from verify_attention_spec_gb300 import workloads as wl

from gpu_common import (ancestor_masks, compare_attention, oracle_attention, run_gpu_attention,
                        run_gpu_attention_tree, to_device)

pytestmark = pytest.mark.gpu


def _case(lens, qlens, Hq, Hkv, D, P, dtype=wl.BF16, seed=3):
    return wl.attention_inputs(lens, qlens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                               page_size=P, kv_dtype=dtype, seed=seed)


# Query lengths that reach every kernel path for GQA groups 1, 4 and 8: a 16-row unit
# (group 8, 2 tokens), 17..64-row units (3..8 tokens at group 8; up to 64 at group 1),
# 128-row blocks (more than 64 rows), a full 64-token tree, decode rows between them, and
# contexts long enough (9000) to be split across SMs.
LENS = [40, 2, 300, 1, 777, 5000, 64, 9000, 130, 2100, 95]
QLENS = [2, 2, 3, 1, 5, 8, 64, 9, 17, 33, 64]


@pytest.mark.parametrize("D,P,Hq,Hkv", [(128, 32, 64, 8), (128, 16, 8, 2), (64, 16, 4, 4),
                                        (64, 32, 16, 2)])
@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_random_trees(vas_lib, D, P, Hq, Hkv, dtype):
    a = _case(LENS, QLENS, Hq, Hkv, D, P, dtype, seed=D + P + Hq)
    parents = wl.draft_tree_parents(QLENS, seed=D + Hkv, extra_roots=0.1)
    ref_o, ref_l = oracle_attention(a, parents=parents)
    out, lse = run_gpu_attention_tree(vas_lib, to_device(a), ancestor_masks(parents, QLENS))
    compare_attention(out, lse, ref_o, ref_l, dtype)
    assert vas_lib.vas_last_device_error() == 0


def test_split_trees(vas_lib):
    """Trees on long contexts with the minimum workspace (no split) and the recommended
    one (split): both match the oracle."""
    lens, qlens = [12000, 6000, 3000], [64, 9, 24]
    a = _case(lens, qlens, 64, 8, 128, 32, seed=41)
    parents = wl.draft_tree_parents(qlens, seed=41)
    ref_o, ref_l = oracle_attention(a, parents=parents)
    ad = to_device(a)
    masks = ancestor_masks(parents, qlens)
    for nbytes in [None, vas_lib.paged_attn_workspace_min(
            vas_lib.attn_dims(ad.q, ad.k_pages, ad.block_table, ad.seq_lens))]:
        out, lse = run_gpu_attention_tree(vas_lib, ad, masks, workspace_bytes=nbytes)
        compare_attention(out, lse, ref_o, ref_l, wl.BF16)


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F32])
def test_chain_is_the_causal_call_bit_for_bit(vas_lib, dtype):
    """A chain (each token's parent the one before it) is the causal window: the tree
    entry point gives paged_attn_fwd's results bit for bit."""
    a = to_device(_case(LENS, QLENS, 64, 8, 128, 32, dtype, seed=9))
    chain = np.concatenate([np.arange(q, dtype=np.int32) - 1 for q in QLENS])
    out_t, lse_t = run_gpu_attention_tree(vas_lib, a, ancestor_masks(chain, QLENS))
    out_c, lse_c = run_gpu_attention(vas_lib, a)
    assert torch.equal(out_t, out_c) and torch.equal(lse_t, lse_c)


def test_masks_ignored_outside_draft_range(vas_lib):
    """Sequences of one query token or more than 64 take the causal window whatever
    their words hold."""
    lens, qlens = [500, 900, 70], [1, 65, 1]
    a = to_device(_case(lens, qlens, 32, 8, 128, 16, seed=13))
    rng = np.random.default_rng(13)
    junk = rng.integers(0, 2**63, size=sum(qlens), dtype=np.int64).astype(np.uint64)
    out_t, lse_t = run_gpu_attention_tree(vas_lib, a, junk)
    out_c, lse_c = run_gpu_attention(vas_lib, a)
    assert torch.equal(out_t, out_c) and torch.equal(lse_t, lse_c)


def test_star_tree(vas_lib):
    """Every draft token a child of the root (a width-63 top-k level): each sees the
    context, the root and itself only."""
    lens, qlens = [3000, 200], [64, 64]
    a = _case(lens, qlens, 64, 8, 128, 32, seed=17)
    parents = np.concatenate([np.r_[-1, np.zeros(63, dtype=np.int32)]] * 2).astype(np.int32)
    ref_o, ref_l = oracle_attention(a, parents=parents)
    out, lse = run_gpu_attention_tree(vas_lib, to_device(a), ancestor_masks(parents, qlens))
    compare_attention(out, lse, ref_o, ref_l, wl.BF16)


def test_tree70b_full_size(vas_lib):
    """The 70B batch whose 64 verify windows are 17-token draft trees, at full size and in
    the bench's launch configuration: tree-masked attention on every row, and the tree
    walk over V = 128256 on every window, against the oracle."""
    import oracle

    a = to_device(wl.workload_attention("tree70b", pool_device="cuda"))
    qlens = a.query_lens.cpu().numpy()
    parents = wl.draft_tree_parents(qlens, seed=wl.WORKLOADS["tree70b"].seed)
    out, lse = run_gpu_attention_tree(vas_lib, a, ancestor_masks(parents, qlens))
    assert vas_lib.vas_last_device_error() == 0
    ref_o, ref_l = oracle_attention(a, parents=parents)
    compare_attention(out, lse, ref_o, ref_l, a.kv_dtype)

    v = wl.workload_verify("tree70b", attn_parents=parents)
    d = "cuda"
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(d)
    acc = torch.empty(v.B, dtype=torch.int32, device=d)
    tok = torch.empty(v.B, v.k + 1, dtype=torch.int32, device=d)
    path = torch.empty(v.B, v.k, dtype=torch.int32, device=d)
    vas_lib.spec_verify_tree(t(v.p), t(v.q), t(v.draft), t(v.parents), v.seed, acc, tok, path)
    torch.cuda.synchronize()
    ref = oracle.spec_verify_tree(v.p, v.q, v.draft, v.parents, v.seed)
    assert ref.status == oracle.OK
    acc, tok, path = acc.cpu().numpy(), tok.cpu().numpy(), path.cpu().numpy()
    flagged = differ = 0
    for b in range(v.B):
        f = int(ref.flag_pos[b])
        if f < 0:
            assert acc[b] == ref.accepted_len[b], (b, acc[b], ref.accepted_len[b])
            np.testing.assert_array_equal(tok[b], ref.out_tokens[b], err_msg=f"window {b}")
            np.testing.assert_array_equal(path[b], ref.path[b], err_msg=f"window {b}")
        else:
            # A uniform within 1e-6 of its threshold (peaked rows over 128256 tokens make
            # such draws common): equal up to the flagged position, and counted.
            flagged += 1
            np.testing.assert_array_equal(tok[b, :f], ref.out_tokens[b, :f])
            np.testing.assert_array_equal(path[b, :f], ref.path[b, :f])
            differ += int(acc[b] != ref.accepted_len[b] or not np.array_equal(tok[b], ref.out_tokens[b]))
    print(f"tree70b: {v.B} windows, {flagged} flagged near a threshold, {differ} of them differ")
    # The GPU's sums sit far inside the 1e-6 window, so even flagged windows rarely differ.
    assert differ <= 1
    assert vas_lib.vas_last_device_error() & ~vas_lib.VAS_DEV_RESIDUAL_FALLBACK == 0
