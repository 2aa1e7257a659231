"""Pins for the oracle's paged attention (CPU only).

The oracle computes softmax attention of each query row over its sequence's KV, read
through the block table ("PagedAttention: making the KV cache schedulable" on the
syslabs.in page; "Anatomy of the KV Cache" on the tempatgunting.com page).  Paging must
be invisible to the result, so the main witness is dense, unpaged attention from a
library routine (torch's scaled_dot_product_attention in float64) on KV laid out
contiguously and scattered into a permuted pool by the layout's definition.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from verify_attention_spec_gb300 import workloads as wl


def scatter_to_pool(dense_k, dense_v, page_size, num_pages, rng):
    """Place per-sequence dense KV [L, Hkv, D] into a pool [num_pages, P, Hkv, D] of
    random pages.  Returns (k_pool, v_pool, block_table)."""
    Hkv, D = dense_k[0].shape[1:]
    npages = [(k.shape[0] + page_size - 1) // page_size for k in dense_k]
    perm = rng.permutation(num_pages)
    kp = rng.standard_normal((num_pages, page_size, Hkv, D))  # garbage in unused slots
    vp = rng.standard_normal((num_pages, page_size, Hkv, D))
    bt = np.full((len(dense_k), max(npages)), -1, dtype=np.int32)
    off = 0
    for i, (k, v) in enumerate(zip(dense_k, dense_v)):
        ids = perm[off:off + npages[i]]
        off += npages[i]
        bt[i, :len(ids)] = ids
        for t in range(k.shape[0]):
            kp[ids[t // page_size], t % page_size] = k[t]
            vp[ids[t // page_size], t % page_size] = v[t]
    return kp, vp, bt


def dense_reference(qs, dense_k, dense_v, qlens, Hq, Hkv, scale):
    """Library witness: float64 SDPA with an explicit boolean mask, per sequence."""
    outs, lses = [], []
    group = Hq // Hkv
    for q, k, v, ql in zip(qs, dense_k, dense_v, qlens):
        L = k.shape[0]
        qt = torch.from_numpy(q).permute(1, 0, 2)                       # [Hq, ql, D]
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(group, 0)  # [Hq, L, D]
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(group, 0)
        pos = L - ql + torch.arange(ql)
        mask = torch.arange(L)[None, :] <= pos[:, None]                   # [ql, L]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                             scale=scale)
        outs.append(o.permute(1, 0, 2).numpy())
        sc = torch.einsum("hqd,hkd->hqk", qt, kt).numpy() * scale
        sc = np.where(mask.numpy()[None], sc, -np.inf)
        lses.append(logsumexp(sc, axis=-1).T)                            # [ql, Hq]
    return np.concatenate(outs), np.concatenate(lses)


def random_case(rng, lens, qlens, Hq, Hkv, D, P, extra_pages=3):
    dense_k = [rng.standard_normal((L, Hkv, D)) for L in lens]
    dense_v = [rng.standard_normal((L, Hkv, D)) for L in lens]
    qs = [rng.standard_normal((ql, Hq, D)) for ql in qlens]
    num_pages = sum((L + P - 1) // P for L in lens) + extra_pages
    kp, vp, bt = scatter_to_pool(dense_k, dense_v, P, num_pages, rng)
    return qs, dense_k, dense_v, kp, vp, bt


@pytest.mark.parametrize("lens,qlens,Hq,Hkv,D,P", [
    ([17, 40, 63, 100], [1, 4, 1, 4], 4, 2, 64, 16),
    ([1, 5, 16, 33], [1, 5, 2, 8], 8, 2, 32, 16),
    ([70, 9], [3, 1], 6, 6, 16, 32),
    ([31], [1], 2, 1, 8, 8),
])
def test_oracle_equals_dense_sdpa(lens, qlens, Hq, Hkv, D, P):
    rng = np.random.default_rng(sum(lens) + Hq)
    qs, dk, dv, kp, vp, bt = random_case(rng, lens, qlens, Hq, Hkv, D, P)
    scale = 1.0 / np.sqrt(D)
    out, lse = oracle.paged_attn(np.concatenate(qs), kp, vp, bt, lens, qlens,
                                 dtype_code=oracle.F64)
    ref_o, ref_l = dense_reference(qs, dk, dv, qlens, Hq, Hkv, scale)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_paging_is_invisible_to_permutation_of_pages():
    rng = np.random.default_rng(5)
    lens, qlens = [50, 23, 7], [4, 1, 2]
    qs, dk, dv, kp, vp, bt = random_case(rng, lens, qlens, 4, 2, 16, 8)
    q = np.concatenate(qs)
    o1, l1 = oracle.paged_attn(q, kp, vp, bt, lens, qlens, dtype_code=oracle.F64)
    perm = rng.permutation(kp.shape[0])            # page i moves to slot perm[i]
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    o2, l2 = oracle.paged_attn(q, kp2, vp2, bt2, lens, qlens, dtype_code=oracle.F64)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    qs, dk, dv, kp, vp, bt = random_case(rng, [1], [1], 4, 2, 8, 4)
    out, lse = oracle.paged_attn(qs[0], kp, vp, bt, [1], [1], dtype_code=oracle.F64)
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], dv[0][0, h // 2])
        np.testing.assert_allclose(lse[0, h], qs[0][0, h] @ dk[0][0, h // 2] / np.sqrt(8),
                                   rtol=0, atol=1e-14)


def test_constant_values_pass_through():
    rng = np.random.default_rng(2)
    lens, qlens = [45, 12], [3, 1]
    qs, dk, dv, kp, vp, bt = random_case(rng, lens, qlens, 2, 1, 8, 8)
    c = rng.standard_normal(8)
    vp[:] = c
    out, _ = oracle.paged_attn(np.concatenate(qs), kp, vp, bt, lens, qlens, dtype_code=oracle.F64)
    np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=0, atol=1e-13)


def test_causal_window_and_gqa_mapping():
    """V = one-hot of the token position (per KV head, offset by the head) makes out the
    attention weights themselves: row j of a verify sequence must put zero weight past
    its own position L - ql + j and positive weight on every position up to it, and
    query head h must read KV head h // (Hq / Hkv)."""
    rng = np.random.default_rng(3)
    L, ql, Hq, Hkv, P = 20, 5, 4, 2, 8
    D = 2 * L
    k = rng.standard_normal((L, Hkv, D))
    v = np.zeros((L, Hkv, D))
    for t in range(L):
        for g in range(Hkv):
            v[t, g, g * L + t] = 1.0
    q = rng.standard_normal((ql, Hq, D))
    kp, vp, bt = scatter_to_pool([k], [v], P, 4, rng)
    out, _ = oracle.paged_attn(q, kp, vp, bt, [L], [ql], dtype_code=oracle.F64)
    for j in range(ql):
        pos = L - ql + j
        for h in range(Hq):
            g = h // (Hq // Hkv)
            wts = out[j, h, g * L:(g + 1) * L]
            assert np.all(wts[:pos + 1] > 0)
            assert np.all(wts[pos + 1:] == 0)
            other = out[j, h, (1 - g) * L:(2 - g) * L]
            assert np.all(other == 0)
            np.testing.assert_allclose(wts.sum(), 1.0, rtol=0, atol=1e-14)


def test_bf16_and_f32_storage_decode_exactly():
    """The oracle's bf16 path (raw bits) equals its f64 path on torch's own upcast."""
    rng = np.random.default_rng(4)
    lens, qlens = [33, 10], [2, 1]
    qs, dk, dv, kp, vp, bt = random_case(rng, lens, qlens, 4, 2, 16, 8)
    q = np.concatenate(qs)
    for dt, code in [(torch.bfloat16, oracle.BF16), (torch.float32, oracle.F32)]:
        tq, tk, tv = (torch.from_numpy(a).to(dt) for a in (q, kp, vp))
        if dt == torch.bfloat16:
            raw = [wl.bf16_bits(t) for t in (tq, tk, tv)]
        else:
            raw = [t.numpy() for t in (tq, tk, tv)]
        o1, l1 = oracle.paged_attn(*raw, bt, lens, qlens, dtype_code=code)
        o2, l2 = oracle.paged_attn(tq.double().numpy(), tk.double().numpy(), tv.double().numpy(),
                                   bt, lens, qlens, dtype_code=oracle.F64)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_tiny_workload_against_dense():
    """The tiny fp32 workload (4 sequences, 4/2 heads, d=64, page 16, 64-page pool)."""
    a = wl.workload_attention("tiny")
    bt = a.block_table.numpy()
    lens, qlens = a.seq_lens.numpy(), a.query_lens.numpy()
    kp, vp = a.k_pages.double().numpy(), a.v_pages.double().numpy()
    q = a.q.double().numpy()
    out, lse = oracle.paged_attn(a.q.numpy(), a.k_pages.numpy(), a.v_pages.numpy(), bt, lens,
                                 qlens, dtype_code=oracle.F32)
    # dense witness built from the pool by the layout's definition
    dk, dv, qs, r = [], [], [], 0
    for i, (L, ql) in enumerate(zip(lens, qlens)):
        t = np.arange(L)
        dk.append(kp[bt[i, t // 16], t % 16])
        dv.append(vp[bt[i, t // 16], t % 16])
        qs.append(q[r:r + ql])
        r += ql
    ref_o, ref_l = dense_reference(qs, dk, dv, qlens, 4, 2, 1 / 8)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_rejects_bad_page_and_lengths():
    rng = np.random.default_rng(6)
    qs, dk, dv, kp, vp, bt = random_case(rng, [20], [1], 2, 1, 8, 8)
    bad = bt.copy()
    bad[0, 1] = kp.shape[0]
    with pytest.raises(ValueError):
        oracle.paged_attn(qs[0], kp, vp, bad, [20], [1], dtype_code=oracle.F64)
    with pytest.raises(ValueError):
        oracle.paged_attn(np.zeros((21, 2, 8)), kp, vp, bt, [20], [21], dtype_code=oracle.F64)


# ---- draft trees ("Tree Attention & Medusa Heads" on the neuralmasteryai.com page) -----
def _tree_case(rng, L, ql, Hq=4, Hkv=2, D=16, P=8):
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    q = rng.standard_normal((ql, Hq, D))
    kp, vp, bt = scatter_to_pool([k], [v], P, (L + P - 1) // P + 2, rng)
    return q, k, v, kp, vp, bt


def test_tree_chain_is_the_causal_window():
    rng = np.random.default_rng(40)
    L, ql = 37, 6
    q, k, v, kp, vp, bt = _tree_case(rng, L, ql)
    args = (q, kp, vp, bt, np.array([L]), np.array([ql]))
    o_c, l_c = oracle.paged_attn(*args, dtype_code=oracle.F64)
    o_t, l_t = oracle.paged_attn(*args, dtype_code=oracle.F64,
                                 parents=np.arange(ql, dtype=np.int32) - 1)
    np.testing.assert_array_equal(o_t, o_c)
    np.testing.assert_array_equal(l_t, l_c)


def test_tree_node_is_decode_over_its_path():
    """Each node of a random tree sees the context and its root-to-node path: the same as
    one decode query over a sequence made of exactly those tokens, in order, placed in a
    fresh paged pool (the causal oracle, pinned above)."""
    rng = np.random.default_rng(41)
    L, ql, P = 45, 9, 8
    Hq, Hkv, D = 4, 2, 16
    q, k, v, kp, vp, bt = _tree_case(rng, L, ql, Hq, Hkv, D, P)
    parents = np.array([-1] + [int(rng.integers(-1, j)) for j in range(1, ql)], dtype=np.int32)
    parents[3] = -1  # at least two roots
    o_t, l_t = oracle.paged_attn(q, kp, vp, bt, np.array([L]), np.array([ql]),
                                 dtype_code=oracle.F64, parents=parents)
    ctx = L - ql
    for j in range(ql):
        path, a = [], j
        while a >= 0:
            path.append(a)
            a = parents[a]
        toks = list(range(ctx)) + [ctx + a for a in reversed(path)]
        kp2, vp2, bt2 = scatter_to_pool([k[toks]], [v[toks]], P,
                                        (len(toks) + P - 1) // P + 1, rng)
        o_d, l_d = oracle.paged_attn(q[j:j + 1], kp2, vp2, bt2, np.array([len(toks)]),
                                     np.array([1]), dtype_code=oracle.F64)
        np.testing.assert_allclose(o_t[j], o_d[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l_t[j], l_d[0], rtol=0, atol=1e-12)


def test_tree_parent_after_child_is_rejected():
    rng = np.random.default_rng(42)
    q, k, v, kp, vp, bt = _tree_case(rng, 20, 4)
    with pytest.raises(ValueError):
        oracle.paged_attn(q, kp, vp, bt, np.array([20]), np.array([4]), dtype_code=oracle.F64,
                          parents=np.array([-1, 0, 3, 1], dtype=np.int32))


def test_tree_batched_sequences_match_alone():
    """Two sequences with their own trees in one call give what each gives alone (the
    parents index the sequence's own query tokens)."""
    rng = np.random.default_rng(43)
    P, Hq, Hkv, D = 8, 4, 2, 16
    L = [30, 26]
    ql = [5, 7]
    par = [np.array([-1, 0, 0, 1, -1], dtype=np.int32),
           np.array([-1, 0, 1, 1, 3, -1, 5], dtype=np.int32)]
    ks = [rng.standard_normal((l, Hkv, D)) for l in L]
    vs = [rng.standard_normal((l, Hkv, D)) for l in L]
    qs = [rng.standard_normal((n, Hq, D)) for n in ql]
    kp, vp, bt = scatter_to_pool(ks, vs, P, sum((l + P - 1) // P for l in L) + 2, rng)
    o, l = oracle.paged_attn(np.concatenate(qs), kp, vp, bt, np.array(L), np.array(ql),
                             dtype_code=oracle.F64, parents=np.concatenate(par))
    r = 0
    for i in range(2):
        kp1, vp1, bt1 = scatter_to_pool([ks[i]], [vs[i]], P, (L[i] + P - 1) // P, rng)
        o1, l1 = oracle.paged_attn(qs[i], kp1, vp1, bt1, np.array([L[i]]), np.array([ql[i]]),
                                   dtype_code=oracle.F64, parents=par[i])
        np.testing.assert_array_equal(o[r:r + ql[i]], o1)
        np.testing.assert_array_equal(l[r:r + ql[i]], l1)
        r += ql[i]
