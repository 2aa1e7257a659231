"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and the
oracle on the same seeded inputs, and compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from verify_attention_spec_gb300 import workloads as wl

# Attention tolerances (output vs the float64 oracle): max-abs 1e-2 and relative L2 5e-3
# for bf16 storage, 1e-5 for fp32 storage.  lse is fp32 in both cases; its error is that
# of an fp32 dot product of length D (bf16 inputs are exact), so 2e-3 / 2e-5 absolute.
# A bf16 output cannot come closer to an exact value than half the bf16 spacing there,
# which passes 1e-2 from |value| = 4 on (spacing 2^-5): for those elements the bound is
# that half spacing plus the 2e-3 the computation is allowed below 4 (1e-2 - 2^-7).
TOL = {wl.BF16: dict(max_abs=1e-2, rel_l2=5e-3, lse=2e-3, format_slack=2e-3),
       wl.F32: dict(max_abs=1e-5, rel_l2=1e-5, lse=2e-5, format_slack=None)}
# Quantised pools: the oracle decodes the same codes exactly, and the output is bf16.
TOL[wl.FP8] = TOL[wl.INT8] = TOL[wl.BF16]


def bf16_half_spacing(x: np.ndarray) -> np.ndarray:
    """Half the gap between adjacent bf16 numbers (8 significant bits) at |x|."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 8)


def to_device(a: wl.AttentionInputs, device="cuda") -> wl.AttentionInputs:
    mv = lambda t: None if t is None else t.to(device, non_blocking=False).contiguous()
    return wl.AttentionInputs(mv(a.q), mv(a.k_pages), mv(a.v_pages), mv(a.block_table),
                              mv(a.seq_lens), mv(a.query_lens), a.num_q_heads, a.num_kv_heads,
                              a.head_dim, a.page_size, a.kv_dtype, mv(a.k_scale), mv(a.v_scale))


def _quant(a: wl.AttentionInputs):
    return a.kv_dtype if a.kv_dtype in wl.QUANTIZED else None


def run_gpu_attention(vas, a: wl.AttentionInputs, workspace_bytes=None, out=None, lse=None,
                      tree_masks=None):
    """One attention call through the C ABI: paged_attn_fwd, paged_attn_fwd_tree (with
    tree_masks) or paged_attn_fwd_quant (quantised pools)."""
    d = a.q.device
    if out is None:
        out = torch.empty_like(a.q)
    if lse is None:
        lse = torch.empty(a.q.shape[0], a.q.shape[1], dtype=torch.float32, device=d)
    dims = vas.attn_dims(a.q, a.k_pages, a.block_table, a.seq_lens, quant=_quant(a))
    ws = vas.alloc_workspace(dims, device=d, nbytes=workspace_bytes)
    tm = None
    if tree_masks is not None:
        tm = torch.from_numpy(np.ascontiguousarray(tree_masks).view(np.int64)).to(d)
    if _quant(a):
        vas.paged_attn_fwd_quant(a.q, a.k_pages, a.v_pages, a.k_scale, a.v_scale, a.block_table,
                                 a.seq_lens, a.query_lens, out, lse, ws, quant=_quant(a),
                                 tree_mask=tm, dims=dims)
    elif tm is not None:
        vas.paged_attn_fwd_tree(a.q, a.k_pages, a.v_pages, a.block_table, a.seq_lens,
                                a.query_lens, tm, out, lse, ws, dims=dims)
    else:
        vas.paged_attn_fwd(a.q, a.k_pages, a.v_pages, a.block_table, a.seq_lens, a.query_lens,
                           out, lse, ws, dims=dims)
    torch.cuda.synchronize()
    return out, lse


def run_gpu_attention_tree(vas, a: wl.AttentionInputs, masks: np.ndarray, workspace_bytes=None):
    return run_gpu_attention(vas, a, workspace_bytes=workspace_bytes, tree_masks=masks)


# The kernel's tree encoding (one uint64 of proper ancestors per query token) has a single
# definition, in the input generator; the tests use that one.
ancestor_masks = wl.ancestor_bits


def oracle_attention(a: wl.AttentionInputs, parents=None):
    np_ = lambda t: t.detach().cpu().contiguous().numpy()
    if a.kv_dtype in wl.QUANTIZED:
        fmt = oracle.Q_E4M3 if a.kv_dtype == wl.FP8 else oracle.Q_INT8
        return oracle.paged_attn_quant(wl.bf16_bits(a.q.cpu()), np_(a.k_pages), np_(a.v_pages),
                                       np_(a.k_scale), np_(a.v_scale), np_(a.block_table),
                                       np_(a.seq_lens), np_(a.query_lens), fmt=fmt,
                                       parents=parents)
    code = oracle.BF16 if a.kv_dtype == wl.BF16 else oracle.F32
    st = lambda t: wl.storage_for_oracle(t, a.kv_dtype)
    return oracle.paged_attn(st(a.q), st(a.k_pages), st(a.v_pages), a.block_table.cpu().numpy(),
                             a.seq_lens.cpu().numpy(), a.query_lens.cpu().numpy(), dtype_code=code,
                             parents=parents)


def compare_attention(out, lse, ref_out, ref_lse, kv_dtype, rows=None):
    tol = TOL[kv_dtype]
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    err = np.abs(o - ref_out)
    max_abs = float(err.max()) if err.size else 0.0
    rel_l2 = float(np.linalg.norm(o - ref_out) / max(np.linalg.norm(ref_out), 1e-30))
    lse_err = float(np.abs(l - ref_lse).max()) if l.size else 0.0
    bound = np.full(err.shape, tol["max_abs"])
    if tol["format_slack"] is not None:
        bound = np.maximum(bound, bf16_half_spacing(ref_out) + tol["format_slack"])
    if err.size and not np.all(err <= bound):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"max-abs {max_abs}: element {i} off by {err[i]} "
                             f"(bound {bound[i]}, exact {ref_out[i]})")
    assert rel_l2 <= tol["rel_l2"], f"rel-L2 {rel_l2}"
    assert lse_err <= tol["lse"], f"lse {lse_err}"
    return dict(max_abs=max_abs, rel_l2=rel_l2, lse=lse_err)


def query_slice_inputs(a: wl.AttentionInputs, seq: int, j0: int, n: int):
    """Query tokens j0 .. j0+n-1 of sequence `seq` as a problem of their own: context
    L - ql + j0 + n (the same pages, so the same positions L - ql + j), query length n.
    Returns (inputs on the CPU, the rows of the full problem they correspond to)."""
    bt = a.block_table.cpu().numpy()
    lens = a.seq_lens.cpu().numpy()
    qlens = a.query_lens.cpu().numpy()
    row0 = int(np.concatenate([[0], np.cumsum(qlens)])[seq])
    L, ql, P = int(lens[seq]), int(qlens[seq]), a.page_size
    Ls = L - ql + j0 + n
    npg = (Ls + P - 1) // P
    ids = torch.from_numpy(bt[seq, :npg].astype(np.int64)).to(a.k_pages.device)
    rows = np.arange(row0 + j0, row0 + j0 + n)
    sc = lambda t: None if t is None else t[ids.to(t.device)].cpu()
    sub = wl.AttentionInputs(a.q[torch.from_numpy(rows).to(a.q.device)].cpu(), a.k_pages[ids].cpu(),
                             a.v_pages[ids].cpu(), torch.arange(npg, dtype=torch.int32)[None, :],
                             torch.tensor([Ls], dtype=torch.int32), torch.tensor([n], dtype=torch.int32),
                             a.num_q_heads, a.num_kv_heads, a.head_dim, a.page_size, a.kv_dtype,
                             sc(a.k_scale), sc(a.v_scale))
    return sub, rows


def compare_verify(acc, out, ref):
    """Bit-exact except sequences the oracle flags (a uniform within 1e-6 of its
    threshold): those must agree before the flagged position, and are counted.
    Returns (flagged, flagged sequences whose outputs differ)."""
    acc = np.asarray(acc)
    out = np.asarray(out)
    flagged = differ = 0
    for b in range(len(acc)):
        f = int(ref.flag_pos[b])
        if f < 0:
            assert acc[b] == ref.accepted_len[b], (b, acc[b], ref.accepted_len[b])
            np.testing.assert_array_equal(out[b], ref.out_tokens[b], err_msg=f"sequence {b}")
        else:
            flagged += 1
            np.testing.assert_array_equal(out[b, :f], ref.out_tokens[b, :f])
            assert acc[b] >= min(f, ref.accepted_len[b])
            if acc[b] != ref.accepted_len[b] or not np.array_equal(out[b], ref.out_tokens[b]):
                differ += 1
    return flagged, differ
