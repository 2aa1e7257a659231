"""paged_attn_fwd_static: the attention entry point that takes no workspace, for callers
that cannot allocate device memory (graph capture, plug-in hosts, exhausted allocators).
Its results must match paged_attn_fwd's, call after call, through the C ABI.

This file is named to be collected last: if it fails, a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from verify_attention_spec_gb300 import workloads as wl

from gpu_common import TOL, compare_attention, oracle_attention, run_gpu_attention, to_device

pytestmark = pytest.mark.gpu


def _static_fn(vas):
    f = vas._lib.paged_attn_fwd_static
    f.argtypes = [ctypes.c_void_p] * 8 + [ctypes.POINTER(vas.vas_attn_dims), ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _call_static(vas, a, out, lse):
    dims = vas.attn_dims(a.q, a.k_pages, a.block_table, a.seq_lens)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return _static_fn(vas)(p(a.q), p(a.k_pages), p(a.v_pages), p(a.block_table), p(a.seq_lens),
                           p(a.query_lens), p(out), p(lse), ctypes.byref(dims), stream)


STATIC_BYTES = 32 << 20  # the library's fixed scratch array


@pytest.mark.parametrize("name", ["verify32", "mixed272"])
def test_static_workspace_matches_caller_workspace_twice(vas_lib, name):
    """Two calls in a row.  Against paged_attn_fwd given a caller workspace of the same
    32 MiB the plan is the same, so the results are bit for bit the same; against the
    recommended workspace they agree within the parity tolerance, and the first call is
    also held to the oracle."""
    a = to_device(wl.workload_attention(name))
    same_o, same_l = run_gpu_attention(vas_lib, a, workspace_bytes=STATIC_BYTES)
    rec_o, rec_l = run_gpu_attention(vas_lib, a)
    tol = TOL[a.kv_dtype]
    for call in range(2):  # the shared array keeps the previous call's contents
        out = torch.full_like(a.q, float("nan"))
        lse = torch.full((a.q.shape[0], a.q.shape[1]), float("nan"), device="cuda")
        assert _call_static(vas_lib, a, out, lse) == vas_lib.VAS_OK
        torch.cuda.synchronize()
        assert torch.equal(out, same_o) and torch.equal(lse, same_l)
        o, r = out.double(), rec_o.double()
        assert (o - r).abs().max().item() <= tol["max_abs"]
        assert ((o - r).norm() / r.norm()).item() <= tol["rel_l2"]
        assert (lse - rec_l).abs().max().item() <= tol["lse"]
        if call == 0:
            ref_o, ref_l = oracle_attention(a)
            compare_attention(out, lse, ref_o, ref_l, a.kv_dtype)
    assert vas_lib.vas_last_device_error() == 0


def test_static_workspace_rejects_batches_beyond_its_size(vas_lib):
    a = to_device(wl.workload_attention("tiny"))
    dims = vas_lib.attn_dims(a.q, a.k_pages, a.block_table, a.seq_lens)
    dims.num_seqs = 2_000_000       # plan space far beyond 32 MiB; nothing is launched
    dims.total_q_tokens = 2_000_000
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = _static_fn(vas_lib)(p(a.q), p(a.k_pages), p(a.v_pages), p(a.block_table), p(a.seq_lens),
                             p(a.query_lens), p(a.q), p(a.q), ctypes.byref(dims), None)
    assert st == vas_lib.VAS_E_WORKSPACE
