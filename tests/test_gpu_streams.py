"""The C ABI's stream argument (include/vas.h): every call runs on the stream it is given,
in order with the work queued there before it, and gives the same bits as on the
default stream."""
import numpy as np
import pytest
import torch

import oracle
from verify_attention_spec_gb300 import workloads as wl

from gpu_common import (compare_attention, compare_verify, oracle_attention, run_gpu_attention,
                        to_device)

pytestmark = pytest.mark.gpu


def test_calls_follow_the_callers_stream(vas_lib):
    if not hasattr(torch.cuda, "_sleep"):
        pytest.skip("torch.cuda._sleep is not available")
    a = wl.workload_attention("verify32")
    ref_o, ref_l = oracle_attention(a)
    v = wl.workload_verify("verify32")
    ref_v = oracle.spec_verify(v.p, v.q, v.draft, v.seed)
    ad = to_device(a)
    base_o, base_l = run_gpu_attention(vas_lib, ad)

    dev = torch.device("cuda")
    p_src = torch.from_numpy(np.ascontiguousarray(v.p)).to(dev)
    q_rows = torch.from_numpy(np.ascontiguousarray(v.q)).to(dev)
    x = torch.from_numpy(np.ascontiguousarray(v.draft, dtype=np.int32)).to(dev)
    q_src = ad.q.clone()
    # The inputs hold zeros until the side stream, after a delay, copies the real ones in.
    # A call launched anywhere but on that stream would read the zeros.
    q_att = torch.zeros_like(ad.q)
    p = torch.zeros_like(p_src)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(40_000_000)  # a fixed spin of 40 M cycles (about 20 ms)
        q_att.copy_(q_src)
        att = wl.AttentionInputs(q_att, ad.k_pages, ad.v_pages, ad.block_table, ad.seq_lens,
                                 ad.query_lens, ad.num_q_heads, ad.num_kv_heads, ad.head_dim,
                                 ad.page_size, ad.kv_dtype, ad.k_scale, ad.v_scale)
        out, lse = run_gpu_attention(vas_lib, att)  # ends with a device synchronize
        torch.cuda._sleep(40_000_000)
        p.copy_(p_src)
        acc = torch.full((v.B,), -7, dtype=torch.int32, device=dev)
        tok = torch.full((v.B, v.k + 1), -7, dtype=torch.int32, device=dev)
        vas_lib.spec_verify(p, q_rows, x, v.seed, acc, tok)
    s.synchronize()
    compare_attention(out, lse, ref_o, ref_l, a.kv_dtype)
    assert torch.equal(out, base_o) and torch.equal(lse, base_l)
    _, differ = compare_verify(acc.cpu().numpy(), tok.cpu().numpy(), ref_v)
    assert differ <= 1
    assert vas_lib.vas_last_device_error() == 0
