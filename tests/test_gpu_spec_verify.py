"""GPU parity of spec_verify (modified rejection sampling) against the oracle, through the
C ABI (include/vas.h: spec_verify).  Accepted lengths and tokens are bit-exact except for
sequences where a uniform lies within 1e-6 of its threshold (flagged by the oracle)."""
import numpy as np
import pytest
import torch
from scipy.stats import chisquare

import oracle
from verify_attention_spec_gb300 import workloads as wl

from gpu_common import compare_verify

pytestmark = pytest.mark.gpu


def run_gpu_verify(vas, p, q, draft, seed):
    B, k1, V = p.shape
    pd = torch.from_numpy(np.ascontiguousarray(p)).cuda()
    qd = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    xd = torch.from_numpy(np.ascontiguousarray(draft, dtype=np.int32)).cuda()
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, k1), -7, dtype=torch.int32, device="cuda")
    vas.spec_verify(pd, qd, xd, seed, acc, out)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "verify32", "mixed272", "stress70b"])
def test_workload_parity(vas_lib, name):
    v = wl.workload_verify(name)
    ref = oracle.spec_verify(v.p, v.q, v.draft, v.seed)
    assert ref.status == oracle.OK
    acc, out = run_gpu_verify(vas_lib, v.p, v.q, v.draft, v.seed)
    flagged, differ = compare_verify(acc, out, ref)
    print(f"{name}: {v.B} sequences, {flagged} flagged near a boundary, {differ} of them differ")
    # The GPU's prefix sums sit within ~1e-9 of the oracle's, far inside the 1e-6 window,
    # so even among flagged sequences a different outcome should be rare.
    assert differ <= 1
    assert vas_lib.vas_last_device_error() == 0


@pytest.mark.parametrize("V", [1, 7, 1001, 5000])
def test_odd_vocab_and_many_sequences(vas_lib, V):
    """Vocabularies that are not a multiple of four take the scalar load path."""
    v = wl.verify_inputs(300, 3, V, seed=V, p_logit_std=2.0, q_noise_std=1.0)
    ref = oracle.spec_verify(v.p, v.q, v.draft, 77)
    acc, out = run_gpu_verify(vas_lib, v.p, v.q, v.draft, 77)
    compare_verify(acc, out, ref)


def test_k0_plain_sampling_and_seed_changes(vas_lib):
    v = wl.verify_inputs(500, 0, 64, seed=2)
    for seed in (0, 1, 2**63 + 5):
        ref = oracle.spec_verify(v.p, v.q, v.draft, seed)
        acc, out = run_gpu_verify(vas_lib, v.p, v.q, v.draft, seed)
        compare_verify(acc, out, ref)
        assert np.all(acc == 0)


def test_chi_square_million_draws(vas_lib):
    """10^6 GPU draws: the first emitted token follows p_0 (the pages' lossless claim) and
    the bonus token after full acceptance follows p_k (chi-square, p > 0.01)."""
    rng = np.random.default_rng(31)
    B, k, V = 1_000_000, 2, 16
    logits = rng.normal(0, 1.0, size=(k + 1, V))
    p1 = np.exp(logits) / np.exp(logits).sum(-1, keepdims=True)
    qq = np.exp(logits[:k] + rng.normal(0, 0.8, size=(k, V)))
    q1 = qq / qq.sum(-1, keepdims=True)
    p32, q32 = p1.astype(np.float32), q1.astype(np.float32)
    x = np.stack([rng.choice(V, size=B, p=q1[i]) for i in range(k)], axis=1).astype(np.int32)
    pd = torch.from_numpy(p32).cuda().expand(B, k + 1, V).contiguous()
    qd = torch.from_numpy(q32).cuda().expand(B, k, V).contiguous()
    xd = torch.from_numpy(x).cuda()
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, k + 1, dtype=torch.int32, device="cuda")
    vas_lib.spec_verify(pd, qd, xd, 20261202, acc, out)
    torch.cuda.synchronize()
    acc, out = acc.cpu().numpy(), out.cpu().numpy()
    p0 = p32[0].astype(np.float64)
    f0 = np.bincount(out[:, 0], minlength=V)
    assert chisquare(f0, B * p0 / p0.sum()).pvalue > 0.01
    full = acc == k
    pk = p32[k].astype(np.float64)
    fk = np.bincount(out[full, k], minlength=V)
    assert chisquare(fk, full.sum() * pk / pk.sum()).pvalue > 0.01


def test_equal_and_disjoint_and_greedy(vas_lib):
    rng = np.random.default_rng(4)
    B, k, V = 64, 4, 40
    p = rng.dirichlet(np.ones(V), size=(B, k + 1)).astype(np.float32)
    x = rng.integers(0, V, size=(B, k)).astype(np.int32)
    acc, out = run_gpu_verify(vas_lib, p, p[:, :k].copy(), x, 9)
    assert np.all(acc == k) and np.all(out[:, :k] == x)
    # disjoint supports
    pd = np.zeros((B, k + 1, V), np.float32)
    qd = np.zeros((B, k, V), np.float32)
    pd[:, :, :20] = 1 / 20
    qd[:, :, 20:] = 1 / 20
    xd = np.full((B, k), 25, np.int32)
    acc, out = run_gpu_verify(vas_lib, pd, qd, xd, 9)
    assert np.all(acc == 0) and np.all(out[:, 0] < 20) and np.all(out[:, 1:] == -1)
    # one-hot rows: greedy exact matching
    tgt = rng.integers(0, V, size=(B, k + 1))
    drf = np.where(rng.random((B, k)) < 0.6, tgt[:, :k], rng.integers(0, V, size=(B, k))).astype(np.int32)
    po = np.zeros((B, k + 1, V), np.float32)
    qo = np.zeros((B, k, V), np.float32)
    po[np.arange(B)[:, None], np.arange(k + 1)[None], tgt] = 1
    qo[np.arange(B)[:, None], np.arange(k)[None], drf] = 1
    ref = oracle.spec_verify(po, qo, drf, 3)
    acc, out = run_gpu_verify(vas_lib, po, qo, drf, 3)
    np.testing.assert_array_equal(acc, ref.accepted_len)
    np.testing.assert_array_equal(out, ref.out_tokens)


def test_error_paths(vas_lib):
    vas_lib.vas_last_device_error()
    p = np.full((3, 3, 5), 0.2, np.float32)
    q = np.full((3, 2, 5), 0.2, np.float32)
    x = np.array([[0, 1], [7, 1], [2, 3]], np.int32)
    acc, out = run_gpu_verify(vas_lib, p, q, x, 1)
    assert vas_lib.vas_last_device_error() & vas_lib.VAS_DEV_BAD_TOKEN
    assert acc[1] == -1 and np.all(out[1] == -1)
    ref = oracle.spec_verify(p, q, x, 1)
    assert acc[0] == ref.accepted_len[0] and acc[2] == ref.accepted_len[2]
    # an empty row to draw from
    pz = np.zeros((2, 1, 9), np.float32)
    acc, out = run_gpu_verify(vas_lib, pz, np.zeros((2, 0, 9), np.float32), np.zeros((2, 0), np.int32), 1)
    assert vas_lib.vas_last_device_error() & vas_lib.VAS_DEV_EMPTY_ROW
    assert np.all(out[:, 0] == -1) and np.all(acc == 0)


def test_zero_residual_fallback_matches_oracle(vas_lib):
    B, V = 200, 6
    p = np.zeros((B, 2, V), np.float32)
    q = np.zeros((B, 1, V), np.float32)
    p[:, 0, :3] = [0.1, 0.2, 0.1]   # p <= q everywhere: a rejection leaves no residual
    q[:, 0, :3] = [0.3, 0.4, 0.3]
    p[:, 1, :] = 1 / V
    x = np.zeros((B, 1), np.int32)
    ref = oracle.spec_verify(p, q, x, 12)
    vas_lib.vas_last_device_error()
    acc, out = run_gpu_verify(vas_lib, p, q, x, 12)
    compare_verify(acc, out, ref)
    if np.any(ref.fallback):
        assert vas_lib.vas_last_device_error() & vas_lib.VAS_DEV_RESIDUAL_FALLBACK


@pytest.mark.parametrize("V", [1_048_576, 999_999])
def test_largest_vocabularies(vas_lib, V):
    """The largest vocabulary the kernel takes (8 slices of 64 stages of 2048 tokens), and
    one just below it that is not a multiple of 4 (rows not 16-byte aligned: staged by
    plain loads)."""
    v = wl.verify_inputs(3, 2, V, seed=V % 1000, p_logit_std=3.0, q_noise_std=1.5)
    for seed in (5, 6):
        ref = oracle.spec_verify(v.p, v.q, v.draft, seed)
        acc, out = run_gpu_verify(vas_lib, v.p, v.q, v.draft, seed)
        compare_verify(acc, out, ref)
    assert vas_lib.vas_last_device_error() == 0


def test_vocabulary_beyond_the_limit_is_rejected(vas_lib):
    """One token past the largest vocabulary: VAS_E_UNSUPPORTED from the host, nothing
    launched (the outputs keep their contents)."""
    V = 1_048_577
    B, k = 1, 1
    p = torch.full((B, k + 1, V), 1.0 / V, device="cuda")
    q = torch.full((B, k, V), 1.0 / V, device="cuda")
    x = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, k + 1), -7, dtype=torch.int32, device="cuda")
    st = vas_lib._lib.spec_verify(p.data_ptr(), q.data_ptr(), x.data_ptr(), 1, acc.data_ptr(),
                                  out.data_ptr(), B, k, V, None)
    assert st == vas_lib.VAS_E_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(acc == -7) and torch.all(out == -7)


def test_misaligned_rows_take_the_plain_path(vas_lib):
    """p and q starting 4 bytes past a 16-byte boundary (a vocabulary that is a multiple
    of 4 but rows that are not 16-byte aligned) give the same tokens as aligned copies."""
    v = wl.verify_inputs(40, 3, 4096, seed=21, p_logit_std=2.0, q_noise_std=1.0)
    ref = oracle.spec_verify(v.p, v.q, v.draft, 8)
    pbuf = torch.empty(v.p.size + 1, dtype=torch.float32, device="cuda")
    qbuf = torch.empty(v.q.size + 1, dtype=torch.float32, device="cuda")
    pd = pbuf[1:].view(v.p.shape)
    qd = qbuf[1:].view(v.q.shape)
    pd.copy_(torch.from_numpy(v.p))
    qd.copy_(torch.from_numpy(v.q))
    assert pd.data_ptr() % 16 == 4
    xd = torch.from_numpy(v.draft).cuda()
    acc = torch.empty(v.B, dtype=torch.int32, device="cuda")
    out = torch.empty(v.B, v.k + 1, dtype=torch.int32, device="cuda")
    vas_lib.spec_verify(pd, qd, xd, 8, acc, out)
    torch.cuda.synchronize()
    compare_verify(acc.cpu().numpy(), out.cpu().numpy(), ref)
    aligned = run_gpu_verify(vas_lib, v.p, v.q, v.draft, 8)
    np.testing.assert_array_equal(acc.cpu().numpy(), aligned[0])
    np.testing.assert_array_equal(out.cpu().numpy(), aligned[1])


def test_longest_draft_window(vas_lib):
    """k = 255, the largest window: random rows, and rows with q = p, where every draft is
    accepted and the token after them comes from the bonus row p_k."""
    v = wl.verify_inputs(3, 255, 64, seed=255, p_logit_std=2.0, q_noise_std=1.0)
    for seed in (3, 4):
        ref = oracle.spec_verify(v.p, v.q, v.draft, seed)
        acc, out = run_gpu_verify(vas_lib, v.p, v.q, v.draft, seed)
        compare_verify(acc, out, ref)
    same_q = np.ascontiguousarray(v.p[:, :255])
    ref = oracle.spec_verify(v.p, same_q, v.draft, 9)
    acc, out = run_gpu_verify(vas_lib, v.p, same_q, v.draft, 9)
    compare_verify(acc, out, ref)
    assert np.all(acc == 255)
    assert vas_lib.vas_last_device_error() == 0


def test_more_clusters_than_fit_at_once(vas_lib):
    """300 windows over V = 128256: 2400 CTAs, about four times what is resident at once,
    so the clusters run in several waves."""
    v = wl.verify_inputs(300, 2, 128256, seed=300)
    ref = oracle.spec_verify(v.p, v.q, v.draft, 11)
    acc, out = run_gpu_verify(vas_lib, v.p, v.q, v.draft, 11)
    flagged, differ = compare_verify(acc, out, ref)
    assert differ <= 1
    assert vas_lib.vas_last_device_error() == 0
