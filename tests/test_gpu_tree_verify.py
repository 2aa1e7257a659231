"""GPU parity of draft-tree verification (include/vas.h: spec_verify_tree) against the
oracle's walk, through the C ABI: bit-exact except sequences whose uniforms fall within
1e-6 of a threshold (flagged by the oracle; compared up to the flagged position), and
the distribution of the first emitted token over 2^17 sequences against p (chi-square).
"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle

pytestmark = pytest.mark.gpu


def _tree_inputs(rng, B, n, V):
    """Random trees (node i + 1 hangs under a uniform earlier node), target rows
    p [B, n+1, V], draft rows q [B, n, V], and each child drafted from its parent's q."""
    parents = np.stack([np.array([rng.integers(0, i + 1) for i in range(n)], np.int32)
                        for _ in range(B)])
    logits = rng.normal(0, 3.0, (B, n + 1, V))
    p = np.exp(logits - logits.max(-1, keepdims=True))
    p = (p / p.sum(-1, keepdims=True)).astype(np.float32)
    ql = logits[:, :n] + rng.normal(0, 1.5, (B, n, V))
    q = np.exp(ql - ql.max(-1, keepdims=True))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    x = np.zeros((B, n), np.int32)
    for b in range(B):
        for i in range(n):
            u = parents[b, i]
            row = q[b, u].astype(np.float64)
            x[b, i] = rng.choice(V, p=row / row.sum())
    return p, q, x, parents


def _gpu(vas, p, q, x, parents, seed):
    d = "cuda"
    B, n1, V = p.shape
    acc = torch.empty(B, dtype=torch.int32, device=d)
    out = torch.empty(B, n1, dtype=torch.int32, device=d)
    path = torch.empty(B, n1 - 1, dtype=torch.int32, device=d)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(d)
    vas.spec_verify_tree(t(p), t(q), t(x), t(parents), seed, acc, out, path)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy(), path.cpu().numpy()


def _compare(acc, out, path, ref):
    flagged = 0
    for b in range(len(acc)):
        f = int(ref.flag_pos[b])
        if f < 0:
            assert acc[b] == ref.accepted_len[b], (b, acc[b], ref.accepted_len[b])
            np.testing.assert_array_equal(out[b], ref.out_tokens[b], err_msg=f"sequence {b}")
            np.testing.assert_array_equal(path[b], ref.path[b], err_msg=f"sequence {b}")
        else:
            flagged += 1
            np.testing.assert_array_equal(out[b, :f], ref.out_tokens[b, :f])
            np.testing.assert_array_equal(path[b, :f], ref.path[b, :f])
    return flagged


# (200, 4, 50003): more trees than fit eight CTAs each, so the clusters shrink to three
# CTAs, with a vocabulary whose rows are not 16-byte aligned; (8, 255, 64): the largest
# tree.
@pytest.mark.parametrize("B,n,V", [(64, 8, 5), (64, 16, 1000), (32, 63, 257), (64, 6, 128256),
                                   (200, 4, 50003), (8, 255, 64)])
def test_random_trees_match_the_oracle(vas_lib, B, n, V):
    rng = np.random.default_rng(B + n + V)
    p, q, x, parents = _tree_inputs(rng, B, n, V)
    for seed in (7, 2 ** 33 + 1):
        ref = oracle.spec_verify_tree(p, q, x, parents, seed)
        assert ref.status == 0
        acc, out, path = _gpu(vas_lib, p, q, x, parents, seed)
        flagged = _compare(acc, out, path, ref)
        assert flagged <= max(1, B // 10)
    assert vas_lib.vas_last_device_error() & ~vas_lib.VAS_DEV_RESIDUAL_FALLBACK == 0


def test_chain_matches_the_plain_rule(vas_lib):
    """A chain through spec_verify_tree gives the oracle's plain rule (spec_verify)."""
    rng = np.random.default_rng(1)
    B, n, V = 64, 4, 32000
    p, q, x, _ = _tree_inputs(rng, B, n, V)
    chain = np.tile(np.arange(n, dtype=np.int32), (B, 1))
    ref = oracle.spec_verify(p, q, x, 99)
    acc, out, path = _gpu(vas_lib, p, q, x, chain, 99)
    ref.path = np.array([[c + 1 if c < ref.accepted_len[b] else -1 for c in range(n)]
                         for b in range(B)], np.int32)
    _compare(acc, out, path, ref)


def test_first_token_follows_p(vas_lib):
    """2^17 sequences with the same rows, each with its own uniforms and its own three
    candidates drafted from q0: the first emitted token follows p0 (chi-square)."""
    rng = np.random.default_rng(4)
    V, n, B = 8, 3, 1 << 17
    p0 = rng.dirichlet(np.ones(V)).astype(np.float32)
    q0 = rng.dirichlet(np.ones(V)).astype(np.float32)
    p = np.broadcast_to(np.stack([p0] * (n + 1)), (B, n + 1, V)).copy()
    q = np.broadcast_to(np.stack([q0] * n), (B, n, V)).copy()
    parents = np.zeros((B, n), np.int32)  # three candidates under the root
    x = rng.choice(V, size=(B, n), p=q0.astype(np.float64) / q0.sum()).astype(np.int32)
    acc, out, path = _gpu(vas_lib, p, q, x, parents, 12345)
    first = out[:, 0]
    counts = np.bincount(first, minlength=V)
    expected = p0.astype(np.float64) / p0.sum() * B
    keep = expected > 5
    chi = stats.chisquare(counts[keep], expected[keep] * counts[keep].sum() / expected[keep].sum())
    assert chi.pvalue > 0.01, chi


def test_bad_tokens_and_parents(vas_lib):
    rng = np.random.default_rng(2)
    p, q, x, parents = _tree_inputs(rng, 4, 3, 16)
    x[1, 2] = 16
    parents[2, 1] = 2  # node 2's parent would be itself
    vas_lib.vas_last_device_error()
    acc, out, path = _gpu(vas_lib, p, q, x, parents, 5)
    err = vas_lib.vas_last_device_error()
    assert err & vas_lib.VAS_DEV_BAD_TOKEN and err & vas_lib.VAS_DEV_BAD_TREE
    for b in (1, 2):
        assert acc[b] == -1 and np.all(out[b] == -1) and np.all(path[b] == -1)
    # the other sequences are untouched: the oracle on the batch with the bad rows
    # repaired (uniforms depend on the sequence index) agrees on rows 0 and 3
    x2, par2 = x.copy(), parents.copy()
    x2[1, 2] = 0
    par2[2, 1] = 0
    ref = oracle.spec_verify_tree(p, q, x2, par2, 5)
    for b in (0, 3):
        if ref.flag_pos[b] < 0:
            assert acc[b] == ref.accepted_len[b]
            np.testing.assert_array_equal(out[b], ref.out_tokens[b])
            np.testing.assert_array_equal(path[b], ref.path[b])
