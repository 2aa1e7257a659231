"""Pins for the oracle's modified rejection sampling (CPU only).

The rule (neuralmasteryai.com, "The Modified Rejection Sampling Algorithm"; syslabs.in,
"The core idea"; tempatgunting.com, "Speculative Decoding: Turning Verification
Parallelism into Latency Wins"): accept draft x_i when r <= min(1, p(x_i)/q(x_i)), halt
at the first rejection and resample from max(0, p - q) normalised, or draw a bonus token
from the last target row when every draft is accepted.  The pages' theorem is that the
emitted tokens are distributed exactly as sampling from the target alone.

Exact enumeration: probabilities are multiples of 1/16 and every draft probability is
0 or a power of two, with total variation 1/16, 2/16, 4/16 or 8/16.  Then every ratio
p/q and every normalised CDF step of the residual or bonus row is a multiple of 1/16, so
each uniform can be integrated exactly on the 32 midpoints (2i+1)/64: no midpoint sits
on a threshold, and the oracle's output is constant on every cell.
"""
import numpy as np
import pytest
from scipy.stats import chisquare

import oracle

N = 32
MID = (np.arange(N) + 0.5) / N


def power_of_two_row(rng, V):
    parts = [16]
    want = int(rng.integers(1, min(V, 6) + 1))
    while len(parts) < want:
        big = [i for i, v in enumerate(parts) if v > 1]
        if not big:
            break
        i = big[int(rng.integers(len(big)))]
        h = parts.pop(i) // 2
        parts += [h, h]
    row = np.zeros(V, dtype=np.int64)
    row[rng.permutation(V)[:len(parts)]] = parts
    return row


def dyadic_pair(rng, V):
    """(p, q) in units of 1/16 with q entries in {0, 1, 2, 4, 8, 16} and
    sum max(0, p - q) in {1, 2, 4, 8}."""
    while True:
        q = power_of_two_row(rng, V)
        p = rng.multinomial(16, np.full(V, 1.0 / V))
        if np.maximum(p - q, 0).sum() in (1, 2, 4, 8):
            return p, q


def as_prob(units):
    return (np.asarray(units, dtype=np.float64) / 16.0).astype(np.float32)


def run_grid(p, q, draft, r_axes, s_axes, k):
    """Evaluate the oracle on the product grid of the given axes.  r_axes/s_axes map an
    axis index to either 'grid' or a fixed value.  Returns (acc, out, cell weight)."""
    grids = []
    names = [("r", i) for i in range(k)] + [("s", j) for j in range(k + 1)]
    spec = {("r", i): r_axes[i] for i in range(k)}
    spec.update({("s", j): s_axes[j] for j in range(k + 1)})
    varying = [n for n in names if isinstance(spec[n], str)]
    mesh = np.meshgrid(*[MID] * len(varying), indexing="ij")
    B = N ** len(varying)
    cols = {}
    for n, m in zip(varying, mesh):
        cols[n] = m.ravel()
    for n in names:
        if n not in cols:
            cols[n] = np.full(B, spec[n])
    r = np.stack([cols[("r", i)] for i in range(k)], axis=1) if k else np.zeros((B, 0))
    s = np.stack([cols[("s", j)] for j in range(k + 1)], axis=1)
    P = np.ascontiguousarray(np.broadcast_to(p, (B,) + p.shape))
    Q = np.ascontiguousarray(np.broadcast_to(q, (B,) + q.shape))
    X = np.ascontiguousarray(np.broadcast_to(np.asarray(draft, dtype=np.int32), (B, k)))
    res = oracle.spec_verify_given_uniforms(P, Q, X, r, s)
    assert res.status == oracle.OK
    return res.accepted_len, res.out_tokens, 1.0 / B


@pytest.mark.parametrize("seed", range(6))
def test_exact_enumeration_k1_first_token_is_target_distribution(seed):
    rng = np.random.default_rng(100 + seed)
    V = int(rng.integers(2, 9))
    p0u, q0u = dyadic_pair(rng, V)
    p1u = rng.multinomial(16, np.full(V, 1.0 / V))
    p = np.stack([as_prob(p0u), as_prob(p1u)])
    q = as_prob(q0u)[None]
    first = np.zeros(V)
    acc1 = 0.0
    bonus = np.zeros(V)
    for x0 in range(V):
        if q0u[x0] == 0:
            continue
        acc, out, w = run_grid(p, q, [x0], ["grid"], ["grid", "grid"], 1)
        wq = q0u[x0] / 16.0 * w
        np.add.at(first, out[:, 0], wq)
        a = acc == 1
        acc1 += wq * a.sum()
        np.add.at(bonus, out[a, 1], wq)
    p0, q0, p1 = p0u / 16.0, q0u / 16.0, p1u / 16.0
    alpha = np.minimum(p0, q0).sum()
    np.testing.assert_allclose(first, p0, rtol=0, atol=1e-12)        # lossless
    np.testing.assert_allclose(acc1, alpha, rtol=0, atol=1e-12)      # acceptance rate
    np.testing.assert_allclose(bonus, alpha * p1, rtol=0, atol=1e-12)  # bonus from p_k


@pytest.mark.parametrize("seed", range(3))
def test_exact_enumeration_k2_second_token_follows_second_row(seed):
    """Given the first draft accepted, the second emitted token is distributed as p_1
    (accepted draft or residual of row 1): P(acc>=1, y0=a, y1=b) = min(p0,q0)(a) p1(b)."""
    rng = np.random.default_rng(200 + seed)
    V = int(rng.integers(2, 6))
    p0u, q0u = dyadic_pair(rng, V)
    p1u, q1u = dyadic_pair(rng, V)
    p2u = rng.multinomial(16, np.full(V, 1.0 / V))
    p = np.stack([as_prob(p0u), as_prob(p1u), as_prob(p2u)])
    q = np.stack([as_prob(q0u), as_prob(q1u)])
    joint = np.zeros((V, V))
    both = 0.0
    for x0 in range(V):
        for x1 in range(V):
            if q0u[x0] == 0 or q1u[x1] == 0:
                continue
            # s_0 is only used after a rejection at 0 and s_2 only for the bonus token,
            # neither of which enters the events below: hold them fixed.
            acc, out, w = run_grid(p, q, [x0, x1], ["grid", "grid"], [0.5, "grid", 0.5], 2)
            wq = q0u[x0] * q1u[x1] / 256.0 * w
            m = acc >= 1
            np.add.at(joint, (out[m, 0], out[m, 1]), wq)
            both += wq * (acc == 2).sum()
    p0, q0, p1, q1 = p0u / 16, q0u / 16, p1u / 16, q1u / 16
    np.testing.assert_allclose(joint, np.outer(np.minimum(p0, q0), p1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(both, np.minimum(p0, q0).sum() * np.minimum(p1, q1).sum(),
                               rtol=0, atol=1e-12)


def test_monte_carlo_with_philox_k3():
    """Full oracle (Philox uniforms): first token ~ p_0; bonus token given all accepted ~ p_3."""
    rng = np.random.default_rng(9)
    B, k, V = 60000, 3, 12
    logits = rng.normal(0, 1.0, size=(k + 1, V))
    p1 = np.exp(logits) / np.exp(logits).sum(-1, keepdims=True)
    ql = np.exp(logits[:k] + rng.normal(0, 0.7, size=(k, V)))
    q1 = ql / ql.sum(-1, keepdims=True)
    p = np.broadcast_to(p1.astype(np.float32), (B, k + 1, V))
    q = np.broadcast_to(q1.astype(np.float32), (B, k, V))
    x = np.stack([rng.choice(V, size=B, p=q1[i] / q1[i].sum()) for i in range(k)], axis=1)
    res = oracle.spec_verify(p, q, x, seed=4242)
    assert res.status == oracle.OK
    f0 = np.bincount(res.out_tokens[:, 0], minlength=V)
    assert chisquare(f0, B * p1[0] / p1[0].sum()).pvalue > 1e-3
    allacc = res.accepted_len == k
    fb = np.bincount(res.out_tokens[allacc, k], minlength=V)
    assert chisquare(fb, allacc.sum() * p1[k] / p1[k].sum()).pvalue > 1e-3
    alpha = np.minimum(p1[:k], q1).sum(-1)
    assert abs(allacc.mean() - np.prod(alpha)) < 5 * np.sqrt(np.prod(alpha) / B)


def test_equal_distributions_accept_everything():
    rng = np.random.default_rng(11)
    B, k, V = 50, 4, 33
    p = rng.dirichlet(np.ones(V), size=(B, k + 1)).astype(np.float32)
    q = p[:, :k].copy()
    x = rng.integers(0, V, size=(B, k))
    res = oracle.spec_verify(p, q, x, seed=3)
    assert np.all(res.accepted_len == k)
    np.testing.assert_array_equal(res.out_tokens[:, :k], x)
    assert np.all(p[np.arange(B), k, res.out_tokens[:, k]] > 0)


def test_disjoint_supports_reject_first_and_draw_from_target():
    B, k, V = 400, 3, 8
    p = np.zeros((B, k + 1, V), dtype=np.float32)
    q = np.zeros((B, k, V), dtype=np.float32)
    p[:, :, :4] = np.array([0.1, 0.2, 0.3, 0.4], dtype=np.float32)
    q[:, :, 4:] = 0.25
    x = np.full((B, k), 5, dtype=np.int32)
    res = oracle.spec_verify(p, q, x, seed=17)
    assert np.all(res.accepted_len == 0)
    assert np.all(res.out_tokens[:, 0] < 4)
    assert np.all(res.out_tokens[:, 1:] == -1)


def test_one_hot_rows_reduce_to_greedy_matching():
    """Temperature 0 (tempatgunting.com FAQ: "reduces to exact token matching")."""
    rng = np.random.default_rng(12)
    B, k, V = 200, 5, 10
    tgt = rng.integers(0, V, size=(B, k + 1))
    drf = np.where(rng.random((B, k)) < 0.7, tgt[:, :k], rng.integers(0, V, size=(B, k)))
    p = np.zeros((B, k + 1, V), dtype=np.float32)
    q = np.zeros((B, k, V), dtype=np.float32)
    p[np.arange(B)[:, None], np.arange(k + 1)[None], tgt] = 1.0
    q[np.arange(B)[:, None], np.arange(k)[None], drf] = 1.0
    res = oracle.spec_verify(p, q, drf, seed=5)
    for b in range(B):
        mism = np.nonzero(drf[b] != tgt[b, :k])[0]
        j = int(mism[0]) if len(mism) else k
        assert res.accepted_len[b] == j
        np.testing.assert_array_equal(res.out_tokens[b, :j + 1], tgt[b, :j + 1])
        assert np.all(res.out_tokens[b, j + 1:] == -1)


def test_k0_is_plain_sampling_from_first_row():
    rng = np.random.default_rng(13)
    B, V = 40000, 6
    p1 = rng.dirichlet(np.ones(V))
    p = np.broadcast_to(p1.astype(np.float32), (B, 1, V))
    res = oracle.spec_verify(p, np.zeros((B, 0, V), np.float32), np.zeros((B, 0), np.int32), seed=8)
    assert np.all(res.accepted_len == 0)
    f = np.bincount(res.out_tokens[:, 0], minlength=V)
    assert chisquare(f, B * p1 / p1.sum()).pvalue > 1e-3


def test_inverse_cdf_convention_and_flags():
    """Smallest x whose inclusive prefix exceeds s*S; zero-weight tokens never drawn;
    a uniform within the window of a CDF step is flagged."""
    p = np.array([[[0.25, 0.0, 0.25, 0.5]]], dtype=np.float32)
    q = np.zeros((1, 0, 4), np.float32)
    x = np.zeros((1, 0), np.int32)
    for s, want in [(0.1, 0), (0.2499, 0), (0.2501, 2), (0.49, 2), (0.51, 3), (0.999, 3)]:
        res = oracle.spec_verify_given_uniforms(p, q, x, np.zeros((1, 0)), np.array([[s]]))
        assert res.out_tokens[0, 0] == want
        assert res.flag_pos[0] == -1
    res = oracle.spec_verify_given_uniforms(p, q, x, np.zeros((1, 0)), np.array([[0.25 + 1e-7]]))
    assert res.out_tokens[0, 0] == 2 and res.flag_pos[0] == 0
    # a ratio test within the window of p/q is flagged at its position
    p2 = np.array([[[0.3, 0.7], [0.5, 0.5]]], dtype=np.float32)
    q2 = np.array([[[0.6, 0.4]]], dtype=np.float32)
    ratio = np.float64(np.float32(0.3)) / np.float64(np.float32(0.6))
    res = oracle.spec_verify_given_uniforms(p2, q2, np.array([[0]]), np.array([[ratio - 5e-7]]),
                                            np.array([[0.3, 0.3]]))
    assert res.accepted_len[0] == 1 and res.flag_pos[0] == 0


def test_zero_residual_falls_back_to_target_row():
    p = np.array([[[0.25, 0.25, 0.0], [0.3, 0.3, 0.4]]], dtype=np.float32)
    q = np.array([[[0.5, 0.5, 0.0]]], dtype=np.float32)
    res = oracle.spec_verify_given_uniforms(p, q, np.array([[0]]), np.array([[0.9]]),
                                            np.array([[0.75, 0.5]]))
    assert res.accepted_len[0] == 0 and res.fallback[0] == 1
    assert res.out_tokens[0, 0] == 1           # 0.75 of the way through [0.5, 0.5, 0]


def test_bad_draft_and_empty_row_are_reported():
    p = np.full((2, 2, 3), 1 / 3, dtype=np.float32)
    q = np.full((2, 1, 3), 1 / 3, dtype=np.float32)
    res = oracle.spec_verify(p, q, np.array([[0], [3]]), seed=1)
    assert res.status == oracle.E_TOKEN
    assert res.accepted_len[1] == -1 and np.all(res.out_tokens[1] == -1)
    assert res.accepted_len[0] == 1
    pz = np.zeros((1, 1, 3), dtype=np.float32)
    res = oracle.spec_verify(pz, np.zeros((1, 0, 3), np.float32), np.zeros((1, 0), np.int32), seed=1)
    assert res.status == oracle.E_DIST and res.out_tokens[0, 0] == -1
