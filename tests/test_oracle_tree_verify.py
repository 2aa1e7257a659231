"""Pins for the oracle's draft-tree verification (CPU only).

The walk is a reading ("Continuous Batching & Speculative Decoding", neuralmasteryai.com,
sections "The Modified Rejection Sampling Algorithm" and "4. Tree Attention & Medusa
Heads"): the modified rejection rule applied to a node's children one after another,
each rejection replacing the target by its normalised positive residual against the
draft distribution.  What pins it:
  - a chain is the plain rule, token for token, with the same uniforms;
  - losslessness, computed exactly: with the children drawn independently from q, the
    token emitted after a node is distributed as the target p at that node.  The
    probabilities come from the oracle as a black box: the threshold of every ratio
    test and every step of the inverse CDF are found by bisection on its uniforms;
  - the normalised residual after each rejection, restated in the pages' own form
    (max(0, p' - q) / sum max(0, p' - q)), fixes every threshold.
"""
import itertools

import numpy as np
import pytest

import oracle


def _rows(rng, V, k):
    """k probability rows that sum to exactly 1 in float32 and in double: multiples of
    2^-20 (the exactness claims hold for normalised rows)."""
    w = np.floor(rng.dirichlet(np.ones(V) * 0.7, k) * 2 ** 20)
    w[np.arange(k), w.argmax(axis=1)] += 2 ** 20 - w.sum(axis=1)
    return (w / 2 ** 20).astype(np.float32)


def test_chain_is_the_plain_rule():
    rng = np.random.default_rng(0)
    for B, n, V in [(16, 4, 32), (8, 7, 1000), (32, 1, 5)]:
        p = _rows(rng, V, B * (n + 1)).reshape(B, n + 1, V)
        q = _rows(rng, V, B * n).reshape(B, n, V)
        # drafts from q, and some forced near-certain acceptances (q = p rows)
        q[: B // 4] = p[: B // 4, :n]
        x = np.array([[rng.choice(V, p=q[b, i] / q[b, i].sum()) for i in range(n)]
                      for b in range(B)], dtype=np.int32)
        chain = np.tile(np.arange(n, dtype=np.int32), (B, 1))
        for seed in (1, 2 ** 40 + 3):
            t = oracle.spec_verify_tree(p, q, x, chain, seed)
            c = oracle.spec_verify(p, q, x, seed)
            assert t.status == 0 and c.status == 0
            np.testing.assert_array_equal(t.accepted_len, c.accepted_len)
            np.testing.assert_array_equal(t.out_tokens, c.out_tokens)
            np.testing.assert_array_equal(t.flag_pos, c.flag_pos)
            for b in range(B):
                acc = t.accepted_len[b]
                np.testing.assert_array_equal(t.path[b, :acc], np.arange(1, acc + 1))
                assert np.all(t.path[b, acc:] == -1)


def _run(p, q, x, par, r, s):
    res = oracle.spec_verify_tree_given_uniforms(p, q, x, par, r, s, flag_window=0.0)
    assert res.status == 0
    return res


def _threshold(query, lo=0.0, hi=1.0, iters=60):
    """Largest u in [lo, hi] with query(u) true, for a query true on [0, t] only."""
    if not query(lo):
        return lo
    if query(hi):
        return hi
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if query(mid):
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _draw_distribution(draw, V):
    """P(token) of an inverse-CDF draw as a function of its uniform s: the length of
    each run of s that yields the token, its ends found by bisection."""
    probs = np.zeros(V)
    s0 = 0.0
    while s0 < 1.0:
        y = draw(s0)
        end = _threshold(lambda s: draw(s) == y, s0, 1.0)
        probs[y] += end - s0
        if end >= 1.0:
            break
        s0 = end + 1e-13
    return probs


def _emitted_after(p_node, q_node, child_rows, V, node, parents, n, rows_p, rows_q):
    """Exact distribution of the token emitted after `node`, whose children are
    nodes node+1 .. node+m (leaves), drafted independently from q_node."""
    kids = [c for c in range(1, n + 1) if parents[c - 1] == node]
    dist = np.zeros(V)
    for xs in itertools.product(range(V), repeat=len(kids)):
        w = np.prod([q_node[x] for x in xs])
        if w == 0:
            continue
        x = np.zeros(n, np.int32)
        for c, xc in zip(kids, xs):
            x[c - 1] = xc
        for c in range(1, n + 1):  # drafts off this node: any fixed token
            if c not in kids:
                x[c - 1] = 0
        p = rows_p[None]
        q = rows_q[None]

        def outcome(rv, sv):
            r = np.ones((1, n))
            r[0, :] = 0.0  # everything before `node` accepted (its tests have r = 0)
            for c, val in zip(kids, rv):
                r[0, c - 1] = val
            s = np.full((1, n + 1), 0.5)
            s[0, node] = sv
            res = _run(p, q, x[None], parents[None], r, s)
            depth = int(np.sum(res.path[0] >= 0))
            return res, depth

        # walk the children: P(reach child i) * P(accept | reached)
        reach = 1.0
        prefix = []
        for i, c in enumerate(kids):
            def accepts(u, i=i):
                rv = list(prefix) + [u] + [1.0] * (len(kids) - i - 1)
                res, _ = outcome(rv, 0.5)
                return c in res.path[0]
            t = _threshold(accepts)
            dist[xs[i]] += w * reach * t
            reach *= 1.0 - t
            prefix.append(1.0)
            if reach == 0.0:
                break
        if reach > 0.0:
            def draw(sv):
                res, depth = outcome([1.0] * len(kids), sv)
                return int(res.out_tokens[0, depth])
            dist += w * reach * _draw_distribution(draw, V)
    return dist


@pytest.mark.parametrize("m", [1, 2, 3])
def test_first_token_is_distributed_as_p(m):
    """A root with m candidate children drafted independently from q0: the first token
    it emits is distributed exactly as p0, whatever q0 (the pages' exactness claim)."""
    rng = np.random.default_rng(10 + m)
    V = 5
    for _ in range(3):
        p0, q0, p1 = _rows(rng, V, 3)
        z = rng.integers(V)  # a token the draft never proposes
        q0[q0.argmax() if q0.argmax() != z else (z + 1) % V] += q0[z]
        q0[z] = 0.0
        n = m
        parents = np.zeros(n, np.int32)
        rows_p = np.stack([p0] + [p1] * n)
        rows_q = np.stack([q0] + [q0] * (n - 1)) if n > 1 else q0[None]
        dist = _emitted_after(p0, q0, None, V, 0, parents, n, rows_p, rows_q)
        np.testing.assert_allclose(dist, p0.astype(np.float64), atol=1e-9)


def test_second_level_is_distributed_as_the_child_row():
    """Depth 2: the root's one child is always accepted (q0 = p0 gives ratio 1); the
    token emitted after it, from three grandchildren drafted from q1, follows p1 (the
    rows of node 1 are used, not the root's)."""
    rng = np.random.default_rng(3)
    V = 4
    p0, p1, q1, p2 = _rows(rng, V, 4)
    n = 4
    parents = np.array([0, 1, 1, 1], np.int32)
    rows_p = np.stack([p0, p1, p2, p2, p2])
    rows_q = np.stack([p0, q1, q1, q1])
    dist = _emitted_after(p1, q1, None, V, 1, parents, n, rows_p, rows_q)
    np.testing.assert_allclose(dist, p1.astype(np.float64), atol=1e-9)


def test_thresholds_follow_the_normalised_residual():
    """Each sibling's acceptance threshold is p'(x) / q(x), with p' the target after the
    earlier siblings' rejections: p, then max(0, p' - q) / sum max(0, p' - q)."""
    rng = np.random.default_rng(5)
    V, n = 6, 3
    p0 = _rows(rng, V, 1)[0]
    q0 = _rows(rng, V, 1)[0]
    x = np.array([[1, 4, 2]], np.int32)
    parents = np.zeros((1, n), np.int32)
    p = np.stack([p0] + [p0] * n)[None]
    q = np.stack([q0] * n)[None]
    pprime = p0.astype(np.float64)
    for i in range(n):
        want = pprime[x[0, i]] / float(q0[x[0, i]])

        def accepts(u, i=i):
            r = np.ones((1, n))
            r[0, i] = u
            res = _run(p, q, x, parents, r, np.full((1, n + 1), 0.5))
            return res.path[0, 0] == i + 1
        assert abs(_threshold(accepts) - min(want, 1.0)) < 1e-12
        res = np.maximum(pprime - q0.astype(np.float64), 0.0)
        pprime = res / res.sum()


def test_bad_parents_and_tokens_are_rejected():
    p = np.full((1, 3, 4), 0.25, np.float32)
    q = np.full((1, 2, 4), 0.25, np.float32)
    r = np.zeros((1, 2))
    s = np.full((1, 3), 0.5)
    assert oracle.spec_verify_tree_given_uniforms(p, q, [[0, 0]], [[0, 2]], r, s).status == oracle.E_ARG
    assert oracle.spec_verify_tree_given_uniforms(p, q, [[0, 9]], [[0, 1]], r, s).status == oracle.E_TOKEN
