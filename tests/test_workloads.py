"""The seeded workload generators produce the shapes and structure stated for each
workload (CPU only; the large pools are not materialised)."""
import numpy as np

from verify_attention_spec_gb300 import workloads as wl


def test_lengths_and_query_lengths():
    for name in wl.ORDER:
        w = wl.WORKLOADS[name]
        L, ql = wl.sample_lengths(w), wl.query_lengths(w)
        assert len(L) == len(ql) == w.num_seqs
        assert np.all(L >= ql) and np.all(ql >= 1)
        assert (ql > 1).sum() == w.num_verify
        if w.num_verify:
            assert np.all(ql[ql > 1] == w.k + 1)
        if w.length_law == "lognormal":
            assert L.min() >= w.length_args[2] and L.max() <= w.length_args[3]
        if w.length_law == "uniform":
            assert L.min() >= w.length_args[0] and L.max() <= w.length_args[1]
        if w.length_law == "pareto":
            assert L.min() >= w.length_args[1] and L.max() <= w.length_args[2]
    np.testing.assert_array_equal(wl.sample_lengths(wl.WORKLOADS["tiny"]), [17, 40, 63, 100])


def test_lognormal_median_and_pareto_tail():
    L = wl.sample_lengths(wl.WORKLOADS["stress70b"])
    assert 1500 < np.median(L) < 2800
    P = wl.sample_lengths(wl.WORKLOADS["mixed272"])
    assert np.median(P) < 200 and P.max() > 1000


def test_pool_is_a_permutation_sized_for_the_total():
    lens = np.array([17, 40, 63, 100])
    bt, n = wl.build_pool(lens, 16, seed=0, pool_pages=64)
    used = bt[bt >= 0]
    assert n == 64 and len(used) == 2 + 3 + 4 + 7 and len(np.unique(used)) == len(used)
    bt2, n2 = wl.build_pool(lens, 16, seed=0)
    assert n2 == 16 and sorted(bt2[bt2 >= 0]) == list(range(16))


def test_tiny_attention_inputs():
    a = wl.workload_attention("tiny")
    assert tuple(a.q.shape) == (10, 4, 64) and tuple(a.k_pages.shape) == (64, 16, 2, 64)
    assert a.q.dtype.is_floating_point and a.kv_dtype == wl.F32


def test_verify_inputs_shapes_and_drafts():
    v = wl.verify_inputs(3, 4, 50, seed=1)
    assert v.p.shape == (3, 5, 50) and v.q.shape == (3, 4, 50) and v.draft.shape == (3, 4)
    np.testing.assert_allclose(v.p.sum(-1), 1, atol=1e-5)
    assert np.all((v.draft >= 0) & (v.draft < 50))
    # drafts come from q: a draft never lands where q is essentially zero
    assert np.all(np.take_along_axis(v.q, v.draft[..., None], -1) > 0)
    again = wl.verify_inputs(3, 4, 50, seed=1)
    np.testing.assert_array_equal(v.p, again.p)
