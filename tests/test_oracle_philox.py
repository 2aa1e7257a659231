"""Pins for the oracle's Philox4x32-10 (Salmon et al., SC'11).

The pages only say "random()"; the counter-based generator and its keying by
(seed, sequence, position) are the method's stated design.  The oracle's own
implementation is checked here against an implementation it shares nothing with:
PyTorch's Philox engine, compiled from its public header into a tiny witness program.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def witness(tmp_path_factory):
    torch = pytest.importorskip("torch")
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    if not os.path.exists(os.path.join(inc, "ATen", "core", "PhiloxRNGEngine.h")):
        pytest.skip("PyTorch's Philox header is not installed")
    exe = str(tmp_path_factory.mktemp("philox") / "witness")
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", inc, os.path.join(HERE, "philox_witness.cpp"),
                    "-o", exe], check=True)

    def run(triples):
        text = "".join(f"{s} {b} {o}\n" for s, b, o in triples)
        res = subprocess.run([exe], input=text, capture_output=True, text=True, check=True)
        rows = [[int(w, 16) for w in line.split()] for line in res.stdout.strip().splitlines()]
        return np.asarray(rows, dtype=np.uint64).astype(np.uint32)

    return run


def test_philox_matches_library_on_random_counters(witness):
    rng = np.random.default_rng(7)
    n = 4000
    seeds = rng.integers(0, 2**64, size=n, dtype=np.uint64)
    subs = rng.integers(0, 2**64, size=n, dtype=np.uint64)
    offs = rng.integers(0, 2**64, size=n, dtype=np.uint64)
    ref = witness(list(zip(seeds.tolist(), subs.tolist(), offs.tolist())))
    ctr = np.stack([offs & 0xFFFFFFFF, offs >> 32, subs & 0xFFFFFFFF, subs >> 32], axis=1)
    for i in range(0, n, 500):
        key = np.array([seeds[i] & 0xFFFFFFFF, seeds[i] >> 32], dtype=np.uint32)
        got = oracle.philox4x32_10(ctr[i:i + 1].astype(np.uint32), key)
        np.testing.assert_array_equal(got, ref[i:i + 1])
    # all rows, each with its own key
    got = np.concatenate([
        oracle.philox4x32_10(ctr[i:i + 1].astype(np.uint32),
                             np.array([seeds[i] & 0xFFFFFFFF, seeds[i] >> 32], dtype=np.uint32))
        for i in range(n)])
    np.testing.assert_array_equal(got, ref)


def test_philox_edge_counters(witness):
    cases = [(0, 0, 0), (2**64 - 1, 2**64 - 1, 2**64 - 1), (1234, 0, 3), (99, 63, 4),
             (0, 2**32, 2**32 - 1)]
    ref = witness(cases)
    for (seed, sub, off), row in zip(cases, ref):
        ctr = np.array([[off & 0xFFFFFFFF, off >> 32, sub & 0xFFFFFFFF, sub >> 32]], dtype=np.uint32)
        key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)
        np.testing.assert_array_equal(oracle.philox4x32_10(ctr, key)[0], row)


def test_uniforms_use_position_sequence_counter(witness):
    """r[b][i] is word 0 and s[b][j] word 1 of the block at counter (position, b, 0, 0):
    in the library's terms offset = position + 2^32 * b, subsequence 0."""
    seed, B, k = 0xDEADBEEF12345678, 5, 4
    r, s = oracle.uniforms(seed, B, k)
    triples = [(seed, 0, pos + (b << 32)) for b in range(B) for pos in range(k + 1)]
    ref = witness(triples).reshape(B, k + 1, 4).astype(np.float64)
    np.testing.assert_array_equal(r, (ref[:, :k, 0] + 0.5) * 2.0**-32)
    np.testing.assert_array_equal(s, (ref[:, :, 1] + 0.5) * 2.0**-32)


def test_uniform_map_open_interval():
    # The map (w + 0.5) 2^-32 sends 0 -> 2^-33 and 2^32-1 -> 1 - 2^-33: strictly inside (0, 1).
    r, s = oracle.uniforms(1, 2000, 3)
    assert np.all(r > 0) and np.all(r < 1) and np.all(s > 0) and np.all(s < 1)
    # uniform on (0,1): mean 1/2, variance 1/12 (loose statistical sanity)
    allu = np.concatenate([r.ravel(), s.ravel()])
    assert abs(allu.mean() - 0.5) < 0.01
    assert abs(allu.var() - 1 / 12) < 0.005
