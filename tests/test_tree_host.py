"""Host-side pieces of draft-tree attention: the seeded tree generator and the parent ->
ancestor-mask encoding the GPU tests hand to paged_attn_fwd_tree."""
import numpy as np

from verify_attention_spec_gb300 import workloads as wl

from gpu_common import ancestor_masks


def test_generated_trees_are_valid_and_seeded():
    qlens = [1, 2, 9, 64, 17]
    par = wl.draft_tree_parents(qlens, seed=5, extra_roots=0.2)
    assert par.dtype == np.int32 and len(par) == sum(qlens)
    assert np.array_equal(par, wl.draft_tree_parents(qlens, seed=5, extra_roots=0.2))
    row0 = 0
    for ql in qlens:
        p = par[row0:row0 + ql]
        assert p[0] == -1
        assert all(-1 <= p[j] < j for j in range(ql))
        row0 += ql


def test_masks_of_a_chain_and_a_star():
    chain = np.arange(5, dtype=np.int32) - 1
    m = ancestor_masks(chain, [5])
    assert [int(x) for x in m] == [0, 1, 3, 7, 15]
    star = np.array([-1, 0, 0, 0], dtype=np.int32)
    assert [int(x) for x in ancestor_masks(star, [4])] == [0, 1, 1, 1]


def test_mask_bits_are_the_path_to_the_root():
    qlens = [64, 30]
    par = wl.draft_tree_parents(qlens, seed=2, extra_roots=0.05)
    masks = ancestor_masks(par, qlens)
    row0 = 0
    for ql in qlens:
        for j in range(ql):
            bits = [a for a in range(64) if (int(masks[row0 + j]) >> a) & 1]
            path, a = [], int(par[row0 + j])
            while a >= 0:
                path.append(a)
                a = int(par[row0 + a])
            assert sorted(path) == bits
            assert all(b < j for b in bits)
        row0 += ql


def test_bf16_half_spacing():
    from gpu_common import bf16_half_spacing
    x = np.array([1.0, 1.5, 3.99, 4.0, 7.9, -5.0, 0.25])
    np.testing.assert_array_equal(bf16_half_spacing(x),
                                  [2**-8, 2**-8, 2**-7, 2**-6, 2**-6, 2**-6, 2**-10])
