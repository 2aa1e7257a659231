"""Host page allocator invariants (include/vas.h: vas_pool_*), CPU only.

What the pages fix: pages are handed out on demand and returned on finish (syslabs.in,
"PagedAttention"; martinuke0.github.io, "PagedAttention: The Other Half of the Story"),
waste is bounded by one partially filled page per sequence (syslabs.in), admission is
gated on can_allocate and the newest sequence is preempted when the pool runs dry
(syslabs.in, "Continuous batching: scheduling per iteration"), rejected drafts are rolled
back (tempatgunting.com, "Speculative Decoding..."), shared prefix pages are reference
counted (tempatgunting.com, "Anatomy of the KV Cache")."""
import numpy as np
import pytest


def check_invariants(pool, model, P):
    """model: dict id -> length.  Every page is free or owned; waste < 1 page per sequence."""
    ids = sorted(model)
    maxp = max([(model[i] + P - 1) // P for i in ids] + [1])
    if ids:
        bt, lens = pool.block_table(ids, maxp)
        np.testing.assert_array_equal(lens, [model[i] for i in ids])
        owned = []
        for r, i in enumerate(ids):
            n = (model[i] + P - 1) // P
            assert np.all(bt[r, :n] >= 0) and np.all(bt[r, n:] == -1)
            owned += list(bt[r, :n])
            assert n * P - model[i] < P  # waste bounded by one partial page
        owned = np.array(owned)
        uniq, counts = np.unique(owned, return_counts=True)
        for pg, c in zip(uniq, counts):
            assert pool.refcount(int(pg)) == c
        used = len(uniq)
    else:
        used = 0
    assert pool.free_pages + used == pool.num_pages
    assert pool.num_seqs == len(ids)


def test_random_admit_grow_rollback_free_preempt(vas_lib):
    rng = np.random.default_rng(0)
    P, N = 16, 200
    pool = vas_lib.PagePool(N, P, seed=42)
    model, order, next_id = {}, [], 0
    for step in range(3000):
        op = rng.integers(0, 6)
        if op == 0 or not model:
            n = int(rng.integers(1, 200))
            fits = pool.can_allocate(n)
            st = pool.admit(next_id, n)
            assert (st == vas_lib.VAS_OK) == fits
            if st == vas_lib.VAS_OK:
                model[next_id] = n
                order.append(next_id)
            else:
                assert st == vas_lib.VAS_E_NOMEM
            next_id += 1
        elif op in (1, 2):
            i = int(rng.choice(list(model)))
            k = int(rng.integers(1, 9))
            need = pool.pages_needed(i, k)
            st = pool.grow(i, k)
            assert (st == vas_lib.VAS_OK) == (need <= pool.free_pages or need == 0) or st == vas_lib.VAS_OK
            if st == vas_lib.VAS_OK:
                model[i] += k
            else:
                assert st == vas_lib.VAS_E_NOMEM
        elif op == 3:
            i = int(rng.choice(list(model)))
            k = int(rng.integers(0, min(model[i], 8) + 1))
            assert pool.rollback(i, k) == vas_lib.VAS_OK
            model[i] -= k
        elif op == 4:
            i = int(rng.choice(list(model)))
            assert pool.free(i) == vas_lib.VAS_OK
            del model[i]
            order.remove(i)
        else:
            st, victim = pool.preempt_newest()
            assert st == vas_lib.VAS_OK and victim == order[-1]
            del model[victim]
            order.pop()
        if step % 50 == 0:
            check_invariants(pool, model, P)
    check_invariants(pool, model, P)


def test_speculative_reservation_and_rollback(vas_lib):
    P = 16
    pool = vas_lib.PagePool(10, P)
    assert pool.admit(7, 30) == 0            # 2 pages
    assert pool.grow(7, 5) == 0              # k=4 verify step reserves 5 slots -> 35, 3 pages
    assert pool.free_pages == 7
    assert pool.rollback(7, 3) == 0          # 1 accepted + bonus: drop 3 rejected -> 32
    assert pool.seq_len(7) == 32 and pool.free_pages == 8
    assert pool.rollback(7, 33) == vas_lib.VAS_E_INVALID_ARG
    assert pool.grow(8, 1) == vas_lib.VAS_E_NOT_FOUND


def test_exhaustion_and_errors(vas_lib):
    pool = vas_lib.PagePool(4, 16)
    assert pool.admit(1, 64) == 0
    assert not pool.can_allocate(1)
    assert pool.admit(2, 1) == vas_lib.VAS_E_NOMEM
    assert pool.admit(1, 1) == vas_lib.VAS_E_EXISTS
    assert pool.grow(1, 1) == vas_lib.VAS_E_NOMEM and pool.seq_len(1) == 64  # all-or-nothing
    assert pool.free(1) == 0 and pool.free(1) == vas_lib.VAS_E_NOT_FOUND
    assert pool.free_pages == 4
    assert pool.preempt_newest()[0] == vas_lib.VAS_E_NOT_FOUND


def test_prefix_sharing_refcounts(vas_lib):
    P = 16
    pool = vas_lib.PagePool(20, P)
    assert pool.admit(1, 70) == 0                    # 5 pages, 4 full
    assert pool.fork(1, 2, 70) == 0                  # shares 4 full pages, 1 fresh
    bt, _ = pool.block_table([1, 2], 5)
    assert list(bt[0, :4]) == list(bt[1, :4]) and bt[0, 4] != bt[1, 4]
    for pg in bt[0, :4]:
        assert pool.refcount(int(pg)) == 2
    assert pool.free(1) == 0
    for pg in bt[1, :4]:
        assert pool.refcount(int(pg)) == 1            # survives its first owner
    assert pool.free_pages == 20 - 5
    # rolling back into a shared page would let the next append overwrite a prefix
    assert pool.fork(2, 3, 64) == 0
    assert pool.rollback(3, 10) == vas_lib.VAS_E_INVALID_ARG
    check_invariants(pool, {2: 70, 3: 64}, P)


def test_seeded_free_list_permutes_pages(vas_lib):
    a = vas_lib.PagePool(64, 16, seed=5)
    b = vas_lib.PagePool(64, 16, seed=0)
    a.admit(1, 64 * 16)
    b.admit(1, 64 * 16)
    ta, _ = a.block_table([1], 64)
    tb, _ = b.block_table([1], 64)
    assert sorted(ta[0]) == list(range(64))
    assert list(tb[0]) == list(range(64))
    assert list(ta[0]) != list(range(64))


def test_block_table_capacity_check(vas_lib):
    pool = vas_lib.PagePool(8, 16)
    pool.admit(1, 40)
    with pytest.raises(vas_lib.VasError):
        pool.block_table([1], 2)
