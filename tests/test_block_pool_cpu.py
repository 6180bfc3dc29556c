"""The library's copy-on-write block pool (host C++, no GPU needed) against
the oracle's model (oracle.CowPool): the same operations give the same
tables, reference counts, free lists and copies; failing calls change
nothing; appends meet the page's waste bound ("KV cache", "The allocator,
not the algorithm")."""
import json
import os

import numpy as np
import pytest

import oracle as O
from kv_cache_decode_gqa_gb300 import _native as N


@pytest.fixture(scope="module")
def K():
    if not os.path.exists(N.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    import kv_cache_decode_gqa_gb300 as K
    return K


def _check_same(pool, model, tables, nb):
    for b in range(nb):
        assert pool.refcount(b) == model.refcount(b), b
    assert pool.free_count() == len(model.free_blocks())
    for name, t in tables.items():
        mt = model.tables[name]
        assert list(t[:len(mt)]) == mt, name
        assert np.all(t[len(mt):] == -1), name


def test_pool_matches_the_model(K):
    rng = np.random.default_rng(100)
    nb, M, bs = 48, 8, 4
    pool, model = K.BlockPool(nb), O.CowPool(nb)
    tables = {}                                  # name -> host table [M]
    for step in range(400):
        op = int(rng.integers(4))
        names = list(tables)
        if op == 0 or not names:
            n = int(rng.integers(1, 4))
            name = f"s{step}"
            if n > pool.free_count():
                with pytest.raises(K.KvdError):
                    pool.alloc(n)
                continue
            t = np.full(M, -1, dtype=np.int32)
            t[:n] = pool.alloc(n)
            tables[name] = t
            model.new_sequence(name, n)
        elif op == 1:
            src = names[int(rng.integers(len(names)))]
            name = f"f{step}"
            pool.share(tables[src][tables[src] >= 0])
            tables[name] = tables[src].copy()
            model.fork(src, name)
        elif op == 2:
            name = names[int(rng.integers(len(names)))]
            p = int(rng.integers(0, M * bs))
            t = tables[name][None, :].copy()
            try:
                src, dst = pool.prepare_append(t, [p], bs)
            except K.KvdError as e:
                assert e.status == 4                 # pool exhausted
                assert np.array_equal(t[0], tables[name])  # unchanged
                continue
            tables[name] = t[0]
            cp = model.prepare_append(name, p, bs)
            assert (list(zip(src, dst)) == [cp]) if cp else len(src) == 0
        else:
            name = names[int(rng.integers(len(names)))]
            pool.release(tables[name][tables[name] >= 0])
            del tables[name]
            model.drop(name)
        _check_same(pool, model, tables, nb)


def test_batched_append_into_one_shared_block(K):
    pool = K.BlockPool(8)
    t = np.full((3, 2), -1, dtype=np.int32)
    t[0, 0] = pool.alloc(1)[0]
    pool.share([t[0, 0]] * 2)
    t[1, 0] = t[2, 0] = t[0, 0]                  # three tables, one block
    src, dst = pool.prepare_append(t, [1, 2, 3], 4)
    # the first two copy, the last keeps the original alone
    assert list(src) == [0, 0] and list(dst) == [1, 2]
    assert list(t[:, 0]) == [1, 2, 0]
    assert [pool.refcount(b) for b in range(3)] == [1, 1, 1]


def test_failing_calls_change_nothing(K):
    pool = K.BlockPool(4)
    a = pool.alloc(2)
    with pytest.raises(K.KvdError):
        pool.release(np.concatenate([a, a]))      # more releases than holds
    assert [pool.refcount(b) for b in a] == [1, 1] and pool.free_count() == 2
    with pytest.raises(K.KvdError):
        pool.alloc(3)                             # exhausted
    assert pool.free_count() == 2
    with pytest.raises(K.KvdError):
        pool.share([3])                           # not held
    assert pool.refcount(3) == 0
    t = np.array([[a[0], a[1]]], dtype=np.int32)
    with pytest.raises(K.KvdError):
        pool.prepare_append(t, [9], 4)            # outside the table
    pool.release(a)
    assert pool.free_count() == 4


def test_appends_meet_the_waste_bound(K, golden_dir):
    with open(os.path.join(golden_dir, "page_figures.json")) as f:
        g = json.load(f)["paged_waste"]
    bs, Lbar = g["block_size"], g["mean_len"]
    rng = np.random.default_rng(101)
    lens = rng.integers(1, 2 * Lbar, 32)
    M = int(lens.max()) // bs + 1
    pool = K.BlockPool(int(lens.sum()) // bs + 64)
    t = np.full((len(lens), M), -1, dtype=np.int32)
    for p in range(int(lens.max())):             # one token per step
        live = np.nonzero(lens > p)[0]
        sub = np.ascontiguousarray(t[live])
        src, _ = pool.prepare_append(sub, np.full(len(live), p), bs)
        assert len(src) == 0                      # nothing is shared
        t[live] = sub
    used = int(lens.sum()) // bs + 64 - pool.free_count()
    assert used == O.blocks_for_lengths(lens, bs)
    waste = used * bs - int(lens.sum())
    assert waste <= len(lens) * (bs - 1)
    assert waste == int(O.paged_waste_slots(lens, bs).sum())
