"""The synthetic workloads' paging: each sequence owns ceil((L + 1) / block)
physical blocks (room for the step's append), the owned blocks of all
sequences and the spares are a permutation of the pool, and only the tiny
workload is laid out contiguously, so every other parity case goes through
a genuinely scattered block table."""
import numpy as np
import pytest

from kv_cache_decode_gqa_gb300 import workloads as W

NAMES = [n for n in W.CONFIGS]


@pytest.mark.parametrize("name", NAMES)
def test_blocks_are_a_partition_of_the_pool(name):
    s = W.config(name)
    pg = W.Paging(s)
    bs = s.block_size
    owned = []
    for b, L in enumerate(s.lengths):
        n = -(-(L + 1) // bs)
        assert pg.counts[b] == n
        row = pg.table[b, :n]
        assert len(set(row.tolist())) == n               # distinct blocks
        owned += row.tolist()
        # entries past the owned ones repeat the last block (valid ids)
        assert np.all(pg.table[b, n:] == row[-1])
    everything = owned + pg.spare.tolist()
    assert sorted(everything) == list(range(pg.num_blocks))
    assert pg.num_blocks == sum(pg.counts) + 2


@pytest.mark.parametrize("name", NAMES)
def test_only_the_tiny_workload_is_contiguous(name):
    s = W.config(name)
    pg = W.Paging(s)
    rows = [pg.table[b, :n] for b, n in enumerate(pg.counts) if n >= 2]
    consecutive = [bool(np.all(np.diff(r) == 1)) for r in rows]
    if name == "tiny_gqa":
        assert all(consecutive)
    else:
        assert not any(consecutive)


def test_paging_is_seeded():
    a = W.Paging(W.config("llama31_70b_gqa")).table
    b = W.Paging(W.config("llama31_70b_gqa")).table
    assert np.array_equal(a, b)
