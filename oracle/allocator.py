"""Copy-on-write prefix sharing over a paged cache, written out plainly.

TEST INFRASTRUCTURE, like the rest of the oracle package.

Page this follows: "KV cache" (this.guide), section "The allocator, not the
algorithm": blocks are indirected, so two sequences with a common prefix
can point their block tables at the same physical blocks, with
copy-on-write when they diverge; each sequence wastes at most
block_size - 1 slots in its final block.

A model of the block pool, not a data structure to be fast: reference
counts are recomputed by counting every table that names a block.

Parity: pinned (tests/test_oracle_pins.py: reference counts equal a
brute-force count over the tables; a fork shares every block and copies
nothing; an append into a shared block copies it once and leaves the other
sequence's view unchanged; blocks used equal ceil(L / block_size) per
unshared sequence, so the waste bound of the page holds).
"""
import numpy as np


class CowPool:
    """num_blocks physical blocks; tables map a sequence's logical blocks to
    physical ones (-1 = none). A block's references are the table entries
    naming it; a block nobody names is free."""

    def __init__(self, num_blocks):
        self.num_blocks = int(num_blocks)
        self.tables = {}                     # sequence -> list of block ids
        self.data = {}                       # block id -> rows (any payload)

    # -- counting --------------------------------------------------------
    def refcount(self, block):
        """References on a block: the table entries naming it."""
        return sum(t.count(block) for t in self.tables.values())

    def free_blocks(self):
        """Ascending ids of the blocks no table names."""
        used = {b for t in self.tables.values() for b in t if b >= 0}
        return [b for b in range(self.num_blocks) if b not in used]

    # -- operations --------------------------------------------------------
    def new_sequence(self, name, n_blocks, payload=None):
        """A sequence owning n_blocks fresh blocks (the lowest free ids)."""
        free = self.free_blocks()
        if n_blocks > len(free):
            raise MemoryError("pool exhausted")
        blocks = free[:n_blocks]
        self.tables[name] = list(blocks)
        for i, b in enumerate(blocks):
            self.data[b] = None if payload is None else payload[i]
        return list(blocks)

    def fork(self, src, name):
        """A new sequence sharing every block of src (no copy)."""
        self.tables[name] = list(self.tables[src])

    def drop(self, name):
        """The sequence ends: its references go."""
        del self.tables[name]

    def prepare_append(self, name, pos, block_size):
        """Make the block that slot pos of the sequence lives in private:
        none yet -> a fresh block; shared -> a fresh block holding a copy of
        the shared one. Returns (src, dst) of the copy, or None."""
        table = self.tables[name]
        lb = pos // block_size
        while len(table) <= lb:
            table.append(-1)
        old = table[lb]
        if old >= 0 and self.refcount(old) == 1:
            return None
        free = self.free_blocks()
        if not free:
            raise MemoryError("pool exhausted")
        fresh = free[0]
        table[lb] = fresh
        if old < 0:
            self.data[fresh] = None
            return None
        self.data[fresh] = self.data.get(old)
        return (old, fresh)

    def blocks_used(self):
        """Blocks some table names."""
        return self.num_blocks - len(self.free_blocks())


def blocks_for_lengths(lengths, block_size):
    """Blocks held by unshared sequences of the given lengths: ceil(L / bs)
    each (so the unused slots are paged_waste_slots)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    return int(((lengths + block_size - 1) // block_size).sum())
