"""Plain-Python model of the block pool, block tables and refcounted copy-on-write.

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the test suite and the benchmark's
CPU-baseline leg may import this module.

Follows spindle, section "Paging":
  * a pool of fixed-size blocks (block size 16) and a per-sequence block table,
    so a sequence wastes at most the unused tail of its final block;
  * reference counts give copy-on-write forking: a fork shares every block of
    its parent; four forks of a 16-token parent hold 64 logical tokens in 16
    physical slots.
and spindle, section "Two bugs worth recording": appends name an explicit
start position; nothing is inferred.

Readings where the page is silent (each listed with the design notes):
  * writing into a block whose refcount is above one first copies it into a
    freshly allocated block (a (src, dst) copy pair), drops one reference to
    the old block and points the writer's table at the copy; a block held
    once is written in place;
  * reference counts count live sequences only, so freeing a parent after
    forking leaves its blocks held by the children alone;
  * blocks are handed out lowest free id first.
"""
from __future__ import annotations

BLOCK = 16


class OutOfBlocks(Exception):
    pass


class OracleBlockManager:
    def __init__(self, num_blocks: int, block_size: int = BLOCK):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.refcount = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lengths: dict[int, int] = {}
        self._next_seq = 0

    # -- bookkeeping -------------------------------------------------------
    def free_blocks(self) -> list[int]:
        return [b for b in range(self.num_blocks) if self.refcount[b] == 0]

    def _take_free(self) -> int:
        for b in range(self.num_blocks):
            if self.refcount[b] == 0:
                self.refcount[b] = 1
                return b
        raise OutOfBlocks()

    # -- operations --------------------------------------------------------
    def add_sequence(self) -> int:
        sid = self._next_seq
        self._next_seq += 1
        self.tables[sid] = []
        self.lengths[sid] = 0
        return sid

    def fork(self, parent: int) -> int:
        """A child that shares every block of ``parent`` (each refcount + 1)."""
        child = self.add_sequence()
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1
        return child

    def free(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self.refcount[b] -= 1
        del self.lengths[seq]

    def blocks_needed(self, seq: int, start: int, n: int) -> int:
        """Blocks an append of n tokens at ``start`` would take from the pool."""
        table = self.tables[seq]
        need = 0
        if n <= 0:
            return 0
        for lb in range(start // self.block_size, (start + n - 1) // self.block_size + 1):
            if lb >= len(table) or self.refcount[table[lb]] > 1:
                need += 1
        return need

    def prepare_append(self, seq: int, start: int, n: int) -> list[tuple[int, int]]:
        """Make positions start .. start+n-1 of ``seq`` writable; return CoW copy pairs."""
        table = self.tables[seq]
        if n < 0 or start < 0:
            raise ValueError("negative position or count")
        if n == 0:
            return []
        if start > len(table) * self.block_size:
            raise ValueError("append would leave a hole in the block table")
        if self.blocks_needed(seq, start, n) > len(self.free_blocks()):
            raise OutOfBlocks()
        pairs = []
        for lb in range(start // self.block_size, (start + n - 1) // self.block_size + 1):
            if lb >= len(table):
                table.append(self._take_free())
            elif self.refcount[table[lb]] > 1:
                old = table[lb]
                new = self._take_free()
                self.refcount[old] -= 1
                table[lb] = new
                pairs.append((old, new))
        self.lengths[seq] = max(self.lengths[seq], start + n)
        return pairs

    # -- accounting --------------------------------------------------------
    def physical_blocks(self) -> int:
        return sum(1 for r in self.refcount if r > 0)

    def logical_tokens(self) -> int:
        return sum(self.lengths.values())

    def stats(self) -> dict:
        return {
            "physical_blocks": self.physical_blocks(),
            "physical_slots": self.physical_blocks() * self.block_size,
            "logical_tokens": self.logical_tokens(),
            "free_blocks": self.num_blocks - self.physical_blocks(),
        }
