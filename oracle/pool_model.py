"""Reference model of a refcounted paged block pool (oracle; test infrastructure only).

Semantics from the pages:

* "KV Cache（键值缓存）" section 2.3: fixed-size blocks (default 16 tokens),
  a block table per sequence mapping logical to physical blocks, blocks
  allocated on demand so only the last block of a sequence can be partly
  empty; sharing between sequences (parallel sampling, beam search) by
  reference counts, with copy-on-write for a shared block that is written.
* "KV缓存原理与显存估算", closing section: a reference count says how many
  holders a block has; at zero the block can be reused; physical capacity is
  counted over the set of unique blocks.

Readings where the pages are silent:

* a new block is the lowest-numbered free block;
* sequence ids are handed out 0, 1, 2, ... and never reused;
* forking copies the parent's table and length and adds one reference to
  each of its blocks;
* appending into a partly filled block that has more than one holder needs
  copy-on-write: ``reserve`` refuses it, ``reserve_cow`` gives the writer a
  fresh block (lowest free id), drops the writer's reference to the shared
  one and reports the pair (shared block, fresh block) whose contents the
  caller copies before the new rows are written. The copy is of the whole
  block; only its first ``length % block_size`` rows are live;
* a reservation that needs more blocks than are free allocates nothing;
* unused table entries are padded with 0.
"""

from __future__ import annotations


class PoolError(Exception):
    pass


class NoBlocks(PoolError):
    pass


class Unsupported(PoolError):
    pass


class PoolModel:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks < 1 or block_size < 1:
            raise ValueError("num_blocks and block_size must be >= 1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.ref = [0] * num_blocks
        self.seqs = {}  # id -> [blocks list, length]
        self.next_id = 0

    def _take_free(self) -> int:
        for b in range(self.num_blocks):
            if self.ref[b] == 0:
                self.ref[b] = 1
                return b
        raise NoBlocks("pool exhausted")

    def free_blocks(self) -> int:
        return sum(1 for r in self.ref if r == 0)

    def add(self) -> int:
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = [[], 0]
        return sid

    def fork(self, parent: int) -> int:
        blocks, n = self.seqs[parent]
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = [list(blocks), n]
        for b in blocks:
            self.ref[b] += 1
        return sid

    def reserve(self, sid: int, n_new: int):
        blocks, n = self.seqs[sid]
        bs = self.block_size
        if n_new < 0:
            raise ValueError("n_new must be >= 0")
        if n_new == 0:
            return []
        if n % bs != 0 and self.ref[blocks[-1]] > 1:
            raise Unsupported("append into a shared partial block needs copy-on-write")
        need = -(-(n + n_new) // bs) - len(blocks)
        if need > self.free_blocks():
            raise NoBlocks("pool exhausted")
        slots = []
        for pos in range(n, n + n_new):
            if pos % bs == 0:
                blocks.append(self._take_free())
            slots.append(blocks[pos // bs] * bs + pos % bs)
        self.seqs[sid][1] = n + n_new
        return slots

    def reserve_cow(self, sid: int, n_new: int):
        """As ``reserve``, but a shared partly filled last block is first replaced
        by a private copy. Returns (slots, copy) with copy = (src, dst) or None."""
        blocks, n = self.seqs[sid]
        bs = self.block_size
        if n_new < 0:
            raise ValueError("n_new must be >= 0")
        copy = None
        if n_new > 0 and n % bs != 0 and self.ref[blocks[-1]] > 1:
            # the fresh block and the new tail blocks must all be available up front
            need = 1 + (-(-(n + n_new) // bs) - len(blocks))
            if need > self.free_blocks():
                raise NoBlocks("pool exhausted")
            old = blocks[-1]
            new = self._take_free()
            self.ref[old] -= 1
            blocks[-1] = new
            copy = (old, new)
        return self.reserve(sid, n_new), copy

    def free(self, sid: int):
        blocks, _ = self.seqs.pop(sid)
        for b in blocks:
            self.ref[b] -= 1

    def length(self, sid: int) -> int:
        return self.seqs[sid][1]

    def table(self, sid: int, max_blocks: int):
        blocks = self.seqs[sid][0]
        if len(blocks) > max_blocks:
            raise ValueError("table wider than max_blocks")
        return list(blocks) + [0] * (max_blocks - len(blocks))

    def stats(self):
        live = [s for s in self.seqs.values()]
        entries = sum(len(b) for b, _ in live)
        tokens = sum(n for _, n in live)
        used = sum(1 for r in self.ref if r > 0)
        return {
            "num_blocks": self.num_blocks,
            "free_blocks": self.num_blocks - used,
            "unique_blocks": used,
            "table_entries": entries,
            "useful_tokens": tokens,
            "live_seqs": len(live),
        }
