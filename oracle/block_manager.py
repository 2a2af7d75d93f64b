"""Ref-counted paged-KV block manager with copy-on-write fork (oracle).

Test infrastructure (see ``oracle/__init__``).  Restates, in my own code, the
rules of the tutorial page "LLM 推理服务引擎深度拆解", section 2.3 "手写一个
Block Manager":

- the pool starts with every block id free, listed in increasing order;
  ``allocate`` takes the id at the END of the free list and gives it ref
  count 1; ``free`` decrements and, at zero, appends the id to the END;
- ``cow`` on a block with ref count 1 returns the same block (write in
  place); otherwise it allocates a fresh block, copies the contents and drops
  one reference from the shared block;
- a sequence appending a token at a block boundary (length % S == 0)
  allocates a new block; otherwise it applies ``cow`` to its last block
  before writing;
- ``fork`` shares every block of the parent (ref count + 1 each), copying
  nothing; ``release`` drops one reference from each block of the table;
- ``usage`` = blocks not on the free list / pool size.

The page's manager stores token ids; this one records, per append, the
physical slot written (block * S + offset) and the copy (src, dst) that a
copy-on-write implies for the device cache, which is what the device side
needs.  Running out of blocks raises ``MemoryError`` as on the page.
"""
from __future__ import annotations


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.ref_count = [0] * num_blocks
        self.free_ids = list(range(num_blocks))

    def allocate(self) -> int | None:
        if not self.free_ids:
            return None
        bid = self.free_ids.pop()
        self.ref_count[bid] = 1
        return bid

    def incref(self, bid: int) -> None:
        self.ref_count[bid] += 1

    def free(self, bid: int) -> None:
        self.ref_count[bid] -= 1
        if self.ref_count[bid] == 0:
            self.free_ids.append(bid)

    def cow(self, bid: int) -> tuple[int, tuple[int, int] | None]:
        """Returns (block to write, (src, dst) copy or None)."""
        if self.ref_count[bid] == 1:
            return bid, None
        new = self.allocate()
        if new is None:
            raise MemoryError("no free block for copy-on-write")
        self.free(bid)
        return new, (bid, new)

    @property
    def usage(self) -> float:
        return (self.num_blocks - len(self.free_ids)) / self.num_blocks


class Sequence:
    def __init__(self, mgr: BlockManager, seq_id: int):
        self.mgr = mgr
        self.seq_id = seq_id
        self.block_table: list[int] = []
        self.length = 0

    def append_slot(self) -> tuple[int, tuple[int, int] | None]:
        """Reserve the slot of the next token.  Returns (slot, copy or None)."""
        S = self.mgr.block_size
        copy = None
        if self.length % S == 0:
            bid = self.mgr.allocate()
            if bid is None:
                raise MemoryError(f"sequence {self.seq_id}: no free block")
            self.block_table.append(bid)
        else:
            bid, copy = self.mgr.cow(self.block_table[-1])
            self.block_table[-1] = bid
        slot = self.block_table[-1] * S + self.length % S
        self.length += 1
        return slot, copy

    def fork(self, new_id: int) -> "Sequence":
        child = Sequence(self.mgr, new_id)
        child.block_table = list(self.block_table)
        child.length = self.length
        for bid in child.block_table:
            self.mgr.incref(bid)
        return child

    def release(self) -> None:
        for bid in self.block_table:
            self.mgr.free(bid)
        self.block_table = []

    @classmethod
    def shared(cls, mgr: BlockManager, seq_id: int, blocks, length: int) -> "Sequence":
        """A sequence whose first blocks are existing ones (a cached prefix):
        each gets one more reference, nothing is copied."""
        S = mgr.block_size
        if blocks and not (len(blocks) - 1) * S < length <= len(blocks) * S:
            raise ValueError("length must end inside the last shared block")
        if not blocks and length != 0:
            raise ValueError("no blocks, no tokens")
        for bid in blocks:
            if mgr.ref_count[bid] < 1:
                raise ValueError(f"block {bid} is not in use")
        seq = cls(mgr, seq_id)
        seq.block_table = list(blocks)
        seq.length = length
        for bid in blocks:
            mgr.incref(bid)
        return seq
