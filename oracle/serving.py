"""Oracle of the KV block pool and the continuous-batching decode step.

TEST INFRASTRUCTURE ONLY.  Only the tests may import this module.  It shares
no code with the CUDA library and never imports it.

What it models (page title, section):
  * forge-engine README, "What it implements": the KV cache is a paged block
    allocator with deterministic cleanup; scheduling is continuous, bounded,
    token-budgeted batching; the engine's report after its workload shows
    zero KV blocks still allocated.
  * "Make the Engine Talk", 1.2: every decode pass appends exactly one token
    to each running sequence's cache.

The pages state those properties and no algorithm, so the policy below is a
reading (the same one the library documents), written the plain way with
Python lists:

  pool   -- a stack of free block ids, 0 handed out first; a released
            sequence's blocks go back last block first; a sequence of n
            tokens owns ceil(n / block_size) blocks, listed in token order.
  step   -- (1) retire every row that has run its max_new_tokens decode
            steps; (2) while the running rows' next tokens need more new
            blocks than are free, send the most recently admitted running
            sequence back to the front of the queue with prompt = its
            length; (3) admit queue heads, first come first served, into the
            lowest free row while a row is free, the pool holds the prompt
            plus one token on top of the running rows' need, and the step's
            admitted prompt tokens stay within the budget (the first
            admission of a step is exempt from the budget), stopping at the
            first head that does not fit; (4) every running row appends one
            token at position len: a new block when len % block_size == 0,
            slot = table[len // block_size] * block_size + len % block_size.

Pins (tests/test_oracle_serving_pins.py): a trace worked out by hand
(tests/golden/serving_trace.json) and invariants checked by brute force
over seeded random request streams: every block is free or owned by exactly
one sequence, each sequence owns ceil(len / block_size) blocks, slots follow
the definition, admission is first come first served, the budget holds, and
the pool is empty once every request has finished.
"""
from __future__ import annotations


def _blocks_for(tokens: int, block_size: int) -> int:
    return -(-tokens // block_size)


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.max_blocks_per_seq = max_blocks_per_seq
        self.free = list(range(num_blocks - 1, -1, -1))   # free[-1] is handed out next
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    def add(self, seq: int, tokens: int) -> None:
        need = _blocks_for(tokens, self.block_size)
        if seq in self.tables or tokens < 0 or need > self.max_blocks_per_seq:
            raise ValueError("bad sequence")
        if need > len(self.free):
            raise MemoryError("pool full")
        self.tables[seq] = [self.free.pop() for _ in range(need)]
        self.lens[seq] = tokens

    def grow(self, seq: int):
        """Append one token; returns (slot, the block it opened or -1)."""
        pos = self.lens[seq]
        opened = -1
        if pos % self.block_size == 0:
            if len(self.tables[seq]) >= self.max_blocks_per_seq:
                raise ValueError("table row full")
            if not self.free:
                raise MemoryError("pool full")
            opened = self.free.pop()
            self.tables[seq].append(opened)
        self.lens[seq] = pos + 1
        slot = self.tables[seq][pos // self.block_size] * self.block_size + pos % self.block_size
        return slot, opened

    def release(self, seq: int) -> None:
        for b in reversed(self.tables.pop(seq)):
            self.free.append(b)
        del self.lens[seq]

    def used(self) -> int:
        return self.num_blocks - len(self.free)


class DecodeBatch:
    def __init__(self, pool: BlockPool, rows: int, token_budget: int):
        self.pool = pool
        self.rows = rows
        self.budget = token_budget
        self.seq = [-1] * rows        # sequence in each row, -1 = none
        self.left = [0] * rows        # decode steps still to run
        self.order = [0] * rows       # admission counter of the row's sequence
        self.admissions = 0
        self.queue: list[list[int]] = []   # [seq, prompt, max_new] in arrival order
        self.live: set[int] = set()

    def submit(self, seq: int, prompt: int, max_new: int) -> None:
        bs = self.pool.block_size
        if seq in self.live or prompt < 0 or max_new < 1:
            raise ValueError("bad request")
        if _blocks_for(prompt + max_new, bs) > self.pool.max_blocks_per_seq:
            raise ValueError("longer than a table row")
        if _blocks_for(prompt + max_new, bs) > self.pool.num_blocks:
            raise MemoryError("larger than the pool")
        self.queue.append([seq, prompt, max_new])
        self.live.add(seq)

    def _len(self, r: int) -> int:
        return self.pool.lens[self.seq[r]] if self.seq[r] >= 0 else 0

    def _need(self) -> int:
        return sum(1 for r in range(self.rows) if self.seq[r] >= 0 and self._len(r) % self.pool.block_size == 0)

    def _vacate(self, r: int) -> None:
        self.seq[r], self.left[r], self.order[r] = -1, 0, 0

    def step(self) -> dict:
        pool, bs = self.pool, self.pool.block_size
        admitted, retired, preempted = [], [], []

        # (1) retire
        for r in range(self.rows):
            if self.seq[r] >= 0 and self.left[r] == 0:
                retired.append((self.seq[r], r, self._len(r)))
                self.live.discard(self.seq[r])
                pool.release(self.seq[r])
                self._vacate(r)

        # (2) preempt the most recently admitted until the growth fits
        while self._need() > len(pool.free):
            running = [r for r in range(self.rows) if self.seq[r] >= 0]
            r = max(running, key=lambda i: self.order[i])
            length = self._len(r)
            preempted.append((self.seq[r], r, length))
            self.queue.insert(0, [self.seq[r], length, self.left[r]])
            pool.release(self.seq[r])
            self._vacate(r)

        # (3) admit, first come first served
        tokens_in = 0
        while self.queue:
            seq, prompt, max_new = self.queue[0]
            free_rows = [r for r in range(self.rows) if self.seq[r] < 0]
            if not free_rows:
                break
            if admitted and tokens_in + prompt > self.budget:
                break
            if _blocks_for(prompt + 1, bs) + self._need() > len(pool.free):
                break
            r = free_rows[0]
            pool.add(seq, prompt)
            self.admissions += 1
            self.seq[r], self.left[r], self.order[r] = seq, max_new, self.admissions
            tokens_in += prompt
            admitted.append((seq, r, prompt))
            self.queue.pop(0)

        # (4) one token for every running row
        slots, opened = [-1] * self.rows, [-1] * self.rows
        for r in range(self.rows):
            if self.seq[r] >= 0:
                slots[r], opened[r] = pool.grow(self.seq[r])
                self.left[r] -= 1

        lens = [self._len(r) for r in range(self.rows)]
        return {
            "seq_ids": list(self.seq), "context_lens": lens, "slots": slots, "new_blocks": opened,
            "admitted": admitted, "retired": retired, "preempted": preempted,
            "report": {"running": sum(1 for s in self.seq if s >= 0), "waiting": len(self.queue),
                       "admitted": len(admitted), "retired": len(retired), "preempted": len(preempted),
                       "free_blocks": len(pool.free), "tokens": sum(lens)},
        }

    def table(self, r: int) -> list[int]:
        """The block-table row of the sequence in row r ([] for an empty row)."""
        return list(self.pool.tables[self.seq[r]]) if self.seq[r] >= 0 else []
