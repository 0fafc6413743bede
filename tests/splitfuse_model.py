"""Plain-Python model of the Dynamic SplitFuse pass planner (test reference).

The same rules as the library's native planner (ds_splitfuse_*), written
plainly so the tests can check the native one pass for pass: one token for
every decoding sequence first, then prompt chunks in arrival order within the
token budget; a sequence whose blocks the ledger cannot supply waits
("DeepSpeed-Inference and DeepSpeed-MII", tutorial ch. 10, sections 10.3 and
10.10; "DeepSpeed Inference v2", pyshine.com/deepspeed-2, section "The front
desk").
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np

from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R


@dataclasses.dataclass
class Request:
    uid: int
    prompt: int          # prompt tokens
    decode: int          # tokens to generate after the prompt
    seen: int = 0        # tokens already in the KV cache
    generated: int = 0
    blocks: List[int] = dataclasses.field(default_factory=list)

    @property
    def prefilling(self) -> bool:
        return self.seen < self.prompt

    @property
    def done(self) -> bool:
        return not self.prefilling and self.generated >= self.decode


class SplitFusePlanner:
    def __init__(self, allocator: "R.BlockAllocator", token_budget: int, max_seqs: int,
                 block_size: int = 64):
        self.alloc = allocator
        self.budget = int(token_budget)
        self.max_seqs = int(max_seqs)
        self.bs = int(block_size)
        self.active: Dict[int, Request] = {}
        self.order: List[int] = []
        self.freed: List[int] = []

    def add(self, uid: int, prompt: int, decode: int) -> None:
        self.active[uid] = Request(uid, int(prompt), int(decode))
        self.order.append(uid)

    def _reserve(self, r: Request, n: int) -> bool:
        extra = R.ds_kv_blocks_required(r.seen, n, len(r.blocks), self.bs)
        if extra > self.alloc.n_free:
            return False
        if extra:
            r.blocks += [int(b) for b in self.alloc.allocate(extra)]
        return True

    def next_batch(self) -> List[Tuple[int, int, int, np.ndarray]]:
        """(uid, seen, new, block_ids) for the next pass: decodes first (one
        token each), then prompt chunks in arrival order; a sequence whose
        blocks cannot be reserved waits for a later pass."""
        batch, left = [], self.budget
        for uid in self.order:
            r = self.active[uid]
            if left == 0 or len(batch) == self.max_seqs:
                break
            if not r.prefilling and not r.done and self._reserve(r, 1):
                batch.append((uid, r.seen, 1))
                left -= 1
        for uid in self.order:
            r = self.active[uid]
            if left == 0 or len(batch) == self.max_seqs:
                break
            if r.prefilling:
                n = min(r.prompt - r.seen, left)
                if self._reserve(r, n):
                    batch.append((uid, r.seen, n))
                    left -= n
        return [(u, s, n, np.array(self.active[u].blocks, np.int32)) for u, s, n in batch]

    def commit(self, batch) -> List[int]:
        """Advance the sequences of a finished pass; flush the ones that are
        done (their blocks go back to the ledger).  Returns the flushed uids."""
        flushed = []
        for uid, seen, new, _ in batch:
            r = self.active[uid]
            r.seen += new
            if r.seen > r.prompt:
                r.generated += new
        for uid in list(self.order):
            r = self.active[uid]
            if r.done:
                self.alloc.free(r.blocks)
                self.freed += r.blocks
                r.blocks = []
                self.order.remove(uid)
                del self.active[uid]
                flushed.append(uid)
        return flushed

    @property
    def idle(self) -> bool:
        return not self.order
