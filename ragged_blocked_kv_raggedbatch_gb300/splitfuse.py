"""Dynamic SplitFuse step planner over the C-ABI block ledger (host logic).

Each forward pass packs, within a token budget, one token for every sequence
that is decoding and then prompt chunks of the sequences still prefilling
("DeepSpeed-Inference and DeepSpeed-MII", tutorial ch. 10, sections 10.3 and
10.10: prefill and decode requests merged into one batch; "DeepSpeed Inference
v2", pyshine.com/deepspeed-2, section "The front desk": blocks are handed out
by the allocator before each pass -- get_kv_requirements / allocate_blocks --
and returned when a sequence is flushed).  This is the minimum driver a
multi-step run needs; it is not a serving scheduler.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import numpy as np

from . import ds_ragged as R


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


class NativeSplitFusePlanner:
    """The same planner in the library (ds_splitfuse_*): state in a host array
    owned here, descriptors written straight into a ds_seq_desc[] that
    ds_ragged_meta_build takes as is."""

    def __init__(self, allocator: "R.BlockAllocator", token_budget: int, max_seqs: int,
                 max_requests: int, max_blocks_per_request: int, block_size: int = 64):
        import ctypes
        lib = R.load()
        self.alloc = allocator
        nbytes = ctypes.c_size_t(0)
        R._check(lib.ds_splitfuse_mem_size(max_requests, max_blocks_per_request, R._ref(nbytes)),
                 "ds_splitfuse_mem_size")
        self.mem = np.zeros((nbytes.value + 7) // 8, np.uint64)
        self.p = R.ds_splitfuse()
        R._check(lib.ds_splitfuse_init(R._ref(self.p), self.mem.ctypes.data, self.mem.nbytes, max_requests,
                                       max_blocks_per_request, token_budget, max_seqs, block_size),
                 "ds_splitfuse_init")
        self.arr = (R.ds_seq_desc * max_seqs)()
        self.uids = np.zeros(max_seqs, np.int32)
        self.flushed = np.zeros(max_requests, np.int32)
        self.n = 0

    def add(self, uid: int, prompt: int, decode: int) -> None:
        R._check(R.load().ds_splitfuse_add(R._ref(self.p), int(uid), int(prompt), int(decode)), "ds_splitfuse_add")

    def plan(self) -> int:
        """Plan the next pass into self.arr[:n] / self.uids[:n]; returns n.
        self (arr, n) is then a descriptor set for ds_ragged_meta_build."""
        import ctypes
        n = ctypes.c_int32(0)
        R._check(R.load().ds_splitfuse_next(R._ref(self.p), R._ref(self.alloc.a), R._ref(self.arr),
                                            self.uids.ctypes.data, R._ref(n)), "ds_splitfuse_next")
        self.n = n.value
        return self.n

    def next_batch(self) -> List[Tuple[int, int, int, np.ndarray]]:
        """The planned pass in SplitFusePlanner.next_batch's form (copies)."""
        n = self.plan()
        out = []
        for i in range(n):
            d = self.arr[i]
            ids = np.ctypeslib.as_array(d.block_ids, shape=(d.n_blocks,)).copy() if d.n_blocks else \
                np.zeros(0, np.int32)
            out.append((int(self.uids[i]), int(d.seen_tokens), int(d.new_tokens), ids))
        return out

    def commit(self, batch=None) -> List[int]:
        import ctypes
        nf = ctypes.c_int32(0)
        R._check(R.load().ds_splitfuse_commit(R._ref(self.p), R._ref(self.alloc.a), self.flushed.ctypes.data,
                                              R._ref(nf)), "ds_splitfuse_commit")
        return [int(u) for u in self.flushed[: nf.value]]

    @property
    def idle(self) -> bool:
        return self.p.n_active == 0
