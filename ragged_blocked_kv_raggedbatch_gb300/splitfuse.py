"""Dynamic SplitFuse pass planner over the C-ABI block ledger: binding of the
library's native planner (ds_splitfuse_*, host logic).

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

from typing import List, Tuple

import numpy as np

from . import ds_ragged as R


class NativeSplitFusePlanner:
    """The library's planner (ds_splitfuse_*): state in a host array owned
    here, descriptors written straight into a ds_seq_desc[] that
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
        """The planned pass as (uid, seen, new, block_ids) tuples (copies)."""
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
