"""Seeded synthetic ragged batches: the inputs of one attention layer's forward.

This module only draws inputs.  It holds none of the layer's arithmetic (no
metadata packing, no rotary embedding, no attention): the CUDA path and the
CPU oracle each derive everything else from what is drawn here.

A batch is a list of sequences, each with ``seen`` tokens already in the KV
cache, ``new`` tokens in this forward pass, and the integer block ids it owns in
a block-indexed KV pool (DeepSpeed-FastGen / Inference-v2 as described on
"DeepSpeed Inference v2" (pyshine.com/deepspeed-2), sections "The front desk"
and "Ragged batches": descriptors keep integer block ids, pools are flat
block-indexed tensors, tokens of all sequences are packed edge to edge).

Draw order (fixed, documented):
  1. sequence lengths (numpy ``Generator(PCG64(seed))``),
  2. the block-id permutation (same numpy generator),
  3. the packed qkv rows (``torch.Generator`` on the target device),
  4. the KV-pool history (same torch generator).
Values are drawn in fp32 from N(0, std) and rounded to the storage dtype with
round-to-nearest-even (torch's ``.to(dtype)``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

BLOCK_SIZE = 64


@dataclasses.dataclass
class RaggedWorkload:
    """Structure of one ragged batch (no tensor values)."""

    name: str
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str  # "fp16" or "bf16"
    rope_theta: float
    value_std: float
    seen: np.ndarray  # int32 [S]
    new: np.ndarray  # int32 [S]
    block_ids: List[np.ndarray]  # per sequence: int32 ids it owns (>= ceil(L/bs))
    num_blocks: int  # pool size in blocks
    seed: int = 0

    @property
    def n_seqs(self) -> int:
        return int(len(self.seen))

    @property
    def n_tokens(self) -> int:
        return int(self.new.sum()) if len(self.new) else 0

    @property
    def qkv_width(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def blocks_needed(self) -> np.ndarray:
        total = self.seen.astype(np.int64) + self.new.astype(np.int64)
        return ((total + self.block_size - 1) // self.block_size).astype(np.int64)

    def max_len(self) -> int:
        if self.n_seqs == 0:
            return 0
        return int((self.seen.astype(np.int64) + self.new.astype(np.int64)).max())

    def pool_shape(self) -> Tuple[int, int, int, int, int]:
        return (self.num_blocks, 2, self.n_kv_heads, self.block_size, self.head_dim)


# Named workloads.  Each entry is the description of one synthetic ragged
# batch; the draws happen in ``make_workload``.
WORKLOADS = {
    # 3 sequences: a 37-token prefill chunk at 0 seen, a decode at 90 seen and
    # a 64-token chunk at 130 seen; 4 query / 2 KV heads, d=64, fp16.
    "tiny_gqa_d64": dict(n_q_heads=4, n_kv_heads=2, head_dim=64, dtype="fp16",
                         rope_theta=1.0e4, value_std=1.0),
    # 256 decodes, seen ~ U{128..4096}; Llama-2-7B attention shape.
    "decode256_mha_d128": dict(n_q_heads=32, n_kv_heads=32, head_dim=128, dtype="bf16",
                               rope_theta=1.0e4, value_std=1.0),
    # Dynamic SplitFuse mix at a 2048-token budget; Llama-3-8B GQA shape.
    "splitfuse2048_gqa_d128": dict(n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
                                   rope_theta=5.0e5, value_std=1.0),
    # Long-context chunked prefill: 2 x 8192 new tokens at seen 0 and 8192.
    "chunked_prefill_2x8192": dict(n_q_heads=64, n_kv_heads=8, head_dim=128, dtype="bf16",
                                   rope_theta=5.0e5, value_std=0.5),
    # Max ragged batch: 8192 tokens over 256 sequences (16 Zipf chunks + 240
    # decodes), seen log-uniform up to 32768, pool 1.25x the blocks needed.
    "max_ragged_8192": dict(n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="fp16",
                            rope_theta=1.0e6, value_std=1.0),
}


def _zipf_chunks(rng: np.random.Generator, n_chunks: int, total: int,
                 lo: int, hi: int, a: float) -> np.ndarray:
    """Chunk sizes: Zipf(a) draws, scaled by a bisected factor c so that
    sum(clip(rint(c*z), lo, hi)) lands on ``total``; the residual is spread
    +1 round-robin in index order over chunks still below ``hi``."""
    z = rng.zipf(a, size=n_chunks).astype(np.float64)
    if not (n_chunks * lo <= total <= n_chunks * hi):
        raise ValueError("total outside the clip bounds")

    def f(c: float) -> np.ndarray:
        return np.clip(np.rint(c * z), lo, hi).astype(np.int64)

    c_lo, c_hi = 0.0, float(hi) / float(z.min()) + 1.0
    for _ in range(200):
        mid = 0.5 * (c_lo + c_hi)
        if f(mid).sum() <= total:
            c_lo = mid
        else:
            c_hi = mid
    sizes = f(c_lo)
    resid = int(total - sizes.sum())
    k = 0
    while resid > 0:
        if sizes[k % n_chunks] < hi:
            sizes[k % n_chunks] += 1
            resid -= 1
        k += 1
    return sizes.astype(np.int32)


def _assign_blocks(seen: np.ndarray, new: np.ndarray, bs: int,
                   ids: np.ndarray) -> List[np.ndarray]:
    """Give each sequence, in batch order, the next ceil(L/bs) ids of ``ids``."""
    need = (seen.astype(np.int64) + new + bs - 1) // bs
    out, pos = [], 0
    for n in need:
        out.append(np.ascontiguousarray(ids[pos:pos + int(n)], dtype=np.int32))
        pos += int(n)
    return out


def make_workload(name: str, seed: int = 0) -> RaggedWorkload:
    """Draw the structure (lengths, block ids) of a named workload."""
    spec = WORKLOADS[name]
    rng = np.random.Generator(np.random.PCG64(seed))
    bs = BLOCK_SIZE
    if name == "tiny_gqa_d64":
        seen = np.array([0, 90, 130], np.int32)
        new = np.array([37, 1, 64], np.int32)
        pool = 16
        ids = rng.permutation(pool).astype(np.int32)
    elif name == "decode256_mha_d128":
        seen = rng.integers(128, 4096, size=256, endpoint=True).astype(np.int32)
        new = np.ones(256, np.int32)
        pool = int(((seen.astype(np.int64) + new + bs - 1) // bs).sum())
        ids = rng.permutation(pool).astype(np.int32)
    elif name == "splitfuse2048_gqa_d128":
        dec_seen = rng.integers(64, 8192, size=512, endpoint=True).astype(np.int32)
        seen = np.concatenate([np.array([0, 1024, 3072], np.int32), dec_seen])
        new = np.concatenate([np.full(3, 512, np.int32), np.ones(512, np.int32)])
        pool = int(((seen.astype(np.int64) + new + bs - 1) // bs).sum())
        ids = rng.permutation(pool).astype(np.int32)
    elif name == "chunked_prefill_2x8192":
        seen = np.array([0, 8192], np.int32)
        new = np.array([8192, 8192], np.int32)
        pool = int(((seen.astype(np.int64) + new + bs - 1) // bs).sum())
        ids = rng.permutation(pool).astype(np.int32)
    elif name == "max_ragged_8192":
        n_pre, n_dec, budget = 16, 240, 8192
        chunks = _zipf_chunks(rng, n_pre, budget - n_dec, 32, 1024, 1.2)
        seen = np.floor(np.exp(rng.uniform(math.log(16.0), math.log(32768.0),
                                           size=n_pre + n_dec))).astype(np.int32)
        new = np.concatenate([chunks, np.ones(n_dec, np.int32)])
        needed = int(((seen.astype(np.int64) + new + bs - 1) // bs).sum())
        pool = int(math.ceil(1.25 * needed))
        ids = rng.permutation(pool)[:needed].astype(np.int32)
    else:  # pragma: no cover - guarded by the dict lookup above
        raise KeyError(name)
    return RaggedWorkload(name=name, block_size=bs, seen=seen, new=new,
                          block_ids=_assign_blocks(seen, new, bs, ids),
                          num_blocks=pool, seed=seed, **spec)


def make_custom(seqs: Sequence[Tuple[int, int]], n_q_heads: int, n_kv_heads: int,
                head_dim: int, dtype: str = "bf16", rope_theta: float = 1.0e4,
                value_std: float = 1.0, seed: int = 0, extra_blocks: int = 0,
                block_size: int = BLOCK_SIZE, name: str = "custom") -> RaggedWorkload:
    """A ragged batch from explicit (seen, new) pairs; block ids are a seeded
    permutation of a pool with ``extra_blocks`` spare blocks."""
    rng = np.random.Generator(np.random.PCG64(seed))
    seen = np.array([s for s, _ in seqs], np.int32).reshape(-1)
    new = np.array([n for _, n in seqs], np.int32).reshape(-1)
    need = int(((seen.astype(np.int64) + new + block_size - 1) // block_size).sum())
    pool = need + int(extra_blocks)
    ids = rng.permutation(pool).astype(np.int32) if pool else np.zeros(0, np.int32)
    return RaggedWorkload(name=name, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
                          head_dim=head_dim, block_size=block_size, dtype=dtype,
                          rope_theta=rope_theta, value_std=value_std, seen=seen, new=new,
                          block_ids=_assign_blocks(seen, new, block_size, ids),
                          num_blocks=pool, seed=seed)


def torch_dtype(wl: RaggedWorkload):
    import torch
    return {"fp16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]


def _randn_into(dst, gen, std: float, chunk_elems: int = 1 << 28) -> None:
    import torch
    flat = dst.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        v = torch.randn(e - s, generator=gen, device=dst.device, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        flat[s:e].copy_(v.to(dst.dtype))


def make_values(wl: RaggedWorkload, device: str = "cpu", seed: Optional[int] = None):
    """Draw the packed qkv rows [N, (Hq+2Hkv)*d] and the KV pool
    [num_blocks, 2, Hkv, bs, d] (every slot drawn; the cache's history is the
    part at positions < seen of each sequence).  Returns (qkv, pool)."""
    import torch
    seed = wl.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) + 0x5EED)
    dt = torch_dtype(wl)
    qkv = torch.empty((wl.n_tokens, wl.qkv_width), dtype=dt, device=device)
    pool = torch.empty(wl.pool_shape(), dtype=dt, device=device)
    if qkv.numel():
        _randn_into(qkv, gen, wl.value_std)
    if pool.numel():
        _randn_into(pool, gen, wl.value_std)
    return qkv, pool


def subset(wl: RaggedWorkload, seq_idx: Sequence[int], name: Optional[str] = None) -> RaggedWorkload:
    """The same workload restricted to some sequences (block ids unchanged)."""
    idx = np.asarray(list(seq_idx), dtype=np.int64)
    return dataclasses.replace(wl, name=name or (wl.name + "_subset"), seen=wl.seen[idx].copy(),
                               new=wl.new[idx].copy(),
                               block_ids=[wl.block_ids[i].copy() for i in idx])


def compact_sequences(wl: RaggedWorkload, keep: Sequence[int], seed: int = 0,
                      suffix: str = "_part") -> RaggedWorkload:
    """Some sequences of a workload over a pool of exactly their blocks (a
    seeded permutation of fresh ids): a smaller case of the same shape."""
    idx = np.asarray(list(keep), dtype=np.int64)
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    seen, new = wl.seen[idx].copy(), wl.new[idx].copy()
    need = int(((seen.astype(np.int64) + new + wl.block_size - 1) // wl.block_size).sum())
    ids = rng.permutation(need).astype(np.int32)
    return dataclasses.replace(wl, name=wl.name + suffix, seen=seen, new=new,
                               block_ids=_assign_blocks(seen, new, wl.block_size, ids),
                               num_blocks=need)


def first_sequences(wl: RaggedWorkload, n: int, seed: int = 0) -> RaggedWorkload:
    """The first n sequences of a workload over a compact pool."""
    return compact_sequences(wl, range(min(n, wl.n_seqs)), seed, suffix="_first%d" % min(n, wl.n_seqs))
