"""Helpers for the GPU parity tests: run the C-ABI layer, run the oracle on a
compact copy of chosen sequences, compare with the stated tolerances.

Tolerances (the layer's stated parity bar): attention output max-abs <= 1e-2
(fp16) / 2e-2 (bf16) and mean-abs <= 1e-3 against the fp64 oracle; appended
keys and rotated queries within 1 unit in the last place of the storage type;
values, slot placement and metadata bit-exact.
"""
import numpy as np
import torch

import oracle
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

MAX_ABS = {"fp16": 1e-2, "bf16": 2e-2}
MEAN_ABS = 1e-3


def ordered(bits: np.ndarray) -> np.ndarray:
    """Sign-magnitude 16-bit patterns as integers whose difference counts ulps."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_diff(a_bits, b_bits) -> np.ndarray:
    return np.abs(ordered(np.asarray(a_bits)) - ordered(np.asarray(b_bits)))


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


class LayerRun:
    """One forward pass of the layer on the GPU through the C ABI."""

    def __init__(self, wl, qkv, pool, rope_style=R.DS_ROPE_HALF, want_q=True, stream=None,
                 capacity_slack=0):
        self.wl = wl
        nb = int(wl.blocks_needed().sum()) if wl.n_seqs else 0
        self.layer = R.RaggedLayer(R.params_for(wl, rope_style), max(1, wl.n_seqs) + capacity_slack,
                                   max(1, wl.n_tokens) + capacity_slack, max(1, nb) + capacity_slack,
                                   max(1, wl.max_len()), stream=stream)
        self.descs = R.SeqDescs.of(wl)
        self.layer.build(self.descs, wl.num_blocks)
        d = wl.n_q_heads * wl.head_dim
        self.q_out = torch.empty((max(1, wl.n_tokens), d), dtype=qkv.dtype, device="cuda") if want_q else None
        self.out = torch.full((max(1, wl.n_tokens), d), float("nan"), dtype=qkv.dtype, device="cuda")
        self.layer.append(qkv, pool, self.q_out)
        self.layer.attention(qkv, pool, self.out)
        torch.cuda.synchronize()
        self.dev_err = self.layer.device_error()


def check_out(wl, got: torch.Tensor, want: np.ndarray, where=""):
    g = got.float().cpu().numpy().reshape(want.shape)
    assert np.isfinite(g).all(), "non-finite output " + where
    err = np.abs(g - want)
    assert err.max() <= MAX_ABS[wl.dtype], "%s max|err| %.4g" % (where, err.max())
    assert err.mean() <= MEAN_ABS, "%s mean|err| %.4g" % (where, err.mean())
    return err.max(), err.mean()


def full_check(wl, qkv, pool_before, run: LayerRun, pool_after, style: int = R.DS_ROPE_HALF):
    """Whole batch against the oracle (small batches); `style` is the rotary
    pairing the run used (the oracle's constants have the same values)."""
    ref = oracle.layer(wl, qkv.cpu(), pool_before.cpu(), style=style)
    meta = run.layer.read_meta()
    for key in ["cu_seqlens", "seq_seen", "seq_new", "blk_off", "block_table", "tok_seq", "tok_pos"]:
        np.testing.assert_array_equal(meta[key], ref["meta"][key], err_msg=key)
    assert run.dev_err == 0
    pa = bits(pool_after).reshape(wl.pool_shape())
    assert ulp_diff(pa, ref["pool"]).max() <= 1  # K within 1 ulp
    np.testing.assert_array_equal(pa[:, 1], ref["pool"][:, 1])  # V exact
    # untouched slots bit-identical (everything except this batch's slots)
    keep = np.ones((wl.num_blocks, wl.block_size), bool)
    keep[ref["slot_block"], ref["slot_off"]] = False
    pb = bits(pool_before).reshape(wl.pool_shape())
    np.testing.assert_array_equal(pa.transpose(0, 3, 1, 2, 4)[keep], pb.transpose(0, 3, 1, 2, 4)[keep])
    if run.q_out is not None:
        assert ulp_diff(bits(run.q_out)[: wl.n_tokens], ref["q_rot"]).max() <= 1
    return check_out(wl, run.out[: wl.n_tokens], ref["out"], wl.name)


def compact(wl, seq_idx, pool_dev, qkv_dev):
    """The chosen sequences as a batch of their own over a compact pool holding
    only their blocks (copied from the device before any kernel ran).  Returns
    (sub_workload, pool_cpu, qkv_cpu, global_token_index, old_block_ids)."""
    seq_idx = list(seq_idx)
    nbs = [int(x) for x in wl.blocks_needed()[seq_idx]]
    old = np.concatenate([wl.block_ids[i][:n] for i, n in zip(seq_idx, nbs)]).astype(np.int64)
    sub = W.subset(wl, seq_idx, name=wl.name + "_sampled")
    new_ids, pos = [], 0
    for n in nbs:
        new_ids.append(np.arange(pos, pos + n, dtype=np.int32))
        pos += n
    sub.block_ids = new_ids
    sub.num_blocks = pos
    pool_c = pool_dev[torch.from_numpy(old).to(pool_dev.device)].cpu()
    cu = np.concatenate([[0], np.cumsum(wl.new)])
    gidx = np.concatenate([np.arange(cu[i], cu[i] + wl.new[i]) for i in seq_idx]).astype(np.int64)
    qkv_c = qkv_dev[torch.from_numpy(gidx).to(qkv_dev.device)].cpu()
    return sub, pool_c, qkv_c, gidx, old


def sample_rows(sub, rng, per_prefill=8):
    """Rows of a compact batch to check: every decode row; for prefill chunks
    the first, second, last and middle tokens, the tokens either side of a
    block boundary, and a few random ones."""
    rows, t0 = [], 0
    for i in range(sub.n_seqs):
        n, s = int(sub.new[i]), int(sub.seen[i])
        if n == 1:
            rows.append(t0)
        else:
            cand = {0, 1, n - 1, n // 2}
            b = (64 - s % 64) % 64  # first new token that starts a block
            for j in (b - 1, b, b + 64):
                if 0 <= j < n:
                    cand.add(j)
            cand |= set(int(x) for x in rng.integers(0, n, size=per_prefill))
            rows += [t0 + j for j in sorted(cand)]
        t0 += n
    return np.array(rows, np.int32)
