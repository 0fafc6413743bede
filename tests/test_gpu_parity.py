"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small batches are compared in full; the full-size workloads are compared on
sampled sequences (the oracle re-runs them as a batch of their own over a
compact copy of their blocks, taken before any kernel ran) plus properties
checked on every row (finite, values bit-exactly placed in their slots).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import LayerRun, bits, check_out, compact, full_check, sample_rows, ulp_diff
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run_full(wl, rope_style=R.DS_ROPE_HALF, poison_unused=False):
    qkv, pool = W.make_values(wl, "cuda")
    if poison_unused:
        # every slot that is not history gets a NaN pattern: a kernel that reads
        # past a sequence's length (or an unused block) shows it in its output
        keep = torch.zeros((wl.num_blocks, wl.block_size), dtype=torch.bool)
        for i in range(wl.n_seqs):
            for u in range(int(wl.seen[i])):
                keep[int(wl.block_ids[i][u // 64]), u % 64] = True
        mask = keep.cuda()[:, None, None, :, None].expand(wl.pool_shape())
        pool.view(torch.int16).masked_fill_(~mask, -1)  # 0xFFFF: NaN in fp16 and bf16
    pool_before = pool.clone()
    run = LayerRun(wl, qkv, pool, rope_style=rope_style)
    if rope_style == R.DS_ROPE_HALF:
        return full_check(wl, qkv, pool_before, run, pool)
    # interleaved pairing: compare with the oracle's interleaved mode
    ref = oracle.layer(wl, qkv.cpu(), pool_before.cpu(), style=oracle.ROPE_INTERLEAVED)
    assert ulp_diff(bits(pool).reshape(wl.pool_shape()), ref["pool"]).max() <= 1
    assert ulp_diff(bits(run.q_out)[: wl.n_tokens], ref["q_rot"]).max() <= 1
    return check_out(wl, run.out[: wl.n_tokens], ref["out"], "interleaved")


def test_tiny_workload_full():
    _run_full(W.make_workload("tiny_gqa_d64", 0))


EDGE = [
    # (name, seqs, Hq, Hkv, d, dtype)
    ("first_token", [(0, 1)], 4, 2, 64, "fp16"),
    ("block_edges_decode", [(63, 1), (64, 1), (127, 1), (128, 1), (0, 1), (1000, 1)], 8, 2, 128, "bf16"),
    ("block_edges_prefill", [(0, 64), (64, 64), (63, 2), (1, 127), (130, 67)], 8, 2, 128, "bf16"),
    ("chunk_crosses_blocks", [(30, 200)], 8, 8, 128, "bf16"),
    ("mha_d64_fp16", [(5, 40), (300, 1), (0, 33)], 4, 4, 64, "fp16"),
    ("gqa8_d128", [(100, 20), (2000, 1), (0, 17)], 32, 4, 128, "bf16"),
    ("gqa2_d128_fp16", [(700, 3), (50, 1), (0, 129)], 4, 2, 128, "fp16"),
    ("long_decode_many_splits", [(5000, 1), (3000, 1), (64 * 16 - 1, 1)], 8, 2, 128, "bf16"),
    ("g1_prefill_long", [(0, 300)], 2, 2, 128, "bf16"),
    # odd query-head counts with an odd number of split items (3 + 2 and
    # 3 + 8 splits of 4 blocks): the split partials' o region must stay
    # 16-byte aligned whatever items * heads is
    ("odd_heads3_split_decode", [(767, 1), (500, 1), (0, 40)], 3, 3, 64, "fp16"),
    ("single_head_split_decode", [(767, 1), (2000, 1), (0, 5)], 1, 1, 128, "bf16"),
]


@pytest.mark.parametrize("case", EDGE, ids=[e[0] for e in EDGE])
def test_edge_cases_full(case):
    name, seqs, hq, hkv, d, dt = case
    wl = W.make_custom(seqs, hq, hkv, d, dtype=dt, rope_theta=1e4 if d == 64 else 5e5, seed=3,
                       extra_blocks=3, name=name)
    _run_full(wl)


def test_interleaved_rotary():
    wl = W.make_custom([(10, 30), (200, 1), (64, 64)], 8, 2, 128, dtype="bf16", seed=4, extra_blocks=1)
    _run_full(wl, rope_style=R.DS_ROPE_INTERLEAVED)


def test_pool_canary_poisoned_slots():
    """Unused blocks and slots past each sequence's length hold NaN patterns;
    the append touches only its own slots and attention never reads the rest."""
    wl = W.make_custom([(37, 29), (90, 1), (130, 64), (0, 1), (250, 1)], 8, 2, 128, dtype="bf16",
                       seed=8, extra_blocks=6)
    _run_full(wl, poison_unused=True)
    wl = W.make_workload("tiny_gqa_d64", 0)
    _run_full(wl, poison_unused=True)


def test_empty_batch_is_a_no_op():
    wl = W.make_custom([], 4, 2, 64, extra_blocks=2)
    qkv = torch.zeros((1, wl.qkv_width), dtype=torch.float16, device="cuda")
    pool = torch.zeros(wl.pool_shape(), dtype=torch.float16, device="cuda")
    run = LayerRun(wl, qkv, pool)
    assert run.dev_err == 0 and run.layer.meta.n_tokens == 0
    assert torch.isnan(run.out).all()  # nothing written


# ------------------------------------------------------------------ full size

FULL = ["decode256_mha_d128", "splitfuse2048_gqa_d128", "chunked_prefill_2x8192", "max_ragged_8192"]
# the workloads whose lengths are drawn at random, also checked at seeds 1 and 2
RANDOM_LENGTHS = ["decode256_mha_d128", "splitfuse2048_gqa_d128", "max_ragged_8192"]


def _pick_sequences(wl, rng, n_pre=4, n_dec=12):
    pre = [i for i in range(wl.n_seqs) if wl.new[i] > 1]
    dec = [i for i in range(wl.n_seqs) if wl.new[i] == 1]
    pick = sorted(pre, key=lambda i: -int(wl.seen[i] + wl.new[i]))[:2] + \
        list(rng.choice(pre, size=min(len(pre), n_pre), replace=False)) if pre else []
    if dec:
        longest = max(dec, key=lambda i: int(wl.seen[i]))
        pick += [longest] + list(rng.choice(dec, size=min(len(dec), n_dec), replace=False))
    return sorted(set(int(i) for i in pick))


@pytest.mark.parametrize("name,seed", [(n, 0) for n in FULL] + [(n, s) for n in RANDOM_LENGTHS for s in (1, 2)])
def test_full_size_sampled(name, seed):
    wl = W.make_workload(name, seed)
    rng = np.random.default_rng(1234 + seed)
    qkv, pool = W.make_values(wl, "cuda")
    seqs = _pick_sequences(wl, rng)
    sub, pool_c, qkv_c, gidx, old_ids = compact(wl, seqs, pool, qkv)
    run = LayerRun(wl, qkv, pool, want_q=False)
    assert run.dev_err == 0
    # metadata bit-exact against the oracle's for the whole batch
    meta = run.layer.read_meta()
    ref_meta = oracle.meta_build(wl)
    for key in ["cu_seqlens", "seq_seen", "seq_new", "blk_off", "block_table", "tok_seq", "tok_pos"]:
        np.testing.assert_array_equal(meta[key], ref_meta[key], err_msg=key)
    # every row finite; every value placed bit-exactly in its slot
    N = wl.n_tokens
    assert torch.isfinite(run.out[:N].float()).all()
    tok_blk = np.array([wl.block_ids[s][p // 64] for s, p in zip(ref_meta["tok_seq"], ref_meta["tok_pos"])])
    tok_off = ref_meta["tok_pos"] % 64
    tb = torch.from_numpy(tok_blk).cuda()
    to = torch.from_numpy(tok_off.astype(np.int64)).cuda()
    v_slots = pool[tb, 1, :, to, :]  # [N, Hkv, d]
    Hq, Hkv, d = wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    v_in = qkv[:, (Hq + Hkv) * d:].view(N, Hkv, d)
    assert torch.equal(v_slots.view(torch.int16), v_in.view(torch.int16))
    # sampled sequences against the oracle
    rows = sample_rows(sub, rng)
    ref = oracle.layer(sub, qkv_c, pool_c, rows=rows)
    got = run.out[torch.from_numpy(gidx[rows]).cuda()]
    check_out(wl, got, ref["out"], name)
    # their blocks after the append: K within 1 ulp, V exact, other slots unchanged
    pa = bits(pool[torch.from_numpy(old_ids).cuda()]).reshape(ref["pool"].shape)
    assert ulp_diff(pa, ref["pool"]).max() <= 1
    np.testing.assert_array_equal(pa[:, 1], ref["pool"][:, 1])


# --------------------------------------------------------- self-consistency

def test_block_id_shuffle_is_bit_identical():
    wl = W.make_custom([(300, 50), (1000, 1), (64, 1), (0, 70)], 8, 2, 128, dtype="bf16", seed=5,
                       extra_blocks=4)
    qkv, pool = W.make_values(wl, "cuda")
    a = LayerRun(wl, qkv, pool.clone(), want_q=False).out
    perm = np.random.default_rng(0).permutation(wl.num_blocks)
    pool2 = torch.empty_like(pool)
    pool2[torch.from_numpy(perm).cuda()] = pool
    wl2 = W.make_custom([(300, 50), (1000, 1), (64, 1), (0, 70)], 8, 2, 128, dtype="bf16", seed=5,
                        extra_blocks=4)
    wl2.block_ids = [perm[b].astype(np.int32) for b in wl.block_ids]
    b = LayerRun(wl2, qkv, pool2, want_q=False).out
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_sequence_order_permutes_rows():
    seqs = [(300, 50), (1000, 1), (64, 1), (0, 70), (129, 5)]
    wl = W.make_custom(seqs, 8, 2, 128, dtype="bf16", seed=6, extra_blocks=4)
    qkv, pool = W.make_values(wl, "cuda")
    a = LayerRun(wl, qkv, pool.clone(), want_q=False).out
    order = [3, 1, 4, 0, 2]
    wl2 = W.subset(wl, order)
    cu = np.concatenate([[0], np.cumsum(wl.new)])
    gidx = np.concatenate([np.arange(cu[i], cu[i] + wl.new[i]) for i in order])
    qkv2 = qkv[torch.from_numpy(gidx).cuda()].contiguous()
    b = LayerRun(wl2, qkv2, pool.clone(), want_q=False).out
    assert torch.equal(a[torch.from_numpy(gidx).cuda()].view(torch.int16), b.view(torch.int16))


def test_device_error_word_on_inconsistent_metadata():
    """A block id outside the pool planted in an uploaded table is caught by
    the kernels' bounds checks (error bit set, access skipped, no fault)."""
    wl = W.make_custom([(100, 3), (200, 1)], 4, 2, 64, dtype="fp16", seed=7, extra_blocks=2)
    qkv, pool = W.make_values(wl, "cuda")
    run = LayerRun(wl, qkv, pool, want_q=False)
    assert run.dev_err == 0
    layer = run.layer
    layer.build(run.descs, wl.num_blocks)  # re-pack into the pinned staging buffer
    torch.cuda.synchronize()
    stage = layer.meta_stage.numpy().view(np.int32)
    off = (layer.meta.block_table - layer.meta.device_buf) // 4
    stage[off + 1] = wl.num_blocks + 5  # sequence 0's second block (holds its new tokens)
    layer.meta_dev[: layer.meta.used_bytes].copy_(layer.meta_stage[: layer.meta.used_bytes])
    layer.append(qkv, pool)
    layer.attention(qkv, pool, run.out)
    torch.cuda.synchronize()
    assert layer.device_error() & R.DS_DEVERR_BLOCK_ID


def test_stream_order_after_overlapped_launches():
    """The decode kernel may start while the prefill kernel still runs; work
    enqueued after the attention call on the same stream must still see both
    kernels' rows.  A long prefill chunk (slow) plus quick decodes, then an
    ordinary copy of the output on the same stream right after the call."""
    wl = W.make_custom([(20000, 256), (100, 1), (3000, 1), (64, 1)], 32, 8, 128, dtype="bf16",
                       seed=12, extra_blocks=2)
    qkv, pool = W.make_values(wl, "cuda")
    nb = int(wl.blocks_needed().sum())
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        layer = R.RaggedLayer(R.params_for(wl), wl.n_seqs, wl.n_tokens, nb, wl.max_len(), stream=stream)
        layer.build(R.SeqDescs.of(wl), wl.num_blocks)
        layer.append(qkv, pool)
        out = torch.full((wl.n_tokens, wl.n_q_heads * wl.head_dim), float("nan"), dtype=qkv.dtype,
                         device="cuda")
        for _ in range(3):
            out.fill_(float("nan"))
            layer.attention(qkv, pool, out)
            snap = out.clone()  # an ordinary kernel right behind the call
            stream.synchronize()
            assert torch.isfinite(snap.float()).all()
            assert torch.equal(snap.view(torch.int16), out.view(torch.int16))
