"""ds_blocked_attention_static_ws: the allocation-free attention entry point.

Some callers cannot allocate device memory (a plugin inside a host program
that owns the allocator, a latency-critical loop that must not call
cudaMalloc, a fixed memory budget reserved at start-up).  For them the library
offers an attention call that keeps its split-decode partials in a scratch
array built into the library instead of a caller workspace.  These tests call
it through the C ABI, twice in a row on two different batches.  Both entry
points run the same kernels on the same work list and differ only in where
the partials live, so each result must be bit-identical to the
workspace-taking entry point's output on the same inputs; one call is also
checked against the CPU oracle within the layer's output tolerance.  The file
is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_out
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _prepared(seqs, hq, hkv, d, dtype, seed):
    """A batch with its K/V appended through the C ABI, ready for attention,
    and the pool as it was before the append (the oracle's input)."""
    wl = W.make_custom(seqs, hq, hkv, d, dtype=dtype, rope_theta=5e5, seed=seed, extra_blocks=3)
    qkv, pool = W.make_values(wl, "cuda")
    pool_before = pool.clone()
    layer = R.RaggedLayer(R.params_for(wl), wl.n_seqs, wl.n_tokens, int(wl.blocks_needed().sum()),
                          wl.max_len())
    layer.build(R.SeqDescs.of(wl), wl.num_blocks)
    layer.append(qkv, pool)
    torch.cuda.synchronize()
    return wl, qkv, pool, layer, pool_before


def _static_call(wl, qkv, pool, layer, _pool_before):
    out = torch.full((wl.n_tokens, wl.n_q_heads * wl.head_dim), float("nan"), dtype=qkv.dtype,
                     device="cuda")
    R.ds_blocked_attention_static_ws(layer.meta, layer.params, layer.rope, qkv,
                                     R.ds_kv_pool(pool.data_ptr(), pool.shape[0]), out)
    return out


def _same_bits(a, b):
    assert torch.isfinite(a.float()).all()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_static_workspace_matches_workspace_entry_point_two_calls():
    # batch A: decode rows with many splits (partials go through the scratch
    # array) plus a prefill chunk; batch B: another shape and dtype
    A = _prepared([(5000, 1), (3000, 1), (100, 50), (1023, 1), (64 * 20, 1)], 8, 2, 128, "bf16", 1)
    B = _prepared([(700, 1), (9000, 1), (0, 33), (130, 1)], 4, 2, 64, "fp16", 2)
    assert A[3].meta.n_decode_items > A[3].meta.n_decode_seqs  # splits really use scratch
    assert B[3].meta.n_decode_items > B[3].meta.n_decode_seqs
    out_a1 = _static_call(*A)
    out_b1 = _static_call(*B)
    torch.cuda.synchronize()
    for wl, qkv, pool, layer, _ in (A, B):
        assert layer.device_error() == 0
    ref = []
    for wl, qkv, pool, layer, _ in (A, B):
        o = torch.empty((wl.n_tokens, wl.n_q_heads * wl.head_dim), dtype=qkv.dtype, device="cuda")
        layer.attention(qkv, pool, o)
        ref.append(o)
    torch.cuda.synchronize()
    _same_bits(out_a1, ref[0])
    _same_bits(out_b1, ref[1])
    # a second round in a row: the array keeps the last call's contents, which
    # must not leak into the next result
    out_b2 = _static_call(*B)
    out_a2 = _static_call(*A)
    torch.cuda.synchronize()
    _same_bits(out_a2, ref[0])
    _same_bits(out_b2, ref[1])
    # and the CPU oracle on batch B (the pool as it was before the append)
    wl, qkv, _, _, pool_before = B
    want = oracle.layer(wl, qkv.cpu(), pool_before.cpu())["out"]
    check_out(wl, out_b2, want, "static workspace vs oracle")


def test_static_workspace_rejects_oversize_batch():
    """A batch whose split partials exceed the built-in array is refused with
    DS_ERR_WORKSPACE before anything is enqueued."""
    # 640 decode rows of 8192 keys, 32 query heads of d=128: 4 splits of 32
    # blocks each, 2560 items x 32 heads x 130 floats = 42.6 MB > 32 MiB
    wl = W.make_custom([(8191, 1)] * 640, 32, 32, 128, dtype="bf16", seed=3)
    params = R.params_for(wl)
    nb = int(wl.blocks_needed().sum())
    dev_b, stg_b = R.ds_meta_buffer_sizes(wl.n_seqs, wl.n_tokens, nb, params)
    meta_dev = torch.empty(dev_b, dtype=torch.uint8, device="cuda")
    stage = np.zeros(stg_b // 4 + 4, np.int32)
    meta = R.ds_meta_init(meta_dev, stage, wl.n_seqs, wl.n_tokens, nb)
    assert R.ds_ragged_meta_pack(R.SeqDescs.of(wl), params, wl.num_blocks, meta) == R.DS_OK
    items, hq = meta.n_decode_items, wl.n_q_heads
    need = (-(-items * hq * 2 // 64) * 64 + items * hq * wl.head_dim) * 4
    assert need > R.DS_STATIC_WORKSPACE_BYTES
    rope = R.ds_rope_table(meta_dev.data_ptr(), wl.max_len(), wl.head_dim, float(wl.rope_theta))
    pool = R.ds_kv_pool(meta_dev.data_ptr(), wl.num_blocks)
    with pytest.raises(R.DSError) as ei:
        R.ds_blocked_attention_static_ws(meta, params, rope, meta_dev.data_ptr(), pool, meta_dev.data_ptr())
    assert ei.value.status == R.DS_ERR_WORKSPACE
