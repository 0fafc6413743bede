"""ds_blocked_attention_static_ws: the allocation-free attention entry point.

Some callers cannot allocate device memory (a plugin inside a host program
that owns the allocator, a latency-critical loop that must not call
cudaMalloc, a fixed memory budget reserved at start-up).  For them the library
offers an attention call that keeps its split-decode partials in a scratch
array built into the library instead of a caller workspace.  These tests call
it through the C ABI, twice in a row on two different batches, and compare
each result with the workspace-taking entry point's output on the same
inputs, within the layer's output tolerance.  The file is named so that
pytest collects it last.
"""
import numpy as np
import pytest
import torch

from gpu_util import MAX_ABS, MEAN_ABS
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _prepared(seqs, hq, hkv, d, dtype, seed):
    """A batch with its K/V appended through the C ABI, ready for attention."""
    wl = W.make_custom(seqs, hq, hkv, d, dtype=dtype, rope_theta=5e5, seed=seed, extra_blocks=3)
    qkv, pool = W.make_values(wl, "cuda")
    layer = R.RaggedLayer(R.params_for(wl), wl.n_seqs, wl.n_tokens, int(wl.blocks_needed().sum()),
                          wl.max_len())
    layer.build(R.SeqDescs.of(wl), wl.num_blocks)
    layer.append(qkv, pool)
    torch.cuda.synchronize()
    return wl, qkv, pool, layer


def _static_call(wl, qkv, pool, layer):
    out = torch.full((wl.n_tokens, wl.n_q_heads * wl.head_dim), float("nan"), dtype=qkv.dtype,
                     device="cuda")
    R.ds_blocked_attention_static_ws(layer.meta, layer.params, layer.rope, qkv,
                                     R.ds_kv_pool(pool.data_ptr(), pool.shape[0]), out)
    return out


def _close(wl, a, b):
    a = a.float().cpu().numpy()
    b = b.float().cpu().numpy()
    assert np.isfinite(a).all() and np.isfinite(b).all()
    err = np.abs(a - b)
    assert err.max() <= MAX_ABS[wl.dtype] and err.mean() <= MEAN_ABS, (err.max(), err.mean())


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
    for wl, qkv, pool, layer in (A, B):
        assert layer.device_error() == 0
    ref = []
    for wl, qkv, pool, layer in (A, B):
        o = torch.empty((wl.n_tokens, wl.n_q_heads * wl.head_dim), dtype=qkv.dtype, device="cuda")
        layer.attention(qkv, pool, o)
        ref.append(o)
    torch.cuda.synchronize()
    _close(A[0], out_a1, ref[0])
    _close(B[0], out_b1, ref[1])
    # a second round in a row: the array keeps the last call's contents, which
    # must not leak into the next result
    out_b2 = _static_call(*B)
    out_a2 = _static_call(*A)
    torch.cuda.synchronize()
    _close(A[0], out_a2, ref[0])
    _close(B[0], out_b2, ref[1])


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
    need = meta.n_decode_items * wl.n_q_heads * (wl.head_dim + 2) * 4
    assert need > R.DS_STATIC_WORKSPACE_BYTES
    rope = R.ds_rope_table(meta_dev.data_ptr(), wl.max_len(), wl.head_dim, float(wl.rope_theta))
    pool = R.ds_kv_pool(meta_dev.data_ptr(), wl.num_blocks)
    with pytest.raises(R.DSError) as ei:
        R.ds_blocked_attention_static_ws(meta, params, rope, meta_dev.data_ptr(), pool, meta_dev.data_ptr())
    assert ei.value.status == R.DS_ERR_WORKSPACE
