"""The fused append + attention call (ds_fused_append_attention).

Against the two-call path (ds_kv_rotary_append, then ds_blocked_attention):
the same pool bits and the same output bits on every batch shape, including
decode rows split many ways, rows whose new token opens a block or fills its
last slot, and the first token of a sequence.  Against the oracle on a small
mixed batch.  Repeated calls and a captured graph replay to the same bits, and
the workspace's split counters are back at zero after every call.
"""
import types

import numpy as np
import pytest
import torch

from gpu_util import bits, full_check
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _layer(wl, rope_style=R.DS_ROPE_HALF, stream=None):
    nb = int(wl.blocks_needed().sum())
    layer = R.RaggedLayer(R.params_for(wl, rope_style), wl.n_seqs, wl.n_tokens, nb, wl.max_len(), stream=stream)
    layer.build(R.SeqDescs.of(wl), wl.num_blocks)
    return layer


def _counters_zero(layer):
    wl_heads = layer.params.n_kv_heads
    n = layer.meta.max_seqs * wl_heads
    c = layer.fused_ws[: 4 * n].view(torch.int32)
    return int(c.abs().sum().item()) == 0


def _both(wl, rope_style=R.DS_ROPE_HALF):
    qkv, pool = W.make_values(wl, "cuda")
    pool_a, pool_b = pool.clone(), pool.clone()
    d = wl.n_q_heads * wl.head_dim
    out_a = torch.full((wl.n_tokens, d), float("nan"), dtype=qkv.dtype, device="cuda")
    out_b = torch.full_like(out_a, float("nan"))
    la = _layer(wl, rope_style)
    la.append(qkv, pool_a)
    la.attention(qkv, pool_a, out_a)
    lb = _layer(wl, rope_style)
    lb.fused(qkv, pool_b, out_b)
    torch.cuda.synchronize()
    assert la.device_error() == 0 and lb.device_error() == 0
    return qkv, pool, pool_a, out_a, pool_b, out_b, lb


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


SMALL = {
    # decode-only, MHA: a first token (seen 0), a token that fills a block's last
    # slot (seen 63) and one that opens a block (seen 64), long rows split many ways
    "decode_only_mha_d128_bf16": ([(300, 1), (1000, 1), (64, 1), (63, 1), (0, 1), (4000, 1), (2049, 1)],
                                  8, 8, 128, "bf16"),
    "decode_only_gqa_d64_fp16": ([(5000, 1), (127, 1), (128, 1), (1, 1), (777, 1)], 8, 2, 64, "fp16"),
    "mixed_gqa_d128_bf16": ([(300, 40), (1000, 1), (64, 1), (0, 70), (2000, 1), (0, 1)], 8, 2, 128, "bf16"),
    "mixed_g8_d128_fp16": ([(500, 33), (3000, 1), (63, 1), (0, 200)], 16, 2, 128, "fp16"),
    "prefill_only_d64_bf16": ([(0, 100), (130, 64), (7, 9)], 4, 2, 64, "bf16"),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_fused_matches_two_calls(name):
    spec, hq, hkv, d, dt = SMALL[name]
    wl = W.make_custom(spec, hq, hkv, d, dtype=dt, seed=len(name), extra_blocks=3)
    qkv, pool, pool_a, out_a, pool_b, out_b, lb = _both(wl)
    assert _same_bits(pool_a, pool_b)
    assert _same_bits(out_a, out_b)
    if lb.fused_ws is not None:
        assert _counters_zero(lb)


def test_fused_interleaved_rotary():
    wl = W.make_custom([(900, 1), (64, 1), (10, 20)], 8, 4, 128, dtype="bf16", seed=3, extra_blocks=1)
    _, _, pool_a, out_a, pool_b, out_b, _ = _both(wl, R.DS_ROPE_INTERLEAVED)
    assert _same_bits(pool_a, pool_b) and _same_bits(out_a, out_b)


@pytest.mark.parametrize("name,n", [("decode256_mha_d128", 64), ("splitfuse2048_gqa_d128", 160),
                                    ("max_ragged_8192", 120)])
def test_fused_matches_two_calls_large(name, n):
    wl = W.first_sequences(W.make_workload(name, 0), n)
    _, _, pool_a, out_a, pool_b, out_b, lb = _both(wl)
    assert _same_bits(pool_a, pool_b)
    assert _same_bits(out_a, out_b)
    assert _counters_zero(lb)


def test_fused_against_oracle():
    wl = W.make_custom([(300, 40), (1000, 1), (64, 1), (0, 70), (2500, 1)], 8, 2, 128, dtype="bf16", seed=9,
                       extra_blocks=2)
    qkv, pool = W.make_values(wl, "cuda")
    pool0 = pool.clone()
    layer = _layer(wl)
    out = torch.full((wl.n_tokens, wl.n_q_heads * wl.head_dim), float("nan"), dtype=qkv.dtype, device="cuda")
    layer.fused(qkv, pool, out)
    torch.cuda.synchronize()
    run = types.SimpleNamespace(layer=layer, dev_err=layer.device_error(), q_out=None, out=out)
    full_check(wl, qkv, pool0, run, pool)


def test_fused_repeat_and_graph_replay():
    wl = W.make_custom([(300, 40), (1000, 1), (64, 1), (0, 70), (2000, 1), (4100, 1)], 8, 2, 128,
                       dtype="bf16", seed=21, extra_blocks=2)
    qkv, pool = W.make_values(wl, "cuda")
    pool0 = pool.clone()
    st = torch.cuda.Stream()
    d = wl.n_q_heads * wl.head_dim
    with torch.cuda.stream(st):
        layer = _layer(wl, stream=st)
        out_e = torch.full((wl.n_tokens, d), float("nan"), dtype=qkv.dtype, device="cuda")
        layer.fused(qkv, pool, out_e)
    st.synchronize()
    pool_e = pool.clone()
    assert _counters_zero(layer)
    # the same call again (the append rewrites the same bits)
    for _ in range(2):
        out_r = torch.full_like(out_e, float("nan"))
        with torch.cuda.stream(st):
            layer.fused(qkv, pool, out_r)
        st.synchronize()
        assert _same_bits(out_r, out_e) and _same_bits(pool, pool_e) and _counters_zero(layer)
    # a captured layer step (metadata upload + fused call) replays to the same bits
    pool.copy_(pool0)
    out_g = torch.full_like(out_e, float("nan"))
    descs = R.SeqDescs.of(wl)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        layer.build(descs, wl.num_blocks)
        layer.fused(qkv, pool, out_g)
    for _ in range(3):
        out_g.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert _same_bits(out_g, out_e) and _same_bits(pool, pool_e) and _counters_zero(layer)
