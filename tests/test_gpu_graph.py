"""A layer step captured in a CUDA graph (metadata upload, KV append,
attention with the prefill/decode programmatic dependency) replays to the
same bits as the eager calls."""
import numpy as np
import pytest
import torch

from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["thread_local", "global"])
def test_graph_replay_matches_eager(mode):
    wl = W.make_custom([(300, 40), (1000, 1), (64, 1), (0, 70), (2000, 1)], 8, 2, 128, dtype="bf16",
                       seed=21, extra_blocks=2)
    qkv, pool = W.make_values(wl, "cuda")
    pool0 = pool.clone()
    nb = int(wl.blocks_needed().sum())
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        layer = R.RaggedLayer(R.params_for(wl), wl.n_seqs, wl.n_tokens, nb, wl.max_len(), stream=st)
        descs = R.SeqDescs.of(wl)
        out_e = torch.empty((wl.n_tokens, wl.n_q_heads * wl.head_dim), dtype=qkv.dtype, device="cuda")
        layer.build(descs, wl.num_blocks)
        layer.append(qkv, pool)
        layer.attention(qkv, pool, out_e)
    st.synchronize()
    pool_e = pool.clone()
    pool.copy_(pool0)
    out_g = torch.full_like(out_e, float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st, capture_error_mode=mode):
        layer.build(descs, wl.num_blocks)
        layer.append(qkv, pool)
        layer.attention(qkv, pool, out_g)
    for _ in range(3):
        out_g.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16))
        assert torch.equal(pool.view(torch.int16), pool_e.view(torch.int16))


# One graph for any batch within the capacities (DS_META_CAPACITY): captured
# once, replayed on batches of other shapes, each checked against the oracle.
CAPS = dict(max_seqs=8, max_tokens=420, max_blocks=170)
POOL_BLOCKS = 200
SHAPES = [
    [(0, 37), (90, 1), (130, 64), (2000, 1)],                          # mixed
    [(500, 1), (64, 1), (63, 1), (3000, 1), (0, 1)],                   # decode rows only
    [(10, 300)],                                                       # one prefill chunk
    [(1000, 150), (5, 1), (777, 1), (0, 100), (2500, 1), (128, 20)],   # mixed, more rows and tokens
]


@pytest.mark.parametrize("path", ["fused", "split"])
@pytest.mark.parametrize("shape", [(8, 2, 128, "bf16"), (4, 4, 64, "fp16")], ids=["gqa4_d128_bf16", "mha_d64_fp16"])
def test_one_graph_replays_any_batch_within_capacity(path, shape):
    import oracle
    from gpu_util import bits, check_out, ulp_diff

    hq, hkv, d, dtype = shape
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    wls = []
    for k, seqs in enumerate(SHAPES):
        need = int(sum(-(-(s + n) // 64) for s, n in seqs))
        wls.append(W.make_custom(seqs, hq, hkv, d, dtype=dtype, rope_theta=5e5, seed=40 + k,
                                 extra_blocks=POOL_BLOCKS - need))
    params = R.params_for(wls[0])
    st = torch.cuda.Stream()
    gen = torch.Generator(device="cuda").manual_seed(7)
    with torch.cuda.stream(st):
        layer = R.RaggedLayer(params, CAPS["max_seqs"], CAPS["max_tokens"], CAPS["max_blocks"], 3200, stream=st,
                              flags=R.DS_META_CAPACITY)
        pool = torch.randn((POOL_BLOCKS, 2, hkv, 64, d), generator=gen, device="cuda").to(tdt)
        qkv = torch.zeros((CAPS["max_tokens"], wls[0].qkv_width), dtype=tdt, device="cuda")
        out = torch.zeros((CAPS["max_tokens"], hq * d), dtype=tdt, device="cuda")
        fb = R.ds_fused_workspace_size(params, CAPS["max_seqs"], CAPS["max_tokens"], CAPS["max_blocks"])
        layer.fused_ws = torch.empty(fb, dtype=torch.uint8, device="cuda")
        R.ds_fused_workspace_init(layer.meta, params, layer.fused_ws, st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        layer.build(R.SeqDescs.of(wls[0]), POOL_BLOCKS)
        if path == "fused":
            layer.fused(qkv, pool, out)
        else:
            layer.append(qkv, pool)
            layer.attention(qkv, pool, out)
    for wl in wls + wls[:1]:
        N = wl.n_tokens
        rows = torch.randn((N, wl.qkv_width), generator=gen, device="cuda").to(tdt)
        st.synchronize()
        layer.pack(R.SeqDescs.of(wl), POOL_BLOCKS)  # the next replay uploads this batch
        qkv[:N].copy_(rows)
        out.fill_(float("nan"))
        pool_before = pool.clone()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert layer.device_error() == 0, wl.seen
        ref = oracle.layer(wl, rows.cpu(), pool_before.cpu())
        check_out(wl, out[:N], ref["out"], "graph replay %s" % list(zip(wl.seen, wl.new)))
        pa = bits(pool).reshape(wl.pool_shape())
        assert ulp_diff(pa, ref["pool"]).max() <= 1
        np.testing.assert_array_equal(pa[:, 1], ref["pool"][:, 1])
    if path == "fused":  # every clean call leaves the split counters at zero
        c = layer.fused_ws[: 4 * CAPS["max_seqs"] * hkv].view(torch.int32)
        assert int(c.abs().sum().item()) == 0
