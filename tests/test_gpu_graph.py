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
