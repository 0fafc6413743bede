"""Multi-step Dynamic SplitFuse run on the GPU (block ledger + planner + the
layer through the C ABI), every pass compared with the oracle running the same
passes on its own pool; at the end the pools agree (K within 1 ulp, V exact)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import MAX_ABS, MEAN_ABS, bits, ulp_diff
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W
from test_ledger_cpu import _requests, run_plan

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [((8, 2), 128, "bf16"), ((4, 2), 64, "fp16")], ids=["gqa4_d128_bf16", "gqa2_d64_fp16"])
def test_multistep_splitfuse_matches_oracle(shape):
    heads, d, dtype = shape
    num_blocks = 40
    passes, _, _ = run_plan(num_blocks=num_blocks)
    f = dict(n_q_heads=heads[0], n_kv_heads=heads[1], head_dim=d, block_size=64, dtype=dtype,
             rope_theta=5e5, value_std=1.0)
    width = (heads[0] + 2 * heads[1]) * d
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    gen = torch.Generator(device="cuda").manual_seed(11)
    pool = torch.randn((num_blocks, 2, heads[1], 64, d), generator=gen, device="cuda").to(tdt)
    pool_oracle = oracle._bits(pool)
    params = R.make_params(heads[0], heads[1], d, dtype, 5e5)
    layer = R.RaggedLayer(params, 8, 128, num_blocks, 2048)
    worst = 0.0
    for k, batch in passes:
        if not batch:
            continue
        wl = W.RaggedWorkload(name="pass%d" % k, seen=np.array([b[1] for b in batch], np.int32),
                              new=np.array([b[2] for b in batch], np.int32),
                              block_ids=[b[3] for b in batch], num_blocks=num_blocks, **f)
        qkv = torch.randn((wl.n_tokens, width), generator=gen, device="cuda").to(tdt)
        out = torch.full((wl.n_tokens, heads[0] * d), float("nan"), dtype=tdt, device="cuda")
        layer.build(R.SeqDescs.of(wl), num_blocks)
        layer.append(qkv, pool)
        layer.attention(qkv, pool, out)
        torch.cuda.synchronize()
        assert layer.device_error() == 0
        ref = oracle.layer(wl, qkv.cpu(), pool_oracle)
        pool_oracle = ref["pool"]
        g = out.float().cpu().numpy().reshape(ref["out"].shape)
        err = np.abs(g - ref["out"])
        assert np.isfinite(g).all()
        assert err.max() <= MAX_ABS[dtype] and err.mean() <= MEAN_ABS, (k, err.max(), err.mean())
        worst = max(worst, err.max())
    pa = bits(pool).reshape(pool_oracle.shape)
    assert ulp_diff(pa, pool_oracle).max() <= 1
    np.testing.assert_array_equal(pa[:, 1], pool_oracle[:, 1])
