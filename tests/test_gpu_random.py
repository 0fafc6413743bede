"""Random small ragged batches through the whole CUDA path, against the oracle.

Each case draws a head ratio (1, 2, 4, 8), a head size (64, 128), a storage
type, a rotary style and a mix of first tokens, decodes and chunks that cross
block boundaries.  The two-call path is checked in full against the oracle
(metadata, appended pool, attention output); the fused call must then give
the same pool and output bits.
"""
import numpy as np
import pytest
import torch

from gpu_util import LayerRun, full_check
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _draw(case):
    rng = np.random.default_rng(9100 + case)
    seqs = []
    for _ in range(int(rng.integers(1, 9))):
        kind = int(rng.integers(0, 3))
        seen = int(rng.choice([0, rng.integers(0, 130), rng.integers(0, 1500)]))
        new = 1 if kind == 0 else int(rng.integers(1, 200))
        seqs.append((seen, new))
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["bf16", "fp16"]))
    style = int(rng.choice([R.DS_ROPE_HALF, R.DS_ROPE_INTERLEAVED]))
    wl = W.make_custom(seqs, hkv * g, hkv, d, dtype=dtype, seed=case, extra_blocks=int(rng.integers(0, 6)),
                       rope_theta=float(rng.choice([1e4, 5e5])))
    return wl, style


@pytest.mark.parametrize("case", range(12))
def test_random_batch_against_oracle_and_fused(case):
    wl, style = _draw(case)
    qkv, pool = W.make_values(wl, "cuda")
    pool0 = pool.clone()
    run = LayerRun(wl, qkv, pool, rope_style=style)
    full_check(wl, qkv, pool0, run, pool, style=style)
    # the fused call on the same inputs: the same bits
    pool_f = pool0.clone()
    nb = int(wl.blocks_needed().sum())
    layer = R.RaggedLayer(R.params_for(wl, style), wl.n_seqs, wl.n_tokens, nb, wl.max_len())
    layer.build(R.SeqDescs.of(wl), wl.num_blocks)
    out_f = torch.full_like(run.out, float("nan"))
    layer.fused(qkv, pool_f, out_f)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(out_f[: wl.n_tokens].view(torch.int16), run.out[: wl.n_tokens].view(torch.int16))
    assert torch.equal(pool_f.view(torch.int16), pool.view(torch.int16))
