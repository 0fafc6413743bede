"""The prefill kernel's atom order does not change a bit of its output.

The kernel takes its (tile, KV head) atoms longest first in rounds of
n_ctas / hg tiles, the heads of a round in groups of hg (header word 14, which
the host picks per batch), and the CTAs take atoms dynamically.  Every atom is
computed by one CTA in a fixed order, so any head grouping and any number of
working CTAs must give the same output bits.  Here the header words are
overwritten on the device after the upload to force each grouping and a grid
of a few CTAs (many rounds), and the output is checked bit for bit against
the host's own choice, which is checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_out
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HDR_PRE_CTAS, HDR_PRE_HG = 10, 14


@pytest.mark.parametrize("shape", [(16, 8, 128, "bf16"), (32, 8, 128, "fp16"), (8, 4, 64, "bf16")],
                         ids=["g2_d128_bf16", "g4_d128_fp16", "g2_d64_bf16"])
def test_atom_order_and_grid_size_leave_the_output_bits_alone(shape):
    hq, hkv, d, dt = shape
    # prefill chunks of several lengths over histories of several lengths,
    # plus decode rows (so the host also sizes the prefill grid)
    seqs = [(1500, 300), (0, 260), (700, 129), (90, 64), (2200, 1), (31, 1), (0, 37)]
    wl = W.make_custom(seqs, hq, hkv, d, dtype=dt, rope_theta=1e4, seed=3, extra_blocks=4)
    qkv, pool = W.make_values(wl, "cuda")
    pool_before = pool.clone()
    layer = R.RaggedLayer(R.params_for(wl), wl.n_seqs, wl.n_tokens, int(wl.blocks_needed().sum()), wl.max_len())
    layer.build(R.SeqDescs.of(wl), wl.num_blocks)
    layer.append(qkv, pool)
    hdr_at = (int(layer.meta.header) - int(layer.meta_dev.data_ptr())) // 4
    words = layer.meta_dev.view(torch.int32)

    def run():
        out = torch.full((wl.n_tokens, hq * d), float("nan"), dtype=qkv.dtype, device="cuda")
        layer.attention(qkv, pool, out)
        torch.cuda.synchronize()
        assert layer.device_error() == 0
        return out

    base = run()
    ref = oracle.layer(wl, qkv.cpu(), pool_before.cpu())
    check_out(wl, base[: wl.n_tokens], ref["out"], "host's atom order")
    want = base.view(torch.int16).cpu().numpy()
    for hg in (0, 1, 2, 4, hkv):
        for ctas in (0, 1, 3, 7):
            words[hdr_at + HDR_PRE_HG] = hg
            words[hdr_at + HDR_PRE_CTAS] = ctas
            got = run().view(torch.int16).cpu().numpy()
            np.testing.assert_array_equal(got, want, err_msg="head group %d, %d CTAs" % (hg, ctas))
