"""GPU: KV block offload/restore round trip (bit-exact) and the ragged
embedding / last-token logits gathers (bit-exact against plain indexing)."""
import numpy as np
import pytest
import torch

from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(8, 128, torch.bfloat16), (2, 64, torch.float16), (32, 128, torch.bfloat16)])
def test_offload_restore_round_trip(shape):
    hkv, d, dt = shape
    params = R.make_params(hkv, hkv, d, "bf16" if dt == torch.bfloat16 else "fp16")
    nblk = 37
    pool = torch.randn((nblk, 2, hkv, 64, d), device="cuda").to(dt)
    bb = R.ds_kv_block_bytes(params)
    assert bb == pool[0].numel() * 2
    ids = np.random.default_rng(0).permutation(nblk)[:1203 % nblk + 5].astype(np.int32)  # scattered ids
    host = torch.empty((len(ids), bb // 2), dtype=dt).pin_memory()
    host.view(torch.int16).fill_(-1)
    pk = R.ds_kv_pool(pool.data_ptr(), nblk)
    R.ds_kv_offload(params, pk, ids, host)
    torch.cuda.synchronize()
    want = pool[torch.from_numpy(ids.astype(np.int64)).cuda()].reshape(len(ids), -1).cpu()
    assert torch.equal(host.view(torch.int16), want.view(torch.int16))
    # restore into other blocks of a second pool
    pool2 = torch.zeros_like(pool)
    dst = np.random.default_rng(1).permutation(nblk)[:len(ids)].astype(np.int32)
    R.ds_kv_restore(params, R.ds_kv_pool(pool2.data_ptr(), nblk), dst, host)
    torch.cuda.synchronize()
    got = pool2[torch.from_numpy(dst.astype(np.int64)).cuda()]
    src = pool[torch.from_numpy(ids.astype(np.int64)).cuda()]
    assert torch.equal(got.view(torch.int16), src.view(torch.int16))
    untouched = np.setdiff1d(np.arange(nblk), dst)
    assert (pool2[torch.from_numpy(untouched).cuda()] == 0).all()


def test_offload_more_than_one_launch():
    params = R.make_params(1, 1, 64, "fp16")
    nblk = 2500
    pool = torch.randn((nblk, 2, 1, 64, 64), device="cuda").half()
    ids = np.random.default_rng(2).permutation(nblk)[:2100].astype(np.int32)
    host = torch.empty((len(ids), 2 * 64 * 64), dtype=torch.float16).pin_memory()
    R.ds_kv_offload(params, R.ds_kv_pool(pool.data_ptr(), nblk), ids, host)
    torch.cuda.synchronize()
    want = pool[torch.from_numpy(ids.astype(np.int64)).cuda()].reshape(len(ids), -1).cpu()
    assert torch.equal(host.view(torch.int16), want.view(torch.int16))


def test_embedding_and_logits_gather():
    wl = W.make_custom([(5, 3), (70, 1), (0, 40), (300, 7)], 4, 2, 64, extra_blocks=1)
    layer = R.RaggedLayer(R.params_for(wl), wl.n_seqs, wl.n_tokens, int(wl.blocks_needed().sum()), wl.max_len())
    layer.build(R.SeqDescs.of(wl), wl.num_blocks)
    vocab, hidden = 1000, 256
    table = torch.randn((vocab, hidden), device="cuda").bfloat16()
    ids = torch.randint(0, vocab, (wl.n_tokens,), device="cuda", dtype=torch.int32)
    out = torch.full((wl.n_tokens, hidden), float("nan"), device="cuda").bfloat16()
    R.ds_ragged_embedding(layer.meta, ids, table, out)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(out.view(torch.int16), table[ids.long()].view(torch.int16))
    # an id outside the table: error bit, zero row, the other rows intact
    ids[5] = vocab + 3
    R.ds_ragged_embedding(layer.meta, ids, table, out)
    torch.cuda.synchronize()
    assert layer.device_error() & R.DS_DEVERR_TOKEN
    assert (out[5] == 0).all() and torch.equal(out[6], table[ids[6].long()])
    # last-token rows
    hs = torch.randn((wl.n_tokens, 512), device="cuda").float()
    lg = torch.zeros((wl.n_seqs, 512), device="cuda")
    R.ds_ragged_logits_gather(layer.meta, hs, lg)
    torch.cuda.synchronize()
    last = np.cumsum(wl.new) - 1
    assert torch.equal(lg, hs[torch.from_numpy(last.astype(np.int64)).cuda()])
