"""C-ABI library on the CPU (no GPU): symbols, host packing, validation.

The library's host half (``ds_ragged_meta_pack``) runs without a device: these
tests compare its packed metadata bit for bit with the oracle's, check the
work lists' coverage invariant, and check every argument error code.  Calls
that would launch kernels are only exercised up to their host-side checks.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from ragged_blocked_kv_raggedbatch_gb300 import build as B
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE_DEV = 0x7F0000000000  # 256-aligned address that is never dereferenced on the host


@pytest.fixture(scope="module")
def lib():
    B.build()
    return R.load()


def test_exports_every_declared_symbol(lib):
    hdr = open(os.path.join(ROOT, "include", "ds_ragged.h")).read()
    declared = set(re.findall(r"^(?:ds_status|const char\*)\s+(ds_\w+)\s*\(", hdr, re.M))
    assert declared, "no declarations found"
    assert declared == set(R.SIGNATURES), declared ^ set(R.SIGNATURES)
    for name in declared:
        assert hasattr(lib, name), name
    assert b"sm_103a" in lib.ds_version()


class Packed:
    def __init__(self, wl, max_seqs=None, max_tokens=None, max_blocks=None, params=None,
                 pool_blocks=None):
        self.params = params or R.params_for(wl)
        self.max_seqs = wl.n_seqs if max_seqs is None else max_seqs
        self.max_tokens = wl.n_tokens if max_tokens is None else max_tokens
        nb = int(wl.blocks_needed().sum()) if wl.n_seqs else 0
        self.max_blocks = nb if max_blocks is None else max_blocks
        dev, stg = R.ds_meta_buffer_sizes(self.max_seqs, self.max_tokens, self.max_blocks, self.params)
        self.stage = np.zeros(stg // 4 + 4, np.int32)
        self.meta = R.ds_ragged_meta()
        self.meta.device_buf = FAKE_DEV
        self.meta.device_bytes = dev
        self.meta.host_staging = self.stage.ctypes.data
        self.meta.staging_bytes = stg
        self.meta.max_seqs, self.meta.max_tokens, self.meta.max_blocks = \
            self.max_seqs, self.max_tokens, self.max_blocks
        self.descs = R.SeqDescs.of(wl)
        self.pool_blocks = wl.num_blocks if pool_blocks is None else pool_blocks

    def pack(self):
        return R.ds_ragged_meta_pack(self.descs, self.params, self.pool_blocks, self.meta)

    def arrays(self):
        return R.unpack_meta(self.meta, self.stage, FAKE_DEV)


ALL = ["tiny_gqa_d64", "decode256_mha_d128", "splitfuse2048_gqa_d128", "chunked_prefill_2x8192",
       "max_ragged_8192"]


@pytest.mark.parametrize("name", ALL)
def test_pack_matches_oracle_bit_exact(lib, name):
    wl = W.make_workload(name, 0)
    pk = Packed(wl)
    assert pk.pack() == R.DS_OK, lib.ds_last_error()
    got = pk.arrays()
    want = oracle.meta_build(wl)
    for key in ["cu_seqlens", "seq_seen", "seq_new", "blk_off", "block_table", "tok_seq", "tok_pos"]:
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)
    assert got["header"][0] == 0 and got["header"][1] == wl.n_seqs and got["header"][2] == wl.n_tokens
    assert pk.meta.max_len == wl.max_len()
    _check_coverage(wl, pk.meta, got)


@pytest.mark.parametrize("case", range(40))
def test_pack_random_batches_bit_exact(lib, case):
    """Random ragged batches (mixes of first tokens, decodes and chunks that
    cross block boundaries; any head ratio and head size; spare pool blocks;
    capacities with slack) pack to the oracle's metadata and a covering work
    list."""
    rng = np.random.default_rng(7000 + case)
    n = int(rng.integers(1, 40))
    seqs = []
    for _ in range(n):
        kind = rng.integers(0, 4)
        seen = int(rng.choice([0, rng.integers(0, 64), rng.integers(0, 5000)]))
        new = 1 if kind < 2 else int(rng.integers(1, 600))
        seqs.append((seen, new))
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    wl = W.make_custom(seqs, hkv * g, hkv, d, dtype=str(rng.choice(["bf16", "fp16"])), seed=case,
                       extra_blocks=int(rng.integers(0, 20)))
    nb = int(wl.blocks_needed().sum())
    pk = Packed(wl, max_seqs=wl.n_seqs + int(rng.integers(0, 5)), max_tokens=wl.n_tokens + int(rng.integers(0, 50)),
                max_blocks=nb + int(rng.integers(0, 30)))
    assert pk.pack() == R.DS_OK, lib.ds_last_error()
    got = pk.arrays()
    want = oracle.meta_build(wl)
    for key in ["cu_seqlens", "seq_seen", "seq_new", "blk_off", "block_table", "tok_seq", "tok_pos"]:
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)
    _check_coverage(wl, pk.meta, got)


@pytest.mark.parametrize("name", ["tiny_gqa_d64", "splitfuse2048_gqa_d128", "max_ragged_8192"])
def test_pack_writes_every_uploaded_word(lib, name):
    """The packed image is the same whatever the staging buffer held before:
    every word up to used_bytes is written (or zeroed) by the pack."""
    wl = W.make_workload(name, 0)
    images = []
    for fill in (0, -0x54545455):  # zeros, then a 0xABABABAB pattern
        pk = Packed(wl)
        pk.stage[:] = fill
        assert pk.pack() == R.DS_OK
        images.append(pk.stage[: pk.meta.used_bytes // 4].copy())
    np.testing.assert_array_equal(images[0], images[1])


def _check_coverage(wl, meta, got):
    """Every prefill token is covered by exactly one tile; every KV block of
    every decode row by exactly one split item; slots are unique."""
    g = wl.n_q_heads // wl.n_kv_heads
    tile_tokens = 256 // g
    cover = {}
    kv_prev = None
    for seq, j0, nt, kv in got["prefill_tiles"]:
        assert wl.new[seq] > 1 and 1 <= nt <= tile_tokens
        assert kv == wl.seen[seq] + j0 + nt
        if kv_prev is not None:
            assert kv <= kv_prev  # longest atoms first
        kv_prev = kv
        for j in range(j0, j0 + nt):
            cover[(seq, j)] = cover.get((seq, j), 0) + 1
    for i in range(wl.n_seqs):
        if wl.new[i] > 1:
            for j in range(int(wl.new[i])):
                assert cover.get((i, j)) == 1
    assert sum(cover.values()) == int(wl.new[wl.new > 1].sum())
    dec = [i for i in range(wl.n_seqs) if wl.new[i] == 1]
    assert len(got["decode_seqs"]) == len(dec)
    # every decode row once, the longest first (ties in batch order)
    order = [int(r[0]) for r in got["decode_seqs"]]
    assert sorted(order) == dec
    assert order == sorted(dec, key=lambda i: -(-(-(int(wl.seen[i]) + 1) // 64)))
    slots = []
    for k, (seq, tok, first, cnt) in enumerate(got["decode_seqs"]):
        assert tok == got["cu_seqlens"][seq]
        nb = -(-(int(wl.seen[seq]) + 1) // 64)
        blocks = []
        split = meta.split_blocks
        # what the fused decode kernel's in-kernel merge derives from one item:
        # the row's split count and its first partial slot
        assert cnt == -(-nb // split)
        for k, it in enumerate(got["decode_items"][first:first + cnt]):
            assert it[0] == seq and it[2] - it[1] <= split
            assert it[1] == k * split
            blocks += list(range(it[1], it[2]))
            if cnt == 1:
                assert it[3] == -1
            else:
                slots.append(int(it[3]))
                assert it[3] - it[1] // split == got["decode_items"][first][3]
        assert blocks == list(range(nb))
    assert len(slots) == len(set(slots))
    assert len(got["decode_items"]) == meta.n_decode_items


def test_pack_edge_cases(lib):
    cases = [
        [],                                     # empty batch
        [(0, 1)],                               # first token of a sequence
        [(63, 1), (64, 1), (127, 2), (0, 64)],  # block boundaries
        [(0, 300), (5, 1)] * 3,
    ]
    for seqs in cases:
        wl = W.make_custom(seqs, 8, 2, 128, extra_blocks=5)
        pk = Packed(wl, max_seqs=max(1, wl.n_seqs), max_tokens=max(1, wl.n_tokens),
                    max_blocks=max(1, int(wl.blocks_needed().sum())))
        assert pk.pack() == R.DS_OK, lib.ds_last_error()
        got = pk.arrays()
        want = oracle.meta_build(wl)
        for key in ["cu_seqlens", "blk_off", "block_table", "tok_seq", "tok_pos"]:
            np.testing.assert_array_equal(got[key], want[key], err_msg=key)
        _check_coverage(wl, pk.meta, got)


def test_extra_block_ids_are_ignored(lib):
    wl = W.make_custom([(10, 5), (100, 1)], 4, 2, 64, extra_blocks=6)
    wl.block_ids[0] = np.concatenate([wl.block_ids[0], [wl.num_blocks - 1]]).astype(np.int32)
    pk = Packed(wl)
    assert pk.pack() == R.DS_OK
    np.testing.assert_array_equal(pk.arrays()["block_table"], oracle.meta_build(wl)["block_table"])


def _status(pk):
    return pk.pack()


def test_error_codes(lib):
    base = W.make_custom([(60, 10), (5, 1)], 4, 2, 64, extra_blocks=2)
    # block list too short
    wl = W.make_custom([(60, 10)], 4, 2, 64)
    wl.block_ids[0] = wl.block_ids[0][:1]
    assert _status(Packed(wl, max_blocks=4)) == R.DS_ERR_CAPACITY
    # id outside the pool
    wl = W.make_custom([(0, 3)], 4, 2, 64)
    wl.block_ids[0] = np.array([wl.num_blocks], np.int32)
    assert _status(Packed(wl)) == R.DS_ERR_BAD_BLOCK
    wl.block_ids[0] = np.array([-1], np.int32)
    assert _status(Packed(wl)) == R.DS_ERR_BAD_BLOCK
    # the same id in two sequences
    wl = W.make_custom([(0, 3), (0, 2)], 4, 2, 64, extra_blocks=1)
    wl.block_ids[1] = wl.block_ids[0].copy()
    assert _status(Packed(wl)) == R.DS_ERR_BAD_BLOCK
    # capacities
    assert _status(Packed(base, max_tokens=base.n_tokens - 1)) == R.DS_ERR_CAPACITY
    assert _status(Packed(base, max_seqs=1)) == R.DS_ERR_CAPACITY
    assert _status(Packed(base, max_blocks=1)) == R.DS_ERR_CAPACITY
    # new_tokens < 1, seen < 0
    wl = W.make_custom([(3, 1)], 4, 2, 64)
    pk = Packed(wl)
    pk.descs.arr[0].new_tokens = 0
    assert _status(pk) == R.DS_ERR_INVALID_ARG
    pk.descs.arr[0].new_tokens = 1
    pk.descs.arr[0].seen_tokens = -1
    assert _status(pk) == R.DS_ERR_INVALID_ARG
    # staging too small
    pk = Packed(base)
    pk.meta.staging_bytes = 8
    assert _status(pk) == R.DS_ERR_WORKSPACE
    # misaligned device buffer, NULL staging
    pk = Packed(base)
    pk.meta.device_buf = FAKE_DEV + 16
    assert _status(pk) == R.DS_ERR_INVALID_ARG
    pk = Packed(base)
    pk.meta.host_staging = None
    assert _status(pk) == R.DS_ERR_INVALID_ARG
    # unsupported shapes
    for kw, code in [(dict(head_dim=96), R.DS_ERR_UNSUPPORTED), (dict(n_q_heads=6, n_kv_heads=4), R.DS_ERR_UNSUPPORTED),
                     (dict(n_q_heads=64, n_kv_heads=2), R.DS_ERR_UNSUPPORTED), (dict(block_size=32), R.DS_ERR_UNSUPPORTED),
                     (dict(dtype=7), R.DS_ERR_UNSUPPORTED), (dict(rope_style=5), R.DS_ERR_UNSUPPORTED),
                     (dict(rope_theta=-1.0), R.DS_ERR_INVALID_ARG), (dict(n_kv_heads=0), R.DS_ERR_INVALID_ARG)]:
        p = R.make_params(4, 2, 64)
        for k, v in kw.items():
            setattr(p, k, v)
        dev, stg = ctypes.c_size_t(), ctypes.c_size_t()
        st = lib.ds_meta_buffer_sizes(4, 4, 4, R._ref(p), R._ref(dev), R._ref(stg))
        assert st == code, (kw, st)
    # NULL params / outputs
    assert lib.ds_meta_buffer_sizes(1, 1, 1, None, None, None) == R.DS_ERR_INVALID_ARG
    assert lib.ds_rope_table_size(R._ref(R.make_params(4, 2, 64)), -1, None) == R.DS_ERR_INVALID_ARG
    assert lib.ds_last_error()  # a message was recorded


def test_call_validation_before_launch(lib):
    """ds_kv_rotary_append / ds_blocked_attention reject bad arguments on the
    host (these cases return before any CUDA call)."""
    wl = W.make_custom([(70, 3), (5, 1)], 4, 2, 64, extra_blocks=1)
    pk = Packed(wl)
    assert pk.pack() == R.DS_OK
    p = pk.params
    rope = R.ds_rope_table(FAKE_DEV, wl.max_len(), 64, float(wl.rope_theta))
    pool = R.ds_kv_pool(FAKE_DEV, wl.num_blocks)
    ws = ctypes.c_size_t()
    assert lib.ds_blocked_attention_workspace_size(R._ref(p), 2, 4, 8, R._ref(ws)) == R.DS_OK
    append = lambda **kw: lib.ds_kv_rotary_append(R._ref(pk.meta), R._ref(p), R._ref(kw.get("rope", rope)),
                                                  kw.get("qkv", FAKE_DEV), kw.get("q_out"),
                                                  R._ref(kw.get("pool", pool)), None)
    attn = lambda **kw: lib.ds_blocked_attention(R._ref(pk.meta), R._ref(p), R._ref(kw.get("rope", rope)),
                                                 kw.get("qkv", FAKE_DEV), R._ref(kw.get("pool", pool)),
                                                 kw.get("out", FAKE_DEV), kw.get("ws", FAKE_DEV),
                                                 kw.get("ws_bytes", ws.value), None)
    assert append(qkv=None) == R.DS_ERR_INVALID_ARG
    assert append(qkv=FAKE_DEV + 2) == R.DS_ERR_INVALID_ARG
    assert append(q_out=FAKE_DEV + 8) == R.DS_ERR_INVALID_ARG
    assert append(rope=R.ds_rope_table(FAKE_DEV, wl.max_len() - 1, 64, float(wl.rope_theta))) == R.DS_ERR_CAPACITY
    assert append(rope=R.ds_rope_table(FAKE_DEV, wl.max_len(), 64, 123.0)) == R.DS_ERR_INVALID_ARG
    assert append(pool=R.ds_kv_pool(FAKE_DEV, wl.num_blocks + 1)) == R.DS_ERR_INVALID_ARG
    assert append(pool=R.ds_kv_pool(FAKE_DEV + 4, wl.num_blocks)) == R.DS_ERR_INVALID_ARG
    assert attn(out=None) == R.DS_ERR_INVALID_ARG
    assert attn(ws_bytes=16) == R.DS_ERR_WORKSPACE
    assert attn(ws=FAKE_DEV + 64) == R.DS_ERR_INVALID_ARG
    assert lib.ds_kv_rotary_append(None, R._ref(p), R._ref(rope), FAKE_DEV, None, R._ref(pool), None) == R.DS_ERR_INVALID_ARG


def test_fused_call_validation_before_launch(lib):
    """ds_fused_* reject bad arguments on the host; the fused workspace is the
    split-path workspace plus one int32 counter per (sequence slot, KV head)."""
    wl = W.make_custom([(70, 3), (5, 1), (200, 1)], 4, 2, 64, extra_blocks=1)
    pk = Packed(wl)
    assert pk.pack() == R.DS_OK
    p = pk.params
    rope = R.ds_rope_table(FAKE_DEV, wl.max_len(), 64, float(wl.rope_theta))
    pool = R.ds_kv_pool(FAKE_DEV, wl.num_blocks)
    ms, mt, mb = pk.meta.max_seqs, pk.meta.max_tokens, pk.meta.max_blocks
    split, fused = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.ds_blocked_attention_workspace_size(R._ref(p), ms, mt, mb, R._ref(split)) == R.DS_OK
    assert lib.ds_fused_workspace_size(R._ref(p), ms, mt, mb, R._ref(fused)) == R.DS_OK
    counters = -(-ms * p.n_kv_heads * 4 // 256) * 256
    assert fused.value == split.value + counters
    call = lambda **kw: lib.ds_fused_append_attention(
        R._ref(pk.meta), R._ref(p), R._ref(kw.get("rope", rope)), kw.get("qkv", FAKE_DEV),
        R._ref(kw.get("pool", pool)), kw.get("out", FAKE_DEV), kw.get("ws", FAKE_DEV),
        kw.get("ws_bytes", fused.value), None)
    assert call(out=None) == R.DS_ERR_INVALID_ARG
    assert call(qkv=FAKE_DEV + 2) == R.DS_ERR_INVALID_ARG
    # partials: (m, l) pairs, then o from the next 256-byte boundary
    items, hq = pk.meta.n_decode_items, p.n_q_heads
    need = counters + (-(-items * hq * 2 // 64) * 64 + items * hq * p.head_dim) * 4
    assert pk.meta.n_decode_items > 0
    assert call(ws_bytes=need - 4) == R.DS_ERR_WORKSPACE
    assert call(ws=FAKE_DEV + 64) == R.DS_ERR_INVALID_ARG
    assert call(rope=R.ds_rope_table(FAKE_DEV, wl.max_len() - 1, 64, float(wl.rope_theta))) == R.DS_ERR_CAPACITY
    assert call(pool=R.ds_kv_pool(FAKE_DEV, wl.num_blocks + 1)) == R.DS_ERR_INVALID_ARG
    init = lambda ws, nbytes: lib.ds_fused_workspace_init(R._ref(pk.meta), R._ref(p), ws, nbytes, None)
    assert init(FAKE_DEV, 16) == R.DS_ERR_WORKSPACE
    assert init(FAKE_DEV + 64, fused.value) == R.DS_ERR_INVALID_ARG
    assert init(None, fused.value) == R.DS_ERR_INVALID_ARG


def test_empty_batch_calls_enqueue_nothing(lib):
    """A batch with no sequences packs, and the layer calls return DS_OK
    before any CUDA call (so they are safe on a host without a GPU)."""
    wl = W.make_custom([], 4, 2, 64)
    pk = Packed(wl, max_seqs=1, max_tokens=1, max_blocks=1, pool_blocks=4)
    assert pk.pack() == R.DS_OK
    assert pk.meta.n_tokens == 0 and pk.meta.n_decode_items == 0 and pk.meta.n_prefill_tiles == 0
    p = pk.params
    rope = R.ds_rope_table(FAKE_DEV, 1, 64, float(wl.rope_theta))
    pool = R.ds_kv_pool(FAKE_DEV, 4)
    assert lib.ds_kv_rotary_append(R._ref(pk.meta), R._ref(p), R._ref(rope), FAKE_DEV, None,
                                   R._ref(pool), None) == R.DS_OK
    assert lib.ds_blocked_attention(R._ref(pk.meta), R._ref(p), R._ref(rope), FAKE_DEV, R._ref(pool),
                                    FAKE_DEV, None, 0, None) == R.DS_OK
    assert lib.ds_fused_append_attention(R._ref(pk.meta), R._ref(p), R._ref(rope), FAKE_DEV, R._ref(pool),
                                         FAKE_DEV, None, 0, None) == R.DS_OK


def test_offload_restore_and_gather_validation(lib):
    """Argument errors of the data-movement calls are found on the host."""
    p = R.make_params(8, 2, 128)
    bb = ctypes.c_size_t()
    assert lib.ds_kv_block_bytes(R._ref(p), R._ref(bb)) == R.DS_OK and bb.value == 2 * 2 * 64 * 128 * 2
    pool = R.ds_kv_pool(FAKE_DEV, 10)
    host = np.zeros(4096, np.uint8)
    ids = lambda *v: np.array(v, np.int32)
    for fn in (lib.ds_kv_offload, lib.ds_kv_restore):
        bad = ids(3, 10)
        assert fn(R._ref(p), R._ref(pool), bad.ctypes.data, 2, host.ctypes.data, None) == R.DS_ERR_BAD_BLOCK
        neg = ids(-1)
        assert fn(R._ref(p), R._ref(pool), neg.ctypes.data, 1, host.ctypes.data, None) == R.DS_ERR_BAD_BLOCK
        assert fn(R._ref(p), R._ref(pool), None, 1, host.ctypes.data, None) == R.DS_ERR_INVALID_ARG
        assert fn(R._ref(p), R._ref(pool), None, 0, None, None) == R.DS_OK
    dup = ids(4, 4)
    assert lib.ds_kv_restore(R._ref(p), R._ref(pool), dup.ctypes.data, 2, host.ctypes.data, None) == R.DS_ERR_BAD_BLOCK
    wl = W.make_custom([(5, 3), (70, 1)], 4, 2, 64)
    pk = Packed(wl)
    assert pk.pack() == R.DS_OK
    tok = FAKE_DEV
    assert lib.ds_ragged_embedding(R._ref(pk.meta), tok, FAKE_DEV, 100, 12, 2, FAKE_DEV, None) == R.DS_ERR_UNSUPPORTED
    assert lib.ds_ragged_embedding(R._ref(pk.meta), tok, FAKE_DEV + 8, 100, 64, 2, FAKE_DEV, None) == R.DS_ERR_INVALID_ARG
    assert lib.ds_ragged_embedding(R._ref(pk.meta), None, FAKE_DEV, 100, 64, 2, FAKE_DEV, None) == R.DS_ERR_INVALID_ARG
    assert lib.ds_ragged_logits_gather(R._ref(pk.meta), FAKE_DEV, 64, 3, FAKE_DEV, None) == R.DS_ERR_UNSUPPORTED
    assert lib.ds_ragged_logits_gather(None, FAKE_DEV, 64, 2, FAKE_DEV, None) == R.DS_ERR_INVALID_ARG


def test_capacity_layout_keeps_every_pointer_and_uploads_the_image(lib):
    """With DS_META_CAPACITY the regions sit at the offsets the capacities
    give: two different batches pack to the same device pointers and the same
    upload size (the whole image), with their counts in the header."""
    a = W.make_custom([(70, 3), (5, 1), (200, 1)], 8, 2, 128, extra_blocks=20, seed=1)
    b = W.make_custom([(0, 40), (1000, 1), (64, 64), (9, 1), (300, 1)], 8, 2, 128, extra_blocks=5, seed=2)
    caps = dict(max_seqs=6, max_tokens=200, max_blocks=40)
    ptr_names = ["header", "cu_seqlens", "seq_seen", "seq_new", "blk_off", "block_table", "tok_seq", "tok_pos",
                 "prefill_tiles", "decode_items", "decode_seqs"]
    got = []
    for wl in (a, b):
        pk = Packed(wl, pool_blocks=64, **caps)
        pk.meta.flags = R.DS_META_CAPACITY
        assert pk.pack() == R.DS_OK
        m = pk.meta
        dev_b, _ = R.ds_meta_buffer_sizes(6, 200, 40, pk.params)
        assert m.used_bytes <= dev_b and m.used_bytes > dev_b - 256
        hdr = pk.arrays()["header"]
        assert list(hdr[[1, 2, 6, 7, 8, 9]]) == [m.n_seqs, m.n_tokens, m.n_prefill_tiles, m.n_decode_items,
                                                 m.n_decode_seqs, m.split_blocks]
        assert hdr[10] == int(np.ceil(m.prefill_sms))
        assert list(hdr[[4, 5, 11, 12]]) == [0, 0, 0, 0]  # the kernels' own counters start at zero
        ref = oracle.meta_build(wl)
        arr = pk.arrays()
        for key in ["cu_seqlens", "seq_seen", "seq_new", "blk_off", "block_table", "tok_seq", "tok_pos"]:
            np.testing.assert_array_equal(arr[key], ref[key], err_msg=key)
        got.append([getattr(m, n) for n in ptr_names])
    assert got[0] == got[1]
    # without the flag the layout follows each batch's counts
    pa, pb = Packed(a, pool_blocks=64, **caps), Packed(b, pool_blocks=64, **caps)
    assert pa.pack() == R.DS_OK and pb.pack() == R.DS_OK
    assert pa.meta.tok_seq != pb.meta.tok_seq and pa.meta.used_bytes < pb.meta.used_bytes


def test_prefill_head_group_follows_the_longest_atom(lib):
    """Header word 14 orders the prefill atoms: one KV head at a time when the
    longest atom is short against a CTA's share of the prefill work (the
    chunked prefill), two otherwise, all heads (tile-major) when one atom
    outlasts that share; 0 when there is no prefill tile."""
    cases = [(W.make_workload("chunked_prefill_2x8192", 0), 1),
             (W.make_workload("max_ragged_8192", 0), 1),
             (W.make_workload("max_ragged_8192", 2), 2),
             (W.make_workload("tiny_gqa_d64", 0), 0),
             (W.make_workload("decode256_mha_d128", 0), 0)]
    for wl, want in cases:
        pk = Packed(wl)
        assert pk.pack() == R.DS_OK
        hdr = pk.arrays()["header"]
        assert hdr[14] == want, (wl.name, hdr[14], pk.meta.prefill_sms)
        assert list(hdr[[4, 5, 11, 12, 13]]) == [0, 0, 0, 0, 0]
