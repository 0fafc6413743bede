"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: a value
derived by hand from the batch description, a library routine (numpy's fp16
rounding, torch's bf16 rounding), a closed form (complex rotation, mean of V,
a single key), an invariant (norm preservation, relative positions, chunked vs
one-shot prefill, GQA vs replicated heads), or an independent brute-force
computation (dense masked attention on an unpadded per-sequence copy).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _runs_const(runs):
    return np.concatenate([np.full(c, v) for v, c in runs]).astype(np.int64)


def _runs_range(runs):
    return np.concatenate([np.arange(s, s + c) for s, c in runs]).astype(np.int64)


# --------------------------------------------------------------------------
# storage rounding: pinned to numpy (fp16) and torch (bf16)
# --------------------------------------------------------------------------

def _special_floats():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-5).astype(np.float32),   # fp16 subnormals
        (rng.standard_normal(5000) * 3e4).astype(np.float32),    # near fp16 max
        np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.0, 65520.0, 65536.0, 1e30, -1e30,
                  6.1035156e-05, 5.9604645e-08, 2.9802322e-08, 2.9802326e-08,
                  np.inf, -np.inf], np.float32),
    ])
    # exact ties of the fp16 grid: 1 + (2k+1) * 2^-11
    ties = (1.0 + (2 * np.arange(64) + 1) * 2.0 ** -11).astype(np.float32)
    return np.concatenate([x, ties, -ties])


def test_fp16_rounding_matches_numpy():
    x = _special_floats()
    got = oracle.f32_to_storage(x, "fp16")
    want = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_bf16_rounding_matches_torch():
    x = _special_floats()
    ties = (1.0 + (2 * np.arange(64) + 1) * 2.0 ** -8).astype(np.float32)  # bf16 ties
    x = np.concatenate([x, ties, -ties])
    got = oracle.f32_to_storage(x, "bf16")
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_storage_decode_matches_libraries():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    h = oracle.storage_to_f64(bits, "fp16")
    ref = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(h[fin], ref[fin])
    assert np.all(np.isnan(h[np.isnan(ref)]))
    b = oracle.storage_to_f64(bits, "bf16")
    refb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    finb = np.isfinite(refb)
    np.testing.assert_array_equal(b[finb], refb[finb])


# --------------------------------------------------------------------------
# rotary embedding
# --------------------------------------------------------------------------

def _complex_rope(x, p, theta):
    """Rotation as a complex product: (x_k + i x_{k+d/2}) * exp(i p theta^(-2k/d))."""
    d = x.shape[-1]
    k = np.arange(d // 2, dtype=np.float64)
    f = theta ** (-2.0 * k / d)
    z = (x[..., : d // 2] + 1j * x[..., d // 2:]) * np.exp(1j * p * f)
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("theta", [1e4, 5e5, 1e6])
def test_rope_matches_complex_rotation(d, theta):
    rng = np.random.default_rng(d)
    for p in [0, 1, 7, 63, 64, 130, 4097, 8191, 16383, 32767, 33791]:
        x = rng.standard_normal(d).astype(np.float32)
        y64 = oracle.rope_vec_f64(x.astype(np.float64), p, theta)
        want = _complex_rope(x.astype(np.float64), p, theta)
        np.testing.assert_allclose(y64, want, rtol=0, atol=1e-9)
        y32 = oracle.rope_vec_f32(x, p, theta)
        # fp32 evaluation: the angle is rounded to fp32 (p*f has relative error
        # 2^-24, i.e. an absolute angle error up to ~2e-3 rad at p = 33791), so
        # compare with the complex rotation by the fp32-rounded angle.
        k = np.arange(d // 2, dtype=np.float64)
        f32 = (theta ** (-2.0 * k / d)).astype(np.float32)
        ang = (np.float32(p) * f32).astype(np.float64)
        z = (x[: d // 2].astype(np.float64) + 1j * x[d // 2:].astype(np.float64)) * np.exp(1j * ang)
        want32 = np.concatenate([z.real, z.imag])
        np.testing.assert_allclose(y32, want32, rtol=0, atol=4e-6 * max(1.0, np.abs(x).max()))


def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(128).astype(np.float32)
    np.testing.assert_array_equal(oracle.rope_vec_f32(x, 0, 1e4), x)
    np.testing.assert_array_equal(oracle.rope_vec_f64(x.astype(np.float64), 0, 1e4), x.astype(np.float64))


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(128)
    y = oracle.rope_vec_f64(x, 12345, 5e5)
    nx = x[:64] ** 2 + x[64:] ** 2
    ny = y[:64] ** 2 + y[64:] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(5)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    for (p, u, c) in [(10, 3, 1000), (16383, 0, 7), (500, 499, 16000)]:
        s1 = oracle.rope_vec_f64(q, p, 5e5) @ oracle.rope_vec_f64(k, u, 5e5)
        s2 = oracle.rope_vec_f64(q, p + c, 5e5) @ oracle.rope_vec_f64(k, u + c, 5e5)
        assert abs(s1 - s2) <= 1e-9 * (1 + abs(s1))


def test_rope_interleaved_is_half_under_permutation():
    d = 64
    rng = np.random.default_rng(6)
    x = rng.standard_normal(d)
    # interleaved pairs (2k, 2k+1) are half pairs (k, k + d/2) after gathering
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])
    yi = oracle.rope_vec_f64(x, 77, 1e4, oracle.ROPE_INTERLEAVED)
    yh = oracle.rope_vec_f64(x[perm], 77, 1e4, oracle.ROPE_HALF)
    np.testing.assert_array_equal(yi[perm], yh)


# --------------------------------------------------------------------------
# metadata and slot placement
# --------------------------------------------------------------------------

def test_meta_tiny_matches_hand_derived_golden():
    g = json.load(open(os.path.join(GOLDEN, "tiny_gqa_d64_meta.json")))
    wl = W.make_workload("tiny_gqa_d64", 0)
    m = oracle.meta_build(wl)
    for key in ["cu_seqlens", "seq_seen", "seq_new", "blk_off"]:
        np.testing.assert_array_equal(m[key], g[key], err_msg=key)
    np.testing.assert_array_equal(m["tok_seq"], _runs_const(g["tok_seq_const_runs"]))
    np.testing.assert_array_equal(m["tok_pos"], _runs_range(g["tok_pos_ranges"]))
    np.testing.assert_array_equal(m["block_table"], np.concatenate(wl.block_ids))
    qkv, pool = W.make_values(wl, "cpu")
    _, _, sb, so = oracle.rope_append(wl, m, qkv, pool)
    np.testing.assert_array_equal(so, _runs_range(g["slot_offset_ranges"]))
    list_idx = _runs_const(g["slot_list_index_const_runs"])
    want_blocks = [wl.block_ids[int(m["tok_seq"][t])][list_idx[t]] for t in range(len(so))]
    np.testing.assert_array_equal(sb, want_blocks)


def test_meta_random_batches_brute_force():
    rng = np.random.default_rng(7)
    for trial in range(20):
        S = int(rng.integers(0, 12))
        seqs = [(int(rng.integers(0, 300)), int(rng.integers(1, 150))) for _ in range(S)]
        wl = W.make_custom(seqs, 4, 2, 64, seed=trial, extra_blocks=int(rng.integers(0, 5)))
        m = oracle.meta_build(wl)
        cu, bo, ts, tp, bt = [0], [0], [], [], []
        for i, (s, n) in enumerate(seqs):
            cu.append(cu[-1] + n)
            nb = -(-(s + n) // 64)
            bo.append(bo[-1] + nb)
            bt += list(wl.block_ids[i][:nb])
            for j in range(n):
                ts.append(i)
                tp.append(s + j)
        np.testing.assert_array_equal(m["cu_seqlens"], cu)
        np.testing.assert_array_equal(m["blk_off"], bo)
        np.testing.assert_array_equal(m["tok_seq"], np.array(ts, dtype=np.int32))
        np.testing.assert_array_equal(m["tok_pos"], np.array(tp, dtype=np.int32))
        np.testing.assert_array_equal(m["block_table"], np.array(bt, dtype=np.int32))


def test_meta_rejects_short_block_list():
    wl = W.make_custom([(60, 10)], 4, 2, 64)
    wl.block_ids[0] = wl.block_ids[0][:1]  # needs 2 blocks for 70 positions
    with pytest.raises(ValueError):
        oracle.meta_build(wl)


def _np_rope32_store(x32, p, theta, dtype):
    """Independent numpy evaluation of the stored rotation (fp32 ops in the
    documented order; cos/sin of the fp32 angle via the math module), rounded by
    numpy (fp16) or torch (bf16)."""
    d = x32.shape[-1]
    k = np.arange(d // 2)
    f = np.array([np.float32(math.pow(theta, -2.0 * kk / d)) for kk in k], np.float32)
    a = (np.float32(p) * f).astype(np.float32)
    c = np.array([np.float32(math.cos(float(v))) for v in a], np.float32)
    s = np.array([np.float32(math.sin(float(v))) for v in a], np.float32)
    x0, x1 = x32[: d // 2], x32[d // 2:]
    y = np.concatenate([(x0 * c) - (x1 * s), (x1 * c) + (x0 * s)]).astype(np.float32)
    if dtype == "fp16":
        return y.astype(np.float16).view(np.uint16)
    return torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _decode_bits(bits, dtype):
    bits = np.asarray(bits, np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


@pytest.mark.parametrize("name", ["tiny_gqa_d64"])
def test_append_places_exact_slots_and_values(name):
    wl = W.make_workload(name, 0)
    qkv, pool = W.make_values(wl, "cpu")
    m = oracle.meta_build(wl)
    before = oracle._bits(pool).reshape(wl.pool_shape())
    after, q_rot, sb, so = oracle.rope_append(wl, m, qkv, pool)
    qkv_b = oracle._bits(qkv).reshape(wl.n_tokens, -1)
    Hq, Hkv, d, bs = wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.block_size
    expect = set()
    t = 0
    for i in range(wl.n_seqs):
        for j in range(int(wl.new[i])):
            p = int(wl.seen[i]) + j
            blk, off = int(wl.block_ids[i][p // bs]), p % bs
            assert (sb[t], so[t]) == (blk, off)
            expect.add((blk, off))
            for h in range(Hkv):
                kin = _decode_bits(qkv_b[t, (Hq + h) * d:(Hq + h + 1) * d], wl.dtype).astype(np.float32)
                np.testing.assert_array_equal(after[blk, 0, h, off], _np_rope32_store(kin, p, wl.rope_theta, wl.dtype))
                np.testing.assert_array_equal(after[blk, 1, h, off], qkv_b[t, (Hq + Hkv + h) * d:(Hq + Hkv + h + 1) * d])
            for h in range(Hq):
                qin = _decode_bits(qkv_b[t, h * d:(h + 1) * d], wl.dtype).astype(np.float32)
                np.testing.assert_array_equal(q_rot[t, h * d:(h + 1) * d], _np_rope32_store(qin, p, wl.rope_theta, wl.dtype))
            t += 1
    changed = np.argwhere(np.any(after != before, axis=(1, 2, 4)))
    for blk, off in changed:
        assert (int(blk), int(off)) in expect
    # untouched slots are bit-identical
    mask = np.ones((wl.num_blocks, bs), bool)
    for blk, off in expect:
        mask[blk, off] = False
    np.testing.assert_array_equal(after.transpose(0, 3, 1, 2, 4)[mask], before.transpose(0, 3, 1, 2, 4)[mask])


# --------------------------------------------------------------------------
# attention: brute force on an unpadded per-sequence copy
# --------------------------------------------------------------------------

def _brute_force(wl, qkv, pool):
    """Dense masked attention per sequence, from the raw inputs only."""
    Hq, Hkv, d, bs = wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.block_size
    g = Hq // Hkv
    qkv_b = oracle._bits(qkv).reshape(wl.n_tokens, -1)
    pool_b = oracle._bits(pool).reshape(wl.pool_shape())
    outs = []
    t0 = 0
    for i in range(wl.n_seqs):
        s, n = int(wl.seen[i]), int(wl.new[i])
        L = s + n
        ids = wl.block_ids[i]
        hist = np.array([[ids[u // bs], u % bs] for u in range(s)], np.int64).reshape(-1, 2)
        Kh = _decode_bits(pool_b[hist[:, 0], 0, :, hist[:, 1]], wl.dtype) if s else np.zeros((0, Hkv, d))
        Vh = _decode_bits(pool_b[hist[:, 0], 1, :, hist[:, 1]], wl.dtype) if s else np.zeros((0, Hkv, d))
        rows = qkv_b[t0:t0 + n]
        Kn = np.zeros((n, Hkv, d))
        Vn = np.zeros((n, Hkv, d))
        Q = np.zeros((n, Hq, d))
        for j in range(n):
            p = s + j
            for h in range(Hkv):
                kin = _decode_bits(rows[j, (Hq + h) * d:(Hq + h + 1) * d], wl.dtype).astype(np.float32)
                Kn[j, h] = _decode_bits(_np_rope32_store(kin, p, wl.rope_theta, wl.dtype), wl.dtype)
                Vn[j, h] = _decode_bits(rows[j, (Hq + Hkv + h) * d:(Hq + Hkv + h + 1) * d], wl.dtype)
            for h in range(Hq):
                Q[j, h] = _complex_rope(_decode_bits(rows[j, h * d:(h + 1) * d], wl.dtype), p, wl.rope_theta)
        K = np.concatenate([Kh, Kn])  # [L, Hkv, d]
        V = np.concatenate([Vh, Vn])
        mask = np.arange(L)[None, :] <= (s + np.arange(n))[:, None]  # [n, L]
        O = np.zeros((n, Hq, d))
        for h in range(Hq):
            S_ = (Q[:, h] @ K[:, h // g].T) / math.sqrt(d)
            S_ = np.where(mask, S_, -np.inf)
            S_ -= S_.max(axis=1, keepdims=True)
            P = np.exp(S_)
            P /= P.sum(axis=1, keepdims=True)
            O[:, h] = P @ V[:, h // g]
        outs.append(O)
        t0 += n
    return np.concatenate(outs) if outs else np.zeros((0, Hq, d))


@pytest.mark.parametrize("case", [
    ("tiny", None),
    ("mha_bf16", dict(seqs=[(0, 5), (64, 1), (63, 2), (1, 70)], hq=2, hkv=2, d=64, dtype="bf16")),
    ("gqa_d128", dict(seqs=[(129, 3), (0, 1), (200, 1)], hq=8, hkv=2, d=128, dtype="bf16")),
    ("gqa_fp16_big_theta", dict(seqs=[(5000, 2), (10, 40)], hq=4, hkv=1, d=64, dtype="fp16", theta=1e6)),
])
def test_attention_matches_brute_force(case):
    name, spec = case
    if spec is None:
        wl = W.make_workload("tiny_gqa_d64", 0)
    else:
        wl = W.make_custom(spec["seqs"], spec["hq"], spec["hkv"], spec["d"], dtype=spec["dtype"],
                           rope_theta=spec.get("theta", 1e4), seed=11, extra_blocks=3)
    qkv, pool = W.make_values(wl, "cpu")
    res = oracle.layer(wl, qkv, pool)
    bf = _brute_force(wl, qkv, pool)
    err = np.abs(res["out"] - bf).max()
    assert err <= 1e-12 * max(1.0, np.abs(bf).max()), err


def test_single_key_returns_its_value_and_zero_query_averages():
    wl = W.make_custom([(0, 1), (100, 1)], 4, 2, 64, dtype="fp16", seed=2)
    qkv, pool = W.make_values(wl, "cpu")
    res = oracle.layer(wl, qkv, pool)
    qkv_b = oracle._bits(qkv).reshape(2, -1)
    d = 64
    # sequence 0: one key (its own) -> output is exactly its V, for every head
    for h in range(4):
        v = _decode_bits(qkv_b[0, (4 + 2 + h // 2) * d:(4 + 2 + h // 2 + 1) * d], "fp16")
        np.testing.assert_array_equal(res["out"][0, h], v)
    # zero queries -> uniform weights -> mean of V over positions 0..p
    qkv2 = qkv.clone()
    qkv2[:, : 4 * d] = 0
    res2 = oracle.layer(wl, qkv2, pool)
    pool_after = res2["pool"]
    ids = wl.block_ids[1]
    for h in range(4):
        vs = np.stack([_decode_bits(pool_after[ids[u // 64], 1, h // 2, u % 64], "fp16") for u in range(101)])
        np.testing.assert_allclose(res2["out"][1, h], vs.mean(axis=0), rtol=0, atol=1e-13)


def test_gqa_equals_replicated_mha():
    gq = W.make_custom([(70, 3), (0, 9)], 4, 2, 64, dtype="bf16", seed=9, extra_blocks=1)
    qkv, pool = W.make_values(gq, "cpu")
    mha = W.make_custom([(70, 3), (0, 9)], 4, 4, 64, dtype="bf16", seed=9, extra_blocks=1)
    mha.block_ids = [b.copy() for b in gq.block_ids]
    d = 64
    qkv_m = torch.empty((gq.n_tokens, (4 + 8) * d), dtype=qkv.dtype)
    qkv_m[:, : 4 * d] = qkv[:, : 4 * d]
    for h in range(4):
        c = h // 2
        qkv_m[:, (4 + h) * d:(5 + h) * d] = qkv[:, (4 + c) * d:(5 + c) * d]
        qkv_m[:, (8 + h) * d:(9 + h) * d] = qkv[:, (6 + c) * d:(7 + c) * d]
    pool_m = pool[:, :, [0, 0, 1, 1]].contiguous()
    a = oracle.layer(gq, qkv, pool)["out"]
    b = oracle.layer(mha, qkv_m, pool_m)["out"]
    np.testing.assert_array_equal(a, b)


def test_chunked_prefill_equals_one_shot():
    one = W.make_custom([(0, 128)], 4, 2, 64, dtype="bf16", seed=21, extra_blocks=2)
    qkv, pool = W.make_values(one, "cpu")
    ref = oracle.layer(one, qkv, pool)
    pool_cur = pool
    outs = []
    start = 0
    for n in [37, 27, 64]:
        step = W.make_custom([(start, n)], 4, 2, 64, dtype="bf16", seed=21, extra_blocks=2)
        step.block_ids = [one.block_ids[0].copy()]
        step.num_blocks = one.num_blocks
        r = oracle.layer(step, qkv[start:start + n], pool_cur)
        pool_cur = torch.from_numpy(r["pool"].view(np.int16)).view(qkv.dtype)
        outs.append(r["out"])
        start += n
    np.testing.assert_array_equal(r["pool"], ref["pool"])
    np.testing.assert_allclose(np.concatenate(outs), ref["out"], rtol=0, atol=1e-12)


def test_thread_count_does_not_change_result():
    wl = W.make_custom([(300, 4), (0, 33)], 8, 2, 64, dtype="bf16", seed=5)
    qkv, pool = W.make_values(wl, "cpu")
    m = oracle.meta_build(wl)
    after, *_ = oracle.rope_append(wl, m, qkv, pool)
    a = oracle.attention(wl, m, qkv, after, n_threads=1)
    b = oracle.attention(wl, m, qkv, after, n_threads=5)
    np.testing.assert_array_equal(a, b)


def test_empty_batch():
    wl = W.make_custom([], 4, 2, 64)
    qkv, pool = W.make_values(wl, "cpu")
    res = oracle.layer(wl, qkv, pool)
    assert res["out"].shape == (0, 4, 64)
    np.testing.assert_array_equal(res["meta"]["cu_seqlens"], [0])


def test_workload_structure_matches_descriptions():
    """The generator's batches have the sizes the workload descriptions state."""
    c2 = W.make_workload("decode256_mha_d128")
    assert c2.n_seqs == 256 and c2.n_tokens == 256 and c2.seen.min() >= 128 and c2.seen.max() <= 4096
    assert c2.num_blocks == int(c2.blocks_needed().sum())
    c3 = W.make_workload("splitfuse2048_gqa_d128")
    assert c3.n_tokens == 2048 and c3.n_seqs == 515
    assert list(c3.seen[:3]) == [0, 1024, 3072] and c3.seen[3:].min() >= 64 and c3.seen[3:].max() <= 8192
    c4 = W.make_workload("chunked_prefill_2x8192")
    assert c4.n_tokens == 16384 and list(c4.seen) == [0, 8192]
    c5 = W.make_workload("max_ragged_8192")
    assert c5.n_seqs == 256 and c5.n_tokens == 8192
    assert c5.new[:16].min() >= 32 and c5.new[:16].max() <= 1024 and (c5.new[16:] == 1).all()
    assert c5.seen.min() >= 16 and c5.seen.max() <= 32768
    need = int(c5.blocks_needed().sum())
    assert c5.num_blocks == math.ceil(1.25 * need)
    all_ids = np.concatenate(c5.block_ids)
    assert len(np.unique(all_ids)) == len(all_ids) and all_ids.max() < c5.num_blocks
