"""Block ledger and SplitFuse planner on the CPU (no GPU).

The ledger (C ABI) is checked against a plain Python free-list model; the
planner's passes are checked for their invariants; and a multi-step run of
the oracle alone checks that a prompt processed in chunks across passes, with
blocks freed and reused in between, gives the one-shot result.
"""
import numpy as np
import pytest

import oracle
from ragged_blocked_kv_raggedbatch_gb300 import build as B
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W
from ragged_blocked_kv_raggedbatch_gb300.splitfuse import NativeSplitFusePlanner
from splitfuse_model import SplitFusePlanner


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return R.load()


def test_allocator_matches_free_list_model():
    rng = np.random.default_rng(0)
    order = rng.permutation(50)
    a = R.BlockAllocator(50, order)
    model = list(order[::-1])  # stack: last element is handed out next
    used = set()
    for step in range(400):
        if rng.random() < 0.55:
            n = int(rng.integers(0, 6))
            if n > len(model):
                with pytest.raises(R.DSError) as ei:
                    a.allocate(n)
                assert ei.value.status == R.DS_ERR_CAPACITY
                continue
            got = a.allocate(n)
            want = [model.pop() for _ in range(n)]
            assert list(got) == want
            used |= set(want)
        elif used:
            k = int(rng.integers(1, min(4, len(used)) + 1))
            ids = list(rng.choice(sorted(used), size=k, replace=False))
            a.free(ids)
            model += ids
            used -= set(ids)
        assert a.n_free == len(model)


def test_allocator_errors_change_nothing():
    a = R.BlockAllocator(8)
    ids = a.allocate(3)
    assert list(ids) == [0, 1, 2]
    for bad in ([5], [99], [-1], [int(ids[0]), int(ids[0])]):
        with pytest.raises(R.DSError) as ei:
            a.free(bad)
        assert ei.value.status == R.DS_ERR_BAD_BLOCK
        assert a.n_free == 5
    a.free(ids)
    with pytest.raises(R.DSError):
        a.free([int(ids[1])])  # double free
    assert a.n_free == 8
    with pytest.raises(R.DSError):
        R.BlockAllocator(4, [0, 1, 1, 2])  # not a permutation


def test_blocks_required_brute_force():
    for seen in range(0, 200, 7):
        for new in range(0, 140, 13):
            for owned in range(0, 6):
                need = -(-(seen + new) // 64)
                assert R.ds_kv_blocks_required(seen, new, owned, 64) == max(0, need - owned)


def _requests():
    # (uid, prompt, decode tokens, arrival pass)
    return [(0, 300, 5, 0), (1, 70, 70, 0), (2, 129, 3, 1), (3, 5, 8, 2), (4, 200, 2, 4), (5, 64, 4, 6)]


def run_plan(budget=128, max_seqs=8, num_blocks=40, seed=0):
    """The passes of a multi-step run: list of (pass, batch)."""
    order = np.random.default_rng(seed).permutation(num_blocks)
    alloc = R.BlockAllocator(num_blocks, order)
    plan = SplitFusePlanner(alloc, budget, max_seqs)
    reqs = _requests()
    passes, k = [], 0
    while k < 200:
        for uid, p, d, arr in reqs:
            if arr == k:
                plan.add(uid, p, d)
        if plan.idle and k > max(r[3] for r in reqs):
            break
        batch = plan.next_batch()
        passes.append((k, batch))
        plan.commit(batch)
        k += 1
    return passes, alloc, plan


def test_planner_invariants():
    passes, alloc, plan = run_plan()
    tot = {u: 0 for u, *_ in _requests()}
    for k, batch in passes:
        assert sum(n for _, _, n, _ in batch) <= 128 and len(batch) <= 8
        owned = {}
        for uid, seen, new, ids in batch:
            assert seen == tot[uid]
            assert len(ids) >= -(-(seen + new) // 64)
            owned[uid] = set(ids.tolist())
            tot[uid] += new
        all_ids = [i for s in owned.values() for i in s]
        assert len(all_ids) == len(set(all_ids))  # no block shared in a pass
    for uid, p, d, _ in _requests():
        assert tot[uid] == p + d
    assert alloc.n_free == 40 and plan.idle
    assert len(plan.freed) > 0


def _drive(plan, alloc, stream, max_passes=10000):
    """Feed (uid, prompt, decode, arrival pass) requests to a planner pass by
    pass; returns the list of (batch, flushed) per pass and the final free count."""
    log, k = [], 0
    last = max(r[3] for r in stream)
    while k < max_passes:
        for uid, p, d, arr in stream:
            if arr == k:
                plan.add(uid, p, d)
        if plan.idle and k > last:
            break
        batch = plan.next_batch()
        flushed = plan.commit(batch)
        log.append(([(u, s_, n, ids.tolist()) for u, s_, n, ids in batch], list(flushed)))
        k += 1
    return log, alloc.n_free


@pytest.mark.parametrize("case", range(6))
def test_native_planner_matches_python_planner(case):
    """ds_splitfuse_* makes the same passes as the Python planner, block for
    block, on random request streams; tight pools make requests wait."""
    rng = np.random.default_rng(100 + case)
    n_req = int(rng.integers(5, 60))
    budget = int(rng.choice([16, 64, 128, 512]))
    max_seqs = int(rng.choice([2, 4, 16, 64]))
    stream = [(int(1000 + i), int(rng.integers(1, 700)), int(rng.integers(0, 40)), int(rng.integers(0, 30)))
              for i in range(n_req)]
    need_max = max(-(-(p + d) // 64) for _, p, d, _ in stream)
    num_blocks = int(max(need_max, rng.integers(need_max, 4 * need_max + 8)))
    order = rng.permutation(num_blocks)
    a_py = R.BlockAllocator(num_blocks, order)
    a_nat = R.BlockAllocator(num_blocks, order)
    py = SplitFusePlanner(a_py, budget, max_seqs)
    nat = NativeSplitFusePlanner(a_nat, budget, max_seqs, max_requests=n_req, max_blocks_per_request=need_max)
    log_py, free_py = _drive(py, a_py, stream)
    log_nat, free_nat = _drive(nat, a_nat, stream)
    assert log_nat == log_py
    assert free_nat == free_py == num_blocks
    assert nat.idle and py.idle
    np.testing.assert_array_equal(a_nat.stack[: a_nat.n_free], a_py.stack[: a_py.n_free])


def test_native_planner_descriptors_pack_like_copies():
    """The planner's own ds_seq_desc[] (block lists in planner memory) packs to
    the same metadata as descriptors built from copied block lists."""
    rng = np.random.default_rng(7)
    stream = [(i, int(rng.integers(1, 400)), int(rng.integers(0, 20)), 0) for i in range(12)]
    alloc = R.BlockAllocator(200, rng.permutation(200))
    nat = NativeSplitFusePlanner(alloc, 256, 8, max_requests=12, max_blocks_per_request=8)
    for uid, p_, d, _ in stream:
        nat.add(uid, p_, d)
    params = R.make_params(4, 2, 64)
    fake_dev = 1 << 40
    for _ in range(30):
        if nat.idle:
            break
        n = nat.plan()
        copies = [(nat.arr[i].seen_tokens, nat.arr[i].new_tokens,
                   np.ctypeslib.as_array(nat.arr[i].block_ids, shape=(nat.arr[i].n_blocks,)).copy())
                  for i in range(n)]
        metas = []
        for descs in (nat, R.SeqDescs([c[0] for c in copies], [c[1] for c in copies], [c[2] for c in copies])):
            dev, stg = R.ds_meta_buffer_sizes(8, 256, 64, params)
            stage = np.zeros(stg // 4 + 4, np.int32)
            meta = R.ds_ragged_meta()
            meta.device_buf, meta.device_bytes = fake_dev, dev
            meta.host_staging, meta.staging_bytes = stage.ctypes.data, stg
            meta.max_seqs, meta.max_tokens, meta.max_blocks = 8, 256, 64
            assert R.ds_ragged_meta_pack(descs, params, 200, meta) == R.DS_OK
            metas.append(stage[: meta.used_bytes // 4].copy())
        np.testing.assert_array_equal(metas[0], metas[1])
        nat.commit()


def test_native_planner_errors():
    alloc = R.BlockAllocator(20)
    nat = NativeSplitFusePlanner(alloc, 64, 4, max_requests=2, max_blocks_per_request=3)
    lib = R.load()
    assert lib.ds_splitfuse_add(R._ref(nat.p), 1, 0, 5) == R.DS_ERR_INVALID_ARG      # empty prompt
    assert lib.ds_splitfuse_add(R._ref(nat.p), 1, 150, 50) == R.DS_ERR_CAPACITY      # 4 blocks > 3
    nat.add(1, 100, 10)
    assert lib.ds_splitfuse_add(R._ref(nat.p), 1, 10, 1) == R.DS_ERR_INVALID_ARG     # uid active
    nat.add(2, 10, 1)
    assert lib.ds_splitfuse_add(R._ref(nat.p), 3, 10, 1) == R.DS_ERR_CAPACITY        # 2 requests max
    nat.plan()
    n = np.zeros(1, np.int32)
    descs = (R.ds_seq_desc * 4)()
    uids = np.zeros(4, np.int32)
    assert lib.ds_splitfuse_next(R._ref(nat.p), R._ref(alloc.a), R._ref(descs), uids.ctypes.data,
                                 n.ctypes.data) == R.DS_ERR_INVALID_ARG            # not committed
    nat.commit()
    flushed = np.zeros(2, np.int32)
    assert lib.ds_splitfuse_commit(R._ref(nat.p), R._ref(alloc.a), flushed.ctypes.data,
                                   n.ctypes.data) == R.DS_ERR_INVALID_ARG          # nothing planned
    small = np.zeros(4, np.uint64)
    p2 = R.ds_splitfuse()
    assert lib.ds_splitfuse_init(R._ref(p2), small.ctypes.data, small.nbytes, 2, 3, 64, 4, 64) == R.DS_ERR_WORKSPACE


def _fields(heads=(4, 2), d=64, dtype="bf16"):
    return dict(n_q_heads=heads[0], n_kv_heads=heads[1], head_dim=d, block_size=64, dtype=dtype,
                rope_theta=1e4, value_std=1.0)


def test_oracle_multistep_chunked_equals_one_shot():
    """Run every pass through the oracle on one evolving pool; each request's
    prompt rows equal a one-shot prefill of that prompt (same rows of qkv) on
    its own, bit for bit."""
    import torch
    passes, _, _ = run_plan(num_blocks=40)
    f = _fields()
    width = (f["n_q_heads"] + 2 * f["n_kv_heads"]) * f["head_dim"]
    gen = torch.Generator().manual_seed(5)
    pool = torch.randn((40, 2, f["n_kv_heads"], 64, f["head_dim"]), generator=gen).to(torch.bfloat16)
    pool_b = oracle._bits(pool)
    rows = {}  # uid -> list of (position, qkv row, output row)
    for k, batch in passes:
        if not batch:
            continue
        wl = W.RaggedWorkload(name="pass%d" % k, seen=np.array([b[1] for b in batch], np.int32),
                              new=np.array([b[2] for b in batch], np.int32),
                              block_ids=[b[3] for b in batch], num_blocks=40, **f)
        qkv = torch.randn((wl.n_tokens, width), generator=gen).to(torch.bfloat16)
        res = oracle.layer(wl, qkv, pool_b)
        pool_b = res["pool"]
        t = 0
        for uid, seen, new, _ in batch:
            for j in range(new):
                rows.setdefault(uid, []).append((seen + j, qkv[t], res["out"][t]))
                t += 1
    for uid, p, d, _ in _requests():
        got = rows[uid]
        assert [r[0] for r in got] == list(range(p + d))
        # one-shot prefill of the prompt alone, from fresh history-free blocks
        one = W.RaggedWorkload(name="one", seen=np.array([0], np.int32), new=np.array([p], np.int32),
                               block_ids=[np.arange(-(-p // 64), dtype=np.int32)], num_blocks=40, **f)
        q1 = torch.stack([r[1] for r in got[:p]])
        ref = oracle.layer(one, q1, pool)
        np.testing.assert_array_equal(np.stack([r[2] for r in got[:p]]), ref["out"])
