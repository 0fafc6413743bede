"""bench.py's accounting on CPU: the algorithmic flops and bytes of a step
(causal pairs only; each byte read or written once), the config object both
arms print, and the source hash that keys the ncu traffic."""
import argparse
import importlib.util
import os

import numpy as np

from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def _brute(wl):
    """The same quantities counted token by token and key by key."""
    e, Hq, Hkv, d = 2, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    flops = bytes_ = 0
    for s, n in zip(wl.seen.tolist(), wl.new.tolist()):
        for j in range(n):
            keys = s + j + 1                              # causal: history plus new tokens up to itself
            flops += Hq * keys * (2 * d + 2 * d)          # q.k and p.v, a multiply and an add each
            bytes_ += e * (Hq + 2 * Hkv) * d              # the token's q, k, v read
            bytes_ += e * 2 * Hkv * d                     # its k, v written to the pool
            bytes_ += e * Hq * d                          # its output written
        bytes_ += e * s * 2 * Hkv * d                     # the history read once
        bytes_ += 4 * ((s + n + 63) // 64)                # its block ids
    return flops, bytes_


def test_algorithmic_counts_match_token_by_token():
    for wl in (W.make_workload("tiny_gqa_d64"),
               W.make_custom([(0, 70), (130, 1), (64, 9), (1000, 1)], 8, 2, 128, dtype="bf16")):
        alg = bench.algorithmic(wl)
        flops, bytes_ = _brute(wl)
        assert alg["flops"] == flops
        assert alg["bytes"] == bytes_


def test_both_arms_share_the_config():
    wl = W.make_workload("tiny_gqa_d64")
    args = argparse.Namespace(path="split")
    c1 = bench.run_config(wl, args, 1)
    c2 = bench.run_config(wl, args, 1)
    assert c1 == c2 and c1["workload"] == wl.name and c1["new_tokens"] == wl.n_tokens
    assert bench.run_config(wl, args, 2)["parallelism"] == "replicas"
    # a step smaller than twice L2 is timed with L2 flushed in between
    assert "flushed" in c1["l2"]
    big = W.make_workload("decode256_mha_d128")
    assert "larger than L2" in bench.run_config(big, args, 1)["l2"]


def test_source_hash_ignores_comments_and_blank_space(tmp_path, monkeypatch):
    csrc = tmp_path / "ragged_blocked_kv_raggedbatch_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("int f(int x) {\n  return x + 1;  // one\n}\n/* note */\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench._src_hash(["k.cu"])
    (csrc / "k.cu").write_text("/* a longer\n   note */\nint f(int x) {   return x + 1; // two\n}\n")
    assert bench._src_hash(["k.cu"]) == h0
    (csrc / "k.cu").write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench._src_hash(["k.cu"]) != h0


def test_spread_order_is_a_permutation_whose_prefixes_track_the_mean():
    vals = W.make_workload("decode256_mha_d128").seen.astype(np.int64)
    order = bench._spread_order(vals, 0)
    assert sorted(order.tolist()) == list(range(len(vals)))
    # the median first; every prefix of 8 or more within 10% of the batch mean
    assert vals[order[0]] == np.sort(vals)[len(vals) // 2]
    for k in (8, 16, 32, 64):
        assert abs(vals[order[:k]].mean() - vals.mean()) <= 0.1 * vals.mean(), k
    odd = np.array([5, 1, 9, 3, 7], np.int64)
    assert sorted(bench._spread_order(odd, 1).tolist()) == list(range(5))


def test_row_work_counts_keys_attended():
    seen, new = [0, 90, 130, 7], [37, 1, 64, 1]
    brute = sum(s + j + 1 for s, n in zip(seen, new) for j in range(n))
    assert bench._row_work(seen, new) == brute
