#!/usr/bin/env python3
"""Benchmark of one ragged blocked-KV attention layer forward (one step =
rotary embedding + KV append + blocked attention over one synthetic ragged
batch), printed as one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on the same workload

value     new tokens/s per layer, inputs resident in HBM, CUDA events on the
          launching stream, max over ranks.
e2e       same metric through the C ABI from pinned HOST buffers: each step
          uploads the step's qkv rows, builds + uploads the batch metadata
          from host descriptors, runs the layer and reads the output back.
roofline  the attention call (the dominant launches) timed live with CUDA
          events: algorithmic bytes (or flops) per launch / mean duration.
Multi-GPU: each rank runs its own copy of the batch (sequences are
independent; no collective on the data path), weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from ragged_blocked_kv_raggedbatch_gb300 import replicas  # noqa: E402
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "decode256_mha_d128"
METRIC = "ragged attn new tokens/s per layer"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# workloads whose oracle is also timed on one thread (the small and the
# HBM-bound ones; the oracle's per-row cost is the same on any thread count)
SINGLE_THREAD_ORACLE = ("tiny_gqa_d64", "decode256_mha_d128", "splitfuse2048_gqa_d128")

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# the dominant kernel from an ncu capture, keyed by workload; reported only
# while the hash of the kernel's source files (comments and blank space
# removed) still matches the capture.
NCU_TRAFFIC = {
    # decode_split_kernel on the first 64 sequences of the decode-only batch:
    # 2.290075 GB read + 6.03 MB written for 2.2576 GB algorithmic (x1.0171);
    # scaled to the full batch by its algorithmic bytes (the KV read dominates
    # and grows in proportion).
    "decode256_mha_d128": {"bytes": 9.3774e9, "files": ["decode.cu", "common.cuh", "tc.cuh"],
                           "src": "eb2b8af3571b7705"},
    # prefill_tc_kernel on the whole chunked-prefill workload (< 1 GB on the
    # device, captured at full size): 461.19 MB read + 231.07 MB written for
    # 637.5 MB algorithmic (x1.086).
    "chunked_prefill_2x8192": {"bytes": 6.92260e8, "files": ["prefill_tc.cu", "common.cuh", "tc.cuh"],
                               "src": "60e9f76d72cc4bee"},
}


def _src_hash(files) -> str:
    """Hash of the kernel's source files with comments and blank space
    removed, so that editing a comment does not invalidate a capture."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ragged_blocked_kv_raggedbatch_gb300", "csrc")
    for f in files:
        text = open(os.path.join(csrc, f), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps") or d.get("hbm")
            tf = d.get("bf16_tflops") or d.get("bf16_dense_tflops")
            tfs = d.get("bf16_tflops_sustained") or tf
            if hbm and tf:
                return {"hbm_gbs": float(hbm), "bf16_tflops": float(tf),
                        "bf16_tflops_sustained": float(tfs), "source": "measured"}
        except Exception:
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


def algorithmic(wl):
    """Algorithmic work of one step (causal pairs only; bytes each read or
    written once): dict of flops and bytes, total and per call."""
    e = 2
    Hq, Hkv, d = wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    s = wl.seen.astype(np.float64)
    n = wl.new.astype(np.float64)
    N = float(n.sum())
    nb = wl.blocks_needed().astype(np.float64)
    flops = 4.0 * d * Hq * float((n * s + n * (n + 1) / 2).sum())
    step_bytes = e * (N * (Hq + 2 * Hkv) * d + N * 2 * Hkv * d + float(s.sum()) * 2 * Hkv * d
                      + N * Hq * d) + 4 * float(nb.sum())
    append_bytes = e * (2 * N * 2 * Hkv * d)
    attn_bytes = e * (N * Hq * d + float((s + n).sum()) * 2 * Hkv * d + N * Hq * d) + 4 * float(nb.sum())
    pre = wl.new > 1
    pre_flops = 4.0 * d * Hq * float((n[pre] * s[pre] + n[pre] * (n[pre] + 1) / 2).sum())
    return dict(flops=flops, bytes=step_bytes, append_bytes=append_bytes, attn_bytes=attn_bytes,
                attn_flops=flops, prefill_flops=pre_flops,
                kv_history_bytes=e * float(s.sum()) * 2 * Hkv * d)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- CPU oracle legs

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.split(":")[0].strip().lower() in ("model name", "cpu model"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def _spread_order(values: np.ndarray, seed: int) -> np.ndarray:
    """Indices of `values` in an order whose every prefix spreads over their
    range: sorted by value (ties shuffled), then visited at quantile midpoints
    level by level -- 1/2; 1/4, 3/4; 3/8, 5/8, 1/8, 7/8; ... -- each level's
    points taken inside-out in symmetric pairs, so that a short prefix already
    has about the mean of the whole."""
    n = len(values)
    rng = np.random.default_rng(seed)
    by_val = np.lexsort((rng.permutation(n), values))
    seen, order = np.zeros(n, bool), []
    levels = int(np.ceil(np.log2(max(n, 2)))) + 2
    for m in range(1, levels + 1):
        half = 1 << (m - 1)
        pts = []
        for j in reversed(range((half + 1) // 2)):
            pts.append((2 * j + 1) / float(1 << m))
            if half - 1 - j != j:
                pts.append((2 * (half - 1 - j) + 1) / float(1 << m))
        for r in pts:
            i = min(n - 1, int(r * n))
            if not seen[i]:
                seen[i] = True
                order.append(i)
    order += [i for i in range(n) if not seen[i]]
    return by_val[np.array(order, np.int64)]


def _row_work(seen, new) -> float:
    """Keys attended, summed over a batch's rows (the oracle's cost grows with it)."""
    s = np.asarray(seen, np.float64)
    n = np.asarray(new, np.float64)
    return float((n * s + n * (n + 1) / 2).sum())


def _oracle_sample(wl, n_rows_target: int, seed: int = 0, max_pool_bytes: float = 256e6):
    """A bounded sample of the workload for the oracle: sequences taken in an
    order spread over the batch's lengths (_spread_order); a prefill chunk
    contributes a random run of up to the remaining row budget (as if it had
    been split there: seen += offset).  Returned as a batch of its own over a
    compact pool (fresh values of the same distribution, CPU generator), capped
    at ~max_pool_bytes of KV."""
    rng = np.random.default_rng(seed)
    order = _spread_order(wl.seen.astype(np.int64) + wl.new, seed)
    block_bytes = 2 * wl.n_kv_heads * 64 * wl.head_dim * 2
    seqs, rows, blocks = [], 0, 0
    for i in order:
        s, n = int(wl.seen[i]), int(wl.new[i])
        take = min(n, max(1, n_rows_target - rows))
        j0 = int(rng.integers(0, n - take + 1))
        nb = -(-(s + j0 + take) // 64)
        if seqs and (blocks + nb) * block_bytes > max_pool_bytes:
            break
        seqs.append((s + j0, take))
        rows += take
        blocks += nb
        if rows >= n_rows_target:
            break
    return W.make_custom(seqs, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, dtype=wl.dtype,
                         rope_theta=wl.rope_theta, value_std=wl.value_std, seed=seed,
                         name=wl.name + "_oracle_sample")


def _grow_sample(wl, seed: int, threads: int, pass_s: float):
    """The smallest sample (_oracle_sample) whose one oracle pass takes about
    pass_s seconds: start at a few rows and grow geometrically.  Returns
    (sample, qkv, pool, seconds of its last pass)."""
    import oracle
    rows, last_n = 4, -1
    while True:
        sub = _oracle_sample(wl, rows, seed)
        qkv, pool = W.make_values(sub, "cpu", seed=seed)
        t0 = time.perf_counter()
        oracle.layer(sub, qkv, pool, n_threads=threads)
        dt = time.perf_counter() - t0
        if dt >= pass_s or sub.n_tokens >= wl.n_tokens or sub.n_tokens == last_n:
            return sub, qkv, pool, dt
        last_n = sub.n_tokens
        rows = min(wl.n_tokens, int(rows * min(8.0, max(2.0, 0.8 * pass_s / max(dt, 1e-4)))))


def time_oracle(wl, seconds: float = 10.0, seed: int = 0, threads: int = 0):
    """The oracle (metadata, append, attention in fp64) on the host cores over a
    bounded sample of the workload, re-run until about `seconds` of work, and
    scaled to the whole batch by the keys its rows attend: tokens/s of the
    batch = N / (sample time x batch work / sample work).  Returns a dict."""
    import oracle
    threads = threads or oracle.default_threads()
    sub, qkv, pool, _ = _grow_sample(wl, seed, threads, seconds / 4)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.layer(sub, qkv, pool, n_threads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    batch_work = _row_work(wl.seen, wl.new)
    sub_work = _row_work(sub.seen, sub.new)
    batch_s = dt / reps * batch_work / sub_work
    return {"value": wl.n_tokens / batch_s, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "seconds": dt, "batch_seconds_est": batch_s,
            "sample": ("%d rows (%d sequences, %d KV-history tokens, mean history %.0f vs the batch's %.0f) "
                       "sampled from %s in length-spread order, fresh values of the same distribution; "
                       "fp64 oracle metadata+append+attention repeated %d times (%.1f s); scaled to the "
                       "whole batch by keys attended (batch/sample = %.1f)"
                       % (sub.n_tokens, sub.n_seqs, int(sub.seen.sum()), float(sub.seen.mean()),
                          float(wl.seen.mean()), wl.name, reps, dt, batch_work / sub_work))}


def _l2_note(wl) -> str:
    step_bytes = algorithmic(wl)["bytes"]
    return ("inputs larger than L2 (%.2f GB per step)" % (step_bytes / 1e9) if step_bytes >= 2 * L2_BYTES
            else "L2 flushed between timed steps (512 MB write, untimed)")


def run_config(wl, args, world: int) -> dict:
    """The workload's config object, the same on both arms' lines."""
    return {"workload": wl.name, "n_seqs": wl.n_seqs, "new_tokens": wl.n_tokens,
            "kv_history_tokens": int(wl.seen.sum()), "n_q_heads": wl.n_q_heads,
            "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim, "block_size": 64,
            "rope_theta": wl.rope_theta, "seed": wl.seed, "l2": _l2_note(wl),
            "path": args.path, "parallelism": "replicas" if world > 1 else "single"}


def reference_arm(args, wl):
    ws, rank, _ = replicas.env()
    if rank != 0:
        return 0
    import oracle
    threads = oracle.default_threads()
    # size each step so that warmup + steps take about two minutes
    budget_s = 120.0
    steps = args.steps + args.warmup
    first = _grow_sample(wl, 0, threads, budget_s / steps)[0]
    rows = first.n_tokens
    batch_work = _row_work(wl.seen, wl.new)
    samples = []
    for k in range(min(steps, 4)):
        sub = _oracle_sample(wl, rows, k)
        samples.append((sub,) + tuple(W.make_values(sub, "cpu", seed=k)))
    batch_s = []
    for k in range(steps):
        sub, qkv, pool = samples[k % len(samples)]
        t0 = time.perf_counter()
        oracle.layer(sub, qkv, pool, n_threads=threads)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            # this step's sample time, scaled to the whole batch by keys attended
            batch_s.append(dt * batch_work / _row_work(sub.seen, sub.new))
    total = float(sum(batch_s))
    value = wl.n_tokens * len(batch_s) / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / max(1, len(batch_s)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": run_config(wl, args, ws),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "cpu_model": cpu_model(), "nproc": os.cpu_count(),
                         "sample": "about %d rows per step (%d in the first sample) drawn from %s in "
                                   "length-spread order (fresh values, same distribution; 4 samples "
                                   "reused); each step's time scaled to the whole batch by keys attended"
                                   % (rows, samples[0][0].n_tokens, wl.name)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm

def _roofline(r_bytes, r_flops, mean_s, peaks, sustained=False):
    """The roofline object of a launch group: the slower of its bytes over the
    HBM peak and its flops over the bf16 tensor peak decides the bound."""
    tf_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    if r_bytes / (peaks["hbm_gbs"] * 1e9) >= r_flops / (tf_peak * 1e12):
        achieved = r_bytes / mean_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "frac_vs_8tbs": achieved / 8000.0}
        if roof["frac"] > 1.0:
            roof["note"] = ("achieved above the measured copy peak: that peak is a read+write copy, "
                            "this launch group mostly reads")
    else:
        achieved = r_flops / mean_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                "frac": achieved / tf_peak}
        if not sustained:
            roof["frac_of_sustained"] = achieved / peaks["bf16_tflops_sustained"]
    return roof


def device_measure(wl, args, grp, local, K, warmup, keep=False, flushed_loop=True):
    """K timed steps of one workload, inputs resident in HBM, CUDA events on
    the launching stream around each step and around its attention call; the
    SM clocks sampled meanwhile.  Returns a dict (and, with keep, the live
    objects the end-to-end leg reuses)."""
    import torch
    from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R

    ws, rank, _ = replicas.env()
    dev = "cuda"
    stream = torch.cuda.Stream()
    nb_total = int(wl.blocks_needed().sum())
    alg = algorithmic(wl)
    with torch.cuda.stream(stream):
        qkv, pool = W.make_values(wl, dev, seed=replicas.rank_seed(wl.seed, rank))
        params = R.params_for(wl)
        layer = R.RaggedLayer(params, wl.n_seqs, wl.n_tokens, nb_total, wl.max_len(), stream=stream)
        descs = R.SeqDescs.of(wl)
        t0 = time.perf_counter()
        layer.build(descs, wl.num_blocks)
        stream.synchronize()
        meta_build_us = 1e6 * (time.perf_counter() - t0)
        out = torch.empty((wl.n_tokens, wl.n_q_heads * wl.head_dim), dtype=qkv.dtype, device=dev)
    m = layer.meta
    fused = args.path == "fused"
    if fused:
        # prefill tiles (their K/V append inside), decode rows (append + split-K,
        # the merge inside on the tensor-core path, beside a prefill grid, or
        # while the CUDA-core kernel's grid is at most two waves)
        sms = torch.cuda.get_device_properties(local).multi_processor_count
        tc_decode = wl.head_dim == 128 and wl.n_q_heads // wl.n_kv_heads >= 2
        merge_inside = tc_decode or m.n_prefill_tiles > 0 or m.n_decode_items * wl.n_kv_heads <= 6 * sms
        launches_per_step = (m.n_prefill_tiles > 0) + (m.n_decode_items > 0) + \
            (not merge_inside and m.n_decode_items > m.n_decode_seqs)
    else:
        launches_per_step = 1 + (m.n_prefill_tiles > 0) + (m.n_decode_items > 0) + \
            (m.n_decode_items > m.n_decode_seqs)

    def run_step(b_event=None):
        if fused:
            if b_event is not None:
                b_event.record(stream)
            layer.fused(qkv, pool, out)
        else:
            layer.append(qkv, pool)
            if b_event is not None:
                b_event.record(stream)
            layer.attention(qkv, pool, out)

    flush = None
    if alg["bytes"] < 2 * L2_BYTES:
        flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run_step()
            if flush is not None:
                flush.zero_()
    stream.synchronize()
    grp.barrier()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for k in range(K):
                a, b, c = ev[k]
                a.record(stream)
                run_step(b)
                c.record(stream)
                if flush is not None:
                    flush.zero_()
        stream.synchronize()
    clocks = clk.summary()
    # the same steps with L2 flushed before each one (a 512 MB write, untimed),
    # next to the main loop's (which flushes only when a step's bytes are
    # below twice L2)
    flushed = None
    if flush is None and flushed_loop:
        fl = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
        K2 = max(3, min(K, 50))
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True)) for _ in range(K2)]
        with torch.cuda.stream(stream):
            for k in range(K2):
                fl.zero_()
                a, b, c = ev2[k]
                a.record(stream)
                run_step(b)
                c.record(stream)
        stream.synchronize()
        flushed = {"ms_per_step": float(np.mean([a.elapsed_time(c) for a, b, c in ev2])),
                   "attention_ms": float(np.mean([b.elapsed_time(c) for a, b, c in ev2])), "steps": K2}
        del fl
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    attn_ms = [b.elapsed_time(c) for a, b, c in ev]
    app_ms = [a.elapsed_time(b) for a, b, c in ev]
    total_ms = grp.max(float(sum(step_ms)), dev)
    torch.cuda.synchronize()
    peaks = load_peaks()
    ms_per_step = total_ms / K
    # roofline of the attention call (the dominant launches); the fused call
    # also does the append, so it is held to the whole step's work.  A loop
    # of a second or more runs at the sustained tensor clock.
    attn_mean_s = float(np.mean(attn_ms)) / 1e3
    r_bytes = alg["bytes"] if fused else alg["attn_bytes"]
    r_flops = alg["flops"] if fused else alg["attn_flops"]
    long_loop = total_ms >= 1000.0
    roof = _roofline(r_bytes, r_flops, attn_mean_s, peaks, sustained=long_loop)
    rec = NCU_TRAFFIC.get(wl.name + (":fused" if fused else ""))
    roof["traffic"] = rec["bytes"] if rec and rec.get("src") == _src_hash(rec["files"]) else None
    parts = ("decode split-K + combine" if m.n_prefill_tiles == 0 else
             "prefill tiles" if m.n_decode_items == 0 else "prefill tiles + decode split-K + combine")
    roof["kernel"] = ("ds_fused_append_attention launches (%s, append inside)" % parts if fused
                      else "ds_blocked_attention launches (%s)" % parts)
    roof["peak_source"] = peaks["source"]
    roof["algorithmic_bytes"] = r_bytes
    roof["algorithmic_flops"] = r_flops
    roof["mean_ms"] = attn_mean_s * 1e3
    # whole-step roofline: T_roof = max(bytes / HBM peak, flops / tensor peak)
    tf = peaks["bf16_tflops_sustained" if long_loop else "bf16_tflops"]
    t_roof = max(alg["bytes"] / (peaks["hbm_gbs"] * 1e9), alg["flops"] / (tf * 1e12))
    res = {
        "value": ws * wl.n_tokens * K / (total_ms / 1e3), "ms_per_step": ms_per_step, "steps": K,
        "roofline": roof, "step_roofline_frac": t_roof / (ms_per_step / 1e3),
        "t_roof_ms": t_roof * 1e3, "clocks": clocks,
        "append_ms": float(np.mean(app_ms)), "attention_ms": float(np.mean(attn_ms)),
        "decode_kv_gbps": alg["kv_history_bytes"] / attn_mean_s / 1e9,
        "algorithmic": {"flops": alg["flops"], "bytes": alg["bytes"]},
        "meta_build_us": meta_build_us, "l2_flushed": flushed, "l2": _l2_note(wl),
        "launches_per_step": int(launches_per_step),
        "workspace_bytes": int(m.n_decode_items * wl.n_q_heads * (wl.head_dim + 2) * 4),
        # bytes the implementation moves: the append (K, V read and written),
        # the attention call (Q, every KV row incl. the new ones, O, block ids)
        # and the split-K partials (written, then read by the merge)
        "implemented_bytes": int(alg["append_bytes"] + alg["attn_bytes"] +
                                 2 * m.n_decode_items * wl.n_q_heads * (wl.head_dim + 2) * 4),
    }
    if keep:
        res["_live"] = dict(stream=stream, qkv=qkv, pool=pool, out=out, layer=layer, params=params,
                            descs=descs, nb_total=nb_total, fused=fused)
    else:
        del qkv, pool, out, layer, flush
        torch.cuda.empty_cache()
    return res


def e2e_measure(wl, args, grp, live, K):
    """The metric end to end through the C ABI: every step copies its qkv rows
    in from pinned host memory, uploads its metadata, runs the layer and copies
    its output rows back to pinned host memory.  Steps are pipelined the way a
    serving loop would run them: copy-in, compute and copy-out on three streams
    over two device buffer sets (and two metadata objects, so a pinned staging
    buffer is never rewritten while its upload may still be pending), ordered
    by events."""
    import torch
    from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R

    ws, _, _ = replicas.env()
    dev = "cuda"
    stream, qkv, pool, out = live["stream"], live["qkv"], live["pool"], live["out"]
    layer, params, descs, fused = live["layer"], live["params"], live["descs"], live["fused"]
    with torch.cuda.stream(stream):
        qkv_host = qkv.cpu().pin_memory()
        out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        qkv_d = [qkv, torch.empty_like(qkv)]
        out_d = [out, torch.empty_like(out)]
        layers = [layer, R.RaggedLayer(params, wl.n_seqs, wl.n_tokens, live["nb_total"], wl.max_len(),
                                       stream=stream)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    ev_meta = [None, None]

    def issue(k):
        b = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_done[b])  # step k-2 no longer reads qkv_d[b]
            qkv_d[b].copy_(qkv_host, non_blocking=True)
            ev_in[b].record(s_in)
        if ev_meta[b] is not None:
            ev_meta[b].synchronize()  # step k-2's metadata upload left the staging buffer
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[b])
            if k >= 2:
                stream.wait_event(ev_out[b])  # step k-2's output is on the host
            layers[b].build(descs, wl.num_blocks)
            ev_meta[b] = torch.cuda.Event()
            ev_meta[b].record(stream)
            if fused:
                layers[b].fused(qkv_d[b], pool, out_d[b])
            else:
                layers[b].append(qkv_d[b], pool)
                layers[b].attention(qkv_d[b], pool, out_d[b])
            ev_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            out_host[b].copy_(out_d[b], non_blocking=True)
            ev_out[b].record(s_out)

    E = max(3, min(K, 200))
    for k in range(4):  # warm-up of the pipeline (both buffer sets)
        issue(k)
    torch.cuda.synchronize()
    grp.barrier()
    t0 = time.perf_counter()
    for k in range(E):
        issue(k)
    torch.cuda.synchronize()  # every step's output is on the host
    e2e_s = grp.max(time.perf_counter() - t0, dev)
    return {"value": ws * wl.n_tokens * E / e2e_s, "unit": "tokens/s",
            "h2d_bytes_per_step": int(qkv.numel() * qkv.element_size() + layer.meta.used_bytes),
            "d2h_bytes_per_step": int(out.numel() * out.element_size()), "steps": E,
            "pipelined": "copy-in / compute / copy-out streams, 2 buffer sets"}


def _per_workload_entry(wl, r) -> dict:
    keep = ("value", "ms_per_step", "steps", "step_roofline_frac", "t_roof_ms", "clocks",
            "attention_ms", "append_ms", "launches_per_step", "l2", "l2_flushed")
    d = {k: r[k] for k in keep}
    d["unit"] = "tokens/s"
    d["roofline"] = {k: r["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac")
                     if k in r["roofline"]}
    for k in ("frac_of_sustained", "frac_vs_8tbs"):
        if k in r["roofline"]:
            d["roofline"][k] = r["roofline"][k]
    d["dtype"] = wl.dtype
    d["seed"] = wl.seed
    return d


def gpu_arm(args, wl):
    import torch

    ws, rank, local = replicas.env()
    torch.cuda.set_device(local)
    grp = replicas.Group("nccl")
    K = args.steps
    head = device_measure(wl, args, grp, local, K, args.warmup, keep=True)
    e2e = None if args.no_e2e else e2e_measure(wl, args, grp, head["_live"], K)
    del head["_live"]
    torch.cuda.empty_cache()

    # every named workload (seed 0) on the same clock, as the headline's
    # neighbours: the headline workload's own entry is its measurement above
    per_workload = None
    if not args.no_per_workload:
        per_workload = {}
        for name in sorted(W.WORKLOADS):
            if name == wl.name and wl.seed == 0:
                per_workload[name] = _per_workload_entry(wl, head)
                continue
            w2 = W.make_workload(name, 0)
            per_workload[name] = _per_workload_entry(
                w2, device_measure(w2, args, grp, local, K, args.warmup, flushed_loop=False))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = time_oracle(wl, seconds=args.cpu_seconds)
        cpu["cpu_model"] = cpu_model()
        cpu["nproc"] = os.cpu_count()
        # the oracle on every workload: all cores, and one thread where a
        # single thread finishes a sample in seconds
        if per_workload is not None:
            per = {}
            for name in sorted(W.WORKLOADS):
                w2 = wl if (name == wl.name and wl.seed == 0) else W.make_workload(name, 0)
                allc = cpu if w2 is wl else time_oracle(w2, seconds=args.cpu_seconds / 3)
                entry = {"all_cores": {"value": allc["value"], "cores": allc["cores"],
                                       "batch_seconds_est": allc["batch_seconds_est"]}}
                if name in SINGLE_THREAD_ORACLE:
                    one = time_oracle(w2, seconds=args.cpu_seconds / 3, threads=1)
                    entry["single_thread"] = {"value": one["value"], "cores": 1,
                                              "batch_seconds_est": one["batch_seconds_est"]}
                per[name] = entry
            cpu["per_workload"] = per

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": run_config(wl, args, ws),
            "roofline": head["roofline"],
            "step_roofline_frac": head["step_roofline_frac"],
            "decode_kv_gbps": head["decode_kv_gbps"],
            "append_ms": head["append_ms"], "attention_ms": head["attention_ms"],
            "algorithmic": head["algorithmic"],
            "hbm_frac_vs_8tbs": head["roofline"].get("frac_vs_8tbs"),
            "meta_build_us": head["meta_build_us"],
            "l2_flushed": head["l2_flushed"],
            "workspace_bytes": head["workspace_bytes"],
            "implemented_bytes": head["implemented_bytes"],
            "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": head["launches_per_step"] * K,
            "clocks": head["clocks"],
            "per_workload": per_workload,
        }
        print(json.dumps(line), flush=True)
    grp.close()
    return 0


# -------------------------------------------------------- component lines

def _line(metric, value, unit, config, **extra):
    d = {"metric": metric, "value": value, "unit": unit, "n_gpus": 1, "higher_is_better": True,
         "data": "synthetic", "config": config}
    d.update(extra)
    print(json.dumps(d), flush=True)


def component_offload(args, wl):
    """BlockedKVCache offload + restore of scattered blocks between the pool
    and page-locked host memory (one kernel each way, per 1000 blocks)."""
    import torch
    from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
    params = R.params_for(wl)
    nblk = min(wl.num_blocks, 4096)
    dt = W.torch_dtype(wl)
    pool = torch.randn((nblk, 2, wl.n_kv_heads, 64, wl.head_dim), device="cuda").to(dt)
    bb = R.ds_kv_block_bytes(params)
    n = min(nblk, max(1, int(2e9 // bb)))
    ids = np.random.default_rng(0).permutation(nblk)[:n].astype(np.int32)
    host = torch.empty((n, bb // 2), dtype=dt).pin_memory()
    pk = R.ds_kv_pool(pool.data_ptr(), nblk)
    st = torch.cuda.current_stream()
    res = {}
    for name, fn in (("offload", R.ds_kv_offload), ("restore", R.ds_kv_restore)):
        for _ in range(args.warmup):
            fn(params, pk, ids, host)
        st.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(args.steps):
            fn(params, pk, ids, host)
        b.record(st)
        st.synchronize()
        res[name] = n * bb * args.steps / (a.elapsed_time(b) / 1e3) / 1e9
    _line("kv block offload+restore GB/s", 2.0 / (1 / res["offload"] + 1 / res["restore"]), "GB/s",
          {"workload": wl.name, "blocks": int(n), "block_bytes": int(bb), "component": "offload"},
          offload_gbs=res["offload"], restore_gbs=res["restore"], steps=args.steps, warmup=args.warmup)


def component_gather(args, wl):
    """Ragged embedding gather (vocab 128k x hidden 4096, bf16) for the
    batch's packed tokens, and the last-token logits gather."""
    import torch
    from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
    layer = R.RaggedLayer(R.params_for(wl), wl.n_seqs, wl.n_tokens, int(wl.blocks_needed().sum()),
                          wl.max_len())
    layer.build(R.SeqDescs.of(wl), wl.num_blocks)
    vocab, hidden = 131072, 4096
    table = torch.randn((vocab, hidden), device="cuda").bfloat16()
    ids = torch.randint(0, vocab, (wl.n_tokens,), device="cuda", dtype=torch.int32)
    out = torch.empty((wl.n_tokens, hidden), device="cuda").bfloat16()
    lg = torch.empty((wl.n_seqs, hidden), device="cuda").bfloat16()
    st = torch.cuda.current_stream()
    t = {}
    for name, fn in (("embedding", lambda: R.ds_ragged_embedding(layer.meta, ids, table, out)),
                     ("logits", lambda: R.ds_ragged_logits_gather(layer.meta, out, lg))):
        for _ in range(args.warmup):
            fn()
        st.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(args.steps):
            fn()
        b.record(st)
        st.synchronize()
        t[name] = a.elapsed_time(b) / args.steps / 1e3
    emb_bytes = 2 * wl.n_tokens * hidden * 2
    _line("ragged embedding gather GB/s", emb_bytes / t["embedding"] / 1e9, "GB/s",
          {"workload": wl.name, "vocab": vocab, "hidden": hidden, "component": "gather"},
          embedding_us=t["embedding"] * 1e6, logits_gather_us=t["logits"] * 1e6,
          logits_gather_gbs=2 * wl.n_seqs * hidden * 2 / t["logits"] / 1e9)


def component_multistep(args, wl):
    """A Dynamic SplitFuse run: 256 requests (prompts log-uniform 32..2048,
    16..256 generated tokens each) through the block ledger, the planner and
    the layer, pass after pass; the workload's head shape, token budget 8192.

    Two numbers.  The live loop: per pass, plan, pack and upload the metadata,
    launch the layer, wait for it (a serving loop samples from its output before
    it can plan the next pass) and commit; its wall time and host time.  The
    device rate: the same passes replayed back to back from metadata built
    beforehand, so the GPU never waits for the host."""
    import torch
    from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
    from ragged_blocked_kv_raggedbatch_gb300.splitfuse import NativeSplitFusePlanner
    rng = np.random.default_rng(args.seed)
    prompts = np.floor(np.exp(rng.uniform(np.log(32), np.log(2048), 256))).astype(int)
    gens = rng.integers(16, 256, 256, endpoint=True)
    nblk = int(sum(-(-(p + g) // 64) for p, g in zip(prompts, gens))) + 64
    params = R.params_for(wl)
    alloc = R.BlockAllocator(nblk, rng.permutation(nblk))
    fused = args.path == "fused"
    plan = NativeSplitFusePlanner(alloc, 8192, 256, max_requests=256, max_blocks_per_request=64)
    for i in range(256):
        plan.add(i, int(prompts[i]), int(gens[i]))
    dt = W.torch_dtype(wl)
    pool = torch.randn((nblk, 2, wl.n_kv_heads, 64, wl.head_dim), device="cuda").to(dt)
    qkv = torch.randn((8192, wl.qkv_width), device="cuda").to(dt)
    out = torch.empty((8192, wl.n_q_heads * wl.head_dim), device="cuda").to(dt)
    st = torch.cuda.Stream()
    layer = R.RaggedLayer(params, 256, 8192, nblk, 4096, stream=st)
    recorded, host_s, rec_s, toks = [], 0.0, 0.0, 0
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    while not plan.idle:
        t0 = time.perf_counter()
        n = plan.plan()
        descs = plan  # its ds_seq_desc[] goes to the metadata build as is
        with torch.cuda.stream(st):
            layer.build(descs, nblk)
            host_s += time.perf_counter() - t0
            if fused:
                layer.fused(qkv, pool, out)
            else:
                layer.append(qkv, pool)
                layer.attention(qkv, pool, out)
        st.synchronize()
        # keep a copy of the pass for the replay below (bench bookkeeping, not timed)
        tr = time.perf_counter()
        rec = [(plan.arr[i].seen_tokens, plan.arr[i].new_tokens,
                np.ctypeslib.as_array(plan.arr[i].block_ids, shape=(plan.arr[i].n_blocks,)).copy())
               for i in range(n)]
        recorded.append(rec)
        toks += sum(r[1] for r in rec)
        t1 = time.perf_counter()
        rec_s += t1 - tr
        plan.commit()
        host_s += time.perf_counter() - t1
    wall_s = time.perf_counter() - t_wall - rec_s
    passes = len(recorded)

    # device rate: replay the recorded passes back to back (one shared
    # workspace; the fused path's counters are back at zero after each call)
    ws_t = layer.fused_ws if fused else layer.workspace
    layers = []
    with torch.cuda.stream(st):
        for rec in recorded:
            L = R.RaggedLayer(params, 256, 8192, nblk, 4096, stream=st, workspace=ws_t)
            if fused:
                L.fused_ws = ws_t
            L.build(R.SeqDescs([r[0] for r in rec], [r[1] for r in rec], [r[2] for r in rec]), nblk)
            layers.append(L)
    st.synchronize()
    rep = []
    for _ in range(max(1, min(args.steps, 5))):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            torch.cuda._sleep(20_000_000)  # the host enqueues every pass before the GPU reaches them
            a.record(st)
            for L in layers:
                if fused:
                    L.fused(qkv, pool, out)
                else:
                    L.append(qkv, pool)
                    L.attention(qkv, pool, out)
            b.record(st)
        st.synchronize()
        rep.append(a.elapsed_time(b) / 1e3)
    dev_s = float(np.median(rep))
    _line("splitfuse multi-pass new tokens/s per layer", toks / dev_s, "tokens/s",
          {"workload": wl.name + "_heads", "requests": 256, "token_budget": 8192, "component": "multistep",
           "planner": "native", "path": args.path},
          passes=passes, tokens=toks, device_ms_per_pass=1e3 * dev_s / passes,
          live_wall_us_per_pass=1e6 * wall_s / passes, live_tokens_per_s=toks / wall_s,
          host_us_per_pass=1e6 * host_s / passes, layer_launches_per_pass=4)


def component_graph(args, wl):
    """One layer step (metadata upload + KV append + attention) replayed from
    a CUDA graph vs. issued call by call, same batch."""
    import torch
    from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
    qkv, pool = W.make_values(wl, "cuda")
    nb = int(wl.blocks_needed().sum())
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        layer = R.RaggedLayer(R.params_for(wl), wl.n_seqs, wl.n_tokens, nb, wl.max_len(), stream=st)
        descs = R.SeqDescs.of(wl)
        out = torch.empty((wl.n_tokens, wl.n_q_heads * wl.head_dim), dtype=qkv.dtype, device="cuda")

    def eager():
        layer.build(descs, wl.num_blocks)
        if args.path == "fused":
            layer.fused(qkv, pool, out)
        else:
            layer.append(qkv, pool)
            layer.attention(qkv, pool, out)

    with torch.cuda.stream(st):
        for _ in range(args.warmup):
            eager()
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        eager()
    res = {}
    for name, fn in (("eager", eager), ("graph", g.replay)):
        with torch.cuda.stream(st):
            for _ in range(args.warmup):
                fn()
            st.synchronize()
            t0 = time.perf_counter()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            for _ in range(args.steps):
                fn()
            b.record(st)
            st.synchronize()
            res[name] = (a.elapsed_time(b) / args.steps, 1e3 * (time.perf_counter() - t0) / args.steps)
    _line("ragged attn layer step, CUDA graph replay (new tokens/s)", wl.n_tokens / (res["graph"][1] / 1e3),
          "tokens/s", {"workload": wl.name, "component": "graph", "path": args.path},
          eager_device_ms=res["eager"][0], eager_wall_ms=res["eager"][1],
          graph_device_ms=res["graph"][0], graph_wall_ms=res["graph"][1], steps=args.steps)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--subset", type=int, default=0,
                    help="profile a smaller case: only the first N sequences, compact pool")
    ap.add_argument("--part", choices=["decode", "prefill"], default=None,
                    help="profile one kernel family: keep only the decode rows or the prefill chunks")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", choices=["split", "fused"], default="split",
                    help="split: ds_kv_rotary_append then ds_blocked_attention; "
                         "fused: ds_fused_append_attention")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle time of the headline workload's CPU baseline (the others take a third)")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only the chosen workload (no per_workload object)")
    ap.add_argument("--component", choices=["offload", "gather", "multistep", "graph"], default=None,
                    help="measure a component next to the layer instead of the layer step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = W.make_workload(args.workload, args.seed)
    if args.part:
        keep = [i for i in range(wl.n_seqs) if (wl.new[i] == 1) == (args.part == "decode")]
        wl = W.compact_sequences(wl, keep, args.seed, suffix="_" + args.part)
    if args.subset:
        wl = W.first_sequences(wl, args.subset, args.seed)
    if args.impl == "reference":
        return reference_arm(args, wl)
    if args.component:
        return {"offload": component_offload, "gather": component_gather,
                "multistep": component_multistep, "graph": component_graph}[args.component](args, wl) or 0
    return gpu_arm(args, wl)


if __name__ == "__main__":
    sys.exit(main())
