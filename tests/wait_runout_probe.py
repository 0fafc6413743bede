"""Subprocess half of test_gpu_wait_runout.py: drives a test build of the
library (compiled with -DDSR_TEST_WAIT_RUNOUT: every mbarrier wait bounded at
~1 ms, and a device flag that stops the tensor-core decode kernel's producers
from issuing copies).

    python wait_runout_probe.py <path of the test build's libds_ragged.so>

1. A grouped-query decode batch (split rows, G = 4, head_dim 128) with the
   copies stalled: the consumers' waits run out while no copy is in flight;
   the call must come back promptly with DS_DEVERR_WORKLIST in the device
   error word.
2. The same batch again (metadata re-uploaded, which clears the error word)
   with the copies released: no error, and the output matches the CPU oracle.
Prints one JSON line; exit status 0 when both hold.
"""
import ctypes
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R  # noqa: E402
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W  # noqa: E402


def main(lib_path):
    R.LIB_PATH = lib_path
    lib = R.load()
    lib.ds_test_stall_copies.restype = ctypes.c_int32
    lib.ds_test_stall_copies.argtypes = [ctypes.c_int32]
    import oracle
    from gpu_util import check_out

    wl = W.make_custom([(3000, 1), (777, 1), (64 * 9, 1), (130, 1)], 16, 4, 128, dtype="bf16",
                       rope_theta=5e5, seed=31, extra_blocks=2)
    qkv, pool = W.make_values(wl, "cuda")
    pool0 = pool.clone()
    layer = R.RaggedLayer(R.params_for(wl), wl.n_seqs, wl.n_tokens, int(wl.blocks_needed().sum()), wl.max_len())
    layer.build(R.SeqDescs.of(wl), wl.num_blocks)
    layer.append(qkv, pool)
    out = torch.full((wl.n_tokens, wl.n_q_heads * wl.head_dim), float("nan"), dtype=qkv.dtype, device="cuda")
    torch.cuda.synchronize()
    res = {"split_items": layer.meta.n_decode_items, "rows": layer.meta.n_decode_seqs}

    assert lib.ds_test_stall_copies(1) == R.DS_OK
    t0 = time.perf_counter()
    layer.attention(qkv, pool, out)
    torch.cuda.synchronize()
    res["stalled_call_s"] = time.perf_counter() - t0
    res["stalled_error_word"] = layer.device_error()
    assert lib.ds_test_stall_copies(0) == R.DS_OK

    layer.build(R.SeqDescs.of(wl), wl.num_blocks)  # a fresh upload clears the error word
    out.fill_(float("nan"))
    layer.attention(qkv, pool, out)
    torch.cuda.synchronize()
    res["next_error_word"] = layer.device_error()
    want = oracle.layer(wl, qkv.cpu(), pool0.cpu())["out"]
    res["next_max_abs"], res["next_mean_abs"] = (float(x) for x in check_out(wl, out, want, "after run-out"))
    ok = (res["stalled_error_word"] & R.DS_DEVERR_WORKLIST) != 0 and res["next_error_word"] == 0 \
        and res["stalled_call_s"] < 30.0
    res["ok"] = bool(ok)
    print(json.dumps(res), flush=True)
    return 0 if ok else 1


if __name__ == "__main__":
    sys.exit(main(sys.argv[1]))
