"""The C ABI driven from a plain C program (tests/c_abi_client.c): metadata
build, RoPE + KV append and blocked attention through include/ds_ragged.h and
libds_ragged.so alone.  Its output is checked against the oracle, and its pool
and output bits against the same step run through the Python binding."""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest
import torch

import oracle
from gpu_util import LayerRun, bits, check_out, ulp_diff
from ragged_blocked_kv_raggedbatch_gb300 import build as B
from ragged_blocked_kv_raggedbatch_gb300 import ds_ragged as R
from ragged_blocked_kv_raggedbatch_gb300 import workloads as W

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _compile(tmp_path) -> str:
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    lib_dir = os.path.dirname(R.LIB_PATH)
    exe = str(tmp_path / "c_abi_client")
    cmd = [cc, "-std=c11", "-O1", "-Wall", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(HERE, "c_abi_client.c"), "-L", lib_dir, "-lds_ragged", "-L", os.path.join(cuda, "lib64"),
           "-lcudart", "-Wl,-rpath," + lib_dir + ":" + os.path.join(cuda, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


@pytest.mark.parametrize("dtype,style", [("bf16", R.DS_ROPE_HALF), ("fp16", R.DS_ROPE_INTERLEAVED)])
def test_c_program_through_the_abi(tmp_path, dtype, style):
    B.build()
    wl = W.make_custom([(0, 37), (90, 1), (130, 64), (2000, 1), (63, 1), (64, 1)], 8, 2, 64, dtype=dtype,
                       seed=11, extra_blocks=3)
    qkv, pool = W.make_values(wl, "cpu")
    words = [wl.n_q_heads, wl.n_kv_heads, wl.head_dim, R.DS_BF16 if dtype == "bf16" else R.DS_FP16, style,
             wl.n_seqs, wl.num_blocks, wl.max_len(), struct.unpack("<i", struct.pack("<f", wl.rope_theta))[0]]
    for i in range(wl.n_seqs):
        ids = [int(b) for b in wl.block_ids[i]]
        words += [int(wl.seen[i]), int(wl.new[i]), len(ids)] + ids
    paths = {k: str(tmp_path / (k + ".bin")) for k in ("batch", "qkv", "pool", "out", "pool_out")}
    np.array(words, np.int32).tofile(paths["batch"])
    bits(qkv).tofile(paths["qkv"])
    bits(pool).tofile(paths["pool"])
    exe = _compile(tmp_path)
    r = subprocess.run([exe, paths["batch"], paths["qkv"], paths["pool"], paths["out"], paths["pool_out"]],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
    out_bits = np.fromfile(paths["out"], np.uint16).reshape(wl.n_tokens, wl.n_q_heads * wl.head_dim)
    pool_bits = np.fromfile(paths["pool_out"], np.uint16).reshape(wl.pool_shape())
    # against the oracle
    ref = oracle.layer(wl, qkv, pool, style=style)
    got = torch.from_numpy(out_bits.view(np.int16)).view(W.torch_dtype(wl))
    check_out(wl, got, ref["out"], "c client")
    assert ulp_diff(pool_bits, ref["pool"]).max() <= 1
    np.testing.assert_array_equal(pool_bits[:, 1], ref["pool"][:, 1])
    # the same step through the Python binding: the same bits
    pool_g = pool.cuda()
    run = LayerRun(wl, qkv.cuda(), pool_g, rope_style=style, want_q=False)
    assert run.dev_err == 0
    np.testing.assert_array_equal(bits(run.out[: wl.n_tokens]), out_bits)
    np.testing.assert_array_equal(bits(pool_g).reshape(wl.pool_shape()), pool_bits)
