"""CPU oracle for one ragged blocked-KV attention layer (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg import this package.  The CUDA library never imports or calls it,
and the two share no code: this wraps ``ragged_oracle.c`` (plain C, fp64)
through ctypes and converts numpy arrays.

Functions (what each computes is documented in ``ragged_oracle.c``):
  meta_build(wl)                       -> dict of int32 metadata arrays
  rope_append(wl, meta, qkv, pool)     -> (pool', q_rot, slot_block, slot_off)
  attention(wl, meta, qkv, pool, rows) -> fp64 [len(rows), Hq, d]
  layer(wl, qkv, pool, rows=None)      -> all of the above in order

Storage arrays are passed as uint16 bit patterns (fp16 or bf16 by ``wl.dtype``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ragged_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libragged_oracle.so")

DTYPE_CODE = {"fp16": 0, "bf16": 1}
ROPE_HALF, ROPE_INTERLEAVED = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add, no fast math)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # RAGGED_ORACLE_LIB lets the mutation test load a deliberately broken
            # copy of the oracle to show the pins reject it.
            lib = ctypes.CDLL(os.environ.get("RAGGED_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
            lib.oracle_meta_build.restype = i64
            lib.oracle_meta_build.argtypes = [i32, P, P, P, P, i32, P, P, P, P, P, P, P]
            lib.oracle_rope_append.restype = ctypes.c_int
            lib.oracle_rope_append.argtypes = [i32, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                               i32, f32, P, P, P, P, P]
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_attention_rows.argtypes = [i32, P, P, P, P, P, i32, i32, i32, i32, i32,
                                                  i32, f32, f32, P, P, P, i32]
            lib.oracle_storage_to_f64.restype = None
            lib.oracle_storage_to_f64.argtypes = [P, i64, i32, P]
            lib.oracle_f32_to_storage.restype = None
            lib.oracle_f32_to_storage.argtypes = [P, i64, i32, P]
            lib.oracle_rope_vec_f32.restype = None
            lib.oracle_rope_vec_f32.argtypes = [P, P, i64, i32, i32, f32]
            lib.oracle_rope_vec_f64.restype = None
            lib.oracle_rope_vec_f64.argtypes = [P, P, i64, i32, i32, f64]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    """uint16 view of an fp16/bf16 tensor or array (torch tensors go via CPU)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


# --------------------------------------------------------------------------
# Element helpers (pins use these)
# --------------------------------------------------------------------------

def storage_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().oracle_storage_to_f64(_ptr(bits), bits.size, DTYPE_CODE[dtype], _ptr(out))
    return out


def f32_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_f32_to_storage(_ptr(x), x.size, DTYPE_CODE[dtype], _ptr(out))
    return out


def rope_vec_f32(x: np.ndarray, p: int, theta: float, style: int = ROPE_HALF) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    _load().oracle_rope_vec_f32(_ptr(x), _ptr(y), int(p), x.size, style, float(theta))
    return y


def rope_vec_f64(x: np.ndarray, p: int, theta: float, style: int = ROPE_HALF) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_rope_vec_f64(_ptr(x), _ptr(y), int(p), x.size, style, float(theta))
    return y


# --------------------------------------------------------------------------
# The layer
# --------------------------------------------------------------------------

def meta_build(wl) -> dict:
    S = wl.n_seqs
    seen = np.ascontiguousarray(wl.seen, np.int32)
    new = np.ascontiguousarray(wl.new, np.int32)
    counts = np.array([len(b) for b in wl.block_ids], np.int64)
    ids_off = np.zeros(S + 1, np.int64)
    ids_off[1:] = np.cumsum(counts)
    ids_flat = (np.concatenate(wl.block_ids).astype(np.int32) if S else np.zeros(1, np.int32))
    ids_flat = np.ascontiguousarray(ids_flat)
    N = int(new.sum()) if S else 0
    total_ids = int(counts.sum())
    m = dict(
        cu_seqlens=np.zeros(S + 1, np.int32), seq_seen=np.zeros(S, np.int32),
        seq_new=np.zeros(S, np.int32), blk_off=np.zeros(S + 1, np.int32),
        block_table=np.zeros(max(total_ids, 1), np.int32), tok_seq=np.zeros(max(N, 1), np.int32),
        tok_pos=np.zeros(max(N, 1), np.int32))
    nb = _load().oracle_meta_build(
        S, _ptr(seen if S else np.zeros(1, np.int32)), _ptr(new if S else np.zeros(1, np.int32)),
        _ptr(ids_off), _ptr(ids_flat), wl.block_size, _ptr(m["cu_seqlens"]), _ptr(m["seq_seen"]) if S else None,
        _ptr(m["seq_new"]) if S else None, _ptr(m["blk_off"]), _ptr(m["block_table"]),
        _ptr(m["tok_seq"]), _ptr(m["tok_pos"]))
    if nb < 0:
        raise ValueError("invalid sequence descriptors")
    m["block_table"] = m["block_table"][:nb].copy()
    m["tok_seq"] = m["tok_seq"][:N].copy()
    m["tok_pos"] = m["tok_pos"][:N].copy()
    m["n_tokens"] = N
    return m


def rope_append(wl, meta: dict, qkv, pool, want_q: bool = True, style: int = ROPE_HALF):
    """Returns (pool_after, q_rot or None, slot_block, slot_off); pool_after is a
    new uint16 array (the input is not modified)."""
    qkv_b = _bits(qkv).reshape(-1)
    pool_b = _bits(pool).reshape(wl.pool_shape()).copy()
    N = meta["n_tokens"]
    q_out = np.zeros((max(N, 1), wl.n_q_heads * wl.head_dim), np.uint16) if want_q else None
    sb = np.zeros(max(N, 1), np.int32)
    so = np.zeros(max(N, 1), np.int32)
    rc = _load().oracle_rope_append(
        N, _ptr(meta["tok_seq"] if N else sb), _ptr(meta["tok_pos"] if N else so),
        _ptr(meta["blk_off"]), _ptr(meta["block_table"] if len(meta["block_table"]) else sb),
        wl.num_blocks, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.block_size,
        DTYPE_CODE[wl.dtype], style, float(wl.rope_theta), _ptr(qkv_b) if qkv_b.size else None,
        _ptr(pool_b) if pool_b.size else None, _ptr(q_out) if want_q else None, _ptr(sb), _ptr(so))
    if rc != 0:
        raise ValueError("block id out of range")
    return pool_b, (q_out[:N] if want_q else None), sb[:N], so[:N]


def attention(wl, meta: dict, qkv, pool_after, rows=None, n_threads: int = 0,
              style: int = ROPE_HALF, scale: float = 0.0) -> np.ndarray:
    """fp64 attention output [len(rows), Hq, d] for the listed packed tokens
    (all tokens when rows is None)."""
    N = meta["n_tokens"]
    rows = np.arange(N, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    out = np.zeros((len(rows), wl.n_q_heads, wl.head_dim), np.float64)
    if len(rows) == 0:
        return out
    qkv_b = _bits(qkv).reshape(-1)
    pool_b = _bits(pool_after).reshape(-1)
    rc = _load().oracle_attention_rows(
        len(rows), _ptr(rows), _ptr(meta["tok_seq"]), _ptr(meta["tok_pos"]), _ptr(meta["blk_off"]),
        _ptr(meta["block_table"]), wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.block_size,
        DTYPE_CODE[wl.dtype], style, float(wl.rope_theta), float(scale), _ptr(qkv_b), _ptr(pool_b),
        _ptr(out), int(n_threads) if n_threads else default_threads())
    if rc != 0:
        raise ValueError("invalid head configuration")
    return out


def layer(wl, qkv, pool, rows=None, n_threads: int = 0, style: int = ROPE_HALF):
    """Metadata, append and attention in order.  Returns a dict."""
    meta = meta_build(wl)
    pool_after, q_rot, sb, so = rope_append(wl, meta, qkv, pool, style=style)
    out = attention(wl, meta, qkv, pool_after, rows=rows, n_threads=n_threads, style=style)
    return dict(meta=meta, pool=pool_after, q_rot=q_rot, slot_block=sb, slot_off=so, out=out)
