"""Thin Python binding of ``libds_ragged.so`` (argument marshalling only).

The functions keep the C ABI's names (``include/ds_ragged.h``); every step of
the layer runs in the library's CUDA kernels.  PyTorch supplies device memory,
pinned host memory and streams.  There is no fallback: if the library is
missing, importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libds_ragged.so")

DS_OK, DS_ERR_INVALID_ARG, DS_ERR_CAPACITY, DS_ERR_BAD_BLOCK = 0, 1, 2, 3
DS_ERR_UNSUPPORTED, DS_ERR_WORKSPACE, DS_ERR_CUDA = 4, 5, 6
DS_DEVERR_BLOCK_ID, DS_DEVERR_POSITION, DS_DEVERR_WORKLIST, DS_DEVERR_TOKEN = 1, 2, 4, 8
DS_FP16, DS_BF16 = 0, 1
DS_ROPE_HALF, DS_ROPE_INTERLEAVED = 0, 1
DS_META_CAPACITY = 1
STATUS_NAMES = {0: "DS_OK", 1: "DS_ERR_INVALID_ARG", 2: "DS_ERR_CAPACITY", 3: "DS_ERR_BAD_BLOCK",
                4: "DS_ERR_UNSUPPORTED", 5: "DS_ERR_WORKSPACE", 6: "DS_ERR_CUDA"}

P = ctypes.c_void_p
i32 = ctypes.c_int32


class ds_seq_desc(ctypes.Structure):
    _fields_ = [("seen_tokens", i32), ("new_tokens", i32),
                ("block_ids", ctypes.POINTER(i32)), ("n_blocks", i32)]


class ds_attn_params(ctypes.Structure):
    _fields_ = [("n_q_heads", i32), ("n_kv_heads", i32), ("head_dim", i32), ("block_size", i32),
                ("dtype", i32), ("rope_style", i32), ("rope_theta", ctypes.c_float),
                ("softmax_scale", ctypes.c_float)]


class ds_kv_pool(ctypes.Structure):
    _fields_ = [("base", P), ("num_blocks", i32)]


class ds_rope_table(ctypes.Structure):
    _fields_ = [("table", P), ("max_positions", i32), ("head_dim", i32),
                ("rope_theta", ctypes.c_float)]


class ds_ragged_meta(ctypes.Structure):
    _fields_ = [("device_buf", P), ("device_bytes", ctypes.c_size_t),
                ("host_staging", P), ("staging_bytes", ctypes.c_size_t),
                ("max_seqs", i32), ("max_tokens", i32), ("max_blocks", i32), ("flags", i32),
                ("n_seqs", i32), ("n_tokens", i32), ("n_blocks", i32),
                ("n_prefill_seqs", i32), ("n_decode_seqs", i32), ("n_prefill_tiles", i32),
                ("n_decode_items", i32), ("max_len", i32), ("pool_num_blocks", i32),
                ("split_blocks", i32), ("prefill_sms", ctypes.c_float), ("used_bytes", ctypes.c_size_t),
                ("header", P), ("cu_seqlens", P), ("seq_seen", P), ("seq_new", P),
                ("blk_off", P), ("block_table", P), ("tok_seq", P), ("tok_pos", P),
                ("prefill_tiles", P), ("decode_items", P), ("decode_seqs", P)]


class ds_block_allocator(ctypes.Structure):
    _fields_ = [("stack", P), ("state", P), ("num_blocks", i32), ("n_free", i32)]


class ds_splitfuse(ctypes.Structure):
    _fields_ = [("mem", P), ("mem_bytes", ctypes.c_size_t), ("max_requests", i32),
                ("max_blocks_per_request", i32), ("token_budget", i32), ("max_seqs", i32),
                ("block_size", i32), ("n_active", i32), ("n_planned", i32)]


# name -> (restype, argtypes); every entry point of include/ds_ragged.h
SIGNATURES = {
    "ds_last_error": (ctypes.c_char_p, []),
    "ds_version": (ctypes.c_char_p, []),
    "ds_meta_buffer_sizes": (i32, [i32, i32, i32, P, P, P]),
    "ds_ragged_meta_pack": (i32, [P, i32, P, i32, P]),
    "ds_ragged_meta_build": (i32, [P, i32, P, i32, P, P]),
    "ds_rope_table_size": (i32, [P, i32, P]),
    "ds_rope_table_build": (i32, [P, i32, P, ctypes.c_size_t, P, P]),
    "ds_kv_rotary_append": (i32, [P, P, P, P, P, P, P]),
    "ds_blocked_attention_workspace_size": (i32, [P, i32, i32, i32, P]),
    "ds_blocked_attention": (i32, [P, P, P, P, P, P, P, ctypes.c_size_t, P]),
    "ds_get_device_error": (i32, [P, P, P]),
    "ds_blocked_attention_static_ws": (i32, [P, P, P, P, P, P, P]),
    "ds_fused_workspace_size": (i32, [P, i32, i32, i32, P]),
    "ds_fused_workspace_init": (i32, [P, P, P, ctypes.c_size_t, P]),
    "ds_fused_append_attention": (i32, [P, P, P, P, P, P, P, ctypes.c_size_t, P]),
    "ds_block_allocator_init": (i32, [P, P, P, i32, P]),
    "ds_block_allocator_allocate": (i32, [P, i32, P]),
    "ds_block_allocator_free": (i32, [P, P, i32]),
    "ds_kv_blocks_required": (i32, [i32, i32, i32, i32, P]),
    "ds_splitfuse_mem_size": (i32, [i32, i32, P]),
    "ds_splitfuse_init": (i32, [P, P, ctypes.c_size_t, i32, i32, i32, i32, i32]),
    "ds_splitfuse_add": (i32, [P, i32, i32, i32]),
    "ds_splitfuse_next": (i32, [P, P, P, P, P]),
    "ds_splitfuse_commit": (i32, [P, P, P, P]),
    "ds_kv_block_bytes": (i32, [P, P]),
    "ds_kv_offload": (i32, [P, P, P, i32, P, P]),
    "ds_kv_restore": (i32, [P, P, P, i32, P, P]),
    "ds_ragged_embedding": (i32, [P, P, P, i32, i32, i32, P, P]),
    "ds_ragged_logits_gather": (i32, [P, P, i32, i32, P, P]),
}

DS_STATIC_WORKSPACE_BYTES = 32 << 20

_lib = None


class DSError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__("%s: %s (%s)" % (where, msg, STATUS_NAMES.get(status, status)))
        self.status = status


def load():
    """Load the library (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libds_ragged.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ref(x):
    return ctypes.cast(ctypes.pointer(x), P) if x is not None else None


def _check(status: int, where: str):
    if status != DS_OK:
        raise DSError(status, where, load().ds_last_error().decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def make_params(n_q_heads: int, n_kv_heads: int, head_dim: int, dtype: str = "bf16",
                rope_theta: float = 1.0e4, rope_style: int = DS_ROPE_HALF,
                block_size: int = 64, softmax_scale: float = 0.0) -> ds_attn_params:
    return ds_attn_params(n_q_heads, n_kv_heads, head_dim, block_size,
                          {"fp16": DS_FP16, "bf16": DS_BF16}[dtype] if isinstance(dtype, str) else dtype,
                          rope_style, rope_theta, softmax_scale)


def params_for(wl, rope_style: int = DS_ROPE_HALF) -> ds_attn_params:
    return make_params(wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.dtype, wl.rope_theta,
                       rope_style, wl.block_size)


class SeqDescs:
    """ds_seq_desc[] for a workload (keeps the id arrays alive)."""

    def __init__(self, seen: Sequence[int], new: Sequence[int], block_ids: Sequence[np.ndarray]):
        self.ids = [np.ascontiguousarray(b, dtype=np.int32) for b in block_ids]
        n = len(self.ids)
        self.arr = (ds_seq_desc * max(n, 1))()
        for i in range(n):
            self.arr[i].seen_tokens = int(seen[i])
            self.arr[i].new_tokens = int(new[i])
            self.arr[i].block_ids = self.ids[i].ctypes.data_as(ctypes.POINTER(i32))
            self.arr[i].n_blocks = len(self.ids[i])
        self.n = n

    @classmethod
    def of(cls, wl):
        return cls(wl.seen, wl.new, wl.block_ids)


# ------------------------------------------------------------ thin wrappers --

def ds_meta_buffer_sizes(max_seqs: int, max_tokens: int, max_blocks: int, params: ds_attn_params):
    dev, stg = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().ds_meta_buffer_sizes(max_seqs, max_tokens, max_blocks, _ref(params),
                                       _ref(dev), _ref(stg)), "ds_meta_buffer_sizes")
    return dev.value, stg.value


def ds_ragged_meta_pack(descs: SeqDescs, params: ds_attn_params, pool_num_blocks: int,
                        meta: ds_ragged_meta) -> int:
    return load().ds_ragged_meta_pack(_ref(descs.arr), descs.n, _ref(params), pool_num_blocks, _ref(meta))


def ds_ragged_meta_build(descs: SeqDescs, params: ds_attn_params, pool_num_blocks: int,
                         meta: ds_ragged_meta, stream=None):
    _check(load().ds_ragged_meta_build(_ref(descs.arr), descs.n, _ref(params), pool_num_blocks,
                                       _ref(meta), _stream(stream)), "ds_ragged_meta_build")


def ds_rope_table_size(params: ds_attn_params, max_positions: int) -> int:
    b = ctypes.c_size_t(0)
    _check(load().ds_rope_table_size(_ref(params), max_positions, _ref(b)), "ds_rope_table_size")
    return b.value


def ds_rope_table_build(params: ds_attn_params, max_positions: int, table, stream=None) -> ds_rope_table:
    out = ds_rope_table()
    nbytes = table.numel() * table.element_size()
    _check(load().ds_rope_table_build(_ref(params), max_positions, _ptr(table), nbytes, _ref(out),
                                      _stream(stream)), "ds_rope_table_build")
    return out


def ds_kv_rotary_append(meta: ds_ragged_meta, params: ds_attn_params, rope: ds_rope_table, qkv,
                        q_out, pool: ds_kv_pool, stream=None):
    _check(load().ds_kv_rotary_append(_ref(meta), _ref(params), _ref(rope), _ptr(qkv), _ptr(q_out),
                                      _ref(pool), _stream(stream)), "ds_kv_rotary_append")


def ds_blocked_attention_workspace_size(params: ds_attn_params, max_seqs: int, max_tokens: int,
                                        max_blocks: int) -> int:
    b = ctypes.c_size_t(0)
    _check(load().ds_blocked_attention_workspace_size(_ref(params), max_seqs, max_tokens, max_blocks,
                                                      _ref(b)), "ds_blocked_attention_workspace_size")
    return b.value


def ds_blocked_attention(meta: ds_ragged_meta, params: ds_attn_params, rope: ds_rope_table, qkv,
                         pool: ds_kv_pool, out, workspace, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().ds_blocked_attention(_ref(meta), _ref(params), _ref(rope), _ptr(qkv), _ref(pool),
                                       _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)),
           "ds_blocked_attention")


def ds_fused_workspace_size(params: ds_attn_params, max_seqs: int, max_tokens: int, max_blocks: int) -> int:
    b = ctypes.c_size_t(0)
    _check(load().ds_fused_workspace_size(_ref(params), max_seqs, max_tokens, max_blocks, _ref(b)),
           "ds_fused_workspace_size")
    return b.value


def ds_fused_workspace_init(meta: ds_ragged_meta, params: ds_attn_params, workspace, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().ds_fused_workspace_init(_ref(meta), _ref(params), _ptr(workspace), ws_bytes, _stream(stream)),
           "ds_fused_workspace_init")


def ds_fused_append_attention(meta: ds_ragged_meta, params: ds_attn_params, rope: ds_rope_table, qkv,
                              pool: ds_kv_pool, out, workspace, stream=None):
    """The append and the attention of one batch (a decode-only batch is one launch)."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().ds_fused_append_attention(_ref(meta), _ref(params), _ref(rope), _ptr(qkv), _ref(pool),
                                            _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)),
           "ds_fused_append_attention")


def ds_blocked_attention_static_ws(meta: ds_ragged_meta, params: ds_attn_params, rope: ds_rope_table,
                                   qkv, pool: ds_kv_pool, out, stream=None):
    """ds_blocked_attention with the split partials in the library's built-in
    scratch array (no workspace argument; nothing is allocated)."""
    _check(load().ds_blocked_attention_static_ws(_ref(meta), _ref(params), _ref(rope), _ptr(qkv),
                                                 _ref(pool), _ptr(out), _stream(stream)),
           "ds_blocked_attention_static_ws")


def ds_kv_block_bytes(params: ds_attn_params) -> int:
    b = ctypes.c_size_t(0)
    _check(load().ds_kv_block_bytes(_ref(params), _ref(b)), "ds_kv_block_bytes")
    return b.value


def ds_kv_offload(params: ds_attn_params, pool: ds_kv_pool, block_ids, host_dst, stream=None):
    ids = np.ascontiguousarray(block_ids, np.int32)
    _check(load().ds_kv_offload(_ref(params), _ref(pool), ids.ctypes.data if len(ids) else None, len(ids),
                                _ptr(host_dst), _stream(stream)), "ds_kv_offload")


def ds_kv_restore(params: ds_attn_params, pool: ds_kv_pool, block_ids, host_src, stream=None):
    ids = np.ascontiguousarray(block_ids, np.int32)
    _check(load().ds_kv_restore(_ref(params), _ref(pool), ids.ctypes.data if len(ids) else None, len(ids),
                                _ptr(host_src), _stream(stream)), "ds_kv_restore")


def ds_ragged_embedding(meta: ds_ragged_meta, token_ids, table, out, stream=None):
    vocab, hidden = table.shape
    _check(load().ds_ragged_embedding(_ref(meta), _ptr(token_ids), _ptr(table), vocab, hidden,
                                      table.element_size(), _ptr(out), _stream(stream)), "ds_ragged_embedding")


def ds_ragged_logits_gather(meta: ds_ragged_meta, hidden_states, out, stream=None):
    hidden = hidden_states.shape[1]
    _check(load().ds_ragged_logits_gather(_ref(meta), _ptr(hidden_states), hidden,
                                          hidden_states.element_size(), _ptr(out), _stream(stream)),
           "ds_ragged_logits_gather")


def ds_get_device_error(meta: ds_ragged_meta, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(load().ds_get_device_error(_ref(meta), _ref(v), _stream(stream)), "ds_get_device_error")
    return v.value


class BlockAllocator:
    """The C-ABI block ledger with its two host arrays."""

    def __init__(self, num_blocks: int, initial_order=None):
        self.stack = np.zeros(max(num_blocks, 1), np.int32)
        self.state = np.zeros(max(num_blocks, 1), np.uint8)
        self.a = ds_block_allocator()
        order = None if initial_order is None else np.ascontiguousarray(initial_order, np.int32)
        self._order = order
        _check(load().ds_block_allocator_init(_ref(self.a), self.stack.ctypes.data, self.state.ctypes.data,
                                              num_blocks, None if order is None else order.ctypes.data),
               "ds_block_allocator_init")

    @property
    def n_free(self) -> int:
        return self.a.n_free

    def allocate(self, n: int) -> np.ndarray:
        out = np.zeros(max(n, 1), np.int32)
        _check(load().ds_block_allocator_allocate(_ref(self.a), n, out.ctypes.data), "ds_block_allocator_allocate")
        return out[:n].copy()

    def free(self, ids) -> None:
        ids = np.ascontiguousarray(ids, np.int32)
        _check(load().ds_block_allocator_free(_ref(self.a), ids.ctypes.data if len(ids) else None, len(ids)),
               "ds_block_allocator_free")


def ds_kv_blocks_required(seen: int, new: int, owned: int, block_size: int = 64) -> int:
    e = ctypes.c_int32(0)
    _check(load().ds_kv_blocks_required(seen, new, owned, block_size, _ref(e)), "ds_kv_blocks_required")
    return e.value


# ------------------------------------------------------- buffer management --

class RaggedLayer:
    """Caller-side buffers for one layer shape and capacity (all allocated with
    torch), plus the three calls of a forward pass."""

    def __init__(self, params: ds_attn_params, max_seqs: int, max_tokens: int, max_blocks: int,
                 max_positions: int, device: str = "cuda", stream=None, workspace=None, flags: int = 0):
        import torch
        self.params = params
        self.device = device
        self.stream = stream
        dev_b, stg_b = ds_meta_buffer_sizes(max_seqs, max_tokens, max_blocks, params)
        self.meta_dev = torch.empty(dev_b, dtype=torch.uint8, device=device)
        self.meta_stage = torch.empty(stg_b, dtype=torch.uint8, pin_memory=True)
        self.meta = ds_meta_init(self.meta_dev, self.meta_stage, max_seqs, max_tokens, max_blocks)
        self.meta.flags = flags
        rb = ds_rope_table_size(params, max_positions)
        self.rope_buf = torch.empty(max(rb, 16), dtype=torch.uint8, device=device)
        self.rope = ds_rope_table_build(params, max_positions, self.rope_buf, stream)
        wb = ds_blocked_attention_workspace_size(params, max_seqs, max_tokens, max_blocks)
        # a caller may share one workspace between layers whose calls are ordered on one stream
        self.workspace = workspace if workspace is not None else torch.empty(wb, dtype=torch.uint8, device=device)
        self.fused_ws = None  # made (and its counters zeroed) on the first fused call

    def build(self, descs: SeqDescs, pool_num_blocks: int):
        ds_ragged_meta_build(descs, self.params, pool_num_blocks, self.meta, self.stream)

    def pack(self, descs: SeqDescs, pool_num_blocks: int):
        """Host half of build (validate and pack into the staging buffer; no
        upload): with DS_META_CAPACITY, what a captured graph's upload then
        copies for the next replay."""
        _check(ds_ragged_meta_pack(descs, self.params, pool_num_blocks, self.meta), "ds_ragged_meta_pack")

    def append(self, qkv, pool_t, q_out=None):
        pool = ds_kv_pool(pool_t.data_ptr(), pool_t.shape[0])
        ds_kv_rotary_append(self.meta, self.params, self.rope, qkv, q_out, pool, self.stream)

    def attention(self, qkv, pool_t, out):
        pool = ds_kv_pool(pool_t.data_ptr(), pool_t.shape[0])
        ds_blocked_attention(self.meta, self.params, self.rope, qkv, pool, out, self.workspace, self.stream)

    def fused(self, qkv, pool_t, out):
        """Append + attention in one call (ds_fused_append_attention)."""
        import torch
        if self.fused_ws is None:
            m = self.meta
            fb = ds_fused_workspace_size(self.params, m.max_seqs, m.max_tokens, m.max_blocks)
            self.fused_ws = torch.empty(fb, dtype=torch.uint8, device=self.device)
            ds_fused_workspace_init(self.meta, self.params, self.fused_ws, self.stream)
        pool = ds_kv_pool(pool_t.data_ptr(), pool_t.shape[0])
        ds_fused_append_attention(self.meta, self.params, self.rope, qkv, pool, out, self.fused_ws, self.stream)

    def device_error(self) -> int:
        return ds_get_device_error(self.meta, self.stream)

    def read_meta(self) -> dict:
        """Copy the uploaded metadata back and split it into named arrays."""
        import torch
        n = self.meta.used_bytes
        raw = self.meta_dev[:n].cpu().numpy().view(np.int32)
        return unpack_meta(self.meta, raw, int(self.meta_dev.data_ptr()))


def ds_meta_init(dev_buf, staging, max_seqs: int, max_tokens: int, max_blocks: int) -> ds_ragged_meta:
    m = ds_ragged_meta()
    m.device_buf = _ptr(dev_buf)
    m.device_bytes = dev_buf.numel() * dev_buf.element_size() if hasattr(dev_buf, "numel") else dev_buf.nbytes
    m.host_staging = _ptr(staging)
    m.staging_bytes = staging.numel() * staging.element_size() if hasattr(staging, "numel") else staging.nbytes
    m.max_seqs, m.max_tokens, m.max_blocks = max_seqs, max_tokens, max_blocks
    return m


def unpack_meta(meta: ds_ragged_meta, words: np.ndarray, base_addr: int) -> dict:
    """Named views of a packed metadata image (staging or device copy)."""
    def at(ptr, count, width=1):
        off = (ptr - base_addr) // 4
        return words[off:off + count * width].reshape(-1, width) if width > 1 else words[off:off + count]
    S, N = meta.n_seqs, meta.n_tokens
    return dict(
        header=at(meta.header, 16),
        cu_seqlens=at(meta.cu_seqlens, S + 1), seq_seen=at(meta.seq_seen, S),
        seq_new=at(meta.seq_new, S), blk_off=at(meta.blk_off, S + 1),
        block_table=at(meta.block_table, meta.n_blocks), tok_seq=at(meta.tok_seq, N),
        tok_pos=at(meta.tok_pos, N),
        prefill_tiles=at(meta.prefill_tiles, meta.n_prefill_tiles, 4),
        decode_items=at(meta.decode_items, meta.n_decode_items, 4),
        decode_seqs=at(meta.decode_seqs, meta.n_decode_seqs, 4))
