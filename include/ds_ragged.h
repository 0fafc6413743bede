/*
 * ds_ragged.h -- C ABI of the ragged blocked-KV attention layer for one GB300
 * (sm_103a): rotary embedding + KV-cache append, then causal attention of every
 * new token over its sequence's whole history read through integer block ids.
 *
 * Source of the design ("DeepSpeed Inference v2", pyshine.com/deepspeed-2):
 *  - section "Ragged batches: packing a whole server into four tensors": the
 *    tokens of all in-flight sequences are concatenated into one stream with
 *    per-sequence metadata in parallel buffers (RaggedBatchWrapper's
 *    insert_sequence packs host buffers, finalize uploads them with a few
 *    non-blocking copies); kernels read block ids from the metadata and address
 *    the KV pools directly, so one kernel serves any batch composition;
 *    attention runs over per-head work "atoms" (AtomBuilder) in a blocked flash
 *    attention kernel (BlockedFlashAttn).
 *  - section "The front desk": a DSSequenceDescriptor keeps the integer block
 *    ids of its sequence; BlockedKVCache pools are flat block-indexed tensors;
 *    the allocator's discipline makes overflow impossible to hide; scheduling
 *    answers with a result instead of throwing.
 *  - "DeepSpeed-Inference and DeepSpeed-MII" tutorial (jwzheng96, ch. 10),
 *    section 10.3: Dynamic SplitFuse mixes prefill chunks and single-token
 *    decodes in one batch; engine limits max_ragged_sequence_count = 256 and
 *    max_ragged_batch_size = 8192 (used as default capacities by callers, not
 *    hard-coded: every capacity is an argument).
 *
 * Conventions (all calls):
 *  - The library never allocates device or pinned memory and owns no stream.
 *    Every buffer is the caller's; sizes come from the *_size functions.
 *  - Device calls are asynchronous on the caller's stream.  Argument errors
 *    are found on the host before anything is enqueued and returned as a
 *    ds_status; nothing is thrown and nothing traps.  ds_last_error() gives a
 *    one-line message for the calling thread.
 *  - Kernels also check every block id and position they use; a violation sets
 *    a device error word (read by ds_get_device_error) and skips the access.
 *  - Storage types: IEEE fp16 or bfloat16 (DS_FP16, DS_BF16).
 */
#ifndef DS_RAGGED_H
#define DS_RAGGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status -- */
typedef int32_t ds_status;
#define DS_OK 0
#define DS_ERR_INVALID_ARG 1  /* null pointer, misaligned buffer, bad field   */
#define DS_ERR_CAPACITY 2     /* over a capacity, or a block list too short   */
#define DS_ERR_BAD_BLOCK 3    /* block id outside the pool, or used twice     */
#define DS_ERR_UNSUPPORTED 4  /* head_dim, block_size, dtype or head ratio    */
#define DS_ERR_WORKSPACE 5    /* a caller buffer is smaller than required     */
#define DS_ERR_CUDA 6         /* a CUDA runtime call failed                   */

/* Device error word bits (ds_get_device_error). */
#define DS_DEVERR_BLOCK_ID 1  /* a kernel met a block id outside the pool     */
#define DS_DEVERR_POSITION 2  /* a position beyond the rotary table or blocks */
#define DS_DEVERR_WORKLIST 4  /* an inconsistent work-list entry              */
#define DS_DEVERR_TOKEN 8     /* a token id outside the embedding table       */

#define DS_FP16 0
#define DS_BF16 1

#define DS_ROPE_HALF 0        /* pairs (x_k, x_{k+d/2})  (default)            */
#define DS_ROPE_INTERLEAVED 1 /* pairs (x_{2k}, x_{2k+1})                     */

/* Thread-local message describing the last non-DS_OK status of this thread. */
const char* ds_last_error(void);

/* ------------------------------------------------------------ descriptors -- */

/* One sequence of the batch (the DSSequenceDescriptor of the pages): tokens
 * already in the cache, tokens in this forward pass, and the integer block ids
 * it owns, in order (HOST memory, read during the call only).  A sequence uses
 * its first ceil((seen+new)/block_size) ids; extra ids are ignored; fewer is
 * DS_ERR_CAPACITY.  new_tokens >= 1, seen_tokens >= 0. */
typedef struct ds_seq_desc {
    int32_t seen_tokens;
    int32_t new_tokens;
    const int32_t* block_ids;
    int32_t n_blocks;
} ds_seq_desc;

/* Layer shape.  Supported: head_dim 64 or 128, block_size 64, n_q_heads a
 * multiple of n_kv_heads with g = n_q_heads/n_kv_heads in {1,2,4,8};
 * rope_theta > 0; softmax_scale <= 0 selects 1/sqrt(head_dim).
 * Query head h reads KV head floor(h / g). */
typedef struct ds_attn_params {
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t dtype;      /* DS_FP16 | DS_BF16 */
    int32_t rope_style; /* DS_ROPE_HALF | DS_ROPE_INTERLEAVED */
    float rope_theta;
    float softmax_scale;
} ds_attn_params;

/* The block-indexed KV pool (one cache group of the BlockedKVCache).
 * base: DEVICE, 16-byte aligned, layout [num_blocks][2][n_kv_heads][block_size]
 * [head_dim] of the storage type: index 0 of the second axis holds rotated
 * keys, index 1 values.  Each (block, K|V, head) tile is contiguous. */
typedef struct ds_kv_pool {
    void* base;
    int32_t num_blocks;
} ds_kv_pool;

/* Rotary table: DEVICE float pairs (cos, sin) [max_positions][head_dim/2] for
 * angle fp32(fp32(p) * fp32(theta^(-2k/d))), each rounded from fp64.  Built once
 * per (theta, head_dim) by ds_rope_table_build, like any per-model constant. */
typedef struct ds_rope_table {
    const void* table;
    int32_t max_positions;
    int32_t head_dim;
    float rope_theta;
} ds_rope_table;

/* ds_ragged_meta.flags: lay every metadata region out at the offset the
 * capacities give (not the batch's counts) and upload the whole image.  Every
 * kernel takes its counts from the uploaded header, so with this flag the
 * device calls make launches that depend only on the capacities: a CUDA
 * graph captured around ds_ragged_meta_build and the layer calls for one
 * batch replays correctly for any other batch within the capacities, once
 * ds_ragged_meta_pack has packed that batch into the same staging buffer
 * (ds_ragged_meta_build's validation then runs outside the graph).  The cost:
 * an upload of the full capacity image, and launches sized by the
 * capacities whose CTAs beyond the batch's work exit at once.  The caller
 * keeps max_len within the rope table and the pool and workspace sized for
 * the capacities. */
#define DS_META_CAPACITY 1

/* Ragged batch metadata (the RaggedBatchWrapper's buffers).
 * Caller fills the first group and keeps it; ds_ragged_meta_build fills the
 * rest on every batch. */
typedef struct ds_ragged_meta {
    /* --- set by the caller (ds_meta_buffer_sizes gives the byte counts) --- */
    void* device_buf;     /* DEVICE, 256-byte aligned                        */
    size_t device_bytes;
    void* host_staging;   /* HOST (pinned for an asynchronous upload)        */
    size_t staging_bytes;
    int32_t max_seqs;
    int32_t max_tokens;
    int32_t max_blocks;   /* capacity of the packed block table              */
    int32_t flags;        /* 0 or DS_META_CAPACITY                           */
    /* --- filled by ds_ragged_meta_build --- */
    int32_t n_seqs;
    int32_t n_tokens;
    int32_t n_blocks;     /* entries of the packed block table               */
    int32_t n_prefill_seqs;
    int32_t n_decode_seqs;
    int32_t n_prefill_tiles;
    int32_t n_decode_items;
    int32_t max_len;      /* max over sequences of seen + new                */
    int32_t pool_num_blocks;
    int32_t split_blocks; /* KV blocks per decode split                      */
    float prefill_sms;    /* SMs the prefill grid takes when decode rows run
                             beside it (0: all SMs)                          */
    size_t used_bytes;    /* bytes uploaded                                  */
    /* DEVICE pointers into device_buf (int32 unless noted):
     *   header[16]        word 0: device error bits, 1: S, 2: N, 3: blocks;
     *                     the rest are the work-list counts, the prefill
     *                     grid size and atom order the pack chose, and the
     *                     kernels' own counters (internal; the counters are
     *                     zero after each upload)
     *   cu_seqlens[S+1]   exclusive prefix sum of new_tokens
     *   seq_seen[S], seq_new[S]
     *   blk_off[S+1]      exclusive prefix sum of ceil((seen+new)/block_size)
     *   block_table[n_blocks]  each sequence's used ids, in batch order
     *   tok_seq[N]        sequence index of each packed token
     *   tok_pos[N]        position seen_i + j of each packed token
     *   prefill_tiles     int4 {seq, first token j0, tokens in tile, kv_len}
     *                     kv_len = keys the tile's last row attends to
     *   decode_items      int4 {seq, first block, end block, partial slot}
     *   decode_seqs       int4 {seq, token, first item, item count} */
    int32_t* header;
    int32_t* cu_seqlens;
    int32_t* seq_seen;
    int32_t* seq_new;
    int32_t* blk_off;
    int32_t* block_table;
    int32_t* tok_seq;
    int32_t* tok_pos;
    int32_t* prefill_tiles;
    int32_t* decode_items;
    int32_t* decode_seqs;
} ds_ragged_meta;

/* ------------------------------------------------------------------ calls -- */

/* Byte counts for a metadata device buffer and its host staging buffer that
 * hold any batch within the capacities.  Returns DS_ERR_INVALID_ARG on
 * negative capacities, DS_ERR_UNSUPPORTED on an unsupported params. */
ds_status ds_meta_buffer_sizes(int32_t max_seqs, int32_t max_tokens, int32_t max_blocks,
                               const ds_attn_params* params, size_t* device_bytes,
                               size_t* staging_bytes);

/* Host half of ds_ragged_meta_build (no CUDA call): validate the descriptors
 * and pack the metadata and the work lists into meta->host_staging; fill the
 * host fields of *meta and its device pointers.  Validation order: argument
 * pointers and params, then per sequence new_tokens >= 1 and seen >= 0
 * (DS_ERR_INVALID_ARG), block list length and the capacities
 * (DS_ERR_CAPACITY), block ids inside [0, pool_num_blocks) and no id used
 * twice in the batch (DS_ERR_BAD_BLOCK). */
ds_status ds_ragged_meta_pack(const ds_seq_desc* seqs, int32_t n_seqs,
                              const ds_attn_params* params, int32_t pool_num_blocks,
                              ds_ragged_meta* meta);

/* RaggedBatchWrapper.insert_sequence + finalize: ds_ragged_meta_pack, then one
 * cudaMemcpyAsync of meta->used_bytes from host_staging to device_buf on
 * `stream`.  host_staging must stay untouched until the stream has passed
 * this point.  stream is a cudaStream_t (0 = legacy default stream). */
ds_status ds_ragged_meta_build(const ds_seq_desc* seqs, int32_t n_seqs,
                               const ds_attn_params* params, int32_t pool_num_blocks,
                               ds_ragged_meta* meta, void* stream);

/* Bytes of a rotary table for positions [0, max_positions). */
ds_status ds_rope_table_size(const ds_attn_params* params, int32_t max_positions,
                             size_t* bytes);

/* Fill a caller-allocated DEVICE table (16-byte aligned) and describe it in
 * *out.  One kernel on `stream`; cos/sin evaluated in fp64 on the device. */
ds_status ds_rope_table_build(const ds_attn_params* params, int32_t max_positions,
                              void* table, size_t table_bytes, ds_rope_table* out,
                              void* stream);

/* Rotary embedding + KV append (one kernel).  For every packed token t
 * (sequence i, position p = seen_i + j): rotate its key heads and store them,
 * with its value heads unchanged, in slot (block_table_i[p / block_size],
 * p % block_size) of the pool.  When q_out is not NULL also write the rotated
 * query heads, storage-rounded, to q_out[N][n_q_heads*head_dim].
 * qkv: DEVICE, 16-byte aligned, [N][(n_q_heads + 2*n_kv_heads)*head_dim], each
 * row = query heads, then key heads, then value heads.  Not modified.
 * Rotation per pair (x0, x1) with (c, s) from the table, all in fp32 and never
 * fused: y0 = x0*c - x1*s, y1 = x1*c + x0*s; then round-to-nearest-even. */
ds_status ds_kv_rotary_append(const ds_ragged_meta* meta, const ds_attn_params* params,
                              const ds_rope_table* rope, const void* qkv, void* q_out,
                              const ds_kv_pool* pool, void* stream);

/* Workspace bytes ds_blocked_attention needs for any batch within the
 * capacities (decode split partials: fp32 (m, l) pairs per item and query
 * head, then the fp32 o vectors from the next 256-byte boundary). */
ds_status ds_blocked_attention_workspace_size(const ds_attn_params* params, int32_t max_seqs,
                                              int32_t max_tokens, int32_t max_blocks,
                                              size_t* bytes);

/* Blocked causal attention (BlockedFlashAttn over the work atoms): for every
 * packed token t of sequence i at position p and every query head h,
 *   out[t][h] = sum_{u<=p} softmax_u(scale * <rot(q_t,h), K[u]>) V[u]
 * with K, V read from the pool through the sequence's block table, KV head
 * floor(h/g), and the query rotated on load (fp32, same rule as the append).
 * Must follow ds_kv_rotary_append of the same batch on the same stream.
 * Prefill tiles (sequences with new_tokens > 1) run on tensor cores; decode
 * rows (new_tokens == 1) run a split-K kernel over KV blocks and a combine.
 * out: DEVICE, 16-byte aligned, [N][n_q_heads*head_dim].  workspace: DEVICE,
 * 256-byte aligned, ws_bytes >= ds_blocked_attention_workspace_size. */
ds_status ds_blocked_attention(const ds_ragged_meta* meta, const ds_attn_params* params,
                               const ds_rope_table* rope, const void* qkv,
                               const ds_kv_pool* pool, void* out, void* workspace,
                               size_t ws_bytes, void* stream);

/* ------------------------------------------------- fused append+attention -- */

/* The append and the attention of one batch in as few launches as the batch
 * allows.  This is operator fusion as "Principle: Deepspeedai DeepSpeed Inference Engine
 * Init" (leeroopedia), section "Theoretical Basis", describes it: fewer, larger
 * kernels cut launch overhead and the round trip of intermediates.  The
 * RoPE-and-append of each new token happens inside an attention kernel, so a
 * call is at most two launches and no separate append kernel runs.
 *
 * Results: exactly those of ds_kv_rotary_append(meta, params, rope, qkv, NULL,
 * pool) followed by ds_blocked_attention on the same stream: the same pool
 * contents and the same output bits.
 * Launches:
 *  - prefill tiles: the prefill kernel, launched cooperatively, first appends
 *    the prefill chunks' new K/V (a prologue over all its CTAs), meets at a
 *    grid barrier, then computes its tiles.
 *  - decode rows: the decode kernel appends each row's new K/V in the split
 *    that holds the row's last KV block, before that block is read, and merges
 *    the split partials of each (row, KV head) in the CTA that finishes last.
 *    Only a decode-only batch on the CUDA-core kernel with a grid above two
 *    waves (n_decode_items * n_kv_heads > 6 * SMs) merges in a separate
 *    kernel instead, which costs less there.
 *  So a batch is 1 launch (prefill only, or decode only) or 2.
 *
 * Workspace: DEVICE, 256-byte aligned, ws_bytes >= ds_fused_workspace_size for
 * the meta object's capacities.  It starts with one int32 counter per
 * (sequence slot, KV head), which must be zero when a call starts; every call
 * that completes without a device error leaves them zero.  Zero them once with
 * ds_fused_workspace_init before the first call, and again after any call that
 * set a bit in the device error word (a CTA that stops early never counts
 * itself done).  The rest holds split partials, as for ds_blocked_attention.
 * Errors: those of ds_kv_rotary_append and ds_blocked_attention. */
ds_status ds_fused_workspace_size(const ds_attn_params* params, int32_t max_seqs, int32_t max_tokens,
                                  int32_t max_blocks, size_t* bytes);
/* Enqueue the zeroing of the workspace's counters (meta gives the capacity). */
ds_status ds_fused_workspace_init(const ds_ragged_meta* meta, const ds_attn_params* params,
                                  void* workspace, size_t ws_bytes, void* stream);
ds_status ds_fused_append_attention(const ds_ragged_meta* meta, const ds_attn_params* params,
                                    const ds_rope_table* rope, const void* qkv,
                                    const ds_kv_pool* pool, void* out, void* workspace,
                                    size_t ws_bytes, void* stream);

/* Allocation-free variant of ds_blocked_attention.  (The source pages have no
 * counterpart: this entry point exists for callers that cannot allocate.)
 *
 * ds_blocked_attention needs a caller-provided workspace for the partial
 * results of split decode rows.  Some callers cannot obtain one: a plugin
 * loaded into a host application that owns all device memory through its own
 * allocator and hands the plugin no way to allocate; a latency-critical loop
 * in which a cudaMalloc, which may synchronize the device, is not acceptable;
 * a deployment that reserves a fixed device-memory budget at start-up and may
 * not allocate afterwards.  This entry point takes the same inputs and
 * outputs (the caller still passes qkv, the pool and out) but keeps the split
 * partials in a scratch array compiled into the library instead of a
 * workspace argument.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 * Limits and behaviour:
 *  - The scratch array is DS_STATIC_WORKSPACE_BYTES (32 MiB) of device memory,
 *    held on every GPU that loads the library until the process exits.  A
 *    batch whose split partials need more (4 * (P + n_decode_items *
 *    n_q_heads * head_dim) bytes, P = 2 * n_decode_items * n_q_heads rounded
 *    up to a multiple of 64) is rejected with DS_ERR_WORKSPACE before
 *    anything is enqueued.
 *  - The first call on each device (with that device current) looks up the
 *    array's device address once; make that first call before any stream
 *    capture begins.  The address stays cached for the life of the process:
 *    after cudaDeviceReset (or anything else that destroys and re-creates
 *    the device's primary context) it is stale, so do not call this entry
 *    point again in that process.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents.  Nothing in it has to start at zero (every partial is written
 *    before it is read), so it is never cleared.  Calls whose work overlaps
 *    on the GPU (different streams, or several host threads) race on the
 *    array: the caller must order them, e.g. on one stream.
 * Arguments, errors and results are otherwise those of ds_blocked_attention. */
#define DS_STATIC_WORKSPACE_BYTES ((size_t)32 << 20)
ds_status ds_blocked_attention_static_ws(const ds_ragged_meta* meta, const ds_attn_params* params,
                                         const ds_rope_table* rope, const void* qkv,
                                         const ds_kv_pool* pool, void* out, void* stream);

/* Wait for `stream` and read the device error word of the last batch built in
 * *meta (0 = none; DS_DEVERR_* bits otherwise). */
ds_status ds_get_device_error(const ds_ragged_meta* meta, int32_t* err, void* stream);

/* ------------------------------------------------- KV offload / restore -- */

/* BlockedKVCache offload and restore ("DeepSpeed Inference v2",
 * pyshine.com/deepspeed-2, section "The front desk": offload copies chosen
 * blocks to host memory to free device room, restore brings them back when
 * their sequence is rescheduled).  One block = all of its K and V tiles,
 * 2*n_kv_heads*block_size*head_dim storage elements, contiguous in the pool. */
ds_status ds_kv_block_bytes(const ds_attn_params* params, size_t* bytes);

/* Copy pool blocks block_ids[0..n) (HOST array, read during the call) into
 * host_dst[i*block_bytes ...] with one kernel per 1000 blocks that writes the
 * page-locked host buffer directly (no staging copy).  host_dst: page-locked
 * (pinned) host memory the device can address, n*block_bytes, 16-byte aligned;
 * DS_ERR_INVALID_ARG otherwise.  Ids outside the pool: DS_ERR_BAD_BLOCK before
 * anything is enqueued. */
ds_status ds_kv_offload(const ds_attn_params* params, const ds_kv_pool* pool,
                        const int32_t* block_ids, int32_t n, void* host_dst, void* stream);

/* The reverse: host_src[i*block_bytes ...] -> pool block block_ids[i].  An id
 * listed twice is DS_ERR_BAD_BLOCK (two sources for one block). */
ds_status ds_kv_restore(const ds_attn_params* params, const ds_kv_pool* pool,
                        const int32_t* block_ids, int32_t n, const void* host_src, void* stream);

/* ----------------------------------------- ragged embedding / logits rows -- */

/* RaggedEmbeddingKernel of the pages ("DeepSpeed Inference v2", section
 * "Ragged batches"): out[t] = table[token_ids[t]] for the batch's packed tokens
 * t < meta->n_tokens.  token_ids: DEVICE int32 [n_tokens]; table: DEVICE
 * [vocab][hidden]; out: DEVICE [n_tokens][hidden]; elements of elem_bytes (2 or
 * 4) bytes; hidden*elem_bytes a multiple of 16 and the pointers 16-byte
 * aligned (DS_ERR_UNSUPPORTED / DS_ERR_INVALID_ARG otherwise).  An id outside
 * [0, vocab) sets DS_DEVERR_TOKEN and writes a zero row. */
ds_status ds_ragged_embedding(const ds_ragged_meta* meta, const int32_t* token_ids,
                              const void* table, int32_t vocab, int32_t hidden, int32_t elem_bytes,
                              void* out, void* stream);

/* RaggedLogitsGather of the pages: out[i] = hidden_states[last packed token of
 * sequence i] (cu_seqlens[i+1] - 1) for i < meta->n_seqs.  hidden_states:
 * DEVICE [n_tokens][hidden]; out: DEVICE [n_seqs][hidden]; same element and
 * alignment rules as ds_ragged_embedding. */
ds_status ds_ragged_logits_gather(const ds_ragged_meta* meta, const void* hidden_states,
                                  int32_t hidden, int32_t elem_bytes, void* out, void* stream);

/* ------------------------------------------------------------ block ledger -- */

/* Host-side ledger of KV-pool block ids (the BlockedAllocator of "DeepSpeed
 * Inference v2", pyshine.com/deepspeed-2, section "The front desk": allocate
 * hands out free indices, free takes them back; the allocator is the whole
 * memory manager, so running out or freeing an id twice is an error, never
 * hidden).  HOST memory only; no CUDA call.  The caller owns both arrays:
 * stack[num_blocks] (free ids) and state[num_blocks] (1 = in use). */
typedef struct ds_block_allocator {
    int32_t* stack;
    uint8_t* state;
    int32_t num_blocks;
    int32_t n_free;
} ds_block_allocator;

/* All blocks free.  initial_order (num_blocks ids, a permutation; NULL = 0, 1,
 * ...) is the order in which allocate hands them out.  DS_ERR_INVALID_ARG on
 * NULL arrays or a non-permutation. */
ds_status ds_block_allocator_init(ds_block_allocator* a, int32_t* stack, uint8_t* state,
                                  int32_t num_blocks, const int32_t* initial_order);

/* Take n free ids into out[n] (DS_ERR_CAPACITY, nothing taken, if fewer than n
 * are free). */
ds_status ds_block_allocator_allocate(ds_block_allocator* a, int32_t n, int32_t* out);

/* Return n ids.  DS_ERR_BAD_BLOCK (nothing returned) if an id is outside the
 * pool, not in use, or listed twice. */
ds_status ds_block_allocator_free(ds_block_allocator* a, const int32_t* ids, int32_t n);

/* Extra blocks a sequence that owns `owned` blocks needs before `new_tokens`
 * more tokens are appended after `seen_tokens` (get_kv_requirements /
 * extend_kv_cache of the pages): max(0, ceil((seen+new)/block_size) - owned). */
ds_status ds_kv_blocks_required(int32_t seen_tokens, int32_t new_tokens, int32_t owned,
                                int32_t block_size, int32_t* extra);

/* ------------------------------------------------------ SplitFuse planner -- */

/* Host-side Dynamic SplitFuse pass planner over the block ledger ("DeepSpeed-
 * Inference and DeepSpeed-MII", tutorial ch. 10, sections 10.3 and 10.10:
 * prefill chunks and single-token decodes merged into one batch under a token
 * budget; "DeepSpeed Inference v2", section "The front desk": blocks are
 * reserved from the allocator before a pass and returned when a sequence is
 * flushed).  HOST memory only; no CUDA call; the state lives in caller memory
 * of ds_splitfuse_mem_size bytes.
 *
 * A pass packs, in arrival order, one token for every request that has
 * finished its prompt and still has tokens to generate, then prompt chunks
 * of the requests still prefilling, until the token budget or max_seqs is
 * reached.  A request whose extra blocks the ledger cannot supply waits for a
 * later pass.  A request is done once its prompt is in the cache and
 * `decode` decode passes have run; commit flushes it. */
typedef struct ds_splitfuse {
    void* mem;                      /* caller memory (8-byte aligned)           */
    size_t mem_bytes;
    int32_t max_requests;           /* requests tracked at once                 */
    int32_t max_blocks_per_request; /* ceil((prompt + decode)/block_size) bound */
    int32_t token_budget;           /* tokens per pass                          */
    int32_t max_seqs;               /* sequences per pass                       */
    int32_t block_size;
    int32_t n_active;               /* requests not yet flushed                 */
    int32_t n_planned;              /* sequences in the pass awaiting commit    */
} ds_splitfuse;

ds_status ds_splitfuse_mem_size(int32_t max_requests, int32_t max_blocks_per_request, size_t* bytes);
/* Empty planner.  DS_ERR_INVALID_ARG on bad sizes or NULL memory,
 * DS_ERR_WORKSPACE if mem_bytes is below ds_splitfuse_mem_size. */
ds_status ds_splitfuse_init(ds_splitfuse* p, void* mem, size_t mem_bytes, int32_t max_requests,
                            int32_t max_blocks_per_request, int32_t token_budget, int32_t max_seqs,
                            int32_t block_size);
/* Queue a request (prompt >= 1 tokens, then decode >= 0 generated tokens).
 * DS_ERR_CAPACITY if max_requests are active or the request would need more
 * than max_blocks_per_request blocks; DS_ERR_INVALID_ARG for bad counts or a
 * uid that is already active. */
ds_status ds_splitfuse_add(ds_splitfuse* p, int32_t uid, int32_t prompt, int32_t decode);
/* Plan the next pass: reserves blocks from `alloc`, writes up to max_seqs
 * descriptors to descs[] and their uids to uids[] (*n_out of them).
 * descs[i].block_ids points into planner memory and stays valid until the
 * next ds_splitfuse_commit.  DS_ERR_INVALID_ARG if the previous pass was not
 * committed.  When the ledger cannot supply any request's blocks the pass is
 * empty (*n_out == 0) while requests stay active; the caller frees blocks
 * (or stops) before planning again. */
ds_status ds_splitfuse_next(ds_splitfuse* p, ds_block_allocator* alloc, ds_seq_desc* descs,
                            int32_t* uids, int32_t* n_out);
/* The planned pass ran: advance its sequences and flush the finished requests
 * (their blocks go back to `alloc`; their uids, in arrival order, to
 * flushed[] -- room for max_requests -- and *n_flushed).  If the ledger
 * rejects a returned block (it no longer matches this planner: another party
 * freed or re-used the block), the ledger's status is returned and the
 * planner must be initialised again. */
ds_status ds_splitfuse_commit(ds_splitfuse* p, ds_block_allocator* alloc, int32_t* flushed,
                              int32_t* n_flushed);

/* Library version string. */
const char* ds_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DS_RAGGED_H */
