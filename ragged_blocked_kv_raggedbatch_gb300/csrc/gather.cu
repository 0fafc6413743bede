// gather.cu -- data movement around the attention layer: KV block offload /
// restore between the pool and page-locked host memory, and the ragged
// embedding / last-token logits row gathers.
//
// "DeepSpeed Inference v2" (pyshine.com/deepspeed-2): section "The front
// desk" (BlockedKVCache offload copies chosen blocks to host memory, restore
// brings them back) and section "Ragged batches" (RaggedEmbeddingKernel gathers
// embedding rows for the packed token stream; RaggedLogitsGather copies only
// the last-token row of each sequence out for sampling).
//
// All copies move 16-byte vectors.  Offload/restore kernels read or write the
// host buffer directly through its device-visible address (over the CPU-GPU
// link on Grace-Blackwell), with the block ids passed as a kernel parameter.
#include <algorithm>
#include <vector>

#include "common.cuh"

namespace dsr {

constexpr int kIdsPerLaunch = 1000;
struct BlockIds {
  int32_t id[kIdsPerLaunch];
};

// grid (blocks in this launch, CTAs per block); each CTA moves a slice of one block.
template <bool TO_HOST>
__global__ void __launch_bounds__(256) kv_block_copy_kernel(uint4* __restrict__ pool,
                                                            uint4* __restrict__ host,
                                                            int64_t block_vec, int32_t first,
                                                            const __grid_constant__ BlockIds ids) {
  const int i = blockIdx.x;
  const int64_t blk = ids.id[i];
  uint4* p = pool + blk * block_vec;
  uint4* h = host + (int64_t)(first + i) * block_vec;
  const int64_t per = (block_vec + gridDim.y - 1) / gridDim.y;
  const int64_t beg = blockIdx.y * per, end = min(block_vec, beg + per);
  for (int64_t v = beg + threadIdx.x; v < end; v += blockDim.x) {
    if (TO_HOST)
      h[v] = p[v];
    else
      p[v] = h[v];
  }
}

cudaError_t launch_kv_block_copy(bool to_host, void* pool, void* host, size_t block_bytes,
                                 const int32_t* ids, int32_t n, cudaStream_t st) {
  const int64_t block_vec = (int64_t)(block_bytes / 16);
  const int slices = (int)std::max<int64_t>(1, std::min<int64_t>(16, block_vec / 4096));
  for (int32_t first = 0; first < n; first += kIdsPerLaunch) {
    const int32_t cnt = std::min(kIdsPerLaunch, n - first);
    BlockIds p;
    std::copy(ids + first, ids + first + cnt, p.id);
    dim3 grid(cnt, slices);
    if (to_host)
      kv_block_copy_kernel<true><<<grid, 256, 0, st>>>(static_cast<uint4*>(pool), static_cast<uint4*>(host),
                                                       block_vec, first, p);
    else
      kv_block_copy_kernel<false><<<grid, 256, 0, st>>>(static_cast<uint4*>(pool), static_cast<uint4*>(host),
                                                        block_vec, first, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// One CTA per output row.
__global__ void __launch_bounds__(128) embedding_kernel(const int32_t* __restrict__ token_ids,
                                                        const uint4* __restrict__ table,
                                                        uint4* __restrict__ out, int32_t vocab,
                                                        int32_t row_vec, int32_t* header) {
  const int t = blockIdx.x;
  const int id = token_ids[t];
  const bool ok = id >= 0 && id < vocab;
  if (!ok && threadIdx.x == 0) set_dev_error(header, DS_DEVERR_TOKEN);
  const uint4* src = table + (int64_t)(ok ? id : 0) * row_vec;
  uint4* dst = out + (int64_t)t * row_vec;
  for (int v = threadIdx.x; v < row_vec; v += blockDim.x) dst[v] = ok ? ld_nc_v4(src + v) : make_uint4(0, 0, 0, 0);
}

__global__ void __launch_bounds__(128) last_token_kernel(const int32_t* __restrict__ cu_seqlens,
                                                         const uint4* __restrict__ hidden,
                                                         uint4* __restrict__ out, int32_t row_vec) {
  const int i = blockIdx.x;
  const int t = cu_seqlens[i + 1] - 1;
  const uint4* src = hidden + (int64_t)t * row_vec;
  uint4* dst = out + (int64_t)i * row_vec;
  for (int v = threadIdx.x; v < row_vec; v += blockDim.x) dst[v] = ld_nc_v4(src + v);
}

cudaError_t launch_embedding(const ds_ragged_meta& m, const int32_t* ids, const void* table, int32_t vocab,
                             int32_t row_bytes, void* out, cudaStream_t st) {
  embedding_kernel<<<m.n_tokens, 128, 0, st>>>(ids, static_cast<const uint4*>(table), static_cast<uint4*>(out),
                                               vocab, row_bytes / 16, m.header);
  return cudaGetLastError();
}

cudaError_t launch_last_token(const ds_ragged_meta& m, const void* hidden, int32_t row_bytes, void* out,
                              cudaStream_t st) {
  last_token_kernel<<<m.n_seqs, 128, 0, st>>>(m.cu_seqlens, static_cast<const uint4*>(hidden),
                                              static_cast<uint4*>(out), row_bytes / 16);
  return cudaGetLastError();
}

}  // namespace dsr

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

ds_status params_ok(const ds_attn_params* p) {
  if (!p || p->n_kv_heads <= 0 || (p->head_dim != 64 && p->head_dim != 128) || p->block_size != 64 ||
      (p->dtype != DS_FP16 && p->dtype != DS_BF16)) {
    dsr::set_last_error("unsupported or missing params");
    return DS_ERR_UNSUPPORTED;
  }
  return DS_OK;
}

// Device-visible address of page-locked host memory, or nullptr.
const void* host_dev_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  return at.devicePointer;
}

ds_status kv_copy(bool to_host, const ds_attn_params* params, const ds_kv_pool* pool, const int32_t* ids,
                  int32_t n, const void* host, void* stream) {
  if (ds_status s = params_ok(params)) return s;
  if (!pool || !pool->base || !aligned16(pool->base) || n < 0 || (n > 0 && (!ids || !host))) {
    dsr::set_last_error("pool, ids or host buffer invalid");
    return DS_ERR_INVALID_ARG;
  }
  if (n == 0) return DS_OK;
  std::vector<uint8_t> seen((size_t)std::max(pool->num_blocks, 0), 0);
  for (int32_t i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= pool->num_blocks) {
      dsr::set_last_error("block id outside the pool");
      return DS_ERR_BAD_BLOCK;
    }
    if (!to_host && seen[ids[i]]) {
      dsr::set_last_error("a block id is listed twice for restore");
      return DS_ERR_BAD_BLOCK;
    }
    seen[ids[i]] = 1;
  }
  const void* hd = host_dev_ptr(host);
  if (!hd || !aligned16(hd)) {
    dsr::set_last_error("host buffer is not page-locked, device-visible and 16-byte aligned");
    return DS_ERR_INVALID_ARG;
  }
  size_t bb = 0;
  ds_kv_block_bytes(params, &bb);
  cudaError_t e = dsr::launch_kv_block_copy(to_host, pool->base, const_cast<void*>(hd), bb, ids, n,
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    dsr::set_last_error(cudaGetErrorString(e));
    return DS_ERR_CUDA;
  }
  return DS_OK;
}

ds_status rows_ok(const ds_ragged_meta* m, int32_t hidden, int32_t elem_bytes, const void* a, const void* b) {
  if (!m || !m->header || m->n_seqs < 0) {
    dsr::set_last_error("meta was not filled by ds_ragged_meta_build");
    return DS_ERR_INVALID_ARG;
  }
  if ((elem_bytes != 2 && elem_bytes != 4) || hidden <= 0 || ((int64_t)hidden * elem_bytes) % 16 != 0) {
    dsr::set_last_error("hidden * elem_bytes must be a positive multiple of 16 (elem_bytes 2 or 4)");
    return DS_ERR_UNSUPPORTED;
  }
  if (!a || !b || !aligned16(a) || !aligned16(b)) {
    dsr::set_last_error("buffers must be non-NULL and 16-byte aligned");
    return DS_ERR_INVALID_ARG;
  }
  return DS_OK;
}

}  // namespace

extern "C" {

ds_status ds_kv_block_bytes(const ds_attn_params* params, size_t* bytes) {
  if (ds_status s = params_ok(params)) return s;
  if (!bytes) {
    dsr::set_last_error("bytes is NULL");
    return DS_ERR_INVALID_ARG;
  }
  *bytes = (size_t)2 * params->n_kv_heads * params->block_size * params->head_dim * 2;
  return DS_OK;
}

ds_status ds_kv_offload(const ds_attn_params* params, const ds_kv_pool* pool, const int32_t* block_ids,
                        int32_t n, void* host_dst, void* stream) {
  return kv_copy(true, params, pool, block_ids, n, host_dst, stream);
}

ds_status ds_kv_restore(const ds_attn_params* params, const ds_kv_pool* pool, const int32_t* block_ids,
                        int32_t n, const void* host_src, void* stream) {
  return kv_copy(false, params, pool, block_ids, n, host_src, stream);
}

ds_status ds_ragged_embedding(const ds_ragged_meta* meta, const int32_t* token_ids, const void* table,
                              int32_t vocab, int32_t hidden, int32_t elem_bytes, void* out, void* stream) {
  if (ds_status s = rows_ok(meta, hidden, elem_bytes, table, out)) return s;
  if (!token_ids || vocab <= 0) {
    dsr::set_last_error("token_ids NULL or vocab <= 0");
    return DS_ERR_INVALID_ARG;
  }
  if (meta->n_tokens == 0) return DS_OK;
  cudaError_t e = dsr::launch_embedding(*meta, token_ids, table, vocab, hidden * elem_bytes, out,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    dsr::set_last_error(cudaGetErrorString(e));
    return DS_ERR_CUDA;
  }
  return DS_OK;
}

ds_status ds_ragged_logits_gather(const ds_ragged_meta* meta, const void* hidden_states, int32_t hidden,
                                  int32_t elem_bytes, void* out, void* stream) {
  if (ds_status s = rows_ok(meta, hidden, elem_bytes, hidden_states, out)) return s;
  if (meta->n_seqs == 0) return DS_OK;
  cudaError_t e = dsr::launch_last_token(*meta, hidden_states, hidden * elem_bytes, out,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    dsr::set_last_error(cudaGetErrorString(e));
    return DS_ERR_CUDA;
  }
  return DS_OK;
}

}  // extern "C"
