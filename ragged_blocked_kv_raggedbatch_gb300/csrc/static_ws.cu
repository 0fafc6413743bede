// static_ws.cu -- ds_blocked_attention_static_ws: blocked attention whose
// split-decode partials live in a scratch array compiled into the library, for
// callers that cannot allocate a workspace (see include/ds_ragged.h).
//
// The array below is a file-scope device variable.  In host code its name is
// only a host-side stand-in for the symbol, not a device address: a kernel
// handed that name would fault, or on systems where the GPU can reach host
// memory silently use the wrong memory.  Host code therefore looks the device
// address up with cudaGetSymbolAddress, once per device with that device
// current, and passes that pointer on.  No allocation happens anywhere here.
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kStaticBytes = DS_STATIC_WORKSPACE_BYTES;

static __device__ __align__(256) float g_static_ws[kStaticBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {};

// Device address of g_static_ws on the current device (looked up on the first
// call per device; later calls reuse it).
cudaError_t static_ws_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ws_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return e;
    g_ws_addr[dev] = p;
  }
  *out = g_ws_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" ds_status ds_blocked_attention_static_ws(const ds_ragged_meta* meta,
                                                    const ds_attn_params* params,
                                                    const ds_rope_table* rope, const void* qkv,
                                                    const ds_kv_pool* pool, void* out,
                                                    void* stream) {
  // Malformed arguments: let ds_blocked_attention report them.
  if (!meta || !params || params->n_q_heads <= 0 || params->head_dim <= 0 || meta->n_decode_items < 0)
    return ds_blocked_attention(meta, params, rope, qkv, pool, out, nullptr, 0, stream);
  const size_t need = (size_t)dsr::ws_partial_bytes(meta->n_decode_items, params->n_q_heads, params->head_dim);
  if (need > kStaticBytes) {
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "batch needs %zu bytes of split-decode scratch; the built-in array holds %zu "
                  "(use ds_blocked_attention with a workspace)",
                  need, kStaticBytes);
    dsr::set_last_error(msg);
    return DS_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  cudaError_t e = static_ws_address(&ws);
  if (e != cudaSuccess) {
    char msg[256];
    std::snprintf(msg, sizeof msg, "looking up the built-in scratch array: %s", cudaGetErrorString(e));
    dsr::set_last_error(msg);
    return DS_ERR_CUDA;
  }
  return ds_blocked_attention(meta, params, rope, qkv, pool, out, ws, kStaticBytes, stream);
}
