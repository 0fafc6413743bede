// ledger.cpp -- host ledger of KV-pool block ids (BlockedAllocator of
// "DeepSpeed Inference v2", pyshine.com/deepspeed-2, section "The front desk":
// allocate returns free indices, free takes them back, and an overflow or a
// double free is an error, never hidden).  Plain host C++; no CUDA call.
#include <cstdio>
#include <vector>

#include "common.cuh"

extern "C" {

ds_status ds_block_allocator_init(ds_block_allocator* a, int32_t* stack, uint8_t* state,
                                  int32_t num_blocks, const int32_t* initial_order) {
  if (!a || num_blocks < 0 || (num_blocks > 0 && (!stack || !state))) {
    dsr::set_last_error("allocator, arrays or size invalid");
    return DS_ERR_INVALID_ARG;
  }
  if (initial_order) {
    std::vector<uint8_t> seen((size_t)num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      const int32_t id = initial_order[i];
      if (id < 0 || id >= num_blocks || seen[id]) {
        dsr::set_last_error("initial_order is not a permutation of the pool's ids");
        return DS_ERR_INVALID_ARG;
      }
      seen[id] = 1;
    }
  }
  a->stack = stack;
  a->state = state;
  a->num_blocks = num_blocks;
  a->n_free = num_blocks;
  // the top of the stack (index n_free - 1) is handed out first
  for (int32_t i = 0; i < num_blocks; ++i) {
    stack[num_blocks - 1 - i] = initial_order ? initial_order[i] : i;
    state[i] = 0;
  }
  return DS_OK;
}

ds_status ds_block_allocator_allocate(ds_block_allocator* a, int32_t n, int32_t* out) {
  if (!a || n < 0 || (n > 0 && !out)) {
    dsr::set_last_error("allocator or output invalid");
    return DS_ERR_INVALID_ARG;
  }
  if (n > a->n_free) {
    char msg[128];
    std::snprintf(msg, sizeof msg, "%d blocks requested, %d free", n, a->n_free);
    dsr::set_last_error(msg);
    return DS_ERR_CAPACITY;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = a->stack[--a->n_free];
    a->state[id] = 1;
    out[i] = id;
  }
  return DS_OK;
}

ds_status ds_block_allocator_free(ds_block_allocator* a, const int32_t* ids, int32_t n) {
  if (!a || n < 0 || (n > 0 && !ids)) {
    dsr::set_last_error("allocator or ids invalid");
    return DS_ERR_INVALID_ARG;
  }
  // validate everything first so that a bad list changes nothing
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= a->num_blocks || a->state[id] != 1) {
      char msg[128];
      std::snprintf(msg, sizeof msg, "block %d is outside the pool or not in use", id);
      dsr::set_last_error(msg);
      for (int32_t j = 0; j < i; ++j) a->state[ids[j]] = 1;  // undo the marks below
      return DS_ERR_BAD_BLOCK;
    }
    a->state[id] = 2;  // marked: catches an id listed twice
  }
  for (int32_t i = 0; i < n; ++i) {
    a->state[ids[i]] = 0;
    a->stack[a->n_free++] = ids[i];
  }
  return DS_OK;
}

ds_status ds_kv_blocks_required(int32_t seen_tokens, int32_t new_tokens, int32_t owned,
                                int32_t block_size, int32_t* extra) {
  if (!extra || seen_tokens < 0 || new_tokens < 0 || owned < 0 || block_size <= 0) {
    dsr::set_last_error("invalid token counts or block size");
    return DS_ERR_INVALID_ARG;
  }
  const int64_t need = ((int64_t)seen_tokens + new_tokens + block_size - 1) / block_size;
  *extra = need > owned ? (int32_t)(need - owned) : 0;
  return DS_OK;
}

}  // extern "C"
