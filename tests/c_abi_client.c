/* A plain C program that drives one layer step through the C ABI alone
 * (include/ds_ragged.h + libds_ragged.so + the CUDA runtime; no Python).
 *
 *   c_abi_client batch.bin qkv.bin pool.bin out.bin pool_out.bin
 *
 * batch.bin (int32 words): n_q_heads, n_kv_heads, head_dim, dtype, rope_style,
 * n_seqs, pool blocks, rotary positions, rope_theta (float bits), then per
 * sequence: seen, new, n_ids, ids[n_ids].  qkv.bin / pool.bin: the storage
 * bytes of qkv [N][(Hq+2Hkv)*d] and of the pool.  Writes the attention output
 * and the pool after the append; prints "ok <version>" on success. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ds_ragged.h"

#define CK(x)                                                                        \
  do {                                                                               \
    ds_status s_ = (x);                                                              \
    if (s_ != DS_OK) {                                                               \
      fprintf(stderr, "%s failed: status %d: %s\n", #x, (int)s_, ds_last_error());   \
      return 1;                                                                      \
    }                                                                                \
  } while (0)
#define CU(x)                                                                        \
  do {                                                                               \
    cudaError_t e_ = (x);                                                            \
    if (e_ != cudaSuccess) {                                                         \
      fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));                \
      return 1;                                                                      \
    }                                                                                \
  } while (0)

static void* slurp(const char* path, size_t* n) {
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  fseek(f, 0, SEEK_END);
  long len = ftell(f);
  fseek(f, 0, SEEK_SET);
  void* buf = malloc(len > 0 ? (size_t)len : 1);
  if (buf && len > 0 && fread(buf, 1, (size_t)len, f) != (size_t)len) {
    free(buf);
    buf = NULL;
  }
  fclose(f);
  *n = (size_t)(len > 0 ? len : 0);
  return buf;
}

static int spill(const char* path, const void* buf, size_t n) {
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  int bad = fwrite(buf, 1, n, f) != n;
  return fclose(f) != 0 || bad;
}

int main(int argc, char** argv) {
  if (argc != 6) {
    fprintf(stderr, "usage: %s batch.bin qkv.bin pool.bin out.bin pool_out.bin\n", argv[0]);
    return 2;
  }
  size_t nb_batch = 0, nb_qkv = 0, nb_pool = 0;
  int32_t* w = (int32_t*)slurp(argv[1], &nb_batch);
  void* qkv_h = slurp(argv[2], &nb_qkv);
  void* pool_h = slurp(argv[3], &nb_pool);
  if (!w || !qkv_h || !pool_h || nb_batch < 9 * 4) {
    fprintf(stderr, "cannot read the inputs\n");
    return 1;
  }
  ds_attn_params p;
  memset(&p, 0, sizeof p);
  p.n_q_heads = w[0];
  p.n_kv_heads = w[1];
  p.head_dim = w[2];
  p.block_size = 64;
  p.dtype = w[3];
  p.rope_style = w[4];
  memcpy(&p.rope_theta, &w[8], 4);
  p.softmax_scale = 0.0f;
  const int32_t n_seqs = w[5], num_blocks = w[6], max_positions = w[7];

  ds_seq_desc* seqs = (ds_seq_desc*)calloc((size_t)(n_seqs > 0 ? n_seqs : 1), sizeof(ds_seq_desc));
  size_t at = 9;
  int32_t n_tokens = 0, n_used_blocks = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    seqs[i].seen_tokens = w[at];
    seqs[i].new_tokens = w[at + 1];
    seqs[i].n_blocks = w[at + 2];
    seqs[i].block_ids = &w[at + 3];
    at += 3 + (size_t)w[at + 2];
    n_tokens += seqs[i].new_tokens;
    n_used_blocks += (seqs[i].seen_tokens + seqs[i].new_tokens + 63) / 64;
  }

  cudaStream_t st;
  CU(cudaStreamCreate(&st));

  /* metadata buffers (device + pinned staging), sized by the library */
  size_t dev_b = 0, stg_b = 0;
  CK(ds_meta_buffer_sizes(n_seqs, n_tokens, n_used_blocks, &p, &dev_b, &stg_b));
  ds_ragged_meta meta;
  memset(&meta, 0, sizeof meta);
  memset(&meta, 0, sizeof meta);
  CU(cudaMalloc(&meta.device_buf, dev_b));
  CU(cudaMallocHost(&meta.host_staging, stg_b));
  meta.device_bytes = dev_b;
  meta.staging_bytes = stg_b;
  meta.max_seqs = n_seqs;
  meta.max_tokens = n_tokens;
  meta.max_blocks = n_used_blocks;

  /* rotary table */
  size_t rope_b = 0;
  CK(ds_rope_table_size(&p, max_positions, &rope_b));
  void* rope_buf = NULL;
  CU(cudaMalloc(&rope_buf, rope_b > 0 ? rope_b : 16));
  ds_rope_table rope;
  CK(ds_rope_table_build(&p, max_positions, rope_buf, rope_b, &rope, st));

  /* inputs on the device */
  void *qkv_d = NULL, *pool_d = NULL, *out_d = NULL, *ws_d = NULL;
  const size_t out_b = (size_t)n_tokens * (size_t)p.n_q_heads * (size_t)p.head_dim * 2;
  CU(cudaMalloc(&qkv_d, nb_qkv));
  CU(cudaMalloc(&pool_d, nb_pool));
  CU(cudaMalloc(&out_d, out_b > 0 ? out_b : 16));
  CU(cudaMemcpyAsync(qkv_d, qkv_h, nb_qkv, cudaMemcpyHostToDevice, st));
  CU(cudaMemcpyAsync(pool_d, pool_h, nb_pool, cudaMemcpyHostToDevice, st));
  ds_kv_pool pool;
  pool.base = pool_d;
  pool.num_blocks = num_blocks;

  /* one layer step: metadata upload, RoPE + KV append, attention */
  CK(ds_ragged_meta_build(seqs, n_seqs, &p, num_blocks, &meta, st));
  CK(ds_kv_rotary_append(&meta, &p, &rope, qkv_d, NULL, &pool, st));
  size_t ws_b = 0;
  CK(ds_blocked_attention_workspace_size(&p, n_seqs, n_tokens, n_used_blocks, &ws_b));
  CU(cudaMalloc(&ws_d, ws_b));
  CK(ds_blocked_attention(&meta, &p, &rope, qkv_d, &pool, out_d, ws_d, ws_b, st));
  int32_t dev_err = -1;
  CK(ds_get_device_error(&meta, &dev_err, st));
  if (dev_err != 0) {
    fprintf(stderr, "device error word %d\n", (int)dev_err);
    return 1;
  }

  void* out_h = malloc(out_b > 0 ? out_b : 1);
  void* pool_out_h = malloc(nb_pool);
  CU(cudaMemcpyAsync(out_h, out_d, out_b, cudaMemcpyDeviceToHost, st));
  CU(cudaMemcpyAsync(pool_out_h, pool_d, nb_pool, cudaMemcpyDeviceToHost, st));
  CU(cudaStreamSynchronize(st));
  if (spill(argv[4], out_h, out_b) || spill(argv[5], pool_out_h, nb_pool)) {
    fprintf(stderr, "cannot write the outputs\n");
    return 1;
  }
  printf("ok %s\n", ds_version());
  return 0;
}
