// common.cuh -- internal helpers shared by the library's kernels and host code.
//
// Nothing here is part of the C ABI (include/ds_ragged.h is).  The metadata
// layout constants below define how ds_ragged_meta_pack lays out the device
// buffer that the kernels read.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ds_ragged.h"

namespace dsr {

// ---------------------------------------------------------------- metadata --
// Header words of the device metadata buffer.
enum : int {
  HDR_ERR = 0,       // device error bits (DS_DEVERR_*), zero after every upload
  HDR_S = 1,
  HDR_N = 2,
  HDR_BLOCKS = 3,
  HDR_DEC_NEXT = 4,  // decode units handed out so far (tensor-core decode kernel)
  HDR_DEC_DONE = 5,  // its CTAs that finished; the last one zeroes both words
  // Counts the kernels read here rather than from launch arguments, so that
  // launches sized by the capacities serve any batch within them.
  HDR_PRE_TILES = 6,  // prefill tiles (atoms = tiles x KV heads)
  HDR_DEC_ITEMS = 7,  // decode split items
  HDR_DEC_SEQS = 8,   // decode rows
  HDR_SPLIT = 9,      // KV blocks per decode split
  HDR_PRE_CTAS = 10,  // CTAs of the prefill grid that work (0: one per SM)
  HDR_PRE_BAR = 11,   // fused prefill: CTAs past the append prologue
  HDR_PRE_DONE = 12,  // prefill CTAs finished; the last one zeroes 11, 12, 13
  HDR_PRE_NEXT = 13,  // prefill atoms handed out so far
  HDR_PRE_HG = 14,    // KV heads per group in the prefill atom order (0: all)
  HDR_WORDS = 16,
};

constexpr int kBlockSize = 64;        // tokens per KV block (only supported value)
constexpr int kPrefillRows = 256;     // rows (tokens x heads of one KV group) per prefill atom
constexpr int kMinSplitBlocks = 4;    // smallest decode split, in KV blocks
constexpr int kMaxSplitBlocks = 32;   // largest decode split, in KV blocks

// Upper bounds of the work lists for given capacities (tiles of up to 256/G
// tokens, splits of at least kMinSplitBlocks blocks).
inline int64_t max_prefill_tiles(int64_t max_seqs, int64_t max_tokens) { return max_seqs + max_tokens; }
inline int64_t max_decode_items(int64_t max_seqs, int64_t max_blocks) {
  return max_seqs + (max_blocks + kMinSplitBlocks - 1) / kMinSplitBlocks;
}

// Split-decode partials in a workspace: the (m, l) pairs [items][Hq][2],
// then o [items][Hq][D] from the next 256-byte boundary, so that the float4
// accesses to o stay 16-byte aligned for any item and head count.
__host__ __device__ constexpr int64_t ws_o_offset(int64_t n_items, int64_t Hq) {
  return (n_items * Hq * 2 + 63) / 64 * 64;
}
// Bytes of the partials of n_items split items.
__host__ __device__ constexpr int64_t ws_partial_bytes(int64_t n_items, int64_t Hq, int64_t D) {
  return (ws_o_offset(n_items, Hq) + n_items * Hq * D) * 4;
}

// Kernel arguments that every launch needs, resolved on the host.
struct LayerArgs {
  int32_t Hq, Hkv, D, G, dtype, style;
  float scale_log2;        // softmax scale * log2(e)
  int32_t num_blocks;      // pool size
  int32_t max_positions;   // rotary table rows
  const float2* rope;      // [max_positions][D/2]
  int32_t* header;         // device error word at header[HDR_ERR], counts at HDR_*
};

// ----------------------------------------------------------- device helpers --
#ifdef __CUDACC__

__device__ __forceinline__ void set_dev_error(int32_t* header, int bits) {
  atomicOr(reinterpret_cast<int*>(header + HDR_ERR), bits);
}

// Storage <-> fp32 (exact up-conversion; round-to-nearest-even down).
template <bool BF16> struct Stor;
template <> struct Stor<true> {
  __device__ __forceinline__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
  __device__ __forceinline__ static float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
  __device__ __forceinline__ static uint32_t pack(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
  }
};
template <> struct Stor<false> {
  __device__ __forceinline__ static float lo(uint32_t w) {
    float f;
    asm("{ .reg .f16 h; mov.b32 {h, _}, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(w));
    return f;
  }
  __device__ __forceinline__ static float hi(uint32_t w) {
    float f;
    asm("{ .reg .f16 h; mov.b32 {_, h}, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(w));
    return f;
  }
  __device__ __forceinline__ static uint32_t pack(float a, float b) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
  }
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Rotation of one pair in fp32 with every product and sum rounded separately
// (never contracted into a fused multiply-add):
//   y0 = x0*c - x1*s,  y1 = x1*c + x0*s.
__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, float& y0,
                                          float& y1) {
  y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
  y1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s));
}

// Rotate 8 pairs.  HALF: a holds x[8c..8c+7], b holds x[d/2+8c..]; the pair of
// element e is (a[e], b[e]) with table index 8c+e.  INTERLEAVED: a, b hold
// x[16c..16c+15]; pairs are adjacent elements, table index 8c + e.
template <bool BF16, bool HALF>
__device__ __forceinline__ void rotate16(uint4& a, uint4& b, const float4* cs /* 4 x float4 */) {
  uint32_t* A = reinterpret_cast<uint32_t*>(&a);
  uint32_t* B = reinterpret_cast<uint32_t*>(&b);
  float c[8], s[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float4 v = cs[q];
    c[2 * q] = v.x;
    s[2 * q] = v.y;
    c[2 * q + 1] = v.z;
    s[2 * q + 1] = v.w;
  }
  if (HALF) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float x0l = Stor<BF16>::lo(A[w]), x0h = Stor<BF16>::hi(A[w]);
      float x1l = Stor<BF16>::lo(B[w]), x1h = Stor<BF16>::hi(B[w]);
      float y0l, y1l, y0h, y1h;
      rope_pair(x0l, x1l, c[2 * w], s[2 * w], y0l, y1l);
      rope_pair(x0h, x1h, c[2 * w + 1], s[2 * w + 1], y0h, y1h);
      A[w] = Stor<BF16>::pack(y0l, y0h);
      B[w] = Stor<BF16>::pack(y1l, y1h);
    }
  } else {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float y0, y1;
      rope_pair(Stor<BF16>::lo(A[w]), Stor<BF16>::hi(A[w]), c[w], s[w], y0, y1);
      A[w] = Stor<BF16>::pack(y0, y1);
      rope_pair(Stor<BF16>::lo(B[w]), Stor<BF16>::hi(B[w]), c[4 + w], s[4 + w], y0, y1);
      B[w] = Stor<BF16>::pack(y0, y1);
    }
  }
}

// ------------------------------------------------ mbarrier + bulk async copy --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of phase `parity` (try_wait may suspend the thread for a
// while; a loop that polls several barriers must not).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after ~`limit_cycles` SM
// cycles (DSR_WAIT_LIMIT: ~2 s at GB300 clocks; a build with
// -DDSR_TEST_WAIT_RUNOUT shortens it to ~1 ms so that a test can make a wait
// run out quickly).  Returns false on timeout (the caller records an error and
// stops issuing work; it never spins forever).
#ifndef DSR_WAIT_LIMIT
#ifdef DSR_TEST_WAIT_RUNOUT
#define DSR_WAIT_LIMIT 2000000LL
#else
#define DSR_WAIT_LIMIT 4000000000LL
#endif
#endif
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit_cycles = DSR_WAIT_LIMIT) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit_cycles) return false;
  }
  return true;
}

// One bulk (non-tensor) global -> shared copy completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// One unit of the KV append for packed token t at position p (sequence block
// blk, slot off): units [0, Hkv*D/16) rotate 16 key elements (8 pairs) into
// the pool's K slot; units [Hkv*D/16, Hkv*(D/16 + D/8)) copy 8 value elements
// into its V slot.  row: the token's qkv row; cs_row: its rotary table row.
template <bool BF16, bool HALF, int D>
__device__ __forceinline__ void append_unit(int u, const uint16_t* row, const float4* cs_row,
                                            uint16_t* pool, int blk, int off, const LayerArgs& a) {
  constexpr int KU = D / 16, VU = D / 8;
  const int n_k = a.Hkv * KU;
  if (u < n_k) {
    const int h = u / KU, c = u % KU;
    const uint16_t* src = row + (a.Hq + h) * D;
    const int i0 = HALF ? 8 * c : 16 * c;
    const int i1 = HALF ? D / 2 + 8 * c : 16 * c + 8;
    uint4 x0 = ld_nc_v4(src + i0);
    uint4 x1 = ld_nc_v4(src + i1);
    float4 cs[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) cs[q] = __ldg(cs_row + 4 * c + q);  // pairs 8c..8c+7
    rotate16<BF16, HALF>(x0, x1, cs);
    uint16_t* dst = pool + ((((int64_t)blk * 2 + 0) * a.Hkv + h) * kBlockSize + off) * D;
    *reinterpret_cast<uint4*>(dst + i0) = x0;
    *reinterpret_cast<uint4*>(dst + i1) = x1;
  } else {
    const int uu = u - n_k;
    const int h = uu / VU, c = uu % VU;
    const uint4 v = ld_nc_v4(row + (a.Hq + a.Hkv + h) * D + 8 * c);
    *reinterpret_cast<uint4*>(pool + ((((int64_t)blk * 2 + 1) * a.Hkv + h) * kBlockSize + off) * D + 8 * c) = v;
  }
}

#endif  // __CUDACC__

// Records the message ds_last_error() returns on this thread (host.cpp).
void set_last_error(const char* msg);

// -------------------------------------------------------------- launchers --
// Implemented in the .cu files; called by the host layer after validation.
cudaError_t launch_rope_table(const ds_attn_params& p, int32_t max_positions, float2* table,
                              cudaStream_t st);
// Launches are sized by the batch's counts, or by the capacities when
// m.flags has DS_META_CAPACITY (the kernels read the batch's counts from the
// uploaded header and their surplus CTAs exit at once).
cudaError_t launch_append(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                          void* q_out, void* pool, cudaStream_t st);
// overlap_previous: launch as a programmatic dependent of the kernel before it
// on the stream (the prefill kernel), so decode CTAs can start while it runs.
// fused_append: the kernel also appends each decode row's new K/V (the append
// kernel then skips decode rows).  counters == nullptr: split partials are
// merged by a separate combine launch; counters != nullptr (fused_append only;
// zero on entry, zero again on exit): the last split CTA of every (row, KV
// head) merges them.
cudaError_t launch_decode(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                          const void* pool, void* out, float* ws, cudaStream_t st,
                          bool overlap_previous, bool fused_append = false,
                          int32_t* counters = nullptr);
// True when launch_decode runs the layer's decode rows on the tensor-core kernel.
bool decode_on_tensor_cores(const LayerArgs& a);
// Decode rows of grouped-query layers (G >= 2, D = 128) on the tensor cores;
// the same arguments and results as launch_decode (decode_tc.cu).
cudaError_t launch_decode_tc(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                             const void* pool, void* out, float* ws, cudaStream_t st,
                             bool overlap_previous, bool fused_append, int32_t* counters);
// The merge of the split partials of multi-split decode rows (decode.cu).
cudaError_t launch_decode_combine(const ds_ragged_meta& m, const LayerArgs& a, const float* ws,
                                  void* out, cudaStream_t st);
// fused_append: the prefill CTAs first append the prefill chunks' new K/V
// (rotated) to the pool, meet at a grid barrier (cooperative launch), then run
// the atoms; decode rows are left to the fused decode kernel.
cudaError_t launch_prefill(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                           void* pool, void* out, cudaStream_t st, bool fused_append = false);

}  // namespace dsr
