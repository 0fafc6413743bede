// prefill_mma.cu -- blocked causal attention for prefill chunks, warp-level
// tensor-core version (mma.sync m16n8k16, fp32 accumulation).
//
// A work atom is (tile of up to 64/G new tokens of one sequence, KV head c):
// its 64 rows are the tile's tokens x the G query heads that share KV head c,
// so every K/V tile staged in shared memory serves all G heads.  The atom
// walks the sequence's KV blocks 0 .. ceil(kv_len/64)-1 through the block
// table, 64 keys (one pool block) at a time, with an fp32 online softmax and
// the causal mask applied only on blocks that reach past the tile's first
// position ("DeepSpeed Inference v2", pyshine.com/deepspeed-2, section
// "Ragged batches": AtomBuilder atoms, BlockedFlashAttn, q-block size chosen
// per head size; "DeepSpeed-Inference and DeepSpeed-MII", ch. 10, section 10.3:
// FlashAttention-2 integration).  The query is rotated on load with the same
// fp32 rule as the KV append and rounded to the storage type.
#include "common.cuh"

namespace dsr {

namespace {

// Copies 16 bytes, or writes 16 zero bytes when `valid` is false (slots past a
// sequence's length may hold anything, and 0 * NaN would poison P*V).
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if (BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `ch` of row `r` in a [rows][D] tile whose
// chunks are XOR-swizzled by the row's low 3 bits (conflict-free ldmatrix).
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int ch) {
  return (uint32_t)(r * (D * 2) + ((ch ^ (r & 7)) << 4));
}

}  // namespace

template <bool BF16, bool HALF, int D, int G>
__global__ void __launch_bounds__(128) prefill_mma_kernel(
    const int4* __restrict__ tiles, const int32_t* __restrict__ cu_seqlens,
    const int32_t* __restrict__ seq_seen, const int32_t* __restrict__ blk_off,
    const int32_t* __restrict__ block_table, const uint16_t* __restrict__ qkv,
    const uint16_t* __restrict__ pool, uint16_t* __restrict__ out, LayerArgs a) {
  constexpr int ROWS = kPrefillRows;      // 64
  constexpr int T = ROWS / G;             // tokens per tile
  constexpr int CPR = D / 8;              // 16-byte chunks per row
  constexpr int TILE = kBlockSize * D * 2;  // bytes of a [64][D] tile
  constexpr int KS = D / 16;              // k-steps over the head dim
  constexpr int NT_O = D / 8;             // output n-tiles
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sQ = smem;                     // [64][D]
  uint8_t* sKV = smem + TILE;             // [2 stages][K, V][64][D]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int4 tl = tiles[blockIdx.x];
  const int seq = tl.x, j0 = tl.y, ntok = tl.z, kv_len = tl.w;
  const int c = blockIdx.y;
  const int s_seen = seq_seen[seq];
  const int tok0 = cu_seqlens[seq] + j0;
  const int W = (a.Hq + 2 * a.Hkv) * D;
  const int* btab = block_table + blk_off[seq];
  const int nb = (kv_len + kBlockSize - 1) / kBlockSize;
  const int pos_first = s_seen + j0;
  if (ntok <= 0 || ntok > T || kv_len != pos_first + ntok) {
    if (tid == 0) set_dev_error(a.header, DS_DEVERR_WORKLIST);
    return;
  }
  if (kv_len > a.max_positions) {
    if (tid == 0) set_dev_error(a.header, DS_DEVERR_POSITION);
    return;
  }

  auto load_kv = [&](int b, int stage) {
    int blk = btab[b];
    if (blk < 0 || blk >= a.num_blocks) {
      if (tid == 0) set_dev_error(a.header, DS_DEVERR_BLOCK_ID);
      blk = 0;
    }
    const uint8_t* kt = reinterpret_cast<const uint8_t*>(
        pool + (((int64_t)blk * 2 + 0) * a.Hkv + c) * (int64_t)(kBlockSize * D));
    const uint8_t* vt = kt + (int64_t)a.Hkv * kBlockSize * D * 2;
    uint8_t* dk = sKV + stage * 2 * TILE;
    uint8_t* dv = dk + TILE;
    const int valid_rows = kv_len - b * kBlockSize;
#pragma unroll
    for (int i = tid; i < kBlockSize * CPR; i += 128) {
      const int r = i / CPR, ch = i % CPR;
      cp_async16_zfill(dk + swz<D>(r, ch), kt + i * 16, r < valid_rows);
      cp_async16_zfill(dv + swz<D>(r, ch), vt + i * 16, r < valid_rows);
    }
  };

  load_kv(0, 0);
  cp_async_commit();

  // ---- Q tile: rotate rows on load, round to the storage type, swizzle.
  {
    const float4* rope4 = reinterpret_cast<const float4*>(a.rope);
    for (int u = tid; u < ROWS * (D / 16); u += 128) {
      const int r = u / (D / 16), cc = u % (D / 16);
      const int j = r / G, hh = c * G + r % G;
      const int ch0 = HALF ? cc : 2 * cc;
      const int ch1 = HALF ? CPR / 2 + cc : 2 * cc + 1;
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
      if (j < ntok) {
        const uint16_t* src = qkv + (int64_t)(tok0 + j) * W + hh * D;
        x0 = ld_nc_v4(src + 8 * ch0);
        x1 = ld_nc_v4(src + 8 * ch1);
        const int p = pos_first + j;
        float4 cs[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) cs[q] = __ldg(rope4 + (int64_t)p * (D / 4) + 4 * cc + q);
        rotate16<BF16, HALF>(x0, x1, cs);
      }
      *reinterpret_cast<uint4*>(sQ + swz<D>(r, ch0)) = x0;
      *reinterpret_cast<uint4*>(sQ + swz<D>(r, ch1)) = x1;
    }
  }
  __syncthreads();

  uint32_t qf[KS][4];
  {
    const int r = warp * 16 + (lane & 15);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      ldsm_x4(smem_u32(sQ + swz<D>(r, 2 * ks + (lane >> 4))), qf[ks][0], qf[ks][1], qf[ks][2],
              qf[ks][3]);
  }

  // rows this thread owns in the MMA fragments and their positions
  const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
  const int pos0 = pos_first + min(r0 / G, ntok - 1);
  const int pos1 = pos_first + min(r1 / G, ntok - 1);

  float o[NT_O][4];
#pragma unroll
  for (int i = 0; i < NT_O; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -1.0e30f, m1 = -1.0e30f, l0 = 0.f, l1 = 0.f;

  for (int b = 0; b < nb; ++b) {
    const int stage = b & 1;
    if (b + 1 < nb) {
      load_kv(b + 1, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint8_t* sK = sKV + stage * 2 * TILE;
    const uint8_t* sV = sK + TILE;

    float sc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = 16 * np + (lane & 7) + ((lane >> 4) << 3);
        const int ch = 2 * ks + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(sK + swz<D>(key, ch)), b0, b1, b2, b3);
        mma16816<BF16>(sc[2 * np], qf[ks], b0, b1);
        mma16816<BF16>(sc[2 * np + 1], qf[ks], b2, b3);
      }
    }
    // scale into log2 units; causal mask where the block reaches past the
    // tile's first position
    const int kbase = b * kBlockSize;
    const bool need_mask = kbase + kBlockSize - 1 > pos_first;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sc[nt][e] * a.scale_log2;
        if (need_mask) {
          const int key = kbase + 8 * nt + 2 * (lane & 3) + (e & 1);
          const int pos = e < 2 ? pos0 : pos1;
          if (key > pos) v = -INFINITY;
        }
        sc[nt][e] = v;
      }
    }
    float mx0 = m0, mx1 = m1;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
    }
#pragma unroll
    for (int mask = 1; mask <= 2; mask <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, mask));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, mask));
    }
    const float al0 = fast_exp2(m0 - mx0), al1 = fast_exp2(m1 - mx1);
    m0 = mx0;
    m1 = mx1;
    float rs0 = 0.f, rs1 = 0.f;
    uint32_t pf[4][4];  // P as A fragments, 4 k-steps of 16 keys
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = fast_exp2(sc[nt][0] - m0), p1 = fast_exp2(sc[nt][1] - m0);
      const float p2 = fast_exp2(sc[nt][2] - m1), p3 = fast_exp2(sc[nt][3] - m1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      pf[nt >> 1][(nt & 1) * 2 + 0] = Stor<BF16>::pack(p0, p1);
      pf[nt >> 1][(nt & 1) * 2 + 1] = Stor<BF16>::pack(p2, p3);
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int i = 0; i < NT_O; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al0;
      o[i][2] *= al1;
      o[i][3] *= al1;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int key = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int ch = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(sV + swz<D>(key, ch)), b0, b1, b2, b3);
        mma16816<BF16>(o[2 * dp], pf[kk], b0, b1);
        mma16816<BF16>(o[2 * dp + 1], pf[kk], b2, b3);
      }
    }
    __syncthreads();  // the stage is free for the load issued next iteration
  }

#pragma unroll
  for (int mask = 1; mask <= 2; mask <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, mask);
    l1 += __shfl_xor_sync(0xffffffffu, l1, mask);
  }
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int j_0 = r0 / G, j_1 = r1 / G;
  uint16_t* out0 = out + (int64_t)(tok0 + j_0) * a.Hq * D + (c * G + r0 % G) * D;
  uint16_t* out1 = out + (int64_t)(tok0 + j_1) * a.Hq * D + (c * G + r1 % G) * D;
#pragma unroll
  for (int nt = 0; nt < NT_O; ++nt) {
    const int dim = 8 * nt + 2 * (lane & 3);
    if (j_0 < ntok)
      *reinterpret_cast<uint32_t*>(out0 + dim) = Stor<BF16>::pack(o[nt][0] * inv0, o[nt][1] * inv0);
    if (j_1 < ntok)
      *reinterpret_cast<uint32_t*>(out1 + dim) = Stor<BF16>::pack(o[nt][2] * inv1, o[nt][3] * inv1);
  }
}

template <bool BF16, bool HALF, int D, int G>
static cudaError_t launch_prefill_t(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                    const void* pool, void* out, cudaStream_t st) {
  constexpr int SMEM = 5 * kBlockSize * D * 2;  // Q + 2 stages of K, V
  auto kern = prefill_mma_kernel<BF16, HALF, D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(m.n_prefill_tiles, a.Hkv);
  kern<<<grid, 128, SMEM, st>>>(reinterpret_cast<const int4*>(m.prefill_tiles), m.cu_seqlens,
                                m.seq_seen, m.blk_off, m.block_table,
                                static_cast<const uint16_t*>(qkv), static_cast<const uint16_t*>(pool),
                                static_cast<uint16_t*>(out), a);
  return cudaGetLastError();
}

template <bool BF16, bool HALF, int D>
static cudaError_t launch_prefill_g(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                    const void* pool, void* out, cudaStream_t st) {
  switch (a.G) {
    case 1: return launch_prefill_t<BF16, HALF, D, 1>(m, a, qkv, pool, out, st);
    case 2: return launch_prefill_t<BF16, HALF, D, 2>(m, a, qkv, pool, out, st);
    case 4: return launch_prefill_t<BF16, HALF, D, 4>(m, a, qkv, pool, out, st);
    case 8: return launch_prefill_t<BF16, HALF, D, 8>(m, a, qkv, pool, out, st);
    default: return cudaErrorInvalidValue;
  }
}

template <bool BF16, bool HALF>
static cudaError_t launch_prefill_d(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                    const void* pool, void* out, cudaStream_t st) {
  return a.D == 128 ? launch_prefill_g<BF16, HALF, 128>(m, a, qkv, pool, out, st)
                    : launch_prefill_g<BF16, HALF, 64>(m, a, qkv, pool, out, st);
}

cudaError_t launch_prefill(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                           const void* pool, void* out, cudaStream_t st) {
  const bool half = a.style == DS_ROPE_HALF;
  if (a.dtype == DS_BF16)
    return half ? launch_prefill_d<true, true>(m, a, qkv, pool, out, st)
                : launch_prefill_d<true, false>(m, a, qkv, pool, out, st);
  return half ? launch_prefill_d<false, true>(m, a, qkv, pool, out, st)
              : launch_prefill_d<false, false>(m, a, qkv, pool, out, st);
}

}  // namespace dsr
