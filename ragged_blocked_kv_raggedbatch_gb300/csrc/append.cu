// append.cu -- rotary table and the rotary-embedding + KV-append kernel.
//
// The KV append scatters each new token's rotated keys and its values into the
// slot its sequence's block list assigns to its position ("DeepSpeed Inference
// v2", pyshine.com/deepspeed-2, sections "The front desk" and "Ragged
// batches": descriptors own integer block ids, kernels address the
// block-indexed pools directly).  HBM-bound: every access is a 16-byte vector.
#include "common.cuh"

namespace dsr {

// (cos, sin) of fp32(fp32(p) * fp32(theta^(-2k/d))), evaluated in fp64 and
// rounded to fp32.  One thread per (p, k).
__global__ void rope_table_kernel(float2* __restrict__ table, int32_t max_positions, int32_t half_d,
                                  float theta) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)max_positions * half_d) return;
  int32_t p = (int32_t)(i / half_d);
  int32_t k = (int32_t)(i % half_d);
  float fk = (float)pow((double)theta, -2.0 * (double)k / (double)(2 * half_d));
  float a = __fmul_rn((float)p, fk);
  double s, c;
  sincos((double)a, &s, &c);
  table[i] = make_float2((float)c, (float)s);
}

cudaError_t launch_rope_table(const ds_attn_params& p, int32_t max_positions, float2* table,
                              cudaStream_t st) {
  int64_t n = (int64_t)max_positions * (p.head_dim / 2);
  int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  rope_table_kernel<<<(unsigned)blocks, threads, 0, st>>>(table, max_positions, p.head_dim / 2,
                                                         p.rope_theta);
  return cudaGetLastError();
}

// One CTA per packed token (CTAs past the batch's token count, in launches
// sized by the capacities, exit at once).  Work units of a token:
//   [0, Hkv*D/16)            rotate 16 key elements (8 pairs) -> pool K slot
//   [.., + Hkv*D/8)          copy 8 value elements           -> pool V slot
//   [.., + Hq*D/16) (q_out)  rotate 16 query elements        -> q_out row
template <bool BF16, bool HALF, int D>
__global__ void __launch_bounds__(128) append_kernel(
    const int32_t* __restrict__ tok_seq, const int32_t* __restrict__ tok_pos,
    const int32_t* __restrict__ blk_off, const int32_t* __restrict__ block_table,
    const uint16_t* __restrict__ qkv, uint16_t* __restrict__ q_out, uint16_t* __restrict__ pool,
    LayerArgs a) {
  const int t = blockIdx.x;
  if (t >= a.header[HDR_N]) return;
  const int seq = tok_seq[t];
  const int p = tok_pos[t];
  const int W = (a.Hq + 2 * a.Hkv) * D;
  const uint16_t* row = qkv + (int64_t)t * W;
  if (p >= a.max_positions) {
    if (threadIdx.x == 0) set_dev_error(a.header, DS_DEVERR_POSITION);
    return;
  }
  const int blk = block_table[blk_off[seq] + p / kBlockSize];
  if (blk < 0 || blk >= a.num_blocks) {
    if (threadIdx.x == 0) set_dev_error(a.header, DS_DEVERR_BLOCK_ID);
    return;
  }
  const int off = p % kBlockSize;
  const float4* cs_row = reinterpret_cast<const float4*>(a.rope + (int64_t)p * (D / 2));
  constexpr int KU = D / 16;  // rotation units per head
  constexpr int VU = D / 8;   // copy units per head
  const int n_kv = a.Hkv * (KU + VU);
  const int n_q = q_out ? a.Hq * KU : 0;
  for (int u = threadIdx.x; u < n_kv + n_q; u += blockDim.x) {
    if (u < n_kv) {
      append_unit<BF16, HALF, D>(u, row, cs_row, pool, blk, off, a);
    } else {
      const int uu = u - n_kv;
      const int h = uu / KU, c = uu % KU;
      const uint16_t* src = row + h * D;
      const int i0 = HALF ? 8 * c : 16 * c;
      const int i1 = HALF ? D / 2 + 8 * c : 16 * c + 8;
      uint4 x0 = ld_nc_v4(src + i0);
      uint4 x1 = ld_nc_v4(src + i1);
      float4 cs[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) cs[q] = __ldg(cs_row + 4 * c + q);  // pairs 8c..8c+7
      rotate16<BF16, HALF>(x0, x1, cs);
      uint16_t* dst = q_out + (int64_t)t * a.Hq * D + h * D;
      *reinterpret_cast<uint4*>(dst + i0) = x0;
      *reinterpret_cast<uint4*>(dst + i1) = x1;
    }
  }
}

template <bool BF16, bool HALF>
static cudaError_t launch_append_t(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                   void* q_out, void* pool, cudaStream_t st) {
  const int n = (m.flags & DS_META_CAPACITY) ? m.max_tokens : m.n_tokens;
  if (n <= 0) return cudaSuccess;
  dim3 grid(n);
  if (a.D == 128)
    append_kernel<BF16, HALF, 128><<<grid, 128, 0, st>>>(
        m.tok_seq, m.tok_pos, m.blk_off, m.block_table, static_cast<const uint16_t*>(qkv),
        static_cast<uint16_t*>(q_out), static_cast<uint16_t*>(pool), a);
  else
    append_kernel<BF16, HALF, 64><<<grid, 128, 0, st>>>(
        m.tok_seq, m.tok_pos, m.blk_off, m.block_table, static_cast<const uint16_t*>(qkv),
        static_cast<uint16_t*>(q_out), static_cast<uint16_t*>(pool), a);
  return cudaGetLastError();
}

cudaError_t launch_append(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv, void* q_out,
                          void* pool, cudaStream_t st) {
  const bool half = a.style == DS_ROPE_HALF;
  if (a.dtype == DS_BF16)
    return half ? launch_append_t<true, true>(m, a, qkv, q_out, pool, st)
                : launch_append_t<true, false>(m, a, qkv, q_out, pool, st);
  return half ? launch_append_t<false, true>(m, a, qkv, q_out, pool, st)
              : launch_append_t<false, false>(m, a, qkv, q_out, pool, st);
}

}  // namespace dsr
