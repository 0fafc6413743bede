// decode.cu -- blocked attention for decode rows (sequences with one new
// token): split-K over KV blocks plus a combine step.
//
// A decode row reads its sequence's whole KV history once, so the kernel is
// bound by HBM bandwidth.  Each CTA owns one (split, KV head) work atom: a run
// of up to split_blocks KV blocks of one sequence ("DeepSpeed Inference v2",
// pyshine.com/deepspeed-2, section "Ragged batches": attention runs over
// per-head work atoms built from the batch metadata; kernels read block ids and
// address the pools directly).  The CTA streams the (block, K|V, head) tiles,
// each contiguous in the pool, into shared memory with bulk asynchronous copies
// (TMA engine) completing on mbarriers, and all G query heads of the KV group
// are scored against each loaded tile, so K/V are read from HBM once.
//
// Thread mapping: a key is handled by D/8 lanes holding 8 dimensions each
// (16-byte shared-memory loads, conflict-free).  Each warp keeps its own online
// softmax state over a fixed slice of every block; the warps' states are
// merged at the end of the split.  A split emits (m, l, o[D]) per query head
// in fp32 (m in log2 units), or the final row when it is its sequence's only
// split; the combine kernel merges the splits of the others.
//
// Fused variant (FUSED): the split holding a row's last KV block also appends
// the row's new token: it rotates K (the append kernel's arithmetic, so the
// stored bits are the same), writes K and V into the pool slot and patches
// them into its staged copy of that block, whose slot the bulk copy read before
// the write.  With a counter array, the splits of a multi-split row also count
// themselves done on a per-(sequence, KV head) counter after writing their
// partials; the last one merges all partials (the combine kernel's arithmetic,
// in its order) and resets the counter, so the decode rows need one launch.
#include "tc.cuh"

// CTA shape: warps per CTA, bulk-copy pipeline stages (each stage one K + V
// tile pair, 32 KB at D=128) and CTAs per SM the registers must allow, for
// G < 4 and G >= 4 query heads per KV head.  Measured on GB300 (decode rows of
// the 2048-token SplitFuse batch, G=4): 4 warps x 2 stages x 3 CTAs/SM
// 6.52 TB/s; 4 x 3 x 2: 5.63; 8 x 2 x 2: 5.35; 8 x 3 x 1: 3.69.  G=1 (256
// decode rows, attention call): 4 x 2 x 3 1.2692 ms; 8 x 2 x 3 1.2681;
// 8 x 3 x 2 1.2732; 4 x 3 x 2 1.2761; 2 x 2 x 3 1.2784; 2 x 3 x 2 1.2905.
#ifndef DSR_DECODE_WARPS
#define DSR_DECODE_WARPS 4
#endif
#ifndef DSR_DECODE_STAGES
#define DSR_DECODE_STAGES 2
#endif
#ifndef DSR_DECODE_WARPS_GQA
#define DSR_DECODE_WARPS_GQA 4
#endif
#ifndef DSR_DECODE_STAGES_GQA
#define DSR_DECODE_STAGES_GQA 2
#endif
#ifndef DSR_DECODE_MINB
#define DSR_DECODE_MINB 3
#endif
#ifndef DSR_DECODE_MINB_GQA
#define DSR_DECODE_MINB_GQA 3
#endif
// 1: the softmax keeps a lagging reference max (rescale only when a score
// outgrows it by 2^8) and per-lane partial row sums; 0: exact running max and
// a warp-wide sum every block.  Measured on GB300 (attention call, 0 -> 1):
// 256 decode rows 1.2878 -> 1.2852 ms, SplitFuse 2048 1.3568 -> 1.3468 ms,
// max ragged 8192 1.2021 -> 1.1922 ms.
#ifndef DSR_DECODE_LAZY
#define DSR_DECODE_LAZY 1
#endif
// 1: decode rows of grouped-query layers with head size 128 run on the
// tensor-core kernel (decode_tc.cu); 0: every decode row runs here.
#ifndef DSR_DECODE_TC
#define DSR_DECODE_TC 1
#endif

namespace dsr {

constexpr float kNegBig = -1.0e30f;  // finite "minus infinity" for running maxima

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = Stor<BF16>::lo(w[i]);
    f[2 * i + 1] = Stor<BF16>::hi(w[i]);
  }
}

template <bool BF16, bool HALF, int D, int G, int WARPS, int STAGES>
struct DecodeCfg {
  static constexpr int LPK = D / 8;             // lanes per key
  static constexpr int KPS = 32 / LPK;          // key groups per warp
  static constexpr int KPW = kBlockSize / WARPS; // keys per warp per block
  static constexpr int KPG = KPW / KPS;         // keys per group per block
  static constexpr int REP = LPK / KPG;         // lanes holding the same reduced key
  static constexpr int TILE_BYTES = kBlockSize * D * 2;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int PBUF_FLOATS = KPS * KPG * G;  // per warp
  static constexpr int MERGE_FLOATS = WARPS * G * (D + 2);
  static constexpr int TILES_BYTES = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = TILES_BYTES;
  static constexpr int PBUF_OFF = BAR_OFF + 8 * STAGES;
  static constexpr int SMEM_BYTES = PBUF_OFF + WARPS * PBUF_FLOATS * 4;
  static_assert(KPG >= 1 && KPG <= LPK, "key split");
  static_assert(MERGE_FLOATS * 4 <= TILES_BYTES, "merge scratch aliases the tiles");
};

template <bool BF16, bool HALF, int D, int G, int WARPS, int STAGES, bool FUSED>
__global__ void __launch_bounds__(WARPS * 32, G >= 4 ? DSR_DECODE_MINB_GQA : DSR_DECODE_MINB) decode_split_kernel(
    const int4* __restrict__ items, const int32_t* __restrict__ cu_seqlens,
    const int32_t* __restrict__ seq_seen, const int32_t* __restrict__ blk_off,
    const int32_t* __restrict__ block_table, const uint16_t* __restrict__ qkv,
    uint16_t* __restrict__ pool, uint16_t* __restrict__ out, float* __restrict__ ws,
    int32_t* __restrict__ counters, LayerArgs a) {
  using C = DecodeCfg<BF16, HALF, D, G, WARPS, STAGES>;
  // the batch's split items (a launch sized by the capacities has more CTAs)
  const int n_items = a.header[HDR_DEC_ITEMS];
  if ((int)blockIdx.x >= n_items) return;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane / C::LPK;       // key group inside the warp
  const int li = lane % C::LPK;        // lane inside the group: dims [8*li, 8*li+8)
  const int4 it = items[blockIdx.x];
  const int seq = it.x, b_begin = it.y, b_end = it.z, slot = it.w;
  const int c = blockIdx.y;            // KV head
  const int t = cu_seqlens[seq];       // the row's packed token
  const int p = seq_seen[seq];         // its position
  const int L = p + 1;
  const int nblk = b_end - b_begin;
  const int* btab = block_table + blk_off[seq];
  if (nblk <= 0 || p >= a.max_positions) {
    if (tid == 0) set_dev_error(a.header, nblk <= 0 ? DS_DEVERR_WORKLIST : DS_DEVERR_POSITION);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  auto issue = [&](int stage, int b) {
    int blk = btab[b];
    uint64_t* bar = &bars[stage];
    if (blk < 0 || blk >= a.num_blocks) {
      set_dev_error(a.header, DS_DEVERR_BLOCK_ID);
      mbar_arrive_expect_tx(bar, 0);  // complete the phase without data
      return;
    }
    const uint16_t* kt = pool + (((int64_t)blk * 2 + 0) * a.Hkv + c) * (int64_t)(kBlockSize * D);
    const uint16_t* vt = pool + (((int64_t)blk * 2 + 1) * a.Hkv + c) * (int64_t)(kBlockSize * D);
    uint8_t* dst = smem + stage * C::STAGE_BYTES;
    mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
    bulk_g2s(dst, kt, C::TILE_BYTES, bar);
    bulk_g2s(dst + C::TILE_BYTES, vt, C::TILE_BYTES, bar);
  };
  if (tid == 0) {
    for (int s = 0; s < STAGES && s < nblk; ++s) issue(s, b_begin + s);
  }

  // ---- fused append of the row's new token (position p) by the split that
  // holds its block: lanes [0, D/16) rotate one 16-element unit of K each,
  // lanes [0, D/8) copy 8 elements of V each.
  const int nb = (L + kBlockSize - 1) / kBlockSize;
  const bool owner = FUSED && b_end == nb;
  const int new_off = p % kBlockSize;
  const int ki0 = HALF ? 8 * lane : 16 * lane;
  const int ki1 = HALF ? D / 2 + 8 * lane : 16 * lane + 8;
  uint4 kn0 = make_uint4(0, 0, 0, 0), kn1 = kn0, vn = kn0;
  if (owner && warp == 0) {
    const int blk = btab[p / kBlockSize];
    const bool blk_ok = blk >= 0 && blk < a.num_blocks;  // else reported by issue()
    const uint16_t* row = qkv + (int64_t)t * (a.Hq + 2 * a.Hkv) * D;
    if (lane < D / 16) {
      kn0 = ld_nc_v4(row + (a.Hq + c) * D + ki0);
      kn1 = ld_nc_v4(row + (a.Hq + c) * D + ki1);
      float4 cs[4];
      const float4* cs_row = reinterpret_cast<const float4*>(a.rope + (int64_t)p * (D / 2));
#pragma unroll
      for (int q = 0; q < 4; ++q) cs[q] = __ldg(cs_row + 4 * lane + q);  // pairs 8*lane ..
      rotate16<BF16, HALF>(kn0, kn1, cs);
      if (blk_ok) {
        uint16_t* dst = pool + ((((int64_t)blk * 2 + 0) * a.Hkv + c) * kBlockSize + new_off) * D;
        *reinterpret_cast<uint4*>(dst + ki0) = kn0;
        *reinterpret_cast<uint4*>(dst + ki1) = kn1;
      }
    }
    if (lane < D / 8) {
      vn = ld_nc_v4(row + (a.Hq + a.Hkv + c) * D + 8 * lane);
      if (blk_ok)
        *reinterpret_cast<uint4*>(pool + ((((int64_t)blk * 2 + 1) * a.Hkv + c) * kBlockSize + new_off) * D +
                                  8 * lane) = vn;
    }
  }

  // ---- query: rotate (fp32, same rule as the append), scale into log2 units.
  float q[G][8];
  {
    const uint16_t* qrow = qkv + (int64_t)t * (a.Hq + 2 * a.Hkv) * D;
    const float2* cs = a.rope + (int64_t)p * (D / 2);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      uint4 raw = ld_nc_v4(qrow + (c * G + h) * D + 8 * li);
      float x[8];
      unpack8<BF16>(raw, x);
      if (HALF) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = __shfl_xor_sync(0xffffffffu, x[e], C::LPK / 2);
        const bool first = li < C::LPK / 2;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float2 r = cs[8 * (li % (C::LPK / 2)) + e];
          float y0, y1;
          if (first) rope_pair(x[e], y[e], r.x, r.y, y0, y1);
          else rope_pair(y[e], x[e], r.x, r.y, y1, y0);
          q[h][e] = y0 * a.scale_log2;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 r = cs[4 * li + e];
          float y0, y1;
          rope_pair(x[2 * e], x[2 * e + 1], r.x, r.y, y0, y1);
          q[h][2 * e] = y0 * a.scale_log2;
          q[h][2 * e + 1] = y1 * a.scale_log2;
        }
      }
    }
  }

  float m[G], l[G], o[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = kNegBig;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[h][e] = 0.f;
  }
  float* pbuf = reinterpret_cast<float*>(smem + C::PBUF_OFF) + warp * C::PBUF_FLOATS;
  const int key0 = warp * C::KPW + grp * C::KPG;  // first key of this group in a block
  const int my_key = (li / C::REP) % C::KPG;        // key this lane holds after reduction
  bool timed_out = false;

  for (int j = 0; j < nblk; ++j) {
    const int stage = j % STAGES;
    bool ok = mbar_wait_bounded(&bars[stage], (j / STAGES) & 1);
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    const uint16_t* Kt = reinterpret_cast<const uint16_t*>(smem + stage * C::STAGE_BYTES);
    const uint16_t* Vt = Kt + kBlockSize * D;
    const int kbase = (b_begin + j) * kBlockSize;
    if (owner && j == nblk - 1) {
      // the new token's slot in the staged last block: the values just appended
      if (warp == 0) {
        uint16_t* Kw = reinterpret_cast<uint16_t*>(smem + stage * C::STAGE_BYTES) + new_off * D;
        uint16_t* Vw = Kw + kBlockSize * D;
        if (lane < D / 16) {
          *reinterpret_cast<uint4*>(Kw + ki0) = kn0;
          *reinterpret_cast<uint4*>(Kw + ki1) = kn1;
        }
        if (lane < D / 8) *reinterpret_cast<uint4*>(Vw + 8 * lane) = vn;
      }
      __syncthreads();
    }

    // scores of this group's KPG keys, partial over the lane's 8 dims
    float part[G][C::KPG];
#pragma unroll
    for (int i = 0; i < C::KPG; ++i) {
      uint4 raw = *reinterpret_cast<const uint4*>(Kt + (key0 + i) * D + 8 * li);
      float k8[8];
      unpack8<BF16>(raw, k8);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int e = 0; e < 8; e += 2) tc::ffma2(a0, a1, q[h][e], q[h][e + 1], k8[e], k8[e + 1], a0, a1);
        part[h][i] = a0 + a1;
      }
    }
    // transposed reduction over the group's lanes: halve the key set at each
    // level (upper half to lanes with the level's bit set), then finish the sum.
    float s[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float v[C::KPG];
#pragma unroll
      for (int i = 0; i < C::KPG; ++i) v[i] = part[h][i];
#pragma unroll
      for (int n = C::KPG, mask = C::LPK / 2; n > 1; n >>= 1, mask >>= 1) {
        const bool upper = (li & mask) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          float send = upper ? v[i] : v[i + n / 2];
          float keep = upper ? v[i + n / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
      }
#pragma unroll
      for (int mask = C::REP / 2; mask >= 1; mask >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
      s[h] = (kbase + key0 + my_key < L) ? v[0] : -INFINITY;
    }
    // online softmax over the warp's keys of this block
#if DSR_DECODE_LAZY
    // The reference max m (warp-uniform, log2 units) is kept unless a score
    // outgrows it by more than 2^8; only then is the warp max taken and O and
    // l rescaled (the final O / l does not depend on the reference).  l holds
    // per-lane partial sums, each key counted by one lane, summed after the
    // last block.
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (__any_sync(0xffffffffu, s[h] > m[h] + 8.0f)) {
        float mx = s[h];
#pragma unroll
        for (int mask = C::REP; mask < 32; mask <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
        const float m_new = fmaxf(m[h], mx);
        const float alpha = fast_exp2(m[h] - m_new);
        l[h] *= alpha;
#pragma unroll
        for (int e = 0; e < 8; e += 2) tc::fmul2(o[h][e], o[h][e + 1], alpha, alpha);
        m[h] = m_new;
      }
      const float pv = fast_exp2(s[h] - m[h]);
      if ((li % C::REP) == 0) {
        l[h] += pv;
        pbuf[(grp * C::KPG + my_key) * G + h] = pv;
      }
    }
#else
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mx = s[h];
#pragma unroll
      for (int mask = C::REP; mask < 32; mask <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
      const float m_new = fmaxf(m[h], mx);
      const float alpha = fast_exp2(m[h] - m_new);
      const float pv = fast_exp2(s[h] - m_new);
      float sum = pv;
#pragma unroll
      for (int mask = C::REP; mask < 32; mask <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, mask);
      l[h] = l[h] * alpha + sum;
      m[h] = m_new;
#pragma unroll
      for (int e = 0; e < 8; e += 2) tc::fmul2(o[h][e], o[h][e + 1], alpha, alpha);
      if ((li % C::REP) == 0) pbuf[(grp * C::KPG + my_key) * G + h] = pv;
    }
#endif
    __syncwarp();
#pragma unroll
    for (int i = 0; i < C::KPG; ++i) {
      // slots past the sequence's length may hold non-finite bytes: skip them
      if (kbase + key0 + i >= L) break;
      uint4 raw = *reinterpret_cast<const uint4*>(Vt + (key0 + i) * D + 8 * li);
      float v8[8];
      unpack8<BF16>(raw, v8);
      const float* pr = pbuf + (grp * C::KPG + i) * G;
      float pw[G];
      if constexpr (G % 4 == 0) {  // 16-byte aligned: G*4 bytes per key
#pragma unroll
        for (int h4 = 0; h4 < G / 4; ++h4) {
          const float4 q4 = reinterpret_cast<const float4*>(pr)[h4];
          pw[4 * h4] = q4.x;
          pw[4 * h4 + 1] = q4.y;
          pw[4 * h4 + 2] = q4.z;
          pw[4 * h4 + 3] = q4.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) pw[h] = pr[h];
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int e = 0; e < 8; e += 2)
          tc::ffma2(o[h][e], o[h][e + 1], v8[e], v8[e + 1], pw[h], pw[h], o[h][e], o[h][e + 1]);
      }
    }
    __syncthreads();  // every warp is done with this stage and with pbuf
    if (tid == 0 && j + STAGES < nblk) issue(stage, b_begin + j + STAGES);
  }

  if (timed_out) {
    if (tid == 0) {
      set_dev_error(a.header, DS_DEVERR_WORKLIST);
      // let copies still in flight land before the CTA's memory is released
      for (int s = 0; s < STAGES; ++s) (void)mbar_wait_bounded(&bars[s], 0, 100000000LL);
    }
    return;
  }

#if DSR_DECODE_LAZY
  // the row sums of the warp: one partial per lane
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int mask = 1; mask < 32; mask <<= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], mask);
#endif
  // ---- merge the key groups of each warp (same m, l; o partial per group)
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int mask = C::LPK; mask < 32; mask <<= 1) o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], mask);

  // ---- merge the warps through shared memory (aliases the tile stages)
  __syncthreads();
  float* mg = reinterpret_cast<float*>(smem);  // [WARPS][G][D+2]
  if (grp == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float* dst = mg + (warp * G + h) * (D + 2);
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[8 * li + e] = o[h][e];
      if (li == 0) {
        dst[D] = m[h];
        dst[D + 1] = l[h];
      }
    }
  }
  __syncthreads();
  const int units = G * (D / 8);
  for (int u = tid; u < units; u += WARPS * 32) {
    const int h = u / (D / 8), d8 = u % (D / 8);
    float M = kNegBig;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, mg[(w * G + h) * (D + 2) + D]);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}, lsum = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float* src = mg + (w * G + h) * (D + 2);
      const float sc = fast_exp2(src[D] - M);
      lsum += sc * src[D + 1];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += sc * src[8 * d8 + e];
    }
    const int hq = c * G + h;
    if (slot < 0) {
      const float inv = 1.f / lsum;
      uint4 pk;
      uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int e = 0; e < 4; ++e) pw[e] = Stor<BF16>::pack(acc[2 * e] * inv, acc[2 * e + 1] * inv);
      *reinterpret_cast<uint4*>(out + (int64_t)t * a.Hq * D + hq * D + 8 * d8) = pk;
    } else {
      float* wml = ws + ((int64_t)slot * a.Hq + hq) * 2;
      float* wo = ws + ws_o_offset(n_items, a.Hq) + ((int64_t)slot * a.Hq + hq) * D + 8 * d8;
      if (d8 == 0) {
        wml[0] = M;
        wml[1] = lsum;
      }
      *reinterpret_cast<float4*>(wo) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      *reinterpret_cast<float4*>(wo + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }

  if (FUSED && counters != nullptr && slot >= 0) {
    // ---- the last split of (row, KV head c) to finish merges all partials
    __shared__ int s_last;
    const int split = a.header[HDR_SPLIT];
    const int cnt = (nb + split - 1) / split;
    const int first = slot - b_begin / split;  // a row's splits hold consecutive slots
    // every thread's partials precede thread 0's fence (barrier), which
    // precedes the count: whoever counts last sees them all
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      s_last = atomicAdd(&counters[seq * a.Hkv + c], 1) == cnt - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* wo_base = ws + ws_o_offset(n_items, a.Hq);
    for (int u = tid; u < units; u += WARPS * 32) {
      const int h = u / (D / 8), d8 = u % (D / 8);
      const int hq = c * G + h;
      float M = kNegBig;
      for (int k = 0; k < cnt; ++k) M = fmaxf(M, __ldcg(ws + ((int64_t)(first + k) * a.Hq + hq) * 2));
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}, lsum = 0.f;
      for (int k = 0; k < cnt; ++k) {
        const float* ml = ws + ((int64_t)(first + k) * a.Hq + hq) * 2;
        const float sc = fast_exp2(__ldcg(ml) - M);
        lsum += sc * __ldcg(ml + 1);
        const float4* src =
            reinterpret_cast<const float4*>(wo_base + ((int64_t)(first + k) * a.Hq + hq) * D + 8 * d8);
        const float4 s0 = __ldcg(src), s1 = __ldcg(src + 1);
        acc[0] += sc * s0.x; acc[1] += sc * s0.y; acc[2] += sc * s0.z; acc[3] += sc * s0.w;
        acc[4] += sc * s1.x; acc[5] += sc * s1.y; acc[6] += sc * s1.z; acc[7] += sc * s1.w;
      }
      const float inv = 1.f / lsum;
      uint4 pk;
      uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int e = 0; e < 4; ++e) pw[e] = Stor<BF16>::pack(acc[2 * e] * inv, acc[2 * e + 1] * inv);
      *reinterpret_cast<uint4*>(out + (int64_t)t * a.Hq * D + hq * D + 8 * d8) = pk;
    }
    if (tid == 0) counters[seq * a.Hkv + c] = 0;  // ready for the next launch
  }
}

// Merge the splits of each multi-split decode row: one warp per (row, head).
template <bool BF16, int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const int4* __restrict__ dseqs,
                                                             const float* __restrict__ ws,
                                                             uint16_t* __restrict__ out,
                                                             const int32_t* __restrict__ header, int32_t Hq) {
  constexpr int DPL = D / 32;  // dims per lane: 4 or 2
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
  if (h >= Hq || (int)blockIdx.x >= header[HDR_DEC_SEQS]) return;
  const int n_items = header[HDR_DEC_ITEMS];
  const int4 ds = dseqs[blockIdx.x];
  const int t = ds.y, first = ds.z, cnt = ds.w;
  if (cnt <= 1) return;
  float M = kNegBig;
  for (int k = 0; k < cnt; ++k) M = fmaxf(M, ws[((int64_t)(first + k) * Hq + h) * 2]);
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  float lsum = 0.f;
  const float* wo = ws + ws_o_offset(n_items, Hq);
  for (int k = 0; k < cnt; ++k) {
    const float* ml = ws + ((int64_t)(first + k) * Hq + h) * 2;
    const float sc = fast_exp2(ml[0] - M);
    lsum += sc * ml[1];
    const float* src = wo + ((int64_t)(first + k) * Hq + h) * D + DPL * lane;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] += sc * src[e];
  }
  const float inv = 1.f / lsum;
  uint16_t* dst = out + (int64_t)t * Hq * D + h * D + DPL * lane;
  if (DPL == 4) {
    uint2 pk;
    pk.x = Stor<BF16>::pack(acc[0] * inv, acc[1] * inv);
    pk.y = Stor<BF16>::pack(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = Stor<BF16>::pack(acc[0] * inv, acc[1] * inv);
  }
}

template <bool BF16, bool HALF, int D, int G>
static cudaError_t launch_decode_t(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                   const void* pool, void* out, float* ws, cudaStream_t st,
                                   bool overlap_previous, bool fused, int32_t* counters) {
  constexpr int WARPS = G >= 4 ? DSR_DECODE_WARPS_GQA : DSR_DECODE_WARPS;
  constexpr int STAGES = G >= 4 ? DSR_DECODE_STAGES_GQA : DSR_DECODE_STAGES;
  using C = DecodeCfg<BF16, HALF, D, G, WARPS, STAGES>;
  auto kern = fused ? decode_split_kernel<BF16, HALF, D, G, WARPS, STAGES, true>
                    : decode_split_kernel<BF16, HALF, D, G, WARPS, STAGES, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  const int64_t items = (m.flags & DS_META_CAPACITY) ? max_decode_items(m.max_seqs, m.max_blocks)
                                                      : m.n_decode_items;
  cfg.gridDim = dim3((unsigned)items, a.Hkv);
  cfg.blockDim = dim3(WARPS * 32);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // After the prefill kernel (which lets dependents start as soon as all its
  // CTAs are running), decode CTAs may fill the SMs that prefill leaves idle:
  // the two read only what the KV append wrote before either started and
  // write disjoint output rows.
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  // the unfused kernel only reads the pool (the append kernel wrote the rows)
  e = cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const int4*>(m.decode_items), m.cu_seqlens,
                         m.seq_seen, m.blk_off, m.block_table, static_cast<const uint16_t*>(qkv),
                         static_cast<uint16_t*>(const_cast<void*>(pool)), static_cast<uint16_t*>(out), ws,
                         counters, a);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (counters == nullptr && ((m.flags & DS_META_CAPACITY) || m.n_decode_items > m.n_decode_seqs))
    e = launch_decode_combine(m, a, ws, out, st);
  return e;
}

cudaError_t launch_decode_combine(const ds_ragged_meta& m, const LayerArgs& a, const float* ws,
                                  void* out, cudaStream_t st) {
  dim3 g2((m.flags & DS_META_CAPACITY) ? m.max_seqs : m.n_decode_seqs, (a.Hq + 3) / 4);
  const int4* dseqs = reinterpret_cast<const int4*>(m.decode_seqs);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (a.dtype == DS_BF16) {
    if (a.D == 128) decode_combine_kernel<true, 128><<<g2, 128, 0, st>>>(dseqs, ws, o, m.header, a.Hq);
    else decode_combine_kernel<true, 64><<<g2, 128, 0, st>>>(dseqs, ws, o, m.header, a.Hq);
  } else {
    if (a.D == 128) decode_combine_kernel<false, 128><<<g2, 128, 0, st>>>(dseqs, ws, o, m.header, a.Hq);
    else decode_combine_kernel<false, 64><<<g2, 128, 0, st>>>(dseqs, ws, o, m.header, a.Hq);
  }
  return cudaGetLastError();
}

template <bool BF16, bool HALF, int D>
static cudaError_t launch_decode_g(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                   const void* pool, void* out, float* ws, cudaStream_t st, bool ov,
                                   bool fu, int32_t* cnt) {
  switch (a.G) {
    case 1: return launch_decode_t<BF16, HALF, D, 1>(m, a, qkv, pool, out, ws, st, ov, fu, cnt);
    case 2: return launch_decode_t<BF16, HALF, D, 2>(m, a, qkv, pool, out, ws, st, ov, fu, cnt);
    case 4: return launch_decode_t<BF16, HALF, D, 4>(m, a, qkv, pool, out, ws, st, ov, fu, cnt);
    case 8: return launch_decode_t<BF16, HALF, D, 8>(m, a, qkv, pool, out, ws, st, ov, fu, cnt);
    default: return cudaErrorInvalidValue;
  }
}

template <bool BF16, bool HALF>
static cudaError_t launch_decode_d(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                   const void* pool, void* out, float* ws, cudaStream_t st, bool ov,
                                   bool fu, int32_t* cnt) {
  return a.D == 128 ? launch_decode_g<BF16, HALF, 128>(m, a, qkv, pool, out, ws, st, ov, fu, cnt)
                    : launch_decode_g<BF16, HALF, 64>(m, a, qkv, pool, out, ws, st, ov, fu, cnt);
}

bool decode_on_tensor_cores(const LayerArgs& a) { return DSR_DECODE_TC && a.D == 128 && a.G >= 2; }

cudaError_t launch_decode(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                          const void* pool, void* out, float* ws, cudaStream_t st,
                          bool overlap_previous, bool fused_append, int32_t* counters) {
  // grouped-query rows of head size 128: the tensor-core kernel (decode_tc.cu)
  if (decode_on_tensor_cores(a))
    return launch_decode_tc(m, a, qkv, pool, out, ws, st, overlap_previous, fused_append, counters);
  const bool half = a.style == DS_ROPE_HALF;
  const bool ov = overlap_previous, fu = fused_append;
  if (a.dtype == DS_BF16)
    return half ? launch_decode_d<true, true>(m, a, qkv, pool, out, ws, st, ov, fu, counters)
                : launch_decode_d<true, false>(m, a, qkv, pool, out, ws, st, ov, fu, counters);
  return half ? launch_decode_d<false, true>(m, a, qkv, pool, out, ws, st, ov, fu, counters)
              : launch_decode_d<false, false>(m, a, qkv, pool, out, ws, st, ov, fu, counters);
}

}  // namespace dsr
