// decode_tc.cu -- blocked attention for decode rows of grouped-query layers
// (G >= 2 query heads per KV head, head_dim 128) on the 5th-generation tensor
// cores: split-K over KV blocks, each split's score and value products as
// tcgen05 MMAs with accumulators in tensor memory, K/V tiles staged by tiled
// TMA loads.
//
// A decode row reads its sequence's whole KV history once, so the work is
// bound by HBM bandwidth; what the tensor cores buy is SM time.  Scoring the G
// query heads of a KV group against a staged 64-key block takes ~700 warp
// instructions on the CUDA cores, which caps how many bytes a single SM can
// consume; as MMAs it is a handful of instructions, so the decode rows reach
// the HBM rate on the SMs a prefill grid leaves free.
//
// Work unit ("DeepSpeed Inference v2", pyshine.com/deepspeed-2, section
// "Ragged batches": attention over per-head work atoms built from the batch
// metadata; kernels read block ids and address the pools directly): one split
// item (a run of up to split_blocks KV blocks of one decode row) x one KV head c.
// Per 128-key tile (two pool blocks):
//   S^T[keys][heads] = K[keys][d] . Q^T[d][heads]    (SS MMA, M=128, N=16, K=128)
//   O^T[d][heads]   += V^T[d][keys] . P[keys][heads]  (SS MMA, M=128, N=16, K=128;
//                                                       V^T read MN-major)
// with the G query heads padded to N = 16 (rows G..15 of Q and P stay zero).
//
// The grid is persistent (one CTA per SM: three 64 KB K+V stages) and takes
// units dynamically from a counter in the batch header, so CTAs that start late
// -- behind a prefill grid -- simply take fewer units; the last CTA to finish
// zeroes the counters for the next launch.  Roles (10 warps):
//   warps 0, 8 TMA producers of the K and of the V halves of 3 stages of
//              128-key x 128-dim tiles (128-byte-swizzled 64x64 boxes of the
//              pool seen as a 2-D tensor), each half refilled once it is free.
//   warp 1     tensor-memory owner; issues the score MMAs S(j) (one elected
//              lane) as soon as tile j landed.
//   warp 3     issues the value MMAs P*V(j) as soon as P(j) is written, so the
//              softmax of one tile overlaps the MMAs of its neighbours.
//   warp 2     unit scheduler: takes the next unit, rotates its G query rows
//              (fp32, the append's arithmetic, rounded to the storage type) into
//              a swizzled Q slot and publishes the unit's record; in the fused
//              variant it also appends the row's new K/V when the unit holds the
//              row's last block (before the producer loads that block).
//   warps 4-7  softmax, one key per thread (tensor-memory lane = key): masked
//              scores, a reference max per head kept unless some score outgrows
//              it by 2^8 (decided by one barrier-OR per tile; then the exact tile
//              max is exchanged and O rescaled: the final O / l does not depend
//              on the reference), P = exp2(S*scale - m) in the storage type;
//              zero the V rows past the last key of a partial tile (those slots
//              may hold anything and 0 * NaN would poison P*V); epilogue O / l
//              -> out, or (m, l, O) partials for the combine step.
//   warp 9     (fused variant with counters) counts each finished split done
//              and merges a row's partials when its last split finishes.
// Tensor memory (64 columns): S[2] at 0 / 16, O[2] at 32 / 48.
// Every mbarrier wait is bounded: on timeout the CTA records an error and stops.
#include <algorithm>

#include "tc.cuh"

#ifndef DSR_DTC_STAGES
#define DSR_DTC_STAGES 3
#endif
// 1: the K/V loads carry an L2 evict_first policy.  Each decode tile is read
// once; without the hint the stream evicts the K/V history that prefill atoms
// running beside it re-read from L2.
#ifndef DSR_DTC_EVICT_FIRST
#define DSR_DTC_EVICT_FIRST 1
#endif
// Largest grid (0: one CTA per SM).
#ifndef DSR_DTC_MAX_CTAS
#define DSR_DTC_MAX_CTAS 0
#endif

namespace dsr {
namespace dtc {

constexpr int D = 128;
constexpr int KEYS = 128;                      // keys per tile: two 64-token blocks
constexpr int NPAD = 16;                       // query heads padded to the MMA's N
constexpr int STAGES = DSR_DTC_STAGES;
constexpr int QN = 4;                          // unit slots (Q tile + unit record)
constexpr int HALF_BYTES = KEYS * 128;         // 128 keys x 64 dims
constexpr int KV_BYTES = 2 * HALF_BYTES;       // a K or V tile: 128 keys x 128 dims
constexpr int STAGE_BYTES = 2 * KV_BYTES;      // K, then V
constexpr int ROWS16_BYTES = NPAD * 128;       // 16 rows x 64 elements
constexpr int QP_BYTES = 2 * ROWS16_BYTES;     // a Q or P operand: 16 rows x 128
constexpr int BOX_BYTES = 64 * 128;            // one TMA box: 64 rows x 64 elements
constexpr int OFF_Q = STAGES * STAGE_BYTES;
constexpr int OFF_P = OFF_Q + QN * QP_BYTES;
constexpr int OFF_RED = OFF_P + 2 * QP_BYTES;  // floats: [2][4][16] maxima, [4][16] sums
constexpr int RED_FLOATS = 2 * 4 * 16 + 4 * 16;
constexpr int OFF_INFO = OFF_RED + RED_FLOATS * 4;
constexpr int INFO_INTS = 16;
constexpr int OFF_BAR = OFF_INFO + QN * INFO_INTS * 4;
// K and V halves of a stage are filled and freed separately: K is free once
// S(j) is done, V once P*V(j) is, so K(j+1) is loaded while tile j's softmax
// and P*V still run, and S(j+1) and its softmax overlap V(j+1)'s load.
enum {
  B_KFULL = 0,
  B_VFULL = B_KFULL + STAGES,
  B_KEMPTY = B_VFULL + STAGES,
  B_VEMPTY = B_KEMPTY + STAGES,
  B_QFULL = B_VEMPTY + STAGES,
  B_QEMPTY = B_QFULL + QN,
  B_SFULL = B_QEMPTY + QN,
  B_PFULL = B_SFULL + 2,
  B_ODONE = B_PFULL + 2,
  B_MMADRAIN = B_ODONE + 2,  // one per MMA warp
  B_MFULL = B_MMADRAIN + 2,  // merge records (fused decode with counters)
  B_MEMPTY = B_MFULL + 4,
  B_COUNT = B_MEMPTY + 4
};
constexpr int MQ = 4;          // merge-record slots
constexpr int MREC_INTS = 8;
// tensor-memory address; then the merge records
constexpr int OFF_MISC = OFF_BAR + 8 * B_COUNT;
constexpr int OFF_MREC = OFF_MISC + 16;
constexpr int SMEM = OFF_MREC + MQ * MREC_INTS * 4 + 1024;  // + room to align the base to 1024
constexpr int TMEM_COLS = 64;
constexpr int COL_S = 0, COL_O = 32;
constexpr int THREADS = 320;
// arrivals that free a unit slot: the two producers, the S warp's commit, the
// P*V warp, four softmax warps
constexpr int QEMPTY_ARRIVALS = 8;
static_assert(SMEM <= 227 * 1024, "shared memory over the per-CTA limit");

// unit record fields
enum { U_UNIT = 0, U_SEQ, U_C, U_TOK, U_POS, U_BBEGIN, U_BEND, U_SLOT, U_NTILES, U_KEYEND };

}  // namespace dtc

#ifdef DSR_TEST_WAIT_RUNOUT
// Test builds only: while set, the producers issue no copies, so every wait
// on a tile runs out with nothing in flight.
__device__ int g_test_stall_copies;
#endif

// One storage-type value (round to nearest even) as raw bits.
template <bool BF16>
__device__ __forceinline__ uint16_t to_bits(float x) {
  uint16_t r;
  if (BF16)
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  else
    asm("{ .reg .f16 h; cvt.rn.f16.f32 h, %1; mov.b16 %0, h; }" : "=h"(r) : "f"(x));
  return r;
}

template <bool BF16, bool HALF, int G, bool FUSED>
__global__ void __launch_bounds__(dtc::THREADS, 1) decode_tc_kernel(
    const __grid_constant__ CUtensorMap pool_map, const int4* __restrict__ items,
    const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ seq_seen,
    const int32_t* __restrict__ blk_off, const int32_t* __restrict__ block_table,
    const uint16_t* __restrict__ qkv, uint16_t* __restrict__ pool, uint16_t* __restrict__ out,
    float* __restrict__ ws, int32_t* __restrict__ counters, LayerArgs a) {
  using namespace dtc;
  static_assert(G >= 2 && G <= 8, "head group");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  int* mrec = reinterpret_cast<int*>(sm + OFF_MREC);
  int* info = reinterpret_cast<int*>(sm + OFF_INFO);
  float* red = reinterpret_cast<float*>(sm + OFF_RED);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* hdr = a.header;
  const int n_items = hdr[HDR_DEC_ITEMS];
  const int n_units = n_items * a.Hkv;

  // Q slots and P buffers start at zero: their rows G..15 are never written.
  for (int i = tid; i < (QN + 2) * QP_BYTES / 16; i += THREADS)
    reinterpret_cast<uint4*>(sm + OFF_Q)[i] = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async();
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bar[B_KFULL + s], 1);
      mbar_init(&bar[B_VFULL + s], 1);
      mbar_init(&bar[B_KEMPTY + s], 1);
      mbar_init(&bar[B_VEMPTY + s], 1);
    }
    for (int s = 0; s < QN; ++s) {
      mbar_init(&bar[B_QFULL + s], 1);
      mbar_init(&bar[B_QEMPTY + s], QEMPTY_ARRIVALS);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[B_SFULL + s], 1);
      mbar_init(&bar[B_PFULL + s], 4);  // one arrival per softmax warp
      mbar_init(&bar[B_ODONE + s], 1);
    }
    mbar_init(&bar[B_MMADRAIN], 1);
    mbar_init(&bar[B_MMADRAIN + 1], 1);
    for (int s = 0; s < MQ; ++s) {
      mbar_init(&bar[B_MFULL + s], 4);  // the four softmax warps
      mbar_init(&bar[B_MEMPTY + s], 1);
    }
    fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, TMEM_COLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  auto warp_wait = [&](int b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait_bounded(&bar[b], parity));
  };

  if (warp == 0 || warp == 8) {
    // ---------------------------------------------------------- producers
    // warp 0 fills the K halves of the stages, warp 8 the V halves, each as
    // soon as its half is free, so K runs up to STAGES tiles ahead of V.
    const int kv = warp == 8 ? 1 : 0;
    const int b_full = kv ? B_VFULL : B_KFULL, b_empty = kv ? B_VEMPTY : B_KEMPTY;
    uint32_t k = 0, r = 0;
    bool ok = true;
#if DSR_DTC_EVICT_FIRST
    const uint64_t pol = tc::policy_evict_first();
#endif
    while (ok) {
      const int slot = k % QN;
      if (!warp_wait(B_QFULL + slot, (k / QN) & 1)) { ok = false; break; }
      const int* inf = info + slot * INFO_INTS;
      const int unit = inf[U_UNIT], seq = inf[U_SEQ], c = inf[U_C];
      const int b_begin = inf[U_BBEGIN], b_end = inf[U_BEND], n_tiles = inf[U_NTILES];
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_QEMPTY + slot]);
      ++k;
      if (unit < 0) break;
      const int* btab = block_table + blk_off[seq];
      for (int tt = 0; tt < n_tiles; ++tt, ++r) {
        const int s = r % STAGES;
        // this half of stage s is free once S (P*V) of tile r - STAGES is done
        if (r >= STAGES && !warp_wait(b_empty + s, ((r / STAGES) - 1) & 1)) { ok = false; break; }
        const int b0 = b_begin + 2 * tt;
        const int nblk = min(2, b_end - b0);
#ifdef DSR_TEST_WAIT_RUNOUT
        const bool stall = *reinterpret_cast<volatile int*>(&g_test_stall_copies) != 0;
#else
        constexpr bool stall = false;
#endif
        if (lane == 0 && !stall) {
          uint64_t* fb = &bar[b_full + s];
          uint8_t* dst = sm + s * STAGE_BYTES + kv * KV_BYTES;
          mbar_arrive_expect_tx(fb, (uint32_t)nblk * 2u * BOX_BYTES);
          for (int i = 0; i < nblk; ++i) {
            int blk = btab[b0 + i];
            if (blk < 0 || blk >= a.num_blocks) {
              set_dev_error(hdr, DS_DEVERR_BLOCK_ID);
              blk = 0;
            }
            const int row = ((blk * 2 + kv) * a.Hkv + c) * 64;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#if DSR_DTC_EVICT_FIRST
              tc::tma_load_2d_hint(dst + h * HALF_BYTES + i * BOX_BYTES, &pool_map, h * 64, row, fb, pol);
#else
              tc::tma_load_2d(dst + h * HALF_BYTES + i * BOX_BYTES, &pool_map, h * 64, row, fb);
#endif
            }
          }
        }
        __syncwarp();
      }
    }
    if (!ok) {
      if (lane == 0) set_dev_error(hdr, DS_DEVERR_WORKLIST);
    }
    // no copy may land after the CTA's shared memory is released: wait for the
    // last fill of every stage (a phase the consumer already saw returns at once)
    if (lane == 0)
      for (uint32_t q = (r > (uint32_t)STAGES ? r - STAGES : 0); q < r; ++q)
        (void)mbar_wait_bounded(&bar[b_full + q % STAGES], (q / STAGES) & 1, DSR_WAIT_LIMIT / 20);
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ---------------------------------------------------------- MMA issuers
    // Warp 1 issues the score MMAs S(j) as soon as tile j landed (and its S
    // buffer is free: the softmax of tile j-2 is done), warp 3 the value MMAs
    // P*V(j) as soon as P(j) is written.  Each blocks on its own barriers; one
    // warp polling both streams reacted ~1000 cycles late.  Each warp's commits
    // track only its own MMAs: S(j)'s completion frees the K half of the stage,
    // P*V(j)'s the V half.
    constexpr uint32_t IS = tc::idesc_f16(BF16, 128, NPAD, false, false);
    constexpr uint32_t IP = tc::idesc_f16(BF16, 128, NPAD, false, true);
    auto commit = [&](int b) {
      if (tc::elect_one()) tc::mma_commit(&bar[b]);
      __syncwarp();
    };
    const bool s_warp = warp == 1;
    uint32_t k = 0, j = 0;
    bool ok = true;
    while (ok) {
      const int slot = k % QN;
      if (!warp_wait(B_QFULL + slot, (k / QN) & 1)) { ok = false; break; }
      const int unit = info[slot * INFO_INTS + U_UNIT];
      const int n_tiles = unit < 0 ? 0 : info[slot * INFO_INTS + U_NTILES];
      const int ob = k & 1;
      ++k;
      if (s_warp) {
        if (n_tiles == 0) commit(B_QEMPTY + slot);
      } else {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_QEMPTY + slot]);
      }
      if (unit < 0) break;
      for (int tt = 0; tt < n_tiles; ++tt, ++j) {
        if (s_warp) {
          if (!warp_wait(B_KFULL + j % STAGES, (j / STAGES) & 1)) { ok = false; break; }
          // S(j) overwrites S(j-2), which the softmax has read once P(j-2) exists
          if (j >= 2 && !warp_wait(B_PFULL + (j & 1), ((j - 2) / 2) & 1)) { ok = false; break; }
          tc::fence_after();
          const uint64_t kd = tc::smem_desc_sw128(smem_u32(sm + (j % STAGES) * STAGE_BYTES), 16, 1024);
          const uint64_t qd = tc::smem_desc_sw128(smem_u32(sm + OFF_Q + slot * QP_BYTES), 16, 1024);
          if (tc::elect_one()) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t ok_ = ((ks / 4) * HALF_BYTES + (ks % 4) * 32) >> 4;
              const uint32_t oq = ((ks / 4) * ROWS16_BYTES + (ks % 4) * 32) >> 4;
              tc::mma_ss(tmem + COL_S + 16 * (j & 1), kd + ok_, qd + oq, IS, ks > 0);
            }
            tc::mma_commit(&bar[B_SFULL + (j & 1)]);
            tc::mma_commit(&bar[B_KEMPTY + j % STAGES]);
            if (tt == n_tiles - 1) tc::mma_commit(&bar[B_QEMPTY + slot]);
          }
          __syncwarp();
        } else {
          if (!warp_wait(B_PFULL + (j & 1), (j / 2) & 1) || !warp_wait(B_VFULL + j % STAGES, (j / STAGES) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after();
          const uint64_t vd =
              tc::smem_desc_sw128(smem_u32(sm + (j % STAGES) * STAGE_BYTES + KV_BYTES), HALF_BYTES, 1024);
          const uint64_t pd = tc::smem_desc_sw128(smem_u32(sm + OFF_P + (j & 1) * QP_BYTES), 16, 1024);
          if (tc::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < KEYS / 16; ++kk) {
              const uint32_t ov = (kk * 2048) >> 4;
              const uint32_t op = ((kk / 4) * ROWS16_BYTES + (kk % 4) * 32) >> 4;
              tc::mma_ss(tmem + COL_O + 16 * ob, vd + ov, pd + op, IP, (tt > 0 || kk > 0));
            }
            tc::mma_commit(&bar[B_ODONE + (j & 1)]);
            tc::mma_commit(&bar[B_VEMPTY + j % STAGES]);
          }
          __syncwarp();
        }
      }
    }
    if (!ok && lane == 0) set_dev_error(hdr, DS_DEVERR_WORKLIST);
    // every MMA this warp issued has completed before tensor memory is freed
    const int drain = B_MMADRAIN + (s_warp ? 0 : 1);
    commit(drain);
    (void)warp_wait(drain, 0);
  } else if (warp == 2) {
    // ---------------------------------------------------------- unit scheduler
    uint32_t k = 0;
    const int W = (a.Hq + 2 * a.Hkv) * D;
    while (true) {
      const int slot = k % QN;
      if (k >= QN && !warp_wait(B_QEMPTY + slot, ((k / QN) - 1) & 1)) {
        if (lane == 0) set_dev_error(hdr, DS_DEVERR_WORKLIST);
        break;  // the others time out on this slot and stop
      }
      int unit = 0;
      if (lane == 0) unit = atomicAdd(&hdr[HDR_DEC_NEXT], 1);
      unit = __shfl_sync(0xffffffffu, unit, 0);
      int* inf = info + slot * INFO_INTS;
      if (unit >= n_units) {
        if (lane == 0) {
          inf[U_UNIT] = -1;
          tc::mbar_arrive(&bar[B_QFULL + slot]);
        }
        break;
      }
      const int4 it = items[unit / a.Hkv];
      const int c = unit % a.Hkv;
      const int seq = it.x, b_begin = it.y, b_end = it.z;
      const int t = cu_seqlens[seq], p = seq_seen[seq];
      const int L = p + 1, nb = (L + 63) / 64;
      int n_tiles = (b_end - b_begin + 1) / 2;
      if (b_end <= b_begin || b_end > nb || p >= a.max_positions) {
        if (lane == 0) set_dev_error(hdr, p >= a.max_positions ? DS_DEVERR_POSITION : DS_DEVERR_WORKLIST);
        n_tiles = 0;
      }
      const uint16_t* row = qkv + (int64_t)t * W;
      const float4* cs4 = reinterpret_cast<const float4*>(a.rope) + (int64_t)min(p, a.max_positions - 1) * (D / 4);
      if (FUSED && n_tiles > 0 && b_end == nb) {
        // the row's new token (position p): rotated K and V into its pool slot,
        // visible to the TMA loads that follow (the producer reads this unit's
        // record only after the fence below)
        const int blk = block_table[blk_off[seq] + p / 64];
        if (blk >= 0 && blk < a.num_blocks) {  // else reported by the producer
          const int off = p % 64;
          if (lane < D / 16) {
            const int i0 = HALF ? 8 * lane : 16 * lane;
            const int i1 = HALF ? D / 2 + 8 * lane : 16 * lane + 8;
            uint4 x0 = ld_nc_v4(row + (a.Hq + c) * D + i0);
            uint4 x1 = ld_nc_v4(row + (a.Hq + c) * D + i1);
            float4 cs[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) cs[q] = __ldg(cs4 + 4 * lane + q);
            rotate16<BF16, HALF>(x0, x1, cs);
            uint16_t* dst = pool + ((((int64_t)blk * 2 + 0) * a.Hkv + c) * 64 + off) * D;
            *reinterpret_cast<uint4*>(dst + i0) = x0;
            *reinterpret_cast<uint4*>(dst + i1) = x1;
          }
          if (lane < D / 8) {
            const uint4 v = ld_nc_v4(row + (a.Hq + a.Hkv + c) * D + 8 * lane);
            *reinterpret_cast<uint4*>(pool + ((((int64_t)blk * 2 + 1) * a.Hkv + c) * 64 + off) * D + 8 * lane) = v;
          }
          tc::fence_proxy_async_global();
        }
      }
      // the G query rows of KV head c: rotate on load, round to the storage
      // type, store 128-byte swizzled (row = head, 16-byte unit ^ (row % 8))
      uint8_t* qs = sm + OFF_Q + slot * QP_BYTES;
      for (int w = lane; w < G * 8; w += 32) {
        const int h = w >> 3, cc = w & 7;
        const int ch0 = HALF ? cc : 2 * cc;
        const int ch1 = HALF ? 8 + cc : 2 * cc + 1;
        const uint16_t* src = row + (c * G + h) * D;
        uint4 x0 = ld_nc_v4(src + 8 * ch0);
        uint4 x1 = ld_nc_v4(src + 8 * ch1);
        float4 cs[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) cs[q] = __ldg(cs4 + 4 * cc + q);
        rotate16<BF16, HALF>(x0, x1, cs);
        const int rb = (h >> 3) * 1024 + (h & 7) * 128;
        *reinterpret_cast<uint4*>(qs + (ch0 >> 3) * ROWS16_BYTES + rb + (((ch0 & 7) ^ (h & 7)) << 4)) = x0;
        *reinterpret_cast<uint4*>(qs + (ch1 >> 3) * ROWS16_BYTES + rb + (((ch1 & 7) ^ (h & 7)) << 4)) = x1;
      }
      if (lane == 0) {
        inf[U_UNIT] = unit;
        inf[U_SEQ] = seq;
        inf[U_C] = c;
        inf[U_TOK] = t;
        inf[U_POS] = p;
        inf[U_BBEGIN] = b_begin;
        inf[U_BEND] = b_end;
        inf[U_SLOT] = it.w;
        inf[U_NTILES] = n_tiles;
        inf[U_KEYEND] = min(b_end * 64, L);
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_QFULL + slot]);
      ++k;
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------- softmax
    // The four warps synchronise on named barrier 1.  A named barrier waits
    // without a bound, so no warp may leave the common sequence of barriers on
    // its own: a wait that runs out only clears the warp's `wok` (it then skips
    // its tensor-memory accesses), and the group leaves together after the
    // next vote (bar_and) sees it.
    const int ts = tid - 128;                               // key row = tensor-memory lane
    const int wq = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * wq) << 16);
    const float sc = a.scale_log2;
    // waits gate warp-collective tensor-memory accesses: decide them per warp
    auto wwait = [&](int b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_bounded(&bar[b], parity));
    };
    uint32_t k = 0, jg = 0, xc = 0, mq = 0;
    bool wok = true, ok = true;
    while (true) {
      const int slot = k % QN;
      wok = wok && wwait(B_QFULL + slot, (k / QN) & 1);
      if (!tc::bar_and(1, 128, wok)) { ok = false; break; }
      const int* inf = info + slot * INFO_INTS;
      const int unit = inf[U_UNIT], seq = inf[U_SEQ], c = inf[U_C], t = inf[U_TOK], pos = inf[U_POS];
      const int b_begin = inf[U_BBEGIN], wslot = inf[U_SLOT];
      const int n_tiles = inf[U_NTILES], key_end = inf[U_KEYEND];
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_QEMPTY + slot]);
      const int ob = k & 1;
      ++k;
      if (unit < 0) break;
      if (n_tiles == 0) continue;
      float m_ref[G], lsum[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m_ref[h] = -INFINITY;
        lsum[h] = 0.f;
      }
      for (int tt = 0; tt < n_tiles; ++tt, ++jg) {
        const bool s_ok = wok && wwait(B_SFULL + (jg & 1), (jg / 2) & 1);
        wok = s_ok;
        uint32_t v[16];
        if (s_ok) {
          tc::fence_after();
          tc::tmem_ld16(lane_addr + COL_S + 16 * (jg & 1), v);
          tc::tmem_wait_ld();
        }
        const int key0 = b_begin * 64 + tt * KEYS;
        const bool valid = s_ok && key0 + ts < key_end;
        float x[G];
        bool want = !wok;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          x[h] = valid ? __uint_as_float(v[h]) * sc : -INFINITY;
          want |= x[h] > m_ref[h] + 8.0f;
        }
        // one barrier per tile: does any score outgrow its head's reference max
        // (or did a wait run out)?
        if (tc::bar_or(1, 128, want)) {
          float* rx = red + (xc & 1) * 64;
          ++xc;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float mx = x[h];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) rx[wq * 16 + h] = mx;
          }
          if (!tc::bar_and(1, 128, wok)) { ok = false; break; }  // also orders rx
          bool resc = false;
          float alpha[G];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float M = fmaxf(fmaxf(rx[h], rx[16 + h]), fmaxf(rx[32 + h], rx[48 + h]));
            alpha[h] = 1.0f;
            if (M > m_ref[h] + 8.0f) {
              alpha[h] = fast_exp2(m_ref[h] - M);
              m_ref[h] = M;
              resc = true;
            }
            lsum[h] *= alpha[h];
          }
          if (resc && tt > 0) {
            // O must hold P*V of the previous tile before it is rescaled
            wok = wok && wwait(B_ODONE + ((jg - 1) & 1), ((jg - 1) / 2) & 1);
            if (wok) {
              tc::fence_after();
              uint32_t o[16];
              tc::tmem_ld16(lane_addr + COL_O + 16 * ob, o);
              tc::tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < G; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
              tc::tmem_st16(lane_addr + COL_O + 16 * ob, o);
              tc::tmem_wait_st();
            }
          }
        }
        float pv[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          pv[h] = valid ? fast_exp2(x[h] - m_ref[h]) : 0.0f;
          lsum[h] += pv[h];
        }
        // rows of this tile past the unit's last key: zero their V (both halves)
        if (key0 + KEYS > key_end && !valid) {
          const uint32_t st = jg % STAGES;
          (void)mbar_wait_bounded(&bar[B_VFULL + st], (jg / STAGES) & 1);  // the tile's V landed
          uint4* vr = reinterpret_cast<uint4*>(sm + st * STAGE_BYTES + KV_BYTES + ts * 128);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            vr[q] = make_uint4(0, 0, 0, 0);
            vr[HALF_BYTES / 16 + q] = make_uint4(0, 0, 0, 0);
          }
        }
        // P(jg) reuses the buffer of P(jg-2): its P*V must be done
        if (jg >= 2) wok = wok && wwait(B_ODONE + (jg & 1), ((jg - 2) / 2) & 1);
        uint8_t* pb = sm + OFF_P + (jg & 1) * QP_BYTES + (ts >> 6) * ROWS16_BYTES;
        const int unit16 = (ts & 63) >> 3, e = ts & 7;
#pragma unroll
        for (int h = 0; h < G; ++h)
          *reinterpret_cast<uint16_t*>(pb + (h >> 3) * 1024 + (h & 7) * 128 + ((unit16 ^ (h & 7)) << 4) + 2 * e) =
              to_bits<BF16>(pv[h]);
        // every lane's P (and V-row) stores are made visible to the MMA (async
        // proxy) and its tensor-memory reads ordered, then one lane arrives for
        // the warp: 128 arrivals on one barrier word cost ~600 cycles
        tc::fence_proxy_async();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_PFULL + (jg & 1)]);
      }
      if (!ok) break;
      // ---- epilogue: row sums over the 128 keys, then O / l or the partials
      float* rs = red + 2 * 64;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float sum = lsum[h];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) rs[wq * 16 + h] = sum;
      }
      wok = wok && wwait(B_ODONE + ((jg - 1) & 1), ((jg - 1) / 2) & 1);
      uint32_t o[16];
      if (wok) {
        tc::fence_after();
        tc::tmem_ld16(lane_addr + COL_O + 16 * ob, o);
        tc::tmem_wait_ld();
      }
      if (!tc::bar_and(1, 128, wok)) { ok = false; break; }  // also orders rs
      float l[G];
#pragma unroll
      for (int h = 0; h < G; ++h) l[h] = (rs[h] + rs[16 + h]) + (rs[32 + h] + rs[48 + h]);
      if (wslot < 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          out[(int64_t)t * a.Hq * D + (c * G + h) * D + ts] = to_bits<BF16>(__uint_as_float(o[h]) * (1.f / l[h]));
      } else {
        float* wo = ws + ws_o_offset(n_items, a.Hq);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const int hq = c * G + h;
          wo[((int64_t)wslot * a.Hq + hq) * D + ts] = __uint_as_float(o[h]);
          if (ts == h) {
            ws[((int64_t)wslot * a.Hq + hq) * 2] = m_ref[h];
            ws[((int64_t)wslot * a.Hq + hq) * 2 + 1] = l[h];
          }
        }
        if (FUSED && counters != nullptr) {
          // hand the unit to the merge warp, which counts it done and, for
          // the last split of (row, KV head c), merges all partials; the
          // softmax warps go on with the next unit meanwhile
          const int q = mq % MQ;
          if (mq >= MQ) wok = wok && wwait(B_MEMPTY + q, ((mq / MQ) - 1) & 1);
          if (ts == 0) {
            int* r = mrec + q * MREC_INTS;
            r[0] = seq;
            r[1] = c;
            r[2] = wslot;
            r[3] = t;
            r[4] = pos;
            r[5] = b_begin;
          }
          ++mq;
          __syncwarp();  // this warp's partials and (lane 0 of warp 4) the record
          if (lane == 0) tc::mbar_arrive(&bar[B_MFULL + q]);
        }
      }
      // the row-sum scratch is reused by the next unit
      tc::bar_sync(1, 128);
    }
    if (!ok) set_dev_error(hdr, DS_DEVERR_WORKLIST);
    if (FUSED && counters != nullptr) {
      // end of the merge warp's records (bounded: the slot's previous record
      // may still be in use)
      const int q = mq % MQ;
      if (mq >= MQ) (void)wwait(B_MEMPTY + q, ((mq / MQ) - 1) & 1);
      if (ts == 0) mrec[q * MREC_INTS] = -1;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[B_MFULL + q]);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- merge warp
    // (fused decode with counters) for each multi-split unit the softmax warps
    // finished: publish its partials (this fence is cumulative: it covers the
    // softmax threads' writes this warp acquired through the record's
    // barrier), count it done on the (row, KV head) counter, and if it is the
    // last split, merge every split's partials (the combine kernel's
    // arithmetic, in its order) into the output row and reset the counter.
    if (FUSED && counters != nullptr) {
      for (uint32_t i = 0;; ++i) {
        const int q = i % MQ;
        if (!warp_wait(B_MFULL + q, (i / MQ) & 1)) {
          if (lane == 0) set_dev_error(hdr, DS_DEVERR_WORKLIST);
          break;
        }
        const int* r = mrec + q * MREC_INTS;
        const int seq = r[0], c = r[1], wslot = r[2], t = r[3], pos = r[4], b_begin = r[5];
        __syncwarp();
        if (seq < 0) break;
        const int split = hdr[HDR_SPLIT];
        const int nb = (pos + 1 + 63) / 64;
        const int cnt = (nb + split - 1) / split;
        const int first = wslot - b_begin / split;  // a row's splits hold consecutive slots
        int last = 0;
        if (lane == 0) {
          __threadfence();
          last = atomicAdd(&counters[seq * a.Hkv + c], 1) == cnt - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          const float* wo = ws + ws_o_offset(n_items, a.Hq);
          for (int h = 0; h < G; ++h) {
            const int hq = c * G + h;
            float M = -1.0e30f;
            for (int k2 = 0; k2 < cnt; ++k2) M = fmaxf(M, __ldcg(ws + ((int64_t)(first + k2) * a.Hq + hq) * 2));
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, lt = 0.f;
            for (int k2 = 0; k2 < cnt; ++k2) {
              const float* ml = ws + ((int64_t)(first + k2) * a.Hq + hq) * 2;
              const float scl = fast_exp2(__ldcg(ml) - M);
              lt += scl * __ldcg(ml + 1);
              const float* src = wo + ((int64_t)(first + k2) * a.Hq + hq) * D;
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[e] += scl * __ldcg(src + lane + 32 * e);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
              out[(int64_t)t * a.Hq * D + hq * D + lane + 32 * e] = to_bits<BF16>(acc[e] * (1.f / lt));
          }
          if (lane == 0) counters[seq * a.Hkv + c] = 0;  // ready for the next launch
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_MEMPTY + q]);
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    // the last CTA to finish resets the unit counter for the next launch (every
    // CTA has stopped taking units before it counts itself done)
    __threadfence();
    if (atomicAdd(&hdr[HDR_DEC_DONE], 1) == (int)gridDim.x - 1) {
      atomicExch(&hdr[HDR_DEC_NEXT], 0);
      atomicExch(&hdr[HDR_DEC_DONE], 0);
    }
  }
}

template <bool BF16, bool HALF, int G>
static cudaError_t launch_dtc_t(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                const void* pool, void* out, float* ws, cudaStream_t st,
                                bool overlap_previous, bool fused, int32_t* counters) {
  CUtensorMap map;
  cudaError_t e = make_pool_map(&map, pool, a);
  if (e != cudaSuccess) return e;
  auto kern = fused ? decode_tc_kernel<BF16, HALF, G, true> : decode_tc_kernel<BF16, HALF, G, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dtc::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM, fewer for a small batch (unless the launch
  // must serve any batch within the capacities)
  const int64_t units = (m.flags & DS_META_CAPACITY) ? (int64_t)sms : (int64_t)m.n_decode_items * a.Hkv;
  const int cap = DSR_DTC_MAX_CTAS > 0 ? std::min(sms, DSR_DTC_MAX_CTAS) : sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>(units, cap)));
  cfg.blockDim = dim3(dtc::THREADS);
  cfg.dynamicSmemBytes = dtc::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // After the prefill kernel, decode CTAs may take the SMs it leaves idle: the
  // two read only what the KV append wrote before either started and write
  // disjoint output rows.
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, map, reinterpret_cast<const int4*>(m.decode_items), m.cu_seqlens,
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

template <bool BF16, bool HALF>
static cudaError_t launch_dtc_g(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                const void* pool, void* out, float* ws, cudaStream_t st, bool ov,
                                bool fu, int32_t* cnt) {
  switch (a.G) {
    case 2: return launch_dtc_t<BF16, HALF, 2>(m, a, qkv, pool, out, ws, st, ov, fu, cnt);
    case 4: return launch_dtc_t<BF16, HALF, 4>(m, a, qkv, pool, out, ws, st, ov, fu, cnt);
    case 8: return launch_dtc_t<BF16, HALF, 8>(m, a, qkv, pool, out, ws, st, ov, fu, cnt);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_tc(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                             const void* pool, void* out, float* ws, cudaStream_t st,
                             bool overlap_previous, bool fused_append, int32_t* counters) {
  const bool half = a.style == DS_ROPE_HALF;
  const bool ov = overlap_previous, fu = fused_append;
  if (a.dtype == DS_BF16)
    return half ? launch_dtc_g<true, true>(m, a, qkv, pool, out, ws, st, ov, fu, counters)
                : launch_dtc_g<true, false>(m, a, qkv, pool, out, ws, st, ov, fu, counters);
  return half ? launch_dtc_g<false, true>(m, a, qkv, pool, out, ws, st, ov, fu, counters)
              : launch_dtc_g<false, false>(m, a, qkv, pool, out, ws, st, ov, fu, counters);
}

}  // namespace dsr

#ifdef DSR_TEST_WAIT_RUNOUT
// Test builds only (not part of the C ABI): stall (1) or release (0) the
// decode producers' copies on the current device.
extern "C" ds_status ds_test_stall_copies(int32_t on) {
  const int v = on ? 1 : 0;
  return cudaMemcpyToSymbol(dsr::g_test_stall_copies, &v, sizeof v) == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}
#endif
