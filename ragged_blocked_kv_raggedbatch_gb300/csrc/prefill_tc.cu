// prefill_tc.cu -- blocked causal attention for prefill chunks on the 5th-gen
// tensor cores (tcgen05 MMAs with accumulators in tensor memory, K/V tiles
// staged by tiled TMA loads).
//
// Work atom ("DeepSpeed Inference v2", pyshine.com/deepspeed-2, section "Ragged
// batches": AtomBuilder atoms executed by BlockedFlashAttn, q-block size chosen
// per head size): up to 256/G consecutive new tokens of one sequence and one
// KV head c, as two Q tiles of 128 rows (tokens x the G query heads that read
// KV head c).  Both tiles share every 128-key K/V tile, which is two 64-token
// pool blocks fetched through the block table.  The grid is persistent: each
// CTA takes the next atom of the longest-first list when it is ready for one;
// the K/V ring, barrier phases and tensor memory carry over from one atom to
// the next.
//
// Roles (12 warps = 3 warpgroups; launched at 168 registers a thread, the
// first warpgroup gives registers back (setmaxnreg 96) and the two softmax
// warpgroups take them (setmaxnreg 200): 128*96 + 2*128*200 <= 384*168):
//   warp 0      takes the atoms (longest first, from a counter in the batch
//               header, one as the previous one's last tile is issued),
//               decodes them and hands them to the others through a ring in
//               shared memory; TMA producer: K and V tiles into
//               2-stage rings whose slots are
//               freed separately (K after the last QK MMA that reads it, V after
//               the last PV MMA), so each K tile is requested about a step and a
//               half before its first QK; zeroes the rows of the final V tile
//               past the chunk's last key (those slots may hold anything and
//               0 * NaN would poison P*V).
//   warp 1      tensor-memory owner and MMA issuer (the warp walks the schedule
//               and builds warp-uniform descriptors; one elected lane issues):
//                 S_X = Q_X K_t^T   (SS MMA, 128 x 128 x D)
//                 O_X += P_X V_t    (TS MMA: P read from tensor memory, in two
//                                    halves of 64 keys, each issued as soon as
//                                    the softmax has written it)
//               issued as QK_A(0) QK_B(0) | PV_A(t) QK_A(t+1) PV_B(t) QK_B(t+1) ...
//               so one tile's softmax overlaps the other tile's MMAs.
//   warps 2-3   no work (they only return their registers)
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: one thread per
//               row (tensor-memory lane = row).  Per atom the tile's 4 warps
//               copy its Q rows into 128-byte-swizzled shared memory with
//               coalesced loads, then each thread rotates its own row in place
//               (fp32, same rule as the append); per KV tile: masked row max,
//               conditional rescale of O (only when the max grows by more than
//               2^8: the reference max may lag, the final O / l is exact),
//               P = exp2(S - m) written back over S as packed 16-bit pairs;
//               epilogue: O / l staged in the tile's Q buffer, written out with
//               coalesced stores.
// Tensor memory: S_A [0,128) S_B [128,256) O_A [256,256+D) O_B [256+D,256+2D).
// Every mbarrier wait is bounded: on timeout the CTA records an error and stops.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "tc.cuh"

// Register split (per thread) between the producer/MMA warpgroup and the two
// softmax warpgroups; 128 * LOW + 256 * HIGH must not exceed 384 * 168.
// 96/200 is the split with no spill in any instance; on GB300 (chunked
// prefill 2x8192, attention) 80/208 2.707 ms, 88/200 2.712-2.717, 96/200 2.703.
#ifndef DSR_PF_REG_LOW
#define DSR_PF_REG_LOW 96
#endif
#ifndef DSR_PF_REG_HIGH
#define DSR_PF_REG_HIGH 200
#endif
static_assert(128 * DSR_PF_REG_LOW + 256 * DSR_PF_REG_HIGH <= 384 * 168, "register split over the launch budget");
// 1: K/V tile loads carry an L2 evict_last policy (every atom of a chunk re-reads
// its sequence's K/V prefix from L2).
#ifndef DSR_PF_EVICT_LAST
#define DSR_PF_EVICT_LAST 0
#endif

namespace dsr {

template <int D>
struct PfCfg {
  static constexpr int ROWS = 128;
  static constexpr int KEYS = 128;
  static constexpr int HALVES = D / 64;
  static constexpr int QHALF = ROWS * 128;      // one 64-column chunk of a Q tile
  static constexpr int KHALF = KEYS * 128;      // one 64-column chunk of a K or V tile
  static constexpr int QTILE = HALVES * QHALF;
  static constexpr int KVTILE = HALVES * KHALF;
  static constexpr int BOX_BYTES = 64 * 128;    // one TMA box: 64 keys x 64 elements
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * QTILE;
  static constexpr int OFF_BAR = OFF_KV + 2 * 2 * KVTILE;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  static constexpr int COL_S0 = 0, COL_O0 = 256;
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 384;
};

// K and V slots of a ring stage are released separately: K once the last
// QK MMA of its step has read it, V once the last PV MMA has, so the next K
// tile is requested a whole step before it is needed.
// P is handed to the P*V MMAs in two halves of 64 keys (B_PFULL + 2x + half):
// the first four K-steps of P*V start while the softmax still computes the
// second half.  B_ODONE0 + x: the first half of P*V(x) is done (its P columns
// may be overwritten).
// B_AFULL / B_AEMPTY: the atom ring (AQ slots) the scheduler warp fills.
constexpr int AQ = 4;
enum {
  B_QREADY = 0, B_KFULL = 2, B_VFULL = 4, B_KEMPTY = 6, B_SFULL = 8, B_PFULL = 10,
  B_ODONE = 14, B_ODONE0 = 16, B_VLAST = 18, B_DONE = 19, B_VEMPTY = 20, B_AFULL = 22,
  B_AEMPTY = B_AFULL + AQ, B_QRAW = B_AEMPTY + AQ, B_OSTG = B_QRAW + 2, B_OFREE = B_OSTG + 2,
  B_COUNT = B_OFREE + 2
};
// arrivals that free an atom slot: the MMA warp, 8 softmax warps
constexpr int AEMPTY_ARRIVALS = 9;
// an atom ring slot: index, valid flag, then the atom's fields as the
// producer decoded them (seq, j0, ntok, kv_len, c, seen, first token, block
// table offset), so the other roles read no metadata from global memory
constexpr int AW = 10;
static_assert(8 * B_COUNT + 4 + 4 * AW * AQ <= 512, "barriers, tensor-memory slot and atom ring fit the reserved bytes");

template <bool BF16, bool HALF, int D, int G, bool FUSED>
__global__ void __launch_bounds__(384, 1) prefill_tc_kernel(
    const __grid_constant__ CUtensorMap pool_map, const int4* __restrict__ tiles,
    const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ seq_seen,
    const int32_t* __restrict__ seq_new, const int32_t* __restrict__ blk_off,
    const int32_t* __restrict__ block_table, const int32_t* __restrict__ tok_seq,
    const int32_t* __restrict__ tok_pos, const uint16_t* __restrict__ qkv, uint16_t* __restrict__ pool,
    uint16_t* __restrict__ out, LayerArgs a) {
  using C = PfCfg<D>;
  constexpr int T = 128 / G;  // tokens per Q tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * B_COUNT);
  int* aring = reinterpret_cast<int*>(sm + C::OFF_BAR + 8 * B_COUNT + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* hdr = a.header;

  // Every CTA of this grid stays resident until the prefill work is done, so
  // the decode launch that follows (it needs nothing from this kernel) may
  // start at once on the SMs this grid does not use.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // The batch's atoms and the CTAs that take them (a launch sized by the
  // capacities has more CTAs; those exit here).
  const int n_atoms = hdr[HDR_PRE_TILES] * a.Hkv;
  int n_ctas = hdr[HDR_PRE_CTAS];
  if (n_ctas <= 0 || n_ctas > (int)gridDim.x) n_ctas = gridDim.x;
  n_ctas = min(n_ctas, n_atoms);
  if ((int)blockIdx.x >= n_ctas) return;

  if (FUSED) {
    // KV append of the prefill chunks' new tokens (decode rows are the decode
    // kernel's), spread over every working CTA; then a grid barrier, so that
    // every atom's K/V tiles hold their chunk's new rows before any is loaded.
    // The launch is cooperative: all n_ctas CTAs are resident, and the wait
    // is bounded.
    // One warp per token; a token's units (Hkv * (D/16 + D/8), at most 192)
    // are spread over the lanes, unrolled so their loads are in flight together.
    const int N = hdr[HDR_N];
    constexpr int U = D / 16 + D / 8;
    const int units = a.Hkv * U;
    const int n_warps = n_ctas * (C::THREADS / 32);
    for (int t = blockIdx.x * (C::THREADS / 32) + warp; t < N; t += n_warps) {
      const int seq = tok_seq[t];
      if (seq_new[seq] == 1) continue;
      const int p = tok_pos[t];
      if (p >= a.max_positions) {
        if (lane == 0) set_dev_error(hdr, DS_DEVERR_POSITION);
        continue;
      }
      const int blk = block_table[blk_off[seq] + p / kBlockSize];
      if (blk < 0 || blk >= a.num_blocks) {
        if (lane == 0) set_dev_error(hdr, DS_DEVERR_BLOCK_ID);
        continue;
      }
      const uint16_t* row = qkv + (int64_t)t * ((a.Hq + 2 * a.Hkv) * D);
      const float4* cs_row = reinterpret_cast<const float4*>(a.rope + (int64_t)p * (D / 2));
#pragma unroll 6
      for (int u = lane; u < units; u += 32) append_unit<BF16, HALF, D>(u, row, cs_row, pool, blk, p % kBlockSize, a);
    }
    tc::fence_proxy_async_global();  // this thread's pool writes -> the TMA loads below
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicAdd(&hdr[HDR_PRE_BAR], 1);
      const long long t0 = clock64();
      while (*reinterpret_cast<volatile int32_t*>(&hdr[HDR_PRE_BAR]) < n_ctas) {
        if (clock64() - t0 > DSR_WAIT_LIMIT) {
          set_dev_error(hdr, DS_DEVERR_WORKLIST);
          break;
        }
      }
      __threadfence();
    }
    __syncthreads();
  }

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar[B_QREADY + s], 128);
      mbar_init(&bar[B_KFULL + s], 1);
      mbar_init(&bar[B_VFULL + s], 1);
      mbar_init(&bar[B_KEMPTY + s], 1);
      mbar_init(&bar[B_VEMPTY + s], 1);
      mbar_init(&bar[B_SFULL + s], 1);
      mbar_init(&bar[B_PFULL + 2 * s], 4);  // one arrival per softmax warp
      mbar_init(&bar[B_PFULL + 2 * s + 1], 4);
      mbar_init(&bar[B_ODONE + s], 1);
      mbar_init(&bar[B_ODONE0 + s], 1);
    }
    mbar_init(&bar[B_VLAST], 1);
    for (int q = 0; q < AQ; ++q) {
      mbar_init(&bar[B_AFULL + q], 1);
      mbar_init(&bar[B_AEMPTY + q], AEMPTY_ARRIVALS);
    }
    mbar_init(&bar[B_DONE], 256);
    for (int s = 0; s < 2; ++s) {  // the 4 softmax warps of a tile
      mbar_init(&bar[B_QRAW + s], 4);
      mbar_init(&bar[B_OSTG + s], 4);
      mbar_init(&bar[B_OFREE + s], 4);
    }
    fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sKV = sm + C::OFF_KV;

  // Atom k of the work list: one (prefill tile, KV head) pair, tiles longest
  // first, KV heads in groups (see below).  Each role walks
  // the same atoms and skips the same malformed ones.
  // Atoms are taken dynamically, longest first: the TMA producer takes the
  // next index from a counter in the batch header when it has issued the
  // last K/V tile of its current atom (so a CTA holds at most about two KV
  // steps of look-ahead), and publishes it in a ring of AQ slots that the
  // MMA and softmax warps read in order (so all walk the same atoms).  A
  // static assignment left a 120 us straggler on the max ragged batch, whose
  // atoms span 32 to 24,872 keys; a scheduler warp filling the ring ahead let
  // one CTA take several of the longest atoms at once.  next_atom returns -1
  // when the atoms are exhausted or a wait ran out (then ok = false).
  struct Atom {
    int seq, j0, ntok, kv_len, c, s_seen, tok0, n_kv;
    bool has_b;
    const int* btab;
  };
  const int n_tiles = hdr[HDR_PRE_TILES];
  auto load_atom = [&](int k, Atom& at) -> bool {
    // Tiles longest first in rounds of R = n_ctas / hg tiles; within a
    // round, the KV heads in groups of hg (the batch header's choice), each
    // group's atoms tile-major.  hg = all heads is plain tile-major order:
    // the atoms running at once then read every head's K/V prefix; with a
    // smaller hg they read those of hg heads, which L2 holds more easily.
    int hg = hdr[HDR_PRE_HG];
    if (hg <= 0 || hg > a.Hkv || a.Hkv % hg != 0) hg = a.Hkv;
    const int R = max(1, n_ctas / hg);        // tiles per round
    const int round = k / (R * a.Hkv);
    const int t0 = round * R;                 // first tile of the round
    const int rt = min(R, n_tiles - t0);      // tiles in the round
    const int j = k - round * R * a.Hkv;      // atom within the round, < rt * Hkv
    const int jj = j % (rt * hg);
    const int4 tl = tiles[t0 + jj / hg];
    at.c = (j / (rt * hg)) * hg + jj % hg;
    at.seq = tl.x; at.j0 = tl.y; at.ntok = tl.z; at.kv_len = tl.w;
    at.s_seen = seq_seen[at.seq];
    at.tok0 = cu_seqlens[at.seq] + at.j0;
    at.btab = block_table + blk_off[at.seq];
    at.has_b = at.ntok > T;
    at.n_kv = (at.kv_len + C::KEYS - 1) / C::KEYS;
    if (at.ntok <= 0 || at.ntok > 2 * T || at.kv_len != at.s_seen + at.j0 + at.ntok) {
      if (tid == 0) set_dev_error(a.header, DS_DEVERR_WORKLIST);
      return false;
    }
    if (at.kv_len > a.max_positions) {
      if (tid == 0) set_dev_error(a.header, DS_DEVERR_POSITION);
      return false;
    }
    return true;
  };
  // The next atom from the ring (AQ slots the producer fills in order): its
  // index (-1 when the atoms are exhausted or a wait ran out, then ok =
  // false), whether it is well formed, and its fields.
  auto next_atom = [&](uint32_t& i, bool& ok, Atom& at, bool& valid) -> int {
    const int q = i % AQ;
    const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&bar[B_AFULL + q], (i / AQ) & 1));
    int k = -1;
    valid = false;
    if (got) {
      const int* sl = aring + q * AW;
      k = sl[0];
      valid = sl[1] != 0;
      at.seq = sl[2]; at.j0 = sl[3]; at.ntok = sl[4]; at.kv_len = sl[5];
      at.c = sl[6]; at.s_seen = sl[7]; at.tok0 = sl[8];
      at.btab = block_table + sl[9];
      at.has_b = at.ntok > T;
      at.n_kv = (at.kv_len + C::KEYS - 1) / C::KEYS;
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bar[B_AEMPTY + q]);
    ++i;
    if (!got) ok = false;
    return k;
  };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(DSR_PF_REG_LOW) : "memory");
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      const uint32_t box_tx = C::HALVES * C::BOX_BYTES;
      uint32_t ring = 0, vlast_uses = 0;
#if DSR_PF_EVICT_LAST
      const uint64_t pol = tc::policy_evict_last();
#define DSR_PF_TMA(dst, c0, c1, b) tc::tma_load_2d_hint(dst, &pool_map, c0, c1, b, pol)
#else
#define DSR_PF_TMA(dst, c0, c1, b) tc::tma_load_2d(dst, &pool_map, c0, c1, b)
#endif
      bool ok = true;
      for (uint32_t ai = 0; ok; ++ai) {
        // take the next atom and hand it to the MMA and softmax warps
        const int q = ai % AQ;
        if (ai >= AQ && !__all_sync(0xffffffffu, mbar_wait_bounded(&bar[B_AEMPTY + q], ((ai / AQ) - 1) & 1))) {
          ok = false;
          break;
        }
        int k = 0;
        if (lane == 0) k = atomicAdd(&hdr[HDR_PRE_NEXT], 1);
        k = __shfl_sync(0xffffffffu, k, 0);
        if (k >= n_atoms) k = -1;
        Atom at;
        const bool valid = k >= 0 && load_atom(k, at);
        if (lane == 0) {
          int* sl = aring + q * AW;
          sl[0] = k;
          sl[1] = valid ? 1 : 0;
          if (valid) {
            sl[2] = at.seq; sl[3] = at.j0; sl[4] = at.ntok; sl[5] = at.kv_len;
            sl[6] = at.c; sl[7] = at.s_seen; sl[8] = at.tok0;
            sl[9] = (int)(at.btab - block_table);
          }
          tc::mbar_arrive(&bar[B_AFULL + q]);
        }
        if (k < 0) break;
        if (!valid) continue;
        for (int t = 0; t < at.n_kv; ++t, ++ring) {
          const int st = ring & 1;
          const uint32_t empty_par = ((ring >> 1) - 1) & 1;
          const bool has1 = t * C::KEYS + 64 < at.kv_len;
          uint8_t* kdst = sKV + st * 2 * C::KVTILE;
          uint8_t* vdst = kdst + C::KVTILE;
          const bool last_partial = (t == at.n_kv - 1) && (at.kv_len % C::KEYS != 0);
          uint64_t* vbar = last_partial ? &bar[B_VLAST] : &bar[B_VFULL + st];
          int blk[2] = {0, 0};
          for (int i = 0; i < (has1 ? 2 : 1); ++i) {
            blk[i] = at.btab[2 * t + i];
            if (blk[i] < 0 || blk[i] >= a.num_blocks) {
              if (lane == 0) set_dev_error(a.header, DS_DEVERR_BLOCK_ID);
              blk[i] = 0;
            }
          }
          const uint32_t tx = (has1 ? 2u : 1u) * box_tx;
          // K slot free (the QK MMAs of ring step ring-2 are done)
          if (ring >= 2 && !mbar_wait_bounded(&bar[B_KEMPTY + st], empty_par)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&bar[B_KFULL + st], tx);
            for (int i = 0; i < (has1 ? 2 : 1); ++i) {
              const int krow = ((blk[i] * 2 + 0) * a.Hkv + at.c) * 64;
#pragma unroll
              for (int h = 0; h < C::HALVES; ++h)
                DSR_PF_TMA(kdst + h * C::KHALF + i * C::BOX_BYTES, h * 64, krow, &bar[B_KFULL + st]);
            }
          }
          // V slot free (the PV MMAs of ring step ring-2 are done)
          if (ring >= 2 && !mbar_wait_bounded(&bar[B_VEMPTY + st], empty_par)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(vbar, tx);
            for (int i = 0; i < (has1 ? 2 : 1); ++i) {
              const int vrow = ((blk[i] * 2 + 1) * a.Hkv + at.c) * 64;
#pragma unroll
              for (int h = 0; h < C::HALVES; ++h)
                DSR_PF_TMA(vdst + h * C::KHALF + i * C::BOX_BYTES, h * 64, vrow, vbar);
            }
          }
          if (last_partial) {
            if (!mbar_wait_bounded(&bar[B_VLAST], vlast_uses & 1)) {
              ok = false;
              break;
            }
            ++vlast_uses;
            const int first_bad = at.kv_len - t * C::KEYS;  // rows [first_bad, 128) hold no key
            const int n16 = (C::KEYS - first_bad) * 8;      // 16-byte chunks per half
            for (int h = 0; h < C::HALVES; ++h)
              for (int i = lane; i < n16; i += 32)
                *reinterpret_cast<uint4*>(vdst + h * C::KHALF + first_bad * 128 + i * 16) =
                    make_uint4(0, 0, 0, 0);
            tc::fence_proxy_async();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar[B_VFULL + st]);
          }
        }
      }
#undef DSR_PF_TMA
      if (!ok && lane == 0) set_dev_error(a.header, DS_DEVERR_WORKLIST);
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      // The whole warp walks the schedule, waits on the barriers and builds the
      // operand descriptors (warp-uniform values); one elected lane issues each
      // group of MMAs and every commit, so all commits track its MMAs.
      {
        constexpr uint32_t IQK = tc::idesc_f16(BF16, 128, 128, false);
        constexpr uint32_t IPV = tc::idesc_f16(BF16, 128, D, true);
        auto wait = [&](int b, uint32_t parity) -> bool {
          return __all_sync(0xffffffffu, mbar_wait_bounded(&bar[b], parity));
        };
        auto commit = [&](int b) {
          if (tc::elect_one()) tc::mma_commit(&bar[b]);
          __syncwarp();
        };
        // descriptor start-address field = byte address / 16 (addresses stay
        // below 256 KB, so adding an offset / 16 never carries out of it)
        auto qk = [&](int x, uint32_t r) {
          const uint64_t qd = tc::smem_desc_sw128(smem_u32(sQ + x * C::QTILE), 16, 1024);
          const uint64_t kd = tc::smem_desc_sw128(smem_u32(sKV + (r & 1) * 2 * C::KVTILE), 16, 1024);
          if (tc::elect_one()) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t oq = ((ks / 4) * C::QHALF + (ks % 4) * 32) >> 4;
              const uint32_t ok_ = ((ks / 4) * C::KHALF + (ks % 4) * 32) >> 4;
              tc::mma_ss(tmem + C::COL_S0 + 128 * x, qd + oq, kd + ok_, IQK, ks > 0);
            }
            tc::mma_commit(&bar[B_SFULL + x]);
          }
          __syncwarp();
        };
        // O_x += P_x V_t in two halves of 64 keys, each issued once the
        // softmax has written that half of P
        auto pv = [&](int x, uint32_t r, bool acc, uint32_t parity) -> bool {
          const uint64_t vd =
              tc::smem_desc_sw128(smem_u32(sKV + (r & 1) * 2 * C::KVTILE + C::KVTILE), C::KHALF, 1024);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (!wait(B_PFULL + 2 * x + half, parity)) return false;
            tc::fence_after();
            if (tc::elect_one()) {
#pragma unroll
              for (int kk = 4 * half; kk < 4 * half + 4; ++kk)
                tc::mma_ts(tmem + C::COL_O0 + D * x, tmem + C::COL_S0 + 128 * x + 8 * kk,
                           vd + ((kk * 2048) >> 4), IPV, (acc || kk > 0));
              tc::mma_commit(&bar[(half ? B_ODONE : B_ODONE0) + x]);
            }
            __syncwarp();
          }
          return true;
        };
        uint32_t ring = 0, qn[2] = {0, 0}, stp[2] = {0, 0};
        bool ok = true;
        for (uint32_t ai = 0; ok;) {
          Atom at;
          bool av;
          const int k = next_atom(ai, ok, at, av);
          if (k < 0) break;
          if (!av) continue;
          ok = wait(B_QREADY + 0, qn[0] & 1) && wait(B_KFULL + (ring & 1), (ring >> 1) & 1);
          ++qn[0];
          if (!ok) break;
          tc::fence_after();
          qk(0, ring);
          if (at.has_b) {
            ok = wait(B_QREADY + 1, qn[1] & 1);
            ++qn[1];
            if (!ok) break;
            tc::fence_after();
            qk(1, ring);
          }
          commit(B_KEMPTY + (ring & 1));
          for (int t = 0; t < at.n_kv; ++t) {
            const uint32_t r = ring + t;
            ok = wait(B_VFULL + (r & 1), (r >> 1) & 1) && pv(0, r, t > 0, stp[0] & 1);
            if (!ok) break;
            ++stp[0];
            if (t + 1 < at.n_kv) {
              ok = wait(B_KFULL + ((r + 1) & 1), ((r + 1) >> 1) & 1);
              if (!ok) break;
              tc::fence_after();
              qk(0, r + 1);
            }
            if (at.has_b) {
              ok = pv(1, r, t > 0, stp[1] & 1);
              if (!ok) break;
              ++stp[1];
            }
            commit(B_VEMPTY + (r & 1));
            if (t + 1 < at.n_kv) {
              if (at.has_b) qk(1, r + 1);
              commit(B_KEMPTY + ((r + 1) & 1));
            }
          }
          ring += at.n_kv;
        }
        if (!ok && lane == 0) set_dev_error(a.header, DS_DEVERR_WORKLIST);
      }
      __syncwarp();
      // free tensor memory once every softmax thread has read its last values
      (void)mbar_wait_bounded(&bar[B_DONE], 0);
      __syncwarp();
      tc::fence_after();
      tc::tmem_dealloc(tmem, C::TMEM_COLS);
      tc::tmem_relinquish();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(DSR_PF_REG_HIGH) : "memory");
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) >> 2;            // 0: tile A, 1: tile B
    const int r = 32 * (warp & 3) + lane;     // row = tensor-memory lane
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t col_s = C::COL_S0 + 128 * x;
    const uint32_t col_o = C::COL_O0 + D * x;
    const float sc = a.scale_log2;
    uint32_t stp = 0;   // KV steps of tile x done by this CTA
    uint32_t qraw = 0;  // Q tiles this tile's warps copied
    uint32_t ostg = 0;  // outputs this tile's warps staged and wrote
    bool ok = true;
    for (uint32_t ai = 0; ok;) {
      Atom at;
      bool av;
      const int k = next_atom(ai, ok, at, av);
      if (k < 0) break;
      if (!av) continue;
      if (x == 1 && !at.has_b) continue;
      const int jt = x * T + r / G;             // token of this row inside the atom
      const bool valid = jt < at.ntok;
      const int pos = at.s_seen + at.j0 + min(jt, at.ntok - 1);

      // Q tile: the tile's 4 warps copy its 128 rows (row r = token r / G,
      // head r % G of KV group c) into 128-byte-swizzled shared memory with
      // coalesced 16-byte loads (the G heads of a token are contiguous), meet
      // at a bounded barrier, then each thread rotates its own row in place
      // (fp32, same rule as the append).  One thread loading its own row took
      // ~9000 cycles between two atoms: 32 rows per warp instruction.
      {
        uint8_t* qt = sQ + x * C::QTILE;
        const int64_t rs = (int64_t)(a.Hq + 2 * a.Hkv) * D;  // qkv row stride
        constexpr int CPR = D / 8;                           // 16-byte chunks per row
        constexpr int PER = 128 * CPR / 128;                 // chunks per thread
        const int tt = 32 * (warp & 3) + lane;               // 0..127 within the tile
        uint4 raw[PER];
#pragma unroll
        for (int k2 = 0; k2 < PER; ++k2) {
          const int i = tt + 128 * k2, row = i / CPR, cc = i % CPR;
          const int tj = x * T + row / G;
          raw[k2] = make_uint4(0, 0, 0, 0);
          if (tj < at.ntok)
            raw[k2] = ld_nc_v4(qkv + (int64_t)(at.tok0 + tj) * rs + (at.c * G + row % G) * D + 8 * cc);
        }
#pragma unroll
        for (int k2 = 0; k2 < PER; ++k2) {
          const int i = tt + 128 * k2, row = i / CPR, cc = i % CPR;
          *reinterpret_cast<uint4*>(qt + (cc / 8) * C::QHALF + row * 128 + (((cc % 8) ^ (row & 7)) << 4)) = raw[k2];
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_QRAW + x]);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bar[B_QRAW + x], qraw & 1))) {
          ok = false;
          break;
        }
        ++qraw;
        if (valid) {
          const float4* cs4 = reinterpret_cast<const float4*>(a.rope) + (int64_t)pos * (D / 4);
#pragma unroll
          for (int cc = 0; cc < D / 16; ++cc) {
            const int ch0 = HALF ? cc : 2 * cc;
            const int ch1 = HALF ? D / 16 + cc : 2 * cc + 1;
            uint4* p0 = reinterpret_cast<uint4*>(qt + (ch0 / 8) * C::QHALF + r * 128 + (((ch0 % 8) ^ (r & 7)) << 4));
            uint4* p1 = reinterpret_cast<uint4*>(qt + (ch1 / 8) * C::QHALF + r * 128 + (((ch1 % 8) ^ (r & 7)) << 4));
            uint4 x0 = *p0, x1 = *p1;
            float4 cs[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) cs[q] = __ldg(cs4 + 4 * cc + q);
            rotate16<BF16, HALF>(x0, x1, cs);
            *p0 = x0;
            *p1 = x1;
          }
        }
        tc::fence_proxy_async();
        tc::mbar_arrive(&bar[B_QREADY + x]);
      }

      float m_ref = -INFINITY, l = 0.f;  // m_ref in log2 units (scaled)
      for (int t = 0; t < at.n_kv; ++t, ++stp) {
        if (!mbar_wait_bounded(&bar[B_SFULL + x], stp & 1)) { ok = false; break; }
        tc::fence_after();
        // the whole S row of this KV tile, one wait
        uint32_t v[128];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tc::tmem_ld32(lane_addr + col_s + 32 * ch, v + 32 * ch);
        tc::tmem_wait_ld();
        const int kbase = t * C::KEYS;
        if (kbase + C::KEYS - 1 > pos) {  // diagonal tile: keys past this row's position
#pragma unroll
          for (int e = 0; e < 128; ++e)
            if (kbase + e > pos) v[e] = __float_as_uint(-INFINITY);
        }
        // row max of the raw scores (scale > 0 commutes with max)
        float m0 = __uint_as_float(v[0]), m1 = __uint_as_float(v[1]);
        float m2 = __uint_as_float(v[2]), m3 = __uint_as_float(v[3]);
#pragma unroll
        for (int e = 4; e < 128; e += 8) {
          m0 = tc::fmax3(m0, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
          m1 = tc::fmax3(m1, __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
          m2 = tc::fmax3(m2, __uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
          m3 = tc::fmax3(m3, __uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
        }
        const float mx = tc::fmax3(m0, m1, fmaxf(m2, m3)) * sc;
        // keep the reference max unless the row max outgrows it by 2^8
        bool mine = false;
        float alpha = 1.0f;
        if (t == 0) {
          m_ref = mx;
        } else if (mx > m_ref + 8.0f) {
          mine = true;
          alpha = fast_exp2(m_ref - mx);
          m_ref = mx;
        }
        // tensor-memory loads/stores are warp-collective: rescale O as a warp
        // whenever any of its rows needs it (alpha = 1 for the others), before
        // any P*V(t) accumulates into it; that needs P*V(t-1) complete
        const bool resc = t > 0 && __any_sync(0xffffffffu, mine);
        if (resc) {
          if (!mbar_wait_bounded(&bar[B_ODONE + x], (stp - 1) & 1)) { ok = false; break; }
          tc::fence_after();
          // 16 columns at a time: the 128 scores of the row are still live
#pragma unroll 1
          for (int ch = 0; ch < D / 16; ++ch) {
            uint32_t o[16];
            tc::tmem_ld16(lane_addr + col_o + 16 * ch, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::tmem_st16(lane_addr + col_o + 16 * ch, o);
          }
        }
        const float nm = -m_ref;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // P(t) overwrites P(t-1): that half of P*V(t-1) must be done
          if (t > 0 && !resc &&
              !mbar_wait_bounded(&bar[(half ? B_ODONE : B_ODONE0) + x], (stp - 1) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after();
#pragma unroll
          for (int ch = 2 * half; ch < 2 * half + 2; ++ch) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float y0, y1;
              tc::ffma2(y0, y1, __uint_as_float(v[32 * ch + 2 * e]), __uint_as_float(v[32 * ch + 2 * e + 1]),
                        sc, sc, nm, nm);
              const float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
              tc::fadd2(s0, s1, p0, p1);
              pk[e] = Stor<BF16>::pack(p0, p1);
            }
            tc::tmem_st16(lane_addr + col_s + 16 * ch, pk);
          }
          tc::tmem_wait_st();
          tc::fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&bar[B_PFULL + 2 * x + half]);
        }
        if (!ok) break;
        l = l * alpha + (s0 + s1);
      }
      if (!ok) break;
      // epilogue: the atom's last P*V, then O / l -> out.  Each thread
      // stages its row in the tile's Q buffer (its last QK is done), the 4
      // warps meet, and they write the rows out with coalesced 16-byte
      // stores (a thread storing its own row: 32 rows per warp instruction).
      if (!mbar_wait_bounded(&bar[B_ODONE + x], (stp - 1) & 1)) { ok = false; break; }
      tc::fence_after();
      {
        const float inv = 1.f / l;
        uint8_t* qt = sQ + x * C::QTILE;
        uint32_t v[D];
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tc::tmem_ld32(lane_addr + col_o + 32 * ch, v + 32 * ch);
        tc::tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < D / 8; ++cc) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = Stor<BF16>::pack(__uint_as_float(v[8 * cc + 2 * e]) * inv,
                                     __uint_as_float(v[8 * cc + 2 * e + 1]) * inv);
          *reinterpret_cast<uint4*>(qt + (cc / 8) * C::QHALF + r * 128 + (((cc % 8) ^ (r & 7)) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_OSTG + x]);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bar[B_OSTG + x], ostg & 1))) {
          ok = false;
          break;
        }
        constexpr int CPR = D / 8;            // 16-byte chunks per row
        const int tt = 32 * (warp & 3) + lane;
#pragma unroll
        for (int k2 = 0; k2 < CPR; ++k2) {
          const int i = tt + 128 * k2, row = i / CPR, cc = i % CPR;
          const int tj = x * T + row / G;
          if (tj < at.ntok)
            *reinterpret_cast<uint4*>(out + (int64_t)(at.tok0 + tj) * a.Hq * D + (at.c * G + row % G) * D + 8 * cc) =
                *reinterpret_cast<const uint4*>(qt + (cc / 8) * C::QHALF + row * 128 + (((cc % 8) ^ (row & 7)) << 4));
        }
        // the staging buffer is the next atom's Q buffer: every warp has read it first
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[B_OFREE + x]);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bar[B_OFREE + x], ostg & 1))) {
          ok = false;
          break;
        }
        ++ostg;
      }
    }
    if (!ok) set_dev_error(a.header, DS_DEVERR_WORKLIST);
    tc::fence_before();
    tc::mbar_arrive(&bar[B_DONE]);
  }
  // the last working CTA to finish re-arms the atom counter (and the fused
  // variant's grid barrier) for the next launch on the same upload: every CTA
  // took its last atom (and passed the barrier) before counting itself
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&hdr[HDR_PRE_DONE], 1) == n_ctas - 1) {
      atomicExch(&hdr[HDR_PRE_NEXT], 0);
      atomicExch(&hdr[HDR_PRE_BAR], 0);
      atomicExch(&hdr[HDR_PRE_DONE], 0);
    }
  }
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// The pool as a 2-D tensor [num_blocks*2*Hkv*64 rows][D]: row
// ((blk*2 + kv)*Hkv + head)*64 + offset; boxes of 64 rows x 64 elements with
// 128-byte swizzle.
cudaError_t make_pool_map(CUtensorMap* map, const void* pool, const LayerArgs& a) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)a.D, (cuuint64_t)a.num_blocks * 2 * a.Hkv * 64};
  cuuint64_t strides[1] = {(cuuint64_t)a.D * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, a.dtype == DS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  2, const_cast<void*>(pool), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool BF16, bool HALF, int D, int G>
static cudaError_t launch_prefill_t(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                    void* pool, void* out, cudaStream_t st, bool fused) {
  using C = PfCfg<D>;
  CUtensorMap map;
  cudaError_t e = make_pool_map(&map, pool, a);
  if (e != cudaSuccess) return e;
  auto kern = fused ? prefill_tc_kernel<BF16, HALF, D, G, true> : prefill_tc_kernel<BF16, HALF, D, G, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // Persistent grid: as many CTAs as SMs, or, with decode rows queued behind
  // this kernel, the SMs the prefill work needs to finish alongside them (the
  // kernel reads the same choice from the header); sized by the SM count
  // alone when the launch must serve any batch within the capacities.
  int ctas = sms;
  if (!(m.flags & DS_META_CAPACITY)) {
    const int n_atoms = m.n_prefill_tiles * a.Hkv;
    if (m.prefill_sms > 0.f) ctas = (int)std::ceil(m.prefill_sms);
    ctas = std::max(1, std::min(ctas, std::min(sms, n_atoms)));
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the fused append's grid barrier
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = fused ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, map, reinterpret_cast<const int4*>(m.prefill_tiles), m.cu_seqlens,
                         m.seq_seen, m.seq_new, m.blk_off, m.block_table, m.tok_seq, m.tok_pos,
                         static_cast<const uint16_t*>(qkv), static_cast<uint16_t*>(pool),
                         static_cast<uint16_t*>(out), a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool BF16, bool HALF, int D>
static cudaError_t launch_prefill_g(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                    void* pool, void* out, cudaStream_t st, bool fu) {
  switch (a.G) {
    case 1: return launch_prefill_t<BF16, HALF, D, 1>(m, a, qkv, pool, out, st, fu);
    case 2: return launch_prefill_t<BF16, HALF, D, 2>(m, a, qkv, pool, out, st, fu);
    case 4: return launch_prefill_t<BF16, HALF, D, 4>(m, a, qkv, pool, out, st, fu);
    case 8: return launch_prefill_t<BF16, HALF, D, 8>(m, a, qkv, pool, out, st, fu);
    default: return cudaErrorInvalidValue;
  }
}

template <bool BF16, bool HALF>
static cudaError_t launch_prefill_d(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv,
                                    void* pool, void* out, cudaStream_t st, bool fu) {
  return a.D == 128 ? launch_prefill_g<BF16, HALF, 128>(m, a, qkv, pool, out, st, fu)
                    : launch_prefill_g<BF16, HALF, 64>(m, a, qkv, pool, out, st, fu);
}

cudaError_t launch_prefill(const ds_ragged_meta& m, const LayerArgs& a, const void* qkv, void* pool,
                           void* out, cudaStream_t st, bool fused_append) {
  const bool half = a.style == DS_ROPE_HALF;
  const bool fu = fused_append;
  if (a.dtype == DS_BF16)
    return half ? launch_prefill_d<true, true>(m, a, qkv, pool, out, st, fu)
                : launch_prefill_d<true, false>(m, a, qkv, pool, out, st, fu);
  return half ? launch_prefill_d<false, true>(m, a, qkv, pool, out, st, fu)
              : launch_prefill_d<false, false>(m, a, qkv, pool, out, st, fu);
}

}  // namespace dsr
