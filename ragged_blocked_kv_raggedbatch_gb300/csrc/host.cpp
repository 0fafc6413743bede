// host.cpp -- C ABI of the ragged blocked-KV attention layer: validation,
// metadata packing (RaggedBatchWrapper.insert_sequence/finalize and the
// AtomBuilder work lists of "DeepSpeed Inference v2", pyshine.com/deepspeed-2,
// section "Ragged batches"), and launch of the kernels.
//
// Every argument error is found here, before anything is enqueued, and
// returned as a status code (the pages' can_schedule answers with a result
// instead of throwing; the allocator's overflow is never hidden -- section
// "The front desk").
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "common.cuh"

// Decode-rate constants of the prefill/decode SM split (GB/s, GB300): the HBM
// rate of the decode rows and the rate one SM of the tensor-core decode kernel
// reaches.
#ifndef DSR_DEC_GBPS
#define DSR_DEC_GBPS 6700.0
#endif
#ifndef DSR_DEC_SM_GBPS
#define DSR_DEC_SM_GBPS 90.0
#endif

namespace {

thread_local char g_err[512] = "";

ds_status fail(ds_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

ds_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ds_status check_params(const ds_attn_params* p) {
  if (!p) return fail(DS_ERR_INVALID_ARG, "params is NULL");
  if (p->n_q_heads <= 0 || p->n_kv_heads <= 0)
    return fail(DS_ERR_INVALID_ARG, "head counts must be positive");
  if (p->n_q_heads % p->n_kv_heads != 0)
    return fail(DS_ERR_UNSUPPORTED, "n_q_heads (%d) not a multiple of n_kv_heads (%d)",
                p->n_q_heads, p->n_kv_heads);
  int g = p->n_q_heads / p->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return fail(DS_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", g);
  if (p->head_dim != 64 && p->head_dim != 128)
    return fail(DS_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", p->head_dim);
  if (p->block_size != dsr::kBlockSize)
    return fail(DS_ERR_UNSUPPORTED, "block_size must be 64 (got %d)", p->block_size);
  if (p->dtype != DS_FP16 && p->dtype != DS_BF16)
    return fail(DS_ERR_UNSUPPORTED, "dtype must be DS_FP16 or DS_BF16");
  if (p->rope_style != DS_ROPE_HALF && p->rope_style != DS_ROPE_INTERLEAVED)
    return fail(DS_ERR_UNSUPPORTED, "unknown rope_style %d", p->rope_style);
  if (!(p->rope_theta > 0.0f) || !std::isfinite(p->rope_theta))
    return fail(DS_ERR_INVALID_ARG, "rope_theta must be a positive finite number");
  if (!std::isfinite(p->softmax_scale))
    return fail(DS_ERR_INVALID_ARG, "softmax_scale must be finite");
  return DS_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// SMs of the GPU the host-side cost models assume (GB300); the launches clamp
// to the device's real count.
constexpr int kModelSMs = 152;

using dsr::max_decode_items;
using dsr::max_prefill_tiles;

// Words (int32) of the packed metadata for the given counts.
struct Layout {
  size_t hdr, cu, seen, newt, boff, btab, tseq, tpos, tiles, items, dseqs, total;
};

Layout layout_for(int64_t S, int64_t N, int64_t B, int64_t tiles, int64_t items, int64_t dseqs) {
  Layout L;
  size_t w = 0;
  L.hdr = w; w += dsr::HDR_WORDS;
  L.cu = w; w += S + 1;
  L.seen = w; w += S;
  L.newt = w; w += S;
  L.boff = w; w += S + 1;
  L.btab = w; w += B;
  L.tseq = w; w += N;
  L.tpos = w; w += N;
  w = align_up(w, 4);
  L.tiles = w; w += 4 * tiles;
  L.items = w; w += 4 * items;
  L.dseqs = w; w += 4 * dseqs;
  L.total = w;
  return L;
}

ds_status check_meta(const ds_ragged_meta* m) {
  if (!m) return fail(DS_ERR_INVALID_ARG, "meta is NULL");
  if (m->n_seqs < 0 || m->n_seqs > m->max_seqs || !m->header)
    return fail(DS_ERR_INVALID_ARG, "meta was not filled by ds_ragged_meta_build");
  return DS_OK;
}

dsr::LayerArgs layer_args(const ds_ragged_meta* m, const ds_attn_params* p,
                          const ds_rope_table* r, int32_t num_blocks) {
  dsr::LayerArgs a;
  a.Hq = p->n_q_heads;
  a.Hkv = p->n_kv_heads;
  a.D = p->head_dim;
  a.G = p->n_q_heads / p->n_kv_heads;
  a.dtype = p->dtype;
  a.style = p->rope_style;
  float scale = p->softmax_scale > 0.0f ? p->softmax_scale : 1.0f / std::sqrt((float)p->head_dim);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.num_blocks = num_blocks;
  a.max_positions = r->max_positions;
  a.rope = static_cast<const float2*>(r->table);
  a.header = m->header;
  return a;
}

ds_status check_rope(const ds_rope_table* r, const ds_attn_params* p, const ds_ragged_meta* m) {
  if (!r || !r->table) return fail(DS_ERR_INVALID_ARG, "rope table is NULL");
  if (!aligned(r->table, 16)) return fail(DS_ERR_INVALID_ARG, "rope table not 16-byte aligned");
  if (r->head_dim != p->head_dim || r->rope_theta != p->rope_theta)
    return fail(DS_ERR_INVALID_ARG, "rope table built for another head_dim or theta");
  if (m->max_len > r->max_positions)
    return fail(DS_ERR_CAPACITY, "batch reaches position %d but the rope table has %d rows",
                m->max_len - 1, r->max_positions);
  return DS_OK;
}

ds_status check_pool(const ds_kv_pool* pool, const ds_ragged_meta* m) {
  if (!pool || !pool->base) return fail(DS_ERR_INVALID_ARG, "pool is NULL");
  if (!aligned(pool->base, 16)) return fail(DS_ERR_INVALID_ARG, "pool base not 16-byte aligned");
  if (pool->num_blocks != m->pool_num_blocks)
    return fail(DS_ERR_INVALID_ARG, "pool has %d blocks but the batch was validated for %d",
                pool->num_blocks, m->pool_num_blocks);
  return DS_OK;
}

}  // namespace

namespace dsr {
// Lets other translation units of the library record a ds_last_error message.
void set_last_error(const char* msg) { std::snprintf(g_err, sizeof g_err, "%s", msg); }
}  // namespace dsr

extern "C" {

const char* ds_last_error(void) { return g_err; }

const char* ds_version(void) { return "ds_ragged 0.1 sm_103a"; }

ds_status ds_meta_buffer_sizes(int32_t max_seqs, int32_t max_tokens, int32_t max_blocks,
                               const ds_attn_params* params, size_t* device_bytes,
                               size_t* staging_bytes) {
  if (ds_status s = check_params(params)) return s;
  if (max_seqs < 0 || max_tokens < 0 || max_blocks < 0)
    return fail(DS_ERR_INVALID_ARG, "negative capacity");
  if (!device_bytes || !staging_bytes) return fail(DS_ERR_INVALID_ARG, "NULL output");
  Layout L = layout_for(max_seqs, max_tokens, max_blocks, max_prefill_tiles(max_seqs, max_tokens),
                        max_decode_items(max_seqs, max_blocks), max_seqs);
  size_t bytes = align_up(L.total * 4, 256);
  *device_bytes = bytes;
  *staging_bytes = bytes;
  return DS_OK;
}

ds_status ds_ragged_meta_pack(const ds_seq_desc* seqs, int32_t n_seqs,
                              const ds_attn_params* params, int32_t pool_num_blocks,
                              ds_ragged_meta* m) {
  if (ds_status s = check_params(params)) return s;
  if (!m) return fail(DS_ERR_INVALID_ARG, "meta is NULL");
  if (n_seqs < 0) return fail(DS_ERR_INVALID_ARG, "n_seqs < 0");
  if (n_seqs > 0 && !seqs) return fail(DS_ERR_INVALID_ARG, "seqs is NULL");
  if (!m->host_staging || !m->device_buf) return fail(DS_ERR_INVALID_ARG, "meta buffers are NULL");
  if (!aligned(m->device_buf, 256) || !aligned(m->host_staging, 16))
    return fail(DS_ERR_INVALID_ARG, "meta device buffer must be 256-byte aligned, staging 16");
  if (pool_num_blocks < 0) return fail(DS_ERR_INVALID_ARG, "pool_num_blocks < 0");
  size_t need_dev = 0, need_stage = 0;
  if (ds_status s = ds_meta_buffer_sizes(m->max_seqs, m->max_tokens, m->max_blocks, params,
                                         &need_dev, &need_stage))
    return s;
  if (m->device_bytes < need_dev || m->staging_bytes < need_stage)
    return fail(DS_ERR_WORKSPACE, "meta buffers hold %zu/%zu bytes, capacities need %zu",
                m->device_bytes, m->staging_bytes, need_dev);
  if (n_seqs > m->max_seqs)
    return fail(DS_ERR_CAPACITY, "%d sequences exceed max_seqs %d", n_seqs, m->max_seqs);

  const int bs = params->block_size;
  const int g = params->n_q_heads / params->n_kv_heads;
  int64_t N = 0, B = 0, max_len = 0;
  int32_t n_pre = 0, n_dec = 0;
  int64_t dec_blocks = 0, pre_tiles = 0;
  const int tile_tokens = dsr::kPrefillRows / g;
  for (int32_t i = 0; i < n_seqs; ++i) {
    const ds_seq_desc& d = seqs[i];
    if (d.new_tokens < 1)
      return fail(DS_ERR_INVALID_ARG, "sequence %d: new_tokens %d < 1", i, d.new_tokens);
    if (d.seen_tokens < 0)
      return fail(DS_ERR_INVALID_ARG, "sequence %d: seen_tokens %d < 0", i, d.seen_tokens);
    int64_t L = (int64_t)d.seen_tokens + d.new_tokens;
    if (L > (int64_t)INT32_MAX - bs) return fail(DS_ERR_CAPACITY, "sequence %d too long", i);
    int64_t nb = (L + bs - 1) / bs;
    if (d.n_blocks < nb)
      return fail(DS_ERR_CAPACITY, "sequence %d owns %d blocks but %lld positions need %lld", i,
                  d.n_blocks, (long long)L, (long long)nb);
    if (nb > 0 && !d.block_ids) return fail(DS_ERR_INVALID_ARG, "sequence %d: block_ids NULL", i);
    N += d.new_tokens;
    B += nb;
    max_len = std::max(max_len, L);
    if (d.new_tokens == 1) {
      ++n_dec;
      dec_blocks += nb;
    } else {
      ++n_pre;
      pre_tiles += (d.new_tokens + tile_tokens - 1) / tile_tokens;
    }
  }
  if (N > m->max_tokens)
    return fail(DS_ERR_CAPACITY, "%lld tokens exceed max_tokens %d", (long long)N, m->max_tokens);
  if (B > m->max_blocks)
    return fail(DS_ERR_CAPACITY, "%lld block-table entries exceed max_blocks %d", (long long)B,
                m->max_blocks);
  // Block ids: inside the pool and never shared inside one batch (one bit
  // per pool block, in a buffer kept per thread; ~1 ns per id).
  thread_local std::vector<uint64_t> used;
  used.assign(((size_t)pool_num_blocks + 63) / 64, 0);
  uint64_t* const bits = used.data();  // one lookup of the thread-local buffer
  for (int32_t i = 0; i < n_seqs; ++i) {
    const ds_seq_desc& d = seqs[i];
    const int64_t nb = ((int64_t)d.seen_tokens + d.new_tokens + bs - 1) / bs;
    const int32_t* ids = d.block_ids;
    for (int64_t b = 0; b < nb; ++b) {
      const int32_t id = ids[b];
      if ((uint32_t)id >= (uint32_t)pool_num_blocks)
        return fail(DS_ERR_BAD_BLOCK, "sequence %d block %lld: id %d outside pool of %d", i,
                    (long long)b, id, pool_num_blocks);
      const uint64_t bit = (uint64_t)1 << (id & 63);
      if (bits[(size_t)id >> 6] & bit) return fail(DS_ERR_BAD_BLOCK, "block id %d used twice in the batch", id);
      bits[(size_t)id >> 6] |= bit;
    }
  }

  // Decode split length in KV blocks: the largest power of two up to
  // kMaxSplitBlocks that still leaves about 8 waves of split CTAs (3 per SM on
  // 152 SMs), at least kMinSplitBlocks.  Longer splits mean fewer partials to
  // combine and less per-CTA set-up (GB300, max ragged batch: 8 blocks
  // 1.341 ms, 16: 1.299, 32: 1.289).
  int split = dsr::kMaxSplitBlocks;
  while (split > dsr::kMinSplitBlocks &&
         dec_blocks * params->n_kv_heads < (int64_t)8 * 3 * kModelSMs * split)
    split >>= 1;
  int64_t n_items = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    if (seqs[i].new_tokens != 1) continue;
    int64_t nb = ((int64_t)seqs[i].seen_tokens + 1 + bs - 1) / bs;
    n_items += (nb + split - 1) / split;
  }

  // capacity layout: every region at the offset the capacities give, so the
  // device pointers are the same for every batch packed into this buffer
  const bool cap = (m->flags & DS_META_CAPACITY) != 0;
  Layout L = cap ? layout_for(m->max_seqs, m->max_tokens, m->max_blocks, max_prefill_tiles(m->max_seqs, m->max_tokens),
                              max_decode_items(m->max_seqs, m->max_blocks), m->max_seqs)
                 : layout_for(n_seqs, N, B, pre_tiles, n_items, n_dec);
  int32_t* w = static_cast<int32_t*>(m->host_staging);
  // Every region below is written in full; only the header and the alignment
  // words before the work lists need clearing.
  std::memset(w + L.hdr, 0, dsr::HDR_WORDS * 4);
  std::memset(w + L.tpos + N, 0, (L.tiles - (L.tpos + N)) * 4);
  w[L.hdr + dsr::HDR_ERR] = 0;
  w[L.hdr + dsr::HDR_S] = n_seqs;
  w[L.hdr + dsr::HDR_N] = (int32_t)N;
  w[L.hdr + dsr::HDR_BLOCKS] = (int32_t)B;
  int32_t* cu = w + L.cu;
  int32_t* seen = w + L.seen;
  int32_t* newt = w + L.newt;
  int32_t* boff = w + L.boff;
  int32_t* btab = w + L.btab;
  int32_t* tseq = w + L.tseq;
  int32_t* tpos = w + L.tpos;
  int32_t* tiles = w + L.tiles;
  int32_t* items = w + L.items;
  int32_t* dseqs = w + L.dseqs;
  cu[0] = 0;
  boff[0] = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    const ds_seq_desc& d = seqs[i];
    int64_t nb = ((int64_t)d.seen_tokens + d.new_tokens + bs - 1) / bs;
    seen[i] = d.seen_tokens;
    newt[i] = d.new_tokens;
    cu[i + 1] = cu[i] + d.new_tokens;
    boff[i + 1] = boff[i] + (int32_t)nb;
    std::memcpy(btab + boff[i], d.block_ids, (size_t)nb * 4);
    for (int32_t j = 0; j < d.new_tokens; ++j) {
      tseq[cu[i] + j] = i;
      tpos[cu[i] + j] = d.seen_tokens + j;
    }
  }
  // Prefill tiles, longest KV range first so the heaviest atoms start first.
  struct Tile { int32_t seq, j0, ntok, kv_len; };
  std::vector<Tile> tv;
  tv.reserve((size_t)pre_tiles);
  for (int32_t i = 0; i < n_seqs; ++i) {
    const ds_seq_desc& d = seqs[i];
    if (d.new_tokens == 1) continue;
    for (int32_t j0 = 0; j0 < d.new_tokens; j0 += tile_tokens) {
      int32_t nt = std::min(tile_tokens, d.new_tokens - j0);
      tv.push_back({i, j0, nt, d.seen_tokens + j0 + nt});
    }
  }
  std::stable_sort(tv.begin(), tv.end(), [](const Tile& a, const Tile& b) { return a.kv_len > b.kv_len; });
  for (size_t k = 0; k < tv.size(); ++k) {
    tiles[4 * k + 0] = tv[k].seq;
    tiles[4 * k + 1] = tv[k].j0;
    tiles[4 * k + 2] = tv[k].ntok;
    tiles[4 * k + 3] = tv[k].kv_len;
  }
  // Decode split items and per-decode-sequence item ranges, the longest rows
  // first: the tensor-core decode kernel takes its units in this order, so
  // the last units taken are the short ones (in batch order, a 32-block unit
  // taken last left a ~60 us tail on the max ragged batch).  A row's items
  // stay consecutive; a row with a single item writes its output directly
  // (partial slot -1).
  thread_local std::vector<std::pair<int32_t, int32_t>> dec_rows;  // (blocks, sequence)
  dec_rows.clear();
  for (int32_t i = 0; i < n_seqs; ++i)
    if (seqs[i].new_tokens == 1)
      dec_rows.push_back({(int32_t)(((int64_t)seqs[i].seen_tokens + 1 + bs - 1) / bs), i});
  std::stable_sort(dec_rows.begin(), dec_rows.end(),
                   [](const std::pair<int32_t, int32_t>& a, const std::pair<int32_t, int32_t>& b) {
                     return a.first > b.first;
                   });
  int64_t it = 0;
  int32_t di = 0;
  for (const auto& row : dec_rows) {
    const int32_t i = row.second;
    const int32_t nb = row.first;
    int32_t cnt = (nb + split - 1) / split;
    dseqs[4 * di + 0] = i;
    dseqs[4 * di + 1] = cu[i];
    dseqs[4 * di + 2] = (int32_t)it;
    dseqs[4 * di + 3] = cnt;
    for (int32_t k = 0; k < cnt; ++k, ++it) {
      items[4 * it + 0] = i;
      items[4 * it + 1] = k * split;
      items[4 * it + 2] = std::min(nb, (k + 1) * split);
      items[4 * it + 3] = cnt == 1 ? -1 : (int32_t)it;
    }
    ++di;
  }

  m->n_seqs = n_seqs;
  m->n_tokens = (int32_t)N;
  m->n_blocks = (int32_t)B;
  m->n_prefill_seqs = n_pre;
  m->n_decode_seqs = n_dec;
  m->n_prefill_tiles = (int32_t)tv.size();
  m->n_decode_items = (int32_t)n_items;
  m->max_len = (int32_t)max_len;
  m->pool_num_blocks = pool_num_blocks;
  m->split_blocks = split;
  // SMs for the persistent prefill grid when decode rows run beside it.  The
  // prefill atoms cost T_PRE (SM-us) in all: ~1.8 us per 128-key step of a
  // two-tile atom, ~1.2 us with one tile (GB300; the sum matches the measured
  // prefill-only time of the max ragged batch within 4%).  The decode rows
  // stream their KV history at up to DSR_DEC_SM_GBPS per SM and DSR_DEC_GBPS
  // in all; decode CTAs take the SMs the prefill grid leaves, and every SM once
  // prefill is done.  The grid is the P minimising the finish time
  //   T(P) = T_PRE / P                        if decode is done by then,
  //          T_PRE / P + (rest of the KV) / rate(all SMs)   otherwise,
  // over P in [1, kModelSMs - 1].  (A fixed share, as an earlier kernel used,
  // let the prefill grid take 143 of 152 SMs on the max ragged batch and left
  // the decode rows to run after it.)
  m->prefill_sms = 0.f;
  if (!tv.empty() && dec_blocks > 0) {
    double pre_us = 0.0;
    for (const Tile& t : tv)
      pre_us += (double)((t.kv_len + 127) / 128) * (t.ntok > tile_tokens / 2 ? 1.8 : 1.2);
    pre_us *= params->n_kv_heads;
    const double dec_bytes = (double)dec_blocks * params->n_kv_heads * 2.0 * bs * params->head_dim * 2.0;
    // the tensor-core decode kernel (G >= 2, d = 128) runs at up to ~90 GB/s
    // per SM; the CUDA-core one needs every SM for the HBM rate
    const bool tc_decode = g >= 2 && params->head_dim == 128;
    const double sm_rate = (tc_decode ? DSR_DEC_SM_GBPS : DSR_DEC_GBPS / kModelSMs) * 1e3;  // bytes/us
    const double bw = DSR_DEC_GBPS * 1e3;
    double t_of[kModelSMs];
    double best_t = 1e300;
    for (int P = 1; P < kModelSMs; ++P) {
      const double t_pre = pre_us / P;
      const double r1 = std::min(bw, (kModelSMs - P) * sm_rate);
      double t = t_pre;
      if (dec_bytes > t_pre * r1) t = t_pre + (dec_bytes - t_pre * r1) / std::min(bw, kModelSMs * sm_rate);
      t_of[P] = t;
      best_t = std::min(best_t, t);
    }
    // T(P) is flat where the decode rows hold the HBM rate throughout; take
    // the middle of the near-optimal range, which hedges both rate estimates
    int lo = kModelSMs, hi = 0;
    for (int P = 1; P < kModelSMs; ++P)
      if (t_of[P] <= best_t * 1.005) {
        lo = std::min(lo, P);
        hi = std::max(hi, P);
      }
    m->prefill_sms = (float)((lo + hi) / 2);
  }
  // Order of the prefill atoms (the kernel takes tiles longest first in
  // rounds; within a round, KV heads in groups of HDR_PRE_HG): the fewer heads
  // the atoms running at once cover, the fewer K/V prefixes L2 must hold, but
  // the later the longest atoms of the last heads start.  So one head at a
  // time when the longest atom is short against a CTA's share of the work,
  // two otherwise, and all heads (plain tile-major) when one atom outlasts
  // that share.  On GB300: chunked prefill 2x8192 (longest atom / share 0.07)
  // DRAM traffic 1.47x -> 1.08x the algorithmic bytes at equal time; max
  // ragged batch, seeds 0 / 1 / 2 (0.24 / 0.34 / 0.54): attention 0.931 ->
  // 0.921, 0.750 -> 0.743, 0.696 -> 0.696 ms.
  int32_t head_group = 0;
  if (!tv.empty()) {
    double total = 0.0, longest = 0.0;
    for (const Tile& t : tv) {
      const double c = (double)((t.kv_len + 127) / 128) * (t.ntok > tile_tokens / 2 ? 1.8 : 1.2);
      total += c;
      longest = std::max(longest, c);
    }
    total *= params->n_kv_heads;
    const double ctas = m->prefill_sms > 0.f ? std::ceil(m->prefill_sms) : (double)kModelSMs;
    const double ratio = longest / (total / ctas);
    head_group = ratio <= 0.3 ? 1 : ratio <= 1.0 ? 2 : 0;
  }
  w[L.hdr + dsr::HDR_PRE_HG] = head_group;
  w[L.hdr + dsr::HDR_PRE_TILES] = (int32_t)tv.size();
  w[L.hdr + dsr::HDR_DEC_ITEMS] = (int32_t)n_items;
  w[L.hdr + dsr::HDR_DEC_SEQS] = n_dec;
  w[L.hdr + dsr::HDR_SPLIT] = split;
  w[L.hdr + dsr::HDR_PRE_CTAS] = (int32_t)std::ceil(m->prefill_sms);
  m->used_bytes = L.total * 4;
  int32_t* base = static_cast<int32_t*>(m->device_buf);
  m->header = base + L.hdr;
  m->cu_seqlens = base + L.cu;
  m->seq_seen = base + L.seen;
  m->seq_new = base + L.newt;
  m->blk_off = base + L.boff;
  m->block_table = base + L.btab;
  m->tok_seq = base + L.tseq;
  m->tok_pos = base + L.tpos;
  m->prefill_tiles = base + L.tiles;
  m->decode_items = base + L.items;
  m->decode_seqs = base + L.dseqs;
  return DS_OK;
}

ds_status ds_ragged_meta_build(const ds_seq_desc* seqs, int32_t n_seqs,
                               const ds_attn_params* params, int32_t pool_num_blocks,
                               ds_ragged_meta* meta, void* stream) {
  if (ds_status s = ds_ragged_meta_pack(seqs, n_seqs, params, pool_num_blocks, meta)) return s;
  cudaError_t e = cudaMemcpyAsync(meta->device_buf, meta->host_staging, meta->used_bytes,
                                  cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "metadata upload");
  return DS_OK;
}

ds_status ds_rope_table_size(const ds_attn_params* params, int32_t max_positions, size_t* bytes) {
  if (ds_status s = check_params(params)) return s;
  if (max_positions < 0 || !bytes) return fail(DS_ERR_INVALID_ARG, "bad max_positions or output");
  *bytes = (size_t)max_positions * (size_t)(params->head_dim / 2) * sizeof(float2);
  return DS_OK;
}

ds_status ds_rope_table_build(const ds_attn_params* params, int32_t max_positions, void* table,
                              size_t table_bytes, ds_rope_table* out, void* stream) {
  size_t need = 0;
  if (ds_status s = ds_rope_table_size(params, max_positions, &need)) return s;
  if (!out) return fail(DS_ERR_INVALID_ARG, "out is NULL");
  if (max_positions > 0 && (!table || !aligned(table, 16)))
    return fail(DS_ERR_INVALID_ARG, "table NULL or not 16-byte aligned");
  if (table_bytes < need) return fail(DS_ERR_WORKSPACE, "table holds %zu bytes, needs %zu", table_bytes, need);
  if (max_positions > 0) {
    cudaError_t e = dsr::launch_rope_table(*params, max_positions, static_cast<float2*>(table),
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "rope table kernel");
  }
  out->table = table;
  out->max_positions = max_positions;
  out->head_dim = params->head_dim;
  out->rope_theta = params->rope_theta;
  return DS_OK;
}

ds_status ds_kv_rotary_append(const ds_ragged_meta* meta, const ds_attn_params* params,
                              const ds_rope_table* rope, const void* qkv, void* q_out,
                              const ds_kv_pool* pool, void* stream) {
  if (ds_status s = check_params(params)) return s;
  if (ds_status s = check_meta(meta)) return s;
  const bool cap = (meta->flags & DS_META_CAPACITY) != 0;
  if (meta->n_tokens == 0 && !cap) return DS_OK;
  if (ds_status s = check_rope(rope, params, meta)) return s;
  if (ds_status s = check_pool(pool, meta)) return s;
  if (!qkv || !aligned(qkv, 16)) return fail(DS_ERR_INVALID_ARG, "qkv NULL or not 16-byte aligned");
  if (q_out && !aligned(q_out, 16)) return fail(DS_ERR_INVALID_ARG, "q_out not 16-byte aligned");
  dsr::LayerArgs a = layer_args(meta, params, rope, pool->num_blocks);
  cudaError_t e = dsr::launch_append(*meta, a, qkv, q_out, pool->base, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append kernel");
  return DS_OK;
}

ds_status ds_blocked_attention_workspace_size(const ds_attn_params* params, int32_t max_seqs,
                                              int32_t max_tokens, int32_t max_blocks,
                                              size_t* bytes) {
  if (ds_status s = check_params(params)) return s;
  if (max_seqs < 0 || max_tokens < 0 || max_blocks < 0 || !bytes)
    return fail(DS_ERR_INVALID_ARG, "negative capacity or NULL output");
  int64_t items = max_decode_items(max_seqs, max_blocks);
  *bytes = align_up((size_t)dsr::ws_partial_bytes(items, params->n_q_heads, params->head_dim), 256);
  return DS_OK;
}

// Split items a call must have workspace for: the batch's, or the capacities'
// when the launches must serve any batch within them.
static int64_t ws_items(const ds_ragged_meta* m) {
  return (m->flags & DS_META_CAPACITY) ? max_decode_items(m->max_seqs, m->max_blocks) : m->n_decode_items;
}

ds_status ds_blocked_attention(const ds_ragged_meta* meta, const ds_attn_params* params,
                               const ds_rope_table* rope, const void* qkv, const ds_kv_pool* pool,
                               void* out, void* workspace, size_t ws_bytes, void* stream) {
  if (ds_status s = check_params(params)) return s;
  if (ds_status s = check_meta(meta)) return s;
  const bool cap = (meta->flags & DS_META_CAPACITY) != 0;
  if (meta->n_tokens == 0 && !cap) return DS_OK;
  if (ds_status s = check_rope(rope, params, meta)) return s;
  if (ds_status s = check_pool(pool, meta)) return s;
  if (!qkv || !aligned(qkv, 16)) return fail(DS_ERR_INVALID_ARG, "qkv NULL or not 16-byte aligned");
  if (!out || !aligned(out, 16)) return fail(DS_ERR_INVALID_ARG, "out NULL or not 16-byte aligned");
  const int64_t items = ws_items(meta);
  const size_t need = (size_t)dsr::ws_partial_bytes(items, params->n_q_heads, params->head_dim);
  if (items > 0) {
    if (!workspace || !aligned(workspace, 256))
      return fail(DS_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
    if (ws_bytes < need)
      return fail(DS_ERR_WORKSPACE, "workspace holds %zu bytes, this batch needs %zu", ws_bytes, need);
  }
  dsr::LayerArgs a = layer_args(meta, params, rope, pool->num_blocks);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool pre = cap || meta->n_prefill_tiles > 0;
  if (pre) {
    cudaError_t e = dsr::launch_prefill(*meta, a, qkv, pool->base, out, st);
    if (e != cudaSuccess) return cuda_fail(e, "prefill kernel");
  }
  if (cap || meta->n_decode_items > 0) {
    cudaError_t e = dsr::launch_decode(*meta, a, qkv, pool->base, out, static_cast<float*>(workspace), st, pre);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernels");
  }
  return DS_OK;
}

static int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 1;
  return n;
}

// Fused workspace: [counters: max_seqs * n_kv_heads int32, 256-aligned][split partials].
static size_t fused_counter_bytes(const ds_attn_params* params, int32_t max_seqs) {
  return align_up((size_t)std::max(max_seqs, 0) * (size_t)params->n_kv_heads * sizeof(int32_t), 256);
}

ds_status ds_fused_workspace_size(const ds_attn_params* params, int32_t max_seqs, int32_t max_tokens,
                                  int32_t max_blocks, size_t* bytes) {
  size_t part = 0;
  if (ds_status s = ds_blocked_attention_workspace_size(params, max_seqs, max_tokens, max_blocks, &part))
    return s;
  *bytes = fused_counter_bytes(params, max_seqs) + part;
  return DS_OK;
}

ds_status ds_fused_workspace_init(const ds_ragged_meta* meta, const ds_attn_params* params,
                                  void* workspace, size_t ws_bytes, void* stream) {
  if (ds_status s = check_params(params)) return s;
  if (!meta) return fail(DS_ERR_INVALID_ARG, "meta is NULL");
  if (!workspace || !aligned(workspace, 256))
    return fail(DS_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
  const size_t cb = fused_counter_bytes(params, meta->max_seqs);
  if (ws_bytes < cb) return fail(DS_ERR_WORKSPACE, "workspace holds %zu bytes, the counters need %zu", ws_bytes, cb);
  cudaError_t e = cudaMemsetAsync(workspace, 0, cb, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "zeroing the workspace counters");
  return DS_OK;
}

ds_status ds_fused_append_attention(const ds_ragged_meta* meta, const ds_attn_params* params,
                                    const ds_rope_table* rope, const void* qkv,
                                    const ds_kv_pool* pool, void* out, void* workspace,
                                    size_t ws_bytes, void* stream) {
  if (ds_status s = check_params(params)) return s;
  if (ds_status s = check_meta(meta)) return s;
  const bool cap = (meta->flags & DS_META_CAPACITY) != 0;
  if (meta->n_tokens == 0 && !cap) return DS_OK;
  if (ds_status s = check_rope(rope, params, meta)) return s;
  if (ds_status s = check_pool(pool, meta)) return s;
  if (!qkv || !aligned(qkv, 16)) return fail(DS_ERR_INVALID_ARG, "qkv NULL or not 16-byte aligned");
  if (!out || !aligned(out, 16)) return fail(DS_ERR_INVALID_ARG, "out NULL or not 16-byte aligned");
  const size_t cb = fused_counter_bytes(params, meta->max_seqs);
  const int64_t items = ws_items(meta);
  const size_t need = cb + (size_t)dsr::ws_partial_bytes(items, params->n_q_heads, params->head_dim);
  if (items > 0) {
    if (!workspace || !aligned(workspace, 256))
      return fail(DS_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
    if (ws_bytes < need)
      return fail(DS_ERR_WORKSPACE, "workspace holds %zu bytes, this batch needs %zu", ws_bytes, need);
  }
  dsr::LayerArgs a = layer_args(meta, params, rope, pool->num_blocks);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // prefill chunks: their K/V append is the prefill kernel's prologue
  const bool pre = cap || meta->n_prefill_tiles > 0;
  if (pre) {
    cudaError_t e = dsr::launch_prefill(*meta, a, qkv, pool->base, out, st, /*fused_append=*/true);
    if (e != cudaSuccess) return cuda_fail(e, "prefill kernel");
  }
  if (cap || meta->n_decode_items > 0) {
    // Decode rows append their own K/V.  Their split partials are merged
    // inside the decode kernel by the tensor-core kernel, and by the CUDA-core
    // one whenever a prefill grid runs too (so a call is at most two launches),
    // its grid is at most two waves of 3 CTAs per SM, or the launch must serve
    // any batch within the capacities.  A larger decode-only grid keeps the
    // separate merge launch, which costs less than holding every CTA for its
    // count: decode-only batch of 256 rows on GB300, 1.304 ms merged in the
    // kernel against 1.297 ms with the merge kernel.
    const bool merge_in_kernel = cap || pre || dsr::decode_on_tensor_cores(a) ||
                                 (int64_t)meta->n_decode_items * params->n_kv_heads <= 6LL * device_sm_count();
    uint8_t* w = static_cast<uint8_t*>(workspace);
    cudaError_t e = dsr::launch_decode(*meta, a, qkv, pool->base, out, reinterpret_cast<float*>(w + cb), st, pre,
                                       /*fused_append=*/true,
                                       merge_in_kernel ? reinterpret_cast<int32_t*>(w) : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "fused decode kernel");
  }
  return DS_OK;
}

ds_status ds_get_device_error(const ds_ragged_meta* meta, int32_t* err, void* stream) {
  if (ds_status s = check_meta(meta)) return s;
  if (!err) return fail(DS_ERR_INVALID_ARG, "err is NULL");
  int32_t v = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&v, meta->header + dsr::HDR_ERR, sizeof v, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *err = v;
  return DS_OK;
}

}  // extern "C"
