// splitfuse.cpp -- Dynamic SplitFuse pass planner over the block ledger
// ("DeepSpeed-Inference and DeepSpeed-MII", tutorial ch. 10, sections 10.3 and
// 10.10: prefill chunks and single-token decodes share one batch under a token
// budget; "DeepSpeed Inference v2", pyshine.com/deepspeed-2, section "The front
// desk": blocks are reserved from the allocator before each pass and returned
// when a sequence is flushed).  Plain host C++; no CUDA call; all state in the
// caller's memory.
//
// Memory layout (int32 words):
//   [0, kHdr)                       header: n_order, n_free_slots, planned
//   Req[max_requests]               per-request state
//   order[max_requests]             active request slots in arrival order
//   free_slots[max_requests]        unused request slots
//   blocks[max_requests][max_bpr]   each request's block ids, in order
#include <cstdio>

#include "common.cuh"

namespace {

struct Req {
  int32_t uid, prompt, decode, seen, generated, n_blocks, planned_new, pad;
};
constexpr int32_t kHdr = 8;
enum { H_ORDER = 0, H_FREE = 1, H_PLANNED = 2 };

struct View {
  int32_t* hdr;
  Req* req;
  int32_t* order;
  int32_t* free_slots;
  int32_t* blocks;
};

size_t mem_words(int64_t max_requests, int64_t max_bpr) {
  return (size_t)kHdr + (size_t)max_requests * (sizeof(Req) / 4 + 2 + (size_t)max_bpr);
}

View view(const ds_splitfuse* p) {
  int32_t* w = static_cast<int32_t*>(p->mem);
  View v;
  v.hdr = w;
  v.req = reinterpret_cast<Req*>(w + kHdr);
  v.order = w + kHdr + (size_t)p->max_requests * (sizeof(Req) / 4);
  v.free_slots = v.order + p->max_requests;
  v.blocks = v.free_slots + p->max_requests;
  return v;
}

bool prefilling(const Req& r) { return r.seen < r.prompt; }
bool done(const Req& r) { return !prefilling(r) && r.generated >= r.decode; }

ds_status fail(ds_status s, const char* msg) {
  dsr::set_last_error(msg);
  return s;
}

// Extend r's blocks for n more tokens; false (nothing taken) if the ledger
// cannot supply them.
bool reserve(Req& r, int32_t* rblocks, int32_t max_bpr, int32_t bs, ds_block_allocator* a, int32_t n) {
  const int64_t need = ((int64_t)r.seen + n + bs - 1) / bs;
  const int64_t extra = need - r.n_blocks;
  if (extra <= 0) return true;
  if (extra > a->n_free || need > max_bpr) return false;
  if (ds_block_allocator_allocate(a, (int32_t)extra, rblocks + r.n_blocks) != DS_OK) return false;
  r.n_blocks += (int32_t)extra;
  return true;
}

}  // namespace

extern "C" {

ds_status ds_splitfuse_mem_size(int32_t max_requests, int32_t max_blocks_per_request, size_t* bytes) {
  if (max_requests < 1 || max_blocks_per_request < 1 || !bytes)
    return fail(DS_ERR_INVALID_ARG, "max_requests and max_blocks_per_request must be >= 1");
  *bytes = mem_words(max_requests, max_blocks_per_request) * 4;
  return DS_OK;
}

ds_status ds_splitfuse_init(ds_splitfuse* p, void* mem, size_t mem_bytes, int32_t max_requests,
                            int32_t max_blocks_per_request, int32_t token_budget, int32_t max_seqs,
                            int32_t block_size) {
  size_t need = 0;
  if (!p) return fail(DS_ERR_INVALID_ARG, "planner is NULL");
  if (ds_status s = ds_splitfuse_mem_size(max_requests, max_blocks_per_request, &need)) return s;
  if (!mem || (reinterpret_cast<uintptr_t>(mem) & 7) != 0)
    return fail(DS_ERR_INVALID_ARG, "memory NULL or not 8-byte aligned");
  if (token_budget < 1 || max_seqs < 1 || block_size < 1)
    return fail(DS_ERR_INVALID_ARG, "token_budget, max_seqs and block_size must be >= 1");
  if (mem_bytes < need) return fail(DS_ERR_WORKSPACE, "planner memory too small");
  p->mem = mem;
  p->mem_bytes = mem_bytes;
  p->max_requests = max_requests;
  p->max_blocks_per_request = max_blocks_per_request;
  p->token_budget = token_budget;
  p->max_seqs = max_seqs;
  p->block_size = block_size;
  p->n_active = 0;
  p->n_planned = 0;
  View v = view(p);
  v.hdr[H_ORDER] = 0;
  v.hdr[H_FREE] = max_requests;
  v.hdr[H_PLANNED] = 0;
  for (int32_t i = 0; i < max_requests; ++i) v.free_slots[i] = max_requests - 1 - i;  // slot 0 first
  return DS_OK;
}

ds_status ds_splitfuse_add(ds_splitfuse* p, int32_t uid, int32_t prompt, int32_t decode) {
  if (!p || !p->mem) return fail(DS_ERR_INVALID_ARG, "planner not initialised");
  if (prompt < 1 || decode < 0) return fail(DS_ERR_INVALID_ARG, "prompt must be >= 1 and decode >= 0");
  View v = view(p);
  for (int32_t k = 0; k < v.hdr[H_ORDER]; ++k)
    if (v.req[v.order[k]].uid == uid) return fail(DS_ERR_INVALID_ARG, "uid is already active");
  const int64_t nb = ((int64_t)prompt + decode + p->block_size - 1) / p->block_size;
  if (nb > p->max_blocks_per_request) return fail(DS_ERR_CAPACITY, "request needs more than max_blocks_per_request");
  if (v.hdr[H_FREE] == 0) return fail(DS_ERR_CAPACITY, "max_requests requests are active");
  const int32_t slot = v.free_slots[--v.hdr[H_FREE]];
  v.req[slot] = Req{uid, prompt, decode, 0, 0, 0, 0, 0};
  v.order[v.hdr[H_ORDER]++] = slot;
  p->n_active = v.hdr[H_ORDER];
  return DS_OK;
}

ds_status ds_splitfuse_next(ds_splitfuse* p, ds_block_allocator* alloc, ds_seq_desc* descs,
                            int32_t* uids, int32_t* n_out) {
  if (!p || !p->mem || !alloc || !descs || !uids || !n_out) return fail(DS_ERR_INVALID_ARG, "NULL argument");
  View v = view(p);
  if (v.hdr[H_PLANNED]) return fail(DS_ERR_INVALID_ARG, "the previous pass was not committed");
  const int32_t bpr = p->max_blocks_per_request;
  int32_t n = 0, left = p->token_budget;
  auto emit = [&](int32_t slot, int32_t tokens) {
    Req& r = v.req[slot];
    r.planned_new = tokens;
    descs[n].seen_tokens = r.seen;
    descs[n].new_tokens = tokens;
    descs[n].block_ids = v.blocks + (size_t)slot * bpr;
    descs[n].n_blocks = r.n_blocks;
    uids[n] = r.uid;
    ++n;
    left -= tokens;
  };
  // decodes first: one token for every request past its prompt and not done
  for (int32_t k = 0; k < v.hdr[H_ORDER]; ++k) {
    if (left == 0 || n == p->max_seqs) break;
    const int32_t slot = v.order[k];
    Req& r = v.req[slot];
    if (!prefilling(r) && !done(r) && reserve(r, v.blocks + (size_t)slot * bpr, bpr, p->block_size, alloc, 1))
      emit(slot, 1);
  }
  // then prompt chunks, as much of each prompt as the budget leaves
  for (int32_t k = 0; k < v.hdr[H_ORDER]; ++k) {
    if (left == 0 || n == p->max_seqs) break;
    const int32_t slot = v.order[k];
    Req& r = v.req[slot];
    if (!prefilling(r)) continue;
    const int32_t tokens = r.prompt - r.seen < left ? r.prompt - r.seen : left;
    if (reserve(r, v.blocks + (size_t)slot * bpr, bpr, p->block_size, alloc, tokens)) emit(slot, tokens);
  }
  v.hdr[H_PLANNED] = 1;
  p->n_planned = n;
  *n_out = n;
  return DS_OK;
}

ds_status ds_splitfuse_commit(ds_splitfuse* p, ds_block_allocator* alloc, int32_t* flushed,
                              int32_t* n_flushed) {
  if (!p || !p->mem || !alloc || !flushed || !n_flushed) return fail(DS_ERR_INVALID_ARG, "NULL argument");
  View v = view(p);
  if (!v.hdr[H_PLANNED]) return fail(DS_ERR_INVALID_ARG, "no pass is awaiting commit");
  const int32_t bpr = p->max_blocks_per_request;
  for (int32_t k = 0; k < v.hdr[H_ORDER]; ++k) {
    Req& r = v.req[v.order[k]];
    if (r.planned_new == 0) continue;
    r.seen += r.planned_new;
    if (r.seen > r.prompt) r.generated += r.planned_new;  // tokens past the prompt were generated
    r.planned_new = 0;
  }
  int32_t nf = 0, kept = 0;
  for (int32_t k = 0; k < v.hdr[H_ORDER]; ++k) {
    const int32_t slot = v.order[k];
    Req& r = v.req[slot];
    if (!done(r)) {
      v.order[kept++] = slot;
      continue;
    }
    if (r.n_blocks > 0) {
      ds_status s = ds_block_allocator_free(alloc, v.blocks + (size_t)slot * bpr, r.n_blocks);
      if (s != DS_OK) return s;  // the ledger no longer matches this planner's blocks
    }
    r.n_blocks = 0;
    flushed[nf++] = r.uid;
    v.free_slots[v.hdr[H_FREE]++] = slot;
  }
  v.hdr[H_ORDER] = kept;
  v.hdr[H_PLANNED] = 0;
  p->n_active = kept;
  p->n_planned = 0;
  *n_flushed = nf;
  return DS_OK;
}

}  // extern "C"
