// Host engine: a page pool with full-input admission and a plan/commit round
// driver over the mixed-step packer.
//
// "Splitting Prefill From Decode Inside a Step", "The arithmetic of chunk
// boundaries": a sequence's pages must be reserved before its first chunk, so
// that a request that cannot finish is refused at admission rather than part
// way through its prompt.  "Chunked Prefill 的 Token 预算" (zwjcode.cn),
// section 11: admission checks the complete input length against the KV
// capacity; section 08: each round schedules, runs the step, then commits the
// request progress.  "Chunked Prefill: Ending the Great Stall", section 05:
// a request's state is its cached length and how much prompt is left.
#include <cstdint>
#include <new>
#include <vector>

#include "mixed_step.h"

namespace {

constexpr int32_t kPage = 16;

struct Live {
  int32_t id;
  int32_t c;        // tokens in the cache
  int32_t rem;      // prompt tokens still to prefill
  int32_t gen;      // tokens generated so far
  int32_t max_new;  // tokens to generate
  std::vector<int32_t> pages;
};

}  // namespace

struct ms_engine {
  int32_t num_pages;
  ms_sched_config cfg;
  std::vector<int32_t> free;  // last in, first out; the back is the next page handed out
  std::vector<Live> live;     // arrival order
  int32_t next_id = 0;
  int64_t rounds = 0;
  bool planned = false;
  std::vector<int32_t> plan_idx;  // live index of each planned row
  std::vector<int32_t> plan_d;    // its new tokens
};

extern "C" MS_API int ms_engine_create(int32_t num_pages, const ms_sched_config* cfg, ms_engine** out) {
  if (out == nullptr || cfg == nullptr || num_pages < 0) return MS_ERR_ARG;
  *out = nullptr;
  ms_engine* e = new (std::nothrow) ms_engine();
  if (e == nullptr) return MS_ERR_ARG;
  e->num_pages = num_pages;
  e->cfg = *cfg;
  e->free.reserve(static_cast<size_t>(num_pages));
  for (int32_t p = num_pages - 1; p >= 0; --p) e->free.push_back(p);
  *out = e;
  return MS_OK;
}

extern "C" MS_API int ms_engine_destroy(ms_engine* e) {
  delete e;
  return MS_OK;
}

extern "C" MS_API int ms_engine_add_request(ms_engine* e, int32_t prompt_len, int32_t max_new_tokens,
                                            int32_t cached_len, int32_t* request_id) {
  if (e == nullptr || request_id == nullptr || prompt_len < 1 || max_new_tokens < 1 || cached_len < 0 ||
      cached_len > prompt_len || (cached_len == prompt_len && max_new_tokens < 2))
    return MS_ERR_ARG;
  const int64_t need = (static_cast<int64_t>(prompt_len) + max_new_tokens + kPage - 1) / kPage;
  if (need > static_cast<int64_t>(e->free.size())) return MS_ERR_NO_PAGES;
  Live r;
  r.id = e->next_id++;
  r.c = cached_len;
  r.rem = prompt_len - cached_len;
  r.gen = r.rem == 0 ? 1 : 0;
  r.max_new = max_new_tokens;
  r.pages.resize(static_cast<size_t>(need));
  for (int64_t k = 0; k < need; ++k) {
    r.pages[k] = e->free.back();
    e->free.pop_back();
  }
  e->live.push_back(std::move(r));
  *request_id = e->live.back().id;
  return MS_OK;
}

extern "C" MS_API int ms_engine_request_pages(const ms_engine* e, int32_t request_id, int32_t* pages,
                                              int32_t cap, int32_t* num_pages) {
  if (e == nullptr || num_pages == nullptr) return MS_ERR_ARG;
  for (const Live& r : e->live) {
    if (r.id != request_id) continue;
    const int32_t n = static_cast<int32_t>(r.pages.size());
    *num_pages = n;
    if (n > cap || (n > 0 && pages == nullptr)) return MS_ERR_ARG;
    for (int32_t k = 0; k < n; ++k) pages[k] = r.pages[k];
    return MS_OK;
  }
  return MS_ERR_ARG;
}

extern "C" MS_API int ms_engine_plan(ms_engine* e, int32_t cap_rows, int32_t cap_tokens, int64_t cap_bt,
                                     int32_t* cu_seqlens_q, int32_t* q_start_pos, int32_t* context_lens,
                                     int32_t* positions, int32_t* slot_mapping, int32_t* block_tables,
                                     int32_t* row_request_id, ms_batch_info* info) {
  if (e == nullptr || info == nullptr || row_request_id == nullptr) return MS_ERR_ARG;
  const int32_t n = static_cast<int32_t>(e->live.size());
  std::vector<ms_request> reqs(static_cast<size_t>(n));
  for (int32_t i = 0; i < n; ++i) {
    const Live& r = e->live[i];
    reqs[i] = {r.c, r.rem, r.pages.data(), static_cast<int32_t>(r.pages.size())};
  }
  std::vector<int32_t> scheduled(static_cast<size_t>(n) + 1);
  std::vector<int32_t> row_req(static_cast<size_t>(cap_rows > 0 ? cap_rows : 0) + 1);
  const int rc = ms_build_batch_metadata(reqs.data(), n, &e->cfg, cap_rows, cap_tokens, cap_bt, cu_seqlens_q,
                                         q_start_pos, context_lens, positions, slot_mapping, block_tables,
                                         row_req.data(), scheduled.data(), info);
  if (rc != MS_OK) return rc;
  e->plan_idx.assign(row_req.begin(), row_req.begin() + info->num_rows);
  e->plan_d.resize(static_cast<size_t>(info->num_rows));
  for (int32_t s = 0; s < info->num_rows; ++s) {
    e->plan_d[s] = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
    row_request_id[s] = e->live[row_req[s]].id;
  }
  e->planned = true;
  return MS_OK;
}

extern "C" MS_API int ms_engine_commit(ms_engine* e, int32_t* finished_ids, int32_t cap_finished,
                                       int32_t* num_finished) {
  if (e == nullptr || num_finished == nullptr || !e->planned) return MS_ERR_ARG;
  // Only planned rows can finish: admission never takes a request that has
  // all its tokens already.  Count them before changing anything.
  int32_t done = 0;
  for (size_t s = 0; s < e->plan_idx.size(); ++s) {
    const Live& r = e->live[e->plan_idx[s]];
    const int32_t gen = r.rem == 0 ? r.gen + 1 : (r.rem == e->plan_d[s] ? 1 : r.gen);
    if (gen >= r.max_new) ++done;
  }
  if (done > cap_finished || (done > 0 && finished_ids == nullptr)) return MS_ERR_ARG;
  for (size_t s = 0; s < e->plan_idx.size(); ++s) {
    Live& r = e->live[e->plan_idx[s]];
    if (r.rem == 0) {
      r.c += 1;
      r.gen += 1;
    } else {
      r.c += e->plan_d[s];
      r.rem -= e->plan_d[s];
      if (r.rem == 0) r.gen = 1;
    }
  }
  e->planned = false;
  e->plan_idx.clear();
  e->plan_d.clear();
  ++e->rounds;
  std::vector<Live> keep;
  keep.reserve(e->live.size());
  int32_t k = 0;
  for (Live& r : e->live) {
    if (r.gen >= r.max_new) {
      finished_ids[k++] = r.id;
      for (int32_t p : r.pages) e->free.push_back(p);
    } else {
      keep.push_back(std::move(r));
    }
  }
  e->live.swap(keep);
  *num_finished = k;
  return MS_OK;
}

extern "C" MS_API int ms_engine_stats(const ms_engine* e, ms_engine_counts* out) {
  if (e == nullptr || out == nullptr) return MS_ERR_ARG;
  out->num_live = static_cast<int32_t>(e->live.size());
  int32_t pre = 0, widest = 0;
  for (const Live& r : e->live) {
    pre += r.rem > 0;
    if (static_cast<int32_t>(r.pages.size()) > widest) widest = static_cast<int32_t>(r.pages.size());
  }
  out->num_prefilling = pre;
  out->max_request_pages = widest;
  out->num_free_pages = static_cast<int32_t>(e->free.size());
  out->num_pages = e->num_pages;
  out->rounds = e->rounds;
  return MS_OK;
}
