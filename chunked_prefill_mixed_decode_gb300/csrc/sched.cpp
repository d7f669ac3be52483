// Host side of the mixed step: token-budget packing, varlen metadata, and the
// rotary cos/sin table.
//
// Default packing follows "Chunked Prefill 的 Token 预算" (zwjcode.cn),
// sections 03-05 and 08, and "Chunked Prefill: Ending the Great Stall",
// sections 03-04: every running decode is placed first at one token each; then
// prompts are visited in arrival order and each takes the largest chunk that
// fits what is left.  Per-prompt limits come from "Prefill head-of-line
// blocking" (a ceiling in "The fix", a floor in "What comes next"), the prefill
// quota from zwjcode section 08, and the prefill-first and fair-share orders
// from "Splitting Prefill From Decode Inside a Step", "Choosing the priority
// order".  The metadata is the zwjcode page's section 06 list: absolute
// positions, one physical slot per new token, the block table, and the context
// length after the round.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "mixed_step.h"

namespace {

constexpr int32_t kPage = 16;

inline int32_t ceil_div(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }

struct Row {
  int32_t req;
  int32_t c;
  int32_t d;
};

// Block-table output of one packing: either rows of `stride` entries padded
// with -1 (block_tables, cap entries) or each row's pages back to back after
// its offset (bt_offsets [rows + 1], bt_pages, cap entries).
struct TableOut {
  int32_t* block_tables;
  int32_t* bt_offsets;
  int32_t* bt_pages;
  int64_t cap;
  bool ragged;
};

int build_metadata(const ms_request* reqs, int32_t n_req, const ms_sched_config* cfg, int32_t cap_rows,
                   int32_t cap_tokens, const TableOut& tab, int32_t* cu_seqlens_q, int32_t* q_start_pos,
                   int32_t* context_lens, int32_t* positions, int32_t* slot_mapping, int32_t* row_req,
                   int32_t* num_scheduled, ms_batch_info* info) {
  int32_t* block_tables = tab.block_tables;
  if (n_req < 0 || cfg == nullptr || info == nullptr || cu_seqlens_q == nullptr || q_start_pos == nullptr ||
      context_lens == nullptr || row_req == nullptr || (n_req > 0 && (reqs == nullptr || num_scheduled == nullptr)))
    return MS_ERR_ARG;
  const int32_t budget = cfg->token_budget;
  const int32_t cap = cfg->max_chunk_per_request;
  const int32_t floor_ = cfg->min_chunk_per_request;
  const int32_t quota = cfg->prefill_quota;
  const int32_t share = cfg->decode_share_permille;
  const int32_t policy = cfg->policy;
  if (budget < 0 || cap < 0 || floor_ < 0 || quota < 0 || share < 0 || share > 1000 ||
      (policy != MS_POLICY_DECODE_FIRST && policy != MS_POLICY_PREFILL_FIRST && policy != MS_POLICY_FAIR_SHARE))
    return MS_ERR_ARG;
  for (int32_t i = 0; i < n_req; ++i) {
    if (reqs[i].cached_len < 0 || reqs[i].remaining_prompt < 0 || reqs[i].num_pages < 0 ||
        (reqs[i].num_pages > 0 && reqs[i].block_table == nullptr))
      return MS_ERR_ARG;
  }

  // 1. the two classes, each in input order
  std::vector<int32_t> dec, pr;
  for (int32_t i = 0; i < n_req; ++i) (reqs[i].remaining_prompt == 0 ? dec : pr).push_back(i);
  const int64_t n_decodes = static_cast<int64_t>(dec.size());
  auto limit = [&](int32_t i) -> int64_t {
    const int64_t rem = reqs[i].remaining_prompt;
    return cap > 0 && rem > cap ? cap : rem;
  };
  // 2. prompts' takes out of an allowance: the floor first, then the leftover, both in arrival order
  std::vector<int64_t> take(static_cast<size_t>(n_req), 0);
  auto prompt_takes = [&](int64_t allowance) -> int64_t {
    int64_t left = allowance;
    if (floor_ > 0) {
      for (int32_t i : pr) {
        if (left == 0) break;
        int64_t t = limit(i) < floor_ ? limit(i) : floor_;
        if (t > left) t = left;
        take[i] += t;
        left -= t;
      }
    }
    for (int32_t i : pr) {
      if (left == 0) break;
      int64_t t = limit(i) - take[i];
      if (t > left) t = left;
      take[i] += t;
      left -= t;
    }
    return allowance - left;
  };
  int64_t n_dec = 0;
  if (policy == MS_POLICY_DECODE_FIRST) {
    int64_t dec_cap = budget;
    if (quota > 0) {
      int64_t demand = 0;  // the quota reserves only what the waiting prompts can use
      for (int32_t i : pr) demand += limit(i);
      dec_cap = budget - (quota < demand ? quota : demand);
    } else if (n_decodes > budget) {
      return MS_ERR_BUDGET;
    }
    n_dec = n_decodes < dec_cap ? n_decodes : (dec_cap > 0 ? dec_cap : 0);
    prompt_takes(budget - n_dec);
  } else if (policy == MS_POLICY_PREFILL_FIRST) {
    const int64_t used_p = prompt_takes(budget);
    n_dec = n_decodes < budget - used_p ? n_decodes : budget - used_p;
  } else {
    const int64_t allow = static_cast<int64_t>(budget) * share / 1000;
    n_dec = n_decodes < allow ? n_decodes : allow;
    const int64_t used_p = prompt_takes(budget - n_dec);
    n_dec = n_decodes < budget - used_p ? n_decodes : budget - used_p;
  }
  std::vector<Row> rows;
  rows.reserve(static_cast<size_t>(n_req));
  for (int64_t k = 0; k < n_dec; ++k) rows.push_back({dec[k], reqs[dec[k]].cached_len, 1});
  int64_t used = n_dec;
  for (int32_t i : pr)
    if (take[i] > 0) {
      rows.push_back({i, reqs[i].cached_len, static_cast<int32_t>(take[i])});
      used += take[i];
    }
  const int32_t num_decodes = static_cast<int32_t>(n_dec);

  // 3. capacities and page coverage
  const int32_t S = static_cast<int32_t>(rows.size());
  int32_t stride = 0;
  for (const Row& r : rows) {
    const int64_t ctx = static_cast<int64_t>(r.c) + r.d;
    if (ctx > INT32_MAX) return MS_ERR_ARG;
    const int32_t need = ceil_div(ctx, kPage);
    if (reqs[r.req].num_pages < need) return MS_ERR_NO_PAGES;
    if (need > stride) stride = need;
    // every page the row reads must be a page id whose slots fit in int32: a
    // negative id could turn into the "no write" slot -1 in slot_mapping
    const int32_t* bt = reqs[r.req].block_table;
    for (int32_t p = 0; p < need; ++p)
      if (bt[p] < 0 || bt[p] > INT32_MAX / kPage - 1) return MS_ERR_ARG;
  }
  int64_t table_entries = static_cast<int64_t>(S) * stride;  // padded rows
  if (tab.ragged) {
    table_entries = 0;  // the pages in use, back to back
    for (const Row& r : rows) table_entries += ceil_div(static_cast<int64_t>(r.c) + r.d, kPage);
    if (table_entries > INT32_MAX) return MS_ERR_ARG;
  }
  if (S > cap_rows || used > cap_tokens || table_entries > tab.cap) return MS_ERR_ARG;
  if (n_req > 0 && num_scheduled == nullptr) return MS_ERR_ARG;
  if (used > 0 && (positions == nullptr || slot_mapping == nullptr)) return MS_ERR_ARG;
  if (tab.ragged ? (tab.bt_offsets == nullptr || (table_entries > 0 && tab.bt_pages == nullptr))
                 : (table_entries > 0 && block_tables == nullptr))
    return MS_ERR_ARG;

  // 4. metadata
  for (int32_t i = 0; i < n_req; ++i) num_scheduled[i] = 0;
  cu_seqlens_q[0] = 0;
  int32_t t = 0;
  int32_t bt_next = 0;  // next free entry of bt_pages
  for (int32_t s = 0; s < S; ++s) {
    const Row& r = rows[s];
    const int32_t* bt = reqs[r.req].block_table;
    cu_seqlens_q[s + 1] = cu_seqlens_q[s] + r.d;
    q_start_pos[s] = r.c;
    context_lens[s] = r.c + r.d;
    row_req[s] = r.req;
    num_scheduled[r.req] = r.d;
    for (int32_t j = 0; j < r.d; ++j, ++t) {
      const int32_t pos = r.c + j;
      positions[t] = pos;
      slot_mapping[t] = bt[pos / kPage] * kPage + pos % kPage;
    }
    const int32_t need = ceil_div(static_cast<int64_t>(r.c) + r.d, kPage);
    if (tab.ragged) {
      std::memcpy(tab.bt_pages + bt_next, bt, static_cast<size_t>(need) * sizeof(int32_t));
      tab.bt_offsets[s] = bt_next;
      bt_next += need;
    } else {
      int32_t* dst = block_tables + static_cast<int64_t>(s) * stride;
      std::memcpy(dst, bt, static_cast<size_t>(need) * sizeof(int32_t));
      std::fill(dst + need, dst + stride, -1);
    }
  }
  if (tab.ragged) tab.bt_offsets[S] = bt_next;
  info->num_rows = S;
  info->num_decodes = num_decodes;
  info->num_tokens = static_cast<int32_t>(used);
  info->bt_stride = stride;
  info->unused_tokens = static_cast<int32_t>(budget - used);
  info->num_deferred = static_cast<int32_t>(n_decodes - n_dec);
  return MS_OK;
}

}  // namespace

extern "C" MS_API int ms_build_batch_metadata(const ms_request* reqs, int32_t n_req, const ms_sched_config* cfg,
                                              int32_t cap_rows, int32_t cap_tokens, int64_t cap_bt,
                                              int32_t* cu_seqlens_q, int32_t* q_start_pos,
                                              int32_t* context_lens, int32_t* positions, int32_t* slot_mapping,
                                              int32_t* block_tables, int32_t* row_req, int32_t* num_scheduled,
                                              ms_batch_info* info) {
  const TableOut tab{block_tables, nullptr, nullptr, cap_bt, false};
  return build_metadata(reqs, n_req, cfg, cap_rows, cap_tokens, tab, cu_seqlens_q, q_start_pos, context_lens,
                        positions, slot_mapping, row_req, num_scheduled, info);
}

extern "C" MS_API int ms_build_batch_metadata_ragged(const ms_request* reqs, int32_t n_req,
                                                     const ms_sched_config* cfg, int32_t cap_rows,
                                                     int32_t cap_tokens, int64_t cap_pages, int32_t* cu_seqlens_q,
                                                     int32_t* q_start_pos, int32_t* context_lens, int32_t* positions,
                                                     int32_t* slot_mapping, int32_t* bt_offsets, int32_t* bt_pages,
                                                     int32_t* row_req, int32_t* num_scheduled, ms_batch_info* info) {
  const TableOut tab{nullptr, bt_offsets, bt_pages, cap_pages, true};
  return build_metadata(reqs, n_req, cfg, cap_rows, cap_tokens, tab, cu_seqlens_q, q_start_pos, context_lens,
                        positions, slot_mapping, row_req, num_scheduled, info);
}

extern "C" MS_API int ms_rope_table(int32_t max_pos, int32_t D, double base, float* cos_tab, float* sin_tab) {
  if (max_pos < 1 || D < 2 || (D & 1) || !(base > 0.0) || cos_tab == nullptr || sin_tab == nullptr)
    return MS_ERR_ARG;
  const int32_t half = D / 2;
  std::vector<double> inv_freq(static_cast<size_t>(half));
  for (int32_t i = 0; i < half; ++i) inv_freq[i] = std::pow(base, -(2.0 * i) / static_cast<double>(D));
  for (int32_t p = 0; p < max_pos; ++p) {
    for (int32_t i = 0; i < half; ++i) {
      const double ang = static_cast<double>(p) * inv_freq[i];
      cos_tab[static_cast<int64_t>(p) * half + i] = static_cast<float>(std::cos(ang));
      sin_tab[static_cast<int64_t>(p) * half + i] = static_cast<float>(std::sin(ang));
    }
  }
  return MS_OK;
}
