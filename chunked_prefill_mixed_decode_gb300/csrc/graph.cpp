// CUDA-graph replay of the mixed step with padded token buckets.
//
// "Chunked Prefill: Ending the Great Stall", section 05: a CUDA graph records
// fixed shapes, while chunked prefill changes the token count every step, so
// an engine captures one graph per token bucket and pads each step up to the
// next bucket; the pad tokens are wasted work and the scheduler's budget and
// the executed token count differ by that padding.
//
// Here one graph per bucket records ms_mixed_step (append + attention)
// at fixed sizes: bucket tokens, max_rows rows, a block-table stride of
// max_row_pages and a context bound of num_pages * 16.  A replay copies the
// step's metadata into fixed device buffers, padded: tokens past the real
// count get slot -1 (no cache write) and position 0; rows past the real count
// get d = 0 (a pad row computes nothing).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "mixed_step.h"

namespace {

constexpr int32_t kPage = 16;
constexpr int32_t kMaxRowsPerStep = 8192;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct MetaLayout {
  size_t cu, q_start, ctx, positions, slots, bt, attn, total;
};

MetaLayout meta_layout(const ms_graph_config& c, int32_t max_bucket) {
  MetaLayout m;
  size_t off = 0;
  m.cu = off;
  off = align_up(off + (static_cast<size_t>(c.max_rows) + 1) * 4, 256);
  m.q_start = off;
  off = align_up(off + static_cast<size_t>(c.max_rows) * 4, 256);
  m.ctx = off;
  off = align_up(off + static_cast<size_t>(c.max_rows) * 4, 256);
  m.positions = off;
  off = align_up(off + static_cast<size_t>(max_bucket) * 4, 256);
  m.slots = off;
  off = align_up(off + static_cast<size_t>(max_bucket) * 4, 256);
  m.bt = off;
  off = align_up(off + static_cast<size_t>(c.max_rows) * c.max_row_pages * 4, 256);
  m.attn = off;
  off += ms_attention_workspace_size(c.max_rows, max_bucket, static_cast<int64_t>(c.num_pages) * kPage, c.H_q,
                                     c.H_kv, c.D);
  m.total = off;
  return m;
}

bool config_ok(const ms_graph_config* c) {
  if (c == nullptr || c->H_q < 1 || c->H_kv < 1 || c->H_q % c->H_kv != 0 || (c->D != 64 && c->D != 128) ||
      c->num_pages < 1 || c->max_rows < 1 || c->max_rows > kMaxRowsPerStep || c->max_row_pages < 1 ||
      c->max_pos < 1 || !(c->scale > 0.f) || c->num_buckets < 1 || c->buckets == nullptr)
    return false;
  for (int32_t i = 0; i < c->num_buckets; ++i)
    if (c->buckets[i] < 1 || (i > 0 && c->buckets[i] <= c->buckets[i - 1])) return false;
  return true;
}

}  // namespace

struct ms_step_graph {
  ms_graph_config cfg;
  ms_graph_buffers buf;
  std::vector<int32_t> buckets;
  std::vector<cudaGraphExec_t> execs;
  MetaLayout lay;
  int32_t* host[2] = {nullptr, nullptr};  // pinned staging, used alternately
  cudaEvent_t copied[2] = {nullptr, nullptr};
  int flip = 0;
  int device = 0;
};

namespace {

uint8_t* ws_base(const ms_step_graph* g) { return static_cast<uint8_t*>(g->buf.workspace); }

// The step that one graph records: append then attention at the bucket's sizes.
int enqueue_step(const ms_step_graph* g, int32_t bucket, cudaStream_t st) {
  const ms_graph_config& c = g->cfg;
  const ms_graph_buffers& b = g->buf;
  uint8_t* ws = ws_base(g);
  const int32_t* positions = reinterpret_cast<const int32_t*>(ws + g->lay.positions);
  const int32_t* slots = reinterpret_cast<const int32_t*>(ws + g->lay.slots);
  return ms_mixed_step(b.q, b.k, b.v, positions, slots, b.cos_tab, b.sin_tab, c.max_pos, b.k_cache, b.v_cache,
                       c.num_pages, b.q_rot, reinterpret_cast<const int32_t*>(ws + g->lay.cu),
                       reinterpret_cast<const int32_t*>(ws + g->lay.q_start),
                       reinterpret_cast<const int32_t*>(ws + g->lay.ctx),
                       reinterpret_cast<const int32_t*>(ws + g->lay.bt), nullptr, 0, c.max_row_pages, c.max_rows,
                       bucket, static_cast<int64_t>(c.num_pages) * kPage, c.H_q, c.H_kv, c.D, kPage, c.scale, b.out,
                       ws + g->lay.attn, g->lay.total - g->lay.attn, b.dev_status, reinterpret_cast<ms_stream_t>(st));
}

void release(ms_step_graph* g) {
  for (cudaGraphExec_t e : g->execs)
    if (e != nullptr) cudaGraphExecDestroy(e);
  for (int i = 0; i < 2; ++i) {
    if (g->copied[i] != nullptr) cudaEventDestroy(g->copied[i]);
    if (g->host[i] != nullptr) cudaFreeHost(g->host[i]);
  }
  delete g;
}

}  // namespace

extern "C" MS_API size_t ms_graph_workspace_size(const ms_graph_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return meta_layout(*cfg, cfg->buckets[cfg->num_buckets - 1]).total;
}

extern "C" MS_API int ms_graph_create(const ms_graph_config* cfg, const ms_graph_buffers* bufs, ms_stream_t stream,
                                      ms_step_graph** out) {
  if (out == nullptr) return MS_ERR_ARG;
  *out = nullptr;
  if (!config_ok(cfg) || bufs == nullptr || stream == nullptr || bufs->workspace == nullptr ||
      (reinterpret_cast<uintptr_t>(bufs->workspace) & 255u) != 0)
    return MS_ERR_ARG;
  const int32_t max_bucket = cfg->buckets[cfg->num_buckets - 1];
  const MetaLayout lay = meta_layout(*cfg, max_bucket);
  if (bufs->ws_bytes < lay.total) return MS_ERR_ARG;
  ms_step_graph* g = new (std::nothrow) ms_step_graph();
  if (g == nullptr) return MS_ERR_ARG;
  g->cfg = *cfg;
  g->buf = *bufs;
  g->buckets.assign(cfg->buckets, cfg->buckets + cfg->num_buckets);
  g->cfg.buckets = g->buckets.data();
  g->lay = lay;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t stage = lay.bt + static_cast<size_t>(cfg->max_rows) * cfg->max_row_pages * 4;
  if (cudaGetDevice(&g->device) != cudaSuccess) {
    release(g);
    return MS_ERR_CUDA;
  }
  for (int i = 0; i < 2; ++i) {
    if (cudaHostAlloc(reinterpret_cast<void**>(&g->host[i]), stage, cudaHostAllocDefault) != cudaSuccess ||
        cudaEventCreateWithFlags(&g->copied[i], cudaEventDisableTiming) != cudaSuccess) {
      release(g);
      return MS_ERR_CUDA;
    }
  }
  // An all-pad step in the fixed buffers: every row d = 0, every token slot -1.
  uint8_t* ws = ws_base(g);
  if (cudaMemsetAsync(ws, 0, lay.slots, st) != cudaSuccess ||
      cudaMemsetAsync(ws + lay.slots, 0xff, lay.attn - lay.slots, st) != cudaSuccess ||
      cudaMemsetAsync(ws + lay.attn, 0, lay.total - lay.attn, st) != cudaSuccess) {
    release(g);
    return MS_ERR_CUDA;
  }
  g->execs.assign(g->buckets.size(), nullptr);
  for (size_t i = 0; i < g->buckets.size(); ++i) {
    // run it once eagerly (one-time setup of the kernels happens outside the capture)
    int rc = enqueue_step(g, g->buckets[i], st);
    if (rc != MS_OK) {
      release(g);
      return rc;
    }
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      release(g);
      return MS_ERR_CUDA;
    }
    rc = enqueue_step(g, g->buckets[i], st);
    const cudaError_t end = cudaStreamEndCapture(st, &graph);
    if (rc != MS_OK || end != cudaSuccess || graph == nullptr) {
      if (graph != nullptr) cudaGraphDestroy(graph);
      release(g);
      return rc != MS_OK ? rc : MS_ERR_CUDA;
    }
    const cudaError_t inst = cudaGraphInstantiate(&g->execs[i], graph, 0);
    cudaGraphDestroy(graph);
    if (inst != cudaSuccess) {
      g->execs[i] = nullptr;
      release(g);
      return MS_ERR_CUDA;
    }
  }
  *out = g;
  return MS_OK;
}

extern "C" MS_API int ms_graph_destroy(ms_step_graph* g) {
  if (g != nullptr) {
    for (int i = 0; i < 2; ++i)
      if (g->copied[i] != nullptr) cudaEventSynchronize(g->copied[i]);
    release(g);
  }
  return MS_OK;
}

extern "C" MS_API int ms_graph_bucket(const ms_step_graph* g, int32_t num_tokens) {
  if (g == nullptr || num_tokens < 0) return MS_ERR_ARG;
  for (int32_t b : g->buckets)
    if (b >= num_tokens) return b;
  return MS_ERR_ARG;
}

extern "C" MS_API int ms_graph_run(ms_step_graph* g, const int32_t* cu_seqlens_q, const int32_t* q_start_pos,
                                   const int32_t* context_lens, const int32_t* positions,
                                   const int32_t* slot_mapping, const int32_t* block_tables, int32_t bt_stride,
                                   int32_t num_rows, int32_t num_tokens, ms_stream_t stream, int32_t* bucket_used) {
  if (g == nullptr || stream == nullptr || num_rows < 0 || num_tokens < 0 || num_rows > g->cfg.max_rows ||
      bt_stride < 0 || bt_stride > g->cfg.max_row_pages)
    return MS_ERR_ARG;
  if (num_rows > 0 && (cu_seqlens_q == nullptr || q_start_pos == nullptr || context_lens == nullptr ||
                       (bt_stride > 0 && block_tables == nullptr)))
    return MS_ERR_ARG;
  if (num_tokens > 0 && (positions == nullptr || slot_mapping == nullptr)) return MS_ERR_ARG;
  size_t k = 0;
  while (k < g->buckets.size() && g->buckets[k] < num_tokens) ++k;
  if (k == g->buckets.size()) return MS_ERR_ARG;
  const int32_t bucket = g->buckets[k];
  const int32_t R = g->cfg.max_rows, P = g->cfg.max_row_pages;
  const MetaLayout& L = g->lay;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  // the staging buffer of two replays ago must have been copied out
  const int h = g->flip;
  if (cudaEventSynchronize(g->copied[h]) != cudaSuccess) return MS_ERR_CUDA;
  uint8_t* host = reinterpret_cast<uint8_t*>(g->host[h]);
  int32_t* cu = reinterpret_cast<int32_t*>(host + L.cu);
  int32_t* qs = reinterpret_cast<int32_t*>(host + L.q_start);
  int32_t* cx = reinterpret_cast<int32_t*>(host + L.ctx);
  int32_t* ps = reinterpret_cast<int32_t*>(host + L.positions);
  int32_t* sl = reinterpret_cast<int32_t*>(host + L.slots);
  int32_t* bt = reinterpret_cast<int32_t*>(host + L.bt);
  const int32_t t_end = num_rows > 0 ? cu_seqlens_q[num_rows] : 0;
  if (num_rows > 0 && (cu_seqlens_q[0] != 0 || t_end != num_tokens)) return MS_ERR_ARG;
  if (num_rows == 0 && num_tokens != 0) return MS_ERR_ARG;
  cu[0] = 0;
  for (int32_t s = 0; s < R; ++s) {  // real rows, then pad rows with d = 0
    const bool real = s < num_rows;
    cu[s + 1] = real ? cu_seqlens_q[s + 1] : t_end;
    qs[s] = real ? q_start_pos[s] : 0;
    cx[s] = real ? context_lens[s] : 0;
  }
  for (int32_t t = 0; t < bucket; ++t) {  // real tokens, then pad tokens (no cache write)
    const bool real = t < num_tokens;
    ps[t] = real ? positions[t] : 0;
    sl[t] = real ? slot_mapping[t] : -1;
  }
  for (int32_t s = 0; s < num_rows; ++s) {  // re-stride the real rows; pad rows read no pages
    const int32_t* src = block_tables + static_cast<int64_t>(s) * bt_stride;
    int32_t* dst = bt + static_cast<int64_t>(s) * P;
    for (int32_t j = 0; j < P; ++j) dst[j] = j < bt_stride ? src[j] : -1;
  }
  uint8_t* ws = ws_base(g);
  const size_t head = L.positions;  // cu, q_start, ctx
  if (cudaMemcpyAsync(ws, host, head, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(ws + L.positions, ps, static_cast<size_t>(bucket) * 4, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(ws + L.slots, sl, static_cast<size_t>(bucket) * 4, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      (num_rows > 0 && cudaMemcpyAsync(ws + L.bt, bt, static_cast<size_t>(num_rows) * P * 4,
                                       cudaMemcpyHostToDevice, st) != cudaSuccess))
    return MS_ERR_CUDA;
  if (cudaEventRecord(g->copied[h], st) != cudaSuccess) return MS_ERR_CUDA;
  g->flip ^= 1;
  if (cudaGraphLaunch(g->execs[k], st) != cudaSuccess) return MS_ERR_CUDA;
  if (bucket_used != nullptr) *bucket_used = bucket;
  return MS_OK;
}

extern "C" MS_API int ms_graph_read_status(ms_step_graph* g, ms_stream_t stream, int32_t* host_status) {
  if (g == nullptr || host_status == nullptr) return MS_ERR_ARG;
  int32_t a = 0, b = 0;
  const int rc = ms_read_status(reinterpret_cast<int32_t*>(ws_base(g) + g->lay.attn), stream, &a);
  if (rc != MS_OK && rc != MS_ERR_DEVICE) return rc;
  if (g->buf.dev_status != nullptr) {
    const int rc2 = ms_read_status(g->buf.dev_status, stream, &b);
    if (rc2 != MS_OK && rc2 != MS_ERR_DEVICE) return rc2;
  }
  *host_status = a | b;
  return (a | b) != 0 ? MS_ERR_DEVICE : MS_OK;
}
