// Mixed-batch attention over a paged KV cache, sm_103a.
//
// A step packs single-token decodes next to prefill chunks ("Chunked Prefill:
// Ending the Great Stall", sections 03-04).  Row s has d_s new tokens at
// absolute positions [c_s, c_s + d_s); its query at position p attends keys
// 0..p ("Chunked Prefill 的 Token 预算" (zwjcode.cn), sections 02 and 07):
// the cached prefix [0, c) plus its own chunk causally.  The two row kinds sit
// on opposite sides of the roofline ("Chunked Prefill: Ending the Great
// Stall", section 03; "Splitting Prefill From Decode Inside a Step", "Two
// kernels with different limiting resources"), so they take two paths:
//
//   decode rows (d = 1): split-KV with warp-level tensor-core MMAs.  One warp
//     owns a work item (row, KV head, span of pages) and streams its pages
//     through a private ring in shared memory with TMA (128-byte swizzled
//     16-row boxes); the G query heads of the KV head share every page read.
//     Per page, S^T = K Q^T (16 tokens x G heads, padded to 8) and
//     O^T += V^T P^T run as mma.sync m16n8k16 on ldmatrix fragments, with P
//     transposed in registers.  Each item leaves a partial (max, sum,
//     accumulator); the last split of a (row, KV head) to finish merges them.
//   chunk rows (d > 1): tcgen05 tensor cores.  A work item is a pair of
//     128-row query tiles (128/G tokens x G heads of one KV head each) that
//     walk 64-key tiles of the prefix and their own chunk together.  TMA loads
//     Q and K pages (one 16-row box per page and 64-column slab, 128-byte
//     swizzle) and V pages (one box per page, both slabs, at D = 128); S = Q K^T
//     lands in TMEM; two groups of four softmax warps, one
//     per query tile and one row per thread, write P (bf16) back over S, and
//     O += P V runs with P as the TMEM operand, accumulating in TMEM and
//     rescaled only when a row's maximum grows by more than a factor 2^8.
//
// A one-CTA prologue validates the metadata, chooses the split size, orders
// rows longest-first, expands the per-row item counts into flat item tables
// and decides how many CTAs start on chunk tiles.  One persistent kernel (a
// CTA per SM) then runs both queues: CTAs on SMs below the split start on
// chunk tiles, the rest on decode items, and each moves to the other queue
// when its own runs dry.  Work comes from atomic counters; no CTA waits on
// another.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "append_rope.cuh"
#include "mixed_step.h"
#include "ptx.cuh"

namespace {

using bf16 = __nv_bfloat16;
using namespace ms;

constexpr int kPage = 16;
constexpr int kMinSplitPages = 32;
constexpr int kMaxSplitPages = 256;
constexpr int kSoftmaxWarps = 8;
constexpr int kChunkThreads = 32 * (4 + kSoftmaxWarps);  // warp 0 TMA + queue, 2-9 softmax, 1/10/11 MMA
constexpr int kSortLimit = 2048;    // rows sorted longest-first up to this count
constexpr int kMaxRows = 8192;      // rows of one step
constexpr int kMaxTokens = 1 << 21;  // tokens of one step (a chunk row's Q-tile pairs fit in 16 bits)
// Cost model that splits the SMs between the two row kinds at the start of a
// step (CTAs then move to whichever queue still has work): the SM time of one
// 128x128 chunk tile, and the decode bandwidth one SM sustains, capped by HBM.
// Both SM-side rates are properties of the kernels' instruction streams, so
// they are kept per SM clock cycle and scaled by the clock the previous call
// ran at (measured on the GPU, see H_CLOCK_MHZ); HBM bandwidth comes from the
// device's memory clock and bus width.  The per-cycle figures come from
// sweeps of the split on the 8B GQA and long bimodal steps, where the kernel
// measured its clock at about 1.94 GHz (3.0 us per tile, 62 GB/s per decode
// SM); a test sweeps the split again and checks the model's choice against
// the best.
constexpr float kChunkTileCycles = 5820.f;    // SM cycles per 128x128 tile, alongside decode traffic
constexpr float kDecodeBytesPerCycle = 32.f;  // decode bytes per SM cycle at G = 1; fewer as G grows
constexpr float kHbmCopyEfficiency = 0.80f;   // sustained share of the nominal HBM rate

// workspace header (int32 words)
enum {
  H_STATUS = 0,
  H_DEC_CTR = 1,
  H_CH_CTR = 2,
  H_NDEC = 3,
  H_NDEC_ITEMS = 4,
  H_NCH = 5,
  H_NCH_ITEMS = 6,
  H_SPLIT = 7,
  H_NPART = 8,
  H_CHUNK_CTAS = 9,  // CTAs that start on chunk work (the rest start on decodes)
  H_CLOCK_MHZ = 10,  // SM clock the last call ran at (kept across calls; 0 in a fresh workspace)
  H_WORDS = 64
};

struct AttnParams {
  // Read by the prologue, which runs once per step from cold caches: kept
  // together at the front so that they span the fewest constant-cache lines.
  const int32_t* cu;
  const int32_t* q_start;
  const int32_t* ctx_lens;
  const int32_t* bt_off;  // ragged block table: row s's pages at bt[bt_off[s] .. bt_off[s + 1]); else nullptr
  int32_t* hdr;
  int64_t bt_len;         // entries of bt
  int64_t context_total;
  int64_t max_dec_items, max_ch_items;  // capacities in items (entries x H_kv)
  int64_t max_partials;
  int32_t bt_stride, num_rows, num_tokens, num_pages;
  int32_t H_q, H_kv, D, G;
  int32_t dec_workers;       // decode worker warps in the grid
  int32_t num_sms;
  int32_t clear_status;      // the prologue zeroes the status word first (scratch owned by the library)
  int32_t force_chunk_ctas;  // test hook: CTAs that start on chunk work (-1: the cost model decides)
  float sm_mhz;              // cost model: the SM clock when no call has measured it yet,
  float hbm_gbs;             // and the HBM bandwidth that caps decode
  float l2_bytes;            // L2 capacity (orders the chunk items)
  float scale_log2;
  int32_t* dec_rows;
  int32_t* dec_part_base;
  int32_t* dec_nsplit;
  int32_t* ch_rows;
  int2* dec_items;  // per decode split (items / H_kv entries): (decode row index, split within the row)
  int32_t* dec_cnt; // per (decode row, KV head): splits finished, for the last one to merge
  int2* ch_items;   // per chunk item: (chunk row index, KV head << 16 | Q-tile pair counted from the last)
  // the attention kernel's alone
  const bf16* q_rot;
  const bf16* k_cache;
  const bf16* v_cache;
  const int32_t* bt;      // padded rows of bt_stride entries, or (bt_off given) every row's pages back to back
  bf16* out;
  float* part_ml;
  float* part_acc;
  uint64_t wait_limit_ns;  // bound of every chunk-phase wait
  int32_t test_stall;      // test hook: chunk-phase producers publish no work item (0 in every real call)
};

__host__ __device__ inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// first block-table entry of row `row`: padded rows or ragged offsets
__device__ __forceinline__ const int32_t* row_table(const AttnParams& p, int row) {
  return p.bt + (p.bt_off != nullptr ? static_cast<int64_t>(__ldg(p.bt_off + row))
                                     : static_cast<int64_t>(row) * p.bt_stride);
}

// ----------------------------------------------------------------------------
// prologue: validate, classify, order longest-first, lay out the work lists
// ----------------------------------------------------------------------------

// Exclusive scan of one int per thread over the block (blockDim.x a multiple
// of 32); returns the thread's prefix and sets `total`.  Each thread adds up
// the warp totals ahead of its own warp, so a scan costs two barriers.
__device__ __forceinline__ int block_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  int before = 0, tot = 0;
  for (int j = 0; j < nw; ++j) {
    const int t = s_warp[j];
    before += j < w ? t : 0;
    tot += t;
  }
  __syncthreads();  // s_warp is free again
  total = tot;
  return before + x - v;
}

// warp sum of values in [0, 2^31): two 32-bit reductions of the 16-bit halves
__device__ __forceinline__ int64_t warp_sum31(int v) {
  const unsigned lo = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(v) & 0xffffu);
  const unsigned hi = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(v) >> 16);
  return (static_cast<int64_t>(hi) << 16) + lo;
}

__device__ __forceinline__ int64_t warp_sum64(int64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Work items of one row: decode splits of `split` pages, or pairs of 128-row Q tiles.
__device__ __forceinline__ int row_items(bool chunk, int c, int d, int tpt, unsigned split) {
  if (!chunk) return static_cast<int>((static_cast<unsigned>(c + kPage) / kPage + split - 1) / split);
  const int n_qt = (d + tpt - 1) / tpt;
  return (n_qt + 1) >> 1;
}

// 128x128 tiles of a chunk row's Q tiles against their causal key ranges (the
// cost model's unit of chunk work)
__device__ __forceinline__ unsigned chunk_tiles(int c, int d, int tpt) {
  unsigned tiles = 0;
  for (int end = tpt; end - tpt < d; end += tpt) tiles += static_cast<unsigned>(c + min(d, end) + 127) >> 7;
  return tiles;
}

// Sort key of the row at position `pos` of its list: the top 19 bits of the
// row's cost as a float (keys to read for a decode, query-key pairs for a
// chunk), then the position reversed.  Keys are unique and nonzero (cost >= 1);
// a larger key means more work or, at about equal cost, an earlier row.
__device__ __forceinline__ uint32_t order_key(float cost, int pos) {
  return ((__float_as_uint(cost) >> 13) << 13) | static_cast<uint32_t>(kMaxRows - 1 - pos);
}

// 32-bit words of the prologue's dynamic shared memory for S rows: sort keys
// (both lists, each padded to 4), list order, each row's d and c, and the item
// prefix in queue order.
__host__ __device__ constexpr int prologue_words(int S) { return 5 * ((S + 3) & ~3) + 16; }

// How many CTAs of the main kernel start on chunk tiles, and which side bounds
// the step.  Chunk time falls as 1/n with n chunk CTAs, in whole items; decode
// time is bytes over the bandwidth of the other SMs, capped by HBM.  Take the
// best split near the balance point, or, while decode stays HBM-bound, as many
// chunk CTAs as keep it so.  Called by one whole warp; the candidate counts go
// one per lane.
//
// It also orders the chunk items.  Longest first by default.  But when decode
// rows stream through L2 beside chunk rows whose K/V (all KV heads) would fill
// more than half of it, the items run KV head by KV head instead: the CTAs on
// chunk work at any time then share one head's K/V tiles in L2, where with
// every head in flight each head's prefix would be pulled from DRAM again and
// again (measured: 7 % more DRAM traffic than the algorithmic bytes on a
// 32K-key chunk next to 512 decodes, 6 % on 40 heads of 4K keys; on 8 heads
// of 10K keys, where the chunk rows bound the step, longest-first is faster).
struct SmSplit {
  int chunk_ctas;
  bool head_major;
};

__device__ SmSplit chunk_cta_split(const AttnParams& p, float tiles, float dec_pages, int n_items,
                                   int n_dec_items, float chunk_keys, int measured, int lane) {
  // the SM clock of the previous call on this workspace (header word H_CLOCK_MHZ, read
  // by the caller early), else the device's rated clock
  const float mhz = measured >= 200 && measured <= 5000 ? static_cast<float>(measured) : p.sm_mhz;
  const float S = static_cast<float>(p.num_sms);
  const float T = tiles * __fdividef(kChunkTileCycles * 1000.f, mhz);         // SM-ns of chunk work
  const float B = dec_pages * p.H_kv * kPage * p.D * 4.f;                     // decode bytes
  const float g = kDecodeBytesPerCycle * mhz * 1e-3f / (1.f + 0.18f * (p.G - 1));  // GB/s per decode SM
  const float n_hbm = fmaxf(0.f, floorf(S - p.hbm_gbs / g));  // most chunk CTAs with decode at HBM rate
  SmSplit r;
  r.head_major = B > 0.f && chunk_keys * p.H_kv * p.D * 4.f > 0.5f * p.l2_bytes;
  // a step whose chunk items and decode items all start at once: a CTA per chunk item
  const int dec_ctas = static_cast<int>((static_cast<int64_t>(n_dec_items) * p.num_sms + p.dec_workers - 1) /
                                        p.dec_workers);
  if (n_items + dec_ctas <= p.num_sms) {
    r.chunk_ctas = n_items;
  } else if (T == 0.f) {
    r.chunk_ctas = static_cast<int>(B == 0.f ? S : n_hbm);
  } else if (B == 0.f) {
    r.chunk_ctas = static_cast<int>(S);
  } else if (T * p.hbm_gbs <= B * n_hbm) {  // chunk done within the HBM-bound decode time
    r.chunk_ctas = static_cast<int>(n_hbm);
  } else {
    // Balance point, then the nearby CTA count that minimizes the step: chunk work
    // comes in whole items, so n chunk CTAs need ceil(items / n) rounds of about
    // T / items each; decode runs on the other CTAs, capped by HBM.  Ties go to
    // the smallest count.
    const float n0 = fminf(S - 1.f, fmaxf(1.f, rintf(__fdividef(T * g * S, B + T * g))));
    const int n_it = max(n_items, 1);
    const float t_item = __fdividef(T, static_cast<float>(n_it));
    const int k_lo = max(1, static_cast<int>(n0) - 16), k_hi = min(static_cast<int>(S) - 1, static_cast<int>(n0) + 16);
    float best = 3.0e38f;
    int bk = static_cast<int>(n0);
    for (int k = k_lo + lane; k <= k_hi; k += 32) {
      const float tc = static_cast<float>((n_it + k - 1) / k) * t_item;
      const float td = __fdividef(B, fminf((S - k) * g, p.hbm_gbs));
      const float tt = fmaxf(tc, td);
      if (tt < best) {
        best = tt;
        bk = k;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int ok = __shfl_xor_sync(0xffffffffu, bk, o);
      if (ob < best || (ob == best && ok < bk)) {
        best = ob;
        bk = ok;
      }
    }
    r.chunk_ctas = bk;
  }
  if (p.force_chunk_ctas >= 0) r.chunk_ctas = min(p.force_chunk_ctas, p.num_sms);
  return r;
}

// Table entry of item i of a chunk row with np Q-tile pairs: (KV head) << 16 |
// (pair counted from the last), KV head by KV head or longest pair first.
__device__ __forceinline__ int chunk_entry(int i, int np, int H_kv, bool head_major) {
  const int hk = head_major ? i / np : i % H_kv;
  const int e = head_major ? i - hk * np : i / H_kv;
  return (hk << 16) | e;
}

// Decode split size: about 8 items per decode worker warp, clamped; at least 32
// pages (64 when G >= 4, whose items carry G heads of partials to merge, and 128
// when chunk rows share the step: decode then runs on the SMs the chunk tiles
// leave, where fewer, longer items cost less than a finer tail saves).
__device__ __forceinline__ int decode_split(const AttnParams& p, int64_t dec_pages, bool with_chunks) {
  const int64_t num = dec_pages * p.H_kv, den = static_cast<int64_t>(p.dec_workers) * 8;
  int64_t split = num + den <= 0xffffffffll
                      ? static_cast<int64_t>(static_cast<uint32_t>(num + den - 1) / static_cast<uint32_t>(den))
                      : cdiv64(num, den);
  const int64_t min_split = p.G >= 4 ? (with_chunks ? 4 : 2) * kMinSplitPages : kMinSplitPages;
  split = split < min_split ? min_split : (split > kMaxSplitPages ? kMaxSplitPages : split);
  return static_cast<int>(split);
}

// Header of a call whose metadata failed validation: status set, no work.
__device__ __forceinline__ void header_bad_meta(int32_t* hdr) {
  atomicOr(hdr + H_STATUS, MS_STATUS_BAD_META);
  hdr[H_DEC_CTR] = hdr[H_CH_CTR] = 0;
  hdr[H_NDEC] = hdr[H_NDEC_ITEMS] = hdr[H_NCH] = hdr[H_NCH_ITEMS] = hdr[H_NPART] = 0;
  hdr[H_SPLIT] = kMinSplitPages;
  hdr[H_CHUNK_CTAS] = 0;
}

// The prologue of a step of at most 32 rows: one warp, a row per lane, with
// ballots and shuffles in place of shared memory and barriers.  Same outputs
// as the block version below.
__device__ __forceinline__ void prologue_warp(const AttnParams& p) {
  const int lane = threadIdx.x, S = p.num_rows;
  int32_t* hdr = p.hdr;
  const int measured_mhz = hdr[H_CLOCK_MHZ];  // loaded beside the row metadata
  int d = 0, c = 0, ctx = 0;
  bool ok = true;
  if (lane < S) {
    const int32_t a = p.cu[lane], b = p.cu[lane + 1];
    d = static_cast<int32_t>(static_cast<uint32_t>(b) - static_cast<uint32_t>(a));  // checked below
    c = p.q_start[lane];
    ctx = p.ctx_lens[lane];
    ok = a >= 0 && b >= a && b <= p.num_tokens && c >= 0 && static_cast<int64_t>(ctx) == static_cast<int64_t>(c) + d;
    if (p.bt_off != nullptr) {
      const int64_t o0 = p.bt_off[lane], o1 = p.bt_off[lane + 1];
      ok = ok && o0 >= 0 && o1 <= p.bt_len && cdiv64(ctx, kPage) <= o1 - o0;
    } else {
      ok = ok && cdiv64(ctx, kPage) <= p.bt_stride;
    }
    if (!ok) d = ctx = 0;
  }
  const bool bad = __any_sync(0xffffffffu, !ok);
  const int64_t ctx_sum = warp_sum31(ctx);  // ctx >= 0 here (valid rows, or 0)
  if (bad || ctx_sum > p.context_total) {
    if (lane == 0) header_bad_meta(hdr);
    return;
  }
  const bool is_dec = d == 1, is_ch = d > 1;
  const int64_t dec_pages = warp_sum31(is_dec ? (ctx + kPage - 1) / kPage : 0);
  const int split = decode_split(p, dec_pages, __any_sync(0xffffffffu, is_ch));
  const int tpt = 128 / p.G;
  const unsigned bd = __ballot_sync(0xffffffffu, is_dec), bc = __ballot_sync(0xffffffffu, is_ch);
  const int n_dec = __popc(bd), n_ch = __popc(bc);
  // position in its list, then rank by key within the list (longest first):
  // the keys sit in shared memory by list position, zero-padded, read 16 bytes at a time
  __shared__ __align__(16) uint32_t s_key[2][32];
  __shared__ int s_items[32], s_pref[32];
  const bool listed = is_dec || is_ch;
  const unsigned list = is_ch ? bc : bd;
  const int pos = __popc(list & ((1u << lane) - 1u));
  const uint32_t key = order_key(is_ch ? 0.5f * d * (2.f * c + d + 1.f) : c + 1.f, pos);
  s_key[0][lane] = 0;
  s_key[1][lane] = 0;
  s_items[lane] = 0;
  __syncwarp();
  if (listed) s_key[is_ch][pos] = key;
  __syncwarp();
  int rank = 0;
  const uint4* k4 = reinterpret_cast<const uint4*>(s_key[is_ch]);
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const uint4 v = k4[m];
    rank += (v.x > key) + (v.y > key) + (v.z > key) + (v.w > key);
  }
  const int items = listed ? row_items(is_ch, c, d, tpt, static_cast<unsigned>(split)) : 0;
  const int q = (is_ch ? n_dec : 0) + rank;  // queue position
  if (listed) s_items[q] = items;
  __syncwarp();
  {  // exclusive prefix over queue positions, one per lane
    const int v = s_items[lane];
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    s_pref[lane] = x - v;
  }
  __syncwarp();
  const int before = listed ? s_pref[q] : 0;  // items of the rows ahead in queue order
  const int dec_tot = __reduce_add_sync(0xffffffffu, is_dec ? items : 0);
  const int ch_tot = __reduce_add_sync(0xffffffffu, is_ch ? items : 0);
  const int64_t n_dec_items = static_cast<int64_t>(dec_tot) * p.H_kv;
  const int64_t n_ch_items = static_cast<int64_t>(ch_tot) * p.H_kv;
  const bool dec_over = n_dec_items > p.max_dec_items || static_cast<int64_t>(dec_tot) * p.H_q > p.max_partials;
  const bool ch_over = n_ch_items > p.max_ch_items;
  const int64_t tiles =
      warp_sum31(is_ch ? static_cast<int>(min(static_cast<int64_t>(chunk_tiles(c, d, tpt)) * p.H_kv,
                                                int64_t{0x7fffffff}))
                       : 0);
  const int64_t chunk_keys = warp_sum31(is_ch ? ctx : 0);
  if (is_dec) {
    p.dec_rows[rank] = lane;
    p.dec_part_base[rank] = static_cast<int32_t>(static_cast<int64_t>(before) * p.H_q);
    p.dec_nsplit[rank] = items;
    if (!dec_over)
      for (int i = 0; i < items; ++i) p.dec_items[before + i] = make_int2(rank, i);
  }
  if (is_ch) p.ch_rows[rank] = lane;
  const SmSplit sp = chunk_cta_split(p, static_cast<float>(tiles), static_cast<float>(dec_pages),
                                     ch_over ? 0 : static_cast<int>(n_ch_items),
                                     dec_over ? 0 : static_cast<int>(n_dec_items), static_cast<float>(chunk_keys),
                                     measured_mhz, lane);
  // the chunk rows' items (pairs x H_kv of them per row), the whole warp on one row at
  // a time; then the split counters, 16 bytes per store
  for (unsigned pend = ch_over ? 0u : bc; pend != 0u; pend &= pend - 1u) {
    const int src = __ffs(pend) - 1;
    const int r_rank = __shfl_sync(0xffffffffu, rank, src), r_items = __shfl_sync(0xffffffffu, items, src);
    const int r_before = __shfl_sync(0xffffffffu, before, src);
    int2* out = p.ch_items + static_cast<int64_t>(r_before - dec_tot) * p.H_kv;
    for (int i = lane; i < r_items * p.H_kv; i += 32)
      out[i] = make_int2(r_rank, chunk_entry(i, r_items, p.H_kv, sp.head_major));
  }
  if (!dec_over) {
    const int n_cnt = n_dec * p.H_kv;  // the counters start 16-byte aligned in the workspace
    for (int i = lane; i < (n_cnt >> 2); i += 32) reinterpret_cast<int4*>(p.dec_cnt)[i] = make_int4(0, 0, 0, 0);
    for (int i = (n_cnt & ~3) + lane; i < n_cnt; i += 32) p.dec_cnt[i] = 0;
  }
  if (lane == 0) {
    hdr[H_NDEC] = dec_over ? 0 : n_dec;
    hdr[H_NDEC_ITEMS] = dec_over ? 0 : static_cast<int32_t>(n_dec_items);
    hdr[H_NPART] = static_cast<int32_t>(static_cast<int64_t>(dec_tot) * p.H_q);
    hdr[H_NCH] = ch_over ? 0 : n_ch;
    hdr[H_NCH_ITEMS] = ch_over ? 0 : static_cast<int32_t>(n_ch_items);
    if (dec_over || ch_over) atomicOr(hdr + H_STATUS, MS_STATUS_BAD_META);
    hdr[H_DEC_CTR] = 0;
    hdr[H_CH_CTR] = 0;
    hdr[H_SPLIT] = split;
    hdr[H_CHUNK_CTAS] = sp.chunk_ctas;
  }
}

// The prologue on one CTA of blockDim.x threads (a multiple of 32, at most
// 1024; warp 0 alone up to 32 rows): validate the rows, split them into decode rows (d = 1)
// and chunk rows (d > 1), order each list longest-first, size the decode
// splits, write the flat item tables (item -> row in queue order, item within
// the row), zero the split counters and pick how many CTAs of the main kernel
// start on chunk work.  Every row's values are read from global memory once;
// the rest happens in shared memory (prologue_words(S) words of dynamic shared
// memory).  It runs once per step from a cold instruction cache, so its loops
// stay rolled and its code short.  It reads only the row metadata, never the
// appended K/V, so it may run alongside the append.
__device__ __forceinline__ void prologue_body(const AttnParams& p) {
  extern __shared__ __align__(16) int32_t psm[];
  __shared__ int s_warp[32];
  __shared__ long long s_sum[3][32];
  __shared__ unsigned s_cnt[2][32];
  __shared__ unsigned long long s_tiles;
  __shared__ SmSplit s_split;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int S = p.num_rows;  // at most kMaxRows (checked by the host, which sizes psm by it)
  int32_t* hdr = p.hdr;
  const int Sp = (S + 3) & ~3;
  uint32_t* key = reinterpret_cast<uint32_t*>(psm);  // Sp + 8 words
  int32_t* lst = psm + Sp + 8;                       // list order: decode rows, then chunk rows
  int32_t* rd = lst + Sp;                            // per row (input order): d (0 for pad rows), c
  int32_t* rc = rd + Sp;
  int32_t* pref = rc + Sp;                           // per queue position: items, then their prefix
  // a library-owned scratch keeps the previous call's status: start this call at zero
  // (ahead of every status write of this call, all of which come after a barrier or from this thread)
  if (tid == 0 && p.clear_status) hdr[H_STATUS] = 0;
  if (S <= 32) {
    if (warp == 0) prologue_warp(p);
    return;
  }
  if (tid == 0) s_tiles = 0;
  const int measured_mhz = warp == 0 ? hdr[H_CLOCK_MHZ] : 0;  // for the SM split, loaded early
  // 1. load and validate the rows; count decodes, chunks, context and decode pages
  int64_t my_ctx = 0, my_pages = 0, my_ch_keys = 0;
  unsigned my_dec = 0, my_ch = 0;
  int my_bad = 0;
  for (int s = tid; s < S; s += nt) {
    const int32_t a = p.cu[s], b = p.cu[s + 1];
    const int32_t d = static_cast<int32_t>(static_cast<uint32_t>(b) - static_cast<uint32_t>(a));  // checked below
    const int32_t c = p.q_start[s], ctx = p.ctx_lens[s];
    // d == 0 is a pad row: valid, and neither a decode nor a chunk
    bool ok = a >= 0 && b >= a && b <= p.num_tokens && c >= 0 && static_cast<int64_t>(ctx) == static_cast<int64_t>(c) + d;
    if (p.bt_off != nullptr) {  // the row's pages must lie inside the table
      const int64_t o0 = p.bt_off[s], o1 = p.bt_off[s + 1];
      ok = ok && o0 >= 0 && o1 <= p.bt_len && cdiv64(ctx, kPage) <= o1 - o0;
    } else {
      ok = ok && cdiv64(ctx, kPage) <= p.bt_stride;
    }
    my_bad |= !ok;
    rd[s] = ok ? d : 0;
    rc[s] = c;
    if (ok) {
      my_ctx += ctx;
      my_dec += d == 1;
      my_ch += d > 1;
      if (d == 1) my_pages += (ctx + kPage - 1) / kPage;
      if (d > 1) my_ch_keys += ctx;
    }
  }
  my_ctx = warp_sum64(my_ctx);
  my_pages = warp_sum64(my_pages);
  my_ch_keys = warp_sum64(my_ch_keys);
  my_dec = __reduce_add_sync(0xffffffffu, my_dec);
  my_ch = __reduce_add_sync(0xffffffffu, my_ch);
  if (lane == 0) {
    s_sum[0][warp] = my_ctx;
    s_sum[1][warp] = my_pages;
    s_sum[2][warp] = my_ch_keys;
    s_cnt[0][warp] = my_dec;
    s_cnt[1][warp] = my_ch;
  }
  const int bad = __syncthreads_or(my_bad);
  int64_t ctx_sum = 0, dec_pages = 0, chunk_keys = 0;
  int n_dec = 0, n_ch = 0;
  for (int j = 0; j < nw; ++j) {
    ctx_sum += s_sum[0][j];
    dec_pages += s_sum[1][j];
    chunk_keys += s_sum[2][j];
    n_dec += static_cast<int>(s_cnt[0][j]);
    n_ch += static_cast<int>(s_cnt[1][j]);
  }
  if (bad || ctx_sum > p.context_total) {
    if (tid == 0) header_bad_meta(hdr);
    return;
  }
  // 2. decode split size
  const int split = decode_split(p, dec_pages, n_ch > 0);
  const int tpt = 128 / p.G;
  const unsigned split32 = static_cast<unsigned>(split);
  // 3. the two lists in input order: decode rows at lst[0, n_dec), chunk rows after them
  const int n_tot = n_dec + n_ch;
  {
    int o_dec = 0, o_ch = 0;
    for (int base = 0; base < S; base += nt) {  // uniform
      const int s = base + tid;  // the row this thread loaded
      const int d = s < S ? rd[s] : 0;
      int tot;
      const int o = block_scan((d == 1) | ((d > 1) << 16), s_warp, tot);  // both counts, 16 bits each
      if (d == 1) lst[o_dec + (o & 0xffff)] = s;
      if (d > 1) lst[n_dec + o_ch + (o >> 16)] = s;
      o_dec += tot & 0xffff;
      o_ch += tot >> 16;
    }
  }
  // 4. sort keys, each list from a 16-byte boundary, padded with zero keys
  const int ch_base = (n_dec + 3) & ~3;
  if (tid < 4) {
    if (n_dec + tid < ch_base) key[n_dec + tid] = 0;
    if (n_ch + tid < ((n_ch + 3) & ~3)) key[ch_base + n_ch + tid] = 0;
  }
  __syncthreads();
  for (int j = tid; j < n_tot; j += nt) {
    const bool ch = j >= n_dec;
    const int pos = ch ? j - n_dec : j, row = lst[j];
    const float d = static_cast<float>(rd[row]), c = static_cast<float>(rc[row]);
    key[(ch ? ch_base : 0) + pos] = order_key(ch ? 0.5f * d * (2.f * c + d + 1.f) : c + 1.f, pos);
  }
  __syncthreads();
  // 5. each list longest first: a row's rank is the number of larger keys in its
  // list (lists longer than kSortLimit keep input order); rows in queue order,
  // and each row's item count at its queue position
  for (int j = tid; j < n_tot; j += nt) {
    const bool ch = j >= n_dec;
    const int pos = ch ? j - n_dec : j, n = ch ? n_ch : n_dec;
    int rank = pos;
    if (n <= kSortLimit) {
      const uint32_t* kl = key + (ch ? ch_base : 0);
      const uint32_t mine = kl[pos];
      const uint4* k4 = reinterpret_cast<const uint4*>(kl);
      rank = 0;
      for (int m = 0; m < (n + 3) >> 2; ++m) {
        const uint4 v = k4[m];
        rank += (v.x > mine) + (v.y > mine) + (v.z > mine) + (v.w > mine);
      }
    }
    const int row = lst[j], c = rc[row], d = rd[row];
    (ch ? p.ch_rows : p.dec_rows)[rank] = row;
    pref[(ch ? n_dec : 0) + rank] = row_items(ch, c, d, tpt, split32);
    if (ch) atomicAdd(&s_tiles, static_cast<unsigned long long>(chunk_tiles(c, d, tpt)) * p.H_kv);
  }
  __syncthreads();
  // 6. exclusive prefix of the item counts in queue order (decode rows, then chunk rows)
  int run = 0;
  for (int base = 0; base < n_tot; base += nt) {  // uniform
    const int q = base + tid;
    const int v = q < n_tot ? pref[q] : 0;
    int tot;
    const int o = block_scan(v, s_warp, tot);
    if (q < n_tot) {
      pref[q] = run + o;
      if (q < n_dec) {
        p.dec_part_base[q] = static_cast<int32_t>(static_cast<int64_t>(run + o) * p.H_q);
        p.dec_nsplit[q] = v;
      }
    }
    run += tot;
  }
  if (tid == 0) pref[n_tot] = run;
  __syncthreads();
  const int dec_tot = pref[n_dec], ch_tot = run - dec_tot;
  const int64_t n_dec_items = static_cast<int64_t>(dec_tot) * p.H_kv;
  const int64_t n_ch_items = static_cast<int64_t>(ch_tot) * p.H_kv;
  const bool dec_over = n_dec_items > p.max_dec_items || static_cast<int64_t>(dec_tot) * p.H_q > p.max_partials;
  const bool ch_over = n_ch_items > p.max_ch_items;
  // 7. item tables.  Decode rows, a thread per row: entry pref[q] + i -> (row
  // k, split i), one entry per split (a work item is an entry and a KV head).
  // Then the SM split, which also orders the chunk items; chunk rows, a warp
  // per row: one entry per item, (row k, KV head and Q-tile pair).  Then the
  // split counters of every (decode row, KV head), zeroed 16 bytes at a time.
  for (int q = tid; q < n_dec && !dec_over; q += nt) {
    const int cnt = pref[q + 1] - pref[q];
    int2* out = p.dec_items + pref[q];
    for (int i = 0; i < cnt; ++i) out[i] = make_int2(q, i);
  }
  if (warp == 0) {
    const SmSplit sp = chunk_cta_split(p, static_cast<float>(s_tiles), static_cast<float>(dec_pages),
                                       ch_over ? 0 : static_cast<int>(n_ch_items),
                                       dec_over ? 0 : static_cast<int>(n_dec_items), static_cast<float>(chunk_keys),
                                       measured_mhz, lane);
    if (lane == 0) s_split = sp;
  }
  __syncthreads();
  for (int q = n_dec + warp; q < n_tot && !ch_over; q += nw) {
    const int np = pref[q + 1] - pref[q];
    int2* out = p.ch_items + static_cast<int64_t>(pref[q] - dec_tot) * p.H_kv;
    for (int i = lane; i < np * p.H_kv; i += 32)
      out[i] = make_int2(q - n_dec, chunk_entry(i, np, p.H_kv, s_split.head_major));
  }
  if (!dec_over) {
    const int n_cnt = n_dec * p.H_kv;  // the counters start 16-byte aligned in the workspace
    for (int i = tid; i < (n_cnt >> 2); i += nt) reinterpret_cast<int4*>(p.dec_cnt)[i] = make_int4(0, 0, 0, 0);
    for (int i = (n_cnt & ~3) + tid; i < n_cnt; i += nt) p.dec_cnt[i] = 0;
  }
  // 8. the header the main kernel starts from
  if (warp == 0) {
    if (lane == 0) {
      hdr[H_NDEC] = dec_over ? 0 : n_dec;
      hdr[H_NDEC_ITEMS] = dec_over ? 0 : static_cast<int32_t>(n_dec_items);
      hdr[H_NPART] = static_cast<int32_t>(static_cast<int64_t>(dec_tot) * p.H_q);
      hdr[H_NCH] = ch_over ? 0 : n_ch;
      hdr[H_NCH_ITEMS] = ch_over ? 0 : static_cast<int32_t>(n_ch_items);
      if (dec_over || ch_over) atomicOr(hdr + H_STATUS, MS_STATUS_BAD_META);
      hdr[H_DEC_CTR] = 0;
      hdr[H_CH_CTR] = 0;
      hdr[H_SPLIT] = static_cast<int32_t>(split);
      hdr[H_CHUNK_CTAS] = s_split.chunk_ctas;
    }
  }
}

// The prologue as its own kernel, launched as a programmatic dependent of the
// kernel before it on the stream (normally the append): it runs alongside that
// kernel and waits for it before it exits, so the kernel after it sees the
// append's writes.
__global__ void __launch_bounds__(1024, 1) prologue_kernel(AttnParams p) {
  griddep_launch_dependents();
  prologue_body(p);
  griddep_wait();
}

// The append and the prologue as one kernel (the step call on small steps):
// CTA 0 runs the prologue, the others the append's work units.  Launched in
// plain stream order, so nothing of the step before is still running.
template <typename Idx>
__global__ void __launch_bounds__(kAppendThreads) append_prologue_kernel(AppendArgs a, AttnParams p) {
  griddep_launch_dependents();  // the attention kernel may start its set-up
  if (blockIdx.x == 0) {
    prologue_body(p);
    return;
  }
  append_rope_units<Idx>(a, static_cast<Idx>(blockIdx.x - 1) * kAppendThreads + threadIdx.x,
                         static_cast<Idx>(gridDim.x - 1) * kAppendThreads);
}

// ----------------------------------------------------------------------------
// decode rows: split-KV, warp-level tensor-core MMAs
// ----------------------------------------------------------------------------

template <int D, int G>
struct DecCfg {
  static constexpr int NST = D == 128 ? 2 : 4;     // ring stages per warp
  static constexpr int PAGE_BYTES = kPage * D * 2;  // one page of one KV head
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;  // K page, then V page
  static constexpr int Q_BYTES = G * D * 2;
  // per-warp tail: two Q buffers, then the ring barriers
  static constexpr int T_BAR = 2 * Q_BYTES;
  static constexpr int TAIL_BYTES = (T_BAR + NST * 8 + 127) / 128 * 128;
  // as many worker warps as the CTA has, while their rings fit in shared memory
  static constexpr int WARPS = 12 * (NST * STAGE_BYTES + TAIL_BYTES) <= 230000 ? 12 : 10;
  // all warps' stages first (each stage 1024-aligned, as 128-byte-swizzled TMA
  // tiles need), then the warps' tails
  static constexpr int TAIL_OFF = WARPS * NST * STAGE_BYTES;
  static constexpr int SMEM = TAIL_OFF + WARPS * TAIL_BYTES;
};


struct DecItem {
  int row;     // row index s
  int k;       // index among decode rows
  int hk;      // KV head
  int p0, np;  // logical pages [p0, p0 + np)
  int ctx;     // keys of the row (c + 1)
  int tok;     // packed token index of the row's query
  int part;    // partial record of query head hk * G (+ g for the others)
  int ns;      // splits of the row
  int w0;      // lane j: page id of the item's page j (its first window of 32 pages)
  const int32_t* btr;  // the row's block table
};

__device__ __forceinline__ DecItem describe_dec(const AttnParams& p, int item, int split) {
  DecItem it;
  // items run (split, KV head) with the head fastest; the table has one entry per split
  const int e = item / p.H_kv;
  const int2 kl = __ldg(p.dec_items + e);  // (decode row index, split within the row)
  const int k = kl.x, sp = kl.y;
  it.hk = item - e * p.H_kv;
  it.k = k;
  it.row = __ldg(p.dec_rows + k);
  it.ctx = __ldg(p.ctx_lens + it.row);
  it.tok = __ldg(p.cu + it.row);
  const int n_pages = (it.ctx + kPage - 1) / kPage;
  it.p0 = sp * split;
  it.np = min(split, n_pages - it.p0);
  it.part = __ldg(p.dec_part_base + k) + sp * p.H_q + it.hk * p.G;
  it.ns = __ldg(p.dec_nsplit + k);
  // the first window of page ids, loaded while the item waits its turn
  const int lane = threadIdx.x & 31;
  it.btr = row_table(p, it.row);
  it.w0 = lane < it.np ? __ldg(it.btr + it.p0 + lane) : 0;
  return it;
}


// Merge the ns split records of decode row k for query heads h0 .. h0+nh-1
// into bf16 output (one warp; lane owns D/32 columns).  Records written by
// other SMs are read past L1.
template <int D>
__device__ __forceinline__ void merge_splits(const AttnParams& p, int k, int h0, int nh, int tok, int ns,
                                             int lane) {
  constexpr int EPL = D / 32;
  const int64_t base0 = __ldcg(p.dec_part_base + k);
  for (int hq = h0; hq < h0 + nh; ++hq) {
    const int64_t base = base0 + hq;
    // lanes over splits for (max, sum); then every lane walks the splits for its columns
    float M = -INFINITY;
    for (int j = lane; j < ns; j += 32)
      M = fmaxf(M, __ldcg(p.part_ml + (base + static_cast<int64_t>(j) * p.H_q) * 2));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f, o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    for (int j0 = 0; j0 < ns; j0 += 32) {
      const int j = j0 + lane;
      float w = 0.f;
      if (j < ns) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (base + static_cast<int64_t>(j) * p.H_q) * 2));
        w = ex2(ml.x - M);
        L += w * ml.y;
      }
      const int nj = min(32, ns - j0);
#pragma unroll 4
      for (int jj = 0; jj < nj; ++jj) {
        const float wj = __shfl_sync(0xffffffffu, w, jj);
        const float* src = p.part_acc + (base + static_cast<int64_t>(j0 + jj) * p.H_q) * D + lane * EPL;
        if constexpr (EPL == 4) {
          const float4 a = __ldcg(reinterpret_cast<const float4*>(src));
          o[0] += wj * a.x; o[1] += wj * a.y; o[2] += wj * a.z; o[3] += wj * a.w;
        } else {
          const float2 a = __ldcg(reinterpret_cast<const float2*>(src));
          o[0] += wj * a.x; o[1] += wj * a.y;
        }
      }
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
    const float inv = 1.f / L;
    bf16* dst = p.out + (static_cast<int64_t>(tok) * p.H_q + hq) * D + lane * EPL;
    if constexpr (EPL == 4) {
      __nv_bfloat162 a = __floats2bfloat162_rn(o[0] * inv, o[1] * inv);
      __nv_bfloat162 b = __floats2bfloat162_rn(o[2] * inv, o[3] * inv);
      *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    } else {
      __nv_bfloat162 a = __floats2bfloat162_rn(o[0] * inv, o[1] * inv);
      *reinterpret_cast<__nv_bfloat162*>(dst) = a;
    }
  }
}

// Decode phase: each worker warp of the CTA (12, or 10 at D = 128, G = 8) is
// independent, with its own ring of page stages, pulling decode items until
// the queue is empty.  Per page it runs mma.sync m16n8k16 on ldmatrix
// fragments: 16 tokens against the G query heads (padded to 8).  tcgen05 does
// not fit here: its M is at least 64 rows, while a decode page is 16 rows per
// warp and a row's G query heads fill only part of N.

// Out of line, as is chunk_phase: each phase gets its own register allocation
// (inlined into one kernel body the two spill).
template <int D, int G>
__device__ __noinline__ void decode_phase(const AttnParams& p, uint8_t* dsmem, const CUtensorMap* tm_k,
                                             const CUtensorMap* tm_v, const CUtensorMap* tm_kp,
                                             const CUtensorMap* tm_vp) {
  using C = DecCfg<D, G>;
  constexpr int NST = C::NST;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp >= DecCfg<D, G>::WARPS) return;  // the CTA's remaining warps have no decode slice
  uint8_t* stg = dsmem + warp * NST * C::STAGE_BYTES;             // this warp's ring stages
  uint8_t* tail = dsmem + C::TAIL_OFF + warp * C::TAIL_BYTES;     // its Q buffers and barriers
  uint64_t* full = reinterpret_cast<uint64_t*>(tail + C::T_BAR);
  const int n_items = p.hdr[H_NDEC_ITEMS];
  const int split = p.hdr[H_SPLIT];
  if (lane == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(full + i, 1);
    fence_mbar_init();
  }
  __syncwarp();


  auto dequeue = [&]() -> int {
    int v = 0;
    if (lane == 0) v = atomicAdd(p.hdr + H_DEC_CTR, 1);
    return __shfl_sync(0xffffffffu, v, 0);
  };

  // issue stream: pages of `cur`, then of `nxt` (one item ahead at most)
  DecItem cur, nxt;
  int cur_id = dequeue();
  if (cur_id >= n_items) return;
  cur = describe_dec(p, cur_id, split);
  int nxt_id = dequeue();
  bool nxt_valid = nxt_id < n_items;
  if (nxt_valid) nxt = describe_dec(p, nxt_id, split);
  uint32_t seq_iss = 0, seq_con = 0;
  int iss_in_nxt = 0, iss_page = 0;
  uint32_t item_par = 0;  // q buffer of the current item
  bool failed = false;

  // lane j: page id of page (window start + j) of the issue-cursor item, and of the
  // window after it: page ids come one coalesced load per 32 pages, a window ahead
  int iss_bt = 0, iss_bt_next = 0;
  auto issue_page = [&](const DecItem& it, int pi, uint32_t qpar) {
    if ((pi & 31) == 0) {
      iss_bt = pi == 0 ? it.w0 : iss_bt_next;
      const int w = pi + 32 + lane;
      if (pi + 32 < it.np) iss_bt_next = w < it.np ? __ldg(it.btr + it.p0 + w) : 0;
    }
    int phys = __shfl_sync(0xffffffffu, iss_bt, pi & 31);
    if (lane == 0) {
      const int st = seq_iss % NST;
      uint8_t* stage = stg + st * C::STAGE_BYTES;
      if (phys < 0 || phys >= p.num_pages) {
        atomicOr(p.hdr + H_STATUS, MS_STATUS_BAD_PAGE);
        phys = 0;
      }
      const uint32_t bytes = 2 * C::PAGE_BYTES + (pi == 0 ? C::Q_BYTES : 0);
      mbar_arrive_expect_tx(full + st, bytes);
      // 16-row x 64-column slabs, 128-byte swizzled, for conflict-free ldmatrix; at
      // D = 128 each of K and V is one box of the whole page (slab 0, then slab 1)
      const int pg = phys * p.H_kv + it.hk;
      if constexpr (D == 128) {
        tma_load_4d(stage, tm_kp, 0, 0, 0, pg, full + st);
        tma_load_4d(stage + C::PAGE_BYTES, tm_vp, 0, 0, 0, pg, full + st);
      } else {
        tma_load_2d(stage, tm_k, 0, pg * kPage, full + st);
        tma_load_2d(stage + C::PAGE_BYTES, tm_v, 0, pg * kPage, full + st);
      }
      if (pi == 0)
        bulk_g2s(tail + qpar * C::Q_BYTES, p.q_rot + (static_cast<int64_t>(it.tok) * p.H_q + it.hk * G) * D,
                 C::Q_BYTES, full + st);
    }
    ++seq_iss;
  };
  auto pump = [&]() {
    while (seq_iss - seq_con < static_cast<uint32_t>(NST)) {
      if (!iss_in_nxt) {
        if (iss_page < cur.np) {
          issue_page(cur, iss_page++, item_par);
          continue;
        }
        iss_in_nxt = 1;
        iss_page = 0;
      }
      if (!nxt_valid || iss_page >= nxt.np) break;
      issue_page(nxt, iss_page++, item_par ^ 1u);
    }
  };
  pump();

  while (true) {
    // Tensor-core MMAs (mma.sync m16n8k16) on each page.  S^T = K Q^T holds
    // 16 tokens x 8 query heads (heads past G are zero); P^T goes back through
    // a register transpose; O^T = V^T P^T accumulates D x 8.
    constexpr int NK = D / 16;  // 16-column steps of a K row, and 16-row blocks of O^T
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t qb[NK][2];
    float acc[NK][4];
#pragma unroll
    for (int j = 0; j < NK; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    float mu0 = -INFINITY, mu1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2 tq and 2 tq + 1
    constexpr float kRescaleLog2 = 8.f;  // raise the reference max only when it grows by 2^8
    for (int pi = 0; pi < cur.np; ++pi) {
      const int st = seq_con % NST;
      if (!mbar_wait(full + st, (seq_con / NST) & 1u, nullptr)) {
        failed = true;
        break;
      }
      const uint32_t kb = smem_u32(stg + st * C::STAGE_BYTES), vb = kb + C::PAGE_BYTES;
      if (pi == 0) {
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(tail + item_par * C::Q_BYTES);
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
          qb[kk][0] = gq < G ? q32[(gq * D + 16 * kk + 2 * tq) >> 1] : 0u;
          qb[kk][1] = gq < G ? q32[(gq * D + 16 * kk + 8 + 2 * tq) >> 1] : 0u;
        }
      }
      const int tok0 = (cur.p0 + pi) * kPage;
      const int nv = min(kPage, cur.ctx - tok0);  // valid keys in this page (>= 1)
      // S^T: lane holds (token gq, heads 2 tq, 2 tq + 1) and (token gq + 8, same heads)
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) {
        const int r = lane & 15, chunk = (kk & 3) * 2 + (lane >> 4);
        uint32_t a[4];
        ldsm_x4(kb + (kk >> 2) * 2048 + r * 128 + ((chunk ^ (r & 7)) << 4), a);
        mma_16816_bf16(c, a, qb[kk][0], qb[kk][1]);
      }
      const float sl2 = p.scale_log2;
      const float s0 = gq < nv ? c[0] * sl2 : -INFINITY, s1 = gq < nv ? c[1] * sl2 : -INFINITY;
      const float s2 = gq + 8 < nv ? c[2] * sl2 : -INFINITY, s3 = gq + 8 < nv ? c[3] * sl2 : -INFINITY;
      float mh0 = fmaxf(s0, s2), mh1 = fmaxf(s1, s3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mh0 = fmaxf(mh0, __shfl_xor_sync(0xffffffffu, mh0, o));
        mh1 = fmaxf(mh1, __shfl_xor_sync(0xffffffffu, mh1, o));
      }
      const bool g0 = mh0 > mu0 + kRescaleLog2, g1 = mh1 > mu1 + kRescaleLog2;
      if (__any_sync(0xffffffffu, g0 || g1)) {
        const float n0 = g0 ? mh0 : mu0, n1 = g1 ? mh1 : mu1;
        const float a0 = g0 ? ex2(mu0 - n0) : 1.f, a1 = g1 ? ex2(mu1 - n1) : 1.f;
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          acc[j][0] *= a0;
          acc[j][1] *= a1;
          acc[j][2] *= a0;
          acc[j][3] *= a1;
        }
        l0 *= a0;
        l1 *= a1;
        mu0 = n0;
        mu1 = n1;
      }
      const float p0 = ex2(s0 - mu0), p1 = ex2(s1 - mu1), p2 = ex2(s2 - mu0), p3 = ex2(s3 - mu1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1), h23 = __floats2bfloat162_rn(p2, p3);
      // P^T as the B operand: lane holds (tokens 2 tq, 2 tq + 1 | + 8, head gq)
      const uint32_t b0 = movmatrix_trans(*reinterpret_cast<uint32_t*>(&h01));
      const uint32_t b1 = movmatrix_trans(*reinterpret_cast<uint32_t*>(&h23));
      if (nv < kPage) {
        // rows past the context in the last page may hold stale (even non-finite) data:
        // zero them in V so that P = 0 times V stays 0
        uint8_t* v0 = stg + st * C::STAGE_BYTES + C::PAGE_BYTES;
        for (int i = lane; i < (kPage - nv) * (D / 8); i += 32) {
          const int r = nv + i / (D / 8), cc = i % (D / 8);  // row, 16-byte chunk of the row
          *reinterpret_cast<uint4*>(v0 + (cc >> 3) * 2048 + r * 128 + (cc & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // ordered before the next copy into this stage
        __syncwarp();
      }
#pragma unroll
      for (int j = 0; j < NK; ++j) {
        const int r = ((lane >> 4) << 3) + (lane & 7), chunk = (j & 3) * 2 + ((lane >> 3) & 1);
        uint32_t a[4];
        ldsm_x4_trans(vb + (j >> 2) * 2048 + r * 128 + ((chunk ^ (r & 7)) << 4), a);
        mma_16816_bf16(acc[j], a, b0, b1);
      }
      __syncwarp();
      ++seq_con;
      pump();
    }
    if (failed) break;
    // O^T: lane holds (d 16 j + gq, heads 2 tq, 2 tq + 1) and (d 16 j + gq + 8, same heads)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hh = 2 * tq + e;
      if (hh >= G) continue;
      const float L = e == 0 ? l0 : l1, M = e == 0 ? mu0 : mu1;
      if (cur.ns == 1) {
        const float inv = 1.f / L;
        bf16* dst = p.out + (static_cast<int64_t>(cur.tok) * p.H_q + cur.hk * G + hh) * D;
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          dst[16 * j + gq] = __float2bfloat16_rn(acc[j][e] * inv);
          dst[16 * j + gq + 8] = __float2bfloat16_rn(acc[j][2 + e] * inv);
        }
      } else {
        const int64_t rec = cur.part + hh;
        float* dst = p.part_acc + rec * D;
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          dst[16 * j + gq] = acc[j][e];
          dst[16 * j + gq + 8] = acc[j][2 + e];
        }
        if (gq == 0) *reinterpret_cast<float2*>(p.part_ml + rec * 2) = make_float2(M, L);
      }
    }
    if (cur.ns > 1) {
      __threadfence();  // this split's records are visible before it is counted
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(p.dec_cnt + cur.k * p.H_kv + cur.hk, 1) == cur.ns - 1;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        merge_splits<D>(p, cur.k, cur.hk * G, G, cur.tok, cur.ns, lane);
      }
    }
    if (!nxt_valid) break;
    // advance: the next item becomes current; dequeue one more
    cur = nxt;
    item_par ^= 1u;
    iss_in_nxt = 0;  // the issue cursor (iss_page) already points into the new current item
    nxt_id = dequeue();
    nxt_valid = nxt_id < n_items;
    if (nxt_valid) nxt = describe_dec(p, nxt_id, split);
    pump();
  }
  if (failed) {
    if (lane == 0) atomicOr(p.hdr + H_STATUS, MS_STATUS_TIMEOUT);
    // let copies already in flight land before the CTA's shared memory is released
    while (seq_con < seq_iss) {
      mbar_wait(full + seq_con % NST, (seq_con / NST) & 1u, nullptr, 200000000ull);
      ++seq_con;
    }
  }
}

// ----------------------------------------------------------------------------
// chunk rows: tcgen05 tensor cores, TMEM accumulators, TMA-staged pages
// ----------------------------------------------------------------------------

constexpr int kQSlab = 128 * 128;  // one 128-row x 64-column bf16 slab of a Q tile (128-byte rows)
constexpr int kKVSlab = 64 * 128;  // one 64-key x 64-column bf16 slab of a K or V tile
constexpr int kKeys = 64;          // keys per KV tile
constexpr int kTilePages = kKeys / kPage;

template <int D>
struct ChCfg {
  static constexpr int NSL = D / 64;                  // 64-column slabs per row
  static constexpr int Q_BYTES = NSL * kQSlab;        // one 128-row Q tile
  static constexpr int Q_OFF = 0;                     // Q tile t at Q_OFF + t * Q_BYTES
  static constexpr int KVS = D == 128 ? 4 : 6;        // K/V pipeline stages
  static constexpr int KV_OFF = 2 * Q_BYTES;          // stage b: K at KV_OFF + b*2*NSL*kKVSlab, V after K
  static constexpr int BAR_OFF = KV_OFF + 2 * KVS * NSL * kKVSlab;
  static constexpr int SMEM = BAR_OFF + 1024;         // dynamic shared memory starts 1024-aligned
  static constexpr int TMEM_COLS = 512;
  static constexpr int O_COL = 128;                   // O of Q tile t at column t * O_COL
  static constexpr int S_COL = 256;                   // S/P buffer b of Q tile t at S_COL + (2t + b) * 64
};

// A work item is a pair of consecutive 128-row Q tiles of one chunk row and KV
// head; both read every K/V tile the pair needs from the same shared stages.
struct ChItem {
  int row, tb, c, hk;
  int n_kt;     // KV tiles the pair needs (those of its later tile)
  int kv0;      // CTA-global index of the item's first KV tile (stage and parity)
  int tok0[2], ntok[2], kv_end[2], nkt[2];  // per Q tile; ntok[1] == 0: no second tile
  int t0[2];    // per Q tile: index of its first KV tile among all tiles its softmax group ran
};

struct ChBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[8], k_empty[8];  // K stage: free once both S issuers' MMAs are done
  uint64_t v_full[8], v_empty[8];  // V stage: free once the PV issuer's MMAs are done
  uint64_t s_full[2][2], p_full[2][2], o_done[2][2];  // [Q tile][S/P buffer]
  uint64_t item_full[2], item_empty[2];
  uint64_t mma_done[3];
  uint32_t tmem;
  int abort;
  ChItem items[2];
};

static_assert(sizeof(ChBars) <= 1024, "chunk-phase barrier block exceeds its reserved space");
static_assert(DecCfg<128, 8>::SMEM <= 232448 && DecCfg<64, 8>::SMEM <= 232448 && DecCfg<128, 4>::WARPS == 12,
              "decode rings exceed the per-CTA shared-memory limit");
static_assert(ChCfg<128>::SMEM <= 232448 && ChCfg<64>::SMEM <= 232448,
              "chunk phase exceeds the per-CTA shared-memory limit");
static_assert(ChCfg<128>::KVS <= 8 && ChCfg<64>::KVS <= 8, "more K/V stages than barriers");

// wait by lane 0, result and ordering shared with the whole warp
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                          uint64_t limit_ns) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, limit_ns) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Chunk phase.  Warp 0 owns the work queue and streams Q and K/V with TMA (K
// one tile ahead of V); warps 2-5 and 6-9 are two softmax groups, group t
// owning Q tile t of the current pair, one query row per thread over 64-key
// tiles.  The S MMAs of the two groups and the PV MMAs are three independent
// streams, so three warps issue them: warp 1 the S MMAs of group 0, warp 10
// those of group 1, and warp 11 the PV MMAs of both (one issuer would queue
// one group's PV behind the other's S).  Each group has two S buffers in
// TMEM, so its next S is computed while it exponentiates the current one, and
// P (bf16) overwrites the S values it came from, where the PV MMA reads it.
// The two groups run a tile apart at most, so one group's exponentials
// overlap the other group's MMAs.  Returns when the chunk queue is empty; the
// caller owns TMEM and the barrier invalidation.
template <int D, int G>
__device__ __noinline__ void chunk_phase(const CUtensorMap* tm_q_p, const CUtensorMap* tm_k_p,
                                            const CUtensorMap* tm_v_p, const CUtensorMap* tm_vp_p,
                                            const AttnParams& p, uint8_t* smem, uint32_t tmem) {
  using C = ChCfg<D>;
  constexpr int NSL = C::NSL;
  constexpr int TPT = 128 / G;  // query tokens per 128-row Q tile
  constexpr int KVS = C::KVS;
  const CUtensorMap& tm_q = *tm_q_p;
  const CUtensorMap& tm_k = *tm_k_p;
  const CUtensorMap& tm_v = *tm_v_p;
  const CUtensorMap& tm_vp = *tm_vp_p;  // V by whole pages (D = 128)
  ChBars* bars = reinterpret_cast<ChBars*>(smem + C::BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.hdr[H_NCH_ITEMS];

  const uint32_t sbase = smem_u32(smem);
  auto k_off = [](int b) { return C::KV_OFF + b * 2 * NSL * kKVSlab; };
  auto v_off = [](int b) { return C::KV_OFF + b * 2 * NSL * kKVSlab + NSL * kKVSlab; };
  // A V stage holds its tile page by page: key k of the tile at
  // (k / 16) * kVPage + slab * 2048 + (k % 16) * 128.  A page is one TMA box
  // (two 2 KB boxes of K cost about as much TMA time as one 4 KB box).
  constexpr int kVPage = NSL * 2048;
  auto s_col = [&](int t, int b) { return tmem + C::S_COL + (2 * t + b) * 64; };

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 2);  // one commit per S issuer
    for (int b = 0; b < 8; ++b) {  // all of them, so that all can be invalidated
      mbar_init(&bars->k_full[b], 1);
      mbar_init(&bars->k_empty[b], 2);
      mbar_init(&bars->v_full[b], 1);
      mbar_init(&bars->v_empty[b], 1);
    }
    for (int t = 0; t < 2; ++t)
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bars->s_full[t][b], 1);
        mbar_init(&bars->p_full[t][b], 128);  // the four warps of group t
        mbar_init(&bars->o_done[t][b], 1);
      }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->item_full[b], 1);
      mbar_init(&bars->item_empty[b], 3 + 32 * kSoftmaxWarps);  // MMA issuers, softmax threads
    }
    for (int i = 0; i < 3; ++i) mbar_init(&bars->mma_done[i], 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &bars->abort;
  const uint64_t lim = p.wait_limit_ns;

  if (warp == 0) {
    // ---------------------------------------------------------------- work queue + TMA producer
    // The whole warp runs this loop: lane 0 owns the queue, the waits and the
    // barrier bookkeeping; a tile's K boxes -- one per (page, 64-column slab)
    // -- go out as one warp-wide TMA instruction, lane L taking page L / NSL,
    // slab L % NSL; its V boxes likewise, one per page (lanes with slab 0).
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(NSL == 2 ? &tm_vp : &tm_v);
    }
    const int my_pg = lane / NSL, my_s = lane % NSL;
    const bool loader = lane < kTilePages * NSL;
    int g = 0;               // CTA-global KV tile counter
    int g_v = 0;             // tiles whose V has been issued
    int n_done = 0;          // items taken by this CTA
    int t_run[2] = {0, 0};   // KV tiles run by each softmax group so far
    // Test hook (never set by a real call): publish no work item and issue no
    // copy, as a producer that stopped would.  Every other role then waits on
    // an item that never comes until its bounded wait gives up, with nothing
    // in flight: the timeout path runs exactly as it would in a real stall.
    const bool stalled = p.test_stall != 0;
    bool ok = !stalled;
    auto lane0_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      int r = 1;
      if (lane == 0) r = mbar_wait(bar, parity, abort_flag, lim) ? 1 : 0;
      r = __shfl_sync(0xffffffffu, r, 0);
      return r != 0;
    };
    // V of tile gv (one tile behind K): its stage was last read by the PV MMAs of gv - KVS
    auto load_v = [&](int gv, int row0, int npg) -> bool {
      const int bv = gv % KVS;
      if (gv >= KVS && !lane0_wait(&bars->v_empty[bv], ((gv / KVS) - 1) & 1)) return false;
      if (lane == 0) mbar_arrive_expect_tx(&bars->v_full[bv], npg * kPage * D * 2);
      __syncwarp();
      if constexpr (NSL == 2) {
        if (loader && my_s == 0 && my_pg < npg)
          tma_load_4d(smem + v_off(bv) + my_pg * kVPage, &tm_vp, 0, 0, 0, row0 / kPage, &bars->v_full[bv]);
      } else {
        if (loader && my_pg < npg)
          tma_load_2d(smem + v_off(bv) + my_pg * kVPage, &tm_v, 0, row0, &bars->v_full[bv]);
      }
      return true;
    };
    while (ok) {
      int item = 0;
      if (lane == 0) item = atomicAdd(p.hdr + H_CH_CTR, 1);
      item = __shfl_sync(0xffffffffu, item, 0);
      const int slot = n_done & 1;
      if (n_done >= 2 && !lane0_wait(&bars->item_empty[slot], ((n_done >> 1) - 1) & 1)) {
        ok = false;
        break;
      }
      ChItem it;
      it.row = -1;
      if (item < n_items) {
        const int2 kl = __ldg(p.ch_items + item);  // (chunk row index, KV head << 16 | pair from the last)
        const int k = kl.x;
        it.row = __ldg(p.ch_rows + k);
        it.tb = __ldg(p.cu + it.row);
        const int d = __ldg(p.cu + it.row + 1) - it.tb;
        it.c = __ldg(p.q_start + it.row);
        const int n_qt = (d + TPT - 1) / TPT;
        const int n_pair = (n_qt + 1) >> 1;
        // the prologue ordered the row's items (KV head by KV head, or longest pair
        // first); later Q-tile pairs see more keys
        it.hk = kl.y >> 16;
        const int pair = n_pair - 1 - (kl.y & 0xffff);
        it.n_kt = 0;
        for (int t = 0; t < 2; ++t) {
          const int qt = 2 * pair + t;
          const bool has = qt < n_qt;
          it.tok0[t] = has ? qt * TPT : 0;
          it.ntok[t] = has ? min(TPT, d - qt * TPT) : 0;
          it.kv_end[t] = has ? it.c + it.tok0[t] + it.ntok[t] : 0;
          it.nkt[t] = (it.kv_end[t] + kKeys - 1) / kKeys;
          it.t0[t] = t_run[t];
          t_run[t] += it.nkt[t];
          it.n_kt = max(it.n_kt, it.nkt[t]);
        }
        it.kv0 = g;
      }
      if (lane == 0) {
        bars->items[slot] = it;
        mbar_arrive(&bars->item_full[slot]);
      }
      ++n_done;
      if (it.row < 0) break;
      // Q tiles: the previous item's S MMAs must be done with them
      if (n_done >= 2 && !lane0_wait(&bars->q_empty, (n_done - 2) & 1)) {
        ok = false;
        break;
      }
      const int nq = it.ntok[1] > 0 ? 2 : 1;
      if (lane == 0) mbar_arrive_expect_tx(&bars->q_full, nq * 128 * D * 2);
      __syncwarp();
      if (lane < nq * NSL) {
        const int t = lane / NSL, s = lane % NSL;
        tma_load_3d(smem + C::Q_OFF + t * C::Q_BYTES + s * kQSlab, &tm_q, s * 64, it.hk * G, it.tb + it.tok0[t],
                    &bars->q_full);
      }
      const int kv_max = max(it.kv_end[0], it.kv_end[1]);
      const int32_t* btrow = row_table(p, it.row);
      const int n_pages = (kv_max + kPage - 1) / kPage;
      // lane L < 4 holds the page id of page L of the current tile; the next tile's is in flight
      int pg_cur = lane < kTilePages && lane < n_pages ? __ldg(btrow + lane) : 0;
      int row0_prev = 0, npg_prev = 0;
      for (int kt = 0; kt < it.n_kt; ++kt, ++g) {
        const int lp = (kt + 1) * kTilePages + lane;
        const int pg_nxt = lane < kTilePages && lp < n_pages ? __ldg(btrow + lp) : 0;
        const int b = g % KVS;
        const int keys = min(kKeys, kv_max - kt * kKeys);
        const int npg = (keys + kPage - 1) / kPage;
        int phys = __shfl_sync(0xffffffffu, pg_cur, my_pg & (kTilePages - 1));
        if (loader && my_pg < npg && (phys < 0 || phys >= p.num_pages)) {
          atomicOr(p.hdr + H_STATUS, MS_STATUS_BAD_PAGE);
          phys = 0;
        }
        const int row0 = (phys * p.H_kv + it.hk) * kPage;
        // K of tile g: its stage was last read by the S MMAs of tile g - KVS
        if (g >= KVS && !lane0_wait(&bars->k_empty[b], ((g / KVS) - 1) & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&bars->k_full[b], npg * kPage * D * 2);
        __syncwarp();
        if (loader && my_pg < npg)
          tma_load_2d(smem + k_off(b) + my_s * kKVSlab + my_pg * 2048, &tm_k, my_s * 64, row0, &bars->k_full[b]);
        if (kt >= 1) {
          if (!load_v(g - 1, row0_prev, npg_prev)) {
            ok = false;
            break;
          }
          g_v = g;
        }
        row0_prev = row0;
        npg_prev = npg;
        pg_cur = pg_nxt;
      }
      if (!ok) break;
      if (!load_v(g - 1, row0_prev, npg_prev)) {
        ok = false;
        break;
      }
      g_v = g;
    }
    if (lane == 0) {
      if (!ok && !stalled) *abort_flag = 1;
      // copies still in flight must land before the CTA moves on
      for (int t = (g > KVS ? g - KVS : 0); t < g; ++t)
        mbar_wait(&bars->k_full[t % KVS], (t / KVS) & 1, nullptr, 200000000ull);
      for (int t = (g_v > KVS ? g_v - KVS : 0); t < g_v; ++t)
        mbar_wait(&bars->v_full[t % KVS], (t / KVS) & 1, nullptr, 200000000ull);
    }
  } else if (warp == 1 || warp == 2 + kSoftmaxWarps) {
    // ---------------------------------------------------------------- S issuer of one group
    // Every S issuer walks every KV tile of the item and commits to the K
    // stage's "empty" barrier (two commits per phase), issuing MMAs only for
    // the tiles its Q tile needs.  It waits for each stage to be full even
    // when it has no MMA for it: that keeps its commits in step with the
    // producer, so a phase can never complete on commits meant for a later one.
    // The issue loops keep every per-item value in registers, step through the
    // stage rings with counters, and build each operand descriptor once per tile:
    // a k-step or a stage only moves the descriptor's start-address field
    // (bytes >> 4, 14 bits, no carry below 256 KB) by a constant.
    const int t = warp == 1 ? 0 : 1;
    if (lane == 0) {
      const uint64_t qdesc = smem_desc_sw128(sbase + C::Q_OFF + t * C::Q_BYTES, 16, 1024);
      const uint64_t kdesc0 = smem_desc_sw128(sbase + C::KV_OFF, 16, 1024);
      const uint32_t s_tm = tmem + C::S_COL + 2 * t * 64;
      constexpr uint32_t idesc_full = idesc_bf16_f32(128, kKeys, 0);
      int bk = 0;        // K stage of the next tile
      uint32_t kph = 0;  // its phase parity
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int slot = n & 1;
        if (!mbar_wait(&bars->item_full[slot], (n >> 1) & 1, abort_flag, lim)) {
          ok = false;
          break;
        }
        const ChItem& it = bars->items[slot];  // stable until this role arrives on item_empty
        const int row = it.row;
        if (row < 0) break;
        const int nkt = it.nkt[t], t0 = it.t0[t], n_kt = it.n_kt;
        const int kv_max = max(it.kv_end[0], it.kv_end[1]);
        if (nkt > 0 && !mbar_wait(&bars->q_full, n & 1, abort_flag, lim)) {
          ok = false;
          break;
        }
        for (int kt = 0; kt < n_kt; ++kt) {
          if (!mbar_wait_fast(&bars->k_full[bk], kph, abort_flag, 16, lim)) {
            ok = false;
            break;
          }
          if (kt < nkt) {
            const int gt = t0 + kt, b = gt & 1;
            // S buffer b last held P of the group's tile gt - 2: its PV MMA must be done
            if (gt >= 2 && !mbar_wait_fast(&bars->o_done[t][b], ((gt - 2) >> 1) & 1, abort_flag, 16, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int keys = kv_max - kt * kKeys;  // at least kKeys but on the last tile
            const uint32_t idesc_s = keys >= kKeys ? idesc_full : idesc_bf16_f32(128, (keys + 15) & ~15, 0);
            const uint64_t kd = kdesc0 + static_cast<uint64_t>((bk * 2 * NSL * kKVSlab) >> 4);
            const uint32_t dcol = s_tm + b * 64;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t qo = static_cast<uint64_t>(((kk >> 2) * kQSlab + (kk & 3) * 32) >> 4);
              const uint64_t ko = static_cast<uint64_t>(((kk >> 2) * kKVSlab + (kk & 3) * 32) >> 4);
              mma_bf16_ss(dcol, qdesc + qo, kd + ko, idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars->s_full[t][b]);
          }
          mma_commit(&bars->k_empty[bk]);
          if (kt == n_kt - 1) mma_commit(&bars->q_empty);
          if (++bk == KVS) {
            bk = 0;
            kph ^= 1u;
          }
        }
        if (!ok) break;
        mbar_arrive(&bars->item_empty[slot]);
      }
      if (!ok) *abort_flag = 1;
      // every MMA this thread issued must finish before TMEM is reused or released
      mma_commit(&bars->mma_done[t]);
      mbar_wait(&bars->mma_done[t], 0, nullptr, 200000000ull);
    }
  } else if (warp == 3 + kSoftmaxWarps) {
    // ---------------------------------------------------------------- PV issuer of both groups
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);
      // V is the MN-major B operand, one page per k-step of 16 keys: the page's
      // 64-column slabs 2048 B apart (LBO), its two 8-key row groups 1024 B apart
      // (SBO).  P (A operand) is in TMEM: 16 keys = 8 packed columns per k-step.
      const uint64_t vdesc0 = smem_desc_sw128(sbase + C::KV_OFF + NSL * kKVSlab, 2048, 1024);
      int bv = 0;        // V stage of the next tile
      uint32_t vph = 0;  // its phase parity
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int slot = n & 1;
        if (!mbar_wait(&bars->item_full[slot], (n >> 1) & 1, abort_flag, lim)) {
          ok = false;
          break;
        }
        const ChItem& it = bars->items[slot];  // stable until this role arrives on item_empty
        const int row = it.row;
        if (row < 0) break;
        const int n_kt = it.n_kt;
        const int nkt_[2] = {it.nkt[0], it.nkt[1]}, t0_[2] = {it.t0[0], it.t0[1]};
        const int ke_[2] = {it.kv_end[0], it.kv_end[1]};
        const int kv_max = max(ke_[0], ke_[1]);
        for (int j = 0; j < n_kt && ok; ++j) {
          if (!mbar_wait_fast(&bars->v_full[bv], vph, abort_flag, 16, lim)) {
            ok = false;
            break;
          }
          const int keys = min(kKeys, kv_max - j * kKeys);  // keys loaded in this tile
          if ((keys & 15) != 0) {
            // rows past the context in the last page may hold stale (even non-finite)
            // data: zero them in V so that P = 0 times V stays 0
            uint8_t* v0 = smem + v_off(bv);
            for (int r = keys; r < ((keys + 15) & ~15); ++r)
              for (int s = 0; s < NSL; ++s)
                for (int q16 = 0; q16 < 8; ++q16)
                  *reinterpret_cast<uint4*>(v0 + (r >> 4) * kVPage + s * 2048 + (r & 15) * 128 + q16 * 16) =
                      make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
          }
          const uint64_t vd = vdesc0 + static_cast<uint64_t>((bv * 2 * NSL * kKVSlab) >> 4);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (j < nkt_[t]) {
              const int gt = t0_[t] + j, b = gt & 1;
              if (!mbar_wait_fast(&bars->p_full[t][b], (gt >> 1) & 1, abort_flag, 16, lim)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t dcol = tmem + t * C::O_COL;
              const uint32_t acol = s_col(t, b);
              const int kr = ke_[t] - j * kKeys;  // keys this Q tile sees in the tile
              if (kr >= kKeys) {
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk)
                  mma_bf16_ts(dcol, acol + kk * 8, vd + static_cast<uint64_t>((kk * kVPage) >> 4), idesc_pv,
                              (j > 0 || kk > 0) ? 1u : 0u);
              } else {
                const int nk_t = (kr + 15) >> 4;
                for (int kk = 0; kk < nk_t; ++kk)
                  mma_bf16_ts(dcol, acol + kk * 8, vd + static_cast<uint64_t>((kk * kVPage) >> 4), idesc_pv,
                              (j > 0 || kk > 0) ? 1u : 0u);
              }
              mma_commit(&bars->o_done[t][b]);
            }
          }
          if (!ok) break;
          mma_commit(&bars->v_empty[bv]);
          if (++bv == KVS) {
            bv = 0;
            vph ^= 1u;
          }
        }
        if (!ok) break;
        mbar_arrive(&bars->item_empty[slot]);
      }
      if (!ok) *abort_flag = 1;
      mma_commit(&bars->mma_done[2]);
      mbar_wait(&bars->mma_done[2], 0, nullptr, 200000000ull);
    }
  } else if (warp >= 2 && warp < 2 + kSoftmaxWarps) {
    // ---------------------------------------------------------------- softmax
    const int t = (warp - 2) >> 2;              // Q tile of this group
    const int quad = warp & 3;                  // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;             // query row of this thread
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tO = tmem + t * C::O_COL + lane_off;
    const float sl2 = p.scale_log2;
    // A row exponentiates against m_use, the largest scaled score seen when it
    // was last raised; it is raised (and O rescaled) only when a tile's max
    // exceeds it by more than 2^8, so P <= 256 and O, l stay exact in fp32.
    constexpr float kRescaleLog2 = 8.f;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int slot = n & 1;
      if (!warp_wait(&bars->item_full[slot], (n >> 1) & 1, abort_flag, lim)) {
        ok = false;
        break;
      }
      const ChItem& it = bars->items[slot];  // stable until this role arrives on item_empty
      if (it.row < 0) break;
      const int nkt = it.nkt[t];
      if (nkt > 0) {
        const int tl = it.tok0[t] + r / G;  // token of this row within the chunk
        const bool valid = (r / G) < it.ntok[t];
        const int pos = it.c + (valid ? tl : it.tok0[t] + it.ntok[t] - 1);
        const int warp_min_pos = it.c + it.tok0[t] + (quad * 32) / G;  // smallest position of this warp's rows
        float m_use = -INFINITY, l = 0.f;
        for (int kt = 0; kt < nkt; ++kt) {
          const int gt = it.t0[t] + kt, b = gt & 1;
          if (!warp_wait(&bars->s_full[t][b], (gt >> 1) & 1, abort_flag, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t r0[32], r1[32];
          const uint32_t ts = s_col(t, b) + lane_off;
          tmem_ld32(ts, r0);
          tmem_ld32(ts + 32, r1);
          tmem_wait_ld();
          reg_fence32(r0);
          reg_fence32(r1);
          float sv[64];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            sv[j] = __uint_as_float(r0[j]);
            sv[32 + j] = __uint_as_float(r1[j]);
          }
          const int key0 = kt * kKeys;
          if (key0 + kKeys - 1 > warp_min_pos) {  // diagonal or ragged tile: causal mask (warp-uniform test)
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (key0 + j > pos) sv[j] = -INFINITY;
          }
          // row max: four chains of three-input maxima
          float mxa[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float m = fmax3(sv[c], sv[c + 4], sv[c + 8]);
#pragma unroll
            for (int j = 12; j < 60; j += 8) m = fmax3(m, sv[j + c], sv[j + 4 + c]);
            mxa[c] = fmaxf(m, sv[60 + c]);
          }
          const float mx = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3]));
          const float mx_s = mx * sl2;
          const bool grow = mx_s > m_use + kRescaleLog2;
          const float m_new = grow ? mx_s : m_use;
          const float alpha = grow ? ex2(m_use - m_new) : 1.f;
          const float neg_m = -m_new;
          // exponentials, two elements per packed FMA and packed add
          const float2 sl2x2 = make_float2(sl2, sl2), negm2 = make_float2(neg_m, neg_m);
          float2 rsa[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float2 x = ffma2(make_float2(sv[j], sv[j + 1]), sl2x2, negm2);
            const float2 e = make_float2(ex2(x.x), ex2(x.y));
            sv[j] = e.x;
            sv[j + 1] = e.y;
            rsa[(j >> 1) & 1] = fadd2(rsa[(j >> 1) & 1], e);
          }
          l = l * alpha + ((rsa[0].x + rsa[0].y) + (rsa[1].x + rsa[1].y));
          m_use = m_new;
          // P (bf16 pairs) over the first 32 columns of the S values it came from.
          // Packing before the rescale keeps 32 registers live through it instead of
          // 64, and the store runs while O is rescaled.
          uint32_t pw[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(sv[2 * j], sv[2 * j + 1]);
            pw[j] = *reinterpret_cast<uint32_t*>(&h2);
          }
          tmem_st32u(ts, pw);
          if (kt > 0 && __any_sync(0xffffffffu, grow)) {  // rescale this row's O
            // the PV MMA of the previous tile must be done with O first
            if (!warp_wait(&bars->o_done[t][(gt - 1) & 1], ((gt - 1) >> 1) & 1, abort_flag, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t rr[32];
              tmem_ld32(tO + cc * 32, rr);
              tmem_wait_ld();
              reg_fence32(rr);
#pragma unroll
              for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * alpha);
              tmem_st32u(tO + cc * 32, rr);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->p_full[t][b]);
        }
        if (!ok) break;
        const int gl = it.t0[t] + nkt - 1;
        if (!warp_wait(&bars->o_done[t][gl & 1], (gl >> 1) & 1, abort_flag, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv = 1.f / l;
        bf16* dst = p.out + (static_cast<int64_t>(it.tb + tl) * p.H_q + it.hk * G + r % G) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(tO + cc * 32, rr);
          tmem_wait_ld();
          reg_fence32(rr);
          if (valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 u;
              __nv_bfloat162 h0 =
                  __floats2bfloat162_rn(__uint_as_float(rr[j]) * inv, __uint_as_float(rr[j + 1]) * inv);
              __nv_bfloat162 h1 =
                  __floats2bfloat162_rn(__uint_as_float(rr[j + 2]) * inv, __uint_as_float(rr[j + 3]) * inv);
              __nv_bfloat162 h2 =
                  __floats2bfloat162_rn(__uint_as_float(rr[j + 4]) * inv, __uint_as_float(rr[j + 5]) * inv);
              __nv_bfloat162 h3 =
                  __floats2bfloat162_rn(__uint_as_float(rr[j + 6]) * inv, __uint_as_float(rr[j + 7]) * inv);
              u.x = *reinterpret_cast<uint32_t*>(&h0);
              u.y = *reinterpret_cast<uint32_t*>(&h1);
              u.z = *reinterpret_cast<uint32_t*>(&h2);
              u.w = *reinterpret_cast<uint32_t*>(&h3);
              *reinterpret_cast<uint4*>(dst + cc * 32 + j) = u;
            }
          }
        }
      }
      // O has been read: the next item's first PV may overwrite it
      tc_fence_before();
      mbar_arrive(&bars->item_empty[slot]);
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(p.hdr + H_STATUS, MS_STATUS_TIMEOUT);
    }
  }
  (void)n_items;
}

// barriers of one finished phase, invalidated before the memory is reused
template <int D, int G>
__device__ __forceinline__ void invalidate_phase_barriers(uint8_t* smem, bool chunk) {
  if (chunk) {
    if (threadIdx.x == 0) {
      ChBars* bars = reinterpret_cast<ChBars*>(smem + ChCfg<D>::BAR_OFF);
      uint64_t* b0 = &bars->q_full;
      uint64_t* b1 = &bars->mma_done[2];
      for (uint64_t* b = b0; b <= b1; ++b) mbar_inval(b);
    }
  } else if ((threadIdx.x & 31) == 0 && (threadIdx.x >> 5) < DecCfg<D, G>::WARPS) {
    using C = DecCfg<D, G>;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::TAIL_OFF + (threadIdx.x >> 5) * C::TAIL_BYTES + C::T_BAR);
    for (int i = 0; i < C::NST; ++i) mbar_inval(full + i);
  }
}

// One persistent CTA per SM.  CTAs on SMs below hdr[H_CHUNK_CTAS] start on chunk
// tiles (tensor cores), the others on decode items (HBM), so the two kinds of
// work run side by side; a CTA whose queue runs dry moves to the other queue.
template <int D, int G>
__global__ void __launch_bounds__(kChunkThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_vp,
                     const __grid_constant__ CUtensorMap tm_kp,
                     AttnParams p) {
  // no static shared memory: the dynamic block starts 1024-aligned, as the
  // 128-byte-swizzled TMA tiles and MMA descriptors require
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  if ((smem_u32(smem) & 1023u) != 0) {
    griddep_wait();
    if (threadIdx.x == 0) atomicOr(p.hdr + H_STATUS, MS_STATUS_INTERNAL);
    return;
  }
  // set-up that needs nothing from the kernels before: it overlaps their tail
  // when this kernel is launched as a programmatic dependent
  uint32_t* tmem_slot = &reinterpret_cast<ChBars*>(smem + ChCfg<D>::BAR_OFF)->tmem;
  if (warp == 1) {
    tmem_alloc(tmem_slot, ChCfg<D>::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // the prologue's item tables (and, through it, the append's q_rot and pages)
  // CTA 0 times its own run in SM cycles and in ns: the SM clock, for the next call's cost model
  const long long clk0 = clock64();
  const uint64_t ns0 = globaltimer_ns();
  const int n_ch_items = p.hdr[H_NCH_ITEMS];
  const int n_dec_items = p.hdr[H_NDEC_ITEMS];
  __syncthreads();  // every thread holds the address before the phases reuse the memory
  if (n_ch_items == 0 && n_dec_items == 0) {
    if (warp == 1) tmem_dealloc(tmem, ChCfg<D>::TMEM_COLS);
    return;
  }
  // Which CTAs start on chunk work goes by the SM they run on, not by block
  // index: as a programmatic dependent, the kernel's blocks reach SMs in an
  // order set by the kernels still draining, and a split by block index then
  // lands differently from step to step (up to 6 % slower on the long bimodal
  // step).  It only sets where a CTA starts; any count of chunk-first CTAs is
  // correct, since a CTA whose queue runs dry takes the other one.
  uint32_t smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  const bool chunk_first = static_cast<int>(smid) < p.hdr[H_CHUNK_CTAS];
  for (int ph = 0; ph < 2; ++ph) {
    const bool chunk = (ph == 0) == chunk_first;
    if (chunk && n_ch_items > 0) {
      chunk_phase<D, G>(&tm_q, &tm_k, &tm_v, &tm_vp, p, smem, tmem);
      tc_fence_before();
      __syncthreads();
      const bool aborted = reinterpret_cast<ChBars*>(smem + ChCfg<D>::BAR_OFF)->abort != 0;
      invalidate_phase_barriers<D, G>(smem, true);
      __syncthreads();
      if (aborted) break;
    } else if (!chunk && n_dec_items > 0) {
      decode_phase<D, G>(p, smem, &tm_k, &tm_v, &tm_kp, &tm_vp);
      __syncwarp();
      invalidate_phase_barriers<D, G>(smem, false);
      __syncthreads();
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ChCfg<D>::TMEM_COLS);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const uint64_t ns = globaltimer_ns() - ns0;
    if (ns >= 20000)  // long enough for the timer's resolution
      p.hdr[H_CLOCK_MHZ] = static_cast<int>(static_cast<double>(clock64() - clk0) * 1e3 / static_cast<double>(ns));
  }
}


}  // namespace

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------

namespace {

struct WsLayout {
  size_t hdr, dec_rows, dec_part_base, dec_nsplit, ch_rows, dec_cnt, dec_items,
      ch_items, part_ml, part_acc, total;
  int64_t max_partials, max_dec_items, max_ch_items;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsLayout ws_layout(int64_t max_rows, int64_t max_tokens, int64_t max_context_total, int64_t H_q, int64_t H_kv,
                   int64_t D) {
  WsLayout w;
  size_t off = 0;
  w.hdr = off;
  off += H_WORDS * 4;
  w.dec_rows = off;
  off = align_up(off + max_rows * 4, 16);
  w.dec_part_base = off;
  off = align_up(off + max_rows * 4, 16);
  w.dec_nsplit = off;
  off = align_up(off + max_rows * 4, 16);
  w.ch_rows = off;
  off = align_up(off + max_rows * 4, 16);
  w.dec_cnt = off;
  off = align_up(off + max_rows * H_kv * 4, 256);
  // every decode split covers >= kMinSplitPages pages: splits <= ctx / (16 * kMinSplitPages) + rows
  const int64_t max_splits = cdiv64(max_context_total, kPage * kMinSplitPages) + 2 * max_rows;
  const int64_t G = H_q / (H_kv > 0 ? H_kv : 1);
  w.max_dec_items = H_kv * max_splits;
  w.max_ch_items = H_kv * (cdiv64(max_tokens * G, 128) + max_rows);
  w.dec_items = off;  // one entry per split: the KV head is not in the table
  off = align_up(off + (w.max_dec_items / H_kv) * 8, 256);
  w.ch_items = off;  // one entry per chunk item
  off = align_up(off + w.max_ch_items * 8, 256);
  w.max_partials = H_q * max_splits;
  w.part_ml = off;
  off = align_up(off + w.max_partials * 2 * 4, 256);
  w.part_acc = off;
  off = align_up(off + w.max_partials * D * 4, 256);
  w.total = off;
  return w;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the driver's tensor-map encoder, looked up once (thread-safe static initialisation)
EncodeTiledFn get_encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return nullptr;
  }();
  return fn;
}

bool encode_bf16(EncodeTiledFn fn, CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                 const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  cuuint32_t elem[5] = {1, 1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides_bytes, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device host state (devices 0 .. kMaxDevices - 1): the SM count and which
// kernels have had their shared-memory limit raised.  Safe to use from
// several host threads: every entry is computed the same way by whoever gets
// there first.
constexpr int kMaxDevices = 64;
std::atomic<int> g_num_sms[kMaxDevices];
std::atomic<uint32_t> g_smem_attr_set[kMaxDevices];

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return -1;
  const int cached = g_num_sms[dev].load(std::memory_order_relaxed);
  if (cached > 0) return cached;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
  g_num_sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

// The cost model's device rates, looked up once per device: the rated SM
// clock (MHz) and the HBM bandwidth (GB/s), nominal (memory clock x bus width,
// double data rate) times the sustained copy share.
std::atomic<float> g_sm_mhz[kMaxDevices], g_hbm_gbs[kMaxDevices], g_l2_bytes[kMaxDevices];

int device_rates(float* sm_mhz, float* hbm_gbs, float* l2_bytes) {
  const int dev = current_device();
  if (dev < 0) return MS_ERR_CUDA;
  float mhz = g_sm_mhz[dev].load(std::memory_order_relaxed);
  float gbs = g_hbm_gbs[dev].load(std::memory_order_relaxed);
  float l2 = g_l2_bytes[dev].load(std::memory_order_relaxed);
  if (!(mhz > 0.f) || !(gbs > 0.f) || !(l2 > 0.f)) {
    int clk_khz = 0, mem_khz = 0, bus_bits = 0, l2_b = 0;
    if (cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&mem_khz, cudaDevAttrMemoryClockRate, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&bus_bits, cudaDevAttrGlobalMemoryBusWidth, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2_b, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return MS_ERR_CUDA;
    mhz = clk_khz > 0 ? clk_khz * 1e-3f : 2000.f;
    gbs = mem_khz > 0 && bus_bits > 0 ? 2.f * mem_khz * 1e3f * (bus_bits / 8.f) * 1e-9f * kHbmCopyEfficiency : 6500.f;
    l2 = l2_b > 0 ? static_cast<float>(l2_b) : 64.f * (1 << 20);
    g_sm_mhz[dev].store(mhz, std::memory_order_relaxed);
    g_hbm_gbs[dev].store(gbs, std::memory_order_relaxed);
    g_l2_bytes[dev].store(l2, std::memory_order_relaxed);
  }
  *sm_mhz = mhz;
  *hbm_gbs = gbs;
  *l2_bytes = l2;
  return MS_OK;
}

// Raise `kernel`'s dynamic shared-memory limit on the current device once
// (bit `slot` of the device's mask).
template <typename Kernel>
int ensure_smem_limit(Kernel kernel, int slot, int bytes) {
  const int dev = current_device();
  if (dev < 0) return MS_ERR_CUDA;
  if (g_smem_attr_set[dev].load(std::memory_order_acquire) & (1u << slot)) return MS_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return MS_ERR_CUDA;
  g_smem_attr_set[dev].fetch_or(1u << slot, std::memory_order_release);
  return MS_OK;
}

// Launch as a programmatic dependent of the previous kernel on the stream: the
// kernel may start while that one finishes and orders itself with
// griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// decode worker warps per CTA for head dim D and group size G
int dec_warps(int D, int G) {
  switch (D * 100 + G) {
    case 6401: return DecCfg<64, 1>::WARPS;
    case 6402: return DecCfg<64, 2>::WARPS;
    case 6404: return DecCfg<64, 4>::WARPS;
    case 6408: return DecCfg<64, 8>::WARPS;
    case 12801: return DecCfg<128, 1>::WARPS;
    case 12802: return DecCfg<128, 2>::WARPS;
    case 12804: return DecCfg<128, 4>::WARPS;
    default: return DecCfg<128, 8>::WARPS;
  }
}

template <int D, int G>
int launch_paths(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& tvp, const CUtensorMap& tkp, int n_ctas, cudaStream_t st) {
  constexpr int smem = ChCfg<D>::SMEM > DecCfg<D, G>::SMEM ? ChCfg<D>::SMEM : DecCfg<D, G>::SMEM;
  static_assert(smem <= 232448, "attention kernel exceeds the per-CTA shared-memory limit");
  const int slot = (D == 128 ? 4 : 0) + (G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3);  // one bit per instance
  if (ensure_smem_limit(attention_kernel<D, G>, slot, smem) != MS_OK) return MS_ERR_CUDA;
  if (launch_dependent(attention_kernel<D, G>, dim3(n_ctas), dim3(kChunkThreads), smem, st, tq, tk, tv, tvp, tkp,
                       p) != cudaSuccess)
    return MS_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MS_OK : MS_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" MS_API size_t ms_attention_workspace_size(int32_t max_rows, int32_t max_tokens, int64_t max_context_total,
                                                     int32_t H_q, int32_t H_kv, int32_t D) {
  if (max_rows < 0 || max_tokens < 0 || max_context_total < 0 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 ||
      (D != 64 && D != 128))
    return 0;
  return ws_layout(max_rows, max_tokens, max_context_total, H_q, H_kv, D).total;
}

extern "C" MS_API int ms_cost_model_rates(float* sm_mhz, float* hbm_gbs) {
  if (sm_mhz == nullptr || hbm_gbs == nullptr) return MS_ERR_ARG;
  float l2 = 0.f;
  return device_rates(sm_mhz, hbm_gbs, &l2);
}

extern "C" MS_API int ms_num_sms(void) {
  const int n = num_sms();
  return n > 0 ? n : MS_ERR_CUDA;
}

namespace {

// An attention call's launch parameters: the kernels' arguments and the four
// tensor maps.
struct AttnPlan {
  AttnParams p;
  CUtensorMap tq, tk, tv, tvp, tkp;
};

// Checks every argument of an attention call and fills *L; enqueues nothing.
// *empty: the step has no tokens, so there is nothing to launch.
// clear_status makes the prologue zero the status word before anything of
// this call can set it.  stall_limit_ns > 0 is the test hook of
// ms_test_attention_stall: chunk-phase producers publish nothing and every
// chunk-phase wait gives up after that many nanoseconds.
int attention_setup(const void* q_rot, const void* k_cache, const void* v_cache, int32_t num_pages,
                    const int32_t* cu_seqlens_q, const int32_t* q_start_pos, const int32_t* context_lens,
                    const int32_t* block_tables, const int32_t* bt_offsets, int64_t bt_len, int32_t bt_stride,
                    int32_t num_rows, int32_t num_tokens, int64_t context_total, int32_t H_q, int32_t H_kv,
                    int32_t D, int32_t page_size, float scale, void* out, void* workspace, size_t ws_bytes,
                    bool clear_status, int64_t stall_limit_ns, AttnPlan* L, bool* empty) {
  *empty = true;
  if (num_rows < 0 || num_tokens < 0 || context_total < 0 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 ||
      (D != 64 && D != 128) || page_size != kPage || bt_stride < 0 || bt_len < 0 || num_pages < 0 ||
      !(scale > 0.f))
    return MS_ERR_ARG;
  const int G = H_q / H_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return MS_ERR_ARG;
  if (num_rows == 0 || num_tokens == 0) return MS_OK;  // no tokens: every row is a pad row
  *empty = false;
  if (!q_rot || !k_cache || !v_cache || !cu_seqlens_q || !q_start_pos || !context_lens || !block_tables || !out ||
      !workspace || num_pages < 1 || (bt_offsets == nullptr && bt_stride < 1) || (bt_offsets != nullptr && bt_len < 1))
    return MS_ERR_ARG;
  if (!aligned16(q_rot) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MS_ERR_ARG;
  if (num_rows > kMaxRows || num_tokens > kMaxTokens) return MS_ERR_ARG;
  const WsLayout w = ws_layout(num_rows, num_tokens, context_total, H_q, H_kv, D);
  if (ws_bytes < w.total) return MS_ERR_ARG;
  const int sms = num_sms();
  if (sms <= 0) return MS_ERR_CUDA;
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return MS_ERR_CUDA;

  CUtensorMap& tq = L->tq;
  CUtensorMap& tk = L->tk;
  CUtensorMap& tv = L->tv;
  CUtensorMap& tvp = L->tvp;
  CUtensorMap& tkp = L->tkp;
  {
    const cuuint64_t dq[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H_q),
                              static_cast<cuuint64_t>(num_tokens)};
    const cuuint64_t sq[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H_q) * D * 2};
    const cuuint32_t bq[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(128 / G)};
    const cuuint64_t dk[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_pages) * H_kv * kPage};
    const cuuint64_t sk[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t bk[2] = {64, static_cast<cuuint32_t>(kPage)};
    if (!encode_bf16(enc, &tq, q_rot, 3, dq, sq, bq) || !encode_bf16(enc, &tk, k_cache, 2, dk, sk, bk) ||
        !encode_bf16(enc, &tv, v_cache, 2, dk, sk, bk))
      return MS_ERR_ARG;
    tvp = tv;  // at D = 64 a page is one 2 KB box of tv (and of tk)
    tkp = tk;
    if (D == 128) {
      // K and V by whole pages (V for the chunk tiles, both for the decode ring):
      // (64 columns, 16 rows, 2 slabs, page x KV head), so that one box lands as
      // the page's slab 0 then its slab 1
      const cuuint64_t dv[4] = {64, static_cast<cuuint64_t>(kPage), 2,
                                static_cast<cuuint64_t>(num_pages) * H_kv};
      const cuuint64_t sv[3] = {static_cast<cuuint64_t>(D) * 2, 128,
                                static_cast<cuuint64_t>(kPage) * D * 2};
      const cuuint32_t bv[4] = {64, static_cast<cuuint32_t>(kPage), 2, 1};
      if (!encode_bf16(enc, &tvp, v_cache, 4, dv, sv, bv) || !encode_bf16(enc, &tkp, k_cache, 4, dv, sv, bv))
        return MS_ERR_ARG;
    }
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AttnParams& p = L->p;
  p.q_rot = static_cast<const bf16*>(q_rot);
  p.k_cache = static_cast<const bf16*>(k_cache);
  p.v_cache = static_cast<const bf16*>(v_cache);
  p.cu = cu_seqlens_q;
  p.q_start = q_start_pos;
  p.ctx_lens = context_lens;
  p.bt = block_tables;
  p.bt_off = bt_offsets;
  p.bt_len = bt_offsets != nullptr ? bt_len : static_cast<int64_t>(num_rows) * bt_stride;
  p.out = static_cast<bf16*>(out);
  p.hdr = reinterpret_cast<int32_t*>(ws + w.hdr);
  p.dec_rows = reinterpret_cast<int32_t*>(ws + w.dec_rows);
  p.dec_part_base = reinterpret_cast<int32_t*>(ws + w.dec_part_base);
  p.dec_nsplit = reinterpret_cast<int32_t*>(ws + w.dec_nsplit);
  p.ch_rows = reinterpret_cast<int32_t*>(ws + w.ch_rows);
  p.dec_items = reinterpret_cast<int2*>(ws + w.dec_items);
  p.dec_cnt = reinterpret_cast<int32_t*>(ws + w.dec_cnt);
  p.ch_items = reinterpret_cast<int2*>(ws + w.ch_items);
  p.max_dec_items = w.max_dec_items;
  p.max_ch_items = w.max_ch_items;
  p.part_ml = reinterpret_cast<float*>(ws + w.part_ml);
  p.part_acc = reinterpret_cast<float*>(ws + w.part_acc);
  p.max_partials = w.max_partials;
  p.context_total = context_total;
  p.bt_stride = bt_stride;
  p.num_rows = num_rows;
  p.num_tokens = num_tokens;
  p.num_pages = num_pages;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.D = D;
  p.G = G;
  p.dec_workers = sms * dec_warps(D, G);
  p.num_sms = sms;
  p.clear_status = clear_status ? 1 : 0;
  p.test_stall = stall_limit_ns > 0 ? 1 : 0;
  p.wait_limit_ns = stall_limit_ns > 0 ? static_cast<uint64_t>(stall_limit_ns) : 2000000000ull;
  p.scale_log2 = scale * 1.4426950408889634f;

  p.force_chunk_ctas = -1;
  if (device_rates(&p.sm_mhz, &p.hbm_gbs, &p.l2_bytes) != MS_OK) return MS_ERR_CUDA;
  return MS_OK;
}

// The prologue as its own kernel, a programmatic dependent of the kernel
// before it: about a thread per row (one warp up to 32 rows, else at least a
// warp per scheduler).
int launch_prologue(const AttnParams& p, cudaStream_t st) {
  if (ensure_smem_limit(prologue_kernel, 8, prologue_words(kMaxRows) * 4) != MS_OK) return MS_ERR_CUDA;
  const int S = p.num_rows;
  const int threads = S <= 32 ? 32 : S >= 1024 ? 1024 : S <= 128 ? 128 : (S + 31) / 32 * 32;
  return launch_dependent(prologue_kernel, dim3(1), dim3(threads), prologue_words(S) * 4, st, p) == cudaSuccess
             ? MS_OK
             : MS_ERR_CUDA;
}

// The persistent attention kernel for the call's head dim and group size.
int launch_attention(const AttnPlan& L, cudaStream_t st) {
  const AttnParams& p = L.p;
  const CUtensorMap &tq = L.tq, &tk = L.tk, &tv = L.tv, &tvp = L.tvp, &tkp = L.tkp;
  const int n_ctas = p.num_sms;  // one persistent CTA per SM
  int rc = MS_ERR_ARG;
  switch (p.D * 100 + p.G) {
    case 6401: rc = launch_paths<64, 1>(p, tq, tk, tv, tvp, tkp, n_ctas, st); break;
    case 6402: rc = launch_paths<64, 2>(p, tq, tk, tv, tvp, tkp, n_ctas, st); break;
    case 6404: rc = launch_paths<64, 4>(p, tq, tk, tv, tvp, tkp, n_ctas, st); break;
    case 6408: rc = launch_paths<64, 8>(p, tq, tk, tv, tvp, tkp, n_ctas, st); break;
    case 12801: rc = launch_paths<128, 1>(p, tq, tk, tv, tvp, tkp, n_ctas, st); break;
    case 12802: rc = launch_paths<128, 2>(p, tq, tk, tv, tvp, tkp, n_ctas, st); break;
    case 12804: rc = launch_paths<128, 4>(p, tq, tk, tv, tvp, tkp, n_ctas, st); break;
    case 12808: rc = launch_paths<128, 8>(p, tq, tk, tv, tvp, tkp, n_ctas, st); break;
    default: break;
  }
  return rc;
}

// The attention call behind the attention entry points: prologue, then the
// persistent kernel.  Every argument check comes before the first enqueue, so
// a call that returns an error has put nothing on the stream.  *launched tells
// whether kernels were enqueued (a step with no tokens enqueues none).
int attention_call(const void* q_rot, const void* k_cache, const void* v_cache, int32_t num_pages,
                   const int32_t* cu_seqlens_q, const int32_t* q_start_pos, const int32_t* context_lens,
                   const int32_t* block_tables, const int32_t* bt_offsets, int64_t bt_len, int32_t bt_stride,
                   int32_t num_rows, int32_t num_tokens,
                   int64_t context_total, int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size, float scale,
                   void* out, void* workspace, size_t ws_bytes, ms_stream_t stream, bool clear_status,
                   int64_t stall_limit_ns, bool* launched, int32_t force_chunk_ctas = -1) {
  *launched = false;
  AttnPlan L;
  bool empty = true;
  const int rc = attention_setup(q_rot, k_cache, v_cache, num_pages, cu_seqlens_q, q_start_pos, context_lens,
                                 block_tables, bt_offsets, bt_len, bt_stride, num_rows, num_tokens, context_total, H_q,
                                 H_kv, D, page_size, scale, out, workspace, ws_bytes, clear_status, stall_limit_ns, &L,
                                 &empty);
  if (rc != MS_OK || empty) return rc;
  L.p.force_chunk_ctas = force_chunk_ctas;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  *launched = true;  // from here on, kernels may be on the stream
  const int rp = launch_prologue(L.p, st);
  return rp != MS_OK ? rp : launch_attention(L, st);
}

// Steps of at most this many rows run the prologue inside the append's launch
// (its shared memory, prologue_words(rows), then sits on every append CTA:
// 20 KB at this bound, under an eighth of the SM's for 8 resident CTAs).
constexpr int kFuseRows = 1024;

}  // namespace

extern "C" MS_API int ms_mixed_step_attention(const void* q_rot, const void* k_cache, const void* v_cache,
                                              int32_t num_pages, const int32_t* cu_seqlens_q,
                                              const int32_t* q_start_pos, const int32_t* context_lens,
                                              const int32_t* block_tables, int32_t bt_stride, int32_t num_rows,
                                              int32_t num_tokens, int64_t context_total, int32_t H_q, int32_t H_kv,
                                              int32_t D, int32_t page_size, float scale, void* out, void* workspace,
                                              size_t ws_bytes, ms_stream_t stream) {
  bool launched = false;
  return attention_call(q_rot, k_cache, v_cache, num_pages, cu_seqlens_q, q_start_pos, context_lens, block_tables,
                        nullptr, 0, bt_stride, num_rows, num_tokens, context_total, H_q, H_kv, D, page_size, scale, out,
                        workspace, ws_bytes, stream, false, 0, &launched);
}

extern "C" MS_API int ms_mixed_step_attention_ragged(const void* q_rot, const void* k_cache, const void* v_cache,
                                                     int32_t num_pages, const int32_t* cu_seqlens_q,
                                                     const int32_t* q_start_pos, const int32_t* context_lens,
                                                     const int32_t* bt_offsets, const int32_t* bt_pages,
                                                     int64_t num_bt_pages, int32_t num_rows, int32_t num_tokens,
                                                     int64_t context_total, int32_t H_q, int32_t H_kv, int32_t D,
                                                     int32_t page_size, float scale, void* out, void* workspace,
                                                     size_t ws_bytes, ms_stream_t stream) {
  if (bt_offsets == nullptr && num_rows > 0 && num_tokens > 0) return MS_ERR_ARG;
  bool launched = false;
  return attention_call(q_rot, k_cache, v_cache, num_pages, cu_seqlens_q, q_start_pos, context_lens, bt_pages,
                        bt_offsets, num_bt_pages, 0, num_rows, num_tokens, context_total, H_q, H_kv, D, page_size,
                        scale, out, workspace, ws_bytes, stream, false, 0, &launched);
}

extern "C" MS_API int ms_mixed_step(const void* q, const void* k, const void* v, const int32_t* positions,
                                   const int32_t* slot_mapping, const float* cos_tab, const float* sin_tab,
                                   int32_t max_pos, void* k_cache, void* v_cache, int32_t num_pages, void* q_rot,
                                   const int32_t* cu_seqlens_q, const int32_t* q_start_pos,
                                   const int32_t* context_lens, const int32_t* block_tables,
                                   const int32_t* bt_offsets, int64_t bt_len, int32_t bt_stride, int32_t num_rows,
                                   int32_t num_tokens, int64_t context_total, int32_t H_q, int32_t H_kv, int32_t D,
                                   int32_t page_size, float scale, void* out, void* workspace, size_t ws_bytes,
                                   int32_t* dev_status, ms_stream_t stream) {
  AppendArgs a;
  int64_t units = 0;
  int rc = append_setup(q, k, v, positions, slot_mapping, num_tokens, cos_tab, sin_tab, max_pos, k_cache, v_cache,
                        num_pages, q_rot, H_q, H_kv, D, page_size, dev_status, &a, &units);
  if (rc != MS_OK) return rc;
  AttnPlan L;
  bool empty = true;
  rc = attention_setup(q_rot, k_cache, v_cache, num_pages, cu_seqlens_q, q_start_pos, context_lens, block_tables,
                       bt_offsets, bt_offsets != nullptr ? bt_len : 0, bt_offsets != nullptr ? 0 : bt_stride, num_rows,
                       num_tokens, context_total, H_q, H_kv, D, page_size, scale, out, workspace, ws_bytes, false, 0,
                       &L, &empty);
  if (rc != MS_OK) return rc;
  if (units == 0) return MS_OK;  // no tokens: nothing to append or attend
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (empty || num_rows > kFuseRows) {
    rc = ms_kv_append_rope(q, k, v, positions, slot_mapping, num_tokens, cos_tab, sin_tab, max_pos, k_cache, v_cache,
                           num_pages, q_rot, H_q, H_kv, D, page_size, dev_status, stream);
    if (rc != MS_OK || empty) return rc;
    rc = launch_prologue(L.p, st);
    return rc != MS_OK ? rc : launch_attention(L, st);
  }
  // CTA 0 runs the prologue beside the append's CTAs; plain stream order, so the
  // step before has finished with the workspace
  const int64_t blocks = 1 + append_blocks(units, L.p.num_sms);
  const int smem = prologue_words(num_rows) * 4;
  if (units + blocks * kAppendThreads < (int64_t{1} << 31)) {
    if (ensure_smem_limit(append_prologue_kernel<uint32_t>, 9, prologue_words(kFuseRows) * 4) != MS_OK)
      return MS_ERR_CUDA;
    append_prologue_kernel<uint32_t><<<static_cast<unsigned>(blocks), kAppendThreads, smem, st>>>(a, L.p);
  } else {
    if (ensure_smem_limit(append_prologue_kernel<int64_t>, 10, prologue_words(kFuseRows) * 4) != MS_OK)
      return MS_ERR_CUDA;
    append_prologue_kernel<int64_t><<<static_cast<unsigned>(blocks), kAppendThreads, smem, st>>>(a, L.p);
  }
  if (cudaGetLastError() != cudaSuccess) return MS_ERR_CUDA;
  return launch_attention(L, st);
}

extern "C" MS_API int ms_test_attention_stall(const void* q_rot, const void* k_cache, const void* v_cache,
                                              int32_t num_pages, const int32_t* cu_seqlens_q,
                                              const int32_t* q_start_pos, const int32_t* context_lens,
                                              const int32_t* block_tables, int32_t bt_stride, int32_t num_rows,
                                              int32_t num_tokens, int64_t context_total, int32_t H_q, int32_t H_kv,
                                              int32_t D, int32_t page_size, float scale, void* out, void* workspace,
                                              size_t ws_bytes, int64_t wait_limit_ns, ms_stream_t stream) {
  if (wait_limit_ns < 100000 || wait_limit_ns > 2000000000ll) return MS_ERR_ARG;  // 0.1 ms .. 2 s
  bool launched = false;
  return attention_call(q_rot, k_cache, v_cache, num_pages, cu_seqlens_q, q_start_pos, context_lens, block_tables,
                        nullptr, 0, bt_stride, num_rows, num_tokens, context_total, H_q, H_kv, D, page_size, scale, out,
                        workspace, ws_bytes, stream, false, wait_limit_ns, &launched);
}

extern "C" MS_API int ms_test_attention_split(const void* q_rot, const void* k_cache, const void* v_cache,
                                              int32_t num_pages, const int32_t* cu_seqlens_q,
                                              const int32_t* q_start_pos, const int32_t* context_lens,
                                              const int32_t* block_tables, const int32_t* bt_offsets, int64_t bt_len,
                                              int32_t bt_stride, int32_t num_rows, int32_t num_tokens,
                                              int64_t context_total, int32_t H_q, int32_t H_kv, int32_t D,
                                              int32_t page_size, float scale, void* out, void* workspace,
                                              size_t ws_bytes, int32_t chunk_ctas, ms_stream_t stream) {
  if (chunk_ctas < 0) return MS_ERR_ARG;
  bool launched = false;
  return attention_call(q_rot, k_cache, v_cache, num_pages, cu_seqlens_q, q_start_pos, context_lens, block_tables,
                        bt_offsets, bt_offsets != nullptr ? bt_len : 0, bt_offsets != nullptr ? 0 : bt_stride,
                        num_rows, num_tokens, context_total, H_q, H_kv, D, page_size, scale, out, workspace, ws_bytes,
                        stream, false, 0, &launched, chunk_ctas);
}

extern "C" MS_API int ms_read_status(int32_t* dev_status, ms_stream_t stream, int32_t* host_status) {
  if (dev_status == nullptr || host_status == nullptr) return MS_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MS_ERR_CUDA;
  if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), st) != cudaSuccess) return MS_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MS_ERR_CUDA;
  *host_status = v;
  return v == 0 ? MS_OK : MS_ERR_DEVICE;
}

// ----------------------------------------------------------------------------
// attention without a caller workspace
// ----------------------------------------------------------------------------
//
// Some callers cannot hand the library a workspace: a serving process that
// reserves nearly all device memory for its KV-cache pool at start-up and
// leaves nothing for a second allocator, or host code that must not call
// cudaMalloc on its per-step path (a device allocation may synchronise the
// device and stall every other stream).  For them the step can run out of a
// fixed scratch array that the library owns.  The array lives in device
// memory from the moment this library's device code is loaded on a GPU until
// the process exits, on every GPU that loads it.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device

static __device__ __align__(256) uint8_t g_step_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_step_scratch on the current device, looked up once per
// device (host code must not pass the symbol itself to a kernel: on the host
// it names a stand-in, not device memory).
int scratch_address(void** out) {
  const int dev = current_device();
  if (dev < 0) return MS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_step_scratch) != cudaSuccess || p == nullptr) return MS_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MS_OK;
}

}  // namespace

extern "C" MS_API int ms_mixed_step_attention_noalloc(const void* q_rot, const void* k_cache, const void* v_cache,
                                                      int32_t num_pages, const int32_t* cu_seqlens_q,
                                                      const int32_t* q_start_pos, const int32_t* context_lens,
                                                      const int32_t* block_tables, int32_t bt_stride,
                                                      int32_t num_rows, int32_t num_tokens, int64_t context_total,
                                                      int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size,
                                                      float scale, void* out, int32_t* dev_status,
                                                      ms_stream_t stream) {
  if (num_rows < 0 || num_tokens < 0 || context_total < 0 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 ||
      (D != 64 && D != 128))
    return MS_ERR_ARG;
  const size_t need = ws_layout(num_rows, num_tokens, context_total, H_q, H_kv, D).total;
  if (need > kNoAllocScratchBytes) return MS_ERR_SCRATCH;
  void* scratch = nullptr;
  const int rc0 = scratch_address(&scratch);
  if (rc0 != MS_OK) return rc0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents.  The prologue zeroes its
  // status word before this call can set a bit (it also resets the queue
  // counters); no separate clearing launch sits between the append and the
  // prologue, so the prologue still overlaps the append.
  bool launched = false;
  const int rc = attention_call(q_rot, k_cache, v_cache, num_pages, cu_seqlens_q, q_start_pos, context_lens,
                                block_tables, nullptr, 0, bt_stride, num_rows, num_tokens, context_total, H_q, H_kv, D,
                                page_size, scale, out, scratch, kNoAllocScratchBytes, stream, true, 0, &launched);
  if (rc != MS_OK) return rc;
  if (dev_status != nullptr) {
    const cudaError_t e = launched ? cudaMemcpyAsync(dev_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, st)
                                   : cudaMemsetAsync(dev_status, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return MS_ERR_CUDA;
  }
  return MS_OK;
}
