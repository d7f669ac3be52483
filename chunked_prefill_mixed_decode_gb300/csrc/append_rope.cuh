// Fused rotary embedding at absolute positions + paged K/V append: the work of
// one thread, shared by the append kernel and the fused append + prologue
// kernel of the step call.
//
// "Chunked Prefill 的 Token 预算" (zwjcode.cn), section 07: a chunk's position
// ids start at its absolute offset and never restart at 0, or the rotary phase
// repeats; section 06: every new token's K/V lands in the physical slot named
// by slot_mapping.  "Chunked Prefill: Ending the Great Stall", section 05: the
// paged blocks are filled token by token whatever chunk writes them.
//
// One thread owns 8 consecutive element pairs (i, i + D/2) of one (token, head)
// row: two 16-byte loads, two 16-byte stores, and one 32-byte read each of the
// cos and sin rows.  The work walks q heads, then k heads, then v heads of all
// tokens; it is HBM-bound: (4 H_q + 8 H_kv) D + 4 D bytes per token.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mixed_step.h"

namespace {

constexpr int kAppendThreads = 256;
constexpr int kAppendVec = 8;  // pairs per thread

struct AppendArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* positions;
  const int32_t* slot_mapping;
  const float* cos_tab;
  const float* sin_tab;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  __nv_bfloat16* q_rot;
  int32_t* status;
  int64_t n_slots;  // num_pages * page_size
  int32_t T, H_q, H_kv, D, max_pos, page;
};

__device__ __forceinline__ void rotate8(const uint4& a, const uint4& b, const float* c, const float* s, uint4& ya,
                                        uint4& yb) {
  const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
  const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
  uint32_t oa[4], ob[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float x1[2] = {__uint_as_float(wa[j] << 16), __uint_as_float(wa[j] & 0xffff0000u)};
    float x2[2] = {__uint_as_float(wb[j] << 16), __uint_as_float(wb[j] & 0xffff0000u)};
    __nv_bfloat16 r1[2], r2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float cs = c[2 * j + e], sn = s[2 * j + e];
      // two products and one sum, each rounded to nearest fp32, never fused
      const float y1 = __fsub_rn(__fmul_rn(x1[e], cs), __fmul_rn(x2[e], sn));
      const float y2 = __fadd_rn(__fmul_rn(x2[e], cs), __fmul_rn(x1[e], sn));
      r1[e] = __float2bfloat16_rn(y1);
      r2[e] = __float2bfloat16_rn(y2);
    }
    oa[j] = static_cast<uint32_t>(__bfloat16_as_ushort(r1[0])) |
            (static_cast<uint32_t>(__bfloat16_as_ushort(r1[1])) << 16);
    ob[j] = static_cast<uint32_t>(__bfloat16_as_ushort(r2[0])) |
            (static_cast<uint32_t>(__bfloat16_as_ushort(r2[1])) << 16);
  }
  ya = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  yb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

// Work units first, first + stride, ... of the step's append.  Idx: the flat
// work index type, 32-bit whenever the step's work fits (the divisions by
// per_row and heads then cost a fraction of 64-bit ones).
template <typename Idx>
__device__ __forceinline__ void append_rope_units(const AppendArgs& a, Idx first, Idx stride) {
  const int half = a.D >> 1;
  const int per_row = half / kAppendVec;  // threads per (token, head) row
  const int heads = a.H_q + 2 * a.H_kv;
  const Idx total = static_cast<Idx>(a.T) * heads * per_row;
  for (Idx g = first; g < total; g += stride) {
    const int part = static_cast<int>(g % per_row);
    const Idx rh = g / per_row;
    const int h = static_cast<int>(rh % heads);
    const int t = static_cast<int>(rh / heads);
    const int i0 = part * kAppendVec;
    const int pos = __ldg(a.positions + t);
    const int slot = __ldg(a.slot_mapping + t);

    if (h >= a.H_q) {  // K or V: the slot first; -1 is the one "no write" value
      if (slot == -1) continue;
      if (slot < 0 || static_cast<int64_t>(slot) >= a.n_slots) {
        if (a.status && part == 0) atomicOr(a.status, MS_STATUS_BAD_SLOT);
        continue;
      }
    }
    // a token at a position outside the table writes nothing: no q_rot, no K, no V
    if (pos < 0 || pos >= a.max_pos) {
      if (a.status && part == 0) atomicOr(a.status, MS_STATUS_BAD_POSITION);
      continue;
    }
    if (h >= a.H_q + a.H_kv) {  // V: plain copy into the slot
      const int hv = h - a.H_q - a.H_kv;
      const __nv_bfloat16* src = a.v + (static_cast<int64_t>(t) * a.H_kv + hv) * a.D;
      const int64_t page = slot / a.page, off = slot % a.page;
      __nv_bfloat16* dst = a.v_cache + ((page * a.H_kv + hv) * a.page + off) * a.D;
      *reinterpret_cast<uint4*>(dst + i0) = __ldg(reinterpret_cast<const uint4*>(src + i0));
      *reinterpret_cast<uint4*>(dst + i0 + half) = __ldg(reinterpret_cast<const uint4*>(src + i0 + half));
      continue;
    }
    float c[kAppendVec], s[kAppendVec];
    {
      const float4* cp = reinterpret_cast<const float4*>(a.cos_tab + static_cast<int64_t>(pos) * half + i0);
      const float4* sp = reinterpret_cast<const float4*>(a.sin_tab + static_cast<int64_t>(pos) * half + i0);
      const float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
      c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w; c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
      s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w; s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
    }
    if (h < a.H_q) {  // q -> q_rot (may alias q: this thread reads before it writes)
      const int64_t base = (static_cast<int64_t>(t) * a.H_q + h) * a.D;
      const uint4 xa = *reinterpret_cast<const uint4*>(a.q + base + i0);
      const uint4 xb = *reinterpret_cast<const uint4*>(a.q + base + i0 + half);
      uint4 ya, yb;
      rotate8(xa, xb, c, s, ya, yb);
      *reinterpret_cast<uint4*>(a.q_rot + base + i0) = ya;
      *reinterpret_cast<uint4*>(a.q_rot + base + i0 + half) = yb;
    } else {  // k -> rotated into the slot
      const int hk = h - a.H_q;
      const int64_t base = (static_cast<int64_t>(t) * a.H_kv + hk) * a.D;
      const uint4 xa = __ldg(reinterpret_cast<const uint4*>(a.k + base + i0));
      const uint4 xb = __ldg(reinterpret_cast<const uint4*>(a.k + base + i0 + half));
      uint4 ya, yb;
      rotate8(xa, xb, c, s, ya, yb);
      const int64_t page = slot / a.page, off = slot % a.page;
      __nv_bfloat16* dst = a.k_cache + ((page * a.H_kv + hk) * a.page + off) * a.D;
      *reinterpret_cast<uint4*>(dst + i0) = ya;
      *reinterpret_cast<uint4*>(dst + i0 + half) = yb;
    }
  }
}

// Host side: check the append's arguments and fill AppendArgs.  Returns
// MS_OK, or MS_ERR_ARG with nothing enqueued; *units is the step's work count
// (0 for an empty step).
inline int append_setup(const void* q, const void* k, const void* v, const int32_t* positions,
                        const int32_t* slot_mapping, int32_t T, const float* cos_tab, const float* sin_tab,
                        int32_t max_pos, void* k_cache, void* v_cache, int32_t num_pages, void* q_rot, int32_t H_q,
                        int32_t H_kv, int32_t D, int32_t page_size, int32_t* dev_status, AppendArgs* a,
                        int64_t* units) {
  *units = 0;
  if (T < 0 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || (D != 64 && D != 128) || page_size != 16 ||
      num_pages < 0 || max_pos < 1)
    return MS_ERR_ARG;
  if (T == 0) return MS_OK;
  if (!q || !k || !v || !positions || !slot_mapping || !cos_tab || !sin_tab || !k_cache || !v_cache || !q_rot)
    return MS_ERR_ARG;
  const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(q) || !al16(k) || !al16(v) || !al16(k_cache) || !al16(v_cache) || !al16(q_rot) || !al16(cos_tab) ||
      !al16(sin_tab))
    return MS_ERR_ARG;
  a->q = static_cast<const __nv_bfloat16*>(q);
  a->k = static_cast<const __nv_bfloat16*>(k);
  a->v = static_cast<const __nv_bfloat16*>(v);
  a->positions = positions;
  a->slot_mapping = slot_mapping;
  a->cos_tab = cos_tab;
  a->sin_tab = sin_tab;
  a->k_cache = static_cast<__nv_bfloat16*>(k_cache);
  a->v_cache = static_cast<__nv_bfloat16*>(v_cache);
  a->q_rot = static_cast<__nv_bfloat16*>(q_rot);
  a->status = dev_status;
  a->n_slots = static_cast<int64_t>(num_pages) * page_size;
  a->T = T;
  a->H_q = H_q;
  a->H_kv = H_kv;
  a->D = D;
  a->max_pos = max_pos;
  a->page = page_size;
  *units = static_cast<int64_t>(T) * (H_q + 2 * H_kv) * (D / 2 / kAppendVec);
  return MS_OK;
}

// CTAs of the append: one unit per thread, grid-stride beyond 16 CTAs per SM
inline int64_t append_blocks(int64_t units, int num_sms) {
  const int64_t blocks = (units + kAppendThreads - 1) / kAppendThreads;
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 152) * 16;
  return blocks < cap ? blocks : cap;
}

}  // namespace
