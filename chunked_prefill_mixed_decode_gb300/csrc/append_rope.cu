// The append entry point: rotary embedding at absolute positions + paged K/V
// append as one kernel (the per-thread work is in append_rope.cuh).
#include <cuda_runtime.h>

#include <cstdint>

#include "append_rope.cuh"
#include "mixed_step.h"

namespace {

template <typename Idx>
__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(AppendArgs a) {
  // the attention call that follows may start its launch now; it waits for
  // this kernel before it reads q_rot or the pages
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  append_rope_units<Idx>(a, static_cast<Idx>(blockIdx.x) * kAppendThreads + threadIdx.x,
                         static_cast<Idx>(gridDim.x) * kAppendThreads);
}

}  // namespace

extern "C" MS_API int ms_kv_append_rope(const void* q, const void* k, const void* v, const int32_t* positions,
                                        const int32_t* slot_mapping, int32_t T, const float* cos_tab,
                                        const float* sin_tab, int32_t max_pos, void* k_cache, void* v_cache,
                                        int32_t num_pages, void* q_rot, int32_t H_q, int32_t H_kv, int32_t D,
                                        int32_t page_size, int32_t* dev_status, ms_stream_t stream) {
  AppendArgs a;
  int64_t units = 0;
  const int rc = append_setup(q, k, v, positions, slot_mapping, T, cos_tab, sin_tab, max_pos, k_cache, v_cache,
                              num_pages, q_rot, H_q, H_kv, D, page_size, dev_status, &a, &units);
  if (rc != MS_OK || units == 0) return rc;
  const int64_t blocks = append_blocks(units, 152);
  if (units + blocks * kAppendThreads < (int64_t{1} << 31))
    append_rope_kernel<uint32_t>
        <<<static_cast<unsigned>(blocks), kAppendThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  else
    append_rope_kernel<int64_t>
        <<<static_cast<unsigned>(blocks), kAppendThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? MS_OK : MS_ERR_CUDA;
}
