// mm_align_noalloc: the grouping step of mm_align for callers that must not
// allocate device memory — for example a serving engine whose memory pool has
// already claimed the whole device, or code running where a cudaMalloc (and
// the device-wide synchronisation that growing mm_align's internal workspace
// implies) is not allowed. Inputs and outputs are still the caller's.
//
// Above 1024 tokens (or 8192 assignments) mm_align keeps per-block expert
// counts in scratch memory. Here that scratch is a fixed file-scope device
// array instead of the library's lazily grown workspace. Every GPU that loads
// this library holds the array (128 KB) until the process exits.
#include <mutex>

#include "mm.h"
#include "mm_internal.h"

namespace {

using mm::kMaxDevices;

// Per-block counts of the multi-block align path: ceil(T/256) * E ints.
__device__ __align__(256) int32_t g_align_noalloc_scratch[MM_ALIGN_NOALLOC_MAX_SCRATCH_INTS];

std::mutex g_setup_mu;
int32_t* g_scratch_dev[kMaxDevices] = {};  // device address of the array, per device

// In host code the array's name is only a host-side stand-in, so its device
// address is looked up once per device, with that device current.
int scratch_for_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_align_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MM_ERR_CUDA;
    }
    g_scratch_dev[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_dev[dev];
  return MM_OK;
}

}  // namespace

extern "C" int mm_align_noalloc(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                                int32_t* sorted_token_ids, int32_t* expert_offsets,
                                int32_t* expert_counts, void* stream) {
  if (T < 0 || top_k <= 0 || E <= 0 || block_m <= 0) return MM_ERR_INVALID_ARG;
  if (E > mm::kMaxExperts || top_k > mm::kMaxTopK || block_m > 256) return MM_ERR_UNSUPPORTED;
  if ((long long)T * top_k + (long long)E * block_m >= (1LL << 31)) return MM_ERR_UNSUPPORTED;
  if (mm::align_scratch_ints(T, E, top_k) > MM_ALIGN_NOALLOC_MAX_SCRATCH_INTS)
    return MM_ERR_UNSUPPORTED;
  if ((T > 0 && !topk_ids) || !sorted_token_ids || !expert_offsets) return MM_ERR_INVALID_ARG;
  int32_t* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc != MM_OK) return rc;
  unsigned* status = nullptr;
  if ((rc = mm::current_status_word(&status)) != MM_OK) return rc;
  // The count kernel writes every scratch entry the place kernel reads, so
  // the previous call's contents never need clearing.
  const cudaError_t e = mm::launch_align(topk_ids, T, top_k, E, block_m,
                                         mm_align_capacity(T, top_k, E, block_m),
                                         sorted_token_ids, expert_offsets, expert_counts,
                                         scratch, status, false,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}
