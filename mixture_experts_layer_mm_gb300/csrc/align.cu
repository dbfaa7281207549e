// Token batching by expert ("mini-sglang guide, chapter 7", paragraph on
// moe/fused.py): a stable, block-padded counting sort of the flat assignment
// ids f = t*k + j by expert.
//
// A token holds each expert at most once, so within one expert increasing f
// is increasing t. Each warp takes 32 consecutive tokens (one per lane) and
// builds, per expert, the ballot of lanes whose token selected it; a lane's
// rank inside its expert is then the popcount of the lower lanes in that
// ballot, plus the counts of the earlier warps and earlier blocks. Nothing is
// ordered by atomics, so the result is deterministic.
//
// Each block first copies its tokens' ids to shared memory (one coalesced
// pass), then works from there.
// Small batches (T <= 1024 and T*k <= 8192): one block does histogram, scan
// and scatter in a single launch. Otherwise: three launches over blocks of
// 256 tokens (per-block counts, one-block scan, scatter); no block ever waits
// on another.
#include "align_block.cuh"

namespace mm {
namespace {

using namespace alignblk;

__global__ void __launch_bounds__(1024) align_single_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, int bm, long long capacity,
    int32_t* __restrict__ sorted, int32_t* __restrict__ offsets, int32_t* __restrict__ counts,
    unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem[];
  align_one_block(ids, T, k, E, bm, capacity, sorted, offsets, counts, err, smem);
}

__global__ void __launch_bounds__(kAlignBlockTokens) align_count_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, int32_t* __restrict__ block_counts,
    unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int W = kAlignBlockTokens / 32;
  const AlignSmem S = carve(smem, W, E);
  const int tok0 = blockIdx.x * kAlignBlockTokens;
  stage_ids(ids, T, k, tok0, S.ids);
  __syncthreads();
  block_ballots(S.ids, T, k, E, tok0, S.bal, err);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) c += __popc(S.bal[w * E + e]);
    block_counts[blockIdx.x * E + e] = c;
  }
}

// One block: per expert, exclusive scan of the block counts (in place, so
// block_counts becomes each block's base slot), padded offsets, padding.
__global__ void __launch_bounds__(256) align_scan_kernel(int nblocks, int T, int k, int E, int bm,
                                                         long long capacity,
                                                         int32_t* __restrict__ block_counts,
                                                         int32_t* __restrict__ sorted,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ counts) {
  __shared__ int tot_s[kMaxExperts];
  __shared__ int off_s[kMaxExperts + 1];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int b = 0; b < nblocks; ++b) {
      const int c = block_counts[b * E + e];
      block_counts[b * E + e] = run;
      run += c;
    }
    tot_s[e] = run;
  }
  __syncthreads();
  if (threadIdx.x < 32) warp_scan_padded(tot_s, E, bm, off_s);
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    offsets[e] = off_s[e];
    if (e < E && counts != nullptr) counts[e] = tot_s[e];
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    for (int b = 0; b < nblocks; ++b) block_counts[b * E + e] += off_s[e];
  fill_padding(off_s, tot_s, E, capacity, T * k, sorted);
}

__global__ void __launch_bounds__(kAlignBlockTokens) align_scatter_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, const int32_t* __restrict__ block_base,
    int32_t* __restrict__ sorted, unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int W = kAlignBlockTokens / 32;
  const AlignSmem S = carve(smem, W, E);
  const int tok0 = blockIdx.x * kAlignBlockTokens;
  stage_ids(ids, T, k, tok0, S.ids);
  for (int e = threadIdx.x; e < E; e += blockDim.x) S.off[e] = block_base[blockIdx.x * E + e];
  __syncthreads();
  // Bad ids were already flagged by the count kernel.
  block_ballots(S.ids, T, k, E, tok0, S.bal, nullptr);
  __syncthreads();
  warp_prefix(S.bal, W, E, S.pre, S.tot);
  __syncthreads();
  block_scatter(S.ids, T, k, E, tok0, S.bal, S.pre, S.off, sorted);
}

}  // namespace

namespace {
inline bool align_single_block(int T, int k) {
  return T <= kAlignSingleMaxTokens && (long long)T * k <= kAlignSingleMaxIds;
}
}  // namespace

long long align_scratch_ints(int T, int E, int k) {
  if (align_single_block(T, k)) return 0;
  return (long long)((T + kAlignBlockTokens - 1) / kAlignBlockTokens) * E;
}

cudaError_t launch_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                         long long capacity, int32_t* sorted, int32_t* offsets, int32_t* counts,
                         int32_t* scratch, unsigned* err, cudaStream_t st) {
  static bool attr_done[kMaxDevices] = {};
  const int dev = current_device();
  if (!attr_done[dev]) {
    cudaError_t e;
    const int single = (int)align_smem_bytes(32, kMaxExperts, 8);  // 32 warps, E=256, 8192 ids
    const int multi = (int)align_smem_bytes(kAlignBlockTokens / 32, kMaxExperts, kMaxTopK);
    if ((e = cudaFuncSetAttribute(align_single_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, single)) !=
        cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(align_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  multi)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(align_scatter_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, multi)) !=
        cudaSuccess)
      return e;
    attr_done[dev] = true;
  }
  if (align_single_block(T, top_k)) {
    const int nwarps = T <= 32 ? 1 : (T + 31) / 32;
    const size_t smem = align_smem_bytes(nwarps, E, top_k);
    align_single_kernel<<<1, nwarps * 32, smem, st>>>(topk_ids, T, top_k, E, block_m, capacity,
                                                      sorted, offsets, counts, err);
    return cudaGetLastError();
  }
  const int nblocks = (T + kAlignBlockTokens - 1) / kAlignBlockTokens;
  const size_t smem = align_smem_bytes(kAlignBlockTokens / 32, E, top_k);
  align_count_kernel<<<nblocks, kAlignBlockTokens, smem, st>>>(topk_ids, T, top_k, E, scratch,
                                                               err);
  align_scan_kernel<<<1, 256, 0, st>>>(nblocks, T, top_k, E, block_m, capacity, scratch, sorted,
                                       offsets, counts);
  align_scatter_kernel<<<nblocks, kAlignBlockTokens, smem, st>>>(topk_ids, T, top_k, E, scratch,
                                                                 sorted, err);
  return cudaGetLastError();
}

}  // namespace mm
