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
// T <= 1024: one block does histogram, scan and scatter in a single launch.
// T >  1024: three launches (per-block counts, one-block scan, scatter);
// no block ever waits on another.
#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

constexpr uint32_t kFull = 0xffffffffu;

// Ballots of the block's tokens: bal_s[w*E + e] = lanes of warp w whose token
// picked expert e.
__device__ __forceinline__ void block_ballots(const int32_t* __restrict__ ids, int T, int k, int E,
                                              int tok0, uint32_t* bal_s, unsigned* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = tok0 + warp * 32 + lane;
  uint32_t bits[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) bits[q] = 0;
  bool bad = false;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int id = ids[(size_t)t * k + j];
      if (id < 0 || id >= E) {
        bad = true;
        continue;
      }
      const uint32_t b = 1u << (id & 31);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if ((id >> 5) == q) {
          if (bits[q] & b) bad = true;
          bits[q] |= b;
        }
    }
  }
  if (bad) atomicOr(err, kDevErrBadIds);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q * 32 >= E) break;
    uint32_t keep = 0;
#pragma unroll 8
    for (int bit = 0; bit < 32; ++bit) {
      const uint32_t bal = __ballot_sync(kFull, (bits[q] >> bit) & 1u);
      if (lane == bit) keep = bal;
    }
    if (q * 32 + lane < E) bal_s[warp * E + q * 32 + lane] = keep;
  }
}

// pre_s[w*E + e] = assignments of expert e in warps before w; tot_s[e] = block total.
__device__ __forceinline__ void warp_prefix(const uint32_t* bal_s, int nwarps, int E, int* pre_s,
                                            int* tot_s) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < nwarps; ++w) {
      pre_s[w * E + e] = run;
      run += __popc(bal_s[w * E + e]);
    }
    tot_s[e] = run;
  }
}

// Warp 0: off[e] = exclusive scan over experts of tot[e] rounded up to bm;
// off[E] = padded total.
__device__ __forceinline__ void warp_scan_padded(const int* tot, int E, int bm, int* off) {
  const int lane = threadIdx.x & 31;
  const int per = (E + 31) / 32, e0 = lane * per;
  int sum = 0;
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    if (e < E) sum += (tot[e] + bm - 1) / bm * bm;
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - sum;
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    if (e < E) {
      off[e] = run;
      run += (tot[e] + bm - 1) / bm * bm;
    }
  }
  if (lane == 31) off[E] = incl;
}

// Writes f = t*k + j of every valid, first-occurrence assignment of the
// block's tokens at base[e] + pre_s + rank-in-warp.
__device__ __forceinline__ void block_scatter(const int32_t* __restrict__ ids, int T, int k, int E,
                                              int tok0, const uint32_t* bal_s, const int* pre_s,
                                              const int* base, int32_t* __restrict__ sorted) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = tok0 + warp * 32 + lane;
  if (t >= T) return;
  const uint32_t lt = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    const int id = ids[(size_t)t * k + j];
    if (id < 0 || id >= E) continue;
    bool dup = false;
    for (int jj = 0; jj < j; ++jj) dup |= ids[(size_t)t * k + jj] == id;
    if (dup) continue;
    const int pos = base[id] + pre_s[warp * E + id] + __popc(bal_s[warp * E + id] & lt);
    sorted[pos] = t * k + j;
  }
}

__device__ __forceinline__ void fill_padding(const int* off, const int* tot, int E,
                                             long long capacity, int sentinel,
                                             int32_t* __restrict__ sorted) {
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    for (int p = off[e] + tot[e]; p < off[e + 1]; ++p) sorted[p] = sentinel;
  for (long long p = off[E] + threadIdx.x; p < capacity; p += blockDim.x) sorted[p] = sentinel;
}

// Shared layout of the block kernels: bal_s [32*E] u32, pre_s [32*E] i32,
// tot_s [E] i32, off_s [E+1] i32.
__host__ __device__ constexpr size_t align_smem_bytes(int E) {
  return (size_t)(2 * 32 * E + E + E + 1) * 4;
}

__global__ void __launch_bounds__(1024) align_single_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, int bm, long long capacity,
    int32_t* __restrict__ sorted, int32_t* __restrict__ offsets, int32_t* __restrict__ counts,
    unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* bal_s = reinterpret_cast<uint32_t*>(smem);
  int* pre_s = reinterpret_cast<int*>(bal_s + 32 * E);
  int* tot_s = pre_s + 32 * E;
  int* off_s = tot_s + E;
  const int nwarps = blockDim.x >> 5;
  block_ballots(ids, T, k, E, 0, bal_s, err);
  __syncthreads();
  warp_prefix(bal_s, nwarps, E, pre_s, tot_s);
  __syncthreads();
  if (threadIdx.x < 32) warp_scan_padded(tot_s, E, bm, off_s);
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    offsets[e] = off_s[e];
    if (e < E && counts != nullptr) counts[e] = tot_s[e];
  }
  block_scatter(ids, T, k, E, 0, bal_s, pre_s, off_s, sorted);
  fill_padding(off_s, tot_s, E, capacity, T * k, sorted);
}

__global__ void __launch_bounds__(1024) align_count_kernel(const int32_t* __restrict__ ids, int T,
                                                           int k, int E,
                                                           int32_t* __restrict__ block_counts,
                                                           unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* bal_s = reinterpret_cast<uint32_t*>(smem);
  const int tok0 = blockIdx.x * kAlignBlockTokens;
  block_ballots(ids, T, k, E, tok0, bal_s, err);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < 32; ++w) c += __popc(bal_s[w * E + e]);
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

__global__ void __launch_bounds__(1024) align_scatter_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, const int32_t* __restrict__ block_base,
    int32_t* __restrict__ sorted, unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* bal_s = reinterpret_cast<uint32_t*>(smem);
  int* pre_s = reinterpret_cast<int*>(bal_s + 32 * E);
  int* tot_s = pre_s + 32 * E;
  int* base_s = tot_s + E;
  const int tok0 = blockIdx.x * kAlignBlockTokens;
  block_ballots(ids, T, k, E, tok0, bal_s, err);
  for (int e = threadIdx.x; e < E; e += blockDim.x) base_s[e] = block_base[blockIdx.x * E + e];
  __syncthreads();
  warp_prefix(bal_s, 32, E, pre_s, tot_s);
  __syncthreads();
  block_scatter(ids, T, k, E, tok0, bal_s, pre_s, base_s, sorted);
}

}  // namespace

long long align_scratch_ints(int T, int E) {
  const long long nb = (T + kAlignBlockTokens - 1) / kAlignBlockTokens;
  return nb <= 1 ? 0 : nb * E;
}

cudaError_t launch_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                         long long capacity, int32_t* sorted, int32_t* offsets, int32_t* counts,
                         int32_t* scratch, unsigned* err, cudaStream_t st) {
  const size_t smem = align_smem_bytes(E);
  static bool attr_done[kMaxDevices] = {};
  const int dev = current_device();
  if (!attr_done[dev]) {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(align_single_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)align_smem_bytes(kMaxExperts))) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(align_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)align_smem_bytes(kMaxExperts))) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(align_scatter_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)align_smem_bytes(kMaxExperts))) != cudaSuccess)
      return e;
    attr_done[dev] = true;
  }
  const int nblocks = (T + kAlignBlockTokens - 1) / kAlignBlockTokens;
  if (nblocks <= 1) {
    const int nwarps = (T + 31) / 32 < 1 ? 1 : (T + 31) / 32;
    align_single_kernel<<<1, nwarps * 32, smem, st>>>(topk_ids, T, top_k, E, block_m, capacity,
                                                      sorted, offsets, counts, err);
    return cudaGetLastError();
  }
  align_count_kernel<<<nblocks, 1024, smem, st>>>(topk_ids, T, top_k, E, scratch, err);
  align_scan_kernel<<<1, 256, 0, st>>>(nblocks, T, top_k, E, block_m, capacity, scratch, sorted,
                                       offsets, counts);
  align_scatter_kernel<<<nblocks, 1024, smem, st>>>(topk_ids, T, top_k, E, scratch, sorted, err);
  return cudaGetLastError();
}

}  // namespace mm
