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
// and scatter in a single launch (for T <= 64 with per-expert 64-bit token
// masks instead of ballots: align_tiny, which the router also runs).
// Otherwise: two launches over blocks of 256 tokens (per-block counts; then
// each block derives its own slot bases from all blocks' counts and
// scatters). When the tensor-core router has already counted each of its
// token tiles, the place step runs alone, from those counts, and in the MoE
// layer it also copies the token rows into segment order
// (align_place_rows_kernel). No block ever waits on another.
#include <algorithm>

#include "align_block.cuh"

namespace mm {
namespace {

using namespace alignblk;

__global__ void __launch_bounds__(1024) align_single_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, int bm, long long capacity,
    int32_t* __restrict__ sorted, int32_t* __restrict__ offsets, int32_t* __restrict__ counts,
    unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_wait();
  pdl_trigger();
  if (T <= kTinyMaxTokens)
    align_tiny(ids, T, k, E, bm, capacity, sorted, offsets, counts, err, smem);
  else
    align_one_block(ids, T, k, E, bm, capacity, sorted, offsets, counts, err, smem);
}

__global__ void __launch_bounds__(kAlignBlockTokens) align_count_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, int32_t* __restrict__ block_counts,
    unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int W = kAlignBlockTokens / 32;
  const AlignSmem S = carve(smem, W, E);
  const int tok0 = blockIdx.x * kAlignBlockTokens;
  pdl_wait();
  pdl_trigger();
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

// Per block: each expert's slot base for this block's tokens (the expert's
// padded offset plus the counts of all earlier blocks, summed here with
// independent loads), then the stable scatter. Block 0 also writes the
// offsets, the counts and the padding sentinels.
// count_rows rows of per-expert counts, each over rows_per_block-th of a
// block's tokens (1 for this file's count kernel; several for the
// tensor-core router's smaller token tiles).
__global__ void __launch_bounds__(kAlignBlockTokens) align_place_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, int bm, long long capacity,
    int count_rows, int rows_per_block, const int32_t* __restrict__ block_counts,
    int32_t* __restrict__ sorted, int32_t* __restrict__ offsets, int32_t* __restrict__ counts) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int W = kAlignBlockTokens / 32;
  const AlignSmem S = carve(smem, W, E);
  int* base_s = reinterpret_cast<int*>(smem + align_smem_bytes(W, E, k));  // [E]
  const int tok0 = blockIdx.x * kAlignBlockTokens;
  pdl_wait();
  pdl_trigger();
  stage_ids(ids, T, k, tok0, S.ids);
  // Per expert, the counts of the rows before this block's first row and of
  // all rows: G = blockDim / E threads per expert each sum every G-th row
  // (partials parked in the ballot / prefix arrays, which are free until the
  // scatter), then one thread per expert adds the G partials.
  const int first_row = (int)blockIdx.x * rows_per_block;  // this block's first count row
  const int G = max(1, min((int)blockDim.x / E, W));  // the arrays hold W x E ints
  int* part_before = S.pre;                               // [G][E]
  int* part_total = reinterpret_cast<int*>(S.bal);        // [G][E]
  for (int i = threadIdx.x; i < G * E; i += blockDim.x) {
    const int e = i % E, g = i / E;
    int before = 0, total = 0;
#pragma unroll 8
    for (int b = g; b < count_rows; b += G) {
      const int c = __ldg(block_counts + (size_t)b * E + e);
      before += b < first_row ? c : 0;
      total += c;
    }
    part_before[g * E + e] = before;
    part_total[g * E + e] = total;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int before = 0, total = 0;
    for (int g = 0; g < G; ++g) {
      before += part_before[g * E + e];
      total += part_total[g * E + e];
    }
    S.tot[e] = total;
    base_s[e] = before;
  }
  __syncthreads();
  if (threadIdx.x < 32) warp_scan_padded(S.tot, E, bm, S.off);
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      offsets[e] = S.off[e];
      if (e < E && counts != nullptr) counts[e] = S.tot[e];
    }
    fill_padding(S.off, S.tot, E, capacity, T * k, sorted);
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) base_s[e] += S.off[e];
  // Bad ids were already flagged by the count kernel.
  block_ballots(S.ids, T, k, E, tok0, S.bal, nullptr);
  __syncthreads();
  warp_prefix(S.bal, W, E, S.pre, S.tot);
  __syncthreads();
  block_scatter(S.ids, T, k, E, tok0, S.bal, S.pre, base_s, sorted);
}

// Counts of every expert before count row `first_row` and over all rows, from
// rows of E ints: G = blockDim / (E/4) threads per column of 4 experts each
// sum every G-th row with 16-byte loads, all of a thread's rows in flight
// (partials parked in part_before / part_total, [G][E]); then one thread per
// expert adds the G partials into before_s and tot_s. E % 4 == 0.
__device__ __forceinline__ void count_prefix4(const int32_t* __restrict__ rows, int count_rows,
                                              int E, int first_row, int gmax, int* part_before,
                                              int* part_total, int* before_s, int* tot_s) {
  const int E4 = E / 4;
  const int G = max(1, min((int)blockDim.x / E4, gmax));
  const int4* r4 = reinterpret_cast<const int4*>(rows);
  for (int i = threadIdx.x; i < G * E4; i += blockDim.x) {
    const int c = i % E4, g = i / E4;
    int4 before = make_int4(0, 0, 0, 0), total = make_int4(0, 0, 0, 0);
#pragma unroll 16
    for (int b = g; b < count_rows; b += G) {
      const int4 v = __ldg(r4 + (size_t)b * E4 + c);
      total.x += v.x;
      total.y += v.y;
      total.z += v.z;
      total.w += v.w;
      if (b < first_row) {
        before.x += v.x;
        before.y += v.y;
        before.z += v.z;
        before.w += v.w;
      }
    }
    *reinterpret_cast<int4*>(part_before + g * E + 4 * c) = before;
    *reinterpret_cast<int4*>(part_total + g * E + 4 * c) = total;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int before = 0, total = 0;
    for (int g = 0; g < G; ++g) {
      before += part_before[g * E + e];
      total += part_total[g * E + e];
    }
    tot_s[e] = total;
    before_s[e] = before;
  }
}

// The grouping and the token-row copy in one launch, from the per-tile
// expert counts of the tensor-core router (count row c covers tokens
// [c*R, (c+1)*R)). One CTA per count row: it derives its tile's slot bases
// from all count rows, ranks its tokens by warp ballots, writes their slots
// of sorted, then copies each token's row of hidden to the token's k slots
// of xs (one read, k writes) and turns the padding rows of the experts
// blockIdx.x, blockIdx.x + gridDim.x, ... into zeros. CTA 0 also writes the
// offsets, the counts and the sentinels. Same output as align_place_kernel
// followed by gather_rows_kernel. E % 4 == 0, R <= 32 * warps.
constexpr int kPlaceRowsThreads = 512;

struct PlaceRowsSmem {
  uint32_t* bal;  // [W*E]
  int* pre;       // [W*E]
  int* tot;       // [E]   all tokens' counts
  int* btot;      // [E]   this CTA's counts
  int* off;       // [E+1]
  int* base;      // [E]
  int* ids;       // [R*k]
  int* pos;       // [R*k]
};

__host__ __device__ constexpr size_t place_rows_smem_bytes(int W, int E, int R, int k) {
  return (size_t)(2 * W * E + 4 * E + 1 + 2 * R * k) * 4;
}

__global__ void __launch_bounds__(kPlaceRowsThreads) align_place_rows_kernel(
    const int32_t* __restrict__ ids, int T, int k, int E, int bm, long long capacity, int R,
    int count_rows, const int32_t* __restrict__ tile_counts, const uint4* __restrict__ hidden,
    int row16, int32_t* __restrict__ sorted, int32_t* __restrict__ offsets,
    int32_t* __restrict__ counts, uint4* __restrict__ xs) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int W = kPlaceRowsThreads / 32;
  PlaceRowsSmem S;
  S.bal = reinterpret_cast<uint32_t*>(smem);
  S.pre = reinterpret_cast<int*>(S.bal + W * E);
  S.tot = S.pre + W * E;
  S.btot = S.tot + E;
  S.off = S.btot + E;
  S.base = S.off + E + 1;
  S.ids = S.base + E;
  S.pos = S.ids + R * k;
  const int tok0 = blockIdx.x * R;
  const int tend = min(T, tok0 + R);  // this CTA's tokens end here
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  stage_ids(ids, tend, k, tok0, S.ids);
  count_prefix4(tile_counts, count_rows, E, blockIdx.x, W, S.pre,
                reinterpret_cast<int*>(S.bal), S.base, S.tot);
  __syncthreads();
  if (threadIdx.x < 32) warp_scan_padded(S.tot, E, bm, S.off);
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      offsets[e] = S.off[e];
      if (e < E && counts != nullptr) counts[e] = S.tot[e];
    }
    fill_padding(S.off, S.tot, E, capacity, T * k, sorted);
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) S.base[e] += S.off[e];
  // Bad ids were already flagged by the router.
  block_ballots(S.ids, tend, k, E, tok0, S.bal, nullptr);
  __syncthreads();
  warp_prefix(S.bal, W, E, S.pre, S.btot);
  __syncthreads();
  block_scatter(S.ids, tend, k, E, tok0, S.bal, S.pre, S.base, sorted, S.pos);
  __syncthreads();
  // Token rows: warp w copies tokens w, w + W, ...; 8 x 16 bytes per lane in
  // flight, each chunk stored to every slot of the token.
  constexpr int kU = 8;
  for (int tl = warp; tl < tend - tok0; tl += W) {
    const uint4* src = hidden + (size_t)(tok0 + tl) * row16;
    const int* pt = S.pos + tl * k;
    for (int c0 = 0; c0 < row16; c0 += 32 * kU) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = c0 + u * 32 + lane;
        if (i < row16) v[u] = __ldg(src + i);
      }
      for (int j = 0; j < k; ++j) {
        const int p = pt[j];
        if (p < 0) continue;
        uint4* dst = xs + (size_t)p * row16;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int i = c0 + u * 32 + lane;
          if (i < row16) dst[i] = v[u];
        }
      }
    }
  }
  // Padding rows of this CTA's experts (at most bm - 1 each).
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int r1 = S.off[e + 1];
    for (int r = S.off[e] + S.tot[e] + warp; r < r1; r += W) {
      uint4* dst = xs + (size_t)r * row16;
      for (int i = lane; i < row16; i += 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// The grouping of a dense MLP: one expert holding every token in order
// (sorted[r] = r, padding T up to a multiple of bm), routing weight 1, and
// the fp32 output accumulator zeroed.
__global__ void __launch_bounds__(256) identity_grouping_kernel(int T, int bm, long long capacity,
                                                                int32_t* __restrict__ sorted,
                                                                int32_t* __restrict__ offsets,
                                                                float* __restrict__ weights,
                                                                float4* __restrict__ zero_buf,
                                                                long long zero4) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  pdl_trigger();
  for (long long r = i0; r < capacity; r += stride) sorted[r] = r < T ? (int32_t)r : T;
  for (long long r = i0; r < T; r += stride) weights[r] = 1.0f;
  for (long long r = i0; r < zero4; r += stride) zero_buf[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (i0 == 0) {
    offsets[0] = 0;
    offsets[1] = (T + bm - 1) / bm * bm;
  }
}

}  // namespace

cudaError_t launch_identity_grouping(int T, int block_m, long long capacity, int32_t* sorted,
                                     int32_t* offsets, float* weights, float* zero_buf,
                                     long long zero_count, int num_sms, cudaStream_t st) {
  long long work = capacity > zero_count / 4 ? capacity : zero_count / 4;
  long long blocks = (work + 255) / 256;
  if (blocks > (long long)num_sms * 4) blocks = (long long)num_sms * 4;
  if (blocks < 1) blocks = 1;
  return launch_k(identity_grouping_kernel, dim3((int)blocks), dim3(256), 0, st, false, T,
                  block_m, capacity, sorted, offsets, weights,
                  reinterpret_cast<float4*>(zero_buf), zero_count / 4);
}

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
                         int32_t* scratch, unsigned* err, bool after_prev, cudaStream_t st) {
  {
    static DeviceFlags single_done, count_done, place_done;
    const int single = (int)align_smem_bytes(32, kMaxExperts, 8);  // 32 warps, E=256, 8192 ids
    const int multi = (int)align_smem_bytes(kAlignBlockTokens / 32, kMaxExperts, kMaxTopK);
    cudaError_t e;
    if ((e = smem_attr_once(single_done, align_single_kernel, single)) != cudaSuccess ||
        (e = smem_attr_once(count_done, align_count_kernel, multi)) != cudaSuccess ||
        (e = smem_attr_once(place_done, align_place_kernel, multi + kMaxExperts * 4)) !=
            cudaSuccess)
      return e;
  }
  if (align_single_block(T, top_k)) {
    // T <= 64: the bitmask grouping, with 8 warps; else one warp per 32 tokens.
    const int nwarps = T <= kTinyMaxTokens ? 8 : (T + 31) / 32;
    const size_t smem = T <= kTinyMaxTokens
                            ? std::max(align_tiny_smem_bytes(E, T * top_k),
                                       align_smem_bytes(nwarps, E, top_k))
                            : align_smem_bytes(nwarps, E, top_k);
    return launch_k(align_single_kernel, dim3(1), dim3(nwarps * 32), smem, st, after_prev,
                    topk_ids, T, top_k, E, block_m, capacity, sorted, offsets, counts, err);
  }
  const int nblocks = (T + kAlignBlockTokens - 1) / kAlignBlockTokens;
  const size_t smem = align_smem_bytes(kAlignBlockTokens / 32, E, top_k);
  cudaError_t e = launch_k(align_count_kernel, dim3(nblocks), dim3(kAlignBlockTokens), smem, st,
                           after_prev, topk_ids, T, top_k, E, scratch, err);
  if (e != cudaSuccess) return e;
  return launch_k(align_place_kernel, dim3(nblocks), dim3(kAlignBlockTokens),
                  smem + (size_t)E * 4, st, true, topk_ids, T, top_k, E, block_m, capacity,
                  nblocks, 1, static_cast<const int32_t*>(scratch), sorted, offsets, counts);
}

cudaError_t launch_align_from_counts(const int32_t* topk_ids, int T, int top_k, int E,
                                     int block_m, long long capacity,
                                     const int32_t* tile_counts, int tile_tokens, int32_t* sorted,
                                     int32_t* offsets, int32_t* counts, bool after_prev,
                                     cudaStream_t st) {
  {
    static DeviceFlags attr_done;
    const int multi = (int)align_smem_bytes(kAlignBlockTokens / 32, kMaxExperts, kMaxTopK);
    const cudaError_t e = smem_attr_once(attr_done, align_place_kernel, multi + kMaxExperts * 4);
    if (e != cudaSuccess) return e;
  }
  const int nblocks = (T + kAlignBlockTokens - 1) / kAlignBlockTokens;
  const int rows = (T + tile_tokens - 1) / tile_tokens;
  const size_t smem = align_smem_bytes(kAlignBlockTokens / 32, E, top_k) + (size_t)E * 4;
  return launch_k(align_place_kernel, dim3(nblocks), dim3(kAlignBlockTokens), smem, st,
                  after_prev, topk_ids, T, top_k, E, block_m, capacity, rows,
                  kAlignBlockTokens / tile_tokens, tile_counts, sorted, offsets, counts);
}

cudaError_t launch_align_place_rows(const int32_t* topk_ids, int T, int top_k, int E,
                                    int block_m, long long capacity, const int32_t* tile_counts,
                                    int tile_tokens, const uint16_t* hidden, int H, int32_t* sorted,
                                    int32_t* offsets, int32_t* counts, uint16_t* xs,
                                    bool after_prev, cudaStream_t st) {
  if (E % 4 != 0 || tile_tokens > kPlaceRowsThreads || H % 8 != 0) return cudaErrorInvalidValue;
  constexpr int W = kPlaceRowsThreads / 32;
  {
    static DeviceFlags attr_done;
    const size_t most = place_rows_smem_bytes(W, kMaxExperts, 128, kMaxTopK);
    const cudaError_t e = smem_attr_once(attr_done, align_place_rows_kernel, (int)most);
    if (e != cudaSuccess) return e;
  }
  if (tile_tokens > 128) return cudaErrorInvalidValue;
  const int rows = (T + tile_tokens - 1) / tile_tokens;
  return launch_k(align_place_rows_kernel, dim3(rows), dim3(kPlaceRowsThreads),
                  place_rows_smem_bytes(W, E, tile_tokens, top_k), st, after_prev, topk_ids, T,
                  top_k, E, block_m, capacity, tile_tokens, rows, tile_counts,
                  reinterpret_cast<const uint4*>(hidden), H / 8, sorted, offsets, counts,
                  reinterpret_cast<uint4*>(xs));
}

}  // namespace mm
