// Block-level routines of the token grouping (stable counting sort of the
// flat assignment ids by expert), shared by the align kernels and by the
// router kernel, which runs them itself when one cluster covers the batch.
#pragma once

#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace alignblk {

constexpr uint32_t kFull = 0xffffffffu;

// ids_s[i] = ids of the block's tokens, row-major (ntok x k), one coalesced copy.
__device__ __forceinline__ void stage_ids(const int32_t* __restrict__ ids, int T, int k, int tok0,
                                          int* ids_s) {
  const int ntok = min((int)(blockDim.x), T - tok0);
  const int n = ntok > 0 ? ntok * k : 0;
  const int32_t* src = ids + (size_t)tok0 * k;
  for (int i = threadIdx.x; i < n; i += blockDim.x) ids_s[i] = src[i];
}

// Ballots of the block's tokens: bal_s[w*E + e] = lanes of warp w whose token
// picked expert e.
__device__ __forceinline__ void block_ballots(const int* ids_s, int T, int k, int E, int tok0,
                                              uint32_t* bal_s, unsigned* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tl = warp * 32 + lane, t = tok0 + tl;
  if (tok0 + warp * 32 >= T) {  // no token in this warp (warp-uniform): empty ballots
    for (int e = lane; e < E; e += 32) bal_s[warp * E + e] = 0u;
    return;
  }
  uint32_t bits[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) bits[q] = 0;
  bool bad = false;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int id = ids_s[tl * k + j];
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
  if (bad && err != nullptr) atomicOr(err, kDevErrBadIds);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q * 32 < E) {  // warp-uniform
      uint32_t keep = 0;
#pragma unroll 8
      for (int bit = 0; bit < 32; ++bit) {
        const uint32_t bal = __ballot_sync(kFull, (bits[q] >> bit) & 1u);
        if (lane == bit) keep = bal;
      }
      if (q * 32 + lane < E) bal_s[warp * E + q * 32 + lane] = keep;
    }
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
// block's tokens at base[e] + pre_s + rank-in-warp. With pos_s, also records
// that slot at pos_s[tl*k + j] (-1 for a dropped id).
__device__ __forceinline__ void block_scatter(const int* ids_s, int T, int k, int E, int tok0,
                                              const uint32_t* bal_s, const int* pre_s,
                                              const int* base, int32_t* __restrict__ sorted,
                                              int* pos_s = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tl = warp * 32 + lane, t = tok0 + tl;
  if (t >= T) return;
  const uint32_t lt = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    const int id = ids_s[tl * k + j];
    bool drop = id < 0 || id >= E;
    for (int jj = 0; jj < j && !drop; ++jj) drop = ids_s[tl * k + jj] == id;
    if (drop) {
      if (pos_s != nullptr) pos_s[tl * k + j] = -1;
      continue;
    }
    const int pos = base[id] + pre_s[warp * E + id] + __popc(bal_s[warp * E + id] & lt);
    sorted[pos] = t * k + j;
    if (pos_s != nullptr) pos_s[tl * k + j] = pos;
  }
}

__device__ __forceinline__ void fill_padding(const int* off, const int* tot, int E,
                                             long long capacity, int sentinel,
                                             int32_t* __restrict__ sorted) {
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    for (int p = off[e] + tot[e]; p < off[e + 1]; ++p) sorted[p] = sentinel;
  for (long long p = off[E] + threadIdx.x; p < capacity; p += blockDim.x) sorted[p] = sentinel;
}

// Shared layout of the block kernels of W warps: bal_s [W*E] u32, pre_s [W*E]
// i32, tot_s [E] i32, off_s [E+1] i32, ids_s [W*32*k] i32.
__host__ __device__ constexpr size_t align_smem_bytes(int W, int E, int k) {
  return (size_t)(2 * W * E + E + E + 1 + W * 32 * k) * 4;
}

struct AlignSmem {
  uint32_t* bal;
  int* pre;
  int* tot;
  int* off;
  int* ids;
};

__device__ __forceinline__ AlignSmem carve(unsigned char* smem, int W, int E) {
  AlignSmem a;
  a.bal = reinterpret_cast<uint32_t*>(smem);
  a.pre = reinterpret_cast<int*>(a.bal + W * E);
  a.tot = a.pre + W * E;
  a.off = a.tot + E;
  a.ids = a.off + E + 1;
  return a;
}

// The whole grouping by one block of W = blockDim.x / 32 warps, for
// T <= 32 * W tokens whose ids are in global memory: histogram, padded scan,
// stable scatter and padding.
__device__ __forceinline__ void align_one_block(const int32_t* __restrict__ ids, int T, int k,
                                                int E, int bm, long long capacity,
                                                int32_t* __restrict__ sorted,
                                                int32_t* __restrict__ offsets,
                                                int32_t* __restrict__ counts, unsigned* err,
                                                unsigned char* smem) {
  const int nwarps = blockDim.x >> 5;
  const AlignSmem S = carve(smem, nwarps, E);
  stage_ids(ids, T, k, 0, S.ids);
  __syncthreads();
  block_ballots(S.ids, T, k, E, 0, S.bal, err);
  __syncthreads();
  warp_prefix(S.bal, nwarps, E, S.pre, S.tot);
  __syncthreads();
  if (threadIdx.x < 32) warp_scan_padded(S.tot, E, bm, S.off);
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    offsets[e] = S.off[e];
    if (e < E && counts != nullptr) counts[e] = S.tot[e];
  }
  block_scatter(S.ids, T, k, E, 0, S.bal, S.pre, S.off, sorted);
  fill_padding(S.off, S.tot, E, capacity, T * k, sorted);
}

// The whole grouping for T <= 64 tokens (ids in global memory), by one block
// of at least 32 threads, with the same output, the same drop rules (ids out
// of range and repeats within a token, the later repeat, are dropped and
// flagged) and the same stable order as align_one_block. A token set fits
// in one 64-bit word: per expert, bit t is set when token t selected it (one
// shared-memory atomicOr per id), so a count is a popcount and the rank of
// token t among the expert's tokens is the popcount of the bits below t. No
// per-warp ballot loops: it runs in a few barrier-separated steps.
constexpr int kTinyMaxTokens = 64;

__host__ __device__ constexpr size_t align_tiny_smem_bytes(int E, int n_ids) {
  return (size_t)E * 8 + (size_t)(E + 1) * 4 + (size_t)E * 4 + (size_t)n_ids * 4 + 32 * 4;
}

__device__ __forceinline__ void align_tiny(const int32_t* __restrict__ ids, int T, int k, int E,
                                           int bm, long long capacity,
                                           int32_t* __restrict__ sorted,
                                           int32_t* __restrict__ offsets,
                                           int32_t* __restrict__ counts, unsigned* err,
                                           unsigned char* smem) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long* mask = reinterpret_cast<unsigned long long*>(smem);  // [E]
  int* off = reinterpret_cast<int*>(mask + E);                            // [E + 1]
  int* cnt = off + E + 1;                                                 // [E]
  int* ids_s = cnt + E;                                                   // [T * k]
  int* wsum = ids_s + T * k;                                              // [32]
  const int n = T * k;
  for (int e = tid; e < E; e += nt) mask[e] = 0ull;
  for (int i = tid; i < n; i += nt) ids_s[i] = ids[i];
  __syncthreads();
  bool bad = false;
  for (int i = tid; i < n; i += nt) {
    const int t = i / k, id = ids_s[i];
    bool drop = id < 0 || id >= E;
    for (int jj = t * k; jj < i && !drop; ++jj) drop = ids_s[jj] == id;  // an earlier repeat
    bad |= drop;
    if (!drop) atomicOr(&mask[id], 1ull << t);
  }
  if (bad && err != nullptr) atomicOr(err, kDevErrBadIds);
  __syncthreads();
  // Exclusive scan of the block-padded counts over the experts (E <= 32 *
  // warps * per-thread loop), one pass per group of nt experts.
  int carry = 0;
  for (int e0 = 0; e0 < E; e0 += nt) {
    const int e = e0 + tid;
    const int c = e < E ? __popcll(mask[e]) : 0;
    const int v = (c + bm - 1) / bm * bm;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int nw = (nt + 31) / 32;
      int w = lane < nw ? wsum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFull, w, o);
        if (lane >= o) w += u;
      }
      if (lane < nw) wsum[lane] = w;  // inclusive totals of the warps
    }
    __syncthreads();
    const int before = carry + (warp > 0 ? wsum[warp - 1] : 0) + incl - v;
    if (e < E) {
      off[e] = before;
      cnt[e] = c;
    }
    carry += wsum[(nt + 31) / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) off[E] = carry;
  __syncthreads();
  for (int e = tid; e <= E; e += nt) {
    offsets[e] = off[e];
    if (e < E && counts != nullptr) counts[e] = cnt[e];
  }
  for (int i = tid; i < n; i += nt) {
    const int t = i / k, id = ids_s[i];
    if (id < 0 || id >= E) continue;
    const unsigned long long m = mask[id];
    if (!((m >> t) & 1ull)) continue;
    bool rep = false;
    for (int jj = t * k; jj < i && !rep; ++jj) rep = ids_s[jj] == id;
    if (rep) continue;
    sorted[off[id] + __popcll(m & ((1ull << t) - 1ull))] = i;
  }
  fill_padding(off, cnt, E, capacity, n, sorted);
}

}  // namespace alignblk
}  // namespace mm
