// Router for batches of more than 4096 tokens, on the sm_103a tensor cores:
// logits = hidden x router_w^T (bf16 in, fp32 accumulated in tensor memory),
// then softmax over all experts and top-k ("mini-sglang guide, chapter 7",
// paragraph on layers/moe.py; "模型与权重加载", ModelConfig: norm_topk_prob).
//
// One tile = 128 tokens x all experts (E <= 128: the MMA's M side is the
// router rows, zero past E; N = the tile's tokens). Persistent CTAs walk the
// tiles; per 64-wide K step, TMA brings 128 router rows and 128 token rows,
// and one MMA thread accumulates into one of two tensor-memory buffers, so
// the epilogue of one tile overlaps the main loop of the next.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = tensor-memory
// allocator + MMA issuer, warps 2-9 = epilogue. The epilogue copies the
// tile's logits from tensor memory (lane = expert, column = token) into a
// shared [token][expert] tile, then each warp finishes four tokens at a
// time (their reduction chains interleave) with the same softmax / top-k
// routine as the cluster router. Every wait is a bounded mbarrier wait (no
// named barriers), so a timeout unwinds all roles.
//
// The launch also zeroes the fp32 output accumulator of the layer: every CTA
// of the grid (one per SM, including those without a tile) clears one slice.
#include <math.h>

#include "mm_device.cuh"
#include "mm_internal.h"
#include "route_finish.cuh"

namespace mm {
namespace {

constexpr int kRcTok = 128;  // tokens per tile (MMA N)
constexpr int kRcK = 64;     // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kRcStages = 4;
constexpr int kRcEpiWarp0 = 2, kRcEpiWarps = 8, kRcEpiThreads = kRcEpiWarps * 32;
constexpr int kRcThreads = (kRcEpiWarp0 + kRcEpiWarps) * 32;  // 320
constexpr int kRcABytes = 128 * kRcK * 2;                       // router rows
constexpr int kRcBBytes = kRcTok * kRcK * 2;                    // token rows
constexpr int kRcStageBytes = kRcABytes + kRcBBytes;
// Logit tile [token][expert] fp32, rows of kRcLd floats: kRcLd = 2 (mod 32)
// makes the finishing reads (thread pair (n, h) reads experts 2j + h of
// token n) hit 32 distinct banks.
constexpr int kRcLd = 130;
constexpr int kRcLogitBytes = kRcTok * kRcLd * 4;
constexpr int kRcSmemBytes = kRcStages * kRcStageBytes + kRcLogitBytes + 1024;
constexpr uint32_t kRcTmemCols = 2 * kRcTok;  // two accumulator buffers
static_assert(kRcSmemBytes <= 227 * 1024 - 4096, "shared memory");

__device__ __forceinline__ bool rc_aborted(const int* flag) {
  return *reinterpret_cast<const volatile int*>(flag) != 0;
}

__device__ __forceinline__ void rc_abort(int* flag, unsigned* err) {
  *reinterpret_cast<volatile int*>(flag) = 1;
  atomicOr(err, kDevErrTimeout);
}

// Zeroes float4 slice [blockIdx.x * per, +per) of zero_buf with `workers`
// threads numbered `w`.
__device__ __forceinline__ void zero_slice(float* zero_buf, long long zero_count, int w,
                                           int workers) {
  if (zero_buf == nullptr) return;
  const long long n4 = zero_count >> 2;
  const long long per = (n4 + gridDim.x - 1) / gridDim.x;
  const long long lo = (long long)blockIdx.x * per;
  const long long hi = lo + per < n4 ? lo + per : n4;
  float4* z = reinterpret_cast<float4*>(zero_buf);
  for (long long i = lo + w; i < hi; i += workers) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Two threads finish token t: thread h of the pair takes experts 2j + h
// (j < 64) of its logit row (bias included), held in registers. Softmax over
// all E experts, top_k rounds of arg-max (the larger logit wins, equal logits
// go to the lower expert id: each round is a tournament over adjacent pairs,
// the left, lower id keeping ties, then one exchange with the partner), ids
// written in ascending order, weights p or p / sum(p) over the selected. A
// logit is compared as an order-preserving uint32 key (-0 folded into +0;
// -inf maps to 0x007fffff), so key 0 can mark "taken or no expert". All 32
// lanes of the warp call this (t < 0: no token).
__device__ __forceinline__ void finish_pair(const float* __restrict__ row, int E, int top_k,
                                            int renorm, int t, int32_t* __restrict__ ids_out,
                                            float* __restrict__ w_out) {
  constexpr uint32_t kAll = 0xffffffffu;
  const int h = threadIdx.x & 1;
  const int nj = t >= 0 ? (E - h + 1) / 2 : 0;  // experts 2j + h < E
  float v[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) v[j] = j < nj ? row[2 * j + h] : -INFINITY;
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < 64; ++j) m = fmaxf(m, v[j]);
  m = fmaxf(m, __shfl_xor_sync(kAll, m, 1));
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 64; ++j)
    if (j < nj) s += expf(v[j] - m);
  s += __shfl_xor_sync(kAll, s, 1);
  uint32_t key[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const uint32_t b = __float_as_uint(v[j] + 0.0f);
    key[j] = j < nj ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
  }
  uint32_t sel0 = 0, sel1 = 0;  // own experts j < 32, j >= 32
  for (int r = 0; r < top_k; ++r) {
    uint32_t a[32];
    int ai[32];
#pragma unroll
    for (int p = 0; p < 32; ++p) {
      const uint32_t sb = p < 16 ? sel0 : sel1;
      const int j0 = 2 * p, j1 = 2 * p + 1;
      const uint32_t x0 = ((sb >> (j0 & 31)) & 1u) ? 0u : key[j0];
      const uint32_t x1 = ((sb >> (j1 & 31)) & 1u) ? 0u : key[j1];
      const bool right = x1 > x0;  // ties keep the lower id
      a[p] = right ? x1 : x0;
      ai[p] = right ? j1 : j0;
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
      for (int p = 0; p < w; ++p) {
        const bool right = a[2 * p + 1] > a[2 * p];
        a[p] = right ? a[2 * p + 1] : a[2 * p];
        ai[p] = right ? ai[2 * p + 1] : ai[2 * p];
      }
    const uint32_t best = a[0];  // 0: no untaken expert in this half
    const int bj = best != 0u ? ai[0] : -1;
    const uint32_t ob = __shfl_xor_sync(kAll, best, 1);
    const int oj = __shfl_xor_sync(kAll, bj, 1);
    // Equal logits: the lower id 2j + h wins.
    const bool win =
        bj >= 0 && (oj < 0 || best > ob || (best == ob && 2 * bj + h < 2 * oj + 1 - h));
    if (win) {
      if (bj < 32)
        sel0 |= 1u << bj;
      else
        sel1 |= 1u << (bj - 32);
    }
  }
  const uint32_t o0 = __shfl_xor_sync(kAll, sel0, 1), o1 = __shfl_xor_sync(kAll, sel1, 1);
  float psel = 0.f;
  for (int w = 0; w < 2; ++w)
    for (uint32_t b = w == 0 ? sel0 : sel1; b != 0; b &= b - 1)
      psel += expf(row[2 * (32 * w + __ffs(b) - 1) + h] - m) / s;
  if (renorm) psel += __shfl_xor_sync(kAll, psel, 1);
  if (t < 0) return;
  // Slot of own expert j: own selected below j, plus the partner's selected
  // experts with a lower id (partner j' < j + h).
  auto below = [](uint32_t lo, uint32_t hi, int j) {  // set bits of (hi:lo) under bit j
    if (j >= 64) return __popc(lo) + __popc(hi);
    if (j >= 32) return __popc(lo) + __popc(hi & ((1u << (j - 32)) - 1u));
    return __popc(lo & ((1u << j) - 1u));
  };
  for (int w = 0; w < 2; ++w)
    for (uint32_t b = w == 0 ? sel0 : sel1; b != 0; b &= b - 1) {
      const int j = 32 * w + __ffs(b) - 1;
      const int slot = below(sel0, sel1, j) + below(o0, o1, j + h);
      const float p = expf(row[2 * j + h] - m) / s;
      ids_out[(size_t)t * top_k + slot] = 2 * j + h;
      w_out[(size_t)t * top_k + slot] = renorm ? p / psel : p;
    }
}

// EP = experts rounded up to a power of two in [32, 128].
template <int EP>
__global__ void __launch_bounds__(kRcThreads, 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmR,
                    const __grid_constant__ CUtensorMap tmH, const float* __restrict__ bias,
                    int T, int H, int E, int top_k, int renorm, int32_t* __restrict__ ids_out,
                    float* __restrict__ w_out, float* __restrict__ zero_buf, long long zero_count,
                    unsigned* err) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kRcStages + 7];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tiles = (T + kRcTok - 1) / kRcTok;
  pdl_trigger();  // the next kernel of the layer may be scheduled (it waits for this one)
  if ((int)blockIdx.x >= tiles) {  // no tile: this CTA only clears its slice
    zero_slice(zero_buf, zero_count, tid, kRcThreads);
    return;
  }

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t smem_base = (raw_addr + 1023u) & ~1023u;
  float* logits = reinterpret_cast<float*>(smem_raw + (smem_base - raw_addr) +
                                           kRcStages * kRcStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + kRcStages;
  uint64_t* tfull = empty + kRcStages;  // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint64_t* lfull = tempty + 2;         // logit tile written
  uint64_t* lfree = lfull + 1;          // logit tile read
  uint64_t* done = lfree + 1;

  if (tid == 0) {
    for (int s = 0; s < kRcStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), kRcEpiThreads);
    }
    mbar_init(smem_u32(lfull), kRcEpiThreads);
    mbar_init(smem_u32(lfree), kRcEpiThreads);
    mbar_init(smem_u32(done), 1);
    abort_s = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmR);
    tma_prefetch_desc(&tmH);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), kRcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;
  const int nk = H / kRcK;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer ---
    if (lane == 0) {
      const uint64_t pol_r = l2_policy_evict_last();   // every tile reads the router rows
      const uint64_t pol_h = l2_policy_evict_first();  // each token row is read once
      int s = 0;
      uint32_t ph = 0;
      for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        if (rc_aborted(&abort_s)) break;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u)) {
            rc_abort(&abort_s, err);
            ok = false;
            break;
          }
          const uint32_t st = smem_base + s * kRcStageBytes;
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, kRcStageBytes);
          tma_load_2d(st, &tmR, fb, kb * kRcK, 0, pol_r);
          tma_load_2d(st + kRcABytes, &tmH, fb, kb * kRcK, tile * kRcTok, pol_h);
          if (++s == kRcStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer ---
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, kRcTok);
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
        if (rc_aborted(&abort_s)) break;
        const int b = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait(smem_u32(&tempty[b]), (use & 1u) ^ 1u)) {
          rc_abort(&abort_s, err);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(b * kRcTok);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(smem_u32(&full[s]), ph)) {
            rc_abort(&abort_s, err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_base + s * kRcStageBytes;
#pragma unroll
          for (int kk = 0; kk < kRcK / 16; ++kk)
            umma_bf16(d, sdesc_kmajor<128>(st + kk * 32),
                      sdesc_kmajor<128>(st + kRcABytes + kk * 32), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&empty[s]));  // frees the stage once these MMAs are done
          if (++s == kRcStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[b]));  // the tile's logits are complete
      }
      umma_commit(smem_u32(done));  // every MMA issued above has finished before teardown
      if (!mbar_wait(smem_u32(done), 0)) rc_abort(&abort_s, err);
    }
  } else {
    // -------------------------------------------------- epilogue (2-9) ---
    const int ew = warp - kRcEpiWarp0;  // 0..7
    const int q = warp & 3;             // tensor-memory lane quarter this warp may read
    const int side = ew >> 2;           // takes 32-token chunks side, side + 2
    zero_slice(zero_buf, zero_count, tid - kRcEpiWarp0 * 32, kRcEpiThreads);
    int it = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
      if (rc_aborted(&abort_s)) break;
      const int b = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      const int t0 = tile * kRcTok;
      const int ntok = min(kRcTok, T - t0);
      if (!mbar_wait(smem_u32(&tfull[b]), use & 1u)) {
        rc_abort(&abort_s, err);
        break;
      }
      // The previous tile's logits have been read by every epilogue thread.
      if (it > 0 && !mbar_wait(smem_u32(lfree), static_cast<uint32_t>((it - 1) & 1))) {
        rc_abort(&abort_s, err);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(b * kRcTok);
      const int el = q * 32 + lane;  // this lane's expert
      const float bl = (bias != nullptr && el < E) ? __ldg(bias + el) : 0.f;
#pragma unroll
      for (int i = 0; i < kRcTok / 64; ++i) {
        const int c0 = (2 * i + side) * 32;
        if (c0 >= ntok) break;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tb + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) logits[(c0 + j) * kRcLd + q * 32 + lane] = __uint_as_float(v[j]) + bl;
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[b]));  // tensor memory buffer b may be overwritten
      mbar_arrive(smem_u32(lfull));
      if (!mbar_wait(smem_u32(lfull), static_cast<uint32_t>(it & 1))) {
        rc_abort(&abort_s, err);
        break;
      }
      // Two threads per token: epilogue thread 2n + h finishes token n.
      {
        const int et = tid - kRcEpiWarp0 * 32, n = et >> 1;
        finish_pair(logits + n * kRcLd, E, top_k, renorm, n < ntok ? t0 + n : -1, ids_out, w_out);
      }
      mbar_arrive(smem_u32(lfree));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kRcTmemCols);
  }
}

template <int EP>
cudaError_t launch_ep(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int T,
                      int H, int E, int top_k, int renorm, int32_t* ids, float* w,
                      float* zero_buf, long long zero_count, int num_sms, unsigned* err,
                      cudaStream_t st) {
  static bool attr_done[kMaxDevices] = {};
  const int dev = current_device();
  if (!attr_done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        route_tc_kernel<EP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRcSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  CUtensorMap tmR, tmH;
  if (!make_tensor_map_2d(&tmR, router_w, (uint64_t)E, (uint64_t)H, 128, kRcK) ||
      !make_tensor_map_2d(&tmH, hidden, (uint64_t)T, (uint64_t)H, kRcTok, kRcK))
    return cudaErrorInvalidValue;
  const int tiles = (T + kRcTok - 1) / kRcTok;
  const int grid = zero_buf != nullptr ? (tiles > num_sms ? tiles : num_sms)
                                       : (tiles < num_sms ? tiles : num_sms);
  return launch_k(route_tc_kernel<EP>, dim3(grid), dim3(kRcThreads), kRcSmemBytes, st, false, tmR,
                  tmH, bias, T, H, E, top_k, renorm, ids, w, zero_buf, zero_count, err);
}

}  // namespace

// Up to 4096 tokens the cluster router is as fast (its 64-token tiles spread
// the softmax / top-k over more SMs); beyond, this router's single pass over
// the router rows per 128 tokens wins (T = 16384: 27 us against 70 us).
bool route_uses_tensor_cores(int T, int E) { return T > 4096 && E <= 128; }

cudaError_t launch_route_tc(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                            int T, int H, int E, int top_k, int renorm, int32_t* topk_ids,
                            float* topk_w, float* zero_buf, long long zero_count, int num_sms,
                            unsigned* err, cudaStream_t st) {
  if (E <= 32)
    return launch_ep<32>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                         zero_buf, zero_count, num_sms, err, st);
  if (E <= 64)
    return launch_ep<64>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                         zero_buf, zero_count, num_sms, err, st);
  return launch_ep<128>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                        zero_buf, zero_count, num_sms, err, st);
}

}  // namespace mm
