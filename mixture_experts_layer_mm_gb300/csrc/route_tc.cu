// Router on the sm_103a tensor cores, for batches of more than 2048 tokens
// and at most 128 experts: logits = hidden x router_w^T (bf16 in, fp32
// accumulated in tensor memory), then softmax over all experts and top-k
// ("mini-sglang guide, chapter 7", paragraph on layers/moe.py;
// "模型与权重加载", ModelConfig: norm_topk_prob).
//
// One tile = TOK tokens x all experts (the MMA's M side is the 128 router
// rows, zero past E; N = the tile's tokens). TOK (32, 64 or 128) is chosen so
// that the tiles about fill the GPU: every tile streams the whole router
// matrix, so a finer split costs L2 reads, not DRAM. Persistent CTAs walk
// the tiles; per 64-wide K step, TMA brings the router rows and the tile's
// token rows, and one MMA thread accumulates into one of two tensor-memory
// buffers, so the epilogue of one tile overlaps the main loop of the next.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = tensor-memory
// allocator + MMA issuer, warps 2-9 = epilogue. The epilogue copies the
// tile's logits (+ bias) from tensor memory (lane = expert, column = token)
// into a shared [token][expert] tile; then P = 256 / TOK threads finish each
// token together (softmax, top-k, ascending slots, renormalisation). Every
// wait is a bounded mbarrier wait (no named barriers), so a timeout unwinds
// all roles.
//
// The epilogue also counts each tile's experts (tile_counts), from which the
// grouping places the tokens in one launch. The launch can zero a buffer on
// the side: every CTA of the grid (one per SM, including those without a
// tile) clears one slice (the layer passes none: its accumulator is zeroed by
// the gate_up kernel).
#include <math.h>

#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

constexpr int kRcK = 64;  // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kRcEpiWarp0 = 2, kRcEpiWarps = 8, kRcEpiThreads = kRcEpiWarps * 32;
constexpr int kRcThreads = (kRcEpiWarp0 + kRcEpiWarps) * 32;  // 320
constexpr int kRcABytes = 128 * kRcK * 2;                       // router rows

template <int TOK>
struct RcCfg {
  static_assert(TOK == 32 || TOK == 64 || TOK == 128, "token tile");
  static constexpr int kP = kRcEpiThreads / TOK;  // threads finishing one token
  static constexpr int kNJ = 128 / kP;             // experts per finishing thread
  static constexpr int kBBytes = TOK * kRcK * 2;
  static constexpr int kStageBytes = kRcABytes + kBBytes;
  static constexpr int kStages = (128 * 1024) / kStageBytes;  // 6, 5, 4
  // Logit rows of kLd floats: kLd = kP (mod 32) makes the finishing reads
  // (thread h of token n reads experts kP*j + h) hit 32 distinct banks.
  static constexpr int kLd = 128 + kP;
  static constexpr int kLogitBytes = TOK * kLd * 4;
  static constexpr int kSmemBytes = kStages * kStageBytes + kLogitBytes + 1024;
  static constexpr uint32_t kTmemCols = 2 * TOK;  // two accumulator buffers
  static_assert(kSmemBytes <= 227 * 1024 - 4096, "shared memory");
};

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

// Order-preserving uint32 key of a logit (-0 folded into +0; -inf maps to
// 0x007fffff), so that key 0 can mark "taken or no expert".
__device__ __forceinline__ uint32_t logit_key(float v) {
  const uint32_t b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// P consecutive lanes finish token t together: lane h of the group holds the
// logits (bias included) of experts P*j + h (j < NJ) of the token's row.
// Softmax over all E experts; top_k rounds of arg-max, the larger logit
// winning and equal logits going to the lower expert id (each round: a
// tournament over adjacent pairs in registers, the left and lower id keeping
// ties, then a butterfly over the group); ids written in ascending order;
// weights p or p / sum(p) over the selected; with cnt (shared, may be NULL)
// each selected expert's count is incremented. All 32 lanes of the warp call
// this (t < 0: no token).
template <int P, int NJ>
__device__ __forceinline__ void finish_group(const float* __restrict__ row, int E, int top_k,
                                             int renorm, int t, int32_t* __restrict__ ids_out,
                                             float* __restrict__ w_out, int* cnt) {
  constexpr uint32_t kAll = 0xffffffffu;
  const int h = threadIdx.x & (P - 1);
  const int nj = t >= 0 ? (E - h + P - 1) / P : 0;  // experts P*j + h < E
  float v[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) v[j] = j < nj ? row[P * j + h] : -INFINITY;
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < NJ; ++j) m = fmaxf(m, v[j]);
#pragma unroll
  for (int o = 1; o < P; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kAll, m, o));
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (j < nj) s += expf(v[j] - m);
#pragma unroll
  for (int o = 1; o < P; o <<= 1) s += __shfl_xor_sync(kAll, s, o);
  uint32_t key[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) key[j] = j < nj ? logit_key(v[j]) : 0u;

  uint32_t own0 = 0, own1 = 0;              // own experts selected: j < 32, j >= 32
  uint32_t g0 = 0, g1 = 0, g2 = 0, g3 = 0;  // the group's selected expert ids (128 bits)
  for (int r = 0; r < top_k; ++r) {
    uint32_t a[NJ / 2];
    int ai[NJ / 2];
#pragma unroll
    for (int p = 0; p < NJ / 2; ++p) {
      const int j0 = 2 * p, j1 = 2 * p + 1;
      const uint32_t sb = j0 < 32 ? own0 : own1;
      const uint32_t x0 = ((sb >> (j0 & 31)) & 1u) ? 0u : key[j0];
      const uint32_t x1 = ((sb >> (j1 & 31)) & 1u) ? 0u : key[j1];
      const bool right = x1 > x0;  // ties keep the lower id
      a[p] = right ? x1 : x0;
      ai[p] = right ? j1 : j0;
    }
#pragma unroll
    for (int w = NJ / 4; w >= 1; w >>= 1)
#pragma unroll
      for (int p = 0; p < w; ++p) {
        const bool right = a[2 * p + 1] > a[2 * p];
        a[p] = right ? a[2 * p + 1] : a[2 * p];
        ai[p] = right ? ai[2 * p + 1] : ai[2 * p];
      }
    uint32_t bk = a[0];                      // 0: no untaken expert here
    int bid = bk != 0u ? P * ai[0] + h : 0;  // expert id of the candidate
#pragma unroll
    for (int o = 1; o < P; o <<= 1) {
      const uint32_t ok = __shfl_xor_sync(kAll, bk, o);
      const int oid = __shfl_xor_sync(kAll, bid, o);
      if (ok > bk || (ok == bk && oid < bid)) {
        bk = ok;
        bid = oid;
      }
    }
    if (bk != 0u) {  // the same winner in every lane of the group
      const uint32_t bit = 1u << (bid & 31);
      const int wd = bid >> 5;
      g0 |= wd == 0 ? bit : 0u;
      g1 |= wd == 1 ? bit : 0u;
      g2 |= wd == 2 ? bit : 0u;
      g3 |= wd == 3 ? bit : 0u;
      if ((bid & (P - 1)) == h) {
        const int j = bid / P;
        if (j < 32)
          own0 |= 1u << j;
        else
          own1 |= 1u << (j - 32);
      }
    }
  }
  float psel = 0.f;
  for (int w = 0; w < 2; ++w)
    for (uint32_t b = w == 0 ? own0 : own1; b != 0; b &= b - 1)
      psel += expf(row[P * (32 * w + __ffs(b) - 1) + h] - m) / s;
  if (renorm) {
#pragma unroll
    for (int o = 1; o < P; o <<= 1) psel += __shfl_xor_sync(kAll, psel, o);
  }
  if (t < 0) return;
  // Slot of a selected expert = selected ids below it (all lanes know them).
  for (int w = 0; w < 2; ++w)
    for (uint32_t b = w == 0 ? own0 : own1; b != 0; b &= b - 1) {
      const int j = 32 * w + __ffs(b) - 1;
      const int id = P * j + h, wd = id >> 5;
      const uint32_t lowbits = (1u << (id & 31)) - 1u;
      const int slot = (wd > 0 ? __popc(g0) : __popc(g0 & lowbits)) +
                       (wd > 1 ? __popc(g1) : wd == 1 ? __popc(g1 & lowbits) : 0) +
                       (wd > 2 ? __popc(g2) : wd == 2 ? __popc(g2 & lowbits) : 0) +
                       (wd == 3 ? __popc(g3 & lowbits) : 0);
      const float p = expf(row[id] - m) / s;
      ids_out[(size_t)t * top_k + slot] = id;
      w_out[(size_t)t * top_k + slot] = renorm ? p / psel : p;
      if (cnt != nullptr) atomicAdd(cnt + id, 1);
    }
}

template <int TOK>
__global__ void __launch_bounds__(kRcThreads, 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmR,
                    const __grid_constant__ CUtensorMap tmH, const float* __restrict__ bias,
                    int T, int H, int E, int top_k, int renorm, int32_t* __restrict__ ids_out,
                    float* __restrict__ w_out, float* __restrict__ zero_buf, long long zero_count,
                    int32_t* __restrict__ tile_counts, unsigned* err) {
  using Cfg = RcCfg<TOK>;
  constexpr int S = Cfg::kStages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * S + 7];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int cnt_s[2][128];  // per-expert counts of the tile (by tile parity)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tiles = (T + TOK - 1) / TOK;
  pdl_wait();  // hidden may come from the kernel before this one (the RMSNorm step)
  pdl_trigger();  // the next kernel of the layer may be scheduled (it waits for this one)
  if ((int)blockIdx.x >= tiles) {  // no tile: this CTA only clears its slice
    zero_slice(zero_buf, zero_count, tid, kRcThreads);
    return;
  }

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t smem_base = (raw_addr + 1023u) & ~1023u;
  float* logits =
      reinterpret_cast<float*>(smem_raw + (smem_base - raw_addr) + S * Cfg::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;   // [2]
  uint64_t* tempty = tfull + 2;  // [2]
  uint64_t* lfull = tempty + 2;  // logit tile written
  uint64_t* lfree = lfull + 1;   // logit tile read
  uint64_t* done = lfree + 1;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
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
    tmem_alloc(smem_u32(&tmem_base_s), Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (tid < 256) cnt_s[tid >> 7][tid & 127] = 0;
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
          const uint32_t st = smem_base + s * Cfg::kStageBytes;
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          tma_load_2d(st, &tmR, fb, kb * kRcK, 0, pol_r);
          tma_load_2d(st + kRcABytes, &tmH, fb, kb * kRcK, tile * TOK, pol_h);
          if (++s == S) {
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
      const uint32_t idesc = idesc_bf16_f32(128, TOK);
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
        const uint32_t d = tmem_base + static_cast<uint32_t>(b * TOK);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(smem_u32(&full[s]), ph)) {
            rc_abort(&abort_s, err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_base + s * Cfg::kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kRcK / 16; ++kk)
            umma_bf16(d, sdesc_kmajor<128>(st + kk * 32),
                      sdesc_kmajor<128>(st + kRcABytes + kk * 32), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&empty[s]));  // frees the stage once these MMAs are done
          if (++s == S) {
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
    const int et = tid - kRcEpiWarp0 * 32;       // 0..255
    const int q = warp & 3;                      // tensor-memory lane quarter this warp may read
    const int side = (warp - kRcEpiWarp0) >> 2;  // takes 32-token chunks side, side + 2
    const int el = q * 32 + lane;                // the expert of this lane's TMEM row
    const float bl = (bias != nullptr && el < E) ? __ldg(bias + el) : 0.f;
    zero_slice(zero_buf, zero_count, et, kRcEpiThreads);
    int it = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
      if (rc_aborted(&abort_s)) break;
      const int b = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      const int t0 = tile * TOK;
      const int ntok = min(TOK, T - t0);
      if (!mbar_wait(smem_u32(&tfull[b]), use & 1u)) {
        rc_abort(&abort_s, err);
        break;
      }
      // The previous tile's logits have been read by every epilogue thread,
      // and its counts are complete: write them out and clear that buffer.
      if (it > 0 && !mbar_wait(smem_u32(lfree), static_cast<uint32_t>((it - 1) & 1))) {
        rc_abort(&abort_s, err);
        break;
      }
      if (it > 0 && tile_counts != nullptr && et < E) {
        int* c = cnt_s[(it - 1) & 1];
        tile_counts[(size_t)(tile - (int)gridDim.x) * E + et] = c[et];
        c[et] = 0;
      }
      tc_fence_after();
      const uint32_t tb =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * TOK);
#pragma unroll
      for (int c0 = side * 32; c0 < TOK; c0 += 64) {
        if (c0 >= ntok) break;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tb + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) logits[(c0 + j) * Cfg::kLd + el] = __uint_as_float(v[j]) + bl;
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[b]));  // tensor memory buffer b may be overwritten
      mbar_arrive(smem_u32(lfull));
      if (!mbar_wait(smem_u32(lfull), static_cast<uint32_t>(it & 1))) {
        rc_abort(&abort_s, err);
        break;
      }
      {
        const int n = et / Cfg::kP;  // the token this thread helps finish
        finish_group<Cfg::kP, Cfg::kNJ>(logits + n * Cfg::kLd, E, top_k, renorm,
                                        n < ntok ? t0 + n : -1, ids_out, w_out,
                                        tile_counts != nullptr ? cnt_s[it & 1] : nullptr);
      }
      mbar_arrive(smem_u32(lfree));
    }
    // The last tile's counts.
    if (it > 0 && tile_counts != nullptr && !rc_aborted(&abort_s)) {
      if (mbar_wait(smem_u32(lfree), static_cast<uint32_t>((it - 1) & 1))) {
        if (et < E)
          tile_counts[(size_t)(blockIdx.x + (it - 1) * (int)gridDim.x) * E + et] =
              cnt_s[(it - 1) & 1][et];
      } else {
        rc_abort(&abort_s, err);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

template <int TOK>
cudaError_t launch_tok(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int T,
                       int H, int E, int top_k, int renorm, int32_t* ids, float* w,
                       float* zero_buf, long long zero_count, int32_t* tile_counts, int num_sms,
                       unsigned* err, bool after_prev, cudaStream_t st) {
  using Cfg = RcCfg<TOK>;
  static DeviceFlags attr_done;
  if (cudaError_t e = smem_attr_once(attr_done, route_tc_kernel<TOK>, Cfg::kSmemBytes);
      e != cudaSuccess)
    return e;
  CUtensorMap tmR, tmH;
  if (!make_tensor_map_2d(&tmR, router_w, (uint64_t)E, (uint64_t)H, 128, kRcK) ||
      !make_tensor_map_2d(&tmH, hidden, (uint64_t)T, (uint64_t)H, TOK, kRcK))
    return cudaErrorInvalidValue;
  const int tiles = (T + TOK - 1) / TOK;
  const int grid = zero_buf != nullptr ? (tiles > num_sms ? tiles : num_sms)
                                       : (tiles < num_sms ? tiles : num_sms);
  return launch_k(route_tc_kernel<TOK>, dim3(grid), dim3(kRcThreads), Cfg::kSmemBytes, st,
                  after_prev, tmR, tmH, bias, T, H, E, top_k, renorm, ids, w, zero_buf,
                  zero_count, tile_counts, err);
}

}  // namespace

// Up to 2048 tokens the cluster router is faster: it splits the router
// matrix over 8 CTAs per 64-token tile, while here one CTA streams all of it
// per tile (about 16 us, bound by one SM's load latency).
bool route_uses_tensor_cores(int T, int E) { return T > 2048 && E <= 128; }

int route_tc_tile_tokens(int T, int num_sms) {
  // The smallest token tile that leaves at most one tile per SM (a CTA's time
  // is mostly its pass over the router matrix); beyond, 128-token tiles.
  if ((T + 31) / 32 <= num_sms) return 32;
  if ((T + 63) / 64 <= num_sms) return 64;
  return 128;
}

cudaError_t launch_route_tc(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                            int T, int H, int E, int top_k, int renorm, int32_t* topk_ids,
                            float* topk_w, float* zero_buf, long long zero_count,
                            int32_t* tile_counts, int num_sms, unsigned* err, bool after_prev,
                            cudaStream_t st) {
  const int tok = route_tc_tile_tokens(T, num_sms);
  if (tok == 32)
    return launch_tok<32>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                          zero_buf, zero_count, tile_counts, num_sms, err, after_prev, st);
  if (tok == 64)
    return launch_tok<64>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                          zero_buf, zero_count, tile_counts, num_sms, err, after_prev, st);
  return launch_tok<128>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                         zero_buf, zero_count, tile_counts, num_sms, err, after_prev, st);
}

}  // namespace mm
