// Grouped expert GEMMs of the MoE layer on the sm_103a tensor cores
// (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
// This file's kernel serves batches with few token rows per expert (decode:
// rows gathered from hidden) and the standalone GEMM's gathered rows; token
// rows already in segment order with many rows per expert (prefill) go to
// the SM-pair kernel of gemm_pair.cu.
//
// Orientation: the expert WEIGHTS are the MMA's M side (128 rows per MMA)
// and the expert's TOKENS are the N side. N may be any multiple of 16 up to
// 256, so an expert segment only has to be padded to 16 rows, not to a
// 128-row tile, and the same kernel serves a decode batch (a few tokens per
// expert, streaming each selected expert's weights once) and a prefill batch.
//
// One tile = (expert e, a chunk of up to BN token rows of e's segment, an
// m-tile of weight rows). Each stage loads two 128x64 weight tiles (A0, A1)
// and one BNx64 token tile (B); two MMAs per 16-wide K step accumulate
//   gate_up mode:  D0 = gate rows [m*128, +128) , D1 = up rows (same + I)
//   down mode:     D0 = H rows [m*256, +128)    , D1 = H rows [m*256+128, +128)
// so the gate_up epilogue finds g and u of one (row, token) in the same thread.
//
// Token rows (B): the contiguous act rows of the down mode come by 2-D TMA
// boxes, and so do gate_up's rows when the layer has copied them into
// segment order first (many rows per expert). Otherwise gate_up gathers them
// from hidden through sorted_token_ids / k: with few rows per expert
// (decode-sized batches) by TMA tile::gather4, four rows per instruction;
// with many rows per expert (the standalone grouped GEMM) by four warps of
// 16-byte cp.async straight into the swizzled layout (the TMA engine would
// spend one gather per four rows of every stage).
//
// Warp roles (448 threads, one CTA per SM, persistent over a static tile
// stride): warp 1 = TMEM allocator + MMA issuer, warps 2-9 = epilogue
// (warps w and w+4 read the same 32-lane quarter of tensor memory and take
// alternate 32-column chunks of the tile), warps 10-13 and 0 = producers,
// one per ring slot: slot s is filled by warp 10 + s (slot 4 by warp 0),
// which issues the slot's weight boxes and its token rows against the
// slot's barrier. A warp's TMA loads that signal a different barrier than
// its previous ones wait for those to land, so a single producer warp would
// keep only one stage in flight; one warp per slot keeps them all in flight.
// (Token rows copied by cp.async, the standalone GEMM's path for many rows
// per expert, use warp 0 for the weights and warps 10-13 for the rows.)
// Two accumulator buffers (256 x BN tiles) let the epilogue of one tile
// overlap the main loop of the next. BN = 128 with a 4-stage ring, or 64 with
// a 5-stage ring when there are few rows per expert.
//
// Epilogues: gate_up writes act = bf16(silu(g) * u) ("模型与权重加载",
// GatedMLP: silu_and_mul of the merged gate_up projection, gate first);
// down multiplies by the routing weight and adds into the fp32 output
// accumulator ("mini-sglang guide, chapter 7": expert outputs weighted by the
// softmax scores and summed).
#include <algorithm>
#include <mutex>

#include "mm.h"
#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

constexpr int kGM = 128;  // weight rows per MMA
// 14 warps: 1 = MMA issuer, 2-9 = epilogue (two warps per tensor-memory lane
// quarter), 10-13 and 0 = producers (one per ring slot).
constexpr int kEpiWarp0 = 2, kEpiWarps = 8, kEpiThreads = kEpiWarps * 32;
constexpr int kBWarp0 = kEpiWarp0 + kEpiWarps;  // 10
constexpr int kGemmThreads = (kBWarp0 + 4) * 32;  // 448
constexpr int kEpiTok = 16;  // tokens per down-epilogue transpose step

struct GemmArgs {
  const int32_t* sorted;   // [capacity]
  const int32_t* offsets;  // [E+1]
  const float* topk_w;     // [T*k] (down mode)
  void* C;                 // act bf16 [capacity, N] | acc fp32 [T, N]
  unsigned* err;
  int E, N, K, Tk, top_k;
  int n_mtiles;  // m-tiles per token chunk
  int ksplit;    // K slices per (chunk, m-tile) (down mode only; 1 for gate_up)
  int w_rows;    // weight rows per expert in the 2-D weight view
  int m_step;    // weight rows per m-tile
  int a1_off;    // row offset of the A1 tile relative to A0
  int w_evict_first;  // weights are read by one token chunk only: stream them past L2
  int b_mode;         // how token rows reach shared memory (kB*)
  const uint16_t* hidden;  // kBLsuGather: token rows are read from here
  const uint16_t* w;       // the weights (the L2 prefetch below)
  int prefetch_guess;      // prefetch the guessed first tile's A0 rows into L2
  float* zero_buf;         // gate_up: zero these floats first (the layer's accumulator)
  long long zero_count;
};

// L2 prefetch of `bytes` (a multiple of 16) contiguous bytes from global memory.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Token-row (B) paths.
constexpr int kBTma = 0;        // 2-D TMA boxes of rows already in segment order
constexpr int kBTmaGather = 1;  // TMA tile::gather4 from hidden (few rows per expert)
constexpr int kBLsuGather = 2;  // four warps of cp.async from hidden (many rows per expert)

// One shared-memory ring of S stages; a stage holds the two weight tiles (A0,
// A1: 32 KB) and the token tile (BN rows) of one K step. The weight producer
// and the token producer fill a stage independently (each arrives on its
// full barrier), but both wait for the same stage to be freed, so loads are
// issued in the order the MMA needs them.
// KB = K per stage: 64 (rows of 128 B, 128-byte swizzle) or 32 (rows of 64 B,
// 64-byte swizzle: twice as many stages of half the size in the same shared
// memory, so more bytes stay in flight while one stage is being consumed).
template <int MODE, int BN, int S, int NACC, int KB>
struct GemmCfg {
  static_assert(KB == 64 || KB == 32, "K per stage");
  static constexpr int kRowBytes = KB * 2;              // one swizzle row
  static constexpr int kABytes = kGM * KB * 2;          // one 128-row weight tile
  static constexpr int kBBytes = BN * KB * 2;
  static constexpr int kStageBytes = 2 * kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = NACC * 2 * BN;  // NACC buffers x (D0, D1) x BN columns
  // down epilogue: one [kEpiTok tokens][32 + 1] fp32 transpose tile per warp
  static constexpr int kEpiBytes = MODE == MM_GEMM_DOWN ? kEpiWarps * kEpiTok * 33 * 4 : 0;
  static constexpr int kEpiOffset = S * kStageBytes;
  static constexpr int kSmemBytes = kEpiOffset + kEpiBytes + 1024;
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                "tensor-memory allocation must be a power of two in [32, 512]");
  static_assert(BN % 64 == 0 && BN <= 256, "BN: whole 32-column chunks for both epilogue sides");
  static_assert(S <= 5, "one producer warp per ring slot: warps 10-13, then warp 0");
  static_assert(kSmemBytes <= 227 * 1024 - 4096, "shared memory");
};

// 16-byte copy global -> shared (L2 only), zero-filled when !valid, with an
// L2 eviction-priority hint.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid,
                                                 uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst),
               "l"(src), "r"(valid ? 16 : 0), "l"(policy)
               : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// One arrival on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

template <int BN>
__device__ __forceinline__ void decode_tile(int tile, int n_mtiles, int E, const int* cs,
                                            const int* off, int& e, int& m, int& row0,
                                            int& nrows) {
  const int ch = tile / n_mtiles;
  m = tile - ch * n_mtiles;
  int lo = 0, hi = E;  // cs[lo] <= ch < cs[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cs[mid] <= ch)
      lo = mid;
    else
      hi = mid;
  }
  e = lo;
  row0 = off[e] + (ch - cs[e]) * BN;
  nrows = min(BN, off[e + 1] - row0);
}

// Tile index -> (expert, m-tile, first row, rows, K slice): tile =
// (chunk * n_mtiles + m) * ksplit + slice.
template <int BN>
__device__ __forceinline__ void decode_tile_k(int tile, const GemmArgs& a, int E, const int* cs,
                                              const int* off, int& e, int& m, int& row0,
                                              int& nrows, int& slice) {
  slice = tile % a.ksplit;
  decode_tile<BN>(tile / a.ksplit, a.n_mtiles, E, cs, off, e, m, row0, nrows);
}

__device__ __forceinline__ bool aborted(const int* flag) {
  return *reinterpret_cast<const volatile int*>(flag) != 0;
}

__device__ __forceinline__ void signal_abort(int* flag, unsigned* err) {
  *reinterpret_cast<volatile int*>(flag) = 1;
  atomicOr(err, kDevErrTimeout);
}

template <int MODE, int BN, int S, int NACC, int KB>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmX, const GemmArgs a) {
  using Cfg = GemmCfg<MODE, BN, S, NACC, KB>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * S + 5];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int off_s[kMaxExperts + 1];
  __shared__ int cs_s[kMaxExperts + 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E;
  // While the kernels before this one still run (the router at decode), start
  // the weight stream: with about one chunk per selected expert and nearly
  // all experts selected, this CTA's first tile is most likely (expert
  // blockIdx / n_mtiles, m-tile blockIdx % n_mtiles). Its A0 rows (contiguous
  // in memory) are prefetched into L2; a wrong guess only costs bandwidth.
  if (a.prefetch_guess && tid == 0) {
    const int ge = (int)blockIdx.x / a.n_mtiles, gm = (int)blockIdx.x % a.n_mtiles;
    if (ge < E) {
      const long long row = (long long)ge * a.w_rows + (long long)gm * a.m_step;
      const uint32_t bytes = (uint32_t)kGM * (uint32_t)a.K * 2u;
      const char* base = reinterpret_cast<const char*>(a.w + row * a.K);
      for (uint32_t off = 0; off < bytes; off += 65536u)
        prefetch_l2_bulk(base + off, bytes - off < 65536u ? bytes - off : 65536u);
    }
  }
  // The fp32 accumulator that the down GEMM of this call adds into is cleared
  // here by every CTA, before the wait: the previous call's last reader of it
  // (finalize) completed before this call's first kernel started, and the
  // down GEMM starts only after this kernel has completed.
  if (a.zero_buf != nullptr) {
    float4* z = reinterpret_cast<float4*>(a.zero_buf);
    const long long n4 = a.zero_count >> 2;
    for (long long i = (long long)blockIdx.x * kGemmThreads + tid; i < n4;
         i += (long long)gridDim.x * kGemmThreads)
      z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();  // the grouping and the token rows come from the kernels before
  pdl_trigger();

  // Chunk table: cs_s[e] = index of expert e's first token chunk.
  for (int i = tid; i <= E; i += kGemmThreads) off_s[i] = a.offsets[i];
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32, e0 = lane * per;
    int sum = 0;
    for (int j = 0; j < per; ++j) {
      const int e = e0 + j;
      if (e < E) sum += (off_s[e + 1] - off_s[e] + BN - 1) / BN;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int j = 0; j < per; ++j) {
      const int e = e0 + j;
      if (e < E) {
        cs_s[e] = run;
        run += (off_s[e + 1] - off_s[e] + BN - 1) / BN;
      }
    }
    if (lane == 31) cs_s[E] = incl;
  }
  __syncthreads();
  const int total_tiles = cs_s[E] * a.n_mtiles * a.ksplit;
  if ((int)blockIdx.x >= total_tiles) return;  // uniform across the CTA

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t smem_base = (raw_addr + 1023u) & ~1023u;
  float* epi_tile =
      reinterpret_cast<float*>(smem_raw + (smem_base - raw_addr) + Cfg::kEpiOffset);
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      // the weight producer + the token side (one TMA producer or 128 loaders)
      // one producer warp per slot, or the weight producer + 128 cp.async threads
      mbar_init(smem_u32(&full[s]), a.b_mode == kBLsuGather ? 1 + 128 : 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), kEpiThreads);
    }
    mbar_init(smem_u32(done), 1);
    abort_s = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;
  const int nk = a.K / KB / a.ksplit;  // K steps per tile (its slice of K)

  // Producers. A warp's TMA loads that signal a different mbarrier than its
  // previous ones wait for those to land, so one warp issuing every stage
  // has at most one stage in flight at a time. Here each ring slot has a
  // warp of its own (slot s: warp 10 + s, slot 4: warp 0), which issues the
  // slot's weight boxes and its token rows against the slot's one barrier;
  // the S slots fill concurrently. (Token rows gathered by cp.async, the
  // standalone GEMM's path for many rows per expert, keep warp 0 for the
  // weights and warps 10-13 for the rows.)
  const bool owners = a.b_mode != kBLsuGather;
  const int slot = warp == 0 ? 4 : warp - kBWarp0;  // the slot a producer warp owns
  if (owners && (warp == 0 || warp >= kBWarp0)) {
    if (slot < S) {
      const uint64_t pol_w = a.w_evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t pol_x = l2_policy_evict_last();
      const bool gather = MODE == MM_GEMM_GATE_UP && a.b_mode == kBTmaGather;
      // Gathered token rows: lane i loads rows 4i..4i+3 of the chunk with one
      // tile::gather4; the rows of the next tile are fetched a tile ahead.
      int nxt[4] = {0, 0, 0, 0};
      auto fetch_rows = [&](int tl, int (&rows)[4]) {
        int e, m, row0, nrows, slice;
        if (tl < total_tiles) decode_tile_k<BN>(tl, a, E, cs_s, off_s, e, m, row0, nrows, slice);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 4 * lane + j;
          const int f = (tl < total_tiles && r < nrows) ? __ldg(a.sorted + row0 + r) : a.Tk;
          rows[j] = f < a.Tk ? f / a.top_k : 0;  // padding rows read row 0 (never stored)
        }
      };
      if (gather) fetch_rows(blockIdx.x, nxt);
      uint32_t use = 0;  // fills of this warp's slot so far
      int q = 0;         // this CTA's K step counter, modulo S
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        if (aborted(&abort_s)) break;
        int rows[4] = {nxt[0], nxt[1], nxt[2], nxt[3]};
        if (gather) fetch_rows(tile + gridDim.x, nxt);
        int e, m, row0, nrows, slice;
        decode_tile_k<BN>(tile, a, E, cs_s, off_s, e, m, row0, nrows, slice);
        const int wrow0 = e * a.w_rows + m * a.m_step;
        const int wrow1 = wrow0 + a.a1_off;
        const int n_g4 = ((nrows + 15) & ~15) / 4;  // gathered rows the MMA reads, 4 per gather
        const uint32_t bbytes = gather ? (uint32_t)(n_g4 * 4 * Cfg::kRowBytes) : Cfg::kBBytes;
        for (int kb = slice * nk; kb < (slice + 1) * nk; ++kb) {
          const bool mine = q == slot;
          if (++q == S) q = 0;
          if (!mine) continue;
          bool w_ok = true;
          if (lane == 0) w_ok = mbar_wait(smem_u32(&empty[slot]), (use & 1u) ^ 1u);
          w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
          if (!w_ok) {
            if (lane == 0) signal_abort(&abort_s, a.err);
            ok = false;
            break;
          }
          const uint32_t st = smem_base + slot * Cfg::kStageBytes;
          const uint32_t fb = smem_u32(&full[slot]);
          if (lane == 0) {
            mbar_arrive_expect_tx(fb, 2 * Cfg::kABytes + bbytes);
            tma_load_2d(st, &tmW, fb, kb * KB, wrow0, pol_w);
            tma_load_2d(st + Cfg::kABytes, &tmW, fb, kb * KB, wrow1, pol_w);
            if (!gather) tma_load_2d(st + 2 * Cfg::kABytes, &tmX, fb, kb * KB, row0, pol_x);
          }
          if (gather) {
            __syncwarp();
            if (lane < n_g4)
              tma_gather4(st + 2 * Cfg::kABytes + lane * 4 * Cfg::kRowBytes, &tmX, fb, kb * KB,
                          rows[0], rows[1], rows[2], rows[3], pol_x);
          }
          ++use;
        }
      }
    }
  } else if (warp == 0) {
    // ----------------------- weight (A) producer of the cp.async token path ---
    if (lane == 0) {
      const uint64_t pol_w = a.w_evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
      int s = 0;
      uint32_t ph = 0;
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        if (aborted(&abort_s)) break;
        int e, m, row0, nrows, slice;
        decode_tile_k<BN>(tile, a, E, cs_s, off_s, e, m, row0, nrows, slice);
        const int wrow0 = e * a.w_rows + m * a.m_step;
        const int wrow1 = wrow0 + a.a1_off;
        bool ok = true;
        for (int kb = slice * nk; kb < (slice + 1) * nk; ++kb) {
          if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u)) {
            signal_abort(&abort_s, a.err);
            ok = false;
            break;
          }
          const uint32_t st = smem_base + s * Cfg::kStageBytes;
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, 2 * Cfg::kABytes);
          tma_load_2d(st, &tmW, fb, kb * KB, wrow0, pol_w);
          tma_load_2d(st + Cfg::kABytes, &tmW, fb, kb * KB, wrow1, pol_w);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp >= kBWarp0) {
    // ------------------------------------ token (B) rows by cp.async (4 warps) ---
    // Warps 10-13 copy the chunk's token rows from hidden with 16-byte
    // cp.async into the swizzled layout the MMA reads (16-byte chunk c of
    // row r at r*RB + ((c ^ sw(r)) * 16), RB = row bytes, sw(r) = r % 8 for
    // the 128-byte swizzle and (r / 2) % 4 for the 64-byte one). Thread
    // (w, l) moves chunk l % CPR of rows p*RPP + w*(32/CPR) + l/CPR. Each
    // thread's copies arrive on the stage's barrier by themselves when they
    // land (cp.async.mbarrier.arrive.noinc, 128 arrivals per stage); the MMA
    // thread then fences the generic-to-async proxy before reading.
    const uint64_t pol_x = l2_policy_evict_last();
    int s = 0;
    uint32_t ph = 0;
    constexpr int kCPR = KB / 8;            // 16-byte chunks per row
    constexpr int kRPP = 128 / kCPR;        // rows per pass of the 128 threads
    constexpr int kPasses = BN / kRPP;
    const int w = warp - kBWarp0, c16 = lane % kCPR;
    const uint16_t* src[kPasses];
    const uint16_t* nxt[kPasses];
    auto fetch_rows = [&](int tl, const uint16_t* (&rows)[kPasses]) {
      int e, m, row0, nrows, slice;
      if (tl < total_tiles) decode_tile_k<BN>(tl, a, E, cs_s, off_s, e, m, row0, nrows, slice);
#pragma unroll
      for (int p = 0; p < kPasses; ++p) {
        const int r = p * kRPP + w * (32 / kCPR) + lane / kCPR;
        const int f = (tl < total_tiles && r < nrows) ? __ldg(a.sorted + row0 + r) : a.Tk;
        rows[p] = f < a.Tk ? a.hidden + (size_t)(f / a.top_k) * a.K + c16 * 8 : nullptr;
      }
    };
    fetch_rows(blockIdx.x, nxt);
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
      if (aborted(&abort_s)) break;
#pragma unroll
      for (int p = 0; p < kPasses; ++p) src[p] = nxt[p];
      fetch_rows(tile + gridDim.x, nxt);
      const int slice = tile % a.ksplit;
      for (int kb = slice * nk; kb < (slice + 1) * nk; ++kb) {
        if (lane == 0) ok = mbar_wait(smem_u32(&empty[s]), ph ^ 1u);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) signal_abort(&abort_s, a.err);
          break;
        }
        const uint32_t st = smem_base + s * Cfg::kStageBytes + 2 * Cfg::kABytes;
#pragma unroll
        for (int p = 0; p < kPasses; ++p) {
          const int r = p * kRPP + w * (32 / kCPR) + lane / kCPR;
          const int sw = KB == 64 ? (r & 7) : ((r >> 1) & 3);
          const uint32_t dst = st + r * Cfg::kRowBytes + ((c16 ^ sw) << 4);
          cp_async16_zfill(dst, src[p] != nullptr ? src[p] + kb * KB : a.hidden,
                           src[p] != nullptr, pol_x);
        }
        cp_async_arrive_noinc(smem_u32(&full[s]));
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    cp_async_wait<0>();  // no copy of this thread is in flight when the CTA ends
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
        if (aborted(&abort_s)) break;
        int e, m, row0, nrows, slice;
        decode_tile_k<BN>(tile, a, E, cs_s, off_s, e, m, row0, nrows, slice);
        const int b = it % NACC;
        const uint32_t use = static_cast<uint32_t>(it / NACC);
        if (!mbar_wait(smem_u32(&tempty[b]), (use & 1u) ^ 1u)) {
          signal_abort(&abort_s, a.err);
          break;
        }
        tc_fence_after();
        const int n_mma = (nrows + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(kGM, n_mma);
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(b * 2 * BN);
        const uint32_t d1 = d0 + BN;
        bool ok = true;
        for (int kb = slice * nk; kb < (slice + 1) * nk; ++kb) {
          if (!mbar_wait(smem_u32(&full[s]), ph)) {
            signal_abort(&abort_s, a.err);
            ok = false;
            break;
          }
          // Rows written by cp.async (generic proxy) are read by the MMA (async proxy).
          if (MODE == MM_GEMM_GATE_UP && a.b_mode == kBLsuGather) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t st = smem_base + s * Cfg::kStageBytes;
#pragma unroll
          for (int kk = 0; kk < KB / 16; ++kk) {
            const uint64_t da0 = sdesc_kmajor<Cfg::kRowBytes>(st + kk * 32);
            const uint64_t da1 = sdesc_kmajor<Cfg::kRowBytes>(st + Cfg::kABytes + kk * 32);
            const uint64_t db = sdesc_kmajor<Cfg::kRowBytes>(st + 2 * Cfg::kABytes + kk * 32);
            const uint32_t acc = (kb != slice * nk || kk != 0) ? 1u : 0u;
            umma_bf16(d0, da0, db, idesc, acc);
            umma_bf16(d1, da1, db, idesc, acc);
          }
          umma_commit(smem_u32(&empty[s]));  // frees the stage once these MMAs are done
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[b]));  // accumulator b is complete
      }
      // Every MMA issued above has finished before the CTA tears down.
      umma_commit(smem_u32(done));
      if (!mbar_wait(smem_u32(done), 0)) signal_abort(&abort_s, a.err);
    }
  } else {
    // ----------------------------------------------------- epilogue (2-9) ---
    const int q = warp & 3;                         // tensor-memory lane quarter this warp may read
    const int side = (warp - kEpiWarp0) >> 2;       // takes 32-column chunks side, side + 2, ...
    constexpr int kCh = BN / 64;                    // chunks per side
    const int r_in = q * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
      if (aborted(&abort_s)) break;
      int e, m, row0, nrows, slice;
      decode_tile_k<BN>(tile, a, E, cs_s, off_s, e, m, row0, nrows, slice);
      const int b = it % NACC;
      const uint32_t use = static_cast<uint32_t>(it / NACC);
      // Down mode: lane j holds the slot id and routing weight of column j of
      // each of this warp's chunks. They are loaded before the wait below, so
      // their latency hides behind the tile's main loop.
      int f_t[kCh];
      float w_t[kCh];
      if (MODE == MM_GEMM_DOWN) {
#pragma unroll
        for (int i = 0; i < kCh; ++i) {
          const int c = (2 * i + side) * 32 + lane;
          f_t[i] = c < nrows ? __ldg(a.sorted + row0 + c) : a.Tk;
        }
#pragma unroll
        for (int i = 0; i < kCh; ++i) w_t[i] = f_t[i] < a.Tk ? __ldg(a.topk_w + f_t[i]) : 0.f;
      }
      if (!mbar_wait(smem_u32(&tfull[b]), use & 1u)) {
        signal_abort(&abort_s, a.err);
        break;
      }
      tc_fence_after();
      const uint32_t tb =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * 2 * BN);
#pragma unroll
      for (int i = 0; i < kCh; ++i) {
        const int c0 = (2 * i + side) * 32;
        if (c0 >= nrows) break;
        uint32_t g[32], u[32];
        tmem_ld_32x32b_x32(tb + c0, g);
        tmem_ld_32x32b_x32(tb + BN + c0, u);
        tmem_wait_ld();
        const int ncol = min(32, nrows - c0);
        if (MODE == MM_GEMM_GATE_UP) {
          const int i_out = m * kGM + r_in;  // intermediate index
          if (i_out < a.N) {
            uint16_t* dst = static_cast<uint16_t*>(a.C) + (size_t)(row0 + c0) * a.N + i_out;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (j < ncol) {
                const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
                // silu(g) * u. The fast divide (about 2 ulp) is far below the
                // bf16 rounding of the result; for g < -87.3, where 1 + e^-g
                // exceeds 2^126, it returns 0 for a |silu(g)| under 1.1e-36.
                dst[(size_t)j * a.N] =
                    f32_to_bf16_bits(__fdividef(gv, 1.0f + __expf(-gv)) * uv);
              }
            }
          }
        } else {
          // Column j's slot id and routing weight come from lane j by
          // shuffle. The weighted values pass through this warp's shared
          // tile (row = token), kEpiTok tokens at a time, so that each lane
          // adds 4 consecutive outputs of one token with one 16-byte vector
          // atomic.
          const int f_l = f_t[i];
          const float w_l = w_t[i];
          const int t_l = f_l / a.top_k;
          float* accp = static_cast<float*>(a.C);
          const uint64_t pol_acc = l2_policy_evict_last();  // keep the accumulator in L2
          float* tr = epi_tile + (warp - kEpiWarp0) * kEpiTok * 33;  // [kEpiTok][32 + 1 pad]
          const int hq = m * 2 * kGM + q * 32;  // first h of this warp's rows
          const int h4 = (lane & 7) * 4;
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const int hb = hq + part * kGM;
#pragma unroll
            for (int grp = 0; grp < 32 / kEpiTok; ++grp) {
              __syncwarp();
#pragma unroll
              for (int j = 0; j < kEpiTok; ++j) {
                const int jj = grp * kEpiTok + j;
                const float wt = __shfl_sync(0xffffffffu, w_l, jj);
                tr[j * 33 + lane] = wt * __uint_as_float(part == 0 ? g[jj] : u[jj]);
              }
              __syncwarp();
#pragma unroll
              for (int s4 = 0; s4 < kEpiTok / 4; ++s4) {
                const int jl = s4 * 4 + (lane >> 3);  // token within the group
                const int jt = grp * kEpiTok + jl;
                const int f = __shfl_sync(0xffffffffu, f_l, jt);
                const int t = __shfl_sync(0xffffffffu, t_l, jt);
                if (jt < ncol && f < a.Tk && hb + h4 < a.N) {
                  const float* v = tr + jl * 33 + h4;
                  red_add_v4_f32(accp + (size_t)t * a.N + hb + h4, v[0], v[1], v[2], v[3], pol_acc);
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[b]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ----------------------------------------------------------------- host ---

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols] read in boxes of kb columns x box_rows
// rows with the 2*kb-byte swizzle (the layout the MMA descriptors expect).
}  // namespace

bool make_tensor_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows, int kb) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kb), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            kb == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tensor_map_sw128(CUtensorMap* m, const void* base, uint32_t rank,
                           const uint64_t* dims, const uint64_t* strides, const uint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || rank < 2 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], estr[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, b, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
template <int MODE, int BN, int S, int NACC, int KB>
cudaError_t launch_cfg(const uint16_t* X, bool x_is_hidden, const uint16_t* W, void* C,
                       const int32_t* sorted, const int32_t* offsets, const float* topk_w, int T,
                       int top_k, int E, int N, int K, long long capacity, long long x_rows,
                       int num_sms, unsigned* err, bool after_prev, cudaStream_t st,
                       float* zero_buf, long long zero_count) {
  using Cfg = GemmCfg<MODE, BN, S, NACC, KB>;
  static DeviceFlags attr_done;
  if (cudaError_t e =
          smem_attr_once(attr_done, grouped_gemm_kernel<MODE, BN, S, NACC, KB>, Cfg::kSmemBytes);
      e != cudaSuccess)
    return e;
  GemmArgs a;
  a.sorted = sorted;
  a.offsets = offsets;
  a.topk_w = topk_w;
  a.C = C;
  a.err = err;
  a.E = E;
  a.N = N;
  a.K = K;
  a.Tk = T * top_k;
  a.top_k = top_k;
  // With more than about half a chunk of rows per expert on average, several
  // token chunks read each weight tile: keep the weights at normal priority.
  a.w_evict_first = (long long)T * top_k <= (long long)E * (BN / 2) ? 1 : 0;
  a.hidden = x_is_hidden ? X : nullptr;
  a.w = W;
  a.zero_buf = zero_buf;
  a.zero_count = zero_count;
  // Decode-sized gate_up (rows gathered from hidden) with enough assignments
  // that nearly every expert is selected (T*k >= 4E: 98 % expected under
  // uniform routing), where the guess of the first tile holds: overlap the
  // router with the first tile's weight stream. With few selected experts
  // (a skewed or tiny batch) the guess is mostly wrong and only costs
  // bandwidth (T=1: 60 -> 63 us), so it is not made.
  a.prefetch_guess = (MODE == MM_GEMM_GATE_UP && x_is_hidden &&
                      gate_up_gathers_rows(T, top_k, E) && (long long)T * top_k >= 4LL * E)
                         ? 1 : 0;
  if (MODE == MM_GEMM_GATE_UP && x_is_hidden)
    a.b_mode = gate_up_gathers_rows(T, top_k, E) ? kBTmaGather : kBLsuGather;
  else
    a.b_mode = kBTma;
  if (MODE == MM_GEMM_GATE_UP) {
    a.w_rows = 2 * N;
    a.m_step = kGM;
    a.a1_off = N;
    a.n_mtiles = (N + kGM - 1) / kGM;
  } else {
    a.w_rows = N;
    a.m_step = 2 * kGM;
    a.a1_off = kGM;
    a.n_mtiles = (N + 2 * kGM - 1) / (2 * kGM);
  }
  // Down mode with too few (chunk, m-tile) pairs to fill the SMs (small
  // batches, the dense MLP at decode): split K into slices whose partial sums
  // the epilogue adds into the fp32 accumulator like any other contribution
  // (so the order of the additions, and the last bits of out, may vary from
  // call to call). With n <= min(E, T*k) experts holding r_e >= 1 rows each,
  // the chunks number sum ceil(r_e / BN) <= n + (T*k - n) / BN, which grows
  // with n: at most min(E, T*k) + (T*k - min(E, T*k)) / BN.
  a.ksplit = 1;
  if (MODE == MM_GEMM_DOWN) {
    const long long rows = (long long)T * top_k;
    const long long busy = std::min<long long>(E, rows);
    const long long tiles = (busy + (rows - busy) / BN) * a.n_mtiles;
    const int nkb = K / KB;
    for (int d = nkb / 2; d >= 2; --d)  // at least two K steps per slice
      if (nkb % d == 0 && tiles * d <= num_sms) {
        a.ksplit = d;
        break;
      }
  }
  CUtensorMap tmW, tmX;
  if (!make_tensor_map_2d(&tmW, W, (uint64_t)E * a.w_rows, (uint64_t)K, kGM, KB))
    return cudaErrorInvalidValue;
  // Gathered rows: X = hidden [T, K], one row per box; otherwise X holds the
  // token rows in segment order [capacity, K].
  // gather4 reads hidden [T, K] one row per box row; 2-D boxes read rows in
  // segment order [capacity, K]; the cp.async path does not use the map.
  const bool ok_x = a.b_mode == kBTma
                        ? make_tensor_map_2d(&tmX, X, (uint64_t)x_rows, (uint64_t)K, BN, KB)
                        : make_tensor_map_2d(&tmX, X, (uint64_t)T, (uint64_t)K, 1, KB);
  if (!ok_x) return cudaErrorInvalidValue;
  const long long max_tiles = (capacity / BN + E) * (long long)a.n_mtiles * a.ksplit;
  const int grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
  return launch_k(grouped_gemm_kernel<MODE, BN, S, NACC, KB>, dim3(grid), dim3(kGemmThreads),
                  Cfg::kSmemBytes, st, after_prev, tmW, tmX, a);
}

// Token rows in segment order: xs[r] = hidden[sorted[r] / k] for the rows of
// the expert segments (r < offsets[E]); padding rows become zeros. One warp
// per row, 16-byte loads and stores.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ hidden,
                                                          const int32_t* __restrict__ sorted,
                                                          const int32_t* __restrict__ offsets,
                                                          int E, int top_k, int Tk, int row16,
                                                          uint4* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  const int rows = __ldg(offsets + E);
  const int wstride = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += wstride) {
    const int f = __ldg(sorted + r);
    const uint4* src = f < Tk ? hidden + (size_t)(f / top_k) * row16 : nullptr;
    uint4* dst = xs + (size_t)r * row16;
#pragma unroll 4
    for (int i = lane; i < row16; i += 32)
      dst[i] = src != nullptr ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  return (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
}
// bf16(o + r) for the two bf16 pairs packed in o and r.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t o, uint32_t r) {
  return bf16x2_bits(__uint_as_float(o << 16) + __uint_as_float(r << 16),
                     __uint_as_float(o & 0xFFFF0000u) + __uint_as_float(r & 0xFFFF0000u));
}

// out = bf16(acc), rounded once; with res_out also the residual add that
// follows the layer, res_out = bf16(out + res_in) (out rounded first, then
// the sum, as a bf16 tensor add does; res_out may be res_in).
__global__ void __launch_bounds__(256) finalize_kernel(const float4* __restrict__ acc,
                                                       uint2* __restrict__ out, long long n4,
                                                       const uint2* res_in, uint2* res_out) {
  pdl_wait();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = acc[i];
    uint2 o;
    o.x = bf16x2_bits(v.x, v.y);
    o.y = bf16x2_bits(v.z, v.w);
    out[i] = o;
    if (res_out != nullptr) {
      const uint2 r = res_in[i];
      res_out[i] = make_uint2(add_bf16x2(o.x, r.x), add_bf16x2(o.y, r.y));
    }
  }
}

}  // namespace

bool gate_up_gathers_rows(int T, int top_k, int E) {
  return (long long)T * top_k <= 64LL * E;  // at most ~64 rows per expert on average
}

cudaError_t launch_grouped_gemm(int mode, const uint16_t* X, bool x_is_hidden, const uint16_t* W,
                                void* C, const int32_t* sorted, const int32_t* offsets,
                                const float* topk_w, int T, int top_k, int E, int N, int K,
                                long long capacity, long long x_rows, int num_sms, unsigned* err,
                                bool after_prev, cudaStream_t st, float* zero_buf,
                                long long zero_count) {
  // 256x128 tiles with two accumulator sets: the epilogue of one tile overlaps
  // the main loop of the next. (256x256 tiles with one set measured slower at
  // every batch size: the epilogue no longer overlaps, and a segment just over
  // 256 rows adds a nearly empty chunk that re-reads the whole weight tile.)
  // (Stages of K = 32 with the 64-byte swizzle, 9 or 8 of them in the same
  // shared memory, measured slower than 4 stages of K = 64 at every size.)
  // With few rows per expert (the decode regime, where gate_up gathers its
  // rows from hidden) the token tile is at most 64 rows, and the 8 KB it
  // frees per stage buys a fifth stage: more weight bytes in flight per SM.
  // Many rows per expert, read in segment order (the layer's row copy and
  // act, a dense MLP's hidden): the SM-pair kernel (gemm_pair.cu).
  if (!gate_up_gathers_rows(T, top_k, E) && (mode == MM_GEMM_DOWN || !x_is_hidden))
    return launch_grouped_gemm_pair(mode, X, W, C, sorted, offsets, topk_w, T, top_k, E, N, K,
                                    capacity, x_rows, num_sms, err, after_prev, st, zero_buf,
                                    zero_count);
  if (gate_up_gathers_rows(T, top_k, E)) {
    if (mode == MM_GEMM_GATE_UP)
      return launch_cfg<MM_GEMM_GATE_UP, 64, 5, 2, 64>(X, x_is_hidden, W, C, sorted, offsets,
                                                       topk_w, T, top_k, E, N, K, capacity,
                                                       x_rows, num_sms, err, after_prev, st,
                                                       zero_buf, zero_count);
    return launch_cfg<MM_GEMM_DOWN, 64, 5, 2, 64>(X, false, W, C, sorted, offsets, topk_w, T,
                                                  top_k, E, N, K, capacity, x_rows, num_sms, err,
                                                  after_prev, st, nullptr, 0);
  }
  if (mode == MM_GEMM_GATE_UP)
    return launch_cfg<MM_GEMM_GATE_UP, 128, 4, 2, 64>(X, x_is_hidden, W, C, sorted, offsets,
                                                      topk_w, T, top_k, E, N, K, capacity, x_rows,
                                                      num_sms, err, after_prev, st, zero_buf,
                                                      zero_count);
  return launch_cfg<MM_GEMM_DOWN, 128, 4, 2, 64>(X, false, W, C, sorted, offsets, topk_w, T, top_k,
                                                 E, N, K, capacity, x_rows, num_sms, err,
                                                 after_prev, st, nullptr, 0);
}

cudaError_t launch_gather_rows(const uint16_t* hidden, const int32_t* sorted,
                               const int32_t* offsets, int T, int top_k, int E, int H,
                               uint16_t* xs, int num_sms, bool after_prev, cudaStream_t st) {
  return launch_k(gather_rows_kernel, dim3(num_sms * 8), dim3(256), 0, st, after_prev,
                  reinterpret_cast<const uint4*>(hidden), sorted, offsets, E, top_k, T * top_k,
                  H / 8, reinterpret_cast<uint4*>(xs));
}

cudaError_t launch_finalize(const float* acc, uint16_t* out, long long n, int num_sms,
                            bool after_prev, cudaStream_t st, const uint16_t* res_in,
                            uint16_t* res_out) {
  const long long n4 = n / 4;
  long long blocks = (n4 + 255) / 256;
  const long long cap_blocks = (long long)num_sms * 8;
  if (blocks > cap_blocks) blocks = cap_blocks;
  if (blocks < 1) blocks = 1;
  return launch_k(finalize_kernel, dim3((int)blocks), dim3(256), 0, st, after_prev,
                  reinterpret_cast<const float4*>(acc), reinterpret_cast<uint2*>(out), n4,
                  reinterpret_cast<const uint2*>(res_in), reinterpret_cast<uint2*>(res_out));
}

}  // namespace mm
