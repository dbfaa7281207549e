// Grouped expert GEMMs of the MoE layer on the sm_103a tensor cores
// (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
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
// Token rows: in gate_up mode with few rows per expert (decode-sized
// batches) they are gathered from hidden by TMA tile::gather4 (four rows per
// instruction, indexed by sorted_token_ids / k), so no permuted copy of the
// activations is written. With many rows per expert the TMA engine would
// spend a gather per four rows of every stage, so the rows are first copied
// into segment order (gather_rows_kernel) and loaded as plain 2-D boxes, like
// the contiguous act rows of the down mode.
//
// Warp roles (192 threads, one CTA per SM, persistent over a static tile
// stride): warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2-5 = epilogue (each reads its 32-lane quarter of tensor memory).
// Two accumulator buffers let the epilogue of one tile overlap the
// main loop of the next.
//
// Epilogues: gate_up writes act = bf16(silu(g) * u) ("模型与权重加载",
// GatedMLP: silu_and_mul of the merged gate_up projection, gate first);
// down multiplies by the routing weight and adds into the fp32 output
// accumulator ("mini-sglang guide, chapter 7": expert outputs weighted by the
// softmax scores and summed).
#include <mutex>

#include "mm.h"
#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

constexpr int kGM = 128;  // weight rows per MMA
constexpr int kGK = 64;   // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kGemmThreads = 192;

struct GemmArgs {
  const int32_t* sorted;   // [capacity]
  const int32_t* offsets;  // [E+1]
  const float* topk_w;     // [T*k] (down mode)
  void* C;                 // act bf16 [capacity, N] | acc fp32 [T, N]
  unsigned* err;
  int E, N, K, Tk, top_k;
  int n_mtiles;  // m-tiles per token chunk
  int w_rows;    // weight rows per expert in the 2-D weight view
  int m_step;    // weight rows per m-tile
  int a1_off;    // row offset of the A1 tile relative to A0
  int w_evict_first;  // weights are read by one token chunk only: stream them past L2
  int gather_rows;    // gate_up: token rows come straight from hidden by tile::gather4
};

template <int BN, int STAGES>
struct GemmCfg {
  static constexpr int kABytes = kGM * kGK * 2;
  static constexpr int kBBytes = BN * kGK * 2;
  static constexpr int kStageBytes = 2 * kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 4 * BN;  // 2 buffers x (D0, D1) x BN columns
  static constexpr int kEpiBytes = 4 * 32 * 33 * 4;  // per epilogue warp: 32x33 fp32 tile
  static constexpr int kSmemBytes = STAGES * kStageBytes + kEpiBytes + 1024;
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                "tensor-memory allocation must be a power of two in [32, 512]");
  static_assert(BN % 32 == 0 && BN <= 256, "BN");
};

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

__device__ __forceinline__ bool aborted(const int* flag) {
  return *reinterpret_cast<const volatile int*>(flag) != 0;
}

__device__ __forceinline__ void signal_abort(int* flag, unsigned* err) {
  *reinterpret_cast<volatile int*>(flag) = 1;
  atomicOr(err, kDevErrTimeout);
}

template <int MODE, int BN, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmX, const GemmArgs a) {
  using Cfg = GemmCfg<BN, STAGES>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * STAGES + 5];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int off_s[kMaxExperts + 1];
  __shared__ int cs_s[kMaxExperts + 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E;

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
  const int total_tiles = cs_s[E] * a.n_mtiles;
  if ((int)blockIdx.x >= total_tiles) return;  // uniform across the CTA

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t smem_base = (raw_addr + 1023u) & ~1023u;
  float* epi_tile = reinterpret_cast<float*>(smem_raw + (smem_base - raw_addr) +
                                             STAGES * Cfg::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 128);
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

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer ---
    const uint64_t pol_w = a.w_evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
    const uint64_t pol_x = l2_policy_evict_last();
    const int nk = a.K / kGK;
    int s = 0;
    uint32_t ph = 0;
    if (MODE == MM_GEMM_GATE_UP && a.gather_rows) {
      // Token rows are gathered straight from hidden: lane i loads rows
      // 4i..4i+3 of the chunk with one tile::gather4 per stage. The rows of the
      // next tile are fetched one tile ahead so their latency is hidden.
      int nxt[4];
      auto fetch_rows = [&](int tl, int (&rows)[4]) {
        int e, m, row0, nrows;
        if (tl < total_tiles) decode_tile<BN>(tl, a.n_mtiles, E, cs_s, off_s, e, m, row0, nrows);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 4 * lane + j;
          const int f = (tl < total_tiles && r < nrows) ? __ldg(a.sorted + row0 + r) : a.Tk;
          rows[j] = f < a.Tk ? f / a.top_k : 0;  // padding rows read row 0 (never stored)
        }
      };
      fetch_rows(blockIdx.x, nxt);
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        if (aborted(&abort_s)) break;
        int rows[4] = {nxt[0], nxt[1], nxt[2], nxt[3]};
        fetch_rows(tile + gridDim.x, nxt);
        int e, m, row0, nrows;
        decode_tile<BN>(tile, a.n_mtiles, E, cs_s, off_s, e, m, row0, nrows);
        const int wrow0 = e * a.w_rows + m * a.m_step;
        const int wrow1 = wrow0 + a.a1_off;
        const int n_g4 = ((nrows + 15) & ~15) / 4;  // rows the MMA reads, 4 per gather
        const uint32_t bytes = 2 * Cfg::kABytes + n_g4 * 4 * kGK * 2;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (lane == 0) ok = mbar_wait(smem_u32(&empty[s]), ph ^ 1u);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            if (lane == 0) signal_abort(&abort_s, a.err);
            break;
          }
          const uint32_t st = smem_base + s * Cfg::kStageBytes;
          const uint32_t fb = smem_u32(&full[s]);
          if (lane == 0) {
            mbar_arrive_expect_tx(fb, bytes);
            tma_load_2d(st, &tmW, fb, kb * kGK, wrow0, pol_w);
            tma_load_2d(st + Cfg::kABytes, &tmW, fb, kb * kGK, wrow1, pol_w);
          }
          __syncwarp();
          if (lane < n_g4)
            tma_gather4(st + 2 * Cfg::kABytes + lane * 4 * kGK * 2, &tmX, fb, kb * kGK, rows[0],
                        rows[1], rows[2], rows[3], pol_x);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
    } else if (lane == 0) {
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        if (aborted(&abort_s)) break;
        int e, m, row0, nrows;
        decode_tile<BN>(tile, a.n_mtiles, E, cs_s, off_s, e, m, row0, nrows);
        const int wrow0 = e * a.w_rows + m * a.m_step;
        const int wrow1 = wrow0 + a.a1_off;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u)) {
            signal_abort(&abort_s, a.err);
            ok = false;
            break;
          }
          const uint32_t st = smem_base + s * Cfg::kStageBytes;
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          tma_load_2d(st, &tmW, fb, kb * kGK, wrow0, pol_w);
          tma_load_2d(st + Cfg::kABytes, &tmW, fb, kb * kGK, wrow1, pol_w);
          tma_load_2d(st + 2 * Cfg::kABytes, &tmX, fb, kb * kGK, row0, pol_x);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      const int nk = a.K / kGK;
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
        if (aborted(&abort_s)) break;
        int e, m, row0, nrows;
        decode_tile<BN>(tile, a.n_mtiles, E, cs_s, off_s, e, m, row0, nrows);
        const int b = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
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
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(smem_u32(&full[s]), ph)) {
            signal_abort(&abort_s, a.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_base + s * Cfg::kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kGK / 16; ++kk) {
            const uint64_t da0 = sdesc_k128(st + kk * 32);
            const uint64_t da1 = sdesc_k128(st + Cfg::kABytes + kk * 32);
            const uint64_t db = sdesc_k128(st + 2 * Cfg::kABytes + kk * 32);
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            umma_bf16(d0, da0, db, idesc, acc);
            umma_bf16(d1, da1, db, idesc, acc);
          }
          umma_commit(smem_u32(&empty[s]));  // frees the stage once these MMAs are done
          if (++s == STAGES) {
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
    // ---------------------------------------------------------- epilogue ---
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    const int r_in = q * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
      if (aborted(&abort_s)) break;
      int e, m, row0, nrows;
      decode_tile<BN>(tile, a.n_mtiles, E, cs_s, off_s, e, m, row0, nrows);
      const int b = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      // Down mode: lane j holds the slot id and routing weight of columns
      // j, j+32, ... of this tile. They are loaded before the wait below, so
      // their latency hides behind the tile's main loop.
      int f_t[BN / 32];
      float w_t[BN / 32];
      if (MODE == MM_GEMM_DOWN) {
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc) {
          const int c = cc * 32 + lane;
          f_t[cc] = c < nrows ? __ldg(a.sorted + row0 + c) : a.Tk;
        }
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc)
          w_t[cc] = f_t[cc] < a.Tk ? __ldg(a.topk_w + f_t[cc]) : 0.f;
      }
      if (!mbar_wait(smem_u32(&tfull[b]), use & 1u)) {
        signal_abort(&abort_s, a.err);
        break;
      }
      tc_fence_after();
      const uint32_t tb =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * 2 * BN);
#pragma unroll
      for (int cc = 0; cc < BN / 32; ++cc) {
        const int c0 = cc * 32;
        if (c0 >= nrows) break;
        uint32_t g[32], u[32];
        tmem_ld_32x32b_x32(tb + c0, g);
        tmem_ld_32x32b_x32(tb + BN + c0, u);
        tmem_wait_ld();
        const int ncol = min(32, nrows - c0);
        if (MODE == MM_GEMM_GATE_UP) {
          const int i = m * kGM + r_in;  // intermediate index
          if (i < a.N) {
            uint16_t* dst = static_cast<uint16_t*>(a.C) + (size_t)(row0 + c0) * a.N + i;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (j < ncol) {
                const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
                dst[(size_t)j * a.N] = f32_to_bf16_bits(gv / (1.0f + __expf(-gv)) * uv);
              }
            }
          }
        } else {
          // Column j's slot id and routing weight come from lane j by
          // shuffle. The weighted 32x32 block of each
          // accumulator goes through this warp's shared tile (row = token) so
          // that each lane adds 4 consecutive outputs of one token with one
          // 16-byte vector atomic.
          const int f_l = f_t[cc];
          const float w_l = w_t[cc];
          const int t_l = f_l / a.top_k;
          float* accp = static_cast<float*>(a.C);
          const uint64_t pol_acc = l2_policy_evict_last();  // keep the accumulator in L2
          float* tr = epi_tile + (warp - 2) * 32 * 33;  // [token 32][h 32 + 1 pad]
          const int hq = m * 2 * kGM + q * 32;            // first h of this warp's rows
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int hb = hq + half * kGM;
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float wt = __shfl_sync(0xffffffffu, w_l, j);
              tr[j * 33 + lane] = wt * __uint_as_float(half == 0 ? g[j] : u[j]);
            }
            __syncwarp();
            const int h4 = (lane & 7) * 4;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int jt = it * 4 + (lane >> 3);
              const int f = __shfl_sync(0xffffffffu, f_l, jt);
              const int t = __shfl_sync(0xffffffffu, t_l, jt);
              if (jt < ncol && f < a.Tk && hb + h4 < a.N) {
                const float* v = tr + jt * 33 + h4;
                red_add_v4_f32(accp + (size_t)t * a.N + hb + h4, v[0], v[1], v[2], v[3], pol_acc);
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

// Row-major bf16 matrix [rows, cols] read in boxes of 64 columns x box_rows
// rows with the 128-byte swizzle (the layout the MMA descriptors expect).
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kGK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int BN, int STAGES>
cudaError_t launch_cfg(const uint16_t* X, bool x_is_hidden, const uint16_t* W, void* C,
                       const int32_t* sorted, const int32_t* offsets, const float* topk_w, int T,
                       int top_k, int E, int N, int K, long long capacity, int num_sms,
                       unsigned* err, cudaStream_t st) {
  using Cfg = GemmCfg<BN, STAGES>;
  static bool attr_done[kMaxDevices] = {};
  const int dev = current_device();
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, BN, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
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
  a.gather_rows = (MODE == MM_GEMM_GATE_UP && x_is_hidden) ? 1 : 0;
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
  CUtensorMap tmW, tmX;
  if (!make_map(&tmW, W, (uint64_t)E * a.w_rows, (uint64_t)K, kGM)) return cudaErrorInvalidValue;
  // Gathered rows: X = hidden [T, K], one row per box; otherwise X holds the
  // token rows in segment order [capacity, K].
  const bool ok_x = a.gather_rows ? make_map(&tmX, X, (uint64_t)T, (uint64_t)K, 1)
                                  : make_map(&tmX, X, (uint64_t)capacity, (uint64_t)K, BN);
  if (!ok_x) return cudaErrorInvalidValue;
  const long long max_tiles = (capacity / BN + E) * (long long)a.n_mtiles;
  const int grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
  grouped_gemm_kernel<MODE, BN, STAGES><<<grid, kGemmThreads, Cfg::kSmemBytes, st>>>(tmW, tmX, a);
  return cudaGetLastError();
}

// x_sorted[r] = hidden[sorted[r] / k] (zeros for padding rows), one warp per
// row, 16-byte loads and stores.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ hidden,
                                                          const int32_t* __restrict__ sorted,
                                                          const int32_t* __restrict__ offsets,
                                                          int E, int Tk, int k, int H,
                                                          uint16_t* __restrict__ xs) {
  const int m_pad = offsets[E];
  const int lane = threadIdx.x & 31;
  const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
  const int vec = H / 8;
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < m_pad;
       r += nw) {
    const int f = sorted[r];
    uint4* dst = reinterpret_cast<uint4*>(xs + r * H);
    if (f < Tk) {
      const uint4* src = reinterpret_cast<const uint4*>(hidden + (size_t)(f / k) * H);
      for (int c = lane; c < vec; c += 32) dst[c] = __ldg(src + c);
    } else {
      for (int c = lane; c < vec; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

__global__ void __launch_bounds__(256) finalize_kernel(const float4* __restrict__ acc,
                                                       uint2* __restrict__ out, long long n4) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = acc[i];
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(v.x) | ((uint32_t)f32_to_bf16_bits(v.y) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(v.z) | ((uint32_t)f32_to_bf16_bits(v.w) << 16);
    out[i] = o;
  }
}

}  // namespace

bool gate_up_gathers_rows(int T, int top_k, int E) {
  return (long long)T * top_k <= 64LL * E;  // at most ~64 rows per expert on average
}

cudaError_t launch_grouped_gemm(int mode, const uint16_t* X, bool x_is_hidden, const uint16_t* W,
                                void* C, const int32_t* sorted, const int32_t* offsets,
                                const float* topk_w, int T, int top_k, int E, int N, int K,
                                long long capacity, int num_sms, unsigned* err, cudaStream_t st) {
  if (mode == MM_GEMM_GATE_UP)
    return launch_cfg<MM_GEMM_GATE_UP, 128, 4>(X, x_is_hidden, W, C, sorted, offsets, topk_w, T,
                                               top_k, E, N, K, capacity, num_sms, err, st);
  return launch_cfg<MM_GEMM_DOWN, 128, 4>(X, false, W, C, sorted, offsets, topk_w, T, top_k, E, N,
                                          K, capacity, num_sms, err, st);
}

cudaError_t launch_gather_rows(const uint16_t* hidden, const int32_t* sorted,
                               const int32_t* offsets, int E, int T, int top_k, int H,
                               long long capacity, uint16_t* x_sorted, int num_sms,
                               cudaStream_t st) {
  long long blocks = (capacity + 7) / 8;
  const long long cap_blocks = (long long)num_sms * 8;
  if (blocks > cap_blocks) blocks = cap_blocks;
  if (blocks < 1) blocks = 1;
  gather_rows_kernel<<<(int)blocks, 256, 0, st>>>(hidden, sorted, offsets, E, T * top_k, top_k, H,
                                                  x_sorted);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* acc, uint16_t* out, long long n, int num_sms,
                            cudaStream_t st) {
  const long long n4 = n / 4;
  long long blocks = (n4 + 255) / 256;
  const long long cap_blocks = (long long)num_sms * 8;
  if (blocks > cap_blocks) blocks = cap_blocks;
  if (blocks < 1) blocks = 1;
  finalize_kernel<<<(int)blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(acc),
                                               reinterpret_cast<uint2*>(out), n4);
  return cudaGetLastError();
}

}  // namespace mm
