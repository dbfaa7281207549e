// Grouped expert GEMMs for batches with many rows per expert (prefill), on
// CTA pairs: tcgen05.mma.cta_group::2 runs one M=256 MMA across the tensor
// cores of two SMs of a cluster. Each CTA holds half of the weight rows (A,
// 128 rows) and half of the token rows (B, N/2 rows) of every K step; the
// pair computes 256 weight rows x N tokens (N <= 256), each CTA keeping its
// 128 rows of the accumulator in its own tensor memory. Per SM that is the
// work of the single-CTA kernel's stage with 32 KB of shared memory instead
// of 48 KB, so six stages fit where four did.
//
// Tiles: (expert e, token chunk of <= 256 rows, m-tile). An expert's segment
// is cut into ceil(L/256) chunks of near-equal size (multiples of 16).
//   gate_up: an m-tile covers 128 intermediate rows; CTA r owns 64 of them,
//     i0 = m*128 + r*64. Its 128 A rows are laid out in four 32-row groups,
//     one per tensor-memory lane quarter: group q = gate rows i0+16q..+15
//     then the matching up rows. A warp therefore finds gate and up of one
//     intermediate row in lanes l and l+16 of its own quarter, and
//     SiLU(gate)*up needs only a shuffle ("模型与权重加载", GatedMLP:
//     silu_and_mul of the merged gate_up projection, gate rows first).
//   down: an m-tile covers 256 rows of H; CTA r owns 128 of them. The
//     epilogue multiplies by the routing weight and adds into the fp32 output
//     accumulator with 16-byte vector atomics ("mini-sglang guide, chapter
//     7": expert outputs weighted by their softmax scores and summed).
//
// Roles per CTA (192 threads): warp 0 = TMA producer (both CTAs load their
// halves; completion is counted on the leader CTA's barrier), warp 1 =
// tensor-memory allocation (both CTAs) and MMA issue (leader only), warps
// 2-5 = epilogue (both CTAs, each on its own tensor memory). Every wait on
// another thread or CTA is bounded and records MM_ERR_TIMEOUT instead of
// hanging; an abort is mirrored to the peer CTA.
#include "mm.h"
#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

constexpr int kPK = 64;          // K per stage (one 128-byte swizzle row of bf16)
constexpr int kPStages = 6;
constexpr int kPThreads = 192;
constexpr int kPMaxN = 256;      // token rows per chunk
constexpr int kPABytes = 128 * kPK * 2;   // 16 KB: this CTA's 128 weight rows
constexpr int kPBBytes = 128 * kPK * 2;   // 16 KB: this CTA's (up to) 128 token rows
constexpr int kPStageBytes = kPABytes + kPBBytes;
constexpr int kPEpiBytes = 4 * 32 * 33 * 4;  // down: per-warp transpose tile
constexpr int kPSmemBytes = kPStages * kPStageBytes + kPEpiBytes + 1024;
constexpr uint32_t kPTmemCols = 512;         // 2 accumulator buffers x 256 columns

struct PairArgs {
  const int32_t* sorted;
  const int32_t* offsets;
  const float* topk_w;
  void* C;
  unsigned* err;
  int E, N, K, Tk, top_k;
  int n_mtiles;
  int w_rows;            // weight rows per expert (2N gate_up, N down)
  int w_evict_first;
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_smem, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem), "r"(rank));
  return r;
}

__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void umma2_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the barrier at offset `bar` in every CTA of `mask` when the
// pair MMAs issued so far have completed.
__device__ __forceinline__ void umma2_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// 2-D box load into this CTA's shared memory whose completion is counted on
// `bar`, a barrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* map, uint32_t bar,
                                                 int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// Announces `bytes` of TMA traffic on a barrier of either CTA of the pair.
// Relaxed: the producer publishes no data of its own here (the bytes are
// tracked by the copies' complete_tx), and a release would make the thread
// wait for its earlier copies, serialising the pipeline stages.
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cluster_bar,
                                                              uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(
          cluster_bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

struct PairShared {
  int off[kMaxExperts + 1];
  int cs[kMaxExperts + 1];   // first chunk of each expert
  int csz[kMaxExperts];      // rows per chunk of each expert
};

__device__ __forceinline__ void decode_pair_tile(int tile, int n_mtiles, int E,
                                                 const PairShared& S, int& e, int& m, int& row0,
                                                 int& nrows) {
  const int ch = tile / n_mtiles;
  m = tile - ch * n_mtiles;
  int lo = 0, hi = E;  // S.cs[lo] <= ch < S.cs[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (S.cs[mid] <= ch)
      lo = mid;
    else
      hi = mid;
  }
  e = lo;
  const int c = ch - S.cs[e];
  row0 = S.off[e] + c * S.csz[e];
  nrows = min(S.csz[e], S.off[e + 1] - row0);
}

template <int MODE>
__global__ void __launch_bounds__(kPThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmW,
                             const __grid_constant__ CUtensorMap tmX, const PairArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kPStages + 5];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ PairShared S;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E;
  const uint32_t rank = cluster_ctarank();  // 0 = leader (issues the MMAs)
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  // Chunk table: balanced chunks of at most kPMaxN rows per expert.
  for (int i = tid; i <= E; i += kPThreads) S.off[i] = a.offsets[i];
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32, e0 = lane * per;
    int sum = 0;
    for (int j = 0; j < per; ++j) {
      const int e = e0 + j;
      if (e < E) sum += (S.off[e + 1] - S.off[e] + kPMaxN - 1) / kPMaxN;
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
        const int L = S.off[e + 1] - S.off[e];
        const int nch = (L + kPMaxN - 1) / kPMaxN;
        S.cs[e] = run;
        S.csz[e] = nch > 0 ? ((L + nch - 1) / nch + 15) / 16 * 16 : 0;
        run += nch;
      }
    }
    if (lane == 31) S.cs[E] = incl;
  }
  __syncthreads();
  const int total_tiles = S.cs[E] * a.n_mtiles;
  if (pair >= total_tiles) return;  // uniform across the pair: no cluster barrier is skipped

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t smem_base = (raw_addr + 1023u) & ~1023u;
  float* epi_tile =
      reinterpret_cast<float*>(smem_raw + (smem_base - raw_addr) + kPStages * kPStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kPStages;
  uint64_t* tfull = bars + 2 * kPStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;

  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(smem_u32(&full[s]), 2);   // each CTA's producer announces its own bytes
      mbar_init(smem_u32(&empty[s]), 1);  // the leader's MMA commit, multicast to both CTAs
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 8);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(smem_u32(done), 1);
    abort_s = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc2(smem_u32(&tmem_base_s), kPTmemCols);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised; allocation visible
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;
  const uint32_t peer_abort = map_to_rank(smem_u32(&abort_s), rank ^ 1u);
  auto fail = [&]() {
    *reinterpret_cast<volatile int*>(&abort_s) = 1;
    st_cluster_u32(peer_abort, 1u);
    atomicOr(a.err, kDevErrTimeout);
  };
  auto aborted_p = [&]() { return *reinterpret_cast<volatile int*>(&abort_s) != 0; };
  const int nk = a.K / kPK;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer ---
    if (lane == 0) {
      const uint64_t pol_w = a.w_evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t pol_x = l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      for (int tile = pair; tile < total_tiles; tile += npairs) {
        if (aborted_p()) break;
        int e, m, row0, nrows;
        decode_pair_tile(tile, a.n_mtiles, E, S, e, m, row0, nrows);
        const int n_mma = (nrows + 15) & ~15;
        const int brow = row0 + (int)rank * (n_mma / 2);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u)) {
            fail();
            ok = false;
            break;
          }
          const uint32_t st = smem_base + s * kPStageBytes;
          const uint32_t fb = map_to_rank(smem_u32(&full[s]), 0);  // the leader's barrier
          mbar_arrive_expect_tx_cluster(fb, kPStageBytes);  // before this CTA's loads
          const int kc = kb * kPK;
          if (MODE == MM_GEMM_GATE_UP) {
            // Four 32-row groups: 16 gate rows, then the same 16 up rows.
            const int g0 = e * a.w_rows + m * 128 + (int)rank * 64;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              tma_load_2d_pair(st + q * 4096, &tmW, fb, kc, g0 + 16 * q, pol_w);
              tma_load_2d_pair(st + q * 4096 + 2048, &tmW, fb, kc, g0 + a.N + 16 * q, pol_w);
            }
          } else {
            tma_load_2d_pair(st, &tmW, fb, kc, e * a.w_rows + m * 256 + (int)rank * 128, pol_w);
          }
          tma_load_2d_pair(st + kPABytes, &tmX, fb, kc, brow, pol_x);
          if (++s == kPStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer (leader) ---
    if (leader && lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      for (int tile = pair; tile < total_tiles; tile += npairs, ++it) {
        if (aborted_p()) break;
        int e, m, row0, nrows;
        decode_pair_tile(tile, a.n_mtiles, E, S, e, m, row0, nrows);
        const int b = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait(smem_u32(&tempty[b]), (use & 1u) ^ 1u)) {
          fail();
          break;
        }
        tc_fence_after();
        const int n_mma = (nrows + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(256, n_mma);
        const uint32_t d = tmem_base + static_cast<uint32_t>(b * kPMaxN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(smem_u32(&full[s]), ph)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_base + s * kPStageBytes;
#pragma unroll
          for (int kk = 0; kk < kPK / 16; ++kk)
            umma2_bf16(d, sdesc_k128(st + kk * 32), sdesc_k128(st + kPABytes + kk * 32), idesc,
                       (kb | kk) != 0 ? 1u : 0u);
          umma2_commit_mc(smem_u32(&empty[s]), 0x3);  // frees stage s in both CTAs
          if (++s == kPStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma2_commit_mc(smem_u32(&tfull[b]), 0x3);  // accumulator b complete in both CTAs
      }
      umma2_commit_mc(smem_u32(done), 0x1);
      if (!mbar_wait(smem_u32(done), 0)) fail();
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue ---
    const int q = warp & 3;  // tensor-memory lane quarter this warp reads
    const uint32_t tempty_leader0 = map_to_rank(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_leader1 = map_to_rank(smem_u32(&tempty[1]), 0);
    float* tr = epi_tile + (warp - 2) * 32 * 33;
    const uint64_t pol_acc = l2_policy_evict_last();
    int it = 0;
    for (int tile = pair; tile < total_tiles; tile += npairs, ++it) {
      if (aborted_p()) break;
      int e, m, row0, nrows;
      decode_pair_tile(tile, a.n_mtiles, E, S, e, m, row0, nrows);
      const int b = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      int f_t[kPMaxN / 32];
      float w_t[kPMaxN / 32];
      if (MODE == MM_GEMM_DOWN) {
#pragma unroll
        for (int cc = 0; cc < kPMaxN / 32; ++cc) {
          const int c = cc * 32 + lane;
          f_t[cc] = c < nrows ? __ldg(a.sorted + row0 + c) : a.Tk;
        }
#pragma unroll
        for (int cc = 0; cc < kPMaxN / 32; ++cc)
          w_t[cc] = f_t[cc] < a.Tk ? __ldg(a.topk_w + f_t[cc]) : 0.f;
      }
      bool ok = true;
      if (lane == 0) ok = mbar_wait(smem_u32(&tfull[b]), use & 1u);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(b * kPMaxN);
#pragma unroll 1
      for (int cc = 0; cc < kPMaxN / 32; ++cc) {
        const int c0 = cc * 32;
        if (c0 >= nrows) break;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tb + c0, v);
        tmem_wait_ld();
        const int ncol = min(32, nrows - c0);
        if (MODE == MM_GEMM_GATE_UP) {
          // Lanes 0-15 hold gate, lanes 16-31 up of the same 16 intermediate
          // rows. Lane l < 16 finishes columns 0-15, lane l + 16 columns 16-31.
          const bool is_gate = lane < 16;
          const int i = m * 128 + (int)rank * 64 + q * 16 + (lane & 15);
          float x[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float send = __uint_as_float(is_gate ? v[16 + j] : v[j]);
            x[j] = __shfl_xor_sync(0xffffffffu, send, 16);
          }
          if (i < a.N) {
            const int cbase = is_gate ? 0 : 16;
            uint16_t* dst = static_cast<uint16_t*>(a.C) + (size_t)(row0 + c0 + cbase) * a.N + i;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (cbase + j < ncol) {
                const float gv = is_gate ? __uint_as_float(v[j]) : x[j];
                const float uv = is_gate ? x[j] : __uint_as_float(v[16 + j]);
                dst[(size_t)j * a.N] = f32_to_bf16_bits(gv / (1.0f + __expf(-gv)) * uv);
              }
            }
          }
        } else {
          // Weighted 32x32 block -> this warp's tile (row = token) -> one
          // 16-byte vector atomic per lane per 4 outputs of a token.
          float wl = 0.f;
          int fl = a.Tk, tl = 0;
#pragma unroll
          for (int c2 = 0; c2 < kPMaxN / 32; ++c2)
            if (c2 == cc) {
              wl = w_t[c2];
              fl = f_t[c2];
            }
          tl = fl / a.top_k;
          const int hb = m * 256 + (int)rank * 128 + q * 32;
          float* accp = static_cast<float*>(a.C);
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float wt = __shfl_sync(0xffffffffu, wl, j);
            tr[j * 33 + lane] = wt * __uint_as_float(v[j]);
          }
          __syncwarp();
          const int h4 = (lane & 7) * 4;
#pragma unroll
          for (int it2 = 0; it2 < 8; ++it2) {
            const int jt = it2 * 4 + (lane >> 3);
            const int f = __shfl_sync(0xffffffffu, fl, jt);
            const int t = __shfl_sync(0xffffffffu, tl, jt);
            if (jt < ncol && f < a.Tk && hb + h4 < a.N) {
              const float* vv = tr + jt * 33 + h4;
              red_add_v4_f32(accp + (size_t)t * a.N + hb + h4, vv[0], vv[1], vv[2], vv[3],
                             pol_acc);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(b == 0 ? tempty_leader0 : tempty_leader1);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs done with tensor memory and with each other's barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, kPTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_map_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kPK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_pair_mode(const uint16_t* X, const uint16_t* W, void* C,
                             const int32_t* sorted, const int32_t* offsets, const float* topk_w,
                             int T, int top_k, int E, int N, int K, long long capacity,
                             int num_sms, unsigned* err, cudaStream_t st) {
  static bool attr_done[kMaxDevices] = {};
  const int dev = current_device();
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  PairArgs a;
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
  a.w_evict_first = 0;
  CUtensorMap tmW, tmX;
  if (MODE == MM_GEMM_GATE_UP) {
    a.w_rows = 2 * N;
    a.n_mtiles = (N + 127) / 128;
    if (!make_map_rows(&tmW, W, (uint64_t)E * a.w_rows, (uint64_t)K, 16))
      return cudaErrorInvalidValue;
  } else {
    a.w_rows = N;
    a.n_mtiles = (N + 255) / 256;
    if (!make_map_rows(&tmW, W, (uint64_t)E * a.w_rows, (uint64_t)K, 128))
      return cudaErrorInvalidValue;
  }
  if (!make_map_rows(&tmX, X, (uint64_t)capacity, (uint64_t)K, 128)) return cudaErrorInvalidValue;
  // At most capacity/16 chunks of >= 16 rows... bounded by E + capacity / 128.
  const long long max_tiles = ((capacity + kPMaxN - 1) / kPMaxN + E) * (long long)a.n_mtiles;
  long long pairs = num_sms / 2;
  if (pairs > max_tiles) pairs = max_tiles;
  if (pairs < 1) pairs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kPThreads, 1, 1);
  cfg.dynamicSmemBytes = kPSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<MODE>, tmW, tmX, a);
}

}  // namespace

cudaError_t launch_grouped_gemm_pair(int mode, const uint16_t* X, const uint16_t* W, void* C,
                                     const int32_t* sorted, const int32_t* offsets,
                                     const float* topk_w, int T, int top_k, int E, int N, int K,
                                     long long capacity, int num_sms, unsigned* err,
                                     cudaStream_t st) {
  if (mode == MM_GEMM_GATE_UP)
    return launch_pair_mode<MM_GEMM_GATE_UP>(X, W, C, sorted, offsets, topk_w, T, top_k, E, N, K,
                                             capacity, num_sms, err, st);
  return launch_pair_mode<MM_GEMM_DOWN>(X, W, C, sorted, offsets, topk_w, T, top_k, E, N, K,
                                        capacity, num_sms, err, st);
}

}  // namespace mm
