// Grouped expert GEMMs for batches with many token rows per expert (prefill),
// on SM pairs: tcgen05.mma.cta_group::2 runs one M = 256 MMA across the
// tensor cores of the two SMs of a cluster. Each CTA holds half of the
// tile's weight rows (A: 128 rows) and half of its token rows (B: N/2 rows)
// for every K step, and keeps its 128 rows x N tokens of the accumulator in
// its own tensor memory. Per SM that is the MMA work of a 256 x 128 tile
// with 32 KB of shared memory per K step instead of 48 KB: a third fewer
// bytes through L2 per flop, and six stages in flight where four fit before.
//
// Tiles: (expert e, token chunk, m-tile). An expert's segment of L rows is
// cut into ceil(L / 256) chunks of near-equal size (multiples of 16), so a
// segment just over 256 rows does not leave a nearly empty chunk behind.
// Tiles are ordered chunk-major (the m-tiles of one chunk, then the next
// chunk of the same expert), so the pairs working at one time share token
// rows and weight tiles through L2.
//   gate_up ("模型与权重加载", GatedMLP: silu_and_mul of the merged gate_up
//   projection, gate rows first): an m-tile covers 128 intermediate rows;
//   CTA r holds 64 of them (i0 = m*128 + r*64) as four 32-row groups, one
//   per tensor-memory lane quarter: group q = gate rows i0+16q .. +15, then
//   the up rows of the same 16 intermediates. A warp thus finds gate and up
//   of one intermediate in lanes l and l + 16 of its own quarter, and
//   SiLU(gate) * up needs one exchange of 16 values by shuffle. The four
//   groups come in with one 5-D TMA box per stage (the weight viewed as
//   [E][gate|up][I/16][16][H]).
//   down: an m-tile covers 256 rows of H; CTA r holds 128 of them. The
//   epilogue multiplies by the routing weight and adds into the fp32 output
//   accumulator with 16-byte vector reductions ("mini-sglang guide, chapter
//   7": expert outputs weighted by their softmax scores and summed).
//
// Roles per CTA (480 threads): warps 0 and 10-14 = TMA producers, one per
// ring slot (each CTA loads its own halves; the bytes are counted on the
// leader CTA's barrier), warp 1 = tensor-memory allocation (both CTAs) and
// MMA issue (leader only), warps 2-9 = epilogue on the CTA's own tensor
// memory (two warps per lane quarter, alternate 32-column chunks). Two accumulator buffers of 256
// columns let the epilogue of one tile overlap the main loop of the next.
// Every wait is bounded (1 s): a wait that runs out records MM_ERR_TIMEOUT,
// the abort is mirrored to the peer CTA, and all roles unwind; the MMA
// thread waits for its MMAs and both CTAs free their tensor memory.
#include "mm.h"
#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

constexpr int kPK = 64;                  // K per stage: one 128-byte swizzle row of bf16
constexpr int kPStages = 6;
constexpr int kPEpiWarp0 = 2, kPEpiWarps = 8;
constexpr int kPProd0 = kPEpiWarp0 + kPEpiWarps;           // 10: producers of slots 1..5
constexpr int kPThreads = (kPProd0 + kPStages - 1) * 32;     // 480
constexpr int kPMaxN = 256;              // token rows per pair tile (half per CTA)
constexpr int kPBox = 16;                // token rows per TMA box
constexpr int kPABytes = 128 * kPK * 2;  // 16 KB: this CTA's 128 weight rows
constexpr int kPBBytes = (kPMaxN / 2) * kPK * 2;  // 16 KB: up to 128 token rows
constexpr int kPStageBytes = kPABytes + kPBBytes;
constexpr int kPEpiTok = 16;             // tokens per down-epilogue transpose step
constexpr int kPEpiBytes = kPEpiWarps * kPEpiTok * 33 * 4;
constexpr int kPSmemBytes = kPStages * kPStageBytes + kPEpiBytes + 1024;
constexpr uint32_t kPTmemCols = 2 * kPMaxN;  // two accumulator buffers
static_assert(kPSmemBytes <= 227 * 1024 - 4096, "shared memory (static arrays need ~3.2 KB)");

// How gate_up's weight rows reach shared memory.
constexpr int kAOneBox = 0;     // one 5-D box: four groups of (16 gate, 16 up) rows
constexpr int kASixteen = 1;    // eight 2-D boxes of 16 rows (same layout)

struct PairArgs {
  const int32_t* sorted;   // [capacity]
  const int32_t* offsets;  // [E+1]
  const float* topk_w;     // [T*k] (down mode)
  void* C;                 // act bf16 [capacity, N] | acc fp32 [T, N]
  unsigned* err;
  float* zero_buf;         // gate_up: zero these floats first (the layer's accumulator)
  long long zero_count;
  int E, N, K, Tk, top_k;
  int n_mtiles;  // m-tiles per token chunk
  int w_rows;    // weight rows per expert in the 2-D weight view
  int a_mode;    // gate_up A path (kAOneBox / kASixteen)
};

__device__ __forceinline__ uint32_t pair_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void pair_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address, in CTA `rank` of the cluster, of the shared variable at `local`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem of both CTAs] (+)= A (128 rows in each CTA) * B (N/2 rows in each
// CTA)^T; issued by one thread of the leader CTA.
__device__ __forceinline__ void umma_pair_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One arrival on the barrier at CTA offset `bar` in every CTA of `mask` once
// the pair MMAs issued so far have completed.
__device__ __forceinline__ void umma_pair_commit(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// Box loads into this CTA's shared memory whose completion is counted on
// `bar`, a barrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* map, uint32_t bar,
                                                 int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const void* map, uint32_t bar,
                                                 int c0, int c1, int c2, int c3, int c4,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(c4), "l"(policy)
      : "memory");
}

// Announces `bytes` of TMA traffic on a barrier of either CTA of the pair.
// Relaxed: the producer publishes no data of its own here (the bytes are
// tracked by the copies' complete_tx), and a release would make the thread
// wait for its earlier copies.
__device__ __forceinline__ void mbar_expect_tx_cluster(uint32_t cluster_bar, uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(
          cluster_bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

struct PairTable {
  int off[kMaxExperts + 1];
  int cs[kMaxExperts + 1];  // first chunk of each expert
  int csz[kMaxExperts];     // rows per chunk of each expert
};

__device__ __forceinline__ void decode_pair_tile(int tile, int n_mtiles, int E, const PairTable& P,
                                                 int& e, int& m, int& row0, int& nrows) {
  const int ch = tile / n_mtiles;
  m = tile - ch * n_mtiles;
  int lo = 0, hi = E;  // P.cs[lo] <= ch < P.cs[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (P.cs[mid] <= ch)
      lo = mid;
    else
      hi = mid;
  }
  e = lo;
  row0 = P.off[e] + (ch - P.cs[e]) * P.csz[e];
  nrows = min(P.csz[e], P.off[e + 1] - row0);
}

template <int MODE>
__global__ void __launch_bounds__(kPThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmW,
                             const __grid_constant__ CUtensorMap tmX, const PairArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kPStages + 5];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ PairTable P;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E;
  const uint32_t rank = pair_rank();  // 0 = leader (issues the MMAs)
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  // The fp32 accumulator that the down GEMM of this call adds into is cleared
  // here, before the wait: its last reader (the previous call's finalize)
  // completed before this call's first kernel started.
  if (a.zero_buf != nullptr) {
    float4* z = reinterpret_cast<float4*>(a.zero_buf);
    const long long n4 = a.zero_count >> 2;
    for (long long i = (long long)blockIdx.x * kPThreads + tid; i < n4;
         i += (long long)gridDim.x * kPThreads)
      z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();  // the grouping and the token rows come from the kernels before
  pdl_trigger();

  // Chunk table: ceil(L / 256) chunks of near-equal size per expert.
  for (int i = tid; i <= E; i += kPThreads) P.off[i] = a.offsets[i];
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32, e0 = lane * per;
    int sum = 0;
    for (int j = 0; j < per; ++j) {
      const int e = e0 + j;
      if (e < E) sum += (P.off[e + 1] - P.off[e] + kPMaxN - 1) / kPMaxN;
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
        const int L = P.off[e + 1] - P.off[e];
        const int nch = (L + kPMaxN - 1) / kPMaxN;
        P.cs[e] = run;
        P.csz[e] = nch > 0 ? ((L + nch - 1) / nch + 15) / 16 * 16 : 0;
        run += nch;
      }
    }
    if (lane == 31) P.cs[E] = incl;
  }
  __syncthreads();
  const int total_tiles = P.cs[E] * a.n_mtiles;
  if (pair >= total_tiles) return;  // the same in both CTAs: no cluster barrier is skipped

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t smem_base = (raw_addr + 1023u) & ~1023u;
  float* epi_tile =
      reinterpret_cast<float*>(smem_raw + (smem_base - raw_addr) + kPStages * kPStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + kPStages;
  uint64_t* tfull = empty + kPStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;

  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(smem_u32(&full[s]), 2);   // each CTA's producer announces its own bytes
      mbar_init(smem_u32(&empty[s]), 1);  // the leader's MMA commit, multicast to both CTAs
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 2 * kPEpiWarps);  // every epilogue warp of both CTAs
    }
    mbar_init(smem_u32(done), 1);
    abort_s = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_base_s), kPTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  pair_sync();  // both CTAs' barriers initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;
  const uint32_t peer_abort = peer_addr(smem_u32(&abort_s), rank ^ 1u);
  auto fail = [&]() {
    *reinterpret_cast<volatile int*>(&abort_s) = 1;
    st_cluster_u32(peer_abort, 1u);
    atomicOr(a.err, kDevErrTimeout);
  };
  auto aborted_p = [&]() { return *reinterpret_cast<volatile int*>(&abort_s) != 0; };
  const int nk = a.K / kPK;

  if (warp == 0 || warp >= kPProd0) {
    // ------------------------------------------------ TMA producers ---
    // One warp per ring slot (slot 0: warp 0, slot s: warp kPProd0 + s - 1):
    // a warp's TMA loads that signal another barrier than its previous ones
    // wait for those to land, so one warp per slot keeps all stages in flight.
    const int slot = warp == 0 ? 0 : warp - kPProd0 + 1;
    if (lane == 0 && slot < kPStages) {
      // Weights: read by every chunk of the expert, so kept at normal
      // priority when the expert has several chunks, and marked first to go
      // when it has one (read once: then they make room for the token rows
      // and the accumulator instead of pushing those out).
      const uint64_t pol_w_multi = l2_policy_evict_normal();
      const uint64_t pol_w_once = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();    // read by every m-tile of the chunk
      uint32_t use = 0;  // fills of this warp's slot so far
      int q = 0;         // K step counter of this pair, modulo the ring size
      bool ok = true;
      for (int tile = pair; tile < total_tiles && ok; tile += npairs) {
        if (aborted_p()) break;
        int e, m, row0, nrows;
        decode_pair_tile(tile, a.n_mtiles, E, P, e, m, row0, nrows);
        const int nh = ((nrows + 15) & ~15) / 2;  // this CTA's token rows (a multiple of 8)
        const int brow = row0 + (int)rank * nh;
        const int nbox = (nh + kPBox - 1) / kPBox;
        const uint32_t bytes = kPABytes + nbox * kPBox * kPK * 2;
        const uint64_t pol_w = P.cs[e + 1] - P.cs[e] > 1 ? pol_w_multi : pol_w_once;
        for (int kb = 0; kb < nk; ++kb) {
          const bool mine = q == slot;
          if (++q == kPStages) q = 0;
          if (!mine) continue;
          if (!mbar_wait(smem_u32(&empty[slot]), (use & 1u) ^ 1u)) {
            fail();
            ok = false;
            break;
          }
          const uint32_t st = smem_base + slot * kPStageBytes;
          const uint32_t fb = peer_addr(smem_u32(&full[slot]), 0);  // the leader's barrier
          mbar_expect_tx_cluster(fb, bytes);                         // before this CTA's loads
          const int kc = kb * kPK;
          if (MODE == MM_GEMM_GATE_UP) {
            const int g0 = m * 8 + (int)rank * 4;  // this CTA's first group of 16 intermediates
            if (a.a_mode == kAOneBox) {
              // coordinates {k, row in group, gate|up, group, expert}
              tma_load_5d_pair(st, &tmW, fb, kc, 0, 0, g0, e, pol_w);
            } else {
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                const int r = e * a.w_rows + 16 * (g0 + g);
                tma_load_2d_pair(st + g * 4096, &tmW, fb, kc, r, pol_w);
                tma_load_2d_pair(st + g * 4096 + 2048, &tmW, fb, kc, r + a.N, pol_w);
              }
            }
          } else {
            tma_load_2d_pair(st, &tmW, fb, kc, e * a.w_rows + m * 256 + (int)rank * 128, pol_w);
          }
          for (int j = 0; j < nbox; ++j)
            tma_load_2d_pair(st + kPABytes + j * (kPBox * kPK * 2), &tmX, fb, kc,
                             brow + j * kPBox, pol_x);
          ++use;
        }
      }
      if (!ok || aborted_p()) {
        // Copies issued just before the abort may still be landing in this
        // CTA's shared memory: give them time (a TMA load completes within
        // microseconds) before the CTA can exit.
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 50000ull) {
        }
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
        decode_pair_tile(tile, a.n_mtiles, E, P, e, m, row0, nrows);
        const int b = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait(smem_u32(&tempty[b]), (use & 1u) ^ 1u)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(256, (nrows + 15) & ~15);
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
            umma_pair_bf16(d, sdesc_kmajor<128>(st + kk * 32),
                           sdesc_kmajor<128>(st + kPABytes + kk * 32), idesc,
                           (kb | kk) != 0 ? 1u : 0u);
          umma_pair_commit(smem_u32(&empty[s]), 0x3);  // frees stage s in both CTAs
          if (++s == kPStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_pair_commit(smem_u32(&tfull[b]), 0x3);  // accumulator b complete in both CTAs
      }
      // Every MMA issued above has finished before tensor memory is freed.
      umma_pair_commit(smem_u32(done), 0x1);
      if (!mbar_wait(smem_u32(done), 0)) fail();
    }
    __syncwarp();
  } else if (warp >= kPEpiWarp0 && warp < kPProd0) {
    // ---------------------------------------------------------- epilogue ---
    const int ew = warp - kPEpiWarp0;  // 0..7
    const int q = warp & 3;            // tensor-memory lane quarter this warp may read
    const int side = ew >> 2;          // takes 32-column chunks side, side + 2, ...
    constexpr int kCh = kPMaxN / 64;   // chunks per side
    const uint32_t tempty_leader0 = peer_addr(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_leader1 = peer_addr(smem_u32(&tempty[1]), 0);
    float* tr = epi_tile + ew * kPEpiTok * 33;  // [kPEpiTok][32 + 1 pad]
    const uint64_t pol_acc = l2_policy_evict_last();
    int it = 0;
    for (int tile = pair; tile < total_tiles; tile += npairs, ++it) {
      if (aborted_p()) break;
      int e, m, row0, nrows;
      decode_pair_tile(tile, a.n_mtiles, E, P, e, m, row0, nrows);
      const int b = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      // Down mode: lane j holds the slot id and routing weight of column j of
      // each of this warp's chunks, loaded before the wait so that their
      // latency hides behind the tile's main loop.
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
#pragma unroll
      for (int i = 0; i < kCh; ++i) {
        const int c0 = (2 * i + side) * 32;
        if (c0 >= nrows) break;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tb + c0, v);
        tmem_wait_ld();
        const int ncol = min(32, nrows - c0);
        if (MODE == MM_GEMM_GATE_UP) {
          // Lanes 0-15 hold gate, lanes 16-31 up of the same 16 intermediate
          // rows, for 32 token columns. Lane l < 16 finishes columns 0-15,
          // lane l + 16 columns 16-31: each sends the 16 values the other
          // needs.
          const bool is_gate = lane < 16;
          const int i_out = m * 128 + (int)rank * 64 + q * 16 + (lane & 15);
          float x[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            x[j] = __shfl_xor_sync(0xffffffffu, __uint_as_float(is_gate ? v[16 + j] : v[j]), 16);
          if (i_out < a.N) {
            const int cb = is_gate ? 0 : 16;
            uint16_t* dst = static_cast<uint16_t*>(a.C) + (size_t)(row0 + c0 + cb) * a.N + i_out;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (cb + j < ncol) {
                const float gv = is_gate ? __uint_as_float(v[j]) : x[j];
                const float uv = is_gate ? x[j] : __uint_as_float(v[16 + j]);
                // silu(g) * u; the fast divide (about 2 ulp) is far below
                // the bf16 rounding of the result, and for g < -87.3 it
                // returns 0 for a |silu(g)| under 1.1e-36.
                dst[(size_t)j * a.N] =
                    f32_to_bf16_bits(__fdividef(gv, 1.0f + __expf(-gv)) * uv);
              }
            }
          }
        } else {
          // Lane = output row h; columns = tokens. The weighted values pass
          // through this warp's shared tile (row = token), kPEpiTok tokens
          // at a time, so that each lane adds 4 consecutive outputs of one
          // token with one 16-byte vector reduction.
          const int f_l = f_t[i];
          const float w_l = w_t[i];
          const int t_l = f_l / a.top_k;
          float* accp = static_cast<float*>(a.C);
          const int hb = m * 256 + (int)rank * 128 + q * 32;  // first h of this warp's rows
          const int h4 = (lane & 7) * 4;
#pragma unroll
          for (int grp = 0; grp < 32 / kPEpiTok; ++grp) {
            __syncwarp();
#pragma unroll
            for (int j = 0; j < kPEpiTok; ++j) {
              const int jj = grp * kPEpiTok + j;
              const float wt = __shfl_sync(0xffffffffu, w_l, jj);
              tr[j * 33 + lane] = wt * __uint_as_float(v[jj]);
            }
            __syncwarp();
#pragma unroll
            for (int s4 = 0; s4 < kPEpiTok / 4; ++s4) {
              const int jl = s4 * 4 + (lane >> 3);  // token within the group
              const int jt = grp * kPEpiTok + jl;
              const int f = __shfl_sync(0xffffffffu, f_l, jt);
              const int t = __shfl_sync(0xffffffffu, t_l, jt);
              if (jt < ncol && f < a.Tk && hb + h4 < a.N) {
                const float* vv = tr + jl * 33 + h4;
                red_add_v4_f32(accp + (size_t)t * a.N + hb + h4, vv[0], vv[1], vv[2], vv[3],
                               pol_acc);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(b == 0 ? tempty_leader0 : tempty_leader1);
    }
  }

  tc_fence_before();
  __syncthreads();
  pair_sync();  // both CTAs are done with tensor memory and with each other's barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPTmemCols);
  }
}

template <int MODE>
cudaError_t launch_pair_mode(const uint16_t* X, const uint16_t* W, void* C,
                             const int32_t* sorted, const int32_t* offsets, const float* topk_w,
                             int T, int top_k, int E, int N, int K, long long capacity,
                             long long x_rows, int num_sms, unsigned* err, bool after_prev,
                             cudaStream_t st, float* zero_buf, long long zero_count) {
  static DeviceFlags attr_done;
  if (cudaError_t e = smem_attr_once(attr_done, grouped_gemm_pair_kernel<MODE>, kPSmemBytes);
      e != cudaSuccess)
    return e;
  PairArgs a;
  a.sorted = sorted;
  a.offsets = offsets;
  a.topk_w = topk_w;
  a.C = C;
  a.err = err;
  a.zero_buf = zero_buf;
  a.zero_count = zero_buf != nullptr ? zero_count : 0;
  a.E = E;
  a.N = N;
  a.K = K;
  a.Tk = T * top_k;
  a.top_k = top_k;
  a.a_mode = kAOneBox;
  CUtensorMap tmW, tmX;
  if (MODE == MM_GEMM_GATE_UP) {
    a.w_rows = 2 * N;
    a.n_mtiles = (N + 127) / 128;
    // w_gate_up [E][2][N/16][16][K] (gate rows, then up rows, of each expert):
    // one box = 4 groups x (16 gate rows, 16 up rows) x 64 of K.
    const uint64_t dims[5] = {(uint64_t)K, 16, 2, (uint64_t)N / 16, (uint64_t)E};
    const uint64_t strides[4] = {(uint64_t)K * 2, (uint64_t)N * K * 2, (uint64_t)16 * K * 2,
                                 (uint64_t)2 * N * K * 2};
    const uint32_t box[5] = {kPK, 16, 2, 4, 1};
    if (!make_tensor_map_sw128(&tmW, W, 5, dims, strides, box)) {
      // The same rows in eight 16-row boxes of the plain [E * 2N, K] view.
      a.a_mode = kASixteen;
      if (!make_tensor_map_2d(&tmW, W, (uint64_t)E * a.w_rows, (uint64_t)K, 16, kPK))
        return cudaErrorInvalidValue;
    }
  } else {
    a.w_rows = N;
    a.n_mtiles = (N + 255) / 256;
    if (!make_tensor_map_2d(&tmW, W, (uint64_t)E * a.w_rows, (uint64_t)K, 128, kPK))
      return cudaErrorInvalidValue;
  }
  if (!make_tensor_map_2d(&tmX, X, (uint64_t)x_rows, (uint64_t)K, kPBox, kPK))
    return cudaErrorInvalidValue;
  // Chunks: sum over experts of ceil(L_e / 256) <= E + capacity / 256.
  const long long max_tiles = ((capacity + kPMaxN - 1) / kPMaxN + E) * (long long)a.n_mtiles;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPThreads, 1, 1);
  cfg.dynamicSmemBytes = kPSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Persistent pairs: as many as can be resident at once (pairs of SMs of
  // one GPC), so that no pair waits for another to finish its tiles.
  static std::atomic<int> resident[kMaxDevices];
  const int dev = current_device();
  int max_pairs = resident[dev].load(std::memory_order_relaxed);
  if (max_pairs <= 0) {
    cfg.gridDim = dim3((unsigned)num_sms, 1, 1);
    if (cudaOccupancyMaxActiveClusters(&max_pairs, grouped_gemm_pair_kernel<MODE>, &cfg) !=
            cudaSuccess ||
        max_pairs <= 0) {
      cudaGetLastError();
      max_pairs = num_sms / 2;
    }
    resident[dev].store(max_pairs, std::memory_order_relaxed);
  }
  long long pairs = max_pairs;
  if (pairs > max_tiles) pairs = max_tiles;
  if (pairs < 1) pairs = 1;
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.numAttrs = after_prev ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<MODE>, tmW, tmX, a);
}

}  // namespace

cudaError_t launch_grouped_gemm_pair(int mode, const uint16_t* X, const uint16_t* W, void* C,
                                     const int32_t* sorted, const int32_t* offsets,
                                     const float* topk_w, int T, int top_k, int E, int N, int K,
                                     long long capacity, long long x_rows, int num_sms,
                                     unsigned* err, bool after_prev, cudaStream_t st,
                                     float* zero_buf, long long zero_count) {
  if (mode == MM_GEMM_GATE_UP)
    return launch_pair_mode<MM_GEMM_GATE_UP>(X, W, C, sorted, offsets, topk_w, T, top_k, E, N, K,
                                             capacity, x_rows, num_sms, err, after_prev, st,
                                             zero_buf, zero_count);
  return launch_pair_mode<MM_GEMM_DOWN>(X, W, C, sorted, offsets, topk_w, T, top_k, E, N, K,
                                        capacity, x_rows, num_sms, err, after_prev, st, nullptr,
                                        0);
}

}  // namespace mm
