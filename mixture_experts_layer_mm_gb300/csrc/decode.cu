// The MoE layer for small batches (T <= 64 tokens) in one launch.
//
// With a handful of tokens the layer is a stream of the selected experts'
// weights ("mini-sglang guide, chapter 7", paragraph on moe/fused.py: each
// selected expert's weights read once, in one kernel call), and what costs
// time besides that stream is latency: the router's dependent steps and the
// boundaries between the kernels of a multi-launch layer. Here one
// cooperative grid (one CTA per SM) runs every step, with three grid-wide
// barriers:
//   A  zero the fp32 sum; router logits, one expert per CTA at a time
//      (fp32 dot products of the token rows with the expert's router row)
//   -- barrier 0
//   B  every CTA reads all logits and finishes every token itself (softmax
//      over all experts, top-k, weights: the router's per-token finish), then
//      groups the assignments by expert in shared memory. No hand-off is
//      needed: all CTAs compute the same grouping. Each CTA also writes its
//      share of the workspace's routing and grouping (as mm_route/mm_align).
//   C  gate_up: units (expert, 8 intermediates) = 8 gate rows and the same 8
//      up rows, full K. One producer warp streams each unit's 16 weight rows
//      into a ring of shared-memory slots with bulk async copies; 8 consumer
//      warps split K, multiply with warp MMAs (m16n8k16: the 16 weight rows x
//      8 of the expert's tokens), add their partial sums in shared memory
//      and write act = bf16(silu(gate) * up) for the unit's 8 intermediates.
//   -- barrier 1 (every act row complete)
//   D  down: units (expert, 16 output rows), full K = I, two units per slot
//      (4 warps each); the routing weight scales each token's result, which
//      is added (fp32 vector atomics) into the layer's sum.
//   -- barrier 2
//   E  out = bf16(sum) (and the residual add after the layer, if asked).
// The producer runs ahead of the consumers through barrier 1: while the
// grid waits there, the ring is already filling with down-projection
// weights. The weights take the M side of the MMA (swap-AB), so one expert
// with up to 8 tokens costs one m16n8 tile per 16 weight rows, and gate and
// up rows of the same intermediates share a tile, so SiLU(gate) * up is
// formed from one lane's accumulators.
//
// A lane (g, q) of an MMA reads 16 bytes (8 consecutive bf16) of weight rows
// g and g + 8 at column 8q of each 32-column step, and 16 bytes of its
// token's row at the same columns; the two MMAs of the step take words
// {0, 1} and {2, 3} as k = {2q, 2q+1} and {2q+8, 2q+9}. That is a fixed
// permutation of the step's 32 columns applied to both operands alike, so
// the dot products are unchanged and no shuffle is needed.
//
// Grid barriers: at barrier 0 each CTA writes the call's epoch (a
// per-launch 64-bit value) into its own flag, then polls all CTAs' flags
// until every one holds the epoch; flags never need clearing (a new call
// brings a new epoch). Barriers 1 and 2 count arrivals on one word each,
// zeroed before barrier 0. Every wait is bounded: after about a second a CTA
// records MM_ERR_TIMEOUT and leaves, the producer first waiting for the
// copies it has in flight.
#include <math.h>

#include <atomic>
#include <chrono>

#include "mm_device.cuh"
#include "mm_internal.h"
#include "route_finish.cuh"

namespace mm {
namespace {

constexpr int kCW = 8;                   // consumer warps
constexpr int kDecThreads = (kCW + 1) * 32;  // + the producer warp (warp kCW)
constexpr int kDecMaxT = 64;             // token sets are 64-bit masks
constexpr int kDecMaxTk = 512;           // assignments per call
constexpr int kDecAutoMaxT = 16;         // mm_moe_forward takes the single launch up to here
constexpr int kSlots = 3;
constexpr int kSlotBytes = 64 * 1024;    // one gate_up unit or two down units
constexpr int kRingBytes = kSlots * kSlotBytes;
constexpr int kGroupsPerPass = 4;        // token groups of 8 per pass over a slot
constexpr int kRedBytes = kCW * kGroupsPerPass * 32 * 16;  // partial sums
constexpr int kDecBarriers = 3;
constexpr int kDecMaxGrid = 256;         // flag slots per barrier
constexpr int kFillEnd = -1;             // control words of a ring fill
constexpr int kFillStop = -2;

struct DecodeArgs {
  const uint16_t* hidden;    // [T, H]
  const uint16_t* router_w;  // [E, H]
  const float* bias;         // [E] or NULL
  const uint16_t* w_gate_up; // [E, 2I, H]
  const uint16_t* w_down;    // [E, H, I]
  int T, H, E, I, k, renorm;
  float* logits;             // [T, E]
  int32_t* ids;              // [T*k]
  float* w;                  // [T*k]
  int32_t* sorted;           // [capacity], segments padded to kForwardBlockM
  int32_t* offsets;          // [E+1]
  int32_t* counts;           // [E]
  long long capacity;
  uint16_t* act;             // [T*k, I] bf16, per assignment
  float* acc;                // [T, H] fp32: the layer's sum (a partial of a TP slice)
  uint16_t* out;             // [T, H] bf16, or NULL (the sum is the result)
  const uint16_t* res_in;    // residual add after the layer: res_out = bf16(out + res_in)
  uint16_t* res_out;
  unsigned long long* flags; // [kDecBarriers, kDecMaxGrid], then 4 u32 counters
  unsigned long long epoch;
  unsigned* err;
  int absent_cta, absent_barrier;  // self-test: that CTA skips that barrier's arrival
};

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// The consumer warps' own barrier (the producer warp does not take part).
__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory");
}
// One half of the consumers (4 warps) in the down phase.
__device__ __forceinline__ void group_bar(int grp) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + grp), "n"(4 * 32) : "memory");
}

// Called by one warp after its CTA's threads have arrived at a CTA barrier:
// publishes the CTA's arrival at grid barrier b and waits (bounded) for all
// CTAs. Returns whether all arrived; lane 0 records a timeout.
__device__ __forceinline__ bool grid_wait_warp(const DecodeArgs& a, int b) {
  const int lane = threadIdx.x & 31;
  unsigned long long* f = a.flags + (size_t)b * kDecMaxGrid;
  if (lane == 0 && !((int)blockIdx.x == a.absent_cta && b == a.absent_barrier)) {
    __threadfence();
    st_release_u64(f + blockIdx.x, a.epoch);
  }
  const uint64_t t0 = global_timer_ns();
  bool done = false, timed_out = false;
  while (!done && !timed_out) {
    bool mine = true;
    // relaxed loads, all in flight together; one acquire fence after
    for (int c = lane; c < (int)gridDim.x; c += 32) mine &= ld_relaxed_u64(f + c) == a.epoch;
    done = __all_sync(0xffffffffu, mine);
    if (!done) timed_out = __shfl_sync(0xffffffffu, global_timer_ns() - t0 > kWaitLimitNs, 0);
  }
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  if (!done && lane == 0) atomicOr(a.err, kDevErrTimeout);
  return done;
}

// Grid barriers 1 and 2: an arrival counter each (zeroed before grid
// barrier 0, so the zero is seen by everyone). Called by one warp after its
// CTA's threads have arrived at a CTA barrier: lane 0 adds the CTA's arrival
// and polls the one counter word until all CTAs have arrived (bounded). One
// word polled by one lane per CTA keeps the L2 traffic of the wait small,
// which matters while the weight stream keeps the memory system busy.
__device__ __forceinline__ bool grid_count_wait(const DecodeArgs& a, unsigned* c, int b) {
  const int lane = threadIdx.x & 31;
  bool done = false;
  if (lane == 0) {
    if (!((int)blockIdx.x == a.absent_cta && b == a.absent_barrier)) {
      __threadfence();
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(c) : "memory");
    }
    const uint64_t t0 = global_timer_ns();
    while (true) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
      if (v >= gridDim.x) {
        done = true;
        break;
      }
      if (global_timer_ns() - t0 > kWaitLimitNs) break;
    }
    if (!done) atomicOr(a.err, kDevErrTimeout);
  }
  return __shfl_sync(0xffffffffu, done ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Token rows: hidden is read-only for the whole launch (non-coherent path);
// act was written earlier in this launch and is read after grid barrier 1,
// whose acquire orders these plain loads after the writes.
template <bool kReadOnly>
__device__ __forceinline__ uint4 ld_row16(const uint16_t* p) {
  if (p == nullptr) return make_uint4(0u, 0u, 0u, 0u);
  return kReadOnly ? __ldg(reinterpret_cast<const uint4*>(p))
                   : *reinterpret_cast<const uint4*>(p);
}

// One warp's share of a unit: 16 weight rows in shared memory (row g at
// a_lo + g * row_bytes, row g + 8 at a_hi + g * row_bytes; both already
// offset by the warp's first column) times NG groups of 8 token rows
// (xrow[n]: the lane's token row of group n, offset likewise, or NULL),
// over nsteps 32-column steps. d[n]: rows g and g + 8, tokens 2q, 2q + 1.
template <int NG, bool kReadOnly>
__device__ __forceinline__ void warp_unit_mma(uint32_t a_lo, uint32_t a_hi,
                                              const uint16_t* const (&xrow)[kGroupsPerPass],
                                              int nsteps, float (&d)[kGroupsPerPass][4]) {
  // kU steps at a time, all their token-row loads issued first: the rows
  // may come from L2 (act, first use), and one round trip then covers kU
  // steps
  constexpr int kU = NG <= 2 ? 4 : 2;
  for (int s0 = 0; s0 < nsteps; s0 += kU) {
    uint4 b[kU][NG];
#pragma unroll
    for (int u = 0; u < kU; ++u)
#pragma unroll
      for (int n = 0; n < NG; ++n)
        b[u][n] = ld_row16<kReadOnly>((xrow[n] && s0 + u < nsteps) ? xrow[n] + 32 * (s0 + u)
                                                                   : nullptr);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (s0 + u >= nsteps) break;
      const uint4 lo = lds128(a_lo + 64 * (s0 + u)), hi = lds128(a_hi + 64 * (s0 + u));
#pragma unroll
      for (int n = 0; n < NG; ++n) {
        mma16816(d[n], lo.x, hi.x, lo.y, hi.y, b[u][n].x, b[u][n].y);
        mma16816(d[n], lo.z, hi.z, lo.w, hi.w, b[u][n].z, b[u][n].w);
      }
    }
  }
}

template <bool kReadOnly>
__device__ __forceinline__ void warp_unit_mma_n(int ng, uint32_t a_lo, uint32_t a_hi,
                                                const uint16_t* const (&xrow)[kGroupsPerPass],
                                                int nsteps, float (&d)[kGroupsPerPass][4]) {
  if (ng <= 1) warp_unit_mma<1, kReadOnly>(a_lo, a_hi, xrow, nsteps, d);
  else if (ng == 2) warp_unit_mma<2, kReadOnly>(a_lo, a_hi, xrow, nsteps, d);
  else if (ng == 3) warp_unit_mma<3, kReadOnly>(a_lo, a_hi, xrow, nsteps, d);
  else warp_unit_mma<4, kReadOnly>(a_lo, a_hi, xrow, nsteps, d);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  // silu(g) * u; the fast divide (about 2 ulp) is far below the bf16
  // rounding of the result.
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

struct Routing {
  unsigned long long* mask;  // [E] tokens that picked e (bit t)
  int* cnt;                  // [E]
  int* start;                // [E+1] unpadded exclusive scan of cnt
  int* offp;                 // [E+1] scan of cnt padded to kForwardBlockM
  int* act_e;                // [E] experts with cnt > 0, ascending
  int* ids;                  // [T*k]
  float* w;                  // [T*k]
  int* slots;                // [T*k] assignments grouped by expert, stable
};

__host__ __device__ constexpr size_t routing_smem_bytes(int E, int Tk) {
  return (size_t)E * 8 + (size_t)(E + 2 * (E + 1) + E) * 4 + (size_t)Tk * 12;
}

__device__ __forceinline__ Routing carve_routing(unsigned char* p, int E, int Tk) {
  Routing r;
  r.mask = reinterpret_cast<unsigned long long*>(p);
  r.cnt = reinterpret_cast<int*>(r.mask + E);
  r.start = r.cnt + E;
  r.offp = r.start + E + 1;
  r.act_e = r.offp + E + 1;
  r.ids = r.act_e + E;
  r.w = reinterpret_cast<float*>(r.ids + Tk);
  r.slots = reinterpret_cast<int*>(r.w + Tk);
  return r;
}

// Every warp of the CTA finishes tokens NT at a time (warp w: tokens
// w*NT .. w*NT + NT - 1, then the next round of all warps), writing the
// routing into ids / w.
template <int Q, int NT>
__device__ __forceinline__ void finish_all(const DecodeArgs& a, int* ids, float* w) {
  constexpr int W = kCW + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t0 = warp * NT; t0 < a.T; t0 += W * NT) {
    float l[NT][Q];
    int tt[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int t = t0 + i;
      tt[i] = t < a.T ? t : -1;
#pragma unroll
      for (int qq = 0; qq < Q; ++qq) {
        const int e = lane + 32 * qq;
        l[i][qq] = (t < a.T && e < a.E) ? __ldcg(a.logits + (size_t)t * a.E + e) : -INFINITY;
      }
    }
    routefin::finish_tokens<Q, NT>(l, tt, a.E, a.k, a.renorm, ids, w);
  }
}

template <int Q>
__global__ void __launch_bounds__(kDecThreads, 1) moe_decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full_bar[kSlots];
  __shared__ __align__(8) uint64_t empty_bar[kSlots];
  __shared__ int ok_s, nact_s;
  __shared__ int wsum_s[kMaxExperts / 32][3];
  __shared__ volatile int abort_s;
  __shared__ volatile int ctl_s[2];
  __shared__ volatile int fill_unit[kSlots];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int Tk = a.T * a.k;
  const uint32_t ring = smem_u32(smem);
  float4* red = reinterpret_cast<float4*>(smem + kRingBytes);
  const Routing R = carve_routing(smem + kRingBytes + kRedBytes, a.E, Tk);

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kCW);
    }
    fence_barrier_init();
    abort_s = 0;
    if (blockIdx.x == 0) {  // the work and arrival counters (read after grid barrier 0)
      unsigned* c = reinterpret_cast<unsigned*>(a.flags + kDecBarriers * kDecMaxGrid);
      c[0] = 0u;
      c[1] = 0u;
      c[2] = 0u;
      c[3] = 0u;
    }
  }
  pdl_wait();

  // ---- A: zero the sum; router logits, expert e on CTA e % G
  {
    const long long gtid = (long long)blockIdx.x * kDecThreads + tid;
    const long long gstride = (long long)G * kDecThreads;
    float4* z = reinterpret_cast<float4*>(a.acc);
    const long long n4 = (long long)a.T * a.H / 4;
    for (long long i = gtid; i < n4; i += gstride) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // warp w: tokens w, w + 9, ...; H / 256 <= 8 16-byte loads per lane and
  // operand, all issued before the sums
  for (int e = blockIdx.x; e < a.E; e += G) {
    const uint4* wr = reinterpret_cast<const uint4*>(a.router_w + (size_t)e * a.H);
    for (int t = warp; t < a.T; t += kCW + 1) {
      const uint4* xr = reinterpret_cast<const uint4*>(a.hidden + (size_t)t * a.H);
      const int nc = a.H / 256;
      uint4 x[8], r[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (c < nc) {
          x[c] = __ldg(xr + lane + 32 * c);
          r[c] = __ldg(wr + lane + 32 * c);
        }
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (c < nc) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t xw = word(x[c], i), rw = word(r[c], i);
            s = fmaf(__uint_as_float(xw << 16), __uint_as_float(rw << 16), s);
            s = fmaf(__uint_as_float(xw & 0xFFFF0000u), __uint_as_float(rw & 0xFFFF0000u), s);
          }
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) a.logits[(size_t)t * a.E + e] = s + (a.bias != nullptr ? a.bias[e] : 0.f);
    }
  }
  __syncthreads();
  if (warp == 0) {
    const bool ok = grid_wait_warp(a, 0);
    if (lane == 0) ok_s = ok ? 1 : 0;
  }
  __syncthreads();
  if (!ok_s) return;

  // ---- B: every CTA finishes every token and groups the assignments
  {
    // NT tokens per warp at a time (their reduction chains interleave); NT
    // is bounded so that NT * Q logits per lane stay in registers
    constexpr int kNTmax = Q >= 8 ? 2 : (Q >= 4 ? 4 : 8);
    const int tpw = (a.T + kCW) / (kCW + 1);
    if (tpw <= 1) {
      finish_all<Q, 1>(a, R.ids, R.w);
    } else if (tpw <= 2 || kNTmax < 4) {
      finish_all<Q, 2>(a, R.ids, R.w);
    } else if constexpr (kNTmax >= 4) {
      if (tpw <= 4 || kNTmax < 8) {
        finish_all<Q, 4>(a, R.ids, R.w);
      } else if constexpr (kNTmax >= 8) {
        finish_all<Q, 8>(a, R.ids, R.w);
      }
    }
  }
  for (int e = tid; e < a.E; e += kDecThreads) R.mask[e] = 0ull;
  __syncthreads();
  for (int i = tid; i < Tk; i += kDecThreads) atomicOr(&R.mask[R.ids[i]], 1ull << (i / a.k));
  __syncthreads();
  {
    // warp w < ceil(E/32) takes experts 32w + lane: counts, the unpadded and
    // the padded scan and the ascending list of selected experts, as
    // warp-local scans and then the warps' totals (conflict-free shared
    // accesses, every warp at once)
    const int nw = (a.E + 31) / 32;
    const int e = warp * 32 + lane;
    int c = 0, pc = 0, ic = 0, ip = 0;
    unsigned bal = 0;
    if (warp < nw) {
      c = e < a.E ? __popcll(R.mask[e]) : 0;
      pc = (c + kForwardBlockM - 1) / kForwardBlockM * kForwardBlockM;
      ic = c;
      ip = pc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, ic, o);
        const int v = __shfl_up_sync(0xffffffffu, ip, o);
        if (lane >= o) {
          ic += u;
          ip += v;
        }
      }
      bal = __ballot_sync(0xffffffffu, c > 0);
      if (lane == 31) {
        wsum_s[warp][0] = ic;
        wsum_s[warp][1] = ip;
        wsum_s[warp][2] = __popc(bal);
      }
    }
    __syncthreads();
    if (warp < nw) {
      int bc = 0, bp = 0, ba = 0;
      for (int w2 = 0; w2 < warp; ++w2) {
        bc += wsum_s[w2][0];
        bp += wsum_s[w2][1];
        ba += wsum_s[w2][2];
      }
      if (e < a.E) {
        R.cnt[e] = c;
        R.start[e] = bc + ic - c;
        R.offp[e] = bp + ip - pc;
        if (c > 0) R.act_e[ba + __popc(bal & ((1u << lane) - 1u))] = e;
      }
      if (warp == nw - 1 && lane == 31) {
        R.start[a.E] = bc + ic;
        R.offp[a.E] = bp + ip;
        nact_s = ba + __popc(bal);
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < Tk; i += kDecThreads) {
    const int e = R.ids[i], t = i / a.k;
    R.slots[R.start[e] + __popcll(R.mask[e] & ((1ull << t) - 1ull))] = i;
  }
  __syncthreads();
  // This CTA's share of the workspace's routing and grouping (tokens t and
  // experts e with t, e = blockIdx.x mod G; the padding tail strided).
  for (int i = tid; i < Tk; i += kDecThreads)
    if ((i / a.k) % G == (int)blockIdx.x) {
      a.ids[i] = R.ids[i];
      a.w[i] = R.w[i];
    }
  for (int e = blockIdx.x; e < a.E; e += G) {
    for (int p = tid; p < R.offp[e + 1] - R.offp[e]; p += kDecThreads)
      a.sorted[R.offp[e] + p] = p < R.cnt[e] ? R.slots[R.start[e] + p] : Tk;
    if (tid == 0) a.counts[e] = R.cnt[e];
  }
  if (blockIdx.x == 0)
    for (int e = tid; e <= a.E; e += kDecThreads) a.offsets[e] = R.offp[e];
  for (long long p = R.offp[a.E] + (long long)blockIdx.x * kDecThreads + tid; p < a.capacity;
       p += (long long)G * kDecThreads)
    a.sorted[p] = Tk;

  // The units: gate_up unit u = (expert act_e[u / (I/8)], intermediates
  // 8 * (u % (I/8)) ..), down pair p = units 2p, 2p + 1, down unit v =
  // (expert act_e[v / (H/16)], output rows 16 * (v % (H/16)) ..). Each CTA
  // takes a contiguous static share of about three quarters of each list (its
  // units mostly of one expert, whose token rows then stay in L1); the rest
  // is handed out one unit (pair) at a time from two counters, so CTAs that
  // stream faster take more and all finish together.
  const int D = nact_s;
  const int gu_per_e = a.I / 8, dn_per_e = a.H / 16;
  const int Ug = D * gu_per_e, Ud = D * dn_per_e, Pd = (Ud + 1) / 2;
  const int sg = (int)((long long)Ug * 3 / 4 / G), sd = (int)((long long)Pd * 3 / 4 / G);
  const uint32_t gu_rows_bytes = 8u * a.H * 2u;   // 8 gate (or up) rows
  const uint32_t dn_unit_bytes = 16u * a.I * 2u;  // 16 rows of w_down[e]
  unsigned* ctr = reinterpret_cast<unsigned*>(a.flags + kDecBarriers * kDecMaxGrid);

  // L1 prefetch of the token rows that this CTA's first gate_up units read
  // (those of the first expert of its static share, up to 32 KB), issued
  // while the first weight copies are in flight: their first loads then hit
  // L1 instead of waiting on L2.
  if (sg > 0) {
    const int e = R.act_e[(blockIdx.x * sg) / gu_per_e];
    const int lines = a.H / 64;  // 128-byte lines of a row
    const int n = min(R.cnt[e] * lines, 256);
    for (int i = tid; i < n; i += kDecThreads)
      prefetch_l1(a.hidden + (size_t)(R.slots[R.start[e] + i / lines] / a.k) * a.H +
                  (i % lines) * 64);
  }

  // ---- producer: fills the ring; fill_unit[slot] tells the consumers what
  // each fill holds (a unit or pair index, or kFillEnd: end of the phase)
  if (warp == kCW) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int i = 0;
      auto acquire = [&](int fill) -> bool {
        if (fill < kSlots) return true;
        const uint32_t bar = smem_u32(&empty_bar[fill % kSlots]);
        const uint32_t par = ((fill / kSlots) - 1) & 1;
        if (mbar_try_wait(bar, par)) return true;
        const uint64_t t0 = global_timer_ns();
        while (true) {
#pragma unroll 1
          for (int r = 0; r < 32; ++r)
            if (mbar_try_wait(bar, par)) return true;
          if (abort_s) return false;
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(a.err, kDevErrTimeout);
            abort_s = 1;
            return false;
          }
        }
      };
      auto issue_gate_up = [&](int u) {
        const int e = R.act_e[u / gu_per_e], i0 = (u % gu_per_e) * 8;
        const uint32_t s = i % kSlots, dst = ring + s * kSlotBytes, bar = smem_u32(&full_bar[s]);
        fill_unit[s] = u;
        mbar_arrive_expect_tx(bar, 2 * gu_rows_bytes);
        bulk_g2s(dst, a.w_gate_up + ((size_t)e * 2 * a.I + i0) * a.H, gu_rows_bytes, bar, pol);
        bulk_g2s(dst + gu_rows_bytes, a.w_gate_up + ((size_t)e * 2 * a.I + a.I + i0) * a.H,
                 gu_rows_bytes, bar, pol);
      };
      auto issue_down = [&](int pr) {
        const int v = 2 * pr, nu = Ud - v < 2 ? Ud - v : 2;
        const uint32_t s = i % kSlots, dst = ring + s * kSlotBytes, bar = smem_u32(&full_bar[s]);
        fill_unit[s] = pr;
        mbar_arrive_expect_tx(bar, nu * dn_unit_bytes);
        for (int j = 0; j < nu; ++j) {
          const int e = R.act_e[(v + j) / dn_per_e], h0 = ((v + j) % dn_per_e) * 16;
          bulk_g2s(dst + j * (kSlotBytes / 2), a.w_down + ((size_t)e * a.H + h0) * a.I,
                   dn_unit_bytes, bar, pol);
        }
      };
      auto mark_end = [&]() {
        const uint32_t s = i % kSlots;
        fill_unit[s] = kFillEnd;
        mbar_arrive(smem_u32(&full_bar[s]));
      };
      bool go = true;
      // Tail claims are made one step ahead: the counter's reply arrives
      // while the producer waits for a free slot, not after it.
      int u_dyn = G * sg + (int)atomicAdd(ctr, 1u);
      for (int u = blockIdx.x * sg; u < (int)(blockIdx.x + 1) * sg && go; ++u)
        if ((go = acquire(i))) issue_gate_up(u), ++i;
      while (go && u_dyn < Ug) {
        const int u_next = G * sg + (int)atomicAdd(ctr, 1u);
        if ((go = acquire(i))) issue_gate_up(u_dyn), ++i;
        u_dyn = u_next;
      }
      int pr_dyn = G * sd + (int)atomicAdd(ctr + 1, 1u);
      if (go && (go = acquire(i))) mark_end(), ++i;
      for (int pr = blockIdx.x * sd; pr < (int)(blockIdx.x + 1) * sd && go; ++pr)
        if ((go = acquire(i))) issue_down(pr), ++i;
      while (go && pr_dyn < Pd) {
        const int pr_next = G * sd + (int)atomicAdd(ctr + 1, 1u);
        if ((go = acquire(i))) issue_down(pr_dyn), ++i;
        pr_dyn = pr_next;
      }
      if (go && (go = acquire(i))) mark_end(), ++i;
      // Every copy lands before the CTA can exit.
      for (int j = i > kSlots ? i - kSlots : 0; j < i; ++j)
        mbar_wait(smem_u32(&full_bar[j % kSlots]), (j / kSlots) & 1);
    }
    return;
  }

  // ---- consumers (warps 0 .. kCW-1)
  const int g = lane >> 2, q = lane & 3;
  int fill = 0;
  // Thread 0 waits for each fill and publishes what it holds (kFillStop
  // when a wait ran out or the CTA is aborting); the consumer barrier after
  // it makes the landed data and the control word visible to all consumers.
  // The word alternates between two slots by fill: thread 0 can write the
  // next fill's word before a slower consumer has read this one, but not the
  // one after (that needs everyone at the next barrier).
  auto next_fill = [&]() -> int {
    if (tid == 0) {
      const bool ok = mbar_wait(smem_u32(&full_bar[fill % kSlots]), (fill / kSlots) & 1);
      if (!ok) {
        atomicOr(a.err, kDevErrTimeout);
        abort_s = 1;
      }
      const int c = fill_unit[fill % kSlots];
      ctl_s[fill & 1] = (ok && !abort_s) ? c : (int)kFillStop;
    }
    consumer_bar();
    return ctl_s[fill & 1];
  };
  auto release = [&](int f) {
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[f % kSlots]));
  };

  // ---- C: gate_up; warp w takes columns [w*H/8, (w+1)*H/8)
  {
    const int kcols = a.H / kCW, nsteps = kcols / 32;
    const uint32_t row_bytes = a.H * 2u;
    while (true) {
      const int u = next_fill();
      if (u == kFillStop) return;
      if (u == kFillEnd) {
        release(fill++);
        break;
      }
      const int e = R.act_e[u / gu_per_e], i0 = (u % gu_per_e) * 8;
      const int cnt = R.cnt[e], base = R.start[e];
      const int ngroups = (cnt + 7) / 8;
      const uint32_t a_lo = ring + (fill % kSlots) * kSlotBytes + g * row_bytes +
                            (warp * kcols + 8 * q) * 2;
      for (int p0 = 0; p0 < ngroups; p0 += kGroupsPerPass) {
        const int ng = ngroups - p0 < kGroupsPerPass ? ngroups - p0 : kGroupsPerPass;
        if (p0 > 0) consumer_bar();  // the previous pass's sums are read
        const uint16_t* xrow[kGroupsPerPass];
#pragma unroll
        for (int n = 0; n < kGroupsPerPass; ++n) {
          const int j = (p0 + n) * 8 + g;
          xrow[n] = (n < ng && j < cnt)
                        ? a.hidden + (size_t)(R.slots[base + j] / a.k) * a.H + warp * kcols + 8 * q
                        : nullptr;
        }
        float d[kGroupsPerPass][4];
#pragma unroll
        for (int n = 0; n < kGroupsPerPass; ++n) d[n][0] = d[n][1] = d[n][2] = d[n][3] = 0.f;
        warp_unit_mma_n<true>(ng, a_lo, a_lo + gu_rows_bytes, xrow, nsteps, d);
#pragma unroll
        for (int n = 0; n < kGroupsPerPass; ++n)
          if (n < ng) red[(warp * kGroupsPerPass + n) * 32 + lane] =
              make_float4(d[n][0], d[n][1], d[n][2], d[n][3]);
        if (p0 + kGroupsPerPass >= ngroups) release(fill);
        consumer_bar();
        if (warp < ng) {
          // group p0 + warp: the 8 warps' sums -> gate, up of intermediate
          // i0 + g for tokens 2q, 2q + 1 of the group
          float4 v = red[warp * 32 + lane];
#pragma unroll
          for (int w2 = 1; w2 < kCW; ++w2) {
            const float4 x = red[(w2 * kGroupsPerPass + warp) * 32 + lane];
            v.x += x.x;
            v.y += x.y;
            v.z += x.z;
            v.w += x.w;
          }
          const int j0 = (p0 + warp) * 8 + 2 * q;
          if (j0 < cnt)
            a.act[(size_t)R.slots[base + j0] * a.I + i0 + g] = f32_to_bf16_bits(silu_mul(v.x, v.z));
          if (j0 + 1 < cnt)
            a.act[(size_t)R.slots[base + j0 + 1] * a.I + i0 + g] =
                f32_to_bf16_bits(silu_mul(v.y, v.w));
        }
      }
      ++fill;
    }
  }

  // ---- barrier 1: every act row is complete
  consumer_bar();
  if (warp == 0) {
    const bool ok = grid_count_wait(a, ctr + 2, 1);
    if (lane == 0) {
      ok_s = ok ? 1 : 0;
      if (!ok) abort_s = 1;
    }
  }
  consumer_bar();
  if (!ok_s) return;
  // L1 prefetch of the act rows of the first expert of this CTA's static
  // down share (written by other SMs before grid barrier 1, so none of their
  // lines can be in this SM's L1 yet).
  if (sd > 0) {
    const int e = R.act_e[(2 * blockIdx.x * sd) / dn_per_e];
    const int lines = a.I / 64;
    const int n = min(R.cnt[e] * lines, 256);
    for (int i = tid; i < n; i += kCW * 32)
      prefetch_l1(a.act + (size_t)R.slots[R.start[e] + i / lines] * a.I + (i % lines) * 64);
  }

  // ---- D: down; a pair of units per slot, warps 4*grp .. 4*grp+3 on unit
  // grp, warp wl of the group on columns [wl*I/4, (wl+1)*I/4)
  {
    const int grp = warp >> 2, wl = warp & 3;
    const int kcols = a.I / 4, nsteps = kcols / 32;
    const uint32_t row_bytes = a.I * 2u;
    const uint64_t pol = l2_policy_evict_last();
    float4* red_g = red + grp * (4 * kGroupsPerPass * 32);
    while (true) {
      const int pr = next_fill();
      if (pr == kFillStop) return;
      if (pr == kFillEnd) {
        release(fill++);
        break;
      }
      const int vv = 2 * pr + grp;
      if (vv < Ud) {
        const int e = R.act_e[vv / dn_per_e], h0 = (vv % dn_per_e) * 16;
        const int cnt = R.cnt[e], base = R.start[e];
        const int ngroups = (cnt + 7) / 8;
        const uint32_t a_lo = ring + (fill % kSlots) * kSlotBytes + grp * (kSlotBytes / 2) +
                              g * row_bytes + (wl * kcols + 8 * q) * 2;
        for (int p0 = 0; p0 < ngroups; p0 += kGroupsPerPass) {
          const int ng = ngroups - p0 < kGroupsPerPass ? ngroups - p0 : kGroupsPerPass;
          if (p0 > 0) group_bar(grp);  // the previous pass's sums are read
          const uint16_t* xrow[kGroupsPerPass];
#pragma unroll
          for (int n = 0; n < kGroupsPerPass; ++n) {
            const int j = (p0 + n) * 8 + g;
            xrow[n] = (n < ng && j < cnt)
                          ? a.act + (size_t)R.slots[base + j] * a.I + wl * kcols + 8 * q
                          : nullptr;
          }
          float d[kGroupsPerPass][4];
#pragma unroll
          for (int n = 0; n < kGroupsPerPass; ++n) d[n][0] = d[n][1] = d[n][2] = d[n][3] = 0.f;
          warp_unit_mma_n<false>(ng, a_lo, a_lo + 8 * row_bytes, xrow, nsteps, d);
#pragma unroll
          for (int n = 0; n < kGroupsPerPass; ++n)
            if (n < ng) red_g[(wl * kGroupsPerPass + n) * 32 + lane] =
                make_float4(d[n][0], d[n][1], d[n][2], d[n][3]);
          if (p0 + kGroupsPerPass >= ngroups) release(fill);
          group_bar(grp);
          if (wl < ng) {
            // token tt of group p0 + wl, output rows h0 + 4*hq .. +3: the 4
            // warps' sums, gathered from the MMA layout (row r, token tt at
            // lane (r & 7) * 4 + tt / 2, word ((r >> 3) << 1) | (tt & 1))
            const int tt = lane >> 2, hq = lane & 3;
            const int j = (p0 + wl) * 8 + tt;
            if (j < cnt) {
              float s4[4];
#pragma unroll
              for (int rr = 0; rr < 4; ++rr) {
                const int r = 4 * hq + rr;
                const int src = (r & 7) * 4 + (tt >> 1), comp = ((r >> 3) << 1) | (tt & 1);
                float acc_v = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < 4; ++w2) {
                  const float* rv =
                      reinterpret_cast<const float*>(&red_g[(w2 * kGroupsPerPass + wl) * 32 + src]);
                  acc_v += rv[comp];
                }
                s4[rr] = acc_v;
              }
              const int f = R.slots[base + j];
              const float wt = R.w[f];
              red_add_v4_f32(a.acc + (size_t)(f / a.k) * a.H + h0 + 4 * hq, wt * s4[0], wt * s4[1],
                             wt * s4[2], wt * s4[3], pol);
            }
          }
        }
      } else {
        release(fill);
      }
      ++fill;
    }
  }
  if (a.out == nullptr) return;  // the caller's fp32 partial is the result

  // ---- barrier 2: the sum is complete
  consumer_bar();
  if (warp == 0) {
    const bool ok = grid_count_wait(a, ctr + 3, 2);
    if (lane == 0) ok_s = ok ? 1 : 0;
  }
  consumer_bar();
  if (!ok_s) return;

  // ---- E: out = bf16(sum), and the residual add after the layer
  {
    const long long ctid = (long long)blockIdx.x * (kCW * 32) + tid;
    const long long cstride = (long long)G * kCW * 32;
    const long long n4 = (long long)a.T * a.H / 4;
    for (long long i = ctid; i < n4; i += cstride) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(a.acc) + i);
      uint2 o;
      o.x = (uint32_t)f32_to_bf16_bits(v.x) | ((uint32_t)f32_to_bf16_bits(v.y) << 16);
      o.y = (uint32_t)f32_to_bf16_bits(v.z) | ((uint32_t)f32_to_bf16_bits(v.w) << 16);
      reinterpret_cast<uint2*>(a.out)[i] = o;
      if (a.res_out != nullptr) {
        const uint2 r = reinterpret_cast<const uint2*>(a.res_in)[i];
        uint2 n;
        n.x = (uint32_t)f32_to_bf16_bits(__uint_as_float(o.x << 16) + __uint_as_float(r.x << 16)) |
              ((uint32_t)f32_to_bf16_bits(__uint_as_float(o.x & 0xFFFF0000u) +
                                          __uint_as_float(r.x & 0xFFFF0000u))
               << 16);
        n.y = (uint32_t)f32_to_bf16_bits(__uint_as_float(o.y << 16) + __uint_as_float(r.y << 16)) |
              ((uint32_t)f32_to_bf16_bits(__uint_as_float(o.y & 0xFFFF0000u) +
                                          __uint_as_float(r.y & 0xFFFF0000u))
               << 16);
        reinterpret_cast<uint2*>(a.res_out)[i] = n;
      }
    }
  }
}

constexpr size_t kMaxDecSmem = kRingBytes + kRedBytes + routing_smem_bytes(kMaxExperts, kDecMaxTk);
static_assert(kMaxDecSmem <= 227 * 1024, "shared memory of the single-launch layer");

template <int Q>
cudaError_t launch_q(const DecodeArgs& a, int grid, size_t smem, cudaStream_t st) {
  static DeviceFlags attr_done;
  const cudaError_t ae = smem_attr_once(attr_done, moe_decode_kernel<Q>, (int)kMaxDecSmem);
  if (ae != cudaSuccess) return ae;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the grid barriers can complete
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_decode_kernel<Q>, a);
}

unsigned long long next_epoch() {
  // Unique per launch, and distinct from anything a flag region can hold
  // from an earlier process: a nanosecond clock reading plus a counter.
  static std::atomic<unsigned long long> seed{0};
  static std::atomic<unsigned long long> ctr{0};
  unsigned long long s = seed.load(std::memory_order_relaxed);
  if (s == 0) {
    const unsigned long long now = (unsigned long long)std::chrono::duration_cast<
        std::chrono::nanoseconds>(std::chrono::system_clock::now().time_since_epoch()).count();
    unsigned long long expect = 0;
    seed.compare_exchange_strong(expect, (now << 16) | 1ull);
    s = seed.load(std::memory_order_relaxed);
  }
  return s + (ctr.fetch_add(1, std::memory_order_relaxed) + 1);
}

}  // namespace

bool decode_supported(int T, int H, int E, int I, int top_k) {
  // gate_up: a unit's 16 rows of H fill at most one slot, and H splits into
  // 8 warps' whole 32-column steps; down: a unit's 16 rows of I fill at most
  // half a slot, and I splits into 4 warps' whole steps.
  return T >= 1 && T <= kDecMaxT && (long long)T * top_k <= kDecMaxTk && E <= kMaxExperts &&
         H % (kCW * 32) == 0 && 16LL * H * 2 <= kSlotBytes && I % (4 * 32) == 0 &&
         16LL * I * 2 <= kSlotBytes / 2;
}

bool decode_preferred(int T, int H, int E, int I, int top_k) {
  // Measured on GB300 (H=2048, E=128, k=8, I=768, Zipf-skewed routing): the
  // single launch takes 36 / 49 / 58 / 73 us at T = 1 / 4 / 8 / 16 against
  // 51 / 55 / 66 / 85 us for the kernel chain, and loses from T = 24 on
  // (92 vs 86 us), where per-CTA routing of every token and the experts
  // holding many of the batch's tokens make it compute-bound.
  return T <= kDecAutoMaxT && decode_supported(T, H, E, I, top_k);
}

// The barriers' flags (grid barrier 0 uses its epoch flags), then two words
// holding the two work counters and the arrival counters of grid barriers 1
// and 2.
int decode_flag_slots() { return kDecBarriers * kDecMaxGrid + 2; }

cudaError_t launch_moe_decode(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                              const uint16_t* w_gate_up, const uint16_t* w_down, int T, int H,
                              int E, int I, int top_k, int renorm, const DecodeBuffers& b,
                              uint16_t* out, const uint16_t* res_in, uint16_t* res_out,
                              int num_sms, unsigned* err, cudaStream_t st, int absent_cta,
                              int absent_barrier) {
  if (!decode_supported(T, H, E, I, top_k)) return cudaErrorInvalidValue;
  DecodeArgs a;
  a.hidden = hidden;
  a.router_w = router_w;
  a.bias = bias;
  a.w_gate_up = w_gate_up;
  a.w_down = w_down;
  a.T = T;
  a.H = H;
  a.E = E;
  a.I = I;
  a.k = top_k;
  a.renorm = renorm;
  a.logits = b.logits;
  a.ids = b.ids;
  a.w = b.w;
  a.sorted = b.sorted;
  a.offsets = b.offsets;
  a.counts = b.counts;
  a.capacity = b.capacity;
  a.act = b.act;
  a.acc = b.acc;
  a.out = out;
  a.res_in = res_in;
  a.res_out = res_out;
  a.flags = b.flags;
  a.epoch = next_epoch();
  a.err = err;
  a.absent_cta = absent_cta;
  a.absent_barrier = absent_barrier;
  const size_t smem = kRingBytes + kRedBytes + routing_smem_bytes(E, T * top_k);
  // one CTA per SM: all resident (cooperative launch)
  const int grid = num_sms < kDecMaxGrid ? num_sms : kDecMaxGrid;
  const int q = (E + 31) / 32;
  if (q <= 1) return launch_q<1>(a, grid, smem, st);
  if (q <= 2) return launch_q<2>(a, grid, smem, st);
  if (q <= 4) return launch_q<4>(a, grid, smem, st);
  return launch_q<8>(a, grid, smem, st);
}

}  // namespace mm
