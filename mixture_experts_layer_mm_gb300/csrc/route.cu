// Router of the MoE layer: logits (bf16 x bf16 -> fp32 on tensor cores),
// softmax over all experts, top-k with ties to the lower id, ascending slot
// order, optional renormalisation ("mini-sglang guide, chapter 7", paragraph
// on layers/moe.py; "模型与权重加载", ModelConfig: norm_topk_prob).
//
// The logits GEMM is 2*T*E*H flops (under 1 % of the layer) but reads the
// whole router matrix for every 64-token tile, so one CTA per tile is
// latency-bound. Here a thread-block cluster of KS CTAs (KS <= 8) shares a
// tile: CTA r loads and multiplies only the K-slice [r*H/KS, (r+1)*H/KS) with
// all its chunks in flight at once (warp-level mma.sync, fp32 accumulate),
// then pushes the partial logits of each token to the CTA that finishes that
// token (remote shared-memory stores into its now free staging buffers).
// After a cluster barrier each CTA sums the KS partials of its 64/KS tokens
// in rank order from its own shared memory (so the result does not depend on
// timing) and runs the softmax and k rounds of warp arg-max (one token per
// warp). Logits never reach global memory.
//
// When one cluster covers the whole batch (T <= 64), CTA 0 of the cluster
// also groups the tokens by expert after the final cluster barrier (which
// makes every CTA's ids visible to it), saving the separate align launch.
#include <float.h>

#include "align_block.cuh"
#include "mm_device.cuh"
#include "mm_internal.h"
#include "route_finish.cuh"

namespace mm {
namespace {

constexpr int kRtTok = 64;        // tokens per cluster tile
constexpr int kRtKc = 64;         // K per cp.async chunk
constexpr int kRtLd = kRtKc + 8;  // padded smem row (bf16): 144 B, conflict-free ldmatrix
constexpr int kRtThreads = 256;  // 8 warps: 4 run the MMAs, all 8 finish tokens
constexpr int kRtMmaWarps = 4;   // 16 token rows each
constexpr int kRtBufs = 4;        // chunks in flight per CTA

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address in CTA `rank` of this cluster of the shared variable at `local`.
__device__ __forceinline__ uint32_t map_rank(uint32_t local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}

__device__ __forceinline__ void st_dsmem_v2(uint32_t cluster_addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(cluster_addr), "f"(a), "f"(b)
               : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes -> the 16 bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// EP = experts rounded up to a power of two >= 32 (E <= EP <= 256).
template <int EP>
__global__ void __launch_bounds__(kRtThreads) route_kernel(
    const uint16_t* __restrict__ hidden, const uint16_t* __restrict__ router_w,
    const float* __restrict__ bias, int T, int H, int E, int top_k, int renorm, int ks,
    int32_t* __restrict__ ids_out, float* __restrict__ w_out, float* __restrict__ zero_buf,
    long long zero_count, const AlignOut fa) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);  // [kRtBufs][kRtTok][kRtLd]
  uint16_t* ws = xs + kRtBufs * kRtTok * kRtLd;       // [kRtBufs][EP][kRtLd]
  float* recv = reinterpret_cast<float*>(smem);       // after the GEMM: [KS][64/KS][EP]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = ks > 1 ? cluster_ctarank() : 0u;
  pdl_wait();  // hidden may come from the kernel before this one (the RMSNorm step)
  pdl_trigger();  // the next kernel of the layer may be scheduled (it waits for this one)
  const int t0 = (blockIdx.x / ks) * kRtTok;
  const int hs = H / ks, hbase = (int)rank * hs;

  const int nk = hs / kRtKc;
  auto load_chunk = [&](int c) {
    if (c < nk) {
      const int buf = c % kRtBufs, kc = hbase + c * kRtKc;
      for (int i = tid; i < kRtTok * 8; i += kRtThreads) {
        const int r = i >> 3, cc = i & 7, t = t0 + r;
        const uint32_t dst = smem_u32(xs + (buf * kRtTok + r) * kRtLd + cc * 8);
        const bool ok = t < T;
        cp_async16(dst, hidden + (ok ? (size_t)t * H + kc + cc * 8 : 0), ok);
      }
      for (int i = tid; i < EP * 8; i += kRtThreads) {
        const int r = i >> 3, cc = i & 7;
        const uint32_t dst = smem_u32(ws + (buf * EP + r) * kRtLd + cc * 8);
        const bool ok = r < E;
        cp_async16(dst, router_w + (ok ? (size_t)r * H + kc + cc * 8 : 0), ok);
      }
    }
    cp_async_commit();  // empty groups keep the group count uniform
  };

  float acc[EP / 8][4];
#pragma unroll
  for (int j = 0; j < EP / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

#pragma unroll
  for (int c = 0; c < kRtBufs; ++c) load_chunk(c);
  // Fused zeroing of the fp32 output accumulator, issued after this CTA's
  // first loads so that those do not queue behind the stores.
  if (zero_buf != nullptr) {
    float4* z = reinterpret_cast<float4*>(zero_buf);
    const long long n4 = zero_count >> 2;
    for (long long i = (long long)blockIdx.x * kRtThreads + tid; i < n4;
         i += (long long)gridDim.x * kRtThreads)
      z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int c = 0; c < nk; ++c) {
    cp_async_wait<kRtBufs - 1>();
    __syncthreads();
    const uint16_t* xb = xs + (c % kRtBufs) * kRtTok * kRtLd;
    const uint16_t* wb = ws + (c % kRtBufs) * EP * kRtLd;
    if (warp < kRtMmaWarps) {
#pragma unroll
      for (int kk = 0; kk < kRtKc / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(smem_u32(xb + (warp * 16 + (lane & 15)) * kRtLd + kk * 16 + (lane >> 4) * 8),
                    a0, a1, a2, a3);
#pragma unroll
        for (int j2 = 0; j2 < EP / 16; ++j2) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(smem_u32(wb + (j2 * 16 + (lane & 7) + ((lane >> 4) << 3)) * kRtLd +
                               kk * 16 + ((lane >> 3) & 1) * 8),
                      b0, b1, b2, b3);
          mma_bf16_16816(acc[2 * j2], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(acc[2 * j2 + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();
    load_chunk(c + kRtBufs);
  }
  cp_async_wait<0>();
  __syncthreads();

  // Every CTA of the cluster has finished with its staging buffers; they now
  // receive partial logits: recv[src][rr][e] holds CTA src's partial sum for
  // token rr of this CTA's share (64/KS tokens). Each CTA pushes its rows to
  // their owners with remote stores, so the reduction below reads only local
  // shared memory.
  const int per = kRtTok / ks;  // tokens each CTA finishes
  if (ks > 1)
    cluster_sync();
  else
    __syncthreads();
  if (warp < kRtMmaWarps) {
    const int r0 = warp * 16 + (lane >> 2), c0 = 2 * (lane & 3);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = r0 + 8 * h;
      const int owner = r / per;
      float* row = recv + ((int)rank * per + (r - owner * per)) * EP;
      if (ks > 1) {
        const uint32_t rbase = map_rank(smem_u32(row), (uint32_t)owner);
#pragma unroll
        for (int j = 0; j < EP / 8; ++j)
          st_dsmem_v2(rbase + (j * 8 + c0) * 4, acc[j][2 * h], acc[j][2 * h + 1]);
      } else {
#pragma unroll
        for (int j = 0; j < EP / 8; ++j) {
          row[j * 8 + c0] = acc[j][2 * h];
          row[j * 8 + c0 + 1] = acc[j][2 * h + 1];
        }
      }
    }
  }
  if (ks > 1)
    cluster_sync();  // all pushes have landed
  else
    __syncthreads();

  constexpr int Q = EP / 32;  // logits per lane
  for (int rr = warp; rr < per; rr += kRtThreads / 32) {
    const int r = (int)rank * per + rr, t = t0 + r;
    if (t >= T) break;
    float l[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int e = lane + 32 * q;
      l[q] = -INFINITY;
      if (e < E) {
        float v = 0.f;
        for (int src = 0; src < ks; ++src)  // fixed order: deterministic sum
          v += recv[(src * per + rr) * EP + e];
        l[q] = v + (bias != nullptr ? bias[e] : 0.f);
      }
    }
    routefin::finish_token<Q>(l, E, top_k, renorm, t, ids_out, w_out);
  }
  // The grouping (T <= 64) needs every CTA's ids: one more cluster barrier.
  if (fa.sorted != nullptr) {
    if (ks > 1)
      cluster_sync();
    else
      __syncthreads();
    if (rank == 0)
      alignblk::align_tiny(ids_out, T, top_k, E, fa.block_m, fa.capacity, fa.sorted,
                           fa.offsets, fa.counts, fa.err, smem);
  }
}

template <int EP>
cudaError_t launch_ep(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int T,
                      int H, int E, int top_k, int renorm, int32_t* ids, float* w, float* zero_buf,
                      long long zero_count, const AlignOut& fa, int num_sms, bool after_prev,
                      cudaStream_t st) {
  const size_t gemm_bytes = (size_t)kRtBufs * (kRtTok + EP) * kRtLd * sizeof(uint16_t);
  const size_t recv_bytes = (size_t)kRtTok * EP * sizeof(float);
  const size_t smem = gemm_bytes > recv_bytes ? gemm_bytes : recv_bytes;
  static DeviceFlags attr_done;
  if (cudaError_t e = smem_attr_once(attr_done, route_kernel<EP>, (int)smem); e != cudaSuccess)
    return e;
  // Cluster size: the largest of 8, 4, 2 that splits H into 64-wide chunks
  // and keeps the whole grid resident at once (CTAs per SM bounded by shared
  // memory). Small batches get the widest split, which shortens each CTA's
  // serial chain of loads; large batches have enough tiles without it.
  const int tiles = (T + kRtTok - 1) / kRtTok;
  const long long resident = (long long)num_sms * (int)((227 * 1024) / (smem + 1024));
  int ks = 1;
  for (int c = 8; c > 1; c >>= 1)
    if (H % (kRtKc * c) == 0 && (long long)tiles * c <= resident) {
      ks = c;
      break;
    }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * ks, 1, 1);
  cfg.blockDim = dim3(kRtThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_prev ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, route_kernel<EP>, hidden, router_w, bias, T, H, E, top_k, renorm,
                            ks, ids, w, zero_buf, zero_count, fa);
}

}  // namespace

bool route_fuses_align(int T, int top_k) { return T <= kRtTok && T * top_k <= kAlignSingleMaxIds; }

cudaError_t launch_route(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                         int T, int H, int E, int top_k, int renorm, int32_t* topk_ids,
                         float* topk_w, float* zero_buf, long long zero_count,
                         const AlignOut* fuse_align, int num_sms, unsigned* err,
                         bool after_prev, cudaStream_t st, int32_t* tile_counts) {
  // More than one 64-token tile and at most 128 experts: the tcgen05 router.
  if (route_uses_tensor_cores(T, E))
    return launch_route_tc(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                           zero_buf, zero_count, tile_counts, num_sms, err, after_prev, st);
  AlignOut fa = {};
  if (fuse_align != nullptr && route_fuses_align(T, top_k)) fa = *fuse_align;
  if (E <= 32)
    return launch_ep<32>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                         zero_buf, zero_count, fa, num_sms, after_prev, st);
  if (E <= 64)
    return launch_ep<64>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                         zero_buf, zero_count, fa, num_sms, after_prev, st);
  if (E <= 128)
    return launch_ep<128>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                          zero_buf, zero_count, fa, num_sms, after_prev, st);
  return launch_ep<256>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w, zero_buf,
                        zero_count, fa, num_sms, after_prev, st);
}

}  // namespace mm
