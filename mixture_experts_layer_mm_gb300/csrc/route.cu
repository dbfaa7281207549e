// Router of the MoE layer: logits (bf16 x bf16 -> fp32 on tensor cores),
// softmax over all experts, top-k with ties to the lower id, ascending slot
// order, optional renormalisation ("mini-sglang guide, chapter 7", paragraph
// on layers/moe.py; "模型与权重加载", ModelConfig: norm_topk_prob).
//
// One CTA = 4 warps = 64 tokens x all experts. The logits GEMM is 2*T*E*H
// flops (under 1 % of the layer), so it runs on warp-level mma.sync with a
// double-buffered cp.async pipeline; each warp then owns 16 tokens and does
// the softmax and the k rounds of warp arg-max on the logits held in shared
// memory. Logits never reach global memory.
#include <float.h>

#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

constexpr int kRtTok = 64;        // tokens per CTA
constexpr int kRtKc = 64;         // K per pipeline stage
constexpr int kRtLd = kRtKc + 8;  // padded smem row (bf16): 144 B, conflict-free ldmatrix
constexpr int kRtThreads = 128;

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
    const float* __restrict__ bias, int T, int H, int E, int top_k, int renorm,
    int32_t* __restrict__ ids_out, float* __restrict__ w_out, float* __restrict__ zero_buf,
    long long zero_count) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);  // [2][kRtTok][kRtLd]
  uint16_t* ws = xs + 2 * kRtTok * kRtLd;             // [2][EP][kRtLd]
  float* logit_s = reinterpret_cast<float*>(smem);    // after the GEMM: [kRtTok][EP + 1]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kRtTok;

  if (zero_buf != nullptr) {  // fused zeroing of the fp32 output accumulator
    float4* z = reinterpret_cast<float4*>(zero_buf);
    const long long n4 = zero_count >> 2;
    for (long long i = (long long)blockIdx.x * kRtThreads + tid; i < n4;
         i += (long long)gridDim.x * kRtThreads)
      z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  auto load_stage = [&](int buf, int kc) {
    for (int i = tid; i < kRtTok * 8; i += kRtThreads) {
      const int r = i >> 3, c = i & 7, t = t0 + r;
      const uint32_t dst = smem_u32(xs + (buf * kRtTok + r) * kRtLd + c * 8);
      const bool ok = t < T;
      cp_async16(dst, hidden + (ok ? (size_t)t * H + kc + c * 8 : 0), ok);
    }
    for (int i = tid; i < EP * 8; i += kRtThreads) {
      const int r = i >> 3, c = i & 7;
      const uint32_t dst = smem_u32(ws + (buf * EP + r) * kRtLd + c * 8);
      const bool ok = r < E;
      cp_async16(dst, router_w + (ok ? (size_t)r * H + kc + c * 8 : 0), ok);
    }
    cp_async_commit();
  };

  float acc[EP / 8][4];
#pragma unroll
  for (int j = 0; j < EP / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  const int nk = H / kRtKc;
  load_stage(0, 0);
  for (int kc = 0; kc < nk; ++kc) {
    if (kc + 1 < nk) {
      load_stage((kc + 1) & 1, (kc + 1) * kRtKc);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint16_t* xb = xs + (kc & 1) * kRtTok * kRtLd;
    const uint16_t* wb = ws + (kc & 1) * EP * kRtLd;
#pragma unroll
    for (int kk = 0; kk < kRtKc / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(smem_u32(xb + (warp * 16 + (lane & 15)) * kRtLd + kk * 16 + (lane >> 4) * 8), a0,
                  a1, a2, a3);
#pragma unroll
      for (int j2 = 0; j2 < EP / 16; ++j2) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(smem_u32(wb + (j2 * 16 + (lane & 7) + ((lane >> 4) << 3)) * kRtLd + kk * 16 +
                             ((lane >> 3) & 1) * 8),
                    b0, b1, b2, b3);
        mma_bf16_16816(acc[2 * j2], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(acc[2 * j2 + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();
  }

  // Accumulators -> shared logits [token][expert].
  {
    const int r0 = warp * 16 + (lane >> 2), c0 = 2 * (lane & 3);
#pragma unroll
    for (int j = 0; j < EP / 8; ++j) {
      logit_s[r0 * (EP + 1) + j * 8 + c0] = acc[j][0];
      logit_s[r0 * (EP + 1) + j * 8 + c0 + 1] = acc[j][1];
      logit_s[(r0 + 8) * (EP + 1) + j * 8 + c0] = acc[j][2];
      logit_s[(r0 + 8) * (EP + 1) + j * 8 + c0 + 1] = acc[j][3];
    }
  }
  __syncthreads();

  constexpr int Q = EP / 32;  // logits per lane
  for (int rr = 0; rr < 16; ++rr) {
    const int r = warp * 16 + rr, t = t0 + r;
    if (t >= T) break;
    float l[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int e = lane + 32 * q;
      l[q] = -INFINITY;
      if (e < E) l[q] = logit_s[r * (EP + 1) + e] + (bias != nullptr ? bias[e] : 0.f);
    }
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < Q; ++q) m = fmaxf(m, l[q]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z[Q], s = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      z[q] = (lane + 32 * q < E) ? expf(l[q] - m) : 0.f;
      s += z[q];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);

    // k rounds of warp arg-max: the larger logit wins, equal logits go to the
    // lower expert id.
    uint32_t sel = 0;
    for (int round = 0; round < top_k; ++round) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int q = 0; q < Q; ++q) {  // ascending ids: strict '>' keeps the lower id on ties
        const int e = lane + 32 * q;
        if (e < E && !((sel >> q) & 1u) && (bi == 0x7fffffff || l[q] > bv)) {
          bv = l[q];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) sel |= 1u << (bi >> 5);
    }

    // Probabilities of the selected experts, renormalised if asked.
    float psel = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q)
      if ((sel >> q) & 1u) psel += z[q] / s;
    float denom = 1.f;
    if (renorm) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psel += __shfl_xor_sync(0xffffffffu, psel, o);
      denom = psel;
    }
    // Ascending expert order: slot = number of selected experts with a lower id.
    int base = 0;
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const bool mine = (sel >> q) & 1u;
      const uint32_t bal = __ballot_sync(0xffffffffu, mine);
      if (mine) {
        const int slot = base + __popc(bal & lt);
        const float p = z[q] / s;
        ids_out[(size_t)t * top_k + slot] = lane + 32 * q;
        w_out[(size_t)t * top_k + slot] = renorm ? p / denom : p;
      }
      base += __popc(bal);
    }
  }
}

template <int EP>
cudaError_t launch_ep(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int T,
                      int H, int E, int top_k, int renorm, int32_t* ids, float* w, float* zero_buf,
                      long long zero_count, cudaStream_t st) {
  const size_t gemm_bytes = (size_t)2 * (kRtTok + EP) * kRtLd * sizeof(uint16_t);
  const size_t logit_bytes = (size_t)kRtTok * (EP + 1) * sizeof(float);
  const size_t smem = gemm_bytes > logit_bytes ? gemm_bytes : logit_bytes;
  cudaError_t e = cudaFuncSetAttribute(route_kernel<EP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = (T + kRtTok - 1) / kRtTok;
  route_kernel<EP><<<grid, kRtThreads, smem, st>>>(hidden, router_w, bias, T, H, E, top_k, renorm,
                                                   ids, w, zero_buf, zero_count);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                         int T, int H, int E, int top_k, int renorm, int32_t* topk_ids,
                         float* topk_w, float* zero_buf, long long zero_count, cudaStream_t st) {
  if (E <= 32)
    return launch_ep<32>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                         zero_buf, zero_count, st);
  if (E <= 64)
    return launch_ep<64>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                         zero_buf, zero_count, st);
  if (E <= 128)
    return launch_ep<128>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w,
                          zero_buf, zero_count, st);
  return launch_ep<256>(hidden, router_w, bias, T, H, E, top_k, renorm, topk_ids, topk_w, zero_buf,
                        zero_count, st);
}

}  // namespace mm
