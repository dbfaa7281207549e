// The residual add + RMSNorm that precedes the MoE block of a decoder layer
// ("The op layer: BaseOP and the layers": the rmsnorm / fused_add_rmsnorm
// listings of "Ops: reference implementations and dispatch"; RMSNormFused
// and DecoderLayer.forward of "RMSNorm and the residual"):
// residual' = bf16(x + residual),
// normed = bf16(weight * bf16(residual' * rsqrt(mean(residual'^2) + eps))).
//
// One warp per row, 16-byte accesses. Lane l takes the 8-element chunks
// c = l, l + 32, ... of the row; the float32 sum of squares runs over its
// chunks in that order (each square rounded, then added: no fused
// multiply-add), then an xor butterfly over the lanes (16, 8, 4, 2, 1).
// rsqrt(v) = 1 / sqrt(v) with both steps rounded. With that order fixed every
// operation is a correctly rounded float32 step, so the normalised rows are
// the same on every call (the pages leave the summation order open; another
// order can move an element by one bf16 rounding step).
#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
}

// Elementwise bf16(a + b) of two chunks of 8 bf16.
__device__ __forceinline__ uint4 add_chunk(uint4 a, uint4 b) {
  uint4 r;
  r.x = pack_bf16(__fadd_rn(bf16_lo(a.x), bf16_lo(b.x)), __fadd_rn(bf16_hi(a.x), bf16_hi(b.x)));
  r.y = pack_bf16(__fadd_rn(bf16_lo(a.y), bf16_lo(b.y)), __fadd_rn(bf16_hi(a.y), bf16_hi(b.y)));
  r.z = pack_bf16(__fadd_rn(bf16_lo(a.z), bf16_lo(b.z)), __fadd_rn(bf16_hi(a.z), bf16_hi(b.z)));
  r.w = pack_bf16(__fadd_rn(bf16_lo(a.w), bf16_lo(b.w)), __fadd_rn(bf16_hi(a.w), bf16_hi(b.w)));
  return r;
}

__device__ __forceinline__ float add_sq(float acc, float v) {
  return __fadd_rn(acc, __fmul_rn(v, v));
}

// Squares of the chunk's 8 elements added to acc in element order.
__device__ __forceinline__ float chunk_sumsq(float acc, uint4 c) {
  acc = add_sq(acc, bf16_lo(c.x));
  acc = add_sq(acc, bf16_hi(c.x));
  acc = add_sq(acc, bf16_lo(c.y));
  acc = add_sq(acc, bf16_hi(c.y));
  acc = add_sq(acc, bf16_lo(c.z));
  acc = add_sq(acc, bf16_hi(c.z));
  acc = add_sq(acc, bf16_lo(c.w));
  acc = add_sq(acc, bf16_hi(c.w));
  return acc;
}

// bf16(w * bf16(r * inv)) for one element pair packed in a word.
__device__ __forceinline__ uint32_t norm_pair(uint32_t r, uint32_t w, float inv) {
  const float ylo = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(bf16_lo(r), inv)));
  const float yhi = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(bf16_hi(r), inv)));
  return pack_bf16(__fmul_rn(bf16_lo(w), ylo), __fmul_rn(bf16_hi(w), yhi));
}

constexpr int kNormBatch = 8;  // chunks a lane has in flight at once

__global__ void __launch_bounds__(256) add_rmsnorm_kernel(const uint4* __restrict__ x,
                                                          uint4* __restrict__ residual,
                                                          const uint4* __restrict__ weight,
                                                          float eps, int T, int H,
                                                          uint4* __restrict__ normed) {
  pdl_wait();  // x may come from the kernel before this one on the stream
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int h8 = H / 8;                 // chunks per row
  const int per = (h8 - lane + 31) / 32;  // this lane's chunks: lane, lane + 32, ...
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
    const uint4* xr = x + (size_t)t * h8 + lane;
    uint4* rr = residual != nullptr ? residual + (size_t)t * h8 + lane : nullptr;
    float acc = 0.f;
    // Pass 1, kNormBatch chunks at a time: all loads of a batch are issued
    // before any of them is used; the squares are added in chunk order.
    for (int b0 = 0; b0 < per; b0 += kNormBatch) {
      uint4 r[kNormBatch], q[kNormBatch];
#pragma unroll
      for (int i = 0; i < kNormBatch; ++i)
        if (b0 + i < per) {
          r[i] = __ldg(xr + 32 * (b0 + i));
          if (rr != nullptr) q[i] = rr[32 * (b0 + i)];
        }
#pragma unroll
      for (int i = 0; i < kNormBatch; ++i)
        if (b0 + i < per) {
          if (rr != nullptr) {
            r[i] = add_chunk(r[i], q[i]);
            rr[32 * (b0 + i)] = r[i];  // residual' in place
          }
          acc = chunk_sumsq(acc, r[i]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    const float mean = __fdiv_rn(acc, (float)H);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
    uint4* nr = normed + (size_t)t * h8 + lane;
    const uint4* wr = weight + lane;
    for (int b0 = 0; b0 < per; b0 += kNormBatch) {
      uint4 r[kNormBatch], w[kNormBatch];
#pragma unroll
      for (int i = 0; i < kNormBatch; ++i)
        if (b0 + i < per) {
          // residual' as this thread wrote it, or x itself
          r[i] = rr != nullptr ? rr[32 * (b0 + i)] : __ldg(xr + 32 * (b0 + i));
          w[i] = __ldg(wr + 32 * (b0 + i));
        }
#pragma unroll
      for (int i = 0; i < kNormBatch; ++i)
        if (b0 + i < per) {
          uint4 o;
          o.x = norm_pair(r[i].x, w[i].x, inv);
          o.y = norm_pair(r[i].y, w[i].y, inv);
          o.z = norm_pair(r[i].z, w[i].z, inv);
          o.w = norm_pair(r[i].w, w[i].w, inv);
          nr[32 * (b0 + i)] = o;
        }
    }
  }
}

}  // namespace

cudaError_t launch_add_rmsnorm(const uint16_t* x, uint16_t* residual, const uint16_t* weight,
                               float eps, int T, int H, uint16_t* normed, int num_sms,
                               bool after_prev, cudaStream_t st) {
  long long blocks = ((long long)T + 7) / 8;  // 8 rows (warps) per block
  if (blocks > (long long)num_sms * 8) blocks = (long long)num_sms * 8;
  if (blocks < 1) blocks = 1;
  return launch_k(add_rmsnorm_kernel, dim3((int)blocks), dim3(256), 0, st, after_prev,
                  reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(residual),
                  reinterpret_cast<const uint4*>(weight), eps, T, H,
                  reinterpret_cast<uint4*>(normed));
}

}  // namespace mm
