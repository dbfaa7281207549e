// The per-token end of the router, shared by both router kernels: softmax
// over all experts, top-k with ties to the lower expert id, ascending slot
// order, optional renormalisation ("mini-sglang guide, chapter 7", paragraph
// on layers/moe.py; "模型与权重加载", ModelConfig: norm_topk_prob).
#pragma once

#include <math.h>

#include "mm_device.cuh"

namespace mm {
namespace routefin {

// One warp finishes NT tokens at once (their reduction chains interleave).
// For token i, lane l holds the logits of experts l + 32*q (q < Q) in
// l[i][q], -INFINITY where l + 32*q >= E (bias already added); t[i] < 0
// marks an unused slot. Writes top_k ids (ascending) and weights at
// ids_out / w_out + t[i]*top_k.
template <int Q, int NT>
__device__ __forceinline__ void finish_tokens(const float (&l)[NT][Q], const int (&t)[NT], int E,
                                              int top_k, int renorm,
                                              int32_t* __restrict__ ids_out,
                                              float* __restrict__ w_out) {
  const int lane = threadIdx.x & 31;
  float m[NT], s[NT], z[NT][Q];
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    m[i] = -INFINITY;
#pragma unroll
    for (int q = 0; q < Q; ++q) m[i] = fmaxf(m[i], l[i][q]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < NT; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], o));
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    s[i] = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      z[i][q] = (lane + 32 * q < E) ? expf(l[i][q] - m[i]) : 0.f;
      s[i] += z[i][q];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < NT; ++i) s[i] += __shfl_xor_sync(0xffffffffu, s[i], o);

  // k rounds of warp arg-max: the larger logit wins, equal logits go to the
  // lower expert id. A logit is compared as an order-preserving uint32 key
  // (exact: -0 is first folded into +0), so one warp-wide max reduction finds
  // the best value and one min reduction picks the lowest id holding it.
  uint32_t key[NT][Q], sel[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    sel[i] = 0;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const uint32_t b = __float_as_uint(l[i][q] + 0.0f);
      key[i][q] = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    }
  }
  for (int round = 0; round < top_k; ++round) {
    uint32_t bk[NT];
    int bq[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      bk[i] = 0;
      bq[i] = Q;  // none
#pragma unroll
      for (int q = 0; q < Q; ++q)  // ascending ids: strict '>' keeps the lower id on ties
        if (lane + 32 * q < E && !((sel[i] >> q) & 1u) && (bq[i] == Q || key[i][q] > bk[i])) {
          bk[i] = key[i][q];
          bq[i] = q;
        }
    }
    uint32_t mk[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) mk[i] = __reduce_max_sync(0xffffffffu, bq[i] < Q ? bk[i] : 0u);
    uint32_t win[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i)
      win[i] = __reduce_min_sync(0xffffffffu, (bq[i] < Q && bk[i] == mk[i])
                                                  ? static_cast<uint32_t>(bq[i] * 32 + lane)
                                                  : 0xffffffffu);
#pragma unroll
    for (int i = 0; i < NT; ++i)
      if ((int)(win[i] & 31u) == lane) sel[i] |= 1u << (win[i] >> 5);
  }

  // Probabilities of the selected experts, renormalised if asked.
  float psel[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    psel[i] = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q)
      if ((sel[i] >> q) & 1u) psel[i] += z[i][q] / s[i];
  }
  if (renorm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int i = 0; i < NT; ++i) psel[i] += __shfl_xor_sync(0xffffffffu, psel[i], o);
  }
  // Ascending expert order: slot = number of selected experts with a lower id.
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    int base = 0;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const bool mine = (sel[i] >> q) & 1u;
      const uint32_t bal = __ballot_sync(0xffffffffu, mine);
      if (mine && t[i] >= 0) {
        const int slot = base + __popc(bal & lt);
        const float p = z[i][q] / s[i];
        ids_out[(size_t)t[i] * top_k + slot] = lane + 32 * q;
        w_out[(size_t)t[i] * top_k + slot] = renorm ? p / psel[i] : p;
      }
      base += __popc(bal);
    }
  }
}

// One token per warp.
template <int Q>
__device__ __forceinline__ void finish_token(const float (&l)[Q], int E, int top_k, int renorm,
                                             int t, int32_t* __restrict__ ids_out,
                                             float* __restrict__ w_out) {
  const float (&ll)[1][Q] = reinterpret_cast<const float (&)[1][Q]>(l);
  const int tt[1] = {t};
  finish_tokens<Q, 1>(ll, tt, E, top_k, renorm, ids_out, w_out);
}

}  // namespace routefin
}  // namespace mm
