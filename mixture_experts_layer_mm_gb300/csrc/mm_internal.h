// Host-side launchers of the MoE layer's kernels (internal; the public C ABI
// is include/mm.h and is implemented in api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mm {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;
// Token rows per expert segment are padded to this multiple by the forward
// path; it is also the granularity of the tensor-core N dimension.
constexpr int kForwardBlockM = 16;
// Align: one block does everything when T <= kAlignSingleMaxTokens and
// T*k <= kAlignSingleMaxIds; otherwise blocks of kAlignBlockTokens tokens.
constexpr int kAlignSingleMaxTokens = 1024;
constexpr int kAlignSingleMaxIds = 8192;
constexpr int kAlignBlockTokens = 256;
constexpr int kMaxDevices = 64;

// Index of the current CUDA device (0 if the query fails).
inline int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) d = 0;
  return d;
}

// Device address of the current device's status word (see
// mm_poll_device_status); sets up the device state on first use.
int current_status_word(unsigned** out);

// Outputs of the grouping step (see mm_align) when the router runs it itself.
struct AlignOut {
  int32_t* sorted;
  int32_t* offsets;
  int32_t* counts;
  int block_m;
  long long capacity;
  unsigned* err;
};

// Whether launch_route can group the tokens by expert in the same launch.
bool route_fuses_align(int T, int top_k);

// Router logits + softmax + top-k (+ renorm). If zero_buf is non-null the same
// launch also zeroes zero_count floats there (zero_count % 4 == 0). If
// fuse_align is non-null and route_fuses_align(T, top_k), the launch also
// produces the grouping. num_sms sizes the cluster split of H.
cudaError_t launch_route(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                         int T, int H, int E, int top_k, int renorm, int32_t* topk_ids,
                         float* topk_w, float* zero_buf, long long zero_count,
                         const AlignOut* fuse_align, int num_sms, cudaStream_t st);

// Scratch ints the align launch needs (0 when one block covers all tokens).
long long align_scratch_ints(int T, int E, int top_k);

cudaError_t launch_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                         long long capacity, int32_t* sorted, int32_t* offsets, int32_t* counts,
                         int32_t* scratch, unsigned* err, cudaStream_t st);

// Grouping of a dense MLP (one expert, every token, weight 1) + zeroed
// accumulator of zero_count floats.
cudaError_t launch_identity_grouping(int T, int block_m, long long capacity, int32_t* sorted,
                                     int32_t* offsets, float* weights, float* zero_buf,
                                     long long zero_count, int num_sms, cudaStream_t st);

// Whether the gate_up GEMM gathers token rows with TMA tile::gather4 (few rows
// per expert) rather than with cp.async loader warps.
bool gate_up_gathers_rows(int T, int top_k, int E);

// Grouped GEMM on tcgen05. mode 0: C = act bf16 [capacity, N] = silu(gate) *
// up; X = hidden [T, K] with rows gathered through sorted / top_k when
// x_is_hidden, else X = token rows already in segment order [x_rows, K]
// (rows at or past x_rows read as zeros).
// mode 1: X = act [x_rows, K], C = fp32 acc [T, N] += topk_w * (X W^T).
cudaError_t launch_grouped_gemm(int mode, const uint16_t* X, bool x_is_hidden, const uint16_t* W,
                                void* C, const int32_t* sorted, const int32_t* offsets,
                                const float* topk_w, int T, int top_k, int E, int N, int K,
                                long long capacity, long long x_rows, int num_sms, unsigned* err,
                                cudaStream_t st);

// out[i] = bf16(acc[i]) for i < n (n % 4 == 0).
// xs[r] = hidden[sorted[r] / top_k] (H bf16 per row) for r < offsets[E];
// padding rows of the segments become zeros. H % 8 == 0.
cudaError_t launch_gather_rows(const uint16_t* hidden, const int32_t* sorted,
                               const int32_t* offsets, int T, int top_k, int E, int H,
                               uint16_t* xs, int num_sms, cudaStream_t st);

cudaError_t launch_finalize(const float* acc, uint16_t* out, long long n, int num_sms,
                            cudaStream_t st);

}  // namespace mm
