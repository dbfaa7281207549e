// Host-side launchers of the MoE layer's kernels (internal; the public C ABI
// is include/mm.h and is implemented in api.cu).
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mm {

// Launches kern<<<grid, block, smem, st>>>(args...). With after_prev the
// launch uses programmatic stream serialisation: it may be scheduled while
// the previous kernel of the layer finishes, and the kernel waits for it
// (griddepcontrol.wait) in every CTA before it touches memory. Only kernels
// that follow another kernel of the same layer call are launched this way.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, bool after_prev, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_prev ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

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

// Per-device first-use flags of kernel attributes. Atomic, so that host
// threads calling into the library at the same time (with distinct
// workspaces) read and set them without a data race; two threads that both
// see the flag unset both set the same attribute value, which CUDA allows.
using DeviceFlags = std::atomic<bool>[kMaxDevices];

// Raises kern's dynamic shared-memory limit to `bytes` on the current device,
// once per device.
template <typename Kern>
inline cudaError_t smem_attr_once(DeviceFlags& done, Kern kern, int bytes) {
  const int dev = current_device();
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
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
// produces the grouping. num_sms sizes the grid; err is the device status
// word (bounded waits that run out set kDevErrTimeout there).
cudaError_t launch_route(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                         int T, int H, int E, int top_k, int renorm, int32_t* topk_ids,
                         float* topk_w, float* zero_buf, long long zero_count,
                         const AlignOut* fuse_align, int num_sms, unsigned* err,
                         bool after_prev, cudaStream_t st, int32_t* tile_counts = nullptr);

// Whether launch_route runs the tensor-core router (route_tc.cu) for this
// batch, its token tile, and its launcher (same arguments, no grouping;
// tile_counts, if not NULL, receives per-tile expert counts [tiles][E] for
// launch_align_from_counts).
bool route_uses_tensor_cores(int T, int E);
int route_tc_tile_tokens(int T, int num_sms);
cudaError_t launch_route_tc(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                            int T, int H, int E, int top_k, int renorm, int32_t* topk_ids,
                            float* topk_w, float* zero_buf, long long zero_count,
                            int32_t* tile_counts, int num_sms, unsigned* err, bool after_prev,
                            cudaStream_t st);

// The grouping from per-tile expert counts the tensor-core router wrote
// (rows of tile_tokens tokens; tile_tokens divides kAlignBlockTokens): one
// launch instead of launch_align's count + place.
cudaError_t launch_align_from_counts(const int32_t* topk_ids, int T, int top_k, int E,
                                     int block_m, long long capacity,
                                     const int32_t* tile_counts, int tile_tokens, int32_t* sorted,
                                     int32_t* offsets, int32_t* counts, bool after_prev,
                                     cudaStream_t st);
// launch_align_from_counts and launch_gather_rows in one launch (one CTA per
// count row): the grouping, then xs[r] = hidden[sorted[r] / top_k] for the
// segment rows and zeros for their padding. E % 4 == 0, tile_tokens <= 128,
// H % 8 == 0 (else cudaErrorInvalidValue).
cudaError_t launch_align_place_rows(const int32_t* topk_ids, int T, int top_k, int E,
                                    int block_m, long long capacity, const int32_t* tile_counts,
                                    int tile_tokens, const uint16_t* hidden, int H, int32_t* sorted,
                                    int32_t* offsets, int32_t* counts, uint16_t* xs,
                                    bool after_prev, cudaStream_t st);

// Scratch ints the align launch needs (0 when one block covers all tokens).
long long align_scratch_ints(int T, int E, int top_k);

cudaError_t launch_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                         long long capacity, int32_t* sorted, int32_t* offsets, int32_t* counts,
                         int32_t* scratch, unsigned* err, bool after_prev, cudaStream_t st);

// Grouping of a dense MLP (one expert, every token, weight 1) + zeroed
// accumulator of zero_count floats.
cudaError_t launch_identity_grouping(int T, int block_m, long long capacity, int32_t* sorted,
                                     int32_t* offsets, float* weights, float* zero_buf,
                                     long long zero_count, int num_sms, cudaStream_t st);

// Tensor map of a row-major bf16 matrix [rows, cols] read in boxes of kb
// columns (64 or 32) x box_rows rows with the 2*kb-byte swizzle the MMA
// descriptors expect; rows past `rows` read as zeros.
bool make_tensor_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows, int kb);

// Tensor map of a bf16 tensor of `rank` (2..5) dimensions, dims[0] the
// contiguous one, strides[i] the byte stride of dimension i + 1, read in
// boxes of box[] elements with the 128-byte swizzle (box[0] * 2 == 128).
// Elements outside the dimensions read as zeros.
bool make_tensor_map_sw128(CUtensorMap* m, const void* base, uint32_t rank,
                           const uint64_t* dims, const uint64_t* strides, const uint32_t* box);

// Whether the gate_up GEMM gathers token rows with TMA tile::gather4 (few rows
// per expert) rather than with cp.async loader warps.
bool gate_up_gathers_rows(int T, int top_k, int E);

// Grouped GEMM on tcgen05. mode 0: C = act bf16 [capacity, N] = silu(gate) *
// up; X = hidden [T, K] with rows gathered through sorted / top_k when
// x_is_hidden, else X = token rows already in segment order [x_rows, K]
// (rows at or past x_rows read as zeros).
// mode 1: X = act [x_rows, K], C = fp32 acc [T, N] += topk_w * (X W^T).
// zero_buf (gate_up mode; may be NULL): zero_count floats the kernel zeroes
// before it waits for the kernels before it (the layer's accumulator).
cudaError_t launch_grouped_gemm(int mode, const uint16_t* X, bool x_is_hidden, const uint16_t* W,
                                void* C, const int32_t* sorted, const int32_t* offsets,
                                const float* topk_w, int T, int top_k, int E, int N, int K,
                                long long capacity, long long x_rows, int num_sms, unsigned* err,
                                bool after_prev, cudaStream_t st, float* zero_buf = nullptr,
                                long long zero_count = 0);

// The same grouped GEMM on SM pairs (tcgen05 cta_group::2): for token rows
// already in segment order and many rows per expert. X = xs (gate_up) or
// act (down) [x_rows, K]; otherwise as launch_grouped_gemm (no split K).
cudaError_t launch_grouped_gemm_pair(int mode, const uint16_t* X, const uint16_t* W, void* C,
                                     const int32_t* sorted, const int32_t* offsets,
                                     const float* topk_w, int T, int top_k, int E, int N, int K,
                                     long long capacity, long long x_rows, int num_sms,
                                     unsigned* err, bool after_prev, cudaStream_t st,
                                     float* zero_buf, long long zero_count);

// out[i] = bf16(acc[i]) for i < n (n % 4 == 0).
// xs[r] = hidden[sorted[r] / top_k] (H bf16 per row) for r < offsets[E];
// padding rows of the segments become zeros. H % 8 == 0.
cudaError_t launch_gather_rows(const uint16_t* hidden, const int32_t* sorted,
                               const int32_t* offsets, int T, int top_k, int E, int H,
                               uint16_t* xs, int num_sms, bool after_prev, cudaStream_t st);

// With res_out (n elements, may be res_in): res_out = bf16(out + res_in).
cudaError_t launch_finalize(const float* acc, uint16_t* out, long long n, int num_sms,
                            bool after_prev, cudaStream_t st, const uint16_t* res_in = nullptr,
                            uint16_t* res_out = nullptr);

// The single-launch layer for small batches (decode.cu): whether it can run
// this shape, whether mm_moe_forward chooses it for this shape (where it
// was measured faster than the kernel chain), the flag words its grid
// barriers need (per workspace), and the launcher. Its workspace regions: logits [T, E] fp32, the routing and the
// grouping (as the multi-kernel path), act [T*k, I] bf16, acc [T, H] fp32
// (the layer's sum, or a caller's fp32 partial), flags [decode_flag_slots]
// uint64.
bool decode_supported(int T, int H, int E, int I, int top_k);
bool decode_preferred(int T, int H, int E, int I, int top_k);
int decode_flag_slots();
struct DecodeBuffers {
  float* logits;
  int32_t* ids;
  float* w;
  int32_t* sorted;
  int32_t* offsets;
  int32_t* counts;
  long long capacity;
  uint16_t* act;
  float* acc;
  unsigned long long* flags;
};
// out NULL: acc is the result (a tensor-parallel partial); res_out: the
// residual add after the layer, res_out = bf16(out + res_in). absent_cta /
// absent_barrier (self-test of the bounded grid-wide wait): that CTA does
// not arrive at that grid barrier, so every CTA's wait there runs out.
cudaError_t launch_moe_decode(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                              const uint16_t* w_gate_up, const uint16_t* w_down, int T, int H,
                              int E, int I, int top_k, int renorm, const DecodeBuffers& b,
                              uint16_t* out, const uint16_t* res_in, uint16_t* res_out,
                              int num_sms, unsigned* err, cudaStream_t st, int absent_cta = -1,
                              int absent_barrier = -1);

// residual' = bf16(x + residual) in place (residual NULL: x is the residual),
// normed = rmsnorm(residual', weight, eps) [T, H] bf16. H % 8 == 0.
cudaError_t launch_add_rmsnorm(const uint16_t* x, uint16_t* residual, const uint16_t* weight,
                               float eps, int T, int H, uint16_t* normed, int num_sms,
                               bool after_prev, cudaStream_t st);

}  // namespace mm
