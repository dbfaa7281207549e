// The C ABI of include/mm.h: argument checks, the per-device state
// (SM count, status word, internal workspace) and the launch sequence of the
// MoE layer. Every computing step runs in the kernels of route.cu,
// route_tc.cu, align.cu, gemm.cu and norm.cu; this file only validates, lays
// out memory and launches.
#include <algorithm>
#include <mutex>

#include "mm.h"
#include "mm_device.cuh"
#include "mm_internal.h"

namespace {

using namespace mm;

// Per-device status word (each device that loads the module has its own copy).
__device__ unsigned g_status_word;

struct DevState {
  bool init = false;
  int sms = 0;
  unsigned* status = nullptr;  // device address of g_status_word
  void* ws = nullptr;          // internal workspace
  size_t ws_bytes = 0;
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Requires g_mu held.
int device_state(DevState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MM_ERR_UNSUPPORTED;
  DevState& s = g_dev[dev];
  if (!s.init) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MM_ERR_CUDA;
    if (major != 10 || minor != 3) return MM_ERR_UNSUPPORTED;  // built for sm_103a only
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&s.status), g_status_word) != cudaSuccess)
      return MM_ERR_CUDA;
    s.init = true;
  }
  *out = &s;
  return MM_OK;
}

// Grows the internal workspace to at least `bytes`. Requires g_mu held.
int ensure_ws(DevState* s, size_t bytes) {
  if (s->ws_bytes >= bytes) return MM_OK;
  if (s->ws != nullptr) {
    if (cudaDeviceSynchronize() != cudaSuccess) return MM_ERR_CUDA;  // work may still use it
    cudaFree(s->ws);
    s->ws = nullptr;
    s->ws_bytes = 0;
  }
  const size_t b = bytes + bytes / 8 + 4096;
  if (cudaMalloc(&s->ws, b) != cudaSuccess) {
    cudaGetLastError();
    s->ws = nullptr;
    return MM_ERR_NO_MEMORY;
  }
  s->ws_bytes = b;
  return MM_OK;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MM_OK : MM_ERR_CUDA; }

int check_route_shape(int T, int H, int E, int top_k) {
  if (T < 0 || H <= 0 || E <= 0 || top_k <= 0) return MM_ERR_INVALID_ARG;
  if (E > kMaxExperts || top_k > kMaxTopK || top_k > E || H % 64 != 0) return MM_ERR_UNSUPPORTED;
  if ((long long)T * top_k >= (1LL << 31) || (long long)T * H >= (1LL << 40))
    return MM_ERR_UNSUPPORTED;
  return MM_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct ForwardLayout {
  size_t normed, ids, w, sorted, offsets, counts, scratch, xs, act, acc, logits, flags,
      total;
  long long capacity;
  bool rows_in_order;  // token rows are copied into segment order before gate_up
  bool single_ok;      // the single-launch small-batch layer (decode.cu) can run
  bool decode;         // ... and mm_moe_forward chooses it
};

// gather_rows: whether a gate_up with many rows per expert reads a copy of
// the token rows in segment order (the MoE layer); a dense MLP's rows are in
// order already.
// normed: room for the rows the add + RMSNorm step hands to the layer.
ForwardLayout forward_layout(int T, int H, int E, int I, int k, bool gather_rows = true,
                             bool normed = false) {
  ForwardLayout L;
  L.capacity = (long long)T * k + (long long)E * (kForwardBlockM - 1);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += round256(bytes);
    return o;
  };
  L.normed = take(normed ? (size_t)T * H * 2 : 0);
  L.ids = take((size_t)T * k * 4);
  L.w = take((size_t)T * k * 4);
  L.sorted = take((size_t)L.capacity * 4);
  L.offsets = take((size_t)(E + 1) * 4);
  L.counts = take((size_t)E * 4);
  // Align block counts, or the tensor-core router's per-tile counts (tiles of
  // at least 32 tokens).
  long long scratch_ints = align_scratch_ints(T, E, k);
  if (route_uses_tensor_cores(T, E))
    scratch_ints = std::max(scratch_ints, ((long long)T / 32 + 1) * E);
  L.scratch = take((size_t)scratch_ints * 4);
  // Many rows per expert: gate_up reads its token rows as 2-D TMA boxes of a
  // copy in segment order (faster than gathering them inside the GEMM).
  L.rows_in_order = gather_rows && !gate_up_gathers_rows(T, k, E);
  L.xs = take(L.rows_in_order ? (size_t)L.capacity * H * 2 : 0);
  L.act = take((size_t)L.capacity * I * 2);
  L.acc = take((size_t)T * H * 4);
  // The single-launch layer of small batches: router logits and the flags
  // of its grid barriers (reserved wherever it can run, so that one
  // workspace size serves mm_moe_forward and mm_moe_forward_single_launch).
  L.single_ok = gather_rows && decode_supported(T, H, E, I, k);
  L.decode = L.single_ok && decode_preferred(T, H, E, I, k);
  L.logits = take(L.single_ok ? (size_t)T * E * 4 : 0);
  L.flags = take(L.single_ok ? (size_t)decode_flag_slots() * 8 : 0);
  L.total = off;
  return L;
}

template <typename Tp>
Tp* at(void* base, size_t off) {
  return reinterpret_cast<Tp*>(static_cast<char*>(base) + off);
}

}  // namespace

namespace mm {

int current_status_word(unsigned** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* s = nullptr;
  const int rc = device_state(&s);
  if (rc == MM_OK) *out = s->status;
  return rc;
}

}  // namespace mm

extern "C" {

const char* mm_status_string(int status) {
  switch (status) {
    case MM_OK: return "MM_OK";
    case MM_ERR_INVALID_ARG: return "MM_ERR_INVALID_ARG: invalid argument";
    case MM_ERR_UNSUPPORTED: return "MM_ERR_UNSUPPORTED: shape or device not supported";
    case MM_ERR_CUDA: return "MM_ERR_CUDA: a CUDA runtime call failed";
    case MM_ERR_NO_MEMORY: return "MM_ERR_NO_MEMORY: workspace allocation failed or too small";
    case MM_ERR_DEVICE: return "MM_ERR_DEVICE: a kernel flagged invalid input";
    case MM_ERR_TIMEOUT: return "MM_ERR_TIMEOUT: a kernel wait timed out";
    default: return "unknown mm status";
  }
}

int mm_route(const uint16_t* hidden, const uint16_t* router_w, const float* router_bias, int T,
             int H, int E, int top_k, int renorm, int32_t* topk_ids, float* topk_w,
             void* stream) {
  int rc = check_route_shape(T, H, E, top_k);
  if (rc != MM_OK) return rc;
  if (T == 0) return MM_OK;  // nothing to read or write; pointers may be NULL
  if (!hidden || !router_w || !topk_ids || !topk_w) return MM_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(router_w) || !aligned16(topk_ids) || !aligned16(topk_w))
    return MM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* s = nullptr;
  if ((rc = device_state(&s)) != MM_OK) return rc;
  return cuda_status(launch_route(hidden, router_w, router_bias, T, H, E, top_k, renorm, topk_ids,
                                  topk_w, nullptr, 0, nullptr, s->sms, s->status, false,
                                  static_cast<cudaStream_t>(stream)));
}

int64_t mm_align_capacity(int T, int top_k, int E, int block_m) {
  if (T < 0 || top_k <= 0 || E <= 0 || block_m <= 0) return -1;
  return (int64_t)T * top_k + (int64_t)E * (block_m - 1);
}

int mm_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
             int32_t* sorted_token_ids, int32_t* expert_offsets, int32_t* expert_counts,
             void* stream) {
  if (T < 0 || top_k <= 0 || E <= 0 || block_m <= 0) return MM_ERR_INVALID_ARG;
  if (E > kMaxExperts || top_k > kMaxTopK || block_m > 256) return MM_ERR_UNSUPPORTED;
  if ((long long)T * top_k + (long long)E * block_m >= (1LL << 31)) return MM_ERR_UNSUPPORTED;
  if ((T > 0 && !topk_ids) || !sorted_token_ids || !expert_offsets) return MM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* s = nullptr;
  int rc = device_state(&s);
  if (rc != MM_OK) return rc;
  const long long scratch_ints = align_scratch_ints(T, E, top_k);
  if (scratch_ints > 0 && (rc = ensure_ws(s, (size_t)scratch_ints * 4)) != MM_OK) return rc;
  return cuda_status(launch_align(topk_ids, T, top_k, E, block_m,
                                  mm_align_capacity(T, top_k, E, block_m), sorted_token_ids,
                                  expert_offsets, expert_counts, static_cast<int32_t*>(s->ws),
                                  s->status, false, static_cast<cudaStream_t>(stream)));
}

int mm_grouped_gemm(int mode, const void* A, const uint16_t* B, void* C,
                    const int32_t* sorted_token_ids, const int32_t* expert_offsets,
                    const float* topk_w, int T, int top_k, int E, int N, int K, int block_m,
                    void* stream) {
  if (mode != MM_GEMM_GATE_UP && mode != MM_GEMM_DOWN) return MM_ERR_INVALID_ARG;
  if (T < 0 || top_k <= 0 || E <= 0 || N <= 0 || K <= 0 || block_m <= 0) return MM_ERR_INVALID_ARG;
  if (E > kMaxExperts || top_k > kMaxTopK || block_m > 256 || N % 64 != 0 || K % 64 != 0)
    return MM_ERR_UNSUPPORTED;
  if (T == 0) return MM_OK;  // nothing to read or write
  if (!A || !B || !C || !sorted_token_ids || !expert_offsets) return MM_ERR_INVALID_ARG;
  if (mode == MM_GEMM_DOWN && !topk_w) return MM_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return MM_ERR_INVALID_ARG;
  const long long capacity = mm_align_capacity(T, top_k, E, block_m);
  if (capacity >= (1LL << 31)) return MM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* s = nullptr;
  int rc = device_state(&s);
  if (rc != MM_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_grouped_gemm(mode, static_cast<const uint16_t*>(A),
                                         mode == MM_GEMM_GATE_UP, B, C, sorted_token_ids,
                                         expert_offsets, topk_w, T, top_k, E, N, K, capacity,
                                         capacity, s->sms, s->status, false, st));
}

int64_t mm_moe_workspace_size(int T, int H, int E, int I, int top_k) {
  if (check_route_shape(T, H, E, top_k) != MM_OK || I <= 0 || I % 64 != 0) return -1;
  return (int64_t)forward_layout(T, H, E, I, top_k).total;
}

int mm_moe_workspace_layout(int T, int H, int E, int I, int top_k, int64_t* layout) {
  if (layout == nullptr) return MM_ERR_INVALID_ARG;
  const int rc = check_route_shape(T, H, E, top_k);
  if (rc != MM_OK) return rc;
  if (I <= 0) return MM_ERR_INVALID_ARG;
  if (I % 64 != 0) return MM_ERR_UNSUPPORTED;
  const ForwardLayout L = forward_layout(T, H, E, I, top_k);
  layout[MM_WS_TOPK_IDS] = (int64_t)L.ids;
  layout[MM_WS_TOPK_W] = (int64_t)L.w;
  layout[MM_WS_SORTED_TOKEN_IDS] = (int64_t)L.sorted;
  layout[MM_WS_EXPERT_OFFSETS] = (int64_t)L.offsets;
  layout[MM_WS_EXPERT_COUNTS] = (int64_t)L.counts;
  layout[MM_WS_CAPACITY] = (int64_t)L.capacity;
  layout[MM_WS_BLOCK_M] = kForwardBlockM;
  layout[MM_WS_TOTAL] = (int64_t)L.total;
  return MM_OK;
}

}  // extern "C"

namespace {

// The add + RMSNorm step before the layer (see mm_moe_forward_add_norm),
// and optionally the residual add after it (res_out = bf16(out + residual')).
struct NormIn {
  const uint16_t* x;
  uint16_t* residual;  // NULL: x is the residual
  const uint16_t* weight;
  float eps;
  uint16_t* res_out;   // NULL: no add after the layer
};

// The launch sequence of the layer. If `ev` is non-null, events ev[0..5] are
// recorded on the stream around the stages: route (which also groups the
// tokens when T <= 64) | align (empty then) | gate_up | down | finalize.
// With `norm`, hidden is ignored: a first kernel writes rmsnorm(x + residual)
// into the workspace and the layer reads it.
int forward_impl(const uint16_t* hidden, const uint16_t* router_w, const float* router_bias,
                 const uint16_t* w_gate_up, const uint16_t* w_down, int T, int H, int E, int I,
                 int top_k, int renorm, uint16_t* out, void* workspace, size_t workspace_bytes,
                 cudaStream_t st, cudaEvent_t const* ev, const NormIn* norm = nullptr,
                 float* partial = nullptr, bool force_single = false,
                 int absent_barrier = -1) {
  if (norm != nullptr) hidden = norm->x;  // for the checks below
  // With `partial` the layer stops before the rounding: the down GEMM adds
  // into partial (fp32, zeroed by the gate_up kernel) and out is not used.
  if (partial != nullptr) out = reinterpret_cast<uint16_t*>(partial);
  int rc = check_route_shape(T, H, E, top_k);
  if (rc != MM_OK) return rc;
  if (I <= 0) return MM_ERR_INVALID_ARG;
  if (I % 64 != 0) return MM_ERR_UNSUPPORTED;
  if (T == 0) return MM_OK;  // nothing to read or write; pointers may be NULL
  if (!hidden || !router_w || !w_gate_up || !w_down || !out) return MM_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(router_w) || !aligned16(w_gate_up) ||
      !aligned16(w_down) || !aligned16(out))
    return MM_ERR_INVALID_ARG;
  if (norm != nullptr && (!norm->weight || !aligned16(norm->weight) ||
                          (norm->residual && !aligned16(norm->residual)) || !(norm->eps >= 0.f) ||
                          (norm->res_out && !aligned16(norm->res_out))))
    return MM_ERR_INVALID_ARG;
  const ForwardLayout L = forward_layout(T, H, E, I, top_k, true, norm != nullptr);
  if (L.capacity >= (1LL << 31)) return MM_ERR_UNSUPPORTED;
  if ((force_single || absent_barrier >= 0) && !L.single_ok) return MM_ERR_UNSUPPORTED;
  const bool single = L.decode || force_single || absent_barrier >= 0;
  if (workspace != nullptr) {
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MM_ERR_INVALID_ARG;
    if (workspace_bytes < L.total) return MM_ERR_NO_MEMORY;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* s = nullptr;
  if ((rc = device_state(&s)) != MM_OK) return rc;
  void* ws = workspace;
  if (ws == nullptr) {
    if ((rc = ensure_ws(s, L.total)) != MM_OK) return rc;
    ws = s->ws;
  }
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* w = at<float>(ws, L.w);
  int32_t* sorted = at<int32_t>(ws, L.sorted);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* scratch = at<int32_t>(ws, L.scratch);
  uint16_t* act = at<uint16_t>(ws, L.act);
  float* acc = partial != nullptr ? partial : at<float>(ws, L.acc);
  const long long nacc = (long long)T * H;
  auto mark = [&](int i) { return ev == nullptr || cudaEventRecord(ev[i], st) == cudaSuccess; };

  if (!mark(0)) return MM_ERR_CUDA;
  if (norm != nullptr) {
    uint16_t* normed = at<uint16_t>(ws, L.normed);
    if (launch_add_rmsnorm(norm->x, norm->residual, norm->weight, norm->eps, T, H, normed, s->sms,
                           false, st) != cudaSuccess)
      return MM_ERR_CUDA;
    hidden = normed;
  }
  if (single) {
    // One cooperative launch for the whole layer (decode.cu). For the stage
    // events its time is the gate_up stage; the other stages are empty.
    const DecodeBuffers b = {at<float>(ws, L.logits), ids, w, sorted, offsets, counts,
                             L.capacity, act, acc, at<unsigned long long>(ws, L.flags)};
    const uint16_t* res_in = nullptr;
    uint16_t* res_out = nullptr;
    if (partial == nullptr && norm != nullptr && norm->res_out != nullptr) {
      res_in = norm->residual != nullptr ? norm->residual : norm->x;
      res_out = norm->res_out;
    }
    if (!mark(1) || !mark(2)) return MM_ERR_CUDA;
    if (launch_moe_decode(hidden, router_w, router_bias, w_gate_up, w_down, T, H, E, I, top_k,
                          renorm, b, partial != nullptr ? nullptr : out, res_in, res_out, s->sms,
                          s->status, st, absent_barrier >= 0 ? 0 : -1,
                          absent_barrier) != cudaSuccess)
      return MM_ERR_CUDA;
    if (!mark(3) || !mark(4) || !mark(5)) return MM_ERR_CUDA;
    return MM_OK;
  }
  const AlignOut fa = {sorted, offsets, counts, kForwardBlockM, L.capacity, s->status};
  const bool fused = route_fuses_align(T, top_k);
  // The accumulator is zeroed by the gate_up kernel (on every SM, while the
  // router runs), not by the router.
  // The tensor-core router also counts each tile's experts, which leaves the
  // grouping one launch.
  const bool router_counts = route_uses_tensor_cores(T, E);
  // Behind the norm kernel the cluster router is launched programmatically
  // (its launch hides behind the norm), the tensor-core router in plain
  // stream order: launched early, its CTAs made the grouping kernel after it
  // slower (T=4096: the layer behind the norm took 447 us with the early
  // launch, 440 us without; the plain layer 418 us either way).
  const bool route_after_norm = norm != nullptr && !router_counts;
  if (launch_route(hidden, router_w, router_bias, T, H, E, top_k, renorm, ids, w, nullptr, 0, &fa,
                   s->sms, s->status, route_after_norm, st,
                   router_counts ? scratch : nullptr) != cudaSuccess ||
      !mark(1))
    return MM_ERR_CUDA;
  uint16_t* xs = at<uint16_t>(ws, L.xs);
  // With the router's counts and token rows wanted in segment order, the
  // grouping and the row copy are one launch.
  const int tile_tokens = router_counts ? route_tc_tile_tokens(T, s->sms) : 0;
  const bool place_rows = router_counts && L.rows_in_order && E % 4 == 0 && tile_tokens <= 128;
  if (place_rows) {
    if (launch_align_place_rows(ids, T, top_k, E, kForwardBlockM, L.capacity, scratch,
                                tile_tokens, hidden, H, sorted, offsets, counts, xs, true,
                                st) != cudaSuccess)
      return MM_ERR_CUDA;
  } else if (router_counts) {
    if (launch_align_from_counts(ids, T, top_k, E, kForwardBlockM, L.capacity, scratch,
                                 tile_tokens, sorted, offsets, counts, true, st) != cudaSuccess)
      return MM_ERR_CUDA;
  } else if (!fused && launch_align(ids, T, top_k, E, kForwardBlockM, L.capacity, sorted, offsets,
                                    counts, scratch, s->status, true, st) != cudaSuccess) {
    return MM_ERR_CUDA;
  }
  if (L.rows_in_order && !place_rows &&
      launch_gather_rows(hidden, sorted, offsets, T, top_k, E, H, xs, s->sms, true, st) !=
          cudaSuccess)
    return MM_ERR_CUDA;
  if (!mark(2)) return MM_ERR_CUDA;
  if (launch_grouped_gemm(MM_GEMM_GATE_UP, L.rows_in_order ? xs : hidden, !L.rows_in_order,
                          w_gate_up, act, sorted, offsets, nullptr, T, top_k, E, I, H, L.capacity,
                          L.capacity, s->sms, s->status, true, st, acc, nacc) != cudaSuccess ||
      !mark(3))
    return MM_ERR_CUDA;
  if (launch_grouped_gemm(MM_GEMM_DOWN, act, false, w_down, acc, sorted, offsets, w, T, top_k, E,
                          H, I, L.capacity, L.capacity, s->sms, s->status, true, st) != cudaSuccess ||
      !mark(4))
    return MM_ERR_CUDA;
  // The rounding of the sum, and with a residual output the add that follows
  // the layer, in one pass.
  if (partial != nullptr) return MM_OK;  // the caller sums the ranks' partials and rounds
  const uint16_t* res_in = nullptr;
  uint16_t* res_out = nullptr;
  if (norm != nullptr && norm->res_out != nullptr) {
    res_in = norm->residual != nullptr ? norm->residual : norm->x;
    res_out = norm->res_out;
  }
  if (launch_finalize(acc, out, nacc, s->sms, true, st, res_in, res_out) != cudaSuccess || !mark(5))
    return MM_ERR_CUDA;
  return MM_OK;
}

}  // namespace

extern "C" {

int mm_moe_forward_ex(const uint16_t* hidden, const uint16_t* router_w, const float* router_bias,
                      const uint16_t* w_gate_up, const uint16_t* w_down, int T, int H, int E,
                      int I, int top_k, int renorm, uint16_t* out, void* workspace,
                      size_t workspace_bytes, void* stream) {
  return forward_impl(hidden, router_w, router_bias, w_gate_up, w_down, T, H, E, I, top_k, renorm,
                      out, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), nullptr);
}

int mm_moe_forward_profiled(const uint16_t* hidden, const uint16_t* router_w,
                            const float* router_bias, const uint16_t* w_gate_up,
                            const uint16_t* w_down, int T, int H, int E, int I, int top_k,
                            int renorm, uint16_t* out, void* workspace, size_t workspace_bytes,
                            void* stream, void* const* events) {
  if (events == nullptr) return MM_ERR_INVALID_ARG;
  for (int i = 0; i < MM_PROFILE_EVENTS; ++i)
    if (events[i] == nullptr) return MM_ERR_INVALID_ARG;
  return forward_impl(hidden, router_w, router_bias, w_gate_up, w_down, T, H, E, I, top_k, renorm,
                      out, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                      reinterpret_cast<cudaEvent_t const*>(events));
}

int mm_moe_forward_partial(const uint16_t* hidden, const uint16_t* router_w,
                           const float* router_bias, const uint16_t* w_gate_up_slice,
                           const uint16_t* w_down_slice, int T, int H, int E, int I_slice,
                           int top_k, int renorm, float* partial, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (T > 0 && partial == nullptr) return MM_ERR_INVALID_ARG;
  return forward_impl(hidden, router_w, router_bias, w_gate_up_slice, w_down_slice, T, H, E,
                      I_slice, top_k, renorm, nullptr, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream), nullptr, nullptr, partial);
}

int mm_selftest_layer_barrier_timeout(const uint16_t* hidden, const uint16_t* router_w,
                                      const uint16_t* w_gate_up, const uint16_t* w_down, int T,
                                      int H, int E, int I, int top_k, int renorm, int barrier,
                                      uint16_t* out, void* stream) {
  if (barrier < 0 || barrier > 2) return MM_ERR_INVALID_ARG;
  return forward_impl(hidden, router_w, nullptr, w_gate_up, w_down, T, H, E, I, top_k, renorm, out,
                      nullptr, 0, static_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr,
                      true, barrier);
}

int mm_moe_forward_single_launch(const uint16_t* hidden, const uint16_t* router_w,
                                 const float* router_bias, const uint16_t* w_gate_up,
                                 const uint16_t* w_down, int T, int H, int E, int I, int top_k,
                                 int renorm, uint16_t* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return forward_impl(hidden, router_w, router_bias, w_gate_up, w_down, T, H, E, I, top_k, renorm,
                      out, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), nullptr,
                      nullptr, nullptr, true);
}

int mm_round_bf16(const float* in, uint16_t* out, int64_t n, void* stream) {
  if (n < 0) return MM_ERR_INVALID_ARG;
  if (n % 4 != 0) return MM_ERR_UNSUPPORTED;
  if (n == 0) return MM_OK;
  if (!in || !out || !aligned16(in) || !aligned16(out)) return MM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* s = nullptr;
  int rc = device_state(&s);
  if (rc != MM_OK) return rc;
  return cuda_status(
      launch_finalize(in, out, (long long)n, s->sms, false, static_cast<cudaStream_t>(stream)));
}

int mm_moe_forward(const uint16_t* hidden, const uint16_t* router_w, const uint16_t* w_gate_up,
                   const uint16_t* w_down, int T, int H, int E, int I, int top_k, int renorm,
                   uint16_t* out, void* stream) {
  return mm_moe_forward_ex(hidden, router_w, nullptr, w_gate_up, w_down, T, H, E, I, top_k, renorm,
                           out, nullptr, 0, stream);
}

int64_t mm_gated_mlp_workspace_size(int T, int H, int I) {
  if (T < 0 || H <= 0 || I <= 0 || H % 64 != 0 || I % 64 != 0) return -1;
  return (int64_t)forward_layout(T, H, 1, I, 1, false).total;
}

int mm_gated_mlp(const uint16_t* hidden, const uint16_t* w_gate_up, const uint16_t* w_down, int T,
                 int H, int I, uint16_t* out, void* stream) {
  if (T < 0 || H <= 0 || I <= 0) return MM_ERR_INVALID_ARG;
  if (H % 64 != 0 || I % 64 != 0 || (long long)T * H >= (1LL << 40)) return MM_ERR_UNSUPPORTED;
  if (T == 0) return MM_OK;
  if (!hidden || !w_gate_up || !w_down || !out) return MM_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(out))
    return MM_ERR_INVALID_ARG;
  const ForwardLayout L = forward_layout(T, H, 1, I, 1, false);  // one expert, k = 1
  if (L.capacity >= (1LL << 31)) return MM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* s = nullptr;
  int rc = device_state(&s);
  if (rc != MM_OK) return rc;
  if ((rc = ensure_ws(s, L.total)) != MM_OK) return rc;
  void* ws = s->ws;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* w = at<float>(ws, L.w);
  int32_t* sorted = at<int32_t>(ws, L.sorted);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  uint16_t* act = at<uint16_t>(ws, L.act);
  float* acc = at<float>(ws, L.acc);
  const long long nacc = (long long)T * H;
  if (launch_identity_grouping(T, kForwardBlockM, L.capacity, sorted, offsets, w, acc, nacc, s->sms,
                               st) != cudaSuccess)
    return MM_ERR_CUDA;
  // The rows are in order already: gate_up reads hidden by 2-D TMA boxes
  // (rows past T read as zeros).
  if (launch_grouped_gemm(MM_GEMM_GATE_UP, hidden, false, w_gate_up, act, sorted, offsets, nullptr,
                          T, 1, 1, I, H, L.capacity, T, s->sms, s->status, true, st) != cudaSuccess)
    return MM_ERR_CUDA;
  if (launch_grouped_gemm(MM_GEMM_DOWN, act, false, w_down, acc, sorted, offsets, w, T, 1, 1, H, I,
                          L.capacity, L.capacity, s->sms, s->status, true, st) != cudaSuccess)
    return MM_ERR_CUDA;
  return cuda_status(launch_finalize(acc, out, nacc, s->sms, true, st));
}

int mm_add_rmsnorm(const uint16_t* x, uint16_t* residual, const uint16_t* norm_w, float eps,
                   int T, int H, uint16_t* normed, void* stream) {
  if (T < 0 || H <= 0 || !(eps >= 0.f)) return MM_ERR_INVALID_ARG;
  if (H % 64 != 0) return MM_ERR_UNSUPPORTED;
  if (T == 0) return MM_OK;
  if (!x || !norm_w || !normed) return MM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(norm_w) || !aligned16(normed) ||
      (residual && !aligned16(residual)))
    return MM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* s = nullptr;
  int rc = device_state(&s);
  if (rc != MM_OK) return rc;
  return cuda_status(launch_add_rmsnorm(x, residual, norm_w, eps, T, H, normed, s->sms, false,
                                        static_cast<cudaStream_t>(stream)));
}

int mm_moe_forward_add_norm(const uint16_t* x, uint16_t* residual, const uint16_t* norm_w,
                            float eps, const uint16_t* router_w, const uint16_t* w_gate_up,
                            const uint16_t* w_down, int T, int H, int E, int I, int top_k,
                            int renorm, uint16_t* out, void* stream) {
  const NormIn norm = {x, residual, norm_w, eps, nullptr};
  return forward_impl(nullptr, router_w, nullptr, w_gate_up, w_down, T, H, E, I, top_k, renorm,
                      out, nullptr, 0, static_cast<cudaStream_t>(stream), nullptr, &norm);
}

int mm_moe_forward_add_norm_residual(const uint16_t* x, uint16_t* residual,
                                     const uint16_t* norm_w, float eps, const uint16_t* router_w,
                                     const uint16_t* w_gate_up, const uint16_t* w_down, int T,
                                     int H, int E, int I, int top_k, int renorm, uint16_t* out,
                                     uint16_t* residual_out, void* stream) {
  if (T > 0 && residual_out == nullptr) return MM_ERR_INVALID_ARG;
  const NormIn norm = {x, residual, norm_w, eps, residual_out};
  return forward_impl(nullptr, router_w, nullptr, w_gate_up, w_down, T, H, E, I, top_k, renorm,
                      out, nullptr, 0, static_cast<cudaStream_t>(stream), nullptr, &norm);
}

int mm_poll_device_status(void* stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* s = nullptr;
  int rc = device_state(&s);
  if (rc != MM_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MM_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, s->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MM_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(s->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return MM_ERR_CUDA;
  }
  if (v & kDevErrTimeout) return MM_ERR_TIMEOUT;
  if (v & kDevErrBadIds) return MM_ERR_DEVICE;
  return MM_OK;
}

void mm_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (int d = 0; d < kMaxDevices; ++d) {
    if (g_dev[d].ws == nullptr) continue;
    if (cudaSetDevice(d) == cudaSuccess) {
      cudaDeviceSynchronize();
      cudaFree(g_dev[d].ws);
    }
    g_dev[d].ws = nullptr;
    g_dev[d].ws_bytes = 0;
  }
  if (have_cur) cudaSetDevice(cur);
}

}  // extern "C"
