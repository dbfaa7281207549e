/*
 * mm.h — C ABI of a fused Mixture-of-Experts layer for one GB300 (sm_103a).
 *
 * The layer is the Qwen3-MoE feed-forward block: for each token a router
 * linear gives one logit per expert, a softmax over all experts turns them
 * into scores, the k best experts are kept (optionally renormalised), each
 * kept expert runs a SwiGLU MLP (gate_up projection, SiLU(gate) * up, down
 * projection) and the expert outputs are summed weighted by their scores.
 * Sources: "mini-sglang guide, chapter 7" (paragraphs on layers/moe.py and
 * moe/fused.py), "The op layer: BaseOP and the layers" (Linear layers table:
 * the router is a replicated linear), "模型与权重加载" (ModelConfig MoE
 * fields; GatedMLP; streaming loader, step 4: experts stacked into [E, ...]).
 *
 * Conventions for every entry point:
 *   - Pointer arguments are DEVICE pointers on the current CUDA device unless
 *     marked host. They are owned by the caller, must be contiguous row-major,
 *     16-byte aligned, and must not alias one another.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     call is asynchronous on that stream and never synchronises the host,
 *     except mm_poll_device_status and the first call on a device (which
 *     allocates the library's state there).
 *   - Errors are returned, never raised: arguments are checked before any
 *     launch, and on error no output is written. Device-side faults that a
 *     kernel can detect (an expert id out of range, a wait that timed out)
 *     are recorded in a per-device status word read by
 *     mm_poll_device_status; kernels never trap.
 *   - Supported shapes: T >= 0, 1 <= E <= 256, 1 <= top_k <= min(E, 32),
 *     H and I multiples of 64, T*top_k < 2^31. Anything else returns
 *     MM_ERR_UNSUPPORTED (or MM_ERR_INVALID_ARG for values that make no sense).
 */
#ifndef MM_H
#define MM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MM_OK = 0,
  MM_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned pointer */
  MM_ERR_UNSUPPORTED = 2,   /* valid but outside the supported shapes */
  MM_ERR_CUDA = 3,          /* a CUDA runtime call failed */
  MM_ERR_NO_MEMORY = 4,     /* workspace allocation failed or too small */
  MM_ERR_DEVICE = 5,        /* a kernel flagged bad input (e.g. expert id out of range) */
  MM_ERR_TIMEOUT = 6        /* a kernel's bounded wait ran out and it returned early */
} mm_status;

/* Gemm modes of mm_grouped_gemm. */
enum { MM_GEMM_GATE_UP = 0, MM_GEMM_DOWN = 1 };

/* Human-readable name of a status code (static storage; never NULL). */
const char* mm_status_string(int status);

/*
 * Routing: router logits, softmax over all E experts, top-k, weights.
 * ("mini-sglang guide, chapter 7", layers/moe.py; "模型与权重加载",
 * ModelConfig: num_experts = E, num_experts_per_tok = top_k, norm_topk_prob.)
 *
 *   logit[t,e]   = sum_h hidden[t,h] * router_w[e,h] (+ router_bias[e]),
 *                  bf16 products accumulated in fp32
 *   p[t,e]       = softmax over all E of logit[t,:]
 *   topk_ids[t,:]= the top_k experts with the largest logit (equal logits: the
 *                  lower id wins), written in ASCENDING expert order
 *   topk_w[t,j]  = p[t, topk_ids[t,j]]; if renorm != 0, divided by the sum
 *                  of the selected p (norm_topk_prob)
 *
 * hidden [T,H] bf16, router_w [E,H] bf16, router_bias [E] fp32 or NULL;
 * outputs topk_ids [T,top_k] int32, topk_w [T,top_k] fp32.
 * T == 0 is a no-op.
 */
int mm_route(const uint16_t* hidden, const uint16_t* router_w, const float* router_bias,
             int T, int H, int E, int top_k, int renorm,
             int32_t* topk_ids, float* topk_w, void* stream);

/*
 * Length of the sorted_token_ids buffer mm_align needs: T*top_k +
 * E*(block_m-1) (each expert wastes fewer than block_m padding slots).
 * Returns -1 for invalid arguments. Host-only, no CUDA call.
 */
int64_t mm_align_capacity(int T, int top_k, int E, int block_m);

/*
 * Token batching by expert ("mini-sglang guide, chapter 7", moe/fused.py:
 * tokens are grouped by their assigned expert so each expert's weights are
 * read once with coalesced accesses).
 *
 * A stable counting sort of the flat assignment ids f = t*top_k + j by
 * expert id topk_ids[f]. Expert e owns slots [expert_offsets[e],
 * expert_offsets[e+1]) of sorted_token_ids: its assignments in increasing f,
 * then padding entries equal to T*top_k up to a multiple of block_m. Experts
 * without assignments own no slots. expert_offsets[E] is the padded total;
 * slots from there up to mm_align_capacity() hold T*top_k as well.
 *
 * topk_ids [T,top_k] int32 (each row: distinct ids in [0,E)); outputs
 * sorted_token_ids [mm_align_capacity()] int32, expert_offsets [E+1] int32,
 * expert_counts [E] int32 or NULL. 1 <= block_m <= 256. Ids outside [0,E) or
 * repeated within a row are dropped and flag MM_ERR_DEVICE in the device
 * status. For T > 1024 (or T*top_k > 8192) the library's internal
 * workspace holds per-block counts, so calls on one device must not overlap;
 * the result is deterministic (bit-identical on every call).
 */
int mm_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
             int32_t* sorted_token_ids, int32_t* expert_offsets, int32_t* expert_counts,
             void* stream);

/*
 * mm_align for callers that cannot allocate device memory: a serving engine
 * whose memory pool already owns the device, or code running where neither a
 * cudaMalloc nor the device-wide synchronisation that growing mm_align's
 * internal workspace implies is allowed. (The pages have no counterpart: this
 * entry point exists for such callers only.)
 *
 * Same arguments, outputs and result as mm_align (bit-identical). The caller
 * still passes every input and output. When mm_align would use scratch memory
 * (T > 1024 or T*top_k > 8192: ceil(T/256) * E per-block counts), this entry
 * point keeps those counts in a fixed device array of
 * MM_ALIGN_NOALLOC_MAX_SCRATCH_INTS int32 (128 KB) that every GPU loading the
 * library holds until exit; sizes needing more (e.g. T > 65536 at E = 128)
 * return MM_ERR_UNSUPPORTED before any CUDA call. The first call on a device
 * looks up the array's device address (a one-time set-up, no allocation);
 * make that first call before any stream capture. Every call shares the one
 * array per device, so calls whose executions overlap on the GPU (other
 * streams, other threads) race and must be serialised by the caller. Each
 * call rewrites every entry it reads, so nothing has to be cleared between
 * calls.
 */
#define MM_ALIGN_NOALLOC_MAX_SCRATCH_INTS 32768
int mm_align_noalloc(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                     int32_t* sorted_token_ids, int32_t* expert_offsets, int32_t* expert_counts,
                     void* stream);

/*
 * One grouped GEMM over the expert segments that mm_align produced, on the
 * 5th-generation tensor cores (bf16 operands, fp32 accumulation in tensor
 * memory). For every expert e and every slot r in its segment:
 *
 * mode MM_GEMM_GATE_UP ("模型与权重加载", GatedMLP: gate_up_proj then
 *   silu_and_mul; rows [0,N) of each expert's matrix are gate, [N,2N) up):
 *     A = hidden [T,K] bf16, row r reads token sorted_token_ids[r] / top_k
 *         (padding rows read zeros)
 *     B = w_gate_up [E, 2N, K] bf16
 *     C = act [capacity, N] bf16:  act[r,n] = silu(g) * u,
 *         g = A_r . B[e,n,:], u = A_r . B[e,N+n,:]   (fp32, one bf16 rounding)
 *     topk_w unused (may be NULL).
 * mode MM_GEMM_DOWN ("模型与权重加载", GatedMLP: down_proj; "mini-sglang
 *   guide, chapter 7": expert outputs weighted by their scores and summed):
 *     A = act [capacity, K] bf16, B = w_down [E, N, K] bf16,
 *     C = acc [T, N] fp32:  acc[f / top_k, n] += topk_w[f] * (A_r . B[e,n,:])
 *         for every real slot (f = sorted_token_ids[r] < T*top_k), by atomic
 *         fp32 adds (summation order is not fixed). The caller zeroes acc.
 *
 * capacity = mm_align_capacity(T, top_k, E, block_m). Token rows are
 * gathered from hidden inside the kernel (TMA tile::gather4 with few rows per
 * expert, cp.async with many); no workspace is used. N and K multiples of 64.
 */
int mm_grouped_gemm(int mode, const void* A, const uint16_t* B, void* C,
                    const int32_t* sorted_token_ids, const int32_t* expert_offsets,
                    const float* topk_w, int T, int top_k, int E, int N, int K, int block_m,
                    void* stream);

/*
 * The whole MoE layer: route, align, gate_up GEMM + SiLU*up, down GEMM +
 * weighted scatter-add, and the fp32 -> bf16 rounding of the sum.
 *
 * hidden [T,H] bf16, router_w [E,H] bf16, w_gate_up [E,2I,H] bf16 (gate rows
 * first), w_down [E,H,I] bf16; out [T,H] bf16. Uses the library's internal
 * per-device workspace (grown on demand with cudaMalloc, which synchronises
 * the device the first time a larger size is needed); calls on one device
 * must therefore not overlap. T == 0 is a no-op.
 *
 * Batches of at most 16 tokens whose shape the single-launch layer takes
 * (see mm_moe_forward_single_launch) run as that one launch; other batches
 * run as a chain of kernels (router, grouping, gate_up, down, rounding).
 * Both give the same routing and grouping and the same result within the
 * rounding of the fp32 accumulation order.
 */
int mm_moe_forward(const uint16_t* hidden, const uint16_t* router_w,
                   const uint16_t* w_gate_up, const uint16_t* w_down,
                   int T, int H, int E, int I, int top_k, int renorm,
                   uint16_t* out, void* stream);

/* Bytes of workspace mm_moe_forward_ex needs for these sizes (-1 if invalid). */
int64_t mm_moe_workspace_size(int T, int H, int E, int I, int top_k);

/*
 * mm_moe_forward with an optional router bias (fp32 [E] added to the
 * logits, NULL for none) and an optional caller workspace: if `workspace` is
 * non-NULL it must hold at least mm_moe_workspace_size() bytes (256-byte
 * aligned) and the call allocates nothing; calls with distinct workspaces may
 * run concurrently. If `workspace` is NULL the internal workspace is used.
 */
int mm_moe_forward_ex(const uint16_t* hidden, const uint16_t* router_w,
                      const float* router_bias,
                      const uint16_t* w_gate_up, const uint16_t* w_down,
                      int T, int H, int E, int I, int top_k, int renorm,
                      uint16_t* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Where a call of mm_moe_forward_ex with a caller workspace leaves its
 * routing and its grouping ("mini-sglang guide, chapter 7": the router's
 * top-k of layers/moe.py, the token batching by expert of moe/fused.py), so
 * that the caller can read them after the call's kernels have completed.
 * Host-only: no CUDA call, nothing allocated.
 *
 * layout: a host array of MM_WS_LAYOUT_FIELDS int64 that receives
 *   [MM_WS_TOPK_IDS]          byte offset of topk_ids [T, top_k] int32 (as mm_route)
 *   [MM_WS_TOPK_W]            byte offset of topk_w [T, top_k] fp32 (as mm_route)
 *   [MM_WS_SORTED_TOKEN_IDS]  byte offset of sorted_token_ids [capacity] int32
 *   [MM_WS_EXPERT_OFFSETS]    byte offset of expert_offsets [E+1] int32
 *   [MM_WS_EXPERT_COUNTS]     byte offset of expert_counts [E] int32
 *   [MM_WS_CAPACITY]          capacity = mm_align_capacity(T, top_k, E, block_m)
 *   [MM_WS_BLOCK_M]           the block_m the forward pads expert segments to
 *   [MM_WS_TOTAL]             mm_moe_workspace_size(T, H, E, I, top_k)
 * Offsets are from the start of the workspace and 256-byte aligned. The
 * grouping is exactly mm_align(topk_ids, T, top_k, E, block_m) (bit for
 * bit), whichever kernels the forward used for this batch size. The contents
 * stay valid until the workspace is passed to another call.
 * Returns MM_OK, or the code mm_moe_workspace_size's checks give
 * (MM_ERR_INVALID_ARG / MM_ERR_UNSUPPORTED; also for layout == NULL).
 */
enum {
  MM_WS_TOPK_IDS = 0,
  MM_WS_TOPK_W = 1,
  MM_WS_SORTED_TOKEN_IDS = 2,
  MM_WS_EXPERT_OFFSETS = 3,
  MM_WS_EXPERT_COUNTS = 4,
  MM_WS_CAPACITY = 5,
  MM_WS_BLOCK_M = 6,
  MM_WS_TOTAL = 7,
  MM_WS_LAYOUT_FIELDS = 8
};
int mm_moe_workspace_layout(int T, int H, int E, int I, int top_k, int64_t* layout);

/*
 * The layer split over W GPUs by tensor parallelism ("The op layer: BaseOP
 * and the layers", "Linear layers": gate_up is a merged column-parallel
 * linear, down a row-parallel linear followed by an all-reduce, the router
 * a replicated linear). Rank r holds, for every expert, the intermediate
 * slice [i0, i0 + I_slice): the gate rows [i0, i0 + I_slice) and the up rows
 * [I + i0, I + i0 + I_slice) of w_gate_up, stored together as
 * w_gate_up_slice [E, 2*I_slice, H] (gate slice first), and the columns
 * [i0, i0 + I_slice) of w_down, stored as w_down_slice [E, H, I_slice].
 * SiLU(gate) * up is elementwise over the intermediates, so the layer is the
 * sum over the slices of
 *   partial[t,:] = sum_j w[t,j] * W_down_slice[e_j] (silu(g_slice) * u_slice)
 * which this call writes, in fp32 and unrounded, to partial [T,H] (caller-
 * owned, overwritten). The routing comes from the replicated router and is
 * the same on every rank. The caller sums the W partials (one all-reduce)
 * and rounds the sum once with mm_round_bf16. Arguments as
 * mm_moe_forward_ex with I = I_slice (a multiple of 64); partial replaces
 * out. The fp32 sum of a rank's own experts' contributions has no fixed
 * order (atomic adds), as in mm_moe_forward.
 */
int mm_moe_forward_partial(const uint16_t* hidden, const uint16_t* router_w,
                           const float* router_bias, const uint16_t* w_gate_up_slice,
                           const uint16_t* w_down_slice, int T, int H, int E, int I_slice,
                           int top_k, int renorm, float* partial, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * out[i] = bf16(in[i]) (round to nearest even) for i < n: the rounding of
 * the all-reduced partials of mm_moe_forward_partial. n % 4 == 0 (else
 * MM_ERR_UNSUPPORTED); in fp32 and out bf16 are device pointers, 16-byte
 * aligned.
 */
int mm_round_bf16(const float* in, uint16_t* out, int64_t n, void* stream);

/*
 * The dense SwiGLU MLP, through the same grouped-GEMM kernels: out =
 * down_proj(silu(gate_proj(x)) * up_proj(x)) for every token ("模型与权重加载",
 * GatedMLP; Qwen3 dense layers, and the MoE model's mlp_only_layers named in
 * its ModelConfig). Equal to mm_moe_forward with one expert, top_k = 1 and a
 * routing weight of 1, without the router.
 *
 * hidden [T,H] bf16, w_gate_up [2I,H] bf16 (gate rows first), w_down [H,I]
 * bf16; out [T,H] bf16 (one rounding of the fp32 result). Uses the internal
 * workspace (mm_gated_mlp_workspace_size bytes), so calls on one device must
 * not overlap. T == 0 is a no-op.
 */
int mm_gated_mlp(const uint16_t* hidden, const uint16_t* w_gate_up, const uint16_t* w_down,
                 int T, int H, int I, uint16_t* out, void* stream);

/* Bytes of internal workspace mm_gated_mlp uses for these sizes (-1 if invalid). */
int64_t mm_gated_mlp_workspace_size(int T, int H, int I);

/*
 * The residual add + RMSNorm that precedes the MoE block in a decoder layer
 * ("The op layer: BaseOP and the layers": the rmsnorm / fused_add_rmsnorm
 * listings of "Ops: reference implementations and dispatch"; RMSNormFused and
 * the post_attention_layernorm of DecoderLayer.forward in "RMSNorm and the
 * residual"):
 *   residual' = bf16(x + residual)                  (written back to residual)
 *   normed    = bf16(norm_w * bf16(residual' * rsqrt(mean(residual'^2) + eps)))
 * With residual == NULL (the first layer) x is the residual and is only read.
 * The float32 sum of squares runs in a fixed order (32 lanes each summing
 * the 8-element chunks c = lane, lane + 32, ... in order, then an xor
 * butterfly) and rsqrt is 1/sqrt with both steps rounded, so normed is the
 * same on every call. Against the exact mean of the squares, that float32
 * sum is off by a few ulps, which can move an element of normed by a bf16
 * rounding step where it sits on a rounding boundary.
 *
 * x, residual, normed [T,H] bf16 row-major; norm_w [H] bf16; eps >= 0.
 * Caller-owned device pointers, 16-byte aligned; x, residual and normed must
 * not overlap. H % 64 != 0 -> MM_ERR_UNSUPPORTED. T == 0 is a no-op.
 */
int mm_add_rmsnorm(const uint16_t* x, uint16_t* residual, const uint16_t* norm_w, float eps,
                   int T, int H, uint16_t* normed, void* stream);

/*
 * The MoE layer behind that step, in one call: residual' and normed as in
 * mm_add_rmsnorm (normed kept in the library's workspace), then
 * out = mm_moe_forward(normed, ...). Same arguments as mm_moe_forward plus
 * x / residual / norm_w / eps (no router bias). The kernels run back to back
 * on `stream`; the normed rows never leave the library.
 */
int mm_moe_forward_add_norm(const uint16_t* x, uint16_t* residual, const uint16_t* norm_w,
                            float eps, const uint16_t* router_w, const uint16_t* w_gate_up,
                            const uint16_t* w_down, int T, int H, int E, int I, int top_k,
                            int renorm, uint16_t* out, void* stream);

/*
 * The MoE half of a decoder layer with both residual adds ("The op layer:
 * BaseOP and the layers", "RMSNorm and the residual": DecoderLayer.forward
 * adds the residual before post_attention_layernorm, and the next layer's
 * fused_add_rmsnorm adds the MLP output to it):
 *   residual'    = bf16(x + residual), normed = rmsnorm(residual')
 *                  (as mm_moe_forward_add_norm; residual == NULL: residual' = x)
 *   out          = mm_moe_forward(normed, ...)
 *   residual_out = bf16(out + residual')   (out rounded to bf16 first)
 * The last add runs in the same pass that rounds the layer's fp32 sum into
 * out (one read of the sum and of residual', one write of out and of
 * residual_out). residual_out [T,H] bf16 is required; it may be
 * residual itself (in-place update of the residual stream) but must not
 * overlap x or out. The next layer then needs only an RMSNorm of
 * residual_out (mm_add_rmsnorm with residual == NULL).
 */
int mm_moe_forward_add_norm_residual(const uint16_t* x, uint16_t* residual,
                                     const uint16_t* norm_w, float eps, const uint16_t* router_w,
                                     const uint16_t* w_gate_up, const uint16_t* w_down, int T,
                                     int H, int E, int I, int top_k, int renorm, uint16_t* out,
                                     uint16_t* residual_out, void* stream);

/*
 * Stage timing of mm_moe_forward_ex, for profiling. Same arguments, plus
 * `events`: a host array of MM_PROFILE_EVENTS cudaEvent_t handles (created
 * by the caller with timing enabled). events[i] is recorded on `stream`
 * before stage i and events[5] after the last one; the stages are
 * 0 route (which also does the grouping when T <= 64), 1 align (then
 * empty), 2 gate_up GEMM, 3 down GEMM, 4 fp32 -> bf16 rounding. No stage is
 * skipped or changed; nothing is synchronised. (Measurement support: the
 * pages describe no counterpart.)
 */
#define MM_PROFILE_EVENTS 6
int mm_moe_forward_profiled(const uint16_t* hidden, const uint16_t* router_w,
                            const float* router_bias,
                            const uint16_t* w_gate_up, const uint16_t* w_down,
                            int T, int H, int E, int I, int top_k, int renorm,
                            uint16_t* out, void* workspace, size_t workspace_bytes, void* stream,
                            void* const* events);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word. Returns MM_OK, MM_ERR_DEVICE (bad ids seen), MM_ERR_TIMEOUT (a kernel
 * gave up waiting and returned early; its outputs are undefined) or
 * MM_ERR_CUDA.
 */
int mm_poll_device_status(void* stream);

/*
 * Self-test of the failure path (no counterpart on the pages): launches one
 * kernel whose mbarrier wait can never complete. Its bounded wait, the one
 * every kernel of the library uses, gives up after about a second, records
 * the timeout in the device status word and returns; the next
 * mm_poll_device_status then reports MM_ERR_TIMEOUT (and clears the word).
 * Nothing faults or hangs, and the context stays usable.
 */
int mm_selftest_wait_timeout(void* stream);

/*
 * The MoE layer for a small batch in one cooperative launch (one CTA per
 * SM), for T <= 64, T*top_k <= 512, E <= 256, H a multiple of 256 up to 2048
 * and I a multiple of 128 up to 1024 (otherwise MM_ERR_UNSUPPORTED; T == 0 is
 * a no-op). Same arguments, outputs and workspace (mm_moe_workspace_size,
 * with the routing and grouping left at mm_moe_workspace_layout's offsets)
 * as mm_moe_forward_ex. Every CTA computes its share of the router logits;
 * after a grid-wide wait every CTA finishes all tokens' routing (softmax
 * over all experts, top-k, weights) and groups them by expert itself; the
 * selected experts' weights then stream through shared memory for gate_up
 * (+ SiLU*up) and down (weighted, added up in fp32), with grid-wide waits
 * before down and before the rounding ("mini-sglang guide, chapter 7",
 * paragraph on moe/fused.py: the fused MoE as a single kernel call). Every
 * grid-wide wait is bounded: after about a second it records MM_ERR_TIMEOUT
 * in the device status word (mm_poll_device_status) and returns.
 * mm_moe_forward takes this path by itself for T <= 16.
 */
int mm_moe_forward_single_launch(const uint16_t* hidden, const uint16_t* router_w,
                                 const float* router_bias, const uint16_t* w_gate_up,
                                 const uint16_t* w_down, int T, int H, int E, int I, int top_k,
                                 int renorm, uint16_t* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Self-test of the single-launch small-batch layer's grid-wide waits (no
 * counterpart on the pages). Runs mm_moe_forward_single_launch on the given
 * inputs (its shape limits apply; otherwise MM_ERR_UNSUPPORTED), with one
 * flag set by
 * the host: CTA 0 does not arrive at grid barrier `barrier` (0: after the
 * router logits, 1: after gate_up, 2: after down). Every CTA's bounded wait
 * at that barrier runs out after about a second, records MM_ERR_TIMEOUT in
 * the device status word and returns (the weight-streaming warp first waits
 * for its copies in flight). `out` is left undefined. barrier outside 0..2:
 * MM_ERR_INVALID_ARG. Nothing faults or hangs, and the context stays usable.
 */
int mm_selftest_layer_barrier_timeout(const uint16_t* hidden, const uint16_t* router_w,
                                      const uint16_t* w_gate_up, const uint16_t* w_down, int T,
                                      int H, int E, int I, int top_k, int renorm, int barrier,
                                      uint16_t* out, void* stream);

/* Frees the internal workspaces of every device. Not thread-safe with calls in flight. */
void mm_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* MM_H */
