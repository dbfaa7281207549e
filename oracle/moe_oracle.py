"""CPU oracle for the fused Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or runs
this module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` do. It shares no code with the CUDA path; the two meet only
through the seeded inputs of ``mixture_experts_layer_mm_gb300.synthetic``.

What it computes (plain numpy, float32 as the layer's definition asks, with a
float64 variant of the expert loop and a dense brute force for pinning it):

  route    router logits -> softmax over ALL experts -> top-k -> weights
           ("mini-sglang guide, chapter 7", paragraph on ``layers/moe.py``:
           the router is a linear layer giving per-expert logits, the top-k are
           picked, and the expert outputs are weighted by softmax scores and
           summed; "模型与权重加载", ModelConfig: ``num_experts``,
           ``num_experts_per_tok``, ``norm_topk_prob``; "The op layer: BaseOP
           and the layers", Linear layers table: the router is a replicated,
           unsharded linear).
  align    token batching by expert: a stable, block-padded grouping of the
           flat (token, slot) ids by expert ("mini-sglang guide, chapter 7",
           paragraph on ``moe/fused.py``).
  norm     the residual add + RMSNorm before the MoE ("The op layer: BaseOP
           and the layers": the ``rmsnorm`` / ``fused_add_rmsnorm`` listings
           of "Ops: reference implementations and dispatch"; RMSNormFused and
           ``DecoderLayer.forward`` of "RMSNorm and the residual"), in the
           pages' rounding order.
  experts  per expert: gate_up projection, SiLU(gate) * up, down projection
           ("模型与权重加载", GatedMLP: gate_up_proj -> silu_and_mul ->
           down_proj, gate rows before up rows; streaming loader, step 4:
           experts stacked into [E, ...]), then the routing-weighted sum.

Readings taken where the pages are silent: fp32 logits (rounding them to
bf16 would make top-k ties common); softmax over all E before top-k; larger logit
wins and equal logits go to the lower expert id; slot order within a token is
ascending expert id; norm_topk_prob divides the selected probabilities by their
sum; grouping within an expert is by increasing flat id f = t*k + j; padding
sentinel = T*k; rows [0, I) of w_gate_up[e] are gate, [I, 2I) are up; the
mean of squares in RMSNorm is the exact mean rounded once to float32.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
closed forms, invariants, brute force over all k-subsets, a dense masked
formulation, the textbook dense SwiGLU MLP, torch's bf16 cast and bf16 add,
torch's float64 rms_norm, and a hand-worked add + RMSNorm example
(``tests/golden/add_rmsnorm_worked.json``). No function is unpinned.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------- inputs ---

def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exactly (bf16 is the top half
    of an IEEE binary32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bit pattern (uint16) of the nearest bf16, ties to even
    (what a cast to bf16 does); NaN stays NaN. Written out on the integer
    bits: add half an ulp of the dropped 16 bits, plus one when the kept part
    is odd (so an exact half rounds to even), then drop them."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    out[nan] = ((b[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)  # quiet NaN
    return out


# ------------------------------------------------------ add + RMSNorm ---
#
# The step before the MoE in a decoder layer ("The op layer: BaseOP and the
# layers", sections "Ops: reference implementations and dispatch" for the
# ``rmsnorm`` / ``fused_add_rmsnorm`` listings and "RMSNorm and the residual"
# for RMSNormFused and ``DecoderLayer.forward``):
# residual <- x + residual (in the bf16 dtype of the tensors); then
# y = r * rsqrt(mean(r^2) + eps) in float32, rounded to bf16, times the
# weight, rounded to bf16. The pages fix the mean of the squares but not the
# order in which a float32 implementation sums them; the oracle takes the
# plain definition: the sum in float64 (the squares of bf16 values are exact
# there, and the sum of a few thousand of them is exact to ~1e-13 relative),
# divided by H and rounded once to float32. An implementation that sums in
# float32 in any order lands within a few float32 ulps of that mean, so its
# bf16 outputs may differ from the oracle's by a rounding step where a value
# sits on a bf16 rounding boundary. rsqrt(v) is read as 1 / sqrt(v), each
# step rounded to float32.

def mean_of_squares(xf: np.ndarray) -> np.ndarray:
    """mean(xf**2) over the last axis: float64 sum / H, rounded to float32."""
    x64 = np.asarray(xf, dtype=np.float32).astype(np.float64)
    return (np.sum(x64 * x64, axis=-1) / x64.shape[-1]).astype(np.float32)


def rmsnorm(x_bits: np.ndarray, weight_bits: np.ndarray, eps: float) -> np.ndarray:
    """bf16 rows x [.., H], bf16 weight [H] -> bf16 bit patterns of
    weight * bf16(x * rsqrt(mean(x^2) + eps))."""
    xf = widen_bf16(x_bits)
    mean = mean_of_squares(xf)
    inv = np.float32(1.0) / np.sqrt(mean + np.float32(eps), dtype=np.float32)
    y = round_bf16(xf * inv[..., None])
    return round_bf16(widen_bf16(weight_bits)[None, :] * widen_bf16(y))


def fused_add_rmsnorm(x_bits, residual_bits, weight_bits, eps: float):
    """Returns (normalised rows, new residual), both bf16 bit patterns:
    residual' = bf16(x + residual); normalised = rmsnorm(residual'). With
    residual None (the first layer) x itself is the residual."""
    if residual_bits is None:
        r = np.asarray(x_bits, dtype=np.uint16).copy()
    else:
        r = round_bf16(widen_bf16(x_bits) + widen_bf16(residual_bits))
    return rmsnorm(r, weight_bits, eps), r


# --------------------------------------------------------------- routing ---

def router_logits(x: np.ndarray, router_w: np.ndarray, bias=None) -> np.ndarray:
    """logit[t, e] = sum_h x[t, h] * Wr[e, h] (+ bias[e]), in float32.

    The router is one linear layer (chapter 7, ``layers/moe.py``; Linear
    layers table: ``LinearReplicated``). Inputs are already-widened fp32."""
    logits = np.matmul(x.astype(np.float32), router_w.astype(np.float32).T)
    if bias is not None:
        logits = logits + np.asarray(bias, dtype=np.float32)[None, :]
    return logits.astype(np.float32)


def softmax_over_experts(logits: np.ndarray) -> np.ndarray:
    """p[t, e] = exp(l[t,e] - max_e l) / sum_e exp(l[t,e] - max_e l), over all
    E experts (the "softmax scores" of chapter 7, ``layers/moe.py``)."""
    l = logits.astype(np.float32)
    m = l.max(axis=1, keepdims=True)
    z = np.exp(l - m)
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """ids[t, :] = the k experts with the largest logits, ties to the lower id,
    returned in ascending expert order (chapter 7: top-k via ``torch.topk``;
    tie-break and slot order are readings, the pages leave them open)."""
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("top_k must be in [1, E]")
    # A stable sort of -logit keeps equal logits in increasing id order.
    order = np.argsort(-logits.astype(np.float32), axis=1, kind="stable")[:, :k]
    return np.sort(order, axis=1).astype(np.int32)


def routing_weights(probs: np.ndarray, ids: np.ndarray, renorm: bool) -> np.ndarray:
    """w[t, j] = p[t, ids[t, j]]; with norm_topk_prob the selected
    probabilities are divided by their sum ("模型与权重加载", ModelConfig:
    ``norm_topk_prob``, default False)."""
    w = np.take_along_axis(probs, ids.astype(np.int64), axis=1).astype(np.float32)
    if renorm:
        w = w / w.sum(axis=1, keepdims=True)
    return w.astype(np.float32)


def route(hidden_bits, router_w_bits, top_k: int, renorm: bool, bias=None):
    """The whole routing step on bf16 inputs: returns (ids int32 [T,k],
    weights fp32 [T,k], logits fp32 [T,E])."""
    logits = router_logits(widen_bf16(hidden_bits), widen_bf16(router_w_bits), bias)
    probs = softmax_over_experts(logits)
    ids = select_topk(logits, top_k)
    return ids, routing_weights(probs, ids, renorm), logits


def near_tie_tokens(logits: np.ndarray, k: int, gap: float = 1e-4) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest logits differ by at most ``gap``.
    For these, either expert is a correct choice and ids may legitimately differ
    between two fp32 implementations that sum in different orders."""
    T, E = logits.shape
    if k >= E:
        return np.zeros(T, dtype=bool)
    s = -np.sort(-logits.astype(np.float64), axis=1)
    return (s[:, k - 1] - s[:, k]) <= gap


# ----------------------------------------------------------------- align ---

def align_capacity(T: int, k: int, E: int, block_m: int) -> int:
    """Upper bound of the padded length: every expert wastes < block_m slots."""
    return T * k + E * (block_m - 1)


def align(ids: np.ndarray, E: int, block_m: int):
    """Token batching by expert (chapter 7, ``moe/fused.py``: the kernel groups
    tokens by their assigned expert).

    Returns (sorted_token_ids [capacity] int32, expert_offsets [E+1] int32,
    expert_counts [E] int32). Expert e owns slots [offsets[e], offsets[e+1]);
    its real entries are the flat ids f = t*k + j with ids[t, j] == e, in
    increasing f, followed by sentinels T*k up to a multiple of block_m.
    Experts with no tokens own no slots. Slots past offsets[E] hold T*k."""
    T, k = ids.shape
    flat = ids.reshape(-1).astype(np.int64)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    padded = (counts + block_m - 1) // block_m * block_m
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    sentinel = T * k
    out = np.full(align_capacity(T, k, E, block_m), sentinel, dtype=np.int64)
    order = np.argsort(flat, kind="stable")  # increasing f within each expert
    pos = 0
    for e in range(E):
        c = int(counts[e])
        out[offsets[e]:offsets[e] + c] = order[pos:pos + c]
        pos += c
    return out.astype(np.int32), offsets.astype(np.int32), counts.astype(np.int32)


# --------------------------------------------------------------- experts ---

def silu_and_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """silu(g) * u with silu(g) = g / (1 + exp(-g)) ("模型与权重加载",
    section 模型结构, GatedMLP: hidden_act "silu", gate_up_proj -> silu x up)."""
    with np.errstate(over="ignore"):
        return g / (1 + np.exp(-g)) * u


def experts_loop(hidden_bits, w_gate_up_bits, w_down_bits, ids, weights,
                 dtype=np.float32) -> np.ndarray:
    """The loop-over-experts MoE: for each expert, run its SwiGLU MLP on the
    tokens routed to it and add the routing-weighted result into out[T, H].

    This is the plain formulation the fused backend replaces (chapter 7,
    ``moe/fused.py``); the expert MLP is GatedMLP ("模型与权重加载"): gate_up
    projection with gate rows [0, I) and up rows [I, 2I) of w_gate_up[e],
    silu(gate) * up, then the down projection w_down[e]. Arithmetic in
    ``dtype`` (float32 by default)."""
    T, H = hidden_bits.shape
    E, twoI, _ = w_gate_up_bits.shape
    I = twoI // 2
    x = widen_bf16(hidden_bits).astype(dtype)
    out = np.zeros((T, H), dtype=dtype)
    for e in range(E):
        tok, slot = np.nonzero(ids == e)  # a token holds expert e at most once
        if tok.size == 0:
            continue
        wgu = widen_bf16(w_gate_up_bits[e]).astype(dtype)
        wd = widen_bf16(w_down_bits[e]).astype(dtype)
        xe = x[tok]
        g = xe @ wgu[:I].T
        u = xe @ wgu[I:].T
        a = silu_and_mul(g, u).astype(dtype)
        y = a @ wd.T
        out[tok] += weights[tok, slot].astype(dtype)[:, None] * y
    return out


def experts_dense_bruteforce(hidden_bits, w_gate_up_bits, w_down_bits, ids, weights):
    """Dense formulation, float64: every expert on every token, then a mask
    that keeps the routed ones, scaled by their weights, summed over experts.
    Independent of the grouping the loop above does; small inputs only."""
    x = widen_bf16(hidden_bits).astype(np.float64)
    wgu = widen_bf16(w_gate_up_bits).astype(np.float64)
    wd = widen_bf16(w_down_bits).astype(np.float64)
    T = x.shape[0]
    E, twoI, _ = wgu.shape
    I = twoI // 2
    gu = np.einsum("th,enh->ten", x, wgu)            # [T, E, 2I]
    a = silu_and_mul(gu[:, :, :I], gu[:, :, I:])    # [T, E, I]
    y = np.einsum("tei,eoi->teo", a, wd)            # [T, E, H]
    mask = np.zeros((T, E), dtype=np.float64)
    for j in range(ids.shape[1]):
        mask[np.arange(T), ids[:, j]] += weights[:, j].astype(np.float64)
    return np.einsum("te,teo->to", mask, y)


# ------------------------------------------------------------ full layer ---

def moe_layer(inputs: dict, top_k: int, renorm: bool, block_m: int = 16,
              dtype=np.float32) -> dict:
    """Route, align and the expert loop on one set of inputs (the dict made
    by the synthetic input generator). Returns every intermediate."""
    ids, w, logits = route(inputs["hidden"], inputs["router_w"], top_k, renorm,
                           inputs.get("router_bias"))
    E = inputs["router_w"].shape[0]
    sorted_ids, offsets, counts = align(ids, E, block_m)
    out = experts_loop(inputs["hidden"], inputs["w_gate_up"], inputs["w_down"],
                       ids, w, dtype=dtype)
    return {"topk_ids": ids, "topk_w": w, "logits": logits,
            "sorted_token_ids": sorted_ids, "expert_offsets": offsets,
            "expert_counts": counts, "out": out}


def moe_layer_after_norm(inputs: dict, x_bits, residual_bits, norm_w_bits, eps: float,
                         top_k: int, renorm: bool, block_m: int = 16) -> dict:
    """The MoE layer fed by the add + RMSNorm step before it: returns the
    normalised rows, the new residual and every output of moe_layer on them."""
    xn, r = fused_add_rmsnorm(x_bits, residual_bits, norm_w_bits, eps)
    res = moe_layer({**inputs, "hidden": xn}, top_k, renorm, block_m)
    return {**res, "normed": xn, "residual": r}
