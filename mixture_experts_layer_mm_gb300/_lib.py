"""Thin ctypes binding of the C ABI in include/mm.h.

Argument marshalling only: torch tensors supply device pointers and the
current CUDA stream; every step of the MoE layer runs in libmm.so's kernels.
There is no fallback: if the library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmm.so")

MM_OK = 0
MM_ERR_INVALID_ARG = 1
MM_ERR_UNSUPPORTED = 2
MM_ERR_CUDA = 3
MM_ERR_NO_MEMORY = 4
MM_ERR_DEVICE = 5
MM_ERR_TIMEOUT = 6
MM_GEMM_GATE_UP = 0
MM_GEMM_DOWN = 1
FORWARD_BLOCK_M = 16  # expert segments are padded to this multiple by mm_moe_forward

# Every entry point include/mm.h declares, with its ctypes signature.
_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "mm_status_string": (ctypes.c_char_p, [_I]),
    "mm_route": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "mm_align_capacity": (_I64, [_I, _I, _I, _I]),
    "mm_align": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "mm_align_noalloc": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "mm_grouped_gemm": (_I, [_I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "mm_moe_forward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "mm_moe_workspace_size": (_I64, [_I, _I, _I, _I, _I]),
    "mm_moe_workspace_layout": (_I, [_I, _I, _I, _I, _I, _P]),
    "mm_moe_forward_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "mm_moe_forward_profiled": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P,
                                     _P]),
    "mm_moe_forward_partial": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "mm_moe_forward_single_launch": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ,
                                          _P]),
    "mm_round_bf16": (_I, [_P, _P, _I64, _P]),
    "mm_gated_mlp": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "mm_gated_mlp_workspace_size": (_I64, [_I, _I, _I]),
    "mm_add_rmsnorm": (_I, [_P, _P, _P, ctypes.c_float, _I, _I, _P, _P]),
    "mm_moe_forward_add_norm": (_I, [_P, _P, _P, ctypes.c_float, _P, _P, _P, _I, _I, _I, _I, _I,
                                     _I, _P, _P]),
    "mm_moe_forward_add_norm_residual": (_I, [_P, _P, _P, ctypes.c_float, _P, _P, _P, _I, _I, _I,
                                              _I, _I, _I, _P, _P, _P]),
    "mm_poll_device_status": (_I, [_P]),
    "mm_selftest_wait_timeout": (_I, [_P]),
    "mm_selftest_layer_barrier_timeout": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                                               _P]),
    "mm_shutdown": (None, []),
}

_lib: Optional[ctypes.CDLL] = None


class MMError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (code {code})")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libmm.so (built by __graft_entry__.build()); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run __graft_entry__.build())")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def status_string(code: int) -> str:
    return lib().mm_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != MM_OK:
        raise MMError(code, where)


def _ptr(t: Optional[torch.Tensor], dtype: torch.dtype, name: str) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def mm_align_capacity(T: int, top_k: int, E: int, block_m: int) -> int:
    return int(lib().mm_align_capacity(T, top_k, E, block_m))


def mm_moe_workspace_size(T: int, H: int, E: int, I: int, top_k: int) -> int:
    return int(lib().mm_moe_workspace_size(T, H, E, I, top_k))


# Fields of mm_moe_workspace_layout, in the order of its MM_WS_* indices.
WS_LAYOUT_FIELDS = ("topk_ids", "topk_w", "sorted_token_ids", "expert_offsets", "expert_counts",
                    "capacity", "block_m", "total")


def mm_moe_workspace_layout(T: int, H: int, E: int, I: int, top_k: int) -> dict:
    """Byte offsets of the routing and grouping inside a caller workspace of
    mm_moe_forward_ex, plus capacity, block_m and the total size."""
    buf = (ctypes.c_int64 * len(WS_LAYOUT_FIELDS))()
    _check(lib().mm_moe_workspace_layout(T, H, E, I, top_k, ctypes.cast(buf, ctypes.c_void_p)),
           "mm_moe_workspace_layout")
    return dict(zip(WS_LAYOUT_FIELDS, (int(v) for v in buf)))


def forward_routing(workspace, T: int, H: int, E: int, I: int, top_k: int) -> dict:
    """Views into a caller workspace that mm_moe_forward_ex just used: its
    own topk_ids, topk_w, sorted_token_ids, expert_offsets and expert_counts
    (valid once the call's kernels have completed)."""
    lay = mm_moe_workspace_layout(T, H, E, I, top_k)
    if workspace.dtype != torch.uint8 or workspace.numel() < lay["total"]:
        raise ValueError("workspace is not a caller workspace of these sizes")

    def view(name, n, dtype):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return workspace[lay[name]:lay[name] + nbytes].view(dtype)

    return {"topk_ids": view("topk_ids", T * top_k, torch.int32).view(T, top_k),
            "topk_w": view("topk_w", T * top_k, torch.float32).view(T, top_k),
            "sorted_token_ids": view("sorted_token_ids", lay["capacity"], torch.int32),
            "expert_offsets": view("expert_offsets", E + 1, torch.int32),
            "expert_counts": view("expert_counts", E, torch.int32),
            "block_m": lay["block_m"]}


def mm_route(hidden, router_w, top_k: int, renorm: bool, router_bias=None,
             topk_ids=None, topk_w=None, stream=None):
    """Router + softmax + top-k. Returns (topk_ids int32 [T,k], topk_w fp32 [T,k])."""
    T, H = hidden.shape
    E = router_w.shape[0]
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=hidden.device)
    if topk_w is None:
        topk_w = torch.empty((T, top_k), dtype=torch.float32, device=hidden.device)
    _check(lib().mm_route(_ptr(hidden, torch.bfloat16, "hidden"),
                          _ptr(router_w, torch.bfloat16, "router_w"),
                          _ptr(router_bias, torch.float32, "router_bias"),
                          T, H, E, top_k, int(bool(renorm)),
                          _ptr(topk_ids, torch.int32, "topk_ids"),
                          _ptr(topk_w, torch.float32, "topk_w"), _stream(stream)), "mm_route")
    return topk_ids, topk_w


def mm_align(topk_ids, E: int, block_m: int, sorted_token_ids=None, expert_offsets=None,
             expert_counts=None, stream=None):
    """Block-padded grouping by expert. Returns (sorted_token_ids, expert_offsets, expert_counts)."""
    T, k = topk_ids.shape
    dev = topk_ids.device
    cap = mm_align_capacity(T, k, E, block_m)
    if cap < 0:
        raise MMError(MM_ERR_INVALID_ARG, "mm_align_capacity")
    if sorted_token_ids is None:
        sorted_token_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    if expert_offsets is None:
        expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if expert_counts is None:
        expert_counts = torch.empty(E, dtype=torch.int32, device=dev)
    _check(lib().mm_align(_ptr(topk_ids, torch.int32, "topk_ids"), T, k, E, block_m,
                          _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
                          _ptr(expert_offsets, torch.int32, "expert_offsets"),
                          _ptr(expert_counts, torch.int32, "expert_counts"),
                          _stream(stream)), "mm_align")
    return sorted_token_ids, expert_offsets, expert_counts


def mm_align_noalloc(topk_ids, E: int, block_m: int, sorted_token_ids, expert_offsets,
                     expert_counts=None, stream=None):
    """mm_align with caller-owned outputs and no device allocation (see include/mm.h)."""
    T, k = topk_ids.shape
    _check(lib().mm_align_noalloc(_ptr(topk_ids, torch.int32, "topk_ids"), T, k, E, block_m,
                                  _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
                                  _ptr(expert_offsets, torch.int32, "expert_offsets"),
                                  _ptr(expert_counts, torch.int32, "expert_counts"),
                                  _stream(stream)), "mm_align_noalloc")
    return sorted_token_ids, expert_offsets, expert_counts


def mm_grouped_gemm(mode: int, A, B, C, sorted_token_ids, expert_offsets, topk_w,
                    T: int, top_k: int, block_m: int, stream=None):
    """One grouped GEMM (MM_GEMM_GATE_UP or MM_GEMM_DOWN); C is written in place."""
    E = B.shape[0]
    if mode == MM_GEMM_GATE_UP:
        N, K = B.shape[1] // 2, B.shape[2]
        cdt = torch.bfloat16
    else:
        N, K = B.shape[1], B.shape[2]
        cdt = torch.float32
    _check(lib().mm_grouped_gemm(mode, _ptr(A, torch.bfloat16, "A"), _ptr(B, torch.bfloat16, "B"),
                                 _ptr(C, cdt, "C"),
                                 _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
                                 _ptr(expert_offsets, torch.int32, "expert_offsets"),
                                 _ptr(topk_w, torch.float32, "topk_w"),
                                 T, top_k, E, N, K, block_m, _stream(stream)), "mm_grouped_gemm")
    return C


def mm_moe_forward(hidden, router_w, w_gate_up, w_down, top_k: int, renorm: bool,
                   out=None, router_bias=None, workspace=None, stream=None):
    """The whole MoE layer; returns out [T, H] bf16."""
    T, H = hidden.shape
    E = router_w.shape[0]
    I = w_down.shape[2]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=hidden.device)
    if router_bias is None and workspace is None:
        _check(lib().mm_moe_forward(_ptr(hidden, torch.bfloat16, "hidden"),
                                    _ptr(router_w, torch.bfloat16, "router_w"),
                                    _ptr(w_gate_up, torch.bfloat16, "w_gate_up"),
                                    _ptr(w_down, torch.bfloat16, "w_down"),
                                    T, H, E, I, top_k, int(bool(renorm)),
                                    _ptr(out, torch.bfloat16, "out"), _stream(stream)),
               "mm_moe_forward")
        return out
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, torch.uint8, "workspace"), workspace.numel()
    _check(lib().mm_moe_forward_ex(_ptr(hidden, torch.bfloat16, "hidden"),
                                   _ptr(router_w, torch.bfloat16, "router_w"),
                                   _ptr(router_bias, torch.float32, "router_bias"),
                                   _ptr(w_gate_up, torch.bfloat16, "w_gate_up"),
                                   _ptr(w_down, torch.bfloat16, "w_down"),
                                   T, H, E, I, top_k, int(bool(renorm)),
                                   _ptr(out, torch.bfloat16, "out"), ws_ptr, ws_bytes,
                                   _stream(stream)), "mm_moe_forward_ex")
    return out


def mm_moe_forward_single_launch(hidden, router_w, w_gate_up, w_down, top_k: int, renorm: bool,
                                 out=None, router_bias=None, workspace=None, stream=None):
    """The whole MoE layer in one cooperative launch (small batches; see
    include/mm.h for the shapes it takes); returns out [T, H] bf16."""
    T, H = hidden.shape
    E = router_w.shape[0]
    I = w_down.shape[2]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=hidden.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, torch.uint8, "workspace"), workspace.numel()
    _check(lib().mm_moe_forward_single_launch(
        _ptr(hidden, torch.bfloat16, "hidden"), _ptr(router_w, torch.bfloat16, "router_w"),
        _ptr(router_bias, torch.float32, "router_bias"),
        _ptr(w_gate_up, torch.bfloat16, "w_gate_up"), _ptr(w_down, torch.bfloat16, "w_down"),
        T, H, E, I, top_k, int(bool(renorm)), _ptr(out, torch.bfloat16, "out"), ws_ptr, ws_bytes,
        _stream(stream)), "mm_moe_forward_single_launch")
    return out


def tp_slice(w_gate_up, w_down, rank: int, world: int):
    """The expert weights rank `rank` of `world` holds under tensor
    parallelism: gate rows [i0, i0 + I/world) and the same up rows of every
    expert, as one [E, 2*I/world, H] tensor (gate slice first), and the same
    columns of w_down, [E, H, I/world]. Weight preparation (done once, like
    the loader's sharding), for torch tensors or numpy arrays."""
    E, twoI, H = w_gate_up.shape
    I = twoI // 2
    if world < 1 or I % world != 0:
        raise ValueError(f"I={I} does not split into {world} equal slices")
    il = I // world
    i0 = rank * il
    gate, up = w_gate_up[:, i0:i0 + il, :], w_gate_up[:, I + i0:I + i0 + il, :]
    if isinstance(w_gate_up, torch.Tensor):
        return torch.cat([gate, up], dim=1).contiguous(), w_down[:, :, i0:i0 + il].contiguous()
    import numpy as np
    return (np.ascontiguousarray(np.concatenate([gate, up], axis=1)),
            np.ascontiguousarray(w_down[:, :, i0:i0 + il]))


def mm_moe_forward_partial(hidden, router_w, w_gate_up_slice, w_down_slice, top_k: int,
                           renorm: bool, partial=None, router_bias=None, workspace=None,
                           stream=None):
    """The layer on one tensor-parallel slice of the experts' intermediates
    (see tp_slice): returns this rank's unrounded fp32 contribution [T, H]."""
    T, H = hidden.shape
    E = router_w.shape[0]
    I = w_down_slice.shape[2]
    if partial is None:
        partial = torch.empty((T, H), dtype=torch.float32, device=hidden.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, torch.uint8, "workspace"), workspace.numel()
    _check(lib().mm_moe_forward_partial(_ptr(hidden, torch.bfloat16, "hidden"),
                                        _ptr(router_w, torch.bfloat16, "router_w"),
                                        _ptr(router_bias, torch.float32, "router_bias"),
                                        _ptr(w_gate_up_slice, torch.bfloat16, "w_gate_up_slice"),
                                        _ptr(w_down_slice, torch.bfloat16, "w_down_slice"),
                                        T, H, E, I, top_k, int(bool(renorm)),
                                        _ptr(partial, torch.float32, "partial"), ws_ptr, ws_bytes,
                                        _stream(stream)), "mm_moe_forward_partial")
    return partial


def mm_round_bf16(x, out=None, stream=None):
    """bf16 rounding (to nearest even) of an fp32 tensor, on the GPU."""
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _check(lib().mm_round_bf16(_ptr(x, torch.float32, "x"), _ptr(out, torch.bfloat16, "out"),
                               x.numel(), _stream(stream)), "mm_round_bf16")
    return out


def mm_gated_mlp_workspace_size(T: int, H: int, I: int) -> int:
    return int(lib().mm_gated_mlp_workspace_size(T, H, I))


def mm_gated_mlp(hidden, w_gate_up, w_down, out=None, stream=None):
    """Dense SwiGLU MLP through the grouped-GEMM kernels; returns out [T, H] bf16."""
    T, H = hidden.shape
    I = w_down.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=hidden.device)
    _check(lib().mm_gated_mlp(_ptr(hidden, torch.bfloat16, "hidden"),
                              _ptr(w_gate_up, torch.bfloat16, "w_gate_up"),
                              _ptr(w_down, torch.bfloat16, "w_down"), T, H, I,
                              _ptr(out, torch.bfloat16, "out"), _stream(stream)), "mm_gated_mlp")
    return out


def mm_add_rmsnorm(x, norm_w, eps: float, residual=None, normed=None, stream=None):
    """residual <- bf16(x + residual) in place (residual None: x is the
    residual); returns normed = rmsnorm(residual, norm_w, eps) [T, H] bf16."""
    T, H = x.shape
    if normed is None:
        normed = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(lib().mm_add_rmsnorm(_ptr(x, torch.bfloat16, "x"),
                                _ptr(residual, torch.bfloat16, "residual"),
                                _ptr(norm_w, torch.bfloat16, "norm_w"), float(eps), T, H,
                                _ptr(normed, torch.bfloat16, "normed"), _stream(stream)),
           "mm_add_rmsnorm")
    return normed


def mm_moe_forward_add_norm(x, norm_w, eps: float, router_w, w_gate_up, w_down, top_k: int,
                            renorm: bool, residual=None, out=None, stream=None):
    """The MoE layer on rmsnorm(x + residual) (residual updated in place, or
    x itself when residual is None); returns out [T, H] bf16."""
    T, H = x.shape
    E = router_w.shape[0]
    I = w_down.shape[2]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(lib().mm_moe_forward_add_norm(_ptr(x, torch.bfloat16, "x"),
                                         _ptr(residual, torch.bfloat16, "residual"),
                                         _ptr(norm_w, torch.bfloat16, "norm_w"), float(eps),
                                         _ptr(router_w, torch.bfloat16, "router_w"),
                                         _ptr(w_gate_up, torch.bfloat16, "w_gate_up"),
                                         _ptr(w_down, torch.bfloat16, "w_down"), T, H, E, I,
                                         top_k, int(bool(renorm)),
                                         _ptr(out, torch.bfloat16, "out"), _stream(stream)),
           "mm_moe_forward_add_norm")
    return out


def mm_moe_forward_add_norm_residual(x, norm_w, eps: float, router_w, w_gate_up, w_down,
                                     top_k: int, renorm: bool, residual=None, residual_out=None,
                                     out=None, stream=None):
    """The MoE half of a decoder layer: residual' = bf16(x + residual) (in
    place; x when residual is None), out = layer(rmsnorm(residual')), and
    residual_out = bf16(out + residual') (default: residual itself, updated
    in place; a new tensor when residual is None). Returns (out, residual_out)."""
    T, H = x.shape
    E = router_w.shape[0]
    I = w_down.shape[2]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    if residual_out is None:
        residual_out = residual if residual is not None else torch.empty_like(x)
    _check(lib().mm_moe_forward_add_norm_residual(
        _ptr(x, torch.bfloat16, "x"), _ptr(residual, torch.bfloat16, "residual"),
        _ptr(norm_w, torch.bfloat16, "norm_w"), float(eps),
        _ptr(router_w, torch.bfloat16, "router_w"), _ptr(w_gate_up, torch.bfloat16, "w_gate_up"),
        _ptr(w_down, torch.bfloat16, "w_down"), T, H, E, I, top_k, int(bool(renorm)),
        _ptr(out, torch.bfloat16, "out"), _ptr(residual_out, torch.bfloat16, "residual_out"),
        _stream(stream)), "mm_moe_forward_add_norm_residual")
    return out, residual_out


PROFILE_STAGES = ("route", "align", "gate_up", "down", "finalize")


def mm_moe_forward_profiled(hidden, router_w, w_gate_up, w_down, top_k: int, renorm: bool,
                            events, out=None, router_bias=None, workspace=None, stream=None):
    """mm_moe_forward that records len(PROFILE_STAGES)+1 torch.cuda.Event
    (timing enabled) around its stages on the stream; returns out."""
    T, H = hidden.shape
    E = router_w.shape[0]
    I = w_down.shape[2]
    if len(events) != len(PROFILE_STAGES) + 1:
        raise ValueError(f"need {len(PROFILE_STAGES) + 1} events")
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=hidden.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace, torch.uint8, "workspace"), workspace.numel()
    for e in events:  # torch creates the CUDA event on its first record
        if e.cuda_event == 0:
            e.record()
    ev = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().mm_moe_forward_profiled(_ptr(hidden, torch.bfloat16, "hidden"),
                                         _ptr(router_w, torch.bfloat16, "router_w"),
                                         _ptr(router_bias, torch.float32, "router_bias"),
                                         _ptr(w_gate_up, torch.bfloat16, "w_gate_up"),
                                         _ptr(w_down, torch.bfloat16, "w_down"),
                                         T, H, E, I, top_k, int(bool(renorm)),
                                         _ptr(out, torch.bfloat16, "out"), ws_ptr, ws_bytes,
                                         _stream(stream), ev), "mm_moe_forward_profiled")
    return out


def mm_poll_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(lib().mm_poll_device_status(_stream(stream)))


def mm_selftest_wait_timeout(stream=None) -> None:
    """Launches the kernel whose bounded wait must time out (see include/mm.h)."""
    _check(lib().mm_selftest_wait_timeout(_stream(stream)), "mm_selftest_wait_timeout")


def mm_selftest_layer_barrier_timeout(hidden, router_w, w_gate_up, w_down, top_k: int,
                                      renorm: bool, barrier: int, out=None, stream=None):
    """Runs the single-launch small-batch layer with CTA 0 absent from grid
    barrier `barrier` (see include/mm.h); every CTA's wait there runs out.
    Returns out (undefined contents)."""
    T, H = hidden.shape
    E = router_w.shape[0]
    I = w_down.shape[2]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=hidden.device)
    _check(lib().mm_selftest_layer_barrier_timeout(
        _ptr(hidden, torch.bfloat16, "hidden"), _ptr(router_w, torch.bfloat16, "router_w"),
        _ptr(w_gate_up, torch.bfloat16, "w_gate_up"), _ptr(w_down, torch.bfloat16, "w_down"),
        T, H, E, I, top_k, int(bool(renorm)), barrier, _ptr(out, torch.bfloat16, "out"),
        _stream(stream)), "mm_selftest_layer_barrier_timeout")
    return out


def mm_shutdown() -> None:
    lib().mm_shutdown()
