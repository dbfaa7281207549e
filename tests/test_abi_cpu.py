"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every entry point include/mm.h declares, and its host-side argument checks
return their codes before any CUDA call is made."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_mm_gb300 as mm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib(mmlib):
    return mm.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "mm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mm_[a-z_0-9]+)\s*\(", src)))


def test_header_and_binding_agree(lib):
    decl = _declared()
    assert decl == sorted(mm.SIGNATURES), (decl, sorted(mm.SIGNATURES))


def test_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(mm.LIB_PATH)
    for name in _declared():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    for code in range(7):
        assert mm.status_string(code).startswith("MM_")
    assert mm.status_string(99) == "unknown mm status"


def test_align_capacity(lib):
    assert mm.mm_align_capacity(64, 8, 128, 16) == 64 * 8 + 128 * 15
    assert mm.mm_align_capacity(0, 2, 8, 1) == 0
    assert mm.mm_align_capacity(-1, 2, 8, 16) == -1
    assert mm.mm_align_capacity(4, 0, 8, 16) == -1


def test_workspace_size(lib):
    n = mm.mm_moe_workspace_size(4096, 2048, 128, 768, 8)
    cap = 4096 * 8 + 128 * 15
    act, acc = cap * 768 * 2, 4096 * 2048 * 4
    xs = cap * 2048 * 2                           # token rows in segment order (T*k > 64*E)
    ids_w, sorted_ = 2 * 4096 * 8 * 4, cap * 4
    tile_counts = (4096 // 32 + 1) * 128 * 4      # the tensor-core router's per-tile counts
    assert n >= act + acc + xs + ids_w + sorted_ + tile_counts
    # decode-sized: rows are gathered inside the GEMM, so no copy of the rows
    cap_d = 64 * 8 + 128 * 15
    n_d = mm.mm_moe_workspace_size(64, 2048, 128, 768, 8)
    assert cap_d * 768 * 2 + 64 * 2048 * 4 <= n_d < cap_d * 2048 * 2
    assert mm.mm_moe_workspace_size(4, 100, 8, 64, 2) == -1   # H % 64
    assert mm.mm_moe_workspace_size(4, 128, 8, 96, 2) == -1   # I % 64
    assert mm.mm_moe_workspace_size(4, 128, 300, 64, 2) == -1  # E > 256


def test_workspace_layout(lib):
    for (T, H, E, I, k) in [(4096, 2048, 128, 768, 8), (64, 2048, 128, 768, 8), (16, 128, 8, 64, 2),
                            (2600, 64, 160, 64, 4), (0, 64, 8, 64, 2)]:
        lay = mm.mm_moe_workspace_layout(T, H, E, I, k)
        assert lay["total"] == mm.mm_moe_workspace_size(T, H, E, I, k)
        assert lay["block_m"] == mm.FORWARD_BLOCK_M
        assert lay["capacity"] == mm.mm_align_capacity(T, k, E, lay["block_m"])
        regions = sorted([(lay["topk_ids"], T * k * 4), (lay["topk_w"], T * k * 4),
                          (lay["sorted_token_ids"], lay["capacity"] * 4),
                          (lay["expert_offsets"], (E + 1) * 4), (lay["expert_counts"], E * 4)])
        for (o, n), (o2, _) in zip(regions, regions[1:] + [(lay["total"], 0)]):
            assert o % 256 == 0 and o + n <= o2, (T, H, E, I, k, regions)
    with pytest.raises(mm.MMError) as ei:
        mm.mm_moe_workspace_layout(4, 128, 8, 96, 2)
    assert ei.value.code == mm.MM_ERR_UNSUPPORTED
    with pytest.raises(mm.MMError) as ei:
        mm.mm_moe_workspace_layout(-1, 128, 8, 64, 2)
    assert ei.value.code == mm.MM_ERR_INVALID_ARG
    assert lib.mm_moe_workspace_layout(4, 128, 8, 64, 2, None) == mm.MM_ERR_INVALID_ARG


def test_host_checks_before_any_cuda_call(lib):
    L = mm.lib()
    # null pointers
    assert L.mm_route(None, None, None, 4, 64, 8, 2, 1, None, None, None) == mm.MM_ERR_INVALID_ARG
    # k > E, H % 64, E > 256, k > 32
    assert L.mm_route(None, None, None, 4, 64, 8, 9, 1, None, None, None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_route(None, None, None, 4, 48, 8, 2, 1, None, None, None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_route(None, None, None, 4, 64, 300, 2, 1, None, None, None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_route(None, None, None, 4, 64, 64, 33, 1, None, None, None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_route(None, None, None, -1, 64, 8, 2, 1, None, None, None) == mm.MM_ERR_INVALID_ARG
    # misaligned pointer
    assert L.mm_route(8, 16, None, 4, 64, 8, 2, 1, 32, 48, None) == mm.MM_ERR_INVALID_ARG
    # align: bad block_m, null outputs
    assert L.mm_align(None, 4, 2, 8, 0, None, None, None, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_align(None, 4, 2, 8, 300, 16, 16, None, None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_align(None, 4, 2, 8, 16, None, None, None, None) == mm.MM_ERR_INVALID_ARG
    # gemm: bad mode, N % 64, missing topk_w in down mode
    assert L.mm_grouped_gemm(7, 16, 16, 16, 16, 16, None, 4, 2, 8, 64, 64, 16, None) == \
        mm.MM_ERR_INVALID_ARG
    assert L.mm_grouped_gemm(0, 16, 16, 16, 16, 16, None, 4, 2, 8, 96, 64, 16, None) == \
        mm.MM_ERR_UNSUPPORTED
    assert L.mm_grouped_gemm(1, 16, 16, 16, 16, 16, None, 4, 2, 8, 64, 64, 16, None) == \
        mm.MM_ERR_INVALID_ARG
    # forward: I % 64, null out, workspace too small or misaligned
    assert L.mm_moe_forward(16, 16, 16, 16, 4, 64, 8, 96, 2, 1, 16, None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_moe_forward(16, 16, 16, 16, 4, 64, 8, 64, 2, 1, None, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_moe_forward_ex(16, 16, None, 16, 16, 4, 64, 8, 64, 2, 1, 16, 256, 1, None) == \
        mm.MM_ERR_NO_MEMORY
    assert L.mm_moe_forward_ex(16, 16, None, 16, 16, 4, 64, 8, 64, 2, 1, 16, 16, 1 << 30, None) == \
        mm.MM_ERR_INVALID_ARG


def test_gated_mlp_host_checks(lib):
    L = mm.lib()
    assert L.mm_gated_mlp(None, None, None, 4, 64, 64, None, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_gated_mlp(16, 16, 16, 4, 96, 64, 16, None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_gated_mlp(16, 16, 16, -1, 64, 64, 16, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_gated_mlp(None, None, None, 0, 64, 64, None, None) == mm.MM_OK
    assert mm.mm_gated_mlp_workspace_size(8, 128, 64) > 0


def test_add_norm_host_checks(lib):
    import ctypes
    L = mm.lib()
    f = ctypes.c_float
    # add + RMSNorm alone: nulls, H % 64, negative or NaN eps, misaligned, T == 0
    assert L.mm_add_rmsnorm(None, None, None, f(1e-6), 4, 64, None, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_add_rmsnorm(16, None, 16, f(1e-6), 4, 96, 16, None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_add_rmsnorm(16, None, 16, f(-1.0), 4, 64, 16, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_add_rmsnorm(16, None, 16, f(float("nan")), 4, 64, 16, None) == \
        mm.MM_ERR_INVALID_ARG
    assert L.mm_add_rmsnorm(16, 8, 16, f(1e-6), 4, 64, 16, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_add_rmsnorm(None, None, None, f(1e-6), 0, 64, None, None) == mm.MM_OK
    # the layer behind it: null norm weight, bad shape, T == 0
    assert L.mm_moe_forward_add_norm(16, None, None, f(1e-6), 16, 16, 16, 4, 64, 8, 64, 2, 1, 16,
                                     None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_moe_forward_add_norm(16, None, 16, f(1e-6), 16, 16, 16, 4, 64, 8, 96, 2, 1, 16,
                                     None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_moe_forward_add_norm(None, None, None, f(1e-6), None, None, None, 0, 64, 8, 64, 2,
                                     1, None, None) == mm.MM_OK


def test_moe_block_residual_host_checks(lib):
    import ctypes
    L = mm.lib()
    f = ctypes.c_float
    # residual_out is required; misaligned residual_out; T == 0 is a no-op
    assert L.mm_moe_forward_add_norm_residual(16, None, 16, f(1e-6), 16, 16, 16, 4, 64, 8, 64, 2,
                                              1, 16, None, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_moe_forward_add_norm_residual(16, None, 16, f(1e-6), 16, 16, 16, 4, 64, 8, 64, 2,
                                              1, 16, 8, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_moe_forward_add_norm_residual(None, None, None, f(1e-6), None, None, None, 0, 64,
                                              8, 64, 2, 1, None, None, None) == mm.MM_OK


def test_tp_host_checks(lib):
    L = mm.lib()
    # the partial output is required; I_slice % 64; T == 0 is a no-op
    assert L.mm_moe_forward_partial(16, 16, None, 16, 16, 4, 64, 8, 64, 2, 1, None, None, 0,
                                    None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_moe_forward_partial(16, 16, None, 16, 16, 4, 64, 8, 96, 2, 1, 16, None, 0,
                                    None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_moe_forward_partial(None, None, None, None, None, 0, 64, 8, 64, 2, 1, None, None,
                                    0, None) == mm.MM_OK
    assert L.mm_round_bf16(16, 16, 6, None) == mm.MM_ERR_UNSUPPORTED
    assert L.mm_round_bf16(16, 16, -4, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_round_bf16(8, 16, 4, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_round_bf16(None, None, 0, None) == mm.MM_OK


def test_binding_raises_without_library(monkeypatch, tmp_path):
    import mixture_experts_layer_mm_gb300._lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        L.lib()
