"""Plant one plausible mistake at a time in the CPU oracle and require that
the pin checks catch it. This shows that the pins constrain every step (a
dropped term, a wrong sign, a swapped operand, a broken tie-break, an unstable
grouping) rather than re-deriving the oracle from itself."""
import numpy as np
import pytest

import pin_checks
from oracle import moe_oracle as O

_orig = {n: getattr(O, n) for n in ("silu_and_mul", "select_topk", "routing_weights",
                                    "softmax_over_experts", "router_logits", "align",
                                    "experts_loop", "widen_bf16", "round_bf16",
                                    "mean_of_squares", "rmsnorm", "fused_add_rmsnorm")}


def _swap_gate_up(g, u):
    return _orig["silu_and_mul"](u, g)


def _silu_sign(g, u):
    with np.errstate(over="ignore"):
        return g / (1 + np.exp(g)) * u


def _tie_high_id(logits, k):
    order = np.argsort(-logits[:, ::-1], axis=1, kind="stable")[:, :k]
    return np.sort(logits.shape[1] - 1 - order, axis=1).astype(np.int32)


def _slots_by_logit(logits, k):
    return np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)


def _smallest_k(logits, k):
    return _orig["select_topk"](-logits, k)


def _always_renorm(p, ids, renorm):
    return _orig["routing_weights"](p, ids, True)


def _never_renorm(p, ids, renorm):
    return _orig["routing_weights"](p, ids, False)


def _softmax_no_max(l):
    z = np.exp(l.astype(np.float32))
    return (z / z.sum(1, keepdims=True)).astype(np.float32)


def _softmax_missing_term(l):
    m = l.max(1, keepdims=True)
    z = np.exp(l - m)
    return (z / (z.sum(1, keepdims=True) - z[:, :1] + 1e-3)).astype(np.float32)


def _logits_drop_bias(x, w, bias=None):
    return _orig["router_logits"](x, w, None)


def _logits_sign(x, w, bias=None):
    return -_orig["router_logits"](x, w, bias)


def _align_unstable(ids, E, block_m):
    s, off, cnt = _orig["align"](ids, E, block_m)
    s = s.copy()
    for e in range(E):
        seg = s[off[e]:off[e] + cnt[e]]
        s[off[e]:off[e] + cnt[e]] = seg[::-1]
    return s, off, cnt


def _align_floor_pad(ids, E, block_m):
    s, off, cnt = _orig["align"](ids, E, block_m)
    pad = cnt // block_m * block_m
    off2 = np.zeros_like(off); off2[1:] = np.cumsum(pad)
    return s, off2, cnt


def _align_sentinel_zero(ids, E, block_m):
    s, off, cnt = _orig["align"](ids, E, block_m)
    s = s.copy(); s[s == ids.size] = 0
    return s, off, cnt


def _loop_no_weights(h, wgu, wd, ids, w, dtype=np.float32):
    return _orig["experts_loop"](h, wgu, wd, ids, np.ones_like(w), dtype=dtype)


def _loop_overwrite(h, wgu, wd, ids, w, dtype=np.float32):
    T, H = h.shape
    E, twoI, _ = wgu.shape
    I = twoI // 2
    x = O.widen_bf16(h).astype(dtype)
    out = np.zeros((T, H), dtype=dtype)
    for e in range(E):
        tok, slot = np.nonzero(ids == e)
        if tok.size == 0:
            continue
        wg = O.widen_bf16(wgu[e]).astype(dtype); wdn = O.widen_bf16(wd[e]).astype(dtype)
        a = O.silu_and_mul(x[tok] @ wg[:I].T, x[tok] @ wg[I:].T)
        out[tok] = w[tok, slot][:, None] * (a @ wdn.T)   # '=' instead of '+='
    return out


def _loop_down_transposed_rows(h, wgu, wd, ids, w, dtype=np.float32):
    # reads w_down[e] with its rows reversed (a wrong index on the H axis)
    return _orig["experts_loop"](h, wgu, wd[:, ::-1, :], ids, w, dtype=dtype)


def _widen_truncate(bits):
    v = _orig["widen_bf16"](bits).copy()
    v[np.abs(v) > 1.5] = np.float32(1.5)
    return v


def _round_truncate(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _round_ties_up(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + np.uint64(0x8000)) >> np.uint64(16)).astype(np.uint16)


def _meansq_drop_last(xf):
    return _orig["mean_of_squares"](np.asarray(xf)[..., :-1])


def _rms_no_eps(x, w, eps):
    return _orig["rmsnorm"](x, w, 0.0)


def _rms_sum_not_mean(x, w, eps):
    xf = O.widen_bf16(x)
    total = O.mean_of_squares(xf) * np.float32(xf.shape[-1])
    inv = np.float32(1.0) / np.sqrt(total + np.float32(eps), dtype=np.float32)
    y = O.round_bf16(xf * inv[..., None])
    return O.round_bf16(O.widen_bf16(w)[None, :] * O.widen_bf16(y))


def _rms_single_round(x, w, eps):
    xf = O.widen_bf16(x)
    mean = O.mean_of_squares(xf)
    inv = np.float32(1.0) / np.sqrt(mean + np.float32(eps), dtype=np.float32)
    return O.round_bf16(O.widen_bf16(w)[None, :] * (xf * inv[..., None]))


def _add_ignores_residual(x, r, w, eps):
    return _orig["fused_add_rmsnorm"](x, None, w, eps)


def _add_keeps_old_residual(x, r, w, eps):
    normed, _ = _orig["fused_add_rmsnorm"](x, r, w, eps)
    return normed, (x if r is None else r)


MUTANTS = {
    "round_truncate": ("round_bf16", _round_truncate),
    "round_ties_up": ("round_bf16", _round_ties_up),
    "meansq_drop_last": ("mean_of_squares", _meansq_drop_last),
    "rms_no_eps": ("rmsnorm", _rms_no_eps),
    "rms_sum_not_mean": ("rmsnorm", _rms_sum_not_mean),
    "rms_single_round": ("rmsnorm", _rms_single_round),
    "add_ignores_residual": ("fused_add_rmsnorm", _add_ignores_residual),
    "add_keeps_old_residual": ("fused_add_rmsnorm", _add_keeps_old_residual),
    "swap_gate_up": ("silu_and_mul", _swap_gate_up),
    "silu_sign": ("silu_and_mul", _silu_sign),
    "tie_high_id": ("select_topk", _tie_high_id),
    "slots_by_logit": ("select_topk", _slots_by_logit),
    "smallest_k": ("select_topk", _smallest_k),
    "always_renorm": ("routing_weights", _always_renorm),
    "never_renorm": ("routing_weights", _never_renorm),
    "softmax_no_max": ("softmax_over_experts", _softmax_no_max),
    "softmax_missing_term": ("softmax_over_experts", _softmax_missing_term),
    "logits_drop_bias": ("router_logits", _logits_drop_bias),
    "logits_sign": ("router_logits", _logits_sign),
    "align_unstable": ("align", _align_unstable),
    "align_floor_pad": ("align", _align_floor_pad),
    "align_sentinel_zero": ("align", _align_sentinel_zero),
    "loop_no_weights": ("experts_loop", _loop_no_weights),
    "loop_overwrite": ("experts_loop", _loop_overwrite),
    "loop_down_rows": ("experts_loop", _loop_down_transposed_rows),
    "widen_truncate": ("widen_bf16", _widen_truncate),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = []
    for check in pin_checks.ALL_CHECKS:
        try:
            check()
        except Exception as exc:  # noqa: BLE001 - any failure counts as caught
            caught.append(f"{check.__name__}: {type(exc).__name__}")
    assert caught, f"planted mistake '{name}' passed every pin"
