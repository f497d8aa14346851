"""Thin ctypes binding of liblrm.so (include/lrm.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensor arguments may be torch tensors (their data_ptr() is passed)
or plain integer device addresses.  Every function raises LrmError on a
non-OK status.  There is no CPU fallback: if the library is missing or the
device is not a GB300, the calls fail loudly.
"""

from __future__ import annotations

import ctypes
import os
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "liblrm.so")

LRM_OK = 0
STATUS_NAMES = [
    "LRM_OK",
    "LRM_ERR_INVALID_ARG",
    "LRM_ERR_SHAPE",
    "LRM_ERR_ALIGN",
    "LRM_ERR_WORKSPACE",
    "LRM_ERR_INDEX",
    "LRM_ERR_QUOTA",
    "LRM_ERR_TIMEOUT",
    "LRM_ERR_ARCH",
    "LRM_ERR_CUDA",
]
(LRM_ERR_INVALID_ARG, LRM_ERR_SHAPE, LRM_ERR_ALIGN, LRM_ERR_WORKSPACE, LRM_ERR_INDEX, LRM_ERR_QUOTA,
 LRM_ERR_TIMEOUT, LRM_ERR_ARCH, LRM_ERR_CUDA) = range(1, 10)
LRM_OP_ROUTE_STATS = 0
LRM_OP_SELECT = 1
LRM_OP_ZERO_DROPPED = 2
LRM_OP_COMBINE = 3

# every entry point declared in include/lrm.h
EXPORTED = (
    "lrm_create",
    "lrm_destroy",
    "lrm_status_string",
    "lrm_abi_version",
    "lrm_sm_count",
    "lrm_workspace_size",
    "lrm_route_stats",
    "lrm_score",
    "lrm_select",
    "lrm_compact",
    "lrm_grouped_dgrad",
    "lrm_grouped_wgrad",
    "lrm_grouped_wgrad_bf16",
    "lrm_compact_padded",
    "lrm_get_device_status",
    "lrm_set_wait_budget",
    "lrm_selftest_wait_timeout",
    "lrm_route_stats_noalloc",
    "lrm_score_metric",
    "lrm_grouped_dgrad_scatter",
    "lrm_zero_dropped_rows",
    "lrm_swiglu_backward",
    "lrm_combine_rows",
    "lrm_capacity",
    "lrm_max_rows",
)

# selection metrics of lrm_score_metric (the ablation of LRMoE sec. 4.7, Table 2)
METRIC_LRM, METRIC_GRAD_L2SQ, METRIC_GRAD_L1, METRIC_RANDOM = 0, 1, 2, 3

# bytes of the library's fixed scratch array used by lrm_route_stats_noalloc
ROUTE_STATS_SCRATCH_BYTES = 4 << 20


class LrmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        name = STATUS_NAMES[code] if 0 <= code < len(STATUS_NAMES) else f"status {code}"
        super().__init__(f"{where}: {name}")


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("h", ctypes.c_int32),
                ("I", ctypes.c_int32)]


class RouteSummary(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int32),
        ("C", ctypes.c_int32),
        ("slots", ctypes.c_int32),
        ("dropped", ctypes.c_int32),
        ("retained", ctypes.c_int32),
        ("max_count", ctypes.c_int32),
        ("min_count", ctypes.c_int32),
        ("nonempty", ctypes.c_int32),
        ("aux_unscaled", ctypes.c_float),
        ("drop_rate", ctypes.c_float),
        ("util", ctypes.c_float),
        ("rho_real", ctypes.c_float),
        ("max_over_mean", ctypes.c_float),
        ("sum_P", ctypes.c_float),
    ]


SUMMARY_BYTES = ctypes.sizeof(RouteSummary)

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load liblrm.so and declare its signatures (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m backward_token_expert_gb300.build`")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    st = ctypes.c_int
    sig = {
        "lrm_create": ([ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)], st),
        "lrm_destroy": ([P], st),
        "lrm_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "lrm_abi_version": ([], i32),
        "lrm_sm_count": ([P, ctypes.POINTER(i32)], st),
        "lrm_workspace_size": ([P, ctypes.c_int, Dims, ctypes.POINTER(ctypes.c_size_t)], st),
        "lrm_route_stats": ([P, P, P, Dims, i32, i32, i32, i32, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], st),
        "lrm_score": ([P, P, P, P, Dims, P, P], st),
        "lrm_select": ([P, P, P, P, P, Dims, i32, P, P, P, ctypes.c_size_t, P], st),
        "lrm_compact": ([P, P, P, P, P, P, Dims, i32, P, P, P, P], st),
        "lrm_grouped_dgrad": ([P, P, P, P, Dims, i32, P, P], st),
        "lrm_grouped_wgrad": ([P, P, P, P, Dims, i32, i32, P, P], st),
        "lrm_grouped_wgrad_bf16": ([P, P, P, P, Dims, i32, i32, P, P], st),
        "lrm_compact_padded": ([P, P, P, P, Dims, i32, P, P, P, P], st),
        "lrm_get_device_status": ([P, P, ctypes.POINTER(ctypes.c_uint32)], st),
        "lrm_set_wait_budget": ([P, ctypes.c_uint64], st),
        "lrm_selftest_wait_timeout": ([P, ctypes.c_uint64, P], st),
        "lrm_route_stats_noalloc": ([P, P, P, Dims, i32, i32, i32, i32, P, P, P, P, P, P, P, P], st),
        "lrm_score_metric": ([P, i32, P, P, P, Dims, ctypes.c_uint64, P, P], st),
        "lrm_grouped_dgrad_scatter": ([P, P, P, P, P, Dims, i32, P, P], st),
        "lrm_zero_dropped_rows": ([P, P, P, Dims, i32, P, P, ctypes.c_size_t, P], st),
        "lrm_swiglu_backward": ([P, P, P, P, Dims, i32, P, P], st),
        "lrm_combine_rows": ([P, P, P, P, Dims, i32, i32, P, P, ctypes.c_size_t, P], st),
        "lrm_capacity": ([Dims, i32, i32, ctypes.POINTER(i32)], st),
        "lrm_max_rows": ([Dims, i32, i32, i32, i32, ctypes.POINTER(i32)], st),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str) -> None:
    if code != LRM_OK:
        raise LrmError(code, where)


def dims_of(T, E, k, h, I) -> Dims:
    return Dims(int(T), int(E), int(k), int(h), int(I))


# ---------------------------------------------------------------------------
# the C entry points, same names, argument marshalling only


def lrm_create(device: int = 0) -> int:
    lib = load_library()
    out = ctypes.c_void_p()
    _check(lib.lrm_create(int(device), ctypes.byref(out)), "lrm_create")
    return out.value


def lrm_destroy(ctx: int) -> None:
    _check(load_library().lrm_destroy(ctx), "lrm_destroy")


def lrm_status_string(code: int) -> str:
    return load_library().lrm_status_string(int(code)).decode()


def lrm_abi_version() -> int:
    return int(load_library().lrm_abi_version())


def lrm_sm_count(ctx: int) -> int:
    out = ctypes.c_int32()
    _check(load_library().lrm_sm_count(ctx, ctypes.byref(out)), "lrm_sm_count")
    return out.value


def lrm_workspace_size(ctx: int, op: int, dims: Dims) -> int:
    out = ctypes.c_size_t()
    _check(load_library().lrm_workspace_size(ctx, int(op), dims, ctypes.byref(out)), "lrm_workspace_size")
    return out.value


def lrm_capacity(dims: Dims, cf) -> int:
    """C = floor(CF * N / E), computed by the library (host only)."""
    cf = Fraction(cf)
    out = ctypes.c_int32()
    _check(load_library().lrm_capacity(dims, cf.numerator, cf.denominator, ctypes.byref(out)), "lrm_capacity")
    return out.value


def lrm_max_rows(dims: Dims, cf, rho) -> int:
    """Upper bound of the retained total over any routing, computed by the library (host only)."""
    cf = Fraction(cf)
    rho = Fraction(rho)
    out = ctypes.c_int32()
    _check(load_library().lrm_max_rows(dims, cf.numerator, cf.denominator, rho.numerator, rho.denominator,
                                       ctypes.byref(out)), "lrm_max_rows")
    return out.value


def lrm_route_stats(ctx, logits, expert_idx, dims: Dims, cf, rho, counts, offsets, bucket, P, f, quota,
                    summary, ws, ws_bytes: int, stream=None) -> None:
    cf = Fraction(cf)
    rho = Fraction(rho)
    _check(load_library().lrm_route_stats(ctx, _ptr(logits), _ptr(expert_idx), dims, cf.numerator,
                                          cf.denominator, rho.numerator, rho.denominator, _ptr(counts),
                                          _ptr(offsets), _ptr(bucket), _ptr(P), _ptr(f), _ptr(quota),
                                          _ptr(summary), _ptr(ws), int(ws_bytes), _stream(stream)),
           "lrm_route_stats")


def lrm_route_stats_noalloc(ctx, logits, expert_idx, dims: Dims, cf, rho, counts, offsets, bucket, P, f, quota,
                            summary, stream=None) -> None:
    """lrm_route_stats with the library's fixed scratch array instead of a workspace."""
    cf = Fraction(cf)
    rho = Fraction(rho)
    _check(load_library().lrm_route_stats_noalloc(ctx, _ptr(logits), _ptr(expert_idx), dims, cf.numerator,
                                                  cf.denominator, rho.numerator, rho.denominator, _ptr(counts),
                                                  _ptr(offsets), _ptr(bucket), _ptr(P), _ptr(f), _ptr(quota),
                                                  _ptr(summary), _stream(stream)),
           "lrm_route_stats_noalloc")


def lrm_score(ctx, g, phi, alpha, dims: Dims, score, stream=None) -> None:
    _check(load_library().lrm_score(ctx, _ptr(g), _ptr(phi), _ptr(alpha), dims, _ptr(score), _stream(stream)),
           "lrm_score")


def lrm_score_metric(ctx, metric: int, g, phi, alpha, dims: Dims, seed: int, score, stream=None) -> None:
    _check(load_library().lrm_score_metric(ctx, int(metric), _ptr(g), _ptr(phi), _ptr(alpha), dims,
                                           int(seed) & ((1 << 64) - 1), _ptr(score), _stream(stream)),
           "lrm_score_metric")


def lrm_grouped_dgrad_scatter(ctx, delta_c, W, sel_offsets, sel_ids, dims: Dims, max_rows: int, dphi_rows,
                              stream=None) -> None:
    _check(load_library().lrm_grouped_dgrad_scatter(ctx, _ptr(delta_c), _ptr(W), _ptr(sel_offsets), _ptr(sel_ids),
                                                    dims, int(max_rows), _ptr(dphi_rows), _stream(stream)),
           "lrm_grouped_dgrad_scatter")


def lrm_zero_dropped_rows(ctx, sel_offsets, sel_ids, dims: Dims, max_rows: int, rows, ws, ws_bytes: int,
                          stream=None) -> None:
    _check(load_library().lrm_zero_dropped_rows(ctx, _ptr(sel_offsets), _ptr(sel_ids), dims, int(max_rows),
                                                _ptr(rows), _ptr(ws), int(ws_bytes), _stream(stream)),
           "lrm_zero_dropped_rows")


def lrm_swiglu_backward(ctx, dphi_c, ab_c, sel_offsets, dims: Dims, max_rows: int, dh1, stream=None) -> None:
    _check(load_library().lrm_swiglu_backward(ctx, _ptr(dphi_c), _ptr(ab_c), _ptr(sel_offsets), dims,
                                              int(max_rows), _ptr(dh1), _stream(stream)), "lrm_swiglu_backward")


def lrm_combine_rows(ctx, rows, sel_offsets, sel_ids, dims: Dims, max_rows: int, width: int, out, ws, ws_bytes: int,
                     stream=None) -> None:
    _check(load_library().lrm_combine_rows(ctx, _ptr(rows), _ptr(sel_offsets), _ptr(sel_ids), dims, int(max_rows),
                                           int(width), _ptr(out), _ptr(ws), int(ws_bytes), _stream(stream)),
           "lrm_combine_rows")


def lrm_select(ctx, score, offsets, bucket, quota, dims: Dims, max_rows: int, sel_offsets, sel_ids, ws=None,
               ws_bytes: int = 0, stream=None) -> None:
    _check(load_library().lrm_select(ctx, _ptr(score), _ptr(offsets), _ptr(bucket), _ptr(quota), dims,
                                     int(max_rows), _ptr(sel_offsets), _ptr(sel_ids), _ptr(ws), int(ws_bytes),
                                     _stream(stream)), "lrm_select")


def lrm_compact(ctx, g, phi, alpha, sel_offsets, sel_ids, dims: Dims, max_rows: int, delta_c, phi_c,
                alpha_c=None, stream=None) -> None:
    _check(load_library().lrm_compact(ctx, _ptr(g), _ptr(phi), _ptr(alpha), _ptr(sel_offsets), _ptr(sel_ids),
                                      dims, int(max_rows), _ptr(delta_c), _ptr(phi_c), _ptr(alpha_c),
                                      _stream(stream)), "lrm_compact")


def lrm_grouped_dgrad(ctx, delta_c, W, sel_offsets, dims: Dims, max_rows: int, dphi_c, stream=None) -> None:
    _check(load_library().lrm_grouped_dgrad(ctx, _ptr(delta_c), _ptr(W), _ptr(sel_offsets), dims, int(max_rows),
                                            _ptr(dphi_c), _stream(stream)), "lrm_grouped_dgrad")


def lrm_grouped_wgrad(ctx, delta_c, phi_c, sel_offsets, dims: Dims, max_rows: int, accumulate: int, dW,
                      stream=None) -> None:
    _check(load_library().lrm_grouped_wgrad(ctx, _ptr(delta_c), _ptr(phi_c), _ptr(sel_offsets), dims,
                                            int(max_rows), int(accumulate), _ptr(dW), _stream(stream)),
           "lrm_grouped_wgrad")


def lrm_grouped_wgrad_bf16(ctx, delta_c, phi_c, sel_offsets, dims: Dims, max_rows: int, accumulate: int, dW,
                           stream=None) -> None:
    _check(load_library().lrm_grouped_wgrad_bf16(ctx, _ptr(delta_c), _ptr(phi_c), _ptr(sel_offsets), dims,
                                                 int(max_rows), int(accumulate), _ptr(dW), _stream(stream)),
           "lrm_grouped_wgrad_bf16")


def lrm_compact_padded(ctx, delta_c, phi_c, sel_offsets, dims: Dims, C: int, delta_pad, phi_pad, pad_offsets,
                       stream=None) -> None:
    _check(load_library().lrm_compact_padded(ctx, _ptr(delta_c), _ptr(phi_c), _ptr(sel_offsets), dims, int(C),
                                             _ptr(delta_pad), _ptr(phi_pad), _ptr(pad_offsets), _stream(stream)),
           "lrm_compact_padded")


def lrm_get_device_status(ctx, stream=None) -> int:
    out = ctypes.c_uint32()
    _check(load_library().lrm_get_device_status(ctx, _stream(stream), ctypes.byref(out)),
           "lrm_get_device_status")
    return out.value


def lrm_set_wait_budget(ctx, ns: int) -> None:
    _check(load_library().lrm_set_wait_budget(ctx, int(ns)), "lrm_set_wait_budget")


def lrm_selftest_wait_timeout(ctx, budget_ns: int, stream=None) -> None:
    _check(load_library().lrm_selftest_wait_timeout(ctx, int(budget_ns), _stream(stream)),
           "lrm_selftest_wait_timeout")


def flag_names(flags: int) -> list[str]:
    return [STATUS_NAMES[c] for c in range(1, len(STATUS_NAMES)) if flags & (1 << c)]
