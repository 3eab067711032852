"""ctypes binding of libpgg.so: the C-ABI functions of include/pgg.h under the
same names, with argument marshalling only. Every step of the computation runs
in the library's CUDA kernels; there is no Python or CPU fallback, and loading
fails loudly when the library has not been built."""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

PGG_F32, PGG_F16, PGG_BF16 = 0, 1, 2

STATUS = {
    0: "PGG_OK", 1: "PGG_ERR_NULL", 2: "PGG_ERR_SHAPE", 3: "PGG_ERR_ATTR", 4: "PGG_ERR_DTYPE",
    5: "PGG_ERR_WORKSPACE", 6: "PGG_ERR_CUDA", 7: "PGG_ERR_ALIGN", 16: "PGG_ERR_INDEX",
    17: "PGG_ERR_GROUPSUM", 18: "PGG_ERR_NOT_PERM", 19: "PGG_ERR_TIMEOUT", 20: "PGG_ERR_CHECK",
}
CODES = {v: k for k, v in STATUS.items()}

_lock = threading.Lock()
_handle = None


class PggError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        super().__init__(f"{where}: {STATUS.get(code, code)} ({code})")
        self.code = code


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("variant", ctypes.c_int32), ("rows_per_block", ctypes.c_int32),
        ("k_per_block", ctypes.c_int32), ("stages", ctypes.c_int32),
        ("k_blocks", ctypes.c_int32), ("band_k_blocks", ctypes.c_int32),
        ("max_row_blocks", ctypes.c_int64), ("workspace_bytes", ctypes.c_size_t),
        ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
        ("cta_pair", ctypes.c_int32),
    ]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_SIZES = [ctypes.c_int64] * 7  # M, N, K, G, L, batch, topK


def load(path: str | None = None):
    """The loaded library (ctypes.CDLL). Raises if it has not been built."""
    global _handle
    with _lock:
        if _handle is None:
            lib_path = path or _build.LIB
            if not os.path.exists(lib_path):
                raise ImportError(f"libpgg.so is not built ({lib_path}); run "
                                  "permute_grouped_gemm_gb300.build.build()")
            lib = ctypes.CDLL(lib_path)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.pgg_dx_workspace_size.argtypes = [*_SIZES, i32, i32, ctypes.POINTER(sz)]
            lib.pgg_dx_plan.argtypes = [*_SIZES, i32, i32, ctypes.POINTER(PlanInfo)]
            lib.pgg_dx_execute.argtypes = [vp, vp, vp, vp, *_SIZES, i32, i32, vp, sz, vp, vp]
            lib.pgg_dx_grouped_gemm.argtypes = [vp, vp, vp, vp, *_SIZES, i32, i32, vp, sz, vp, vp]
            lib.pgg_dx_route_prep.argtypes = [vp, vp, *_SIZES, i32, i32, vp, sz, vp]
            lib.pgg_dx_execute_static_scratch.argtypes = [vp, vp, vp, vp, *_SIZES, i32, i32, vp,
                                                          vp, vp]
            lib.pgg_dw_workspace_size.argtypes = [*_SIZES, i32, i32, ctypes.POINTER(sz)]
            lib.pgg_dw_plan.argtypes = [*_SIZES, i32, i32, ctypes.POINTER(PlanInfo)]
            lib.pgg_dw_execute.argtypes = [vp, vp, vp, vp, *_SIZES, i32, i32, i32, vp, sz, vp, vp]
            lib.pgg_dw_grouped_gemm.argtypes = [vp, vp, vp, vp, *_SIZES, i32, i32, i32, vp, sz,
                                                vp, vp]
            lib.pgg_fwd_workspace_size.argtypes = [*_SIZES, i32, i32, ctypes.POINTER(sz)]
            lib.pgg_fwd_plan.argtypes = [*_SIZES, i32, i32, ctypes.POINTER(PlanInfo)]
            lib.pgg_fwd_execute.argtypes = [vp, vp, vp, vp, *_SIZES, i32, i32, i32, vp, sz, vp,
                                            vp]
            lib.pgg_fwd_grouped_gemm.argtypes = [vp, vp, vp, vp, *_SIZES, i32, i32, i32, vp, sz,
                                                 vp, vp]
            lib.pgg_fwd_route_prep.argtypes = [vp, vp, *_SIZES, i32, i32, vp, sz, vp]
            lib.pgg_unpermute_grad_workspace_size.argtypes = [ctypes.c_int64] * 3 + [
                ctypes.POINTER(sz)]
            lib.pgg_unpermute_grad.argtypes = [vp, vp, vp, vp] + [ctypes.c_int64] * 4 + [
                i32, i32, i32, vp, sz, vp, vp, vp]
            lib.pgg_unpermute_grad_apply.argtypes = lib.pgg_unpermute_grad.argtypes
            lib.pgg_unpermute_grad_prep.argtypes = [vp] + [ctypes.c_int64] * 3 + [i32, vp, sz, vp]
            for f in ("pgg_unpermute_grad_workspace_size", "pgg_unpermute_grad",
                      "pgg_unpermute_grad_prep", "pgg_unpermute_grad_apply"):
                getattr(lib, f).restype = ctypes.c_int
            for f in ("pgg_fwd_workspace_size", "pgg_fwd_plan", "pgg_fwd_execute",
                      "pgg_fwd_grouped_gemm", "pgg_fwd_route_prep"):
                getattr(lib, f).restype = ctypes.c_int
            for f in ("pgg_dx_workspace_size", "pgg_dx_plan", "pgg_dx_execute",
                      "pgg_dx_grouped_gemm", "pgg_dx_route_prep", "pgg_dx_execute_static_scratch",
                      "pgg_dw_workspace_size", "pgg_dw_plan", "pgg_dw_execute",
                      "pgg_dw_grouped_gemm"):
                getattr(lib, f).restype = ctypes.c_int
            lib.pgg_status_string.argtypes = [ctypes.c_int]
            lib.pgg_status_string.restype = ctypes.c_char_p
            lib.pgg_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            lib.pgg_debug_set_ticket_bias.argtypes = [ctypes.c_uint32]
            lib.pgg_debug_force_variant.argtypes = [ctypes.c_int]
            lib.pgg_debug_set_band_k_blocks.argtypes = [ctypes.c_int]
            lib.pgg_debug_set_hold_release.argtypes = [ctypes.c_int]
            for f in ("pgg_debug_set_wait_limit_ns", "pgg_debug_set_ticket_bias",
                      "pgg_debug_force_variant", "pgg_debug_set_band_k_blocks",
                      "pgg_debug_set_hold_release"):
                getattr(lib, f).restype = None
            _handle = lib
    return _handle


def _check(rc: int, where: str):
    if rc != 0:
        raise PggError(rc, where)


def pgg_dx_workspace_size(M, N, K, G, L, batch, topK, rowIdxType, dtype) -> int:
    out = ctypes.c_size_t(0)
    _check(load().pgg_dx_workspace_size(M, N, K, G, L, batch, topK, rowIdxType, dtype,
                                        ctypes.byref(out)), "pgg_dx_workspace_size")
    return out.value


def pgg_dx_plan(M, N, K, G, L, batch, topK, rowIdxType, dtype) -> dict:
    info = PlanInfo()
    _check(load().pgg_dx_plan(M, N, K, G, L, batch, topK, rowIdxType, dtype,
                              ctypes.byref(info)), "pgg_dx_plan")
    return info.as_dict()


def pgg_dx_execute(gradY, weight, expandedRowIdx, groupList, M, N, K, G, L, batch, topK,
                   rowIdxType, dtype, workspace, workspace_bytes, out, stream) -> int:
    """Raw call with integer device addresses; returns the pgg_status code."""
    return load().pgg_dx_execute(gradY, weight, expandedRowIdx, groupList, M, N, K, G, L, batch,
                                 topK, rowIdxType, dtype, workspace, workspace_bytes, out, stream)


def pgg_dx_route_prep(expandedRowIdx, groupList, M, N, K, G, L, batch, topK, rowIdxType, dtype,
                      workspace, workspace_bytes, stream) -> int:
    return load().pgg_dx_route_prep(expandedRowIdx, groupList, M, N, K, G, L, batch, topK,
                                    rowIdxType, dtype, workspace, workspace_bytes, stream)


def pgg_dx_grouped_gemm(gradY, weight, expandedRowIdx, groupList, M, N, K, G, L, batch, topK,
                        rowIdxType, dtype, workspace, workspace_bytes, out, stream) -> int:
    return load().pgg_dx_grouped_gemm(gradY, weight, expandedRowIdx, groupList, M, N, K, G, L,
                                      batch, topK, rowIdxType, dtype, workspace, workspace_bytes,
                                      out, stream)


def pgg_dx_execute_static_scratch(gradY, weight, expandedRowIdx, groupList, M, N, K, G, L, batch,
                                  topK, rowIdxType, dtype, out, status, stream) -> int:
    """pgg_dx_execute without a workspace argument, for callers that cannot
    allocate device memory: the library's fixed 8 MiB device scratch is used.
    `status` is an optional device address (0 = none) that receives the
    device-detected status word. Returns the pgg_status code."""
    return load().pgg_dx_execute_static_scratch(gradY, weight, expandedRowIdx, groupList, M, N, K,
                                                G, L, batch, topK, rowIdxType, dtype, out,
                                                status or None, stream)


def pgg_dw_workspace_size(M, N, K, G, L, batch, topK, rowIdxType, dtype) -> int:
    out = ctypes.c_size_t(0)
    _check(load().pgg_dw_workspace_size(M, N, K, G, L, batch, topK, rowIdxType, dtype,
                                        ctypes.byref(out)), "pgg_dw_workspace_size")
    return out.value


def pgg_dw_plan(M, N, K, G, L, batch, topK, rowIdxType, dtype) -> dict:
    info = PlanInfo()
    _check(load().pgg_dw_plan(M, N, K, G, L, batch, topK, rowIdxType, dtype,
                              ctypes.byref(info)), "pgg_dw_plan")
    return info.as_dict()


def pgg_dw_execute(x, gradY, expandedRowIdx, groupList, M, N, K, G, L, batch, topK, rowIdxType,
                   dtype, out_dtype, workspace, workspace_bytes, dweight, stream) -> int:
    """Raw call with integer device addresses; returns the pgg_status code."""
    return load().pgg_dw_execute(x, gradY, expandedRowIdx, groupList, M, N, K, G, L, batch, topK,
                                 rowIdxType, dtype, out_dtype, workspace, workspace_bytes,
                                 dweight, stream)


def pgg_dw_grouped_gemm(x, gradY, expandedRowIdx, groupList, M, N, K, G, L, batch, topK,
                        rowIdxType, dtype, out_dtype, workspace, workspace_bytes, dweight,
                        stream) -> int:
    return load().pgg_dw_grouped_gemm(x, gradY, expandedRowIdx, groupList, M, N, K, G, L, batch,
                                      topK, rowIdxType, dtype, out_dtype, workspace,
                                      workspace_bytes, dweight, stream)


def pgg_fwd_workspace_size(M, N, K, G, L, batch, topK, rowIdxType, dtype) -> int:
    out = ctypes.c_size_t(0)
    _check(load().pgg_fwd_workspace_size(M, N, K, G, L, batch, topK, rowIdxType, dtype,
                                         ctypes.byref(out)), "pgg_fwd_workspace_size")
    return out.value


def pgg_fwd_plan(M, N, K, G, L, batch, topK, rowIdxType, dtype) -> dict:
    info = PlanInfo()
    _check(load().pgg_fwd_plan(M, N, K, G, L, batch, topK, rowIdxType, dtype,
                               ctypes.byref(info)), "pgg_fwd_plan")
    return info.as_dict()


def pgg_fwd_execute(x, weight, expandedRowIdx, groupList, M, N, K, G, L, batch, topK,
                    rowIdxType, dtype, out_dtype, workspace, workspace_bytes, y, stream) -> int:
    """Raw call with integer device addresses; returns the pgg_status code."""
    return load().pgg_fwd_execute(x, weight, expandedRowIdx, groupList, M, N, K, G, L, batch,
                                  topK, rowIdxType, dtype, out_dtype, workspace, workspace_bytes,
                                  y, stream)


def pgg_fwd_route_prep(expandedRowIdx, groupList, M, N, K, G, L, batch, topK, rowIdxType, dtype,
                       workspace, workspace_bytes, stream) -> int:
    return load().pgg_fwd_route_prep(expandedRowIdx, groupList, M, N, K, G, L, batch, topK,
                                      rowIdxType, dtype, workspace, workspace_bytes, stream)


def pgg_fwd_grouped_gemm(x, weight, expandedRowIdx, groupList, M, N, K, G, L, batch, topK,
                         rowIdxType, dtype, out_dtype, workspace, workspace_bytes, y,
                         stream) -> int:
    return load().pgg_fwd_grouped_gemm(x, weight, expandedRowIdx, groupList, M, N, K, G, L,
                                       batch, topK, rowIdxType, dtype, out_dtype, workspace,
                                       workspace_bytes, y, stream)


def pgg_unpermute_grad_workspace_size(M, batch, topK) -> int:
    out = ctypes.c_size_t(0)
    _check(load().pgg_unpermute_grad_workspace_size(M, batch, topK, ctypes.byref(out)),
           "pgg_unpermute_grad_workspace_size")
    return out.value


def pgg_unpermute_grad(permuted, d_out, probs, expandedRowIdx, M, H, batch, topK, rowIdxType,
                       dtype, probs_grad_dtype, workspace, workspace_bytes, perm_grad, probs_grad,
                       stream) -> int:
    """Raw call with integer device addresses (0 for an absent optional one)."""
    return load().pgg_unpermute_grad(permuted or None, d_out, probs or None, expandedRowIdx, M,
                                     H, batch, topK, rowIdxType, dtype, probs_grad_dtype,
                                     workspace, workspace_bytes, perm_grad, probs_grad or None,
                                     stream)


def pgg_unpermute_grad_prep(expandedRowIdx, M, batch, topK, rowIdxType, workspace,
                            workspace_bytes, stream) -> int:
    """Raw call: index validation and inverse map into the workspace."""
    return load().pgg_unpermute_grad_prep(expandedRowIdx, M, batch, topK, rowIdxType, workspace,
                                          workspace_bytes, stream)


def pgg_unpermute_grad_apply(permuted, d_out, probs, expandedRowIdx, M, H, batch, topK,
                             rowIdxType, dtype, probs_grad_dtype, workspace, workspace_bytes,
                             perm_grad, probs_grad, stream) -> int:
    """Raw call: the unpermute kernel on a workspace filled by the prep step."""
    return load().pgg_unpermute_grad_apply(permuted or None, d_out, probs or None,
                                           expandedRowIdx, M, H, batch, topK, rowIdxType, dtype,
                                           probs_grad_dtype, workspace, workspace_bytes,
                                           perm_grad, probs_grad or None, stream)


def pgg_status_string(code: int) -> str:
    return load().pgg_status_string(code).decode()


def pgg_debug_set_wait_limit_ns(ns: int):
    load().pgg_debug_set_wait_limit_ns(ns)


def pgg_debug_set_ticket_bias(bias: int):
    load().pgg_debug_set_ticket_bias(bias)


def pgg_debug_force_variant(variant: int):
    load().pgg_debug_force_variant(variant)


def pgg_debug_set_band_k_blocks(k_blocks: int):
    load().pgg_debug_set_band_k_blocks(k_blocks)


def pgg_debug_set_hold_release(hold: int):
    load().pgg_debug_set_hold_release(hold)
