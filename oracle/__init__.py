"""Oracle for the MoE permute + grouped matmul: the backward (d_x, d_weight),
the forward y it differentiates, and the probs-weighted unpermute backward.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``permute_grouped_gemm_gb300``) never imports, links or calls it, and this
package never imports the product.

The arithmetic lives in ``oracle_dx.cpp`` (plain C++17 loops, fp64
accumulation, multithreaded over tokens); this module compiles it with g++
and marshals arguments. It follows the element-wise gradient formula of the
page "MoeInitRoutingGroupedMatmulGrad design" (section "数学定义和公式"):

    d_x[b, k] = sum_{i : batch(i) = b} sum_n d_y[i, n] * weight[g(i), k, n]

with batch(i) = original_pos(i) // topK (same section, Step 2) and
expandedRowIdx read in gather (rowIdxType 0) or scatter (rowIdxType 1) form
(section "输入输出", note 1); and the weight gradient of the separate operator
the same page describes (section 1.2, "为何不计算 d_weight" item 3:
expanded_x^T @ d_y per expert, expanded_x[i] = x[batch(i)] from the forward's
MoeInitRouting of section 1.1):

    d_weight[g, k, n] = sum_{i in expert g} x[batch(i), k] * d_y[i, n]

Pins (``tests/test_oracle_pins.py``, ``tests/test_oracle_dw_pins.py``): a
pure-Python indicator-sum brute force,
the unfused two-step form written with numpy, ``torch.matmul`` for the
one-expert identity-routing case, hand-derived closed forms, a hand-worked
example in ``tests/golden/``, and invariants (column sums, expert relabelling,
empty experts, gather vs scatter index, linearity), and for d_weight the
adjoint identity sum(d_weight * weight) == sum(d_x * x), which ties the two
functions to each other. The dtype decoders are pinned against numpy / torch
conversions of every 16-bit pattern.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_dx.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle_dx.so")

F32, F16, BF16 = 0, 1, 2

ERRORS = {
    0: "ok",
    1: "null pointer",
    2: "shape",
    3: "attribute",
    4: "dtype",
    16: "index out of range",
    17: "groupList sum != M or negative count",
    18: "index is not a permutation",
}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with g++ (no CUDA)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
        )
        os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """ctypes handle with the oracle's signatures (also used by the mutation tests)."""
    lib = ctypes.CDLL(path)
    i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.oracle_dx.argtypes = [vp, vp, ctypes.c_int, vp, vp, i64, i64, i64, i64,
                              i64, i64, ctypes.c_int, vp, i64, dp, ctypes.c_int]
    lib.oracle_dx.restype = ctypes.c_int
    lib.oracle_decode.argtypes = [vp, ctypes.c_int, i64, dp]
    lib.oracle_decode.restype = ctypes.c_int
    lib.oracle_dw.argtypes = [vp, vp, ctypes.c_int, vp, vp, i64, i64, i64, i64,
                              i64, i64, ctypes.c_int, vp, vp, i64, dp, ctypes.c_int]
    lib.oracle_dw.restype = ctypes.c_int
    lib.oracle_fwd.argtypes = [vp, vp, ctypes.c_int, vp, vp, i64, i64, i64, i64,
                               i64, i64, ctypes.c_int, vp, i64, dp, ctypes.c_int]
    lib.oracle_fwd.restype = ctypes.c_int
    lib.oracle_unpermute_grad.argtypes = [vp, vp, vp, ctypes.c_int, vp, i64, i64, i64, i64,
                                          ctypes.c_int, dp, dp, ctypes.c_int]
    lib.oracle_unpermute_grad.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _raw(a):
    """(contiguous numpy array of the raw element bits, dtype code)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(a, torch.Tensor):
        a = a.detach().cpu().contiguous()
        if a.dtype == torch.bfloat16:
            return a.view(torch.int16).numpy(), BF16
        if a.dtype == torch.float16:
            return a.view(torch.int16).numpy(), F16
        if a.dtype == torch.float32:
            return a.numpy(), F32
        raise TypeError(f"unsupported dtype {a.dtype}")
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.int16), F16
    if a.dtype == np.float32:
        return a, F32
    raise TypeError(f"unsupported dtype {a.dtype}")


def _i64(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=np.int64)


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle rejected the inputs: {ERRORS.get(code, code)} (code {code})")
        self.code = code


def dx(grad_y, weight, expanded_row_idx, group_list, batch: int, top_k: int,
       row_idx_type: int, tokens=None, nthreads: int = 0, lib=None) -> np.ndarray:
    """fp64 d_x rows for ``tokens`` (all tokens if None): array [len(tokens), K].

    grad_y: [M, N], weight: [G, K, N] (torch CPU/CUDA tensors or numpy; fp32,
    fp16 or bf16, same dtype), expanded_row_idx: int64 [M], group_list: int64
    [G] counts. Raises OracleError with the constraint that failed. ``lib``
    selects another build of the same source (mutation tests only).
    """
    lib = lib or _load()
    dy, dt = _raw(grad_y)
    w, dtw = _raw(weight)
    if dt != dtw:
        raise OracleError(4)
    M, N = dy.shape
    G, K, Nw = w.shape
    if Nw != N:
        raise OracleError(2)
    idx = _i64(expanded_row_idx)
    gl = _i64(group_list)
    if idx.shape != (M,) or gl.shape != (G,):
        raise OracleError(2)
    if tokens is None:
        tok = None
        nt = batch
    else:
        tok = _i64(tokens)
        nt = tok.shape[0]
    out = np.empty((nt, K), dtype=np.float64)
    rc = lib.oracle_dx(dy.ctypes.data, w.ctypes.data, dt, idx.ctypes.data, gl.ctypes.data,
                       M, N, K, G, batch, top_k, row_idx_type,
                       None if tok is None else tok.ctypes.data, nt, out.ctypes.data,
                       int(nthreads))
    if rc != 0:
        raise OracleError(rc)
    return out


def dw(x, grad_y, expanded_row_idx, group_list, batch: int, top_k: int, row_idx_type: int,
       sel=None, nthreads: int = 0, lib=None) -> np.ndarray:
    """fp64 d_weight. With ``sel`` None: array [G, K, N]; otherwise ``sel`` is a
    pair (g, k) of int arrays and the result is [len(g), N], row s being
    d_weight[g[s], k[s], :].

    x: [batch, K] (the forward input, original token order), grad_y: [M, N],
    same dtype; expanded_row_idx, group_list as for ``dx``. ``group_list`` also
    fixes G.
    """
    lib = lib or _load()
    xr, dt = _raw(x)
    dy, dty = _raw(grad_y)
    if dt != dty:
        raise OracleError(4)
    B, K = xr.shape
    M, N = dy.shape
    idx = _i64(expanded_row_idx)
    gl = _i64(group_list)
    G = gl.shape[0]
    if B != batch or idx.shape != (M,):
        raise OracleError(2)
    if sel is None:
        sg = sk = None
        ns = G * K
    else:
        sg, sk = _i64(sel[0]), _i64(sel[1])
        if sg.shape != sk.shape or sg.ndim != 1:
            raise OracleError(2)
        ns = sg.shape[0]
    out = np.empty((ns, N), dtype=np.float64)
    rc = lib.oracle_dw(xr.ctypes.data, dy.ctypes.data, dt, idx.ctypes.data, gl.ctypes.data,
                       M, N, K, G, batch, top_k, row_idx_type,
                       None if sg is None else sg.ctypes.data,
                       None if sk is None else sk.ctypes.data, ns, out.ctypes.data,
                       int(nthreads))
    if rc != 0:
        raise OracleError(rc)
    return out.reshape(G, K, N) if sel is None else out


def fwd(x, weight, expanded_row_idx, group_list, batch: int, top_k: int, row_idx_type: int,
        rows=None, nthreads: int = 0, lib=None) -> np.ndarray:
    """fp64 forward y [M, N] in expanded order (or the listed ``rows``):
    y[i] = x[batch(i)] @ weight[g(i)]. x: [batch, K], weight: [G, K, N], same
    dtype."""
    lib = lib or _load()
    xr, dt = _raw(x)
    w, dtw = _raw(weight)
    if dt != dtw:
        raise OracleError(4)
    B, K = xr.shape
    G, Kw, N = w.shape
    idx = _i64(expanded_row_idx)
    gl = _i64(group_list)
    M = idx.shape[0]
    if B != batch or Kw != K or gl.shape != (G,):
        raise OracleError(2)
    if rows is None:
        rw = None
        nr = M
    else:
        rw = _i64(rows)
        nr = rw.shape[0]
    out = np.empty((nr, N), dtype=np.float64)
    rc = lib.oracle_fwd(xr.ctypes.data, w.ctypes.data, dt, idx.ctypes.data, gl.ctypes.data,
                        M, N, K, G, batch, top_k, row_idx_type,
                        None if rw is None else rw.ctypes.data, nr, out.ctypes.data,
                        int(nthreads))
    if rc != 0:
        raise OracleError(rc)
    return out


def unpermute_grad(permuted, d_out, probs, expanded_row_idx, batch: int, top_k: int,
                   row_idx_type: int, nthreads: int = 0, lib=None):
    """fp64 (perm_grad [M, H], probs_grad [batch, topK] or None) of the
    probs-weighted unpermute: permuted [M, H] (may be None without probs),
    d_out [batch, H], probs [batch, topK] or None, same dtype."""
    lib = lib or _load()
    d, dt = _raw(d_out)
    B, H = d.shape
    idx = _i64(expanded_row_idx)
    M = idx.shape[0]
    if B != batch:
        raise OracleError(2)
    pr = pm = None
    if probs is not None:
        pr, dtp = _raw(probs)
        pm, dtm = _raw(permuted)
        if dtp != dt or dtm != dt:
            raise OracleError(4)
        if pr.shape != (batch, top_k) or pm.shape != (M, H):
            raise OracleError(2)
    pg = np.empty((M, H), dtype=np.float64)
    qg = np.empty((batch, top_k), dtype=np.float64) if probs is not None else None
    rc = lib.oracle_unpermute_grad(None if pm is None else pm.ctypes.data, d.ctypes.data,
                                   None if pr is None else pr.ctypes.data, dt, idx.ctypes.data,
                                   M, H, batch, top_k, row_idx_type, pg.ctypes.data,
                                   None if qg is None else qg.ctypes.data, int(nthreads))
    if rc != 0:
        raise OracleError(rc)
    return pg, qg


def decode(raw_bits: np.ndarray, dtype_code: int, lib=None) -> np.ndarray:
    """Widen raw element bits (uint16 for fp16/bf16, float32 for fp32) to fp64."""
    lib = lib or _load()
    src = np.ascontiguousarray(raw_bits)
    out = np.empty(src.size, dtype=np.float64)
    rc = lib.oracle_decode(src.ctypes.data, dtype_code, src.size, out.ctypes.data)
    if rc != 0:
        raise OracleError(rc)
    return out.reshape(src.shape)


def host_cores() -> int:
    """Threads the oracle uses by default (std::thread::hardware_concurrency)."""
    return os.cpu_count() or 1
