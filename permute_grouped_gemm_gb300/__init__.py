"""GB300 (sm_103a) fused MoE permute + grouped-matmul backward, input gradient.

    d_x[b, k] = sum_{i : batch(i) = b} sum_n grad_y[i, n] * weight[g(i), k, n]

("MoeInitRoutingGroupedMatmulGrad design", section "数学定义和公式".) The work
runs in libpgg.so (include/pgg.h); this package is its thin binding. PyTorch
supplies device memory and the current stream only.
"""

from __future__ import annotations

from ._lib import (  # noqa: F401
    CODES, PGG_BF16, PGG_F16, PGG_F32, STATUS, PggError, load,
    pgg_debug_force_variant, pgg_debug_set_band_k_blocks, pgg_debug_set_hold_release,
    pgg_debug_set_ticket_bias, pgg_debug_set_wait_limit_ns,
    pgg_dw_execute, pgg_dw_grouped_gemm, pgg_dw_plan, pgg_dw_workspace_size,
    pgg_fwd_execute, pgg_fwd_grouped_gemm, pgg_fwd_plan, pgg_fwd_route_prep,
    pgg_fwd_workspace_size, pgg_unpermute_grad, pgg_unpermute_grad_apply,
    pgg_unpermute_grad_prep, pgg_unpermute_grad_workspace_size,
    pgg_dx_execute, pgg_dx_execute_static_scratch, pgg_dx_grouped_gemm, pgg_dx_plan,
    pgg_dx_route_prep,
    pgg_dx_workspace_size, pgg_status_string,
)

_DT = None


def dtype_code(torch_dtype) -> int:
    global _DT
    if _DT is None:
        import torch
        _DT = {torch.float32: PGG_F32, torch.float16: PGG_F16, torch.bfloat16: PGG_BF16}
    if torch_dtype not in _DT:
        raise PggError(CODES["PGG_ERR_DTYPE"], "dtype_code")
    return _DT[torch_dtype]


def _args(grad_y, weight, expanded_row_idx, group_list, batch, top_k):
    M, N = grad_y.shape
    G, K, _ = weight.shape
    return M, N, K, G, expanded_row_idx.shape[0], batch, top_k


def workspace_bytes(grad_y, weight, expanded_row_idx, group_list, batch, top_k,
                    row_idx_type) -> int:
    sizes = _args(grad_y, weight, expanded_row_idx, group_list, batch, top_k)
    return pgg_dx_workspace_size(*sizes, row_idx_type, dtype_code(grad_y.dtype))


def dx(grad_y, weight, expanded_row_idx, group_list, batch: int, top_k: int,
       row_idx_type: int, out=None, workspace=None, stream=None):
    """d_x [batch, K] fp32 on grad_y's device (torch tensors, contiguous, CUDA).

    Allocates ``out`` and the workspace through torch when not given. The call
    is asynchronous on ``stream`` (default: torch's current stream); the
    device-detected status is the first int32 of the workspace.
    Returns (out, workspace).
    """
    import torch
    for t in (grad_y, weight, expanded_row_idx, group_list):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    if expanded_row_idx.dtype != torch.int64 or group_list.dtype != torch.int64:
        raise ValueError("expandedRowIdx and groupList must be int64")
    sizes = _args(grad_y, weight, expanded_row_idx, group_list, batch, top_k)
    dt = dtype_code(grad_y.dtype)
    if weight.dtype != grad_y.dtype:
        raise PggError(CODES["PGG_ERR_DTYPE"], "dx")
    need = pgg_dx_workspace_size(*sizes, row_idx_type, dt)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=grad_y.device)
    if out is None:
        out = torch.empty(batch, sizes[2], dtype=torch.float32, device=grad_y.device)
    if stream is None:
        stream = torch.cuda.current_stream(grad_y.device)
    rc = pgg_dx_execute(grad_y.data_ptr(), weight.data_ptr(), expanded_row_idx.data_ptr(),
                        group_list.data_ptr(), *sizes, row_idx_type, dt, workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), out.data_ptr(),
                        stream.cuda_stream)
    if rc != 0:
        raise PggError(rc, "pgg_dx_execute")
    return out, workspace


def dw(x, grad_y, expanded_row_idx, group_list, batch: int, top_k: int, row_idx_type: int,
       G: int | None = None, out_dtype=None, out=None, workspace=None, stream=None):
    """d_weight [G, K, N] (``out_dtype``: grad_y's dtype by default, or
    torch.float32) from the forward input x [batch, K] and grad_y [M, N].
    G defaults to len(group_list). Returns (out, workspace)."""
    import torch
    for t in (x, grad_y, expanded_row_idx, group_list):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    if expanded_row_idx.dtype != torch.int64 or group_list.dtype != torch.int64:
        raise ValueError("expandedRowIdx and groupList must be int64")
    if x.dtype != grad_y.dtype:
        raise PggError(CODES["PGG_ERR_DTYPE"], "dw")
    M, N = grad_y.shape
    _, K = x.shape
    G = group_list.shape[0] if G is None else G
    sizes = (M, N, K, G, expanded_row_idx.shape[0], batch, top_k)
    dt = dtype_code(grad_y.dtype)
    out_dtype = grad_y.dtype if out_dtype is None else out_dtype
    odt = dtype_code(out_dtype)
    need = pgg_dw_workspace_size(*sizes, row_idx_type, dt)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=grad_y.device)
    if out is None:
        out = torch.empty(G, K, N, dtype=out_dtype, device=grad_y.device)
    if stream is None:
        stream = torch.cuda.current_stream(grad_y.device)
    rc = pgg_dw_execute(x.data_ptr(), grad_y.data_ptr(), expanded_row_idx.data_ptr(),
                        group_list.data_ptr(), *sizes, row_idx_type, dt, odt,
                        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        out.data_ptr(), stream.cuda_stream)
    if rc != 0:
        raise PggError(rc, "pgg_dw_execute")
    return out, workspace


def fwd(x, weight, expanded_row_idx, group_list, batch: int, top_k: int, row_idx_type: int,
        out_dtype=None, out=None, workspace=None, stream=None):
    """Forward y [M, N] (expanded order; ``out_dtype``: x's dtype by default, or
    torch.float32) from x [batch, K] and weight [G, K, N]. Returns (y, workspace)."""
    import torch
    for t in (x, weight, expanded_row_idx, group_list):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    if expanded_row_idx.dtype != torch.int64 or group_list.dtype != torch.int64:
        raise ValueError("expandedRowIdx and groupList must be int64")
    if x.dtype != weight.dtype:
        raise PggError(CODES["PGG_ERR_DTYPE"], "fwd")
    G, K, N = weight.shape
    M = expanded_row_idx.shape[0]
    sizes = (M, N, K, G, M, batch, top_k)
    dt = dtype_code(x.dtype)
    out_dtype = x.dtype if out_dtype is None else out_dtype
    odt = dtype_code(out_dtype)
    need = pgg_fwd_workspace_size(*sizes, row_idx_type, dt)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    rc = pgg_fwd_execute(x.data_ptr(), weight.data_ptr(), expanded_row_idx.data_ptr(),
                         group_list.data_ptr(), *sizes, row_idx_type, dt, odt,
                         workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                         out.data_ptr(), stream.cuda_stream)
    if rc != 0:
        raise PggError(rc, "pgg_fwd_execute")
    return out, workspace


def unpermute_grad(permuted, d_out, probs, expanded_row_idx, top_k: int, row_idx_type: int,
                   probs_grad_dtype=None, perm_grad=None, probs_grad=None, workspace=None,
                   stream=None):
    """(perm_grad [M, H], probs_grad [batch, topK] or None, workspace) of the
    probs-weighted unpermute (probs None: plain scatter copy)."""
    import torch
    for t in (d_out, expanded_row_idx) + ((permuted, probs) if probs is not None else ()):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    batch, H = d_out.shape
    M = expanded_row_idx.shape[0]
    dt = dtype_code(d_out.dtype)
    pdt = d_out.dtype if probs_grad_dtype is None else probs_grad_dtype
    need = pgg_unpermute_grad_workspace_size(M, batch, top_k)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=d_out.device)
    if perm_grad is None:
        perm_grad = torch.empty(M, H, dtype=d_out.dtype, device=d_out.device)
    if probs is not None and probs_grad is None:
        probs_grad = torch.empty(batch, top_k, dtype=pdt, device=d_out.device)
    if stream is None:
        stream = torch.cuda.current_stream(d_out.device)
    rc = pgg_unpermute_grad(permuted.data_ptr() if probs is not None else 0, d_out.data_ptr(),
                            probs.data_ptr() if probs is not None else 0,
                            expanded_row_idx.data_ptr(), M, H, batch, top_k, row_idx_type, dt,
                            dtype_code(pdt), workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), perm_grad.data_ptr(),
                            probs_grad.data_ptr() if probs is not None else 0,
                            stream.cuda_stream)
    if rc != 0:
        raise PggError(rc, "pgg_unpermute_grad")
    return perm_grad, (probs_grad if probs is not None else None), workspace


def status(workspace) -> int:
    """Device-detected status word of a finished call (synchronises)."""
    import torch
    return int(workspace[:4].view(torch.int32).item())
