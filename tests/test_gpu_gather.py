"""GPU parity of plan variant 5: the ticketed CTA-pair d_x kernel whose
operands are copied by gather warps (4-byte cp.async into the 128-byte swizzle
layout) instead of the tensor-memory-access unit.

It serves rows of N * 2 bytes that are not a multiple of 16 (even N, 16-bit
dtypes: the page's N = 286 tail case of the white-box list) and gradY / weight
pointers that are 4-byte but not 16-byte aligned. Its shared-memory operands,
MMAs, tile order and epilogue are those of variant 0, so on rows both can
read it must agree with variant 0 bit for bit; everywhere it must match the
fp64 oracle within 1e-4 * max |d_x_ref| and repeat bitwise.
"""

import numpy as np
import pytest
import torch

import oracle
import permute_grouped_gemm_gb300 as pgg
from workloads import make_case
from workloads.moe import with_row_idx_type

pytestmark = pytest.mark.gpu

TOL = 1e-4
GATHER = 5


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from permute_grouped_gemm_gb300 import build as pbuild
    pbuild.build()
    oracle.build()
    pgg.load()
    yield
    pgg.pgg_debug_force_variant(-1)
    pgg.pgg_debug_set_ticket_bias(0)
    pgg.pgg_debug_set_wait_limit_ns(0)


def run(inp, variant=-1, grad_y=None, weight=None):
    try:
        pgg.pgg_debug_force_variant(variant)
        out, ws = pgg.dx(inp.grad_y if grad_y is None else grad_y,
                         inp.weight if weight is None else weight, inp.expanded_row_idx,
                         inp.group_list, inp.batch, inp.top_k, inp.row_idx_type)
        torch.cuda.synchronize()
    finally:
        pgg.pgg_debug_force_variant(-1)
    assert pgg.status(ws) == 0, pgg.STATUS.get(pgg.status(ws))
    return out


def check(inp, out, what=""):
    ref = oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                    inp.top_k, inp.row_idx_type)
    err = np.abs(out.double().cpu().numpy() - ref).max()
    assert err <= TOL * np.abs(ref).max(), f"{what}: max|diff| {err:.3e}"


def plan_variant(inp):
    M, N = inp.grad_y.shape
    G, K, _ = inp.weight.shape
    return pgg.pgg_dx_plan(M, N, K, G, M, inp.batch, inp.top_k, inp.row_idx_type,
                           pgg.dtype_code(inp.grad_y.dtype))["variant"]


def _shifted(t, elems):
    buf = torch.empty(t.numel() + elems, dtype=t.dtype, device=t.device)
    v = buf[elems:].view(t.shape)
    v.copy_(t)
    return v


# aligned rows: forced variant 5 against variant 0, bit for bit
ALIGNED = {
    "ragged_k_n": dict(batch=300, top_k=4, G=7, K=400, N=328, routing="zipf", zipf_zero=2),
    "many_tiles": dict(batch=2048, top_k=8, G=12, K=1024, N=512),
    "tail_k178_n280": dict(batch=10, K=178, N=280, top_k=3, G=4),
    "k_is_1": dict(batch=128, K=1, N=256, top_k=3, G=4),
    "top1": dict(batch=700, K=256, N=192, top_k=1, G=5),
    "duplicate_experts": dict(batch=200, top_k=4, G=3, K=384, N=128, routing="replacement"),
}


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("case", sorted(ALIGNED))
def test_gathered_operands_equal_the_tma_kernel_bitwise(case, dtype):
    inp = make_case(dtype=dtype, seed=81, device="cuda", **ALIGNED[case])
    tma = run(inp, 0)
    gat = run(inp, GATHER)
    assert torch.equal(tma.view(torch.int32), gat.view(torch.int32)), case
    check(inp, gat, case)


# rows of N * 2 bytes, N even but not a multiple of 8: the automatic plan
@pytest.mark.parametrize("n", [2, 6, 286, 1022, 1030, 2046])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("row_idx_type", [0, 1])
def test_unaligned_rows_on_the_tensor_cores(n, dtype, row_idx_type):
    inp = make_case(batch=400, top_k=4, G=9, K=300, N=n, dtype=dtype, routing="zipf",
                    zipf_zero=2, row_idx_type=row_idx_type, seed=82, device="cuda")
    assert plan_variant(inp) == GATHER
    out = run(inp)
    check(inp, out, f"N={n}")
    again = run(inp)
    assert torch.equal(out.view(torch.int32), again.view(torch.int32))


def test_index_forms_agree_bitwise():
    inp0 = make_case(batch=1000, top_k=6, G=12, K=640, N=1022, dtype="bf16", seed=83,
                     device="cuda")
    a = run(inp0)
    b = run(with_row_idx_type(inp0, 1))
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_odd_rows_and_fp32_keep_the_fp32_pipes():
    for n, dtype in ((1031, "bf16"), (1, "fp16"), (1030, "fp32")):
        inp = make_case(batch=64, top_k=2, G=4, K=128, N=n, dtype=dtype, seed=84, device="cuda")
        assert plan_variant(inp) == 3, (n, dtype)
        check(inp, run(inp), f"{dtype} N={n}")


@pytest.mark.parametrize("shift_y,shift_w", [(2, 0), (0, 2), (6, 4)])
def test_four_byte_aligned_pointers_take_the_gather_warps(shift_y, shift_w):
    # gradY / weight 4-byte but not 16-byte aligned: the same kernel and the
    # same bits as forced variant 5 on aligned copies of the same values
    inp = make_case(batch=300, top_k=4, G=6, K=256, N=128, dtype="bf16", seed=85, device="cuda")
    want = run(inp, GATHER)
    got = run(inp, grad_y=_shifted(inp.grad_y, shift_y), weight=_shifted(inp.weight, shift_w))
    assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    check(inp, got, "shifted")


def test_large_unaligned_problem_sampled():
    # many row blocks and k blocks: 16 experts, K = 2048, N = 1022
    inp = make_case(batch=4096, top_k=8, G=16, K=2048, N=1022, dtype="bf16", seed=86,
                    device="cuda")
    out = run(inp)
    toks = np.sort(np.random.default_rng(4).choice(inp.batch, 512, replace=False))
    ref = oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                    inp.top_k, inp.row_idx_type, tokens=toks)
    err = np.abs(out.double().cpu().numpy()[toks] - ref).max()
    assert err <= TOL * np.abs(ref).max()


def test_bounded_wait_reports_timeout_and_recovers():
    inp = make_case(batch=256, top_k=4, G=8, K=256, N=126, dtype="bf16", seed=87, device="cuda")
    assert plan_variant(inp) == GATHER
    pgg.pgg_debug_set_wait_limit_ns(20_000_000)  # 20 ms
    pgg.pgg_debug_set_ticket_bias(1000)          # no ticket ever reaches rank + 1000
    try:
        _, ws = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                       inp.top_k, inp.row_idx_type)
        torch.cuda.synchronize()
        assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_TIMEOUT"
    finally:
        pgg.pgg_debug_set_ticket_bias(0)
        pgg.pgg_debug_set_wait_limit_ns(0)
    check(inp, run(inp), "after timeout")
