"""The entry point for callers that cannot allocate device memory.

Some callers have no allocator when they need d_x: a plugin inside a
framework that owns all device memory, a serving or real-time runtime that
reserved HBM at start-up and forbids cudaMalloc afterwards, plain C code with
no allocator handle. pgg_dx_execute_static_scratch takes the same inputs and
output as pgg_dx_execute but no workspace; the library's fixed device scratch
array stands in for it. These checks call it through the C ABI and compare its
output with that of the workspace-taking entry point and with the fp64 oracle,
on two calls in a row (the second call finds the first call's leftovers in the
shared array).
"""

import numpy as np
import pytest
import torch

import oracle
import permute_grouped_gemm_gb300 as pgg
from workloads import make_case

pytestmark = pytest.mark.gpu

TOL = 1e-4
SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from permute_grouped_gemm_gb300 import build as pbuild
    pbuild.build()
    oracle.build()
    pgg.load()


def oracle_dx(inp):
    return oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                     inp.top_k, inp.row_idx_type)


def call_static(inp, out, status):
    w = inp.workload
    return pgg.pgg_dx_execute_static_scratch(
        inp.grad_y.data_ptr(), inp.weight.data_ptr(), inp.expanded_row_idx.data_ptr(),
        inp.group_list.data_ptr(), w.M, w.N, w.K, w.G, w.M, w.batch, w.top_k, w.row_idx_type,
        pgg.dtype_code(inp.grad_y.dtype), out.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,row_idx_type", [("bf16", 0), ("fp16", 1)])
def test_static_scratch_matches_workspace_entry_point(dtype, row_idx_type):
    inp = make_case(batch=1536, top_k=8, G=12, K=640, N=320, dtype=dtype,
                    row_idx_type=row_idx_type, seed=21, device="cuda")
    ref, ws = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list,
                     inp.batch, inp.top_k, inp.row_idx_type)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    ref = ref.double().cpu().numpy()
    exact = oracle_dx(inp)
    scale = np.abs(exact).max()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = torch.full((inp.batch, inp.workload.K), float("nan"), device="cuda")
        rc = call_static(inp, out, status)
        assert rc == 0, pgg.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.double().cpu().numpy()
        for want, what in ((ref, "workspace entry point"), (exact, "oracle")):
            err = np.abs(got - want).max()
            assert err <= TOL * scale, f"{what}: max|diff| {err:.3e} > {TOL} * {scale:.3e}"


def test_static_scratch_with_the_owner_plan():
    # few experts per token: the automatic plan is the owner kernel, whose workspace also
    # holds the slab bounds; both entry points run the same plan, so they agree bit for bit
    inp = make_case(batch=2048, top_k=8, G=16, K=4096, N=128, dtype="bf16", seed=22,
                    device="cuda")
    w = inp.workload
    assert pgg.pgg_dx_plan(w.M, w.N, w.K, w.G, w.M, w.batch, w.top_k, 0,
                           pgg.PGG_BF16)["variant"] == 4
    ref, ws = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list,
                     inp.batch, inp.top_k, inp.row_idx_type)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    toks = np.sort(np.random.default_rng(23).choice(inp.batch, 256, replace=False))
    exact = oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                      inp.top_k, inp.row_idx_type, tokens=toks)
    scale = np.abs(exact).max()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = torch.full((inp.batch, w.K), float("nan"), device="cuda")
        rc = call_static(inp, out, status)
        assert rc == 0, pgg.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
        err = np.abs(out.double().cpu().numpy()[toks] - exact).max()
        assert err <= TOL * scale, f"oracle: max|diff| {err:.3e} > {TOL} * {scale:.3e}"


def test_sizes_beyond_the_scratch_are_rejected():
    # batch 1M tokens x topK 8 at K = 7168 needs far more than 8 MiB of index
    # tables; the call is refused on the host before any pointer is used
    M, K, N, G, batch = 8 << 20, 7168, 2048, 64, 1 << 20
    need = pgg.pgg_dx_workspace_size(M, N, K, G, M, batch, 8, 0, pgg.PGG_BF16)
    assert need > SCRATCH_BYTES
    fake = 1 << 20
    rc = pgg.pgg_dx_execute_static_scratch(fake, fake, fake, fake, M, N, K, G, M, batch, 8, 0,
                                           pgg.PGG_BF16, fake, 0, None)
    assert pgg.STATUS[rc] == "PGG_ERR_WORKSPACE"
