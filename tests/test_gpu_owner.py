"""GPU parity of the slab-owner variant of the fused d_x backward (plan variant 4).

The owner kernel adds each token's rows in the same order as the ticketed
kernel (increasing expanded index), so the two agree bit for bit; both match
the fp64 oracle within 1e-4 * max |d_x_ref|. When some expert's rows are not in
increasing original position the ticketed kernel launched after it does the
work.
"""

import numpy as np
import pytest
import torch

import oracle
import permute_grouped_gemm_gb300 as pgg
from workloads import WORKLOADS, make_case, make_inputs
from workloads.moe import Inputs, with_row_idx_type

pytestmark = pytest.mark.gpu

TOL = 1e-4


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


def run(inp, variant=-1):
    try:
        pgg.pgg_debug_force_variant(variant)
        out, ws = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                         inp.top_k, inp.row_idx_type)
        torch.cuda.synchronize()
    finally:
        pgg.pgg_debug_force_variant(-1)
    assert pgg.status(ws) == 0, pgg.STATUS.get(pgg.status(ws))
    return out


def check(inp, out, tokens=None, what=""):
    ref = oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                    inp.top_k, inp.row_idx_type, tokens=tokens)
    got = out.double().cpu().numpy()
    if tokens is not None:
        got = got[np.asarray(tokens)]
    err = np.abs(got - ref).max()
    assert err <= TOL * np.abs(ref).max(), f"{what}: {err:.3e}"


def test_uniform_workload_plans_the_owner_variant():
    w = WORKLOADS["uniform-bf16"]
    p = pgg.pgg_dx_plan(w.M, w.N, w.K, w.G, w.M, w.batch, w.top_k, 0, pgg.PGG_BF16)
    assert p["variant"] == 4 and p["rows_per_block"] == 224 and p["cta_pair"] == 1


CASES = {
    "uniform_small": dict(batch=1024, top_k=8, G=16, K=512, N=256),
    "ragged_k_n_batch": dict(batch=700, top_k=4, G=7, K=400, N=328),
    "empty_experts": dict(batch=600, top_k=3, G=9, K=256, N=192, routing="zipf", zipf_zero=3),
    "same_expert_twice": dict(batch=500, top_k=4, G=3, K=384, N=128, routing="replacement"),
    "top1": dict(batch=900, top_k=1, G=4, K=256, N=256),
    "k_is_1": dict(batch=300, top_k=3, G=4, K=1, N=256),
    "many_rows_per_expert": dict(batch=2000, top_k=2, G=2, K=256, N=128),
    # 32-token slabs of 256 rows over two experts: chunks of 128 rows and a tail
    "chunk_split": dict(batch=1000, top_k=8, G=2, K=512, N=192, routing="replacement"),
    # many experts: 256-token slabs with a few rows of each expert
    "wide_slabs": dict(batch=800, top_k=2, G=40, K=300, N=256),
    # one two-panel stage whose second panel is past N (read as zero)
    "n_is_64": dict(batch=600, top_k=4, G=4, K=256, N=64),
    # one 64-n stage whose box reaches past the 16 values of a row
    "n_is_16": dict(batch=600, top_k=4, G=4, K=256, N=16),
}


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_owner_matches_oracle_and_ticketed_kernel_bitwise(case, dtype):
    inp = make_case(dtype=dtype, seed=51, device="cuda", **CASES[case])
    owner = run(inp, 4)
    check(inp, owner, what=case)
    ticketed = run(inp, 0)
    assert torch.equal(owner.view(torch.int32), ticketed.view(torch.int32)), case


def test_index_forms_and_repeat_bitwise():
    inp = make_case(batch=1024, top_k=8, G=16, K=512, N=256, dtype="bf16", seed=52,
                    device="cuda")
    a = run(inp, 4)
    for _ in range(3):
        assert torch.equal(run(inp, 4).view(torch.int32), a.view(torch.int32))
    b = run(with_row_idx_type(inp, 1), 4)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def _unsorted(inp):
    """The same problem with two rows of expert 0 swapped in the expanded order
    (still a valid routing; the expert's rows no longer in increasing position)."""
    gather = inp.gather.clone()
    i, j = 0, 1  # rows 0 and 1 both belong to expert 0 (its count is large here)
    assert int(inp.group_list[0]) >= 2
    gather[i], gather[j] = gather[j].clone(), gather[i].clone()
    dy = inp.grad_y.clone()
    dy[[i, j]] = dy[[j, i]]
    idx = gather if inp.row_idx_type == 0 else torch.argsort(gather)
    return Inputs(inp.workload, dy, inp.weight, idx.to(dy.device), inp.group_list, inp.experts,
                  gather)


@pytest.mark.parametrize("row_idx_type", [0, 1])
def test_unsorted_rows_fall_back_to_the_ticketed_kernel(row_idx_type):
    base = make_case(batch=1024, top_k=8, G=16, K=512, N=256, dtype="bf16", seed=53,
                     row_idx_type=row_idx_type, device="cuda")
    inp = _unsorted(base)
    out = run(inp, 4)
    check(inp, out, what="unsorted")
    assert torch.equal(out.view(torch.int32), run(inp, 0).view(torch.int32))


def test_device_errors_zero_the_output_in_owner_mode():
    base = make_case(batch=512, top_k=8, G=16, K=256, N=128, dtype="bf16", seed=54, device="cuda")
    idx = base.expanded_row_idx.clone()
    idx[5] = idx[6]
    out = torch.full((512, 256), 7.0, device="cuda")
    try:
        pgg.pgg_debug_force_variant(4)
        _, ws = pgg.dx(base.grad_y, base.weight, idx, base.group_list, 512, 8, 0, out=out)
        torch.cuda.synchronize()
    finally:
        pgg.pgg_debug_force_variant(-1)
    assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_NOT_PERM"
    assert torch.count_nonzero(out) == 0


def test_bounded_wait_reports_timeout_and_recovers():
    # the epilogue withholds its first release of accumulator 0 (test hook), so
    # the MMA thread of that pipeline waits for it until the limit: every role
    # of every CTA gives up, the call reports PGG_ERR_TIMEOUT, and the next call
    # on the same context is correct
    inp = make_case(batch=2048, top_k=8, G=16, K=512, N=512, dtype="bf16", seed=58,
                    device="cuda")
    pgg.pgg_debug_set_wait_limit_ns(20_000_000)  # 20 ms
    pgg.pgg_debug_set_hold_release(1)
    try:
        pgg.pgg_debug_force_variant(4)
        _, ws = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                       inp.top_k, inp.row_idx_type)
        torch.cuda.synchronize()
        assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_TIMEOUT"
    finally:
        pgg.pgg_debug_force_variant(-1)
        pgg.pgg_debug_set_hold_release(0)
        pgg.pgg_debug_set_wait_limit_ns(0)
    check(inp, run(inp, 4), what="after timeout")


def test_uniform_workload_full_size():
    w = WORKLOADS["uniform-bf16"]
    inp = make_inputs(w, device="cuda")
    out = run(inp)
    check(inp, out, what=w.name)  # every token
    assert torch.equal(out.view(torch.int32), run(inp, 0).view(torch.int32))


def test_large_few_expert_problem_plans_and_matches_the_owner_kernel():
    # 16384 tokens, topK 4, 8 experts: 224-token slabs (74) x 4 k ranges = 296 units,
    # some experts' slab rows above 128 (chunk splits), N a multiple of 64 (two-panel stages)
    inp = make_case(batch=16384, top_k=4, G=8, K=1024, N=512, dtype="bf16", seed=55,
                    device="cuda")
    M = inp.grad_y.shape[0]
    p = pgg.pgg_dx_plan(M, 512, 1024, 8, M, 16384, 4, 0, pgg.PGG_BF16)
    assert p["variant"] == 4 and p["rows_per_block"] == 224
    out = run(inp)
    toks = np.sort(np.random.default_rng(9).choice(inp.batch, 64, replace=False))
    check(inp, out, tokens=toks, what="large few-expert")
    assert torch.equal(out.view(torch.int32), run(inp, 0).view(torch.int32))


def _random_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        top_k = int(rng.integers(1, 9))
        G = int(rng.integers(top_k, 25))
        cases.append(dict(batch=int(rng.integers(1, 3000)), top_k=top_k, G=G,
                          K=int(rng.integers(1, 1000)),
                          N=int(rng.choice([16, 48, 64, 96, 128, 200, 256, 320])),
                          dtype=str(rng.choice(["bf16", "fp16"])),
                          row_idx_type=int(rng.integers(0, 2)), seed=100 + i))
    return cases


@pytest.mark.parametrize("case", _random_cases(24, 2026),
                         ids=lambda c: "b{batch}k{top_k}g{G}K{K}N{N}".format(**c))
def test_random_shapes_owner_equals_ticketed(case):
    # random sizes cross every slab size, partial last slab, chunk split, K tail,
    # N tail and both stage kinds; the owner kernel must match the ticketed one
    # bit for bit, and both the oracle
    inp = make_case(device="cuda", **case)
    owner = run(inp, 4)
    ticketed = run(inp, 0)
    assert torch.equal(owner.view(torch.int32), ticketed.view(torch.int32))
    toks = None
    if inp.batch > 256:
        toks = np.sort(np.random.default_rng(case["seed"]).choice(inp.batch, 64, replace=False))
    check(inp, owner, tokens=toks, what=str(case))
