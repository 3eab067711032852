"""GPU parity of the weight gradient against the fp64 oracle, through the C ABI.

Tolerance, derived from the arithmetic: the kernels accumulate in fp32, so an
fp32 output must satisfy max |GPU - oracle| <= 1e-4 * max |oracle| (as d_x); a
16-bit output is that fp32 sum rounded to nearest even once more, which adds
at most half a unit in the last place: per element |GPU - oracle| <=
2^-8 * |oracle| (bf16; 2^-11 for fp16) + 1e-4 * max |oracle|.
"""

import numpy as np
import pytest
import torch

import oracle
import permute_grouped_gemm_gb300 as pgg
import sampling
from workloads import WORKLOADS, make_case, make_inputs
from workloads.moe import forward_input, with_row_idx_type

pytestmark = pytest.mark.gpu

TOL = 1e-4
ROUND = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11, torch.float32: 0.0}


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


def run(inp, x, **kw):
    out, ws = pgg.dw(x, inp.grad_y, inp.expanded_row_idx, inp.group_list, inp.batch,
                     inp.top_k, inp.row_idx_type, **kw)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0, pgg.STATUS.get(pgg.status(ws))
    return out


def ref_of(inp, x, sel=None):
    return oracle.dw(x, inp.grad_y, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k,
                     inp.row_idx_type, sel=sel)


def assert_close(got_t, ref, what=""):
    got = got_t.double().cpu().numpy()
    scale = np.abs(ref).max()
    bound = ROUND[got_t.dtype] * np.abs(ref) + TOL * scale
    err = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"{what}: |diff| {err[worst]:.3e} > bound {bound[worst]:.3e} "
                                  f"at {worst} (ref {ref[worst]:.4e})")


def plan_variant(inp, x):
    M, N = inp.grad_y.shape
    K = x.shape[1]
    G = inp.group_list.shape[0]
    return pgg.pgg_dw_plan(M, N, K, G, M, inp.batch, inp.top_k, inp.row_idx_type,
                           pgg.dtype_code(x.dtype))["variant"]


# The page's white-box shapes (section 4.2.1) plus multi-stage / ragged cases.
CASES = {
    "one_token_one_expert": dict(batch=1, K=128, N=256, top_k=1, G=1),
    "one_token_multi_expert": dict(batch=1, K=128, N=256, top_k=3, G=3),
    "multi_token_one_expert": dict(batch=128, K=128, N=256, top_k=1, G=1),
    "multi_token_multi_expert": dict(batch=128, K=128, N=256, top_k=3, G=10),
    "empty_expert": dict(batch=10, K=128, N=256, top_k=2, G=4, empty=(1,)),
    "tail_k178_n286": dict(batch=10, K=178, N=286, top_k=3, G=4),
    "n_is_1": dict(batch=128, K=128, N=1, top_k=3, G=4),
    "k_is_1": dict(batch=128, K=1, N=256, top_k=3, G=4),
    "ragged_tc": dict(batch=700, K=184, N=328, top_k=3, G=5),
}


@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_cases(case, dtype, out_f32):
    inp = make_case(dtype=dtype, seed=21, device="cuda", **CASES[case])
    x = forward_input(inp)
    out = run(inp, x, out_dtype=torch.float32 if out_f32 else None)
    assert_close(out, ref_of(inp, x), case)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_tensor_and_fp32_pipe_kernels_agree_with_the_oracle(dtype):
    # rows of several stages per expert, a partial last stage, ragged k and n
    inp = make_case(batch=900, top_k=4, G=7, K=312, N=520, dtype=dtype, routing="zipf",
                    zipf_zero=2, seed=22, device="cuda")
    x = forward_input(inp)
    assert plan_variant(inp, x) == 0
    ref = ref_of(inp, x)
    tc = run(inp, x, out_dtype=torch.float32)
    assert_close(tc, ref, "tensor cores")
    try:
        pgg.pgg_debug_force_variant(3)
        simt = run(inp, x, out_dtype=torch.float32)
    finally:
        pgg.pgg_debug_force_variant(-1)
    assert_close(simt, ref, "FP32 pipes")
    assert (inp.group_list == 0).sum() == 2
    for g in torch.nonzero(inp.group_list == 0).flatten().tolist():
        assert torch.count_nonzero(tc[g]) == 0 and torch.count_nonzero(simt[g]) == 0


@pytest.mark.parametrize("force_simt", [False, True])
def test_bitwise_repeatable_and_index_form_independent(force_simt):
    inp = make_case(batch=1500, top_k=6, G=12, K=256, N=512, dtype="bf16", seed=23,
                    device="cuda")
    x = forward_input(inp)
    try:
        if force_simt:
            pgg.pgg_debug_force_variant(3)
        first = run(inp, x, out_dtype=torch.float32)
        for _ in range(3):
            assert torch.equal(run(inp, x, out_dtype=torch.float32).view(torch.int32),
                               first.view(torch.int32))
        other = run(with_row_idx_type(inp, 1), x, out_dtype=torch.float32)
        assert torch.equal(other.view(torch.int32), first.view(torch.int32))
    finally:
        pgg.pgg_debug_force_variant(-1)
    assert_close(first, ref_of(inp, x))


def test_expanded_x_input_gives_the_same_bits():
    # a caller that kept expanded_x [M, K] passes it as x with topK = 1 and the
    # identity index: same rows, same order of additions
    inp = make_case(batch=400, top_k=4, G=6, K=192, N=256, dtype="fp16", seed=24, device="cuda")
    x = forward_input(inp)
    gathered = run(inp, x)
    pos = inp.gather.to("cuda")
    ex = x[pos // inp.top_k].contiguous()
    M = ex.shape[0]
    ident = torch.arange(M, dtype=torch.int64, device="cuda")
    out, ws = pgg.dw(ex, inp.grad_y, ident, inp.group_list, M, 1, 0)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    assert torch.equal(out.view(torch.int16), gathered.view(torch.int16))


def _shifted(t, elems):
    buf = torch.empty(t.numel() + elems, dtype=t.dtype, device=t.device)
    v = buf[elems:].view(t.shape)
    v.copy_(t)
    return v


def test_misaligned_pointers_take_the_fp32_pipes():
    # x 2-byte aligned: the FP32-pipe kernel, whose result does not depend on
    # the addresses; an output that is 4-byte but not 16-byte aligned: the
    # tensor cores with 4-byte stores, bitwise equal to the aligned run
    inp = make_case(batch=300, top_k=4, G=6, K=256, N=256, dtype="bf16", seed=25, device="cuda")
    x = forward_input(inp)
    tc = run(inp, x, out_dtype=torch.float32)
    try:
        pgg.pgg_debug_force_variant(3)
        simt = run(inp, x, out_dtype=torch.float32)
    finally:
        pgg.pgg_debug_force_variant(-1)
    out, ws = pgg.dw(_shifted(x, 1), _shifted(inp.grad_y, 3), inp.expanded_row_idx,
                     inp.group_list, inp.batch, inp.top_k, 0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    assert torch.equal(out.view(torch.int32), simt.view(torch.int32))
    obuf = torch.empty(6 * 256 * 256 + 1, dtype=torch.float32, device="cuda")
    o = obuf[1:].view(6, 256, 256)
    _, ws = pgg.dw(x, inp.grad_y, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k, 0,
                   out_dtype=torch.float32, out=o)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    assert torch.equal(o.view(torch.int32), tc.view(torch.int32))


def test_device_detected_errors_zero_the_output():
    base = make_case(batch=64, top_k=2, G=4, K=128, N=64, dtype="bf16", seed=26, device="cuda")
    x = forward_input(base)
    for variant in (-1, 3):
        idx = base.expanded_row_idx.clone()
        idx[5] = idx[6]
        out = torch.full((4, 128, 64), 7.0, dtype=torch.bfloat16, device="cuda")
        try:
            pgg.pgg_debug_force_variant(variant)
            _, ws = pgg.dw(x, base.grad_y, idx, base.group_list, 64, 2, 0, out=out)
            torch.cuda.synchronize()
        finally:
            pgg.pgg_debug_force_variant(-1)
        assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_NOT_PERM"
        assert torch.count_nonzero(out) == 0
    assert_close(run(base, x), ref_of(base, x), "after errors")


def test_gpu_results_satisfy_the_adjoint_identity():
    # sum(dW * W) == sum(d_x * x), both from the GPU (fp32 outputs)
    inp = make_case(batch=512, top_k=4, G=8, K=256, N=192, dtype="bf16", seed=27, device="cuda")
    x = forward_input(inp)
    dwt = run(inp, x, out_dtype=torch.float32).double()
    dx, _ = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                   inp.top_k, 0)
    lhs = float((dwt * inp.weight.double()).sum())
    rhs = float((dx.double() * x.double()).sum())
    assert abs(lhs - rhs) <= 1e-4 * (abs(lhs) + abs(rhs))


@pytest.mark.parametrize("name", ["uniform-bf16", "skewed-fp16", "large-bf16", "skinny-bf16",
                                  "unaligned-bf16"])
def test_workload_full_size(name):
    # every (expert, k) row of d_weight against the oracle; large-bf16 and
    # skinny-bf16 (7.5 GB of output) on a seeded 1/16 of the rows
    w = WORKLOADS[name]
    inp = make_inputs(w, device="cuda")
    x = forward_input(inp)
    out = run(inp, x)
    flat = out.view(w.G * w.K, w.N)
    sel = sampling.units(name, w.G * w.K, seed=2, full=sampling.FULL - {"skinny-bf16"})
    pieces = sampling.chunks(w.G * w.K if sel is None else sel, max(1, (1 << 25) // w.N))
    for part in pieces:
        ref = ref_of(inp, x, sel=(part // w.K, part % w.K))
        assert_close(flat[torch.as_tensor(part, device="cuda")], ref, name)
    again = run(inp, x)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def _random_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        top_k = int(rng.integers(1, 7))
        cases.append(dict(batch=int(rng.integers(1, 600)), top_k=top_k,
                          G=int(rng.integers(top_k, 17)), K=int(rng.integers(1, 400)),
                          N=int(rng.integers(1, 400)),
                          dtype=str(rng.choice(["bf16", "fp16", "fp32"])),
                          row_idx_type=int(rng.integers(0, 2)), seed=300 + i,
                          out_f32=bool(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("case", _random_cases(16, 4343),
                         ids=lambda c: "b{batch}k{top_k}g{G}K{K}N{N}{dtype}".format(**c))
def test_random_shapes(case):
    # random sizes, dtypes and index forms: tensor-core and FP32-pipe plans alike
    c = dict(case)
    out_f32 = c.pop("out_f32")
    inp = make_case(device="cuda", **c)
    x = forward_input(inp)
    got = run(inp, x, out_dtype=torch.float32 if out_f32 else None)
    assert_close(got, ref_of(inp, x), what=str(case))


# ---------------------------------------------------------------- rows the TMA cannot stream

def _plan(inp):
    M, N = inp.grad_y.shape
    G, K, _ = inp.weight.shape
    return pgg.pgg_dw_plan(M, N, K, G, M, inp.batch, inp.top_k, inp.row_idx_type,
                           pgg.dtype_code(inp.grad_y.dtype))["variant"]


@pytest.mark.parametrize("n", [2, 6, 286, 1022])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("out_f32", [False, True])
def test_unaligned_dy_rows_on_the_tensor_cores(n, dtype, out_f32):
    # d_y and d_weight rows of N * 2 bytes (N even, not a multiple of 8): the
    # gather warps copy the d_y panels 4 bytes at a time (plan variant 5); the
    # empty experts of the Zipf routing get zeros through 4-byte stores
    inp = make_case(batch=400, top_k=4, G=9, K=320, N=n, dtype=dtype, routing="zipf",
                    zipf_zero=2, seed=27, device="cuda")
    assert _plan(inp) == 5
    x = forward_input(inp)
    out = run(inp, x, out_dtype=torch.float32 if out_f32 else None)
    assert_close(out, ref_of(inp, x), f"N={n}")
    again = run(inp, x, out_dtype=torch.float32 if out_f32 else None)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("out_f32", [False, True])
def test_four_byte_aligned_dy_and_output_equal_the_tma_path_bitwise(out_f32):
    inp = make_case(batch=300, top_k=4, G=6, K=256, N=320, dtype="bf16", seed=28,
                    routing="zipf", zipf_zero=1, device="cuda")
    x = forward_input(inp)
    od = torch.float32 if out_f32 else torch.bfloat16
    want = run(inp, x, out_dtype=od)
    G, K, N = want.shape
    obuf = torch.empty(G * K * N + 2, dtype=od, device="cuda")
    o = obuf[(1 if out_f32 else 2):][:G * K * N].view(G, K, N)
    got, ws = pgg.dw(x, _shifted(inp.grad_y, 2), inp.expanded_row_idx, inp.group_list,
                     inp.batch, inp.top_k, inp.row_idx_type, out_dtype=od, out=o)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("n", [1024, 1022])
def test_bounded_wait_reports_timeout_and_recovers(n):
    # every epilogue warp withholds its first release of accumulator 0 (test
    # hook), so the MMA thread's wait for it runs out at each CTA pair's third
    # tile (16 experts x 4 k blocks x 4 n blocks = 256 tiles over 76 pairs):
    # every role of both CTAs gives up, the call reports PGG_ERR_TIMEOUT, and
    # the next call on the same context is correct. N = 1022 takes the d_y
    # panels copied by the gather warps.
    inp = make_case(batch=2048, top_k=8, G=16, K=1024, N=n, dtype="bf16", seed=60,
                    device="cuda")
    x = forward_input(inp)
    assert plan_variant(inp, x) == (0 if n == 1024 else 5)
    pgg.pgg_debug_set_wait_limit_ns(20_000_000)  # 20 ms
    pgg.pgg_debug_set_hold_release(1)
    try:
        _, ws = pgg.dw(x, inp.grad_y, inp.expanded_row_idx, inp.group_list, inp.batch,
                       inp.top_k, inp.row_idx_type)
        torch.cuda.synchronize()
        assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_TIMEOUT"
    finally:
        pgg.pgg_debug_set_hold_release(0)
        pgg.pgg_debug_set_wait_limit_ns(0)
    rng = np.random.default_rng(60)
    g = rng.integers(0, 16, 256)
    k = rng.integers(0, 1024, 256)
    out = run(inp, x)
    got = out[torch.from_numpy(g).cuda(), torch.from_numpy(k).cuda()]
    assert_close(got, ref_of(inp, x, sel=(g, k)), "after timeout")
