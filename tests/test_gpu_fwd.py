"""GPU parity of the forward grouped matmul against the fp64 oracle, through the C ABI.

Tolerance, derived from the arithmetic as for the weight gradient: fp32
accumulation gives max |GPU - oracle| <= 1e-4 * max |oracle| for an fp32
output; a 16-bit output adds one rounding to nearest even, per element
2^-8 * |oracle| (bf16; 2^-11 fp16) on top.
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
    y, ws = pgg.fwd(x, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k,
                    inp.row_idx_type, **kw)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0, pgg.STATUS.get(pgg.status(ws))
    return y


def ref_of(inp, x, rows=None):
    return oracle.fwd(x, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k,
                      inp.row_idx_type, rows=rows)


def assert_close(got_t, ref, what=""):
    got = got_t.double().cpu().numpy()
    scale = np.abs(ref).max()
    bound = ROUND[got_t.dtype] * np.abs(ref) + TOL * scale
    err = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), (f"{what}: |diff| {err[worst]:.3e} > bound {bound[worst]:.3e} "
                                  f"at {worst} (ref {ref[worst]:.4e})")


def variant(inp, x):
    G, K, N = inp.weight.shape
    M = inp.expanded_row_idx.shape[0]
    return pgg.pgg_fwd_plan(M, N, K, G, M, inp.batch, inp.top_k, inp.row_idx_type,
                            pgg.dtype_code(x.dtype))["variant"]


CASES = {
    "one_token_one_expert": dict(batch=1, K=128, N=256, top_k=1, G=1),
    "one_token_multi_expert": dict(batch=1, K=128, N=256, top_k=3, G=3),
    "multi_token_one_expert": dict(batch=128, K=128, N=256, top_k=1, G=1),
    "multi_token_multi_expert": dict(batch=128, K=128, N=256, top_k=3, G=10),
    "empty_expert": dict(batch=10, K=128, N=256, top_k=2, G=4, empty=(1,)),
    "tail_k178_n286": dict(batch=10, K=178, N=286, top_k=3, G=4),
    "n_is_1": dict(batch=128, K=128, N=1, top_k=3, G=4),
    "k_is_1": dict(batch=128, K=1, N=256, top_k=3, G=4),
    "ragged_tc": dict(batch=700, K=200, N=328, top_k=3, G=5),
}


@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_cases(case, dtype, out_f32):
    inp = make_case(dtype=dtype, seed=31, device="cuda", **CASES[case])
    x = forward_input(inp)
    y = run(inp, x, out_dtype=torch.float32 if out_f32 else None)
    assert_close(y, ref_of(inp, x), case)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_tensor_and_fp32_pipe_kernels_agree_with_the_oracle(dtype):
    # experts of several 256-row blocks with a ragged last block (rows written
    # one by one where a 32-row box would cross into the next expert), k and n
    # with ragged tails, empty experts
    inp = make_case(batch=900, top_k=4, G=7, K=328, N=520, dtype=dtype, routing="zipf",
                    zipf_zero=2, seed=32, device="cuda")
    x = forward_input(inp)
    assert variant(inp, x) == 0
    assert (inp.group_list > 256).any()
    ref = ref_of(inp, x)
    tc = run(inp, x, out_dtype=torch.float32)
    assert_close(tc, ref, "tensor cores")
    try:
        pgg.pgg_debug_force_variant(3)
        simt = run(inp, x, out_dtype=torch.float32)
    finally:
        pgg.pgg_debug_force_variant(-1)
    assert_close(simt, ref, "FP32 pipes")


def test_output_rows_are_written_exactly_once_per_row():
    # guard bands around y: nothing outside [M, N] is touched
    inp = make_case(batch=333, top_k=3, G=5, K=256, N=384, dtype="bf16", seed=33, device="cuda")
    x = forward_input(inp)
    M, N = inp.grad_y.shape[0], 384
    buf = torch.full((M * N + 2 * 4096,), -7.0, dtype=torch.bfloat16, device="cuda")
    y = buf[4096:4096 + M * N].view(M, N)
    run(inp, x, out=y)
    assert (buf[:4096] == -7.0).all() and (buf[4096 + M * N:] == -7.0).all()
    assert_close(y, ref_of(inp, x))


@pytest.mark.parametrize("force_simt", [False, True])
def test_bitwise_repeatable_and_index_form_independent(force_simt):
    inp = make_case(batch=1500, top_k=6, G=12, K=512, N=256, dtype="bf16", seed=34,
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


def _shifted(t, elems):
    buf = torch.empty(t.numel() + elems, dtype=t.dtype, device=t.device)
    v = buf[elems:].view(t.shape)
    v.copy_(t)
    return v


def test_misaligned_pointers_take_the_fp32_pipes():
    inp = make_case(batch=300, top_k=4, G=6, K=256, N=256, dtype="bf16", seed=35, device="cuda")
    x = forward_input(inp)
    try:
        pgg.pgg_debug_force_variant(3)
        simt = run(inp, x, out_dtype=torch.float32)
    finally:
        pgg.pgg_debug_force_variant(-1)
    y, ws = pgg.fwd(_shifted(x, 1), _shifted(inp.weight, 3), inp.expanded_row_idx,
                    inp.group_list, inp.batch, inp.top_k, 0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    assert torch.equal(y.view(torch.int32), simt.view(torch.int32))


def test_device_detected_errors_zero_the_output():
    base = make_case(batch=64, top_k=2, G=4, K=128, N=64, dtype="bf16", seed=36, device="cuda")
    x = forward_input(base)
    for v in (-1, 3):
        gl = base.group_list.clone()
        gl[0] += 1
        y = torch.full((128, 64), 7.0, dtype=torch.bfloat16, device="cuda")
        try:
            pgg.pgg_debug_force_variant(v)
            _, ws = pgg.fwd(x, base.weight, base.expanded_row_idx, gl, 64, 2, 0, out=y)
            torch.cuda.synchronize()
        finally:
            pgg.pgg_debug_force_variant(-1)
        assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_GROUPSUM"
        assert torch.count_nonzero(y) == 0
    assert_close(run(base, x), ref_of(base, x), "after errors")


def test_gpu_results_satisfy_the_adjoint_identity():
    # <d_y, y> == sum(d_x * x), y and d_x both from the GPU (fp32 outputs)
    inp = make_case(batch=512, top_k=4, G=8, K=256, N=192, dtype="bf16", seed=37, device="cuda")
    x = forward_input(inp)
    y = run(inp, x, out_dtype=torch.float32).double()
    dx, _ = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                   inp.top_k, 0)
    lhs = float((y * inp.grad_y.double()).sum())
    rhs = float((dx.double() * x.double()).sum())
    assert abs(lhs - rhs) <= 1e-4 * (abs(lhs) + abs(rhs))


@pytest.mark.parametrize("name", ["uniform-bf16", "skewed-fp16", "large-bf16", "skinny-bf16",
                                  "unaligned-bf16"])
def test_workload_full_size(name):
    # every row of y against the oracle (large-bf16: a seeded 1/16 of them)
    w = WORKLOADS[name]
    inp = make_inputs(w, device="cuda")
    x = forward_input(inp)
    y = run(inp, x)
    rows = sampling.units(name, w.M, seed=3)
    got = y if rows is None else y[torch.as_tensor(rows, device="cuda")]
    assert_close(got, ref_of(inp, x, rows=rows), name)
    again = run(inp, x)
    assert torch.equal(y.view(torch.int16), again.view(torch.int16))


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


@pytest.mark.parametrize("case", _random_cases(16, 4242),
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
    return pgg.pgg_fwd_plan(M, N, K, G, M, inp.batch, inp.top_k, inp.row_idx_type,
                            pgg.dtype_code(inp.grad_y.dtype))["variant"]


@pytest.mark.parametrize("n", [2, 6, 286, 1022])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("out_f32", [False, True])
def test_unaligned_weight_rows_on_the_tensor_cores(n, dtype, out_f32):
    # weight and y rows of N * 2 bytes (N even, not a multiple of 8): the gather
    # warps copy the weight panels 4 bytes at a time (plan variant 5)
    inp = make_case(batch=400, top_k=4, G=9, K=320, N=n, dtype=dtype, routing="zipf",
                    zipf_zero=2, seed=38, device="cuda")
    assert _plan(inp) == 5
    x = forward_input(inp)
    y = run(inp, x, out_dtype=torch.float32 if out_f32 else None)
    assert_close(y, ref_of(inp, x), f"N={n}")
    again = run(inp, x, out_dtype=torch.float32 if out_f32 else None)
    assert torch.equal(y.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("out_f32", [False, True])
def test_four_byte_aligned_weight_and_y_equal_the_tma_path_bitwise(out_f32):
    # weight / y 4-byte but not 16-byte aligned: the gathered weight panels and
    # the 4-byte stores give the bits of the TMA path
    inp = make_case(batch=300, top_k=4, G=6, K=256, N=320, dtype="bf16", seed=39, device="cuda")
    x = forward_input(inp)
    od = torch.float32 if out_f32 else torch.bfloat16
    want = run(inp, x, out_dtype=od)
    M, N = want.shape
    ybuf = torch.empty(M * N + 2, dtype=od, device="cuda")
    y = ybuf[(1 if out_f32 else 2):][:M * N].view(M, N)
    got, ws = pgg.fwd(x, _shifted(inp.weight, 2), inp.expanded_row_idx, inp.group_list,
                      inp.batch, inp.top_k, 0, out_dtype=od, out=y)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("n", [1024, 1022])
def test_bounded_wait_reports_timeout_and_recovers(n):
    # every epilogue warp withholds its first release of accumulator 0 (test
    # hook), so the MMA thread's wait for it runs out at each CTA pair's third
    # tile (256 tiles over 76 pairs): every role of both CTAs gives up, the call
    # reports PGG_ERR_TIMEOUT, and the next call on the same context is correct.
    # N = 1022 takes the weight panels copied by the gather warps.
    inp = make_case(batch=2048, top_k=8, G=16, K=512, N=n, dtype="bf16", seed=59,
                    device="cuda")
    x = forward_input(inp)
    assert variant(inp, x) == (0 if n == 1024 else 5)
    pgg.pgg_debug_set_wait_limit_ns(20_000_000)  # 20 ms
    pgg.pgg_debug_set_hold_release(1)
    try:
        _, ws = pgg.fwd(x, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                        inp.top_k, inp.row_idx_type)
        torch.cuda.synchronize()
        assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_TIMEOUT"
    finally:
        pgg.pgg_debug_set_hold_release(0)
        pgg.pgg_debug_set_wait_limit_ns(0)
    rows = np.sort(np.random.default_rng(59).choice(inp.grad_y.shape[0], 512, replace=False))
    y = run(inp, x)
    assert_close(y[torch.from_numpy(rows).cuda()], ref_of(inp, x, rows=rows), "after timeout")
