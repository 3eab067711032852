"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerance for every dtype: max |GPU - oracle| <= 1e-4 * max |oracle| over the
compared rows. The GPU result must also be bitwise identical from run to run.
"""

import numpy as np
import pytest
import torch

import oracle
import permute_grouped_gemm_gb300 as pgg
import sampling
from workloads import WORKLOADS, make_case, make_inputs
from workloads.moe import with_row_idx_type

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
    pgg.pgg_debug_set_band_k_blocks(0)
    pgg.pgg_debug_set_ticket_bias(0)
    pgg.pgg_debug_set_wait_limit_ns(0)


def run(inp, **kw):
    out, ws = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list,
                     inp.batch, inp.top_k, inp.row_idx_type, **kw)
    torch.cuda.synchronize()
    return out, ws


def ref_rows(inp, tokens=None):
    return oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list,
                     inp.batch, inp.top_k, inp.row_idx_type, tokens=tokens)


def assert_close(got, ref, what=""):
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    assert err <= TOL * scale, f"{what}: max|diff| {err:.3e} > {TOL} * {scale:.3e}"


def check(inp, tokens=None, what=""):
    out, ws = run(inp)
    assert pgg.status(ws) == 0, pgg.STATUS.get(pgg.status(ws))
    got = out.double().cpu().numpy()
    if tokens is not None:
        got = got[np.asarray(tokens)]
    assert_close(got, ref_rows(inp, tokens), what)
    return out


# The page's white-box list (section 4.2.1). N = 1 and the tail case's
# N = 286 have rows whose byte length is not a multiple of 16 and run on the
# FP32-pipe kernel; "tail_k178_n280" keeps a ragged tail on the tensor cores.
WHITE_BOX = {
    "one_token_one_expert": dict(batch=1, K=128, N=256, top_k=1, G=1),
    "one_token_multi_expert": dict(batch=1, K=128, N=256, top_k=3, G=3),
    "multi_token_one_expert": dict(batch=128, K=128, N=256, top_k=1, G=1),
    "multi_token_multi_expert": dict(batch=128, K=128, N=256, top_k=3, G=10),
    "empty_expert": dict(batch=10, K=128, N=256, top_k=2, G=4, empty=(1,)),
    "tail_k178_n286": dict(batch=10, K=178, N=286, top_k=3, G=4),
    "tail_k178_n280": dict(batch=10, K=178, N=280, top_k=3, G=4),
    "m_is_1": dict(batch=1, K=128, N=256, top_k=1, G=1),
    "n_is_1": dict(batch=128, K=128, N=1, top_k=3, G=4),
    "k_is_1": dict(batch=128, K=1, N=256, top_k=3, G=4),
}


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("row_idx_type", [0, 1])
@pytest.mark.parametrize("case", sorted(WHITE_BOX))
def test_white_box(case, dtype, row_idx_type):
    inp = make_case(dtype=dtype, row_idx_type=row_idx_type, seed=3, device="cuda",
                    **WHITE_BOX[case])
    if case == "empty_expert":
        assert int(inp.group_list[1]) == 0
    check(inp, what=case)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_large_m_white_box(dtype):
    # "大 token 数": batch = 108 * 1024, topK = 2, G = 60, K = 128, N = 256
    inp = make_case(batch=108 * 1024, top_k=2, G=60, K=128, N=256, dtype=dtype, seed=4,
                    device="cuda")
    toks = np.random.default_rng(0).choice(inp.batch, 256, replace=False)
    check(inp, tokens=toks, what="large M")


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 5])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_multi_tile_ragged(dtype, variant):
    if dtype == "fp32" and variant in (2, 5):
        pytest.skip("variants 2 and 5 exist for 16-bit inputs only")
    # several k blocks with a ragged tail, a ragged reduction tail, groups of
    # 0 .. several hundred rows
    pgg.pgg_debug_force_variant(variant)
    try:
        inp = make_case(batch=300, top_k=4, G=7, K=400, N=328 if dtype != "fp32" else 332,
                        dtype=dtype, routing="zipf", zipf_zero=2, seed=5, device="cuda")
        assert (inp.group_list == 0).sum() == 2
        check(inp, what=f"variant {variant}")
    finally:
        pgg.pgg_debug_force_variant(-1)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_same_expert_twice_for_a_token(dtype):
    # degenerate routing: rows of one token inside one tile must still be
    # added in order (no deadlock, correct sum)
    for variant in ((0, 1, 2, 3, 5) if dtype != "fp32" else (0, 1, 3)):
        pgg.pgg_debug_force_variant(variant)
        try:
            inp = make_case(batch=200, top_k=4, G=3, K=384, N=128, dtype=dtype,
                            routing="replacement", seed=6, device="cuda")
            check(inp, what=f"replacement variant {variant}")
        finally:
            pgg.pgg_debug_force_variant(-1)


@pytest.mark.parametrize("n", [256, 250])
def test_bitwise_repeatable(n):
    inp = make_case(batch=2048, top_k=8, G=16, K=512, N=n, dtype="bf16", seed=7,
                    device="cuda")
    first, ws = run(inp)
    for _ in range(4):
        again, _ = run(inp, workspace=ws)
        assert torch.equal(again.view(torch.int32), first.view(torch.int32))


def test_tile_order_does_not_change_a_bit():
    inp = make_case(batch=1024, top_k=8, G=12, K=1024, N=256, dtype="bf16", seed=13,
                    device="cuda")
    base, ws = run(inp)
    try:
        for band in (1, 3, 5):
            pgg.pgg_debug_set_band_k_blocks(band)
            again, _ = run(inp, workspace=ws)
            assert torch.equal(again.view(torch.int32), base.view(torch.int32)), band
    finally:
        pgg.pgg_debug_set_band_k_blocks(0)
    assert_close(base.double().cpu().numpy(), ref_rows(inp))


def test_variants_agree():
    # CTA-pair tiles, single-CTA tiles and narrow tiles: same additions in the
    # same order per element; the tensor-core sums may differ only by rounding
    inp = make_case(batch=640, top_k=6, G=9, K=896, N=448, dtype="bf16", seed=14,
                    device="cuda")
    ref = ref_rows(inp)
    outs = []
    try:
        for variant in (0, 1, 2, 3, 5):
            pgg.pgg_debug_force_variant(variant)
            out, _ = run(inp)
            outs.append(out)
            assert_close(out.double().cpu().numpy(), ref, f"variant {variant}")
    finally:
        pgg.pgg_debug_force_variant(-1)
    # the gathered operands are those the tensor-memory-access unit loads
    assert torch.equal(outs[0].view(torch.int32), outs[4].view(torch.int32))


@pytest.mark.parametrize("n", [192, 190])
def test_gather_and_scatter_forms_agree_bitwise(n):
    inp0 = make_case(batch=500, top_k=6, G=12, K=256, N=n, dtype="fp16", seed=8,
                     device="cuda")
    inp1 = with_row_idx_type(inp0, 1)
    a, _ = run(inp0)
    b, _ = run(inp1)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


# The routing step ranks a token's rows with one lane per position when
# topK <= 32 (topK lanes per token, 32 // topK tokens per warp, idle lanes when
# topK does not divide 32) and with one thread per token above that.
@pytest.mark.parametrize("top_k", [5, 32, 40])
@pytest.mark.parametrize("row_idx_type", [0, 1])
def test_many_experts_per_token(top_k, row_idx_type):
    inp = make_case(batch=97, top_k=top_k, G=48, K=256, N=128, dtype="bf16", seed=17,
                    row_idx_type=row_idx_type, device="cuda")
    a = check(inp, what=f"topK {top_k}")
    b, _ = run(inp)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    try:  # the owner kernel adds the same rows in the same order
        pgg.pgg_debug_force_variant(4)
        c, ws = run(inp)
    finally:
        pgg.pgg_debug_force_variant(-1)
    assert pgg.status(ws) == 0
    assert torch.equal(a.view(torch.int32), c.view(torch.int32))
    # a position without an expanded row is still detected
    idx = inp.expanded_row_idx.clone()
    idx[3] = idx[4]
    out = torch.full((97, 256), 7.0, device="cuda")
    _, ws = pgg.dx(inp.grad_y, inp.weight, idx, inp.group_list, 97, top_k, row_idx_type, out=out)
    torch.cuda.synchronize()
    assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_NOT_PERM"
    assert torch.count_nonzero(out) == 0


@pytest.mark.parametrize("n", [64, 63])
def test_device_detected_errors_zero_the_output(n):
    base = make_case(batch=64, top_k=2, G=4, K=128, N=n, dtype="bf16", seed=9, device="cuda")
    cases = {}
    idx = base.expanded_row_idx.clone()
    idx[5] = base.batch * base.top_k  # out of range
    cases["PGG_ERR_INDEX"] = (idx, base.group_list)
    idx = base.expanded_row_idx.clone()
    idx[5] = idx[6]
    cases["PGG_ERR_NOT_PERM"] = (idx, base.group_list)
    gl = base.group_list.clone()
    gl[0] += 1
    cases["PGG_ERR_GROUPSUM"] = (base.expanded_row_idx, gl)
    gl = base.group_list.clone()
    gl[1] += gl[0] + 1
    gl[0] = -1
    cases["PGG_ERR_GROUPSUM_NEG"] = (base.expanded_row_idx, gl)
    for name, (idx, gl) in cases.items():
        out = torch.full((64, 128), 7.0, device="cuda")
        _, ws = pgg.dx(base.grad_y, base.weight, idx, gl, 64, 2, 0, out=out)
        torch.cuda.synchronize()
        assert pgg.STATUS[pgg.status(ws)] == name.replace("_NEG", ""), name
        assert torch.count_nonzero(out) == 0
    # the context is still usable
    check(base, what="after errors")


@pytest.mark.parametrize("n", [128, 127, 126])
def test_bounded_wait_reports_timeout_and_recovers(n):
    inp = make_case(batch=256, top_k=4, G=8, K=256, N=n, dtype="bf16", seed=10,
                    device="cuda")
    pgg.pgg_debug_set_wait_limit_ns(20_000_000)  # 20 ms
    pgg.pgg_debug_set_ticket_bias(1000)          # no ticket ever reaches rank + 1000
    try:
        _, ws = run(inp)
        assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_TIMEOUT"
    finally:
        pgg.pgg_debug_set_ticket_bias(0)
        pgg.pgg_debug_set_wait_limit_ns(0)
    check(inp, what="after timeout")


@pytest.mark.parametrize("variant,dtype", [(1, "bf16"), (2, "fp16"), (0, "fp32"), (1, "fp32")])
def test_bounded_wait_timeout_single_cta_forms(variant, dtype):
    """The single-CTA instantiations of the ticketed kernel (narrow and wide
    row blocks, and the 3xTF32 fp32 form) give up on a ticket that never comes
    the same way the CTA-pair form does."""
    inp = make_case(batch=256, top_k=4, G=8, K=256, N=128, dtype=dtype, seed=11,
                    device="cuda")
    pgg.pgg_debug_force_variant(variant)
    pgg.pgg_debug_set_wait_limit_ns(20_000_000)  # 20 ms
    pgg.pgg_debug_set_ticket_bias(1000)
    try:
        plan = pgg.pgg_dx_plan(*_sizes(inp), inp.row_idx_type, pgg.dtype_code(inp.grad_y.dtype))
        assert plan["variant"] == variant and plan["cta_pair"] == 0
        _, ws = run(inp)
        assert pgg.STATUS[pgg.status(ws)] == "PGG_ERR_TIMEOUT"
    finally:
        pgg.pgg_debug_set_ticket_bias(0)
        pgg.pgg_debug_set_wait_limit_ns(0)
        pgg.pgg_debug_force_variant(-1)
    check(inp, what="after timeout")


def test_no_writes_outside_out_and_workspace():
    inp = make_case(batch=100, top_k=3, G=5, K=200, N=96, dtype="bf16", seed=11, device="cuda")
    need = pgg.workspace_bytes(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list,
                               inp.batch, inp.top_k, 0)
    guard = 4096
    ws_buf = torch.full((need + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
    out_buf = torch.full((100 * 200 + 2 * 1024,), -3.0, device="cuda")
    ws = ws_buf[guard:guard + need]
    out = out_buf[1024:1024 + 100 * 200].view(100, 200)
    _, _ = run(inp, out=out, workspace=ws)
    assert pgg.status(ws) == 0
    assert (ws_buf[:guard] == 0xA5).all() and (ws_buf[guard + need:] == 0xA5).all()
    assert (out_buf[:1024] == -3.0).all() and (out_buf[1024 + 100 * 200:] == -3.0).all()
    assert_close(out.double().cpu().numpy(), ref_rows(inp))


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_unaligned_rows_many_tiles(dtype):
    # rows of 2 * 1030 (or 4 * 1031) bytes over many row blocks, k blocks with
    # a ragged tail, and a ragged reduction tail: 16-bit rows on the gather
    # warps of variant 5, fp32 rows on the FP32-pipe kernel; then 16-bit rows
    # of an odd length (2 * 1031 bytes), also on the FP32 pipes
    n = 1031 if dtype == "fp32" else 1030
    inp = make_case(batch=1000, top_k=4, G=9, K=300, N=n, dtype=dtype, routing="zipf",
                    zipf_zero=2, seed=12, device="cuda")
    want = 3 if dtype == "fp32" else 5
    assert pgg.pgg_dx_plan(*_sizes(inp), 0, pgg.dtype_code(inp.grad_y.dtype))["variant"] == want
    check(inp, what=f"unaligned rows {dtype}")
    if dtype != "fp32":
        inp = make_case(batch=1000, top_k=4, G=9, K=300, N=1031, dtype=dtype, routing="zipf",
                        zipf_zero=2, seed=12, device="cuda")
        assert pgg.pgg_dx_plan(*_sizes(inp), 0, pgg.dtype_code(inp.grad_y.dtype))["variant"] == 3
        check(inp, what=f"odd rows {dtype}")


def _sizes(inp):
    M, N = inp.grad_y.shape
    G, K, _ = inp.weight.shape
    return M, N, K, G, M, inp.batch, inp.top_k


def _shifted(t, elems):
    # the same values in a contiguous tensor whose address is `elems` elements
    # past an allocation boundary
    buf = torch.empty(t.numel() + elems, dtype=t.dtype, device=t.device)
    v = buf[elems:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_misaligned_pointers(dtype):
    # gradY / weight not 16-byte aligned: the FP32-pipe kernel, whose result
    # does not depend on the addresses; out not 16-byte aligned: scalar
    # epilogue stores, bitwise equal to the vector ones
    inp = make_case(batch=300, top_k=4, G=6, K=256, N=128, dtype=dtype, seed=15, device="cuda")
    ref = ref_rows(inp)
    try:
        pgg.pgg_debug_force_variant(3)
        simt, _ = run(inp)
    finally:
        pgg.pgg_debug_force_variant(-1)
    assert_close(simt.double().cpu().numpy(), ref, "forced FP32-pipe kernel")
    for shift_y, shift_w in ((1, 0), (0, 1), (3, 5)):
        out, ws = pgg.dx(_shifted(inp.grad_y, shift_y), _shifted(inp.weight, shift_w),
                         inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k, 0)
        torch.cuda.synchronize()
        assert pgg.status(ws) == 0
        assert torch.equal(out.view(torch.int32), simt.view(torch.int32)), (shift_y, shift_w)
    tc, _ = run(inp)
    assert_close(tc.double().cpu().numpy(), ref, "tensor cores")
    out_buf = torch.empty(300 * 256 + 1, dtype=torch.float32, device="cuda")
    out = out_buf[1:].view(300, 256)
    _, ws = run(inp, out=out)
    assert pgg.status(ws) == 0
    assert torch.equal(out.view(torch.int32), tc.view(torch.int32))
    _, ws = pgg.dx(_shifted(inp.grad_y, 1), inp.weight, inp.expanded_row_idx, inp.group_list,
                   inp.batch, inp.top_k, 0, out=out)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    assert torch.equal(out.view(torch.int32), simt.view(torch.int32))


# ---------------------------------------------------------------- full-size workloads

@pytest.mark.parametrize("name", ["tiny-fp32", "uniform-bf16", "skewed-fp16", "large-bf16",
                                  "skinny-bf16", "unaligned-bf16"])
def test_workload_full_size(name):
    # every token against the oracle (large-bf16: a seeded 1/16 of them), in the
    # launch configuration the benchmark times; bitwise equal on a second run
    w = WORKLOADS[name]
    inp = make_inputs(w, device="cuda")
    out, ws = run(inp)
    assert pgg.status(ws) == 0
    toks = sampling.units(name, w.batch, seed=1)
    got = out.double().cpu().numpy()
    if toks is not None:
        got = got[toks]
    assert_close(got, ref_rows(inp, toks), name)
    again, _ = run(inp, workspace=ws)
    assert torch.equal(out.view(torch.int32), again.view(torch.int32))
    assert torch.isfinite(out).all()


def _random_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        top_k = int(rng.integers(1, 9))
        cases.append(dict(batch=int(rng.integers(1, 2500)), top_k=top_k,
                          G=int(rng.integers(top_k, 40)), K=int(rng.integers(1, 700)),
                          N=int(rng.integers(1, 400)),
                          dtype=str(rng.choice(["bf16", "fp16", "fp32"])),
                          row_idx_type=int(rng.integers(0, 2)), seed=700 + i))
    return cases


@pytest.mark.parametrize("case", _random_cases(20, 4545),
                         ids=lambda c: "b{batch}k{top_k}g{G}K{K}N{N}{dtype}".format(**c))
def test_random_shapes(case):
    # random sizes, dtypes and index forms through the automatic plan (ticketed,
    # narrow, FP32-pipe or owner kernel), against the oracle, and repeatable
    inp = make_case(device="cuda", **case)
    toks = None
    if inp.batch > 256:
        toks = np.sort(np.random.default_rng(case["seed"]).choice(inp.batch, 64, replace=False))
    a = check(inp, tokens=toks, what=str(case))
    b, _ = run(inp)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
