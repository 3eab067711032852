"""GPU parity of the probs-weighted unpermute backward against the fp64 oracle.

perm_grad is d_out * prob rounded once to the dtype: per element |GPU - oracle|
<= 2^-8 |oracle| (bf16; 2^-11 fp16; 2^-23 fp32), or half the subnormal spacing
for results below the dtype's smallest normal number (2^-25 for fp16). probs_grad is an fp32 sum
over h: |GPU - oracle| <= 1e-4 * max |oracle| plus the same one rounding when
it is returned in a 16-bit dtype.
"""

import numpy as np
import pytest
import torch

import oracle
import permute_grouped_gemm_gb300 as pgg
from workloads import WORKLOADS, make_case, make_inputs
from workloads.moe import unpermute_inputs, with_row_idx_type

pytestmark = pytest.mark.gpu

TOL = 1e-4
ROUND = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11, torch.float32: 2.0 ** -23}
SUBNORMAL_HALF_ULP = {torch.bfloat16: 2.0 ** -134, torch.float16: 2.0 ** -25,
                      torch.float32: 2.0 ** -150}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from permute_grouped_gemm_gb300 import build as pbuild
    pbuild.build()
    oracle.build()
    pgg.load()
    yield


def run(inp, d_out, probs, **kw):
    pg, qg, ws = pgg.unpermute_grad(inp.grad_y, d_out, probs, inp.expanded_row_idx, inp.top_k,
                                    inp.row_idx_type, **kw)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0, pgg.STATUS.get(pgg.status(ws))
    return pg, qg


def ref_of(inp, d_out, probs):
    return oracle.unpermute_grad(inp.grad_y, d_out, probs, inp.expanded_row_idx, inp.batch,
                                 inp.top_k, inp.row_idx_type)


def check_pg(pg, ref):
    got = pg.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= ROUND[pg.dtype] * np.abs(ref) + SUBNORMAL_HALF_ULP[pg.dtype])


def check_qg(qg, ref):
    got = qg.double().cpu().numpy()
    r = ROUND[qg.dtype] if qg.dtype != torch.float32 else 0.0
    bound = r * np.abs(ref) + TOL * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= bound), np.abs(got - ref).max()


@pytest.mark.parametrize("qg_f32", [False, True])
@pytest.mark.parametrize("row_idx_type", [0, 1])
@pytest.mark.parametrize("n", [256, 286, 1])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_cases(dtype, n, row_idx_type, qg_f32):
    inp = make_case(batch=150, top_k=3, G=5, K=16, N=n, dtype=dtype, seed=41,
                    row_idx_type=row_idx_type, device="cuda")
    d_out, probs = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, probs, probs_grad_dtype=torch.float32 if qg_f32 else None)
    rpg, rqg = ref_of(inp, d_out, probs)
    check_pg(pg, rpg)
    check_qg(qg, rqg)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_without_probs_is_an_exact_scatter_copy(dtype):
    inp = make_case(batch=300, top_k=4, G=6, K=16, N=512, dtype=dtype, seed=42, device="cuda")
    d_out, _ = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, None)
    assert qg is None
    b = inp.gather.to("cuda") // inp.top_k
    assert torch.equal(pg.view(torch.int16 if dtype != "fp32" else torch.int32),
                       d_out[b].view(torch.int16 if dtype != "fp32" else torch.int32))


def test_bitwise_repeatable_and_index_forms():
    inp = make_case(batch=400, top_k=8, G=16, K=16, N=1024, dtype="bf16", seed=43, device="cuda")
    d_out, probs = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, probs)
    for _ in range(2):
        pg2, qg2 = run(inp, d_out, probs)
        assert torch.equal(pg.view(torch.int16), pg2.view(torch.int16))
        assert torch.equal(qg.view(torch.int16), qg2.view(torch.int16))
    pg3, qg3 = run(with_row_idx_type(inp, 1), d_out, probs)
    assert torch.equal(pg.view(torch.int16), pg3.view(torch.int16))
    assert torch.equal(qg.view(torch.int16), qg3.view(torch.int16))



def test_prep_then_apply_equals_the_one_call():
    inp = make_case(batch=300, top_k=6, G=8, K=16, N=520, dtype="fp16", seed=44,
                    row_idx_type=1, device="cuda")
    d_out, probs = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, probs)
    M, H = inp.grad_y.shape
    need = pgg.pgg_unpermute_grad_workspace_size(M, inp.batch, inp.top_k)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    pg2 = torch.empty_like(pg)
    qg2 = torch.empty_like(qg)
    dt = pgg.dtype_code(inp.grad_y.dtype)
    sp = torch.cuda.current_stream().cuda_stream
    idx = inp.expanded_row_idx
    assert pgg.pgg_unpermute_grad_prep(idx.data_ptr(), M, inp.batch, inp.top_k,
                                       inp.row_idx_type, ws.data_ptr(), need, sp) == 0
    assert pgg.pgg_unpermute_grad_apply(inp.grad_y.data_ptr(), d_out.data_ptr(), probs.data_ptr(),
                                        idx.data_ptr(), M, H, inp.batch, inp.top_k,
                                        inp.row_idx_type, dt, dt, ws.data_ptr(), need,
                                        pg2.data_ptr(), qg2.data_ptr(), sp) == 0
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    assert torch.equal(pg.view(torch.int16), pg2.view(torch.int16))
    assert torch.equal(qg.view(torch.int16), qg2.view(torch.int16))

@pytest.mark.parametrize("shift", [1, 2])
def test_misaligned_pointers_use_the_narrower_paths(shift):
    # shift 1 element: 2-byte accesses; 2 elements: 4-byte pairs
    inp = make_case(batch=200, top_k=4, G=6, K=16, N=512, dtype="bf16", seed=44, device="cuda")
    d_out, probs = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, probs)
    buf = torch.empty(d_out.numel() + shift, dtype=d_out.dtype, device="cuda")
    d_shift = buf[shift:].view(d_out.shape)
    d_shift.copy_(d_out)
    pg2, qg2, ws = pgg.unpermute_grad(inp.grad_y, d_shift, probs, inp.expanded_row_idx,
                                      inp.top_k, 0)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    assert torch.equal(pg.view(torch.int16), pg2.view(torch.int16))
    rpg, rqg = ref_of(inp, d_out, probs)
    check_qg(qg2, rqg)


def test_index_errors_zero_the_outputs():
    inp = make_case(batch=64, top_k=2, G=4, K=16, N=64, dtype="bf16", seed=45, device="cuda")
    d_out, probs = unpermute_inputs(inp)
    for name, mutate in (("PGG_ERR_NOT_PERM", lambda i: i.__setitem__(5, int(i[6]))),
                         ("PGG_ERR_INDEX", lambda i: i.__setitem__(5, 128))):
        idx = inp.expanded_row_idx.clone()
        mutate(idx)
        pg = torch.full((128, 64), 7.0, dtype=torch.bfloat16, device="cuda")
        qg = torch.full((64, 2), 7.0, dtype=torch.bfloat16, device="cuda")
        _, _, ws = pgg.unpermute_grad(inp.grad_y, d_out, probs, idx, 2, 0, perm_grad=pg,
                                      probs_grad=qg)
        torch.cuda.synchronize()
        assert pgg.STATUS[pgg.status(ws)] == name
        assert torch.count_nonzero(pg) == 0 and torch.count_nonzero(qg) == 0


def test_chained_into_the_fused_input_gradient():
    # perm_grad is the gradY of the fused d_x backward
    inp = make_case(batch=256, top_k=4, G=8, K=384, N=256, dtype="bf16", seed=46, device="cuda")
    d_out, probs = unpermute_inputs(inp)
    pg, _ = run(inp, d_out, probs)
    dx, ws = pgg.dx(pg, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k, 0)
    torch.cuda.synchronize()
    assert pgg.status(ws) == 0
    ref = oracle.dx(pg, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k, 0)
    got = dx.double().cpu().numpy()
    assert np.abs(got - ref).max() <= TOL * np.abs(ref).max()


@pytest.mark.parametrize("name", ["uniform-bf16", "skewed-fp16", "large-bf16", "skinny-bf16",
                                  "unaligned-bf16"])
def test_workload_full_size(name):
    # every element of perm_grad and probs_grad against the oracle
    w = WORKLOADS[name]
    inp = make_inputs(w, device="cuda")
    d_out, probs = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, probs)
    rpg, rqg = ref_of(inp, d_out, probs)
    check_pg(pg, rpg)
    check_qg(qg, rqg)
    pg2, qg2 = run(inp, d_out, probs)
    assert torch.equal(pg.view(torch.int16), pg2.view(torch.int16))
    assert torch.equal(qg.view(torch.int16), qg2.view(torch.int16))


def _random_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        top_k = int(rng.integers(1, 9))
        cases.append(dict(batch=int(rng.integers(1, 800)), top_k=top_k,
                          G=int(rng.integers(top_k, 17)), K=16, N=int(rng.integers(1, 700)),
                          dtype=str(rng.choice(["bf16", "fp16", "fp32"])),
                          row_idx_type=int(rng.integers(0, 2)), seed=500 + i,
                          qg_f32=bool(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("case", _random_cases(16, 4444),
                         ids=lambda c: "b{batch}k{top_k}H{N}{dtype}".format(**c))
def test_random_shapes(case):
    # random hidden sizes cross the 16-byte, 4-byte-pair and element paths
    c = dict(case)
    qg_f32 = c.pop("qg_f32")
    inp = make_case(device="cuda", **c)
    d_out, probs = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, probs, probs_grad_dtype=torch.float32 if qg_f32 else None)
    rpg, rqg = ref_of(inp, d_out, probs)
    check_pg(pg, rpg)
    check_qg(qg, rqg)
