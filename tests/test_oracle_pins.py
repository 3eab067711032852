"""Pins for the oracle: checks against things other than the oracle itself.

Every check here is independent of the oracle's code path: a hand-worked
example, a pure-Python brute force of the scalar indicator-sum formula, the
unfused two-step form (grouped matmul then scatter-add) written with numpy,
torch.matmul for the one-expert identity case, closed forms, and invariants
of the formula ("MoeInitRoutingGroupedMatmulGrad design", section
"数学定义和公式"; golden structure from section 4.1 "测试标杆").
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import make_case
from workloads.moe import with_row_idx_type

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- helpers

def as_f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def brute_force(inp):
    """Scalar form: sum over all i, n of 1[batch(i) == b] * dy[i,n] * W[g(i),k,n],
    written with plain Python loops and an independent reading of the index."""
    dy = as_f64(inp.grad_y).tolist()
    w = as_f64(inp.weight).tolist()
    idx = inp.expanded_row_idx.cpu().tolist()
    gl = inp.group_list.cpu().tolist()
    M, N = len(dy), len(dy[0])
    G, K = len(w), len(w[0])
    top_k = inp.top_k

    def group_of(i):
        start = 0
        for g in range(G):
            if start <= i < start + gl[g]:
                return g
            start += gl[g]
        raise AssertionError("row outside all groups")

    def batch_of(i):
        if inp.row_idx_type == 0:
            return idx[i] // top_k
        return idx.index(i) // top_k

    out = [[0.0] * K for _ in range(inp.batch)]
    for b in range(inp.batch):
        for k in range(K):
            s = 0.0
            for i in range(M):
                ind = 1.0 if batch_of(i) == b else 0.0
                g = group_of(i)
                for n in range(N):
                    s += ind * dy[i][n] * w[g][k][n]
            out[b][k] = s
    return np.array(out)


def unfused_numpy(inp):
    """Step 1 (d_expanded_x = d_y @ W[g]^T per expert, materialised) then
    Step 2 (scatter-add of row i into token original_pos(i) // topK)."""
    dy = as_f64(inp.grad_y)
    w = as_f64(inp.weight)
    gl = inp.group_list.cpu().numpy()
    M = dy.shape[0]
    d_exp = np.zeros((M, w.shape[1]))
    starts = np.concatenate([[0], np.cumsum(gl)])
    for g in range(w.shape[0]):
        lo, hi = starts[g], starts[g + 1]
        d_exp[lo:hi] = dy[lo:hi] @ w[g].T
    idx = inp.expanded_row_idx.cpu().numpy()
    if inp.row_idx_type == 0:
        orig = idx
    else:
        orig = np.empty(M, dtype=np.int64)
        orig[idx] = np.arange(M)
    dx = np.zeros((inp.batch, w.shape[1]))
    np.add.at(dx, orig // inp.top_k, d_exp)
    return dx, d_exp


def run(inp, **kw):
    return oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list,
                     inp.batch, inp.top_k, inp.row_idx_type, **kw)


def rel_err(a, b):
    scale = max(np.abs(b).max(), 1e-300)
    return np.abs(a - b).max() / scale


# ---------------------------------------------------------------- decoders

def test_decode_fp16_every_pattern(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.decode(bits, oracle.F16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_decode_bf16_every_pattern(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.decode(bits, oracle.BF16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_decode_fp32_is_exact(oracle_lib):
    x = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    assert np.array_equal(oracle.decode(x, oracle.F32), x.astype(np.float64))


# ---------------------------------------------------------------- worked example

def test_hand_worked_example(oracle_lib):
    ex = json.load(open(os.path.join(HERE, "golden", "hand_example.json")))
    dy = np.array(ex["grad_y"], dtype=np.float32)
    w = np.array(ex["weight"], dtype=np.float32)
    gl = np.array(ex["groupList"], dtype=np.int64)
    for rit, key in ((0, "gather"), (1, "scatter")):
        idx = np.array(ex[key], dtype=np.int64)
        got = oracle.dx(dy, w, idx, gl, ex["batch"], ex["topK"], rit)
        assert np.array_equal(got, np.array(ex["d_x"], dtype=np.float64))


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("row_idx_type", [0, 1])
@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_matches_indicator_sum_brute_force(oracle_lib, seed, row_idx_type, dtype):
    inp = make_case(batch=5, top_k=2, G=3, K=6, N=7, dtype=dtype, seed=seed,
                    row_idx_type=row_idx_type)
    ref = brute_force(inp)
    got = run(inp)
    assert rel_err(got, ref) <= 1e-12


def test_brute_force_empty_expert_and_duplicate_experts(oracle_lib):
    # an expert with no rows (page white-box case "空 expert") ...
    inp = make_case(batch=4, top_k=2, G=4, K=5, N=4, dtype="fp32", empty=(1,), seed=3)
    assert int(inp.group_list[1]) == 0
    assert rel_err(run(inp), brute_force(inp)) <= 1e-12
    # ... and a token that picks the same expert twice
    inp = make_case(batch=6, top_k=3, G=2, K=4, N=3, dtype="fp32", routing="replacement", seed=4)
    assert rel_err(run(inp), brute_force(inp)) <= 1e-12


# ---------------------------------------------------------------- unfused form

@pytest.mark.parametrize("row_idx_type", [0, 1])
@pytest.mark.parametrize("shape", [(128, 3, 10, 128, 256), (10, 3, 4, 178, 286), (1, 3, 3, 128, 256)])
def test_matches_unfused_two_step(oracle_lib, row_idx_type, shape):
    batch, top_k, G, K, N = shape
    inp = make_case(batch=batch, top_k=top_k, G=G, K=K, N=N, dtype="bf16",
                    row_idx_type=row_idx_type, seed=batch)
    ref, _ = unfused_numpy(inp)
    assert rel_err(run(inp), ref) <= 1e-12


def test_column_sums_equal_expanded_column_sums(oracle_lib):
    # sum_b d_x[b, k] == sum_i d_expanded_x[i, k]
    inp = make_case(batch=64, top_k=4, G=8, K=32, N=48, dtype="fp16", seed=7)
    _, d_exp = unfused_numpy(inp)
    got = run(inp)
    assert np.abs(got.sum(0) - d_exp.sum(0)).max() <= 1e-10 * np.abs(d_exp).sum(0).max()


# ---------------------------------------------------------------- library special case

def test_one_expert_identity_routing_is_plain_matmul(oracle_lib):
    inp = make_case(batch=96, top_k=1, G=1, K=40, N=72, dtype="fp32", seed=5)
    assert torch.equal(inp.expanded_row_idx, torch.arange(96))
    ref = torch.matmul(inp.grad_y.double(), inp.weight[0].double().T).numpy()
    assert rel_err(run(inp), ref) <= 1e-12


# ---------------------------------------------------------------- closed forms

def test_closed_form_all_ones(oracle_lib):
    inp = make_case(batch=9, top_k=3, G=4, K=11, N=13, dtype="bf16", seed=6)
    inp.grad_y.fill_(1.0)
    inp.weight.fill_(1.0)
    got = run(inp)
    assert np.array_equal(got, np.full((9, 11), 3.0 * 13))


def test_closed_form_shifted_identity_weights(oracle_lib):
    # weight[g, k, n] = (g + 1) if n == (k + s) mod N else 0, with K == N:
    # d_x[b, k] = sum_j (g_j + 1) * d_y[i_j, (k + s) mod N]
    # (distinguishes weight[g,k,n] from its transpose weight[g,n,k]).
    batch, top_k, G, N, s = 7, 3, 5, 12, 5
    inp = make_case(batch=batch, top_k=top_k, G=G, K=N, N=N, dtype="fp32", seed=8)
    w = torch.zeros(G, N, N)
    for g in range(G):
        for k in range(N):
            w[g, k, (k + s) % N] = g + 1
    inp.weight.copy_(w)
    dy = inp.grad_y.double()
    gather = inp.gather.tolist()
    expert_of_row = np.repeat(np.arange(G), inp.group_list.numpy())
    ref = np.zeros((batch, N))
    for i, p in enumerate(gather):
        b = p // top_k
        for k in range(N):
            ref[b, k] += (expert_of_row[i] + 1) * float(dy[i, (k + s) % N])
    assert rel_err(run(inp), ref) <= 1e-13


# ---------------------------------------------------------------- invariants

def test_gather_and_scatter_index_give_identical_result(oracle_lib):
    inp0 = make_case(batch=50, top_k=4, G=6, K=24, N=40, dtype="fp16", seed=9, row_idx_type=0)
    inp1 = with_row_idx_type(inp0, 1)
    assert np.array_equal(run(inp0), run(inp1))


def test_expert_relabelling_invariance(oracle_lib):
    inp = make_case(batch=40, top_k=3, G=5, K=16, N=24, dtype="bf16", seed=10)
    M = inp.batch * inp.top_k
    base = run(inp)
    relabel = torch.tensor([3, 0, 4, 1, 2])  # old expert e -> new expert relabel[e]
    expert_of_row = torch.repeat_interleave(torch.arange(5), inp.group_list)
    new_expert = relabel[expert_of_row]
    key = new_expert * M + inp.gather  # re-sort rows stably by new id, then position
    order = torch.argsort(key)
    dy = inp.grad_y[order]
    gather = inp.gather[order]
    w = torch.empty_like(inp.weight)
    w[relabel] = inp.weight
    gl = torch.bincount(new_expert, minlength=5)
    got = oracle.dx(dy, w, gather, gl, inp.batch, inp.top_k, 0)
    assert np.array_equal(got, base)


def test_empty_experts_contribute_nothing(oracle_lib):
    inp = make_case(batch=30, top_k=2, G=4, K=20, N=16, dtype="fp32", seed=11)
    base = run(inp)
    # insert three experts with random weights and no rows
    extra = torch.randn(3, 20, 16)
    w = torch.cat([extra[:1], inp.weight[:2], extra[1:], inp.weight[2:]])
    gl = torch.cat([torch.zeros(1, dtype=torch.int64), inp.group_list[:2],
                    torch.zeros(2, dtype=torch.int64), inp.group_list[2:]])
    got = oracle.dx(inp.grad_y, w, inp.expanded_row_idx, gl, inp.batch, inp.top_k, 0)
    assert np.array_equal(got, base)


def test_linear_in_grad_y(oracle_lib):
    a = make_case(batch=20, top_k=3, G=4, K=12, N=10, dtype="fp32", seed=12)
    b = make_case(batch=20, top_k=3, G=4, K=12, N=10, dtype="fp32", seed=13)
    b_dy = b.grad_y
    s = (a.grad_y.double() * 0.5 + b_dy.double() * 2.0).float()
    exact_ok = torch.equal(s.double(), a.grad_y.double() * 0.5 + b_dy.double() * 2.0)
    ra = run(a)
    rb = oracle.dx(b_dy, a.weight, a.expanded_row_idx, a.group_list, a.batch, a.top_k, 0)
    rs = oracle.dx(s, a.weight, a.expanded_row_idx, a.group_list, a.batch, a.top_k, 0)
    tol = 1e-12 if exact_ok else 1e-6
    assert rel_err(rs, 0.5 * ra + 2.0 * rb) <= tol


def test_token_subset_equals_rows_of_full(oracle_lib):
    inp = make_case(batch=33, top_k=2, G=3, K=9, N=8, dtype="bf16", seed=14)
    full = run(inp)
    toks = np.array([32, 0, 7, 7, 15])
    assert np.array_equal(run(inp, tokens=toks), full[toks])
    assert np.array_equal(run(inp, nthreads=1), full)


# ---------------------------------------------------------------- constraint table

def test_rejects_inputs_outside_the_constraints(oracle_lib):
    inp = make_case(batch=8, top_k=2, G=3, K=4, N=4, dtype="fp32", seed=15)
    args = lambda **o: dict(dict(grad_y=inp.grad_y, weight=inp.weight,  # noqa: E731
                                 expanded_row_idx=inp.expanded_row_idx,
                                 group_list=inp.group_list, batch=8, top_k=2,
                                 row_idx_type=0), **o)

    def code(**o):
        with pytest.raises(oracle.OracleError) as e:
            oracle.dx(**args(**o))
        return e.value.code

    gl = inp.group_list.clone()
    gl[0] += 1
    assert code(group_list=gl) == 17                      # sum != M
    gl = inp.group_list.clone()
    gl[1] += gl[0] + 1
    gl[0] = -1                                            # sum still M
    assert int(gl.sum()) == 16
    assert code(group_list=gl) == 17                      # negative count
    idx = inp.expanded_row_idx.clone()
    idx[3] = 16
    assert code(expanded_row_idx=idx) == 16              # out of range
    idx = inp.expanded_row_idx.clone()
    idx[3] = idx[4]
    assert code(expanded_row_idx=idx) == 18              # not a permutation
    assert code(row_idx_type=1, expanded_row_idx=idx) == 18
    assert code(batch=7) == 2                            # M != batch * topK
    assert code(row_idx_type=2) == 3
    assert code(top_k=0) == 3
