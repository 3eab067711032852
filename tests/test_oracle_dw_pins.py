"""Pins for the oracle's weight gradient, by means other than the oracle itself.

d_weight[g, k, n] = sum over the expanded rows i of expert g of
x[batch(i), k] * d_y[i, n]: the separate operator expanded_x^T @ d_y of
"MoeInitRoutingGroupedMatmulGrad design", section 1.2 ("为何不计算 d_weight",
item 3), with expanded_x[i] = x[batch(i)] from the forward's MoeInitRouting
(section 1.1). Checked against a hand-worked example, a pure-Python
indicator-sum brute force, the unfused form with expanded_x materialised
(numpy), torch.matmul for one expert with identity routing, and the adjoint
identity sum(d_weight * weight) == sum(d_x * x), which holds because both are
gradients of <d_y, y> for the same forward y = GroupedMatmul(Permute(x), weight).
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import make_case
from workloads.moe import forward_input, with_row_idx_type

HERE = os.path.dirname(os.path.abspath(__file__))


def as_f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def rel_err(a, b):
    scale = max(np.abs(b).max(), 1e-300)
    return np.abs(a - b).max() / scale


def run_dw(inp, x, **kw):
    return oracle.dw(x, inp.grad_y, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k,
                     inp.row_idx_type, **kw)


def run_dx(inp):
    return oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                     inp.top_k, inp.row_idx_type)


def brute_force_dw(inp, x):
    """sum over all i of 1[g(i) == g] * x[batch(i), k] * dy[i, n], plain loops,
    with its own reading of the index."""
    dy = as_f64(inp.grad_y).tolist()
    xs = as_f64(x).tolist()
    idx = inp.expanded_row_idx.cpu().tolist()
    gl = inp.group_list.cpu().tolist()
    M, N = len(dy), len(dy[0])
    G, K = len(gl), len(xs[0])

    def group_of(i):
        start = 0
        for g in range(G):
            if start <= i < start + gl[g]:
                return g
            start += gl[g]
        raise AssertionError("row outside all groups")

    def batch_of(i):
        if inp.row_idx_type == 0:
            return idx[i] // inp.top_k
        return idx.index(i) // inp.top_k

    out = np.zeros((G, K, N))
    for g in range(G):
        for k in range(K):
            for n in range(N):
                s = 0.0
                for i in range(M):
                    ind = 1.0 if group_of(i) == g else 0.0
                    s += ind * xs[batch_of(i)][k] * dy[i][n]
                out[g, k, n] = s
    return out


def unfused_dw(inp, x):
    """expanded_x materialised (row i = x[batch(i)]), then expanded_x[rows g]^T
    @ d_y[rows g] per expert with numpy."""
    dy = as_f64(inp.grad_y)
    xs = as_f64(x)
    gl = inp.group_list.cpu().numpy()
    idx = inp.expanded_row_idx.cpu().numpy()
    M = dy.shape[0]
    if inp.row_idx_type == 0:
        pos = idx
    else:
        pos = np.empty(M, dtype=np.int64)
        pos[idx] = np.arange(M)
    ex = xs[pos // inp.top_k]
    starts = np.concatenate([[0], np.cumsum(gl)])
    out = np.zeros((len(gl), xs.shape[1], dy.shape[1]))
    for g in range(len(gl)):
        lo, hi = starts[g], starts[g + 1]
        out[g] = ex[lo:hi].T @ dy[lo:hi]
    return out


def test_hand_worked_example(oracle_lib):
    ex = json.load(open(os.path.join(HERE, "golden", "hand_example.json")))
    dy = np.array(ex["grad_y"], dtype=np.float32)
    x = np.array(ex["x"], dtype=np.float32)
    gl = np.array(ex["groupList"], dtype=np.int64)
    for rit, key in ((0, "gather"), (1, "scatter")):
        idx = np.array(ex[key], dtype=np.int64)
        got = oracle.dw(x, dy, idx, gl, ex["batch"], ex["topK"], rit)
        assert np.array_equal(got, np.array(ex["d_weight"], dtype=np.float64))
        w = np.array(ex["weight"], dtype=np.float64)
        assert (got * w).sum() == ex["adjoint"]


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("row_idx_type", [0, 1])
@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_matches_indicator_sum_brute_force(oracle_lib, seed, row_idx_type, dtype):
    inp = make_case(batch=5, top_k=2, G=3, K=6, N=7, dtype=dtype, seed=seed,
                    row_idx_type=row_idx_type)
    x = forward_input(inp)
    assert rel_err(run_dw(inp, x), brute_force_dw(inp, x)) <= 1e-12


def test_brute_force_empty_expert_and_duplicate_experts(oracle_lib):
    inp = make_case(batch=4, top_k=2, G=4, K=5, N=4, dtype="fp32", empty=(1,), seed=3)
    x = forward_input(inp)
    got = run_dw(inp, x)
    assert np.all(got[1] == 0.0)
    assert rel_err(got, brute_force_dw(inp, x)) <= 1e-12
    inp = make_case(batch=6, top_k=3, G=2, K=4, N=3, dtype="fp32", routing="replacement", seed=4)
    x = forward_input(inp)
    assert rel_err(run_dw(inp, x), brute_force_dw(inp, x)) <= 1e-12


@pytest.mark.parametrize("row_idx_type", [0, 1])
@pytest.mark.parametrize("shape", [(128, 3, 10, 128, 256), (10, 3, 4, 178, 286), (1, 3, 3, 128, 256)])
def test_matches_unfused_form(oracle_lib, row_idx_type, shape):
    batch, top_k, G, K, N = shape
    inp = make_case(batch=batch, top_k=top_k, G=G, K=K, N=N, dtype="bf16",
                    row_idx_type=row_idx_type, seed=batch)
    x = forward_input(inp)
    assert rel_err(run_dw(inp, x), unfused_dw(inp, x)) <= 1e-12


def test_one_expert_identity_routing_is_plain_matmul(oracle_lib):
    inp = make_case(batch=96, top_k=1, G=1, K=40, N=72, dtype="fp32", seed=5)
    assert torch.equal(inp.expanded_row_idx, torch.arange(96))
    x = forward_input(inp)
    ref = torch.matmul(x.double().T, inp.grad_y.double()).numpy()
    assert rel_err(run_dw(inp, x)[0], ref) <= 1e-12


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("routing", ["uniform", "zipf", "replacement"])
def test_adjoint_identity_with_d_x(oracle_lib, dtype, routing):
    # <d_y, y> differentiated w.r.t. weight and w.r.t. x: sum(dW * W) == sum(d_x * x)
    inp = make_case(batch=40, top_k=3, G=6, K=24, N=20, dtype=dtype, routing=routing,
                    zipf_zero=1 if routing == "zipf" else 0, seed=8)
    x = forward_input(inp)
    lhs = (run_dw(inp, x) * as_f64(inp.weight)).sum()
    rhs = (run_dx(inp) * as_f64(x)).sum()
    assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + abs(rhs) + 1.0)


def test_selected_rows_equal_the_full_gradient(oracle_lib):
    inp = make_case(batch=30, top_k=2, G=5, K=9, N=11, dtype="fp16", seed=9, empty=(2,))
    x = forward_input(inp)
    full = run_dw(inp, x)
    g = np.array([4, 0, 2, 1, 4])
    k = np.array([8, 0, 3, 5, 0])
    assert np.array_equal(run_dw(inp, x, sel=(g, k)), full[g, k])


def test_invariants(oracle_lib):
    inp = make_case(batch=50, top_k=4, G=7, K=12, N=10, dtype="fp32", seed=10)
    x = forward_input(inp)
    base = run_dw(inp, x)
    # gather and scatter forms, bitwise
    assert np.array_equal(run_dw(with_row_idx_type(inp, 1), x), base)
    # linear in x (a power-of-two scale is exact in every dtype)
    assert np.array_equal(run_dw(inp, 4.0 * x), 4.0 * base)
