"""Pins for the oracle's forward, by means other than the oracle itself.

y[i, n] = sum_k x[batch(i), k] * weight[g(i), k, n]: MoeInitRouting (x ->
expanded_x, rows laid out by expert) followed by GroupedMatmul(expanded_x,
weight), the forward chain of "MoeInitRoutingGroupedMatmulGrad design",
sections 1.1 and 1.2. Checked against a hand-worked example, a pure-Python
indicator-sum brute force, the unfused form (expanded_x materialised, one
numpy matmul per expert), torch.matmul for one expert with identity routing,
and the two adjoint identities <d_y, y> == sum(d_x * x) == sum(d_weight *
weight), which tie the forward to both backward functions.
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


def run_fwd(inp, x, **kw):
    return oracle.fwd(x, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k,
                      inp.row_idx_type, **kw)


def brute_force_fwd(inp, x):
    """sum over all b, g, k of 1[batch(i) == b] 1[g(i) == g] x[b, k] W[g, k, n],
    plain loops with their own reading of the index."""
    xs = as_f64(x).tolist()
    w = as_f64(inp.weight).tolist()
    idx = inp.expanded_row_idx.cpu().tolist()
    gl = inp.group_list.cpu().tolist()
    M = len(idx)
    G, K, N = len(w), len(w[0]), len(w[0][0])

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

    out = np.zeros((M, N))
    for i in range(M):
        for n in range(N):
            s = 0.0
            for b in range(len(xs)):
                for g in range(G):
                    ind = (1.0 if batch_of(i) == b else 0.0) * (1.0 if group_of(i) == g else 0.0)
                    if ind:
                        for k in range(K):
                            s += xs[b][k] * w[g][k][n]
            out[i, n] = s
    return out


def unfused_fwd(inp, x):
    xs = as_f64(x)
    w = as_f64(inp.weight)
    gl = inp.group_list.cpu().numpy()
    idx = inp.expanded_row_idx.cpu().numpy()
    M = idx.shape[0]
    if inp.row_idx_type == 0:
        pos = idx
    else:
        pos = np.empty(M, dtype=np.int64)
        pos[idx] = np.arange(M)
    ex = xs[pos // inp.top_k]
    starts = np.concatenate([[0], np.cumsum(gl)])
    y = np.zeros((M, w.shape[2]))
    for g in range(len(gl)):
        lo, hi = starts[g], starts[g + 1]
        y[lo:hi] = ex[lo:hi] @ w[g]
    return y


def test_hand_worked_example(oracle_lib):
    # the example of tests/golden/hand_example.json; its forward, by hand:
    # expanded_x rows i0..i3 = x[b0], x[b1], x[b0], x[b1] = [1,-1], [2,0.5], [1,-1], [2,0.5];
    # experts e0 (i0, i1) with W0 = [[1,0],[2,1]], e1 (i2, i3) with W1 = [[0,3],[1,-1]];
    # y[i0] = [1*1 - 1*2, 1*0 - 1*1] = [-1, -1]; y[i1] = [2*1 + 0.5*2, 0 + 0.5*1] = [3, 0.5];
    # y[i2] = [0 - 1*1, 3 + 1] = [-1, 4]; y[i3] = [0 + 0.5, 6 - 0.5] = [0.5, 5.5].
    # <d_y, y> = (1*-1 + 2*-1) + (3*3 - 1*0.5) + (0.5*-1 + 4*4) + (-2*0.5 + 1*5.5) = 25.5,
    # the same number as sum(d_x * x) and sum(d_weight * weight) in that file.
    ex = json.load(open(os.path.join(HERE, "golden", "hand_example.json")))
    x = np.array(ex["x"], dtype=np.float32)
    w = np.array(ex["weight"], dtype=np.float32)
    gl = np.array(ex["groupList"], dtype=np.int64)
    dy = np.array(ex["grad_y"], dtype=np.float64)
    want = np.array([[-1, -1], [3, 0.5], [-1, 4], [0.5, 5.5]], dtype=np.float64)
    for rit, key in ((0, "gather"), (1, "scatter")):
        idx = np.array(ex[key], dtype=np.int64)
        y = oracle.fwd(x, w, idx, gl, ex["batch"], ex["topK"], rit)
        assert np.array_equal(y, want)
        assert (y * dy).sum() == ex["adjoint"]


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("row_idx_type", [0, 1])
@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_matches_indicator_sum_brute_force(oracle_lib, seed, row_idx_type, dtype):
    inp = make_case(batch=5, top_k=2, G=3, K=6, N=7, dtype=dtype, seed=seed,
                    row_idx_type=row_idx_type)
    x = forward_input(inp)
    assert rel_err(run_fwd(inp, x), brute_force_fwd(inp, x)) <= 1e-12


def test_brute_force_empty_expert_and_duplicate_experts(oracle_lib):
    inp = make_case(batch=4, top_k=2, G=4, K=5, N=4, dtype="fp32", empty=(1,), seed=3)
    x = forward_input(inp)
    assert rel_err(run_fwd(inp, x), brute_force_fwd(inp, x)) <= 1e-12
    inp = make_case(batch=6, top_k=3, G=2, K=4, N=3, dtype="fp32", routing="replacement", seed=4)
    x = forward_input(inp)
    assert rel_err(run_fwd(inp, x), brute_force_fwd(inp, x)) <= 1e-12


@pytest.mark.parametrize("row_idx_type", [0, 1])
@pytest.mark.parametrize("shape", [(128, 3, 10, 128, 256), (10, 3, 4, 178, 286), (1, 3, 3, 128, 256)])
def test_matches_unfused_form(oracle_lib, row_idx_type, shape):
    batch, top_k, G, K, N = shape
    inp = make_case(batch=batch, top_k=top_k, G=G, K=K, N=N, dtype="bf16",
                    row_idx_type=row_idx_type, seed=batch)
    x = forward_input(inp)
    assert rel_err(run_fwd(inp, x), unfused_fwd(inp, x)) <= 1e-12


def test_one_expert_identity_routing_is_plain_matmul(oracle_lib):
    inp = make_case(batch=96, top_k=1, G=1, K=40, N=72, dtype="fp32", seed=5)
    x = forward_input(inp)
    ref = torch.matmul(x.double(), inp.weight[0].double()).numpy()
    assert rel_err(run_fwd(inp, x), ref) <= 1e-12


@pytest.mark.parametrize("routing", ["uniform", "zipf", "replacement"])
def test_adjoint_identities(oracle_lib, routing):
    inp = make_case(batch=40, top_k=3, G=6, K=24, N=20, dtype="bf16", routing=routing,
                    zipf_zero=1 if routing == "zipf" else 0, seed=8)
    x = forward_input(inp)
    dy = as_f64(inp.grad_y)
    inner = (run_fwd(inp, x) * dy).sum()
    dx = oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                   inp.top_k, inp.row_idx_type)
    dw = oracle.dw(x, inp.grad_y, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k,
                   inp.row_idx_type)
    for other in ((dx * as_f64(x)).sum(), (dw * as_f64(inp.weight)).sum()):
        assert abs(inner - other) <= 1e-12 * (abs(inner) + abs(other) + 1.0)


def test_selected_rows_and_index_forms(oracle_lib):
    inp = make_case(batch=30, top_k=2, G=5, K=9, N=11, dtype="fp16", seed=9, empty=(2,))
    x = forward_input(inp)
    full = run_fwd(inp, x)
    rows = np.array([59, 0, 17, 3, 59])
    assert np.array_equal(run_fwd(inp, x, rows=rows), full[rows])
    assert np.array_equal(run_fwd(with_row_idx_type(inp, 1), x), full)
