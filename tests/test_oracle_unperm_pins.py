"""Pins for the oracle's probs-weighted unpermute backward.

"NPU DeepSeek-V3.2-Exp TileLang operator practice", section
moe_token_unpermute_grad: for the combine out[b] = sum_j prob[b, j] *
permuted[row(b, j)],
    perm_grad[row(b, j)] = d_out[b] * prob[b, j]   (prob = 1 without probs)
    probs_grad[b, j]     = <d_out[b], permuted[row(b, j)]>.
Checked against a hand-worked example, plain-loop brute force, a vectorised
numpy form, the plain scatter copy without probs, and the adjoint identities
sum(prob * probs_grad) == <d_out, out> == <perm_grad, permuted>.
"""

import numpy as np
import pytest
import torch

import oracle
from workloads import make_case
from workloads.moe import unpermute_inputs, with_row_idx_type


def as_f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def rel_err(a, b):
    scale = max(np.abs(b).max(), 1e-300)
    return np.abs(a - b).max() / scale


def row_of_position(inp):
    idx = inp.expanded_row_idx.cpu().numpy()
    if inp.row_idx_type == 1:
        return idx.copy()
    r = np.empty_like(idx)
    r[idx] = np.arange(idx.shape[0])
    return r


def brute(inp, d_out, probs):
    perm = as_f64(inp.grad_y).tolist()
    d = as_f64(d_out).tolist()
    pr = as_f64(probs).tolist()
    idx = inp.expanded_row_idx.cpu().tolist()
    M, H = len(perm), len(perm[0])
    pg = np.zeros((M, H))
    qg = np.zeros((inp.batch, inp.top_k))
    for b in range(inp.batch):
        for j in range(inp.top_k):
            p = b * inp.top_k + j
            i = idx.index(p) if inp.row_idx_type == 0 else idx[p]
            for h in range(H):
                pg[i][h] = d[b][h] * pr[b][j]
                qg[b][j] += d[b][h] * perm[i][h]
    return pg, qg


def run(inp, d_out, probs):
    return oracle.unpermute_grad(inp.grad_y, d_out, probs, inp.expanded_row_idx, inp.batch,
                                 inp.top_k, inp.row_idx_type)


def test_hand_worked_example(oracle_lib):
    # the routing of tests/golden/hand_example.json: gather [1, 2, 0, 3], so
    # position p0 -> row i2, p1 -> i0, p2 -> i1, p3 -> i3; permuted rows
    # i0..i3 = [1,2], [3,-1], [0.5,4], [-2,1]; d_out = [[1,-1],[2,0.5]];
    # probs = [[0.25, 0.75], [0.5, 0.5]].
    # perm_grad: i2 = 0.25*[1,-1], i0 = 0.75*[1,-1], i1 = i3 = 0.5*[2,0.5];
    # probs_grad: <[1,-1],[0.5,4]> = -3.5, <[1,-1],[1,2]> = -1,
    #             <[2,0.5],[3,-1]> = 5.5, <[2,0.5],[-2,1]> = -3.5.
    perm = np.array([[1, 2], [3, -1], [0.5, 4], [-2, 1]], dtype=np.float32)
    d_out = np.array([[1, -1], [2, 0.5]], dtype=np.float32)
    probs = np.array([[0.25, 0.75], [0.5, 0.5]], dtype=np.float32)
    want_pg = np.array([[0.75, -0.75], [1, 0.25], [0.25, -0.25], [1, 0.25]])
    want_qg = np.array([[-3.5, -1], [5.5, -3.5]])
    for rit, idx in ((0, [1, 2, 0, 3]), (1, [2, 0, 1, 3])):
        pg, qg = oracle.unpermute_grad(perm, d_out, probs, np.array(idx), 2, 2, rit)
        assert np.array_equal(pg, want_pg) and np.array_equal(qg, want_qg)


@pytest.mark.parametrize("row_idx_type", [0, 1])
@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_matches_brute_force(oracle_lib, row_idx_type, dtype):
    inp = make_case(batch=6, top_k=3, G=4, K=8, N=5, dtype=dtype, seed=2,
                    row_idx_type=row_idx_type)
    d_out, probs = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, probs)
    bpg, bqg = brute(inp, d_out, probs)
    assert rel_err(pg, bpg) <= 1e-15 and rel_err(qg, bqg) <= 1e-12


@pytest.mark.parametrize("row_idx_type", [0, 1])
def test_matches_vectorised_form(oracle_lib, row_idx_type):
    inp = make_case(batch=200, top_k=4, G=8, K=16, N=96, dtype="bf16", seed=3,
                    row_idx_type=row_idx_type)
    d_out, probs = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, probs)
    rows = row_of_position(inp)
    d = as_f64(d_out)
    pr = as_f64(probs).reshape(-1)
    perm = as_f64(inp.grad_y)
    b = np.arange(inp.batch * inp.top_k) // inp.top_k
    want_pg = np.empty_like(perm)
    want_pg[rows] = d[b] * pr[:, None]
    want_qg = np.einsum("ph,ph->p", d[b], perm[rows]).reshape(inp.batch, inp.top_k)
    assert np.array_equal(pg, want_pg)
    assert rel_err(qg, want_qg) <= 1e-12


def test_without_probs_is_the_scatter_copy(oracle_lib):
    inp = make_case(batch=50, top_k=2, G=4, K=8, N=33, dtype="fp16", seed=4)
    d_out, _ = unpermute_inputs(inp)
    pg, qg = oracle.unpermute_grad(None, d_out, None, inp.expanded_row_idx, inp.batch,
                                   inp.top_k, 0)
    assert qg is None
    rows = row_of_position(inp)
    assert np.array_equal(pg[rows], as_f64(d_out)[np.arange(100) // 2])


def test_adjoint_identities(oracle_lib):
    inp = make_case(batch=60, top_k=3, G=5, K=8, N=40, dtype="bf16", seed=5)
    d_out, probs = unpermute_inputs(inp)
    pg, qg = run(inp, d_out, probs)
    rows = row_of_position(inp)
    perm = as_f64(inp.grad_y)
    pr = as_f64(probs)
    out = (perm[rows].reshape(inp.batch, inp.top_k, -1) * pr[:, :, None]).sum(1)
    inner = (as_f64(d_out) * out).sum()
    for other in ((pr * qg).sum(), (pg * perm).sum()):
        assert abs(inner - other) <= 1e-12 * (abs(inner) + abs(other) + 1.0)


def test_index_forms_agree_bitwise(oracle_lib):
    inp = make_case(batch=40, top_k=4, G=6, K=8, N=24, dtype="fp32", seed=6)
    d_out, probs = unpermute_inputs(inp)
    a = run(inp, d_out, probs)
    b = run(with_row_idx_type(inp, 1), d_out, probs)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
