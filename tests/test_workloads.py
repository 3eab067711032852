"""The seeded input generator produces what its recipe states."""

import torch

from workloads import WORKLOADS, make_case, expanded_order, route_experts, Workload


def check_routing(inp):
    w = inp.workload
    M = w.M
    gather = inp.gather
    assert torch.equal(torch.sort(gather).values, torch.arange(M))
    assert int(inp.group_list.sum()) == M
    assert (inp.group_list >= 0).all()
    # rows are sorted by (expert, original position)
    expert_of_row = torch.repeat_interleave(torch.arange(w.G), inp.group_list)
    flat = inp.experts.reshape(-1)
    assert torch.equal(flat[gather], expert_of_row)
    key = expert_of_row * M + gather
    assert (key[1:] > key[:-1]).all()
    if w.row_idx_type == 1:
        assert torch.equal(inp.expanded_row_idx[gather], torch.arange(M))
    else:
        assert torch.equal(inp.expanded_row_idx, gather)


def test_small_cases_are_valid_and_deterministic():
    for rit in (0, 1):
        a = make_case(batch=37, top_k=3, G=7, K=8, N=16, row_idx_type=rit, seed=3)
        b = make_case(batch=37, top_k=3, G=7, K=8, N=16, row_idx_type=rit, seed=3)
        check_routing(a)
        assert torch.equal(a.grad_y, b.grad_y) and torch.equal(a.weight, b.weight)
        assert torch.equal(a.expanded_row_idx, b.expanded_row_idx)
        # distinct experts per token
        s = torch.sort(a.experts, dim=1).values
        assert (s[:, 1:] != s[:, :-1]).all()


def test_tiny_workload_has_expert_one_empty():
    w = WORKLOADS["tiny-fp32"]
    gen = torch.Generator()
    gen.manual_seed(w.seed)
    experts = route_experts(w, gen)
    _, _, gl = expanded_order(experts, w.G)
    assert int(gl[1]) == 0 and (gl[[0, 2, 3]] > 0).all() and int(gl.sum()) == 128


def test_zipf_workload_has_ten_empty_experts():
    w = WORKLOADS["skewed-fp16"]
    gen = torch.Generator()
    gen.manual_seed(w.seed)
    experts = route_experts(w, gen)
    gather, scatter, gl = expanded_order(experts, w.G)
    assert int((gl == 0).sum()) == 10
    assert int(gl.sum()) == w.M
    # skewed: the most popular expert gets far more than the mean
    assert int(gl.max()) > 4 * w.M // w.G
    assert torch.equal(scatter[gather], torch.arange(w.M))


def test_value_distributions():
    w = Workload("v", batch=512, top_k=4, G=4, K=64, N=128, dtype="bf16")
    from workloads import make_inputs
    inp = make_inputs(w)
    assert inp.grad_y.dtype == torch.bfloat16 and inp.grad_y.shape == (2048, 128)
    assert abs(float(inp.grad_y.float().std()) - 1.0) < 0.05
    assert abs(float(inp.weight.float().std()) - 0.02) < 0.002
    check_routing(inp)


def test_replacement_routing_allows_repeats():
    inp = make_case(batch=200, top_k=4, G=3, K=8, N=8, routing="replacement", dtype="fp32")
    check_routing(inp)
    s = torch.sort(inp.experts, dim=1).values
    assert (s[:, 1:] == s[:, :-1]).any()
