"""Plausible mistakes planted in copies of the oracle source are caught.

Each mutant is the oracle's C++ source with one edit (a dropped term, a wrong
index, a transposed operand, swapped index forms, a wrong exponent bias, in
the input gradient, the weight gradient, the forward or the probs-weighted
unpermute backward),
compiled to a temporary library on the CPU. The check fails if any mutant
passes every pin below, i.e. if the pins could not tell it from the real
oracle. Every mutant keeps all memory accesses in bounds.
"""

import os
import subprocess

import numpy as np
import pytest

import oracle
from workloads import make_case

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle_dx.cpp")

MUTANTS = {
    "drop_last_topk_term": ("for (int64_t j = 0; j < job.topK; ++j) {\n      const int64_t i = job.routing->row_of_pos[b * job.topK + j];",
                            "for (int64_t j = 0; j < job.topK - 1; ++j) {\n      const int64_t i = job.routing->row_of_pos[b * job.topK + j];"),
    "j_major_original_position": ("row_of_pos[b * job.topK + j]",
                                  "row_of_pos[b + j * static_cast<int64_t>("
                                  "job.routing->row_of_pos.size() / job.topK)]"),
    "transposed_weight": ("const int64_t wbase = (g * K + k) * N;\n        double s = 0.0;\n"
                          "        for (int64_t n = 0; n < N; ++n) s += dy_row[n] * job.dec->at(job.w, wbase + n);",
                          "const int64_t wbase = g * K * N;\n        double s = 0.0;\n"
                          "        for (int64_t n = 0; n < N; ++n) s += dy_row[n] * "
                          "job.dec->at(job.w, wbase + (n * K + k) % (K * N));"),
    "swapped_index_forms": ("if (row_idx_type == 0) {", "if (row_idx_type == 1) {"),
    "group_off_by_one": ("r->group_of_row[i++] = g;", "r->group_of_row[i++] = (g + 1) % G;"),
    "fp16_exponent_bias": ("e - 25", "e - 24"),
    "bf16_wrong_half": ("static_cast<uint32_t>(h) << 16;", "static_cast<uint32_t>(h) << 15;"),
    # weight gradient
    "dw_drop_last_row": ("i < job.routing->first_row[g + 1]; ++i)",
                         "i + 1 < job.routing->first_row[g + 1]; ++i)"),
    "dw_rows_from_start": ("for (int64_t i = job.routing->first_row[g];",
                           "for (int64_t i = 0;"),
    "dw_token_of_row_not_position": ("const int64_t b = job.routing->pos_of_row[i] / job.topK;\n      const double xv",
                                     "const int64_t b = i / job.topK;\n      const double xv"),
    "dw_k_n_swapped_in_x": ("const double xv = job.dec->at(job.x, b * K + k);",
                            "const double xv = job.dec->at(job.x, b * K + (K - 1 - k));"),
    # forward
    "fwd_transposed_weight": ("acc += x_row[k] * job.dec->at(job.w, (g * K + k) * N + n);",
                              "acc += x_row[k] * job.dec->at(job.w, (g * K + n) * N + k);"),
    "fwd_group_of_previous_row": ("    const int64_t g = job.routing->group_of_row[i];\n    for (int64_t k = 0; k < K; ++k) x_row[k]",
                                  "    const int64_t g = job.routing->group_of_row[i > 0 ? i - 1 : 0];\n    for (int64_t k = 0; k < K; ++k) x_row[k]"),
    "fwd_token_of_row_not_position": ("const int64_t b = job.routing->pos_of_row[i] / job.topK;\n    const int64_t g",
                                      "const int64_t b = i / job.topK;\n    const int64_t g"),
    "unperm_prob_of_first_j": ("const double pr = job.probs ? job.dec->at(job.probs, p) : 1.0;",
                               "const double pr = job.probs ? job.dec->at(job.probs, b * job.topK) : 1.0;"),
    "unperm_dot_drops_last_h": ("if (job.probs) dot += d[h] * job.dec->at(job.perm, i * H + h);",
                                "if (job.probs && h + 1 < H) dot += d[h] * job.dec->at(job.perm, i * H + h);"),
    "unperm_maps_confused": ("const int64_t i = job.routing->row_of_pos[p];",
                             "const int64_t i = job.routing->pos_of_row[p];"),
    "fwd_drop_last_k": ("for (int64_t k = 0; k < K; ++k) acc += x_row[k]",
                        "for (int64_t k = 0; k < K - 1; ++k) acc += x_row[k]"),
}


def build_mutant(tmp_path, name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / f"{name}.cpp"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread",
                           str(path), "-o", str(lib)])
    return oracle.load_library(str(lib))


def pins_pass(lib) -> bool:
    from test_oracle_pins import brute_force, unfused_numpy, rel_err
    from test_oracle_dw_pins import brute_force_dw
    from test_oracle_fwd_pins import brute_force_fwd
    from test_oracle_unperm_pins import brute as brute_unperm
    from workloads.moe import unpermute_inputs
    from workloads.moe import forward_input
    # decoders against numpy / torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref16 = bits.view(np.float16).astype(np.float64)
    got16 = oracle.decode(bits, oracle.F16, lib=lib)
    fin = np.isfinite(ref16)
    if not np.array_equal(got16[fin], ref16[fin]):
        return False
    import torch
    refb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    gotb = oracle.decode(bits, oracle.BF16, lib=lib)
    fin = np.isfinite(refb)
    if not np.array_equal(gotb[fin], refb[fin]):
        return False
    # brute force and unfused form, both index forms, K == N so that a
    # transposed weight stays in bounds
    for rit in (0, 1):
        for dt in ("fp32", "fp16"):
            inp = make_case(batch=5, top_k=3, G=3, K=6, N=6, dtype=dt, seed=21, row_idx_type=rit)
            try:
                got = oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list,
                                inp.batch, inp.top_k, rit, lib=lib)
            except oracle.OracleError:
                return False
            if rel_err(got, brute_force(inp)) > 1e-12:
                return False
            if rel_err(got, unfused_numpy(inp)[0]) > 1e-12:
                return False
            # weight gradient against its brute force
            x = forward_input(inp)
            try:
                gw = oracle.dw(x, inp.grad_y, inp.expanded_row_idx, inp.group_list, inp.batch,
                               inp.top_k, rit, lib=lib)
            except oracle.OracleError:
                return False
            if rel_err(gw, brute_force_dw(inp, x)) > 1e-12:
                return False
            # forward against its brute force
            try:
                y = oracle.fwd(x, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                               inp.top_k, rit, lib=lib)
            except oracle.OracleError:
                return False
            if rel_err(y, brute_force_fwd(inp, x)) > 1e-12:
                return False
            # probs-weighted unpermute backward against its brute force
            d_out, probs = unpermute_inputs(inp)
            try:
                pg, qg = oracle.unpermute_grad(inp.grad_y, d_out, probs, inp.expanded_row_idx,
                                               inp.batch, inp.top_k, rit, lib=lib)
            except oracle.OracleError:
                return False
            bpg, bqg = brute_unperm(inp, d_out, probs)
            if rel_err(pg, bpg) > 1e-12 or rel_err(qg, bqg) > 1e-12:
                return False
    return True


def test_real_oracle_passes_the_pins(oracle_lib):
    assert pins_pass(oracle._load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    assert not pins_pass(build_mutant(tmp_path, name))
