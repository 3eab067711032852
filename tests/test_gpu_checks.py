"""The checked build (libpgg_checks.so: the same sources compiled with
-DPGG_CHECKS) on the GPU.

Its kernels check every index they read from the routing tables (row blocks,
row records, slab bounds, the unpermute index) against the table's bounds; a
failed check writes PGG_ERR_CHECK to the status word (the check's site to the
diagnostic word after it) and keeps the access in bounds, so nothing traps or
hangs. The checks run in a child process that loads the checked library in
place of libpgg.so:

1. every kernel path (ticketed pair, narrow and FP32-pipe d_x kernels, the
   owner kernel, the weight-gradient and forward kernels on the tensor cores
   and on the FP32 pipes, the unpermute backward) gives status 0 and matches
   the fp64 oracle within the tolerance of the other parity tests;
2. a routing table corrupted on purpose between the two stages of the call
   (a row block's expert, a row's token, a slab bound: values the routing step
   never writes) is caught by the check at its site, and the next clean call
   on the same context is correct again.
"""

import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
import oracle
import permute_grouped_gemm_gb300 as pgg
from permute_grouped_gemm_gb300 import build as pbuild
from workloads import make_case
from workloads.moe import forward_input, unpermute_inputs

pgg.load(pbuild.LIB_CHECKS)
oracle.build()
res = {}

def rel(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))

def dx_case(name, variant, **kw):
    inp = make_case(device="cuda", **kw)
    pgg.pgg_debug_force_variant(variant)
    try:
        out, ws = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list,
                         inp.batch, inp.top_k, inp.row_idx_type)
        torch.cuda.synchronize()
    finally:
        pgg.pgg_debug_force_variant(-1)
    ref = oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                    inp.top_k, inp.row_idx_type)
    res[name] = [pgg.status(ws), rel(out.double().cpu().numpy(), ref)]

dx_case("dx_pair", 0, batch=300, top_k=4, G=7, K=400, N=320, dtype="bf16", seed=61)
dx_case("dx_narrow", 1, batch=300, top_k=4, G=7, K=400, N=320, dtype="fp16", seed=62,
        row_idx_type=1)
dx_case("dx_fp32", 0, batch=200, top_k=3, G=5, K=200, N=96, dtype="fp32", seed=63)
dx_case("dx_simt", 3, batch=300, top_k=4, G=7, K=400, N=286, dtype="bf16", seed=64)
dx_case("dx_owner", 4, batch=1024, top_k=8, G=16, K=512, N=256, dtype="bf16", seed=65)

for name, variant, n in (("dw_tensor", -1, 256), ("dw_simt", 3, 286)):
    inp = make_case(batch=300, top_k=4, G=7, K=192, N=n, dtype="bf16", seed=66, device="cuda")
    x = forward_input(inp)
    pgg.pgg_debug_force_variant(variant)
    try:
        out, ws = pgg.dw(x, inp.grad_y, inp.expanded_row_idx, inp.group_list, inp.batch,
                         inp.top_k, inp.row_idx_type, out_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        pgg.pgg_debug_force_variant(-1)
    ref = oracle.dw(x, inp.grad_y, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k,
                    inp.row_idx_type)
    res[name] = [pgg.status(ws), rel(out.double().cpu().numpy(), ref)]

for name, variant, n in (("fwd_tensor", -1, 256), ("fwd_simt", 3, 286)):
    inp = make_case(batch=300, top_k=4, G=7, K=192, N=n, dtype="bf16", seed=67, device="cuda")
    x = forward_input(inp)
    pgg.pgg_debug_force_variant(variant)
    try:
        y, ws = pgg.fwd(x, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                        inp.top_k, inp.row_idx_type, out_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        pgg.pgg_debug_force_variant(-1)
    ref = oracle.fwd(x, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch, inp.top_k,
                     inp.row_idx_type)
    res[name] = [pgg.status(ws), rel(y.double().cpu().numpy(), ref)]

inp = make_case(batch=300, top_k=4, G=7, K=16, N=320, dtype="fp32", seed=68, row_idx_type=1,
                device="cuda")
d_out, probs = unpermute_inputs(inp)
pg, qg, ws = pgg.unpermute_grad(inp.grad_y, d_out, probs, inp.expanded_row_idx, inp.top_k,
                                inp.row_idx_type, probs_grad_dtype=torch.float32)
torch.cuda.synchronize()
rpg, rqg = oracle.unpermute_grad(inp.grad_y, d_out, probs, inp.expanded_row_idx, inp.batch,
                                 inp.top_k, inp.row_idx_type)
res["unperm"] = [pgg.status(ws), max(rel(pg.double().cpu().numpy(), rpg),
                                     rel(qg.double().cpu().numpy(), rqg))]

# --- routing tables corrupted between the two stages of the d_x call

def layout(M, G, batch, plan, n_slabs):
    # the workspace sections of the d_x call, each 256-byte aligned
    at = [0]
    def take(n):
        o = at[0]
        at[0] = (at[0] + n + 255) // 256 * 256
        return o
    L = {}
    L["hdr"] = take(64)
    L["off"] = take(8 * (G + 1))
    L["rbstart"] = take(4 * (G + 1))
    L["rblist"] = take(16 * plan["max_row_blocks"])
    L["inv"] = take(4 * M)
    L["rowinfo"] = take(8 * M)
    L["tickets"] = take(4 * ((batch * plan["k_blocks"] + 3) // 4 * 4))
    L["seg"] = take(4 * G * (n_slabs + 1))
    L["total"] = at[0]
    return L

def corrupted(name, variant, section, word, value, **kw):
    inp = make_case(device="cuda", **kw)
    w = inp.workload
    sizes = (w.M, w.N, w.K, w.G, w.M, w.batch, w.top_k)
    dt = pgg.dtype_code(inp.grad_y.dtype)
    pgg.pgg_debug_force_variant(variant)
    try:
        plan = pgg.pgg_dx_plan(*sizes, w.row_idx_type, dt)
        need = pgg.pgg_dx_workspace_size(*sizes, w.row_idx_type, dt)
        n_slabs = -(-w.batch // plan["rows_per_block"]) if plan["variant"] == 4 else 0
        L = layout(w.M, w.G, w.batch, plan, n_slabs)
        assert L["total"] == need, (L["total"], need)
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        out = torch.empty(w.batch, w.K, dtype=torch.float32, device="cuda")
        sp = torch.cuda.current_stream().cuda_stream
        pgg.pgg_debug_set_wait_limit_ns(200_000_000)
        rc = pgg.pgg_dx_route_prep(inp.expanded_row_idx.data_ptr(), inp.group_list.data_ptr(),
                                   *sizes, w.row_idx_type, dt, ws.data_ptr(), need, sp)
        assert rc == 0
        torch.cuda.synchronize()
        assert pgg.status(ws) == 0
        # one 32-bit word of the section, a value the routing step never writes
        ws[L[section]:L[section] + need - L[section]].view(torch.int32)[word] = value
        rc = pgg.pgg_dx_grouped_gemm(inp.grad_y.data_ptr(), inp.weight.data_ptr(),
                                     inp.expanded_row_idx.data_ptr(), inp.group_list.data_ptr(),
                                     *sizes, w.row_idx_type, dt, ws.data_ptr(), need,
                                     out.data_ptr(), sp)
        assert rc == 0
        torch.cuda.synchronize()
        words = ws[:16].view(torch.int32).cpu().tolist()
    finally:
        pgg.pgg_debug_set_wait_limit_ns(0)
        pgg.pgg_debug_force_variant(-1)
    # a clean call afterwards on the same context
    out2, ws2 = pgg.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                       inp.top_k, inp.row_idx_type)
    torch.cuda.synchronize()
    ref = oracle.dx(inp.grad_y, inp.weight, inp.expanded_row_idx, inp.group_list, inp.batch,
                    inp.top_k, inp.row_idx_type)
    res[name] = [words[0], words[3], pgg.status(ws2), rel(out2.double().cpu().numpy(), ref)]

case = dict(batch=300, top_k=4, G=7, K=400, N=320, dtype="bf16", seed=69)
# the expert of row block 0 (word 0 of the list)
corrupted("bad_row_block", 0, "rblist", 0, 1 << 20, **case)
# the token of expanded row 5 (word 10 of the row records: {token, rank} pairs)
corrupted("bad_token", 0, "rowinfo", 10, 1 << 30, **case)
# the first slab bound of expert 0 in the owner kernel's table
corrupted("bad_slab_bound", 4, "seg", 0, 1 << 30, batch=1024, top_k=8, G=16, K=512, N=256,
          dtype="bf16", seed=70)
print(json.dumps(res))
"""

CLEAN = ["dx_pair", "dx_narrow", "dx_fp32", "dx_simt", "dx_owner", "dw_tensor", "dw_simt",
         "fwd_tensor", "fwd_simt", "unperm"]
# corruption -> the site of the check that must catch it
SITES = {"bad_row_block": 41, "bad_token": 43, "bad_slab_bound": 30}
PGG_ERR_CHECK = 20
TOL = 1e-4


@pytest.fixture(scope="module")
def results():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from permute_grouped_gemm_gb300 import build as pbuild
    pbuild.build(checks=True)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("name", CLEAN)
def test_checked_build_runs_clean_and_matches_the_oracle(results, name):
    status, err = results[name]
    assert status == 0, f"{name}: status {status}"
    assert err <= TOL, f"{name}: max|diff| / max|ref| = {err:.3e}"


@pytest.mark.parametrize("name", sorted(SITES))
def test_checked_build_catches_a_corrupted_table(results, name):
    status, site, clean_status, clean_err = results[name]
    assert status == PGG_ERR_CHECK, f"{name}: status {status}"
    assert site == SITES[name], f"{name}: caught at site {site}"
    assert clean_status == 0 and clean_err <= TOL
