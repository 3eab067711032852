"""The C-ABI library builds, loads without a GPU, exports every declared entry
point, and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re

import pytest

import permute_grouped_gemm_gb300 as pgg
from permute_grouped_gemm_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return pgg.load()


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pgg_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert "pgg_dx_execute" in names and "pgg_dx_workspace_size" in names
    raw = ctypes.CDLL(pbuild.LIB)
    for n in names:
        assert hasattr(raw, n), n


def test_checked_build_compiles_loads_and_exports_every_declared_function():
    # the same sources with -DPGG_CHECKS (device bounds checks), in a library of its own
    path = pbuild.build(checks=True)
    assert path == pbuild.LIB_CHECKS and os.path.isfile(path) and path != pbuild.LIB
    raw = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(raw, n), n
    raw.pgg_status_string.argtypes = [ctypes.c_int]
    raw.pgg_status_string.restype = ctypes.c_char_p
    assert b"bounds check" in raw.pgg_status_string(20)
    assert pgg.STATUS[20] == "PGG_ERR_CHECK"


# large-config sizes (pages' scale): M = 108000, G = 60, K = 7168, N = 2048
LARGE = dict(M=108000, N=2048, K=7168, G=60, L=108000, batch=13500, topK=8)


def ws(**o):
    a = dict(LARGE, rowIdxType=0, dtype=pgg.PGG_BF16)
    a.update(o)
    return pgg.pgg_dx_workspace_size(a["M"], a["N"], a["K"], a["G"], a["L"], a["batch"],
                                     a["topK"], a["rowIdxType"], a["dtype"])


def code_of(**o):
    with pytest.raises(pgg.PggError) as e:
        ws(**o)
    return pgg.STATUS[e.value.code]


def test_workspace_is_small_and_independent_of_n(lib):
    w = ws()
    assert w <= 16 * 2**20
    assert ws(N=4096) == w            # no dependence on N
    assert ws(M=2048, L=2048, batch=256, G=256) < 256 * 1024  # skinny
    # grows with M (index tables) but never holds an [M, K] array
    assert w < LARGE["M"] * LARGE["K"] // 64


def test_host_errors(lib):
    assert code_of(L=107999) == "PGG_ERR_SHAPE"           # L != M
    assert code_of(batch=13499) == "PGG_ERR_SHAPE"        # M != batch * topK
    assert code_of(topK=0) == "PGG_ERR_ATTR"
    assert code_of(batch=0) == "PGG_ERR_ATTR"
    assert code_of(rowIdxType=2) == "PGG_ERR_ATTR"
    assert code_of(dtype=3) == "PGG_ERR_DTYPE"
    assert code_of(M=2**31, L=2**31, batch=2**28) == "PGG_ERR_SHAPE"
    assert code_of(K=0) == "PGG_ERR_SHAPE"
    assert code_of(G=0) == "PGG_ERR_SHAPE"


def test_execute_rejects_before_any_cuda_call(lib):
    # null pointers and a short workspace are reported without a GPU
    a = LARGE
    rc = pgg.pgg_dx_execute(0, 0, 0, 0, a["M"], a["N"], a["K"], a["G"], a["L"], a["batch"],
                            a["topK"], 0, pgg.PGG_BF16, 0, 0, 0, None)
    assert pgg.STATUS[rc] == "PGG_ERR_NULL"
    fake = 1 << 20  # aligned non-null addresses: never dereferenced on these paths
    need = ws()
    rc = pgg.pgg_dx_execute(fake, fake, fake, fake, a["M"], a["N"], a["K"], a["G"], a["L"],
                            a["batch"], a["topK"], 0, pgg.PGG_BF16, fake, need - 1, fake, None)
    assert pgg.STATUS[rc] == "PGG_ERR_WORKSPACE"
    # gradY and weight need element alignment, out 4 bytes, the workspace 256
    rc = pgg.pgg_dx_execute(fake + 1, fake, fake, fake, a["M"], a["N"], a["K"], a["G"], a["L"],
                            a["batch"], a["topK"], 0, pgg.PGG_BF16, fake, need, fake, None)
    assert pgg.STATUS[rc] == "PGG_ERR_ALIGN"
    rc = pgg.pgg_dx_execute(fake, fake + 2, fake, fake, a["M"], a["N"], a["K"], a["G"], a["L"],
                            a["batch"], a["topK"], 0, pgg.PGG_F32, fake, need, fake, None)
    assert pgg.STATUS[rc] == "PGG_ERR_ALIGN"
    rc = pgg.pgg_dx_execute(fake, fake, fake, fake, a["M"], a["N"], a["K"], a["G"], a["L"],
                            a["batch"], a["topK"], 0, pgg.PGG_BF16, fake, need, fake + 2, None)
    assert pgg.STATUS[rc] == "PGG_ERR_ALIGN"
    rc = pgg.pgg_dx_execute(fake, fake, fake, fake, a["M"], a["N"], a["K"], a["G"], a["L"],
                            a["batch"], a["topK"], 0, pgg.PGG_BF16, fake + 64, need, fake, None)
    assert pgg.STATUS[rc] == "PGG_ERR_ALIGN"
    rc = pgg.pgg_dx_route_prep(0, fake, a["M"], a["N"], a["K"], a["G"], a["L"], a["batch"],
                               a["topK"], 0, pgg.PGG_BF16, fake, need, None)
    assert pgg.STATUS[rc] == "PGG_ERR_NULL"


def test_every_compiled_configuration_fits_one_sm(lib):
    # each (dtype, variant) the plan can report asks for at most the 227 KB of
    # shared memory a CTA may use and at most 1024 threads
    sizes = (108000, 2048, 7168, 60, 108000, 13500, 8, 0)
    seen = set()
    try:
        for dt in (pgg.PGG_BF16, pgg.PGG_F16, pgg.PGG_F32):
            for v in (0, 1, 2, 3, 4, 5):
                pgg.pgg_debug_force_variant(v)
                for plan in (pgg.pgg_dx_plan, pgg.pgg_dw_plan, pgg.pgg_fwd_plan):
                    try:
                        p = plan(*sizes, dt)
                    except pgg.PggError as e:
                        # a variant that does not exist for this dtype is refused
                        assert pgg.STATUS[e.code] == "PGG_ERR_DTYPE", (plan.__name__, dt, v)
                        continue
                    seen.add((plan.__name__, dt, p["variant"]))
                    assert 0 < p["smem_bytes"] <= 227 * 1024, (plan.__name__, dt, v, p)
                    assert 0 < p["threads"] <= 1024 and p["threads"] % 32 == 0, \
                        (plan.__name__, dt, v, p)
    finally:
        pgg.pgg_debug_force_variant(-1)
    assert len(seen) >= 10


def test_plan_variants(lib):
    big = pgg.pgg_dx_plan(108000, 2048, 7168, 60, 108000, 13500, 8, 0, pgg.PGG_BF16)
    skinny = pgg.pgg_dx_plan(2048, 2048, 7168, 256, 2048, 256, 8, 0, pgg.PGG_BF16)
    assert big["variant"] == 0 and big["rows_per_block"] == 256 and big["k_blocks"] == 56
    assert skinny["variant"] == 1 and skinny["rows_per_block"] == 32
    for p in (big, skinny):
        assert p["smem_bytes"] <= 227 * 1024
        assert p["k_per_block"] == 128
    pgg.pgg_debug_force_variant(1)
    try:
        assert pgg.pgg_dx_plan(108000, 2048, 7168, 60, 108000, 13500, 8, 0,
                               pgg.PGG_BF16)["variant"] == 1
    finally:
        pgg.pgg_debug_force_variant(-1)


def test_owner_plan(lib):
    # few experts per token: the owner variant, slabs of T = 112 G / topK tokens
    # rounded down to 32 (at most 224: tensor-memory columns 480-511 stay free),
    # 256 threads (two TMA warps, two MMA-issuing warps, four epilogue warps)
    uni = pgg.pgg_dx_plan(32768, 1024, 2048, 16, 32768, 4096, 8, 0, pgg.PGG_BF16)
    assert uni["variant"] == 4 and uni["rows_per_block"] == 224
    assert uni["threads"] == 256 and uni["cta_pair"] == 1 and uni["stages"] == 4
    assert uni["smem_bytes"] <= 227 * 1024
    # 112 G > 224 topK: the ticketed kernel, unless forced; forced, the slab is capped
    wide = pgg.pgg_dx_plan(16000, 256, 2048, 40, 16000, 8000, 2, 0, pgg.PGG_BF16)
    assert wide["variant"] == 0
    pgg.pgg_debug_force_variant(4)
    try:
        p = pgg.pgg_dx_plan(16000, 256, 2048, 40, 16000, 8000, 2, 0, pgg.PGG_BF16)
        assert p["variant"] == 4 and p["rows_per_block"] == 224
        # N not a multiple of 64: one-panel stages, eight of them
        p = pgg.pgg_dx_plan(32768, 1000, 2048, 16, 32768, 4096, 8, 0, pgg.PGG_F16)
        assert p["variant"] == 4 and p["stages"] == 8 and p["smem_bytes"] <= 227 * 1024
        # fp32 never takes the owner variant
        assert pgg.pgg_dx_plan(32768, 1024, 2048, 16, 32768, 4096, 8, 0, pgg.PGG_F32)["variant"] == 0
    finally:
        pgg.pgg_debug_force_variant(-1)


def test_status_strings(lib):
    for code, name in pgg.STATUS.items():
        assert pgg.pgg_status_string(code) != "unknown status", name


def test_rows_the_tma_cannot_stream_take_the_gather_warps_or_the_fp32_pipes(lib):
    # row bytes N * sizeof(dtype) not a multiple of 16 (the page's N = 1 and
    # N = 286 white-box cases): 16-bit rows of an even length are copied by the
    # gather warps of variant 5 (tensor cores); odd lengths and fp32 plan the
    # FP32-pipe kernel; never an error
    for n, dt in ((286, pgg.PGG_BF16), (2046, pgg.PGG_F16), (2, pgg.PGG_BF16)):
        p = pgg.pgg_dx_plan(1280, n, 178, 4, 1280, 640, 2, 0, dt)
        assert p["variant"] == 5 and p["rows_per_block"] == 256 and p["cta_pair"] == 1, (n, dt)
        assert p["threads"] == 704 and p["smem_bytes"] <= 227 * 1024, (n, dt)
    for n, dt in ((1, pgg.PGG_BF16), (287, pgg.PGG_BF16), (2047, pgg.PGG_F16), (6, pgg.PGG_F32),
                  (1, pgg.PGG_F32)):
        p = pgg.pgg_dx_plan(1280, n, 178, 4, 1280, 640, 2, 0, dt)
        assert p["variant"] == 3 and p["rows_per_block"] == 64 and p["threads"] == 128, (n, dt)
        assert p["cta_pair"] == 0 and p["smem_bytes"] <= 227 * 1024 // 3  # 3 CTAs per SM
    # forcing variant 5 where it cannot copy the rows gives the FP32-pipe kernel
    pgg.pgg_debug_force_variant(5)
    try:
        assert pgg.pgg_dx_plan(1280, 287, 178, 4, 1280, 640, 2, 0, pgg.PGG_BF16)["variant"] == 3
        assert pgg.pgg_dx_plan(1280, 288, 178, 4, 1280, 640, 2, 0, pgg.PGG_F32)["variant"] == 3
        assert pgg.pgg_dx_plan(1280, 288, 178, 4, 1280, 640, 2, 0, pgg.PGG_BF16)["variant"] == 5
    finally:
        pgg.pgg_debug_force_variant(-1)
    for n, dt in ((8, pgg.PGG_BF16), (4, pgg.PGG_F32), (280, pgg.PGG_F16)):
        assert pgg.pgg_dx_plan(1280, n, 178, 4, 1280, 640, 2, 0, dt)["variant"] != 3, (n, dt)
    # the workspace stays small at the pages' scale
    assert ws(N=2047) <= 16 * 2**20
    assert ws(N=2047) < LARGE["M"] * LARGE["K"] // 64


def test_weight_gradient_plan_and_host_errors(lib):
    a = LARGE
    sizes = (a["M"], a["N"], a["K"], a["G"], a["L"], a["batch"], a["topK"], 0)
    p = pgg.pgg_dw_plan(*sizes, pgg.PGG_BF16)
    assert p["variant"] == 0 and p["k_per_block"] == 256 and p["threads"] % 32 == 0
    assert p["cta_pair"] == 1 and p["stages"] == 6 and p["threads"] == 16 * 32
    assert p["k_blocks"] == 28 and p["band_k_blocks"] == 8 and p["smem_bytes"] <= 227 * 1024
    assert pgg.pgg_dw_plan(*sizes, pgg.PGG_F32)["variant"] == 3
    assert pgg.pgg_dw_plan(a["M"], 286, 178, a["G"], a["L"], a["batch"], a["topK"], 0,
                           pgg.PGG_BF16)["variant"] == 3
    # d_y rows of 572 bytes, x rows of 384: d_y gathered by warps (variant 5)
    assert pgg.pgg_dw_plan(a["M"], 286, 192, a["G"], a["L"], a["batch"], a["topK"], 0,
                           pgg.PGG_BF16)["variant"] == 5
    assert pgg.pgg_dw_plan(a["M"], 287, 192, a["G"], a["L"], a["batch"], a["topK"], 0,
                           pgg.PGG_BF16)["variant"] == 3
    assert pgg.pgg_dw_workspace_size(*sizes, pgg.PGG_BF16) == ws()
    fake = 1 << 20
    need = ws()
    args = (fake, fake, fake, fake, *sizes[:-1], 0, pgg.PGG_BF16)
    assert pgg.STATUS[pgg.pgg_dw_execute(*args, pgg.PGG_F16, fake, need, fake, None)] == \
        "PGG_ERR_DTYPE"
    assert pgg.STATUS[pgg.pgg_dw_execute(*args, pgg.PGG_BF16, fake, need - 1, fake, None)] == \
        "PGG_ERR_WORKSPACE"
    assert pgg.STATUS[pgg.pgg_dw_execute(*args, pgg.PGG_BF16, fake, need, 0, None)] == \
        "PGG_ERR_NULL"
    assert pgg.STATUS[pgg.pgg_dw_execute(*args, pgg.PGG_F32, fake, need, fake + 2, None)] == \
        "PGG_ERR_ALIGN"
    assert pgg.STATUS[pgg.pgg_dw_execute(fake + 1, *args[1:], pgg.PGG_BF16, fake, need, fake,
                                         None)] == "PGG_ERR_ALIGN"


def test_forward_plan_and_host_errors(lib):
    a = LARGE
    sizes = (a["M"], a["N"], a["K"], a["G"], a["L"], a["batch"], a["topK"], 0)
    p = pgg.pgg_fwd_plan(*sizes, pgg.PGG_BF16)
    assert p["variant"] == 0 and p["rows_per_block"] == 256 and p["cta_pair"] == 1
    assert p["k_per_block"] == 64 and p["k_blocks"] == 112 and p["band_k_blocks"] == 8
    assert p["smem_bytes"] <= 227 * 1024 and p["stages"] == 7 and p["threads"] == 13 * 32
    assert pgg.pgg_fwd_plan(*sizes, pgg.PGG_F32)["variant"] == 3
    # the gather warps hold an x row's offset in 16-byte units in 32 bits: x of
    # 64 GiB or more (batch x K / 8 >= 2^32 - 1) takes the FP32-pipe kernel
    for batch, want in ((2**22 - 1, 0), (2**22, 3)):
        assert pgg.pgg_fwd_plan(batch, 256, 8192, 1, batch, batch, 1, 0,
                                pgg.PGG_BF16)["variant"] == want, batch
    assert pgg.pgg_fwd_plan(a["M"], 286, 178, a["G"], a["L"], a["batch"], a["topK"], 0,
                            pgg.PGG_BF16)["variant"] == 3
    # weight and y rows of 572 bytes, x rows of 384: weight gathered by warps (variant 5)
    assert pgg.pgg_fwd_plan(a["M"], 286, 192, a["G"], a["L"], a["batch"], a["topK"], 0,
                            pgg.PGG_BF16)["variant"] == 5
    assert pgg.pgg_fwd_plan(a["M"], 287, 192, a["G"], a["L"], a["batch"], a["topK"], 0,
                            pgg.PGG_BF16)["variant"] == 3
    need = pgg.pgg_fwd_workspace_size(*sizes, pgg.PGG_BF16)
    assert need <= 16 * 2**20
    fake = 1 << 20
    args = (fake, fake, fake, fake, *sizes[:-1], 0, pgg.PGG_BF16)
    assert pgg.STATUS[pgg.pgg_fwd_execute(*args, pgg.PGG_F16, fake, need, fake, None)] == \
        "PGG_ERR_DTYPE"
    assert pgg.STATUS[pgg.pgg_fwd_execute(*args, pgg.PGG_BF16, fake, need - 1, fake, None)] == \
        "PGG_ERR_WORKSPACE"
    assert pgg.STATUS[pgg.pgg_fwd_execute(*args, pgg.PGG_BF16, fake, need, 0, None)] == \
        "PGG_ERR_NULL"
    assert pgg.STATUS[pgg.pgg_fwd_execute(fake + 1, *args[1:], pgg.PGG_BF16, fake, need, fake,
                                          None)] == "PGG_ERR_ALIGN"


def test_unpermute_grad_host_errors(lib):
    assert pgg.pgg_unpermute_grad_workspace_size(108000, 13500, 8) == 256 + 432128  # 4 M, 256-aligned
    with pytest.raises(pgg.PggError):
        pgg.pgg_unpermute_grad_workspace_size(108000, 13499, 8)
    fake = 1 << 20
    need = pgg.pgg_unpermute_grad_workspace_size(1000, 250, 4)
    base = dict(permuted=fake, d_out=fake, probs=fake, expandedRowIdx=fake, M=1000, H=512,
                batch=250, topK=4, rowIdxType=0, dtype=pgg.PGG_BF16,
                probs_grad_dtype=pgg.PGG_BF16, workspace=fake, workspace_bytes=need,
                perm_grad=fake, probs_grad=fake, stream=None)

    def code(**o):
        a = dict(base, **o)
        return pgg.STATUS[pgg.pgg_unpermute_grad(**a)]

    assert code(probs_grad_dtype=pgg.PGG_F16) == "PGG_ERR_DTYPE"
    assert code(workspace_bytes=need - 1) == "PGG_ERR_WORKSPACE"
    assert code(probs_grad=0) == "PGG_ERR_NULL"
    assert code(d_out=fake + 1) == "PGG_ERR_ALIGN"
    assert code(rowIdxType=2) == "PGG_ERR_ATTR"
    assert code(M=999) == "PGG_ERR_SHAPE"


def test_unpermute_grad_two_stage_host_errors(lib):
    fake = 1 << 20
    need = pgg.pgg_unpermute_grad_workspace_size(1000, 250, 4)
    prep = dict(expandedRowIdx=fake, M=1000, batch=250, topK=4, rowIdxType=0, workspace=fake,
                workspace_bytes=need, stream=None)

    def prep_code(**o):
        return pgg.STATUS[pgg.pgg_unpermute_grad_prep(**dict(prep, **o))]

    assert prep_code(expandedRowIdx=0) == "PGG_ERR_NULL"
    assert prep_code(workspace_bytes=need - 1) == "PGG_ERR_WORKSPACE"
    assert prep_code(rowIdxType=2) == "PGG_ERR_ATTR"
    assert prep_code(M=999) == "PGG_ERR_SHAPE"
    assert prep_code(workspace=fake + 128) == "PGG_ERR_ALIGN"
    apply = dict(permuted=fake, d_out=fake, probs=fake, expandedRowIdx=fake, M=1000, H=512,
                 batch=250, topK=4, rowIdxType=0, dtype=pgg.PGG_BF16,
                 probs_grad_dtype=pgg.PGG_BF16, workspace=fake, workspace_bytes=need,
                 perm_grad=fake, probs_grad=fake, stream=None)

    def apply_code(**o):
        return pgg.STATUS[pgg.pgg_unpermute_grad_apply(**dict(apply, **o))]

    assert apply_code(probs_grad_dtype=pgg.PGG_F16) == "PGG_ERR_DTYPE"
    assert apply_code(workspace_bytes=need - 1) == "PGG_ERR_WORKSPACE"
    assert apply_code(probs_grad=0) == "PGG_ERR_NULL"
    assert apply_code(perm_grad=fake + 1) == "PGG_ERR_ALIGN"
    assert apply_code(H=0) == "PGG_ERR_SHAPE"
