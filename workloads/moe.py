"""Seeded input recipes for the MoE permute + grouped-matmul backward.

Recipe (the same for every workload, seed 0 unless stated):

1. Routing. Each token b picks ``top_k`` experts:
   * ``uniform``: ``top_k`` distinct experts uniformly at random (argsort of
     uniform noise over the allowed experts); experts listed in ``empty``
     are never chosen.
   * ``zipf``: expert popularity w_r = r^-s over popularity ranks r = 1..G,
     with the ``zipf_zero`` least popular ranks set to weight 0 (so exactly
     that many experts receive no rows); ranks map to expert ids through a
     seeded permutation; ``top_k`` distinct experts per token are drawn
     without replacement in proportion to w.
   * ``replacement``: ``top_k`` experts uniformly with replacement (a token
     may pick the same expert twice; a degenerate routing kept for tests).
2. Expanded order. The pairs (expert, p) with original position
   p = b * top_k + j are sorted by expert, then by p. Row i of the sorted list
   has ``gather[i] = p`` (rowIdxType 0 form); the scatter form (rowIdxType 1)
   is its inverse, ``scatter[p] = i``. groupList[g] is the number of rows of
   expert g (counts, not a cumulative sum).
3. Values. d_y ~ N(0, 1) with shape [M, N] in expanded order and
   weight ~ N(0, w_std^2) with shape [G, K, N], drawn in fp32 and rounded to
   the workload dtype (round to nearest even). The weight is drawn one
   expert at a time so that the fp32 staging stays small. For the weight
   gradient, the forward input x ~ N(0, 1) with shape [batch, K] (seed + 2,
   ``forward_input``).
4. Unpermute backward (``unpermute_inputs``): grad_y [M, N] stands for the
   expert outputs being combined; d_out ~ N(0, 1) with shape [batch, N]
   (seed + 3); probs uniform in (0, 1] plus 1e-3, normalised per token
   (seed + 4); both rounded to the workload dtype.

The pages' shapes: M ~ 108K expanded tokens, K = 7168, G = 60, N = 2048
("MoeInitRoutingGroupedMatmulGrad design", section 1.2 and the d_weight
memory example). No public dataset is involved.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    top_k: int
    G: int
    K: int
    N: int
    dtype: str
    routing: str = "uniform"
    row_idx_type: int = 0
    seed: int = 0
    w_std: float = 0.02
    zipf_s: float = 1.2
    zipf_zero: int = 0
    empty: tuple = field(default_factory=tuple)

    @property
    def M(self) -> int:
        return self.batch * self.top_k

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def describe(self) -> dict:
        return {
            "workload": self.name, "batch": self.batch, "topK": self.top_k, "M": self.M,
            "G": self.G, "K": self.K, "N": self.N, "dtype": self.dtype,
            "routing": self.routing, "rowIdxType": self.row_idx_type, "seed": self.seed,
        }


# The workloads the benchmarks and full-size parity tests run.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny-fp32", batch=64, top_k=2, G=4, K=128, N=64, dtype="fp32",
                 routing="uniform", empty=(1,)),
        Workload("uniform-bf16", batch=4096, top_k=8, G=16, K=2048, N=1024, dtype="bf16"),
        Workload("skewed-fp16", batch=8192, top_k=8, G=64, K=4096, N=1536, dtype="fp16",
                 routing="zipf", zipf_s=1.2, zipf_zero=10, row_idx_type=1),
        Workload("large-bf16", batch=13500, top_k=8, G=60, K=7168, N=2048, dtype="bf16"),
        Workload("skinny-bf16", batch=256, top_k=8, G=256, K=7168, N=2048, dtype="bf16"),
        # rows of 2044 bytes (not a multiple of 16): the FP32-pipe kernel
        Workload("unaligned-bf16", batch=4096, top_k=8, G=16, K=2048, N=1022, dtype="bf16"),
    ]
}


@dataclass
class Inputs:
    workload: Workload
    grad_y: torch.Tensor          # [M, N] dtype, expanded order
    weight: torch.Tensor          # [G, K, N] dtype
    expanded_row_idx: torch.Tensor  # int64 [M], in the workload's rowIdxType form
    group_list: torch.Tensor      # int64 [G] counts
    experts: torch.Tensor         # int64 [batch, top_k] expert chosen by (b, j)
    gather: torch.Tensor          # int64 [M]: original position of expanded row i

    @property
    def batch(self):
        return self.workload.batch

    @property
    def top_k(self):
        return self.workload.top_k

    @property
    def row_idx_type(self):
        return self.workload.row_idx_type

    def to(self, device) -> "Inputs":
        return Inputs(self.workload, self.grad_y.to(device), self.weight.to(device),
                      self.expanded_row_idx.to(device), self.group_list.to(device),
                      self.experts, self.gather)


def route_experts(w: Workload, gen: torch.Generator) -> torch.Tensor:
    """[batch, top_k] int64 expert ids, drawn on the CPU generator ``gen``."""
    B, T, G = w.batch, w.top_k, w.G
    if w.routing == "uniform":
        allowed = torch.tensor([e for e in range(G) if e not in set(w.empty)], dtype=torch.int64)
        if T > allowed.numel():
            raise ValueError("top_k larger than the number of allowed experts")
        noise = torch.rand(B, allowed.numel(), generator=gen)
        return allowed[noise.argsort(dim=1)[:, :T]]
    if w.routing == "zipf":
        ranks = torch.arange(1, G + 1, dtype=torch.float64)
        pop = ranks.pow(-w.zipf_s)
        if w.zipf_zero:
            pop[G - w.zipf_zero:] = 0.0
        perm = torch.randperm(G, generator=gen)  # popularity rank r -> expert perm[r]
        weight = torch.empty(G, dtype=torch.float64)
        weight[perm] = pop
        for e in w.empty:
            weight[e] = 0.0
        return torch.multinomial(weight.expand(B, G), T, replacement=False, generator=gen)
    if w.routing == "replacement":
        return torch.randint(0, G, (B, T), generator=gen)
    raise ValueError(f"unknown routing {w.routing!r}")


def expanded_order(experts: torch.Tensor, G: int):
    """(gather [M], scatter [M], group_list [G]) for the stable (expert, p) sort."""
    B, T = experts.shape
    M = B * T
    flat = experts.reshape(-1).to(torch.int64)
    pos = torch.arange(M, dtype=torch.int64)
    key = flat * M + pos
    gather = torch.argsort(key)  # unique keys: the sort is stable by construction
    scatter = torch.empty(M, dtype=torch.int64)
    scatter[gather] = torch.arange(M, dtype=torch.int64)
    group_list = torch.bincount(flat, minlength=G).to(torch.int64)
    return gather, scatter, group_list


def _values(w: Workload, device, seed: int):
    dt = DTYPES[w.dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 1)
    dy = torch.randn(w.M, w.N, generator=gen, device=device, dtype=torch.float32).to(dt)
    weight = torch.empty(w.G, w.K, w.N, dtype=dt, device=device)
    for g in range(w.G):
        weight[g] = (torch.randn(w.K, w.N, generator=gen, device=device, dtype=torch.float32)
                     * w.w_std).to(dt)
    return dy, weight


def make_inputs(w: Workload, device="cpu") -> Inputs:
    """Seeded inputs for ``w``. Routing is drawn on the CPU; values on ``device``
    (the value stream therefore depends on the device type)."""
    gen = torch.Generator()
    gen.manual_seed(w.seed)
    experts = route_experts(w, gen)
    gather, scatter, group_list = expanded_order(experts, w.G)
    idx = gather if w.row_idx_type == 0 else scatter
    dy, weight = _values(w, device, w.seed)
    return Inputs(w, dy, weight, idx.to(device), group_list.to(device), experts, gather)


def forward_input(inp: Inputs, device=None) -> torch.Tensor:
    """The forward input x [batch, K] that goes with ``inp`` (the operand of the
    weight gradient): x ~ N(0, 1) drawn in fp32 on ``device`` (default: the
    device of ``inp``) with seed + 2 and rounded to the workload dtype."""
    w = inp.workload
    device = inp.grad_y.device if device is None else device
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed + 2)
    x = torch.randn(w.batch, w.K, generator=gen, device=device, dtype=torch.float32)
    return x.to(DTYPES[w.dtype])


def unpermute_inputs(inp: Inputs, device=None):
    """(d_out [batch, N], probs [batch, top_k]) for the probs-weighted unpermute
    backward that goes with ``inp`` (whose grad_y [M, N] stands for the expert
    outputs being combined): d_out ~ N(0, 1) (seed + 3); probs drawn uniform in
    (0, 1] and normalised per token (seed + 4); both in fp32, rounded to the
    workload dtype."""
    w = inp.workload
    device = inp.grad_y.device if device is None else device
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed + 3)
    d_out = torch.randn(w.batch, w.N, generator=gen, device=device, dtype=torch.float32)
    gen.manual_seed(w.seed + 4)
    p = torch.rand(w.batch, w.top_k, generator=gen, device=device, dtype=torch.float32) + 1e-3
    p = p / p.sum(dim=1, keepdim=True)
    return d_out.to(DTYPES[w.dtype]), p.to(DTYPES[w.dtype])


def make_case(batch, top_k, G, K, N, dtype="bf16", routing="uniform", row_idx_type=0,
              seed=0, empty=(), device="cpu", name="case", **kw) -> Inputs:
    w = Workload(name, batch=batch, top_k=top_k, G=G, K=K, N=N, dtype=dtype, routing=routing,
                 row_idx_type=row_idx_type, seed=seed, empty=tuple(empty), **kw)
    return make_inputs(w, device)


def with_row_idx_type(inp: Inputs, row_idx_type: int) -> Inputs:
    """The same problem with the index in the other form."""
    gather = inp.gather
    if row_idx_type == 0:
        idx = gather
    else:
        idx = torch.empty_like(gather)
        idx[gather] = torch.arange(gather.numel(), dtype=torch.int64)
    w = replace(inp.workload, row_idx_type=row_idx_type)
    return Inputs(w, inp.grad_y, inp.weight, idx.to(inp.grad_y.device), inp.group_list,
                  inp.experts, inp.gather)
