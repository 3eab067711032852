"""Which units of a full-size workload the parity tests compare with the oracle.

The oracle (fp64 loops on the host cores) covers every unit of these workloads
in seconds to tens of seconds, so they are compared in full; the others on a
seeded subset of ceil(n / 16) units (tokens of d_x, rows of y, (expert, k) rows
of d_weight), spread over the whole problem.
"""

import numpy as np

FULL = frozenset({"tiny-fp32", "uniform-bf16", "skewed-fp16", "skinny-bf16", "unaligned-bf16"})
FRACTION = 16


def units(name: str, n: int, seed: int, full=FULL):
    """None (compare all n units) or the sorted seeded subset to compare."""
    if name in full:
        return None
    k = -(-n // FRACTION)
    return np.sort(np.random.default_rng(seed).choice(n, k, replace=False))


def chunks(n_or_units, size: int):
    """The units (all of range(n) when given an int) in consecutive pieces of
    at most ``size``."""
    u = np.arange(n_or_units) if isinstance(n_or_units, (int, np.integer)) else n_or_units
    for i in range(0, len(u), size):
        yield u[i:i + size]
