"""Seeded synthetic inputs for the attention-scored KV decode path.

This package holds only input recipes: shapes, seeds, value distributions and the
planted structure of each workload.  It contains none of the method's arithmetic
(no attention, quantisation, scoring or selection), and it is shared by the tests,
the oracle-driven checks and the benchmark.  It imports neither ``oracle`` nor the
CUDA package.
"""

from .recipes import (  # noqa: F401
    Workload, WORKLOADS, get, Inputs, scaled_down, as_f64, tensor_seed,
)
