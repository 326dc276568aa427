"""Seeded synthetic workloads shared by the oracle, the CUDA path and the bench.

Only random draws and index structure live here (block tables, lengths,
first-block offsets, token lists, padding masks, raw K/V/Q values).  None of
the paged-cache arithmetic does: slot numbers, copies and attention are
computed separately by ``oracle/`` and by the CUDA library.
"""

from .gen import (  # noqa: F401
    PoolSpec,
    Batch,
    TokenStream,
    Workload,
    CONFIGS,
    make_workload,
    small_workload,
    fill_pool,
    fill_pool_i8,
    new_pool,
    rand_rows,
    to_numpy_bits,
)
