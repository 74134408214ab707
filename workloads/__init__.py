"""Seeded synthetic inputs for the sharded MLP block and the vocab-parallel
cross-entropy.

This package is shared by the tests, the benchmark and the oracle's callers.
It holds workload shapes and random-number recipes only: none of the
method's arithmetic lives here (no matmul, activation, reduction or loss).
"""

from .configs import MLPConfig, CEConfig, MLP_CONFIGS, CE_CONFIGS, config_by_name  # noqa: F401
from .gen import (  # noqa: F401
    gen_mlp_inputs,
    gen_ce_inputs,
    gen_random_mlp,
    gen_integer_mlp,
    MLPInputs,
    CEInputs,
)
