"""CPU oracle for exact softmax attention (test infrastructure only).

This package is a plain, slow, fp64 statement of what fused tiled attention
computes. It exists so that the CUDA kernels can be checked against something
obviously correct. It shares no code with the CUDA path and must only be used
by the tests, by the package's smoke check and by the benchmark's CPU-baseline
leg; the product path never calls it.

Every function here is pinned by ``tests/test_oracle.py`` against closed forms,
invariants, finite differences and an independent library routine.
"""

from .attention import (  # noqa: F401
    visible,
    scores,
    probabilities,
    forward,
    backward,
    tiled_forward,
    row_stat_D,
)
from .varlen import forward_varlen, backward_varlen  # noqa: F401
from .decode import decode_forward, split_decode  # noqa: F401
from .fp8 import fp8_forward, fp8_forward_online, fp8_shift_bound, e4m3_round  # noqa: F401
from . import dropout  # noqa: F401
