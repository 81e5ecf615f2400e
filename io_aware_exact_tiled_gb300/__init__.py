"""Fused, tiled, exact softmax attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libfa.so`` built from ``csrc/``
(declared in ``include/fa.h``); :mod:`.binding` only marshals arguments.
"""

from .binding import (  # noqa: F401
    FAError,
    forward,
    backward,
    forward_varlen,
    backward_varlen,
    decode,
    forward_fp8,
    forward_dropout,
    backward_dropout,
    backward_noalloc,
    noalloc_status,
    fwd_workspace_size,
    bwd_workspace_size,
    get_status,
    last_launch_count,
    load,
    set_timing_events,
    workspace,
)
from .binding import C_NAMES as _C_NAMES

globals().update(_C_NAMES)  # fa_fwd, fa_bwd, ...: the header's names
