"""fp64 CPU oracle for the gated delta-rule recurrence (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
import this package. The CUDA library and its Python binding never do.
"""
from .oracle import (  # noqa: F401
    Oracle,
    default,
    build,
    conv1d_decode,
    conv1d_split,
    decode_multi,
    decode_step,
    prefill,
    prefill_chunked,
    prefill_varlen,
    unit_lower_inverse,
    EPS_L2,
    EPS_RMS,
)
