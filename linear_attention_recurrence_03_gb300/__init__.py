"""Gated delta-rule (GDN) linear-attention recurrence for one NVIDIA GB300 (sm_103a).

A C-ABI CUDA library (include/gdn.h, built into ``libgdn.so`` by ``build.py``) with a
thin Python binding of the same names:

* ``gdn_prefill``      -- chunked prefill ("GDN CTE Kernel API Reference").
* ``gdn_prefill_noalloc`` -- the same, with the library's own static scratch.
* ``gdn_prefill_varlen`` -- the same over sequences packed by ``cu_seqlens``.
* ``gdn_decode_step``  -- fused single-token decode step ("GDN TKG Kernel API Reference").
* ``gdn_decode_multi`` -- T consecutive decode tokens in one call (state read once).
* ``gdn_unit_lower_inverse`` -- the intra-chunk (I + A)^-1 by forward substitution or
  the Neumann product (the prefill's selectable inverse method, on its own).
* ``gdn_conv1d_decode`` -- the conv1d decode token feeding the decode step ("GDN Block
  TKG Kernel API Reference").
"""
from .gdn import (  # noqa: F401
    EXPORTS,
    GDN_DTYPE_BF16,
    GDN_DTYPE_F32,
    GDN_ECUDA,
    GDN_EINVAL,
    GDN_ETIMEOUT,
    GDN_EUNSUPPORTED,
    GDN_OK,
    GDN_TRIL_NEUMANN,
    GDN_TRIL_SUBSTITUTION,
    GDNError,
    gdn_conv1d_decode,
    gdn_decode_multi,
    gdn_decode_step,
    gdn_get_device_status,
    gdn_last_error,
    gdn_launch_count,
    gdn_prefill,
    gdn_prefill_noalloc,
    gdn_prefill_varlen,
    gdn_prefill_varlen_workspace_bytes,
    gdn_prefill_workspace_bytes,
    gdn_unit_lower_inverse,
    load_library,
)
