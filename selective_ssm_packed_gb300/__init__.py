"""Packed variable-length Mamba-1 conv1d + selective scan for GB300 (sm_103a).

The compute lives in libvarlen_ssm.so (C ABI, include/varlen_ssm.h); this
package builds it (``build.build()``) and exposes a thin ctypes binding with
the C entry points' names.
"""
from .binding import (  # noqa: F401
    VssmError,
    chunk_states_shape,
    pack_sequences,
    read_status,
    varlen_conv1d_bwd,
    varlen_conv1d_fwd,
    varlen_conv1d_scan_fwd,
    varlen_position_indices,
    varlen_selective_scan_bwd,
    varlen_selective_scan_fwd,
)
