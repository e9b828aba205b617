"""GB300 selective-SSM (Mamba2 SSD) serving hot path.

Python binding of the C ABI in ``include/ssd.h``: ``ssd_chunk_metadata``
(host), ``ssd_prefill_varlen`` and ``ssm_decode_update`` (CUDA, sm_103a), both parts of a
mixed batch in one call, ``ssd_mixed_step``, and the
depthwise causal conv1d in front of them, ``ssd_conv1d_varlen`` / ``ssd_conv1d_update``, and the
Mamba1 selective scan with per-channel states, ``mamba1_scan_varlen`` / ``mamba1_state_update``.
The CUDA library is loaded on first use; if it is missing the call raises.
"""
from ._binding import (  # noqa: F401
    DEVERR_COLUMN, DEVERR_METADATA, DEVERR_SLOT, DEVERR_TIMEOUT, EXPORTED_SYMBOLS, LIB_PATH, SSDError,
    conv1d_args, decode_args, lib, mamba1_args, mamba1_scan_varlen, mamba1_state_update, prefill_args,
    ssd_chunk_metadata, ssd_conv1d_update, ssd_conv1d_varlen, ssd_mixed_step,
    ssd_max_chunks, ssd_prefill_kernel_count, ssd_prefill_varlen,
    ssd_prefill_workspace_size, ssm_decode_update)


def build(verbose_ptxas: bool = False) -> str:
    """Compile ``libssd_gb300.so`` in-tree (nvcc, sm_103a); returns its path."""
    from ._build import build as _b
    return _b(verbose_ptxas)
