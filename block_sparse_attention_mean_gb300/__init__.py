"""GB300 block-sparse attention forward: mean-pooled top-k / static block masks
and a tcgen05 block-sparse FlashAttention kernel behind a C ABI (libbsa.so).

The compute path is the CUDA library only; this package marshals arguments.
"""
from .binding import (  # noqa: F401
    BF16, FP32, BsaError, Index, StaticSpec, band_spec, bsa_build_mask, bsa_check_device_error,
    bsa_debug_config, bsa_forward, bsa_mask_nnz, bsa_status_string, bsa_validate_index,
    bsa_workspace_size, build_mask, cuboid_spec, explicit_spec, forward, load, workspace)
