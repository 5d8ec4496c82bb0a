"""GB300 block-sparse attention forward: mean-pooled top-k / static block masks
and a tcgen05 block-sparse FlashAttention kernel behind a C ABI (libbsa.so).

The compute path is the CUDA library only; this package marshals arguments.
The binding (and with it torch) is imported on first use of one of its names, so
that the seeded input generator (``workloads``) can be used without either.
"""
_BINDING_NAMES = (
    "BF16", "FP32", "BsaError", "Index", "StaticSpec", "band_spec", "bsa_build_mask", "bsa_check_device_error",
    "bsa_debug_config", "bsa_forward", "bsa_mask_nnz", "bsa_status_string", "bsa_validate_index",
    "bsa_workspace_size", "build_mask", "cuboid_spec", "explicit_spec", "forward", "load", "workspace")

__all__ = list(_BINDING_NAMES)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
