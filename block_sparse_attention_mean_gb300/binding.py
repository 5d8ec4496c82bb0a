"""ctypes binding of libbsa.so: the C ABI of include/bsa.h, one Python function per
entry point with the same name (argument marshalling only), plus small helpers
that allocate outputs and workspaces with torch.

There is no fallback: if libbsa.so cannot be loaded every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbsa.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_SHAPE = 2
ERR_DTYPE = 3
ERR_CAPACITY = 4
ERR_NONFINITE = 5
ERR_TIMEOUT = 6
ERR_CUDA = 7
ERR_UNSUPPORTED = 8
ERR_WORKSPACE = 9

BF16 = 0
FP32 = 1

STATIC_EXPLICIT = 0
STATIC_MODALITY_BAND = 1
STATIC_CUBOID = 2
MAX_ANCHORS = 8

# every symbol declared in include/bsa.h
EXPORTS = ("bsa_build_mask", "bsa_forward", "bsa_mask_nnz", "bsa_workspace_size",
           "bsa_check_device_error", "bsa_validate_index", "bsa_debug_config",
           "bsa_status_string", "bsa_build_mask_noalloc", "bsa_residual_capture", "bsa_forward_residual",
           "bsa_build_mask_modal", "bsa_mask_nnz_modal", "bsa_build_mask_exact", "bsa_forward_tokens",
           "bsa_select_tokens", "bsa_query_groups", "bsa_tokens_per_group", "bsa_forward_plan",
           "bsa_forward_lse")
NOALLOC_SCRATCH_BYTES = 16 << 20  # BSA_NOALLOC_SCRATCH_BYTES
# bsa_debug_config flag bits
DBG_STALL = 1       # skip loads and MMAs: the first device wait runs out
DBG_NO_SPLIT = 2    # never split a query tile over several CTAs
DBG_SPLIT_ALL = 4   # split every tile with two or more steps (within the partial budget)
INDEX_PLANNED = 0x100  # BSA_INDEX_PLANNED: index_mode flag, reuse the work list of bsa_forward_plan


class StaticSpec(ctypes.Structure):
    """Mirror of bsa_static_spec."""
    _fields_ = [("kind", ctypes.c_int), ("bitmap", ctypes.c_void_p), ("broadcast_bh", ctypes.c_int),
                ("n_text_blocks", ctypes.c_int), ("band", ctypes.c_int), ("n_anchors", ctypes.c_int),
                ("anchors", ctypes.c_int * MAX_ANCHORS), ("grid_t", ctypes.c_int),
                ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int)]


class BsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (status {code})")
        self.code = code


_lib = None


def load():
    """Load libbsa.so (raises OSError if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise OSError(f"libbsa.so not built at {LIB_PATH}; run block_sparse_attention_mean_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    I64, SZ, U32, U64 = ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint64
    lib.bsa_build_mask.argtypes = [P, P, I, I, I, I, I, I, F, ctypes.POINTER(StaticSpec), P, P, I64, P, P,
                                   SZ, P]
    lib.bsa_forward.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P, I, F, P, P, P, SZ, P]
    lib.bsa_forward_residual.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P, I, F, P, P, P, P, SZ, P]
    lib.bsa_forward_plan.argtypes = [I, I, I, I, I, I, P, P, P, I, P, SZ, P]
    lib.bsa_forward_lse.argtypes = [P, P, I, I, I, I, I, I, P, P, P, I, F, P, P, SZ, P]
    lib.bsa_residual_capture.argtypes = [P, P, I, I64, P, P]
    lib.bsa_forward_tokens.argtypes = [P, P, P, I, I, I, I, I, P, P, I, F, P, P, P, SZ, P]
    lib.bsa_select_tokens.argtypes = [P, P, I, I, I, I, I, P, P, F, F, P, I64, P, SZ, P]
    lib.bsa_query_groups.argtypes = [P, I, I, I, I, I, P, P, SZ, P]
    lib.bsa_tokens_per_group.argtypes = [I, F, ctypes.POINTER(I)]
    lib.bsa_build_mask_modal.argtypes = [P, P, I, I, I, I, I, I, I, P, P, P, I64, P, P, SZ, P]
    lib.bsa_mask_nnz_modal.argtypes = [I, I, I, I, I, P, ctypes.POINTER(I64)]
    lib.bsa_build_mask_exact.argtypes = [P, P, I, I, I, I, I, I, F, F, P, P, P, I64, P, P, SZ, P]
    lib.bsa_build_mask_noalloc.argtypes = [P, P, I, I, I, I, I, I, F, ctypes.POINTER(StaticSpec), P, P, I64, P,
                                           P, P]
    lib.bsa_mask_nnz.argtypes = [I, I, I, I, F, ctypes.POINTER(StaticSpec), ctypes.POINTER(I64)]
    lib.bsa_workspace_size.argtypes = [I, I, I, I, I, I, ctypes.POINTER(SZ)]
    lib.bsa_check_device_error.argtypes = [P, P]
    lib.bsa_validate_index.argtypes = [I, I, I, I, P, P, P, P, SZ, P]
    lib.bsa_debug_config.argtypes = [U32, U64]
    lib.bsa_status_string.argtypes = [I]
    lib.bsa_status_string.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name != "bsa_status_string":
            getattr(lib, name).restype = I
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str):
    if code != OK:
        raise BsaError(code, where)


def status_string(code: int) -> str:
    return load().bsa_status_string(int(code)).decode()


# ------------------------------------------------------------------ C ABI mirror


def bsa_build_mask(Q, K, dt: int, B: int, H: int, N: int, d: int, block: int, density: float,
                   spec: Optional[StaticSpec], row_ptr, col_idx, col_capacity: int, bitmap, workspace,
                   workspace_bytes: int, stream=None) -> None:
    code = load().bsa_build_mask(_ptr(Q), _ptr(K), dt, B, H, N, d, block, float(density),
                                 ctypes.byref(spec) if spec is not None else None, _ptr(row_ptr),
                                 _ptr(col_idx), int(col_capacity), _ptr(bitmap), _ptr(workspace),
                                 int(workspace_bytes), _stream(stream))
    _check(code, "bsa_build_mask")


def bsa_forward(Q, K, V, dt: int, B: int, H: int, N: int, d: int, block: int, row_ptr, col_idx, bitmap,
                index_mode: int, scale: float, O, LSE, workspace, workspace_bytes: int, stream=None) -> None:
    code = load().bsa_forward(_ptr(Q), _ptr(K), _ptr(V), dt, B, H, N, d, block, _ptr(row_ptr), _ptr(col_idx),
                              _ptr(bitmap), int(index_mode), float(scale), _ptr(O), _ptr(LSE),
                              _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(code, "bsa_forward")


def bsa_forward_lse(Q, K, dt: int, B: int, H: int, N: int, d: int, block: int, row_ptr, col_idx, bitmap,
                    index_mode: int, scale: float, LSE, workspace, workspace_bytes: int, stream=None) -> None:
    code = load().bsa_forward_lse(_ptr(Q), _ptr(K), dt, B, H, N, d, block, _ptr(row_ptr), _ptr(col_idx),
                                  _ptr(bitmap), int(index_mode), float(scale), _ptr(LSE), _ptr(workspace),
                                  int(workspace_bytes), _stream(stream))
    _check(code, "bsa_forward_lse")


def bsa_forward_plan(dt: int, B: int, H: int, N: int, d: int, block: int, row_ptr, col_idx, bitmap,
                     index_mode: int, workspace, workspace_bytes: int, stream=None) -> None:
    code = load().bsa_forward_plan(dt, B, H, N, d, block, _ptr(row_ptr), _ptr(col_idx), _ptr(bitmap),
                                   int(index_mode), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(code, "bsa_forward_plan")


def bsa_forward_residual(Q, K, V, dt: int, B: int, H: int, N: int, d: int, block: int, row_ptr, col_idx,
                         bitmap, index_mode: int, scale: float, R, O, LSE, workspace, workspace_bytes: int,
                         stream=None) -> None:
    code = load().bsa_forward_residual(_ptr(Q), _ptr(K), _ptr(V), dt, B, H, N, d, block, _ptr(row_ptr),
                                       _ptr(col_idx), _ptr(bitmap), int(index_mode), float(scale), _ptr(R),
                                       _ptr(O), _ptr(LSE), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(code, "bsa_forward_residual")


def _densities(density) -> ctypes.Array:
    d4 = [float(x) for x in density]
    if len(d4) != 4:
        raise ValueError("density: four values (text->text, text->image, image->text, image->image)")
    return (ctypes.c_float * 4)(*d4)


def bsa_mask_nnz_modal(B: int, H: int, N: int, block: int, n_text_blocks: int, density) -> int:
    out = ctypes.c_int64(0)
    _check(load().bsa_mask_nnz_modal(B, H, N, block, n_text_blocks, _densities(density), ctypes.byref(out)),
           "bsa_mask_nnz_modal")
    return int(out.value)


def bsa_build_mask_modal(Q, K, dt: int, B: int, H: int, N: int, d: int, block: int, n_text_blocks: int, density,
                         row_ptr, col_idx, col_capacity: int, bitmap, workspace, workspace_bytes: int,
                         stream=None) -> None:
    code = load().bsa_build_mask_modal(_ptr(Q), _ptr(K), dt, B, H, N, d, block, int(n_text_blocks),
                                       _densities(density), _ptr(row_ptr), _ptr(col_idx), int(col_capacity),
                                       _ptr(bitmap), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(code, "bsa_build_mask_modal")


def build_mask_modal(q: torch.Tensor, k: torch.Tensor, block: int, n_text_blocks: int, density,
                     ws: Optional[torch.Tensor] = None, stream=None) -> "Index":
    """Per-modality top-k index (bsa_build_mask_modal) with freshly allocated buffers."""
    B, H, N, d = q.shape
    nB = -(-N // block)  # a ragged last block counts
    W = (nB + 31) // 32
    nnz = bsa_mask_nnz_modal(B, H, N, block, n_text_blocks, density)
    row_ptr = torch.empty(B * H * nB + 1, dtype=torch.int32, device=q.device)
    col_idx = torch.empty(max(nnz, 1), dtype=torch.int32, device=q.device)
    bitmap = torch.empty(B * H * nB * W, dtype=torch.int32, device=q.device)
    if ws is None:
        ws = workspace(0, B, H, N, d, block, q.device)
    bsa_build_mask_modal(q, k, _dtype_code(q), B, H, N, d, block, n_text_blocks, density, row_ptr, col_idx,
                         col_idx.numel(), bitmap, ws, ws.numel(), stream)
    _check(bsa_check_device_error(ws, stream), "bsa_build_mask_modal (device)")
    return Index(row_ptr, col_idx, bitmap, nnz, block)


def bsa_build_mask_exact(Q, K, dt: int, B: int, H: int, N: int, d: int, block: int, density: float, scale: float,
                         LSE, row_ptr, col_idx, col_capacity: int, bitmap, workspace, workspace_bytes: int,
                         stream=None) -> None:
    code = load().bsa_build_mask_exact(_ptr(Q), _ptr(K), dt, B, H, N, d, block, float(density), float(scale),
                                       _ptr(LSE), _ptr(row_ptr), _ptr(col_idx), int(col_capacity), _ptr(bitmap),
                                       _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(code, "bsa_build_mask_exact")


def build_mask_exact(q: torch.Tensor, k: torch.Tensor, lse_dense: torch.Tensor, block: int, density: float,
                     scale: float = 0.0, ws: Optional[torch.Tensor] = None, stream=None):
    """Block-oracle index from the dense LSE (bsa_build_mask_exact); returns (Index, workspace)."""
    B, H, N, d = q.shape
    nB = -(-N // block)  # a ragged last block counts
    W = (nB + 31) // 32
    nnz = bsa_mask_nnz(B, H, N, block, density, None)  # the same count rule as the pooled selector
    row_ptr = torch.empty(B * H * nB + 1, dtype=torch.int32, device=q.device)
    col_idx = torch.empty(nnz, dtype=torch.int32, device=q.device)
    bitmap = torch.empty(B * H * nB * W, dtype=torch.int32, device=q.device)
    if ws is None:
        ws = workspace(2, B, H, N, d, block, q.device)
    bsa_build_mask_exact(q, k, _dtype_code(q), B, H, N, d, block, density, scale, lse_dense, row_ptr, col_idx,
                         col_idx.numel(), bitmap, ws, ws.numel(), stream)
    _check(bsa_check_device_error(ws, stream), "bsa_build_mask_exact (device)")
    return Index(row_ptr, col_idx, bitmap, col_idx.numel(), block), ws


def bsa_forward_tokens(Q, K, V, dt: int, B: int, H: int, N: int, d: int, perm, tokens, n_tokens: int,
                       scale: float, O, LSE, ws, ws_bytes: int, stream=None) -> None:
    _check(load().bsa_forward_tokens(_ptr(Q), _ptr(K), _ptr(V), dt, B, H, N, d, _ptr(perm), _ptr(tokens), n_tokens,
                                     ctypes.c_float(scale), _ptr(O), _ptr(LSE), _ptr(ws), ctypes.c_size_t(ws_bytes),
                                     _stream(stream)), "bsa_forward_tokens")


def bsa_query_groups(Q, dt: int, B: int, H: int, N: int, d: int, perm, ws, ws_bytes: int, stream=None) -> None:
    _check(load().bsa_query_groups(_ptr(Q), dt, B, H, N, d, _ptr(perm), _ptr(ws), ctypes.c_size_t(ws_bytes),
                                   _stream(stream)), "bsa_query_groups")


def bsa_select_tokens(Q, K, dt: int, B: int, H: int, N: int, d: int, perm, LSE, density: float, scale: float,
                      tokens, tokens_capacity: int, ws, ws_bytes: int, stream=None) -> None:
    _check(load().bsa_select_tokens(_ptr(Q), _ptr(K), dt, B, H, N, d, _ptr(perm), _ptr(LSE), ctypes.c_float(density),
                                    ctypes.c_float(scale), _ptr(tokens), ctypes.c_int64(tokens_capacity), _ptr(ws),
                                    ctypes.c_size_t(ws_bytes), _stream(stream)), "bsa_select_tokens")


def bsa_residual_capture(O_dense, O_sparse, dt: int, count: int, R, stream=None) -> None:
    code = load().bsa_residual_capture(_ptr(O_dense), _ptr(O_sparse), dt, int(count), _ptr(R), _stream(stream))
    _check(code, "bsa_residual_capture")


def bsa_build_mask_noalloc(Q, K, dt: int, B: int, H: int, N: int, d: int, block: int, density: float,
                           spec: Optional[StaticSpec], row_ptr, col_idx, col_capacity: int, bitmap,
                           device_status=None, stream=None) -> None:
    """bsa_build_mask without a workspace, for callers that cannot allocate device memory."""
    code = load().bsa_build_mask_noalloc(_ptr(Q), _ptr(K), dt, B, H, N, d, block, float(density),
                                         ctypes.byref(spec) if spec is not None else None, _ptr(row_ptr),
                                         _ptr(col_idx), int(col_capacity), _ptr(bitmap), _ptr(device_status),
                                         _stream(stream))
    _check(code, "bsa_build_mask_noalloc")


def bsa_mask_nnz(B: int, H: int, N: int, block: int, density: float, spec: Optional[StaticSpec]) -> int:
    out = ctypes.c_int64(0)
    code = load().bsa_mask_nnz(B, H, N, block, float(density),
                               ctypes.byref(spec) if spec is not None else None, ctypes.byref(out))
    _check(code, "bsa_mask_nnz")
    return out.value


def bsa_workspace_size(which: int, B: int, H: int, N: int, d: int, block: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().bsa_workspace_size(which, B, H, N, d, block, ctypes.byref(out)), "bsa_workspace_size")
    return out.value


def bsa_check_device_error(workspace, stream=None) -> int:
    """Status recorded on the device (0 = none); synchronises the stream and clears it."""
    return int(load().bsa_check_device_error(_ptr(workspace), _stream(stream)))


def bsa_validate_index(B: int, H: int, N: int, block: int, row_ptr, col_idx, bitmap, workspace,
                       workspace_bytes: int, stream=None) -> None:
    _check(load().bsa_validate_index(B, H, N, block, _ptr(row_ptr), _ptr(col_idx), _ptr(bitmap),
                                     _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "bsa_validate_index")


def bsa_debug_config(flags: int, wait_limit_ns: int = 0) -> None:
    _check(load().bsa_debug_config(int(flags), int(wait_limit_ns)), "bsa_debug_config")


def bsa_status_string(code: int) -> str:
    return status_string(code)


# ------------------------------------------------------------------ helpers


def band_spec(n_text_blocks: int, band: int, anchors: Sequence[int]) -> StaticSpec:
    s = StaticSpec()
    s.kind = STATIC_MODALITY_BAND
    s.n_text_blocks = n_text_blocks
    s.band = band
    s.n_anchors = len(anchors)
    for i, a in enumerate(anchors):
        s.anchors[i] = a
    return s


def cuboid_spec(n_text_blocks: int, grid: Tuple[int, int, int]) -> StaticSpec:
    s = StaticSpec()
    s.kind = STATIC_CUBOID
    s.n_text_blocks = n_text_blocks
    s.grid_t, s.grid_h, s.grid_w = grid
    return s


def explicit_spec(bitmap: torch.Tensor, broadcast_bh: bool = False) -> StaticSpec:
    s = StaticSpec()
    s.kind = STATIC_EXPLICIT
    s.bitmap = bitmap.data_ptr()
    s.broadcast_bh = 1 if broadcast_bh else 0
    s._keep = bitmap  # keep the device buffer alive with the spec
    return s


def _dtype_code(t: Optional[torch.Tensor], default: int = BF16) -> int:
    if t is None:
        return default
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise BsaError(ERR_DTYPE, f"tensor dtype {t.dtype}")


def workspace(which: int, B: int, H: int, N: int, d: int, block: int, device="cuda") -> torch.Tensor:
    """Zero-initialised device workspace (the device error word starts cleared)."""
    return torch.zeros(bsa_workspace_size(which, B, H, N, d, block), dtype=torch.uint8, device=device)


class Index:
    """Device CSR + bitmap index of a block mask."""

    def __init__(self, row_ptr, col_idx, bitmap, nnz, block):
        self.row_ptr, self.col_idx, self.bitmap, self.nnz, self.block = row_ptr, col_idx, bitmap, nnz, block


def build_mask(q: Optional[torch.Tensor], k: Optional[torch.Tensor], block: int, density: float = 0.0,
               spec: Optional[StaticSpec] = None, shape: Optional[Tuple[int, int, int, int]] = None,
               ws: Optional[torch.Tensor] = None, stream=None, check: bool = True) -> Index:
    """Allocate the index and run bsa_build_mask. `shape` = (B, H, N, d) when q is None."""
    if q is not None:
        B, H, N, d = q.shape
        device = q.device
    else:
        B, H, N, d = shape
        device = torch.device("cuda")
    nB = -(-N // block)  # a ragged last block counts
    nnz = bsa_mask_nnz(B, H, N, block, density, spec)
    W = (nB + 31) // 32
    row_ptr = torch.empty(B * H * nB + 1, dtype=torch.int32, device=device)
    col_idx = torch.empty(max(nnz, 1), dtype=torch.int32, device=device)
    bitmap = torch.empty(B * H * nB * W, dtype=torch.int32, device=device)
    if ws is None:
        ws = workspace(0, B, H, N, d, block, device)
    bsa_build_mask(q, k, _dtype_code(q), B, H, N, d, block, density, spec, row_ptr, col_idx, nnz, bitmap,
                   ws, ws.numel(), stream)
    if check:
        _check(bsa_check_device_error(ws, stream), "bsa_build_mask (device)")
    if spec is not None and spec.kind == STATIC_EXPLICIT and check:
        nnz = int(row_ptr[-1].item())
    return Index(row_ptr, col_idx, bitmap, nnz, block)


def forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, index: Index, index_mode: int = 0,
            scale: float = 0.0, ws: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, stream=None, check: bool = True,
            residual: Optional[torch.Tensor] = None):
    """Run bsa_forward (or bsa_forward_residual when `residual` is given); returns (O, LSE)."""
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(1, B, H, N, d, index.block, q.device)
    if residual is None:
        bsa_forward(q, k, v, _dtype_code(q), B, H, N, d, index.block, index.row_ptr, index.col_idx, index.bitmap,
                    index_mode, scale, out, lse, ws, ws.numel(), stream)
    else:
        bsa_forward_residual(q, k, v, _dtype_code(q), B, H, N, d, index.block, index.row_ptr, index.col_idx,
                             index.bitmap, index_mode, scale, residual, out, lse, ws, ws.numel(), stream)
    if check:
        _check(bsa_check_device_error(ws, stream), "bsa_forward (device)")
    return out, lse


def forward_lse(q: torch.Tensor, k: torch.Tensor, index: Index, index_mode: int = 0, scale: float = 0.0,
                ws: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, stream=None,
                check: bool = True) -> torch.Tensor:
    """Run bsa_forward_lse; returns LSE fp32 [B, H, N]."""
    B, H, N, d = q.shape
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(1, B, H, N, d, index.block, q.device)
    bsa_forward_lse(q, k, _dtype_code(q), B, H, N, d, index.block, index.row_ptr, index.col_idx, index.bitmap,
                    index_mode, scale, lse, ws, ws.numel(), stream)
    if check:
        _check(bsa_check_device_error(ws, stream), "bsa_forward_lse (device)")
    return lse


def forward_plan(q: torch.Tensor, index: Index, index_mode: int = 0, ws: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """Run bsa_forward_plan into `ws` (allocated when None); returns the workspace to pass to
    forward(..., index_mode=index_mode | INDEX_PLANNED, ws=ws)."""
    B, H, N, d = q.shape
    if ws is None:
        ws = workspace(1, B, H, N, d, index.block, q.device)
    bsa_forward_plan(_dtype_code(q), B, H, N, d, index.block, index.row_ptr, index.col_idx, index.bitmap,
                     index_mode, ws, ws.numel(), stream)
    return ws


def residual_capture(o_dense: torch.Tensor, o_sparse: torch.Tensor, out: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """R = O_dense - O_sparse in fp32 (bsa_residual_capture)."""
    if out is None:
        out = torch.empty(o_dense.shape, dtype=torch.float32, device=o_dense.device)
    bsa_residual_capture(o_dense, o_sparse, _dtype_code(o_dense), o_dense.numel(), out, stream)
    return out


def forward_tokens(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, perm: torch.Tensor, tokens: torch.Tensor,
                   scale: float = 0.0, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   ws: Optional[torch.Tensor] = None, stream=None, check: bool = True):
    """Run bsa_forward_tokens: perm int32 [B*H, N] (groups of 128 rows), tokens int32
    [B*H, N/128, n_tokens]; returns (O, LSE)."""
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = torch.zeros(256, dtype=torch.uint8, device=q.device)
    bsa_forward_tokens(q, k, v, _dtype_code(q), B, H, N, d, perm, tokens, int(tokens.shape[-1]), scale, out, lse,
                       ws, ws.numel(), stream)
    if check:
        _check(bsa_check_device_error(ws, stream), "bsa_forward_tokens (device)")
    return out, lse


def bsa_tokens_per_group(N: int, density: float) -> int:
    out = ctypes.c_int(0)
    _check(load().bsa_tokens_per_group(int(N), float(density), ctypes.byref(out)), "bsa_tokens_per_group")
    return int(out.value)


def tokens_per_group(N: int, density: float) -> int:
    """Tokens each query group keeps (the library's host count, bsa_tokens_per_group)."""
    return bsa_tokens_per_group(N, density)


def query_groups(q: torch.Tensor, stream=None, check: bool = True) -> torch.Tensor:
    """Run bsa_query_groups; returns perm int32 [B*H, N] (groups of 128 rows)."""
    B, H, N, d = q.shape
    perm = torch.empty((B * H, N), dtype=torch.int32, device=q.device)
    ws = workspace(4, B, H, N, d, 64, q.device)
    bsa_query_groups(q, _dtype_code(q), B, H, N, d, perm, ws, ws.numel(), stream)
    if check:
        _check(bsa_check_device_error(ws, stream), "bsa_query_groups (device)")
    return perm


def select_tokens(q: torch.Tensor, k: torch.Tensor, perm: torch.Tensor, lse: torch.Tensor, density: float,
                  scale: float = 0.0, stream=None, check: bool = True):
    """Run bsa_select_tokens; returns (tokens int32 [B*H, N/128, K], workspace)."""
    B, H, N, d = q.shape
    K = tokens_per_group(N, density)
    tokens = torch.empty((B * H, N // 128, K), dtype=torch.int32, device=q.device)
    ws = workspace(3, B, H, N, d, 64, q.device)
    bsa_select_tokens(q, k, _dtype_code(q), B, H, N, d, perm, lse, density, scale, tokens, tokens.numel(), ws,
                      ws.numel(), stream)
    if check:
        _check(bsa_check_device_error(ws, stream), "bsa_select_tokens (device)")
    return tokens, ws


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
