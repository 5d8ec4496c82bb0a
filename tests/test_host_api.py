"""C-ABI library checks that need no GPU: it loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from block_sparse_attention_mean_gb300 import binding as bb
from block_sparse_attention_mean_gb300 import build as bbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    bbuild.build()
    return bb.load()


def _header_functions():
    src = open(os.path.join(ROOT, "include", "bsa.h")).read()
    return sorted(set(re.findall(r"^(?:bsa_status|const char \*)\s*(bsa_\w+)\s*\(", src, re.M)))


def test_header_symbols_exported(lib):
    names = _header_functions()
    assert len(names) == 20
    assert sorted(bb.EXPORTS) == names
    for n in names:
        assert getattr(lib, n) is not None  # dlsym succeeds


def test_header_is_plain_c_and_cpp():
    # the boundary is a C ABI: the header must compile as C99 and as C++17 with no other include
    import shutil
    import subprocess
    header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bsa.h")
    for cc, std, lang in (("gcc", "-std=c99", "c"), ("g++", "-std=c++17", "c++")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not available")
        r = subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", lang, header],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_status_strings(lib):
    assert bb.status_string(0) == "ok"
    assert "capacity" in bb.status_string(bb.ERR_CAPACITY)
    assert bb.status_string(99) == "unknown status"


def test_workspace_sizes(lib):
    ws0 = bb.bsa_workspace_size(0, 2, 24, 4224, 64, 64)
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    BH, nB, d, W = 48, 66, 64, 3
    dynamic = 256 + 2 * up(BH * nB * d * 4) + up(BH * nB * nB * 4)                # Qbar, Kbar, score keys
    static = 256 + up(BH * nB * 4) + up((nB + 1) * 4) + up(nB * W * 4)  # counts, pattern
    assert ws0 == max(dynamic, static)
    ws1 = bb.bsa_workspace_size(1, 2, 24, 4224, 64, 64)
    tiles = 2 * 24 * 33  # 128-row query tiles
    budget = min(640, 8 * tiles)  # partial slots for chunks of split tiles
    # header, items (tiles + chunks), tile lengths, split bases, merge counters (8 per slot),
    # partial row stats (16 B per row), partial O (fp32, d per row)
    assert ws1 == (256 + up((tiles + budget) * 4) + 2 * up(tiles * 4) + up(budget * 8 * 4)
                   + up(budget * 128 * 16) + up(budget * 128 * d * 4))
    # a tiny problem gets at most 8 partial slots per tile
    tiny = bb.bsa_workspace_size(1, 1, 1, 128, 64, 64)
    assert tiny == 256 + up(9 * 4) + 2 * up(4) + up(8 * 8 * 4) + up(8 * 128 * 16) + up(8 * 128 * 64 * 4)
    # a ragged sequence (N not a multiple of the block) has ceil(N / 128) query tiles
    assert bb.bsa_workspace_size(1, 1, 1, 100, 64, 64) == tiny
    assert bb.bsa_workspace_size(0, 1, 1, 100, 64, 64) == bb.bsa_workspace_size(0, 1, 1, 128, 64, 64)
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_workspace_size(1, 1, 1, 0, 64, 64)
    assert e.value.code == bb.ERR_SHAPE
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_workspace_size(5, 1, 1, 128, 64, 64)  # 0 mask, 1 forward, 2 exact, 3 tokens, 4 groups
    assert e.value.code == bb.ERR_INVALID_ARG


def test_ragged_sequence_block_counts(lib):
    # N = 500 at block 64: 8 blocks, the last one holding 52 tokens; k = floor(0.5 * 8) = 4
    assert bb.bsa_mask_nnz(1, 2, 500, 64, 0.5, None) == 2 * 8 * 4
    assert bb.bsa_mask_nnz(1, 1, 500, 128, 0.25, None) == 4 * 1
    assert bb.bsa_mask_nnz_modal(1, 1, 500, 64, 2, [1.0, 1.0, 1.0, 0.5]) == 2 * 8 + 6 * (2 + 3)


def test_mask_nnz_counts(lib):
    # 812 active blocks per (b, h) for the t2i band spec, 3600 for the video cuboids
    assert bb.bsa_mask_nnz(2, 24, 4224, 64, 0.0, bb.band_spec(2, 2, [0, 32])) == 812 * 48
    assert bb.bsa_mask_nnz(1, 24, 16640, 64, 0.0, bb.cuboid_spec(4, (4, 8, 8))) == 3600 * 24
    assert bb.bsa_mask_nnz(1, 24, 8192, 64, 0.15, None) == 24 * 128 * 19
    assert bb.bsa_mask_nnz(1, 16, 65536, 128, 0.05, None) == 16 * 512 * 25
    ex = bb.StaticSpec()
    ex.kind = bb.STATIC_EXPLICIT
    ex.bitmap = 256
    assert bb.bsa_mask_nnz(1, 2, 512, 64, 0.0, ex) == 2 * 8 * 8  # upper bound
    with pytest.raises(bb.BsaError):
        bb.bsa_mask_nnz(1, 1, 8192, 64, 0.0, None)  # density 0
    with pytest.raises(bb.BsaError):
        bb.bsa_mask_nnz(1, 1, 8192, 64, 1.5, None)
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_mask_nnz(1, 1, 4224, 64, 0.0, bb.cuboid_spec(4, (4, 8, 8)))  # grid does not match N
    assert e.value.code == bb.ERR_SHAPE


FAKE = 1 << 20  # a 256-aligned non-null address that is never dereferenced on these paths


def _build(**kw):
    args = dict(Q=FAKE, K=FAKE, dt=bb.BF16, B=1, H=2, N=512, d=64, block=64, density=0.5, spec=None,
                row_ptr=FAKE, col_idx=FAKE, col_capacity=1 << 20, bitmap=FAKE, workspace=FAKE,
                workspace_bytes=1 << 30)
    args.update(kw)
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_build_mask(**args, stream=0)
    return e.value.code


def _fwd(**kw):
    args = dict(Q=FAKE, K=FAKE, V=FAKE, dt=bb.BF16, B=1, H=2, N=512, d=64, block=64, row_ptr=FAKE,
                col_idx=FAKE, bitmap=FAKE, index_mode=0, scale=0.0, O=FAKE, LSE=FAKE, workspace=FAKE,
                workspace_bytes=1 << 30)
    args.update(kw)
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_forward(**args, stream=0)
    return e.value.code


def test_build_mask_rejects_bad_arguments(lib):
    assert _build(N=0) == bb.ERR_SHAPE              # empty sequence
    assert _build(d=96) == bb.ERR_SHAPE
    assert _build(block=32) == bb.ERR_SHAPE
    assert _build(dt=7) == bb.ERR_DTYPE
    assert _build(Q=None) == bb.ERR_INVALID_ARG
    assert _build(row_ptr=None) == bb.ERR_INVALID_ARG
    assert _build(density=0.0) == bb.ERR_INVALID_ARG
    assert _build(density=float("nan")) == bb.ERR_INVALID_ARG
    assert _build(workspace=None) == bb.ERR_WORKSPACE
    assert _build(workspace_bytes=16) == bb.ERR_WORKSPACE
    assert _build(workspace=FAKE + 16) == bb.ERR_WORKSPACE  # misaligned
    assert _build(Q=FAKE + 2) == bb.ERR_INVALID_ARG          # TMA-incompatible alignment
    assert _build(col_capacity=2 * 8 * 4 - 1) == bb.ERR_CAPACITY  # k = 4 per row, 16 rows
    assert _build(spec=bb.band_spec(2, 2, [0, 99])) == bb.ERR_INVALID_ARG  # anchor out of range
    assert _build(spec=bb.band_spec(2, 2, [0]), col_capacity=10) == bb.ERR_CAPACITY
    ex = bb.StaticSpec()
    ex.kind = bb.STATIC_EXPLICIT
    assert _build(spec=ex) == bb.ERR_INVALID_ARG  # null bitmap
    bad = bb.StaticSpec()
    bad.kind = 9
    assert _build(spec=bad) == bb.ERR_INVALID_ARG


def test_forward_rejects_bad_arguments(lib):
    assert _fwd(N=0) == bb.ERR_SHAPE
    assert _fwd(d=32) == bb.ERR_SHAPE
    assert _fwd(dt=5) == bb.ERR_DTYPE
    assert _fwd(V=None) == bb.ERR_INVALID_ARG
    assert _fwd(LSE=None) == bb.ERR_INVALID_ARG
    assert _fwd(O=FAKE + 8) == bb.ERR_INVALID_ARG
    assert _fwd(index_mode=2) == bb.ERR_INVALID_ARG
    assert _fwd(index_mode=0, col_idx=None) == bb.ERR_INVALID_ARG
    assert _fwd(index_mode=1, bitmap=None) == bb.ERR_INVALID_ARG
    assert _fwd(scale=float("nan")) == bb.ERR_INVALID_ARG
    assert _fwd(scale=float("inf")) == bb.ERR_INVALID_ARG
    assert _fwd(workspace_bytes=100) == bb.ERR_WORKSPACE
    assert _fwd(B=0) == bb.ERR_SHAPE
    # the planned flag rides on either index mode and is checked with it
    assert _fwd(index_mode=2 | bb.INDEX_PLANNED) == bb.ERR_INVALID_ARG
    assert _fwd(index_mode=1 | bb.INDEX_PLANNED, bitmap=None) == bb.ERR_INVALID_ARG
    assert _fwd(index_mode=0 | bb.INDEX_PLANNED, row_ptr=None) == bb.ERR_INVALID_ARG


def _lse(**kw):
    args = dict(Q=FAKE, K=FAKE, dt=bb.BF16, B=1, H=2, N=512, d=64, block=64, row_ptr=FAKE, col_idx=FAKE,
                bitmap=FAKE, index_mode=0, scale=0.0, LSE=FAKE, workspace=FAKE, workspace_bytes=1 << 30)
    args.update(kw)
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_forward_lse(**args, stream=0)
    return e.value.code


def test_forward_lse_rejects_bad_arguments(lib):
    assert _lse(N=0) == bb.ERR_SHAPE
    assert _lse(d=32) == bb.ERR_SHAPE
    assert _lse(dt=5) == bb.ERR_DTYPE
    assert _lse(K=None) == bb.ERR_INVALID_ARG
    assert _lse(LSE=None) == bb.ERR_INVALID_ARG
    assert _lse(Q=FAKE + 8) == bb.ERR_INVALID_ARG
    assert _lse(index_mode=2) == bb.ERR_INVALID_ARG
    assert _lse(index_mode=bb.INDEX_PLANNED) == bb.ERR_INVALID_ARG  # no planned LSE-only call
    assert _lse(index_mode=1, bitmap=None) == bb.ERR_INVALID_ARG
    assert _lse(scale=float("nan")) == bb.ERR_INVALID_ARG
    assert _lse(workspace_bytes=100) == bb.ERR_WORKSPACE


def _plan(**kw):
    args = dict(dt=bb.BF16, B=1, H=2, N=512, d=64, block=64, row_ptr=FAKE, col_idx=FAKE, bitmap=FAKE,
                index_mode=0, workspace=FAKE, workspace_bytes=1 << 30)
    args.update(kw)
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_forward_plan(**args, stream=0)
    return e.value.code


def test_forward_plan_rejects_bad_arguments(lib):
    assert _plan(N=0) == bb.ERR_SHAPE
    assert _plan(d=96) == bb.ERR_SHAPE
    assert _plan(block=32) == bb.ERR_SHAPE
    assert _plan(dt=3) == bb.ERR_DTYPE
    assert _plan(index_mode=2) == bb.ERR_INVALID_ARG
    assert _plan(index_mode=bb.INDEX_PLANNED) == bb.ERR_INVALID_ARG  # a plan takes a plain index mode
    assert _plan(index_mode=0, col_idx=None) == bb.ERR_INVALID_ARG
    assert _plan(index_mode=1, bitmap=None) == bb.ERR_INVALID_ARG
    assert _plan(workspace=None) == bb.ERR_WORKSPACE
    assert _plan(workspace=FAKE + 16) == bb.ERR_WORKSPACE
    assert _plan(workspace_bytes=100) == bb.ERR_WORKSPACE
    # fp32 keeps no work list: a valid call launches nothing and succeeds without a device
    bb.bsa_forward_plan(bb.FP32, 1, 2, 512, 64, 64, FAKE, FAKE, FAKE, 0, FAKE, 1 << 30, stream=0)


def test_validate_index_rejects_bad_arguments(lib):
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_validate_index(1, 1, 512, 64, None, FAKE, FAKE, FAKE, 1 << 20, stream=0)
    assert e.value.code == bb.ERR_INVALID_ARG
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_validate_index(1, 1, 512, 64, FAKE, FAKE, FAKE, FAKE, 8, stream=0)
    assert e.value.code == bb.ERR_WORKSPACE


def test_debug_config_roundtrip(lib):
    bb.bsa_debug_config(0, 0)


def test_static_spec_layout_matches_header(lib):
    # int kind; ptr; 4 ints; int[8]; 3 ints  (x86-64 and aarch64 LP64 layout)
    assert ctypes.sizeof(bb.StaticSpec) == 4 + 4 + 8 + 4 * 4 + 4 * 8 + 4 * 3 + 4


def _fwd_res(**kw):
    args = dict(Q=FAKE, K=FAKE, V=FAKE, dt=bb.BF16, B=1, H=2, N=512, d=64, block=64, row_ptr=FAKE,
                col_idx=FAKE, bitmap=FAKE, index_mode=0, scale=0.0, R=FAKE, O=FAKE, LSE=FAKE, workspace=FAKE,
                workspace_bytes=1 << 30)
    args.update(kw)
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_forward_residual(**args, stream=0)
    return e.value.code


def _fwd_tok(**kw):
    args = dict(Q=FAKE, K=FAKE, V=FAKE, dt=bb.BF16, B=1, H=2, N=512, d=64, perm=FAKE, tokens=FAKE, n_tokens=32,
                scale=0.0, O=FAKE, LSE=FAKE, ws=FAKE, ws_bytes=256)
    args.update(kw)
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_forward_tokens(**args, stream=0)
    return e.value.code


def test_token_selection_workspace_and_arguments(lib):
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    rows = 2 * 3 * (1024 // 128)
    assert bb.bsa_workspace_size(3, 2, 3, 1024, 128, 64) == 256 + up(rows * 1024 * 4) + up(rows * 32 * 4)
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_workspace_size(3, 1, 1, 1000, 64, 64)
    assert e.value.code == bb.ERR_SHAPE
    assert bb.tokens_per_group(1024, 0.1) == 102 and bb.tokens_per_group(1024, 1e-6) == 1

    def sel(**kw):
        args = dict(Q=FAKE, K=FAKE, dt=bb.BF16, B=1, H=2, N=512, d=64, perm=FAKE, LSE=FAKE, density=0.25,
                    scale=0.0, tokens=FAKE, tokens_capacity=2 * 4 * 128, ws=FAKE, ws_bytes=1 << 30)
        args.update(kw)
        with pytest.raises(bb.BsaError) as e:
            bb.bsa_select_tokens(**args, stream=0)
        return e.value.code

    assert sel(N=500) == bb.ERR_SHAPE
    # fp32 runs on CUDA cores with one shared-memory key per token; bf16 (tcgen05 masses in the
    # workspace, radix top-k) has no such limit and reaches the capacity check instead
    assert sel(N=1 << 16, d=128, dt=bb.FP32) == bb.ERR_SHAPE
    assert sel(N=1 << 16, d=128) == bb.ERR_CAPACITY
    assert sel(dt=3) == bb.ERR_DTYPE
    assert sel(LSE=None) == bb.ERR_INVALID_ARG
    assert sel(density=0.0) == bb.ERR_INVALID_ARG
    assert sel(tokens_capacity=2 * 4 * 128 - 1) == bb.ERR_CAPACITY
    assert sel(ws_bytes=256) == bb.ERR_WORKSPACE


def test_query_groups_workspace_and_arguments(lib):
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for d in (64, 128):
        n = 2 * 3 * 1024
        slots = 2 * 3 * (1024 // 128)  # one per group of each head
        # working permutation, 64-bit (projection, row) keys, scratch copy; per slot a slice's
        # row sum, its scatter blocks (136 of (d/16)^2 entries), a segment's mean and direction
        want = (256 + up(n * 4) + up(n * 8) + up(n * 4) + up(slots * d * 4)
                + up(slots * (d * d // 256 * 136) * 4) + up(slots * 2 * d * 4))
        assert bb.bsa_workspace_size(4, 2, 3, 1024, d, 64) == want

    def grp(**kw):
        args = dict(Q=FAKE, dt=bb.BF16, B=1, H=2, N=512, d=64, perm=FAKE, ws=FAKE, ws_bytes=1 << 30)
        args.update(kw)
        with pytest.raises(bb.BsaError) as e:
            bb.bsa_query_groups(**args, stream=0)
        return e.value.code

    assert grp(N=500) == bb.ERR_SHAPE
    assert grp(N=128 * 513) == bb.ERR_SHAPE  # at most 512 groups per head
    assert grp(d=32) == bb.ERR_SHAPE
    assert grp(B=300, H=300) == bb.ERR_SHAPE  # one grid row per head
    assert grp(dt=2) == bb.ERR_DTYPE
    assert grp(perm=None) == bb.ERR_INVALID_ARG
    assert grp(ws_bytes=1024) == bb.ERR_WORKSPACE


def test_token_forward_rejects_bad_arguments(lib):
    assert _fwd_tok(N=500) == bb.ERR_SHAPE          # groups of 128 queries
    assert _fwd_tok(d=96) == bb.ERR_SHAPE
    assert _fwd_tok(B=300, H=300) == bb.ERR_SHAPE   # one grid row per head
    assert _fwd_tok(dt=7) == bb.ERR_DTYPE
    assert _fwd_tok(perm=None) == bb.ERR_INVALID_ARG
    assert _fwd_tok(tokens=FAKE + 2) == bb.ERR_INVALID_ARG
    assert _fwd_tok(n_tokens=0) == bb.ERR_INVALID_ARG
    assert _fwd_tok(n_tokens=513) == bb.ERR_INVALID_ARG
    assert _fwd_tok(scale=float("nan")) == bb.ERR_INVALID_ARG
    assert _fwd_tok(ws=None) == bb.ERR_WORKSPACE
    assert _fwd_tok(ws_bytes=255) == bb.ERR_WORKSPACE


def test_residual_entry_points_reject_bad_arguments(lib):
    # bsa_forward_residual: the residual pointer, then every bsa_forward check
    assert _fwd_res(R=None) == bb.ERR_INVALID_ARG
    assert _fwd_res(R=FAKE + 4) == bb.ERR_INVALID_ARG  # fp32 rows read 16 bytes at a time
    assert _fwd_res(N=0) == bb.ERR_SHAPE
    assert _fwd_res(dt=5) == bb.ERR_DTYPE
    assert _fwd_res(workspace=None) == bb.ERR_WORKSPACE
    # bsa_residual_capture
    for kw, code in [(dict(dt=9), bb.ERR_DTYPE), (dict(count=-1), bb.ERR_INVALID_ARG),
                     (dict(R=None), bb.ERR_INVALID_ARG), (dict(O_dense=FAKE + 2), bb.ERR_INVALID_ARG)]:
        args = dict(O_dense=FAKE, O_sparse=FAKE, dt=bb.BF16, count=1024, R=FAKE)
        args.update(kw)
        with pytest.raises(bb.BsaError) as e:
            bb.bsa_residual_capture(**args, stream=0)
        assert e.value.code == code
    bb.bsa_residual_capture(None, None, bb.BF16, 0, None, stream=0)  # nothing to do, nothing enqueued


def test_modal_counts_and_rejects_bad_arguments(lib):
    # 2 text + 64 image blocks (t2i): text rows keep 2 + 32, image rows 1 + 9
    dens = [1.0, 0.5, 0.5, 0.15]
    assert bb.bsa_mask_nnz_modal(2, 24, 4224, 64, 2, dens) == 48 * (2 * (2 + 32) + 64 * (1 + 9))
    assert bb.bsa_mask_nnz_modal(1, 1, 512, 64, 0, [0.5, 0.5, 0.5, 0.25]) == 8 * 2  # the plain selector
    assert bb.bsa_mask_nnz_modal(1, 1, 512, 64, 8, [0.0, 0.0, 0.0, 0.0]) == 0
    for bad in ([1.5, 0, 0, 0], [-0.1, 0, 0, 0], [float("nan"), 0, 0, 0]):
        with pytest.raises(bb.BsaError) as e:
            bb.bsa_mask_nnz_modal(1, 1, 512, 64, 2, bad)
        assert e.value.code == bb.ERR_INVALID_ARG
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_mask_nnz_modal(1, 1, 512, 64, 9, dens)  # more text blocks than blocks
    assert e.value.code == bb.ERR_INVALID_ARG
    args = dict(Q=FAKE, K=FAKE, dt=bb.BF16, B=1, H=2, N=512, d=64, block=64, n_text_blocks=2, density=dens,
                row_ptr=FAKE, col_idx=FAKE, col_capacity=1 << 20, bitmap=FAKE, workspace=FAKE,
                workspace_bytes=1 << 30)
    for kw, code in [(dict(N=0), bb.ERR_SHAPE), (dict(dt=4), bb.ERR_DTYPE), (dict(Q=None), bb.ERR_INVALID_ARG),
                     (dict(n_text_blocks=-1), bb.ERR_INVALID_ARG), (dict(density=[2.0, 0, 0, 0]), bb.ERR_INVALID_ARG),
                     (dict(workspace=None), bb.ERR_WORKSPACE), (dict(col_capacity=3), bb.ERR_CAPACITY)]:
        a = dict(args)
        a.update(kw)
        with pytest.raises(bb.BsaError) as e:
            bb.bsa_build_mask_modal(**a, stream=0)
        assert e.value.code == code


def test_exact_selector_workspace_and_bad_arguments(lib):
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # partial masses: 4 per 128-row tile and KV block
    assert bb.bsa_workspace_size(2, 1, 24, 8192, 128, 64) == 256 + up(24 * 64 * 4 * 128 * 4)
    args = dict(Q=FAKE, K=FAKE, dt=bb.BF16, B=1, H=2, N=512, d=64, block=64, density=0.25, scale=0.0, LSE=FAKE,
                row_ptr=FAKE, col_idx=FAKE, col_capacity=1 << 20, bitmap=FAKE, workspace=FAKE,
                workspace_bytes=1 << 30)
    for kw, code in [(dict(dt=bb.FP32), bb.ERR_UNSUPPORTED), (dict(dt=7), bb.ERR_DTYPE),
                     (dict(LSE=None), bb.ERR_INVALID_ARG), (dict(density=0.0), bb.ERR_INVALID_ARG),
                     (dict(scale=float("inf")), bb.ERR_INVALID_ARG), (dict(N=0), bb.ERR_SHAPE),
                     (dict(workspace_bytes=16), bb.ERR_WORKSPACE), (dict(col_capacity=15), bb.ERR_CAPACITY)]:
        a = dict(args)
        a.update(kw)
        with pytest.raises(bb.BsaError) as e:
            bb.bsa_build_mask_exact(**a, stream=0)
        assert e.value.code == code


def test_tokens_per_group_count(lib):
    # K = max(1, floor(density * N)), density as fp32, at most N
    assert bb.bsa_tokens_per_group(8192, 0.15) == 1228
    assert bb.bsa_tokens_per_group(1024, 0.1) == 102
    assert bb.bsa_tokens_per_group(128, 1e-6) == 1
    assert bb.bsa_tokens_per_group(128, 1.0) == 128
    # 0.3 in fp32 is 0.30000001192..., so 10 * it floors to 3, not 2
    assert bb.bsa_tokens_per_group(10, 0.3) == 3
    for bad in (0.0, -0.1, 1.5, float("nan")):
        with pytest.raises(bb.BsaError) as e:
            bb.bsa_tokens_per_group(1024, bad)
        assert e.value.code == bb.ERR_INVALID_ARG
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_tokens_per_group(0, 0.5)
    assert e.value.code == bb.ERR_SHAPE
