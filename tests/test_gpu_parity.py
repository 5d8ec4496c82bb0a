"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Index (bitmap, row_ptr, col_idx) must match bit for bit; O within max-abs 2e-2
and mean-abs 2e-3, LSE within 1e-3 (bf16 inputs, fp32 accumulation). Small
cases compare every row; the full-size workloads compare a seeded sample of
rows plus the whole index.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_mean_gb300 import binding as bb
from block_sparse_attention_mean_gb300 import build as bbuild
from block_sparse_attention_mean_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bbuild.build()
    bb.load()
    bb.bsa_debug_config(0, 0)


def run_workload(w, index_mode=None, rows=None, scale=None):
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    mask = gu.oracle_mask(w, inp)
    idx = gu.device_index(w, q, k, mask)
    gu.assert_index_equal(idx, mask)
    mode = w.index_mode if index_mode is None else index_mode
    O, L = bb.forward(q, k, v, idx, index_mode=mode, scale=0.0 if scale is None else scale)
    torch.cuda.synchronize()
    return gu.assert_attention_close(O, L, inp, mask, w, rows=rows, scale=scale)


# ------------------------------------------------------------ small, all rows


def test_tiny_fp32_explicit():
    run_workload(wl.WORKLOADS["tiny"])


def test_tiny_bf16_both_index_modes():
    w = wl.scaled(wl.WORKLOADS["tiny"], dtype="bf16")
    run_workload(w, index_mode=0)
    run_workload(w, index_mode=1)


def test_t2i_two_heads_all_rows():
    run_workload(wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2))


def test_t2i_ragged_tile_tail_all_rows():
    # 67 blocks of 64: the last 128-row tile holds a single Q block
    w = wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2, N=64 * 67)
    run_workload(w)


def test_dynamic_topk_small_all_rows():
    run_workload(wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2048))


@pytest.mark.parametrize("nB", [128, 130, 200, 257])
def test_selector_score_tiles_all_columns(nB):
    # the scorer works on 64 x 64 tiles of (Q block, KV block) pairs: full tiles (128), and
    # ragged last tiles of Q rows and of KV columns holding 2, 8 and 1 blocks (130, 200, 257)
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=1, N=64 * nB, density=0.2)
    inp = wl.make_inputs(w)
    q, k = gu.upload(inp, "q"), gu.upload(inp, "k")
    mask = gu.oracle_mask(w, inp)
    gu.assert_index_equal(gu.device_index(w, q, k, mask), mask)


def test_long_block128_small_all_rows():
    run_workload(wl.scaled(wl.WORKLOADS["long_topk"], H=2, N=4096))


def test_video_small_grid_all_rows():
    w = wl.scaled(wl.WORKLOADS["video_cuboid"], H=2, N=256 + 8 * 16 * 16, grid=(2, 4, 4),
                  video_shape=(8, 16, 16))
    run_workload(w)


# ------------------------------------------------------------ ragged last block
#
# N not a multiple of the block size: the last block holds the keys and query rows up to
# N (the tile loop's padding mask) and pooling averages the tokens it holds. Index bit for
# bit, then the forward in both index modes and with every tile split.

RAGGED_CASES = {
    "tiny_fp32": wl.scaled(wl.WORKLOADS["tiny"], N=475),                           # SIMT path
    "t2i_d64_bs64": wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2, N=4224 - 40),  # last block: 24 rows
    "dynamic_d128_bs64": wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=1000),     # last block: 40 rows
    "long_d128_bs128": wl.scaled(wl.WORKLOADS["long_sweep_bs128"], H=2, N=1000, density=0.5),
    "d64_bs128": wl.scaled(wl.WORKLOADS["long_sweep_bs128"], H=2, N=900, d=64, density=0.5),
}


@pytest.mark.parametrize("name", sorted(RAGGED_CASES))
def test_ragged_sequence_matches_oracle(name):
    w = RAGGED_CASES[name]
    assert w.N % w.block != 0
    run_workload(w)
    if w.dtype == "bf16":
        run_workload(w, index_mode=1 - w.index_mode)
        _run_with_flags(w, bb.DBG_SPLIT_ALL)


# ------------------------------------------------------------ split query tiles
#
# A tile whose step count is well above the per-CTA share is split by KV block
# range into chunks that separate CTAs run; the last to finish merges the partial
# (O, max, sums). The debug flags force the split for every tile (with empty
# chunks, ragged ranges and many merges) or forbid it; both must match the oracle.

SPLIT_CASES = {
    "t2i": wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2),
    "dynamic": wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2048),
    "video": wl.scaled(wl.WORKLOADS["video_cuboid"], H=2, N=256 + 8 * 16 * 16, grid=(2, 4, 4),
                       video_shape=(8, 16, 16)),
    # block 128, bitmap index; 16 of 64 blocks per row so that tiles have steps to split
    "long_bitmap": wl.scaled(wl.WORKLOADS["long_topk"], H=2, N=8192, density=0.25),
}


def _run_with_flags(w, flags):
    """Forward under debug `flags`; checks the outputs and returns the launch's item count."""
    bb.bsa_debug_config(flags, 0)
    try:
        inp = wl.make_inputs(w)
        q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
        mask = gu.oracle_mask(w, inp)
        idx = gu.device_index(w, q, k, mask)
        ws = bb.workspace(1, w.B, w.H, w.N, w.d, w.block)
        O, L = bb.forward(q, k, v, idx, index_mode=w.index_mode, ws=ws)
        torch.cuda.synchronize()
        n_items = int(ws[12:16].view(torch.int32).item())  # workspace header: work items of the launch
        gu.assert_attention_close(O, L, inp, mask, w)
        return n_items
    finally:
        bb.bsa_debug_config(0, 0)


@pytest.mark.parametrize("name", sorted(SPLIT_CASES))
def test_split_tiles_match_oracle(name):
    w = SPLIT_CASES[name]
    tiles = w.B * w.H * ((w.N + 127) // 128)
    assert _run_with_flags(w, bb.DBG_SPLIT_ALL) > tiles
    assert _run_with_flags(w, bb.DBG_NO_SPLIT) == tiles


@pytest.mark.parametrize("flags", [0, bb.DBG_SPLIT_ALL])
def test_many_tiles_multi_cta_ordering(flags):
    # more than 8192 query tiles: the work list is built by the multi-CTA ordering
    # launch (smaller problems use the single-CTA one); sampled rows against the oracle
    w = wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=128, N=64 * 130)
    tiles = w.B * w.H * ((w.N + 127) // 128)
    assert tiles > 8192
    bb.bsa_debug_config(flags, 0)
    try:
        inp = wl.make_inputs(w)
        q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
        mask = gu.oracle_mask(w, inp)
        idx = gu.device_index(w, q, k, mask)
        ws = bb.workspace(1, w.B, w.H, w.N, w.d, w.block)
        O, L = bb.forward(q, k, v, idx, index_mode=w.index_mode, ws=ws)
        torch.cuda.synchronize()
        n_items = int(ws[12:16].view(torch.int32).item())
        assert n_items > tiles if flags else n_items >= tiles
        rows = gu.sample_rows(w, np.random.default_rng(23), blocks_per_head=2, rows_per_block=4)
        gu.assert_attention_close(O, L, inp, mask, w, rows=rows)
    finally:
        bb.bsa_debug_config(0, 0)


def _expected_work_list(w, mask):
    """Unsplit tiles in the kernel's order: tiles of at least share / 8 steps longest first
    (ties in tile order), then the rest in tile order. A tile's length is the sum of its Q
    blocks' active counts (clamped like the kernel's 1024 length buckets); the share is the
    total over the resident CTAs of the launch (SMs x CTAs per SM, at most the tiles plus the
    partial slots), at least 4."""
    counts = mask.reshape(w.B * w.H, w.nQB, w.nKB).sum(axis=2)
    per = 2 if w.block == 64 else 1
    tiles_per_bh = (w.N + 127) // 128
    lens = []
    for bh in range(w.B * w.H):
        for qt in range(tiles_per_bh):
            lens.append(int(counts[bh, per * qt:per * qt + per].sum()))
    lens = np.array(lens)
    n_tiles = lens.size
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid = min(n_tiles + min(8 * n_tiles, 640), sms * (2 if w.block == 64 else 1))
    share = max(-(-int(lens.sum()) // grid), 4)
    long_min = max(share // 8, 1)
    tiles = np.arange(n_tiles)
    is_long = lens >= long_min
    clamped = np.minimum(lens, 1022)
    head = tiles[is_long][np.lexsort((tiles[is_long], -clamped[is_long]))]
    return np.concatenate([head, tiles[~is_long]]).astype(np.int32)


ORDER_CASES = {
    "t2i_csr": wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=4),
    "video_csr": wl.scaled(wl.WORKLOADS["video_cuboid"], H=2),
    "long_bitmap": wl.scaled(wl.WORKLOADS["long_topk"], H=16, N=8192),
    "t2i_csr_multi_cta": wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=128, N=64 * 130),
}


@pytest.mark.parametrize("name", sorted(ORDER_CASES))
def test_work_list_is_longest_first_then_tile_order(name):
    # row a6: the work list is a stable counting sort (long tiles by length descending, ties
    # in tile order, then the rest in tile order), which keeps a head's tiles together;
    # single-CTA (CSR) and multi-CTA (bitmap, or more than 8192 tiles) ordering launches, no
    # splitting
    w = ORDER_CASES[name]
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    mask = gu.oracle_mask(w, inp)
    idx = gu.device_index(w, q, k, mask)
    ws = bb.workspace(1, w.B, w.H, w.N, w.d, w.block)
    bb.bsa_debug_config(bb.DBG_NO_SPLIT, 0)
    try:
        bb.forward(q, k, v, idx, index_mode=w.index_mode, ws=ws)
        torch.cuda.synchronize()
    finally:
        bb.bsa_debug_config(0, 0)
    expect = _expected_work_list(w, mask)
    n_items = int(ws[12:16].view(torch.int32).item())
    assert n_items == expect.size
    items = ws[256:256 + 4 * n_items].view(torch.int32).cpu().numpy()
    assert np.array_equal(items, expect)


# ------------------------------------------------------------ residual compensation
#
# [P3] section "残差补偿找回被丢弃的尾部": R = O_dense - O_sparse at an anchor step, and
# later steps output O_sparse + R. The capture must equal the fp32 difference bit
# for bit; the compensated forward of a later step (other inputs) must match the
# oracle's sparse attention plus the same R; at the anchor it gives the dense output.

RESIDUAL_CASES = {
    "t2i": wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2),
    "dynamic": wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2048),
    "long_bitmap": wl.scaled(wl.WORKLOADS["long_topk"], H=2, N=8192, density=0.25),
    "tiny_fp32": wl.WORKLOADS["tiny"],
}


def _step(w, inp):
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    mask = gu.oracle_mask(w, inp)
    return q, k, v, mask, gu.device_index(w, q, k, mask)


def _full_index(w):
    """Every KV block active for every Q block: the dense reference of the anchor step."""
    ones = np.ones((w.B, w.H, w.nQB, w.nKB), dtype=np.uint8)
    dev = torch.from_numpy(gu.mask_bitmap_words(ones).reshape(-1)).cuda()
    return bb.build_mask(None, None, w.block, spec=bb.explicit_spec(dev), shape=(w.B, w.H, w.N, w.d))


@pytest.mark.parametrize("flags", [0, bb.DBG_SPLIT_ALL])
@pytest.mark.parametrize("name", sorted(RESIDUAL_CASES))
def test_residual_compensation_matches_oracle(name, flags):
    w = RESIDUAL_CASES[name]
    bb.bsa_debug_config(flags, 0)
    try:
        # anchor step: dense (every block active) and sparse outputs, then R
        inp0 = wl.make_inputs(w)
        q0, k0, v0, mask0, idx0 = _step(w, inp0)
        full = np.ones_like(mask0)
        idx_full = _full_index(w)
        gu.assert_index_equal(idx_full, full)
        O_dense, _ = bb.forward(q0, k0, v0, idx_full, index_mode=w.index_mode)
        O_sparse, _ = bb.forward(q0, k0, v0, idx0, index_mode=w.index_mode)
        R = bb.residual_capture(O_dense, O_sparse)
        torch.cuda.synchronize()
        expect = (O_dense.float() - O_sparse.float()).cpu().numpy()
        assert np.array_equal(R.cpu().numpy(), expect)  # fp32 difference, bit for bit
        R_np = R.cpu().numpy().reshape(-1, w.d).astype(np.float64)
        # at the anchor, compensation gives the dense output (oracle, full mask)
        O_a, L_a = bb.forward(q0, k0, v0, idx0, index_mode=w.index_mode, residual=R)
        torch.cuda.synchronize()
        Od_ref, _ = oracle.attention(inp0["q"], inp0["k"], inp0["v"], full, w.block)
        err = np.abs(O_a.float().reshape(-1, w.d).cpu().numpy() - Od_ref)
        assert err.max() <= gu.O_MAX_ABS and err.mean() <= gu.O_MEAN_ABS
        # a later step: other inputs, the anchor's R
        inp1 = wl.make_inputs(wl.scaled(w, seed=w.seed + 1000))
        q1, k1, v1, mask1, idx1 = _step(w, inp1)
        O1, L1 = bb.forward(q1, k1, v1, idx1, index_mode=w.index_mode, residual=R)
        torch.cuda.synchronize()
        Os_ref, L_ref = oracle.attention(inp1["q"], inp1["k"], inp1["v"], mask1, w.block)
        O_ref = oracle.compensate(Os_ref, R_np)
        err = np.abs(O1.float().reshape(-1, w.d).cpu().numpy() - O_ref)
        assert err.max() <= gu.O_MAX_ABS, f"O max-abs {err.max():.3e}"
        assert err.mean() <= gu.O_MEAN_ABS, f"O mean-abs {err.mean():.3e}"
        Lg = L1.reshape(-1).cpu().numpy().astype(np.float64)
        live = ~np.isneginf(L_ref)
        assert np.array_equal(np.isneginf(Lg), ~live)
        assert np.abs(Lg[live] - L_ref[live]).max() <= gu.LSE_MAX_ABS  # the LSE stays the sparse one
    finally:
        bb.bsa_debug_config(0, 0)


# ------------------------------------------------------------ per-modality top-k
#
# [P1] §3.3: a density per (query modality, key modality) group. The index must equal
# the oracle's bit for bit, and the forward over it must match the oracle.

MODAL_CASES = {
    # t2i recipe (rank-8 shared component), 2 text blocks: text rows dense over text, half of the image
    "t2i_text2": (wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2, mask=wl.TOPK, density=0.1), 2,
                  [1.0, 0.5, 0.5, 0.15]),
    # clustered recipe at d = 128, 4 "text" blocks, one group switched off
    "dynamic_text4": (wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2048), 4, [0.75, 0.0, 0.25, 0.2]),
    # block 128, bitmap index
    "long_text2": (wl.scaled(wl.WORKLOADS["long_topk"], H=2, N=4096), 2, [1.0, 0.1, 1.0, 0.05]),
}


@pytest.mark.parametrize("name", sorted(MODAL_CASES))
def test_modal_index_and_forward_match_oracle(name):
    w, n_text, dens = MODAL_CASES[name]
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    mask = oracle.select_mask_modal(inp["q"], inp["k"], w.block, n_text, dens)
    idx = bb.build_mask_modal(q, k, w.block, n_text, dens)
    assert idx.nnz == int(mask.sum())
    gu.assert_index_equal(idx, mask)
    O, L = bb.forward(q, k, v, idx, index_mode=w.index_mode)
    torch.cuda.synchronize()
    gu.assert_attention_close(O, L, inp, mask, w)


def test_modal_builder_without_text_is_the_plain_selector():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=4096)
    inp = wl.make_inputs(w)
    q, k = gu.upload(inp, "q"), gu.upload(inp, "k")
    plain = bb.build_mask(q, k, w.block, density=w.density, shape=(w.B, w.H, w.N, w.d))
    modal = bb.build_mask_modal(q, k, w.block, 0, [0.5, 0.5, 0.5, w.density])
    torch.cuda.synchronize()
    assert torch.equal(plain.row_ptr, modal.row_ptr)
    assert torch.equal(plain.col_idx[:plain.nnz], modal.col_idx[:modal.nnz])
    assert torch.equal(plain.bitmap, modal.bitmap)


# ------------------------------------------------------------ planned work list
#
# bsa_forward_plan makes the forward's work list once; bsa_forward with BSA_INDEX_PLANNED
# reuses it. Planned calls must equal the unplanned call bit for bit, call after call (the
# forward resets its scheduler and merge counters itself), with and without split tiles.

PLAN_CASES = {
    "t2i_csr": (wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=4), 0),
    "video_bitmap": (wl.scaled(wl.WORKLOADS["video_cuboid"], H=2), 1),
    "dynamic_csr": (wl.scaled(wl.WORKLOADS["dynamic_topk"], H=3, N=4096), 0),
    "long_bitmap": (wl.scaled(wl.WORKLOADS["long_topk"], H=2, N=8192), 1),
}


@pytest.mark.parametrize("flags", [0, bb.DBG_SPLIT_ALL])
@pytest.mark.parametrize("name", sorted(PLAN_CASES))
def test_planned_forward_equals_unplanned(name, flags):
    w, mode = PLAN_CASES[name]
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    mask = gu.oracle_mask(w, inp)
    idx = gu.device_index(w, q, k, mask)
    bb.bsa_debug_config(flags, 0)
    try:
        O0, L0 = bb.forward(q, k, v, idx, index_mode=mode)
        ws = bb.forward_plan(q, idx, index_mode=mode)
        outs = [bb.forward(q, k, v, idx, index_mode=mode | bb.INDEX_PLANNED, ws=ws) for _ in range(3)]
        split_items = int(ws[12:16].view(torch.int32).item())  # n_items in the header
    finally:
        bb.bsa_debug_config(0, 0)
    torch.cuda.synchronize()
    if flags:
        assert split_items > w.B * w.H * (-(-w.N // 128))  # the plan holds chunks of split tiles
    for O, L in outs:
        assert torch.equal(O, O0)
        assert torch.equal(L, L0)
    gu.assert_attention_close(O0, L0, inp, mask, w)


@pytest.mark.parametrize("name", ["t2i_static", "video_cuboid"])
def test_planned_forward_full_size_static_masks(name):
    # the configurations the bench plans once: at full size, three planned calls equal the
    # unplanned call bit for bit, and sampled rows match the oracle
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    mask = gu.oracle_mask(w, inp)
    idx = gu.device_index(w, q, k, mask)
    O0, L0 = bb.forward(q, k, v, idx, index_mode=w.index_mode)
    ws = bb.forward_plan(q, idx, index_mode=w.index_mode)
    for _ in range(3):
        O, L = bb.forward(q, k, v, idx, index_mode=w.index_mode | bb.INDEX_PLANNED, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(O, O0) and torch.equal(L, L0)
    rng = np.random.default_rng(21)
    gu.assert_attention_close(O0, L0, inp, mask, w, rows=gu.sample_rows(w, rng, blocks_per_head=4, rows_per_block=4))


def test_planned_fp32_forward_is_the_plain_forward():
    # the CUDA-core fp32 forward keeps no work list: planning is a no-op and the planned flag
    # changes nothing
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    mask = gu.oracle_mask(w, inp)
    idx = gu.device_index(w, q, k, mask)
    O0, L0 = bb.forward(q, k, v, idx)
    ws = bb.forward_plan(q, idx)
    O, L = bb.forward(q, k, v, idx, index_mode=bb.INDEX_PLANNED, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(O, O0)
    assert torch.equal(L, L0)
    gu.assert_attention_close(O, L, inp, mask, w)


def test_planned_residual_forward_equals_unplanned():
    w = wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2)
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    idx = gu.device_index(w, q, k, gu.oracle_mask(w, inp))
    R = torch.randn(q.shape, dtype=torch.float32, device="cuda") * 0.01
    O0, L0 = bb.forward(q, k, v, idx, residual=R)
    ws = bb.forward_plan(q, idx)
    for _ in range(2):
        O, L = bb.forward(q, k, v, idx, index_mode=bb.INDEX_PLANNED, ws=ws, residual=R)
        torch.cuda.synchronize()
        assert torch.equal(O, O0)
        assert torch.equal(L, L0)


def test_planned_forward_needs_its_own_plan():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2048)
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    mask = gu.oracle_mask(w, inp)
    idx = gu.device_index(w, q, k, mask)
    ws = bb.workspace(1, w.B, w.H, w.N, w.d, w.block)
    # no plan in a fresh workspace: an argument error raised on the device, nothing run
    bb.forward(q, k, v, idx, index_mode=bb.INDEX_PLANNED, ws=ws, check=False)
    assert bb.bsa_check_device_error(ws) == bb.ERR_INVALID_ARG
    # a plan for the bitmap index is not a plan for the CSR one
    bb.forward_plan(q, idx, index_mode=1, ws=ws)
    bb.forward(q, k, v, idx, index_mode=0 | bb.INDEX_PLANNED, ws=ws, check=False)
    assert bb.bsa_check_device_error(ws) == bb.ERR_INVALID_ARG
    # the matching plan runs, and an unplanned call leaves a usable plan too
    bb.forward_plan(q, idx, index_mode=0, ws=ws)
    O, L = bb.forward(q, k, v, idx, index_mode=bb.INDEX_PLANNED, ws=ws)
    gu.assert_attention_close(O, L, inp, mask, w)
    bb.forward(q, k, v, idx, index_mode=1, ws=ws)
    O, L = bb.forward(q, k, v, idx, index_mode=1 | bb.INDEX_PLANNED, ws=ws)
    gu.assert_attention_close(O, L, inp, mask, w)


# ------------------------------------------------------------ LSE only
#
# bsa_forward_lse runs the forward's QK^T and softmax sums only. Its LSE must be the full
# forward's bit for bit (the full forward without split tiles: a split tile's LSE is merged in
# another order) and match the oracle.

LSE_CASES = {
    "dynamic_csr": (wl.scaled(wl.WORKLOADS["dynamic_topk"], H=3, N=4096), 0),        # d128 bs64, one thread per row
    "long_bitmap": (wl.scaled(wl.WORKLOADS["long_topk"], H=2, N=8192), 1),           # d128 bs128, four lanes per row
    "t2i_csr": (wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=4), 0),                 # d64 bs64
    "d64_bs128": (wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2, N=2048, block=128, mask=wl.TOPK,
                            density=0.25), 1),
    "ragged": (wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2000), 0),
    "fp32_tiny": (wl.WORKLOADS["tiny"], 0),
}


@pytest.mark.parametrize("name", sorted(LSE_CASES))
def test_forward_lse_is_the_forward_lse(name):
    w, mode = LSE_CASES[name]
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    mask = gu.oracle_mask(w, inp)
    idx = gu.device_index(w, q, k, mask)
    bb.bsa_debug_config(bb.DBG_NO_SPLIT, 0)
    try:
        _, L0 = bb.forward(q, k, v, idx, index_mode=mode)
    finally:
        bb.bsa_debug_config(0, 0)
    L = bb.forward_lse(q, k, idx, index_mode=mode)
    torch.cuda.synchronize()
    assert torch.equal(L, L0)
    _, L_ref = oracle.attention(inp["q"], inp["k"], inp["v"], mask, w.block, rows=None)
    assert np.abs(L.reshape(-1).cpu().numpy().astype(np.float64) - L_ref).max() <= gu.LSE_MAX_ABS


def test_forward_lse_dense_and_empty_rows():
    # every block active (the exact selectors' pass 1) and rows with no active block (-inf)
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2048)
    inp = wl.make_inputs(w)
    q, k = gu.upload(inp, "q"), gu.upload(inp, "k")
    full = np.ones((w.B, w.H, w.nQB, w.nKB), dtype=np.uint8)
    full[0, 1, 3:5, :] = 0  # two Q blocks of head 1 attend to nothing
    idx = bb.build_mask(None, None, w.block, spec=bb.explicit_spec(
        torch.from_numpy(gu.mask_bitmap_words(full).reshape(-1)).cuda()), shape=(w.B, w.H, w.N, w.d))
    L = bb.forward_lse(q, k, idx).reshape(-1).cpu().numpy().astype(np.float64)
    _, L_ref = oracle.attention(inp["q"], inp["k"], inp["v"], full, w.block, rows=None)
    empty = np.isneginf(L_ref)
    assert empty.sum() == 2 * w.block and np.all(np.isneginf(L[empty]))
    assert np.abs(L[~empty] - L_ref[~empty]).max() <= gu.LSE_MAX_ABS


def test_forward_lse_full_size_dense_anchor_pass():
    # the token path's anchor pass at its working shape (B1 H24 N8192 d128): the LSE-only
    # forward over an all-active block-128 index equals the full forward's LSE bit for bit and
    # the oracle's dense LSE on sampled rows
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], block=128)
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    nb = w.N // 128
    full = np.ones((w.B, w.H, nb, nb), dtype=np.uint8)
    idx = bb.build_mask(None, None, 128, spec=bb.explicit_spec(
        torch.from_numpy(gu.mask_bitmap_words(full).reshape(-1)).cuda()), shape=(w.B, w.H, w.N, w.d))
    L = bb.forward_lse(q, k, idx)
    bb.bsa_debug_config(bb.DBG_NO_SPLIT, 0)
    try:
        _, L0 = bb.forward(q, k, v, idx)
    finally:
        bb.bsa_debug_config(0, 0)
    torch.cuda.synchronize()
    assert torch.equal(L, L0)
    rng = np.random.default_rng(22)
    rows = gu.sample_rows(w, rng, blocks_per_head=4, rows_per_block=4)
    _, L_ref = oracle.attention(inp["q"], inp["k"], inp["v"], full, 128, rows=rows)
    assert np.abs(L.reshape(-1).cpu().numpy().astype(np.float64)[rows] - L_ref).max() <= gu.LSE_MAX_ABS


# ------------------------------------------------------------ block-oracle selector
#
# [P3] section "质量差距有三个可分离来源": keep the blocks with the most exact attention
# mass. Pass 1 is the dense LSE; bsa_build_mask_exact is pass 2 and the selection.
# The masses are floating point, so the selection is checked for validity: every
# kept block is within the tolerance of the k-th largest mass, and rows whose k-th
# and (k+1)-th masses are clearly apart select exactly the oracle's blocks.

EXACT_CASES = {
    "d64_bs64": (wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2, N=2048), 0.15),
    "d128_bs64": (wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2048), 0.15),
    "d64_bs128": (wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2, N=2048, block=128), 0.25),
    "d128_bs128": (wl.scaled(wl.WORKLOADS["long_topk"], H=2, N=4096), 0.1),
    # ragged last block: 32 blocks of 64, the last holding 16 keys (zero-filled loads, masked)
    "d128_bs64_ragged": (wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2000), 0.15),
}
MASS_RTOL = 2e-3


def _gpu_masses(ws, w):
    """Block masses from the selector's workspace partials, summed in the kernel's order."""
    BH, nB, tpb = w.B * w.H, w.nQB, (w.N + 127) // 128
    part = ws[256:256 + BH * tpb * 4 * nB * 4].view(torch.float32).reshape(BH, tpb, 4, nB).cpu().numpy()
    out = np.empty((BH, nB, nB), np.float32)
    for i in range(nB):
        if w.block == 128:
            p = part[:, i]
            out[:, i] = ((p[:, 0] + p[:, 1]) + p[:, 2]) + p[:, 3]
        else:
            h = i % 2
            out[:, i] = part[:, i // 2, 2 * h] + part[:, i // 2, 2 * h + 1]
    return out


def _check_selection(idx, mass_ref, k):
    """Counts, bitmap/CSR agreement, and the kept set against the exact masses."""
    R, nB = int(np.prod(mass_ref.shape[:-1])), mass_ref.shape[-1]
    rp = idx.row_ptr.cpu().numpy()
    ci = idx.col_idx.cpu().numpy()
    assert np.array_equal(rp, np.arange(R + 1) * k)
    m = mass_ref.reshape(R, nB)
    sel = np.zeros((R, nB), np.uint8)
    exact_rows = 0
    for r in range(R):
        cols = ci[rp[r]:rp[r + 1]]
        assert np.all(np.diff(cols) > 0)
        sel[r, cols] = 1
        order = np.sort(m[r])[::-1]
        kth = order[k - 1]
        tol = MASS_RTOL * kth
        assert np.all(m[r, cols] >= kth - tol), f"row {r} keeps a block below the k-th mass"
        if k < nB and order[k - 1] - order[k] > 2 * tol:
            exact_rows += 1
            assert set(cols.tolist()) == set(np.argsort(-m[r], kind="stable")[:k].tolist())
    _, _, bitmap_ref = oracle.mask_to_index(sel.reshape(mass_ref.shape))
    assert np.array_equal(idx.bitmap.cpu().numpy().view(np.uint32), bitmap_ref.reshape(-1))
    assert exact_rows > R // 2  # most rows have no near tie at the boundary
    return sel


@pytest.mark.parametrize("name", sorted(EXACT_CASES))
def test_exact_selector_masses_and_selection(name):
    w, density = EXACT_CASES[name]
    inp = wl.make_inputs(w)
    q, k = gu.upload(inp, "q"), gu.upload(inp, "k")
    full = np.ones((w.B, w.H, w.nQB, w.nKB), dtype=np.uint8)
    _, lse = oracle.attention(inp["q"], inp["k"], inp["k"], full, w.block)  # pass 1 in double
    lse_dev = torch.from_numpy(lse.astype(np.float32)).cuda()
    idx, ws = bb.build_mask_exact(q, k, lse_dev, w.block, density)
    torch.cuda.synchronize()
    mass_ref = oracle.block_mass(inp["q"], inp["k"], lse, w.block)
    np.testing.assert_allclose(_gpu_masses(ws, w), mass_ref.reshape(-1, w.nQB, w.nKB), rtol=MASS_RTOL,
                               atol=1e-6 * w.block)
    _check_selection(idx, mass_ref, oracle.topk_count(density, w.nKB))


def test_exact_selector_end_to_end_with_gpu_pass_one():
    # pass 1 on the GPU (dense forward), pass 2 + selection, then the sparse forward on that index
    w, density = EXACT_CASES["d128_bs64"]
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    ones = np.ones((w.B, w.H, w.nQB, w.nKB), dtype=np.uint8)
    dense_idx = bb.build_mask(None, None, w.block, spec=bb.explicit_spec(
        torch.from_numpy(gu.mask_bitmap_words(ones).reshape(-1)).cuda()), shape=(w.B, w.H, w.N, w.d))
    _, lse_dense = bb.forward(q, k, v, dense_idx)
    idx, _ = bb.build_mask_exact(q, k, lse_dense, w.block, density)
    torch.cuda.synchronize()
    _, lse = oracle.attention(inp["q"], inp["k"], inp["k"], ones, w.block)
    sel = _check_selection(idx, oracle.block_mass(inp["q"], inp["k"], lse, w.block),
                           oracle.topk_count(density, w.nKB))
    O, L = bb.forward(q, k, v, idx, index_mode=w.index_mode)
    torch.cuda.synchronize()
    gu.assert_attention_close(O, L, inp, sel, w)


@pytest.mark.parametrize("d,block,mode", [(64, 128, 0), (64, 128, 1), (128, 64, 1), (64, 64, 1)])
def test_shape_combinations(d, block, mode):
    w = wl.scaled(wl.WORKLOADS["long_topk"], H=3, N=2048, d=d, block=block, density=0.3)
    run_workload(w, index_mode=mode)


def test_custom_scale():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=1, N=1024)
    run_workload(w, scale=0.05)


def test_single_block_sequences():
    for block in (64, 128):
        w = wl.scaled(wl.WORKLOADS["tiny"], dtype="bf16", N=block, block=block, d=128)
        run_workload(w)
    w = wl.scaled(wl.WORKLOADS["tiny"], dtype="bf16", N=128, block=64)
    run_workload(w)


def test_empty_and_full_rows():
    w = wl.scaled(wl.WORKLOADS["tiny"], dtype="bf16", H=3, N=1024, d=128)
    inp = wl.make_inputs(w)
    mask = inp["mask"].copy()
    mask[0, 0, 3, :] = 0          # one empty Q block (its tile partner is not empty)
    mask[0, 1, 4:6, :] = 0        # a whole empty 128-row tile
    mask[0, 2, :, :] = 0          # a head with one full row block and one single-block row
    mask[0, 2, 0, :] = 1
    mask[0, 2, 7, 15] = 1
    inp["mask"] = mask
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    for mode in (0, 1):
        idx = gu.device_index(w, q, k, mask)
        gu.assert_index_equal(idx, mask)
        O, L = bb.forward(q, k, v, idx, index_mode=mode)
        gu.assert_attention_close(O, L, inp, mask, w)


def test_fp32_shapes():
    for d, block in ((128, 128), (128, 64), (64, 128)):
        w = wl.scaled(wl.WORKLOADS["tiny"], H=1, N=512, d=d, block=block)
        run_workload(w)


def test_random_fuzz():
    rng = np.random.default_rng(7)
    for t in range(6):
        d = int(rng.choice([64, 128]))
        block = int(rng.choice([64, 128]))
        nb = int(rng.integers(1, 12))
        w = wl.scaled(wl.WORKLOADS["tiny"], dtype="bf16", H=int(rng.integers(1, 4)), N=nb * block, d=d,
                      block=block, mask_seed=100 + t, mask_p=float(rng.uniform(0.05, 0.9)), seed=50 + t)
        run_workload(w, index_mode=t % 2)


# ------------------------------------------------------------ properties


def test_csr_and_bitmap_bitwise_identical_and_deterministic():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=4, N=4096)
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    idx = bb.build_mask(q, k, w.block, density=w.density)
    idx2 = bb.build_mask(q, k, w.block, density=w.density)
    assert torch.equal(idx.col_idx, idx2.col_idx) and torch.equal(idx.bitmap, idx2.bitmap)
    O0, L0 = bb.forward(q, k, v, idx, index_mode=0)
    O1, L1 = bb.forward(q, k, v, idx, index_mode=1)
    O2, L2 = bb.forward(q, k, v, idx, index_mode=0)
    assert torch.equal(O0, O1) and torch.equal(L0, L1)
    assert torch.equal(O0, O2) and torch.equal(L0, L2)


@pytest.mark.parametrize("H", [13])
def test_build_eager_and_graph_replayed(H):
    # the builder's launches (the scoring and the selection with programmatic dependent
    # launch) captured in a CUDA graph: the eager build and two replays of the captured one
    # all give the oracle's index
    w = wl.scaled(wl.WORKLOADS["long_sweep_bs64"], H=H)
    inp = wl.make_inputs(w)
    q, k = gu.upload(inp, "q"), gu.upload(inp, "k")
    mask = gu.oracle_mask(w, inp)
    gu.assert_index_equal(gu.device_index(w, q, k), mask)
    nB, W = w.nQB, (w.nQB + 31) // 32
    cap = bb.bsa_mask_nnz(w.B, w.H, w.N, w.block, w.density, None)
    rp = torch.empty(w.B * w.H * nB + 1, dtype=torch.int32, device="cuda")
    ci = torch.empty(cap, dtype=torch.int32, device="cuda")
    bm = torch.empty(w.B * w.H * nB * W, dtype=torch.int32, device="cuda")
    ws = bb.workspace(0, w.B, w.H, w.N, w.d, w.block, q.device)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bb.bsa_build_mask(q, k, bb.BF16, w.B, w.H, w.N, w.d, w.block, w.density, None, rp, ci, cap, bm, ws,
                          ws.numel(), torch.cuda.current_stream())
    for _ in range(2):
        rp.fill_(-1), ci.fill_(-1), bm.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert bb.bsa_check_device_error(ws, s) == 0
        gu.assert_index_equal(bb.Index(rp, ci, bm, cap, w.block), mask)


def test_validate_index():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=2048)
    inp = wl.make_inputs(w)
    q, k = gu.upload(inp, "q"), gu.upload(inp, "k")
    idx = bb.build_mask(q, k, w.block, density=w.density)
    ws = bb.workspace(0, w.B, w.H, w.N, w.d, w.block)
    bb.bsa_validate_index(w.B, w.H, w.N, w.block, idx.row_ptr, idx.col_idx, idx.bitmap, ws, ws.numel())
    assert bb.bsa_check_device_error(ws) == bb.OK
    bad = idx.col_idx.clone()
    bad[5], bad[6] = bad[6].clone(), bad[5].clone()  # breaks ascending order within a row
    bb.bsa_validate_index(w.B, w.H, w.N, w.block, idx.row_ptr, bad, idx.bitmap, ws, ws.numel())
    assert bb.bsa_check_device_error(ws) == bb.ERR_INVALID_ARG
    assert bb.bsa_check_device_error(ws) == bb.OK  # cleared by the read


# ------------------------------------------------------------ device-raised errors


def test_nan_score_raises_nonfinite():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=1, N=1024)
    inp = wl.make_inputs(w)
    q, k = gu.upload(inp, "q"), gu.upload(inp, "k")
    q[0, 0, 5, 3] = float("nan")
    with pytest.raises(bb.BsaError) as e:
        bb.build_mask(q, k, w.block, density=w.density)
    assert e.value.code == bb.ERR_NONFINITE


@pytest.mark.parametrize("N", [512, 16384])
def test_broadcast_explicit_mask(N):
    # one bitmap for every (b, h), built once and copied into every head: index bit for bit
    # against the oracle's at two sizes, and the forward on the small one
    w = wl.scaled(wl.WORKLOADS["tiny"], dtype="bf16", B=2, H=3, N=N)
    rng = np.random.default_rng(N)
    one = (rng.random((w.nQB, w.nKB)) < 0.3).astype(np.uint8)
    one[np.arange(w.nQB), np.arange(w.nKB)] = 1
    mask = np.broadcast_to(one, (w.B, w.H, w.nQB, w.nKB)).copy()
    words = torch.from_numpy(gu.mask_bitmap_words(one[None, None]).reshape(-1)).cuda()
    idx = bb.build_mask(None, None, w.block, spec=bb.explicit_spec(words, broadcast_bh=True),
                        shape=(w.B, w.H, w.N, w.d))
    gu.assert_index_equal(idx, mask)
    if N == 512:
        inp = wl.make_inputs(w)
        q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
        O, L = bb.forward(q, k, v, idx)
        torch.cuda.synchronize()
        gu.assert_attention_close(O, L, inp, mask, w)


def test_explicit_capacity_overflow_is_reported():
    w = wl.scaled(wl.WORKLOADS["tiny"], dtype="bf16")
    inp = wl.make_inputs(w)
    words = torch.from_numpy(gu.mask_bitmap_words(inp["mask"]).reshape(-1)).cuda()
    spec = bb.explicit_spec(words)
    B, H, N, d = w.B, w.H, w.N, w.d
    nB = N // w.block
    row_ptr = torch.empty(B * H * nB + 1, dtype=torch.int32, device="cuda")
    cap = 10
    col_idx = torch.full((cap + 64,), -7, dtype=torch.int32, device="cuda")
    bitmap = torch.empty(B * H * nB, dtype=torch.int32, device="cuda")
    ws = bb.workspace(0, B, H, N, d, w.block)
    bb.bsa_build_mask(None, None, bb.BF16, B, H, N, d, w.block, 0.0, spec, row_ptr, col_idx, cap, bitmap, ws,
                      ws.numel())
    assert bb.bsa_check_device_error(ws) == bb.ERR_CAPACITY
    assert torch.all(col_idx[cap:] == -7)  # nothing written past the capacity


def test_bounded_wait_times_out_and_context_survives():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=1024)
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    idx = bb.build_mask(q, k, w.block, density=w.density)
    ws = bb.workspace(1, w.B, w.H, w.N, w.d, w.block)
    try:
        # loads and MMAs are skipped, so the softmax warps wait for a score tile nothing produces
        bb.bsa_debug_config(1, 20_000_000)
        O = torch.empty_like(q)
        L = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
        bb.bsa_forward(q, k, v, bb.BF16, w.B, w.H, w.N, w.d, w.block, idx.row_ptr, idx.col_idx, idx.bitmap,
                       0, 0.0, O, L, ws, ws.numel())
        assert bb.bsa_check_device_error(ws) == bb.ERR_TIMEOUT
    finally:
        bb.bsa_debug_config(0, 0)
    mask = gu.oracle_mask(w, inp)
    O, L = bb.forward(q, k, v, idx)
    gu.assert_attention_close(O, L, inp, mask, w)


# ------------------------------------------------------------ full-size workloads


def test_full_t2i_static():
    w = wl.WORKLOADS["t2i_static"]
    rng = np.random.default_rng(11)
    run_workload(w, rows=gu.sample_rows(w, rng, blocks_per_head=8, rows_per_block=8))


def test_full_dynamic_topk():
    w = wl.WORKLOADS["dynamic_topk"]
    rng = np.random.default_rng(12)
    run_workload(w, rows=gu.sample_rows(w, rng))


def test_full_video_cuboid():
    w = wl.WORKLOADS["video_cuboid"]
    rng = np.random.default_rng(13)
    run_workload(w, rows=gu.sample_rows(w, rng, blocks_per_head=12, rows_per_block=6, text_rows_heads=2))


def test_full_long_topk_bitmap():
    w = wl.WORKLOADS["long_topk"]
    rng = np.random.default_rng(14)
    run_workload(w, rows=gu.sample_rows(w, rng, blocks_per_head=10, rows_per_block=4))


@pytest.mark.parametrize("N", [65536, 131072])
def test_selector_at_the_largest_key_block_counts(N):
    # 1024 and 2048 key blocks per row (the selector's widest register path, 64 keys per lane;
    # 2048 is the limit): the index bit for bit and sampled rows of the forward over it
    w = wl.scaled(wl.WORKLOADS["long_sweep_bs64"], H=1, N=N)
    rng = np.random.default_rng(N)
    run_workload(w, rows=gu.sample_rows(w, rng, blocks_per_head=8, rows_per_block=4))


@pytest.mark.parametrize("nB,density", [(1500, 0.01), (2048, 0.015)])
def test_selector_widest_rows_small_k(nB, density):
    # 64 keys per lane with k = 14 / 30 <= 32: the search over the keys above the lane-maximum
    # bound on the widest register rows (a ragged last word at 1500); the index bit for bit
    w = wl.scaled(wl.WORKLOADS["long_sweep_bs64"], H=2, N=64 * nB, density=density)
    assert 1 <= oracle.topk_count(density, nB) <= 32
    inp = wl.make_inputs(w)
    q, k = gu.upload(inp, "q"), gu.upload(inp, "k")
    mask = gu.oracle_mask(w, inp)
    gu.assert_index_equal(gu.device_index(w, q, k, mask), mask)


@pytest.mark.parametrize("name", ["long_sweep_bs64", "long_sweep_bs128"])
def test_full_block_size_sweep(name):
    w = wl.WORKLOADS[name]
    rng = np.random.default_rng(15)
    run_workload(w, rows=gu.sample_rows(w, rng, blocks_per_head=8, rows_per_block=4))
