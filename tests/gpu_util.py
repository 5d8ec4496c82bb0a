"""Shared helpers of the GPU parity tests: upload seeded inputs, build the oracle's
mask for a workload, compare indexes bit for bit and outputs within tolerance."""
import numpy as np
import torch

import oracle
from block_sparse_attention_mean_gb300 import binding as bb
from block_sparse_attention_mean_gb300 import workloads as wl

# Parity bar for bf16 inputs with fp32 accumulation (fp32 inputs use the same bar).
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def upload(inp, name):
    w = inp["workload"]
    if w.dtype == "bf16":
        bits = np.ascontiguousarray(inp[name + "_bits"]).view(np.int16)
        return torch.from_numpy(bits).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(inp[name])).cuda()


def spec_for(w, mask_dev=None):
    if w.mask == wl.BAND:
        return bb.band_spec(w.n_text_blocks, w.band, list(w.anchors))
    if w.mask == wl.CUBOID:
        return bb.cuboid_spec(w.n_text_blocks, w.grid)
    if w.mask == wl.EXPLICIT:
        return bb.explicit_spec(mask_dev)
    return None


def mask_bitmap_words(mask):
    return wl.pack_bitmap_words(mask)


def oracle_mask(w, inp):
    """uint8 [B, H, nQB, nKB] block mask of the workload, from the oracle only."""
    shape = (w.B, w.H, w.nQB, w.nKB)
    if w.mask == wl.EXPLICIT:
        return inp["mask"]
    if w.mask == wl.BAND:
        return np.broadcast_to(oracle.band_mask(w.nQB, w.n_text_blocks, w.band, w.anchors), shape).copy()
    if w.mask == wl.CUBOID:
        return np.broadcast_to(oracle.cuboid_mask(w.n_text_blocks, w.grid), shape).copy()
    return oracle.select_mask(inp["q"], inp["k"], w.block, w.density)


def device_index(w, q, k, mask=None):
    mask_dev = None
    if w.mask == wl.EXPLICIT:
        mask_dev = torch.from_numpy(mask_bitmap_words(mask).reshape(-1)).cuda()
    spec = spec_for(w, mask_dev)
    return bb.build_mask(q if spec is None else None, k if spec is None else None, w.block,
                         density=w.density, spec=spec, shape=(w.B, w.H, w.N, w.d))


def assert_index_equal(idx, mask):
    row_ptr, col_idx, bitmap = oracle.mask_to_index(mask)
    nnz = int(row_ptr[-1])
    assert np.array_equal(idx.row_ptr.cpu().numpy(), row_ptr)
    assert np.array_equal(idx.col_idx[:nnz].cpu().numpy(), col_idx)
    assert np.array_equal(idx.bitmap.cpu().numpy().view(np.uint32), bitmap.reshape(-1))


def sample_rows(w, rng, blocks_per_head=16, rows_per_block=8, heads=None, text_rows_heads=0):
    """Global row ids: per head the first and last Q block plus random blocks,
    a few rows from each (always the block's first and last row)."""
    heads = range(w.B * w.H) if heads is None else heads
    out = []
    for h in heads:
        blocks = {0, w.nQB - 1} | set(rng.choice(w.nQB, size=min(blocks_per_head, w.nQB), replace=False).tolist())
        for i in sorted(blocks):
            rr = {0, w.block - 1} | set(rng.choice(w.block, size=rows_per_block - 2, replace=False).tolist())
            out += [h * w.N + i * w.block + r for r in sorted(rr)]
    for h in range(text_rows_heads):
        out += [h * w.N + r for r in range(w.n_text_blocks * w.block)]
    return np.unique(np.array(out, np.int64))


def assert_attention_close(O, LSE, inp, mask, w, rows=None, scale=None):
    O_ref, L_ref = oracle.attention(inp["q"], inp["k"], inp["v"], mask, w.block, scale=scale, rows=rows)
    Og = O.float().reshape(-1, w.d).cpu().numpy().astype(np.float64)
    Lg = LSE.reshape(-1).cpu().numpy().astype(np.float64)
    if rows is not None:
        Og, Lg = Og[rows], Lg[rows]
    err = np.abs(Og - O_ref)
    assert np.all(np.isfinite(Og)), "non-finite output"
    assert err.max() <= O_MAX_ABS, f"O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"O mean-abs {err.mean():.3e}"
    empty = np.isneginf(L_ref)
    assert np.array_equal(np.isneginf(Lg), empty), "empty-row LSE mismatch"
    assert np.all(Og[empty] == 0.0)
    if (~empty).any():
        lerr = np.abs(Lg[~empty] - L_ref[~empty])
        assert lerr.max() <= LSE_MAX_ABS, f"LSE max-abs {lerr.max():.3e}"
    return float(err.max()), float(err.mean())
