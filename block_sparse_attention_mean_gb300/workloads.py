"""Seeded synthetic workloads for the block-sparse attention forward.

This module only *draws inputs* and *describes masks*: shapes, value recipes,
and the parameters of the static mask specs. It contains none of the method's
arithmetic (no pooling, scoring, selection, softmax or index building), so both
the CUDA path and the CPU oracle can take their inputs from here without
sharing any computation.

Workloads follow the shapes the pages describe for multimodal and video DiTs
("多模态DiT中的块稀疏注意力：从原理到工程落地", §1.1 for the 1024² image ->
4096 patch + text token count, §3.1-§3.2 for text/image/video regions and
cuboids, §5.1 for the density range) and the mean-pooled top-k selector of
"Can sparse attention close the quality gap in diffusion transformers"
(naive BSA). Recipes that the pages leave open are fixed as follows:

* ``rank``: per (b, h) draw U ~ N(0,1)^{N x r} and C ~ N(0,1)^{r x d}/sqrt(r)
  once; X = Z_X + s * U @ C for X in {Q, K, V} with fresh Z_X ~ N(0,1).
* ``clustered``: per head, 16 centroids ~ N(0,1)^d shared by Q and K; token
  cluster ids run in contiguous segments of uniform length in [32, 512];
  Q = c[id] + 0.3 Z_Q, K = c[id] + 0.3 Z_K, V = Z_V.
* ``blurred``: text tokens N(0,1); each (head, channel) video field of shape
  (T, Hh, Ww) is N(0,1) smoothed by a separable Gaussian (sigma 1.5, radius 5,
  numpy 'reflect' padding) and divided by the blur's analytic standard
  deviation, then tokens are permuted so each 4x4x4 cuboid is contiguous
  (cuboids t-major raster, tokens inside a cuboid (dt, dh, dw) raster).

bf16 workloads are rounded to bf16 (round-to-nearest-even) here; the float32
arrays returned hold exactly the bf16 values, so both sides see identical
inputs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Tuple

import numpy as np

# mask kinds
EXPLICIT = "explicit"
BAND = "band"
CUBOID = "cuboid"
TOPK = "topk"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    block: int
    dtype: str              # "fp32" or "bf16"
    seed: int
    mask: str               # EXPLICIT | BAND | CUBOID | TOPK
    values: str             # "iid" | "rank" | "clustered" | "blurred"
    density: float = 0.0    # TOPK: fraction of KV blocks kept per Q block
    index_mode: int = 0     # 0: CSR, 1: bitmap + popcount
    rank: int = 0           # "rank": rank of the shared component
    rank_scale: float = 0.0
    n_text_blocks: int = 0  # BAND / CUBOID: leading text blocks (dense rows and columns)
    band: int = 0           # BAND: |r - c| <= band over image block rows
    anchors: Tuple[int, ...] = ()      # BAND: global image blocks (row- and column-dense)
    grid: Tuple[int, int, int] = (0, 0, 0)  # CUBOID: (gt, gh, gw) cuboid grid
    video_shape: Tuple[int, int, int] = (0, 0, 0)  # "blurred": latent (T, Hh, Ww)
    n_text_tokens: int = 0  # "blurred": leading text tokens
    mask_seed: int = 0      # EXPLICIT: seed of the Bernoulli block mask
    mask_p: float = 0.5     # EXPLICIT: Bernoulli probability

    @property
    def nQB(self) -> int:
        return -(-self.N // self.block)  # a ragged last block counts

    @property
    def nKB(self) -> int:
        return -(-self.N // self.block)  # a ragged last block counts


WORKLOADS: Dict[str, Workload] = {
    # B=1 H=2 N=512 d=64, 8x8 block grid, fp32 i.i.d., random block mask p=0.5 + diagonal
    "tiny": Workload("tiny", 1, 2, 512, 64, 64, "fp32", seed=1, mask=EXPLICIT, values="iid",
                     mask_seed=101, mask_p=0.5),
    # text-to-image DiT: 128 text + 64x64 patch tokens = 4224 = 66 blocks of 64
    "t2i_static": Workload("t2i_static", 2, 24, 4224, 64, 64, "bf16", seed=2, mask=BAND,
                           values="rank", rank=8, rank_scale=0.5,
                           n_text_blocks=2, band=2, anchors=(0, 32)),
    # dynamic mean-pooled top-k, 15% of KV blocks per Q block
    "dynamic_topk": Workload("dynamic_topk", 1, 24, 8192, 128, 64, "bf16", seed=3, mask=TOPK,
                             values="clustered", density=0.15),
    # video: 256 text tokens + 16x32x32 latent tokens, 4x4x4 cuboids as blocks
    "video_cuboid": Workload("video_cuboid", 1, 24, 16640, 128, 64, "bf16", seed=4, mask=CUBOID,
                             values="blurred", n_text_blocks=4, grid=(4, 8, 8),
                             video_shape=(16, 32, 32), n_text_tokens=256),
    # long sequence, block 128, 5% top-k through the bitmap index
    "long_topk": Workload("long_topk", 1, 16, 65536, 128, 128, "bf16", seed=5, mask=TOPK,
                          values="rank", rank=16, rank_scale=0.5, density=0.05, index_mode=1),
    # block-size sweep at N=32768
    "long_sweep_bs64": Workload("long_sweep_bs64", 1, 16, 32768, 128, 64, "bf16", seed=5,
                                mask=TOPK, values="rank", rank=16, rank_scale=0.5,
                                density=0.05, index_mode=1),
    "long_sweep_bs128": Workload("long_sweep_bs128", 1, 16, 32768, 128, 128, "bf16", seed=5,
                                 mask=TOPK, values="rank", rank=16, rank_scale=0.5,
                                 density=0.05, index_mode=1),
}


def scaled(w: Workload, **changes) -> Workload:
    """Same recipe with some fields changed (smaller parity cases, fuzzing)."""
    return dataclasses.replace(w, **changes)


# ---------------------------------------------------------------------------
# value recipes


def round_to_bf16(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Round float32 -> bf16 (nearest, ties to even) for finite inputs.

    Returns (float32 array holding the bf16 values, uint16 bf16 bit patterns).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)
    bits = (r >> np.uint32(16)).astype(np.uint16)
    return r.view(np.float32), bits


def _gauss_taps(sigma: float, radius: int) -> np.ndarray:
    t = np.arange(-radius, radius + 1, dtype=np.float64)
    w = np.exp(-0.5 * (t / sigma) ** 2)
    return w / w.sum()


def _blur_axis(x: np.ndarray, taps: np.ndarray, axis: int) -> np.ndarray:
    r = (len(taps) - 1) // 2
    pad = [(0, 0)] * x.ndim
    pad[axis] = (r, r)
    xp = np.pad(x, pad, mode="reflect")
    out = np.zeros_like(x)
    n = x.shape[axis]
    for i, wt in enumerate(taps):
        sl = [slice(None)] * x.ndim
        sl[axis] = slice(i, i + n)
        out += np.float32(wt) * xp[tuple(sl)]
    return out


def cuboid_permutation(video_shape: Tuple[int, int, int], cuboid: int = 4) -> np.ndarray:
    """perm[new_index] = raster index (t, h, w) of the token placed there."""
    T, Hh, Ww = video_shape
    gt, gh, gw = T // cuboid, Hh // cuboid, Ww // cuboid
    t = np.arange(T).reshape(T, 1, 1)
    h = np.arange(Hh).reshape(1, Hh, 1)
    w = np.arange(Ww).reshape(1, 1, Ww)
    cub = ((t // cuboid) * gh + (h // cuboid)) * gw + (w // cuboid)
    inner = ((t % cuboid) * cuboid + (h % cuboid)) * cuboid + (w % cuboid)
    new_index = (cub * cuboid ** 3 + inner).reshape(-1)
    perm = np.empty_like(new_index)
    perm[new_index] = np.arange(new_index.size)
    return perm


def _draw_values(w: Workload, rng: np.random.Generator):
    B, H, N, d = w.B, w.H, w.N, w.d
    shape = (B, H, N, d)
    if w.values == "iid":
        return [rng.standard_normal(shape, dtype=np.float32) for _ in range(3)]
    if w.values == "rank":
        out = [np.empty(shape, np.float32) for _ in range(3)]
        for b in range(B):
            for h in range(H):
                U = rng.standard_normal((N, w.rank), dtype=np.float32)
                C = rng.standard_normal((w.rank, d), dtype=np.float32) / np.float32(math.sqrt(w.rank))
                shared = np.float32(w.rank_scale) * (U @ C)
                for t in range(3):
                    out[t][b, h] = rng.standard_normal((N, d), dtype=np.float32) + shared
        return out
    if w.values == "clustered":
        q = np.empty(shape, np.float32)
        k = np.empty(shape, np.float32)
        for b in range(B):
            for h in range(H):
                cent = rng.standard_normal((16, d), dtype=np.float32)
                ids = np.empty(N, np.int64)
                pos = 0
                while pos < N:
                    ln = int(rng.integers(32, 513))
                    ids[pos:pos + ln] = int(rng.integers(0, 16))
                    pos += ln
                q[b, h] = cent[ids] + np.float32(0.3) * rng.standard_normal((N, d), dtype=np.float32)
                k[b, h] = cent[ids] + np.float32(0.3) * rng.standard_normal((N, d), dtype=np.float32)
        v = rng.standard_normal(shape, dtype=np.float32)
        return [q, k, v]
    if w.values == "blurred":
        T, Hh, Ww = w.video_shape
        nv = T * Hh * Ww
        assert w.n_text_tokens + nv == N
        taps = _gauss_taps(1.5, 5)
        # std of the separable blur of unit white noise is (sum w^2)^(3/2)
        norm = np.float32(1.0 / float(np.sum(taps ** 2)) ** 1.5)
        perm = cuboid_permutation(w.video_shape)
        out = [np.empty(shape, np.float32) for _ in range(3)]
        for t in range(3):
            for b in range(B):
                for h in range(H):
                    text = rng.standard_normal((w.n_text_tokens, d), dtype=np.float32)
                    f = rng.standard_normal((T, Hh, Ww, d), dtype=np.float32)
                    for ax in range(3):
                        f = _blur_axis(f, taps, ax)
                    f = (f * norm).reshape(nv, d)
                    out[t][b, h, :w.n_text_tokens] = text
                    out[t][b, h, w.n_text_tokens:] = f[perm]
        return out
    raise ValueError(f"unknown value recipe {w.values!r}")


def explicit_block_mask(w: Workload) -> Optional[np.ndarray]:
    """Bernoulli(p) block bits per (b, h, i, j) with the diagonal forced on (uint8)."""
    if w.mask != EXPLICIT:
        return None
    rng = np.random.default_rng(w.mask_seed)
    m = (rng.random((w.B, w.H, w.nQB, w.nKB)) < w.mask_p).astype(np.uint8)
    idx = np.arange(min(w.nQB, w.nKB))
    m[:, :, idx, idx] = 1
    return m


def make_inputs(w: Workload) -> dict:
    """Draw the workload's Q, K, V (and explicit mask) from its seed.

    Returns a dict with float32 arrays ``q``, ``k``, ``v`` of shape [B, H, N, d]
    holding exactly the values the GPU sees, ``*_bits`` (uint16 bf16 patterns)
    for bf16 workloads, and ``mask`` (uint8 [B, H, nQB, nKB]) for explicit masks.
    """
    rng = np.random.default_rng(w.seed)
    q, k, v = _draw_values(w, rng)
    out = {"workload": w}
    for name, x in (("q", q), ("k", k), ("v", v)):
        if w.dtype == "bf16":
            xf, bits = round_to_bf16(x)
            out[name] = xf.reshape(x.shape)
            out[name + "_bits"] = bits.reshape(x.shape)
        else:
            out[name] = np.ascontiguousarray(x, dtype=np.float32)
    out["mask"] = explicit_block_mask(w)
    return out



def pack_bitmap_words(mask: np.ndarray) -> np.ndarray:
    """Explicit block mask -> the bitmap input format of the static explicit spec.

    uint8 [..., nKB] -> int32 words [..., ceil(nKB/32)]; bit j % 32 of word j / 32
    is block j.
    """
    nKB = mask.shape[-1]
    W = (nKB + 31) // 32
    pad = np.zeros((*mask.shape[:-1], W * 32), np.uint64)
    pad[..., :nKB] = mask
    words = (pad.reshape(*mask.shape[:-1], W, 32) << np.arange(32, dtype=np.uint64)).sum(-1)
    return words.astype(np.uint32).view(np.int32)
