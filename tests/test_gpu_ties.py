"""GPU parity of the pooled top-k selector on exact ties ("Can sparse attention close the
quality gap in diffusion transformers", section "均值池化块打分漏掉高权重 token", with the
per-Q-block count of "多模态DiT中的块稀疏注意力" §5.3).

Q and K are block-constant, so each pooled mean is exact, and their values are drawn from a
small palette, so many block scores are exactly equal: small-integer dot products, +0 from
all-zero key blocks, -0 from one tiny product that underflows in the last channel, and +inf /
-inf from one product that overflows. The selection must equal the oracle's bit for bit
(value descending with -0 equal to +0, ties to the lower block index) in CSR and bitmap, at
both block sizes, with 72 or 300 key blocks so that tie groups straddle the 32-bit words of the
bitmap. The data are checked to contain each kind of tie at the k-th position. The three
densities take the selector's three searches: k = 36 of 72 the full-row search (k > 32); k = 18
of 72 the search over the keys above the lane-maximum bound (at most 72 of them); k = 30 of 300
both, about half the rows holding more than 128 keys above the bound and falling back.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_mean_gb300 import binding as bb
from block_sparse_attention_mean_gb300 import build as bbuild
from tests import gpu_util as gu

TINY = 2.0 ** -80   # TINY * -TINY = -2^-160 rounds to -0 in fp32
HUGE = 2.0 ** 100   # HUGE * HUGE overflows fp32 to +inf


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bbuild.build()
    bb.load()


def tie_inputs(H, nB, bs, d, seed):
    """Block-constant Q, K [1, H, nB*bs, d] (fp32 values, all exact in bf16) with a palette of
    key blocks: 0 all-zero (score +0), 1 negative zero (score -0), 2 / 3 overflow (+inf / -inf
    for query blocks whose channel 1 is HUGE, +0 otherwise), 4.. small-integer vectors."""
    rng = np.random.default_rng(seed)
    n_int = 6
    qb = np.zeros((H, nB, d), np.float32)
    kb = np.zeros((H, nB, d), np.float32)
    for h in range(H):
        pal = np.zeros((4 + n_int, d), np.float32)
        pal[1, d - 1] = -TINY
        pal[2, 1] = HUGE
        pal[3, 1] = -HUGE
        ints = rng.integers(-1, 2, size=(n_int, d)).astype(np.float32)
        ints[:, 1] = 0.0
        ints[:, d - 1] = 0.0
        pal[4:] = ints
        choice = rng.choice(pal.shape[0], size=nB, p=[0.2, 0.2, 0.05, 0.05] + [0.5 / n_int] * n_int)
        kb[h] = pal[choice]
        qi = rng.integers(-2, 3, size=(nB, d)).astype(np.float32)
        qi[:, 1] = np.where(rng.random(nB) < 0.3, HUGE, 0.0)
        qi[:, d - 1] = TINY
        qb[h] = qi
    q = np.repeat(qb, bs, axis=1)[None]
    k = np.repeat(kb, bs, axis=1)[None]
    return q, k


def to_bf16_device(x):
    bits = (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), x)  # every value exact in bf16
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def tie_coverage(q, k, bs, kk):
    """Rows whose k-th score sits in a tie group that the cut splits, and what that group holds."""
    H = q.shape[1]
    qbar = oracle.block_mean(q.reshape(H, -1, q.shape[-1]), bs)
    kbar = oracle.block_mean(k.reshape(H, -1, k.shape[-1]), bs)
    s = oracle.block_scores(qbar, kbar).reshape(-1, kbar.shape[1])
    stats = {"split": 0, "signed_zeros": 0, "word": 0, "pinf": 0, "ninf": 0}
    for row in s:
        order = np.lexsort((np.arange(row.size), -row))
        kth = row[order[kk - 1]]
        group = np.flatnonzero(row == kth)  # -0 == +0 here, as in the selector
        kept, dropped = group[np.isin(group, order[:kk])], group[~np.isin(group, order[:kk])]
        stats["pinf"] += bool(np.isposinf(row).any())
        stats["ninf"] += bool(np.isneginf(row).any())
        if kept.size and dropped.size:
            stats["split"] += 1
            stats["signed_zeros"] += bool(kth == 0 and np.signbit(row[group]).any() and (~np.signbit(row[group])).any())
            stats["word"] += bool(kept.max() // 32 != dropped.min() // 32)
    return stats


@pytest.mark.gpu
@pytest.mark.parametrize("nB,density", [(72, 0.5), (72, 0.25), (300, 0.1)])
@pytest.mark.parametrize("block,d", [(64, 128), (128, 128), (64, 64)])
def test_selection_on_exact_ties_matches_oracle(block, d, nB, density):
    H = 4
    q, k = tie_inputs(H, nB, block, d, seed=block + d)
    N = nB * block
    kk = oracle.topk_count(density, nB)
    cov = tie_coverage(q, k, block, kk)
    for key in cov:
        assert cov[key] > 0, (key, cov)  # the data exercise every kind of tie
    mask = oracle.select_mask(q, k, block, density)
    idx = bb.build_mask(to_bf16_device(q), to_bf16_device(k), block, density=density, shape=(1, H, N, d))
    torch.cuda.synchronize()
    gu.assert_index_equal(idx, mask)
