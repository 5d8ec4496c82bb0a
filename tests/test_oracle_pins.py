"""Pins of the CPU oracle to things other than itself.

Each oracle function is tied to closed forms, library routines, brute force on
tiny inputs or hand-derived fixtures under tests/golden/, chosen so that a
plausible slip (a dropped term, a wrong sign or index, a transposed operand, a
different summation order, a lost tie-break) fails at least one test.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special

import oracle
from tests.conftest import read_golden

RNG = np.random.default_rng(12345)


def _rand(*shape):
    return RNG.standard_normal(shape).astype(np.float32)


# ---------------------------------------------------------------- attention


def _dense_library(q, k, v, scale, allowed):
    """softmax/logsumexp from scipy over an explicit token-level allow matrix."""
    s = (q.astype(np.float64) @ k.astype(np.float64).T) * scale
    s = np.where(allowed, s, -np.inf)
    lse = scipy.special.logsumexp(s, axis=-1)
    p = scipy.special.softmax(s, axis=-1)
    return p @ v.astype(np.float64), lse


def test_all_ones_mask_equals_dense_attention():
    H, N, d, bs = 2, 96, 16, 32
    q, k, v = _rand(H, N, d), _rand(H, N, d), _rand(H, N, d)
    mask = np.ones((H, N // bs, N // bs), np.uint8)
    O, L = oracle.attention(q, k, v, mask, bs)
    for h in range(H):
        Od, Ld = _dense_library(q[h], k[h], v[h], 1.0 / math.sqrt(d), np.ones((N, N), bool))
        np.testing.assert_allclose(O[h * N:(h + 1) * N], Od, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L[h * N:(h + 1) * N], Ld, rtol=1e-12, atol=1e-12)


def test_random_mask_equals_library_on_token_mask():
    H, N, d, bs = 3, 64, 8, 16
    q, k, v = _rand(H, N, d), _rand(H, N, d), _rand(H, N, d)
    nB = N // bs
    mask = (RNG.random((H, nB, nB)) < 0.5).astype(np.uint8)
    mask[:, np.arange(nB), np.arange(nB)] = 1
    O, L = oracle.attention(q, k, v, mask, bs, scale=0.3)
    for h in range(H):
        tok = np.kron(mask[h], np.ones((bs, bs), np.uint8)).astype(bool)
        Od, Ld = _dense_library(q[h], k[h], v[h], 0.3, tok)
        np.testing.assert_allclose(O[h * N:(h + 1) * N], Od, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L[h * N:(h + 1) * N], Ld, rtol=1e-12, atol=1e-12)


def test_block_diagonal_mask_is_independent_block_attention():
    N, d, bs = 64, 8, 16
    q, k, v = _rand(1, N, d), _rand(1, N, d), _rand(1, N, d)
    mask = np.eye(N // bs, dtype=np.uint8)[None]
    O, L = oracle.attention(q, k, v, mask, bs)
    for i in range(N // bs):
        sl = slice(i * bs, (i + 1) * bs)
        Ob, Lb = _dense_library(q[0, sl], k[0, sl], v[0, sl], 1 / math.sqrt(d),
                                np.ones((bs, bs), bool))
        np.testing.assert_allclose(O[sl], Ob, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L[sl], Lb, rtol=1e-12)


def test_single_active_block_brute_force():
    N, d, bs = 16, 3, 4
    q, k, v = _rand(1, N, d), _rand(1, N, d), _rand(1, N, d)
    nB = N // bs
    mask = np.zeros((1, nB, nB), np.uint8)
    pick = [2, 0, 3, 1]
    for i, j in enumerate(pick):
        mask[0, i, j] = 1
    O, L = oracle.attention(q, k, v, mask, bs, scale=0.7)
    for r in range(N):
        j = pick[r // bs]
        ss = []
        for c in range(j * bs, (j + 1) * bs):
            ss.append(0.7 * sum(float(q[0, r, e]) * float(k[0, c, e]) for e in range(d)))
        mx = max(ss)
        w = [math.exp(s - mx) for s in ss]
        tot = sum(w)
        for e in range(d):
            ref = sum(w[t] * float(v[0, j * bs + t, e]) for t in range(bs)) / tot
            assert abs(O[r, e] - ref) < 1e-12
        assert abs(L[r] - (mx + math.log(tot))) < 1e-12


def test_zero_keys_closed_form():
    """K = 0: every active score is 0, so LSE = ln(#active keys), O = mean of active values."""
    N, d, bs = 64, 8, 16
    q, v = _rand(1, N, d), _rand(1, N, d)
    k = np.zeros((1, N, d), np.float32)
    nB = N // bs
    mask = (RNG.random((1, nB, nB)) < 0.5).astype(np.uint8)
    mask[0, :, 0] = 1
    O, L = oracle.attention(q, k, v, mask, bs)
    for r in range(N):
        act = np.nonzero(mask[0, r // bs])[0]
        keys = np.concatenate([np.arange(j * bs, (j + 1) * bs) for j in act])
        assert L[r] == pytest.approx(math.log(len(keys)), abs=1e-13)
        np.testing.assert_allclose(O[r], v[0, keys].astype(np.float64).mean(0), atol=1e-13)


def test_constant_values_and_unit_row_mass():
    N, d, bs = 64, 4, 16
    q, k = _rand(2, N, d) * 3, _rand(2, N, d) * 3
    nB = N // bs
    mask = (RNG.random((2, nB, nB)) < 0.6).astype(np.uint8)
    mask[:, :, 1] = 1
    v = np.full((2, N, d), 1.0, np.float32)
    O, _ = oracle.attention(q, k, v, mask, bs)
    np.testing.assert_allclose(O, 1.0, atol=1e-13)  # sum_c p_c = 1 per row
    v2 = np.broadcast_to(np.array([2.5, -1.0, 0.0, 7.0], np.float32), (2, N, d)).copy()
    O2, _ = oracle.attention(q, k, v2, mask, bs)
    np.testing.assert_allclose(O2, np.broadcast_to(v2[0, 0], O2.shape), atol=1e-12)


def test_key_permutation_inside_blocks_is_invariant():
    N, d, bs = 64, 8, 16
    q, k, v = _rand(1, N, d), _rand(1, N, d), _rand(1, N, d)
    nB = N // bs
    mask = (RNG.random((1, nB, nB)) < 0.5).astype(np.uint8)
    mask[0, np.arange(nB), np.arange(nB)] = 1
    perm = np.concatenate([RNG.permutation(bs) + j * bs for j in range(nB)])
    O1, L1 = oracle.attention(q, k, v, mask, bs)
    O2, L2 = oracle.attention(q, k[:, perm], v[:, perm], mask, bs)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(L1, L2, atol=1e-12)


def test_masked_keys_do_not_matter():
    """Changing K/V inside skipped blocks leaves the result bit-identical (they are -inf)."""
    N, d, bs = 64, 8, 16
    q, k, v = _rand(1, N, d), _rand(1, N, d), _rand(1, N, d)
    mask = np.zeros((1, 4, 4), np.uint8)
    mask[0, :, 1] = 1
    mask[0, 2, 3] = 1
    O1, L1 = oracle.attention(q, k, v, mask, bs)
    k2, v2 = k.copy(), v.copy()
    k2[0, 0:16] *= 100
    v2[0, 0:16] = 1e6
    O2, L2 = oracle.attention(q, k2, v2, mask, bs)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_empty_row_convention():
    N, d, bs = 32, 4, 16
    q, k, v = _rand(1, N, d), _rand(1, N, d), _rand(1, N, d)
    mask = np.array([[[0, 0], [1, 1]]], np.uint8)
    O, L = oracle.attention(q, k, v, mask, bs)
    assert np.all(O[:16] == 0.0) and np.all(np.isneginf(L[:16]))
    assert np.all(np.isfinite(L[16:]))


def test_default_scale_is_inverse_sqrt_d():
    N, d, bs = 32, 16, 16
    q, k, v = _rand(1, N, d), _rand(1, N, d), _rand(1, N, d)
    mask = np.ones((1, 2, 2), np.uint8)
    O1, L1 = oracle.attention(q, k, v, mask, bs)
    O2, L2 = oracle.attention(q, k, v, mask, bs, scale=0.25)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_attention_golden_two_keys():
    q = np.array([[[1.0], [0.0]]], np.float32)
    k = np.array([[[0.0], [1.0]]], np.float32)
    v = np.array([[[0.0], [1.0]]], np.float32)
    for bits, o_ref, l_ref in read_golden("attention_two_keys.txt"):
        mask = np.zeros((1, 2, 2), np.uint8)
        mask[0, 0] = [int(c) for c in bits]
        mask[0, 1] = 1
        O, L = oracle.attention(q, k, v, mask, 1, scale=1.0, rows=np.array([0]))
        assert O[0, 0] == pytest.approx(float(o_ref), abs=1e-15)
        if l_ref == "-inf":
            assert np.isneginf(L[0])
        else:
            assert L[0] == pytest.approx(float(l_ref), abs=1e-15)


def test_row_subset_matches_full():
    N, d, bs = 64, 8, 16
    q, k, v = _rand(2, N, d), _rand(2, N, d), _rand(2, N, d)
    mask = (RNG.random((2, 4, 4)) < 0.5).astype(np.uint8)
    mask[:, :, 2] = 1
    O, L = oracle.attention(q, k, v, mask, bs)
    rows = np.array([5, 70, 127, 0])
    Os, Ls = oracle.attention(q, k, v, mask, bs, rows=rows)
    np.testing.assert_array_equal(Os, O[rows])
    np.testing.assert_array_equal(Ls, L[rows])


# ---------------------------------------------------------------- selector


def test_block_mean_golden_order():
    for bs, toks, ref in read_golden("block_mean_order.txt"):
        bs = int(bs)
        x = np.array([float(t) for t in toks.split()], np.float32).reshape(1, bs, 1)
        out = oracle.block_mean(x, bs)
        assert out.shape == (1, 1, 1)
        assert float(out[0, 0, 0]) == float(ref)


def test_block_mean_exact_integers_and_layout():
    H, N, d, bs = 3, 64, 5, 16
    x = RNG.integers(-50, 50, size=(H, N, d)).astype(np.float32)
    out = oracle.block_mean(x, bs)
    ref = x.astype(np.float64).reshape(H, N // bs, bs, d).mean(axis=2)
    assert np.array_equal(out.astype(np.float64), ref)  # sums of small ints are exact


def test_block_scores_golden_fma():
    for qs, ks, ref in read_golden("score_fma.txt"):
        qb = np.array([float(t) for t in qs.split()], np.float32).reshape(1, 1, -1)
        kb = np.array([float(t) for t in ks.split()], np.float32).reshape(1, 1, -1)
        assert float(oracle.block_scores(qb, kb)[0, 0, 0]) == float(ref)


def test_block_scores_exact_small_integers_and_orientation():
    qb = RNG.integers(-8, 8, size=(2, 5, 7)).astype(np.float32)
    kb = RNG.integers(-8, 8, size=(2, 3, 7)).astype(np.float32)
    s = oracle.block_scores(qb, kb)
    assert s.shape == (2, 5, 3)
    ref = np.einsum("hic,hjc->hij", qb.astype(np.int64), kb.astype(np.int64))
    assert np.array_equal(s.astype(np.int64), ref)


def test_topk_golden_ties_and_signed_zero():
    for scores, k, kept in read_golden("topk_ties.txt"):
        s = np.array([float(t) for t in scores.split()], np.float32).reshape(1, -1)
        m = oracle.topk_mask(s, int(k))
        assert list(np.nonzero(m[0])[0]) == [int(t) for t in kept.split()]


def test_topk_brute_force_with_ties():
    nKB = 40
    for trial in range(30):
        s = RNG.integers(-4, 4, size=(3, nKB)).astype(np.float32)  # many exact ties
        if trial % 3 == 0:
            s[s == 0] = -0.0
        k = int(RNG.integers(1, nKB + 1))
        m = oracle.topk_mask(s, k)
        for r in range(3):
            order = sorted(range(nKB), key=lambda j: (-float(s[r, j]), j))
            ref = np.zeros(nKB, np.uint8)
            ref[order[:k]] = 1
            assert np.array_equal(m[r], ref)
            assert int(m[r].sum()) == k


def test_topk_rejects_nan():
    s = np.array([[0.0, np.nan, 1.0]], np.float32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.topk_mask(s, 1)
    assert e.value.code == oracle.ERR_NONFINITE


@pytest.mark.parametrize("density,nKB,k", [(0.15, 128, 19), (0.05, 512, 25), (0.05, 256, 12),
                                           (0.001, 64, 1), (1.0, 66, 66), (0.5, 8, 4),
                                           (0.25, 128, 32)])
def test_topk_count(density, nKB, k):
    assert oracle.topk_count(density, nKB) == k


def test_select_mask_is_pool_score_topk():
    """End to end on clustered blocks: blocks built from one centroid rank first."""
    bs, d = 16, 8
    cent = np.zeros((4, d), np.float32)
    cent[np.arange(4), np.arange(4)] = 4.0
    order = [0, 1, 2, 3, 0, 1, 2, 3]
    x = np.concatenate([np.repeat(cent[c][None], bs, 0) for c in order])[None]
    m = oracle.select_mask(x, x, bs, 0.25)
    for i, c in enumerate(order):
        assert list(np.nonzero(m[0, i])[0]) == [j for j, cc in enumerate(order) if cc == c]


# ---------------------------------------------------------------- static masks


def _golden_bits(name):
    return np.array([[int(c) for c in row[0]] for row in read_golden(name)], np.uint8)


def test_band_mask_golden_small():
    assert np.array_equal(oracle.band_mask(6, 1, 1, [3]), _golden_bits("band_mask_small.txt"))


def test_band_mask_t2i_count():
    """66 blocks: 2 text + 64 image rows, band 2, anchors {0, 32}.

    Text rows 2*66 = 132, text columns of image rows 64*2 = 128. Image-image:
    band 64*5 - 2*(1+2) = 314; anchor rows/cols 2*64 + 2*64 - 4 = 252; band
    cells on anchor rows/cols: row0 3 + row32 5 + col0 3 + col32 5 - 2 = 14;
    total 314 + 252 - 14 = 552. Sum 812.
    """
    m = oracle.band_mask(66, 2, 2, [0, 32])
    assert int(m.sum()) == 812
    assert np.array_equal(m, m.T)


def test_cuboid_mask_golden_small():
    assert np.array_equal(oracle.cuboid_mask(1, (1, 2, 2)), _golden_bits("cuboid_mask_small.txt"))


def test_cuboid_mask_video_count():
    """4 text + 4x8x8 cuboids: self 256; face pairs t 2*3*64 = 384, h 2*4*7*8 = 448,
    w 2*4*8*7 = 448 -> 1536; text rows 4*260 = 1040; text cols 256*4 = 1024. Sum 3600."""
    m = oracle.cuboid_mask(4, (4, 8, 8))
    assert m.shape == (260, 260)
    assert int(m.sum()) == 3600
    assert np.array_equal(m, m.T)
    assert np.all(m[np.arange(260), np.arange(260)] == 1)


def test_cuboid_mask_degree_brute_force():
    grid = (3, 2, 4)
    m = oracle.cuboid_mask(2, grid)
    cells = list(itertools.product(range(3), range(2), range(4)))
    for a, ca in enumerate(cells):
        for b, cb in enumerate(cells):
            want = sum(abs(x - y) for x, y in zip(ca, cb)) <= 1
            assert m[2 + a, 2 + b] == want


# ---------------------------------------------------------------- index forms


def test_mask_to_index_brute_force():
    for nKB in (1, 8, 31, 32, 33, 70):
        mask = (RNG.random((5, nKB)) < 0.4).astype(np.uint8)
        mask[2] = 0
        row_ptr, col_idx, bitmap = oracle.mask_to_index(mask)
        assert row_ptr[0] == 0 and row_ptr[-1] == mask.sum()
        for r in range(5):
            js = [j for j in range(nKB) if mask[r, j]]
            assert list(col_idx[row_ptr[r]:row_ptr[r + 1]]) == js
            for j in range(nKB):
                assert ((int(bitmap[r, j // 32]) >> (j % 32)) & 1) == mask[r, j]
            assert sum(bin(int(w)).count("1") for w in bitmap[r]) == len(js)


# ------------------------------------------------------------ residual compensation


def test_residual_and_compensate_hand_values():
    # R = dense - sparse (not sparse - dense), and compensation adds it
    r = oracle.residual(np.array([1.0, 2.0, -4.0]), np.array([0.5, 3.0, -4.0]))
    assert r.tolist() == [0.5, -1.0, 0.0]
    assert oracle.compensate(np.array([1.0, 1.0, 2.0]), r).tolist() == [1.5, 0.0, 2.0]


def test_compensation_at_the_anchor_gives_the_dense_output():
    rng = np.random.default_rng(7)
    N, d, bs = 256, 64, 64
    q, k, v = (rng.standard_normal((1, 1, N, d)) for _ in range(3))
    nB = N // bs
    full = np.ones((1, 1, nB, nB), dtype=np.uint8)
    sparse = np.eye(nB, dtype=np.uint8)[None, None]
    o_dense, _ = oracle.attention(q, k, v, full, bs)
    o_sparse, _ = oracle.attention(q, k, v, sparse, bs)
    r = oracle.residual(o_dense, o_sparse)
    assert np.abs(r).max() > 0.01  # the dropped blocks matter here
    np.testing.assert_allclose(oracle.compensate(o_sparse, r), o_dense, rtol=0, atol=1e-14)
    # a full mask drops nothing: no residual
    assert np.array_equal(oracle.residual(o_dense, oracle.attention(q, k, v, full, bs)[0]), np.zeros_like(r))


# ------------------------------------------------------------ per-modality top-k


def test_modal_counts_rules():
    # 2 text + 14 image blocks: groups of 2 and 14 key blocks
    assert oracle.modal_counts([1.0, 0.5, 0.5, 0.15], 2, 16) == [[2, 7], [1, 2]]
    assert oracle.modal_counts([0.0, 0.0, 1.0, 0.01], 2, 16) == [[0, 0], [2, 1]]  # rho 0 keeps none; >0 keeps >= 1
    # no text blocks: no text rows and no text columns (the text-row counts are unused)
    assert oracle.modal_counts([0.3, 0.3, 0.3, 0.3], 0, 8) == [[0, 2], [0, 2]]


def test_modal_selection_brute_force():
    rng = np.random.default_rng(12)
    nB, n_text = 13, 3
    scores = rng.integers(-3, 4, size=(2, nB, nB)).astype(np.float32)  # many ties
    dens = [0.7, 0.3, 0.4, 0.25]
    kq = oracle.modal_counts(dens, n_text, nB)
    spans = ((0, n_text), (n_text, nB))
    got = np.zeros_like(scores, dtype=np.uint8)
    for a in (0, 1):
        for b in (0, 1):
            (r0, r1), (c0, c1) = spans[a], spans[b]
            if kq[a][b]:
                got[:, r0:r1, c0:c1] = oracle.topk_mask(np.ascontiguousarray(scores[:, r0:r1, c0:c1]), kq[a][b])
    for h in range(2):
        for i in range(nB):
            a = 0 if i < n_text else 1
            want = set()
            for b in (0, 1):
                c0, c1 = spans[b]
                order = sorted(range(c0, c1), key=lambda j: (-scores[h, i, j], j))
                want |= set(order[:kq[a][b]])
            assert set(np.flatnonzero(got[h, i]).tolist()) == want


def test_modal_selector_reduces_to_plain_without_text():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((2, 1, 1, 512, 64)).astype(np.float32)
    plain = oracle.select_mask(q, k, 64, 0.3)
    modal = oracle.select_mask_modal(q, k, 64, 0, [0.9, 0.9, 0.9, 0.3])
    assert np.array_equal(plain, modal)


# ------------------------------------------------------------ exact block mass (block-oracle selector)


def _dense_lse(q, k):
    nB = q.shape[-2] // 64
    full = np.ones((*q.shape[:-2], nB, nB), dtype=np.uint8)
    _, lse = oracle.attention(q, k, k, full, 64)
    return lse.reshape(q.shape[:-1])


def test_block_mass_rows_hold_one_unit_per_query_row():
    # with the dense LSE every query row's probabilities sum to 1: a Q block's masses sum to bs
    rng = np.random.default_rng(21)
    q, k = rng.standard_normal((2, 1, 2, 256, 64)).astype(np.float32)  # the inputs both functions see
    m = oracle.block_mass(q, k, _dense_lse(q, k), 64)
    np.testing.assert_allclose(m.sum(axis=-1), 64.0, rtol=1e-12)
    assert (m > 0).all()


def test_block_mass_brute_force_small():
    rng = np.random.default_rng(22)
    N, d, bs = 8, 4, 4
    q, k = rng.standard_normal((2, N, d))
    lse = rng.standard_normal(N)
    got = oracle.block_mass(q, k, lse, bs, scale=0.7)
    for i in range(2):
        for j in range(2):
            want = sum(math.exp(0.7 * float(q[r] @ k[c]) - lse[r])
                       for r in range(i * bs, (i + 1) * bs) for c in range(j * bs, (j + 1) * bs))
            assert abs(got[i, j] - want) <= 1e-12 * want


def test_exact_selector_keeps_the_block_that_holds_the_attention():
    rng = np.random.default_rng(23)
    q, k = (rng.standard_normal((2, 1, 1, 512, 64)) * 0.1).astype(np.float32)
    k[0, 0, 5 * 64 + 7] = 4.0 * q[0, 0, 2 * 64 + 3]  # one key aligned with one query of block 2
    m = oracle.block_mass(q, k, _dense_lse(q, k), 64)
    sel = oracle.select_mask_exact(m, 1.0 / 8)  # k = 1
    assert sel[0, 0, 2].tolist() == [0, 0, 0, 0, 0, 1, 0, 0]


# ---------------------------------------------------------------- ragged last block (reading R20)


def test_ragged_all_ones_mask_equals_dense_attention():
    # N = 75 at block 16: five blocks, the last holding 11 keys; every key of the row counts once
    H, N, d, bs = 2, 75, 8, 16
    q, k, v = _rand(H, N, d), _rand(H, N, d), _rand(H, N, d)
    nB = -(-N // bs)
    O, L = oracle.attention(q, k, v, np.ones((H, nB, nB), np.uint8), bs)
    assert O.shape == (H * N, d)
    for h in range(H):
        Od, Ld = _dense_library(q[h], k[h], v[h], 1.0 / math.sqrt(d), np.ones((N, N), bool))
        np.testing.assert_allclose(O[h * N:(h + 1) * N], Od, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L[h * N:(h + 1) * N], Ld, rtol=1e-12, atol=1e-12)


def test_ragged_block_diagonal_is_independent_block_attention():
    N, d, bs = 70, 4, 16   # blocks of 16, 16, 16, 16 and 6 tokens
    q, k, v = _rand(1, N, d), _rand(1, N, d), _rand(1, N, d)
    nB = -(-N // bs)
    O, L = oracle.attention(q, k, v, np.eye(nB, dtype=np.uint8)[None], bs, scale=0.5)
    for i in range(nB):
        sl = slice(i * bs, min((i + 1) * bs, N))
        n = sl.stop - sl.start
        Ob, Lb = _dense_library(q[0, sl], k[0, sl], v[0, sl], 0.5, np.ones((n, n), bool))
        np.testing.assert_allclose(O[sl], Ob, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L[sl], Lb, rtol=1e-12)


def test_ragged_block_mean_is_the_mean_of_the_tokens_it_holds():
    # integer tokens: every partial sum is exact in fp32, so the pooled value is the fp32
    # quotient of the exact sum by the block's token count (3 here, not the block size)
    N, d, bs = 11, 5, 4
    x = RNG.integers(-50, 50, size=(2, N, d)).astype(np.float32)
    m = oracle.block_mean(x, bs)
    assert m.shape == (2, 3, d)
    for i, (a, b) in enumerate([(0, 4), (4, 8), (8, 11)]):
        want = (x[:, a:b].astype(np.float64).sum(axis=1) / (b - a)).astype(np.float32)
        s = x[:, a:b].sum(axis=1, dtype=np.float64).astype(np.float32)
        np.testing.assert_array_equal(m[:, i], np.float32(s) / np.float32(b - a))
        np.testing.assert_allclose(m[:, i], want, rtol=1e-7)


def test_ragged_block_mass_rows_hold_one_unit_per_query_row():
    # with the dense LSE each query row's probabilities sum to 1, so a Q block's masses add up
    # to its row count: 16 for full blocks, 6 for the ragged last one
    N, d, bs = 38, 8, 16
    q, k = _rand(1, N, d), _rand(1, N, d)
    s = (q[0].astype(np.float64) @ k[0].astype(np.float64).T) / math.sqrt(d)
    lse = scipy.special.logsumexp(s, axis=-1)
    mass = oracle.block_mass(q, k, lse[None], bs)
    assert mass.shape == (1, 3, 3)
    np.testing.assert_allclose(mass[0].sum(axis=1), [16, 16, 6], rtol=1e-12)
    # the ragged block's mass against a brute-force sum over its 6 keys
    np.testing.assert_allclose(mass[0, 0, 2], np.exp(s[:16, 32:] - lse[:16, None]).sum(), rtol=1e-12)


# ---------------------------------------------------------------- token-level selection (readings R21-R23)


def test_query_groups_partition_and_sizes():
    q = _rand(384, 8)
    perm = oracle.query_groups(q, 128)
    assert sorted(perm.tolist()) == list(range(384))
    for g in range(3):
        grp = perm[g * 128:(g + 1) * 128]
        assert np.all(np.diff(grp) > 0)  # ascending inside a group
    with pytest.raises(ValueError):
        oracle.query_groups(_rand(300, 8), 128)


@pytest.mark.parametrize("m", [2, 3, 4, 5])
def test_query_groups_on_a_line_are_sorted_chunks(m):
    # points on one line: the principal direction is that line, so every median split keeps
    # the order along it and the groups are consecutive runs of the sorted coordinate
    C = 4
    t = RNG.permutation(m * C).astype(np.float64) * 0.37 + RNG.random(m * C) * 0.01
    e = np.array([3.0, -4.0, 0.0]) / 5.0
    q = (t[:, None] * e[None, :]).astype(np.float32)
    perm = oracle.query_groups(q, C)
    order = np.argsort(t)
    got = {frozenset(perm[g * C:(g + 1) * C].tolist()) for g in range(m)}
    # the direction's sign decides which end comes first; the runs themselves do not change
    want = {frozenset(order[g * C:(g + 1) * C].tolist()) for g in range(m)}
    assert got == want


def test_query_groups_separate_two_clusters():
    C = 16
    a = _rand(C, 6) * 0.1 + np.array([10, 0, 0, 0, 0, 0], np.float32)
    b = _rand(C, 6) * 0.1 - np.array([10, 0, 0, 0, 0, 0], np.float32)
    idx = RNG.permutation(2 * C)
    q = np.concatenate([a, b])[idx]
    perm = oracle.query_groups(q, C)
    in_b = set(np.where(idx >= C)[0].tolist())  # rows holding cluster b (the lower projections)
    assert set(perm[:C].tolist()) == in_b


def test_query_groups_follow_a_row_permutation():
    q = _rand(256, 5)
    perm = oracle.query_groups(q, 32)
    shuffle = RNG.permutation(256)
    perm2 = oracle.query_groups(q[shuffle], 32)
    for g in range(8):
        assert set(shuffle[perm2[g * 32:(g + 1) * 32]].tolist()) == set(perm[g * 32:(g + 1) * 32].tolist())


def test_token_mass_rows_hold_one_unit_per_query():
    N, d, C = 64, 8, 16
    q, k = _rand(N, d), _rand(N, d)
    s = (q.astype(np.float64) @ k.astype(np.float64).T) / math.sqrt(d)
    lse = scipy.special.logsumexp(s, axis=-1)
    perm = oracle.query_groups(q, C)
    mass = oracle.token_mass(q, k, lse, perm, C)
    np.testing.assert_allclose(mass.sum(axis=1), C, rtol=1e-12)
    # brute force of one entry, and the block mass when the groups are the blocks
    g, t = 2, 37
    want = sum(math.exp(s[r, t] - lse[r]) for r in perm[g * C:(g + 1) * C])
    assert math.isclose(mass[g, t], want, rel_tol=1e-12)
    ident = np.arange(N)
    mb = oracle.token_mass(q, k, lse, ident, C).reshape(N // C, N // C, C).sum(axis=2)
    np.testing.assert_allclose(mb, oracle.block_mass(q[None], k[None], lse[None], C)[0], rtol=1e-12)


def test_select_tokens_keeps_the_largest_with_low_index_ties():
    mass = RNG.integers(0, 6, size=(5, 40)).astype(np.float64)
    sel = oracle.select_tokens(mass, 0.25)
    K = 10
    assert sel.shape == (5, K)
    for g in range(5):
        chosen = set(sel[g].tolist())
        assert np.all(np.diff(sel[g]) > 0)
        rest = [t for t in range(40) if t not in chosen]
        lo = min(mass[g, t] for t in chosen)
        assert all(mass[g, t] <= lo for t in rest)
        # a tie at the boundary goes to the lower indices
        assert all(t > max(c for c in chosen if mass[g, c] == lo) for t in rest if mass[g, t] == lo)


def test_token_attention_all_tokens_is_dense_and_subset_is_masked_dense():
    N, d, C = 48, 6, 16
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    perm = oracle.query_groups(q, C)
    full = np.tile(np.arange(N), (N // C, 1))
    O, L = oracle.token_attention(q, k, v, perm, full, C, scale=0.4)
    Od, Ld = _dense_library(q, k, v, 0.4, np.ones((N, N), bool))
    np.testing.assert_allclose(O, Od, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(L, Ld, rtol=1e-12)
    tokens = np.stack([np.sort(RNG.choice(N, size=7, replace=False)) for _ in range(N // C)])
    O, L = oracle.token_attention(q, k, v, perm, tokens, C, scale=0.4)
    allowed = np.zeros((N, N), bool)
    for g in range(N // C):
        allowed[np.ix_(perm[g * C:(g + 1) * C], tokens[g])] = True
    Od, Ld = _dense_library(q, k, v, 0.4, allowed)
    np.testing.assert_allclose(O, Od, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(L, Ld, rtol=1e-12)
    one = np.full((N // C, 1), 5)
    O, L = oracle.token_attention(q, k, v, perm, one, C, scale=0.4)
    np.testing.assert_allclose(O, np.tile(v[5].astype(np.float64), (N, 1)), rtol=1e-12)
    np.testing.assert_allclose(L, 0.4 * (q.astype(np.float64) @ k[5].astype(np.float64)), rtol=1e-12)
