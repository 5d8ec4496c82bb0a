"""CPU oracle for block-sparse attention with a mean-pooled top-k selector.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check
and by the benchmark's CPU-baseline leg. The product path never imports it.

The arithmetic lives in ``bsa_oracle.c`` (plain C, double precision for the
attention, the fp32 rules of the selector spelled out there). This module
compiles it with gcc and wraps it with ctypes and numpy. The residual
compensation definitions (``residual``, ``compensate``) are one-line numpy
expressions in double precision.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

OK = 0
ERR_ARG = 1
ERR_NONFINITE = 5


def build(force: bool = False) -> str:
    """Compile liboracle.so (gcc, -O2, OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
    lib.bsa_oracle_block_mean.argtypes = [P, i64, i64, i32, i32, P]
    lib.bsa_oracle_block_scores.argtypes = [P, P, i64, i32, i32, i32, P]
    lib.bsa_oracle_topk_count.argtypes = [f32, i32]
    lib.bsa_oracle_topk.argtypes = [P, i64, i32, i32, P]
    lib.bsa_oracle_band_mask.argtypes = [i32, i32, i32, P, i32, P]
    lib.bsa_oracle_cuboid_mask.argtypes = [i32, i32, i32, i32, P]
    lib.bsa_oracle_mask_to_index.argtypes = [P, i64, i32, P, P, P]
    lib.bsa_oracle_mask_to_index.restype = i64
    lib.bsa_oracle_attention.argtypes = [P, P, P, i64, i64, i32, i32, P, f64, P, i64, P, P]
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def _check(code: int, what: str):
    if code != OK:
        raise OracleError(code, what)


def block_mean(x: np.ndarray, bs: int) -> np.ndarray:
    """Mean-pooled block representation: x [..., N, d] fp32 -> [..., ceil(N/bs), d] fp32
    (a ragged last block averages the tokens it holds)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    *lead, N, d = x.shape
    heads = int(np.prod(lead)) if lead else 1
    out = np.empty((*lead, -(-N // bs), d), np.float32)
    _check(_load().bsa_oracle_block_mean(_ptr(x), heads, N, d, bs, _ptr(out)), "block_mean")
    return out


def block_scores(qbar: np.ndarray, kbar: np.ndarray) -> np.ndarray:
    """Scores [..., nQB, nKB] of pooled blocks (fmaf chain over channels)."""
    qbar = np.ascontiguousarray(qbar, dtype=np.float32)
    kbar = np.ascontiguousarray(kbar, dtype=np.float32)
    *lead, nQB, d = qbar.shape
    nKB = kbar.shape[-2]
    heads = int(np.prod(lead)) if lead else 1
    out = np.empty((*lead, nQB, nKB), np.float32)
    _check(_load().bsa_oracle_block_scores(_ptr(qbar), _ptr(kbar), heads, nQB, nKB, d, _ptr(out)),
           "block_scores")
    return out


def topk_count(density: float, nKB: int) -> int:
    return int(_load().bsa_oracle_topk_count(float(density), int(nKB)))


def topk_mask(scores: np.ndarray, k: int) -> np.ndarray:
    """uint8 mask [..., nQB, nKB] of the k best blocks per row (ties -> lower index)."""
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    *lead, nKB = scores.shape
    rows = int(np.prod(lead)) if lead else 1
    out = np.empty(scores.shape, np.uint8)
    _check(_load().bsa_oracle_topk(_ptr(scores), rows, nKB, int(k), _ptr(out)), "topk")
    return out


def band_mask(nB: int, n_text: int, band: int, anchors: Sequence[int]) -> np.ndarray:
    a = np.ascontiguousarray(np.array(list(anchors) or [0], dtype=np.int32))
    out = np.empty((nB, nB), np.uint8)
    _check(_load().bsa_oracle_band_mask(nB, n_text, band, _ptr(a), len(anchors), _ptr(out)),
           "band_mask")
    return out


def cuboid_mask(n_text: int, grid: Tuple[int, int, int]) -> np.ndarray:
    gt, gh, gw = grid
    nB = n_text + gt * gh * gw
    out = np.empty((nB, nB), np.uint8)
    _check(_load().bsa_oracle_cuboid_mask(n_text, gt, gh, gw, _ptr(out)), "cuboid_mask")
    return out


def mask_to_index(mask: np.ndarray):
    """(row_ptr int32 [R+1], col_idx int32 [nnz], bitmap uint32 [R, ceil(nKB/32)])."""
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    nKB = mask.shape[-1]
    R = mask.size // nKB
    W = (nKB + 31) // 32
    row_ptr = np.empty(R + 1, np.int32)
    col_idx = np.empty(max(int(mask.sum()), 1), np.int32)
    bitmap = np.empty((R, W), np.uint32)
    nnz = _load().bsa_oracle_mask_to_index(_ptr(mask), R, nKB, _ptr(row_ptr), _ptr(col_idx),
                                           _ptr(bitmap))
    if nnz < 0:
        raise OracleError(ERR_ARG, "mask_to_index")
    return row_ptr, col_idx[:nnz].copy(), bitmap


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray, bs: int,
              scale: Optional[float] = None, rows: Optional[np.ndarray] = None):
    """Masked attention in double for selected rows.

    q, k, v: fp32 [..., N, d]; mask: uint8 [..., nQB, nKB] (same leading dims);
    rows: int64 global row ids (flattened head * N + r); default all rows.
    Returns (O float64 [n_rows, d], LSE float64 [n_rows]).
    """
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    *lead, N, d = q.shape
    heads = int(np.prod(lead)) if lead else 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if rows is None:
        rows = np.arange(heads * N, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    O = np.empty((rows.size, d), np.float64)
    L = np.empty(rows.size, np.float64)
    _check(_load().bsa_oracle_attention(_ptr(q), _ptr(k), _ptr(v), heads, N, d, bs, _ptr(mask),
                                        float(scale), _ptr(rows), rows.size, _ptr(O), _ptr(L)),
           "attention")
    return O, L


def select_mask(q: np.ndarray, k: np.ndarray, bs: int, density: float) -> np.ndarray:
    """Naive BSA selector end to end: pool, score, top-k -> uint8 mask [..., nQB, nKB]."""
    qbar = block_mean(q, bs)
    kbar = block_mean(k, bs)
    s = block_scores(qbar, kbar)
    return topk_mask(s, topk_count(density, s.shape[-1]))


def modal_counts(density: Sequence[float], n_text: int, nB: int):
    """Blocks kept by a query block of modality a among the key blocks of modality b.

    [P1] "多模态DiT中的块稀疏注意力：从原理到工程落地" §3.3: a density per modality group
    instead of one global rate. Blocks [0, n_text) are text (0), the rest image (1);
    density = (text->text, text->image, image->text, image->image). A group of n
    key blocks with density rho keeps the selector's count for n blocks, and none
    when rho is 0 (or the group is empty).
    """
    n = (n_text, nB - n_text)
    kq = [[0, 0], [0, 0]]
    for a in (0, 1):
        for b in (0, 1):
            rho, nb = float(density[2 * a + b]), n[b]
            kq[a][b] = 0 if (nb == 0 or rho <= 0.0) else topk_count(rho, nb)
    return kq


def select_mask_modal(q: np.ndarray, k: np.ndarray, bs: int, n_text: int, density: Sequence[float]) -> np.ndarray:
    """Per-modality selector: pool, score, then the top-k of every (query, key) modality group."""
    qbar = block_mean(q, bs)
    kbar = block_mean(k, bs)
    s = block_scores(qbar, kbar)
    nB = s.shape[-1]
    kq = modal_counts(density, n_text, nB)
    spans = ((0, n_text), (n_text, nB))
    out = np.zeros(s.shape, np.uint8)
    for a in (0, 1):
        r0, r1 = spans[a]
        for b in (0, 1):
            c0, c1 = spans[b]
            if kq[a][b] == 0 or r1 <= r0:
                continue
            out[..., r0:r1, c0:c1] = topk_mask(np.ascontiguousarray(s[..., r0:r1, c0:c1]), kq[a][b])
    return out


def block_mass(q: np.ndarray, k: np.ndarray, lse: np.ndarray, bs: int, scale: Optional[float] = None) -> np.ndarray:
    """Exact attention mass of every (Q block, KV block) pair, in double.

    [P3] "Can sparse attention close the quality gap in diffusion transformers",
    section "质量差距有三个可分离来源" (the oracle selectors): with the dense row
    logsumexp LSE_r, mass_ij = sum over rows r of Q block i and keys c of KV block j
    of exp(scale * q_r . k_c - LSE_r). Returns [..., nQB, nKB].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    *lead, N, d = q.shape
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nB = -(-N // bs)  # a ragged last block holds the rows and keys up to N
    out = np.empty((*lead, nB, nB))
    qf, kf = q.reshape(-1, N, d), k.reshape(-1, N, d)
    lf = np.asarray(lse, dtype=np.float64).reshape(-1, N)
    of = out.reshape(-1, nB, nB)
    pp = np.zeros((nB * bs, nB * bs))
    for h in range(qf.shape[0]):
        pp[:N, :N] = np.exp(sc * (qf[h] @ kf[h].T) - lf[h][:, None])
        of[h] = pp.reshape(nB, bs, nB, bs).sum(axis=(1, 3))
    return out


def select_mask_exact(mass: np.ndarray, density: float) -> np.ndarray:
    """The block-oracle selector: top-k blocks per Q block by mass (ties -> lower index)."""
    return topk_mask(np.asarray(mass, dtype=np.float32), topk_count(density, mass.shape[-1]))


def residual(o_dense: np.ndarray, o_sparse: np.ndarray) -> np.ndarray:
    """Residual of sparse attention at an anchor step, in double.

    [P3] "Can sparse attention close the quality gap in diffusion transformers",
    section "残差补偿找回被丢弃的尾部": the dense-minus-sparse residual R = O_dense - O_sparse
    is measured at an anchor step and reused at later steps.
    """
    return np.asarray(o_dense, dtype=np.float64) - np.asarray(o_sparse, dtype=np.float64)


def compensate(o_sparse: np.ndarray, r: np.ndarray) -> np.ndarray:
    """Residual-compensated output of a later step, O_sparse + R, in double (same section)."""
    return np.asarray(o_sparse, dtype=np.float64) + np.asarray(r, dtype=np.float64)


# ---------------------------------------------------------------- token-level selection
#
# [P3] "Can sparse attention close the quality gap in diffusion transformers", section
# "token 级选择需要瓦片对齐的查询分组": queries of a head are put in groups of exactly C
# similar queries (C = the kernel's query tile) by a median split along the principal
# direction, applied recursively; each group then shares one set of individually
# selected KV tokens, gathered by index. The exact token selection uses the dense
# probabilities (the token oracle of section "质量差距有三个可分离来源"): per group and key
# token, the attention mass the group's queries give it under dense attention.


def query_groups(q: np.ndarray, C: int, splits: Optional[list] = None) -> np.ndarray:
    """Median-split principal-direction grouping of one head's queries (reading R21).

    q: [N, d] (N a multiple of C). A group of m*C rows (m >= 2) is centred, projected on the
    eigenvector of the largest eigenvalue of its scatter matrix (sign: its entry of largest
    magnitude positive), its rows ordered by (projection, row index), and cut after the
    first ceil(m/2)*C rows; the two halves are split again until every group holds C rows.
    Returns perm [N]: group g is rows perm[g*C:(g+1)*C], groups in depth-first order
    (first half before second half), rows inside a group in ascending index order.
    If `splits` is a list, one record per split is appended to it (for tests that bound how
    far an inexact computation may be from this one): the two largest eigenvalues, the gap
    between the projections on either side of the cut, and the largest centred row norm.
    """
    x = np.asarray(q, dtype=np.float64)
    N = x.shape[0]
    if C <= 0 or N % C != 0:
        raise ValueError("N must be a positive multiple of C")
    out = []

    def split(rows: np.ndarray):
        m = rows.size // C
        if m == 1:
            out.append(np.sort(rows))
            return
        xc = x[rows] - x[rows].mean(axis=0)
        w, vecs = np.linalg.eigh(xc.T @ xc)
        u = vecs[:, np.argmax(w)]
        if u[np.argmax(np.abs(u))] < 0:
            u = -u
        proj = xc @ u
        order = rows[np.lexsort((rows, proj))]
        cut = -(-m // 2) * C
        if splits is not None:
            p = np.sort(proj)
            splits.append({"lam1": float(w[-1]), "lam2": float(w[-2]), "gap": float(p[cut] - p[cut - 1]),
                           "rmax": float(np.sqrt((xc * xc).sum(axis=1)).max())})
        split(order[:cut])
        split(order[cut:])

    split(np.arange(N))
    return np.concatenate(out)


def token_mass(q: np.ndarray, k: np.ndarray, lse: np.ndarray, perm: np.ndarray, C: int,
               scale: Optional[float] = None) -> np.ndarray:
    """Exact attention mass of every (query group, key token) pair of one head, in double:
    mass[g, t] = sum over rows r of group g of exp(scale * q_r . k_t - LSE_r), with the dense
    row logsumexp LSE_r. Returns [N/C, N]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    sc = 1.0 / math.sqrt(q.shape[1]) if scale is None else float(scale)
    G = q.shape[0] // C
    out = np.empty((G, k.shape[0]))
    for g in range(G):
        rows = perm[g * C:(g + 1) * C]
        out[g] = np.exp(sc * (q[rows] @ k.T) - lse[rows][:, None]).sum(axis=0)
    return out


def select_tokens(mass: np.ndarray, density: float) -> np.ndarray:
    """The token oracle's selection (reading R22): per group the K = max(1, floor(density * N))
    tokens of largest mass, ties to the lower index; returns [groups, K], ascending per row."""
    G, N = mass.shape
    K = topk_count(density, N)
    sel = np.empty((G, K), np.int64)
    for g in range(G):
        order = np.lexsort((np.arange(N), -mass[g]))  # mass descending, then index ascending
        sel[g] = np.sort(order[:K])
    return sel


def token_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, perm: np.ndarray, tokens: np.ndarray,
                    C: int, scale: Optional[float] = None):
    """Token-sparse attention of one head in double (reading R23): each row r of group g attends
    to the keys tokens[g] only, O_r = sum_t softmax_t(scale * q_r . k_t) v_t and
    LSE_r = ln sum_t exp(scale * q_r . k_t), t over tokens[g]. Returns O [N, d], LSE [N] in row order."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    N, d = q.shape
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    O = np.empty((N, v.shape[1]))
    L = np.empty(N)
    for g in range(N // C):
        rows = perm[g * C:(g + 1) * C]
        t = tokens[g]
        s = sc * (q[rows] @ k[t].T)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        O[rows] = (p @ v[t]) / l
        L[rows] = (m + np.log(l))[:, 0]
    return O, L
