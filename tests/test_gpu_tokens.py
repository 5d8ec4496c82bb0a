"""GPU parity of bsa_forward_tokens (token-sparse attention over tile-aligned query groups)
against the CPU oracle.

The groups (median-split principal-direction grouping) and each group's tokens (the exact
per-group token mass from the dense LSE, top-K) come from the oracle and are the kernel's
inputs, as the index is bsa_forward's. O within max-abs 2e-2 and mean-abs 2e-3, LSE within
1e-3, every row; an out-of-range index raises BSA_ERR_INVALID_ARG without a fault.
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
C = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bbuild.build()
    bb.load()
    bb.bsa_debug_config(0, 0)


def _groups_and_tokens(inp, w, density):
    BH = w.B * w.H
    q = inp["q"].reshape(BH, w.N, w.d)
    k = inp["k"].reshape(BH, w.N, w.d)
    full = np.ones((BH, w.nQB, w.nKB), np.uint8)
    _, lse = oracle.attention(q, k, k, full, w.block)  # dense LSE (values unused)
    lse = lse.reshape(BH, w.N)
    perms, toks = [], []
    for h in range(BH):
        perm = oracle.query_groups(q[h], C)
        mass = oracle.token_mass(q[h], k[h], lse[h], perm, C)
        perms.append(perm)
        toks.append(oracle.select_tokens(mass, density))
    return np.stack(perms), np.stack(toks)


CASES = {
    "bf16_d128": (wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, N=1024), 0.1),
    "bf16_d64": (wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2, N=1024), 0.2),
    "fp32_d64": (wl.scaled(wl.WORKLOADS["tiny"], N=512), 0.25),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_token_forward_matches_oracle(name):
    w, density = CASES[name]
    inp = wl.make_inputs(w)
    perm, toks = _groups_and_tokens(inp, w, density)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    perm_d = torch.from_numpy(perm.astype(np.int32)).cuda()
    toks_d = torch.from_numpy(toks.astype(np.int32)).cuda()
    O, L = bb.forward_tokens(q, k, v, perm_d, toks_d)
    torch.cuda.synchronize()
    BH = w.B * w.H
    Og = O.float().reshape(BH, w.N, w.d).cpu().numpy().astype(np.float64)
    Lg = L.reshape(BH, w.N).cpu().numpy().astype(np.float64)
    qf, kf, vf = (inp[n].reshape(BH, w.N, w.d) for n in ("q", "k", "v"))
    for h in range(BH):
        O_ref, L_ref = oracle.token_attention(qf[h], kf[h], vf[h], perm[h], toks[h], C)
        err = np.abs(Og[h] - O_ref)
        assert err.max() <= gu.O_MAX_ABS and err.mean() <= gu.O_MEAN_ABS, (h, err.max(), err.mean())
        assert np.abs(Lg[h] - L_ref).max() <= gu.LSE_MAX_ABS


@pytest.mark.parametrize("d,density", [(128, 0.15), (64, 0.1)])
def test_token_forward_working_size_sampled_groups(d, density):
    # the dynamic_topk shape (N = 8192, 64 groups of 128 per head) at 15% / 10% of the keys:
    # 1228 / 819 tokens per group, so the last 128-key step is ragged. Groups from the
    # oracle, token sets seeded (the forward must hold for any ascending set); every row
    # of a seeded sample of groups against the oracle's token attention.
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=2, d=d)
    inp = wl.make_inputs(w)
    BH, G = w.B * w.H, w.N // C
    K = bb.tokens_per_group(w.N, density)
    assert K % C != 0
    qf, kf, vf = (inp[n].reshape(BH, w.N, w.d) for n in ("q", "k", "v"))
    perm = np.stack([oracle.query_groups(qf[h], C) for h in range(BH)])
    rng = np.random.default_rng(d)
    toks = np.stack([[np.sort(rng.choice(w.N, size=K, replace=False)) for _ in range(G)] for _ in range(BH)])
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    O, L = bb.forward_tokens(q, k, v, torch.from_numpy(perm.astype(np.int32)).cuda(),
                             torch.from_numpy(toks.astype(np.int32)).cuda())
    torch.cuda.synchronize()
    Og = O.float().reshape(BH, w.N, w.d).cpu().numpy().astype(np.float64)
    Lg = L.reshape(BH, w.N).cpu().numpy().astype(np.float64)
    for h in range(BH):
        for g in sorted({0, G - 1} | set(rng.choice(G, size=6, replace=False).tolist())):
            rows = perm[h, g * C:(g + 1) * C]
            sub = np.arange(C)  # the group alone: its own permutation is 0..127
            O_ref, L_ref = oracle.token_attention(qf[h][rows], kf[h], vf[h], sub, toks[h, g][None], C)
            err = np.abs(Og[h][rows] - O_ref)
            assert err.max() <= gu.O_MAX_ABS and err.mean() <= gu.O_MEAN_ABS, (h, g, err.max(), err.mean())
            assert np.abs(Lg[h][rows] - L_ref).max() <= gu.LSE_MAX_ABS


def test_token_forward_out_of_range_index_is_reported():
    w, density = CASES["bf16_d64"]
    inp = wl.make_inputs(w)
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    BH = w.B * w.H
    perm = torch.arange(w.N, dtype=torch.int32).repeat(BH, 1).cuda()
    toks = torch.zeros((BH, w.N // C, 8), dtype=torch.int32).cuda()
    toks[0, 1, 3] = w.N + 5  # past the sequence: skipped and reported
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    bb.forward_tokens(q, k, v, perm, toks, ws=ws, check=False)
    assert bb.bsa_check_device_error(ws) == bb.ERR_INVALID_ARG
    O, L = bb.forward_tokens(q, k, v, perm, torch.zeros_like(toks))  # the context is still usable
    torch.cuda.synchronize()
    assert torch.isfinite(L).all()


MASS_RTOL = 2e-3


@pytest.mark.parametrize("name", sorted(CASES))
def test_token_selection_matches_oracle(name):
    # masses against the oracle's (double); the kept tokens bit for bit against the oracle's
    # selection rule applied to the kernel's own fp32 masses (the decision taken in the kernel's
    # precision: at token granularity many masses sit within rounding of the K-th one), and
    # within rounding of the K-th double mass; then the token forward on the GPU's selection
    w, density = CASES[name]
    inp = wl.make_inputs(w)
    BH, G = w.B * w.H, w.N // C
    qf, kf, vf = (inp[n].reshape(BH, w.N, w.d) for n in ("q", "k", "v"))
    full = np.ones((BH, w.nQB, w.nKB), np.uint8)
    _, lse = oracle.attention(qf, kf, kf, full, w.block)
    lse = lse.reshape(BH, w.N)
    perm = np.stack([oracle.query_groups(qf[h], C) for h in range(BH)])
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    perm_d = torch.from_numpy(perm.astype(np.int32)).cuda()
    lse_d = torch.from_numpy(lse.astype(np.float32)).cuda()
    toks, ws = bb.select_tokens(q, k, perm_d, lse_d, density)
    torch.cuda.synchronize()
    K = bb.tokens_per_group(w.N, density)
    got = ws[256:256 + BH * G * w.N * 4].view(torch.float32).reshape(BH, G, w.N).cpu().numpy()
    sel = toks.cpu().numpy()
    for h in range(BH):
        ref = oracle.token_mass(qf[h], kf[h], lse[h], perm[h], C)
        np.testing.assert_allclose(got[h], ref, rtol=MASS_RTOL, atol=1e-6 * C)
        np.testing.assert_array_equal(sel[h], oracle.select_tokens(got[h].astype(np.float64), density))
        for g in range(G):
            order = np.sort(ref[g])[::-1]
            assert np.all(ref[g][sel[h, g]] >= order[K - 1] * (1 - 2 * MASS_RTOL))
    O, L = bb.forward_tokens(q, k, v, perm_d, toks)
    torch.cuda.synchronize()
    Og = O.float().reshape(BH, w.N, w.d).cpu().numpy().astype(np.float64)
    Lg = L.reshape(BH, w.N).cpu().numpy().astype(np.float64)
    for h in range(BH):
        O_ref, L_ref = oracle.token_attention(qf[h], kf[h], vf[h], perm[h], sel[h], C)
        err = np.abs(Og[h] - O_ref)
        assert err.max() <= gu.O_MAX_ABS and err.mean() <= gu.O_MEAN_ABS
        assert np.abs(Lg[h] - L_ref).max() <= gu.LSE_MAX_ABS


@pytest.mark.parametrize("N,density", [(8192, 0.15), (40960, 0.05)])
def test_token_selection_working_sizes(N, density):
    # the selection at the dynamic_topk size and above the former shared-memory limit of
    # about 37k keys: the dense LSE from the GPU's full-index forward (pass 1), groups from
    # a seeded permutation; masses of sampled groups against the oracle's (double, same
    # LSE), and every group's kept tokens bit for bit against the oracle's rule on the
    # kernel's own fp32 masses
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=1, N=N)
    inp = wl.make_inputs(w)
    BH, G = w.B * w.H, N // C
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    ones = np.ones((w.B, w.H, w.nQB, w.nKB), dtype=np.uint8)
    full = bb.build_mask(None, None, w.block, spec=bb.explicit_spec(
        torch.from_numpy(gu.mask_bitmap_words(ones).reshape(-1)).cuda()), shape=(w.B, w.H, N, w.d))
    _, lse = bb.forward(q, k, v, full)
    del full
    rng = np.random.default_rng(N)
    perm = np.stack([rng.permutation(N) for _ in range(BH)]).astype(np.int32)
    perm_d = torch.from_numpy(perm).cuda()
    toks, ws = bb.select_tokens(q, k, perm_d, lse, density)
    torch.cuda.synchronize()
    K = bb.tokens_per_group(N, density)
    got = ws[256:256 + BH * G * N * 4].view(torch.float32).reshape(BH, G, N).cpu().numpy()
    sel = toks.cpu().numpy()
    lse_h = lse.reshape(BH, N).cpu().numpy().astype(np.float64)
    qf, kf = (inp[n].reshape(BH, N, w.d) for n in ("q", "k"))
    for h in range(BH):
        for g in sorted({0, G - 1} | set(rng.choice(G, size=4, replace=False).tolist())):
            rows = perm[h, g * C:(g + 1) * C]
            ref = oracle.token_mass(qf[h][rows], kf[h], lse_h[h][rows], np.arange(C), C)[0]
            np.testing.assert_allclose(got[h, g], ref, rtol=MASS_RTOL, atol=1e-6 * C)
        np.testing.assert_array_equal(sel[h], oracle.select_tokens(got[h].astype(np.float64), density))
        assert sel.shape[-1] == K


def _sse(x, perm):
    """Within-group sum of squared distances to the group mean (double)."""
    g = x[perm].reshape(-1, C, x.shape[1]).astype(np.float64)
    return float(((g - g.mean(axis=1, keepdims=True)) ** 2).sum())


def test_query_groups_on_a_line_match_the_oracle():
    # points on one line: every median split is an exact cut of the sorted coordinate, so
    # the GPU's groups are the oracle's, bit for bit (4 and 5 groups: even and odd splits)
    for m in (4, 5):
        N, d = m * C, 64
        rng = np.random.default_rng(m)
        t = rng.permutation(N).astype(np.float64) * 0.5 + rng.random(N) * 0.1
        e = rng.standard_normal(d)
        e /= np.linalg.norm(e)
        q = (t[:, None] * e[None, :]).astype(np.float32)
        perm = bb.query_groups(torch.from_numpy(q).reshape(1, 1, N, d).cuda())
        torch.cuda.synchronize()
        assert np.array_equal(perm.cpu().numpy()[0], oracle.query_groups(q, C))


def anisotropic_queries(N, d, seed):
    """Gaussian queries with distinct leading variances (scales 81, 27, 9, 3, 1.5, then 1) in a
    seeded random orientation: every split of the grouping has a clear principal direction."""
    rng = np.random.default_rng(seed)
    sc = np.ones(d)
    sc[:5] = [81, 27, 9, 3, 1.5]
    rot, _ = np.linalg.qr(rng.standard_normal((d, d)))
    return ((rng.standard_normal((N, d)) * sc) @ rot.T / 8).astype(np.float32)


@pytest.mark.parametrize("d,seed,dtype", [(128, 1, "fp32"), (64, 2, "fp32"), (128, 3, "bf16"), (64, 4, "bf16")])
def test_query_groups_anisotropic_match_the_oracle_exactly(d, seed, dtype):
    # The GPU takes each principal direction by 32 fp32 power-iteration steps. Against the
    # exact eigenvector its direction errs by at most ~ T * rho^32 (rho = lam2/lam1, T the
    # tangent of the start vector's angle, <= 10 here) plus fp32 rounding ~ 4*d*2^-24, so a
    # difference of two projections errs by at most eps = 2 * rmax * (10 * rho^32 + 4*d*2^-24)
    # (rmax: largest centred row norm). When every cut's gap exceeds its eps, no row can change
    # sides and the groups must equal the oracle's bit for bit.
    # bf16 at d = 128 takes the tcgen05 scatter pass (raw sums of exact products in fp32, the
    # segment's mean term taken off afterwards); the oracle sees the same bf16-rounded values.
    N = 1024
    x = anisotropic_queries(N, d, seed)
    if dtype == "bf16":
        xt = torch.from_numpy(x).to(torch.bfloat16)
        x = xt.float().numpy()
    splits = []
    ref = oracle.query_groups(x, C, splits=splits)
    for sp in splits:
        rho = sp["lam2"] / sp["lam1"]
        eps = 2.0 * sp["rmax"] * (10.0 * rho ** 32 + 4.0 * d * 2.0 ** -24)
        assert sp["gap"] > eps, (sp, eps)  # the data leave no row within eps of a cut
    qdev = (xt if dtype == "bf16" else torch.from_numpy(x)).reshape(1, 1, N, d).cuda()
    perm = bb.query_groups(qdev)
    torch.cuda.synchronize()
    assert np.array_equal(perm.cpu().numpy()[0], ref)


@pytest.mark.parametrize("name", sorted(CASES))
def test_query_groups_partition_and_quality(name):
    # a valid partition into ascending groups of 128, as tight as the oracle's (its direction
    # is an fp32 power iteration, so a row within rounding of a median may change sides)
    w, _ = CASES[name]
    inp = wl.make_inputs(w)
    BH = w.B * w.H
    q = gu.upload(inp, "q")
    perm = bb.query_groups(q)
    torch.cuda.synchronize()
    got = perm.cpu().numpy()
    qf = inp["q"].reshape(BH, w.N, w.d)
    for h in range(BH):
        assert sorted(got[h].tolist()) == list(range(w.N))
        assert np.all(np.diff(got[h].reshape(-1, C), axis=1) > 0)
        ref = oracle.query_groups(qf[h], C)
        assert _sse(qf[h], got[h]) <= 1.01 * _sse(qf[h], ref)


def test_query_groups_repeat_run_to_run():
    # every sum of the grouping runs in a fixed order (slices in order, blocks in order), so
    # the same queries give the same groups on every call, at a size with several slices
    # per segment on the top levels
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=4)
    q = gu.upload(wl.make_inputs(w), "q")
    first = bb.query_groups(q)
    for _ in range(2):
        assert torch.equal(bb.query_groups(q), first)


def test_token_path_end_to_end_on_the_gpu():
    # groups, dense LSE, selection and the token forward all on the GPU; the forward checked
    # against the oracle's token attention over the GPU's own groups and tokens
    w, density = CASES["bf16_d128"]
    inp = wl.make_inputs(w)
    BH = w.B * w.H
    q, k, v = (gu.upload(inp, n) for n in ("q", "k", "v"))
    perm = bb.query_groups(q)
    ones = np.ones((w.B, w.H, w.nQB, w.nKB), dtype=np.uint8)
    full = bb.build_mask(None, None, w.block, spec=bb.explicit_spec(
        torch.from_numpy(gu.mask_bitmap_words(ones).reshape(-1)).cuda()), shape=(w.B, w.H, w.N, w.d))
    _, lse = bb.forward(q, k, v, full)
    toks, _ = bb.select_tokens(q, k, perm, lse, density)
    O, L = bb.forward_tokens(q, k, v, perm, toks)
    torch.cuda.synchronize()
    pg, tg = perm.cpu().numpy(), toks.cpu().numpy()
    Og = O.float().reshape(BH, w.N, w.d).cpu().numpy().astype(np.float64)
    Lg = L.reshape(BH, w.N).cpu().numpy().astype(np.float64)
    qf, kf, vf = (inp[n].reshape(BH, w.N, w.d) for n in ("q", "k", "v"))
    for h in range(BH):
        O_ref, L_ref = oracle.token_attention(qf[h], kf[h], vf[h], pg[h], tg[h], C)
        err = np.abs(Og[h] - O_ref)
        assert err.max() <= gu.O_MAX_ABS and err.mean() <= gu.O_MEAN_ABS
        assert np.abs(Lg[h] - L_ref).max() <= gu.LSE_MAX_ABS
