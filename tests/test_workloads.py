"""Input generator checks: determinism, bf16 rounding, recipe structure."""
import numpy as np
import torch

from block_sparse_attention_mean_gb300 import workloads as wl


def test_round_to_bf16_matches_torch():
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32) * 37
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 3.0]
    xf, bits = wl.round_to_bf16(x)
    t = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(t.view(torch.int16).numpy().view(np.uint16), bits)
    assert np.array_equal(t.float().numpy(), xf)


def test_generator_is_deterministic_and_exact_bf16():
    w = wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=2)
    a, b = wl.make_inputs(w), wl.make_inputs(w)
    for n in ("q", "k", "v"):
        assert np.array_equal(a[n], b[n])
        assert a[n].shape == (1, 2, 4224, 64)
        # float32 copy holds exactly the bf16 values
        assert np.array_equal(a[n].view(np.uint32) >> 16, a[n + "_bits"].astype(np.uint32))
        assert np.all((a[n].view(np.uint32) & 0xFFFF) == 0)


def test_tiny_mask_has_diagonal():
    inp = wl.make_inputs(wl.WORKLOADS["tiny"])
    m = inp["mask"]
    assert m.shape == (1, 2, 8, 8)
    assert np.all(m[:, :, np.arange(8), np.arange(8)] == 1)
    assert inp["q"].dtype == np.float32 and "q_bits" not in inp


def test_cuboid_permutation_groups_cuboids():
    perm = wl.cuboid_permutation((8, 8, 8))
    assert np.array_equal(np.sort(perm), np.arange(512))
    t, h, w = np.unravel_index(perm, (8, 8, 8))
    for c in range(8):
        sl = slice(c * 64, (c + 1) * 64)
        assert len({(a, b, cc) for a, b, cc in zip(t[sl] // 4, h[sl] // 4, w[sl] // 4)}) == 1


def test_blurred_recipe_is_smooth_and_unit_variance():
    w = wl.scaled(wl.WORKLOADS["video_cuboid"], H=1, d=16)
    q = wl.make_inputs(w)["q"][0, 0, 256:]
    assert 0.7 < float(q.std()) < 1.3
    # neighbouring tokens inside a cuboid are strongly correlated
    c = np.corrcoef(q[0:63].ravel(), q[1:64].ravel())[0, 1]
    assert c > 0.5


def test_clustered_recipe_blocks_are_coherent():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=1, N=2048)
    inp = wl.make_inputs(w)
    q = inp["q"][0, 0]
    # mean over a block of one cluster keeps the centroid norm (noise averages out)
    norms = np.linalg.norm(q.reshape(-1, 64, 128).mean(1), axis=1)
    assert np.median(norms) > 5.0
