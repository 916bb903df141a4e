"""Pins for the oracle's randomized Hadamard transform and residual VQ."""
import math

import numpy as np
import pytest

import synth
from oracle import rvq as R


@pytest.mark.parametrize("n", [1, 2, 4, 8, 64])
def test_sylvester_is_orthogonal_and_symmetric(n):
    h = R.sylvester(n)
    assert np.allclose(h @ h, np.eye(n), atol=1e-14)
    assert np.array_equal(h, h.T)
    assert np.allclose(np.abs(h), 1 / np.sqrt(n))


def test_sylvester_small_explicit():
    h4 = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]]) / 2.0
    assert np.array_equal(R.sylvester(4), h4)


@pytest.mark.parametrize("n", [2, 8, 32, 64])
def test_fwht_equals_matrix_product(n):
    v = np.random.default_rng(n).standard_normal((5, n))
    assert np.allclose(R.fwht(v, axis=1), v @ R.sylvester(n), atol=1e-13)
    assert np.allclose(R.fwht(v.T, axis=0), (v @ R.sylvester(n)).T, atol=1e-13)


def test_rotation_round_trip_and_product_identity():
    w = synth.rvq_weight(4, 0, 0, 64, 128)
    so, si = synth.rvq_signs(4, 0, 0, 64, 128)
    wr = R.rotate_weight(w, so, si)
    assert np.max(np.abs(R.unrotate_weight(wr, so, si) - w)) < 1e-12
    # Frobenius norm is preserved by the orthogonal change of basis
    assert np.isclose(np.linalg.norm(wr), np.linalg.norm(w), rtol=1e-13)
    # the transform-aware product on the exact rotated weight equals the plain product
    x = synth.bf16_to_f64(synth.activations_bf16(4, 3, 128))
    assert np.allclose(R.linear(x, wr, so, si), x @ w.T, rtol=0, atol=1e-12)


def test_nearest_lowest_index_ties():
    cb = np.array([[1.0, 0.0], [-1.0, 0.0], [1.0, 0.0]])
    u = np.array([[0.0, 0.0], [1.0, 0.1], [0.9, 0.0]])
    assert R.nearest(u, cb).tolist() == [0, 0, 0]
    rng = np.random.default_rng(0)
    u = rng.standard_normal((300, 8))
    cb = rng.standard_normal((17, 8))
    brute = [min(range(17), key=lambda j: (float(((u[i] - cb[j]) ** 2).sum()), j)) for i in range(300)]
    assert R.nearest(u, cb).tolist() == brute


def _objective(v, cent):
    a = R.nearest(v, cent)
    return float(((v - cent[a]) ** 2).sum())


def test_kmeans_objective_non_increasing():
    v = np.random.default_rng(1).standard_normal((4000, 8))
    objs = [_objective(v, R.kmeans(v, 32, it, seed=3)) for it in range(0, 8)]
    assert all(a >= b - 1e-9 for a, b in zip(objs, objs[1:]))
    assert objs[-1] < objs[0]


def test_kmeans_empty_cluster_keeps_centroid():
    # two far clusters and four centroids initialised from the data: after one
    # step every centroid is either a member mean or its previous value
    v = np.concatenate([np.zeros((50, 2)) + [0.0, 0.0], np.zeros((50, 2)) + [10.0, 10.0]])
    v = v + np.random.default_rng(2).standard_normal(v.shape) * 1e-3
    c0 = R.kmeans(v, 4, 0, seed=1)
    c1 = R.kmeans(v, 4, 1, seed=1)
    a = R.nearest(v, c0)
    for j in range(4):
        m = v[a == j]
        assert np.allclose(c1[j], m.mean(axis=0) if len(m) else c0[j])


def test_decode_definition_float32():
    cb = np.zeros((2, 256, 8), dtype=np.float16)
    cb[0, 3] = np.float16(0.5)
    cb[1, 7] = np.float16(-0.125)
    cb[0, 9] = np.float16(1.0 / 3.0)
    cb[1, 9] = np.float16(1.0 / 7.0)
    idx = np.array([[[3, 7], [9, 9]]], dtype=np.uint8)
    s = np.array([np.float16(0.0213)]).view(np.uint16)
    w = R.decode(idx, cb.view(np.uint16), s)
    sf = np.float32(np.float16(0.0213))
    assert w.dtype == np.float32
    assert w[0, 0] == sf * (np.float32(0.5) + np.float32(-0.125))
    assert w[0, 8] == sf * (np.float32(np.float16(1 / 3)) + np.float32(np.float16(1 / 7)))


def test_rvq_codec_quality():
    rng = np.random.default_rng(5)
    w = rng.normal(0, 0.02, size=(128, 256))
    so, si = synth.rvq_signs(5, 0, 0, 128, 256)
    wr = R.rotate_weight(w, so, si)
    scale = R.row_scale_f16(wr)
    u = R.normalised_vectors(wr, scale, 8)
    cb = R.fit_codebooks(u, k=256, iters=10, seed=7)
    assert np.array_equal(cb, cb.astype(np.float16).astype(np.float64))
    idx, sc = R.encode(wr, cb)
    assert np.array_equal(sc, scale)
    dec = R.decode(idx, cb.astype(np.float16).view(np.uint16), sc).astype(np.float64)
    rel = np.linalg.norm(dec - wr) / np.linalg.norm(wr)
    # one stage alone is worse than two
    i1 = R.nearest(u, cb[0])
    one = (cb[0][i1].reshape(128, 256) * synth.f16_to_f64(sc)[:, None])
    rel1 = np.linalg.norm(one - wr) / np.linalg.norm(wr)
    assert rel < rel1 < 1.0
    assert rel < 0.45


def test_silu_closed_form():
    assert R.silu(np.array([0.0]))[0] == 0.0
    assert np.isclose(R.silu(np.array([1.0]))[0], 1.0 / (1.0 + np.exp(-1.0)))
    assert np.isclose(R.silu(np.array([-20.0]))[0], -20.0 * np.exp(-20.0) / (1 + np.exp(-20.0)))


# ------------------------------------------------------ frequency-conditioned stages
def test_stage_allocation_thirds_by_rank():
    """E = 64, s = 2: the 21 most popular experts (ranks 1..21 of the layer's Zipf order) get 3
    stages, the 21 least popular 1, the 22 others 2; the mean is exactly 2 (rate-matched)."""
    cfg = synth.OLMOE_RVQ_FREQ
    pop = synth.zipf_popularity(cfg.seed, cfg.E, cfg.zipf_s)
    st = R.stage_allocation(pop, cfg.stages)
    # the layer's rank -> expert order, rebuilt from the generator's permutation
    rng = np.random.default_rng(np.random.SeedSequence([cfg.seed, synth.TAG_ZIPF_RANK, cfg.E]))
    perm = rng.permutation(cfg.E)
    assert sorted(np.nonzero(st == 3)[0].tolist()) == sorted(perm[:21].tolist())
    assert sorted(np.nonzero(st == 1)[0].tolist()) == sorted(perm[-21:].tolist())
    assert (st == 2).sum() == 22
    assert st.sum() == 2 * cfg.E


def test_stage_allocation_follows_water_filling_order():
    """The reverse-water-filling rates r_e = r + log2(pi_e / geomean(pi)) / 2 order experts the same
    way: every 3-stage expert has a higher rate than every 2-stage one, and so on."""
    pop = np.random.default_rng(3).dirichlet(np.ones(30))
    st = R.stage_allocation(pop, 2)
    r = 2 + 0.5 * np.log2(pop / np.exp(np.mean(np.log(pop))))
    for hi, lo in ((3, 2), (2, 1)):
        assert r[st == hi].min() > r[st == lo].max()
    assert st.sum() == 60


def test_stage_allocation_ties_and_small_layers():
    assert R.stage_allocation(np.ones(6), 2).tolist() == [3, 3, 2, 2, 1, 1]
    assert R.stage_allocation(np.ones(2), 2).tolist() == [2, 2]      # floor(2/3) = 0 per third


def test_one_stage_decode_is_scale_times_first_codeword():
    rng = np.random.default_rng(5)
    cb = (rng.standard_normal((3, 256, 8)) * 0.3).astype(np.float16)
    idx = rng.integers(0, 256, size=(4, 3, 1)).astype(np.uint8)
    sc = np.array([0.5, 1.25, 0.01, 3.0], np.float16)
    w = R.decode(idx, cb.view(np.uint16), sc.view(np.uint16))
    for r in range(4):
        for v in range(3):
            exp = np.float32(sc[r]) * cb[0][idx[r, v, 0]].astype(np.float32)
            assert np.array_equal(w[r, 8 * v:8 * v + 8], exp)


def test_three_stage_decode_with_zero_third_codebook_equals_two_stage():
    rng = np.random.default_rng(6)
    cb = (rng.standard_normal((3, 256, 8)) * 0.3).astype(np.float16)
    cb[2] = 0
    idx3 = rng.integers(0, 256, size=(5, 4, 3)).astype(np.uint8)
    sc = (rng.random(5) + 0.1).astype(np.float16)
    w3 = R.decode(idx3, cb.view(np.uint16), sc.view(np.uint16))
    w2 = R.decode(idx3[:, :, :2], cb[:2].view(np.uint16), sc.view(np.uint16))
    assert np.array_equal(w3, w2)
    # explicit float32 sums, left to right
    c = cb.astype(np.float32)
    exp = np.float32(sc[1]) * ((c[0][idx3[1, 2, 0]] + c[1][idx3[1, 2, 1]]) + c[2][idx3[1, 2, 2]])
    assert np.array_equal(w3[1, 16:24], exp)


def test_encode_prefix_consistency_across_stage_counts():
    """Stage s's index depends only on stages before it: the S-stage code is a prefix of the
    (S+1)-stage code, and a 2-codebook set gives the same first two stages as a 3-codebook set."""
    cfg = synth.OLMOE_RVQ
    w = synth.rvq_weight(cfg.seed, 0, synth.GATE, 16, 64)
    so, si = synth.rvq_signs(cfg.seed, 0, synth.GATE, 16, 64)
    wr = R.rotate_weight(w, so, si)
    u = R.normalised_vectors(wr, R.row_scale_f16(wr), 8)
    cb3 = R.fit_codebooks(u, k=16, iters=5, seed=1, stages=3)
    cb2 = R.fit_codebooks(u, k=16, iters=5, seed=1, stages=2)
    assert np.array_equal(cb3[:2], cb2)
    i1, _ = R.encode(wr, cb3, stages=1)
    i2, _ = R.encode(wr, cb2)
    i3, _ = R.encode(wr, cb3)
    assert np.array_equal(i3[:, :, :2], i2) and np.array_equal(i2[:, :, :1], i1)
    # more stages never leave a larger total squared error on the fitted data
    errs = []
    for idx in (i1, i2, i3):
        d = R.decode(idx, R.f16_round(cb3).astype(np.float16).view(np.uint16), R.row_scale_f16(wr))
        errs.append(float(np.sum((d - wr) ** 2)))
    assert errs[0] > errs[1] > errs[2]


# ---------------------------------------------------------------- pins of the expert FFN and the row scale
def _h2():
    """The 2 x 2 normalised Hadamard matrix written out (independent of the oracle's builder)."""
    r = 1.0 / math.sqrt(2.0)
    return np.array([[r, r], [r, -r]])


def _rotated(w, sign_out, sign_in):
    """W' = H D_out W D_in H for 2 x 2 matrices, so that the transform-aware product gives W x."""
    h = _h2()
    return h @ np.diag(sign_out) @ np.asarray(w, np.float64) @ np.diag(sign_in) @ h


def test_swiglu_expert_hand_computed():
    # [QCA] expert FFN (SwiGLU): y = down(bf16(SiLU(gate x) * (up x))).  Plain weights
    # gate = I, up = [[0, 1], [1, 0]], down = [[1, 1], [1, -1]], x = (1, 2):
    #   g = (1, 2), u = (2, 1)
    #   SiLU(1) * 2 = 2 / (1 + e^-1) = 1.46211715726...  -> bf16 1 + 59/128 = 1.4609375
    #   SiLU(2) * 1 = 2 / (1 + e^-2) = 1.76159415595...  -> bf16 1 + 97/128 = 1.7578125
    #   y = (1.4609375 + 1.7578125, 1.4609375 - 1.7578125) = (3.21875, -0.296875)
    # Swapping gate and up gives y[1] = +0.296875; dropping the bf16 rounding of h gives
    # (3.22371131..., -0.29947699...).
    so, si = np.array([1.0, -1.0]), np.array([-1.0, -1.0])
    gate = (_rotated(np.eye(2), so, si), so, si)
    up = (_rotated([[0, 1], [1, 0]], so[::-1].copy(), si), so[::-1].copy(), si)
    down = (_rotated([[1, 1], [1, -1]], si, so), si, so)
    y = R.swiglu_expert(np.array([[1.0, 2.0]]), gate, up, down)
    assert np.allclose(y, [[3.21875, -0.296875]], rtol=0, atol=1e-12)


def test_swiglu_expert_one_dimensional():
    # one-dimensional layers (the 1 x 1 Hadamard is 1) with unit weights: SiLU(0) * u = 0, and
    # for x = 1, h = SiLU(1) * 1 = 0.73105857... rounds to the nearest bf16, 187/256 (spacing
    # 2^-8 on [0.5, 1); 187.15 units); down = 1 passes h through.
    one = (np.ones((1, 1)), np.ones(1), np.ones(1))
    assert R.swiglu_expert(np.array([[0.0]]), one, one, one)[0, 0] == 0.0
    assert R.swiglu_expert(np.array([[1.0]]), one, one, one)[0, 0] == 187.0 / 256.0
    # x = -1: h = SiLU(-1) * (-1) = 0.26894142... -> 0.26953125 (138/512, spacing 2^-9)
    assert R.swiglu_expert(np.array([[-1.0]]), one, one, one)[0, 0] == 138.0 / 512.0


@pytest.mark.parametrize("row,expected", [
    # a constant row c: RMS = |c|
    ([0.02] * 16, np.float16(0.02)),
    ([-0.375] * 8, np.float16(0.375)),
    # (a, -a, 0, 0): RMS = |a| / sqrt(2)
    ([0.5, -0.5, 0.0, 0.0], np.float16(0.5 / math.sqrt(2.0))),
    # (3, 4) / (5 * sqrt(2)) scaled: RMS of (3, 4) is 5 / sqrt(2)
    ([3.0, 4.0], np.float16(5.0 / math.sqrt(2.0))),
    # one nonzero among n = 8: RMS = |v| / sqrt(8)
    ([0.0, 0.0, 0.0, 0.1, 0.0, 0.0, 0.0, 0.0], np.float16(0.1 / math.sqrt(8.0))),
])
def test_row_scale_f16_closed_forms(row, expected):
    # [QCA] "Residual vector quantization": per-row RMS scale, stored in fp16.  A scale of
    # max|w|, or a root of the sum without the division by n, fails every row but the first.
    got = R.row_scale_f16(np.array([row]))
    assert got.dtype == np.uint16
    assert got[0] == np.array([expected], np.float16).view(np.uint16)[0]
