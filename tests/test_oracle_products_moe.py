"""Pins for the oracle's dense products, router, bucketing and MoE layer."""
from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import moe as M
from oracle import products as P


def _exact_xwt(x, w):
    T, K = x.shape
    R = w.shape[0]
    out = [[Fraction(0)] * R for _ in range(T)]
    for t in range(T):
        for r in range(R):
            acc = Fraction(0)
            for c in range(K):
                acc += Fraction(float(x[t, c])) * Fraction(float(w[r, c]))
            out[t][r] = acc
    return out


def test_products_exact_on_tiny():
    rng = np.random.default_rng(0)
    tern = rng.integers(-1, 2, size=(7, 24)).astype(np.int8)
    s = synth.f16_to_f64(synth.row_scales(0, 0, 0, 7))
    w = tern * s[:, None]
    x = synth.bf16_to_f64(synth.activations_bf16(0, 3, 24))
    y = P.matmul_xwt(x, w)
    ex = _exact_xwt(x, w)
    for t in range(3):
        for r in range(7):
            # bf16 x fp16 products and short sums are exact in float64 here
            assert Fraction(y[t, r]) == ex[t][r]
            assert Fraction(P.ternary_dot(tern[r], s[r], x[t])) == ex[t][r]


def test_special_cases():
    rng = np.random.default_rng(1)
    w = rng.integers(-1, 2, size=(5, 9)).astype(np.float64) * 0.5
    assert np.all(P.matmul_xwt(np.zeros((2, 9)), w) == 0)
    assert np.all(P.matmul_xwt(rng.standard_normal((2, 9)), np.zeros((5, 9))) == 0)
    onehot = np.zeros((1, 9)); onehot[0, 4] = 1.0
    assert np.array_equal(P.matmul_xwt(onehot, w)[0], w[:, 4])
    assert np.array_equal(P.matmul_xwt(np.eye(9), w), w.T)


def test_normwise_rel_err():
    assert P.normwise_rel_err([1.0, 2.0], [1.0, 2.0]) == 0.0
    assert P.normwise_rel_err([1.0, 2.1], [1.0, 2.0]) == pytest.approx(0.05)
    assert P.normwise_rel_err([0.0], [0.0]) == 0.0


def test_bf16_round_halfway_cases():
    h = 2.0 ** -8          # half a bf16 ulp at 1
    vals = np.array([1 + h, 1 + 3 * h, -(1 + h), 1 + h + 2.0 ** -30, 0.0, 3.0])
    assert list(M.bf16_round(vals)) == [1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7, 0.0, 3.0]


def test_bf16_round_matches_float32_bit_rounding():
    x = (np.random.default_rng(2).standard_normal(50000) * 5).astype(np.float32)
    assert np.array_equal(M.bf16_round(x.astype(np.float64)), synth.bf16_to_f64(synth.bf16_bits_from_f32(x)))


def test_route_top1_and_gates():
    lg = np.array([[0.0, 2.0, 1.0], [5.0, 5.0, -1.0]], dtype=np.float32)
    ids, gates = M.route(lg, 1)
    assert ids.tolist() == [[1], [0]]          # equal logits: lower id first
    z0 = np.exp(0.0) + np.exp(2.0) + np.exp(1.0)
    assert gates[0, 0] == pytest.approx(np.exp(2.0) / z0, rel=1e-15)
    assert gates[1, 0] == pytest.approx(0.5 / (1 + 0.5 * np.exp(-6.0)), rel=1e-15)


def test_route_topk_brute_force():
    lg = synth.zipf_logits(4, 64, 64, 0.9)
    ids, gates = M.route(lg, 8)
    for t in range(64):
        order = sorted(range(64), key=lambda e: (-float(lg[t, e]), e))[:8]
        assert ids[t].tolist() == order
        sm = np.exp(lg[t].astype(np.float64) - lg[t].max())
        sm /= sm.sum()
        assert np.allclose(gates[t], sm[order], rtol=1e-13, atol=0)
    assert np.all(gates.sum(axis=1) <= 1 + 1e-12)


def test_bucketise_stable_and_conserving():
    ids = np.array([[3, 1], [1, 0], [3, 3], [2, 1]], dtype=np.int32)
    counts, offsets, perm = M.bucketise(ids, 5)
    assert counts.tolist() == [1, 3, 1, 3, 0]
    assert offsets.tolist() == [0, 1, 4, 5, 8, 8]
    assert perm.tolist() == [3, 1, 2, 7, 6, 0, 4, 5]
    big = np.argmax(synth.zipf_logits(3, 4096, 2048, 1.0), axis=1).astype(np.int32)[:, None]
    counts, offsets, perm = M.bucketise(big, 2048)
    assert counts.sum() == 4096 and offsets[-1] == 4096
    assert sorted(perm.tolist()) == list(range(4096))
    for e in range(2048):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.all(big[seg, 0] == e)


def test_moe_layer_equals_per_token_loop():
    rng = np.random.default_rng(3)
    E, d, f, T, k = 4, 6, 10, 9, 2
    wi = rng.integers(-1, 2, size=(E, f, d)) * 0.03
    wo = rng.integers(-1, 2, size=(E, d, f)) * 0.02
    x = synth.bf16_to_f64(synth.activations_bf16(9, T, d))
    ids, gates = M.route(rng.standard_normal((T, E)).astype(np.float32), k)
    y = M.moe_layer(x, ids, gates, lambda e, xs: M.relu_expert(xs, wi[e], wo[e]), d)
    for t in range(T):
        ref = np.zeros(d)
        for j in range(k):
            e = ids[t, j]
            h = np.maximum(wi[e] @ x[t], 0.0)
            h = M.bf16_round(h)
            ref = ref + gates[t, j] * (wo[e] @ h)
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-15)
