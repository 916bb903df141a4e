"""Pins for the oracle's E8P lattice codebook ([M8.5] 0x06E): counts from combinatorics, the
lattice's definition, hand-derived code words, a textbook lattice decoder and a quantiser
bound, none of them recomputed with the oracle's own formulas."""
import itertools
import math

import numpy as np
import pytest

import synth
from oracle import e8p as P
from oracle import rvq as R


def test_base_patterns_are_the_smallest_norm_half_integer_patterns():
    pat = P.base_patterns()
    assert pat.shape == (256, 8)
    assert len({tuple(p) for p in pat}) == 256
    assert set(np.unique(pat).tolist()) <= {1, 3, 5}
    # ordered 8-tuples over {1/2, 3/2, 5/2} by squared norm, counted with binomials:
    # norm^2 = 2 + (number of 3/2) * 2 + (number of 5/2) * 6
    def count(n2):
        return sum(math.comb(8, b) * math.comb(8 - b, c) for b in range(9) for c in range(9 - b)
                   if 2 + 2 * b + 6 * c == n2)
    n2 = (pat.astype(np.int64) ** 2).sum(axis=1) // 4
    for v in (2, 4, 6, 8, 10):
        assert int(np.sum(n2 == v)) == count(v)
    assert count(2) + count(4) + count(6) + count(8) + count(10) == 227
    assert int(np.sum(n2 == 12)) == 256 - 227 and count(12) == 224
    assert np.all(np.diff(n2) >= 0)
    # every pattern below squared norm 12, including those with a 7/2 coordinate, is present
    have = {tuple(p) for p in pat}
    for t in itertools.product((1, 3, 5, 7), repeat=8):
        if sum(v * v for v in t) // 4 < 12:
            assert t in have


def test_base_table_is_one_kib_of_nibbles():
    words = P.base_table_words()
    assert words.dtype == np.uint32 and words.nbytes == 1024
    pat = P.base_patterns()
    for e in (0, 1, 100, 255):
        assert [(int(words[e]) >> (4 * i)) & 15 for i in range(8)] == pat[e].tolist()


def test_hand_derived_code_words():
    quarter = np.full(8, 0.25)
    # pattern 0 is (1/2, ..., 1/2): sum 4 is even with no negative sign
    assert np.array_equal(P.decode_codes(np.array([0]))[0], quarter)
    assert np.array_equal(P.decode_codes(np.array([0x8000]))[0], np.full(8, 0.75))
    # coordinate 0 negative makes the sum 3: the parity makes coordinate 7 negative too
    v = P.decode_codes(np.array([0x0100]))[0]
    assert np.array_equal(v, np.array([-0.75, 0.25, 0.25, 0.25, 0.25, 0.25, 0.25, -0.75]))
    # two negatives keep the sum even: coordinate 7 stays positive
    v = P.decode_codes(np.array([0x0300 | 0x8000]))[0]
    assert np.array_equal(v, np.array([-0.25, -0.25, 0.75, 0.75, 0.75, 0.75, 0.75, 0.75]))
    # pattern 1 is (1/2, ..., 1/2, 3/2): sum 5 is odd, so coordinate 7 is negative with no other
    assert P.base_patterns()[1].tolist() == [1, 1, 1, 1, 1, 1, 1, 3]
    v = P.decode_codes(np.array([1]))[0]
    assert np.array_equal(v, np.array([0.25] * 7 + [-1.75]))


def test_codebook_is_the_shifted_e8_points_of_the_table_patterns():
    cb = P.codebook()
    assert cb.shape == (65536, 8)
    assert len({tuple(r) for r in cb}) == 65536
    # enumerate D8^ (half-integer vectors with an even coordinate sum) over the table's
    # absolute patterns and all 256 sign vectors, then add +-1/4
    want = set()
    for p in P.base_patterns() / 2.0:
        for signs in itertools.product((1.0, -1.0), repeat=8):
            x = p * np.array(signs)
            if x.sum() % 2 == 0:
                for c in (0.25, -0.25):
                    want.add(tuple(x + c))
    assert want == {tuple(r) for r in cb}
    # every codeword: v - c has odd doubled coordinates and an even sum, c = +1/4 for bit 15
    codes = np.arange(65536)
    c = np.where(codes >> 15, 0.25, -0.25)
    x = cb - c[:, None]
    assert np.all(np.mod(2 * x, 2) == 1) and np.all(np.mod(x.sum(axis=1), 2) == 0)


def test_half_integer_roots_of_e8():
    """E8 has 240 roots; 128 of them are the half-integer vectors (+-1/2)^8 with an even
    number of minus signs: pattern 0 without the shift."""
    codes = np.array([c for c in range(65536) if c & 0xFF == 0 and not c >> 15])
    x = P.decode_codes(codes) + 0.25
    assert len({tuple(r) for r in x}) == 128
    assert np.all((x * x).sum(axis=1) == 2.0)
    assert np.all((x < 0).sum(axis=1) % 2 == 0)


def test_kappa_is_the_codebook_power():
    cb = P.codebook()
    assert P.kappa_squared() == pytest.approx(float((cb * cb).sum()) / cb.size, rel=1e-15)
    assert P.kappa_squared() == 2450 / 2048


def _d8_nearest(y):
    """Conway and Sloane's decoder for D8 (integer vectors with an even sum): round every
    coordinate; if the sum is odd, round the worst coordinate the other way."""
    f = np.floor(y + 0.5)
    if int(f.sum()) % 2 == 0:
        return f
    err = y - f
    k = int(np.argmax(np.abs(err)))
    f[k] += 1.0 if err[k] > 0 else -1.0
    return f


def test_encoder_agrees_with_the_lattice_decoder():
    """Within the table the brute-force nearest codeword is the nearest point of the shifted
    lattice E8 + 1/4 = (D8 + 1/2 + 1/4) u (D8 + 1/2 - 1/4)."""
    rng = np.random.default_rng(7)
    u = rng.standard_normal((600, 8)) * math.sqrt(P.kappa_squared())
    codes = P.nearest_codes(u)
    v = P.decode_codes(codes)
    have = {tuple(p) for p in P.base_patterns()}
    inside = 0
    for i in range(u.shape[0]):
        best = None
        for c in (0.25, -0.25):
            pt = _d8_nearest(u[i] - 0.5 - c) + 0.5 + c
            d = float(((u[i] - pt) ** 2).sum())
            if best is None or d < best[0]:
                best = (d, pt, c)
        d_code = float(((u[i] - v[i]) ** 2).sum())
        assert d_code >= best[0] - 1e-12            # nothing in the codebook beats the lattice
        x = best[1] - best[2]
        if tuple(np.rint(2 * np.abs(x)).astype(int)) in have:
            inside += 1
            assert np.array_equal(v[i], best[1])
    assert inside > 300                              # most of them (58 % for this seed)


def test_encoder_is_brute_force_argmin_with_small_code_ties():
    cb = P.codebook()
    rng = np.random.default_rng(3)
    u = rng.standard_normal((4, 8))
    u = np.vstack([u, np.zeros((1, 8))])            # the origin is equally far from +-1/4
    got = P.nearest_codes(u)
    for i in range(u.shape[0]):
        d = [sum((u[i, j] - cb[c, j]) ** 2 for j in range(8)) for c in range(65536)]
        m = min(d)
        assert int(got[i]) == d.index(m)
    assert int(got[-1]) == 0


def test_encoder_round_trips_codewords():
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 65536, 300)
    assert np.array_equal(P.nearest_codes(P.decode_codes(codes)), codes.astype(np.uint16))


def test_e8p_beats_the_scalar_two_bit_quantiser():
    """At 2 bits per weight the lattice codebook's mean squared error on i.i.d. Gaussian
    vectors is below that of the optimal 4-level scalar (Lloyd-Max) quantiser, 0.1175 sigma^2."""
    rng = np.random.default_rng(5)
    k = math.sqrt(P.kappa_squared())
    u = rng.standard_normal((3000, 8)) * k
    v = P.decode_codes(P.nearest_codes(u))
    mse = float(((u - v) ** 2).mean()) / P.kappa_squared()
    assert mse < 0.1175


def test_scale_and_encode_of_a_rotated_weight():
    rows, cols = 16, 64
    w = synth.rvq_weight(4, 0, 1, rows, cols)
    so, si = synth.rvq_signs(4, 0, 1, rows, cols)
    wr = R.rotate_weight(w, so, si)
    codes, scale = P.encode(wr)
    assert codes.shape == (rows, cols // 8) and codes.dtype == np.uint16
    s = scale.view(np.float16).astype(np.float64)
    u = wr / s[:, None]
    # u has the codebook's power per coordinate, up to the fp16 rounding of the scale
    rms = np.sqrt((u * u).mean(axis=1))
    assert np.all(np.abs(rms / math.sqrt(P.kappa_squared()) - 1) < 2.0 ** -10)
    wd = P.decode(codes, scale)
    assert wd.dtype == np.float32
    # decode is fp32(s) * v exactly; the rotated-basis error is the quantiser's
    assert np.array_equal(wd, (s[:, None].astype(np.float32) * P.decode_codes(codes).reshape(rows, cols)
                               .astype(np.float32)))
    rel = np.linalg.norm(wd - wr) / np.linalg.norm(wr)
    assert 0.2 < rel < 0.35


def test_codewords_keep_the_e8_minimal_distance():
    """E8 has minimal squared norm 2, so distinct points of E8 + 1/4 are at squared distance >= 2,
    with equality for neighbours; a wrong parity rule or shift would bring codewords closer."""
    cb = P.codebook()
    rng = np.random.default_rng(13)
    pick = rng.choice(65536, 300, replace=False)
    best = np.inf
    for c in pick:
        d = ((cb - cb[c]) ** 2).sum(axis=1)
        d[c] = np.inf
        best = min(best, float(d.min()))
        assert d.min() >= 2.0
    assert best == 2.0
