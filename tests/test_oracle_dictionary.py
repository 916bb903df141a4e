"""Pins for the oracle's Algorithm 1 and the Figure 4 entry layout (QMoE page)."""
import itertools
import math

import numpy as np
import pytest

from oracle import dictionary as D


@pytest.fixture(scope="module")
def dict886():
    return D.generate(0.886)


def _class_enumeration(p0, n):
    """The n most probable pair sequences of 2..28 ternary values, independently of any heap.

    Under the independence model a sequence's probability depends only on its
    length L and its count of nonzeros z, so sequences fall into classes (L, z).
    Classes are visited in order of decreasing probability; inside a class the
    members are listed in lexicographic order and appended until n are taken.
    """
    lp0, lq = math.log(p0), math.log((1 - p0) / 2)
    classes = []
    for L in range(2, 29, 2):
        for z in range(0, L + 1):
            classes.append(((L - z) * lp0 + z * lq, L, z))
    classes.sort(key=lambda c: -c[0])
    out = []
    for _, L, z in classes:
        if len(out) >= n:
            break
        members = []
        for pos in itertools.combinations(range(L), z):
            for vals in itertools.product((1, 2), repeat=z):
                seq = [0] * L
                for p, v in zip(pos, vals):
                    seq[p] = v
                members.append(tuple(seq))
        members.sort()
        out.extend(members[: n - len(out)])
    return out


def test_size_and_lengths(dict886):
    assert len(dict886) == 65536
    assert len(set(dict886)) == 65536
    lengths = {len(s) for s in dict886}
    assert lengths <= set(range(2, 29, 2))
    assert 28 in lengths and 2 in lengths


def test_all_nine_pairs_present(dict886):
    for pair in D.PAIRS:
        assert pair in set(dict886)


def test_prefix_closed_at_pair_granularity(dict886):
    s = set(dict886)
    for seq in dict886:
        for cut in range(2, len(seq), 2):
            assert seq[:cut] in s


def test_probability_non_increasing(dict886):
    lp0, lq = D.log_probs(0.886)
    pr = [D.priority(s, lp0, lq) for s in dict886]
    assert all(a >= b for a, b in zip(pr, pr[1:]))


def test_equals_most_probable_sequences(dict886):
    # Algorithm 1 is a best-first enumeration: it must return exactly the 2**16
    # most probable sequences, most probable first, equal ones in lexicographic order.
    assert dict886 == _class_enumeration(0.886, 65536)


@pytest.mark.parametrize("p0", [0.857, 0.87])
def test_equals_most_probable_sequences_other_p0(p0):
    assert D.generate(p0, 4000) == _class_enumeration(p0, 4000)


def test_no_cross_class_near_ties(dict886):
    # Distinct (length, nonzero-count) classes adjacent in the order must not be
    # within rounding distance of each other, so the order cannot depend on the
    # last bit of a logarithm.
    lp0, lq = D.log_probs(0.886)
    pr = np.array([D.priority(s, lp0, lq) for s in dict886])
    key = [(len(s), len(s) - s.count(0)) for s in dict886]
    for i in range(1, len(dict886)):
        if key[i] != key[i - 1]:
            assert pr[i - 1] - pr[i] > 1e-9


def test_most_probable_entry_is_zero_pair(dict886):
    # the single most probable sequence is one pair of zeros, P = p0**2
    assert dict886[0] == (0, 0)


def test_entry_layout_matches_listing_extraction(dict886):
    # QMoE Listing 1 as described on the page: lanes 0-27 read word 2*enc + lane/14,
    # take (w >> (4 + 2*(lane % 14))) & 3, and advance by 2*(w & 0xf) weights.
    words = D.pack(dict886[:2000] + [dict886[-1]])
    for e in range(len(words) // 2):
        seq = (dict886[:2000] + [dict886[-1]])[e]
        w = words[2 * e: 2 * e + 2]
        assert 2 * (int(w[0]) & 0xF) == len(seq)
        assert 2 * (int(w[1]) & 0xF) == len(seq)
        lanes = [(int(w[lane // 14]) >> (4 + 2 * (lane % 14))) & 3 for lane in range(28)]
        assert tuple(lanes[:len(seq)]) == seq
        assert all(v == 0 for v in lanes[len(seq):])       # padding decodes to the zero weight


def test_pack_handmade_entry():
    # (w_min, w_max, 0, 0): pair count 2, symbols 1 and 2 in the first two fields
    w0, w1 = D.pack_entry((1, 2, 0, 0))
    assert w0 == 2 | (1 << 4) | (2 << 6)
    assert w1 == 2
    # 16 symbols: the 15th and 16th land in word 1 fields 0 and 1
    seq = (0,) * 14 + (2, 1)
    w0, w1 = D.pack_entry(seq)
    assert w0 == 8 and w1 == 8 | (2 << 4) | (1 << 6)
    assert D.unpack_entry(np.array([w0, w1], dtype=np.uint32), 0) == seq


def test_nonzero_counts_per_entry(dict886):
    # At p0 = 0.886 every entry has at most 3 nonzero weights; the longest entries
    # (28 values) are exactly those with at most 2 nonzeros: 1 + 2*28 + 4*C(28,2).
    nnz = [len(s) - s.count(0) for s in dict886]
    assert max(nnz) == 3
    assert sum(1 for s in dict886 if len(s) == 28) == 1 + 2 * 28 + 4 * math.comb(28, 2)


def test_measured_p0():
    t = np.array([[0, 1, -1, 0], [0, 0, 0, 1]], dtype=np.int8)
    assert D.measured_p0(t) == 5 / 8
