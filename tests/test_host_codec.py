"""The C-ABI library without a GPU: exported symbols and the host codec against the oracle."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import synth
from oracle import codec as C
from oracle import dictionary as D
from oracle import rvq as R

Q = pytest.importorskip("decode_matvec_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "qmoe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported():
    names = _declared_functions()
    assert len(names) >= 17
    out = subprocess.run(["nm", "-D", "--defined-only", Q.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    for n in names:
        assert n in exported, n
        assert getattr(Q.lib(), n) is not None
    assert sorted(Q.EXPORTED) == names


@pytest.mark.parametrize("p0", [0.857, 0.87, 0.886, 0.89, 0.5])
def test_dictionary_matches_oracle(p0):
    words, used = Q.qmoe_encode_dictionary(p0)
    assert used == p0
    assert np.array_equal(words, D.build(p0))


def test_dictionary_from_measured_symbols():
    tern = synth.ternary_matrix(0, 0, 0, 64, 512, 0.89)
    words, used = Q.qmoe_encode_dictionary(symbols=tern)
    assert used == D.measured_p0(tern)
    assert np.array_equal(words, D.build(used))


def test_dictionary_rejects_bad_p0():
    for bad in (0.0, 1.0, -0.5, 2.0):
        with pytest.raises(Q.QmoeError):
            Q.qmoe_encode_dictionary(bad)
    with pytest.raises(Q.QmoeError):
        Q.qmoe_encode_dictionary(symbols=np.zeros(10, np.int8))      # measured p0 = 1


@pytest.fixture(scope="module")
def words886():
    return D.build(0.886)


@pytest.mark.parametrize("rows,cols,block,p0", [(7, 2080, 256, 0.886), (5, 300, 256, 0.857), (3, 2, 256, 0.886),
                                               (4, 1030, 64, 0.87), (2, 512, 256, 0.0), (2, 512, 256, 1.0)])
def test_pack_matches_oracle(words886, rows, cols, block, p0):
    if p0 in (0.0, 1.0):
        tern = np.zeros((rows, cols), np.int8) if p0 == 1.0 else \
            np.where(np.arange(rows * cols).reshape(rows, cols) % 5 < 2, 1, -1).astype(np.int8)
    else:
        tern = synth.ternary_matrix(17, 2, 1, rows, cols, p0)
    codes, off = Q.qmoe_pack(tern, words886, block)
    rc, ro = C.encode(tern, words886, block)
    assert np.array_equal(codes, rc) and np.array_equal(off, ro)


def test_pack_rejects_bad_input(words886):
    with pytest.raises(Q.QmoeError):
        Q.qmoe_pack(np.zeros((2, 7), np.int8), words886)
    with pytest.raises(Q.QmoeError):
        Q.qmoe_pack(np.full((1, 4), 2, np.int8), words886)
    broken = words886.copy()
    broken[0] = 0                    # pair count 0 in one half
    with pytest.raises(Q.QmoeError):
        Q.qmoe_pack(np.zeros((1, 4), np.int8), broken)


def test_pack_capacity_error(words886):
    tern = synth.ternary_matrix(1, 0, 0, 2, 256, 0.886)
    codes = np.zeros(3, np.uint16)
    off = np.zeros(3, np.uint32)
    with pytest.raises(Q.QmoeError) as ei:
        Q.qmoe_pack_into(tern, words886, 256, codes, off)
    assert ei.value.status == Q.QMOE_ECAPACITY


@pytest.mark.parametrize("p0", [0.886, 0.857, 0.75])
def test_compact_table_lists_every_nonzero(p0):
    # up to three nonzeros: three 6-bit slots; four nonzeros within the first eight positions: four
    # 4-bit slots (flag 0x40); anything else (p0 0.75 has five-nonzero entries): the canonical words
    ents = D.generate(p0)
    words = D.pack(ents)
    comp = Q.qmoe_dict_compact(words)
    plane_a = comp[:2 * 65536].view(np.uint16)
    plane_b = comp[2 * 65536:3 * 65536]
    # the third plane repeats both entries as one uint32
    plane_w = comp[3 * 65536:7 * 65536].view(np.uint32)
    assert np.array_equal(plane_w, plane_a.astype(np.uint32) | (plane_b.astype(np.uint32) << 16))
    kinds = set()
    for e, seq in enumerate(ents):
        a, b = int(plane_a[e]), int(plane_b[e])
        assert (a & 15) == len(seq) // 2
        nz = [2 * i + (1 if s == 1 else 0) for i, s in enumerate(seq) if s]
        if len(nz) <= 3:
            slots = [(a >> 4) & 63, (a >> 10) & 63, b & 63]
            assert slots == nz + [63] * (3 - len(nz))
            assert b & 0xC0 == 0
            kinds.add(3)
        elif len(nz) == 4 and nz[3] < 16:
            assert [(a >> 4) & 15, (a >> 8) & 15, (a >> 12) & 15, b & 15] == nz
            assert b & 0xF0 == 0x40
            kinds.add(4)
        else:
            assert a >> 4 == 0xFFF and b == 0xBF
            kinds.add(5)
    assert kinds == {0.886: {3}, 0.857: {3, 4}, 0.75: {3, 4, 5}}[p0]


def test_rvq_pack_matches_oracle():
    rows, cols = 64, 256
    w = synth.rvq_weight(4, 1, 2, rows, cols)
    so, si = synth.rvq_signs(4, 1, 2, rows, cols)
    wr = R.rotate_weight(w, so, si)
    u = R.normalised_vectors(wr, R.row_scale_f16(wr), 8)
    cb = R.fit_codebooks(u, k=256, iters=4, seed=3)
    cb_bits = cb.astype(np.float16).view(np.uint16)
    idx, sc = Q.rvq_pack(w, so, si, cb_bits)
    ridx, rsc = R.encode(wr, cb)
    assert np.array_equal(sc, rsc)
    assert np.array_equal(idx, ridx)


def test_native_ternary_generator_matches_python():
    lib = ctypes.CDLL(os.path.join(ROOT, "synth", "libsynth.so"))
    lib.synth_ternary_rows.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64,
                                       ctypes.c_uint32, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    for (seed, e, m, cols, p0, r0, n) in [(3, 17, 1, 2080, 0.886, 5, 7), (1, 0, 0, 3072, 0.857, 0, 3)]:
        out = np.zeros((n, cols), np.int8)
        lib.synth_ternary_rows(seed, e, m, cols, synth.zero_threshold(p0), r0, n, out.ctypes.data)
        assert np.array_equal(out, synth.ternary_rows(seed, e, m, cols, p0, r0, n))


@pytest.mark.parametrize("stages", [1, 2, 3])
def test_rvq_pack_stages_matches_oracle(stages):
    rows, cols = 32, 128
    w = synth.rvq_weight(4, 2, 0, rows, cols)
    so, si = synth.rvq_signs(4, 2, 0, rows, cols)
    wr = R.rotate_weight(w, so, si)
    u = R.normalised_vectors(wr, R.row_scale_f16(wr), 8)
    cb = R.fit_codebooks(u, k=256, iters=3, seed=5, stages=3)
    idx, sc = Q.rvq_pack(w, so, si, cb.astype(np.float16).view(np.uint16), stages)
    ridx, rsc = R.encode(wr, cb, stages=stages)
    assert idx.shape == (rows, cols // 8, stages)
    assert np.array_equal(sc, rsc) and np.array_equal(idx, ridx)


def test_rvq_stage_allocation_matches_oracle():
    for E, seed in ((64, 4), (7, 1), (2, 3), (30, 9)):
        pop = synth.zipf_popularity(seed, E, 0.9)
        assert np.array_equal(Q.rvq_stage_allocation(pop, 2), R.stage_allocation(pop, 2))
    ties = np.array([1.0, 2.0, 2.0, 1.0, 2.0, 0.5])
    assert np.array_equal(Q.rvq_stage_allocation(ties, 2), R.stage_allocation(ties, 2))
    with pytest.raises(Q.QmoeError):
        Q.rvq_stage_allocation(np.ones(6), 3)          # s_bar + 1 = 4 stages is beyond the maximum


def test_three_stage_codebook_fixture_extends_the_two_stage_one():
    """The committed codebook sets: the first two stages of the three-stage set are the two-stage set."""
    golden = os.path.join(ROOT, "tests", "golden")
    cb2 = np.load(os.path.join(golden, "olmoe_rvq_codebooks.npy"))
    cb3 = np.load(os.path.join(golden, "olmoe_rvq_codebooks3.npy"))
    assert cb2.shape == (2, 256, 8) and cb3.shape == (3, 256, 8)
    assert np.array_equal(cb3[:2].view(np.uint16), cb2.view(np.uint16))


def test_e8p_base_table_matches_oracle():
    from oracle import e8p as P8
    assert np.array_equal(Q.e8p_base_table(), P8.base_table_words())


@pytest.mark.parametrize("rows,cols,seed", [(16, 64, 0), (8, 256, 1), (32, 32, 2)])
def test_e8p_pack_matches_oracle(rows, cols, seed):
    from oracle import e8p as P8
    w = synth.rvq_weight(4, seed, 2, rows, cols)
    so, si = synth.rvq_signs(4, seed, 2, rows, cols)
    codes, sc = Q.e8p_pack(w, so, si)
    rcodes, rsc = P8.encode(R.rotate_weight(w, so, si))
    assert np.array_equal(sc, rsc)
    assert np.array_equal(codes, rcodes)


def test_e8p_nearest_matches_brute_force_on_boundaries_and_far_points():
    """The host search (lattice decoder first, all patterns when that is ambiguous or outside
    the table) against the oracle's brute force: Voronoi-boundary inputs, where ties go to the
    smaller code word, points far outside the codebook, and exact codewords."""
    from oracle import e8p as P8
    rng = np.random.default_rng(4)
    special = np.array([[0.0] * 8, [1.0] * 8, [0.25] * 8, [-0.25] * 8, [0.5] * 8, [-0.75] * 8,
                        [-0.25, 0.25, 1.0, -1.0, 2.0, 0.5, -0.5, 0.0], [3.0, -3.0, 0.0, 0.0, 1.0, 1.0, -1.0, 2.0],
                        [0.75, 0.75, 0.75, 0.75, 0.25, 0.25, 0.25, 0.25], [9.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, -9.0]])
    far = rng.standard_normal((200, 8)) * 3.0
    near = rng.standard_normal((600, 8)) * np.sqrt(P8.kappa_squared())
    grid = rng.integers(-8, 9, (200, 8)) / 4.0                      # quarter-integers: many exact ties
    cw = P8.decode_codes(rng.integers(0, 65536, 100))
    u = np.vstack([special, far, near, grid, cw])
    assert np.array_equal(Q.e8p_nearest(u), P8.nearest_codes(u))
    with pytest.raises(Q.QmoeError):
        Q.e8p_nearest(np.full((1, 8), np.nan))


def test_e8p_pack_codewords_round_trip():
    """A weight whose rotated rows are scaled codewords encodes to those code words."""
    from oracle import e8p as P8
    rng = np.random.default_rng(5)
    rows, cols = 8, 64
    codes = rng.integers(0, 65536, (rows, cols // 8)).astype(np.uint16)
    wr = P8.decode_codes(codes).reshape(rows, cols)
    so, si = synth.rvq_signs(4, 9, 0, rows, cols)
    w = R.unrotate_weight(wr, so, si)
    got, sc = Q.e8p_pack(w, so, si)
    want, wsc = P8.encode(R.rotate_weight(w, so, si))
    assert np.array_equal(sc, wsc) and np.array_equal(got, want)


def test_e8p_pack_rejects_bad_inputs():
    w = synth.rvq_weight(4, 0, 0, 16, 64)
    so, si = synth.rvq_signs(4, 0, 0, 16, 64)
    with pytest.raises(Q.QmoeError):
        Q.e8p_pack(w[:, :48], so, si[:48])                  # 48 columns: not a power of two
    with pytest.raises(Q.QmoeError):
        Q.e8p_pack(w[:12], so[:12], si)                     # 12 rows: not a power of two
    bad = si.copy()
    bad[3] = 0
    with pytest.raises(Q.QmoeError):
        Q.e8p_pack(w, so, bad)                              # a sign that is not +-1
    with pytest.raises(Q.QmoeError):
        Q.e8p_pack(np.zeros((16, 64)), so, si)             # a zero row has no scale
    assert Q.e8p_nearest(np.zeros((0, 8))).shape == (0,)


def test_offsets_compact_round_trip(words886):
    # the device layout's row starts and per-block codeword counts re-encode qmoe_pack's offsets exactly
    tern = synth.ternary_matrix(4, 0, 0, 37, 1030, 0.886)
    codes, off = Q.qmoe_pack(tern, words886)
    nb = (1030 + 255) // 256
    row_off, blk_len = Q.qmoe_offsets_compact(off, 37, nb)
    assert row_off.dtype == np.uint32 and blk_len.dtype == np.uint8
    assert row_off.size == 38 and blk_len.size == 37 * (nb - 1)
    rebuilt = np.zeros_like(off)
    for r in range(37):
        starts = row_off[r] + np.concatenate([[0], np.cumsum(blk_len[r * (nb - 1):(r + 1) * (nb - 1)])])
        rebuilt[r * nb:(r + 1) * nb] = starts
    rebuilt[-1] = row_off[-1]
    assert np.array_equal(rebuilt, off)
    # two matrices back to back
    ro2, bl2 = Q.qmoe_offsets_compact(np.concatenate([off, off]), 37, nb, count=2)
    assert np.array_equal(ro2[:38], row_off) and np.array_equal(ro2[38:], row_off)
    assert np.array_equal(bl2[:blk_len.size], blk_len)


def test_offsets_compact_rejects_bad_offsets():
    with pytest.raises(Q.QmoeError):
        Q.qmoe_offsets_compact(np.array([0, 5, 3, 8], np.uint32), 1, 3)          # decreasing
    with pytest.raises(Q.QmoeError):
        Q.qmoe_offsets_compact(np.array([0, 300, 310], np.uint32), 1, 2)         # a block of 300 codewords
    with pytest.raises(Q.QmoeError):
        Q.qmoe_offsets_compact(np.array([1, 5, 9], np.uint32), 1, 2)             # not starting at 0
