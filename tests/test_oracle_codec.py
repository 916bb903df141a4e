"""Pins for the oracle's encoder, reference decoder and rate ledger."""
import math

import numpy as np
import pytest

import synth
from oracle import codec as C
from oracle import dictionary as D


@pytest.fixture(scope="module")
def words886():
    return D.build(0.886)


@pytest.fixture(scope="module")
def table886(words886):
    return C.entry_table(words886)


def _scales(rows, seed=5):
    return synth.row_scales(seed, 0, 0, rows)


@pytest.mark.parametrize("rows,cols,p0", [(3, 256, 0.886), (5, 2, 0.886), (4, 300, 0.5), (2, 1030, 0.886),
                                         (3, 512, 0.0), (3, 512, 1.0)])
def test_round_trip(words886, table886, rows, cols, p0):
    if p0 in (0.0, 1.0):
        tern = np.zeros((rows, cols), np.int8) if p0 == 1.0 else \
            np.where(np.arange(rows * cols).reshape(rows, cols) % 3 == 0, 1, -1).astype(np.int8)
    else:
        tern = synth.ternary_matrix(11, 0, 0, rows, cols, p0)
    codes, off = C.encode(tern, words886, table=table886)
    assert off[0] == 0 and off[-1] == len(codes) and np.all(np.diff(off.astype(np.int64)) >= 0)
    sym = C.decode_symbols(codes, off, words886, rows, cols)
    assert np.array_equal(C.ternary_of_symbols(sym), tern)
    s = _scales(rows)
    w = C.decode(codes, off, words886, s, rows, cols)
    sv = synth.f16_to_f64(s)
    assert np.array_equal(w, tern.astype(np.float64) * sv[:, None])


def test_round_trip_other_block(words886, table886):
    tern = synth.ternary_matrix(12, 0, 0, 3, 100, 0.886)
    codes, off = C.encode(tern, words886, block=32, table=table886)
    assert len(off) == 3 * 4 + 1
    assert np.array_equal(C.ternary_of_symbols(C.decode_symbols(codes, off, words886, 3, 100, 32)), tern)


def test_greedy_takes_longest_match(words886, table886):
    tern = synth.ternary_matrix(13, 0, 0, 2, 512, 0.886)
    codes, off = C.encode(tern, words886, table=table886)
    length, sym = C.expansion(words886)
    entries = set(table886)
    symrow = np.where(tern == 0, 0, np.where(tern < 0, 1, 2))
    nb = C.n_blocks(512)
    for r in range(2):
        for b in range(nb):
            pos = b * 256
            for c in codes[off[r * nb + b]:off[r * nb + b + 1]]:
                L = length[c]
                assert tuple(symrow[r, pos:pos + L]) == tuple(sym[c, :L])
                # no longer entry matches here inside the block
                for L2 in range(L + 2, min(28, 256 * (b + 1) - pos) + 1, 2):
                    assert tuple(symrow[r, pos:pos + L2]) not in entries
                pos += L


def test_all_zero_block_uses_longest_zero_run(words886, table886):
    tern = np.zeros((1, 56), np.int8)
    codes, off = C.encode(tern, words886, table=table886)
    assert len(codes) == 2
    assert D.unpack_entry(words886, int(codes[0])) == (0,) * 28


def test_odd_lengths_rejected(words886):
    with pytest.raises(ValueError):
        C.encode(np.zeros((1, 7), np.int8), words886)


def test_decoder_rejects_overrun(words886, table886):
    tern = np.zeros((1, 256), np.int8)
    codes, off = C.encode(tern, words886, table=table886)
    bad = off.copy()
    bad[-1] = len(codes) - 1
    with pytest.raises(ValueError):
        C.decode_symbols(codes[:-1], bad, words886, 1, 256)


def test_decoder_reads_handmade_words():
    # two handmade entries: e0 = (w_min, w_max), e1 = (0, 0, 0, w_max)
    words = np.array([D.pack_entry((1, 2))[0], D.pack_entry((1, 2))[1],
                      D.pack_entry((0, 0, 0, 2))[0], D.pack_entry((0, 0, 0, 2))[1]], dtype=np.uint32)
    codes = np.array([1, 0], dtype=np.uint16)
    off = np.array([0, 2], dtype=np.uint32)
    s = np.array([np.float16(0.25)]).view(np.uint16)
    w = C.decode(codes, off, words, s, 1, 6, block=256)
    assert list(w[0]) == [0.0, 0.0, 0.0, 0.25, -0.25, 0.25]


# ---------------------------------------------------------------------- rates
def test_entropy_printed_values():
    # QMoE page: about 0.63 bits per weight at p0 = 0.885, a limit of 25.40x vs bf16.
    h = C.entropy_bits(0.885)
    assert abs(h - 0.63) < 0.005
    assert abs(16.0 / h - 25.40) < 0.01


@pytest.mark.slow
def test_synthetic_rate_near_printed(words886):
    # QMoE page: 21.11x on synthetic i.i.d. ternary weights at p0 = 0.885.
    words = D.build(0.885)
    tern = synth.ternary_matrix(21, 0, 0, 96, 4096, 0.885)
    codes, off = C.encode(tern, words)
    led = C.ledger(len(codes), 96, 4096, 0, 0, p0_hat=D.measured_p0(tern))
    assert abs(led["payload_compression_vs_bf16"] / 21.11 - 1.0) < 0.05
    # a code cannot beat the entropy of its source
    assert led["payload_bits_per_weight"] > led["entropy_bits_per_weight"]
    # sub-1-bit payload exactly when the mean expansion exceeds 16 weights per codeword
    assert (led["payload_bits_per_weight"] < 1.0) == (led["mean_run"] > 16.0)


@pytest.mark.slow
def test_rate_improves_with_sparsity():
    # Table 7 trend: compression grows as the zero fraction grows.
    rates = []
    for p0 in (0.857, 0.87, 0.886):
        words = D.build(p0)
        tern = synth.ternary_matrix(22, 0, 0, 32, 4096, p0)
        codes, _ = C.encode(tern, words)
        rates.append(16.0 * len(codes) / tern.size)
    assert rates[0] > rates[1] > rates[2]


def test_ledger_counts_everything():
    led = C.ledger(n_codes=1000, rows=10, cols=2000, offset_bytes=4 * 81, scale_bytes=20, p0_hat=0.9)
    assert led["payload_bits_per_weight"] == 16000 / 20000
    assert math.isclose(led["effective_bits_per_weight"], 8 * (2000 + 324 + 20) / 20000)
    assert math.isclose(led["effective_with_dictionary"], led["effective_bits_per_weight"] + 8 * 524288 / 20000)
    assert math.isclose(led["bitmask_bits_per_weight"], 1.1)


def test_ledger_of_a_hand_counted_artifact(words886):
    # [M8.5] 0x01A / 0x08A: the effective rate counts every stored byte.  A 2 x 512 all-zero matrix in
    # 256-weight blocks: each block is nine 28-zero runs and one 4-zero run (greedy longest match
    # over the 14 all-zero entries), so 2 rows x 2 blocks x 10 = 40 codewords = 80 bytes; block
    # offsets 2 x 2 + 1 = 5 uint32 = 20 bytes; row scales 2 fp16 = 4 bytes; 1024 weights.
    tern = np.zeros((2, 512), np.int8)
    words86 = words886
    codes, off = C.encode(tern, words86)
    scales = np.array([0x2000, 0x2400], np.uint16)
    assert len(codes) == 40 and codes.nbytes == 80 and off.nbytes == 20 and scales.nbytes == 4
    led = C.ledger(len(codes), 2, 512, off.nbytes, scales.nbytes)
    assert led["payload_bits_per_weight"] == 16 * 40 / 1024                  # 0.625
    assert led["effective_bits_per_weight"] == 8 * (80 + 20 + 4) / 1024      # 0.8125
    # the shared dictionary: 2^16 entries x two uint32 words = 524,288 bytes
    assert words86.nbytes == 524288
    assert led["effective_with_dictionary"] == 8 * (80 + 20 + 4 + 524288) / 1024
    assert led["compression_vs_bf16"] == 16 / 0.8125
    assert led["mean_run"] == 1024 / 40


def test_ledger_one_nonzero_per_block(words886):
    # one +1 at the start of each block: a 28-run with one nonzero, then eight 28-zero runs and a
    # 4-zero run, again 10 codewords per block; one row of 768 weights = 3 blocks = 30 codewords.
    tern = np.zeros((1, 768), np.int8)
    tern[0, [0, 256, 512]] = 1
    codes, off = C.encode(tern, words886)
    assert len(codes) == 30 and off.nbytes == 16
    led = C.ledger(len(codes), 1, 768, off.nbytes, 2)
    assert led["effective_bits_per_weight"] == 8 * (60 + 16 + 2) / 768
