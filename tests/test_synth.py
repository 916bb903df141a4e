"""The seeded generators: published SplitMix64 outputs and the ternary draw rule."""
import numpy as np

import synth


def test_splitmix64_published_sequence():
    # First outputs of SplitMix64 seeded with 0 (Steele, Lea, Flood 2014; the
    # public reference implementation's sequence).
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [synth.splitmix64_scalar(0, i) for i in range(3)] == expect
    assert [int(v) for v in synth.splitmix64(0, np.arange(3))] == expect


def test_ternary_rows_are_independent_of_the_window():
    full = synth.ternary_matrix(7, 3, 1, 40, 300, 0.886)
    part = synth.ternary_rows(7, 3, 1, 300, 0.886, 17, 5)
    assert np.array_equal(full[17:22], part)


def test_ternary_frequencies():
    t = synth.ternary_matrix(3, 0, 0, 256, 4096, 0.886)
    n = t.size
    p0 = (t == 0).mean()
    # binomial standard error at n = 1M is ~3e-4
    assert abs(p0 - 0.886) < 2e-3
    assert abs((t == 1).mean() - (t == -1).mean()) < 2e-3
    assert set(np.unique(t)) <= {-1, 0, 1} and n == 256 * 4096


def test_bf16_bits_round_to_nearest_even():
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -8)      # half a bf16 ulp at 1.0
    vals = np.array([one + ulp, one + 3 * ulp, -(one + ulp)], dtype=np.float32)
    got = synth.bf16_to_f64(synth.bf16_bits_from_f32(vals))
    assert list(got) == [1.0, 1.0 + 2.0 ** -6, -1.0]


def test_scales_in_range_and_fp16():
    s = synth.f16_to_f64(synth.row_scales(1, 2, 0, 5000))
    assert s.min() >= 0.00999 and s.max() <= 0.05001
    assert np.array_equal(s, s.astype(np.float16).astype(np.float64))


def test_zipf_logits_skew():
    lg = synth.zipf_logits(2, 2048, 128, 1.1)
    top = np.argmax(lg, axis=1)
    counts = np.bincount(top, minlength=128)
    # Gumbel-top-1 picks rank r with probability ~ r**-s: the hottest expert
    # takes ~1/H_{128,1.1} of the tokens (about 23%), and many experts see
    # only a handful of tokens.
    assert 0.15 < counts.max() / 2048 < 0.32
    assert (counts <= 4).sum() >= 10
