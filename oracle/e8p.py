"""E8P structured lattice codebook (2 bits per weight).  Test infrastructure.

[M8.5] 0x06E "Why The E8P Codebook Is Structured": an 8-dimensional vector is
coded by one 16-bit word built from the E8 lattice: 8 bits choose one of 256
stored absolute-value patterns (a 256 x 8 base table of 1 KiB), 7 bits are
explicit signs, 1 bit picks the lattice shift, and the last sign follows from
parity.  [M8.5] 0x05H lists this "fused decode-multiply" form among the runtime
choices, and 0x06C / 0x06H give the transform around it, the same randomized
Hadamard transform as the residual-VQ format (``oracle.rvq``).

Readings (the page fixes the decoder's shape, not the table's contents):

* The lattice.  E8 = D8 u (D8 + 1/2), and D8 + 1/2 = D8^ is the set of
  half-integer vectors whose coordinates sum to an even integer.  Shifting by
  1/4: E8 + 1/4 = (D8^ + 1/4) u (D8^ - 1/4), because D8^ + 1 = D8^.  So a
  codeword is a point of D8^ plus a shift of +1/4 or -1/4 on every coordinate,
  and the point of D8^ is an absolute pattern with signs.  Flipping the sign of
  one half-integer coordinate changes the sum by an odd integer, so for any
  pattern and any 7 signs exactly one sign of the last coordinate puts the
  point in D8^: "the last sign is recovered from parity".
* The base table.  The 256 absolute patterns a in {1/2, 3/2, 5/2, ...}^8 of
  smallest squared norm, equal norms in lexicographic order of the tuple
  (2 a_0, ..., 2 a_7).  All 227 patterns with squared norm <= 10 are in it and
  29 of the 224 with squared norm 12; no coordinate exceeds 5/2.  Stored as
  8 nibbles 2 a_i (1, 3 or 5) per entry: 256 x 32 bits = 1 KiB.
* The code word: bits 0-7 the pattern index, bit 8 + i (i = 0 .. 6) set when
  coordinate i is negative, bit 15 the shift (0: -1/4, 1: +1/4).
* The scale.  Rows of the rotated weight W' carry one fp16 scale
  s_r = fp16(RMS(W'_r) / kappa), kappa^2 = the mean power per coordinate of the
  65 536 codewords (2450 / 2048), so that u = W'_r / s_r has the codebook's
  power; the RMS is summed left to right as in ``oracle.rvq.row_scale_f16``.
* Encoding: the codeword nearest to u in Euclidean distance, the squared
  distance accumulated over coordinates 0 .. 7 in float64; ties go to the
  smaller code word.
* The decoded rotated-basis weight is fp32(s_r) * v with v the codeword, exact
  in float32 (every coordinate is a multiple of 1/4 below 3).
"""
from __future__ import annotations

import functools
import itertools

import numpy as np

from . import rvq as R

DIM = 8
N_PATTERNS = 256
N_CODES = 1 << 16


# ------------------------------------------------------------------ base table
def base_patterns() -> np.ndarray:
    """The 256 absolute patterns as int [256, 8] of 2|a_i| (odd), by (squared norm, tuple)."""
    # 2|a| = 7 gives a squared norm >= 12.25 + 7 / 4 > 12, beyond the 256th pattern
    cands = [t for t in itertools.product((1, 3, 5), repeat=DIM)]
    cands.sort(key=lambda t: (sum(v * v for v in t), t))
    return np.array(cands[:N_PATTERNS], dtype=np.int64)


def base_table_words() -> np.ndarray:
    """The 1 KiB table as uint32 [256]: nibble i (bits 4i .. 4i+3) = 2|a_i|."""
    pat = base_patterns()
    words = np.zeros(N_PATTERNS, dtype=np.uint64)
    for i in range(DIM):
        words |= pat[:, i].astype(np.uint64) << np.uint64(4 * i)
    return words.astype(np.uint32)


def kappa_squared() -> float:
    """Mean squared coordinate of the codebook, averaged over all 65 536 code words."""
    pat = base_patterns() / 2.0
    # every pattern appears with 128 sign choices and 2 shifts; the sign-shift cross terms
    # cancel over the shift bit
    return float(np.mean(np.sum(pat * pat, axis=1)) / DIM + 1.0 / 16.0)


# ------------------------------------------------------------------ decoder
def decode_codes(codes: np.ndarray) -> np.ndarray:
    """Codewords v, float64 [..., 8], of 16-bit code words."""
    codes = np.asarray(codes, dtype=np.int64)
    pat = base_patterns()[codes & 0xFF] / 2.0                      # |a|, [..., 8]
    neg = np.zeros(codes.shape + (DIM,), dtype=bool)
    for i in range(DIM - 1):
        neg[..., i] = (codes >> (8 + i)) & 1 == 1
    # the last sign: the one that makes sum_i s_i a_i an even integer
    partial = np.sum(np.where(neg[..., :DIM - 1], -pat[..., :DIM - 1], pat[..., :DIM - 1]), axis=-1)
    plus_sum = partial + pat[..., DIM - 1]
    neg[..., DIM - 1] = np.mod(plus_sum, 2.0) != 0.0
    shift = np.where((codes >> 15) & 1 == 1, 0.25, -0.25)
    return np.where(neg, -pat, pat) + shift[..., None]


def codebook() -> np.ndarray:
    """All 65 536 codewords, float64 [65536, 8], row c = the codeword of code word c."""
    return _codebook_t().T.copy()


@functools.lru_cache(maxsize=1)
def _codebook_t() -> np.ndarray:
    t = np.ascontiguousarray(decode_codes(np.arange(N_CODES)).T)
    t.setflags(write=False)
    return t


# ------------------------------------------------------------------ encoder
def row_scale_f16(wr: np.ndarray) -> np.ndarray:
    """Per-row fp16 scale bits: fp16(RMS(W'_r) / kappa), the RMS summed left to right."""
    sq = np.asarray(wr, np.float64) ** 2
    rms = np.sqrt(np.cumsum(sq, axis=1)[:, -1] / wr.shape[1])
    return (rms / np.sqrt(kappa_squared())).astype(np.float16).view(np.uint16)


def nearest_codes(u: np.ndarray, chunk: int = 8) -> np.ndarray:
    """Code word of the codeword nearest to every row of u [n, 8], by brute force over all
    65 536 codewords (ties: the smaller code word).

    Squared distances are accumulated coordinate by coordinate, j = 0 .. 7, in float64,
    d = d + (u_j - v_j)^2, exactly as ``oracle.rvq.nearest`` does; only the buffers are
    reused between coordinates."""
    u = np.asarray(u, np.float64)
    cbt = _codebook_t()                                            # [8, 65536]
    out = np.empty(u.shape[0], dtype=np.uint16)
    diff = np.empty((chunk, N_CODES))
    dist = np.empty((chunk, N_CODES))
    for lo in range(0, u.shape[0], chunk):
        part = u[lo:lo + chunk]
        n = part.shape[0]
        d, df = dist[:n], diff[:n]
        d.fill(0.0)
        for j in range(DIM):
            np.subtract(part[:, j, None], cbt[j][None, :], out=df)
            np.multiply(df, df, out=df)
            np.add(d, df, out=d)
        out[lo:lo + n] = np.argmin(d, axis=1)
    return out


def encode(wr: np.ndarray):
    """Code words uint16 [rows, cols/8] and fp16 scale bits [rows] of a rotated weight."""
    rows, cols = wr.shape
    scale = row_scale_f16(wr)
    u = R.normalised_vectors(wr, scale, DIM)
    return nearest_codes(u).reshape(rows, cols // DIM), scale


def decode(codes: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """Decoded rotated-basis weight, float32 [rows, cols]: fp32(s_r) * v (one float32 multiply)."""
    codes = np.asarray(codes)
    rows, nv = codes.shape
    v = decode_codes(codes).astype(np.float32)                     # exact
    s = np.asarray(scale_bits, np.uint16).view(np.float16).astype(np.float32)
    return (s[:, None, None] * v).reshape(rows, nv * DIM).astype(np.float32)
