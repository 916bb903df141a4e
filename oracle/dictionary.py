"""QMoE dictionary: Algorithm 1 and the Figure 4 entry format.  Test infrastructure.

[QMoE] section "The Fixed-to-Variable Dictionary Code", paragraph
"Dictionary generation (Algorithm 1)": a max-priority queue seeded with the
empty sequence; pop the most probable sequence, keep it when it holds 1 to 28
ternary values, push its extensions by every one of the 9 ternary pairs with
probability multiplied by P(t1)P(t2); stop at 2**16 entries; the dictionary
is ordered from most to least probable.  Symbol probabilities follow the
independence model: P(0) = p0, P(1) = P(2) = (1 - p0)/2.

Readings taken where the page is silent:
* priority of a sequence = n0*ln(p0) + nz*ln((1-p0)/2) recomputed from its
  counts, so sequences with equal counts tie exactly;
* ties are broken by the symbol tuple in lexicographic order, smallest first
  (0 < 1 < 2), i.e. Python's tuple order, which ``heapq`` applies after the
  priority;
* a sequence of 28 values is not expanded (its extensions could never be kept).

Entry format, [QMoE] "Dictionary storage format (Figure 4)" and the kernel
walk-through of Listing 1: an entry is two uint32 words; in both words bits
[3:0] hold the total pair count; word h holds symbol 14*h + i at bits
[5+2i : 4+2i]; symbol 0 is the zero weight, 1 is w_min, 2 is w_max; unused
symbol fields are 0 (the listing multiplies every one of the 28 lanes, so
padding must decode to a zero weight).
"""
from __future__ import annotations

import heapq
import math

import numpy as np

N_ENTRIES = 1 << 16
MAX_LEN = 28          # ternary values per entry
PAIRS = tuple((a, b) for a in range(3) for b in range(3))


def log_probs(p0: float) -> tuple[float, float]:
    """(ln P(0), ln P(nonzero symbol)) of the independence model."""
    if not (0.0 < p0 < 1.0):
        raise ValueError("p0 must lie in (0, 1)")
    return math.log(p0), math.log((1.0 - p0) / 2.0)


def priority(seq: tuple, lp0: float, lq: float) -> float:
    n0 = seq.count(0)
    return n0 * lp0 + (len(seq) - n0) * lq


def generate(p0: float, n_entries: int = N_ENTRIES) -> list[tuple]:
    """Algorithm 1: the ``n_entries`` most probable pair sequences, most probable first."""
    lp0, lq = log_probs(p0)
    heap = [(-0.0, ())]
    entries = []
    while len(entries) < n_entries:
        negp, seq = heapq.heappop(heap)
        if 1 <= len(seq) <= MAX_LEN:
            entries.append(seq)
        if len(seq) < MAX_LEN:
            for t1, t2 in PAIRS:
                child = seq + (t1, t2)
                heapq.heappush(heap, (-priority(child, lp0, lq), child))
    return entries


def pack_entry(seq: tuple) -> tuple[int, int]:
    """Figure 4 layout of one entry as (word0, word1)."""
    if len(seq) % 2 or not (2 <= len(seq) <= MAX_LEN):
        raise ValueError("entry length must be even and in [2, 28]")
    pairs = len(seq) // 2
    words = [pairs, pairs]
    for j, s in enumerate(seq):
        h, i = divmod(j, 14)
        words[h] |= (s & 3) << (4 + 2 * i)
    return words[0], words[1]


def pack(entries: list[tuple]) -> np.ndarray:
    """All entries as the flat uint32 array ``dec`` with entry e at dec[2e], dec[2e+1]."""
    out = np.zeros(2 * len(entries), dtype=np.uint32)
    for e, seq in enumerate(entries):
        out[2 * e], out[2 * e + 1] = pack_entry(seq)
    return out


def unpack_entry(words: np.ndarray, code: int) -> tuple:
    """Symbols of entry ``code`` read back the way Listing 1 reads them."""
    w0, w1 = int(words[2 * code]), int(words[2 * code + 1])
    if (w0 & 0xF) != (w1 & 0xF):
        raise ValueError(f"entry {code}: pair counts disagree")
    n = 2 * (w0 & 0xF)
    out = []
    for lane in range(n):
        w = w0 if lane < 14 else w1
        out.append((w >> (4 + 2 * (lane % 14))) & 3)
    return tuple(out)


def build(p0: float) -> np.ndarray:
    """Dictionary words for the independence model with zero probability p0."""
    return pack(generate(p0))


def measured_p0(tern: np.ndarray) -> float:
    """Zero fraction of a ternary matrix, for building the dictionary from real weights."""
    t = np.asarray(tern)
    return float(np.count_nonzero(t == 0)) / float(t.size)
