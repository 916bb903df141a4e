"""QMoE dictionary codec: encoder, reference decoder, rate ledger.  Test infrastructure.

Encoder -- [QMoE] section "The GPU Decoding Kernel", paragraph "Encoding
(compression time)": scan each row and emit the codeword of the longest
dictionary sequence that is a prefix of what remains; rows are independent and
packed densely with start offsets.  Reading taken here: rows are cut into
blocks of ``block`` weights (256 unless stated; the last block of a row may be
shorter), a codeword never crosses a block boundary, and offsets are kept per
(row, block) instead of per row, so that a row can be decoded from any block.
Blocks are stored in row-major block order; ``blk_off[r*nb + b]`` is the index
of the first codeword of block b of row r and a final sentinel holds the
total.  Row and block lengths must be even (entries hold whole pairs).

Decoder -- [M8.5] section 0x08A, the reference decoder: expand every codeword
of a row through the dictionary and map symbols (0, 1, 2) to the row's
(zero, negative, positive) values; here the row values are (0, -s, +s) with
one fp16 scale s per row ([QMoE] "Quantization grid": per-row
{w_min, 0, w_max}; the synthetic layers use w_min = -w_max).

Rate ledger -- [M8.5] 0x00A/0x01A (effective rate counts every byte the
loader needs) and 0x08A (a codeword expanding to L weights costs 16/L bits;
sub-one-bit payload needs E[L] > 16).  The entropy of the independence model
is from [QMoE] "The entropy perspective"; the bitmask and column-index
alternatives from "Why standard sparse formats don't work well enough".
"""
from __future__ import annotations

import math

import numpy as np

from . import dictionary as D

BLOCK = 256
SYMBOL_OF_TERNARY = {0: 0, -1: 1, 1: 2}


def n_blocks(cols: int, block: int = BLOCK) -> int:
    return (cols + block - 1) // block


def entry_table(words: np.ndarray) -> dict:
    """Map symbol tuple -> codeword, read back from the packed entries."""
    table = {}
    for code in range(len(words) // 2):
        table.setdefault(D.unpack_entry(words, code), code)
    return table


def encode_block(symbols: tuple, table: dict) -> list[int]:
    """Greedy longest match of one block's symbols."""
    out = []
    pos = 0
    n = len(symbols)
    while pos < n:
        for L in range(min(D.MAX_LEN, n - pos), 0, -2):
            code = table.get(symbols[pos:pos + L])
            if code is not None:
                out.append(code)
                pos += L
                break
        else:
            raise ValueError("no dictionary entry matches at this position")
    return out


def encode(tern: np.ndarray, words: np.ndarray, block: int = BLOCK, table: dict | None = None):
    """Encode a rows x cols ternary int8 matrix.  Returns (codes uint16, blk_off uint32)."""
    tern = np.asarray(tern)
    rows, cols = tern.shape
    if cols % 2 or block % 2 or block <= 0:
        raise ValueError("row length and block length must be even")
    if table is None:
        table = entry_table(words)
    nb = n_blocks(cols, block)
    sym = np.where(tern == 0, 0, np.where(tern < 0, 1, 2))
    codes: list[int] = []
    offs = np.zeros(rows * nb + 1, dtype=np.uint32)
    for r in range(rows):
        row = tuple(int(v) for v in sym[r])
        for b in range(nb):
            offs[r * nb + b] = len(codes)
            codes.extend(encode_block(row[b * block:(b + 1) * block], table))
    offs[rows * nb] = len(codes)
    return np.asarray(codes, dtype=np.uint16), offs


def expansion(words: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(length [n], symbols [n, 28]) of every entry, read through the Fig. 4 bit layout."""
    w = np.asarray(words, dtype=np.uint32).reshape(-1, 2)
    c0, c1 = w[:, 0] & 0xF, w[:, 1] & 0xF
    if np.any(c0 != c1):
        raise ValueError("pair counts of the two halves disagree")
    length = 2 * c0.astype(np.int64)
    lanes = np.arange(28)
    half = lanes // 14
    shift = (4 + 2 * (lanes % 14)).astype(np.uint32)
    sym = (w[:, half] >> shift[None, :]) & 3
    return length, sym.astype(np.int64)


def decode_symbols(codes: np.ndarray, blk_off: np.ndarray, words: np.ndarray,
                   rows: int, cols: int, block: int = BLOCK) -> np.ndarray:
    """Ternary symbols (0, 1, 2) of the whole matrix; checks every block expands exactly."""
    length, sym = expansion(words)
    codes = np.asarray(codes, dtype=np.int64)
    nb = n_blocks(cols, block)
    blk_off = np.asarray(blk_off, dtype=np.int64)
    if blk_off.shape != (rows * nb + 1,) or blk_off[0] != 0 or blk_off[-1] != len(codes):
        raise ValueError("malformed block offsets")
    if np.any(np.diff(blk_off) < 0):
        raise ValueError("block offsets must be non-decreasing")
    out = np.empty((rows, cols), dtype=np.int64)
    for r in range(rows):
        for b in range(nb):
            lo, hi = blk_off[r * nb + b], blk_off[r * nb + b + 1]
            cs = codes[lo:hi]
            seq = np.concatenate([sym[c, :length[c]] for c in cs]) if len(cs) else np.zeros(0, np.int64)
            c0, c1 = b * block, min(cols, (b + 1) * block)
            if len(seq) != c1 - c0:
                raise ValueError(f"row {r} block {b}: expands to {len(seq)} weights, expected {c1 - c0}")
            out[r, c0:c1] = seq
    return out


def decode(codes, blk_off, words, scales_f16_bits, rows, cols, block: int = BLOCK) -> np.ndarray:
    """Reference decoder: float64 weights, symbol 0/1/2 -> 0/-s/+s with s the row's fp16 scale."""
    sym = decode_symbols(codes, blk_off, words, rows, cols, block)
    s = np.asarray(scales_f16_bits, dtype=np.uint16).view(np.float16).astype(np.float64)
    values = np.stack([np.zeros(rows), -s, s], axis=1)     # (zero, negative, positive) per row
    return np.take_along_axis(values, sym, axis=1)


def ternary_of_symbols(sym: np.ndarray) -> np.ndarray:
    return np.array([0, -1, 1], dtype=np.int8)[np.asarray(sym)]


# ---------------------------------------------------------------- rate ledger
def entropy_bits(p0: float) -> float:
    """Bits per weight of the independence model ([QMoE] "The entropy perspective")."""
    q = (1.0 - p0) / 2.0
    return -p0 * math.log2(p0) - 2.0 * q * math.log2(q)


def ledger(n_codes: int, rows: int, cols: int, offset_bytes: int, scale_bytes: int,
           dict_bytes: int = 8 * D.N_ENTRIES, p0_hat: float | None = None) -> dict:
    """Effective rate of one stored matrix (or layer), everything counted at its stored width."""
    P = rows * cols
    payload = 16.0 * n_codes / P
    eff = 8.0 * (2 * n_codes + offset_bytes + scale_bytes) / P
    out = {
        "weights": P,
        "codes": n_codes,
        "mean_run": P / n_codes if n_codes else float("inf"),
        "payload_bits_per_weight": payload,
        "effective_bits_per_weight": eff,
        "effective_with_dictionary": eff + 8.0 * dict_bytes / P,
        "compression_vs_bf16": 16.0 / eff,
        "payload_compression_vs_bf16": 16.0 / payload,
    }
    if p0_hat is not None:
        out["entropy_bits_per_weight"] = entropy_bits(p0_hat)
        out["bitmask_bits_per_weight"] = 1.0 + (1.0 - p0_hat)      # mask + one sign bit per nonzero
        out["colindex_bits_per_weight"] = (1.0 - p0_hat) * (math.ceil(math.log2(cols)) + 1.0)
    return out
