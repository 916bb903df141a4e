"""Shared builders for the GPU parity tests: seeded inputs -> oracle artifacts."""
from __future__ import annotations

import functools

import numpy as np

import synth
from oracle import codec as C
from oracle import dictionary as D

BLOCK = 256


@functools.lru_cache(maxsize=8)
def dictionary(p0: float) -> np.ndarray:
    return D.build(p0)


@functools.lru_cache(maxsize=8)
def entry_table(p0: float) -> dict:
    return C.entry_table(dictionary(p0))


def oracle_matrix(seed, expert, matrix, rows, cols, p0, block=BLOCK):
    """Ternary weights, oracle-encoded stream and fp16 scales of one matrix."""
    tern = synth.ternary_matrix(seed, expert, matrix, rows, cols, p0)
    codes, off = C.encode(tern, dictionary(p0), block, table=entry_table(p0))
    scale = synth.row_scales(seed, expert, matrix, rows)
    return tern, codes, off, scale


def oracle_matrix_set(seed, E, matrix, rows, cols, p0, block=BLOCK):
    """Concatenated streams of E experts' matrices: (codes, code_base, blk_off, scales, decoded W list)."""
    all_codes, bases, offs, scales, dense = [], [], [], [], []
    base = 0
    words = dictionary(p0)
    for e in range(E):
        tern, codes, off, sc = oracle_matrix(seed, e, matrix, rows, cols, p0, block)
        bases.append(base)
        base += len(codes)
        all_codes.append(codes)
        offs.append(off)
        scales.append(sc)
        dense.append(C.decode(codes, off, words, sc, rows, cols, block))
    return (np.concatenate(all_codes), np.asarray(bases, np.uint64), np.concatenate(offs),
            np.concatenate(scales), dense)


def bf16_tensor(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16).copy()).to(device)


def bf16_values(t) -> np.ndarray:
    """Device bf16 (int16 view) -> float64 host values."""
    return synth.bf16_to_f64(t.cpu().numpy().view(np.uint16))
