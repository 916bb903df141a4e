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


@functools.lru_cache(maxsize=1)
def _native_synth():
    import ctypes
    import os
    lib = ctypes.CDLL(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "synth",
                                   "libsynth.so"))
    lib.synth_ternary_rows.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64,
                                       ctypes.c_uint32, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    lib.synth_ternary_rows.restype = None
    return lib


def fill_ternary(seed, expert, matrix, p0, out):
    """Fill int8 out[rows, cols] with synth.ternary_rows(...) through the native twin of the generator
    (same numbers; the twin is checked against the Python definition in test_host_codec)."""
    rows, cols = out.shape
    _native_synth().synth_ternary_rows(seed, expert, matrix, cols, synth.zero_threshold(p0), 0, rows,
                                       out.ctypes.data)
    return out


def seeded_weights(seed, expert, matrix, rows, cols, p0):
    """float64 weights s_r * t_rc of one seeded ternary matrix (the oracle's definition of the layer)."""
    tern = fill_ternary(seed, expert, matrix, p0, np.empty((rows, cols), np.int8))
    s = synth.f16_to_f64(synth.row_scales(seed, expert, matrix, rows))
    return tern.astype(np.float64) * s[:, None]


def rvq_oracle_matrix(args):
    """Oracle-coded RVQ matrix (decoded W', sign_out, sign_in) of one seeded expert matrix: rotate,
    encode with the given fp16 codebooks, decode.  A plain function so that a spawn pool can run it."""
    from oracle import rvq as R
    seed, e, m, rows, cols, cb_bits = args
    w = synth.rvq_weight(seed, e, m, rows, cols)
    so, si = synth.rvq_signs(seed, e, m, rows, cols)
    cb = np.asarray(cb_bits, np.uint16).view(np.float16).astype(np.float64)
    idx, sc = R.encode(R.rotate_weight(w, so, si), cb)
    return R.decode(idx, cb_bits, sc), so, si
