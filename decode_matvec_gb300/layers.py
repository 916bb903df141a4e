"""Assembles device-resident dictionary-coded and RVQ-coded expert layers.

The caller supplies the weights (a function returning one expert matrix as
int8 ternary, or as float64 for RVQ); matrices are encoded with the library's
host encoders (``qmoe_pack`` / ``rvq_pack``, which release the GIL) on a thread
pool and uploaded as the concatenated per-set arrays that ``qmoe_matrix_set`` /
``rvq_matrix_set`` describe.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

from . import (Dictionary, MatrixSet, RvqMatrixSet, e8p_pack, qmoe_encode_dictionary, qmoe_pack_into, rvq_pack)


def _threads(n: int | None) -> int:
    if n:
        return n
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 4


class DictLayerArtifact:
    """Host copy of one matrix set: codes, per-expert code bases, offsets, scales."""

    def __init__(self, count, rows, cols, block, codes, code_base, blk_off, scales, n_codes):
        self.count, self.rows, self.cols, self.block = count, rows, cols, block
        self.codes, self.code_base, self.blk_off, self.scales = codes, code_base, blk_off, scales
        self.n_codes = n_codes          # int64 [count]

    @property
    def nb(self) -> int:
        return (self.cols + self.block - 1) // self.block

    def expert_bytes(self, e: int) -> int:
        """Stored bytes of matrix e as the device holds it: codes (uint16), row starts (uint32, rows + 1),
        block lengths (uint8, rows x (nb - 1)) and row scales (fp16)."""
        return 2 * int(self.n_codes[e]) + 4 * (self.rows + 1) + self.rows * (self.nb - 1) + 2 * self.rows

    def expert_offset_bytes_unread_by_cuda_cores(self, e: int) -> int:
        """The block lengths of matrix e: the CUDA-core kernel reads only the row starts."""
        return self.rows * (self.nb - 1)

    def to_device(self, device="cuda") -> MatrixSet:
        return MatrixSet.from_host(self.codes, self.blk_off, self.scales, self.rows, self.cols, self.block,
                                   code_base=self.code_base, count=self.count, device=device)


def pack_matrix_set(count: int, rows: int, cols: int, dict_words: np.ndarray, tern_fn, scale_fn,
                    block: int = 256, threads: int | None = None) -> DictLayerArtifact:
    """Encode `count` matrices: tern_fn(e, out_int8[rows, cols]) fills weights, scale_fn(e) -> fp16 bits."""
    nb = (cols + block - 1) // block
    words = np.ascontiguousarray(dict_words, dtype=np.uint32)
    offs = np.zeros((count, rows * nb + 1), dtype=np.uint32)
    scales = np.zeros((count, rows), dtype=np.uint16)
    per = [None] * count
    nthreads = _threads(threads)
    scratch = {}

    def work(e):
        import threading
        tid = threading.get_ident()
        bufs = scratch.get(tid)
        if bufs is None:
            bufs = (np.empty((rows, cols), np.int8), np.empty(rows * cols // 2 + 1, np.uint16))
            scratch[tid] = bufs
        tern, cbuf = bufs
        tern_fn(e, tern)
        n = qmoe_pack_into(tern, words, block, cbuf, offs[e])
        per[e] = cbuf[:n].copy()
        scales[e] = scale_fn(e)
        return n

    with cf.ThreadPoolExecutor(max_workers=nthreads) as ex:
        n_codes = np.asarray(list(ex.map(work, range(count))), dtype=np.int64)
    base = np.zeros(count, dtype=np.uint64)
    base[1:] = np.cumsum(n_codes[:-1]).astype(np.uint64)
    codes = np.concatenate(per) if count else np.zeros(0, np.uint16)
    return DictLayerArtifact(count, rows, cols, block, codes, base, offs.reshape(-1), scales.reshape(-1), n_codes)


class DictLayer:
    """A dictionary-coded Switch-style MoE FFN layer resident on the device."""

    def __init__(self, p0: float, E: int, d_model: int, d_ff: int, wi_tern_fn, wo_tern_fn, wi_scale_fn, wo_scale_fn,
                 block: int = 256, device="cuda", threads: int | None = None):
        self.words, _ = qmoe_encode_dictionary(p0)
        self.E, self.d_model, self.d_ff, self.block = E, d_model, d_ff, block
        self.wi_host = pack_matrix_set(E, d_ff, d_model, self.words, wi_tern_fn, wi_scale_fn, block, threads)
        self.wo_host = pack_matrix_set(E, d_model, d_ff, self.words, wo_tern_fn, wo_scale_fn, block, threads)
        self.dictionary = Dictionary(self.words, device=device)
        self.wi = self.wi_host.to_device(device)
        self.wo = self.wo_host.to_device(device)

    def stream_bytes(self, experts) -> int:
        """Stored bytes (codes + offsets + scales, both matrices) of the given experts."""
        return int(sum(self.wi_host.expert_bytes(e) + self.wo_host.expert_bytes(e) for e in experts))

    def total_bytes(self) -> int:
        return self.stream_bytes(range(self.E))


def pack_rvq_set(count: int, rows: int, cols: int, codebooks_f16: np.ndarray, weight_fn, sign_fn,
                 threads: int | None = None, device="cuda", stages=None) -> RvqMatrixSet:
    """Encode `count` RVQ matrices: weight_fn(e) -> float64 [rows, cols], sign_fn(e) -> (sign_out, sign_in).
    stages: None (two stages each, two codebooks given) or per-matrix stage counts (1 .. codebooks given)."""
    scales = np.zeros((count, rows), dtype=np.uint16)
    so = np.zeros((count, rows), dtype=np.int8)
    si = np.zeros((count, cols), dtype=np.int8)
    cb = np.ascontiguousarray(codebooks_f16, dtype=np.uint16)
    per = [None] * count

    def work(e):
        w = weight_fn(e)
        s_out, s_in = sign_fn(e)
        per[e], scales[e] = rvq_pack(w, s_out, s_in, cb, 2 if stages is None else int(stages[e]))
        so[e], si[e] = s_out, s_in

    with cf.ThreadPoolExecutor(max_workers=_threads(threads)) as ex:
        list(ex.map(work, range(count)))
    idx = np.stack(per) if stages is None else per
    return RvqMatrixSet.from_host(idx, cb if stages is not None else cb[:2], scales.reshape(-1), so.reshape(-1),
                                  si.reshape(-1), count, rows, cols, device=device)


def pack_e8p_set(count: int, rows: int, cols: int, weight_fn, sign_fn, threads: int | None = None,
                 device="cuda") -> RvqMatrixSet:
    """Encode `count` matrices with the E8P lattice code: weight_fn(e) -> float64 [rows, cols],
    sign_fn(e) -> (sign_out, sign_in)."""
    codes = np.zeros((count, rows, cols // 8), dtype=np.uint16)
    scales = np.zeros((count, rows), dtype=np.uint16)
    so = np.zeros((count, rows), dtype=np.int8)
    si = np.zeros((count, cols), dtype=np.int8)

    def work(e):
        w = weight_fn(e)
        s_out, s_in = sign_fn(e)
        codes[e], scales[e] = e8p_pack(w, s_out, s_in)
        so[e], si[e] = s_out, s_in

    with cf.ThreadPoolExecutor(max_workers=_threads(threads)) as ex:
        list(ex.map(work, range(count)))
    return RvqMatrixSet.e8p_from_host(codes, scales.reshape(-1), so.reshape(-1), si.reshape(-1), count, rows, cols,
                                      device=device)
