"""Python binding of ``libqmoe.so``: the GB300 fused decode-and-multiply library.

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels (``include/qmoe.h`` documents each call).  PyTorch supplies device
memory and streams.  Importing this package fails loudly when the library has
not been built (``python decode_matvec_gb300/build.py``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python decode_matvec_gb300/build.py` "
                      "(or __graft_entry__.build()); there is no non-CUDA fallback")
_lib = ctypes.CDLL(LIB_PATH)

QMOE_OK, QMOE_EINVAL, QMOE_ECAPACITY, QMOE_ECUDA, QMOE_EFORMAT, QMOE_ETIMEOUT, QMOE_EUNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
STATUS_NAMES = {0: "QMOE_OK", -1: "QMOE_EINVAL", -2: "QMOE_ECAPACITY", -3: "QMOE_ECUDA", -4: "QMOE_EFORMAT",
                -5: "QMOE_ETIMEOUT", -6: "QMOE_EUNSUPPORTED"}
DICT_ENTRIES = 65536
DICT_WORDS = 2 * DICT_ENTRIES
COMPACT_BYTES = 7 * DICT_ENTRIES
QMOE_VQ_RVQ, QMOE_VQ_E8P = 0, 1      # code formats of an RVQ matrix set

EXPORTED = [
    "qmoe_encode_dictionary", "qmoe_pack", "qmoe_dict_compact", "qmoe_expert_matvec", "qmoe_route",
    "qmoe_bucketise", "qmoe_moe_layer_ws_size", "qmoe_moe_layer", "rvq_expert_matmul_ws_size",
    "rvq_expert_matmul", "rvq_moe_layer_ws_size", "rvq_moe_layer", "rvq_pack", "qmoe_check_status",
    "qmoe_last_error", "qmoe_decode_dense", "rvq_decode_dense", "qmoe_set_phase_events",
    "qmoe_moe_layer_noalloc", "qmoe_pack_device_ws_size", "qmoe_pack_device", "rvq_pack_stages",
    "rvq_stage_allocation", "e8p_base_table", "e8p_pack", "e8p_nearest", "qmoe_offsets_compact",
    "qmoe_moe_layer_kernels",
]


class QmoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.qmoe_last_error().decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != QMOE_OK:
        raise QmoeError(status, where)


# ------------------------------------------------------------------ C structs
class CDict(ctypes.Structure):
    _fields_ = [("words", ctypes.c_void_p), ("compact", ctypes.c_void_p)]


class CMatrixSet(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("code_base", ctypes.c_void_p), ("row_off", ctypes.c_void_p),
                ("blk_len", ctypes.c_void_p),
                ("scale_f16", ctypes.c_void_p), ("count", ctypes.c_int), ("rows", ctypes.c_int),
                ("cols", ctypes.c_int), ("block", ctypes.c_int)]


class CRvqSet(ctypes.Structure):
    _fields_ = [("idx", ctypes.c_void_p), ("codebooks", ctypes.c_void_p), ("scale_f16", ctypes.c_void_p),
                ("sign_out", ctypes.c_void_p), ("sign_in", ctypes.c_void_p), ("count", ctypes.c_int),
                ("rows", ctypes.c_int), ("cols", ctypes.c_int), ("stages", ctypes.c_void_p),
                ("idx_base", ctypes.c_void_p), ("n_stages", ctypes.c_int), ("format", ctypes.c_int)]


_vp, _i, _sz, _d = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_double
_sig = {
    "qmoe_encode_dictionary": [_vp, _sz, _d, _vp, _vp],
    "qmoe_pack": [_vp, _i, _i, _i, _vp, _vp, _sz, _vp, _vp],
    "qmoe_dict_compact": [_vp, _vp],
    "qmoe_expert_matvec": [_vp, _vp, _vp, _i, _vp, _i, _vp],
    "qmoe_route": [_vp, _i, _i, _i, _vp, _vp, _vp],
    "qmoe_bucketise": [_vp, _i, _i, _i, _vp, _vp, _vp, _vp],
    "qmoe_moe_layer_ws_size": [_i, _i, _i, _i, _i, _vp],
    "qmoe_moe_layer_kernels": [_i, _i, _i, _i, _i, _vp, _vp, _vp],
    "qmoe_moe_layer": [_vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _i, _vp, _sz, _vp],
    "rvq_expert_matmul_ws_size": [_i, _i, _i, _vp],
    "rvq_expert_matmul": [_vp, _vp, _i, _vp, _i, _vp, _sz, _vp],
    "rvq_moe_layer_ws_size": [_i, _i, _i, _i, _i, _vp],
    "rvq_moe_layer": [_vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _i, _vp, _sz, _vp],
    "rvq_pack": [_vp, _i, _i, _vp, _vp, _vp, _vp, _vp],
    "qmoe_check_status": [_vp],
    "qmoe_decode_dense": [_vp, _vp, _vp, _vp],
    "rvq_decode_dense": [_vp, _vp, _vp],
    "qmoe_set_phase_events": [_vp, _i],
    "qmoe_moe_layer_noalloc": [_vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _i, _vp],
    "qmoe_pack_device_ws_size": [_i, _i, _i, _vp],
    "qmoe_pack_device": [_vp, _vp, _i, _i, _i, _vp, _sz, _vp, _vp, _sz, _vp],
    "rvq_pack_stages": [_vp, _i, _i, _vp, _vp, _vp, _i, _vp, _vp],
    "rvq_stage_allocation": [_vp, _i, _i, _vp],
    "e8p_base_table": [_vp],
    "e8p_pack": [_vp, _i, _i, _vp, _vp, _vp, _vp],
    "e8p_nearest": [_vp, _sz, _vp],
    "qmoe_offsets_compact": [_vp, _i, _i, _vp, _vp],
}
for _name, _args in _sig.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_lib.qmoe_last_error.argtypes = []
_lib.qmoe_last_error.restype = ctypes.c_char_p


def lib() -> ctypes.CDLL:
    return _lib


def _np_ptr(a: np.ndarray) -> int:
    return a.ctypes.data if a is not None else None


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


# ================================================================ host codec
def qmoe_encode_dictionary(p0: float | None = None, symbols: np.ndarray | None = None):
    """Algorithm 1 dictionary as uint32[2*65536], plus the p0 it was built for."""
    words = np.zeros(DICT_WORDS, dtype=np.uint32)
    used = ctypes.c_double(0.0)
    sym = None if symbols is None else np.ascontiguousarray(symbols, dtype=np.int8)
    _check(_lib.qmoe_encode_dictionary(_np_ptr(sym), 0 if sym is None else sym.size,
                                       float(p0 if p0 is not None else 0.0), _np_ptr(words), ctypes.byref(used)),
           "qmoe_encode_dictionary")
    return words, used.value


def qmoe_pack(tern: np.ndarray, dict_words: np.ndarray, block: int = 256):
    """Greedy longest-match codewords (uint16) and per-block offsets (uint32) of a ternary matrix."""
    tern = np.ascontiguousarray(tern, dtype=np.int8)
    rows, cols = tern.shape
    words = np.ascontiguousarray(dict_words, dtype=np.uint32)
    n = ctypes.c_size_t(0)
    _check(_lib.qmoe_pack(_np_ptr(tern), rows, cols, block, _np_ptr(words), None, 0, ctypes.byref(n), None),
           "qmoe_pack(count)")
    nb = (cols + block - 1) // block
    codes = np.zeros(max(n.value, 1), dtype=np.uint16)
    off = np.zeros(rows * nb + 1, dtype=np.uint32)
    _check(_lib.qmoe_pack(_np_ptr(tern), rows, cols, block, _np_ptr(words), _np_ptr(codes), codes.size,
                          ctypes.byref(n), _np_ptr(off)), "qmoe_pack")
    return codes[:n.value], off


def qmoe_pack_into(tern: np.ndarray, dict_words: np.ndarray, block: int, codes_out: np.ndarray,
                   off_out: np.ndarray) -> int:
    """Pack into caller buffers (views); returns the codeword count.  Releases the GIL while packing."""
    tern = np.ascontiguousarray(tern, dtype=np.int8)
    rows, cols = tern.shape
    n = ctypes.c_size_t(0)
    _check(_lib.qmoe_pack(_np_ptr(tern), rows, cols, block, _np_ptr(dict_words), _np_ptr(codes_out),
                          codes_out.size, ctypes.byref(n), _np_ptr(off_out)), "qmoe_pack")
    return n.value


def qmoe_dict_compact(dict_words: np.ndarray) -> np.ndarray:
    words = np.ascontiguousarray(dict_words, dtype=np.uint32)
    out = np.zeros(COMPACT_BYTES, dtype=np.uint8)
    _check(_lib.qmoe_dict_compact(_np_ptr(words), _np_ptr(out)), "qmoe_dict_compact")
    return out


def rvq_pack(w: np.ndarray, sign_out: np.ndarray, sign_in: np.ndarray, codebooks_f16: np.ndarray,
             stages: int | None = None):
    """Host RVQ encoder: (idx uint8 [rows, cols/8, S], scale fp16 bits [rows]); S = stages, by default
    the number of codebooks given ([S_max, 256, 8] fp16 bits; the first S are used)."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    rows, cols = w.shape
    so = np.ascontiguousarray(sign_out, dtype=np.int8)
    si = np.ascontiguousarray(sign_in, dtype=np.int8)
    cb = np.ascontiguousarray(codebooks_f16, dtype=np.uint16)
    n_st = cb.shape[0] if stages is None else int(stages)
    if not 1 <= n_st <= cb.shape[0]:
        raise ValueError("stage count outside 1 .. number of codebooks")
    idx = np.zeros((rows, cols // 8, n_st), dtype=np.uint8)
    sc = np.zeros(rows, dtype=np.uint16)
    _check(_lib.rvq_pack_stages(_np_ptr(w), rows, cols, _np_ptr(so), _np_ptr(si), _np_ptr(cb), n_st, _np_ptr(idx),
                                _np_ptr(sc)), "rvq_pack_stages")
    return idx, sc


def rvq_stage_allocation(popularity: np.ndarray, s_bar: int = 2) -> np.ndarray:
    """Stages per expert by popularity thirds (s_bar + 1 / s_bar / s_bar - 1), uint8 [E]."""
    pop = np.ascontiguousarray(popularity, dtype=np.float64)
    out = np.zeros(pop.shape[0], dtype=np.uint8)
    _check(_lib.rvq_stage_allocation(_np_ptr(pop), pop.shape[0], int(s_bar), _np_ptr(out)), "rvq_stage_allocation")
    return out


def e8p_base_table() -> np.ndarray:
    """The E8P base table: uint32 [256], nibble j of entry p = 2|a_j| of absolute pattern p."""
    out = np.zeros(256, dtype=np.uint32)
    _check(_lib.e8p_base_table(_np_ptr(out)), "e8p_base_table")
    return out


def e8p_pack(w: np.ndarray, sign_out: np.ndarray, sign_in: np.ndarray):
    """Host E8P encoder: (code words uint16 [rows, cols/8], scale fp16 bits [rows])."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    rows, cols = w.shape
    so = np.ascontiguousarray(sign_out, dtype=np.int8)
    si = np.ascontiguousarray(sign_in, dtype=np.int8)
    codes = np.zeros((rows, cols // 8), dtype=np.uint16)
    sc = np.zeros(rows, dtype=np.uint16)
    _check(_lib.e8p_pack(_np_ptr(w), rows, cols, _np_ptr(so), _np_ptr(si), _np_ptr(codes), _np_ptr(sc)), "e8p_pack")
    return codes, sc


def e8p_nearest(u: np.ndarray) -> np.ndarray:
    """Code words (uint16 [n]) of the E8P codewords nearest to the rows of u [n, 8]."""
    u = np.ascontiguousarray(u, dtype=np.float64).reshape(-1, 8)
    out = np.zeros(u.shape[0], dtype=np.uint16)
    _check(_lib.e8p_nearest(_np_ptr(u), u.shape[0], _np_ptr(out)), "e8p_nearest")
    return out


def qmoe_last_error() -> str:
    return _lib.qmoe_last_error().decode()


def qmoe_check_status(stream=None) -> int:
    return _lib.qmoe_check_status(_stream_ptr(stream))


# ================================================================ device objects
class Dictionary:
    """Canonical words and the derived compact table, resident on the device."""

    def __init__(self, words: np.ndarray, device="cuda"):
        import torch
        w = np.ascontiguousarray(words, dtype=np.uint32)
        compact = qmoe_dict_compact(w)
        self.words_host = w
        self.words = torch.from_numpy(w.view(np.int32)).to(device)
        self.compact = torch.from_numpy(compact).to(device)
        self.c = CDict(_dptr(self.words), _dptr(self.compact))


class MatrixSet:
    """`count` dictionary-coded matrices of one shape, resident on the device, with compact offsets:
    row_off uint32 [count][rows + 1] and blk_len uint8 [count][rows][nb - 1] (qmoe_offsets_compact)."""

    def __init__(self, codes, code_base, row_off, blk_len, scale_f16, count, rows, cols, block=256):
        self.codes, self.code_base, self.row_off, self.blk_len, self.scale = codes, code_base, row_off, blk_len, scale_f16
        self.count, self.rows, self.cols, self.block = count, rows, cols, block
        self.c = CMatrixSet(_dptr(codes), _dptr(code_base), _dptr(row_off), _dptr(blk_len), _dptr(scale_f16), count,
                            rows, cols, block)

    @property
    def nb(self) -> int:
        return (self.cols + self.block - 1) // self.block

    @classmethod
    def from_host(cls, codes: np.ndarray, blk_off: np.ndarray, scale_f16: np.ndarray, rows, cols, block=256,
                  code_base: np.ndarray | None = None, count: int = 1, device="cuda"):
        """From qmoe_pack's output (uint32 block offsets [count][rows*nb + 1]), re-encoded compactly."""
        import torch
        codes = np.ascontiguousarray(codes, dtype=np.uint16)
        padded = np.zeros((codes.size + 15) // 8 * 8, dtype=np.uint16)     # whole 16-byte chunks, plus one
        padded[:codes.size] = codes
        c = torch.from_numpy(padded.view(np.int16)).to(device)
        row_off, blk_len = qmoe_offsets_compact(blk_off, rows, (cols + block - 1) // block, count)
        o = torch.from_numpy(row_off.view(np.int32).copy()).to(device)
        bl = torch.from_numpy(blk_len.copy()).to(device) if blk_len.size else None
        s = torch.from_numpy(np.ascontiguousarray(scale_f16, dtype=np.uint16).view(np.int16).copy()).to(device)
        b = None
        if code_base is not None:
            b = torch.from_numpy(np.ascontiguousarray(code_base, dtype=np.uint64).view(np.int64).copy()).to(device)
        return cls(c, b, o, bl, s, count, rows, cols, block)

    def expert(self, e: int, code_base_host=None) -> "MatrixSet":
        """A one-matrix set for matrix e (views into the same device buffers); code_base_host: the host copy
        of the set's code bases (needed when count > 1)."""
        base = int(code_base_host[e]) if self.count > 1 else 0
        nb1 = self.nb - 1
        return MatrixSet(self.codes[base:], None, self.row_off[e * (self.rows + 1):(e + 1) * (self.rows + 1)],
                         self.blk_len[e * self.rows * nb1:(e + 1) * self.rows * nb1] if nb1 else None,
                         self.scale[e * self.rows:(e + 1) * self.rows], 1, self.rows, self.cols, self.block)


def qmoe_offsets_compact(blk_off: np.ndarray, rows: int, nb: int, count: int = 1):
    """Compact offsets of `count` matrices from their uint32 block offsets [count][rows*nb + 1]:
    (row_off uint32 [count*(rows + 1)], blk_len uint8 [count*rows*(nb - 1)])."""
    bo = np.ascontiguousarray(blk_off, dtype=np.uint32).reshape(count, rows * nb + 1)
    row_off = np.zeros((count, rows + 1), dtype=np.uint32)
    blk_len = np.zeros((count, rows * (nb - 1)), dtype=np.uint8)
    for e in range(count):
        _check(_lib.qmoe_offsets_compact(_np_ptr(bo[e]), rows, nb, _np_ptr(row_off[e]),
                                         _np_ptr(blk_len[e]) if nb > 1 else None), "qmoe_offsets_compact")
    return row_off.reshape(-1), blk_len.reshape(-1)


class RvqMatrixSet:
    """`count` RVQ-coded matrices of one shape, resident on the device.  With `stages` (device uint8 per
    matrix) and `idx_base` (device int64 byte offsets), matrices may have 1 .. n_stages stages each."""

    def __init__(self, idx, codebooks, scale_f16, sign_out, sign_in, count, rows, cols, stages=None, idx_base=None,
                 n_stages=0, fmt=QMOE_VQ_RVQ):
        self.idx, self.codebooks, self.scale, self.sign_out, self.sign_in = idx, codebooks, scale_f16, sign_out, sign_in
        self.count, self.rows, self.cols = count, rows, cols
        self.stages, self.idx_base, self.n_stages, self.fmt = stages, idx_base, n_stages, fmt
        self.c = CRvqSet(_dptr(idx), _dptr(codebooks), _dptr(scale_f16), _dptr(sign_out), _dptr(sign_in), count,
                         rows, cols, _dptr(stages), _dptr(idx_base), n_stages, fmt)

    @classmethod
    def e8p_from_host(cls, codes, scale_f16, sign_out, sign_in, count, rows, cols, device="cuda"):
        """E8P set: codes uint16 [count, rows, cols/8]; the base table comes from e8p_base_table."""
        import torch

        def up(a, dt, view):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=dt).view(view).copy()).to(device)
        return cls(up(codes, np.uint16, np.int16), up(e8p_base_table(), np.uint32, np.int32),
                   up(scale_f16, np.uint16, np.int16), up(sign_out, np.int8, np.int8), up(sign_in, np.int8, np.int8),
                   count, rows, cols, fmt=QMOE_VQ_E8P)

    @classmethod
    def from_host(cls, idx, codebooks_f16, scale_f16, sign_out, sign_in, count, rows, cols, device="cuda"):
        """idx: uint8 [count, rows, cols/8, 2] (two stages each), or a list of count arrays
        [rows, cols/8, S_e] with per-matrix stage counts (each matrix's codes start 16-byte aligned)."""
        import torch

        def up(a, dt, view):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=dt).view(view).copy()).to(device)
        cb = np.ascontiguousarray(codebooks_f16, dtype=np.uint16)
        if isinstance(idx, (list, tuple)):
            st = np.array([a.shape[2] for a in idx], dtype=np.uint8)
            sizes = [a.size for a in idx]
            base = np.zeros(count, dtype=np.int64)
            off = 0
            for e, n in enumerate(sizes):
                base[e] = off
                off += (n + 15) // 16 * 16
            flat = np.zeros(max(off, 16), dtype=np.uint8)
            for e, a in enumerate(idx):
                flat[base[e]:base[e] + sizes[e]] = np.ascontiguousarray(a, dtype=np.uint8).reshape(-1)
            return cls(up(flat, np.uint8, np.uint8), up(cb, np.uint16, np.int16), up(scale_f16, np.uint16, np.int16),
                       up(sign_out, np.int8, np.int8), up(sign_in, np.int8, np.int8), count, rows, cols,
                       stages=up(st, np.uint8, np.uint8), idx_base=up(base, np.int64, np.int64), n_stages=cb.shape[0])
        return cls(up(idx, np.uint8, np.uint8), up(cb, np.uint16, np.int16),
                   up(scale_f16, np.uint16, np.int16), up(sign_out, np.int8, np.int8), up(sign_in, np.int8, np.int8),
                   count, rows, cols, n_stages=cb.shape[0])


# ================================================================ device calls
def qmoe_expert_matvec(d: Dictionary, m: MatrixSet, x, y, y_is_f32: bool = True, stream=None):
    """y[T, rows] = x[T, cols] W^T (x: int16-viewed bf16 tensor on the device)."""
    T = int(x.shape[0]) if x.dim() == 2 else 1
    _check(_lib.qmoe_expert_matvec(ctypes.byref(d.c), ctypes.byref(m.c), _dptr(x), T, _dptr(y), int(bool(y_is_f32)),
                                   _stream_ptr(stream)), "qmoe_expert_matvec")
    return y


def qmoe_decode_dense(d: Dictionary, m: MatrixSet, w_out, stream=None):
    _check(_lib.qmoe_decode_dense(ctypes.byref(d.c), ctypes.byref(m.c), _dptr(w_out), _stream_ptr(stream)),
           "qmoe_decode_dense")
    return w_out


def qmoe_route(logits, k: int, ids, gates, stream=None):
    T, E = logits.shape
    _check(_lib.qmoe_route(_dptr(logits), T, E, k, _dptr(ids), _dptr(gates), _stream_ptr(stream)), "qmoe_route")
    return ids, gates


def qmoe_bucketise(ids, E: int, counts, offsets, perm, stream=None):
    T, k = ids.shape
    _check(_lib.qmoe_bucketise(_dptr(ids), T, k, E, _dptr(counts), _dptr(offsets), _dptr(perm), _stream_ptr(stream)),
           "qmoe_bucketise")


def qmoe_pack_device_ws_size(rows: int, cols: int, block: int = 256) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.qmoe_pack_device_ws_size(rows, cols, block, ctypes.byref(n)), "qmoe_pack_device_ws_size")
    return n.value


def qmoe_pack_device(d: Dictionary, tern, codes, blk_off, workspace, block: int = 256, stream=None):
    """Device encoder: codewords and block offsets of the int8 ternary matrix `tern` (device tensor
    [rows, cols]) into `codes` (int16-viewed uint16) and `blk_off` (int32-viewed uint32, rows*nb + 1).
    The codeword count is blk_off[-1] once the stream has reached the end of the call."""
    rows, cols = tern.shape
    _check(_lib.qmoe_pack_device(ctypes.byref(d.c), _dptr(tern), rows, cols, block, _dptr(codes),
                                 int(codes.numel()), _dptr(blk_off), _dptr(workspace), int(workspace.numel()),
                                 _stream_ptr(stream)), "qmoe_pack_device")
    return codes, blk_off


def qmoe_moe_layer_ws_size(E, d_model, d_ff, T, k) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.qmoe_moe_layer_ws_size(E, d_model, d_ff, T, k, ctypes.byref(n)), "qmoe_moe_layer_ws_size")
    return n.value


QMOE_KERNEL_FLAT, QMOE_KERNEL_ROWS, QMOE_KERNEL_FLAT_L2 = 0, 1, 2
KERNEL_NAMES = {QMOE_KERNEL_FLAT: "dict_gemm_kernel", QMOE_KERNEL_ROWS: "dict_rows_kernel",
                QMOE_KERNEL_FLAT_L2: "dict_gemm_kernel"}


def qmoe_moe_layer_kernels(E, d_model, d_ff, T, k):
    """(wi kernel, wo kernel, tensor-core launch) of a qmoe_moe_layer call with these shapes."""
    wi, wo, tc = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(_lib.qmoe_moe_layer_kernels(E, d_model, d_ff, T, k, ctypes.byref(wi), ctypes.byref(wo), ctypes.byref(tc)),
           "qmoe_moe_layer_kernels")
    return wi.value, wo.value, bool(tc.value)


def qmoe_moe_layer(d: Dictionary, wi: MatrixSet, wo: MatrixSet, x, ids, gates, y, workspace, y_is_f32=True,
                   stream=None):
    T, k = ids.shape
    _check(_lib.qmoe_moe_layer(ctypes.byref(d.c), ctypes.byref(wi.c), ctypes.byref(wo.c), _dptr(x), T, k, _dptr(ids),
                               _dptr(gates), _dptr(y), int(bool(y_is_f32)), _dptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream)), "qmoe_moe_layer")
    return y


def qmoe_moe_layer_noalloc(d: Dictionary, wi: MatrixSet, wo: MatrixSet, x, ids, gates, y, y_is_f32=True,
                           stream=None):
    """qmoe_moe_layer with its scratch in the library's static device buffer (no workspace)."""
    T, k = ids.shape
    _check(_lib.qmoe_moe_layer_noalloc(ctypes.byref(d.c), ctypes.byref(wi.c), ctypes.byref(wo.c), _dptr(x), T, k,
                                       _dptr(ids), _dptr(gates), _dptr(y), int(bool(y_is_f32)), _stream_ptr(stream)),
           "qmoe_moe_layer_noalloc")
    return y


def rvq_expert_matmul_ws_size(rows, cols, T) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.rvq_expert_matmul_ws_size(rows, cols, T, ctypes.byref(n)), "rvq_expert_matmul_ws_size")
    return n.value


def rvq_expert_matmul(m: RvqMatrixSet, x, y, workspace, y_is_f32=True, stream=None):
    T = int(x.shape[0])
    _check(_lib.rvq_expert_matmul(ctypes.byref(m.c), _dptr(x), T, _dptr(y), int(bool(y_is_f32)), _dptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "rvq_expert_matmul")
    return y


def rvq_moe_layer_ws_size(E, d_model, d_ff, T, k) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.rvq_moe_layer_ws_size(E, d_model, d_ff, T, k, ctypes.byref(n)), "rvq_moe_layer_ws_size")
    return n.value


def rvq_moe_layer(gate: RvqMatrixSet, up: RvqMatrixSet, down: RvqMatrixSet, x, ids, gates, y, workspace,
                  y_is_f32=True, stream=None):
    T, k = ids.shape
    _check(_lib.rvq_moe_layer(ctypes.byref(gate.c), ctypes.byref(up.c), ctypes.byref(down.c), _dptr(x), T, k,
                              _dptr(ids), _dptr(gates), _dptr(y), int(bool(y_is_f32)), _dptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream_ptr(stream)), "rvq_moe_layer")
    return y


def rvq_decode_dense(m: RvqMatrixSet, w_out, stream=None):
    _check(_lib.rvq_decode_dense(ctypes.byref(m.c), _dptr(w_out), _stream_ptr(stream)), "rvq_decode_dense")
    return w_out


def qmoe_set_phase_events(events) -> None:
    """Install (list of torch.cuda.Event, 6..8 of them) or clear (None) the phase-event hook."""
    if not events:
        _check(_lib.qmoe_set_phase_events(None, 0), "qmoe_set_phase_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[int(e.cuda_event) for e in events])
    _check(_lib.qmoe_set_phase_events(arr, len(events)), "qmoe_set_phase_events")
