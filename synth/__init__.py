"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no dictionary, no encoding, no product, no routing
decision, no transform).  Both the CPU oracle and the CUDA path take their
inputs from here, so the two never feed each other.

Ternary expert weights are drawn from a counter-based generator so that any
row of any expert matrix can be regenerated on its own (the oracle checks
sampled rows of layers too large to regenerate whole) and so that the native
twin in ``synth/csrc/synth.cpp`` can regenerate the 52-billion-weight
c2048-shaped layer in seconds.  The generator is SplitMix64 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014; the
64-bit finaliser with shifts 30/27/31), used in counter mode: output number
``i`` of the stream seeded with ``key`` is ``mix(key + (i + 1) * gamma)``.

Everything else (scales, activations, router logits, RVQ weights and sign
vectors) comes from numpy's seeded ``default_rng`` and is generated on the
host, where it is cheap at every size used here.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
M64 = (1 << 64) - 1

# stream tags: one per kind of drawn quantity
TAG_TERNARY = 1
TAG_SCALE = 2
TAG_X = 3
TAG_LOGITS = 4
TAG_ZIPF = 5
TAG_RVQ_W = 6
TAG_RVQ_SIGN = 7
TAG_KMEANS = 8
TAG_ZIPF_RANK = 9
TAG_E8P = 10


def splitmix64_scalar(key: int, idx: int) -> int:
    """Output ``idx`` (0-based) of the SplitMix64 stream seeded with ``key``."""
    z = (key + (idx + 1) * GAMMA) & M64
    z = ((z ^ (z >> 30)) * MIX1) & M64
    z = ((z ^ (z >> 27)) * MIX2) & M64
    return z ^ (z >> 31)


def splitmix64(key: int, idx: np.ndarray) -> np.ndarray:
    """Vectorised :func:`splitmix64_scalar` over an array of stream indices."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx + np.uint64(1)) * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
        z = z ^ (z >> np.uint64(31))
    return z


def stream_key(seed: int, tag: int, expert: int = 0, matrix: int = 0) -> int:
    """Key of the stream for one (configuration seed, quantity, expert, matrix)."""
    assert 0 <= expert < (1 << 32) and 0 <= matrix < 256 and 0 <= tag < 256
    return splitmix64_scalar(seed, (tag << 48) | (expert << 8) | matrix)


def zero_threshold(p0: float) -> int:
    """32-bit threshold: a weight is zero when the high word of its draw is below it."""
    t = int(round(p0 * 4294967296.0))
    assert 0 <= t <= 0xFFFFFFFF
    return t


def ternary_rows(seed: int, expert: int, matrix: int, cols: int, p0: float,
                 row_start: int, row_count: int) -> np.ndarray:
    """Rows ``[row_start, row_start+row_count)`` of a ternary matrix, int8 in {-1,0,+1}.

    Weight (r, c) uses stream index ``r*cols + c``: zero when the draw's high
    32 bits are below :func:`zero_threshold`, otherwise +1 if the draw is odd
    and -1 if it is even.  P(0) = threshold / 2**32, P(+1) = P(-1).
    """
    key = stream_key(seed, TAG_TERNARY, expert, matrix)
    idx = (np.arange(row_start, row_start + row_count, dtype=np.uint64)[:, None] * np.uint64(cols)
           + np.arange(cols, dtype=np.uint64)[None, :])
    u = splitmix64(key, idx)
    hi = (u >> np.uint64(32)).astype(np.uint64)
    zero = hi < np.uint64(zero_threshold(p0))
    sign = np.where((u & np.uint64(1)) == np.uint64(1), 1, -1).astype(np.int8)
    out = np.where(zero, np.int8(0), sign).astype(np.int8)
    return out


def ternary_matrix(seed: int, expert: int, matrix: int, rows: int, cols: int, p0: float) -> np.ndarray:
    return ternary_rows(seed, expert, matrix, cols, p0, 0, rows)


def f16_bits(values: np.ndarray) -> np.ndarray:
    """Round float64 values to IEEE binary16 (numpy rounds to nearest even) and return the bits."""
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_bits_from_f32(values: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16, nearest-even, and return the 16-bit patterns."""
    b = np.ascontiguousarray(values, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def row_scales(seed: int, expert: int, matrix: int, rows: int) -> np.ndarray:
    """Per-row fp16 scale bits, U(0.01, 0.05) rounded to fp16."""
    key = stream_key(seed, TAG_SCALE, expert, matrix)
    u = splitmix64(key, np.arange(rows, dtype=np.uint64))
    unit = (u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return f16_bits(0.01 + 0.04 * unit)


def activations_bf16(seed: int, T: int, d: int, tag: int = TAG_X) -> np.ndarray:
    """T x d bf16 bit patterns of N(0,1) draws (float64 -> float32 -> bf16, nearest even)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, tag, T, d]))
    v = rng.standard_normal((T, d)).astype(np.float32)
    return bf16_bits_from_f32(v).reshape(T, d)


def zipf_logits(seed: int, T: int, E: int, s: float) -> np.ndarray:
    """Router logits whose top-k picks experts without replacement with P ~ rank**-s.

    log pi_rank + Gumbel(0,1) noise (the Gumbel-top-k construction); ranks map
    to expert ids through a seeded permutation.  float32 [T, E].
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, TAG_ZIPF, T, E]))
    perm = rng.permutation(E)             # perm[rank-1] = expert id
    ranks = np.arange(1, E + 1, dtype=np.float64)
    logpi = -s * np.log(ranks)
    logpi -= np.log(np.exp(logpi).sum())
    base = np.empty(E, dtype=np.float64)
    base[perm] = logpi
    u = rng.random((T, E))
    u = np.clip(u, 1e-300, None)
    gumbel = -np.log(-np.log(u))
    return (base[None, :] + gumbel).astype(np.float32)


def zipf_popularity(seed: int, E: int, s: float) -> np.ndarray:
    """Selection weights pi_e ~ rank**-s of a layer's experts, summing to 1; ranks map to
    expert ids through a seeded permutation that belongs to the layer (not to a batch)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, TAG_ZIPF_RANK, E]))
    perm = rng.permutation(E)             # perm[rank-1] = expert id
    pi = np.arange(1, E + 1, dtype=np.float64) ** -s
    pi /= pi.sum()
    out = np.empty(E, dtype=np.float64)
    out[perm] = pi
    return out


def zipf_layer_logits(seed: int, T: int, E: int, s: float) -> np.ndarray:
    """Router logits log pi_e + Gumbel(0,1) noise with the layer's fixed popularity
    (zipf_popularity): top-k picks experts without replacement with P ~ pi.  float32 [T, E]."""
    logpi = np.log(zipf_popularity(seed, E, s))
    rng = np.random.default_rng(np.random.SeedSequence([seed, TAG_ZIPF_RANK, T, E]))
    u = np.clip(rng.random((T, E)), 1e-300, None)
    return (logpi[None, :] - np.log(-np.log(u))).astype(np.float32)


def normal_logits(seed: int, T: int, E: int) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence([seed, TAG_LOGITS, T, E]))
    return rng.standard_normal((T, E)).astype(np.float32)


def rvq_weight(seed: int, expert: int, matrix: int, rows: int, cols: int, std: float = 0.02) -> np.ndarray:
    """Dense float64 weight ~ N(0, std^2) for one RVQ-coded matrix (rows = outputs)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, TAG_RVQ_W, expert, matrix]))
    return rng.normal(0.0, std, size=(rows, cols))


def e8p_random_matrix(seed: int, expert: int, matrix: int, rows: int, cols: int, std: float = 0.02):
    """Uniform 16-bit code words uint16 [rows, cols/8] (every word is an E8P code word) and fp16
    row-scale bits [rows] drawn from U(0.5, 1.5) * std / 1.094 (the scale a N(0, std^2) weight
    gets), for parity cases that need no encoder."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, TAG_E8P, expert, matrix]))
    codes = rng.integers(0, 1 << 16, size=(rows, cols // 8)).astype(np.uint16)
    scale = (rng.uniform(0.5, 1.5, size=rows) * std / 1.094).astype(np.float16).view(np.uint16)
    return codes, scale


def rvq_signs(seed: int, expert: int, matrix: int, n_out: int, n_in: int) -> tuple[np.ndarray, np.ndarray]:
    """Random sign diagonals (output side, input side) as int8 +-1."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, TAG_RVQ_SIGN, expert, matrix]))
    s_out = (rng.integers(0, 2, size=n_out) * 2 - 1).astype(np.int8)
    s_in = (rng.integers(0, 2, size=n_in) * 2 - 1).astype(np.int8)
    return s_out, s_in


# --------------------------------------------------------------------------
# Workload shapes (synthetic stand-ins for the SwitchTransformer and OLMoE
# expert layers that the QMoE and cache-amplification papers measure on).
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class DictLayer:
    name: str
    E: int
    d_model: int
    d_ff: int
    p0: float
    seed: int
    top_k: int
    routing: str          # "normal" (logits N(0,1)) or "zipf"
    zipf_s: float
    tokens: tuple


@dataclasses.dataclass(frozen=True)
class LinearCfg:
    name: str
    rows: int
    cols: int
    p0: float
    seed: int
    tokens: tuple


@dataclasses.dataclass(frozen=True)
class RvqLayer:
    name: str
    E: int
    d_model: int
    d_ff: int
    seed: int
    top_k: int
    zipf_s: float
    tokens: tuple
    vec_dim: int = 8
    stages: int = 2
    codebook_size: int = 256
    # frequency-conditioned stages: router with the layer's fixed Zipf popularity, and per-expert
    # stage counts stages-1 / stages / stages+1 for the least / middle / most popular thirds
    freq_stages: bool = False
    # "rvq": residual k-means codebooks; "e8p": the E8P lattice code (one 16-bit word per 8 weights)
    vq: str = "rvq"


LINEAR_1024x4096 = LinearCfg("linear-1024x4096-p0.89", 1024, 4096, 0.89, 0, (1, 8, 32))
SWITCH_BASE_128 = DictLayer("switch-base-128", 128, 768, 3072, 0.857, 1, 1, "normal", 0.0, (512,))
SWITCH_LARGE_128 = DictLayer("switch-large-128", 128, 1024, 4096, 0.87, 2, 1, "zipf", 1.1, (2048,))
SWITCH_C2048 = DictLayer("switch-c2048", 2048, 2080, 6144, 0.886, 3, 1, "zipf", 1.0, (1, 64, 4096))
OLMOE_RVQ = RvqLayer("olmoe-rvq-2bit", 64, 2048, 1024, 4, 8, 0.9, (1, 32))
OLMOE_RVQ_FREQ = RvqLayer("olmoe-rvq-freq-2bit", 64, 2048, 1024, 4, 8, 0.9, (1, 32), freq_stages=True)
OLMOE_E8P = RvqLayer("olmoe-e8p-2bit", 64, 2048, 1024, 4, 8, 0.9, (1, 32), vq="e8p")

# matrix ids inside a dictionary-coded expert
WI, WO = 0, 1
# matrix ids inside an RVQ-coded SwiGLU expert
GATE, UP, DOWN = 0, 1, 2


def dict_matrix_shape(cfg: DictLayer, matrix: int) -> tuple[int, int]:
    """(rows, cols) with rows = output features: wi is d_ff x d_model, wo is d_model x d_ff."""
    return (cfg.d_ff, cfg.d_model) if matrix == WI else (cfg.d_model, cfg.d_ff)


def rvq_matrix_shape(cfg: RvqLayer, matrix: int) -> tuple[int, int]:
    return (cfg.d_ff, cfg.d_model) if matrix in (GATE, UP) else (cfg.d_model, cfg.d_ff)


def layer_logits(cfg, T: int) -> np.ndarray:
    if getattr(cfg, "routing", "zipf") == "normal":
        return normal_logits(cfg.seed, T, cfg.E)
    if getattr(cfg, "freq_stages", False):
        return zipf_layer_logits(cfg.seed, T, cfg.E, cfg.zipf_s)
    return zipf_logits(cfg.seed, T, cfg.E, cfg.zipf_s)


def layer_tokens(cfg, T: int) -> np.ndarray:
    return activations_bf16(cfg.seed, T, cfg.d_model)
