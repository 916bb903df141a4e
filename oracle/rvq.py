"""Randomized Hadamard transform + residual vector quantisation.  Test infrastructure.

[QCA] section "Codec", paragraph "Incoherence processing": a two-sided
randomized Hadamard transform with random sign diagonals and the normalised
Walsh-Hadamard matrix, undone at run time on the activations,
y = D_l H_o (W' (H_i D_r x)).  The page's weight-side formula and its runtime
formula disagree about the order of signs and Hadamards; the runtime formula is
followed (it also matches the sign order of [M8.5] 0x06H "Runtime Trace":
input signs before the Hadamard, output signs after it), so that

    W' = H_o D_l W D_r H_i   and   W = D_l H_o W' H_i D_r.

[QCA] "Residual vector quantization": rows of W' are normalised by an fp16
per-row RMS scale and cut into d-dimensional subvectors; each subvector is coded
by S residual stages, each an 8-bit index into a 256-entry codebook; stage s's
codebook is k-means-fit on the residual left by earlier stages.  The
workloads here use d = 8 and S = 2 (2 bits per weight) with fp16 codebooks and
one codebook set per layer.  [QCA] "Frequency-Conditioned Bit Allocation":
with an average of S stages, the most-activated third of a layer's experts get
S + 1 stages and the least-activated third S - 1 (the page's rank-based
approximation of the reverse-water-filling rates r_e = r + log2(pi_e / pi~) / 2),
so the mean rate is unchanged; an expert with S_e stages uses the first S_e
codebooks of the layer's set.

k-means follows the conventions of [M8.5] 0x02B/0x02D: nearest-centroid ties
go to the lowest index; a cluster that receives no point keeps its previous
centroid; the final assignment is made against the final (here fp16-rounded)
codebook.  Initialisation (a seeded sample of distinct vectors) and the stop
rule (25 Lloyd iterations or stable assignments) are readings, as the pages
leave them open.

The decoded rotated-basis weight is defined in float32 as
fp32(s_r) * (fp32(C1[i1]) + fp32(C2[i2])): one add, then one multiply, each
rounded to nearest even; with S stages the adds run left to right,
((C1 + C2) + C3) ..., and one stage is fp32(s_r) * fp32(C1[i1]).  The fast Walsh-Hadamard transform is the O(n log n)
butterfly of [M8.5] 0x06C.
"""
from __future__ import annotations

import numpy as np

from .moe import bf16_round


# ------------------------------------------------------------------ Hadamard
def sylvester(n: int) -> np.ndarray:
    """Normalised Sylvester-Hadamard matrix H_n (n a power of two), H_n @ H_n = I."""
    if n < 1 or n & (n - 1):
        raise ValueError("n must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(n)


def fwht(v: np.ndarray, axis: int = -1) -> np.ndarray:
    """Normalised fast Walsh-Hadamard transform along ``axis`` (float64 butterfly)."""
    a = np.moveaxis(np.array(v, dtype=np.float64), axis, -1)
    n = a.shape[-1]
    if n < 1 or n & (n - 1):
        raise ValueError("length must be a power of two")
    h = 1
    while h < n:
        a = a.reshape(a.shape[:-1] + (n // (2 * h), 2, h))
        top = a[..., 0, :] + a[..., 1, :]
        bot = a[..., 0, :] - a[..., 1, :]
        a = np.stack([top, bot], axis=-2).reshape(a.shape[:-3] + (n,))
        h *= 2
    a = a / np.sqrt(n)
    return np.moveaxis(a, -1, axis)


def rotate_weight(w: np.ndarray, sign_out: np.ndarray, sign_in: np.ndarray) -> np.ndarray:
    """W' = H_o D_l W D_r H_i."""
    dw = np.asarray(w, np.float64) * np.asarray(sign_out, np.float64)[:, None] * np.asarray(sign_in, np.float64)[None, :]
    return fwht(fwht(dw, axis=0), axis=1)


def unrotate_weight(wr: np.ndarray, sign_out: np.ndarray, sign_in: np.ndarray) -> np.ndarray:
    """W = D_l H_o W' H_i D_r."""
    w = fwht(fwht(np.asarray(wr, np.float64), axis=0), axis=1)
    return w * np.asarray(sign_out, np.float64)[:, None] * np.asarray(sign_in, np.float64)[None, :]


# ------------------------------------------------------------ vector quantiser
def nearest(u: np.ndarray, cb: np.ndarray, chunk: int = 8192) -> np.ndarray:
    """Index of the nearest codeword for every row of u (squared Euclidean distance).

    The distance is accumulated coordinate by coordinate, j = 0 .. d-1, in
    float64; ties go to the lowest index (numpy's argmin returns the first).
    """
    u = np.asarray(u, dtype=np.float64)
    cb = np.asarray(cb, dtype=np.float64)
    out = np.empty(u.shape[0], dtype=np.int64)
    for lo in range(0, u.shape[0], chunk):
        part = u[lo:lo + chunk]
        dist = np.zeros((part.shape[0], cb.shape[0]))
        for j in range(u.shape[1]):
            diff = part[:, j, None] - cb[None, :, j]
            dist = dist + diff * diff
        out[lo:lo + chunk] = np.argmin(dist, axis=1)
    return out


def kmeans(vectors: np.ndarray, k: int, iters: int, seed: int) -> np.ndarray:
    """Lloyd's k-means (float64 centroids) from a seeded sample of k distinct vectors."""
    v = np.asarray(vectors, dtype=np.float64)
    uniq = np.unique(v, axis=0)
    if uniq.shape[0] < k:
        raise ValueError("fewer distinct vectors than centroids")
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x6B6D]))
    cent = uniq[np.sort(rng.choice(uniq.shape[0], size=k, replace=False))].copy()
    assign = None
    for _ in range(iters):
        new = nearest(v, cent)
        if assign is not None and np.array_equal(new, assign):
            break
        assign = new
        for j in range(k):
            members = v[assign == j]
            if members.shape[0]:
                cent[j] = members.mean(axis=0)
    return cent


def f16_round(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float16).astype(np.float64)


def row_scale_f16(wr: np.ndarray) -> np.ndarray:
    """Per-row fp16 RMS scale bits of the rotated weight.

    The sum of squares is taken left to right (cumulative sum), then divided by
    the row length; reading of "fp16 per-row RMS scale" ([QCA] "Residual vector
    quantization") with a fixed summation order so that any exact encoder can
    reproduce the scale bit for bit.
    """
    sq = np.asarray(wr, np.float64) ** 2
    rms = np.sqrt(np.cumsum(sq, axis=1)[:, -1] / wr.shape[1])
    return rms.astype(np.float16).view(np.uint16)


def normalised_vectors(wr: np.ndarray, scale_bits: np.ndarray, d: int) -> np.ndarray:
    """u = W' / s_r cut into consecutive d-input vectors of each row: [rows * cols/d, d]."""
    s = np.asarray(scale_bits, np.uint16).view(np.float16).astype(np.float64)
    rows, cols = wr.shape
    if cols % d:
        raise ValueError("row length must be a multiple of the vector dimension")
    return (np.asarray(wr, np.float64) / s[:, None]).reshape(rows * (cols // d), d)


def fit_codebooks(vectors: np.ndarray, k: int = 256, iters: int = 25, seed: int = 0, stages: int = 2) -> np.ndarray:
    """`stages` residual stages: fp16 codebooks [stages, k, d] as float64 values; stage s (seed + s)
    is fit on what the earlier stages leave, each vector taking its nearest rounded codeword."""
    cbs = []
    resid = np.asarray(vectors, np.float64)
    for st in range(stages):
        c = f16_round(kmeans(resid, k, iters, seed + st))
        resid = resid - c[nearest(resid, c)]
        cbs.append(c)
    return np.stack(cbs)


def encode(wr: np.ndarray, codebooks: np.ndarray, d: int = 8, stages: int | None = None):
    """Indices uint8 [rows, cols/d, S] and fp16 scale bits [rows] of a rotated weight, S = stages
    (default: every codebook of the set): stage s takes the codeword nearest to what stages
    0 .. s-1 leave of u."""
    rows, cols = wr.shape
    cb = np.asarray(codebooks, np.float64)
    n_st = cb.shape[0] if stages is None else stages
    if not 1 <= n_st <= cb.shape[0]:
        raise ValueError("stage count outside 1 .. number of codebooks")
    scale = row_scale_f16(wr)
    resid = normalised_vectors(wr, scale, d)
    idx = []
    for st in range(n_st):
        i = nearest(resid, cb[st])
        idx.append(i)
        resid = resid - cb[st][i]
    return np.stack(idx, axis=1).astype(np.uint8).reshape(rows, cols // d, n_st), scale


def decode(idx: np.ndarray, codebooks_f16_bits: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """Decoded rotated-basis weight, float32 [rows, cols]:
    fp32(s) * (((fp32(C1[i1]) + fp32(C2[i2])) + fp32(C3[i3])) ...), as many stages as idx holds."""
    idx = np.asarray(idx)
    rows, nv, n_st = idx.shape
    cb = np.asarray(codebooks_f16_bits, np.uint16).view(np.float16).astype(np.float32)
    d = cb.shape[2]
    s = np.asarray(scale_bits, np.uint16).view(np.float16).astype(np.float32)
    summed = cb[0][idx[:, :, 0]]
    for st in range(1, n_st):
        summed = summed + cb[st][idx[:, :, st]]                      # float32 adds, left to right
    w = s[:, None, None] * summed                                    # float32 multiply
    return w.reshape(rows, nv * d).astype(np.float32)


def stage_allocation(popularity: np.ndarray, s_bar: int) -> np.ndarray:
    """Stages per expert ([QCA] "Frequency-Conditioned Bit Allocation", rank-based form):
    the floor(E/3) most popular experts get s_bar + 1, the floor(E/3) least popular s_bar - 1, the
    rest s_bar.  Equal popularity ranks the lower expert id as more popular."""
    pop = np.asarray(popularity, np.float64)
    E = pop.shape[0]
    third = E // 3
    order = sorted(range(E), key=lambda e: (-pop[e], e))
    st = np.full(E, s_bar, dtype=np.int64)
    st[order[:third]] = s_bar + 1
    st[order[E - third:]] = s_bar - 1
    return st


def linear(x: np.ndarray, w_dec: np.ndarray, sign_out: np.ndarray, sign_in: np.ndarray) -> np.ndarray:
    """y = D_l H_o (W'_hat (H_i D_r x)) for rows of x, float64."""
    x = np.asarray(x, np.float64)
    xr = fwht(x * np.asarray(sign_in, np.float64)[None, :], axis=1)
    yr = xr @ np.asarray(w_dec, np.float64).T
    return fwht(yr, axis=1) * np.asarray(sign_out, np.float64)[None, :]


def silu(g: np.ndarray) -> np.ndarray:
    g = np.asarray(g, np.float64)
    return g / (1.0 + np.exp(-g))


def swiglu_expert(x: np.ndarray, gate, up, down) -> np.ndarray:
    """OLMoE-shaped expert: down(bf16(silu(gate(x)) * up(x))); each of gate/up/down is
    a tuple (decoded W', sign_out, sign_in)."""
    g = linear(x, *gate)
    u = linear(x, *up)
    h = bf16_round(silu(g) * u)
    return linear(h, *down)
