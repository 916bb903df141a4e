"""Router, expert bucketing and the MoE feed-forward layer.  Test infrastructure.

[QMoE] "Inference Execution": at run time each token's router picks an
expert and the expert's matrix-vector products run through the fused decode
kernel; experts that receive no token are skipped ("skip empty CUDA calls").
The list-buffer idea of [QMoE] "List buffer" (one flat token buffer plus
per-expert index lists) is the bucketing below: a stable counting sort of the
(token, slot) pairs by expert.

Readings where the pages are silent:
* top-k takes the k largest logits in descending order, equal logits going to
  the lower expert id;
* gates are the softmax over all E logits, read at the chosen experts, with no
  renormalisation over the k chosen ones;
* a dictionary-coded (SwitchTransformer-shaped) expert is relu(W_i x) followed
  by W_o, with no bias; the intermediate h is rounded to bfloat16, because
  activations travel in bfloat16;
* a token's output is the sum over its k slots, in slot order, of gate * o.
"""
from __future__ import annotations

import numpy as np


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits: for |v| in [2**(e-1), 2**e) the spacing
    is 2**(e-8), so v * 2**(8-e) is rounded to an integer (numpy's rint rounds
    half to even) and scaled back.  The exponent is clamped at bfloat16's
    smallest normal binade so tiny values land on the subnormal grid 2**-133.
    """
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    e = np.maximum(e, -125)
    return np.ldexp(np.rint(np.ldexp(v, 8 - e)), e - 8)


def route(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-k expert ids int32 [T, k] and softmax gates float64 [T, k]."""
    logits = np.asarray(logits)
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("k out of range")
    ids = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        row = logits[t].astype(np.float64)
        # stable sort on -logit keeps the lower id first among equal logits
        order = np.argsort(-row, kind="stable")[:k]
        m = row.max()
        z = np.exp(row - m).sum()
        ids[t] = order
        gates[t] = np.exp(row[order] - m) / z
    return ids, gates


def bucketise(ids: np.ndarray, E: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Stable counting sort of flat slots (t*k + j) by expert.

    Returns counts int32 [E], offsets int32 [E+1] (exclusive prefix sum) and
    perm int32 [T*k]: perm[offsets[e] : offsets[e+1]] lists, in increasing
    order, the flat slots routed to expert e.
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    cursor = offsets[:-1].copy()
    perm = np.empty(flat.size, dtype=np.int64)
    for slot, e in enumerate(flat):
        perm[cursor[e]] = slot
        cursor[e] += 1
    return counts.astype(np.int32), offsets.astype(np.int32), perm.astype(np.int32)


def relu_expert(x: np.ndarray, w_i: np.ndarray, w_o: np.ndarray) -> np.ndarray:
    """One SwitchTransformer-shaped expert on rows of x: W_o . bf16(relu(W_i . x))."""
    h = np.maximum(np.asarray(x, np.float64) @ w_i.T, 0.0)
    return bf16_round(h) @ w_o.T


def moe_layer(x: np.ndarray, ids: np.ndarray, gates: np.ndarray, expert_fn, d_out: int) -> np.ndarray:
    """y[t] = sum_j gates[t, j] * expert_fn(ids[t, j], x[t]) with slots summed in order.

    ``expert_fn(e, xs)`` maps rows xs [n, d] to expert e's outputs [n, d_out].  It
    is called once per used expert with all of that expert's tokens (each row is
    computed independently, so the grouping does not change any value).
    """
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    T, k = ids.shape
    out_slot = np.zeros((T, k, d_out), dtype=np.float64)
    for e in np.unique(ids):
        where = np.argwhere(ids == e)
        out_slot[where[:, 0], where[:, 1]] = expert_fn(int(e), x[where[:, 0]])
    y = np.zeros((T, d_out), dtype=np.float64)
    for j in range(k):
        y = y + np.asarray(gates, dtype=np.float64)[:, j:j + 1] * out_slot[:, j]
    return y
