"""Oracle parity of the layer calls at the full shapes of the five workloads.

Every layer here is built at its workload's own sizes (experts, d_model, d_ff,
token batch, zero probability, routing) from the seeded generators, encoded by
the library's host encoder and run through the C ABI exactly as the benchmark
runs it.  The expected values come from the oracle alone: the float64 MoE layer
of ``oracle.moe`` over the seeded weights s_r * t_rc (dictionary path), or the
oracle's own residual-VQ encoding, decoding and SwiGLU expert (VQ path).  At
these sizes the oracle checks sampled tokens (chosen to cover every expert load
class: the tensor-core experts, several-token chunks, single tokens) and
sampled experts' decoded weights, which must be bit-exact.

Tolerance: fp32-mode outputs, max|y - y_ref| / max|y_ref| per token <= 2e-3.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest

import synth
from oracle import moe as M
from oracle import products as P
from oracle import rvq as R

from helpers import bf16_tensor, fill_ternary, seeded_weights

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
TOL = 2e-3

Q = pytest.importorskip("decode_matvec_gb300")
from decode_matvec_gb300.layers import DictLayer, pack_rvq_set  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda")


def build_dict_layer(cfg, dev, tern_fns=None):
    """The workload's layer on the device; tern_fns optionally overrides (wi_fill, wo_fill)."""
    def tern(m):
        return lambda e, out: fill_ternary(cfg.seed, e, m, cfg.p0, out)

    def scale(m):
        rows = synth.dict_matrix_shape(cfg, m)[0]
        return lambda e: synth.row_scales(cfg.seed, e, m, rows)

    fi, fo = tern_fns or (tern(synth.WI), tern(synth.WO))
    return DictLayer(cfg.p0, cfg.E, cfg.d_model, cfg.d_ff, fi, fo, scale(synth.WI), scale(synth.WO), device=dev)


def expert_view(ms, host, e):
    """A one-matrix set for expert e of a device matrix set (views into the same buffers)."""
    return ms.expert(e, host.code_base)


class SeededExperts:
    """The oracle's float64 expert weights from the seeded generators, built on demand (the last two
    kept: a c2048-shaped expert is 200 MB in float64)."""

    def __init__(self, cfg, weights_fn=None):
        self.cfg, self.cache = cfg, {}
        self.weights_fn = weights_fn or (lambda e, m, r, c: seeded_weights(cfg.seed, e, m, r, c, cfg.p0))

    def __call__(self, e):
        if e not in self.cache:
            if len(self.cache) >= 2:
                self.cache.pop(next(iter(self.cache)))
            self.cache[e] = tuple(self.weights_fn(e, m, *synth.dict_matrix_shape(self.cfg, m))
                                  for m in (synth.WI, synth.WO))
        return self.cache[e]


def run_dict_layer(layer, x_bits, ids, gates, dev, y_is_f32=True):
    T, k = ids.shape
    ws = torch.empty(Q.qmoe_moe_layer_ws_size(layer.E, layer.d_model, layer.d_ff, T, k), dtype=torch.uint8,
                     device=dev)
    y = torch.empty((T, layer.d_model), dtype=torch.float32 if y_is_f32 else torch.int16, device=dev)
    Q.qmoe_moe_layer(layer.dictionary, layer.wi, layer.wo, bf16_tensor(x_bits), ids, gates, y, ws,
                     y_is_f32=y_is_f32)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    return y


def routed(cfg, T, dev):
    """Device routing of the workload's logits, checked equal to the oracle router; returns the
    device (ids, gates) and the oracle's (ids, gates)."""
    lg = synth.layer_logits(cfg, T)
    ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, cfg.top_k), dtype=torch.float32, device=dev)
    Q.qmoe_route(torch.from_numpy(lg).to(dev), cfg.top_k, ids, gates)
    rid, rg = M.route(lg, cfg.top_k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(gates.cpu().numpy(), rg, rtol=1e-5, atol=1e-7)
    return ids, gates, rid, rg


def check_tokens(y, x_bits, rid, rg, tokens, experts, d_model):
    """Per-token normwise error of the fp32-mode output against the float64 oracle layer."""
    x = synth.bf16_to_f64(x_bits)
    sel = np.asarray(sorted(set(int(t) for t in tokens)))
    ref = M.moe_layer(x[sel], rid[sel], rg[sel], lambda e, xs: M.relu_expert(xs, *experts(e)), d_model)
    got = y.cpu().numpy().astype(np.float64)[sel]
    worst = max(P.normwise_rel_err(got[i], ref[i]) for i in range(len(sel)))
    assert worst < TOL, worst
    return worst


def tokens_by_load(rid, picks_per_class=2):
    """Sampled tokens covering every expert load class of a top-1 batch: the busiest expert, experts
    with >= 32 tokens (tensor-core kernel), 9-31, 5-8, 3-4, 2 and 1 tokens."""
    ids = rid[:, 0]
    counts = np.bincount(ids)
    out = [int(np.nonzero(ids == np.argmax(counts))[0][0])]
    for lo, hi in ((32, 1 << 30), (9, 31), (5, 8), (3, 4), (2, 2), (1, 1)):
        experts = np.nonzero((counts >= lo) & (counts <= hi))[0][:picks_per_class]
        for e in experts:
            toks = np.nonzero(ids == e)[0]
            out += [int(toks[0]), int(toks[-1])]
    return sorted(set(out))


def check_decoded(layer, e, experts):
    """qmoe_decode_dense of expert e's wi and wo equals the seeded weights exactly."""
    for ms, host, ref in ((layer.wi, layer.wi_host, experts(e)[0]), (layer.wo, layer.wo_host, experts(e)[1])):
        w = torch.empty((ms.rows, ms.cols), dtype=torch.float32, device=ms.codes.device)
        Q.qmoe_decode_dense(layer.dictionary, expert_view(ms, host, e), w)
        assert Q.qmoe_check_status() == Q.QMOE_OK
        assert np.array_equal(w.cpu().numpy().astype(np.float64), ref)


# ------------------------------------------------------------------ switch-base-128 and switch-large-128
@pytest.mark.parametrize("cfg", [synth.SWITCH_BASE_128, synth.SWITCH_LARGE_128], ids=lambda c: c.name)
def test_switch_layers_full_shape_every_token(dev, cfg):
    """switch-base-128 (p0 0.857: entries with four nonzeros in every warp window, near-uniform
    top-1) at T=512 and switch-large-128 (p0 0.87, Zipf(1.1): skewed loads up to hundreds of
    tokens on one expert) at T=2048; every token is checked."""
    layer = build_dict_layer(cfg, dev)
    experts = SeededExperts(cfg)
    for T in cfg.tokens:
        ids, gates, rid, rg = routed(cfg, T, dev)
        xb = synth.layer_tokens(cfg, T)
        y = run_dict_layer(layer, xb, ids, gates, dev)
        check_tokens(y, xb, rid, rg, range(T), experts, cfg.d_model)
        counts = np.bincount(rid[:, 0], minlength=cfg.E)
        for e in (int(np.argmax(counts)), int(np.nonzero(counts == counts[counts > 0].min())[0][0])):
            check_decoded(layer, e, experts)


# ------------------------------------------------------------------ switch-c2048
@pytest.fixture(scope="module")
def c2048(dev):
    cfg = synth.SWITCH_C2048
    layer = build_dict_layer(cfg, dev)
    yield cfg, layer, SeededExperts(cfg)
    del layer
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [1, 64])
def test_c2048_full_shape_small_batches(dev, c2048, T):
    cfg, layer, experts = c2048
    ids, gates, rid, rg = routed(cfg, T, dev)
    xb = synth.layer_tokens(cfg, T)
    y = run_dict_layer(layer, xb, ids, gates, dev)
    check_tokens(y, xb, rid, rg, range(T), experts, cfg.d_model)
    # bf16 output: the fp32 result rounded to nearest even
    yb = run_dict_layer(layer, xb, ids, gates, dev, y_is_f32=False)
    assert np.array_equal(yb.cpu().numpy().view(np.uint16), synth.bf16_bits_from_f32(y.cpu().numpy()))


def test_c2048_full_shape_t4096(dev, c2048):
    """The benchmark's step: sampled tokens of every load class, decoded weights of the busiest
    expert and of a one-token expert."""
    cfg, layer, experts = c2048
    T = 4096
    ids, gates, rid, rg = routed(cfg, T, dev)
    xb = synth.layer_tokens(cfg, T)
    y = run_dict_layer(layer, xb, ids, gates, dev)
    toks = tokens_by_load(rid)
    assert len(toks) >= 10
    check_tokens(y, xb, rid, rg, toks, experts, cfg.d_model)
    counts = np.bincount(rid[:, 0], minlength=cfg.E)
    check_decoded(layer, int(np.argmax(counts)), experts)
    check_decoded(layer, int(np.nonzero(counts == 1)[0][0]), experts)


def test_c2048_shaped_token_counts_around_tensor_core_threshold(dev):
    """Six c2048-shaped experts (d_model 2080, d_ff 6144) with 31, 32, 33, 3, 300 and 7 tokens routed
    by hand (T = 406, k = 1, enough slots for the tensor-core kernel): its threshold from both sides,
    a 300-token expert split into two tensor-core jobs (at most 256 tokens each), several-token chunks
    with odd remainders on the CUDA-core kernels (wi and wo token classes of the full-size layer)."""
    cfg = synth.SWITCH_C2048
    import dataclasses
    small = dataclasses.replace(cfg, E=6)
    layer = build_dict_layer(small, dev)
    experts = SeededExperts(small)
    counts = [31, 32, 33, 3, 300, 7]
    rid = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(counts)])
    rid = rid[np.random.default_rng(5).permutation(rid.size)].reshape(-1, 1)
    rg = np.random.default_rng(6).uniform(0.2, 1.0, size=rid.shape)
    T = rid.shape[0]
    xb = synth.activations_bf16(17, T, cfg.d_model)
    y = run_dict_layer(layer, xb, torch.from_numpy(rid).to(dev), torch.from_numpy(rg.astype(np.float32)).to(dev), dev)
    check_tokens(y, xb, rid, rg.astype(np.float32).astype(np.float64), range(T), experts, cfg.d_model)


@pytest.mark.parametrize("p0", [0.857, 0.886])
def test_degenerate_experts_in_a_layer_call(dev, p0):
    """switch-base-shaped experts (d_model 768, d_ff 3072) with degenerate weights in one layer call:
    expert 0 all zero (every codeword a run of zeros), expert 1 with no zero at all (the shortest
    codewords: two-nonzero pairs at p0 0.886, four-nonzero entries taken through the escape path at
    p0 0.857, the most codewords a block can have), expert 2 drawn as usual."""
    import dataclasses
    cfg = dataclasses.replace(synth.SWITCH_BASE_128, E=3, p0=p0)

    def fill(m):
        def f(e, out):
            if e == 0:
                out[:] = 0
            elif e == 1:
                rng = np.random.default_rng(100 + m)
                out[:] = rng.integers(0, 2, size=out.shape, dtype=np.int8) * 2 - 1
            else:
                fill_ternary(cfg.seed, e, m, cfg.p0, out)
            return out
        return f

    layer = build_dict_layer(cfg, dev, (fill(synth.WI), fill(synth.WO)))

    def weights(e, m, rows, cols):
        t = fill(m)(e, np.empty((rows, cols), np.int8)).astype(np.float64)
        return t * synth.f16_to_f64(synth.row_scales(cfg.seed, e, m, rows))[:, None]

    experts = SeededExperts(cfg, weights)
    # each degenerate expert once on the tensor-core kernel (200 tokens) and once on the CUDA-core one
    # (256 slots: enough for the tensor-core kernel to run)
    for counts in ((200, 5, 51), (5, 200, 51)):
        rid = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(counts)])
        rid = rid[np.random.default_rng(7).permutation(rid.size)].reshape(-1, 1)
        rg = np.ones(rid.shape, np.float32)
        xb = synth.activations_bf16(19, rid.shape[0], cfg.d_model)
        y = run_dict_layer(layer, xb, torch.from_numpy(rid).to(dev), torch.from_numpy(rg).to(dev), dev)
        assert np.all(y.cpu().numpy()[rid[:, 0] == 0] == 0.0)
        check_tokens(y, xb, rid, rg.astype(np.float64), np.nonzero(rid[:, 0] != 0)[0], experts, cfg.d_model)
    for e in range(3):
        check_decoded(layer, e, experts)


# ------------------------------------------------------------------ OLMoE-shaped two-stage RVQ
def test_olmoe_rvq_layer_full_shape(dev):
    """The OLMoE-shaped SwiGLU layer (E=64, d_model 2048, d_ff 1024, top-8, Zipf(0.9)) coded as
    two-stage RVQ with the layer's k-means codebooks (tests/golden), at T=1 (CUDA-core path) and
    T=32 (tensor-core path).  The oracle encodes the needed experts itself (a spawn pool over the
    host cores) and compares every token at T=1 and two tokens at T=32."""
    cfg = synth.OLMOE_RVQ
    cb = np.load(os.path.join(ROOT, "tests", "golden", "olmoe_rvq_codebooks.npy")).view(np.uint16)
    sets = []
    for m in (synth.GATE, synth.UP, synth.DOWN):
        rows, cols = synth.rvq_matrix_shape(cfg, m)
        sets.append(pack_rvq_set(cfg.E, rows, cols, cb,
                                 lambda e, m=m, r=rows, c=cols: synth.rvq_weight(cfg.seed, e, m, r, c),
                                 lambda e, m=m, r=rows, c=cols: synth.rvq_signs(cfg.seed, e, m, r, c), device=dev))
    runs = []
    for T, n_check in ((1, 1), (32, 2)):
        ids, gates, rid, rg = routed(cfg, T, dev)
        xb = synth.layer_tokens(cfg, T)
        ws = torch.empty(Q.rvq_moe_layer_ws_size(cfg.E, cfg.d_model, cfg.d_ff, T, cfg.top_k), dtype=torch.uint8,
                         device=dev)
        y = torch.empty((T, cfg.d_model), dtype=torch.float32, device=dev)
        Q.rvq_moe_layer(sets[0], sets[1], sets[2], bf16_tensor(xb), ids, gates, y, ws)
        assert Q.qmoe_check_status() == Q.QMOE_OK
        runs.append((xb, rid, rg, y.cpu().numpy().astype(np.float64), list(range(0, T, max(1, T // n_check)))[:n_check]))
    need = sorted({int(e) for xb, rid, rg, y, toks in runs for t in toks for e in rid[t]})
    jobs = [(cfg.seed, e, m, *synth.rvq_matrix_shape(cfg, m), cb) for e in need
            for m in (synth.GATE, synth.UP, synth.DOWN)]
    from helpers import rvq_oracle_matrix
    with mp.get_context("spawn").Pool(min(len(jobs), max(1, len(os.sched_getaffinity(0))))) as pool:
        mats = pool.map(rvq_oracle_matrix, jobs)
    coded = {e: mats[3 * i:3 * i + 3] for i, e in enumerate(need)}
    for xb, rid, rg, y, toks in runs:
        sel = np.asarray(toks)
        ref = M.moe_layer(synth.bf16_to_f64(xb)[sel], rid[sel], rg[sel],
                          lambda e, xs: R.swiglu_expert(xs, *coded[e]), cfg.d_model)
        for i, t in enumerate(sel):
            assert P.normwise_rel_err(y[t], ref[i]) < TOL
