"""GPU parity of the RHT + residual-VQ path against the oracle, through the C ABI.

Decoded weights are compared exactly; fp32-mode outputs normwise within 2e-3;
bf16-mode outputs must be the fp32-mode outputs rounded to nearest even.
"""
import numpy as np
import pytest

import synth
from oracle import moe as M
from oracle import products as P
from oracle import rvq as R

from helpers import bf16_tensor, bf16_values

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
TOL = 2e-3

Q = pytest.importorskip("decode_matvec_gb300")


def _matrix(seed, e, m, rows, cols, cb=None, iters=4):
    w = synth.rvq_weight(seed, e, m, rows, cols)
    so, si = synth.rvq_signs(seed, e, m, rows, cols)
    wr = R.rotate_weight(w, so, si)
    if cb is None:
        cb = R.fit_codebooks(R.normalised_vectors(wr, R.row_scale_f16(wr), 8), k=256, iters=iters, seed=seed)
    idx, sc = R.encode(wr, cb)
    return dict(w=w, so=so, si=si, idx=idx, scale=sc, cb=cb.astype(np.float16).view(np.uint16))


def _set(mats, rows, cols):
    return Q.RvqMatrixSet.from_host(np.stack([m["idx"] for m in mats]), mats[0]["cb"],
                                    np.concatenate([m["scale"] for m in mats]),
                                    np.concatenate([m["so"] for m in mats]), np.concatenate([m["si"] for m in mats]),
                                    len(mats), rows, cols)


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    return torch.device("cuda")


@pytest.mark.parametrize("rows,cols", [(128, 256), (64, 2048), (2048, 64), (8, 8)])
def test_rvq_decode_bit_exact(dev, rows, cols):
    mt = _matrix(2, 0, 0, rows, cols) if rows * cols >= 2048 * 8 else None
    if mt is None:
        rng = np.random.default_rng(0)
        cb = R.f16_round(rng.standard_normal((2, 256, 8)))
        mt = _matrix(2, 0, 0, rows, cols, cb=cb)
    s = _set([mt], rows, cols)
    w = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    Q.rvq_decode_dense(s, w)
    ref = R.decode(mt["idx"], mt["cb"], mt["scale"])
    assert np.array_equal(w.cpu().numpy(), ref)


@pytest.mark.parametrize("T", [1, 2, 3, 8, 13, 32])
def test_rvq_expert_matmul_parity(dev, T):
    rows, cols = 256, 512
    mt = _matrix(3, 1, 0, rows, cols)
    s = _set([mt], rows, cols)
    xb = synth.activations_bf16(3, T, cols)
    y = torch.empty((T, rows), dtype=torch.float32, device=dev)
    ws = torch.empty(Q.rvq_expert_matmul_ws_size(rows, cols, T), dtype=torch.uint8, device=dev)
    Q.rvq_expert_matmul(s, bf16_tensor(xb), y, ws)
    yb = torch.empty((T, rows), dtype=torch.int16, device=dev)
    Q.rvq_expert_matmul(s, bf16_tensor(xb), yb, ws, y_is_f32=False)
    wdec = R.decode(mt["idx"], mt["cb"], mt["scale"])
    ref = R.linear(synth.bf16_to_f64(xb), wdec, mt["so"], mt["si"])
    assert P.normwise_rel_err(y.cpu().numpy(), ref) < TOL
    assert np.array_equal(yb.cpu().numpy().view(np.uint16), synth.bf16_bits_from_f32(y.cpu().numpy()))
    assert P.normwise_rel_err(bf16_values(yb), ref) < 2.0 ** -8 + TOL


def test_rvq_product_approximates_dense_weight(dev):
    # the whole pipeline approximates the original (unrotated) dense product
    rows, cols = 256, 512
    mt = _matrix(3, 2, 0, rows, cols, iters=8)
    s = _set([mt], rows, cols)
    xb = synth.activations_bf16(7, 4, cols)
    y = torch.empty((4, rows), dtype=torch.float32, device=dev)
    ws = torch.empty(Q.rvq_expert_matmul_ws_size(rows, cols, 4), dtype=torch.uint8, device=dev)
    Q.rvq_expert_matmul(s, bf16_tensor(xb), y, ws)
    dense = synth.bf16_to_f64(xb) @ mt["w"].T
    rel = np.linalg.norm(y.cpu().numpy() - dense) / np.linalg.norm(dense)
    assert rel < 0.45


@pytest.mark.parametrize("E,d,f,T,k", [(8, 256, 128, 20, 4), (16, 512, 256, 32, 8), (4, 128, 64, 1, 2)])
def test_rvq_moe_layer_parity(dev, E, d, f, T, k):
    seed = 31
    gate = [_matrix(seed, e, synth.GATE, f, d) for e in range(E)]
    cb = R.f16_round(gate[0]["cb"].view(np.float16).astype(np.float64))
    gate = [_matrix(seed, e, synth.GATE, f, d, cb=cb) for e in range(E)]
    up = [_matrix(seed, e, synth.UP, f, d, cb=cb) for e in range(E)]
    down = [_matrix(seed, e, synth.DOWN, d, f, cb=cb) for e in range(E)]
    sg, su, sd = _set(gate, f, d), _set(up, f, d), _set(down, d, f)
    lg = synth.zipf_logits(seed, T, E, 0.9)
    xb = synth.activations_bf16(seed, T, d)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, k), dtype=torch.float32, device=dev)
    Q.qmoe_route(torch.from_numpy(lg).to(dev), k, ids, gates)
    ws = torch.empty(Q.rvq_moe_layer_ws_size(E, d, f, T, k), dtype=torch.uint8, device=dev)
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    Q.rvq_moe_layer(sg, su, sd, bf16_tensor(xb), ids, gates, y, ws)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    rid, rg = M.route(lg, k)

    def expert(e, xs):
        trip = [(R.decode(m["idx"], m["cb"], m["scale"]), m["so"], m["si"]) for m in (gate[e], up[e], down[e])]
        return R.swiglu_expert(xs, *trip)

    ref = M.moe_layer(synth.bf16_to_f64(xb), rid, rg, expert, d)
    assert P.normwise_rel_err(y.cpu().numpy(), ref) < TOL


# ------------------------------------------------------ per-matrix stage counts
def _matrix_st(seed, e, m, rows, cols, cb, stages):
    w = synth.rvq_weight(seed, e, m, rows, cols)
    so, si = synth.rvq_signs(seed, e, m, rows, cols)
    wr = R.rotate_weight(w, so, si)
    idx, sc = R.encode(wr, cb, stages=stages)
    return dict(w=w, so=so, si=si, idx=idx, scale=sc, cb=cb.astype(np.float16).view(np.uint16))


def _set_st(mats, rows, cols):
    return Q.RvqMatrixSet.from_host([m["idx"] for m in mats], mats[0]["cb"],
                                    np.concatenate([m["scale"] for m in mats]),
                                    np.concatenate([m["so"] for m in mats]), np.concatenate([m["si"] for m in mats]),
                                    len(mats), rows, cols)


def _cb3(seed, rows, cols):
    w = synth.rvq_weight(seed, 0, 0, rows, cols)
    so, si = synth.rvq_signs(seed, 0, 0, rows, cols)
    wr = R.rotate_weight(w, so, si)
    return R.fit_codebooks(R.normalised_vectors(wr, R.row_scale_f16(wr), 8), k=256, iters=3, seed=seed, stages=3)


@pytest.mark.parametrize("stages", [1, 2, 3])
def test_rvq_decode_bit_exact_any_stage_count(dev, stages):
    rows, cols = 128, 256
    cb = _cb3(8, rows, cols)
    mt = _matrix_st(8, 1, 0, rows, cols, cb, stages)
    s = _set_st([mt], rows, cols)
    w = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    Q.rvq_decode_dense(s, w)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    assert np.array_equal(w.cpu().numpy(), R.decode(mt["idx"], mt["cb"], mt["scale"]))


@pytest.mark.parametrize("stages,T", [(1, 1), (3, 1), (1, 32), (3, 32), (3, 5)])
def test_rvq_expert_matmul_any_stage_count(dev, stages, T):
    rows, cols = 256, 512
    cb = _cb3(9, rows, cols)
    mt = _matrix_st(9, 2, 0, rows, cols, cb, stages)
    s = _set_st([mt], rows, cols)
    xb = synth.activations_bf16(9, T, cols)
    y = torch.empty((T, rows), dtype=torch.float32, device=dev)
    ws = torch.empty(Q.rvq_expert_matmul_ws_size(rows, cols, T), dtype=torch.uint8, device=dev)
    Q.rvq_expert_matmul(s, bf16_tensor(xb), y, ws)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    ref = R.linear(synth.bf16_to_f64(xb), R.decode(mt["idx"], mt["cb"], mt["scale"]), mt["so"], mt["si"])
    assert P.normwise_rel_err(y.cpu().numpy(), ref) < TOL


@pytest.mark.parametrize("E,d,f,T,k", [(9, 256, 128, 24, 4), (6, 128, 256, 3, 2), (4, 256, 128, 64, 2)])
def test_rvq_moe_layer_frequency_conditioned_parity(dev, E, d, f, T, k):
    """Experts with 3 / 2 / 1 stages by popularity thirds (the layer's fixed Zipf popularity)."""
    seed = 41
    pop = synth.zipf_popularity(seed, E, 0.9)
    st = Q.rvq_stage_allocation(pop, 2)
    assert np.array_equal(st, R.stage_allocation(pop, 2))
    cb = _cb3(seed, f, d)
    gate = [_matrix_st(seed, e, synth.GATE, f, d, cb, int(st[e])) for e in range(E)]
    up = [_matrix_st(seed, e, synth.UP, f, d, cb, int(st[e])) for e in range(E)]
    down = [_matrix_st(seed, e, synth.DOWN, d, f, cb, int(st[e])) for e in range(E)]
    sg, su, sd = _set_st(gate, f, d), _set_st(up, f, d), _set_st(down, d, f)
    lg = synth.zipf_layer_logits(seed, T, E, 0.9)
    xb = synth.activations_bf16(seed, T, d)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, k), dtype=torch.float32, device=dev)
    Q.qmoe_route(torch.from_numpy(lg).to(dev), k, ids, gates)
    ws = torch.empty(Q.rvq_moe_layer_ws_size(E, d, f, T, k), dtype=torch.uint8, device=dev)
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    Q.rvq_moe_layer(sg, su, sd, bf16_tensor(xb), ids, gates, y, ws)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    rid, rg = M.route(lg, k)

    def expert(e, xs):
        trip = [(R.decode(m["idx"], m["cb"], m["scale"]), m["so"], m["si"]) for m in (gate[e], up[e], down[e])]
        return R.swiglu_expert(xs, *trip)

    ref = M.moe_layer(synth.bf16_to_f64(xb), rid, rg, expert, d)
    assert P.normwise_rel_err(y.cpu().numpy(), ref) < TOL


def test_rvq_bad_stage_count_reported(dev):
    rows, cols = 64, 128
    cb = _cb3(10, rows, cols)
    mt = _matrix_st(10, 0, 0, rows, cols, cb, 2)
    s = _set_st([mt], rows, cols)
    s.stages.fill_(5)                       # more stages than the set's three codebooks
    w = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    Q.rvq_decode_dense(s, w)
    assert Q.qmoe_check_status() == Q.QMOE_EFORMAT


# ------------------------------------------------------ activation range of the tensor-core split
def _scaled_tokens(seed, T, cols, exps):
    """bf16 tokens N(0,1) * 10**exps[t] (token t's magnitude set by its own exponent)."""
    v = np.random.default_rng(seed).standard_normal((T, cols)) * (10.0 ** np.asarray(exps, np.float64))[:, None]
    return synth.bf16_bits_from_f32(v.astype(np.float32))


@pytest.mark.parametrize("T", [1, 3, 16, 32])
def test_rvq_expert_matmul_activation_range(dev, T):
    """Tokens of very different magnitudes in one batch (|x| up to ~1e6 and down to ~1e-4): the
    CUDA-core path (T < 16) takes fp32 activations as they are; the tensor-core path (T >= 16)
    splits each token into fp16 high and low parts after a per-token power-of-two scale, so no
    part leaves fp16's range.  Every token is compared with the oracle on its own."""
    rows, cols = 256, 512
    mt = _matrix(3, 1, 0, rows, cols)
    s = _set([mt], rows, cols)
    exps = np.resize(np.array([6.0, -4.0, 0.0, 5.0, -3.0, 2.5, 4.7]), T)
    xb = _scaled_tokens(8, T, cols, exps)
    y = torch.empty((T, rows), dtype=torch.float32, device=dev)
    ws = torch.empty(Q.rvq_expert_matmul_ws_size(rows, cols, T), dtype=torch.uint8, device=dev)
    Q.rvq_expert_matmul(s, bf16_tensor(xb), y, ws)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    ref = R.linear(synth.bf16_to_f64(xb), R.decode(mt["idx"], mt["cb"], mt["scale"]), mt["so"], mt["si"])
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    for t in range(T):
        assert P.normwise_rel_err(got[t], ref[t]) < TOL, (t, exps[t])


def test_rvq_moe_layer_activation_range(dev):
    """The SwiGLU layer on the tensor-core path with tokens scaled by 1e5 and 1e-3: gate/up inputs,
    the bf16 h (up to ~1e9 here) and the down input all pass through the fp16 split."""
    E, d, f, T, k, seed = 8, 256, 128, 32, 4, 33
    gate = [_matrix(seed, e, synth.GATE, f, d) for e in range(E)]
    cb = R.f16_round(gate[0]["cb"].view(np.float16).astype(np.float64))
    gate = [_matrix(seed, e, synth.GATE, f, d, cb=cb) for e in range(E)]
    up = [_matrix(seed, e, synth.UP, f, d, cb=cb) for e in range(E)]
    down = [_matrix(seed, e, synth.DOWN, d, f, cb=cb) for e in range(E)]
    sg, su, sd = _set(gate, f, d), _set(up, f, d), _set(down, d, f)
    lg = synth.zipf_logits(seed, T, E, 0.9)
    xb = _scaled_tokens(9, T, d, np.where(np.arange(T) % 2 == 0, 5.0, -3.0))
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, k), dtype=torch.float32, device=dev)
    Q.qmoe_route(torch.from_numpy(lg).to(dev), k, ids, gates)
    ws = torch.empty(Q.rvq_moe_layer_ws_size(E, d, f, T, k), dtype=torch.uint8, device=dev)
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    Q.rvq_moe_layer(sg, su, sd, bf16_tensor(xb), ids, gates, y, ws)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    rid, rg = M.route(lg, k)

    def expert(e, xs):
        trip = [(R.decode(m["idx"], m["cb"], m["scale"]), m["so"], m["si"]) for m in (gate[e], up[e], down[e])]
        return R.swiglu_expert(xs, *trip)

    ref = M.moe_layer(synth.bf16_to_f64(xb), rid, rg, expert, d)
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    for t in range(T):
        assert P.normwise_rel_err(got[t], ref[t]) < TOL, t
