"""GPU parity of the E8P lattice-code path ([M8.5] 0x06E) against the oracle, through the C ABI.

Decoded weights are compared exactly (all 65 536 code words included); fp32-mode outputs
normwise within 2e-3; bf16-mode outputs must be the fp32-mode outputs rounded to nearest even.
Large cases use seeded uniform code words (every 16-bit word is a code word), so they depend
on no encoder; small cases use the oracle's encoder.
"""
import numpy as np
import pytest

import synth
from oracle import e8p as P8
from oracle import moe as M
from oracle import products as P
from oracle import rvq as R

from helpers import bf16_tensor, bf16_values

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
TOL = 2e-3

Q = pytest.importorskip("decode_matvec_gb300")


def _random(seed, e, m, rows, cols):
    codes, sc = synth.e8p_random_matrix(seed, e, m, rows, cols)
    so, si = synth.rvq_signs(seed, e, m, rows, cols)
    return dict(codes=codes, scale=sc, so=so, si=si)


def _encoded(seed, e, m, rows, cols):
    w = synth.rvq_weight(seed, e, m, rows, cols)
    so, si = synth.rvq_signs(seed, e, m, rows, cols)
    codes, sc = P8.encode(R.rotate_weight(w, so, si))
    return dict(w=w, codes=codes, scale=sc, so=so, si=si)


def _set(mats, rows, cols):
    return Q.RvqMatrixSet.e8p_from_host(np.stack([m["codes"] for m in mats]), np.concatenate([m["scale"] for m in mats]),
                                        np.concatenate([m["so"] for m in mats]),
                                        np.concatenate([m["si"] for m in mats]), len(mats), rows, cols)


def _triple(m):
    return P8.decode(m["codes"], m["scale"]), m["so"], m["si"]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    return torch.device("cuda")


def test_e8p_decode_every_code_word(dev):
    rows, cols = 512, 1024                                   # 65 536 vectors: code word c at vector c
    codes = np.arange(65536, dtype=np.uint16).reshape(rows, cols // 8)
    so, si = synth.rvq_signs(1, 0, 0, rows, cols)
    ones = np.full(rows, 0x3C00, dtype=np.uint16)            # fp16 1.0
    s = _set([dict(codes=codes, scale=ones, so=so, si=si)], rows, cols)
    w = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    Q.rvq_decode_dense(s, w)
    assert np.array_equal(w.cpu().numpy().reshape(65536, 8), P8.codebook().astype(np.float32))
    mt = _random(2, 0, 0, rows, cols)
    s = _set([mt], rows, cols)
    Q.rvq_decode_dense(s, w)
    assert np.array_equal(w.cpu().numpy(), P8.decode(mt["codes"], mt["scale"]))


@pytest.mark.parametrize("rows,cols", [(64, 128), (8, 8), (32, 256)])
def test_e8p_decode_oracle_encoded(dev, rows, cols):
    mt = _encoded(3, 0, 1, rows, cols)
    s = _set([mt], rows, cols)
    w = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    Q.rvq_decode_dense(s, w)
    assert np.array_equal(w.cpu().numpy(), P8.decode(mt["codes"], mt["scale"]))


@pytest.mark.parametrize("rows,cols,T", [(256, 512, 1), (256, 512, 2), (256, 512, 3), (256, 512, 8), (256, 512, 13),
                                         (256, 512, 16), (256, 512, 32), (256, 512, 40), (64, 128, 33),
                                         (2048, 64, 32), (8, 8, 5), (1024, 2048, 32), (1024, 2048, 1)])
def test_e8p_expert_matmul_parity(dev, rows, cols, T):
    """T < 16 (or K not a multiple of 128) runs on CUDA cores, T >= 16 on tcgen05; 64-row and
    2048-row matrices leave part of a 128-row tile empty or need many tiles, T = 33 and 40 leave
    a ragged 32-token tile."""
    mt = _random(4, 1, 0, rows, cols)
    s = _set([mt], rows, cols)
    xb = synth.activations_bf16(5, T, cols)
    y = torch.empty((T, rows), dtype=torch.float32, device=dev)
    ws = torch.empty(Q.rvq_expert_matmul_ws_size(rows, cols, T), dtype=torch.uint8, device=dev)
    Q.rvq_expert_matmul(s, bf16_tensor(xb), y, ws)
    yb = torch.empty((T, rows), dtype=torch.int16, device=dev)
    Q.rvq_expert_matmul(s, bf16_tensor(xb), yb, ws, y_is_f32=False)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    ref = R.linear(synth.bf16_to_f64(xb), *_triple(mt))
    assert P.normwise_rel_err(y.cpu().numpy(), ref) < TOL
    assert np.array_equal(yb.cpu().numpy().view(np.uint16), synth.bf16_bits_from_f32(y.cpu().numpy()))
    assert P.normwise_rel_err(bf16_values(yb), ref) < 2.0 ** -8 + TOL


@pytest.mark.parametrize("T", [1, 32])
def test_e8p_product_approximates_dense_weight(dev, T):
    """Oracle-encoded weights: the whole pipeline approximates the original dense product."""
    rows, cols = 128, 256
    mt = _encoded(3, 2, 0, rows, cols)
    s = _set([mt], rows, cols)
    xb = synth.activations_bf16(7, T, cols)
    y = torch.empty((T, rows), dtype=torch.float32, device=dev)
    ws = torch.empty(Q.rvq_expert_matmul_ws_size(rows, cols, T), dtype=torch.uint8, device=dev)
    Q.rvq_expert_matmul(s, bf16_tensor(xb), y, ws)
    dense = synth.bf16_to_f64(xb) @ mt["w"].T
    rel = np.linalg.norm(y.cpu().numpy() - dense) / np.linalg.norm(dense)
    assert rel < 0.35
    ref = R.linear(synth.bf16_to_f64(xb), *_triple(mt))
    assert P.normwise_rel_err(y.cpu().numpy(), ref) < TOL


def _layer(dev, gate, up, down, E, d, f, T, k, seed, sample=None):
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
    assert np.array_equal(ids.cpu().numpy(), rid)
    rows = np.arange(T) if sample is None else np.asarray(sample)
    x = synth.bf16_to_f64(xb)
    ref = np.zeros((rows.size, d))
    for i, t in enumerate(rows):
        for j in range(k):
            e = int(rid[t, j])
            o = R.swiglu_expert(x[t:t + 1], _triple(gate[e]), _triple(up[e]), _triple(down[e]))
            ref[i] = ref[i] + rg[t, j] * o[0]
    return y.cpu().numpy()[rows], ref


@pytest.mark.parametrize("E,d,f,T,k", [(8, 256, 128, 20, 4), (16, 512, 256, 32, 8), (4, 128, 64, 1, 2),
                                       (6, 256, 512, 40, 2), (5, 128, 256, 7, 3), (12, 128, 256, 3, 10),
                                       (16, 256, 128, 2, 12)])
def test_e8p_moe_layer_parity(dev, E, d, f, T, k):
    """k <= 8: the output transform runs on a thread-block cluster per token; k > 8 on one block."""
    seed = 37
    gate = [_random(seed, e, synth.GATE, f, d) for e in range(E)]
    up = [_random(seed, e, synth.UP, f, d) for e in range(E)]
    down = [_random(seed, e, synth.DOWN, d, f) for e in range(E)]
    got, ref = _layer(dev, gate, up, down, E, d, f, T, k, seed)
    assert P.normwise_rel_err(got, ref) < TOL


@pytest.mark.parametrize("T", [1, 32])
def test_e8p_olmoe_layer_full_size_sampled(dev, T):
    """The OLMoE-shaped layer of the benchmark (E=64, d_model=2048, d_ff=1024, top-8) at its
    token counts; the oracle evaluates a few sampled tokens."""
    cfg = synth.OLMOE_E8P
    E, d, f, k = cfg.E, cfg.d_model, cfg.d_ff, cfg.top_k
    gate = [_random(cfg.seed, e, synth.GATE, f, d) for e in range(E)]
    up = [_random(cfg.seed, e, synth.UP, f, d) for e in range(E)]
    down = [_random(cfg.seed, e, synth.DOWN, d, f) for e in range(E)]
    sample = [0] if T == 1 else [0, 17, T - 1]
    got, ref = _layer(dev, gate, up, down, E, d, f, T, k, cfg.seed, sample=sample)
    assert P.normwise_rel_err(got, ref) < TOL


def test_e8p_bad_sets_rejected(dev):
    rows, cols = 64, 128
    mt = _random(1, 0, 0, rows, cols)
    s = _set([mt], rows, cols)
    xb = bf16_tensor(synth.activations_bf16(1, 2, cols))
    y = torch.empty((2, rows), dtype=torch.float32, device=dev)
    ws = torch.empty(Q.rvq_expert_matmul_ws_size(rows, cols, 2), dtype=torch.uint8, device=dev)
    st = torch.ones(1, dtype=torch.uint8, device=dev)
    for bad in (dict(format=7), dict(n_stages=2), dict(stages=st.data_ptr())):
        c = Q.CRvqSet.from_buffer_copy(s.c)
        for key, v in bad.items():
            setattr(c, key, v)
        s.c = c
        with pytest.raises(Q.QmoeError):
            Q.rvq_expert_matmul(s, xb, y, ws)
        s = _set([mt], rows, cols)
    assert Q.qmoe_check_status() == Q.QMOE_OK


@pytest.mark.parametrize("T", [3, 24])
def test_mixed_formats_in_one_layer(dev, T):
    """Each matrix set carries its own format: E8P gate and down with a two-stage RVQ up matrix."""
    E, d, f, k, seed = 6, 256, 128, 2, 41
    gate = [_random(seed, e, synth.GATE, f, d) for e in range(E)]
    down = [_random(seed, e, synth.DOWN, d, f) for e in range(E)]
    rng = np.random.default_rng(seed)
    cb = R.f16_round(rng.standard_normal((2, 256, 8)) * 0.5)
    cb_bits = cb.astype(np.float16).view(np.uint16)
    up = []
    for e in range(E):
        idx = rng.integers(0, 256, (f, d // 8, 2)).astype(np.uint8)
        sc = (rng.uniform(0.5, 1.5, f) * 0.02).astype(np.float16).view(np.uint16)
        so, si = synth.rvq_signs(seed, e, synth.UP, f, d)
        up.append(dict(idx=idx, scale=sc, so=so, si=si))
    su = Q.RvqMatrixSet.from_host(np.stack([m["idx"] for m in up]), cb_bits, np.concatenate([m["scale"] for m in up]),
                                  np.concatenate([m["so"] for m in up]), np.concatenate([m["si"] for m in up]), E, f, d)
    sg, sd = _set(gate, f, d), _set(down, d, f)
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
        u = (R.decode(up[e]["idx"], cb_bits, up[e]["scale"]), up[e]["so"], up[e]["si"])
        return R.swiglu_expert(xs, _triple(gate[e]), u, _triple(down[e]))

    ref = M.moe_layer(synth.bf16_to_f64(xb), rid, rg, expert, d)
    assert P.normwise_rel_err(y.cpu().numpy(), ref) < TOL
