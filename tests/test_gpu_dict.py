"""GPU parity of the dictionary path against the oracle, through the C ABI.

Tolerance: fp32-mode outputs are compared normwise, max|y - y_ref| / max|y_ref|
<= 2e-3 (bf16 activations, fp32 accumulation; in practice ~1e-7).  bf16-mode
outputs must equal the fp32-mode result rounded to nearest even, bit for bit;
bf16 keeps 8 significant bits, so that rounding alone may move an output by
2**-8 of its value.  Decoded weights, routing ids and bucketing are compared
exactly.
"""
import numpy as np
import pytest

import synth
from oracle import codec as C
from oracle import moe as M
from oracle import products as P

from helpers import BLOCK, bf16_tensor, bf16_values, dictionary, oracle_matrix, oracle_matrix_set

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
TOL = 2e-3
TOL_BF16_OUT = 2.0 ** -8 + TOL

Q = pytest.importorskip("decode_matvec_gb300")


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda")


@pytest.fixture(scope="module")
def dict886(dev):
    return Q.Dictionary(dictionary(0.886))


@pytest.fixture(scope="module")
def dict857(dev):
    return Q.Dictionary(dictionary(0.857))


def _single(codes, off, scale, rows, cols, block=BLOCK):
    return Q.MatrixSet.from_host(codes, off, scale, rows, cols, block)


@pytest.mark.parametrize("rows,cols,block,p0", [(96, 4096, 256, 0.886), (33, 1030, 256, 0.886),
                                               (20, 3072, 256, 0.857), (5, 100, 32, 0.886), (3, 2, 256, 0.886)])
def test_decode_dense_bit_exact(dev, rows, cols, block, p0):
    d = Q.Dictionary(dictionary(p0))
    tern, codes, off, scale = oracle_matrix(11, 0, 0, rows, cols, p0, block)
    m = _single(codes, off, scale, rows, cols, block)
    w = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    Q.qmoe_decode_dense(d, m, w)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    ref = C.decode(codes, off, dictionary(p0), scale, rows, cols, block)
    assert np.array_equal(w.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8, 13, 32])
def test_expert_matvec_parity(dev, dict886, T):
    rows, cols = 200, 2080
    tern, codes, off, scale = oracle_matrix(5, 1, 0, rows, cols, 0.886)
    m = _single(codes, off, scale, rows, cols)
    xb = synth.activations_bf16(5, T, cols)
    x = bf16_tensor(xb)
    y = torch.empty((T, rows), dtype=torch.float32, device=dev)
    Q.qmoe_expert_matvec(dict886, m, x, y, y_is_f32=True)
    yb = torch.empty((T, rows), dtype=torch.int16, device=dev)
    Q.qmoe_expert_matvec(dict886, m, x, yb, y_is_f32=False)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    W = C.decode(codes, off, dictionary(0.886), scale, rows, cols)
    ref = P.matmul_xwt(synth.bf16_to_f64(xb), W)
    got = y.cpu().numpy().astype(np.float64)
    assert P.normwise_rel_err(got, ref) < 1e-5
    assert P.normwise_rel_err(bf16_values(yb), ref) < TOL_BF16_OUT
    # bf16 mode is the fp32 result rounded to nearest even
    assert np.array_equal(yb.cpu().numpy().view(np.uint16), synth.bf16_bits_from_f32(y.cpu().numpy()))


@pytest.mark.parametrize("p0,most", [(0.857, 4), (0.75, 5)])
def test_expert_matvec_escape_entries(dev, p0, most):
    # p0 = 0.857 dictionaries hold entries with four nonzeros (the four-slot compact form); p0 = 0.75
    # ones also entries with five (read through their canonical words)
    d = Q.Dictionary(dictionary(p0))
    rows, cols = 64, 3072
    tern, codes, off, scale = oracle_matrix(6, 0, 1, rows, cols, p0)
    L, sym = C.expansion(dictionary(p0))
    nnz = (sym != 0).sum(axis=1)
    assert nnz[codes].max() == most
    m = _single(codes, off, scale, rows, cols)
    W = C.decode(codes, off, dictionary(p0), scale, rows, cols)
    for T in (1, 2, 4, 7):
        xb = synth.activations_bf16(6, T, cols)
        y = torch.empty((T, rows), dtype=torch.float32, device=dev)
        Q.qmoe_expert_matvec(d, m, bf16_tensor(xb), y)
        assert P.normwise_rel_err(y.cpu().numpy(), P.matmul_xwt(synth.bf16_to_f64(xb), W)) < 1e-5
    assert Q.qmoe_check_status() == Q.QMOE_OK


def test_identity_probe_recovers_weights(dev, dict886):
    # X = I gives y[t][r] = s_r * w_rt exactly: the decoded weights seen through the fused kernel
    rows, cols = 48, 512
    tern, codes, off, scale = oracle_matrix(8, 0, 0, rows, cols, 0.886)
    m = _single(codes, off, scale, rows, cols)
    eye = np.eye(cols, dtype=np.float32)
    y = torch.empty((cols, rows), dtype=torch.float32, device=dev)
    Q.qmoe_expert_matvec(dict886, m, bf16_tensor(synth.bf16_bits_from_f32(eye)), y)
    W = C.decode(codes, off, dictionary(0.886), scale, rows, cols)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), W.T)


def test_linear_1024x4096_full_size(dev):
    cfg = synth.LINEAR_1024x4096
    d = Q.Dictionary(dictionary(cfg.p0))
    tern, codes, off, scale = oracle_matrix(cfg.seed, 0, 0, cfg.rows, cfg.cols, cfg.p0)
    m = _single(codes, off, scale, cfg.rows, cfg.cols)
    W = C.decode(codes, off, dictionary(cfg.p0), scale, cfg.rows, cfg.cols)
    for T in cfg.tokens:
        xb = synth.activations_bf16(cfg.seed, T, cfg.cols)
        y = torch.empty((T, cfg.rows), dtype=torch.float32, device=dev)
        Q.qmoe_expert_matvec(d, m, bf16_tensor(xb), y)
        assert P.normwise_rel_err(y.cpu().numpy(), P.matmul_xwt(synth.bf16_to_f64(xb), W)) < 1e-5
    w = torch.empty((cfg.rows, cfg.cols), dtype=torch.float32, device=dev)
    Q.qmoe_decode_dense(d, m, w)
    assert np.array_equal(w.cpu().numpy().astype(np.float64), W)
    assert Q.qmoe_check_status() == Q.QMOE_OK


def test_corrupt_stream_reports_format_error(dev, dict886):
    rows, cols = 8, 512
    tern, codes, off, scale = oracle_matrix(9, 0, 0, rows, cols, 0.886)
    lengths = C.expansion(dictionary(0.886))[0]
    bad = codes.copy()
    # replace a shorter codeword by a 28-weight one: its block now expands past its end
    i = int(np.argmax(lengths[codes] < 28))
    bad[i] = int(np.argmax(lengths))
    m = _single(bad, off, scale, rows, cols)
    y = torch.empty((1, rows), dtype=torch.float32, device=dev)
    Q.qmoe_expert_matvec(dict886, m, bf16_tensor(synth.activations_bf16(1, 1, cols)), y)
    assert Q.qmoe_check_status() == Q.QMOE_EFORMAT
    w = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    Q.qmoe_decode_dense(dict886, m, w)
    assert Q.qmoe_check_status() == Q.QMOE_EFORMAT
    assert Q.qmoe_check_status() == Q.QMOE_OK          # the error word was cleared


@pytest.mark.parametrize("which", ["wi", "wo"])
def test_corrupt_stream_in_a_layer_call(dev, which):
    """A codeword of expert 0 replaced by a 28-weight run (its block now expands past its end) in a
    layer call that stages the table in shared memory: the row-per-lane kernel (wi, 512 rows) and the
    flat-stream kernel (wo, 256 rows) both record QMOE_EFORMAT; their activation reads stay inside the
    staged row and its zero padding."""
    E, d, f, T, p0 = 2, 256, 512, 32, 0.886
    assert Q.qmoe_moe_layer_kernels(E, d, f, T, 1)[:2] == (Q.QMOE_KERNEL_ROWS, Q.QMOE_KERNEL_FLAT)
    wi = oracle_matrix_set(21, E, synth.WI, f, d, p0)
    wo = oracle_matrix_set(21, E, synth.WO, d, f, p0)
    lengths = C.expansion(dictionary(p0))[0]
    tgt = wi if which == "wi" else wo
    codes = tgt[0].copy()
    i = int(np.argmax(lengths[codes[: int(tgt[1][1])]] < 28))      # inside expert 0's stream
    codes[i] = int(np.argmax(lengths))
    wi_codes, wo_codes = (codes, wo[0]) if which == "wi" else (wi[0], codes)
    mwi = Q.MatrixSet.from_host(wi_codes, wi[2], wi[3], f, d, code_base=wi[1], count=E)
    mwo = Q.MatrixSet.from_host(wo_codes, wo[2], wo[3], d, f, code_base=wo[1], count=E)
    dd = Q.Dictionary(dictionary(p0))
    x = bf16_tensor(synth.activations_bf16(21, T, d))
    ids = torch.zeros((T, 1), dtype=torch.int32, device=dev)       # every token to expert 0
    gates = torch.ones((T, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(Q.qmoe_moe_layer_ws_size(E, d, f, T, 1), dtype=torch.uint8, device=dev)
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    Q.qmoe_moe_layer(dd, mwi, mwo, x, ids, gates, y, ws, y_is_f32=True)
    assert Q.qmoe_check_status() == Q.QMOE_EFORMAT
    assert Q.qmoe_check_status() == Q.QMOE_OK          # the error word was cleared


def test_bad_arguments_rejected_on_host(dev, dict886):
    tern, codes, off, scale = oracle_matrix(9, 0, 0, 4, 64, 0.886)
    m = _single(codes, off, scale, 4, 64)
    bad = Q.MatrixSet(m.codes, None, m.row_off, m.blk_len, m.scale, 1, 4, 63, 256)
    y = torch.empty((1, 4), dtype=torch.float32, device=dev)
    with pytest.raises(Q.QmoeError):
        Q.qmoe_expert_matvec(dict886, bad, bf16_tensor(synth.activations_bf16(1, 1, 64)), y)


@pytest.mark.parametrize("T,E,k", [(64, 128, 1), (37, 64, 8), (5, 7, 3), (1, 64, 8), (3, 256, 32),
                                   (33, 2048, 1), (9, 300, 4), (2, 257, 32), (600, 300, 4)])
def test_route_parity(dev, T, E, k):
    """E <= 256: a warp per token with the logits in registers; larger E: a block per token up to
    512 tokens, a warp per token beyond."""
    lg = synth.zipf_logits(4, T, E, 0.9)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, k), dtype=torch.float32, device=dev)
    Q.qmoe_route(torch.from_numpy(lg).to(dev), k, ids, gates)
    rid, rg = M.route(lg, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(gates.cpu().numpy(), rg, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("E", [40, 600])
def test_route_ties_go_to_lower_id(dev, E):
    lg = np.zeros((3, E), np.float32)
    lg[1, [5, 9, 30]] = 2.0
    lg[2, [E - 1, 3, 33]] = -1.0
    ids = torch.empty((3, 4), dtype=torch.int32, device=dev)
    gates = torch.empty((3, 4), dtype=torch.float32, device=dev)
    Q.qmoe_route(torch.from_numpy(lg).to(dev), 4, ids, gates)
    assert ids.cpu().numpy().tolist() == M.route(lg, 4)[0].tolist()


@pytest.mark.parametrize("T,k,E", [(512, 1, 128), (40, 8, 64), (4096, 1, 2048), (1, 1, 5), (300, 2, 8192)])
def test_bucketise_exact(dev, T, k, E):
    ids_np = M.route(synth.zipf_logits(3, T, E, 1.0), k)[0]
    ids = torch.from_numpy(ids_np).to(dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    Q.qmoe_bucketise(ids, E, counts, offsets, perm)
    rc, ro, rp = M.bucketise(ids_np, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)


def _layer(E, d, f, p0, seed):
    wi = oracle_matrix_set(seed, E, synth.WI, f, d, p0)
    wo = oracle_matrix_set(seed, E, synth.WO, d, f, p0)
    mwi = Q.MatrixSet.from_host(wi[0], wi[2], wi[3], f, d, code_base=wi[1], count=E)
    mwo = Q.MatrixSet.from_host(wo[0], wo[2], wo[3], d, f, code_base=wo[1], count=E)
    return mwi, mwo, wi[4], wo[4]


@pytest.mark.parametrize("E,d,f,T,k,p0", [(8, 256, 512, 40, 1, 0.857), (6, 128, 384, 33, 2, 0.886),
                                           (16, 768, 768, 200, 1, 0.87), (4, 256, 256, 3, 1, 0.886),
                                           # experts with >= 32 tokens take the tensor-core kernel:
                                           (4, 776, 1040, 300, 1, 0.857), (6, 520, 264, 160, 2, 0.886),
                                           # ~75 tensor-core jobs: 4-tile (wi) and 2-tile (wo) work items
                                           (2, 512, 1024, 4700, 1, 0.886),
                                           # 3-tile (wi) work items, entries with more than three nonzeros
                                           (2, 384, 768, 4700, 1, 0.857),
                                           # entries with five nonzeros (canonical words) on both kernels
                                           (6, 256, 512, 300, 1, 0.75)])
def test_moe_layer_parity(dev, E, d, f, T, k, p0):
    dd = Q.Dictionary(dictionary(p0))
    mwi, mwo, Wi, Wo = _layer(E, d, f, p0, seed=21)
    lg = synth.zipf_logits(21, T, E, 1.0)
    xb = synth.activations_bf16(21, T, d)
    x = bf16_tensor(xb)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, k), dtype=torch.float32, device=dev)
    Q.qmoe_route(torch.from_numpy(lg).to(dev), k, ids, gates)
    ws = torch.empty(Q.qmoe_moe_layer_ws_size(E, d, f, T, k), dtype=torch.uint8, device=dev)
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    Q.qmoe_moe_layer(dd, mwi, mwo, x, ids, gates, y, ws, y_is_f32=True)
    yb = torch.empty((T, d), dtype=torch.int16, device=dev)
    Q.qmoe_moe_layer(dd, mwi, mwo, x, ids, gates, yb, ws, y_is_f32=False)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    rid, rg = M.route(lg, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    ref = M.moe_layer(synth.bf16_to_f64(xb), rid, rg, lambda e, xs: M.relu_expert(xs, Wi[e], Wo[e]), d)
    assert P.normwise_rel_err(y.cpu().numpy(), ref) < TOL
    assert np.array_equal(yb.cpu().numpy().view(np.uint16), synth.bf16_bits_from_f32(y.cpu().numpy()))
    assert P.normwise_rel_err(bf16_values(yb), ref) < TOL_BF16_OUT
    # run-to-run determinism: the same bits again
    y2 = torch.empty_like(y)
    Q.qmoe_moe_layer(dd, mwi, mwo, x, ids, gates, y2, ws, y_is_f32=True)
    assert torch.equal(y, y2)
