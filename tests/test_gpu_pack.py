"""GPU device encoder (qmoe_pack_device) against the oracle encoder and the host
encoder: codewords and block offsets must be equal bit for bit."""
import numpy as np
import pytest

import synth
from oracle import codec as C

from helpers import dictionary, entry_table

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

Q = pytest.importorskip("decode_matvec_gb300")


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda", 0)


def _device_pack(dd, tern, block, dev, cap=None):
    rows, cols = tern.shape
    nb = (cols + block - 1) // block
    t = torch.from_numpy(np.ascontiguousarray(tern, dtype=np.int8)).to(dev)
    cap = rows * cols // 2 if cap is None else cap
    codes = torch.zeros(max(cap, 1), dtype=torch.int16, device=dev)
    off = torch.zeros(rows * nb + 1, dtype=torch.int32, device=dev)
    ws = torch.empty(Q.qmoe_pack_device_ws_size(rows, cols, block), dtype=torch.uint8, device=dev)
    Q.qmoe_pack_device(dd, t, codes, off, ws, block)
    status = Q.qmoe_check_status()
    off_h = off.cpu().numpy().view(np.uint32)
    n = int(off_h[-1])
    return status, codes.cpu().numpy().view(np.uint16)[:min(n, cap)], off_h


@pytest.mark.parametrize("rows,cols,block,p0", [(7, 512, 256, 0.886), (5, 1030, 256, 0.857), (3, 96, 256, 0.89),
                                                (4, 300, 64, 0.87), (2, 2, 256, 0.886)])
def test_device_pack_equals_oracle(dev, rows, cols, block, p0):
    words = dictionary(p0)
    dd = Q.Dictionary(words)
    tern = synth.ternary_matrix(5, 1, 0, rows, cols, p0)
    status, codes, off = _device_pack(dd, tern, block, dev)
    assert status == Q.QMOE_OK
    ref_codes, ref_off = C.encode(tern, words, block, table=entry_table(p0))
    assert np.array_equal(off, np.asarray(ref_off, dtype=np.uint32))
    assert np.array_equal(codes, np.asarray(ref_codes, dtype=np.uint16))


def test_device_pack_equals_host_pack_large(dev):
    """c2048-shaped wi matrix (6144 x 2080) and a wo-shaped one, against the host encoder."""
    p0 = 0.886
    words = dictionary(p0)
    dd = Q.Dictionary(words)
    for rows, cols, m in ((6144, 2080, synth.WI), (2080, 6144, synth.WO)):
        tern = synth.ternary_matrix(3, 11, m, rows, cols, p0)
        status, codes, off = _device_pack(dd, tern, 256, dev)
        assert status == Q.QMOE_OK
        hc, ho = Q.qmoe_pack(tern, words, 256)
        assert np.array_equal(off, ho)
        assert np.array_equal(codes, hc)


def test_device_pack_edge_rows(dev):
    """All-zero rows, all-nonzero rows, alternating signs and zero rows count."""
    p0 = 0.886
    words = dictionary(p0)
    dd = Q.Dictionary(words)
    cols = 520
    tern = np.zeros((4, cols), dtype=np.int8)
    tern[1] = 1
    tern[2] = -1
    tern[3, ::2] = 1
    tern[3, 1::2] = -1
    status, codes, off = _device_pack(dd, tern, 256, dev)
    assert status == Q.QMOE_OK
    hc, ho = Q.qmoe_pack(tern, words, 256)
    assert np.array_equal(off, ho) and np.array_equal(codes, hc)
    empty = np.zeros((0, cols), dtype=np.int8)
    status, codes, off = _device_pack(dd, empty, 256, dev)
    assert status == Q.QMOE_OK and off.tolist() == [0]


def test_device_pack_repeated_entry_takes_first_code(dev):
    """A dictionary that repeats an entry: both encoders emit the smaller codeword."""
    p0 = 0.886
    words = dictionary(p0).copy()
    # entry 40000 becomes a copy of entry 5
    words[2 * 40000], words[2 * 40000 + 1] = words[2 * 5], words[2 * 5 + 1]
    dd = Q.Dictionary(words)
    tern = synth.ternary_matrix(9, 0, 0, 16, 1024, p0)
    status, codes, off = _device_pack(dd, tern, 256, dev)
    assert status == Q.QMOE_OK
    hc, ho = Q.qmoe_pack(tern, words, 256)
    assert np.array_equal(off, ho) and np.array_equal(codes, hc)
    assert not np.any(codes == 40000)


def test_device_pack_errors(dev):
    p0 = 0.886
    words = dictionary(p0)
    dd = Q.Dictionary(words)
    tern = synth.ternary_matrix(5, 2, 0, 8, 512, p0)
    # a weight outside {-1, 0, 1}: reported through the device error word
    bad = tern.copy()
    bad[3, 77] = 2
    status, _, _ = _device_pack(dd, bad, 256, dev)
    assert status == Q.QMOE_EINVAL
    # too small a codeword buffer: the excess is dropped and reported
    status, _, _ = _device_pack(dd, tern, 256, dev, cap=10)
    assert status == Q.QMOE_ECAPACITY
    # host-side shape checks
    t = torch.zeros((4, 7), dtype=torch.int8, device=dev)
    with pytest.raises(Q.QmoeError):
        Q.qmoe_pack_device_ws_size(4, 7, 256)
    ws = torch.empty(16, dtype=torch.uint8, device=dev)
    codes = torch.zeros(16, dtype=torch.int16, device=dev)
    off = torch.zeros(8, dtype=torch.int32, device=dev)
    with pytest.raises(Q.QmoeError):
        Q.qmoe_pack_device(dd, torch.zeros((4, 8), dtype=torch.int8, device=dev), codes, off, ws, 256)
    assert Q.qmoe_check_status() == Q.QMOE_OK
    del t
