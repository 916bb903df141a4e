"""The MoE layer entry point that allocates nothing (static device scratch).

Callers hosted in a framework that owns all device memory, or serving loops
that forbid cudaMalloc after start-up, use qmoe_moe_layer_noalloc; it must give
what qmoe_moe_layer gives with a caller workspace.  This file is collected last
so that a run stopping at its first failure has run every other test first.
"""
import numpy as np
import pytest

import synth
from oracle import products as P

from helpers import bf16_tensor, dictionary, oracle_matrix_set

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
TOL = 2e-3

Q = pytest.importorskip("decode_matvec_gb300")


def _layer(E, d, f, p0, seed, dev):
    wi = oracle_matrix_set(seed, E, synth.WI, f, d, p0)
    wo = oracle_matrix_set(seed, E, synth.WO, d, f, p0)
    mwi = Q.MatrixSet.from_host(wi[0], wi[2], wi[3], f, d, code_base=wi[1], count=E, device=dev)
    mwo = Q.MatrixSet.from_host(wo[0], wo[2], wo[3], d, f, code_base=wo[1], count=E, device=dev)
    return mwi, mwo


@pytest.mark.parametrize("E,d,f,T,k,p0", [(8, 256, 512, 40, 1, 0.886), (6, 256, 384, 33, 2, 0.857)])
def test_noalloc_matches_workspace_entry_point_twice(E, d, f, T, k, p0):
    assert torch.cuda.is_available()
    dev = torch.device("cuda")
    dd = Q.Dictionary(dictionary(p0), device=dev)
    mwi, mwo = _layer(E, d, f, p0, 41, dev)
    x = bf16_tensor(synth.activations_bf16(41, T, d))
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, k), dtype=torch.float32, device=dev)
    Q.qmoe_route(torch.from_numpy(synth.zipf_logits(41, T, E, 1.0)).to(dev), k, ids, gates)
    ws = torch.empty(Q.qmoe_moe_layer_ws_size(E, d, f, T, k), dtype=torch.uint8, device=dev)
    ref = torch.empty((T, d), dtype=torch.float32, device=dev)
    Q.qmoe_moe_layer(dd, mwi, mwo, x, ids, gates, ref, ws, y_is_f32=True)
    for _ in range(2):
        y = torch.full((T, d), float("nan"), dtype=torch.float32, device=dev)
        Q.qmoe_moe_layer_noalloc(dd, mwi, mwo, x, ids, gates, y, y_is_f32=True)
        assert Q.qmoe_check_status() == Q.QMOE_OK
        assert P.normwise_rel_err(y.cpu().numpy(), ref.cpu().numpy()) <= TOL
        assert torch.equal(y, ref)            # same kernels, same order: the same bits


def test_noalloc_rejects_oversize_calls():
    dev = torch.device("cuda")
    dd = Q.Dictionary(dictionary(0.886), device=dev)
    E, d, f = 2, 256, 512
    mwi, mwo = _layer(E, d, f, 0.886, 42, dev)
    T = 20000                              # T * d_ff * 2 bytes of h alone exceed 16 MiB
    x = torch.zeros((T, d), dtype=torch.int16, device=dev)
    ids = torch.zeros((T, 1), dtype=torch.int32, device=dev)
    gates = torch.zeros((T, 1), dtype=torch.float32, device=dev)
    y = torch.zeros((T, d), dtype=torch.float32, device=dev)
    with pytest.raises(Q.QmoeError) as ei:
        Q.qmoe_moe_layer_noalloc(dd, mwi, mwo, x, ids, gates, y)
    assert ei.value.status == Q.QMOE_ECAPACITY
    assert "16777216" in str(ei.value)
