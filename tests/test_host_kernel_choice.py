"""Host logic: which dictionary kernel a layer call launches for each matrix (no GPU needed)."""
import pytest

import decode_matvec_gb300 as Q


def test_c2048_shapes():
    # wi: 6144 rows, 4-token chunks, 20 warps: 192 groups of 32 rows in 10 full rounds -> row-per-lane;
    # wo: 2080 rows, 2-token chunks, 24 warps: 65 groups in 3 rounds (90 % busy) -> flat stream
    assert Q.qmoe_moe_layer_kernels(2048, 2080, 6144, 4096, 1) == (Q.QMOE_KERNEL_ROWS, Q.QMOE_KERNEL_FLAT, True)
    # 64 slots: the table still goes to shared memory, no tensor-core launch below 256 slots
    assert Q.qmoe_moe_layer_kernels(2048, 2080, 6144, 64, 1) == (Q.QMOE_KERNEL_ROWS, Q.QMOE_KERNEL_FLAT, False)
    # fewer than 16 slots: the table is read through L1/L2
    assert Q.qmoe_moe_layer_kernels(2048, 2080, 6144, 8, 1) == (Q.QMOE_KERNEL_FLAT_L2, Q.QMOE_KERNEL_FLAT_L2, False)


def test_switch_base_shapes():
    # wi: 3072 rows, 8-token chunks, 16 warps: 96 groups in 6 full rounds -> row-per-lane;
    # wo: 768 rows, 4-token chunks, 20 warps: 24 groups in 2 rounds (60 % busy) -> flat stream
    assert Q.qmoe_moe_layer_kernels(128, 768, 3072, 512, 1) == (Q.QMOE_KERNEL_ROWS, Q.QMOE_KERNEL_FLAT, True)


def test_bad_sizes_rejected():
    with pytest.raises(Q.QmoeError):
        Q.qmoe_moe_layer_kernels(0, 2080, 6144, 4096, 1)
    with pytest.raises(Q.QmoeError):
        Q.qmoe_moe_layer_kernels(8, 2080, 6144, 4096, 9)
