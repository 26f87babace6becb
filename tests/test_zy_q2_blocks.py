"""Q2 weights packed from their stored block form (qmv_pack_q2_blocks).

The block form is {f16 d; u8 qs[group/4]} per group of weights, row by row,
as the weights come from a file; the pack entry point takes it from host
memory, rewrites it on the host and packs it on the device.  The host
rewrite is also checked without a GPU (test_abi.py).  This file is collected
after the kernel tests, so a run that stops at the first failure has run
those first."""
import numpy as np
import pytest

import oracle
from gemm_decode_prefill_gb300 import synth
from gpu_helpers import TOL_GEMV, assert_within, d16, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qmv():
    from gemm_decode_prefill_gb300 import qmv as m
    return m


def to_blocks(codes, d, group):
    """Planar (codes [rows][cols/4], d bits [rows][cols/group]) -> blocks."""
    rows = codes.shape[0]
    nb, qb = d.shape[1], group // 4
    b = np.empty((rows, nb, 2 + qb), np.uint8)
    b[:, :, 0] = d & 0xFF
    b[:, :, 1] = d >> 8
    b[:, :, 2:] = codes.reshape(rows, nb, qb)
    return b.reshape(rows, -1)


@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("rows,cols", [(1000, 5120), (37, 256)])
def test_pack_from_blocks_equals_planar_pack(qmv, group, rows, cols):
    codes, d, x = synth.q2_inputs(rows, cols, group, seed=61 + group + rows)
    blocks = to_blocks(codes, d, group)
    wb = qmv.qmv_pack_q2_blocks(blocks, group)
    wp = qmv.qmv_pack_q2(dev(codes), d16(d), group)
    assert (wb.rows, wb.cols) == (rows, cols)
    fn = qmv.qmv_q2g64 if group == 64 else qmv.qmv_q2g128
    yb = host(fn(wb, dev(x)))
    yp = host(fn(wp, dev(x)))
    assert np.array_equal(yb, yp)
    y_ref = oracle.q2_blocks(blocks, group, x)
    _, mag = oracle.q2(codes, d, group, x, with_mag=True)
    assert_within(yb, y_ref, mag, TOL_GEMV, f"q2 g{group} {rows}x{cols} from blocks")


def test_pack_from_blocks_rejects_a_ragged_row(qmv):
    with pytest.raises(ValueError):
        qmv.qmv_pack_q2_blocks(np.zeros((4, 19), np.uint8), 64)
