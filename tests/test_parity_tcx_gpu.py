"""GPU parity of the f32-accurate tensor-core path (B200Q_PATH_TCX) against the
CPU oracle.

The path scales each row of x by an exact power of two and splits it exactly
into three bf16 pieces, so every product on the tensor cores is exact and only
the f32 accumulation rounds: the bar is the f32 path's, 1e-5 of
|scale| * sum_i |deq * x|, and results are bit-exact where one rounding is the
whole computation (one-hot x).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_F32, assert_within, gpu_matmul, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import torch
    torch.cuda.set_device(0)
    import quantized_weight_quant_gb300 as q
    return q


def _check(q, fmt, O, I, S, seed=0):
    codes, scales, x = inputs(fmt, O, I, S, seed)
    y_ref, bound = oracle.matmul(fmt, O, I, codes, scales, x)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        y = gpu_matmul(q, t, x, S, O, q.PATH_TCX)
    assert_within(y, y_ref, bound, TOL_F32, "tcx fmt%d O%d I%d S%d" % (fmt, O, I, S))


@pytest.mark.parametrize("fmt", [1, 2], ids=["i8", "i4"])
@pytest.mark.parametrize("O,I", [(1, 1), (127, 63), (129, 64), (300, 65), (77, 1000), (256, 512)])
@pytest.mark.parametrize("S", [1, 2, 5, 6, 10, 11, 15, 16, 31])
def test_tcx_ragged(q, fmt, O, I, S):
    _check(q, fmt, O, I, S, seed=O * 17 + I + S)


@pytest.mark.parametrize("fmt", [1, 2], ids=["i8", "i4"])
def test_tcx_onehot_bit_exact(q, fmt):
    """One-hot x: y = RN_f32(scale * deq), bit for bit (pieces 1, 0, 0)."""
    O, I = 256, 15
    codes, scales, _ = inputs(fmt, O, I, 1, seed=9)
    x = np.eye(I, dtype=np.float32)
    y_ref, _ = oracle.matmul(fmt, O, I, codes, scales, x)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        y = gpu_matmul(q, t, x, I, O, q.PATH_TCX)
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("fmt", [1, 2], ids=["i8", "i4"])
def test_tcx_extreme_rows(q, fmt):
    """Rows whose largest |x| is subnormal, near 1e33, or an outlier, and an
    all-zero row: the per-row power of two keeps the split exact."""
    O, I, S = 72, 300, 4
    codes, scales, x = inputs(fmt, O, I, S, seed=17)
    g = synth.rng(17, 5)
    x = x.astype(np.float64)
    x[0] = np.sign(x[0]) * g.uniform(1.0, 3.0, I) * 2.0 ** -140
    x[1] = x[1] * 1e33
    x[2, 7] = 1e3
    x[3] = 0.0
    x = x.astype(np.float32)
    y_ref, bound = oracle.matmul(fmt, O, I, codes, scales, x)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        y = gpu_matmul(q, t, x, S, O, q.PATH_TCX)
    assert_within(y, y_ref, bound, TOL_F32, "tcx extreme fmt%d" % fmt)
    assert np.all(y[3] == 0)


@pytest.mark.parametrize("S", [2, 4, 8, 15])
def test_tcx_int4_12288x6144(q, S):
    """Config-2 shape at S = 4 (and neighbours), every output."""
    _check(q, 2, 12288, 6144, S, seed=S)


def test_tcx_gate_up_shares_pieces(q):
    import torch
    from gpu_util import empty, to_dev
    fmt, O, I, S = 2, 2048, 6144, 6
    cg, sg = synth.quant_tensor(fmt, O, I, 0, 71, 5e-3, 2e-2)
    cu, su = synth.quant_tensor(fmt, O, I, 0, 72, 5e-3, 2e-2)
    x = synth.activations(S, I, 0, 73)
    yg_ref, bg, yu_ref, bu = oracle.matmul_gate_up(fmt, O, I, cg, sg, cu, su, x)
    with q.tensor_upload(fmt, O, I, cg, sg) as tg, q.tensor_upload(fmt, O, I, cu, su) as tu:
        if q.matmul_path(tg, S) != q.PATH_TCX:
            pytest.skip("the three-piece path is not AUTO's choice at this S")
        xd, yg, yu = to_dev(x), empty(S, O), empty(S, O)
        q.matmul_gate_up(tg, tu, xd, yg, yu, S)
        torch.cuda.synchronize()
        assert_within(yg.cpu().numpy(), yg_ref, bg, TOL_F32, "gate tcx")
        assert_within(yu.cpu().numpy(), yu_ref, bu, TOL_F32, "up tcx")
