"""GPU parity of the tensor-core (bf16 x, tcgen05) path against the CPU oracle.

Contract bar: |y_gpu - y_ref| <= 4e-3 * |scale| * sum_i |deq * x| against the
oracle on the unrounded f32 x.  Diagnostic bar: against the oracle run on x
rounded to bf16 (what the tensor cores actually multiply), the f32
accumulation alone must stay within 1e-5 of that bound.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_F32, TOL_TC, assert_within, empty, gpu_matmul, inputs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import torch
    torch.cuda.set_device(0)
    import quantized_weight_quant_gb300 as q
    return q


def _check_tc(q, fmt, O, I, S, seed=0, path=None):
    codes, scales, x = inputs(fmt, O, I, S, seed)
    y_ref, bound = oracle.matmul(fmt, O, I, codes, scales, x)
    y_b, bound_b, _ = oracle.matmul_bf16x(fmt, O, I, codes, scales, x)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        y = gpu_matmul(q, t, x, S, O, q.PATH_TC if path is None else path)
    assert_within(y, y_ref, bound, TOL_TC, "tc vs oracle fmt%d O%d I%d S%d" % (fmt, O, I, S))
    assert_within(y, y_b, bound_b, TOL_F32, "tc vs bf16-x oracle fmt%d O%d I%d S%d" % (fmt, O, I, S))
    return y


@pytest.mark.parametrize("fmt", [1, 2], ids=["i8", "i4"])
@pytest.mark.parametrize("O,I", [(1, 1), (127, 63), (129, 64), (300, 65), (128, 200), (77, 1000), (256, 512)])
@pytest.mark.parametrize("S", [1, 16, 17, 176, 177, 400])
def test_tc_ragged(q, fmt, O, I, S):
    _check_tc(q, fmt, O, I, S, seed=O * 31 + I)


@pytest.mark.parametrize("fmt", [1, 2], ids=["i8", "i4"])
def test_threshold_15_16(q, fmt):
    """S = 15 takes an f32-accurate path (1e-5), S = 16 the bf16 tensor-core path."""
    O, I = 200, 300
    thr = q.tc_min_s()
    codes, scales, x = inputs(fmt, O, I, thr, seed=5)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        assert q.matmul_path(t, thr - 1) in (q.PATH_F32, q.PATH_TCX)
        assert q.matmul_path(t, thr) == q.PATH_TC
        y15 = gpu_matmul(q, t, x[:thr - 1], thr - 1, O)
        y16 = gpu_matmul(q, t, x, thr, O)
    r15, b15 = oracle.matmul(fmt, O, I, codes, scales, x[:thr - 1])
    r16, b16 = oracle.matmul(fmt, O, I, codes, scales, x)
    assert_within(y15, r15, b15, TOL_F32, "S=15 f32 path")
    assert_within(y16, r16, b16, TOL_TC, "S=16 tc path")


@pytest.mark.parametrize("fmt", [1, 2], ids=["i8", "i4"])
def test_tc_onehot_bit_exact(q, fmt):
    """One-hot x is exact in bf16, so y = RN_f32(scale * deq) bit for bit."""
    O, I = 256, 64
    codes, scales, _ = inputs(fmt, O, I, 1, seed=9)
    x = np.eye(I, dtype=np.float32)
    y_ref, _ = oracle.matmul(fmt, O, I, codes, scales, x)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        y = gpu_matmul(q, t, x, I, O, q.PATH_TC)
    assert np.array_equal(y, y_ref)


def test_tc_repeatable(q):
    codes, scales, x = inputs(2, 384, 640, 200, seed=3)
    with q.tensor_upload(2, 384, 640, codes, scales) as t:
        y1 = gpu_matmul(q, t, x, 200, 384, q.PATH_TC)
        y2 = gpu_matmul(q, t, x, 200, 384, q.PATH_TC)
    assert np.array_equal(y1, y2)


def test_f32_and_int2_reject_tc(q):
    for fmt in (0, 3):
        codes, scales, x = inputs(fmt, 16, 64, 20)
        with q.tensor_upload(fmt, 16, 64, codes, scales) as t:
            assert q.matmul_path(t, 100) == q.PATH_F32
            for path in (q.PATH_TC, q.PATH_TCX):
                with pytest.raises(q.B200QError):
                    q.matmul_ex(t, to_dev(x), empty(20, 16), 20, path)


def _sample_idx(n, k, seed, must):
    g = synth.rng(seed, 0)
    idx = set(int(v) for v in g.choice(n, size=min(k, n), replace=False))
    idx.update(m for m in must if 0 <= m < n)
    return np.array(sorted(idx))


@pytest.mark.parametrize("fmt", [2, 1], ids=["i4", "i8"])
def test_prefill_12288x6144_s1571_sampled(q, fmt):
    """W4A16 (and W8A16) prefill O=12288, I=6144, S=1571 in the launch
    configuration the benchmark times; sampled outputs (tile edges included)
    against the oracle."""
    O, I, S = 12288, 6144, 1571
    codes, scales, x = inputs(fmt, O, I, S, seed=0)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        assert q.matmul_path(t, S) == q.PATH_TC
        y = gpu_matmul(q, t, x, S, O)
    rows = _sample_idx(O, 120, 1, [0, 1, 127, 128, 255, 6143, 12160, 12287])
    toks = _sample_idx(S, 160, 2, [0, 1, 175, 176, 351, 1407, 1408, 1569, 1570])
    y_ref, bound = oracle.matmul(fmt, len(rows), I, codes[rows], scales[rows], x[toks])
    assert_within(y[np.ix_(toks, rows)], y_ref, bound, TOL_TC, "prefill sampled")
    assert np.all(np.isfinite(y))


@pytest.mark.slow
@pytest.mark.parametrize("fmt", [2, 1], ids=["i4", "i8"])
def test_prefill_12288x6144_s1571_full(q, fmt):
    """Every output of the W4A16 (and W8A16) prefill call O=12288, I=6144,
    S=1571, in the launch configuration the benchmark times, against the
    oracle (118.6 G double multiply-adds, about ten seconds on 16 host cores):
    the persistent walk over all 96 x 9 output tiles, each over 96 k-blocks, is
    compared in full, not only at sampled rows and tokens."""
    O, I, S = 12288, 6144, 1571
    codes, scales, x = inputs(fmt, O, I, S, seed=0)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        assert q.matmul_path(t, S) == q.PATH_TC
        y = gpu_matmul(q, t, x, S, O)
    y_ref, bound = oracle.matmul(fmt, O, I, codes, scales, x)
    assert_within(y, y_ref, bound, TOL_TC, "prefill full fmt%d" % fmt)


def test_gate_up_tc(q):
    import torch
    fmt, O, I, S = 2, 2048, 6144, 40
    cg, sg = synth.quant_tensor(fmt, O, I, 0, 41, 5e-3, 2e-2)
    cu, su = synth.quant_tensor(fmt, O, I, 0, 42, 5e-3, 2e-2)
    x = synth.activations(S, I, 0, 43)
    yg_ref, bg, yu_ref, bu = oracle.matmul_gate_up(fmt, O, I, cg, sg, cu, su, x)
    with q.tensor_upload(fmt, O, I, cg, sg) as tg, q.tensor_upload(fmt, O, I, cu, su) as tu:
        xd, yg, yu = to_dev(x), empty(S, O), empty(S, O)
        q.matmul_gate_up(tg, tu, xd, yg, yu, S)
        torch.cuda.synchronize()
        assert_within(yg.cpu().numpy(), yg_ref, bg, TOL_TC, "gate tc")
        assert_within(yu.cpu().numpy(), yu_ref, bu, TOL_TC, "up tc")


def test_device_status_clean(q):
    codes, scales, x = inputs(2, 256, 256, 64)
    with q.tensor_upload(2, 256, 256, codes, scales) as t:
        gpu_matmul(q, t, x, 64, 256)
        gpu_matmul(q, t, x[:2], 2, 256)
    assert q.device_status() == q.OK
