"""GPU parity of tensors with group-wise scales (b200q_tensor_upload_grouped)
against the CPU oracle: one scale per row and group of gs columns, the f32
path's bar (1e-5 of sum_i |scale_g * deq * x|)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_F32, assert_within, empty, gpu_matmul, to_dev

pytestmark = pytest.mark.gpu

GS = {0: [4, 8, 64], 1: [16, 32, 128], 2: [16, 32, 64, 128], 3: [16, 32, 64, 128]}


@pytest.fixture(scope="module")
def q():
    import torch
    torch.cuda.set_device(0)
    import quantized_weight_quant_gb300 as q
    return q


def _grouped(fmt, O, I, gs, seed):
    codes = synth.codes(fmt, O, I, seed, 1)
    G = -(-I // gs)
    gsc = synth.uniform_f32((O, G), 5e-3, 2e-2, seed, 2)
    return codes, gsc


@pytest.mark.parametrize("fmt,gs", [(f, g) for f in (0, 1, 2, 3) for g in GS[f]],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("O,I", [(8, 64), (77, 300), (130, 1000)])
@pytest.mark.parametrize("S", [1, 3, 17])
def test_group_scales_vs_oracle(q, fmt, gs, O, I, S):
    codes, gsc = _grouped(fmt, O, I, gs, O + I + gs)
    x = synth.activations(S, I, gs, 3)
    y_ref, bound = oracle.matmul_gs(fmt, O, I, gs, codes, gsc, x)
    with q.tensor_upload(fmt, O, I, codes, gsc, gs=gs) as t:
        assert q.tensor_group_size(t) == gs
        assert q.matmul_path(t, S) == q.PATH_F32
        y = gpu_matmul(q, t, x, S, O)
    assert_within(y, y_ref, bound, TOL_F32, "gs fmt%d gs%d O%d I%d S%d" % (fmt, gs, O, I, S))


def test_group_scales_int4_12288x6144_gs128(q):
    fmt, O, I, gs = 2, 12288, 6144, 128
    codes, gsc = _grouped(fmt, O, I, gs, 1)
    x = synth.activations(1, I, 1, 3)
    y_ref, bound = oracle.matmul_gs(fmt, O, I, gs, codes, gsc, x)
    with q.tensor_upload(fmt, O, I, codes, gsc, gs=gs) as t:
        y = gpu_matmul(q, t, x, 1, O)
    assert_within(y, y_ref, bound, TOL_F32, "gs int4 12288x6144")


def test_group_scales_gate_up_and_grouped_call(q):
    import torch
    fmt, O, I, gs, S = 2, 256, 512, 64, 2
    (cg, sg), (cu, su) = _grouped(fmt, O, I, gs, 7), _grouped(fmt, O, I, gs, 8)
    x = synth.activations(S, I, 9, 3)
    yg_ref, bg = oracle.matmul_gs(fmt, O, I, gs, cg, sg, x)
    yu_ref, bu = oracle.matmul_gs(fmt, O, I, gs, cu, su, x)
    with q.tensor_upload(fmt, O, I, cg, sg, gs=gs) as tg, q.tensor_upload(fmt, O, I, cu, su, gs=gs) as tu:
        xd, yg, yu = to_dev(x), empty(S, O), empty(S, O)
        q.matmul_gate_up(tg, tu, xd, yg, yu, S)
        zg, zu = empty(S, O), empty(S, O)
        q.matmul_grouped([tg, tu], [xd, xd], [zg, zu], S)
        torch.cuda.synchronize()
        for got, ref, b, what in ((yg, yg_ref, bg, "gate"), (yu, yu_ref, bu, "up"), (zg, yg_ref, bg, "grouped gate"),
                                  (zu, yu_ref, bu, "grouped up")):
            assert_within(got.cpu().numpy(), ref, b, TOL_F32, what)


def test_group_scales_refusals(q):
    fmt, O, I, gs = 2, 16, 64, 32
    codes, gsc = _grouped(fmt, O, I, gs, 3)
    with q.tensor_upload(fmt, O, I, codes, gsc, gs=gs) as t:
        x = to_dev(synth.activations(20, I, 3, 3))
        for path in (q.PATH_TC, q.PATH_TCX):
            with pytest.raises(q.B200QError):
                q.matmul_ex(t, x, empty(20, O), 20, path)
        with pytest.raises(q.B200QError):
            q.matmul_tc_noalloc(t, x, empty(20, O), 20)
    big = np.ones(O * I, np.float32)                 # enough scales for any group size
    for bad in (0, -1, 24, 48):                      # through the C entry point itself
        assert not q.lib.b200q_tensor_upload_grouped(fmt, O, I, bad, codes.ctypes.data, big.ctypes.data)
        assert "group size" in q.last_error()
    with q.tensor_upload(fmt, O, I, codes, np.ones(O, np.float32)) as t:
        assert q.tensor_group_size(t) == 0
