"""GPU parity of the layer glue kept on the device: RMSNorm with an optional
residual (b200q_rmsnorm) against the CPU oracle.

h = x + r is one f32 addition on both sides, so h is compared bit for bit; y
is compared within 1e-5 of |y_ref| (f32 sum of squares, correctly rounded
square root and division against the oracle's double).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import torch
    torch.cuda.set_device(0)
    import quantized_weight_quant_gb300 as q
    return q


def _inputs(S, D, seed):
    x = synth.normal_f32((S, D), seed, 1, std=2.0)
    r = synth.normal_f32((S, D), seed, 2)
    w = synth.uniform_f32((D,), 0.5, 1.5, seed, 3)
    return x, r, w


def _check_y(y, y_ref, what):
    err = np.abs(y.astype(np.float64) - y_ref)
    ok = err <= 1e-5 * np.abs(y_ref)
    assert ok.all(), "%s: max rel err %.3g" % (what, np.max(err / np.maximum(np.abs(y_ref), 1e-300)))


@pytest.mark.parametrize("D", [1, 5, 6, 33, 1024, 6144, 7168, 8192, 8196, 10000])
@pytest.mark.parametrize("S", [1, 3, 64])
@pytest.mark.parametrize("residual", [False, True], ids=["x", "x+r"])
def test_rmsnorm_vs_oracle(q, D, S, residual):
    import torch
    x, r, w = _inputs(S, D, D * 7 + S)
    eps = 1e-6
    h_ref, _, y_ref = oracle.rmsnorm(x, w, eps, r=r if residual else None)
    xd, rd, wd = to_dev(x), to_dev(r), to_dev(w)
    y = torch.full((S, D), float("nan"), device=xd.device)
    h = torch.full((S, D), float("nan"), device=xd.device)
    q.rmsnorm(xd, wd, y, S, D, eps, r=rd if residual else None, h=h)
    torch.cuda.synchronize()
    assert np.array_equal(h.cpu().numpy(), h_ref)
    _check_y(y.cpu().numpy(), y_ref, "rmsnorm D%d S%d" % (D, S))


def test_rmsnorm_1571_rows(q):
    """A prefill-sized batch: 1571 rows of 6144."""
    import torch
    S, D = 1571, 6144
    x, r, w = _inputs(S, D, 11)
    _, _, y_ref = oracle.rmsnorm(x, w, 1e-5, r=r)
    xd, rd, wd = to_dev(x), to_dev(r), to_dev(w)
    y = torch.empty((S, D), device=xd.device)
    q.rmsnorm(xd, wd, y, S, D, 1e-5, r=rd)
    torch.cuda.synchronize()
    _check_y(y.cpu().numpy(), y_ref, "rmsnorm 1571x6144")


@pytest.mark.parametrize("D", [6144, 10000, 33])
@pytest.mark.parametrize("alias", ["h=x", "h=r"])
def test_rmsnorm_residual_in_place(q, D, alias):
    """The residual stream updated in place: h written over x, or over r."""
    import torch
    S = 2
    x, r, w = _inputs(S, D, 5)
    h_ref, _, y_ref = oracle.rmsnorm(x, w, 1e-6, r=r)
    xd, rd, wd = to_dev(x), to_dev(r), to_dev(w)
    y = torch.empty((S, D), device=xd.device)
    h = xd if alias == "h=x" else rd
    q.rmsnorm(xd, wd, y, S, D, 1e-6, r=rd, h=h)
    torch.cuda.synchronize()
    assert np.array_equal(h.cpu().numpy(), h_ref)
    _check_y(y.cpu().numpy(), y_ref, "in place " + alias)


def test_rmsnorm_zero_row_and_errors(q):
    import torch
    D = 64
    x = np.zeros((1, D), np.float32)
    w = np.ones(D, np.float32)
    xd, wd = to_dev(x), to_dev(w)
    y = torch.full((1, D), float("nan"), device=xd.device)
    q.rmsnorm(xd, wd, y, 1, D, 1e-6)
    torch.cuda.synchronize()
    assert np.all(y.cpu().numpy() == 0)
    with pytest.raises(q.B200QError):
        q.rmsnorm(xd, wd, xd, 1, D, 1e-6)                  # y over x
    with pytest.raises(q.B200QError):
        q.rmsnorm(xd, wd, y, 1, D, -1.0)                   # negative eps
    q.rmsnorm(xd, wd, y, 0, D, 1e-6)                       # S = 0: no-op
