"""Shared helpers of the GPU parity tests: run the library through the C ABI and
compare with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np

import oracle
import synth

TOL_F32 = 1e-5      # f32 path:        |y - y_ref| <= 1e-5 * |scale| * sum |deq * x|
TOL_TC = 4e-3       # tensor-core path: |y - y_ref| <= 4e-3 * |scale| * sum |deq * x|

SCALE_RANGE = {0: (1e-3, 2e-2), 1: (1e-3, 1e-2), 2: (5e-3, 2e-2), 3: (1e-3, 2e-2)}


def device():
    import torch
    return torch.device("cuda:0")


def inputs(fmt, O, I, S, seed=0, stream=1):
    lo, hi = SCALE_RANGE[fmt]
    codes, scales = synth.quant_tensor(fmt, O, I, seed, stream, lo, hi)
    x = synth.activations(S, I, seed, stream + 100)
    return codes, scales, x


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device())


def empty(S, O):
    import torch
    return torch.full((S, O), float("nan"), dtype=torch.float32, device=device())


def gpu_matmul(q, t, x, S, O, path=None):
    import torch
    xd = to_dev(x)
    yd = empty(S, O)
    if path is None:
        q.matmul(t, xd, yd, S)
    else:
        q.matmul_ex(t, xd, yd, S, path)
    torch.cuda.synchronize()
    return yd.cpu().numpy()


def assert_within(y, y_ref, bound, tol, what=""):
    y = np.asarray(y, np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), "%s: non-finite output (unwritten or NaN)" % what
    err = np.abs(y - y_ref.astype(np.float64))
    ok = err <= tol * bound
    if not ok.all():
        bad = np.argwhere(~ok)
        s, o = bad[0]
        ratio = np.max(err[bound > 0] / bound[bound > 0]) if (bound > 0).any() else float("inf")
        raise AssertionError("%s: %d/%d outside tol %.1e (max err/bound %.3g); first (s=%d,o=%d): "
                             "gpu %r ref %r bound %r" % (what, len(bad), y.size, tol, ratio, s, o,
                                                          y[s, o], y_ref[s, o], bound[s, o]))
    return float(np.max(err / np.where(bound > 0, bound, 1.0)))
