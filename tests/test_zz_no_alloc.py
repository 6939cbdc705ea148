"""The allocation-free tensor-core entry point, b200q_matmul_tc_noalloc.

It serves callers that cannot allocate device memory while they run (their
device memory belongs to another allocator, or they must not wait on an
allocator call).  It must give the same results as the regular tensor-core
path, b200q_matmul_ex(..., B200Q_PATH_TC), within the tensor-core tolerance,
on consecutive calls that share its fixed workspace, and must refuse sizes
beyond that workspace with a clear error.  This file is collected last so a
run that stops at the first failure has run every other test before it.
"""
import numpy as np
import pytest

import oracle
from gpu_util import TOL_TC, assert_within, empty, gpu_matmul, inputs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import torch
    torch.cuda.set_device(0)
    import quantized_weight_quant_gb300 as q
    return q


def _noalloc(q, t, x, S, O):
    import torch
    xd = to_dev(x)
    yd = empty(S, O)
    q.matmul_tc_noalloc(t, xd, yd, S)
    torch.cuda.synchronize()
    return yd.cpu().numpy()


def test_noalloc_matches_tc_path_two_calls():
    import quantized_weight_quant_gb300 as q
    import torch
    torch.cuda.set_device(0)
    cases = [(2, 256, 1024, 200, 1), (1, 300, 640, 64, 2)]   # (fmt, O, I, S, seed): int4 then int8
    for fmt, O, I, S, seed in cases:
        codes, scales, x = inputs(fmt, O, I, S, seed=seed)
        _, bound = oracle.matmul(fmt, O, I, codes, scales, x)
        with q.tensor_upload(fmt, O, I, codes, scales) as t:
            y_tc = gpu_matmul(q, t, x, S, O, q.PATH_TC)
            y1 = _noalloc(q, t, x, S, O)
            # second call in a row: a different, shorter x over the same array
            x2 = x[: S // 2][::-1].copy()
            y2 = _noalloc(q, t, x2, S // 2, O)
            y2_tc = gpu_matmul(q, t, x2, S // 2, O, q.PATH_TC)
        _, bound2 = oracle.matmul(fmt, O, I, codes, scales, x2)
        assert_within(y1, y_tc, bound, TOL_TC, "noalloc call 1 vs tc path")
        assert_within(y2, y2_tc, bound2, TOL_TC, "noalloc call 2 vs tc path")
        assert np.array_equal(y1, y_tc) and np.array_equal(y2, y2_tc)   # same kernels, same order


def test_noalloc_rejects_oversize_and_bad_format():
    import quantized_weight_quant_gb300 as q
    import torch
    torch.cuda.set_device(0)
    cap = q.tc_noalloc_capacity()
    assert cap == 24 * 2 ** 20
    O, I = 128, 6144                     # 6144 padded int4 columns -> 12288 bytes per row of x
    codes, scales, x = inputs(2, O, I, 1)
    with q.tensor_upload(2, O, I, codes, scales) as t:
        S = cap // (I * 2) + 1           # one row past the capacity
        with pytest.raises(q.B200QError) as ei:
            q.matmul_tc_noalloc(t, 16, 16, S)        # refused before any pointer is touched
        assert ei.value.status == q.EINVAL and "workspace" in q.last_error()
    codes, scales, x = inputs(3, 8, 64, 1)
    with q.tensor_upload(3, 8, 64, codes, scales) as t:
        with pytest.raises(q.B200QError):
            q.matmul_tc_noalloc(t, to_dev(np.zeros((1, 64), np.float32)), empty(1, 8), 1)
