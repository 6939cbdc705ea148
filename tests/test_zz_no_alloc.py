"""The allocation-free tensor-core entry point, b200q_matmul_tc_noalloc.

It serves callers that cannot allocate device memory while they run (their
device memory belongs to another allocator, or they must not wait on an
allocator call).  It must match the CPU oracle within the tensor-core
tolerance and give the same results as the regular tensor-core path,
b200q_matmul_ex(..., B200Q_PATH_TC), on consecutive calls that share its
fixed workspace; it must allocate nothing (checked in a fresh process whose
first library call is this one); and it must refuse sizes beyond that
workspace with a clear error.  This file is collected last so a run that
stops at the first failure has run every other test before it.
"""
import os
import subprocess
import sys
import textwrap

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
        y_ref, bound = oracle.matmul(fmt, O, I, codes, scales, x)
        with q.tensor_upload(fmt, O, I, codes, scales) as t:
            y_tc = gpu_matmul(q, t, x, S, O, q.PATH_TC)
            y1 = _noalloc(q, t, x, S, O)
            # second call in a row: a different, shorter x over the same array
            x2 = x[: S // 2][::-1].copy()
            y2 = _noalloc(q, t, x2, S // 2, O)
            y2_tc = gpu_matmul(q, t, x2, S // 2, O, q.PATH_TC)
        y2_ref, bound2 = oracle.matmul(fmt, O, I, codes, scales, x2)
        assert_within(y1, y_ref, bound, TOL_TC, "noalloc call 1 vs oracle")
        assert_within(y2, y2_ref, bound2, TOL_TC, "noalloc call 2 vs oracle")
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


_FRESH = textwrap.dedent("""
    import sys
    sys.path.insert(0, sys.argv[1])
    import numpy as np
    import torch
    torch.cuda.set_device(0)
    import quantized_weight_quant_gb300 as q
    import synth
    O, I, S = 256, 1024, 64
    codes, scales = synth.quant_tensor(q.I4, O, I, 0, 1, 5e-3, 2e-2)
    x = torch.from_numpy(synth.activations(S, I, 0, 2)).cuda()
    y = torch.empty((S, O), dtype=torch.float32, device="cuda")
    t = q.tensor_upload(q.I4, O, I, codes, scales)
    torch.cuda.synchronize()
    n0 = q.workspace_allocations()
    q.matmul_tc_noalloc(t, x, y, S)
    q.matmul_tc_noalloc(t, x, y, S)
    torch.cuda.synchronize()
    n1 = q.workspace_allocations()
    q.matmul_ex(t, x, y, S, q.PATH_TC)          # the regular path does allocate: the counter works
    torch.cuda.synchronize()
    n2 = q.workspace_allocations()
    t.free()
    print("allocs", n0, n1, n2)
""")


def test_noalloc_allocates_nothing_in_a_fresh_process():
    """The first library calls of a fresh process are the two no-alloc calls:
    the library's workspace counter (pool creation, pool allocations, staging
    buffers) must not move, while one regular tensor-core call afterwards
    must move it."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("allocs")][-1]
    n0, n1, n2 = (int(v) for v in line.split()[1:])
    assert n0 == 0 and n1 == 0, line
    assert n2 > n1, line
