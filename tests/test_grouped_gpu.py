"""GPU parity of the grouped calls (b200q_matmul_grouped and
b200q_matmul_grouped_silu) against the CPU oracle, one tensor at a time.

A grouped call must give every tensor of the group the result the oracle
gives that tensor alone, within the bar of the path it takes (1e-5 of
sum |scale * deq * x| on the f32 path, 4e-3 on the tensor-core path), for
shared and distinct inputs, ragged shapes, every format, and groups whose
blocks span many tensors.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import SCALE_RANGE, TOL_F32, TOL_TC, assert_within, empty, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import torch
    torch.cuda.set_device(0)
    import quantized_weight_quant_gb300 as q
    return q


def _tensors(fmt, Os, I, seed):
    lo, hi = SCALE_RANGE[fmt]
    return [synth.quant_tensor(fmt, O, I, seed, 200 + j, lo, hi) for j, O in enumerate(Os)]


def _run_grouped(q, fmt, Os, I, S, x_of, seed=0):
    """x_of[j]: index of set j's input among the distinct inputs."""
    import torch
    ws = _tensors(fmt, Os, I, seed)
    xs = [synth.activations(S, I, seed, 300 + k) for k in range(max(x_of) + 1)]
    handles = [q.tensor_upload(fmt, O, I, c, s) for O, (c, s) in zip(Os, ws)]
    try:
        xd = [to_dev(x) for x in xs]
        ys = [empty(S, O) for O in Os]
        q.matmul_grouped(handles, [xd[k] for k in x_of], ys, S)
        torch.cuda.synchronize()
        out = [y.cpu().numpy() for y in ys]
    finally:
        for h in handles:
            h.free()
    for j, (O, (c, s)) in enumerate(zip(Os, ws)):
        y_ref, bound = oracle.matmul(fmt, O, I, c, s, xs[x_of[j]])
        assert_within(out[j], y_ref, bound, TOL_F32, "set %d (O=%d) fmt%d I%d S%d" % (j, O, fmt, I, S))
    return out


GROUPS = {
    "shared": ([256, 100, 8, 513, 64], [0, 0, 0, 0, 0]),
    "distinct": ([300, 17, 640, 129], [0, 1, 2, 3]),
    "repeat": ([200, 72, 136, 96], [0, 0, 1, 0]),     # a non-consecutive repeat is a new slot
    "pairs": ([128, 128, 256, 256, 64, 64], [0, 0, 1, 1, 2, 2]),
}


@pytest.mark.parametrize("fmt", [0, 1, 2, 3], ids=["f32", "i8", "i4", "i2"])
@pytest.mark.parametrize("S", [1, 2, 3, 5])
@pytest.mark.parametrize("name", sorted(GROUPS))
def test_grouped_vs_oracle(q, fmt, S, name):
    Os, x_of = GROUPS[name]
    _run_grouped(q, fmt, Os, 1000, S, x_of, seed=fmt * 7 + S)


@pytest.mark.parametrize("fmt", [1, 2, 3], ids=["i8", "i4", "i2"])
@pytest.mark.parametrize("S", [1, 3])
def test_grouped_blocks_span_many_inputs(q, fmt, S):
    """Fifteen one-row-group tensors ahead of a tall one, every input distinct:
    the first blocks stage several inputs each."""
    Os = [8] * 15 + [4096]
    _run_grouped(q, fmt, Os, 512, S, list(range(16)), seed=3)


def test_grouped_one_launch_per_token_pair(q):
    import torch
    fmt, I = 2, 256
    Os = [64] * 16
    ws = _tensors(fmt, Os, I, 0)
    handles = [q.tensor_upload(fmt, O, I, c, s) for O, (c, s) in zip(Os, ws)]
    try:
        x = to_dev(synth.activations(3, I, 0, 1))
        ys = [empty(3, O) for O in Os]
        n0 = q.kernel_launches()
        q.matmul_grouped(handles, [x] * 16, ys, 1)
        n1 = q.kernel_launches()
        q.matmul_grouped(handles, [x] * 16, ys, 3)
        n2 = q.kernel_launches()
        torch.cuda.synchronize()
    finally:
        for h in handles:
            h.free()
    assert n1 - n0 == 1 and n2 - n1 == 2


def test_grouped_pair_equals_gate_up(q):
    """[tg, tu] on one x is the fused gate/up call: the same launch, bit for bit
    (at S = 1, where both run the SIMT decode kernel)."""
    import torch
    fmt, O, I, S = 2, 2048, 6144, 1
    (cg, sg), (cu, su) = _tensors(fmt, [O, O], I, 5)
    x = to_dev(synth.activations(S, I, 5, 9))
    with q.tensor_upload(fmt, O, I, cg, sg) as tg, q.tensor_upload(fmt, O, I, cu, su) as tu:
        yg, yu, zg, zu = empty(S, O), empty(S, O), empty(S, O), empty(S, O)
        q.matmul_gate_up(tg, tu, x, yg, yu, S)
        q.matmul_grouped([tg, tu], [x, x], [zg, zu], S)
        torch.cuda.synchronize()
        assert torch.equal(yg, zg) and torch.equal(yu, zu)


@pytest.mark.parametrize("fmt", [0, 2, 3], ids=["f32", "i4", "i2"])
@pytest.mark.parametrize("S", [1, 2])
def test_grouped_silu_vs_oracle(q, fmt, S):
    import torch
    Os, I = [384, 96, 256], 700
    ws = _tensors(fmt, Os, I, 11)
    gs = [synth.normal_f32((S, I), 11, 400 + j, std=3.0) for j in range(3)]
    us = [synth.activations(S, I, 11, 500 + j) for j in range(3)]
    handles = [q.tensor_upload(fmt, O, I, c, s) for O, (c, s) in zip(Os, ws)]
    try:
        ys = [empty(S, O) for O in Os]
        q.matmul_grouped_silu(handles, [to_dev(g) for g in gs], [to_dev(u) for u in us], ys, S)
        torch.cuda.synchronize()
        out = [y.cpu().numpy() for y in ys]
    finally:
        for h in handles:
            h.free()
    for j, (O, (c, s)) in enumerate(zip(Os, ws)):
        h32, _ = oracle.silu_mul(gs[j], us[j])
        y_ref, bound = oracle.matmul(fmt, O, I, c, s, h32)
        assert_within(out[j], y_ref, bound, TOL_F32, "silu set %d" % j)


@pytest.mark.parametrize("silu", [False, True], ids=["plain", "silu"])
def test_grouped_tensor_core_rows(q, silu):
    """From the tensor-core threshold on, each tensor runs its own
    tensor-core call (silu(g) * u formed in a workspace first)."""
    import torch
    fmt, Os, I, S = 2, [256, 130], 512, max(q.tc_min_s(), 20)
    ws = _tensors(fmt, Os, I, 13)
    gs = [synth.normal_f32((S, I), 13, 600 + j, std=2.0) for j in range(2)]
    us = [synth.activations(S, I, 13, 700 + j) for j in range(2)]
    handles = [q.tensor_upload(fmt, O, I, c, s) for O, (c, s) in zip(Os, ws)]
    try:
        ys = [empty(S, O) for O in Os]
        if silu:
            q.matmul_grouped_silu(handles, [to_dev(g) for g in gs], [to_dev(u) for u in us], ys, S)
        else:
            q.matmul_grouped(handles, [to_dev(g) for g in gs], ys, S)
        torch.cuda.synchronize()
        out = [y.cpu().numpy() for y in ys]
    finally:
        for h in handles:
            h.free()
    for j, (O, (c, s)) in enumerate(zip(Os, ws)):
        xin = oracle.silu_mul(gs[j], us[j])[0] if silu else gs[j]
        y_ref, bound = oracle.matmul(fmt, O, I, c, s, xin)
        assert_within(out[j], y_ref, bound, TOL_TC, "tc set %d" % j)


def test_moe_layer_grouped_stage_isolated(q):
    """A mixture-of-experts layer at S=1 in two launches: the gate and up
    tensors of 8 experts ([2048, 6144] int4) on one x, then the 8 down
    tensors ([6144, 2048] int4) on silu(g) * u of their own expert.  Each
    stage is checked against the oracle fed the GPU's own input to it."""
    import torch
    fmt, D, F, k = 2, 6144, 2048, 8
    lo, hi = SCALE_RANGE[fmt]
    gu = [synth.quant_tensor(fmt, F, D, 0, 800 + j, lo, hi) for j in range(2 * k)]
    dn = [synth.quant_tensor(fmt, D, F, 0, 900 + e, lo, hi) for e in range(k)]
    x = synth.activations(1, D, 0, 99)
    th = [q.tensor_upload(fmt, F, D, c, s) for c, s in gu]
    td = [q.tensor_upload(fmt, D, F, c, s) for c, s in dn]
    try:
        xd = to_dev(x)
        G, U, Y = empty(k, F), empty(k, F), empty(k, D)
        n0 = q.kernel_launches()
        q.matmul_grouped(th, [xd] * (2 * k), [t for e in range(k) for t in (G[e], U[e])], 1)
        q.matmul_grouped_silu(td, [G[e] for e in range(k)], [U[e] for e in range(k)],
                              [Y[e] for e in range(k)], 1)
        launches = q.kernel_launches() - n0
        torch.cuda.synchronize()
        g_np, u_np, y_np = G.cpu().numpy(), U.cpu().numpy(), Y.cpu().numpy()
    finally:
        for h in th + td:
            h.free()
    assert launches == 2
    for e in range(k):
        cg, sg = gu[2 * e]
        cu, su = gu[2 * e + 1]
        yg_ref, bg, yu_ref, bu = oracle.matmul_gate_up(fmt, F, D, cg, sg, cu, su, x)
        assert_within(g_np[e:e + 1], yg_ref, bg, TOL_F32, "expert %d gate" % e)
        assert_within(u_np[e:e + 1], yu_ref, bu, TOL_F32, "expert %d up" % e)
        h32, _ = oracle.silu_mul(g_np[e:e + 1], u_np[e:e + 1])
        y_ref, bd = oracle.matmul(fmt, D, F, dn[e][0], dn[e][1], h32)
        assert_within(y_np[e:e + 1], y_ref, bd, TOL_F32, "expert %d down" % e)


def test_grouped_argument_errors(q):
    import torch
    (c1, s1), (c2, s2) = _tensors(2, [16, 16], 64, 0)
    c3, s3 = synth.quant_tensor(1, 16, 64, 0, 1, 1e-3, 1e-2)
    with q.tensor_upload(2, 16, 64, c1, s1) as a, q.tensor_upload(2, 16, 128, *_tensors(2, [16], 128, 0)[0]) as b, \
            q.tensor_upload(1, 16, 64, c3, s3) as c:
        x = to_dev(np.zeros((1, 128), np.float32))
        y1, y2 = empty(1, 16), empty(1, 16)
        with pytest.raises(q.B200QError):
            q.matmul_grouped([a, b], [x, x], [y1, y2], 1)          # I differs
        with pytest.raises(q.B200QError):
            q.matmul_grouped([a, c], [x, x], [y1, y2], 1)          # format differs
        with pytest.raises(q.B200QError):
            q.matmul_grouped([a, a], [x, x], [y1, y1], 1)          # outputs overlap
        with pytest.raises(q.B200QError):
            q.matmul_grouped([a], [x], [x], 1)                     # output overlaps input
        with pytest.raises(q.B200QError) as ei:
            q.matmul_grouped([a] * 17, [x] * 17, [empty(1, 16) for _ in range(17)], 1)
        assert ei.value.status == q.EINVAL
        q.matmul_grouped([a], [x], [y1], 0)                        # S = 0: no-op
        torch.cuda.synchronize()
