"""GPU parity of tensors with group-wise scales (b200q_tensor_upload_grouped)
against the CPU oracle: one scale per row and group of gs columns, the f32
path's bar (1e-5 of sum_i |scale_g * deq * x|)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_F32, TOL_TC, assert_within, empty, gpu_matmul, to_dev

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
        tc = fmt in (1, 2) and S >= q.tc_min_s()           # int8 / int4 from the threshold: bf16 tensor cores
        assert q.matmul_path(t, S) == (q.PATH_TC if tc else q.PATH_F32)
        y = gpu_matmul(q, t, x, S, O)
    assert_within(y, y_ref, bound, TOL_TC if tc else TOL_F32, "gs fmt%d gs%d O%d I%d S%d" % (fmt, gs, O, I, S))


def test_group_scales_int4_12288x6144_gs128(q):
    fmt, O, I, gs = 2, 12288, 6144, 128
    codes, gsc = _grouped(fmt, O, I, gs, 1)
    x = synth.activations(1, I, 1, 3)
    y_ref, bound = oracle.matmul_gs(fmt, O, I, gs, codes, gsc, x)
    with q.tensor_upload(fmt, O, I, codes, gsc, gs=gs) as t:
        y = gpu_matmul(q, t, x, 1, O)
    assert_within(y, y_ref, bound, TOL_F32, "gs int4 12288x6144")


@pytest.mark.parametrize("S", [2, 20], ids=["decode", "tensor_cores"])
def test_group_scales_gate_up_and_grouped_call(q, S):
    import torch
    fmt, O, I, gs = 2, 256, 512, 64
    tol = TOL_TC if S >= q.tc_min_s() else TOL_F32
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
            assert_within(got.cpu().numpy(), ref, b, tol, what)


def test_group_scales_refusals(q):
    fmt, O, I, gs = 2, 16, 64, 32
    codes, gsc = _grouped(fmt, O, I, gs, 3)
    with q.tensor_upload(fmt, O, I, codes, gsc, gs=gs) as t:
        x = to_dev(synth.activations(20, I, 3, 3))
        with pytest.raises(q.B200QError):                      # the three-piece path needs exact weights
            q.matmul_ex(t, x, empty(20, O), 20, q.PATH_TCX)
        assert q.matmul_path(t, 8) == q.PATH_F32
    big = np.ones(O * I, np.float32)                 # enough scales for any group size
    for bad in (0, -1, 24, 48):                      # through the C entry point itself
        assert not q.lib.b200q_tensor_upload_grouped(fmt, O, I, bad, codes.ctypes.data, big.ctypes.data)
        assert "group size" in q.last_error()
    with q.tensor_upload(fmt, O, I, codes, np.ones(O, np.float32)) as t:
        assert q.tensor_group_size(t) == 0


# rows of several decode stages (512 code bytes each) with a ragged tail, and
# group sizes whose groups straddle stages or span several
WIDE = [(0, 12, 700), (0, 260, 1500), (1, 48, 2100), (1, 16, 1300), (2, 96, 3000), (2, 2048, 5000),
        (2, 16, 2500), (3, 192, 6000), (3, 16, 4100), (3, 32, 2200)]


@pytest.mark.parametrize("fmt,gs,I", WIDE, ids=lambda v: str(v))
@pytest.mark.parametrize("S", [1, 2, 5])
def test_group_scales_wide_rows(q, fmt, gs, I, S):
    O = 200
    codes, gsc = _grouped(fmt, O, I, gs, gs + I)
    x = synth.activations(S, I, I, 4)
    y_ref, bound = oracle.matmul_gs(fmt, O, I, gs, codes, gsc, x)
    with q.tensor_upload(fmt, O, I, codes, gsc, gs=gs) as t:
        y = gpu_matmul(q, t, x, S, O)
    assert_within(y, y_ref, bound, TOL_F32, "gs fmt%d gs%d I%d S%d" % (fmt, gs, I, S))


@pytest.mark.parametrize("fmt,gs", [(1, 32), (2, 128), (2, 16), (3, 32)], ids=lambda v: str(v))
@pytest.mark.parametrize("silu", [False, True], ids=["plain", "silu"])
def test_group_scales_grouped_many_sets(q, fmt, gs, silu):
    """Six tensors of different heights in one grouped call (blocks span
    several tensors and inputs), every tensor checked on its own."""
    import torch
    Os, I, S = [300, 8, 640, 17, 129, 1024], 1536, 2
    ws = [_grouped(fmt, O, I, gs, 40 + j) for j, O in enumerate(Os)]
    xa = [synth.normal_f32((S, I), 41, 10 + j, std=2.0) for j in range(len(Os))]
    xb = [synth.activations(S, I, 41, 20 + j) for j in range(len(Os))]
    handles = [q.tensor_upload(fmt, O, I, c, s, gs=gs) for O, (c, s) in zip(Os, ws)]
    try:
        ys = [empty(S, O) for O in Os]
        if silu:
            q.matmul_grouped_silu(handles, [to_dev(a) for a in xa], [to_dev(b) for b in xb], ys, S)
        else:
            q.matmul_grouped(handles, [to_dev(a) for a in xa], ys, S)
        torch.cuda.synchronize()
        out = [y.cpu().numpy() for y in ys]
    finally:
        for h in handles:
            h.free()
    for j, (O, (c, s)) in enumerate(zip(Os, ws)):
        xin = oracle.silu_mul(xa[j], xb[j])[0] if silu else xa[j]
        y_ref, bound = oracle.matmul_gs(fmt, O, I, gs, c, s, xin)
        assert_within(out[j], y_ref, bound, TOL_F32, "set %d" % j)


def test_group_scales_mixed_layouts_in_a_group(q):
    """Per-row and group-wise tensors in one grouped call run one at a time."""
    import torch
    fmt, O, I, S = 2, 96, 640, 1
    c0, s0 = synth.quant_tensor(fmt, O, I, 3, 1, 5e-3, 2e-2)
    c1, s1 = _grouped(fmt, O, I, 64, 4)
    c2, s2 = _grouped(fmt, O, I, 128, 5)
    x = synth.activations(S, I, 3, 9)
    with q.tensor_upload(fmt, O, I, c0, s0) as a, q.tensor_upload(fmt, O, I, c1, s1, gs=64) as b, \
            q.tensor_upload(fmt, O, I, c2, s2, gs=128) as c:
        xd = to_dev(x)
        ys = [empty(S, O) for _ in range(3)]
        q.matmul_grouped([a, b, c], [xd] * 3, ys, S)
        torch.cuda.synchronize()
        out = [y.cpu().numpy() for y in ys]
    refs = [oracle.matmul(fmt, O, I, c0, s0, x), oracle.matmul_gs(fmt, O, I, 64, c1, s1, x),
            oracle.matmul_gs(fmt, O, I, 128, c2, s2, x)]
    for j, (y_ref, bound) in enumerate(refs):
        assert_within(out[j], y_ref, bound, TOL_F32, "mixed set %d" % j)


@pytest.mark.parametrize("fmt,gs", [(0, 8), (1, 16), (2, 128), (2, 16), (3, 16), (3, 32), (3, 64)],
                         ids=lambda v: str(v))
def test_group_scales_run_the_decode_kernel(q, fmt, gs):
    """Below 16 rows a group-wise tensor runs the staged decode kernel, one
    launch per two rows (5 rows: 3 launches); from 16 rows f32 and int2 run
    the general SIMT kernel (one launch), int8 and int4 the bf16 tensor-core
    path (x to bf16, then the GEMM: two launches)."""
    import torch
    O, I = 256, 1024
    codes, gsc = _grouped(fmt, O, I, gs, 6)
    with q.tensor_upload(fmt, O, I, codes, gsc, gs=gs) as t:
        xd = to_dev(synth.activations(16, I, 6, 1))
        y = empty(16, O)
        n0 = q.kernel_launches()
        q.matmul(t, xd, y, 5)
        n1 = q.kernel_launches()
        q.matmul(t, xd, y, 16)
        n2 = q.kernel_launches()
        torch.cuda.synchronize()
    assert (n1 - n0, n2 - n1) == (3, 2 if fmt in (1, 2) else 1)


TC_CASES = [  # fmt, gs, O, I, S
    (2, 128, 300, 1000, 40), (2, 16, 129, 640, 17), (2, 32, 256, 2048, 200), (2, 96, 130, 3000, 33),
    (1, 16, 200, 700, 64), (1, 48, 128, 1536, 100), (1, 128, 77, 4096, 18),
]


@pytest.mark.parametrize("fmt,gs,O,I,S", TC_CASES, ids=lambda v: str(v))
def test_group_scales_tensor_core_path(q, fmt, gs, O, I, S):
    """bf16 tensor-core path with group scales (dequantizer forms
    bf16((code - zero point) * scale)), within the path's 4e-3 bar; tiles
    span several k-blocks, groups that straddle k-blocks, ragged O and I."""
    codes, gsc = _grouped(fmt, O, I, gs, O + gs)
    x = synth.activations(S, I, I, 5)
    y_ref, bound = oracle.matmul_gs(fmt, O, I, gs, codes, gsc, x)
    with q.tensor_upload(fmt, O, I, codes, gsc, gs=gs) as t:
        y = gpu_matmul(q, t, x, S, O, path=q.PATH_TC)
        y2 = empty(S, O)
        q.matmul_tc_noalloc(t, to_dev(x), y2, S)
        import torch
        torch.cuda.synchronize()
        y2 = y2.cpu().numpy()
    assert_within(y, y_ref, bound, TOL_TC, "tc gs fmt%d gs%d" % (fmt, gs))
    assert np.array_equal(y, y2)                            # the no-alloc call runs the same kernel


def test_group_scales_prefill_full_size_sampled(q):
    """int4 [12288, 6144] gs=128 at S=1571 on the tensor cores: 96 sampled rows
    (every tile row block) against the oracle run on those rows."""
    fmt, O, I, gs, S = 2, 12288, 6144, 128, 1571
    codes, gsc = _grouped(fmt, O, I, gs, 11)
    x = synth.activations(S, I, 11, 6)
    with q.tensor_upload(fmt, O, I, codes, gsc, gs=gs) as t:
        assert q.matmul_path(t, S) == q.PATH_TC
        y = gpu_matmul(q, t, x, S, O)
    rows = np.sort(synth.rng(11, 7).choice(O, 96, replace=False))
    y_ref, bound = oracle.matmul_gs(fmt, len(rows), I, gs, codes[rows], gsc[rows], x)
    assert_within(y[:, rows], y_ref, bound, TOL_TC, "tc gs full size")
