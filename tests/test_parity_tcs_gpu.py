"""GPU parity of the f32-accurate tensor-core path for few tokens
(B200Q_PATH_TCS: weights dequantized into tensor memory, x in two fp16 pieces
per token) against the CPU oracle, at the f32 bar:
|y - y_ref| <= 1e-5 * |scale| * sum |deq * x|.

Shapes cover tiles whose k-blocks are shared by several CTAs (partial planes
added by the second kernel) and tiles one CTA owns whole, ragged O and I,
S across the 16- and 32-column token tiles and past 16 rows (chunked),
one-hot rows (bit-exact), every code value, extreme token magnitudes and
tokens whose columns are zero in whole k-ranges.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_F32, assert_within, empty, gpu_matmul, inputs, to_dev

pytestmark = pytest.mark.gpu

FMTS = [(1, "i8"), (2, "i4"), (3, "i2")]


@pytest.fixture(scope="module")
def q():
    import torch
    torch.cuda.set_device(0)
    import quantized_weight_quant_gb300 as q
    return q


def _check(q, fmt, O, I, S, seed=0, x=None):
    codes, scales, x0 = inputs(fmt, O, I, S, seed)
    if x is None:
        x = x0
    y_ref, bound = oracle.matmul(fmt, O, I, codes, scales, x)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        y = gpu_matmul(q, t, x, S, O, q.PATH_TCS)
    assert_within(y, y_ref, bound, TOL_F32, "tcs fmt%d O%d I%d S%d" % (fmt, O, I, S))
    return y


@pytest.mark.parametrize("fmt", [f for f, _ in FMTS], ids=[n for _, n in FMTS])
@pytest.mark.parametrize("O,I", [(1, 1), (127, 63), (129, 256), (300, 257), (256, 1000), (77, 1024), (640, 3000)])
@pytest.mark.parametrize("S", [1, 2, 3, 8, 9, 16, 17])
def test_tcs_ragged(q, fmt, O, I, S):
    _check(q, fmt, O, I, S, seed=O * 7 + I)


@pytest.mark.parametrize("fmt", [f for f, _ in FMTS], ids=[n for _, n in FMTS])
@pytest.mark.parametrize("O,I", [(1024, 8192), (19456, 256), (152 * 128, 512), (12288, 640)])
def test_tcs_partitions(q, fmt, O, I):
    """Item counts that split tiles over CTAs at several offsets, and counts
    where every CTA owns whole tiles (no partial planes)."""
    for S in (1, 5):
        _check(q, fmt, O, I, S, seed=O + I + S)


@pytest.mark.parametrize("fmt", [f for f, _ in FMTS], ids=[n for _, n in FMTS])
@pytest.mark.parametrize("O,I,S", [(4000, 16384, 5), (4000, 16384, 8), (3000, 20000, 8)])
def test_tcs_several_ranges(q, fmt, O, I, S):
    """Long rows at 5-8 tokens: every CTA's k-blocks no longer fit its B
    slots at once, so K is cut into ranges (8 to 53 of them here), each tile
    is shared by the CTAs of all its ranges, and the CTA that brings the
    tile's arrival count to its number of pieces adds them."""
    _check(q, fmt, O, I, S, seed=O + S)


def test_tcs_several_ranges_extreme_x(q):
    """The same shared-tile path with tokens of very different magnitudes:
    every CTA's pieces carry their own power of two."""
    fmt, O, I, S = 2, 4000, 16384, 8
    codes, scales, x = inputs(fmt, O, I, S, seed=31)
    x = x.astype(np.float64)
    x[0] *= 2.0 ** -135
    x[1] *= 1e30
    x[2, : I // 2] = 0.0
    x[3] = 0.0
    x[4, 5] = 1e4
    y = _check(q, fmt, O, I, S, x=x.astype(np.float32))
    assert np.all(y[3] == 0)


@pytest.mark.parametrize("S", [1, 4])
def test_tcs_int4_12288x6144(q, S):
    """The headline decode shape, every output."""
    _check(q, 2, 12288, 6144, S)


@pytest.mark.parametrize("fmt", [f for f, _ in FMTS], ids=[n for _, n in FMTS])
@pytest.mark.parametrize("S", [1, 2, 8])
def test_tcs_format_sweep_8192(q, fmt, S):
    _check(q, fmt, 8192, 8192, S, seed=fmt)


@pytest.mark.parametrize("fmt", [f for f, _ in FMTS], ids=[n for _, n in FMTS])
def test_tcs_onehot_bit_exact(q, fmt):
    """One-hot x rows make each output a single rounding of scale * deq:
    bit-exact against the oracle (and the dequantization with it)."""
    O, I = 384, 256
    codes, scales, _ = inputs(fmt, O, I, 1, seed=9)
    x = np.eye(I, dtype=np.float32)[:48]
    y_ref, _ = oracle.matmul(fmt, O, I, codes, scales, x)
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        y = gpu_matmul(q, t, x, 48, O, q.PATH_TCS)
    assert np.array_equal(y, y_ref)


def test_tcs_exhaustive_codes(q):
    """Every int8 byte, int4 nibble and int2 field value through this path."""
    for fmt, I in ((1, 256), (2, 512), (3, 1024)):
        row = np.arange(256, dtype=np.uint8)[None, :]
        codes = np.repeat(row, 2, axis=0)
        scales = np.array([1.0, 0.5], np.float32)
        want = oracle.dequant_row(fmt, I, row[0])
        with q.tensor_upload(fmt, 2, I, codes, scales) as t:
            for s0 in range(0, I, 16):
                x = np.zeros((16, I), np.float32)
                x[np.arange(16), s0 + np.arange(16)] = 1.0
                y = gpu_matmul(q, t, x, 16, 2, q.PATH_TCS)
                assert np.array_equal(y[:, 0], want[s0:s0 + 16].astype(np.float32))
                assert np.array_equal(y[:, 1], (want[s0:s0 + 16] * 0.5).astype(np.float32))


@pytest.mark.parametrize("fmt", [f for f, _ in FMTS], ids=[n for _, n in FMTS])
def test_tcs_extreme_x_magnitudes(q, fmt):
    """Tokens far from unit scale (all subnormal, near 1e33, a 1e3 outlier,
    all zero): the per-token power of two keeps the pieces exact and in range."""
    O, I, S = 1024, 4096, 4
    codes, scales, x = inputs(fmt, O, I, S, seed=17)
    g = synth.rng(17, 5)
    x = x.astype(np.float64)
    x[0] = np.sign(x[0]) * g.uniform(1.0, 3.0, I) * 2.0 ** -140
    x[1] = x[1] * 1e33
    x[2, 7] = 1e3
    x[3] = 0.0
    x = x.astype(np.float32)
    y = _check(q, fmt, O, I, S, x=x)
    assert np.all(y[3] == 0)


@pytest.mark.parametrize("fmt", [f for f, _ in FMTS], ids=[n for _, n in FMTS])
def test_tcs_zero_column_ranges(q, fmt):
    """Tokens whose columns are zero over whole k-ranges (some CTAs of a shared
    tile see only zeros) next to tiny or huge values elsewhere: the partial
    planes' exponents must combine without losing the nonzero parts."""
    O, I, S = 512, 8192, 4
    codes, scales, x = inputs(fmt, O, I, S, seed=23)
    x = x.astype(np.float64)
    x[0, : I // 2] = 0.0
    x[0, I // 2:] *= 2.0 ** -130
    x[1, I // 3:] = 0.0
    x[1, : I // 3] *= 1e30
    x[2, : 7 * I // 8] = 0.0
    x[3, 100:] = 0.0
    _check(q, fmt, O, I, S, x=x.astype(np.float32))


def _digits(S):
    """Digits per token of a launch of S (<= 8) tokens: N = 16 ceil((7S+1)/16)
    columns, 8 digits where 8S + 1 of them fit, else 7."""
    n = 16 * -(-(7 * S + 1) // 16)
    return 8 if 8 * S + 1 <= n else 7


@pytest.mark.parametrize("fmt", [f for f, _ in FMTS], ids=[n for _, n in FMTS])
@pytest.mark.parametrize("S", [1, 2, 3, 4, 8])
def test_tcs_error_bound(q, fmt, S):
    """The path's own bound, far inside the f32 bar: x is the only thing
    rounded (to 4J-2 bits below its token's largest magnitude), so
    |y - y_exact| <= 2^(1-4J) max|x_s| sum_i |scale deq| plus y's rounding."""
    O, I = 1024, 4096
    codes, scales, x = inputs(fmt, O, I, S, seed=7 + S)
    _, _, ydbl = oracle.matmul(fmt, O, I, codes, scales, x, want_dbl=True)
    _, absrow = oracle.matmul(fmt, O, I, codes, scales, np.ones((1, I), np.float32))   # sum_i |scale deq|
    with q.tensor_upload(fmt, O, I, codes, scales) as t:
        y = gpu_matmul(q, t, x, S, O, q.PATH_TCS).astype(np.float64)
    J = _digits(S)
    xmax = np.abs(x.astype(np.float64)).max(axis=1, keepdims=True)
    tol = 2.0 ** (1 - 4 * J) * xmax * absrow[0][None, :] + 2.0 ** -24 * np.abs(ydbl) + 1e-300
    err = np.abs(y - ydbl)
    assert np.all(err <= tol), float((err / tol).max())


def test_tcs_repeatable(q):
    codes, scales, x = inputs(2, 1024, 4096, 5, seed=3)
    with q.tensor_upload(2, 1024, 4096, codes, scales) as t:
        y1 = gpu_matmul(q, t, x, 5, 1024, q.PATH_TCS)
        y2 = gpu_matmul(q, t, x, 5, 1024, q.PATH_TCS)
    assert np.array_equal(y1, y2)


def test_tcs_gate_up_pair(q):
    import torch
    fmt, O, I, S = 2, 2048, 6144, 3
    cg, sg = synth.quant_tensor(fmt, O, I, 0, 41, 5e-3, 2e-2)
    cu, su = synth.quant_tensor(fmt, O, I, 0, 42, 5e-3, 2e-2)
    x = synth.activations(S, I, 0, 43)
    yg_ref, bg, yu_ref, bu = oracle.matmul_gate_up(fmt, O, I, cg, sg, cu, su, x)
    with q.tensor_upload(fmt, O, I, cg, sg) as tg, q.tensor_upload(fmt, O, I, cu, su) as tu:
        yg = gpu_matmul(q, tg, x, S, O, q.PATH_TCS)
        yu = gpu_matmul(q, tu, x, S, O, q.PATH_TCS)
    assert_within(yg, yg_ref, bg, TOL_F32, "gate")
    assert_within(yu, yu_ref, bu, TOL_F32, "up")


def test_tcs_rejects_f32_and_group_scales(q):
    codes, scales, x = inputs(0, 16, 64, 2)
    with q.tensor_upload(0, 16, 64, codes, scales) as t:
        with pytest.raises(q.B200QError):
            q.matmul_ex(t, to_dev(x), empty(2, 16), 2, q.PATH_TCS)
    codes = synth.codes(2, 16, 64, 0, 1)
    gsc = synth.uniform_f32((16, 2), 5e-3, 2e-2, 0, 2)
    with q.tensor_upload(2, 16, 64, codes, gsc, gs=32) as t:
        with pytest.raises(q.B200QError):
            q.matmul_ex(t, to_dev(np.zeros((2, 64), np.float32)), empty(2, 16), 2, q.PATH_TCS)


def test_tcs_device_status_clean(q):
    codes, scales, x = inputs(2, 256, 2048, 3)
    with q.tensor_upload(2, 256, 2048, codes, scales) as t:
        gpu_matmul(q, t, x, 3, 256, q.PATH_TCS)
    assert q.device_status() == q.OK
