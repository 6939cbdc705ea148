"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each ``check_*`` raises AssertionError on a mismatch.  They call the oracle only
through the ``oracle`` module's functions, so the mutation tests can run the
same checks against copies of ``qref.c`` with planted mistakes and require that
every planted mistake is caught.

What fixes each expected value (none of them is the oracle's own output):
  * worked examples expanded by hand (tests/golden/worked_examples.txt);
  * code tables written out literally, or read off by numpy's int8 view and by
    Python's hex / base-4 digit formatting (all 256 byte values);
  * one-hot rows with power-of-two x, so the position a code lands in is read
    off the exponent of the result;
  * closed forms (constant codes against x = 1 or alternating +-1, identity W);
  * invariants (power-of-two scaling is exact, linearity in x, bound >= |y|);
  * reductions to library routines (numpy float64 matmul on the int8 / f32
    views of the codes, numpy unpackbits for int4 / int2, torch silu, torch
    bfloat16 rounding).
"""
from __future__ import annotations

import os

import numpy as np

import oracle as Q
import synth

F32, I8, I4, I2 = Q.F32, Q.I8, Q.I4, Q.I2
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "worked_examples.txt")

# Values of every code, written out (int4: code - 8; int2: code - 2).
INT4_VALUES = [-8, -7, -6, -5, -4, -3, -2, -1, 0, 1, 2, 3, 4, 5, 6, 7]
INT2_VALUES = [-2, -1, 0, 1]


def load_golden(path: str = GOLDEN):
    cases, cur = [], None
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0], "codes": [], "weights": [], "x": [], "y": [], "bound": []}
            cases.append(cur)
        elif key in ("fmt", "O", "I"):
            cur[key] = int(vals[0])
        elif key == "codes":
            cur["codes"] = [bytes.fromhex(v) for v in vals]
        elif key == "scales":
            cur["scales"] = [float(v) for v in vals]
        else:
            cur[key].append([float(v) for v in vals])
    return cases


def _golden_codes(c):
    if c["fmt"] == F32:
        return np.array(c["weights"], np.float32).view(np.uint8)
    return np.frombuffer(b"".join(c["codes"]), np.uint8).reshape(c["O"], -1)


def check_worked_examples():
    cases = load_golden()
    assert len(cases) == 4
    for c in cases:
        y, bound = Q.matmul(c["fmt"], c["O"], c["I"], _golden_codes(c),
                            np.array(c["scales"], np.float32), np.array(c["x"], np.float32))
        assert np.array_equal(y, np.array(c["y"], np.float32)), (c["name"], y)
        assert np.array_equal(bound, np.array(c["bound"], np.float64)), (c["name"], bound)


def check_int8_table():
    row = np.arange(256, dtype=np.uint8)
    got = Q.dequant_row(I8, 256, row)
    want = row.view(np.int8).astype(np.float64)          # numpy's two's-complement view
    assert np.array_equal(got, want)
    assert got[0x7F] == 127 and got[0x80] == -128 and got[0xFF] == -1 and got[0x81] == -127


def check_int4_table():
    row = np.arange(256, dtype=np.uint8)
    got = Q.dequant_row(I4, 512, row)
    want = []
    for b in range(256):
        hi, lo = "%02x" % b                               # hex digits: high, low nibble
        want += [INT4_VALUES[int(lo, 16)], INT4_VALUES[int(hi, 16)]]
    assert np.array_equal(got, np.array(want, np.float64))
    # code 8 is zero, code 0 is -8, code 15 is +7
    assert Q.dequant_row(I4, 2, np.array([0x88], np.uint8)).tolist() == [0.0, 0.0]
    assert Q.dequant_row(I4, 2, np.array([0xF0], np.uint8)).tolist() == [-8.0, 7.0]


def check_int2_table():
    row = np.arange(256, dtype=np.uint8)
    got = Q.dequant_row(I2, 1024, row)
    want = []
    for b in range(256):
        d = np.base_repr(b, 4).zfill(4)                   # base-4 digits, most significant first
        want += [INT2_VALUES[int(ch)] for ch in reversed(d)]
    assert np.array_equal(got, np.array(want, np.float64))
    assert Q.dequant_row(I2, 4, np.array([0xAA], np.uint8)).tolist() == [0.0] * 4
    assert Q.dequant_row(I2, 4, np.array([0xE4], np.uint8)).tolist() == [-2.0, -1.0, 0.0, 1.0]


def check_zero_point_rows():
    x = synth.activations(3, 40, 0, 1)
    for fmt, byte in ((I4, 0x88), (I2, 0xAA), (I8, 0x00)):
        rb = Q.row_bytes(fmt, 40)
        codes = np.full((5, rb), byte, np.uint8)
        y, bound = Q.matmul(fmt, 5, 40, codes, np.ones(5, np.float32), x)
        assert not y.any() and not bound.any()


# One-hot rows, written out byte by byte: the value +7 (int4 code 15), +1
# (int2 code 3) or +5 (int8) at position p, zero-point codes elsewhere.
ONE_HOT = {
    I4: (4, [bytes([0x8F, 0x88]), bytes([0xF8, 0x88]), bytes([0x88, 0x8F]), bytes([0x88, 0xF8])], 7.0),
    I2: (4, [bytes([0xAB]), bytes([0xAE]), bytes([0xBA]), bytes([0xEA])], 1.0),
    I8: (4, [bytes([5, 0, 0, 0]), bytes([0, 5, 0, 0]), bytes([0, 0, 5, 0]), bytes([0, 0, 0, 5])], 5.0),
}


def check_bit_order():
    for fmt, (I, rows, v) in ONE_HOT.items():
        O = len(rows)
        codes = np.frombuffer(b"".join(rows), np.uint8).reshape(O, -1)
        scales = np.array([1.0, 0.5, 2.0, 4.0], np.float32)
        # x row 0 = 2^i, x row 1 = 3 * 2^(i+4): the result names the position
        x = np.array([[2.0 ** i for i in range(I)], [3.0 * 2.0 ** (i + 4) for i in range(I)]],
                     np.float32)
        y, _ = Q.matmul(fmt, O, I, codes, scales, x)
        for p in range(O):
            assert y[0, p] == scales[p] * v * 2.0 ** p, (fmt, p, y[:, p])
            assert y[1, p] == scales[p] * v * 3.0 * 2.0 ** (p + 4), (fmt, p, y[:, p])


def check_closed_forms():
    I = 1000
    ones = np.ones((1, I), np.float32)
    alt = np.array([[1.0 if i % 2 == 0 else -1.0 for i in range(I)]], np.float32)
    for fmt, byte, value in ((I4, 0xFF, 7), (I4, 0x00, -8), (I2, 0x00, -2), (I2, 0xFF, 1),
                             (I8, 0x9C, -100), (I8, 0x64, 100)):
        rb = Q.row_bytes(fmt, I)
        codes = np.full((3, rb), byte, np.uint8)
        sc = np.array([0.25, 1.0, 3.0], np.float32)
        y, b = Q.matmul(fmt, 3, I, codes, sc, ones)
        assert np.array_equal(y[0], sc * value * I)
        assert np.array_equal(b[0], np.abs(sc).astype(np.float64) * abs(value) * I)
        y, _ = Q.matmul(fmt, 3, I, codes, sc, alt)
        assert not y.any()
    # f32 identity with no scales gives x back
    n = 5
    W = np.eye(n, dtype=np.float32)
    x = synth.activations(3, n, 0, 7)
    y, _ = Q.matmul(F32, n, n, W.view(np.uint8), None, x)
    assert np.array_equal(y, x)


def check_single_rounding():
    # The result is the exact scale * sum rounded once to f32.  Worked by hand:
    # W = [1, 2^-24, 2^-40] (f32), x = 1, scale = 1.5.  Exact value
    # 1.5 + 0.75*2^-23*(1 + 2^-16) lies nearest to 1.5 + 2^-23.  Rounding the
    # sum to f32 first (1 + 2^-23) and then scaling would land on the tie
    # 1.5 + 1.5*2^-23 and round to 1.5 + 2^-22 instead.
    W = np.array([[1.0, 2.0 ** -24, 2.0 ** -40]], np.float32)
    y, _ = Q.matmul(F32, 1, 3, W.view(np.uint8), np.array([1.5], np.float32),
                    np.ones((1, 3), np.float32))
    assert y[0, 0] == np.float32(1.5 + 2.0 ** -23)


def check_scale_power_of_two():
    for fmt in (F32, I8, I4, I2):
        O, I, S = 9, 37, 3
        codes, sc = synth.quant_tensor(fmt, O, I, 3, 10 + fmt, 1e-3, 2e-2)
        x = synth.activations(S, I, 3, 20 + fmt)
        y1, b1 = Q.matmul(fmt, O, I, codes, sc, x)
        for k in (-3, 5):
            y2, b2 = Q.matmul(fmt, O, I, codes, sc * np.float32(2.0 ** k), x)
            assert np.array_equal(y2, y1 * np.float32(2.0 ** k))
            assert np.array_equal(b2, b1 * 2.0 ** k)
        # a negative scale flips y and keeps the bound
        y3, b3 = Q.matmul(fmt, O, I, codes, -sc, x)
        assert np.array_equal(y3, -y1) and np.array_equal(b3, b1)


def check_linearity():
    # small-integer x so that a*x1 + b*x2 is exact in f32 and every partial
    # sum is exact in double: then linearity holds exactly
    g = synth.rng(5, 1)
    for fmt in (I8, I4, I2):
        O, I = 7, 64
        codes, _ = synth.quant_tensor(fmt, O, I, 5, 30 + fmt, 1e-3, 2e-2)
        x1 = g.integers(-50, 51, size=(2, I)).astype(np.float32)
        x2 = g.integers(-50, 51, size=(2, I)).astype(np.float32)
        a, b = 3.0, -2.0
        _, _, y1 = Q.matmul(fmt, O, I, codes, None, x1, want_dbl=True)
        _, _, y2 = Q.matmul(fmt, O, I, codes, None, x2, want_dbl=True)
        _, _, y12 = Q.matmul(fmt, O, I, codes, None, a * x1 + b * x2, want_dbl=True)
        assert np.array_equal(y12, a * y1 + b * y2)


def check_bound_dominates():
    for fmt in (F32, I8, I4, I2):
        O, I, S = 11, 50, 2
        codes, sc = synth.quant_tensor(fmt, O, I, 6, 40 + fmt, 1e-3, 2e-2)
        x = synth.activations(S, I, 6, 50 + fmt)
        y, b, yd = Q.matmul(fmt, O, I, codes, sc, x, want_dbl=True)
        assert (b >= np.abs(yd)).all() and (b > 0).all()
        # all terms non-negative: bound equals y
        xp = np.abs(x)
        codes_p = np.full_like(codes, {F32: 0, I8: 0x11, I4: 0xCC, I2: 0xFF}[fmt])
        if fmt == F32:
            codes_p = np.abs(codes.view(np.float32)).view(np.uint8)
        y, b, yd = Q.matmul(fmt, O, I, codes_p, sc, xp, want_dbl=True)
        assert np.allclose(b, yd, rtol=1e-15, atol=0)


def _unpack_fields(codes, fmt, I):
    """Library route for int4 / int2: numpy unpackbits (LSB first) then a
    weighted sum of bit planes."""
    bits = np.unpackbits(codes, axis=1, bitorder="little").astype(np.int64)
    b = {I4: 4, I2: 2}[fmt]
    fields = bits.reshape(codes.shape[0], -1, b) @ (1 << np.arange(b))
    return fields[:, :I]


def check_library_reduction():
    O, I, S = 13, 45, 3                                   # O != I != S, ragged I
    for fmt in (F32, I8, I4, I2):
        codes, sc = synth.quant_tensor(fmt, O, I, 8, 60 + fmt, 1e-3, 2e-2)
        x = synth.activations(S, I, 8, 70 + fmt)
        _, bound, yd = Q.matmul(fmt, O, I, codes, sc, x, want_dbl=True)
        if fmt == F32:
            W = codes.view(np.float32).astype(np.float64)
        elif fmt == I8:
            W = codes.view(np.int8).astype(np.float64)
        else:
            W = (_unpack_fields(codes, fmt, I) - {I4: 8, I2: 2}[fmt]).astype(np.float64)
        ref = (x.astype(np.float64) @ W.T) * sc.astype(np.float64)
        assert np.all(np.abs(ref - yd) <= 1e-13 * bound), fmt
        absref = np.abs(x.astype(np.float64)) @ np.abs(W.T) * np.abs(sc.astype(np.float64))
        assert np.allclose(absref, bound, rtol=1e-13, atol=0)


def check_gate_up():
    O, I, S = 6, 33, 2
    cg, sg = synth.quant_tensor(I4, O, I, 9, 1, 5e-3, 2e-2)
    cu, su = synth.quant_tensor(I4, O, I, 9, 2, 5e-3, 2e-2)
    x = synth.activations(S, I, 9, 3)
    yg, bg, yu, bu = Q.matmul_gate_up(I4, O, I, cg, sg, cu, su, x)
    yg1, bg1 = Q.matmul(I4, O, I, cg, sg, x)
    yu1, bu1 = Q.matmul(I4, O, I, cu, su, x)
    assert np.array_equal(yg, yg1) and np.array_equal(yu, yu1)
    assert np.array_equal(bg, bg1) and np.array_equal(bu, bu1)
    assert not np.array_equal(yg, yu)


def check_silu():
    import torch
    g = np.array([0.0, 1.0, -1.0, 5.0, -5.0, 30.0, -30.0, 0.125], np.float32)
    u = np.array([1.0, 2.0, 0.5, -1.0, 3.0, 1.0, 1.0, -4.0], np.float32)
    h, hd = Q.silu_mul(g, u)
    ref = torch.nn.functional.silu(torch.from_numpy(g.astype(np.float64))).numpy() * u
    assert np.allclose(hd, ref, rtol=1e-15, atol=1e-300)
    assert hd[0] == 0.0
    assert abs(hd[5] - 30.0) < 1e-11                     # silu(z) -> z for large z
    assert abs(hd[6]) < 1e-11                            # silu(z) -> 0 for very negative z
    assert np.array_equal(h, hd.astype(np.float32))


def check_group_scales():
    """Group-wise scales: one group is the per-row scale exactly; a hand-worked
    group size 1; a short last group; per-group linearity; the bound."""
    # gs = I: bit for bit the per-row matmul
    c, sc = synth.quant_tensor(2, 5, 40, 0, 1, 5e-3, 2e-2)
    x = synth.activations(3, 40, 0, 2)
    y1, b1 = Q.matmul(2, 5, 40, c, sc, x)
    y2, b2 = Q.matmul_gs(2, 5, 40, 40, c, sc.reshape(5, 1), x)
    assert np.array_equal(y1, y2) and np.allclose(b1, b2, rtol=1e-15, atol=0)
    # gs = 1, int8 codes [1, -2, 3], scales [0.5, 2, -1], x [2, 1, 4]:
    # 0.5*1*2 + 2*(-2)*1 + (-1)*3*4 = -15, bound 1 + 4 + 12 = 17
    codes = np.array([[1, 0xFE, 3]], np.uint8)
    y, b, yd = Q.matmul_gs(1, 1, 3, 1, codes, np.array([[0.5, 2.0, -1.0]], np.float32),
                           np.array([[2.0, 1.0, 4.0]], np.float32), want_dbl=True)
    assert yd[0, 0] == -15.0 and b[0, 0] == 17.0
    # int4, I = 5, gs = 2: groups {0, 1}, {2, 3}, {4}; codes 9, 10, 6, 8, 15 -> 1, 2, -2, 0, 7
    codes = np.array([[0xA9, 0x86, 0x0F]], np.uint8)
    gsc = np.array([[1.0, 0.25, -0.5]], np.float32)
    xx = np.array([[1.0, 2.0, 3.0, 4.0, 2.0]], np.float32)
    _, b, yd = Q.matmul_gs(2, 1, 5, 2, codes, gsc, xx, want_dbl=True)
    # 1*(1*1 + 2*2) + 0.25*(-2*3 + 0*4) + (-0.5)*(7*2) = 5 - 1.5 - 7 = -3.5; bound 5 + 1.5 + 7
    assert yd[0, 0] == -3.5 and b[0, 0] == 13.5
    # doubling one group's scale adds exactly that group's contribution again
    gs, I = 16, 70
    c, _ = synth.quant_tensor(2, 3, I, 0, 3, 5e-3, 2e-2)
    G = -(-I // gs)
    gsc = synth.uniform_f32((3, G), 5e-3, 2e-2, 0, 4)
    x = synth.activations(2, I, 0, 5)
    _, _, y0 = Q.matmul_gs(2, 3, I, gs, c, gsc, x, want_dbl=True)
    g2 = gsc.copy()
    g2[:, 2] *= 2.0
    _, _, y2 = Q.matmul_gs(2, 3, I, gs, c, g2, x, want_dbl=True)
    only = np.zeros_like(gsc)
    only[:, 2] = gsc[:, 2]
    _, _, yg = Q.matmul_gs(2, 3, I, gs, c, only, x, want_dbl=True)
    assert np.allclose(y2 - y0, yg, rtol=1e-12, atol=1e-18)
    # the last (short) group matters: zeroing its scale removes element 64..69
    z = gsc.copy()
    z[:, G - 1] = 0.0
    _, _, yz = Q.matmul_gs(2, 3, I, gs, c, z, x, want_dbl=True)
    lastonly = np.zeros_like(gsc)
    lastonly[:, G - 1] = gsc[:, G - 1]
    _, _, yl = Q.matmul_gs(2, 3, I, gs, c, lastonly, x, want_dbl=True)
    assert np.allclose(y0 - yz, yl, rtol=1e-12, atol=1e-18) and np.any(yl != 0)


def check_rmsnorm():
    """RMSNorm (textbook, the pages name it without printing it): a worked
    example by hand, closed forms, the residual sum, the eps term, row
    independence and scale invariance."""
    one = np.ones(2, np.float32)
    # [3, 4]: mean square 12.5, y = [3, 4] / sqrt(12.5)
    _, y, yd = Q.rmsnorm(np.array([[3.0, 4.0]], np.float32), one, 0.0)
    assert np.allclose(yd, [[0.848528137423857, 1.131370849898476]], rtol=1e-14, atol=0)
    # the weight multiplies per element
    _, _, yd = Q.rmsnorm(np.array([[3.0, 4.0]], np.float32), np.array([2.0, -1.0], np.float32), 0.0)
    assert np.allclose(yd, [[1.697056274847714, -1.131370849898476]], rtol=1e-14, atol=0)
    # a constant row c: h / |c| = sign(c), so y = -w exactly for c = -2
    w5 = np.array([1.0, 0.5, -3.0, 2.0, 0.25], np.float32)
    _, y, yd = Q.rmsnorm(np.full((1, 5), -2.0, np.float32), w5, 0.0)
    assert np.array_equal(yd[0], -w5.astype(np.float64)) and np.array_equal(y[0], -w5)
    # eps enters under the root: [1, 1] with eps 3 -> 1 / sqrt(1 + 3) = 0.5
    _, _, yd = Q.rmsnorm(np.array([[1.0, 1.0]], np.float32), one, 3.0)
    assert np.array_equal(yd, [[0.5, 0.5]])
    # residual: h = x + r = [4, 0], mean square 8, y = [sqrt 2, 0]
    h, _, yd = Q.rmsnorm(np.array([[1.0, 2.0]], np.float32), one, 0.0, r=np.array([[3.0, -2.0]], np.float32))
    assert np.array_equal(h, [[4.0, 0.0]])
    assert abs(yd[0, 0] - np.sqrt(2.0)) < 1e-15 and yd[0, 1] == 0.0
    # rows are normalized independently; a power-of-two scale of a row cancels exactly
    g = synth.rng(5, 0)
    x = g.standard_normal((2, 7)).astype(np.float32)
    w7 = g.uniform(0.5, 2.0, 7).astype(np.float32)
    _, y, yd = Q.rmsnorm(x, w7, 0.0)
    _, y4, yd4 = Q.rmsnorm(np.stack([x[0] * 4.0, x[1]]).astype(np.float32), w7, 0.0)
    assert np.array_equal(y4, y) and np.allclose(yd4, yd, rtol=1e-15)
    _, y1, _ = Q.rmsnorm(x[1:], w7, 0.0)
    assert np.array_equal(y1[0], y[1])
    # mean of squares: sum of y^2 / w^2 equals D (eps = 0)
    assert abs(np.sum((yd[0] / w7) ** 2) - 7.0) < 1e-12


def check_round_bf16():
    import torch
    one = 1.0
    cases = {
        one: one,
        one + 2.0 ** -8: one,                             # tie -> even (1.0)
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,             # tie -> even (1 + 2^-6)
        one + 2.0 ** -8 + 2.0 ** -20: one + 2.0 ** -7,    # above the tie
        -(one + 2.0 ** -8): -one,
        0.0: 0.0,
    }
    for v, want in cases.items():
        got = float(Q.round_bf16(np.array([v], np.float32))[0])
        want_bf = float(torch.tensor([want], dtype=torch.float32).to(torch.bfloat16).float()[0])
        assert got == want_bf, (v, got, want_bf)
    v = synth.activations(1, 2000, 11, 1)[0] * np.float32(37.0)
    v = v * np.float32(2.0) ** synth.rng(11, 2).integers(-100, 100, size=v.shape).astype(np.float32)
    got = Q.round_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    assert np.array_equal(got, ref)


def check_row_bytes():
    assert [Q.row_bytes(I4, n) for n in (0, 1, 2, 3, 6144)] == [0, 1, 1, 2, 3072]
    assert [Q.row_bytes(I2, n) for n in (1, 4, 5, 8192)] == [1, 1, 2, 2048]
    assert [Q.row_bytes(I8, n) for n in (1, 513)] == [1, 513]
    assert [Q.row_bytes(F32, n) for n in (1, 3)] == [4, 12]
    assert Q.row_bytes(7, 4) == -1


def _dense_weights(fmt, codes, sc, O, I):
    """Weight values scale * (code - zero point) by the library routes of
    check_library_reduction, [O, I] float64."""
    if fmt == F32:
        W = codes.view(np.float32).astype(np.float64)
    elif fmt == I8:
        W = codes.view(np.int8).astype(np.float64)
    else:
        W = (_unpack_fields(codes, fmt, I) - {I4: 8, I2: 2}[fmt]).astype(np.float64)
    return W * sc.astype(np.float64)[:, None]


def _mla_case(fmt, H, Dn, Dv, K, R, S, T, seed, gs=0):
    codes, sc = synth.quant_tensor(fmt, H * (Dn + Dv), K, seed, 1, 5e-3, 2e-2)
    if gs:
        sc = synth.uniform_f32((H * (Dn + Dv), -(-K // gs)), 5e-3, 2e-2, seed, 6)
    qn = synth.normal_f32((S, H, Dn), seed, 2, std=4.0)
    qr = synth.normal_f32((S, H, R), seed, 3)
    lat = synth.normal_f32((T, K), seed, 4)
    rope = synth.normal_f32((T, R), seed, 5)
    return codes, sc, qn, qr, lat, rope


MLA_CASES = [  # fmt, H, Dn, Dv, K, R, S, T, st0, scale, gs
    (I4, 3, 8, 5, 40, 6, 3, 11, 2, 0.3, 0),
    (I8, 2, 4, 7, 33, 4, 1, 9, 0, 0.5, 0),
    (F32, 2, 6, 6, 20, 2, 2, 5, 3, 1.0, 0),
    (I2, 4, 3, 2, 27, 3, 4, 12, 1, 0.7, 0),
    (I4, 2, 5, 4, 48, 4, 2, 10, 1, 0.4, 16),     # group-wise scales, 3 groups per row
    (I8, 3, 4, 6, 40, 4, 1, 8, 0, 0.6, 12),      # a short last group
]


def check_mla_naive():
    """Absorption is an identity: decompress every position's keys and values
    (k_t = Wk L_t, v_t = Wv L_t, the non-absorbed MLA form), then textbook
    causal attention over [st0, T-S+s] in numpy float64.  The error bound is
    recomputed from its definition."""
    for fmt, H, Dn, Dv, K, R, S, T, st0, scale, gs in MLA_CASES:
        codes, sc, qn, qr, lat, rope = _mla_case(fmt, H, Dn, Dv, K, R, S, T, 11 + fmt, gs)
        _, bound, cd = Q.mla_absorb(fmt, H, Dn, Dv, K, codes, sc, qn, qr, lat, rope, st0, scale, gs=gs,
                                    want_dbl=True)
        if gs:      # scale of column i: its group's, expanded over the row
            ones = np.ones(H * (Dn + Dv), np.float32)
            W = _dense_weights(fmt, codes, ones, H * (Dn + Dv), K) * np.repeat(sc.astype(np.float64), gs, 1)[:, :K]
        else:
            W = _dense_weights(fmt, codes, sc, H * (Dn + Dv), K)
        W = W.reshape(H, Dn + Dv, K)
        Wk, Wv = W[:, :Dn], W[:, Dn:]
        L, Rr = lat.astype(np.float64), rope.astype(np.float64)
        keys = np.einsum("hdk,tk->thd", Wk, L)
        vals = np.einsum("hvk,tk->thv", Wv, L)
        for s in range(S):
            win = np.arange(st0, T - S + s + 1)
            for h in range(H):
                z = (keys[win, h] @ qn[s, h].astype(np.float64) + Rr[win] @ qr[s, h].astype(np.float64)) * scale
                p = np.exp(z - z.max())
                p /= p.sum()
                ref = p @ vals[win, h]
                assert np.all(np.abs(cd[s, h] - ref) <= 1e-12 * bound[s, h]), (fmt, s, h)
                qa = np.abs(Wk[h] * qn[s, h].astype(np.float64)[:, None]).sum(0)
                A = (np.abs(L[win]) @ qa + np.abs(Rr[win] * qr[s, h].astype(np.float64)).sum(1)).max() * abs(scale)
                b = (1 + A) * (np.abs(Wv[h]) @ (p @ np.abs(L[win])))
                assert np.allclose(bound[s, h], b, rtol=1e-12, atol=0), (fmt, s, h)


def check_mla_uniform_window():
    """With q = 0 (or scale = 0) every score is equal: the context is the plain
    mean of the latent rows in the window, through the value rows."""
    fmt, H, Dn, Dv, K, R, S, T = I4, 2, 5, 4, 24, 4, 3, 10
    codes, sc, qn, qr, lat, rope = _mla_case(fmt, H, Dn, Dv, K, R, S, T, 21)
    Wv = _dense_weights(fmt, codes, sc, H * (Dn + Dv), K).reshape(H, Dn + Dv, K)[:, Dn:]
    for st0 in (0, 4, T - S):
        for args in ((np.zeros_like(qn), np.zeros_like(qr), 0.9), (qn, qr, 0.0)):
            _, bound, cd = Q.mla_absorb(fmt, H, Dn, Dv, K, codes, sc, args[0], args[1], lat, rope, st0, args[2],
                                        want_dbl=True)
            for s in range(S):
                mean = lat[st0:T - S + s + 1].astype(np.float64).mean(0)
                for h in range(H):
                    assert np.all(np.abs(cd[s, h] - Wv[h] @ mean) <= 1e-12 * bound[s, h]), (st0, s, h)


def check_mla_window_edges():
    """Latent and rope rows outside a token's window do not move its context;
    the first and last rows inside it do."""
    fmt, H, Dn, Dv, K, R, S, T, st0 = I8, 2, 4, 3, 16, 4, 3, 9, 2
    codes, sc, qn, qr, lat, rope = _mla_case(fmt, H, Dn, Dv, K, R, S, T, 31)
    base, _ = Q.mla_absorb(fmt, H, Dn, Dv, K, codes, sc, qn, qr, lat, rope, st0, 0.4)
    for t in range(T):
        for which in ("lat", "rope"):
            l2, r2 = lat.copy(), rope.copy()
            (l2 if which == "lat" else r2)[t] += np.float32(3.0)
            got, _ = Q.mla_absorb(fmt, H, Dn, Dv, K, codes, sc, qn, qr, l2, r2, st0, 0.4)
            for s in range(S):
                inside = st0 <= t <= T - S + s
                same = np.array_equal(got[s], base[s])
                assert same != inside, (which, t, s)


def check_mla_shift_invariance():
    """Adding one vector to every rope row shifts all of a token's scores by the
    same amount, which the softmax ignores."""
    fmt, H, Dn, Dv, K, R, S, T = I4, 2, 4, 4, 24, 6, 2, 8
    codes, sc, qn, qr, lat, rope = _mla_case(fmt, H, Dn, Dv, K, R, S, T, 41)
    rope = np.round(rope * 64) / np.float32(64)               # on a 1/64 grid: the shift below is exact
    _, bound, cd = Q.mla_absorb(fmt, H, Dn, Dv, K, codes, sc, qn, qr, lat, rope, 1, 0.5, want_dbl=True)
    shifted = rope + synth.rng(41, 9).integers(-3, 4, size=(1, R)).astype(np.float32)
    _, _, cd2 = Q.mla_absorb(fmt, H, Dn, Dv, K, codes, sc, qn, qr, lat, shifted, 1, 0.5, want_dbl=True)
    assert np.all(np.abs(cd - cd2) <= 1e-12 * bound)
    assert not np.array_equal(Q.mla_absorb(fmt, H, Dn, Dv, K, codes, sc, qn, qr * 2, lat, rope, 1, 0.5)[0],
                              Q.mla_absorb(fmt, H, Dn, Dv, K, codes, sc, qn, qr, lat, rope, 1, 0.5)[0])


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
