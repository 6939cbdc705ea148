"""ctypes binding of the CPU oracle in ``qref.c``.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain definition of the
quantized-weight matmul that the CUDA library is checked against.  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
import this package; the library under ``quantized_weight_quant_gb300`` never
does, and this package imports nothing from it.

Every function takes and returns numpy arrays in the host layout the pages
describe: codes are row-major ``[O, row_bytes(fmt, I)]`` bytes (int4 low nibble
first, int2 low bits first), scales ``[O]`` f32 (or None = 1.0), x ``[S, I]``
f32.  Results: y ``[S, O]`` f32 rounded once from a double accumulation, and
bound ``[S, O]`` f64 = |scale| * sum |deq(W) x| for the parity tolerance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, I8, I4, I2 = 0, 1, 2, 3
ZERO_POINT = {F32: 0, I8: 0, I4: 8, I2: 2}
BITS = {F32: 32, I8: 8, I4: 4, I2: 2}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qref.c")
_LIB = os.path.join(_HERE, "libqref.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile qref.c (plain C99, -O2, no fast-math, OpenMP) into libqref.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-std=c99", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-Wall", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    L = ctypes.CDLL(path)
    c_long, c_int, vp = ctypes.c_long, ctypes.c_int, ctypes.c_void_p
    L.qref_row_bytes.argtypes = [c_int, c_long]
    L.qref_row_bytes.restype = c_long
    L.qref_weight.argtypes = [c_int, vp, c_long]
    L.qref_weight.restype = ctypes.c_double
    L.qref_dequant_row.argtypes = [c_int, c_long, vp, vp]
    L.qref_dequant_row.restype = c_int
    L.qref_set_threads.argtypes = [c_int]
    L.qref_set_threads.restype = None
    L.qref_max_threads.argtypes = []
    L.qref_max_threads.restype = c_int
    L.qref_matmul.argtypes = [c_int, c_long, c_long, vp, vp, vp, c_long, vp, vp, vp]
    L.qref_matmul.restype = c_int
    L.qref_matmul_gate_up.argtypes = [c_int, c_long, c_long, vp, vp, vp, vp, vp,
                                      c_long, vp, vp, vp, vp]
    L.qref_matmul_gate_up.restype = c_int
    L.qref_silu_mul.argtypes = [vp, vp, c_long, vp, vp]
    L.qref_silu_mul.restype = None
    L.qref_matmul_gs.argtypes = [c_int, c_long, c_long, c_long, vp, vp, vp, c_long, vp, vp, vp]
    L.qref_matmul_gs.restype = c_int
    L.qref_rmsnorm.argtypes = [vp, vp, vp, c_long, c_long, ctypes.c_double, vp, vp, vp]
    L.qref_rmsnorm.restype = c_int
    L.qref_mla_absorb.argtypes = [c_int, c_long, c_long, c_long, c_long, c_long, vp, vp, c_long, vp, vp, vp, vp,
                                  c_long, c_long, ctypes.c_double, c_long, vp, vp, vp]
    L.qref_mla_absorb.restype = c_int
    L.qref_round_bf16.argtypes = [ctypes.c_float]
    L.qref_round_bf16.restype = ctypes.c_float
    L.qref_matmul_bf16x.argtypes = [c_int, c_long, c_long, vp, vp, vp, c_long, vp,
                                    vp, vp, vp]
    L.qref_matmul_bf16x.restype = c_int
    return L


def lib():
    """The compiled oracle (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


_override = threading.local()


def _L():
    o = getattr(_override, "lib", None)
    return o if o is not None else lib()


class using:
    """Context manager: route this module's functions to another compiled copy
    of qref.c (the mutation tests plant mistakes in copies of the source)."""

    def __init__(self, so_path: str):
        self._L = _bind(so_path)

    def __enter__(self):
        self._prev = getattr(_override, "lib", None)
        _override.lib = self._L
        return self

    def __exit__(self, *exc):
        _override.lib = self._prev
        return False


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def row_bytes(fmt: int, I: int) -> int:
    return int(_L().qref_row_bytes(fmt, I))


def set_threads(n: int) -> None:
    """Number of OpenMP threads the oracle uses (0 = all)."""
    _L().qref_set_threads(int(n))


def max_threads() -> int:
    return int(_L().qref_max_threads())


def dequant_row(fmt: int, I: int, row: np.ndarray) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    assert row.size >= row_bytes(fmt, I)
    out = np.empty(I, np.float64)
    rc = _L().qref_dequant_row(fmt, I, _ptr(row), _ptr(out))
    if rc:
        raise ValueError("bad format")
    return out


def _check_codes(fmt, O, I, codes):
    codes = np.ascontiguousarray(codes)
    if codes.dtype != np.uint8:
        codes = codes.view(np.uint8)
    rb = row_bytes(fmt, I)
    if rb < 0:
        raise ValueError("bad format %r" % fmt)
    if codes.size != O * rb:
        raise ValueError("codes have %d bytes, expected %d" % (codes.size, O * rb))
    return codes


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def matmul(fmt: int, O: int, I: int, codes, scales, x, *, want_dbl: bool = False):
    """Returns (y f32 [S,O], bound f64 [S,O]) or (y, bound, ydbl) with want_dbl."""
    codes = _check_codes(fmt, O, I, codes)
    scales = _f32(scales)
    x = _f32(x).reshape(-1, I) if I > 0 else _f32(x).reshape(-1, 0)
    S = x.shape[0]
    y = np.empty((S, O), np.float32)
    bound = np.empty((S, O), np.float64)
    ydbl = np.empty((S, O), np.float64) if want_dbl else None
    rc = _L().qref_matmul(fmt, O, I, _ptr(codes), _ptr(scales), _ptr(x), S, _ptr(y),
                           _ptr(ydbl), _ptr(bound))
    if rc:
        raise ValueError("qref_matmul: bad argument")
    return (y, bound, ydbl) if want_dbl else (y, bound)


def matmul_gs(fmt: int, O: int, I: int, gs: int, codes, gscales, x, *, want_dbl: bool = False):
    """Group-wise scales gscales [O, ceil(I / gs)]: returns (y f32 [S,O], bound
    f64 [S,O]) or (y, bound, ydbl) with want_dbl."""
    codes = _check_codes(fmt, O, I, codes)
    G = -(-I // gs)
    gscales = _f32(gscales).reshape(O, G)
    x = _f32(x).reshape(-1, I)
    S = x.shape[0]
    y = np.empty((S, O), np.float32)
    bound = np.empty((S, O), np.float64)
    ydbl = np.empty((S, O), np.float64) if want_dbl else None
    rc = _L().qref_matmul_gs(fmt, O, I, gs, _ptr(codes), _ptr(gscales), _ptr(x), S, _ptr(y),
                             _ptr(ydbl), _ptr(bound))
    if rc:
        raise ValueError("qref_matmul_gs: bad argument")
    return (y, bound, ydbl) if want_dbl else (y, bound)


def matmul_gate_up(fmt, O, I, codes_g, scales_g, codes_u, scales_u, x):
    """Returns (yg, bound_g, yu, bound_u)."""
    codes_g = _check_codes(fmt, O, I, codes_g)
    codes_u = _check_codes(fmt, O, I, codes_u)
    scales_g, scales_u = _f32(scales_g), _f32(scales_u)
    x = _f32(x).reshape(-1, I)
    S = x.shape[0]
    yg = np.empty((S, O), np.float32)
    yu = np.empty((S, O), np.float32)
    bg = np.empty((S, O), np.float64)
    bu = np.empty((S, O), np.float64)
    rc = _L().qref_matmul_gate_up(fmt, O, I, _ptr(codes_g), _ptr(scales_g), _ptr(codes_u),
                                   _ptr(scales_u), _ptr(x), S, _ptr(yg), _ptr(bg), _ptr(yu),
                                   _ptr(bu))
    if rc:
        raise ValueError("qref_matmul_gate_up: bad argument")
    return yg, bg, yu, bu


def silu_mul(g, u):
    """h = silu(g) * u in double; returns (h rounded to f32, h f64)."""
    g, u = _f32(g), _f32(u)
    assert g.shape == u.shape
    h = np.empty(g.shape, np.float32)
    hd = np.empty(g.shape, np.float64)
    _L().qref_silu_mul(_ptr(g), _ptr(u), g.size, _ptr(h), _ptr(hd))
    return h, hd


def rmsnorm(x, w, eps: float, r=None):
    """h = x + r (f32, or x when r is None); y = h * w / sqrt(mean(h^2) + eps)
    per row, in double.  Returns (h f32, y f32, y f64)."""
    x = _f32(x)
    S, D = x.shape
    w = _f32(w).reshape(D)
    if r is not None:
        r = _f32(r).reshape(S, D)
    h = np.empty((S, D), np.float32)
    y = np.empty((S, D), np.float32)
    yd = np.empty((S, D), np.float64)
    rc = _L().qref_rmsnorm(_ptr(x), _ptr(r) if r is not None else None, _ptr(w), S, D, float(eps),
                           _ptr(h), _ptr(y), _ptr(yd))
    if rc:
        raise ValueError("qref_rmsnorm: bad argument")
    return h, y, yd


def mla_absorb(fmt: int, H: int, Dn: int, Dv: int, K: int, codes, scales, q_nope, q_rope, lat, rope,
               st0: int, scale: float, *, gs: int = 0, want_dbl: bool = False):
    """MLA decode attention with weight absorption over a [H*(Dn+Dv), K]
    weight tensor (per-row scales or None = 1.0; gs >= 1: group-wise scales
    [H*(Dn+Dv), ceil(K / gs)]).  q_nope [S, H, Dn], q_rope
    [S, H, R], lat [T, K], rope [T, R]; the S new tokens are the last S
    positions of the caches.  Returns (ctx f32 [S, H, Dv], bound f64) or
    (ctx, bound, ctx f64) with want_dbl."""
    codes = _check_codes(fmt, H * (Dn + Dv), K, codes)
    scales = _f32(scales)
    q_nope = _f32(q_nope)
    S = q_nope.shape[0]
    q_nope = q_nope.reshape(S, H, Dn)
    lat = _f32(lat)
    T = lat.shape[0]
    lat = lat.reshape(T, K)
    rope = _f32(rope).reshape(T, -1)
    R = rope.shape[1]
    q_rope = _f32(q_rope).reshape(S, H, R)
    ctx = np.empty((S, H, Dv), np.float32)
    bound = np.empty((S, H, Dv), np.float64)
    cd = np.empty((S, H, Dv), np.float64) if want_dbl else None
    rc = _L().qref_mla_absorb(fmt, H, Dn, Dv, K, R, _ptr(codes), _ptr(scales), gs, _ptr(q_nope), _ptr(q_rope),
                              _ptr(lat), _ptr(rope), T, st0, float(scale), S, _ptr(ctx), _ptr(cd),
                              _ptr(bound))
    if rc == -2:
        raise MemoryError("qref_mla_absorb: out of host memory for the per-row scratch vectors")
    if rc:
        raise ValueError("qref_mla_absorb: bad argument")
    return (ctx, bound, cd) if want_dbl else (ctx, bound)


def round_bf16(v) -> np.ndarray:
    """Round every f32 of v to the nearest bf16 (ties to even), as f32."""
    v = _f32(v)
    f = _L().qref_round_bf16
    out = np.empty_like(v)
    flat_in, flat_out = v.reshape(-1), out.reshape(-1)
    for k in range(flat_in.size):
        flat_out[k] = f(float(flat_in[k]))
    return out


def matmul_bf16x(fmt: int, O: int, I: int, codes, scales, x):
    """The matmul on x rounded to bf16 (diagnostic for the tensor-core path)."""
    codes = _check_codes(fmt, O, I, codes)
    scales = _f32(scales)
    x = _f32(x).reshape(-1, I)
    S = x.shape[0]
    xr = np.empty_like(x)
    y = np.empty((S, O), np.float32)
    bound = np.empty((S, O), np.float64)
    rc = _L().qref_matmul_bf16x(fmt, O, I, _ptr(codes), _ptr(scales), _ptr(x), S, _ptr(xr),
                                 _ptr(y), None, _ptr(bound))
    if rc:
        raise ValueError("qref_matmul_bf16x: bad argument")
    return y, bound, xr
