"""Python binding of the b200q C ABI (``include/b200q.h``).

Argument marshalling only: every step of the matmul runs in the CUDA library
``libb200q.so`` built from ``csrc/``.  There is no CPU fallback; importing the
package without the built library raises.

Device arrays are passed as torch CUDA tensors (their ``data_ptr()``) or as
raw integer device pointers.  ``stream`` is None (torch's current stream on
the current device), a ``torch.cuda.Stream``, or a raw ``cudaStream_t`` int.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

F32, I8, I4, I2 = 0, 1, 2, 3
OK, EINVAL, ENOMEM, ECUDA, ETIMEOUT = 0, -1, -2, -3, -4
PATH_AUTO, PATH_F32, PATH_TC, PATH_TCX, PATH_TCS = 0, 1, 2, 3, 4
GROUP_MAX = 16
FORMATS = {"f32": F32, "i8": I8, "i4": I4, "i2": I2}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libb200q.so")


class B200QError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("b200q status %d: %s" % (status, message))
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libb200q.so is not built: run `python -c \"import __graft_entry__ as g; g.build()\"` "
                          "or `python quantized_weight_quant_gb300/build.py`")
    L = ctypes.CDLL(LIB_PATH)
    vp, ci, cl, cll, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_longlong, ctypes.c_float
    L.b200q_tensor_upload.argtypes = [ci, ci, ci, vp, vp]
    L.b200q_tensor_upload.restype = vp
    L.b200q_tensor_upload_grouped.argtypes = [ci, ci, ci, ci, vp, vp]
    L.b200q_tensor_upload_grouped.restype = vp
    L.b200q_tensor_group_size.argtypes = [vp]
    L.b200q_tensor_group_size.restype = ci
    L.b200q_tensor_free.argtypes = [vp]
    L.b200q_tensor_free.restype = None
    L.b200q_matmul.argtypes = [vp, vp, vp, ci, vp]
    L.b200q_matmul.restype = ci
    L.b200q_matmul_ex.argtypes = [vp, vp, vp, ci, ci, vp]
    L.b200q_matmul_ex.restype = ci
    L.b200q_matmul_path.argtypes = [vp, ci]
    L.b200q_matmul_path.restype = ci
    L.b200q_tc_min_s.argtypes = []
    L.b200q_tc_min_s.restype = ci
    L.b200q_tcx_min_s.argtypes = []
    L.b200q_tcx_min_s.restype = ci
    L.b200q_matmul_gate_up.argtypes = [vp, vp, vp, vp, vp, ci, vp]
    L.b200q_matmul_gate_up.restype = ci
    L.b200q_matmul_grouped.argtypes = [vp, ci, vp, vp, ci, vp]
    L.b200q_matmul_grouped.restype = ci
    L.b200q_matmul_grouped_silu.argtypes = [vp, ci, vp, vp, vp, ci, vp]
    L.b200q_matmul_grouped_silu.restype = ci
    L.b200q_rmsnorm.argtypes = [vp, vp, vp, vp, vp, ci, ci, cf, vp]
    L.b200q_rmsnorm.restype = ci
    L.b200q_mla_absorb.argtypes = [vp, ci, ci, ci, vp, vp, vp, vp, ci, ci, ci, cf, vp, ci, vp]
    L.b200q_mla_absorb.restype = ci
    L.b200q_kv_append.argtypes = [vp, vp, ci, ci, ci, vp, vp, ci, vp]
    L.b200q_kv_append.restype = ci
    L.b200q_selftest_timeout.argtypes = [ci, vp]
    L.b200q_selftest_timeout.restype = ci
    L.b200q_silu_mul.argtypes = [vp, vp, vp, cl, vp]
    L.b200q_silu_mul.restype = ci
    L.b200q_matmul_host.argtypes = [vp, vp, vp, ci, vp]
    L.b200q_matmul_host.restype = ci
    L.b200q_tensor_info.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(ci), ctypes.POINTER(ci),
                                    ctypes.POINTER(ci), ctypes.POINTER(cll)]
    L.b200q_tensor_info.restype = ci
    L.b200q_matmul_tc_noalloc.argtypes = [vp, vp, vp, ci, vp]
    L.b200q_matmul_tc_noalloc.restype = ci
    L.b200q_tc_noalloc_capacity.argtypes = []
    L.b200q_tc_noalloc_capacity.restype = cll
    L.b200q_device_status.argtypes = []
    L.b200q_device_status.restype = ci
    L.b200q_kernel_launches.argtypes = []
    L.b200q_kernel_launches.restype = cll
    L.b200q_workspace_allocations.argtypes = []
    L.b200q_workspace_allocations.restype = cll
    L.b200q_last_error.argtypes = []
    L.b200q_last_error.restype = ctypes.c_char_p
    return L


lib = _load()


def last_error() -> str:
    return lib.b200q_last_error().decode()


def kernel_launches() -> int:
    """Kernels launched through the library so far in this process."""
    return int(lib.b200q_kernel_launches())


def workspace_allocations() -> int:
    """Device workspace allocations the library has made so far in this process."""
    return int(lib.b200q_workspace_allocations())


def device_status() -> int:
    """Synchronize the device; raise if a kernel gave up on a bounded wait."""
    return _check(lib.b200q_device_status())


def tc_min_s() -> int:
    return int(lib.b200q_tc_min_s())


def tcx_min_s() -> int:
    return int(lib.b200q_tcx_min_s())


def _check(rc: int) -> int:
    if rc < 0:
        raise B200QError(rc, last_error())
    return rc


def _dptr(a) -> int:
    """Device pointer of a torch CUDA tensor (checked contiguous f32) or an int."""
    if a is None:
        return 0
    if isinstance(a, int):
        return a
    import torch
    if not isinstance(a, torch.Tensor):
        raise TypeError("expected a torch CUDA tensor or an int device pointer")
    if not a.is_cuda:
        raise ValueError("expected a CUDA tensor, got a %s tensor" % a.device)
    if a.dtype != torch.float32 or not a.is_contiguous():
        raise ValueError("expected a contiguous float32 tensor")
    return a.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class QTensor:
    """A weight tensor resident on the GPU (owns its b200q_tensor handle)."""

    def __init__(self, handle: int, fmt: int, O: int, I: int):
        self.handle, self.fmt, self.O, self.I = handle, fmt, O, I

    def free(self):
        if self.handle:
            lib.b200q_tensor_free(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.free()
        return False

    def info(self):
        return tensor_info(self)


def _h(t) -> int:
    return t.handle if isinstance(t, QTensor) else t


def tensor_upload(fmt: int, O: int, I: int, codes, scales, gs: int = 0) -> QTensor:
    """Upload host codes ([O, row_bytes] uint8, or f32 [O, I] for fmt F32) and
    host scales (f32 [O], or None for F32; with gs >= 1 group-wise scales
    [O, ceil(I / gs)]) to the current device."""
    codes = np.ascontiguousarray(codes)
    if codes.dtype != np.uint8:
        codes = codes.view(np.uint8)
    n_scales = O * (-(-I // gs) if gs else 1)
    if scales is not None:
        scales = np.ascontiguousarray(scales, dtype=np.float32)
        if scales.size != n_scales:
            raise ValueError("scales must hold %d floats" % n_scales)
    bits = {F32: 32, I8: 8, I4: 4, I2: 2}.get(fmt)
    if bits is not None and codes.size != O * ((I * bits + 7) // 8):
        raise ValueError("codes hold %d bytes, expected O * row_bytes = %d"
                         % (codes.size, O * ((I * bits + 7) // 8)))
    sp = None if scales is None else scales.ctypes.data
    if gs:
        h = lib.b200q_tensor_upload_grouped(fmt, O, I, gs, codes.ctypes.data, sp)
    else:
        h = lib.b200q_tensor_upload(fmt, O, I, codes.ctypes.data, sp)
    if not h:
        msg = last_error()
        raise B200QError(ENOMEM if "memory" in msg else EINVAL, msg)
    return QTensor(h, fmt, O, I)


def tensor_upload_grouped(fmt: int, O: int, I: int, gs: int, codes, scales) -> QTensor:
    """tensor_upload with group-wise scales (b200q_tensor_upload_grouped)."""
    return tensor_upload(fmt, O, I, codes, scales, gs=gs)


def tensor_group_size(t) -> int:
    return _check(lib.b200q_tensor_group_size(_h(t)))


def tensor_free(t) -> None:
    if isinstance(t, QTensor):
        t.free()
    else:
        lib.b200q_tensor_free(t)


def tensor_info(t):
    f, o, i, d = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    nb = ctypes.c_longlong()
    _check(lib.b200q_tensor_info(_h(t), ctypes.byref(f), ctypes.byref(o), ctypes.byref(i),
                                 ctypes.byref(d), ctypes.byref(nb)))
    return {"fmt": f.value, "O": o.value, "I": i.value, "device": d.value,
            "device_bytes": nb.value}


def matmul(t, x, y, S: int, stream=None) -> None:
    _check(lib.b200q_matmul(_h(t), _dptr(x), _dptr(y), S, _stream(stream)))


def matmul_ex(t, x, y, S: int, path: int, stream=None) -> None:
    _check(lib.b200q_matmul_ex(_h(t), _dptr(x), _dptr(y), S, path, _stream(stream)))


def matmul_path(t, S: int) -> int:
    return _check(lib.b200q_matmul_path(_h(t), S))


def matmul_gate_up(tg, tu, x, yg, yu, S: int, stream=None) -> None:
    _check(lib.b200q_matmul_gate_up(_h(tg), _h(tu), _dptr(x), _dptr(yg), _dptr(yu), S,
                                    _stream(stream)))


def _ptr_array(items, conv):
    """A host array of pointers (kept alive by the caller's reference)."""
    arr = (ctypes.c_void_p * max(len(items), 1))()
    for j, a in enumerate(items):
        arr[j] = conv(a) or None
    return arr


def matmul_grouped(ts, xs, ys, S: int, stream=None) -> None:
    """ys[j] = matmul(ts[j], xs[j]) for every j, in one launch per two rows on
    the f32 path (b200q_matmul_grouped).  ts, xs, ys: equal-length sequences."""
    if not (len(ts) == len(xs) == len(ys)):
        raise ValueError("ts, xs and ys must have the same length")
    th, xh, yh = _ptr_array(ts, _h), _ptr_array(xs, _dptr), _ptr_array(ys, _dptr)
    _check(lib.b200q_matmul_grouped(th, len(ts), xh, yh, S, _stream(stream)))


def matmul_grouped_silu(ts, gs, us, ys, S: int, stream=None) -> None:
    """ys[j] = matmul(ts[j], silu(gs[j]) * us[j]) for every j
    (b200q_matmul_grouped_silu)."""
    if not (len(ts) == len(gs) == len(us) == len(ys)):
        raise ValueError("ts, gs, us and ys must have the same length")
    th, gh, uh, yh = (_ptr_array(ts, _h), _ptr_array(gs, _dptr), _ptr_array(us, _dptr),
                      _ptr_array(ys, _dptr))
    _check(lib.b200q_matmul_grouped_silu(th, len(ts), gh, uh, yh, S, _stream(stream)))


def matmul_tc_noalloc(t, x, y, S: int, stream=None) -> None:
    """Tensor-core matmul with no allocation: the bf16 copy of x lives in a
    fixed per-device array (see b200q_matmul_tc_noalloc in include/b200q.h)."""
    _check(lib.b200q_matmul_tc_noalloc(_h(t), _dptr(x), _dptr(y), S, _stream(stream)))


def tc_noalloc_capacity() -> int:
    return int(lib.b200q_tc_noalloc_capacity())


def silu_mul(g, u, h, n: int, stream=None) -> None:
    _check(lib.b200q_silu_mul(_dptr(g), _dptr(u), _dptr(h), n, _stream(stream)))


def rmsnorm(x, w, y, S: int, D: int, eps: float, r=None, h=None, stream=None) -> None:
    """y = (x + r) * w / sqrt(mean((x + r)^2) + eps) per row; h receives x + r
    when given (b200q_rmsnorm)."""
    _check(lib.b200q_rmsnorm(_dptr(x), _dptr(r), _dptr(h), _dptr(w), _dptr(y), S, D, eps, _stream(stream)))


def selftest_timeout(wait_us: int, stream=None) -> None:
    """A kernel waits wait_us on an mbarrier nothing completes and records a
    timeout (b200q_selftest_timeout); device_status() then reports it."""
    _check(lib.b200q_selftest_timeout(wait_us, _stream(stream)))


KV_PAGE_TOKENS = 64


def _page_table(a) -> int:
    """Device address of a page-pointer array: an int64 CUDA tensor or an int."""
    if a is None:
        return 0
    if isinstance(a, int):
        return a
    import torch
    if not a.is_cuda or a.dtype != torch.int64 or not a.is_contiguous():
        raise ValueError("expected a contiguous int64 CUDA tensor of page pointers")
    return a.data_ptr()


def mla_absorb(t, H: int, Dn: int, Dv: int, q_nope, q_rope, lat_pages, rope_pages, R: int, T: int, st0: int,
               scale: float, ctx, S: int, stream=None) -> None:
    """MLA decode attention with weight absorption (b200q_mla_absorb): ctx
    [S, H, Dv] from q_nope [S, H, Dn], q_rope [S, H, R] and the paged caches
    (lat_pages / rope_pages: device arrays of page pointers, e.g. PagedKV's)."""
    _check(lib.b200q_mla_absorb(_h(t), H, Dn, Dv, _dptr(q_nope), _dptr(q_rope), _page_table(lat_pages),
                                _page_table(rope_pages), R, T, st0, scale, _dptr(ctx), S, _stream(stream)))


def kv_append(lat_pages, rope_pages, K: int, R: int, pos: int, lat_rows, rope_rows, n: int, stream=None) -> None:
    """Rows n of lat_rows [n, K] / rope_rows [n, R] into the paged caches at
    positions pos .. pos+n-1 (b200q_kv_append)."""
    _check(lib.b200q_kv_append(_page_table(lat_pages), _page_table(rope_pages), K, R, pos, _dptr(lat_rows),
                               _dptr(rope_rows), n, _stream(stream)))


class PagedKV:
    """A paged latent / rope cache in torch device memory: pages of 64
    positions ([64, K] and [64, R] f32) carved from one pool each, and the
    device page tables b200q_mla_absorb reads.  `order` places logical page p
    at pool slot order[p] (any permutation), so the tables need not be in
    address order."""

    def __init__(self, K: int, R: int, max_tokens: int, device="cuda", order=None):
        import torch
        n = max(1, -(-max_tokens // KV_PAGE_TOKENS))
        self.K, self.R, self.n_pages = K, R, n
        self.lat_pool = torch.zeros((n, KV_PAGE_TOKENS, K), dtype=torch.float32, device=device)
        self.rope_pool = torch.zeros((n, KV_PAGE_TOKENS, max(R, 1)), dtype=torch.float32, device=device)
        slots = list(range(n)) if order is None else [int(v) for v in order]
        if sorted(slots) != list(range(n)):
            raise ValueError("order must be a permutation of range(n_pages)")
        lb, rb = self.lat_pool.data_ptr(), self.rope_pool.data_ptr()
        self.lat_pages = torch.tensor([lb + q * KV_PAGE_TOKENS * K * 4 for q in slots], dtype=torch.int64,
                                      device=device)
        self.rope_pages = torch.tensor([rb + q * KV_PAGE_TOKENS * max(R, 1) * 4 for q in slots],
                                       dtype=torch.int64, device=device)
        self.slots = slots

    def append(self, lat_rows, rope_rows, pos: int, n: int, stream=None) -> None:
        kv_append(self.lat_pages, self.rope_pages if self.R else None, self.K, self.R, pos, lat_rows,
                  rope_rows if self.R else None, n, stream)

    def attend(self, t, H: int, Dn: int, Dv: int, q_nope, q_rope, T: int, st0: int, scale: float, ctx, S: int,
               stream=None) -> None:
        mla_absorb(t, H, Dn, Dv, q_nope, q_rope, self.lat_pages, self.rope_pages if self.R else None, self.R, T,
                   st0, scale, ctx, S, stream)


def matmul_host(t, x_host, y_host, S: int, stream=None) -> None:
    """x_host / y_host: host f32 buffers (numpy arrays or pinned torch CPU tensors)."""
    def hptr(a):
        if isinstance(a, np.ndarray):
            if a.dtype != np.float32 or not a.flags.c_contiguous:
                raise ValueError("expected a contiguous float32 array")
            return a.ctypes.data
        if isinstance(a, int):
            return a
        if a.is_cuda or not a.is_contiguous():
            raise ValueError("expected a contiguous host tensor")
        return a.data_ptr()
    _check(lib.b200q_matmul_host(_h(t), hptr(x_host), hptr(y_host), S, _stream(stream)))
