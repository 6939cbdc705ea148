"""The C-ABI library loads and exports every declared symbol; host-side error
paths that need no GPU (CPU only: no compute call is made)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "b200q.h")


@pytest.fixture(scope="module")
def built_lib():
    import __graft_entry__
    return __graft_entry__._build_module().build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(b200q_\w+)\s*\(", text)))


def test_header_declares_the_core_calls():
    names = declared_functions()
    for n in ("b200q_tensor_upload", "b200q_matmul", "b200q_matmul_gate_up", "b200q_tensor_free",
              "b200q_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(built_lib):
    L = ctypes.CDLL(built_lib)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_names_match_the_abi(built_lib):
    import quantized_weight_quant_gb300 as q
    for n in declared_functions():
        assert hasattr(q, n[len("b200q_"):]), n


def test_upload_argument_errors(built_lib):
    import quantized_weight_quant_gb300 as q
    L = q.lib
    codes = np.zeros(64, np.uint8)
    sc = np.ones(4, np.float32)
    assert not L.b200q_tensor_upload(9, 4, 16, codes.ctypes.data, sc.ctypes.data)
    assert "format" in q.last_error()
    assert not L.b200q_tensor_upload(q.I8, 0, 16, codes.ctypes.data, sc.ctypes.data)
    assert "O and I" in q.last_error()
    assert not L.b200q_tensor_upload(q.I8, 4, -1, codes.ctypes.data, sc.ctypes.data)
    assert not L.b200q_tensor_upload(q.I8, 4, 16, None, sc.ctypes.data)
    assert "NULL" in q.last_error()
    assert not L.b200q_tensor_upload(q.I4, 4, 16, codes.ctypes.data, None)
    assert "scales" in q.last_error()


def test_fault_injection_alloc(built_lib, monkeypatch):
    import quantized_weight_quant_gb300 as q
    monkeypatch.setenv("B200Q_FAULT_INJECT", "alloc")
    codes = np.zeros(64, np.uint8)
    sc = np.ones(4, np.float32)
    with pytest.raises(q.B200QError) as ei:
        q.tensor_upload(q.I8, 4, 16, codes, sc)
    assert ei.value.status == q.ENOMEM
    assert "injected" in q.last_error()


def test_null_tensor_calls(built_lib):
    import quantized_weight_quant_gb300 as q
    L = q.lib
    assert L.b200q_matmul(None, None, None, 1, None) == q.EINVAL
    assert L.b200q_matmul_gate_up(None, None, None, None, None, 1, None) == q.EINVAL
    assert L.b200q_matmul_path(None, 1) == q.EINVAL
    assert L.b200q_matmul_host(None, None, None, 1, None) == q.EINVAL
    assert L.b200q_tensor_info(None, None, None, None, None, None) == q.EINVAL
    L.b200q_tensor_free(None)            # no-op


def test_silu_mul_argument_errors(built_lib):
    import quantized_weight_quant_gb300 as q
    L = q.lib
    assert L.b200q_silu_mul(None, None, None, 0, None) == q.OK      # n == 0 is a no-op
    assert L.b200q_silu_mul(None, None, None, -1, None) == q.EINVAL
    assert L.b200q_silu_mul(None, None, None, 4, None) == q.EINVAL
    assert L.b200q_silu_mul(16, 32, 49, 4, None) == q.EINVAL         # misaligned h
    assert L.b200q_silu_mul(16, 64, 32, 8, None) == q.EINVAL         # h partially overlaps g


def test_tc_threshold_default(built_lib):
    import quantized_weight_quant_gb300 as q
    if "B200Q_TC_MIN_S" not in os.environ:
        assert q.tc_min_s() == 16


def test_grouped_argument_errors_without_gpu(built_lib):
    import quantized_weight_quant_gb300 as q
    L = q.lib
    arr = (ctypes.c_void_p * 17)()
    assert L.b200q_matmul_grouped(arr, 0, arr, arr, 1, None) == q.EINVAL
    assert "n must be" in q.last_error()
    assert L.b200q_matmul_grouped(arr, 17, arr, arr, 1, None) == q.EINVAL
    assert L.b200q_matmul_grouped(None, 2, arr, arr, 1, None) == q.EINVAL
    assert "NULL host array" in q.last_error()
    assert L.b200q_matmul_grouped(arr, 2, arr, arr, 1, None) == q.EINVAL    # NULL handles
    assert "tensor is NULL" in q.last_error()
    assert L.b200q_matmul_grouped_silu(arr, 2, arr, None, arr, 1, None) == q.EINVAL
    assert L.b200q_matmul_grouped_silu(arr, 2, arr, arr, arr, 1, None) == q.EINVAL
    assert q.GROUP_MAX == 16
    with pytest.raises(ValueError):
        q.matmul_grouped([1, 2], [3], [4, 5], 1)


def test_rmsnorm_argument_errors_without_gpu(built_lib):
    import quantized_weight_quant_gb300 as q
    L = q.lib
    assert L.b200q_rmsnorm(None, None, None, None, None, 0, 8, 1e-6, None) == q.OK      # S == 0
    assert L.b200q_rmsnorm(None, None, None, None, None, 1, 0, 1e-6, None) == q.EINVAL  # D == 0
    assert L.b200q_rmsnorm(None, None, None, None, None, 1, 8, -1.0, None) == q.EINVAL  # eps < 0
    assert L.b200q_rmsnorm(None, None, None, None, None, 1, 8, 1e-6, None) == q.EINVAL  # NULL x
    assert L.b200q_rmsnorm(16, None, None, 32, 48 + 4, 1, 8, 1e-6, None) == q.EINVAL    # misaligned y
    assert L.b200q_rmsnorm(4096, None, None, 0x10000, 4096 + 16, 1, 8, 1e-6, None) == q.EINVAL   # y overlaps x
    assert "overlap" in q.last_error()


def test_mla_argument_errors_without_gpu(built_lib):
    import quantized_weight_quant_gb300 as q
    L = q.lib
    # no tensor: refused before anything touches a device
    assert L.b200q_mla_absorb(None, 2, 4, 4, 16, 32, 48, 64, 4, 8, 0, 0.5, 80, 1, None) == q.EINVAL
    assert "NULL" in q.last_error() or "tensor" in q.last_error()
    # cache appends: bad counts and NULL pointers
    assert L.b200q_kv_append(16, 32, 8, 4, 0, 48, 64, -1, None) == q.EINVAL
    assert L.b200q_kv_append(16, 32, 8, 4, -3, 48, 64, 2, None) == q.EINVAL
    assert L.b200q_kv_append(None, 32, 8, 4, 0, 48, 64, 2, None) == q.EINVAL
    assert "NULL" in q.last_error()
    assert L.b200q_kv_append(16, None, 8, 4, 0, 48, None, 2, None) == q.EINVAL
    assert L.b200q_kv_append(16, None, 8, 0, 0, 48, None, 0, None) == q.OK     # n = 0: no-op
    assert q.KV_PAGE_TOKENS == 64


def test_selftest_timeout_argument_errors_without_gpu(built_lib):
    import quantized_weight_quant_gb300 as q
    assert q.lib.b200q_selftest_timeout(0, None) == q.EINVAL
    assert q.lib.b200q_selftest_timeout(2000000, None) == q.EINVAL
