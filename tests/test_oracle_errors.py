"""The oracle fails loudly instead of skipping work (CPU only).

A row of the MLA oracle whose scratch vectors cannot be allocated must make
the whole call return an error, never a status of success with some outputs
left unwritten.  The scratch for one row is a few vectors of K doubles, so a
latent width near 2^58 asks for far more host memory than any address space
holds; the allocation fails before any input is read, which is why the input
pointers here only need to be non-NULL.
"""
import ctypes

import numpy as np
import pytest

import oracle


def test_mla_absorb_reports_allocation_failure():
    L = oracle.lib()
    K = 1 << 58                                   # 8 * K bytes per scratch vector: cannot be allocated
    dummy = np.zeros(16, np.float32)
    p = dummy.ctypes.data_as(ctypes.c_void_p)
    ctx = np.full(1, np.nan, np.float32)
    rc = L.qref_mla_absorb(oracle.I8, 1, 1, 1, K, 0, p, None, 0, p, None, p, None, 1, 0, 1.0, 1,
                           ctx.ctypes.data_as(ctypes.c_void_p), None, None)
    assert rc == -2
    assert np.isnan(ctx[0])                       # nothing was written


def test_mla_absorb_bad_argument_is_minus_one():
    L = oracle.lib()
    dummy = np.zeros(16, np.float32)
    p = dummy.ctypes.data_as(ctypes.c_void_p)
    # st0 > T - S: the window would hold no position
    rc = L.qref_mla_absorb(oracle.I8, 1, 1, 1, 4, 0, p, None, 0, p, None, p, None, 2, 2, 1.0, 1, p, None, None)
    assert rc == -1
    with pytest.raises(ValueError):
        oracle.mla_absorb(oracle.I8, 1, 1, 1, 4, np.zeros((2, 4), np.uint8), np.ones(2, np.float32),
                          np.zeros((1, 1, 1), np.float32), np.zeros((1, 1, 0), np.float32),
                          np.zeros((2, 4), np.float32), np.zeros((2, 0), np.float32), 2, 1.0)
