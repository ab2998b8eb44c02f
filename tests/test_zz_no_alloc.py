"""The non-allocating entry point, fsa_attention_fwd_noalloc.

It exists for callers that may not allocate device memory while running: it
keeps the MX copies of Q, K, V in a fixed 64 MiB array inside the library
instead of a cudaMalloc'ed workspace.  Called here through the C ABI, twice
in a row on different inputs and formats, and compared with the allocating
entry point, fsa_attention_fwd, within the parity tolerance of the other
attention tests.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import fsa_inputs
import oracle
from gpu_util import to_dev, to_f64

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def fsa():
    import __graft_entry__
    __graft_entry__.build()
    import matrix_core_softmax_gb300 as m
    return m


def _noalloc(fsa, q, k, v, fmt, theta=8.0):
    B, H, S, D = q.shape
    o = torch.empty_like(q)
    st = fsa.load().fsa_attention_fwd_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()), B, H, S, D,
        fsa.FORMATS[fmt], ctypes.c_float(theta), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, fsa.status_string(st)
    return o


def test_noalloc_matches_allocating_entry_point_on_two_calls(fsa):
    cases = [((1, 4, 1000, 128), "mxfp8", 31), ((2, 3, 777, 64), "mxfp4", 32)]
    for (B, H, S, D), fmt, seed in cases:
        q, k, v = (to_dev(x) for x in fsa_inputs.qkv(B, H, S, D, seed=seed))
        got = _noalloc(fsa, q, k, v, fmt)
        torch.cuda.synchronize()
        ref = fsa.attention_fwd(q, k, v, fmt=fmt)
        assert fsa.get_device_error() == 0
        a, b = to_f64(got).reshape(-1, D), to_f64(ref).reshape(-1, D)
        assert np.all(np.isfinite(a))
        assert oracle.rel_l2(a, b) <= TOL


def test_noalloc_rejects_shapes_beyond_its_array(fsa):
    q = torch.zeros(1, 1, 16, 128, dtype=torch.bfloat16, device="cuda")
    st = fsa.load().fsa_attention_fwd_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(q.data_ptr()), 1, 40, 75600, 128, 0, ctypes.c_float(8.0), None)
    assert st == 1  # FSA_ERR_INVALID_ARGUMENT, nothing launched
