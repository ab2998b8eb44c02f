"""C-ABI library checks that need no GPU: the library loads, exports every
symbol include/fsa.h declares, and rejects bad arguments on the host before
touching the device."""
import ctypes
import os
import re

import pytest

import matrix_core_softmax_gb300 as fsa
from matrix_core_softmax_gb300 import build as fsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fsa_build.build()
    return fsa.load()


def _declared():
    txt = open(os.path.join(ROOT, "include", "fsa.h")).read()
    return sorted(set(re.findall(r"FSA_API\s+[\w\s\*]+?\b(fsa_\w+)\s*\(", txt)))


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(fsa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(6):
        assert fsa.status_string(s)
    assert fsa.status_string(0) == "ok"


def test_workspace_size(lib):
    assert fsa.workspace_size(1, 2, 512, 64) > 3 * 2 * 512 * 64
    assert lib.fsa_attention_workspace_size(1, 1, 100, 96, 0) == 0   # unsupported D
    assert lib.fsa_attention_workspace_size(0, 1, 100, 64, 0) == 0
    assert lib.fsa_attention_workspace_size(1, 1, 100, 64, 7) == 0


def _attn(lib, q=16, k=16, v=16, o=16, B=1, H=1, S=8, D=64, fmt=0, theta=8.0):
    P = ctypes.c_void_p
    return lib.fsa_attention_fwd(P(q) if q else None, P(k) if k else None, P(v) if v else None,
                                 P(o) if o else None, B, H, S, D, fmt, theta, None)


def test_attention_argument_validation(lib):
    assert _attn(lib, q=0) == 1
    assert _attn(lib, o=0) == 1
    assert _attn(lib, S=0) == 1
    assert _attn(lib, B=-1) == 1
    assert _attn(lib, D=96) == 2
    assert _attn(lib, q=8) == 1                     # not 16-byte aligned
    assert _attn(lib, fmt=4) == 1
    assert _attn(lib, theta=float("nan")) == 1
    assert _attn(lib, theta=-1.0) == 1
    assert _attn(lib, theta=81.0) == 1
    assert _attn(lib, B=300, H=300) == 1            # more than 65535 heads


def test_cross_attention_workspace_and_validation(lib):
    # Sq = Sk is the self-attention workspace; each length sizes its own part
    assert lib.fsa_cross_attention_workspace_size(1, 2, 512, 512, 64, 0) == \
        lib.fsa_attention_workspace_size(1, 2, 512, 64, 0)
    small, big = (lib.fsa_cross_attention_workspace_size(1, 2, 100, sk, 128, 1) for sk in (300, 3000))
    assert big - small >= 2 * 2 * 2700 * 128            # K and V^T copies grow with Sk
    assert lib.fsa_cross_attention_workspace_size(1, 2, 0, 300, 64, 0) == 0
    assert lib.fsa_cross_attention_workspace_size(1, 2, 300, 0, 64, 0) == 0
    P = ctypes.c_void_p

    def cross(q=16, Sq=8, Sk=8, D=64):
        return lib.fsa_cross_attention_fwd(P(q) if q else None, P(16), P(16), P(16), 1, 1, Sq, Sk, D,
                                           0, 8.0, None, None)
    assert cross(q=0) == 1
    assert cross(Sq=0) == 1
    assert cross(Sk=0) == 1
    assert cross(Sk=-3) == 1
    assert cross(D=96) == 2


def test_bf16_attention_argument_validation(lib):
    P = ctypes.c_void_p
    assert lib.fsa_bf16_attention_fwd(None, P(16), P(16), P(16), 1, 1, 8, 64, None) == 1
    assert lib.fsa_bf16_attention_fwd(P(16), P(16), P(16), P(16), 1, 1, 8, 80, None) == 2


def test_quantize_argument_validation(lib):
    P = ctypes.c_void_p
    assert lib.fsa_quantize_mx(None, 1, 4, 4, 1, 0, P(16), P(16), None) == 1
    assert lib.fsa_quantize_mx(P(16), 1, 4, 4, 2, 0, P(16), P(16), None) == 1
    assert lib.fsa_quantize_mx(P(16), 1, 4, 4, 1, 3, P(16), P(16), None) == 1
    assert lib.fsa_quantize_mx(P(16), -1, 4, 4, 1, 0, P(16), P(16), None) == 1
    assert lib.fsa_quantize_mx(P(17), 1, 4, 4, 1, 0, P(16), P(16), None) == 1
    # empty tensor: nothing to do, no device needed
    assert lib.fsa_quantize_mx(P(16), 0, 4, 4, 1, 0, P(16), P(16), None) == 0


def test_mma_rate_probe_argument_validation(lib):
    # every check is on the host, before the device is touched
    fl = ctypes.c_double(0.0)
    for kind, ctas, iters in [(-1, 1, 1), (5, 1, 1), (0, 0, 1), (0, 65536, 1), (0, 1, 0),
                              (0, 1, (1 << 24) + 1)]:
        assert lib.fsa_mma_rate_probe(kind, ctas, iters, ctypes.byref(fl), None) == 1


def test_host_attention_argument_validation(lib):
    # host-buffer entry points: shape, format and threshold checks happen on
    # the host before any device call (host pointers need no alignment)
    P = ctypes.c_void_p

    def host(q=16, B=1, H=1, Sq=8, Sk=8, D=64, fmt=0, theta=8.0):
        return lib.fsa_cross_attention_fwd_host(P(q) if q else None, P(16), P(16), P(16), B, H, Sq, Sk,
                                                D, fmt, theta, None, None)
    assert host(q=0) == 1
    assert host(Sq=0) == 1
    assert host(Sk=-1) == 1
    assert host(D=96) == 2
    assert host(fmt=4) == 1
    assert host(theta=float("inf")) == 1
    assert host(B=300, H=300) == 1
    assert lib.fsa_attention_fwd_host(None, P(16), P(16), P(16), 1, 1, 8, 64, 0, 8.0, None, None) == 1
    assert lib.fsa_attention_fwd_host(P(16), P(16), P(16), P(16), 1, 1, 8, 80, 0, 8.0, None, None) == 2


def test_host_attention_binding_rejects_device_or_mismatched_tensors():
    import torch
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fsa.attention_fwd_host(q, q, q.float())                      # not bf16
    with pytest.raises(ValueError):
        fsa.attention_fwd_host(q, q, torch.zeros(1, 2, 9, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        fsa.cross_attention_fwd_host(q, torch.zeros(1, 2, 5, 64, dtype=torch.bfloat16),
                                     torch.zeros(1, 2, 6, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        fsa.attention_fwd_host(q, q, q, out=torch.zeros(1, 2, 8, 32, dtype=torch.bfloat16))
