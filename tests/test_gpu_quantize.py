"""GPU parity of the MX quantizer (fsa_quantize_mx) against the oracle:
codes and scales must be bit-exact for all three element formats, both block
axes, ragged tails and special blocks."""
import numpy as np
import pytest
import torch

import fsa_inputs
import oracle
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fsa():
    import __graft_entry__
    __graft_entry__.build()
    import matrix_core_softmax_gb300 as m
    return m


def _special_bits():
    """bf16 patterns covering zero blocks, signed zeros, subnormals, the
    largest finite bf16, exact format maxima and round-to-even midpoints."""
    rng = np.random.default_rng(9)
    blocks = [
        np.zeros(32, np.uint16),
        np.full(32, 0x8000, np.uint16),                                   # -0.0
        rng.integers(1, 0x80, 32).astype(np.uint16),                      # subnormals
        (rng.integers(1, 0x80, 32) | 0x8000).astype(np.uint16),
        np.concatenate([[0x7F7F], rng.integers(0, 0x7F7F, 31)]).astype(np.uint16),  # max bf16
        fsa_inputs.to_bf16_bits(np.array([448.0, 464.0, 240.0, 7.5, 6.0, 5.0, 0.0625, 1e-3] * 4,
                                         np.float32)),
        fsa_inputs.to_bf16_bits(rng.standard_normal(32).astype(np.float32) * 1e-30),
        fsa_inputs.to_bf16_bits(rng.standard_normal(32).astype(np.float32) * 1e30),
    ]
    return np.concatenate(blocks)


@pytest.mark.parametrize("elem", [0, 1, 2])
@pytest.mark.parametrize("shape", [(1, 64, 128), (2, 75, 45), (3, 33, 64), (1, 1, 1), (1, 512, 64)])
@pytest.mark.parametrize("axis", [1, 0])
def test_quantize_bit_exact(fsa, elem, shape, axis):
    rng = np.random.default_rng(sum(shape) + elem)
    x = fsa_inputs.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) *
                                np.float32(rng.choice([1e-3, 1.0, 40.0])))
    codes, scales = fsa.quantize_mx(to_dev(x), axis, elem)
    rc, rs = oracle.mx_quantize(x, axis, elem)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("elem", [0, 1, 2])
@pytest.mark.parametrize("axis", [1, 0])
def test_quantize_special_blocks(fsa, elem, axis):
    sp = _special_bits().reshape(-1, 32)          # each row one block
    x = sp if axis == 1 else np.ascontiguousarray(sp.T)
    codes, scales = fsa.quantize_mx(to_dev(x), axis, elem)
    rc, rs = oracle.mx_quantize(x, axis, elem)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("elem", [0, 1, 2])
def test_quantize_qkv_layouts_at_config_size(fsa, elem):
    # Q/K blocks along D, V blocks along keys (transposed), 8192 x 128 heads
    q, k, v = fsa_inputs.qkv(1, 2, 8192, 128, seed=0)
    for x, axis in ((q, 1), (v, 0)):
        x3 = x.reshape(2, 8192, 128)
        codes, scales = fsa.quantize_mx(to_dev(x3), axis, elem)
        rc, rs = oracle.mx_quantize(x3, axis, elem)
        assert np.array_equal(scales.cpu().numpy(), rs)
        assert np.array_equal(codes.cpu().numpy(), rc)
