"""GPU parity of the six-bit P conversion at the edges of its norm bound, and
of operands at the edge of the scale range.

For MXFP6 and MXFP4 the fused kernel skips the block minima for a warp whose
rows satisfy 2 |alpha| |q^_i| max_j |k^_j| <= 15000 (alpha = 128 log2(e) sm),
a Cauchy-Schwarz bound under which no weight of the row can underflow the
scaled conversion; other warps, and the masked tail tile, keep the exact
test.  These cases put score spreads right inside and right outside that
bound, and mix bounded and unbounded warps in one CTA; every output must
still match the oracle (relative L2 <= 5e-3)."""
import math

import numpy as np
import pytest

import fsa_inputs
import oracle
import parity
from gpu_util import to_dev, to_f64

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def fsa():
    import __graft_entry__
    __graft_entry__.build()
    import matrix_core_softmax_gb300 as m
    return m


def _check(fsa, q, k, v, fmt, theta=8.0):
    B, H, S, D = q.shape
    o = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt, threshold=theta)
    st = fsa.get_device_error()
    assert st == 0, fsa.status_string(st)
    got = to_f64(o).reshape(-1, D)
    ref = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=theta)["out"]
    assert np.all(np.isfinite(got))
    parity.check_out(f"norm bound {q.shape} {fmt} theta={theta}", got, ref)


def _spread_inputs(D, S, ek, seed):
    """q rows all +1.5, key rows +-ek (random sign per key): every score is
    exactly +-1.5 ek D in accumulator units, the widest spread Cauchy-Schwarz
    allows for these norms.  1.5 and 2 or 3 are exact in E4M3, E2M3 and
    E2M1 at their block scales."""
    rng = np.random.default_rng(seed)
    q = np.full((1, 1, S, D), 1.5, np.float32)
    sign = np.where(rng.random(S) < 0.5, -1.0, 1.0).astype(np.float32)
    k = (sign[:, None] * np.float32(ek)) * np.ones((S, D), np.float32)
    k = k.reshape(1, 1, S, D)
    v = rng.standard_normal((1, 1, S, D)).astype(np.float32)
    return (fsa_inputs.to_bf16_bits(q), fsa_inputs.to_bf16_bits(k), fsa_inputs.to_bf16_bits(v))


@pytest.mark.parametrize("fmt", ["mxfp6", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("ek", [2.0, 3.0])
def test_widest_spread_inside_and_outside_the_bound(fsa, fmt, D, ek):
    S = 300  # three KV tiles, a ragged tail
    alpha = 128.0 * math.log2(math.e) / math.sqrt(D)
    a = 1.5 * ek * D  # |q^| |k^| = the largest |accumulator|
    spread = 2.0 * alpha * a
    # D = 128: 12535 (inside) and 18803 (outside); D = 64: 8864 and 13296
    assert (spread <= 15000.0) == (ek == 2.0 or D == 64)
    q, k, v = _spread_inputs(D, S, ek, seed=int(ek * 10) + D)
    _check(fsa, q, k, v, fmt, theta=80.0)


@pytest.mark.parametrize("fmt", ["mxfp6", "mxfp4"])
@pytest.mark.parametrize("D", [64, 128])
def test_bounded_and_unbounded_warps_in_one_tile(fsa, fmt, D):
    # query rows 0-31 (warp 0 of the first query tile) scaled x40: that warp
    # fails the bound and takes the exact test; rows 32-127 and the second
    # query tile pass it
    B, H, S = 1, 2, 400
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=77 + D)
    qf = fsa_inputs.bf16_bits_to_f32(q)
    qf[:, :, :32, :] *= np.float32(40.0)
    q = fsa_inputs.to_bf16_bits(qf)
    _check(fsa, q, k, v, fmt, theta=80.0)


@pytest.mark.parametrize("fmt", ["mxfp6", "mxfp4"])
def test_one_large_key_tile_unbounds_the_head(fsa, fmt):
    # one key row x30 in the last tile raises the head's key bound: every warp
    # of that head takes the exact test, the other head keeps the shortcut
    B, H, S, D = 1, 2, 520, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=91)
    kf = fsa_inputs.bf16_bits_to_f32(k)
    kf[0, 1, 515, :] *= np.float32(30.0)
    k = fsa_inputs.to_bf16_bits(kf)
    _check(fsa, q, k, v, fmt, theta=80.0)


@pytest.mark.parametrize("fmt", ["mxfp6", "mxfp4", "mxfp8"])
def test_near_bf16_maximum_values_in_v(fsa, fmt):
    # one key row of V at 2^126 (scale exponent X > 121: the six-bit
    # quantizer keeps the exact decode there instead of the v / 64 pattern
    # with exponent X + 6, which E8M0 could not hold); the output stays
    # finite because that key carries one weight among many
    B, H, S, D = 1, 2, 700, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=88)
    vf = fsa_inputs.bf16_bits_to_f32(v)
    vf[0, 0, 333, :] = np.float32(2.0 ** 126) * np.sign(vf[0, 0, 333, :] + 0.5)
    v = fsa_inputs.to_bf16_bits(vf)
    _check(fsa, q, k, v, fmt)
