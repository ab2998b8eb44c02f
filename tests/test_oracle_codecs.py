"""Pins of the oracle's element codecs, MX scale rule, bf16 rounding and
Schraudolph code against things other than the oracle itself: torch's own
float8 types, exhaustive brute force, values printed on the pages or in
Schraudolph's paper, and closed-form error bounds."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import E2M1, E2M3, E4M3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NBITS = {E4M3: 8, E2M3: 6, E2M1: 4}
MAXV = {E4M3: 448.0, E2M3: 7.5, E2M1: 6.0}


def _decode_all(fmt):
    return np.array([oracle.decode_elem(fmt, c) for c in range(1 << NBITS[fmt])])


def test_e4m3_decode_matches_torch_float8():
    ours = _decode_all(E4M3)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e2m1_largest_code_is_the_pages_value():
    with open(os.path.join(GOLDEN, "e2m1_largest_code.txt")) as f:
        code, value = [l.split() for l in f if l.strip() and not l.startswith("#")][0]
    assert oracle.decode_elem(E2M1, int(code)) == float(value)
    vals = _decode_all(E2M1)[:8]
    assert vals.max() == float(value)


@pytest.mark.parametrize("fmt", [E2M3, E2M1])
def test_narrow_formats_embed_exactly_in_e4m3(fmt):
    # every value of the narrow formats must survive an E4M3 round trip in
    # torch; a wrong bias or subnormal rule would leave the E4M3 grid
    vals = torch.tensor(_decode_all(fmt), dtype=torch.float32)
    back = vals.to(torch.float8_e4m3fn).float()
    assert torch.equal(vals, back)


@pytest.mark.parametrize("fmt", [E4M3, E2M3, E2M1])
def test_grid_structure(fmt):
    """Textbook structure of a binary format with gradual underflow: the
    non-negative codes are strictly increasing, the subnormal spacing equals
    the spacing of the first normal binade, and each binade above doubles
    the spacing of the one below."""
    half = 1 << (NBITS[fmt] - 1)
    v = _decode_all(fmt)[:half]
    if fmt == E4M3:
        v = v[:-1]  # 0x7F is NaN
    assert np.all(np.diff(v) > 0)
    assert v[0] == 0.0 and v[-1] == MAXV[fmt]
    neg = _decode_all(fmt)[half:half + len(v)]
    assert np.array_equal(neg, -v)
    mbits = {E4M3: 3, E2M3: 3, E2M1: 1}[fmt]
    per = 1 << mbits
    vv = _decode_all(fmt)[:half]  # includes E4M3's NaN slot at the end
    nb = half // per              # binades, exponent field 0 .. nb-1
    step = [None] * nb
    for b in range(1, nb):
        step[b] = vv[b * per] / per          # 2^(e - mbits)
        seg = vv[b * per: (b + 1) * per]
        seg = seg[~np.isnan(seg)]
        assert np.all(np.diff(seg) == step[b])
    step[0] = vv[1] - vv[0]
    assert np.all(np.diff(vv[:per]) == step[0])
    assert step[0] == step[1]                 # gradual underflow
    for b in range(2, nb):
        assert step[b] == 2 * step[b - 1]
    for b in range(1, nb):
        assert vv[b * per] - vv[b * per - 1] == step[b - 1]


def _brute_force_encode(fmt, x):
    """Nearest representable value by exhaustive search; ties go to the code
    with an even last mantissa bit.  Saturates at the largest finite value."""
    half = 1 << (NBITS[fmt] - 1)
    vals = _decode_all(fmt)[:half]
    if fmt == E4M3:
        vals = vals[:-1]
    a = np.minimum(np.abs(x), MAXV[fmt])
    dist = np.abs(a[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    codes = np.arange(len(vals))
    # prefer even code (mantissa LSB 0) among ties
    score = np.where(cand, (codes[None, :] & 1), 9)
    c = np.argmin(score, axis=1)
    sign = np.signbit(x).astype(np.int64) << (NBITS[fmt] - 1)
    return c | sign


@pytest.mark.parametrize("fmt", [E4M3, E2M3, E2M1])
def test_encode_is_round_to_nearest_even(fmt):
    rng = np.random.default_rng(1)
    # all finite bf16 patterns in the format's range, and midpoints
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    x = (bits << 16).view(np.float32).astype(np.float64)
    x = x[x <= MAXV[fmt] * 1.2]
    vals = _decode_all(fmt)[: 1 << (NBITS[fmt] - 1)]
    vals = vals[~np.isnan(vals)]
    mids = (vals[1:] + vals[:-1]) / 2
    x = np.concatenate([x, mids, -x[::97], rng.uniform(0, MAXV[fmt], 5000)])
    ours = np.array([oracle.encode_elem(fmt, float(t)) for t in x])
    ref = _brute_force_encode(fmt, x)
    assert np.array_equal(ours, ref)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(20000) * 30, rng.uniform(-448, 448, 20000),
                        rng.standard_normal(5000) * 1e-3])
    ours = np.array([oracle.encode_elem(E4M3, float(t)) for t in x], dtype=np.uint8)
    ref = torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch converts float64 via float32; x values are float32-exact above
    assert np.array_equal(ours, ref)


def test_double_to_bf16_matches_torch_for_float32_inputs():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-38,
                        rng.standard_normal(2000) * 1e30]).astype(np.float32)
    ours = np.array([oracle.double_to_bf16(float(t)) for t in x], dtype=np.uint16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_e8m0_scale_byte_decodes_with_torch():
    # the scale byte X + 127 must be the E8M0 encoding of 2^X (torch type)
    for X in (-127, -8, -2, 0, 5, 127):
        b = torch.tensor([X + 127], dtype=torch.uint8).view(torch.float8_e8m0fnu).double().item()
        assert b == 2.0 ** X


@pytest.mark.parametrize("fmt", [E4M3, E2M3, E2M1])
def test_scale_rule_smallest_non_saturating_power(fmt):
    """For every positive finite bf16 amax, 2^X is the smallest power of two
    whose scaled block maximum still encodes without saturation -- checked
    by brute force over candidate exponents with the exhaustive encoder."""
    bits = np.arange(1, 0x7F80, 37, dtype=np.uint32)
    amax = (bits << 16).view(np.float32).astype(np.float64)
    for a in amax:
        X = oracle.mx_scale_exp(fmt, float(a))
        lo = max(-127, X - 3)
        fits = [Y for Y in range(lo, min(127, X + 3) + 1) if a / 2.0 ** Y <= MAXV[fmt]]
        assert X == max(fits[0], -127)


def test_scale_rule_zero_block():
    for fmt in (E4M3, E2M3, E2M1):
        assert oracle.mx_scale_exp(fmt, 0.0) == -127


def test_scale_rule_power_of_two_equivariance():
    rng = np.random.default_rng(4)
    for fmt in (E4M3, E2M3, E2M1):
        for a in rng.uniform(1e-3, 1e3, 200):
            X = oracle.mx_scale_exp(fmt, a)
            for k in (-5, 3, 17):
                assert oracle.mx_scale_exp(fmt, a * 2.0 ** k) == X + k


def test_mx_quantize_layouts_and_tails():
    rng = np.random.default_rng(5)
    from fsa_inputs import to_bf16_bits
    x = to_bf16_bits(rng.standard_normal((2, 70, 45)).astype(np.float32))
    c1, s1 = oracle.mx_quantize(x, 1, E4M3)
    assert c1.shape == (2, 70, 45) and s1.shape == (2, 70, 2)
    c0, s0 = oracle.mx_quantize(x, 0, E4M3)
    assert c0.shape == (2, 45, 70) and s0.shape == (2, 45, 3)
    # block_axis 0 equals block_axis 1 on the transposed input
    xt = np.ascontiguousarray(np.swapaxes(x, 1, 2))
    c1t, s1t = oracle.mx_quantize(xt, 1, E4M3)
    assert np.array_equal(c0, c1t) and np.array_equal(s0, s1t)
    # dequantized values are within half an E4M3 step (relative 2^-4)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    dq = np.vectorize(lambda c: oracle.decode_elem(E4M3, int(c)))(c1)
    sc = 2.0 ** (np.repeat(s1.astype(np.float64) - 127, 32, axis=2)[:, :, :45])
    err = np.abs(dq * sc - xf)
    assert np.all(err <= np.maximum(np.abs(xf) * 2.0 ** -4, sc * 2.0 ** -10))


def _schraudolph_constants():
    vals = {}
    with open(os.path.join(GOLDEN, "schraudolph_1999.txt")) as f:
        for l in f:
            if l.strip() and not l.startswith("#"):
                k, v = l.split()
                vals[k] = int(v)
    return vals


def test_schraudolph_constants_follow_the_1999_paper():
    c = _schraudolph_constants()
    # b is the bias 1023 in the exponent field above 20 mantissa bits
    assert c["b"] == 1023 * 2 ** c["mantissa_bits_double_hi"]
    shift = c["mantissa_bits_double_hi"] - c["mantissa_bits_bf16"]
    c_bf16 = round(c["c"] / 2 ** shift)
    # x = 0: y = 2^7 * 127 - c_bf16
    assert oracle.schraudolph_y(0.0) == 128 * 127 - c_bf16
    assert oracle.schraudolph_code(oracle.schraudolph_y(0.0)) == 0x3F79
    assert oracle.bf16_to_double(0x3F79) == 0.97265625
    # slope: one unit of x moves y by 2^7 / ln 2 (a scaled from 2^20 to 2^7)
    slope = oracle.schraudolph_y(1.0) - oracle.schraudolph_y(0.0)
    assert slope == pytest.approx(c["a_num"] / 2 ** shift / math.log(2), rel=1e-12)


def test_schraudolph_relative_error_closed_form_bounds():
    """Ignoring integer rounding, the code represents 2^floor(v)(1+frac(v))
    with v = x log2 e - c/128, so the ratio to e^x is (1+f)/2^f * 2^(-c/128):
    between 2^(-7/128) = 0.96280 and max_f (1+f)/2^f * 2^(-7/128) = 1.02194
    (maximum at f = 1/ln2 - 1).  Rounding y to an integer widens that by a
    factor 2^(+-1/256)."""
    x = np.linspace(-20, 0, 200001)
    p = np.array([oracle.bf16_to_double(oracle.schraudolph_code(oracle.schraudolph_y(t)))
                  for t in x])
    r = p / np.exp(x) - 1
    f = 1 / math.log(2) - 1
    lo = 2 ** (-7 / 128) * 2 ** (-1 / 256) - 1
    hi = (1 + f) / 2 ** f * 2 ** (-7 / 128) * 2 ** (1 / 256) - 1
    assert r.min() >= lo - 1e-12 and r.max() <= hi + 1e-12
    # and the bounds are nearly reached (a dropped shift or a wrong slope
    # moves them by far more than this)
    assert r.min() < lo + 2e-3 and r.max() > hi - 2e-3
    assert lo == pytest.approx(-0.0398, abs=1e-3) and hi == pytest.approx(0.0248, abs=1e-3)


def test_schraudolph_clamps_to_non_negative_finite_bf16():
    assert oracle.schraudolph_code(-5.0) == 0
    assert oracle.schraudolph_code(1e9) == 0x7F7F
    assert oracle.schraudolph_code(2.5) == 2 and oracle.schraudolph_code(3.5) == 4  # RNE
