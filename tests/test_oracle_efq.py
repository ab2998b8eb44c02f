"""The oracle's EFQ-Softmax producer and online-attention mode, pinned by what
the definitions fix rather than by restating the rule: online attention with
exact exp is softmax attention; a single key, or equal scores, make the
output the (mean) dequantized value row whatever the codes; powers of two in
V pass through exactly; the block maximum always lands on one of the two
largest E2M1 codes (its residual lies in (log2 6 - 1, log2 6]); and the
library's calibrated (tau, h) is a local optimum of the calibration
objective."""
import math
import os

import numpy as np
import pytest

import fsa_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "efq_calibration.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if line:
            vals[line[0]] = float(line[1])
    return vals


def _vhat(v, D):
    # MXFP4-dequantized V along the keys: V's blocks run along the keys, so a
    # one-key head is a block of one element
    return oracle.attention(v, v, v, fmt="mxfp4", mode="operands_only")["out"]


def test_online_attention_is_softmax_attention():
    q, k, v = fsa_inputs.qkv(1, 2, 700, 64, seed=61)
    a = oracle.attention(q, k, v, fmt=None, mode="online")["out"]
    b = oracle.attention(q, k, v, fmt=None, mode="exact")["out"]
    assert np.max(np.abs(a - b)) <= 1e-12


def test_single_key_returns_its_value_row():
    q, _, _ = fsa_inputs.qkv(1, 3, 50, 64, seed=62)
    _, k, v = fsa_inputs.qkv(1, 3, 1, 64, seed=63)
    r = oracle.attention(q, k, v, fmt="mxfp4", mode="efq")["out"].reshape(3, 50, 64)
    # the same single key through the fused pipeline gives V-hat exactly as well
    ref = oracle.attention(q, k, v, fmt="mxfp4", mode="fused")["out"].reshape(3, 50, 64)
    assert np.array_equal(r, ref)
    assert np.all(np.abs(r[:, 1:] - r[:, :1]) == 0)


def test_equal_scores_give_the_mean_value_row():
    q, k, v = fsa_inputs.qkv(1, 1, 40, 64, seed=64)
    k[...] = k[:, :, :1]                        # every key the same row
    r = oracle.attention(q, k, v, fmt="mxfp4", mode="efq")["out"]
    # all weights equal, so the output is the mean of the dequantized V rows:
    # the same as exact softmax attention on the dequantized operands
    ref = oracle.attention(q, k, v, fmt="mxfp4", mode="operands_only")["out"]
    assert np.max(np.abs(r - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_value_power_of_two_equivariance():
    q, k, v = fsa_inputs.qkv(1, 2, 300, 64, seed=65)
    v2 = fsa_inputs.to_bf16_bits(fsa_inputs.bf16_bits_to_f32(v) * np.float32(8.0))
    a = oracle.attention(q, k, v, fmt="mxfp4", mode="efq")["out"]
    b = oracle.attention(q, k, v2, fmt="mxfp4", mode="efq")["out"]
    assert np.array_equal(b, 8.0 * a)


def test_block_maximum_takes_a_top_code():
    # one-hot value rows expose the quantized weights: with V_j = e_j (exact
    # in MXFP4), O_j / l is p-hat_j / sum(p-hat); inside one 32-key block the
    # largest weight must be 4 or 6 times the block scale, so p-hat_max /
    # p-hat_min over nonzero weights is bounded by 6 / 0.5 and the largest
    # weight of the block is one of the two top E2M1 values
    D = 32
    q, k, _ = fsa_inputs.qkv(1, 1, 32, D, seed=66)
    v = fsa_inputs.to_bf16_bits(np.eye(32, D, dtype=np.float32)[None, None])
    r = oracle.attention(q, k, v, fmt="mxfp4", mode="efq")["out"]
    w = r / r.sum(axis=1, keepdims=True)
    for row in w:
        nz = row[row > 0]
        top = nz.max()
        # every nonzero weight is an E2M1 value times the same scale
        ratios = nz / (top / 6.0), nz / (top / 4.0)
        grid = np.array([0.5, 1, 1.5, 2, 3, 4, 6])
        ok6 = np.all(np.min(np.abs(ratios[0][:, None] - grid[None]), axis=1) < 1e-9)
        ok4 = np.all(np.min(np.abs(ratios[1][:, None] - grid[None]), axis=1) < 1e-9)
        assert ok6 or ok4


@pytest.mark.slow
def test_calibration_is_a_local_optimum():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "efq_calibrate", os.path.join(os.path.dirname(__file__), "..", "oracle", "efq_calibrate.py"))
    cal = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(cal)
    g = _golden()
    assert (g["tau"], g["h"]) == (oracle.EFQ_TAU, oracle.EFQ_H)
    sets = cal.data()
    e0 = cal.objective(sets, g["tau"], g["h"])
    assert abs(e0 - g["error"]) < 1e-6
    for dt, dh in ((0.04, 0), (-0.04, 0), (0, 0.02), (0, -0.02)):
        assert cal.objective(sets, g["tau"] + dt, g["h"] + dh) >= e0 - 1e-9


def test_library_defaults_match_calibration():
    g = _golden()
    assert (g["tau"], g["h"]) == (oracle.EFQ_TAU, oracle.EFQ_H)


def _grid_row(dot):
    """A key row of 32 elements, every one on the E2M1 grid at scale 1 with
    a 6 among them (so the row's MX block has scale 2^0 and is exact), whose
    elements sum to `dot` (a multiple of 0.5).  Input construction only."""
    mags = [6.0, 4.0, 3.0, 2.0, 1.5, 1.0, 0.5]
    row, rest = [6.0], dot - 6.0
    while rest != 0.0:
        m = next(x for x in mags if x <= abs(rest))
        row.append(math.copysign(m, rest))
        rest -= math.copysign(m, rest)
    assert len(row) <= 32
    return row + [0.0] * (32 - len(row))


def test_code_mapping_hand_computed():
    """The code rule of the EFQ page's "Code mapping" step, code =
    clip(floor((r - tau) / h), 0, 7) with r = u - X, checked on a block whose
    residuals straddle chosen thresholds, the codes worked out by hand.

    One query row of 32 ones and 32 keys whose dot products with it are the
    values in DOTS (exact in MXFP4: q is 4 x 2^-2 everywhere, every key row is
    on the E2M1 grid at scale 1); sm = ln(2) / 16, so u_j = (s_j - m) log2(e)
    = (dot_j - 18) / 16 with m the largest score (dot 18).  The block's scale
    exponent is X = ceil(0 - log2 6) = -2, so r = u + 2, and with tau = -2,
    h = 0.5: code = clip(floor(2 u + 8), 0, 7) = clip(floor((dot - 18) / 8 +
    8), 0, 7).  Each pair in DOTS sits half a unit of dot on either side of a
    threshold (a wrong rounding, sign of tau, scale of h, offset of X or clip
    moves at least one code).  V is one-hot (V_j = e_j, exact in MXFP4), so
    output column j is p^_j / sum(p^) and o_j / o_0 = E2M1(code_j) / 6."""
    DOTS = [18, 10.5, 9.5, 2.5, 1.5, -5.5, -6.5, -13.5, -14.5, -21.5, -22.5, -29.5, -30.5,
            -37.5, -38.5, -60, 14, 6, -2, -10, -18, -26, -34, -42, -100, 17.5, 0, 4, 12, -16,
            -24, -32]
    CODES = [7, 7, 6, 6, 5, 5, 4, 4, 3, 3, 2, 2, 1, 1, 0, 0, 7, 6, 5, 4, 3, 2, 1, 0, 0, 7, 5,
             6, 7, 3, 2, 1]
    E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    q = fsa_inputs.to_bf16_bits(np.ones((1, 1, 1, 32), np.float32))
    k = fsa_inputs.to_bf16_bits(np.array([_grid_row(d) for d in DOTS], np.float32)[None, None])
    v = fsa_inputs.to_bf16_bits(np.eye(32, dtype=np.float32)[None, None])
    o = oracle.attention(q, k, v, fmt="mxfp4", mode="efq", sm_scale=math.log(2.0) / 16.0,
                         efq_tau=-2.0, efq_h=0.5)["out"][0]
    ratios = o / o[0]
    expected = np.array([E2M1[c] / 6.0 for c in CODES])
    assert np.max(np.abs(ratios - expected)) < 1e-12, list(zip(DOTS, ratios * 6.0, CODES))
