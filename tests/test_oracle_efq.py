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
