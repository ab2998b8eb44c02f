"""The gate shortcut on converted values (the oracle's gate="shortcut"),
pinned by a closed form: X (the P block scale) is a step function of the
largest weight code, so the shortcut is exactly the FP32 gate with the
threshold raised to theta*, the score excess at which the Schraudolph code
first reaches a larger scale than theta's own code.  theta* is computed here
from the scale rule written out independently of the oracle."""
import math

import numpy as np
import pytest

import fsa_inputs
import oracle

LOG2E = 1.4426950408889634
MAXV = {"mxfp8": 448.0, "mxfp6": 7.5, "mxfp4": 7.5}   # P element: E4M3, E2M3, E2M3


def code_of(d):
    y = 128.0 * (d * LOG2E + 127.0) - 7.0
    return int(min(max(np.rint(y), 0), 0x7F7F))


def bf16_value(code):
    return float(np.array([code << 16], np.uint32).view(np.float32)[0])


def scale_exp(amax, maxv):
    # smallest X with amax <= maxv * 2^X
    x = math.ceil(math.log2(amax / maxv))
    while amax > math.ldexp(maxv, x):
        x += 1
    while amax <= math.ldexp(maxv, x - 1):
        x -= 1
    return x


def theta_star(theta, fmt):
    xt = scale_exp(bf16_value(code_of(theta)), MAXV[fmt])
    c = code_of(theta)
    while scale_exp(bf16_value(c + 1), MAXV[fmt]) <= xt:
        c += 1
    # the shortcut fires iff rne(y(d)) > c, i.e. y(d) > c + 0.5
    return ((c + 0.5 + 7.0) / 128.0 - 127.0) / LOG2E


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
def test_shortcut_is_fp32_gate_at_raised_threshold(fmt):
    theta = 8.0
    ts = theta_star(theta, fmt)
    assert theta < ts < theta + math.log(2.0)       # within one scale binade of theta
    q, k, v = fsa_inputs.qkv(1, 2, 4096, 128, seed=51, stress_from=2048)
    a = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=theta, gate="shortcut",
                         want_bits=True)
    b = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=ts, gate="fp32", want_bits=True)
    assert a["rollback_count"] > 0
    assert np.array_equal(a["bits"], b["bits"])
    assert np.array_equal(a["out"], b["out"])


def test_shortcut_misses_only_within_the_band():
    # the FP32 gate's firings the shortcut misses are exactly those whose
    # excess lies in (theta, theta*], read at the first difference per row
    theta, fmt = 8.0, "mxfp4"
    ts = theta_star(theta, fmt)
    q, k, v = fsa_inputs.qkv(1, 2, 4096, 128, seed=52, stress_from=2048)
    f = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=theta, want_bits=True,
                         want_margins=True)
    s = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=theta, gate="shortcut",
                         want_bits=True)
    for row in range(f["bits"].shape[0]):
        diff = np.nonzero(f["bits"][row] != s["bits"][row])[0]
        if len(diff) == 0:
            continue
        t = diff[0]
        excess = f["margins"][row, t] + theta
        assert f["bits"][row, t] == 1 and s["bits"][row, t] == 0
        assert theta < excess <= ts + 1e-9
