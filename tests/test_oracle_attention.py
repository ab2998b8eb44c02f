"""Pins of the attention oracle against mathematics and the pages:

* with quantization and the approximate exponential switched off the method
  is exact softmax attention, whatever the gate threshold, so the frozen
  reference, the gate and the rescale must reproduce a direct FP64 softmax;
* at S <= 8 (one partial tile, no gate) a brute-force few-line restatement
  built on torch's float8 cast and exhaustive grid search must agree exactly;
* power-of-two scalings of V and of K rows act exactly (block axes);
* the pages' error split (ten seeds, N(0,1) inputs) is reproduced.
"""
import math
import os

import numpy as np
import pytest
import torch

import fsa_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f(bits):
    return fsa_inputs.bf16_bits_to_f32(bits).astype(np.float64)


def _softmax_attention(q, k, v):
    """Direct FP64 softmax(Q K^T / sqrt(D)) V per head."""
    qf, kf, vf = _f(q), _f(k), _f(v)
    D = qf.shape[-1]
    s = np.einsum("hid,hjd->hij", qf, kf) / math.sqrt(D)
    s -= s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    return np.einsum("hij,hjd->hid", p, vf) / p.sum(-1)[..., None]


@pytest.mark.parametrize("S", [1, 5, 130, 300])
def test_exact_mode_is_softmax_attention(S):
    q, k, v = fsa_inputs.qkv(1, 2, S, 64, seed=S)
    ref = _softmax_attention(q[0], k[0], v[0]).reshape(-1, 64)
    got = oracle.attention(q, k, v, fmt=None, mode="exact", threads=2)["out"]
    assert oracle.rel_l2(got, ref) < 1e-12


@pytest.mark.parametrize("theta", [0.0, 0.25, 8.0])
@pytest.mark.parametrize("stress", [False, True])
def test_frozen_reference_gate_and_rescale_are_exact(theta, stress):
    # with exact exp and no quantization, freezing the reference at tile 0
    # and rolling back on a gate hit must give softmax attention exactly
    S = 700
    q, k, v = fsa_inputs.qkv(1, 2, S, 64, seed=7, stress_from=200 if stress else None,
                             stress_frac=0.05)
    ref = _softmax_attention(q[0], k[0], v[0]).reshape(-1, 64)
    r = oracle.attention(q, k, v, fmt=None, mode="exact_frozen", threshold=theta, threads=2,
                         want_bits=True)
    assert oracle.rel_l2(r["out"], ref) < 1e-12
    if theta == 0.0 or stress:
        assert r["rollback_count"] > 0       # the rescale path really ran
    assert r["rollback_count"] == int(r["bits"].sum())
    assert not r["bits"][:, 0].any()           # tile 0 initialises, never rolls back


def test_gate_does_not_fire_on_normal_inputs_and_fires_under_stress():
    q, k, v = fsa_inputs.qkv(1, 1, 2048, 128, seed=0)
    r = oracle.attention(q, k, v, fmt="mxfp8", mode="fused", threads=4, want_bits=True)
    assert r["rollback_count"] == 0
    q, k, v = fsa_inputs.qkv(1, 1, 2048, 128, seed=0, stress_from=1024)
    r = oracle.attention(q, k, v, fmt="mxfp8", mode="fused", threads=4, want_bits=True)
    assert r["rollback_count"] > 0
    assert not r["bits"][:, : 1024 // 128].any()   # no stressed keys before 1024


# ---------------------------------------------------------------- brute force
_GRID = {}


def _grid(name):
    """Non-negative values of a narrow format, by exhaustive enumeration of
    the E4M3 grid restricted to the narrow format's mantissa width and range
    (torch decodes E4M3; no oracle code involved)."""
    if name not in _GRID:
        e4 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
        if name == "e4m3":
            g = e4
        elif name == "e2m3":   # step 1/8 below 1, 3 mantissa bits above, max 7.5
            g = np.array([x for x in e4 if x <= 7.5 and (x * 8) == np.floor(x * 8)
                          and (x < 1 or (x / 2 ** np.floor(np.log2(x)) * 8) % 1 == 0)])
        elif name == "e2m1":   # step 1/2 below 1, 1 mantissa bit above, max 6
            g = np.array([x for x in e4 if x <= 6 and (x * 2) == np.floor(x * 2)
                          and (x < 1 or (x / 2 ** np.floor(np.log2(x)) * 2) % 1 == 0)])
        _GRID[name] = np.unique(g)
    return _GRID[name]


def _rne_to_grid(x, g):
    """Nearest grid value, ties to the one with even index (even mantissa)."""
    a = np.abs(x)
    d = np.abs(a[..., None] - g)
    best = d.min(-1, keepdims=True)
    idx = np.argmin(np.where(d == best, np.arange(len(g)) & 1, 9), axis=-1)
    return np.sign(x) * g[idx]


def _mx(x, name, axis):
    """MX quantization along `axis` in blocks of 32 (last block short)."""
    g = _grid(name)
    x = np.moveaxis(np.asarray(x, np.float64), axis, -1)
    out = np.empty_like(x)
    n = x.shape[-1]
    for b0 in range(0, n, 32):
        blk = x[..., b0:b0 + 32]
        amax = np.abs(blk).max(-1, keepdims=True)
        X = np.where(amax > 0, np.ceil(np.log2(np.where(amax > 0, amax, 1) / g[-1])), -127)
        X = np.where(amax > g[-1] * 2.0 ** (X - 1), X, X - 1)   # exact fix-up
        X = np.where(amax > g[-1] * 2.0 ** X, X + 1, X)
        out[..., b0:b0 + 32] = _rne_to_grid(blk / 2.0 ** X, g) * 2.0 ** X
    return np.moveaxis(out, -1, axis)


def _brute_force_fused(q, k, v, qkv_name, p_name):
    """The whole method on one short tile: frozen reference = row max, no gate
    can fire, Schraudolph code by numpy bit view, two-stage MX P, l = sum P."""
    qh = _mx(_f(q), qkv_name, -1)
    kh = _mx(_f(k), qkv_name, -1)
    vh = _mx(_f(v), qkv_name, -2)
    D = qh.shape[-1]
    s = np.einsum("hid,hjd->hij", qh, kh) / math.sqrt(D)
    x = s - s.max(-1, keepdims=True)
    y = 128 * (x / math.log(2) + 127) - 7
    code = np.clip(np.round(y), 0, 0x7F7F).astype(np.uint32)   # numpy rounds half to even
    p = (code << 16).view(np.float32).astype(np.float64)
    ph = _mx(p, p_name, -1)
    return np.einsum("hij,hjd->hid", ph, vh) / ph.sum(-1)[..., None]


@pytest.mark.parametrize("fmt,names", [("mxfp8", ("e4m3", "e4m3")),
                                       ("mxfp6", ("e2m3", "e2m3")),
                                       ("mxfp4", ("e2m1", "e2m3"))])
@pytest.mark.parametrize("S,D", [(1, 64), (5, 64), (8, 128), (7, 96)])
def test_brute_force_tiny(fmt, names, S, D):
    q, k, v = fsa_inputs.qkv(1, 3, S, D, seed=11 * S + D)
    ref = _brute_force_fused(q[0], k[0], v[0], *names).reshape(-1, D)
    got = oracle.attention(q, k, v, fmt=fmt, mode="fused", threads=1)["out"]
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_brute_force_grids_have_the_format_sizes():
    assert len(_grid("e4m3")) == 127 and _grid("e4m3")[-1] == 448
    assert len(_grid("e2m3")) == 32 and _grid("e2m3")[-1] == 7.5
    assert len(_grid("e2m1")) == 8 and _grid("e2m1")[-1] == 6


# ---------------------------------------------------------- invariances
@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
def test_v_column_power_of_two_scaling_is_exact(fmt):
    # V blocks run along the keys, so doubling one column of V doubles only
    # that output column, bit for bit; blocks along D would break this
    q, k, v = fsa_inputs.qkv(1, 1, 300, 64, seed=3)
    base = oracle.attention(q, k, v, fmt=fmt, mode="fused", threads=2)["out"]
    v2 = v.copy()
    v2[..., 5] = fsa_inputs.to_bf16_bits(fsa_inputs.bf16_bits_to_f32(v2[..., 5]) * 4)
    got = oracle.attention(q, k, v2, fmt=fmt, mode="fused", threads=2)["out"]
    assert np.array_equal(got[:, 5], 4 * base[:, 5])
    other = np.arange(64) != 5
    assert np.array_equal(got[:, other], base[:, other])


def test_k_row_scaling_by_8_shifts_scales_only():
    q, k, v = fsa_inputs.qkv(1, 1, 64, 128, seed=4)
    k8 = fsa_inputs.to_bf16_bits(fsa_inputs.bf16_bits_to_f32(k) * 8)
    for fmt in (oracle.E4M3, oracle.E2M3, oracle.E2M1):
        c, s = oracle.mx_quantize(k[0, 0], 1, fmt)
        c8, s8 = oracle.mx_quantize(k8[0, 0], 1, fmt)
        assert np.array_equal(c, c8)
        assert np.array_equal(s8.astype(int), s.astype(int) + 3)


def test_row_subset_gives_the_same_bytes():
    # rows are independent: computing a subset of rows gives the same bytes
    q, k, v = fsa_inputs.qkv(1, 2, 260, 64, seed=5)
    full = oracle.attention(q, k, v, fmt="mxfp8", mode="fused", threads=3)
    rows = np.array([519, 3, 260, 130, 0])
    sub = oracle.attention(q, k, v, fmt="mxfp8", mode="fused", rows=rows, threads=2)
    assert np.array_equal(sub["out"], full["out"][rows])


# ----------------------------------------------------- pages' error split
def _pages_numbers():
    tot, inc = {}, None
    with open(os.path.join(GOLDEN, "pages_error_split.txt")) as f:
        for l in f:
            if l.strip() and not l.startswith("#"):
                a, b = l.split()
                if a == "increment":
                    inc = float(b)
                else:
                    tot[a] = float(b)
    return tot, inc


@pytest.mark.slow
def test_error_split_matches_the_pages():
    """Ten seeds of N(0,1) inputs (S=8192, D=128, a 64-row sample per seed):
    the fused pipeline's relative error vs exact attention is within 1 pp of
    the pages' totals, and exceeds conventional softmax on the same
    quantized operands by at most the pages' 0.3 pp (+0.1 pp sampling
    tolerance)."""
    tot, inc = _pages_numbers()
    S, D = 8192, 128
    acc = {}
    for seed in range(10):
        q, k, v = fsa_inputs.qkv(1, 1, S, D, seed=seed)
        rows = np.arange(0, S, S // 64)
        ex = oracle.attention(q, k, v, fmt=None, mode="exact", rows=rows)["out"]
        for fmt in tot:
            for mode in ("fused", "conventional"):
                o = oracle.attention(q, k, v, fmt=fmt, mode=mode, rows=rows)["out"]
                a = acc.setdefault((fmt, mode), [0.0, 0.0])
                a[0] += float(np.sum((o - ex) ** 2))
                a[1] += float(np.sum(ex ** 2))
    for fmt, page in tot.items():
        fused = 100 * math.sqrt(acc[(fmt, "fused")][0] / acc[(fmt, "fused")][1])
        conv = 100 * math.sqrt(acc[(fmt, "conventional")][0] / acc[(fmt, "conventional")][1])
        assert abs(fused - page) < 1.0, (fmt, fused, page)
        assert fused - conv <= inc + 0.1, (fmt, fused, conv)
        assert fused - conv > 0.0
