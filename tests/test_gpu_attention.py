"""GPU parity of the fused attention (fsa_attention_fwd_ex, through the C
ABI) and of the BF16 baseline against the CPU oracle.

Bar (tests/parity.py): output relative L2 <= 5e-3 against the oracle's
FP64 result for the fused kernel over the compared rows, every row within
0.1 and at most 1 % of them above 5e-3 (1e-2 against exact attention for
the BF16 kernel); rollback decisions identical
per (row, tile) except near-ties, i.e. tiles whose gate margin |max s - m -
theta| is below 1e-4 in score units, where FP32 accumulation order on the
GPU may legitimately decide the other way -- counted, and at most 0.1 % of
the decisions.  The full-size workloads the bench measures are in
test_gpu_configs.py."""
import math

import numpy as np
import pytest
import torch

import fsa_inputs
import oracle
import parity
from gpu_util import to_dev, to_f64

pytestmark = pytest.mark.gpu
TOL = parity.TOL


@pytest.fixture(scope="module")
def fsa():
    import __graft_entry__
    __graft_entry__.build()
    import matrix_core_softmax_gb300 as m
    return m


def _run(fsa, q, k, v, fmt, theta=8.0, want_bits=False):
    B, H, S, D = q.shape
    n_t = (S + 127) // 128
    rb = torch.full((B * H * S, n_t), 7, dtype=torch.uint8, device="cuda") if want_bits else None
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    o = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt, threshold=theta,
                          rollback_bits=rb, rollback_count=cnt)
    st = fsa.get_device_error()
    assert st == 0, fsa.status_string(st)
    return o, rb, int(cnt.item())


# up to 2048 keys (16 KV tiles) the persistent kernel runs; beyond, one CTA
# per (query tile, head): 2049 and 2200 keys put a ragged tail of 1 and 24
# keys on the one-CTA kernel
SMALL = [(1, 2, 512, 64), (1, 1, 1, 64), (1, 2, 31, 128), (2, 1, 33, 64), (1, 1, 129, 128),
         (1, 3, 300, 64), (1, 1, 1000, 128), (2, 2, 257, 128), (1, 1, 2049, 128), (1, 2, 2200, 64)]


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
@pytest.mark.parametrize("shape", SMALL)
def test_fused_matches_oracle_small(fsa, fmt, shape):
    B, H, S, D = shape
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=S + D)
    o, rb, _ = _run(fsa, q, k, v, fmt, want_bits=True)
    got = to_f64(o).reshape(-1, D)
    r = oracle.attention(q, k, v, fmt=fmt, mode="fused", want_bits=True, want_margins=True)
    skip, _ = parity.check_bits(f"small {shape} {fmt} bits", rb.cpu().numpy(), r["bits"], r["margins"])
    parity.check_out(f"small {shape} {fmt}", got, r["out"], skip_rows=skip)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
def test_rollback_decisions_match_oracle(fsa, fmt):
    B, H, S, D = 1, 2, 4096, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=3, stress_from=2048)
    o, rb, cnt = _run(fsa, q, k, v, fmt, want_bits=True)
    r = oracle.attention(q, k, v, fmt=fmt, mode="fused", want_bits=True, want_margins=True)
    bits = rb.cpu().numpy()
    skip, _ = parity.check_bits(f"stress h2 s4096 {fmt} bits", bits, r["bits"], r["margins"])
    assert r["rollback_count"] > 0
    assert cnt == int(bits.sum())
    parity.check_out(f"stress h2 s4096 {fmt}", to_f64(o).reshape(-1, D), r["out"], skip_rows=skip)


def _sample(BH, S, per_head=96, seed=0):
    rng = np.random.default_rng(seed + 1000)
    heads = sorted({0, BH // 2, BH - 1})
    last0 = ((S - 1) // 128) * 128
    rows = []
    for h in heads:
        rows += [h * S + np.arange(0, min(128, S)), h * S + np.arange(last0, S),
                 h * S + rng.integers(0, S, per_head)]
    return np.unique(np.concatenate(rows)).astype(np.int64)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
def test_fused_full_size_h16_s8192(fsa, fmt):
    B, H, S, D = 1, 16, 8192, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=0)
    o, _, cnt = _run(fsa, q, k, v, fmt)
    got = to_f64(o).reshape(-1, D)
    assert np.all(np.isfinite(got))
    rows = _sample(B * H, S)
    ref = oracle.attention(q, k, v, fmt=fmt, mode="fused", rows=rows)
    parity.check_out(f"h16-s8192 seed 0 {fmt}", got[rows], ref["out"])
    assert cnt == 0          # N(0,1) inputs never pass the frozen reference by 8


@pytest.mark.parametrize("shape", [(1, 2, 512, 64), (1, 1, 300, 128), (2, 2, 1000, 128), (1, 1, 5, 64)])
def test_bf16_kernel_matches_exact_attention(fsa, shape):
    B, H, S, D = shape
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=1)
    o = fsa.bf16_attention_fwd(to_dev(q), to_dev(k), to_dev(v))
    assert fsa.get_device_error() == 0
    ref = oracle.attention(q, k, v, fmt=None, mode="exact")["out"]
    assert oracle.rel_l2(to_f64(o).reshape(-1, D), ref) <= 1e-2


def test_bounded_wait_reports_timeout_and_context_survives(fsa):
    # the loader skips KV tile 1: every wait on it must give up, the kernel
    # must exit cleanly, and the next call on the same context must work
    # (18 KV tiles: the one-CTA-per-item kernel; the persistent kernel's own
    # case is in test_gpu_persistent.py)
    B, H, S, D = 1, 1, 2304, 64
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=2)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    fsa.attention_fwd(tq, tk, tv, fmt="mxfp8", wait_timeout_ms=200,
                      debug_flags=fsa.DEBUG_SKIP_KV_ARRIVE)
    assert fsa.get_device_error() == 5
    assert fsa.get_device_error() == 0          # cleared
    o = fsa.attention_fwd(tq, tk, tv, fmt="mxfp8")
    assert fsa.get_device_error() == 0
    ref = oracle.attention(q, k, v, fmt="mxfp8", mode="fused")["out"]
    parity.check_out("after timeout", to_f64(o).reshape(-1, D), ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
@pytest.mark.parametrize("qscale", [16.0, 0.02])
def test_fused_wide_and_narrow_score_ranges(fsa, fmt, qscale):
    # q x 16: scores spread over hundreds of natural-log units, so weights
    # underflow (clamped codes, subnormal P blocks); q x 0.02: nearly flat rows
    B, H, S, D = 1, 2, 600, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=21)
    q = fsa_inputs.to_bf16_bits(fsa_inputs.bf16_bits_to_f32(q) * np.float32(qscale))
    o, _, _ = _run(fsa, q, k, v, fmt, theta=80.0)
    ref = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=80.0)["out"]
    parity.check_out(f"q x {qscale} {fmt}", to_f64(o).reshape(-1, D), ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_gate_at_theta_zero(fsa, fmt):
    # theta = 0: every tile whose max passes the reference rolls back
    B, H, S, D = 1, 2, 1500, 64
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=22)
    o, rb, cnt = _run(fsa, q, k, v, fmt, theta=0.0, want_bits=True)
    r = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=0.0, want_bits=True,
                         want_margins=True)
    skip, _ = parity.check_bits(f"theta 0 {fmt} bits", rb.cpu().numpy(), r["bits"], r["margins"])
    assert r["rollback_count"] > 100
    assert cnt == int(rb.sum().item())
    parity.check_out(f"theta 0 {fmt}", to_f64(o).reshape(-1, D), r["out"], skip_rows=skip)


@pytest.mark.parametrize("fmt,gate", [("mxfp8", "fp32"), ("mxfp6", "fp32"), ("mxfp4_efq", "fp32"),
                                      ("mxfp8", "shortcut")])
def test_maximum_head_count(fsa, fmt, gate):
    # B * H = 65535, the largest the entry points accept (the launch grids'
    # y limit): the quantizers' per-head grids, the persistent kernel with
    # 65535 work items and, through the shortcut gate's one-CTA-per-item
    # kernel, a grid of 65535 heads; three keys and ragged query tiles
    B, H, S, D = 3, 21845, 3, 64
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=91)
    o = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt, threshold=8.0, gate=gate)
    st = fsa.get_device_error()
    assert st == 0, fsa.status_string(st)
    rng = np.random.default_rng(91)
    BHS = B * H * S
    rows = np.unique(np.concatenate([np.arange(6), BHS - 6 + np.arange(6),
                                     rng.integers(0, BHS, 512)])).astype(np.int64)
    got = to_f64(o).reshape(-1, D)[rows]
    if fmt == "mxfp4_efq":
        ref = oracle.attention(q, k, v, fmt="mxfp4", mode="efq", rows=rows)["out"]
    else:
        ref = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=8.0, gate=gate, rows=rows)["out"]
    parity.check_out(f"max heads {fmt} {gate}", got, ref)
