"""GPU parity of the shortcut rollback gate (fsa_options.gate_mode = 1,
"Fused-Softmax shifts ...", paragraph 12: the fastest four-bit kernel gates
on converted values and can miss a recovery trigger) against the oracle's
gate="shortcut" mode, through the C ABI: the rollback decision of every
(row, tile) identical except near-ties -- here tiles whose excess lies within
1e-4 of the raised threshold theta*, where the shortcut's decision flips --
and the output within the parity bar.  On the rollback-stress workload the
GPU's own bits also give the miss rate against the FP32 gate: every miss has
its excess in (theta, theta*]."""
import numpy as np
import pytest
import torch

import fsa_inputs
import oracle
import parity
from gpu_util import to_dev, to_f64
from test_oracle_gate_shortcut import theta_star

pytestmark = pytest.mark.gpu
THETA = 8.0


@pytest.fixture(scope="module")
def fsa():
    import __graft_entry__
    __graft_entry__.build()
    import matrix_core_softmax_gb300 as m
    return m


def _run(fsa, q, k, v, fmt, gate, theta=THETA):
    B, H, S, D = q.shape
    n_t = (S + 127) // 128
    rb = torch.full((B * H * S, n_t), 7, dtype=torch.uint8, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    o = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt, threshold=theta,
                          rollback_bits=rb, rollback_count=cnt, gate=gate)
    st = fsa.get_device_error()
    assert st == 0, fsa.status_string(st)
    return o, rb, int(cnt.item())


def _star_margins(margins, fmt, theta=THETA):
    # the shortcut fires iff the excess passes theta*: its gate margin
    return margins + theta - theta_star(theta, fmt)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
def test_shortcut_gate_matches_oracle(fsa, fmt):
    B, H, S, D = 1, 2, 4096, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=51, stress_from=2048)
    o, rb, cnt = _run(fsa, q, k, v, fmt, "shortcut")
    r = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=THETA, gate="shortcut",
                         want_bits=True, want_margins=True)
    bits = rb.cpu().numpy()
    skip, _ = parity.check_bits(f"shortcut h2 s4096 {fmt} bits", bits, r["bits"],
                                _star_margins(r["margins"], fmt))
    assert r["rollback_count"] > 0
    assert cnt == int(bits.sum())
    parity.check_out(f"shortcut h2 s4096 {fmt}", to_f64(o).reshape(-1, D), r["out"], skip_rows=skip)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_shortcut_gate_on_the_small_shapes(fsa, fmt):
    # ragged tails and one-tile heads: nothing to gate or a partial last tile
    for B, H, S, D in [(1, 1, 1, 64), (2, 1, 33, 64), (1, 3, 300, 64), (2, 2, 257, 128)]:
        q, k, v = fsa_inputs.qkv(B, H, S, D, seed=S + 5 * D)
        o, rb, _ = _run(fsa, q, k, v, fmt, "shortcut")
        r = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=THETA, gate="shortcut",
                             want_bits=True, want_margins=True)
        skip, _ = parity.check_bits(f"shortcut {(B, H, S, D)} {fmt} bits", rb.cpu().numpy(),
                                    r["bits"], _star_margins(r["margins"], fmt))
        parity.check_out(f"shortcut {(B, H, S, D)} {fmt}", to_f64(o).reshape(-1, D), r["out"],
                         skip_rows=skip)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
def test_shortcut_on_rollback_stress_and_its_miss_rate(fsa, fmt):
    B, H, S, D = 1, 8, 32768, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=0, stress_from=16384)
    o_s, rb_s, cnt_s = _run(fsa, q, k, v, fmt, "shortcut")
    o_f, rb_f, cnt_f = _run(fsa, q, k, v, fmt, "fp32")
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([np.arange(128), (B * H - 1) * S + np.arange(S - 128, S),
                                     rng.integers(0, B * H * S, 256)])).astype(np.int64)
    r = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=THETA, gate="shortcut", rows=rows,
                         want_bits=True, want_margins=True)
    sel = torch.from_numpy(rows).cuda()
    skip, _ = parity.check_bits(f"shortcut rollback-stress {fmt} bits", rb_s[sel].cpu().numpy(),
                                r["bits"], _star_margins(r["margins"], fmt))
    parity.check_out(f"shortcut rollback-stress {fmt}", to_f64(o_s).reshape(-1, D)[rows], r["out"],
                     skip_rows=skip)
    # misses against the FP32 gate, from the GPU's own bits over every row:
    # at a row's first differing tile the FP32 gate fired and the shortcut
    # did not, and the oracle's excess there lies in (theta, theta*]
    bs, bf = rb_s.cpu().numpy(), rb_f.cpu().numpy()
    differ = bs != bf
    first = np.where(differ.any(axis=1), differ.argmax(axis=1), -1)
    miss_rows = np.nonzero(first >= 0)[0]
    assert cnt_f > cnt_s > 0
    assert np.all(bf[miss_rows, first[miss_rows]] == 1) and np.all(bs[miss_rows, first[miss_rows]] == 0)
    check = miss_rows[:64]
    m = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=THETA, rows=check.astype(np.int64),
                         want_margins=True)["margins"]
    excess = m[np.arange(len(check)), first[check]] + THETA
    ts = theta_star(THETA, fmt)
    assert np.all((excess > THETA - 1e-4) & (excess <= ts + 1e-4)), (excess.min(), excess.max(), ts)
    parity.log(f"shortcut miss rate {fmt} (GPU bits, every row)", fp32_firings=cnt_f,
               shortcut_firings=cnt_s, rows_with_a_miss=int(len(miss_rows)),
               miss_rate_per_fp32_firing=len(miss_rows) / cnt_f, theta_star=ts)
