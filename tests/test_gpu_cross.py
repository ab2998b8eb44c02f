"""GPU parity of the fused attention with Sq != Sk (fsa_cross_attention_fwd
and the prepare/run halves, through the C ABI) and of D = 64 at scale,
against the CPU oracle.  Same bar as the self-attention tests: output
relative L2 <= 5e-3 against the oracle's FP64 result, rollback decisions
identical per (row, tile) except near-ties (|max s - m - theta| < 1e-4)."""
import numpy as np
import pytest
import torch

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


def _qkv(B, H, Sq, Sk, D, seed, stress_from=None):
    q, _, _ = fsa_inputs.qkv(B, H, Sq, D, seed=seed)
    _, k, v = fsa_inputs.qkv(B, H, Sk, D, seed=seed + 1, stress_from=stress_from)
    return q, k, v


CROSS = [(1, 2, 37, 300, 64), (1, 2, 300, 37, 128), (2, 1, 129, 1000, 128), (1, 2, 1000, 129, 64),
         (1, 1, 1, 513, 128), (1, 3, 640, 128, 64), (1, 1, 256, 1, 128),
         # one query row against many KV tiles (one CTA walks 157 of them), and
         # a few rows against one key more than 32 tiles (a one-key tail tile)
         (1, 1, 1, 20000, 128), (2, 1, 3, 4097, 64)]


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
@pytest.mark.parametrize("shape", CROSS)
def test_cross_matches_oracle(fsa, fmt, shape):
    B, H, Sq, Sk, D = shape
    q, k, v = _qkv(B, H, Sq, Sk, D, seed=Sq + 7 * Sk)
    o = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt)
    assert fsa.get_device_error() == 0
    got = to_f64(o).reshape(-1, D)
    ref = oracle.attention(q, k, v, fmt=fmt, mode="fused")["out"]
    assert got.shape == ref.shape == (B * H * Sq, D)
    assert np.all(np.isfinite(got))
    parity.check_out(f"cross {shape} {fmt}", got, ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_cross_rollback_decisions(fsa, fmt):
    B, H, Sq, Sk, D = 1, 2, 700, 4096, 128
    q, k, v = _qkv(B, H, Sq, Sk, D, seed=41, stress_from=2048)
    n_t = (Sk + 127) // 128
    bits = torch.full((B * H * Sq, n_t), 7, dtype=torch.uint8, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    o = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt, rollback_bits=bits,
                                rollback_count=cnt)
    assert fsa.get_device_error() == 0
    r = oracle.attention(q, k, v, fmt=fmt, mode="fused", want_bits=True, want_margins=True)
    b = bits.cpu().numpy()
    skip, _ = parity.check_bits(f"cross rollback {fmt} bits", b, r["bits"], r["margins"])
    assert r["rollback_count"] > 0
    assert int(cnt.item()) == int(b.sum())
    parity.check_out(f"cross rollback {fmt}", to_f64(o).reshape(-1, D), r["out"], skip_rows=skip)


def test_cross_with_equal_lengths_is_self_attention(fsa):
    B, H, S, D = 1, 2, 777, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=43)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    for fmt in ("mxfp8", "mxfp6"):
        a = fsa.cross_attention_fwd(tq, tk, tv, fmt=fmt)
        b = fsa.attention_fwd(tq, tk, tv, fmt=fmt)
        assert fsa.get_device_error() == 0
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_cross_prepare_run_halves(fsa):
    B, H, Sq, Sk, D = 1, 2, 300, 1200, 64
    q, k, v = _qkv(B, H, Sq, Sk, D, seed=44)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    ws = fsa.new_cross_workspace(B, H, Sq, Sk, D)
    o = torch.empty_like(tq)
    fsa.cross_attention_prepare(tq, tk, tv, ws, "mxfp6")
    fsa.cross_attention_run(ws, o, Sk, "mxfp6")
    want = fsa.cross_attention_fwd(tq, tk, tv, fmt="mxfp6")
    assert fsa.get_device_error() == 0
    assert torch.equal(o.view(torch.int16), want.view(torch.int16))


def _sample(BH, S, per_head, seed):
    rng = np.random.default_rng(seed + 1000)
    heads = sorted({0, BH // 2, BH - 1})
    last0 = ((S - 1) // 128) * 128
    rows = []
    for h in heads:
        rows += [h * S + np.arange(0, min(128, S)), h * S + np.arange(last0, S),
                 h * S + rng.integers(0, S, per_head)]
    return np.unique(np.concatenate(rows)).astype(np.int64)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_d64_at_scale(fsa, fmt):
    B, H, S, D = 1, 16, 32768, 64
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=45)
    o = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt)
    assert fsa.get_device_error() == 0
    rows = _sample(B * H, S, 32, seed=45)
    got = to_f64(o).reshape(-1, D)[rows]
    ref = oracle.attention(q, k, v, fmt=fmt, mode="fused", rows=rows)["out"]
    assert np.all(np.isfinite(got))
    parity.check_out(f"d64 at scale {fmt}", got, ref)


@pytest.mark.parametrize("Sq,Sk", [(75600, 512), (4096, 32768)])
def test_cross_at_scale(fsa, Sq, Sk):
    # a video-token query against a short context (Sk = 512), and a short
    # query against a long context
    B, H, D = 1, 8, 128
    q, k, v = _qkv(B, H, Sq, Sk, D, seed=46)
    o = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp8")
    assert fsa.get_device_error() == 0
    rows = _sample(B * H, Sq, 32, seed=46)
    got = to_f64(o).reshape(-1, D)[rows]
    ref = oracle.attention(q, k, v, fmt="mxfp8", mode="fused", rows=rows)["out"]
    assert np.all(np.isfinite(got))
    parity.check_out(f"cross at scale Sq={Sq} Sk={Sk}", got, ref)
