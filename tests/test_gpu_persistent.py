"""GPU parity of the persistent kernel (work items of at most 16 KV tiles,
128 for the EFQ producer, whose larger items tests/test_gpu_efq.py covers:
one CTA per SM, at most one per item, walks the items with double-buffered Q
and barrier phases carried across items; the cases here have more items than
SMs, so every CTA walks several) against the CPU oracle.  Same bar as the
other fused-attention tests (tests/parity.py)."""
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


@pytest.fixture(scope="module")
def n_sm():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _qkv(B, H, Sq, Sk, D, seed, stress_from=None):
    q, _, _ = fsa_inputs.qkv(B, H, Sq, D, seed=seed)
    _, k, v = fsa_inputs.qkv(B, H, Sk, D, seed=seed + 1, stress_from=stress_from)
    return q, k, v


# (B, H, Sq, Sk, D): 3 KV tiles with a ragged tail (odd: consecutive items start
# on alternating softmax warpgroups), 8 full tiles, a single one-key tile,
# D = 64 with 2 tiles and ragged query rows, B = 2, 16 tiles with a tail
SHAPES = [(1, 4, 5000, 300, 128), (1, 4, 4900, 1024, 128), (1, 4, 5000, 1, 128),
          (1, 8, 2500, 200, 64), (2, 2, 5000, 640, 128), (1, 2, 9800, 2000, 128)]


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4", "mxfp4_efq"])
@pytest.mark.parametrize("shape", SHAPES)
def test_persistent_matches_oracle(fsa, n_sm, fmt, shape):
    B, H, Sq, Sk, D = shape
    assert (Sk + 127) // 128 <= 16 and B * H * ((Sq + 127) // 128) > n_sm  # the persistent path
    q, k, v = _qkv(B, H, Sq, Sk, D, seed=Sq + 3 * Sk + D)
    o = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt)
    assert fsa.get_device_error() == 0
    got = to_f64(o).reshape(-1, D)
    if fmt == "mxfp4_efq":
        ref = oracle.attention(q, k, v, fmt="mxfp4", mode="efq")["out"]
    else:
        ref = oracle.attention(q, k, v, fmt=fmt, mode="fused")["out"]
    assert np.all(np.isfinite(got))
    parity.check_out(f"persistent {shape} {fmt}", got, ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_persistent_rollback_decisions(fsa, n_sm, fmt):
    # 1 % of the keys from 512 on scaled x8: later tiles pass the frozen maxima
    B, H, Sq, Sk, D = 1, 4, 5000, 1000, 128
    q, k, v = _qkv(B, H, Sq, Sk, D, seed=52, stress_from=512)
    n_t = (Sk + 127) // 128
    bits = torch.full((B * H * Sq, n_t), 7, dtype=torch.uint8, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    o = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt, rollback_bits=bits,
                                rollback_count=cnt)
    assert fsa.get_device_error() == 0
    r = oracle.attention(q, k, v, fmt=fmt, mode="fused", want_bits=True, want_margins=True)
    got_bits = bits.cpu().numpy()
    skip, _ = parity.check_bits(f"persistent rollback {fmt} bits", got_bits, r["bits"], r["margins"])
    assert r["rollback_count"] > 0
    assert int(cnt.item()) == int(got_bits.sum())
    parity.check_out(f"persistent rollback {fmt}", to_f64(o).reshape(-1, D), r["out"], skip_rows=skip)


def test_persistent_six_bit_mixed_norm_bounds(fsa, n_sm):
    # head 1's keys include one row x30: its warps fail the norm bound and
    # take the exact test, head 0's keep the shortcut, in the same CTAs
    B, H, Sq, Sk, D = 1, 2, 10000, 520, 128
    q, k, v = _qkv(B, H, Sq, Sk, D, seed=61)
    kf = fsa_inputs.bf16_bits_to_f32(k)
    kf[0, 1, 515, :] *= np.float32(30.0)
    k = fsa_inputs.to_bf16_bits(kf)
    o = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp6", threshold=80.0)
    assert fsa.get_device_error() == 0
    ref = oracle.attention(q, k, v, fmt="mxfp6", mode="fused", threshold=80.0)["out"]
    parity.check_out(f"persistent mixed norm bounds mxfp6", to_f64(o).reshape(-1, D), ref)


def test_persistent_equals_self_attention_path(fsa):
    # Sq = Sk = 1024 goes through the same persistent kernel as the cross call
    # with those sizes; the self-attention entry point must agree bit for bit
    B, H, S, D = 1, 20, 1024, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=71)
    a = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp8")
    b = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp8")
    assert fsa.get_device_error() == 0
    assert torch.equal(a, b)


def test_persistent_bounded_wait_reports_timeout_and_context_survives(fsa, n_sm):
    # every persistent CTA's K tile 1 never arrives: the waits on it give up,
    # all CTAs leave their item loops, and the next call on the context works
    B, H, S, D = 1, 20, 1024, 128
    assert H * ((S + 127) // 128) > n_sm
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=81)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    fsa.attention_fwd(tq, tk, tv, fmt="mxfp4", wait_timeout_ms=200,
                      debug_flags=fsa.DEBUG_SKIP_KV_ARRIVE)
    assert fsa.get_device_error() == 5
    assert fsa.get_device_error() == 0
    o = fsa.attention_fwd(tq, tk, tv, fmt="mxfp4")
    assert fsa.get_device_error() == 0
    ref = oracle.attention(q, k, v, fmt="mxfp4", mode="fused")["out"]
    parity.check_out(f"persistent after timeout mxfp4", to_f64(o).reshape(-1, D), ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "mxfp4_efq"])
def test_persistent_rollback_at_tile_one_with_many_items(fsa, n_sm, fmt):
    # theta = 0 (every tile whose maximum passes the reference rolls back, so
    # tile 1 of most items does) with several items per CTA: the rescale of
    # tile 1 waits for the item's first PV product, which waits for the
    # previous item's epilogue -- written first by the warpgroup that owes it.
    # The EFQ producer's growing running maximum takes the same path.
    B, H, Sq, Sk, D = 1, 8, 10000, 1000, 128
    assert B * H * ((Sq + 127) // 128) > 3 * n_sm and (Sk + 127) // 128 <= 16
    q, k, v = _qkv(B, H, Sq, Sk, D, seed=91)
    n_t = (Sk + 127) // 128
    bits = torch.full((B * H * Sq, n_t), 7, dtype=torch.uint8, device="cuda")
    o = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt, threshold=0.0,
                                rollback_bits=bits if fmt != "mxfp4_efq" else None)
    st = fsa.get_device_error()
    assert st == 0, fsa.status_string(st)
    rows = np.arange(0, B * H * Sq, 7).astype(np.int64)
    if fmt == "mxfp4_efq":
        r = oracle.attention(q, k, v, fmt="mxfp4", mode="efq", rows=rows)
        parity.check_out(f"persistent theta 0 {fmt}", to_f64(o).reshape(-1, D)[rows], r["out"])
        return
    r = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=0.0, rows=rows, want_bits=True,
                         want_margins=True)
    sel = bits[torch.from_numpy(rows).cuda()].cpu().numpy()
    skip, _ = parity.check_bits(f"persistent theta 0 {fmt} bits", sel, r["bits"], r["margins"])
    assert r["bits"][:, 1].sum() > len(rows) // 10      # tile 1 rolls back in many rows
    parity.check_out(f"persistent theta 0 {fmt}", to_f64(o).reshape(-1, D)[rows], r["out"],
                     skip_rows=skip)
