"""GPU parity of the EFQ-Softmax format (FSA_MXFP4_EFQ: MXFP4 Q/K/V, online
attention with the running row maximum, E2M1 P generated directly from the
shifted scores) against the oracle's "efq" mode, through the C ABI.  Same
bar as the other formats: output relative L2 <= 5e-3 against the oracle's
FP64 result."""
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


SMALL = [(1, 1, 2049, 128), (1, 2, 512, 64), (1, 1, 1, 64), (1, 2, 31, 128), (2, 1, 33, 64), (1, 1, 129, 128),
         (1, 3, 300, 64), (1, 1, 1000, 128), (2, 2, 257, 128)]


@pytest.mark.parametrize("shape", SMALL)
def test_efq_matches_oracle_small(fsa, shape):
    B, H, S, D = shape
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=S + 3 * D)
    o = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp4_efq")
    assert fsa.get_device_error() == 0
    got = to_f64(o).reshape(-1, D)
    ref = oracle.attention(q, k, v, fmt="mxfp4", mode="efq")["out"]
    assert np.all(np.isfinite(got))
    parity.check_out(f"efq {shape}", got, ref)


def test_efq_custom_rule_parameters(fsa):
    B, H, S, D = 1, 2, 900, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=71)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    for tau, h in ((-1.5, 0.55), (-3.0, 0.8)):
        o = fsa.attention_fwd(tq, tk, tv, fmt="mxfp4_efq", efq_tau=tau, efq_h=h)
        assert fsa.get_device_error() == 0
        ref = oracle.attention(q, k, v, fmt="mxfp4", mode="efq", efq_tau=tau, efq_h=h)["out"]
        parity.check_out(f"efq tau={tau} h={h}", to_f64(o).reshape(-1, D), ref)


def test_efq_growing_maximum(fsa):
    # keys scaled by 8 after position 2048 make the running maximum grow often
    B, H, S, D = 1, 2, 4096, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=72, stress_from=2048)
    o = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp4_efq")
    assert fsa.get_device_error() == 0
    ref = oracle.attention(q, k, v, fmt="mxfp4", mode="efq")["out"]
    parity.check_out(f"efq growing maximum", to_f64(o).reshape(-1, D), ref)


def test_efq_full_size_sampled(fsa):
    B, H, S, D = 1, 16, 8192, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=73)
    o = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp4_efq")
    assert fsa.get_device_error() == 0
    rng = np.random.default_rng(73)
    rows = np.unique(np.concatenate([np.arange(128), S * 15 + np.arange(S - 128, S),
                                     rng.integers(0, B * H * S, 256)])).astype(np.int64)
    got = to_f64(o).reshape(-1, D)[rows]
    ref = oracle.attention(q, k, v, fmt="mxfp4", mode="efq", rows=rows)["out"]
    parity.check_out(f"efq h16-s8192", got, ref)


@pytest.mark.parametrize("S", [16384, 16385])
def test_efq_at_the_persistent_boundary(fsa, S):
    # 128 KV tiles per item run the EFQ producer's persistent kernel, 129 (a
    # ragged last tile of one key) the one-CTA-per-item kernel; the growing
    # maximum of the second half rescales O and l in both
    B, H, D = 1, 2, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=74, stress_from=S // 2)
    o = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp4_efq")
    assert fsa.get_device_error() == 0
    rng = np.random.default_rng(74)
    rows = np.unique(np.concatenate([np.arange(128), (B * H - 1) * S + np.arange(S - 128, S),
                                     rng.integers(0, B * H * S, 128)])).astype(np.int64)
    got = to_f64(o).reshape(-1, D)[rows]
    ref = oracle.attention(q, k, v, fmt="mxfp4", mode="efq", rows=rows)["out"]
    parity.check_out(f"efq boundary S={S}", got, ref)
