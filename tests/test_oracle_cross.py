"""The oracle with Sq != Sk (queries and keys of different lengths), pinned
to what the definition fixes: exact mode is FP64 softmax attention written
with library matrix products, and rows are independent, so every row of a
cross-attention call equals the same row of a self-attention call on the
same keys and values."""
import numpy as np
import pytest

import fsa_inputs
import oracle


def _f64(bits):
    return fsa_inputs.bf16_bits_to_f32(bits).astype(np.float64)


def _direct_softmax(q, k, v):
    D = q.shape[-1]
    s = np.einsum("bid,bjd->bij", q, k) / np.sqrt(D)
    s -= s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    return np.einsum("bij,bjd->bid", p, v) / p.sum(axis=-1)[..., None]


@pytest.mark.parametrize("Sq,Sk,D", [(37, 300, 64), (300, 37, 64), (130, 257, 128), (1, 129, 32)])
def test_exact_cross_is_softmax_attention(Sq, Sk, D):
    q, _, _ = fsa_inputs.qkv(1, 2, Sq, D, seed=31)
    _, k, v = fsa_inputs.qkv(1, 2, Sk, D, seed=32)
    r = oracle.attention(q, k, v, fmt=None, mode="exact")
    want = _direct_softmax(_f64(q).reshape(2, Sq, D), _f64(k).reshape(2, Sk, D),
                           _f64(v).reshape(2, Sk, D)).reshape(-1, D)
    assert r["out"].shape == (2 * Sq, D)
    assert np.max(np.abs(r["out"] - want)) <= 1e-12 * np.max(np.abs(want))


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
def test_cross_rows_equal_self_attention_rows(fmt):
    # Sq < Sk: the queries extended to Sk rows give a self-attention call
    # whose first Sq rows must be bit-identical
    Sq, Sk, D = 90, 400, 64
    qe, k, v = fsa_inputs.qkv(1, 2, Sk, D, seed=33, stress_from=200)
    q = np.ascontiguousarray(qe[:, :, :Sq])
    cross = oracle.attention(q, k, v, fmt=fmt, mode="fused", want_bits=True)
    self_rows = np.concatenate([np.arange(Sq) + h * Sk for h in range(2)])
    ref = oracle.attention(qe, k, v, fmt=fmt, mode="fused", rows=self_rows, want_bits=True)
    assert np.array_equal(cross["out"], ref["out"])
    assert np.array_equal(cross["bits"], ref["bits"])
    assert cross["bits"].shape == (2 * Sq, (Sk + 127) // 128)
    assert cross["rollback_count"] == ref["rollback_count"] > 0


def test_cross_more_queries_than_keys_rows_independent():
    # Sq > Sk: a row subset computed alone equals the same rows of the full call
    Sq, Sk, D = 300, 70, 128
    q, _, _ = fsa_inputs.qkv(1, 1, Sq, D, seed=34)
    _, k, v = fsa_inputs.qkv(1, 1, Sk, D, seed=35)
    full = oracle.attention(q, k, v, fmt="mxfp8", mode="fused")
    rows = np.array([0, 69, 70, 128, 299], dtype=np.int64)
    part = oracle.attention(q, k, v, fmt="mxfp8", mode="fused", rows=rows)
    assert np.array_equal(part["out"], full["out"][rows])
    # and the first Sk rows equal self-attention on the first Sk queries
    self_att = oracle.attention(np.ascontiguousarray(q[:, :, :Sk]), k, v, fmt="mxfp8", mode="fused")
    assert np.array_equal(full["out"][:Sk], self_att["out"])
