"""GPU parity of the MX quantizer (fsa_quantize_mx) against the oracle:
codes and scales must be bit-exact for all three element formats, both block
axes, ragged tails and special blocks."""
import numpy as np
import pytest
import torch

import fsa_inputs
import oracle
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fsa():
    import __graft_entry__
    __graft_entry__.build()
    import matrix_core_softmax_gb300 as m
    return m


def _special_bits():
    """bf16 patterns covering zero blocks, signed zeros, subnormals, the
    largest finite bf16, exact format maxima and round-to-even midpoints."""
    rng = np.random.default_rng(9)
    blocks = [
        np.zeros(32, np.uint16),
        np.full(32, 0x8000, np.uint16),                                   # -0.0
        rng.integers(1, 0x80, 32).astype(np.uint16),                      # subnormals
        (rng.integers(1, 0x80, 32) | 0x8000).astype(np.uint16),
        np.concatenate([[0x7F7F], rng.integers(0, 0x7F7F, 31)]).astype(np.uint16),  # max bf16
        fsa_inputs.to_bf16_bits(np.array([448.0, 464.0, 240.0, 7.5, 6.0, 5.0, 0.0625, 1e-3] * 4,
                                         np.float32)),
        fsa_inputs.to_bf16_bits(rng.standard_normal(32).astype(np.float32) * 1e-30),
        fsa_inputs.to_bf16_bits(rng.standard_normal(32).astype(np.float32) * 1e30),
    ]
    return np.concatenate(blocks)


@pytest.mark.parametrize("elem", [0, 1, 2])
@pytest.mark.parametrize("shape", [(1, 64, 128), (2, 75, 45), (3, 33, 64), (1, 1, 1), (1, 512, 64)])
@pytest.mark.parametrize("axis", [1, 0])
def test_quantize_bit_exact(fsa, elem, shape, axis):
    rng = np.random.default_rng(sum(shape) + elem)
    x = fsa_inputs.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) *
                                np.float32(rng.choice([1e-3, 1.0, 40.0])))
    codes, scales = fsa.quantize_mx(to_dev(x), axis, elem)
    rc, rs = oracle.mx_quantize(x, axis, elem)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("elem", [0, 1, 2])
@pytest.mark.parametrize("axis", [1, 0])
def test_quantize_special_blocks(fsa, elem, axis):
    sp = _special_bits().reshape(-1, 32)          # each row one block
    x = sp if axis == 1 else np.ascontiguousarray(sp.T)
    codes, scales = fsa.quantize_mx(to_dev(x), axis, elem)
    rc, rs = oracle.mx_quantize(x, axis, elem)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("elem", [0, 1, 2])
def test_quantize_qkv_layouts_at_config_size(fsa, elem):
    # Q/K blocks along D, V blocks along keys (transposed), 8192 x 128 heads
    q, k, v = fsa_inputs.qkv(1, 2, 8192, 128, seed=0)
    for x, axis in ((q, 1), (v, 0)):
        x3 = x.reshape(2, 8192, 128)
        codes, scales = fsa.quantize_mx(to_dev(x3), axis, elem)
        rc, rs = oracle.mx_quantize(x3, axis, elem)
        assert np.array_equal(scales.cpu().numpy(), rs)
        assert np.array_equal(codes.cpu().numpy(), rc)


# ---- the fused attention's own quantizer (fsa_attention_prepare) ----------
# Its output is the documented attention layout: E4M3 bit patterns of the
# quantized elements (a six-bit E2M3 block with scale exponent X <= 121 stored
# as the patterns of v / 64 with exponent X + 6), scale bytes in 128-row x
# 4-block atoms (row r, block kb at byte (r % 32) * 16 + (r / 32) * 4 + kb,
# unused entries 127), V transposed with its keys padded to a multiple of 16,
# and for MXFP6 / MXFP4 upper bounds of the quantized rows' norms.


def _a256(x):
    return (x + 255) // 256 * 256


def _carve(ws, BH, S, D):
    S16, nt = (S + 15) // 16 * 16, (S + 127) // 128
    o, parts = 0, {}
    for name, size in (("qc", BH * S * D), ("kc", BH * S * D), ("vt", BH * D * S16)):
        parts[name] = ws[o:o + size]
        o += _a256(size)
    atoms = BH * nt * 512
    parts["qsf"], parts["ksf"], parts["vsf"] = ws[o:o + atoms], ws[o + atoms:o + 2 * atoms], \
        ws[o + 2 * atoms:o + 3 * atoms]
    o += _a256(3 * atoms)
    parts["qnorm"] = ws[o:o + BH * S * 4].view(np.float32)
    o += _a256(BH * S * 4)
    parts["knorm"] = ws[o:o + BH * nt * 4].view(np.float32)
    return parts


def _luts(elem):
    n = {0: 256, 1: 64, 2: 16}[elem]
    vals = np.array([oracle.decode_elem(elem, c) for c in range(n)])
    plain = np.array([oracle.encode_elem(0, x) for x in vals], np.uint8)
    shifted = np.array([oracle.encode_elem(0, x / 64.0) for x in vals], np.uint8)
    return vals, plain, shifted


def _expected_rows(x, elem, D):
    """Attention-layout codes [BH][S][D], per-block stored exponents
    [BH][S][D/32] and exact quantized values of rows x[BH][S][D]."""
    codes, scales = oracle.mx_quantize(x, 1, elem)
    vals, plain, shifted = _luts(elem)
    X = scales.astype(np.int64) - 127
    shift = np.where((X <= 121) & (elem == 1), 6, 0)
    blk = np.repeat(shift, 32, axis=-1)[..., :D]
    cont = np.where(blk == 6, shifted[codes], plain[codes])
    qv = vals[codes] * np.exp2(np.repeat(X, 32, axis=-1)[..., :D])
    return cont, X + shift, qv


def _expected_atoms(exps, n_rows_total, nblk, BH, nt):
    """Scale atoms [BH][nt][512] from stored exponents [BH][rows][nblk]."""
    at = np.full((BH, nt, 512), 127, np.uint8)
    for r in range(n_rows_total):
        t, rr = divmod(r, 128)
        for kb in range(nblk):
            at[:, t, (rr % 32) * 16 + (rr // 32) * 4 + kb] = exps[:, r, kb] + 127
    return at


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4"])
@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (1, 1, 200, 64)])
def test_attention_layout_quantizer_matches_oracle(fsa, fmt, shape):
    B, H, S, D = shape
    BH, nt, S16 = B * H, (S + 127) // 128, (S + 15) // 16 * 16
    elem = {"mxfp8": 0, "mxfp6": 1, "mxfp4": 2}[fmt]
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=S + D)
    # a query row and a key column near the bf16 maximum (scale exponents
    # above 121, where E2M3 keeps its own exponent)
    qf, vf = fsa_inputs.bf16_bits_to_f32(q), fsa_inputs.bf16_bits_to_f32(v)
    qf[0, 0, 5, :] = np.float32(2.0 ** 126)
    vf[0, 0, 7, :] = np.float32(-2.0 ** 126)
    q, v = fsa_inputs.to_bf16_bits(qf), fsa_inputs.to_bf16_bits(vf)
    ws = fsa.new_workspace(B, H, S, D, fmt)
    fsa.attention_prepare(to_dev(q), to_dev(k), to_dev(v), ws, fmt)
    torch.cuda.synchronize()
    assert fsa.get_device_error() == 0
    got = _carve(ws.cpu().numpy(), BH, S, D)
    nblk = D // 32
    for name, x in (("q", q), ("k", k)):
        cont, exps, qv = _expected_rows(x.reshape(BH, S, D), elem, D)
        assert np.array_equal(got[name + "c"].reshape(BH, S, D), cont), name
        assert np.array_equal(got[name + "sf"].reshape(BH, nt, 512),
                              _expected_atoms(exps, S, nblk, BH, nt)), name
        if elem != 0:  # norm bounds: above the exact norm, and tight
            norms = np.sqrt((qv ** 2).sum(-1))  # [BH][S]
            if name == "q":
                bnd = got["qnorm"].reshape(BH, S).astype(np.float64)
                ref = norms
            else:
                bnd = got["knorm"].reshape(BH, nt).astype(np.float64)
                ref = np.stack([norms[:, 128 * t:128 * (t + 1)].max(1) for t in range(nt)], 1)
            # (rows whose squares overflow FP32 give an infinite bound: the
            # kernel then takes its exact test)
            tight = (bnd <= ref * (1 + 2.0 ** -9) + 1e-15) | (np.isinf(bnd) & (ref > 1e18))
            assert np.all(bnd >= ref) and np.all(tight), name
    # V: blocks along keys, transposed [BH][D][S16], padding keys zero
    vc, vs = oracle.mx_quantize(v.reshape(BH, S, D), 0, elem)   # [BH][D][S], [BH][D][ceil(S/32)]
    vals, plain, shifted = _luts(elem)
    X = vs.astype(np.int64) - 127
    shift = np.where((X <= 121) & (elem == 1), 6, 0)
    blk = np.repeat(shift, 32, axis=-1)[..., :S]
    exp_vt = np.zeros((BH, D, S16), np.uint8)
    exp_vt[..., :S] = np.where(blk == 6, shifted[vc], plain[vc])
    assert np.array_equal(got["vt"].reshape(BH, D, S16), exp_vt)
    at = np.full((BH, nt, 512), 127, np.uint8)
    exps = X + shift  # [BH][D][blocks along keys]
    for d in range(D):
        for b32 in range(exps.shape[-1]):
            t, kb = divmod(b32, 4)
            at[:, t, (d % 32) * 16 + (d // 32) * 4 + kb] = exps[:, d, b32] + 127
    assert np.array_equal(got["vsf"].reshape(BH, nt, 512), at)
