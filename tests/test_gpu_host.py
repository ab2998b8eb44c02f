"""GPU tests of the host-buffer entry points (fsa_attention_fwd_host,
fsa_cross_attention_fwd_host, through the C ABI): the heads are streamed
through the device in chunks with copies overlapping the computation, which
must change nothing -- every head is computed independently, so the output
equals the device-buffer call bit for bit, and matches the oracle."""
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


def _host(bits, pinned):
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t.clone()


# (B, H, Sq, Sk, D): one chunk; two chunks (10 + 6 heads); three chunks with
# a partial last one (19 + 19 + 2 heads); cross-attention; D = 64
SHAPES = [(1, 2, 300, 300, 128), (1, 16, 4096, 4096, 128), (1, 40, 2048, 2048, 128),
          (2, 8, 3000, 700, 128), (1, 24, 2500, 2500, 64)]


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp6", "mxfp4", "mxfp4_efq"])
@pytest.mark.parametrize("shape", SHAPES)
def test_host_call_equals_device_call(fsa, fmt, shape):
    B, H, Sq, Sk, D = shape
    q, _, _ = fsa_inputs.qkv(B, H, Sq, D, seed=Sq + H)
    _, k, v = fsa_inputs.qkv(B, H, Sk, D, seed=Sk + H + 1)
    hq, hk, hv = (_host(x, pinned=True) for x in (q, k, v))
    o_host = fsa.cross_attention_fwd_host(hq, hk, hv, fmt=fmt)
    torch.cuda.synchronize()
    o_dev = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt)
    assert fsa.get_device_error() == 0
    assert torch.equal(o_host, o_dev.cpu())


@pytest.mark.parametrize("pinned", [True, False])
def test_host_call_matches_oracle(fsa, pinned):
    B, H, S, D = 1, 16, 4096, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=5)
    hq, hk, hv = (_host(x, pinned) for x in (q, k, v))
    o = fsa.attention_fwd_host(hq, hk, hv, fmt="mxfp4")
    torch.cuda.synchronize()
    assert fsa.get_device_error() == 0
    got = o.float().numpy().astype(np.float64).reshape(-1, D)
    rows = np.arange(0, B * H * S, 97)
    ref = oracle.attention(q, k, v, fmt="mxfp4", mode="fused", rows=rows)["out"]
    parity.check_out(f"host call pinned={pinned} mxfp4", got[rows], ref)


def test_host_call_rollback_bits_follow_the_chunks(fsa):
    # rollback bits and count of a multi-chunk call equal the device call's
    B, H, S, D = 1, 16, 4096, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=9, stress_from=2048)
    n_t = (S + 127) // 128
    bits_h = torch.full((B * H * S, n_t), 7, dtype=torch.uint8, device="cuda")
    bits_d = torch.full((B * H * S, n_t), 7, dtype=torch.uint8, device="cuda")
    cnt_h = torch.zeros(1, dtype=torch.int64, device="cuda")
    cnt_d = torch.zeros(1, dtype=torch.int64, device="cuda")
    hq, hk, hv = (_host(x, True) for x in (q, k, v))
    fsa.attention_fwd_host(hq, hk, hv, fmt="mxfp8", rollback_bits=bits_h, rollback_count=cnt_h)
    fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp8", rollback_bits=bits_d,
                      rollback_count=cnt_d)
    assert fsa.get_device_error() == 0
    assert int(cnt_d.item()) > 0
    assert torch.equal(bits_h, bits_d) and int(cnt_h.item()) == int(cnt_d.item())


def test_host_calls_on_two_streams_and_growing_buffers(fsa):
    # a small call, then a larger one on another stream (the chunk buffers
    # grow), then the small one again: every result equals the device call
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    shapes = [(1, 4, 1000, 128), (1, 20, 3000, 128), (1, 4, 1000, 128)]
    outs, refs = [], []
    for i, (B, H, S, D) in enumerate(shapes):
        q, k, v = fsa_inputs.qkv(B, H, S, D, seed=30 + i)
        hq, hk, hv = (_host(x, True) for x in (q, k, v))
        st = s1 if i % 2 == 0 else s2
        outs.append(fsa.attention_fwd_host(hq, hk, hv, fmt="mxfp6", stream=st))
        refs.append(fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt="mxfp6"))
    torch.cuda.synchronize()
    assert fsa.get_device_error() == 0
    for o, r in zip(outs, refs):
        assert torch.equal(o, r.cpu())


def test_host_call_rejects_device_tensors(fsa):
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fsa.attention_fwd_host(q, q, q)


def test_host_calls_with_inputs_ready_overlap_and_stay_exact(fsa):
    # consecutive calls whose copy-in may start before the previous call
    # finished (host inputs declared final): every output equals the
    # device call's, the output buffers reused call after call
    B, H, S, D = 1, 16, 4096, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=40)
    hq, hk, hv = (_host(x, True) for x in (q, k, v))
    outs = [torch.empty(B, H, S, D, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    for i, fmt in enumerate(("mxfp8", "mxfp6", "mxfp4", "mxfp8")):
        fsa.attention_fwd_host(hq, hk, hv, fmt=fmt, out=outs[i % 2], host_inputs_ready=True)
        if i % 2 == 1:
            torch.cuda.synchronize()
            for j, f in ((i - 1, ("mxfp8", "mxfp6", "mxfp4", "mxfp8")[i - 1]), (i, fmt)):
                ref = fsa.attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=f)
                assert torch.equal(outs[j % 2], ref.cpu()), (j, f)
    assert fsa.get_device_error() == 0


def test_overlapping_host_calls_with_different_layouts_stay_exact(fsa):
    # consecutive calls with the host inputs declared final, alternating
    # between shapes whose chunk buffer sets are carved at different offsets
    # (different Sq, Sk and heads per chunk) and between two streams: a
    # call with a new layout must not overwrite buffers the previous call's
    # kernels or copies still use, so every output equals the device call's
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    shapes = [(1, 16, 4096, 1000, 128), (1, 20, 2000, 3000, 128), (1, 16, 4096, 1000, 128),
              (1, 12, 3000, 3000, 64)]
    cases = []
    for i, (B, H, Sq, Sk, D) in enumerate(shapes):
        q, _, _ = fsa_inputs.qkv(B, H, Sq, D, seed=50 + i)
        _, k, v = fsa_inputs.qkv(B, H, Sk, D, seed=60 + i)
        cases.append((q, k, v, tuple(_host(x, True) for x in (q, k, v))))
    # the largest layout first, so the buffers are not reallocated (and the
    # device not synchronised) between the overlapping calls below
    B, H, Sq, Sk, D = shapes[1]
    fsa.cross_attention_fwd_host(*cases[1][3], fmt="mxfp8", host_inputs_ready=True)
    torch.cuda.synchronize()
    fmts = ("mxfp8", "mxfp4", "mxfp6", "mxfp8")
    outs = []
    for i, (q, k, v, h) in enumerate(cases):
        st = s1 if i % 2 == 0 else s2
        outs.append(fsa.cross_attention_fwd_host(*h, fmt=fmts[i], host_inputs_ready=True, stream=st))
    torch.cuda.synchronize()
    assert fsa.get_device_error() == 0
    for (q, k, v, _), fmt, o in zip(cases, fmts, outs):
        ref = fsa.cross_attention_fwd(to_dev(q), to_dev(k), to_dev(v), fmt=fmt)
        assert torch.equal(o, ref.cpu()), fmt
    assert fsa.get_device_error() == 0
