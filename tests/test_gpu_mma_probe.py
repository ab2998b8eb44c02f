"""The tensor-core rate probe (fsa_mma_rate_probe), whose measured rates are
the denominators of every roofline fraction the benchmark reports: each kind
runs to completion without a timed-out wait, reports the operation count its
declaration states (2 M N K per instruction, four instructions per group; the
attention tile's 4 * 128^3 per group), and its rates order as the hardware's
do -- packed FP4 above the eight- and six-bit formats, those above BF16 --
and stay below twice the nominal dense peaks of a GB300."""
import pytest
import torch

pytestmark = pytest.mark.gpu

# M, N, K of one instruction; four instructions per group
SHAPES = {"mxf8f6f4_e4m3": (128, 256, 32), "mxf8f6f4_e2m3": (128, 256, 32), "mxf4_e2m1": (128, 256, 64),
          "f16_bf16": (128, 256, 16)}
NOMINAL_TFLOPS = {"mxf8f6f4_e4m3": 4500.0, "mxf8f6f4_e2m3": 4500.0, "mxf4_e2m1": 13500.0,
                  "attention_tile_e4m3": 4500.0, "f16_bf16": 2250.0}


@pytest.fixture(scope="module")
def fsa():
    import __graft_entry__
    __graft_entry__.build()
    import matrix_core_softmax_gb300 as m
    return m


def _rate(fsa, kind, ctas, iters):
    stream = torch.cuda.current_stream()
    fsa.mma_rate_probe(kind, ctas, iters, stream)           # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    flops = fsa.mma_rate_probe(kind, ctas, iters, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    st = fsa.get_device_error()
    assert st == 0, fsa.status_string(st)
    return flops, flops / (e0.elapsed_time(e1) / 1e3) / 1e12


def test_probe_counts_and_rates(fsa):
    assert set(fsa.PROBE_KINDS) == set(NOMINAL_TFLOPS)
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    iters = 2048
    rates = {}
    for kind in fsa.PROBE_KINDS:
        flops, rate = _rate(fsa, kind, ctas, iters)
        if kind == "attention_tile_e4m3":
            want = 4.0 * 128 ** 3
        else:
            m, n, k = SHAPES[kind]
            want = 4 * 2.0 * m * n * k
        assert flops == want * iters * ctas, kind
        assert 0.0 < rate < 2.0 * NOMINAL_TFLOPS[kind], (kind, rate)
        rates[kind] = rate
    assert rates["mxf4_e2m1"] > rates["mxf8f6f4_e4m3"] > rates["f16_bf16"], rates
    assert rates["mxf8f6f4_e2m3"] > rates["f16_bf16"], rates
    assert rates["attention_tile_e4m3"] <= rates["mxf8f6f4_e4m3"] * 1.05, rates
