"""The denoising-step precision schedules (host logic) and, on the GPU, that
every step of a schedule is exactly the library call of its format."""
import os

import numpy as np
import pytest

from matrix_core_softmax_gb300 import schedule as sch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hybrid_schedule.txt")


def _golden():
    steps, fmts = None, {}
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if not line:
            continue
        if line[0] == "steps":
            steps = int(line[1])
        else:
            fmts[int(line[0])] = line[1]
    return steps, [fmts[i] for i in range(steps)]


def test_hybrid_schedule_is_the_pages_schedule():
    steps, want = _golden()
    assert sch.DENOISING_STEPS == steps
    assert sch.hybrid_schedule() == want
    assert want.count("mxfp6") == 6 and want.count("mxfp4") == 14


def test_schedule_edge_cases():
    assert sch.hybrid_schedule(0) == []
    assert sch.hybrid_schedule(4, 3) == ["mxfp6"] * 4          # edges overlap
    assert sch.hybrid_schedule(7, 0) == ["mxfp4"] * 7
    assert sch.hybrid_schedule(5, 1, "mxfp8", "bf16") == ["mxfp8", "bf16", "bf16", "bf16", "mxfp8"]
    assert sch.uniform_schedule("bf16", 3) == ["bf16"] * 3
    for bad in (lambda: sch.hybrid_schedule(-1), lambda: sch.hybrid_schedule(5, -2),
                lambda: sch.uniform_schedule("fp16"), lambda: sch.hybrid_schedule(5, 1, "e4m3")):
        with pytest.raises(ValueError):
            bad()


@pytest.mark.gpu
def test_schedule_steps_equal_direct_calls():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import fsa_inputs
    import matrix_core_softmax_gb300 as fsa
    from gpu_util import to_dev
    B, H, S, D = 1, 2, 700, 128
    q, k, v = (to_dev(x) for x in fsa_inputs.qkv(B, H, S, D, seed=5))
    plan = sch.hybrid_schedule(8, 2) + ["mxfp8", "bf16"]
    ws = fsa.new_workspace(B, H, S, D)
    for fmt in plan:
        got = sch.attention_step(q, k, v, fmt, 8.0, workspace=ws)
        want = (fsa.bf16_attention_fwd(q, k, v) if fmt == "bf16"
                else fsa.attention_fwd(q, k, v, fmt=fmt, threshold=8.0))
        assert fsa.get_device_error() == 0
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), fmt
