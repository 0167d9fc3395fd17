"""The forward's segment plan (slim_attn_segments) against a restatement of
its makespan model here, on the GPU's own SM count: for each candidate count
of segments, waves x (tiles per segment + 2) for the forward plus 0.4 x waves
x (tiles per segment + 2) for the state pass over all but the last segment;
the plan is the first candidate of least cost (waves capped at 8)."""
import pytest
import torch

from sub_linear_memory_gb300 import inputs

pytestmark = pytest.mark.gpu


def model_segments(bh, tiles, sms):
    cap = max(1, 8 * ((sms + bh - 1) // bh))
    best, pick = None, 1
    for cand in range(1, min(tiles, cap) + 1):
        cps = -(-tiles // cand)
        segs = -(-tiles // cps)
        waves = -(-(segs * bh) // sms)
        waves_s = -(-((segs - 1) * bh) // sms)
        span = waves * (cps + 2.0) + 0.4 * waves_s * (cps + 2.0)
        if best is None or span < best - 1e-9:
            best, pick = span, segs
    cps = -(-tiles // pick)
    return -(-tiles // cps)


@pytest.mark.parametrize("name", ["l4k", "l32k", "l1m", "elu16k"])
@pytest.mark.parametrize("heads", [None, (1, 8), (2, 8)])
def test_forward_plan_follows_the_model(name, heads):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sub_linear_memory_gb300 import binding

    binding.set_option(binding.OPT_SEGMENTS, 0)
    wl = inputs.WORKLOADS[name]
    b, h = heads or (wl.B, wl.H)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    got = binding.segments(b, h, wl.L, wl.d, wl.M, wl.chunk)
    want = model_segments(b * h, -(-wl.L // 128), sms)
    print(name, (b, h), "segments", got, "model", want, "SMs", sms)
    assert got == want
