"""The exponential-unit probe the benchmark times (slim_attn_probe_ex2): it
runs, leaves every chain's value where x <- 2^(-x/2) keeps it (in (0, 1],
eight chains summed), and takes longer for more work."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_probe_ex2_runs_and_scales():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sub_linear_memory_gb300 import binding

    blocks = 4
    sink = torch.full((blocks * 256,), -1.0, dtype=torch.float32, device="cuda")
    binding.probe_ex2(blocks, 64, sink)
    binding.sync_status()
    assert torch.isfinite(sink).all()
    # the fixed point of x = 2^(-x/2) is about 0.7667; eight chains sum to about 6.13
    assert torch.allclose(sink, torch.full_like(sink, 8 * 0.7667), atol=0.05)
    times = []
    for iters in (1024, 8192):
        binding.probe_ex2(blocks, iters, sink)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        binding.probe_ex2(blocks, iters, sink)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert times[1] > 2 * times[0]
