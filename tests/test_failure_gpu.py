"""The failure path of the bounded on-chip waits, on the GPU, without a fault.

Every tensor-core kernel waits on mbarriers with a time limit; a wait that
runs out records SLIM_ERR_TIMEOUT in the device status word and the kernel
winds down instead of hanging.  Production kernels are never made to time out
here (they would have copies and tensor-core work in flight); the library's
self-test kernel runs the same bounded wait on a barrier nothing ever arms,
with nothing else in flight, and this test checks what the host sees: the
timeout is reported once, the status is cleared by reading it, and the next
attention call on the same context is correct.
"""
import numpy as np
import pytest
import torch

import oracle
from sub_linear_memory_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sub_linear_memory_gb300 import binding as b

    b.sync_status()  # start from a clean status word
    return b


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("limit_ns", [1_000_000, 20_000_000])
def test_bounded_wait_gives_up_and_reports_timeout(binding, limit_ns):
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    binding.selftest_timeout(limit_ns, waited)
    with pytest.raises(binding.SlimError) as err:
        binding.sync_status()
    assert err.value.code == 5  # SLIM_ERR_TIMEOUT
    binding.sync_status()  # reading the status cleared it
    ns = int(waited.item())
    assert ns != 1, "the wait saw a barrier phase complete that nothing armed"
    assert limit_ns <= ns < limit_ns + 50_000_000, ns


def test_context_is_usable_after_a_timeout(binding):
    binding.selftest_timeout(1_000_000)
    with pytest.raises(binding.SlimError):
        binding.sync_status()
    wl = inputs.WORKLOADS["l32k"].with_(B=1, H=2, L=700, index=500)
    q, k, v, dy, w = (t.cuda() for t in inputs.make_inputs(wl))
    y = binding.slim_attn_fwd(q, k, v, w, wl.chunk)
    dq, dk, dv, _ = binding.slim_attn_bwd(q, k, v, w, dy, wl.chunk)
    binding.sync_status()
    qn, kn, vn, dyn, wn = _np(q), _np(k), _np(v), _np(dy), _np(w)
    ref_y = oracle.recurrence_forward(qn, kn, vn, wn)
    ref = oracle.recurrence_backward(qn, kn, vn, wn, dyn, want_dw=False)
    for got, exp in ((y, ref_y), (dq, ref[0]), (dk, ref[1]), (dv, ref[2])):
        assert oracle.rel_l2(_np(got), exp) <= 2e-2


def test_bad_limits_are_refused_before_any_launch(binding):
    for bad in (0, 999, 100_000_001):
        with pytest.raises(binding.SlimError) as err:
            binding.selftest_timeout(bad)
        assert err.value.code == 1
    binding.sync_status()
