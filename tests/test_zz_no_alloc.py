"""slim_attn_fwd_noalloc: the forward for callers that cannot allocate.

Some callers of this library cannot allocate device memory (a memory-capped
pool, an allocation-free real-time loop, code that must not risk the device
synchronisation an allocation can cause).  For them the library has one
forward entry point whose scratch is a fixed array compiled into the
library instead of a caller-registered workspace.  These tests call it
directly through the C ABI and check:
  * its output against the fp64 oracle and against slim_attn_fwd, on FAVOR+
    and elu+1 problems, several calls in a row on different problems (the
    shared array must not carry anything over);
  * that a call allocates nothing: after a warm-up call, neither torch's
    allocator nor the device's free-memory count moves across a call;
  * that a problem too large for the array is refused before any launch.
The file name makes pytest collect it last, so that a run stopped at its
first failure (pytest -x) has already run every other test when one of
these fails.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from sub_linear_memory_gb300 import inputs

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 64 << 20  # SLIM_NOALLOC_SCRATCH_BYTES
BF16_TOL = 2e-2


def _lib():
    from sub_linear_memory_gb300 import binding

    return binding, binding.raw().slim_attn_fwd_noalloc


def _problem(B, H, L, d, M, C, seed, feature="favor"):
    base = inputs.WORKLOADS["l4k"] if feature == "favor" else inputs.WORKLOADS["elu16k"]
    wl = base.with_(B=B, H=H, L=L, d=d, M=M, chunk=C, index=200 + seed)
    q, k, v, _, w = inputs.make_inputs(wl, want_dy=False)
    return q.cuda(), k.cuda(), v.cuda(), (None if w is None else w.cuda()), C


def _noalloc_forward(fn, q, k, v, w, chunk, y=None):
    b, h, length, d = q.shape
    m = d if w is None else w.shape[1]
    if y is None:
        y = torch.full_like(q, float("nan"))
    stream = torch.cuda.current_stream().cuda_stream
    rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), None if w is None else w.data_ptr(), y.data_ptr(),
            b, h, length, d, m, chunk, stream)
    assert rc == 0, rc
    return y


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _rel_l2(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm((a - b).ravel()) / np.linalg.norm(b.ravel()))


PROBLEMS = [
    # (B, H, L, d, M, C, seed, feature)
    (2, 4, 2048, 64, 128, 64, 0, "favor"),
    (1, 3, 777, 32, 64, 32, 1, "favor"),
    (1, 2, 600, 64, 64, 64, 2, "elu"),
]


def test_noalloc_forward_matches_oracle_and_slim_attn_fwd():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding, fn = _lib()
    for B, H, L, d, M, C, seed, feature in PROBLEMS:
        q, k, v, w, chunk = _problem(B, H, L, d, M, C, seed, feature)
        assert binding.noalloc_bytes(B, H, L, d, M, chunk) <= NOALLOC_BYTES
        y = _noalloc_forward(fn, q, k, v, w, chunk)
        y_ref = binding.slim_attn_fwd(q, k, v, w, chunk)
        binding.sync_status()
        assert torch.isfinite(y.float()).all()
        exact = oracle.recurrence_forward(_np(q), _np(k), _np(v), None if w is None else _np(w))
        assert oracle.rel_l2(_np(y), exact) <= BF16_TOL, (feature, d, M)
        assert _rel_l2(y, y_ref) <= BF16_TOL


def test_noalloc_forward_allocates_nothing():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding, fn = _lib()
    q, k, v, w, chunk = _problem(1, 3, 777, 32, 64, 32, 3)
    y = torch.empty_like(q)
    _noalloc_forward(fn, q, k, v, w, chunk, y)  # warm-up: loads the device code if needed
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc_forward(fn, q, k, v, w, chunk, y)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_after == free_before
    binding.sync_status()


def test_noalloc_refuses_problems_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding, fn = _lib()
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64, 256, dtype=torch.float32, device="cuda")
    assert binding.noalloc_bytes(2, 16, 32768, 64, 256, 128) > NOALLOC_BYTES
    rc = fn(t.data_ptr(), t.data_ptr(), t.data_ptr(), w.data_ptr(), t.data_ptr(),
            2, 16, 32768, 64, 256, 128, torch.cuda.current_stream().cuda_stream)
    assert rc == 3  # SLIM_ERR_WORKSPACE, returned before any launch
