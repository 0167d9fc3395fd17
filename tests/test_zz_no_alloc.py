"""slim_attn_fwd_noalloc: the forward for callers that cannot allocate.

Some callers of this library cannot allocate device memory (a memory-capped
pool, an allocation-free real-time loop, code that must not risk the device
synchronisation an allocation can cause).  For them the library has one
forward entry point whose scratch is a fixed array compiled into the
library instead of a caller-registered workspace.  This test calls it
directly through the C ABI and checks it against slim_attn_fwd, twice in a
row on different problems (the shared array must not carry anything over),
and checks that a problem too large for the array is refused.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from sub_linear_memory_gb300 import inputs

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 64 << 20  # SLIM_NOALLOC_SCRATCH_BYTES
BF16_TOL = 2e-2


def _lib():
    from sub_linear_memory_gb300 import binding

    lib = binding.raw()
    fn = lib.slim_attn_fwd_noalloc
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return binding, fn


def _problem(B, H, L, d, M, C, seed):
    wl = inputs.WORKLOADS["l4k"].with_(B=B, H=H, L=L, d=d, M=M, chunk=C, index=200 + seed)
    q, k, v, _, w = inputs.make_inputs(wl, want_dy=False)
    return q.cuda(), k.cuda(), v.cuda(), w.cuda(), C


def _noalloc_forward(fn, q, k, v, w, chunk):
    b, h, length, d = q.shape
    y = torch.full_like(q, float("nan"))
    stream = torch.cuda.current_stream().cuda_stream
    rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), w.data_ptr(), y.data_ptr(),
            b, h, length, d, w.shape[1], chunk, stream)
    assert rc == 0, rc
    return y


def _rel_l2(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm((a - b).ravel()) / np.linalg.norm(b.ravel()))


def test_noalloc_forward_matches_slim_attn_fwd_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding, fn = _lib()
    for problem in (_problem(2, 4, 2048, 64, 128, 64, 0), _problem(1, 3, 777, 32, 64, 32, 1)):
        q, k, v, w, chunk = problem
        b, h, length, d = q.shape
        assert binding.workspace_bytes(b, h, length, d, w.shape[1], chunk, 0) <= NOALLOC_BYTES
        y = _noalloc_forward(fn, q, k, v, w, chunk)
        y_ref = binding.slim_attn_fwd(q, k, v, w, chunk)
        binding.sync_status()
        assert torch.isfinite(y.float()).all()
        assert _rel_l2(y, y_ref) <= BF16_TOL


def test_noalloc_refuses_problems_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding, fn = _lib()
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64, 256, dtype=torch.float32, device="cuda")
    assert binding.workspace_bytes(2, 16, 32768, 64, 256, 128, 0) > NOALLOC_BYTES
    rc = fn(t.data_ptr(), t.data_ptr(), t.data_ptr(), w.data_ptr(), t.data_ptr(),
            2, 16, 32768, 64, 256, 128, torch.cuda.current_stream().cuda_stream)
    assert rc == 3  # SLIM_ERR_WORKSPACE, returned before any launch
