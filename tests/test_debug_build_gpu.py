"""The -DSLIM_DEBUG build on the GPU: the same small cases through every
kernel family, loaded in a child process (SLIM_ATTN_LIBRARY=debug) so this
process keeps the release library.  Every call of the debug build waits for
its work and returns the device status, so a failed bounds check
(SLIM_ERR_BOUNDS) or a timed-out wait would fail the call that caused it;
the results must also match the fp64 oracle."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import numpy as np, torch
import oracle
from sub_linear_memory_gb300 import binding, inputs
assert binding.library_path.endswith("libslim_attn_debug.so"), binding.library_path
f = lambda t: t.detach().to("cpu", torch.float64).numpy()
cases = [("l32k", dict(B=1, H=2, L=700), 2e-2), ("l4k", dict(B=2, H=1, L=1000, M=64), 2e-2),
         ("tiny", dict(B=1, H=2, L=250), 1e-4), ("elu16k", dict(B=1, H=2, L=300), 2e-2)]
for name, kw, tol in cases:
    wl = inputs.WORKLOADS[name].with_(index=77, **kw)
    for segments in (0, 3):
        binding.set_option(binding.OPT_SEGMENTS, segments)
        q, k, v, dy, w = (None if t is None else t.cuda() for t in inputs.make_inputs(wl))
        y = binding.slim_attn_fwd(q, k, v, w, wl.chunk)
        dq, dk, dv, _ = binding.slim_attn_bwd(q, k, v, w, dy, wl.chunk)
        binding.sync_status()
        wn = None if w is None else f(w)
        ry = oracle.recurrence_forward(f(q), f(k), f(v), wn)
        ref = oracle.recurrence_backward(f(q), f(k), f(v), wn, f(dy), want_dw=False)
        for got, exp in ((y, ry), (dq, ref[0]), (dk, ref[1]), (dv, ref[2])):
            err = oracle.rel_l2(f(got), exp)
            assert err <= tol, (name, segments, err)
binding.set_option(binding.OPT_SEGMENTS, 0)
print("debug build ok")
'''


def test_debug_build_runs_clean_and_matches_oracle():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sub_linear_memory_gb300 import build

    build.build(debug=True)
    env = dict(os.environ, SLIM_ATTN_LIBRARY="debug", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    print(r.stdout[-2000:], r.stderr[-4000:])
    assert r.returncode == 0, r.stderr[-4000:]
    assert "debug build ok" in r.stdout
