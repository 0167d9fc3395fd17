"""GPU parity of the serving form (prefill state, one-row decode) against the
fp64 oracle's ``prefill_state`` / ``decode_step`` ("Sub-Linear Memory: How to
Make Performers SLiM", section 2.1, eq. (3)-(4) one row at a time).

Bars as for the forward (relative L2 in fp64): fp32 I/O 1e-4, bf16 I/O 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from sub_linear_memory_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sub_linear_memory_gb300 import binding

    binding.set_option(binding.OPT_SEGMENTS, 0)
    binding.set_option(binding.OPT_PATH, 0)
    yield binding
    binding.set_option(binding.OPT_SEGMENTS, 0)
    binding.set_option(binding.OPT_PATH, 0)


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _wnp(w):
    return None if w is None else _np(w)


def rel(got, ref):
    den = float(np.linalg.norm(np.ravel(ref)))
    return float(np.linalg.norm(np.ravel(np.asarray(got, np.float64) - ref))) / max(den, 1e-30)


def case(B, H, L, d, M, C, dtype, feature, seed):
    base = inputs.WORKLOADS["tiny" if dtype == torch.float32 else "l4k"]
    wl = base.with_(B=B, H=H, L=L, d=d, M=M, chunk=C, index=300 + seed,
                    dtype="fp32" if dtype == torch.float32 else "bf16", feature=feature,
                    qk_scale=(1.0 if feature == "elu" else d ** -0.25),
                    w_kind=("none" if feature == "elu" else base.w_kind))
    q, k, v, dy, w = inputs.make_inputs(wl)
    return q.cuda(), k.cuda(), v.cuda(), None if w is None else w.cuda()


def profiled(_lib, fn):
    _lib.profile_reset()
    _lib.profile_enable(True)
    try:
        out = fn()
        _lib.sync_status()
        names = set(_lib.profile_read())
    finally:
        _lib.profile_enable(False)
    return out, names


STATE_CASES = [
    # (B, H, L, d, M, C, dtype, feature, expected state kernel)
    (2, 3, 1000, 64, 256, 128, torch.bfloat16, "favor", "tc_segment_state"),
    (1, 2, 700, 64, 128, 64, torch.bfloat16, "favor", "tc_segment_state"),
    (2, 1, 129, 64, 64, 128, torch.bfloat16, "favor", "tc_segment_state"),
    (1, 2, 333, 64, 64, 128, torch.bfloat16, "elu", "tc_segment_state"),
    (1, 1, 300, 128, 128, 64, torch.bfloat16, "elu", "tc_segment_state"),
    (1, 2, 257, 16, 32, 32, torch.float32, "favor", "gen_segment_state"),
    (2, 1, 100, 32, 48, 16, torch.float32, "favor", "gen_segment_state"),
    (1, 2, 90, 32, 32, 16, torch.float32, "elu", "gen_segment_state"),
    (1, 1, 77, 16, 32, 32, torch.bfloat16, "favor", "gen_segment_state"),
]


@pytest.mark.parametrize("c", STATE_CASES, ids=lambda c: "x".join(map(str, c[:6])) + "-" + c[7] + "-" + str(c[6])[6:])
def test_prefill_state_matches_oracle(c, _lib):
    B, H, L, d, M, C, dtype, feature, kernel = c
    q, k, v, w = case(B, H, L, d, M, C, dtype, feature, seed=1)
    st, names = profiled(_lib, lambda: _lib.slim_attn_state(k, v, w, C))
    assert kernel in names, names
    ref = oracle.prefill_state(_np(k), _np(v), _wnp(w))
    err = rel(_np(st), ref)
    print("state rel L2 %.3e" % err)
    assert err <= TOL[dtype]


def test_prefill_state_of_no_rows_is_zero(_lib):
    q, k, v, w = case(1, 2, 64, 64, 128, 64, torch.bfloat16, "favor", seed=2)
    st = torch.full((1, 2, 65, 128), 7.0, device="cuda")
    _lib.slim_attn_state(k[:, :, :0].contiguous(), v[:, :, :0].contiguous(), w, 64, state=st)
    _lib.sync_status()
    assert bool((st == 0).all())


DECODE_CASES = [
    # (B, H, d, M, dtype, feature)
    (4, 8, 64, 256, torch.bfloat16, "favor"),
    (3, 5, 64, 128, torch.float32, "favor"),
    (2, 3, 16, 32, torch.float32, "favor"),
    (2, 2, 32, 48, torch.float32, "favor"),   # M not a multiple of 32
    (1, 3, 128, 128, torch.bfloat16, "elu"),
    (2, 2, 64, 64, torch.float32, "elu"),
]


@pytest.mark.parametrize("c", DECODE_CASES, ids=lambda c: "x".join(map(str, c[:4])) + "-" + c[5] + "-" + str(c[4])[6:])
def test_decode_step_matches_oracle(c, _lib):
    """One decode step from a state built over 40 earlier rows."""
    B, H, d, M, dtype, feature = c
    q, k, v, w = case(B, H, 41, d, M, 16, dtype, feature, seed=3)
    ref_state = oracle.prefill_state(_np(k[:, :, :40]), _np(v[:, :, :40]), _wnp(w))
    state = torch.tensor(ref_state, dtype=torch.float32, device="cuda")
    ref_state = state.double().cpu().numpy()  # the fp32 state the library starts from
    ql, kl, vl = (x[:, :, 40].contiguous() for x in (q, k, v))
    y, names = profiled(_lib, lambda: _lib.slim_attn_decode(ql, kl, vl, w, state))
    assert "decode" in names, names
    y_ref = oracle.decode_step(_np(ql), _np(kl), _np(vl), _wnp(w), ref_state)
    e_y, e_s = rel(_np(y), y_ref), rel(_np(state), ref_state)
    print("decode y rel L2 %.3e, state %.3e" % (e_y, e_s))
    assert e_y <= TOL[dtype] and e_s <= TOL[torch.float32]


@pytest.mark.parametrize("feature,dtype,M", [("favor", torch.bfloat16, 256), ("favor", torch.float32, 64),
                                             ("elu", torch.bfloat16, 64)])
def test_prefill_then_decode_continues_the_forward(feature, dtype, M, _lib):
    """State over rows < l, then decode rows l .. l + 9: each output row is row
    l + i of the forward over the whole sequence (library and oracle)."""
    B, H, L, d = 1, 4, 300, 64
    q, k, v, w = case(B, H, L, d, M, 64, dtype, feature, seed=4)
    y_fwd = _np(_lib.slim_attn_fwd(q, k, v, w, 64))
    y_ref = oracle.recurrence_forward(_np(q), _np(k), _np(v), _wnp(w))
    for l in (0, 128, 287):
        state = _lib.slim_attn_state(k[:, :, :l].contiguous(), v[:, :, :l].contiguous(), w, 64)
        rows = []
        for i in range(l, min(l + 10, L)):
            rows.append(_np(_lib.slim_attn_decode(q[:, :, i].contiguous(), k[:, :, i].contiguous(),
                                                  v[:, :, i].contiguous(), w, state)))
        _lib.sync_status()
        got = np.stack(rows, axis=2)
        n = got.shape[2]
        assert rel(got, y_ref[:, :, l:l + n]) <= TOL[dtype]
        assert rel(got, y_fwd[:, :, l:l + n]) <= TOL[dtype]
