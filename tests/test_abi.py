"""CPU-only checks of the C ABI: the library loads, exports every function the
header declares, and rejects bad arguments on the host (no GPU work)."""
import ctypes
import os
import re

import pytest

from sub_linear_memory_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "slim_attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    from sub_linear_memory_gb300 import binding

    return binding.raw()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(slim_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("slim_attn_fwd", "slim_attn_bwd", "slim_attn_fwd_f32", "slim_attn_bwd_f32",
              "slim_attn_workspace_bytes", "slim_attn_set_workspace", "slim_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(6):
        assert lib.slim_status_string(code).startswith(b"SLIM_")
    assert b"unknown" in lib.slim_status_string(99)


def test_bad_shapes_are_rejected_before_any_launch(lib):
    vp = ctypes.c_void_p
    dummy = vp(256)
    # d not supported
    assert lib.slim_attn_fwd(dummy, dummy, dummy, dummy, dummy, 1, 1, 64, 48, 64, 32, None) == 2
    # M not a multiple of 16
    assert lib.slim_attn_fwd(dummy, dummy, dummy, dummy, dummy, 1, 1, 64, 64, 40, 32, None) == 2
    # chunk not a power of two / out of range
    assert lib.slim_attn_fwd(dummy, dummy, dummy, dummy, dummy, 1, 1, 64, 64, 64, 48, None) == 2
    assert lib.slim_attn_fwd(dummy, dummy, dummy, dummy, dummy, 1, 1, 64, 64, 64, 512, None) == 2
    # elu+1 (w NULL) needs M == d
    assert lib.slim_attn_fwd(dummy, dummy, dummy, None, dummy, 1, 1, 64, 64, 128, 32, None) == 1
    # negative sizes
    assert lib.slim_attn_fwd(dummy, dummy, dummy, dummy, dummy, -1, 1, 64, 64, 64, 32, None) == 1
    # dw requested with elu+1
    assert lib.slim_attn_bwd(dummy, dummy, dummy, None, dummy, dummy, dummy, dummy, dummy,
                             1, 1, 64, 64, 64, 32, None) == 1
    # NULL tensors with work to do
    assert lib.slim_attn_fwd(None, dummy, dummy, dummy, dummy, 1, 1, 64, 64, 64, 32, None) == 1
    assert lib.slim_attn_bwd(dummy, dummy, dummy, dummy, None, dummy, dummy, dummy, None,
                             1, 1, 64, 64, 64, 32, None) == 1


def test_empty_problem_is_a_no_op(lib):
    vp = ctypes.c_void_p
    assert lib.slim_attn_fwd(None, None, None, vp(256), None, 0, 4, 128, 64, 64, 32, None) == 0
    assert lib.slim_attn_fwd(None, None, None, vp(256), None, 2, 4, 0, 64, 64, 32, None) == 0


def test_workspace_registration_rules(lib):
    assert lib.slim_attn_set_workspace(ctypes.c_void_p(4096), 0) == 1
    assert lib.slim_attn_set_workspace(ctypes.c_void_p(4100), 1024) == 1  # not 256-B aligned
    assert lib.slim_attn_set_workspace(None, 0) == 0
    assert lib.slim_attn_set_option(99, 0) == 1
    assert lib.slim_attn_set_option(1, -1) == 1


def test_probe_ex2_rejects_bad_arguments_before_any_launch(lib):
    vp = ctypes.c_void_p
    assert lib.slim_attn_probe_ex2(0, 1, vp(256), None) == 1
    assert lib.slim_attn_probe_ex2(1, 0, vp(256), None) == 1
    assert lib.slim_attn_probe_ex2(1, 1 << 21, vp(256), None) == 1
    assert lib.slim_attn_probe_ex2(1, 1, None, None) == 1


def test_reuse_states_option(lib):
    """SLIM_OPT_REUSE_STATES takes 0 or 1; it leaves the forward's plan alone
    (the backward may take the forward's segments), no GPU needed."""
    assert lib.slim_attn_set_option(5, 2) == 1
    assert lib.slim_attn_set_option(5, -1) == 1
    shape = (2, 16, 32768, 64, 256, 128)
    off = [lib.slim_attn_workspace_bytes(*shape, b) for b in (0, 1)]
    assert lib.slim_attn_set_option(5, 1) == 0
    try:
        on = [lib.slim_attn_workspace_bytes(*shape, b) for b in (0, 1)]
    finally:
        assert lib.slim_attn_set_option(5, 0) == 0
    assert on[0] == off[0] and min(off + on) > 0


def test_workspace_does_not_grow_with_sequence_length(lib):
    """Sub-linear memory: past the point where every SM has a segment, the
    workspace is independent of L (only boundary states and chunk scratch)."""
    sizes = [lib.slim_attn_workspace_bytes(1, 8, 1 << e, 64, 64, 256, 1) for e in (16, 18, 20)]
    assert sizes[0] > 0 and sizes[0] == sizes[1] == sizes[2]
    # an L x d x M prefix-sum tensor at L = 2^20 would be 8 GiB per head-group
    assert sizes[2] < (1 << 30)


def test_state_and_decode_reject_bad_arguments_before_any_launch(lib):
    vp = ctypes.c_void_p
    dummy = vp(256)
    # decode: d, M outside the supported set; elu+1 needs M == d; NULL buffers
    assert lib.slim_attn_decode(dummy, dummy, dummy, dummy, dummy, dummy, 1, 1, 48, 64, None) == 2
    assert lib.slim_attn_decode(dummy, dummy, dummy, dummy, dummy, dummy, 1, 1, 64, 40, None) == 2
    assert lib.slim_attn_decode(dummy, dummy, dummy, None, dummy, dummy, 1, 1, 64, 128, None) == 1
    assert lib.slim_attn_decode(None, dummy, dummy, dummy, dummy, dummy, 1, 1, 64, 64, None) == 1
    assert lib.slim_attn_decode(dummy, dummy, dummy, dummy, None, dummy, 1, 1, 64, 64, None) == 1
    assert lib.slim_attn_decode_f32(dummy, dummy, dummy, dummy, dummy, dummy, -1, 1, 64, 64, None) == 1
    # no heads: nothing to do
    assert lib.slim_attn_decode(dummy, dummy, dummy, dummy, dummy, dummy, 0, 4, 64, 64, None) == 0
    # state: shape checks as for the forward; NULL state
    assert lib.slim_attn_state(dummy, dummy, dummy, dummy, 1, 1, 64, 48, 64, 32, None) == 2
    assert lib.slim_attn_state(dummy, dummy, dummy, dummy, 1, 1, 64, 64, 64, 48, None) == 2
    assert lib.slim_attn_state(dummy, dummy, dummy, None, 1, 1, 64, 64, 64, 32, None) == 1
    assert lib.slim_attn_state_f32(dummy, dummy, None, dummy, 1, 1, 64, 64, 128, 32, None) == 1


def test_selftest_rejects_bad_limits_on_the_host(lib):
    # limits outside [1 us, 100 ms] return SLIM_ERR_INVALID_ARG before any launch
    for bad in (0, 999, 100_000_001, -5):
        assert lib.slim_attn_selftest_timeout(bad, None, None) == 1


def test_noalloc_size_query(lib):
    """slim_attn_noalloc_bytes is the CUDA-core forward plan's size: never more
    than the registered-workspace size for the same shape, 0 when empty."""
    assert lib.slim_attn_noalloc_bytes(0, 4, 128, 64, 64, 64) == 0
    assert lib.slim_attn_noalloc_bytes(1, 1, 64, 48, 64, 32) == 0  # d unsupported
    for shape in ((2, 4, 2048, 64, 128, 64), (1, 3, 777, 32, 64, 32), (2, 16, 32768, 64, 256, 128)):
        n = lib.slim_attn_noalloc_bytes(*shape)
        assert 0 < n <= lib.slim_attn_workspace_bytes(*shape, 0)
    assert lib.slim_attn_noalloc_bytes(2, 16, 32768, 64, 256, 128) > (64 << 20)


def test_debug_build_exports_every_declared_symbol():
    """The -DSLIM_DEBUG variant (device-side bounds checks that record
    SLIM_ERR_BOUNDS; every call waits and reports device errors itself)
    builds and exports the same C ABI."""
    path = build.build(debug=True)
    dbg = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    dbg.slim_status_string.restype = ctypes.c_char_p
    assert dbg.slim_status_string(6).startswith(b"SLIM_ERR_BOUNDS")
