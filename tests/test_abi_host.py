"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every entry point
include/dspark.h declares, and rejects invalid arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_ragged_gb300 import build
    build.build()
    from speculative_decoding_ragged_gb300 import _binding
    return _binding.lib()


def header_functions():
    with open(os.path.join(ROOT, "include", "dspark.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert {"dspark_schedule", "dspark_pack", "dspark_verify", "dspark_scatter"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name
    from speculative_decoding_ragged_gb300 import _binding
    assert set(names) == set(_binding.SYMBOLS)


def test_version(lib):
    # 1.1: the dspark_graph_* capture and replay calls
    assert lib.dspark_version() == 102


def test_argument_errors_are_reported_on_the_host(lib):
    from speculative_decoding_ragged_gb300 import _binding as bd
    cost = bd._Cost(1.0, None, 0, None, 0)
    rc = lib.dspark_schedule(None, -1, 4, ctypes.byref(cost), None, None, None, None)
    assert rc == -1 and "B = -1" in bd.last_error()
    rc = lib.dspark_schedule(None, 4, 40, ctypes.byref(cost), None, None, None, None)
    assert rc == -1 and "gamma" in bd.last_error()
    rc = lib.dspark_schedule(None, 8192, 4, ctypes.byref(cost), None, None, None, None)
    assert rc == -2 and "B*(gamma-1)" in bd.last_error()     # 24576 candidates > 16384
    rc = lib.dspark_pack(None, None, 2, 4, None, 0, None, None, None, None, 0, None, None, None)
    assert rc == -1 and "n_tiers" in bd.last_error()
    rc = lib.dspark_verify(7, 0, None, 0, None, 0, 16, None, None, None, 1, 2, 1.0, 0, 0,
                           None, None, None, None, None, 0, None, None)
    assert rc == -1 and "mode" in bd.last_error()
    rc = lib.dspark_verify(1, 1, None, 0, None, 0, 16, None, None, None, 1, 2, 0.0, 0, 0,
                           None, None, None, None, None, 0, None, None)
    assert rc == -1 and "temperature" in bd.last_error()
    rc = lib.dspark_verify(1, 0, None, 0, None, 0, 16, None, None, None, 1, 2, 1.0, 0, 0,
                           None, None, None, None, None, 0, None, None)
    assert rc == -1 and "required" in bd.last_error()
    rc = lib.dspark_scatter(None, None, 3, 33, None, None, 4, None, None)
    assert rc == -1


def test_fused_entry_points_check_both_halves(lib):
    from speculative_decoding_ragged_gb300 import _binding as bd
    cost = bd._Cost(1.0, None, 0, None, 0)
    rc = lib.dspark_schedule_pack(None, -1, 4, ctypes.byref(cost), None, None, 1, None, None,
                                  None, None, None, None, 0, None, None, None)
    assert rc == -1 and "dspark_schedule_pack: B = -1" in bd.last_error()
    rc = lib.dspark_schedule_pack(None, 8192, 4, ctypes.byref(cost), None, None, 1, None, None,
                                  None, None, None, None, 0, None, None, None)
    assert rc == -2 and "B*(gamma-1)" in bd.last_error()
    # the schedule half is valid (B == 0), the pack half is not (no tiers)
    k = ctypes.c_int32(0)
    rc = lib.dspark_schedule_pack(None, 0, 4, ctypes.byref(cost), None, None, 0, None,
                                  ctypes.byref(k), None, None, None, None, 0, None, None, None)
    assert rc == -1 and "n_tiers" in bd.last_error()
    rc = lib.dspark_verify_scatter(1, 0, None, 0, None, 0, 16, None, None, None, 1, 2, 1.0, 0,
                                   0, None, None, None, None, None, 0, None, None, 4, None, None)
    assert rc == -1 and "dspark_verify_scatter" in bd.last_error()
    # the verify half is valid (B == 0), the scatter half is not (negative capacity)
    rc = lib.dspark_verify_scatter(1, 0, None, 0, None, 0, 16, None, None, None, 0, 2, 1.0, 0,
                                   0, None, None, None, None, None, 0, None, None, -1, None, None)
    assert rc == -1 and "out_cap=-1" in bd.last_error()
    rc = lib.dspark_verify_scatter(1, 0, None, 0, None, 0, 16, None, None, None, 0, 2, 1.0, 0,
                                   0, None, None, None, None, None, 0, None, None, 4, None, None)
    assert rc == 0


def test_workspace_size_is_a_function_of_sizes(lib):
    from speculative_decoding_ragged_gb300 import _binding as bd
    assert bd.dspark_verify_workspace_bytes(0, 8, 1000, False) == 0
    g = bd.dspark_verify_workspace_bytes(256, 8, 151936, False)
    s = bd.dspark_verify_workspace_bytes(256, 8, 151936, True)
    # a 256-byte head, then the target partials (8 B per chunk of each of the B*gamma rows);
    # stochastic adds the draft partials (as many, 8 B each), a 4-byte counter per request and
    # two fp32 sums per 256-token tile per request
    align = lambda x: (x + 255) // 256 * 256
    part = g - 256
    assert part > 0 and part % 256 == 0
    assert s == 256 + 2 * part + align(4 * 256) + align(8 * 256 * ((151936 + 255) // 256))
    assert bd.dspark_verify_workspace_bytes(-1, 8, 10, False) == 0
    assert "bad sizes" in bd.last_error()


def test_stream_kernel_setting_is_checked(lib):
    from speculative_decoding_ragged_gb300 import _binding as bd
    assert lib.dspark_set_stream_kernel(7) == -1 and "unknown kernel 7" in bd.last_error()
    assert lib.dspark_set_stream_kernel(bd.STREAM_BULK) == 0
    assert lib.dspark_set_stream_kernel(bd.STREAM_AUTO) == 0


def test_stream_events_need_both_or_neither(lib):
    from speculative_decoding_ragged_gb300 import _binding as bd
    assert lib.dspark_set_stream_events(ctypes.c_void_p(8), None) == -1
    assert "both events or neither" in bd.last_error()
    assert lib.dspark_set_stream_events(None, None) == 0
