"""The C ABI without a GPU: the library loads, exports every function that
include/ep.h declares, and rejects bad arguments on the host before any CUDA
call (no compute is launched here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")


@pytest.fixture(scope="module")
def L():
    from combine_ep_get_dispatch_gb300 import build
    build.build()
    import combine_ep_get_dispatch_gb300 as ep
    return ep.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(ep_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["ep_get_dispatch_layout", "ep_dispatch", "ep_combine", "ep_ll_dispatch_send",
              "ep_ll_dispatch_recv", "ep_ll_combine", "ep_layout_workspace_bytes", "ep_ll_workspace_bytes"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_version_and_error_strings(L):
    import combine_ep_get_dispatch_gb300 as ep
    assert L.ep_version() >= 100
    assert ep.ep_error_string(ep.EP_ERR_LL_CAPACITY).startswith("low-latency")
    assert ep.ep_error_string(ep.EP_ST_NOT_SENT).startswith("status")
    assert "zero-fill" in ep.ep_error_string(ep.EP_ST_WORKSPACE)
    assert ep.ep_error_string(0) == "ok"


def test_workspace_sizes(L):
    import combine_ep_get_dispatch_gb300 as ep
    assert ep.ep_layout_workspace_bytes(16384, 6, 256, 8) > 0
    assert ep.ep_layout_workspace_bytes(16, 6, 250, 8) == 0     # E % R != 0
    assert ep.ep_layout_workspace_bytes(16, 0, 256, 8) == 0     # K < 1
    assert ep.ep_layout_workspace_bytes(16, 33, 256, 8) == 0    # K > EP_MAX_TOPK
    assert ep.ep_layout_workspace_bytes(16, 8, 2048, 8) == 0    # E > EP_MAX_EXPERTS
    a = ep.ep_ll_workspace_bytes(4096, 8, 256, 32, 128)
    assert a >= 4096 * 8 * 4 + 256 * 32 * 8
    assert ep.ep_ll_workspace_bytes(4096, 8, 256, 32, 0) == 0


def test_host_validation_rejects_before_cuda(L):
    import combine_ep_get_dispatch_gb300 as ep
    P = ctypes.c_void_p
    # null layout handle
    assert L.ep_get_dispatch_layout(None, None, 0, None, None) == ep.EP_ERR_INVALID_ARG
    # sizes out of range
    lay = ep.ep_layout_t(10, 8, 250, 8, P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16))
    assert L.ep_get_dispatch_layout(ctypes.byref(lay), P(256), 1 << 20, None, None) == ep.EP_ERR_INVALID_ARG
    # workspace too small
    lay = ep.ep_layout_t(10, 8, 256, 8, P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16))
    assert L.ep_get_dispatch_layout(ctypes.byref(lay), P(256), 16, None, None) == ep.EP_ERR_WORKSPACE
    # workspace not 16-byte aligned
    assert L.ep_get_dispatch_layout(ctypes.byref(lay), P(264), 1 << 20, None, None) == ep.EP_ERR_ALIGNMENT
    # dispatch: misaligned x, bad hidden sizes
    assert L.ep_dispatch(ctypes.byref(lay), P(18), 64, 0, None, None, None, None, None) == ep.EP_ERR_ALIGNMENT
    assert L.ep_dispatch(ctypes.byref(lay), P(16), 60, 0, None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(ctypes.byref(lay), P(16), 64, 1, None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(ctypes.byref(lay), P(16), 32768, 0, None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    # layout + dispatch in one call: the dispatch arguments are checked first, then the layout's
    LD = L.ep_layout_dispatch
    assert LD(None, P(256), 1 << 20, P(16), 64, 0, None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert LD(ctypes.byref(lay), P(256), 1 << 20, P(18), 64, 0, None, None, None, None, None) \
        == ep.EP_ERR_ALIGNMENT
    assert LD(ctypes.byref(lay), P(256), 1 << 20, P(16), 60, 0, None, None, None, None, None) \
        == ep.EP_ERR_INVALID_ARG
    assert LD(ctypes.byref(lay), P(256), 1 << 20, P(16), 128, ep.EP_FP8_UE8M0, None, None, None, None, None) \
        == ep.EP_ERR_INVALID_ARG
    assert LD(ctypes.byref(lay), P(256), 16, P(16), 64, 0, None, None, None, None, None) == ep.EP_ERR_WORKSPACE
    assert LD(ctypes.byref(lay), P(264), 1 << 20, P(16), 64, 0, None, None, None, None, None) \
        == ep.EP_ERR_ALIGNMENT
    # combine: misaligned output
    assert L.ep_combine(ctypes.byref(lay), P(16), 10, 64, P(16), None, P(24), None, None) == ep.EP_ERR_ALIGNMENT
    assert L.ep_combine(ctypes.byref(lay), P(16), 10, 64, P(16), P(40), P(32), None, None) == ep.EP_ERR_ALIGNMENT
    # alignment of the expert segments must be sane
    bad = ep.ep_layout_t(10, 8, 256, 8, P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16), -3)
    assert L.ep_get_dispatch_layout(ctypes.byref(bad), P(256), 1 << 20, None, None) == ep.EP_ERR_INVALID_ARG
    # low latency: tokens per rank above T, N not divisible by R, missing workspace
    ll = L.ep_ll_dispatch_send
    assert ll(P(16), P(16), 160, 8, 256, 256, 8, 16, 0, P(16), None, P(16), P(256), 1 << 30, None, None) \
        == ep.EP_ERR_LL_CAPACITY
    assert ll(P(16), P(16), 130, 8, 256, 256, 8, 128, 0, P(16), None, P(16), P(256), 1 << 30, None, None) \
        == ep.EP_ERR_INVALID_ARG
    assert ll(P(16), P(16), 128, 8, 256, 256, 8, 128, 0, P(16), None, P(16), None, 0, None, None) \
        == ep.EP_ERR_WORKSPACE
    assert ll(P(16), P(16), 128, 8, 256, 256, 8, 128, 1, P(16), None, P(16), P(256), 1 << 30, None, None) \
        == ep.EP_ERR_INVALID_ARG  # FP8 without a scale buffer
    assert L.ep_ll_dispatch_recv(P(256), 16, 128, 8, 256, 8, 128, P(16), None, None, None, None) \
        == ep.EP_ERR_WORKSPACE
    # FP8 flag words: scale options need EP_FP8; unknown bits are refused
    assert L.ep_dispatch(ctypes.byref(lay), P(16), 128, ep.EP_FP8_ROUND_SCALE, None, None, None, None, None) \
        == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(ctypes.byref(lay), P(16), 128, 0x8 | ep.EP_FP8, None, None, None, None, None) \
        == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(ctypes.byref(lay), P(16), 128, ep.EP_FP8 | ep.EP_FP8_UE8M0, None, None, None, None,
                         None) == ep.EP_OK  # valid flags; no buffer given, so nothing to launch
    assert L.ep_ll_combine(P(16), P(16), None, P(256), 1 << 30, 128, 8, 100, 256, 8, 128, P(16), None, None) \
        == ep.EP_ERR_INVALID_ARG  # hidden % 8 != 0
    assert L.ep_fp8_e4m3_encode(None, None, -1, None) == ep.EP_ERR_INVALID_ARG
    # quantisation on its own: FP8 flag required, hidden % 128, 16-byte rows, buffers for rows > 0
    Q = L.ep_fp8_quantize
    assert Q(P(16), 4, 256, 0, P(16), P(16), None) == ep.EP_ERR_INVALID_ARG          # BF16 flag word
    assert Q(P(16), 4, 200, ep.EP_FP8, P(16), P(16), None) == ep.EP_ERR_INVALID_ARG  # hidden % 128 != 0
    assert Q(P(16), -1, 256, ep.EP_FP8, P(16), P(16), None) == ep.EP_ERR_INVALID_ARG
    assert Q(P(16), 4, 256, ep.EP_FP8, P(16), None, None) == ep.EP_ERR_INVALID_ARG   # no scale buffer
    assert Q(P(24), 4, 256, ep.EP_FP8, P(16), P(16), None) == ep.EP_ERR_ALIGNMENT
    assert Q(P(16), 4, 256, ep.EP_FP8, P(40), P(16), None) == ep.EP_ERR_ALIGNMENT
    assert Q(None, 0, 256, ep.EP_FP8 | ep.EP_FP8_UE8M0, None, None, None) == ep.EP_OK  # nothing to do
    # shrink-mode mask calls: rank range, rank count, workspace size
    assert L.ep_ll_update_mask(P(256), 1 << 20, 8, 8, 1, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_ll_update_mask(P(256), 1 << 20, 0, 0, 1, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_ll_update_mask(P(256), 64, 8, 0, 1, None) == ep.EP_ERR_WORKSPACE
    assert L.ep_ll_query_mask(P(256), 1 << 20, 8, None, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_ll_clean_mask(None, 0, 8, None) == ep.EP_ERR_WORKSPACE


def test_package_has_no_cpu_fallback():
    """The product package never imports the oracle (test infrastructure)."""
    pkg = os.path.join(ROOT, "combine_ep_get_dispatch_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "ep_oracle" not in text, f
