"""The layout entry point that allocates nothing (ep_get_dispatch_layout_noalloc).

It serves callers that cannot allocate device memory where they need the
layout (a host framework's caching allocator owns the GPU's memory, a
plug-in only gets its input and output buffers, or a latency-critical loop
must not risk a synchronising cudaMalloc). It keeps its scratch in a fixed
device array inside the library instead of a caller-provided workspace.

Checked here through the C ABI: two calls in a row, on different routings,
give exactly the results of ep_get_dispatch_layout and of the CPU oracle (the
layout is integer work, so the tolerance is zero); a size whose scratch would
exceed the fixed array is refused on the host; and an argument error queues
nothing on the stream (seen by capturing the call into a CUDA graph).

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import combine_ep_get_dispatch_gb300 as ep
import epinputs as ei
import oracle

pytestmark = pytest.mark.gpu

KEYS = ("num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "expert_offset",
        "rank_offset", "expert_slot", "rank_slot")


@pytest.fixture(scope="module")
def noalloc():
    import __graft_entry__ as g
    g.build()
    f = ep.lib().ep_get_dispatch_layout_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ep.ep_layout_t), ctypes.c_void_p, ctypes.c_void_p]
    return f


def _call(f, lay, status):
    c = lay.c_struct()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(ctypes.byref(c), ctypes.c_void_p(status.data_ptr()), stream)


@pytest.mark.parametrize("cfgs", [(4, 5), (3, 2)])
def test_noalloc_matches_workspace_entry_point_twice(noalloc, cfgs):
    for c in cfgs:  # two calls in a row on different routings
        cfg = ei.WORKLOADS[c]
        idx, _ = ei.make_routing(cfg, seed=11 + c)
        idx_d = torch.from_numpy(idx).cuda()
        st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = ep.get_dispatch_layout(idx_d, cfg.E, cfg.R, status=st_ref)
        got = ep.new_layout(idx_d, cfg.E, cfg.R)
        for k in KEYS:
            getattr(got, k).fill_(-3)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _call(noalloc, got, st) == ep.EP_OK
        torch.cuda.synchronize()
        want = oracle.layout(idx, cfg.E, cfg.R)
        for k in KEYS:
            assert torch.equal(getattr(got, k), getattr(ref, k)), (c, k)
            assert np.array_equal(getattr(got, k).cpu().numpy(), want[k]), (c, k)
        assert int(st.item()) == int(st_ref.item()) == 0


def test_noalloc_refuses_sizes_beyond_its_scratch(noalloc):
    # E = R = 1024: the scratch needs 8 KiB per layout block; 2**20 entries
    # need 171 blocks, more than the fixed 1 MiB array holds.
    N, K, E, R = 1 << 17, 8, 1024, 1024
    assert ep.ep_layout_workspace_bytes(N, K, E, R) > (1 << 20)
    idx_d = torch.zeros((N, K), dtype=torch.int32, device="cuda")
    lay = ep.new_layout(idx_d, E, R)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call(noalloc, lay, st) == ep.EP_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def _captured_nodes(fn) -> int:
    """(return code, nodes enqueued) of a call captured on a fresh stream."""
    rt = ctypes.CDLL("libcudart.so.13")
    rt.cudaStreamBeginCapture.argtypes = [ctypes.c_void_p, ctypes.c_int]
    rt.cudaStreamEndCapture.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    rt.cudaGraphGetNodes.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)]
    rt.cudaGraphDestroy.argtypes = [ctypes.c_void_p]
    s = torch.cuda.Stream()
    h = ctypes.c_void_p(s.cuda_stream)
    assert rt.cudaStreamBeginCapture(h, 2) == 0        # cudaStreamCaptureModeRelaxed
    rc = fn(h)
    g = ctypes.c_void_p()
    assert rt.cudaStreamEndCapture(h, ctypes.byref(g)) == 0
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetNodes(g, None, ctypes.byref(n)) == 0
    rt.cudaGraphDestroy(g)
    return rc, n.value


def test_noalloc_argument_error_queues_nothing(noalloc):
    cfg = ei.WORKLOADS[5].scaled(N=1000)
    idx, _ = ei.make_routing(cfg, seed=3)
    lay = ep.new_layout(torch.from_numpy(idx).cuda(), cfg.E, cfg.R)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call(noalloc, lay, st) == ep.EP_OK          # the device's first call happens outside any capture
    torch.cuda.synchronize()
    c = lay.c_struct()
    stp = ctypes.c_void_p(st.data_ptr())
    rc, n = _captured_nodes(lambda h: noalloc(ctypes.byref(c), stp, h))
    assert rc == ep.EP_OK and n >= 2                    # the barrier reset and the layout kernel
    bad = ep.ep_layout_t.from_buffer_copy(c)
    bad.rank_slot = None
    rc, n = _captured_nodes(lambda h: noalloc(ctypes.byref(bad), stp, h))
    assert rc == ep.EP_ERR_INVALID_ARG and n == 0
