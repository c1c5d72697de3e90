"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bar: bit-exact for counts, masks, slots, source indices, BF16 and FP8
payloads and scales; combine within 1 BF16 step of the oracle (the design
makes it bit-exact too: the same fp32 fused multiply-add chain in slot order,
and that is asserted as well).

Sizes: ragged slices of every workload that span several CTAs and warps,
edge shapes and the maximum sizes the ABI accepts; the full workloads are
compared array by array in test_gpu_full_size.py.
"""
import numpy as np
import pytest
import torch

import combine_ep_get_dispatch_gb300 as ep
import epinputs as ei
import oracle
from helpers import bf16_ulp_diff, status_value, to_dev, to_dev_bf16, u16, u8

pytestmark = pytest.mark.gpu

LAYOUT_KEYS = ("num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "expert_offset",
               "rank_offset", "expert_slot", "rank_slot")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available()


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _layout_equal(lay, ref):
    for k in LAYOUT_KEYS:
        got = getattr(lay, k).cpu().numpy()
        assert np.array_equal(got, ref[k]), k


# ------------------------------------------------------------------ layout ----
@pytest.mark.parametrize("c", [1, 2, 3, 4, 5])
def test_layout_full_configs(c):
    cfg = ei.WORKLOADS[c]
    idx, _ = ei.make_routing(cfg, 0)
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(idx), cfg.E, cfg.R, status=st)
    _layout_equal(lay, oracle.layout(idx, cfg.E, cfg.R))
    assert status_value(st) == 0


def _rand_idx(N, K, E, seed, p_mask=0.0, distinct=True):
    key = ei.stream_key(seed, 900)
    u = ei.uniform01(key, N * E).reshape(N, E)
    if distinct:
        idx = np.argsort(u, axis=1)[:, :K].astype(np.int32)
    else:
        idx = (ei.uniform01(ei.stream_key(seed, 901), N * K).reshape(N, K) * E).astype(np.int32)
    if p_mask:
        m = ei.uniform01(ei.stream_key(seed, 902), N * K).reshape(N, K) < p_mask
        idx[m] = -1
    return idx


@pytest.mark.parametrize("N,K,E,R,p_mask,distinct", [
    (0, 8, 256, 8, 0.0, True),
    (1, 8, 256, 8, 0.0, True),
    (1000, 6, 256, 8, 0.0, True),
    (7777, 8, 128, 8, 0.1, True),
    (5000, 4, 64, 1, 0.0, True),
    (3000, 4, 64, 64, 0.3, True),
    (2000, 32, 1024, 16, 0.05, True),
    (4097, 1, 32, 4, 0.0, True),
    (999, 8, 16, 4, 0.2, False),       # repeated experts within a row
    (40000, 8, 256, 32, 0.0, True),    # many CTAs
])
def test_layout_edge_cases(N, K, E, R, p_mask, distinct):
    idx = _rand_idx(N, K, E, seed=N + K, p_mask=p_mask, distinct=distinct) if N else np.zeros((0, K), np.int32)
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(idx) if N else torch.zeros((0, K), dtype=torch.int32, device="cuda"),
                                 E, R, status=st)
    _layout_equal(lay, oracle.layout(idx, E, R))
    assert status_value(st) == 0


def test_layout_all_masked_and_bad_indices():
    idx = np.full((300, 4), -1, np.int32)
    lay = ep.get_dispatch_layout(to_dev(idx), 32, 4)
    _layout_equal(lay, oracle.layout(idx, 32, 4))
    idx = _rand_idx(500, 4, 32, seed=3)
    idx[::7, 1] = 32
    idx[::11, 2] = -5
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(idx), 32, 4, status=st)
    ref = oracle.layout(idx, 32, 4)
    _layout_equal(lay, ref)
    assert ref["status"] & oracle.BAD_INDEX
    assert status_value(st) & ep.EP_ST_BAD_INDEX


def test_layout_deterministic_repeat():
    cfg = ei.WORKLOADS[4]
    idx, _ = ei.make_routing(cfg, 0)
    a = ep.get_dispatch_layout(to_dev(idx), cfg.E, cfg.R)
    b = ep.get_dispatch_layout(to_dev(idx), cfg.E, cfg.R)
    for k in LAYOUT_KEYS:
        assert torch.equal(getattr(a, k), getattr(b, k))


def test_layout_workspace_left_clean_and_dirty_one_flagged():
    """The grid barrier clears its own arrival count: calls on one zero-filled
    workspace stay exact with no reset in between; a leftover count (a
    workspace never zero-filled) is reported with EP_ST_WORKSPACE."""
    cfg = ei.WORKLOADS[4].scaled(N=2048)          # 12288 entries: a dozen CTAs, so a real grid barrier
    idx, _ = ei.make_routing(cfg, 50)
    ref = oracle.layout(idx, cfg.E, cfg.R)
    ws = torch.zeros(ep.ep_layout_workspace_bytes(cfg.N, cfg.K, cfg.E, cfg.R), dtype=torch.uint8, device="cuda")
    lay = ep.new_layout(to_dev(idx), cfg.E, cfg.R)
    for _ in range(3):
        st = _status()
        ep.ep_get_dispatch_layout(lay, ws, st)
        _layout_equal(lay, ref)
        assert status_value(st) == 0
        assert int(ws[:4].view(torch.int32).item()) == 0    # the arrival count is zero again
    # Leftover bytes: an arrival count of 0x01010101 is far above the block
    # count, so every block reports it and none waits.
    ws[:8] = 1
    st = _status()
    ep.ep_get_dispatch_layout(lay, ws, st)
    assert status_value(st) & ep.EP_ST_WORKSPACE
    ws[:8] = 0
    st = _status()
    ep.ep_get_dispatch_layout(lay, ws, st)
    _layout_equal(lay, ref)
    assert status_value(st) == 0


def test_layout_grid_wait_runs_out_and_reports_it():
    """A bounded in-kernel wait that runs out: the layout's arrival count is
    seeded with 0xFFFFFFFF, so the first block to arrive sees a count above
    the block count (EP_ST_WORKSPACE) and wraps it to zero, and no later block
    is ever the last arrival. The others wait their one-second limit, set
    EP_ST_TIMEOUT and finish (every access stays inside the arrays). The
    context stays usable: after a zero fill the next call is exact."""
    import time
    cfg = ei.WORKLOADS[4].scaled(N=2048)          # a dozen CTAs
    idx, _ = ei.make_routing(cfg, 51)
    ref = oracle.layout(idx, cfg.E, cfg.R)
    ws = torch.zeros(ep.ep_layout_workspace_bytes(cfg.N, cfg.K, cfg.E, cfg.R), dtype=torch.uint8, device="cuda")
    lay = ep.new_layout(to_dev(idx), cfg.E, cfg.R)
    ws[:4] = 0xFF
    st = _status()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ep.ep_get_dispatch_layout(lay, ws, st)
    val = status_value(st)
    waited = time.perf_counter() - t0
    assert val & ep.EP_ST_TIMEOUT and val & ep.EP_ST_WORKSPACE, val
    assert 0.5 < waited < 30.0, waited
    ws.zero_()
    st = _status()
    ep.ep_get_dispatch_layout(lay, ws, st)
    _layout_equal(lay, ref)
    assert status_value(st) == 0


# ---------------------------------------------------------------- dispatch ----
def _check_dispatch(res, ref, use_fp8, K, with_rank=True):
    conv = u8 if use_fp8 else u16
    D_e = ref["exp_x"].shape[0]
    assert np.array_equal(conv(res.expert_x[:D_e]), ref["exp_x"])
    assert np.array_equal(res.expert_src[:D_e].cpu().numpy(), ref["exp_src"])
    if use_fp8:
        assert np.array_equal(res.expert_scales[:D_e].cpu().numpy(), ref["exp_scales"])
    if with_rank:
        D_r = ref["rank_x"].shape[0]
        assert np.array_equal(conv(res.rank_x[:D_r]), ref["rank_x"])
        assert np.array_equal(res.rank_src[:D_r].cpu().numpy(), ref["rank_src"])
        assert np.array_equal(res.rank_topk_idx[:D_r].cpu().numpy(), ref["rank_topk_idx"])
        assert np.array_equal(res.rank_topk_weights[:D_r].cpu().numpy(), ref["rank_topk_weights"])
        if use_fp8:
            assert np.array_equal(res.rank_scales[:D_r].cpu().numpy(), ref["rank_scales"])


@pytest.mark.parametrize("c,N,H", [(3, 1000, 7168), (4, 777, 7168), (5, 1500, 4096), (3, 257, 128),
                                   (4, 333, 8), (5, 64, 1024)])
@pytest.mark.parametrize("use_fp8", [False, True])
def test_dispatch_parity(c, N, H, use_fp8):
    if use_fp8 and H % 128:
        pytest.skip("FP8 needs hidden % 128 == 0")
    cfg = ei.WORKLOADS[c].scaled(N=N, H=H)
    d = ei.make_inputs(cfg, seed=c)
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(d["topk_idx"]), cfg.E, cfg.R, status=st)
    res = ep.dispatch(to_dev_bf16(d["x"]), lay, to_dev(d["topk_weights"]), use_fp8=use_fp8, exact=False,
                      status=st)
    ref = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], cfg.E, cfg.R, use_fp8)
    _check_dispatch(res, ref, use_fp8, cfg.K)
    assert status_value(st) == 0


@pytest.mark.parametrize("use_fp8", [False, True])
def test_maximum_sizes(use_fp8):
    """The largest shapes the ABI accepts: hidden 16384, top-32, 1024 experts
    on 1024 ranks (one expert each): layout, both receive buffers and combine
    against the oracle."""
    N, H, K, E, R = 70, ep.EP_MAX_HIDDEN, ep.EP_MAX_TOPK, ep.EP_MAX_EXPERTS, ep.EP_MAX_EXPERTS
    idx = _rand_idx(N, K, E, seed=11, p_mask=0.1)
    x = ei.make_x(N, H, seed=12)
    w = ei.uniform01(ei.stream_key(13, 0), N * K).reshape(N, K).astype(np.float32)
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(idx), E, R, status=st)
    _layout_equal(lay, oracle.layout(idx, E, R))
    res = ep.dispatch(to_dev_bf16(x), lay, to_dev(w), use_fp8=use_fp8, status=st)
    ref = oracle.dispatch(x, idx, w, E, R, use_fp8)
    _check_dispatch(res, ref, use_fp8, K)
    y = ep.dispatch(to_dev_bf16(x), lay, to_dev(w), with_rank=False).expert_x
    out = ep.combine(y, lay, to_dev(w), status=st)
    ref_out, _ = oracle.combine(u16(y), ref["layout"]["expert_slot"], w)
    assert np.array_equal(u16(out), ref_out)
    assert status_value(st) == 0


def test_dispatch_expert_only_and_rank_only():
    cfg = ei.WORKLOADS[4].scaled(N=500, H=1024)
    d = ei.make_inputs(cfg, seed=9)
    lay = ep.get_dispatch_layout(to_dev(d["topk_idx"]), cfg.E, cfg.R)
    ref = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], cfg.E, cfg.R, False)
    res = ep.dispatch(to_dev_bf16(d["x"]), lay, to_dev(d["topk_weights"]), with_rank=False, exact=True)
    assert res.rank_x is None
    _check_dispatch(res, ref, False, cfg.K, with_rank=False)
    res = ep.dispatch(to_dev_bf16(d["x"]), lay, to_dev(d["topk_weights"]), with_expert=False, exact=True)
    D_r = ref["rank_x"].shape[0]
    assert np.array_equal(u16(res.rank_x), ref["rank_x"]) and res.rank_x.shape[0] == D_r


@pytest.mark.parametrize("c,N,H,use_fp8", [(3, 1000, 7168, True), (4, 777, 7168, False), (5, 1500, 4096, True),
                                           (4, 333, 8, False), (3, 257, 128, False), (5, 64, 1024, True)])
def test_layout_and_dispatch_in_one_call(c, N, H, use_fp8):
    """ep_layout_dispatch (the dispatch launched as the layout's programmatic
    dependent) gives the oracle's layout and receive rows."""
    cfg = ei.WORKLOADS[c].scaled(N=N, H=H)
    d = ei.make_inputs(cfg, seed=c + 20)
    st = _status()
    lay, res = ep.get_layout_and_dispatch(to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), cfg.E, cfg.R,
                                          to_dev(d["topk_weights"]), use_fp8=use_fp8, status=st)
    _layout_equal(lay, oracle.layout(d["topk_idx"], cfg.E, cfg.R))
    ref = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], cfg.E, cfg.R, use_fp8)
    _check_dispatch(res, ref, use_fp8, cfg.K)
    assert status_value(st) == 0


def _same_dispatch(lay1, r1, lay2, r2):
    for k in LAYOUT_KEYS:
        assert torch.equal(getattr(lay1, k), getattr(lay2, k)), k
    D_e, D_r = int(lay1.expert_offset[-1].item()), int(lay1.rank_offset[-1].item())
    for name, D in (("expert_x", D_e), ("expert_scales", D_e), ("expert_src", D_e), ("rank_x", D_r),
                    ("rank_scales", D_r), ("rank_src", D_r), ("rank_topk_idx", D_r), ("rank_topk_weights", D_r)):
        a, b = getattr(r1, name), getattr(r2, name)
        assert (a is None) == (b is None), name
        if a is not None:
            assert torch.equal(a[:D], b[:D]), name


@pytest.mark.parametrize("c", [3, 4, 5])
def test_layout_and_dispatch_full_size_matches_two_calls(c):
    """On the full workloads the one-call path writes exactly what
    ep_get_dispatch_layout + ep_dispatch write (checked against the oracle above)."""
    cfg = ei.WORKLOADS[c]
    d = ei.make_inputs(cfg, seed=0)
    x, idx, w = to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), to_dev(d["topk_weights"])
    st = _status()
    lay1 = ep.get_dispatch_layout(idx, cfg.E, cfg.R, status=st)
    r1 = ep.dispatch(x, lay1, w, use_fp8=cfg.fp8, status=st)
    lay2, r2 = ep.get_layout_and_dispatch(x, idx, cfg.E, cfg.R, w, use_fp8=cfg.fp8, status=st)
    _same_dispatch(lay1, r1, lay2, r2)
    assert status_value(st) == 0
    del r1, r2
    torch.cuda.empty_cache()


def test_layout_and_dispatch_empty_masked_and_bad_indices():
    """The one-call path on an empty batch, and on a routing with masked slots and
    out-of-range indices: the same rows and status bits as the two calls."""
    H = 256
    x0 = torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
    st = _status()
    lay, res = ep.get_layout_and_dispatch(x0, torch.empty((0, 4), dtype=torch.int32, device="cuda"), 32, 4,
                                          torch.empty((0, 4), dtype=torch.float32, device="cuda"), status=st)
    assert lay.expert_offset.cpu().numpy().tolist() == [0] * 33
    assert status_value(st) == 0
    idx = _rand_idx(500, 4, 32, seed=5)
    idx[::7, 1] = 32
    idx[::11, 2] = -5
    idx[::13, 3] = -1
    d = ei.make_inputs(ei.WORKLOADS[4].scaled(N=500, H=H, K=4, E=32, R=4), seed=6)
    x, w = to_dev_bf16(d["x"]), to_dev(d["topk_weights"])
    for fp8 in (False, True):
        st1, st2 = _status(), _status()
        lay1 = ep.get_dispatch_layout(to_dev(idx), 32, 4, status=st1)
        r1 = ep.dispatch(x, lay1, w, use_fp8=fp8, status=st1)
        lay2, r2 = ep.get_layout_and_dispatch(x, to_dev(idx), 32, 4, w, use_fp8=fp8, status=st2)
        _same_dispatch(lay1, r1, lay2, r2)
        assert status_value(st1) == status_value(st2) == ep.EP_ST_BAD_INDEX
        _layout_equal(lay2, oracle.layout(idx, 32, 4))


@pytest.mark.parametrize("round_scale,ue8m0", [(False, False), (True, False), (False, True)])
def test_layout_and_dispatch_aligned_with_padding(round_scale, ue8m0):
    """Expert segments padded to 128 rows, with each FP8 scale format: the
    one-call path writes the same rows, scales and zero-filled padding rows."""
    cfg = ei.WORKLOADS[3].scaled(N=600, H=1024)
    d = ei.make_inputs(cfg, seed=31)
    x, idx, w = to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), to_dev(d["topk_weights"])
    st = _status()
    opts = dict(use_fp8=True, round_scale=round_scale, use_ue8m0=ue8m0)
    lay1 = ep.get_dispatch_layout(idx, cfg.E, cfg.R, status=st, expert_alignment=128)
    r1 = ep.dispatch(x, lay1, w, status=st, **opts)
    lay2, r2 = ep.get_layout_and_dispatch(x, idx, cfg.E, cfg.R, w, status=st, expert_alignment=128, **opts)
    _same_dispatch(lay1, r1, lay2, r2)
    assert status_value(st) == 0


def test_dispatch_capacity_overflow_flagged():
    cfg = ei.WORKLOADS[4].scaled(N=400, H=256)
    d = ei.make_inputs(cfg, seed=4)
    lay = ep.get_dispatch_layout(to_dev(d["topk_idx"]), cfg.E, cfg.R)
    D_e = int(lay.expert_offset[-1].item())
    cap = D_e - 37
    ex = torch.zeros((cap, cfg.H), dtype=torch.bfloat16, device="cuda")
    src = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    st = _status()
    x = to_dev_bf16(d["x"])
    ep.ep_dispatch(lay, x, False, None, None, ep._recv_struct(ex, None, src), st)
    assert status_value(st) & ep.EP_ST_CAPACITY
    ref = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], cfg.E, cfg.R, False, exp_cap=cap)
    assert np.array_equal(u16(ex), ref["exp_x"])


# ----------------------------------------------------------------- combine ----
def _expert_outputs(n_rows, H, seed):
    z = ei.normal(ei.stream_key(seed, 500), n_rows * H).astype(np.float32) * 3.0
    return ei.bf16_bits_from_f32(z).reshape(n_rows, H)


# Batches of at least eight blocks per SM (1216 tokens on 152 SMs) split the
# last partial wave's tokens into spans: 1500 and 2500 tokens (ragged spans at
# H 7296), 1217 (a one-token tail of two spans at H 1032), 2432 (no tail).
@pytest.mark.parametrize("c,N,H", [(3, 1000, 7168), (4, 777, 7168), (5, 1500, 4096), (4, 129, 8),
                                   (5, 100, 1032), (4, 2500, 7296), (3, 1217, 1032), (3, 2432, 7168)])
def test_combine_parity(c, N, H):
    cfg = ei.WORKLOADS[c].scaled(N=N, H=H)
    idx, w = ei.make_routing(cfg, seed=c + 10)
    lay_ref = oracle.layout(idx, cfg.E, cfg.R)
    D_e = int(lay_ref["expert_offset"][-1])
    y = _expert_outputs(D_e, H, seed=c)
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(idx), cfg.E, cfg.R, status=st)
    out = ep.combine(to_dev_bf16(y), lay, to_dev(w), status=st)
    ref, _ = oracle.combine(y, lay_ref["expert_slot"], w)
    got = u16(out)
    assert bf16_ulp_diff(got, ref).max() <= 1
    assert np.array_equal(got, ref)
    assert status_value(st) == 0


def test_combine_identity_round_trip():
    cfg = ei.WORKLOADS[4].scaled(N=600, H=2048)
    d = ei.make_inputs(cfg, seed=5)
    lay = ep.get_dispatch_layout(to_dev(d["topk_idx"]), cfg.E, cfg.R)
    x = to_dev_bf16(d["x"])
    res = ep.dispatch(x, lay, with_rank=False, exact=True)
    out = ep.combine(res.expert_x, lay, to_dev(d["topk_weights"]))
    xf = oracle.f32_from_bf16(d["x"]).astype(np.float64)
    of = oracle.f32_from_bf16(u16(out)).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(xf), 2.0 ** -126))) - 7)
    assert np.all(np.abs(of - xf) <= ulp)


def test_combine_masked_and_capacity():
    idx = np.array([[-1, -1], [0, -1], [1, 0]], np.int32)
    w = np.array([[1, 1], [2, 0], [0.5, 0.25]], np.float32)
    y = ei.bf16_bits_from_f32(np.array([[1, 2, 3, 4, 5, 6, 7, 8], [8, 7, 6, 5, 4, 3, 2, 1]], np.float32))
    lay = ep.get_dispatch_layout(to_dev(idx), 2, 1)
    out = ep.combine(to_dev_bf16(y), lay, to_dev(w))
    ref, _ = oracle.combine(y, oracle.layout(idx, 2, 1)["expert_slot"], w)
    assert np.array_equal(u16(out), ref)
    assert np.all(u16(out)[0] == 0)  # +0 for a token with every slot masked
    st = _status()
    out = torch.empty((3, 8), dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(lay, to_dev_bf16(y)[:1], to_dev(w), out, st)
    assert status_value(st) & ep.EP_ST_CAPACITY


# ------------------------------------------------------------ low latency ----
@pytest.mark.parametrize("c,n_s,H,T", [(1, 16, 7168, 16), (1, 5, 256, 128), (2, 16, 512, 128),
                                       (2, 128, 1024, 128)])
def test_ll_dispatch_parity(c, n_s, H, T):
    # T only sizes the fixed regions (packed rows do not depend on it); the
    # full-width case uses a small T so the oracle's host buffers stay small.
    base = ei.WORKLOADS[c]
    cfg = base.scaled(N=base.R * n_s, H=H, T=T)
    use_fp8 = cfg.fp8
    d = ei.make_inputs(cfg, seed=c + n_s)
    st = _status()
    x = to_dev_bf16(d["x"])
    recv, cnt, handle, hook = ep.low_latency_dispatch(x, to_dev(d["topk_idx"]), cfg.T, cfg.E, cfg.R,
                                                      use_fp8=use_fp8, status=st)
    hook()
    ref = oracle.ll_dispatch(d["x"], d["topk_idx"], cfg.E, cfg.R, cfg.T, use_fp8)
    cnt = cnt.cpu().numpy()
    assert np.array_equal(cnt, ref["recv_count"])
    assert np.array_equal(handle.layout_range.cpu().numpy(), ref["layout_range"])
    rx, rs = recv if use_fp8 else (recv, None)
    gx = u8(rx) if use_fp8 else u16(rx)
    src = handle.recv_src.cpu().numpy()
    for e in range(cfg.E):
        n = cnt[e]
        assert np.array_equal(gx[e, :n], ref["recv_x"][e, :n])
        assert np.array_equal(src[e, :n], ref["recv_src"][e, :n])
        if use_fp8:
            assert np.array_equal(rs[e, :n].cpu().numpy(), ref["recv_scales"][e, :n])
    assert status_value(st) == 0
    # combine: experts y = x (dequantised for FP8 -> BF16 round trip is not needed: use BF16 copies)
    yb = torch.zeros((cfg.E, cfg.R * cfg.T, H), dtype=torch.bfloat16, device="cuda")
    ref_y = np.zeros((cfg.E, cfg.R * cfg.T, H), np.uint16)
    z = _expert_outputs(cfg.E * cfg.R * cfg.T, H, seed=c).reshape(cfg.E, cfg.R * cfg.T, H)
    for e in range(cfg.E):
        ref_y[e, :cnt[e]] = z[e, :cnt[e]]
    yb.copy_(to_dev_bf16(ref_y))
    out = ep.low_latency_combine(yb, to_dev(d["topk_weights"]), handle, status=st)
    ref_out, _ = oracle.ll_combine(ref_y, ref["slot_map"], d["topk_weights"])
    got = u16(out)
    assert bf16_ulp_diff(got, ref_out).max() <= 1
    assert np.array_equal(got, ref_out)
    assert status_value(st) == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_empty_batches(fp8):
    """Zero tokens through every call: layout, dispatch and combine of the
    normal path; low-latency send, receive and combine (all counts and ranges
    zero, no status bit)."""
    H, K, E, R, T = 256, 4, 32, 4, 8
    st = _status()
    x0 = torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
    i0 = torch.empty((0, K), dtype=torch.int32, device="cuda")
    w0 = torch.empty((0, K), dtype=torch.float32, device="cuda")
    lay = ep.get_dispatch_layout(i0, E, R, status=st)
    _layout_equal(lay, oracle.layout(np.zeros((0, K), np.int32), E, R))
    ep.dispatch(x0, lay, w0, use_fp8=fp8, status=st)
    out = ep.combine(torch.zeros((1, H), dtype=torch.bfloat16, device="cuda"), lay, w0, status=st)
    assert tuple(out.shape) == (0, H)
    recv, cnt, handle, hook = ep.low_latency_dispatch(x0, i0, T, E, R, use_fp8=fp8, status=st)
    hook()
    assert cnt.cpu().numpy().tolist() == [0] * E
    assert not handle.layout_range.cpu().numpy().any()
    outl = ep.low_latency_combine(torch.zeros((E, R * T, H), dtype=torch.bfloat16, device="cuda"), w0, handle,
                                  status=st)
    assert tuple(outl.shape) == (0, H)
    assert status_value(st) == 0


@pytest.mark.parametrize("E,R,n_s,K", [
    (4, 2, 2, 4),        # 16 entries: the one-launch send
    (1024, 32, 4, 8),    # E * R above the one-launch table: one-CTA layout + dispatch
    (4, 2, 600, 4),      # 4800 entries: the multi-CTA layout + dispatch
])
@pytest.mark.parametrize("fp8", [False, True])
def test_ll_masked_bad_repeated_and_overflow(E, R, n_s, K, fp8):
    """Every low-latency send path against the oracle on a routing with masked
    slots, out-of-range indices and repeated experts, the first half of the
    tokens sending two slots each to expert 0 so that its region (R * T rows)
    overflows: counts, ranges (rows that landed), rows, scales, sources,
    status bits, and the combine (overflowed slots are skipped)."""
    N, H, T = R * n_s, 256, n_s
    idx = _rand_idx(N, K, E, seed=E + n_s + K, p_mask=0.15, distinct=False)
    idx[: N // 2 + 1, 0:2] = 0
    idx[1::5, K - 1] = E
    idx[2::7, K - 2] = -9
    x = ei.make_x(N, H, seed=n_s)
    w = ei.uniform01(ei.stream_key(n_s, 1), N * K).reshape(N, K).astype(np.float32)
    st = _status()
    recv, cnt, handle, hook = ep.low_latency_dispatch(to_dev_bf16(x), to_dev(idx), T, E, R, use_fp8=fp8, status=st)
    hook()
    ref = oracle.ll_dispatch(x, idx, E, R, T, fp8)
    assert ref["status"] == oracle.BAD_INDEX | oracle.LL_OVERFLOW
    assert status_value(st) == ep.EP_ST_BAD_INDEX | ep.EP_ST_LL_OVERFLOW
    cnt = cnt.cpu().numpy()
    assert np.array_equal(cnt, ref["recv_count"])
    assert np.array_equal(handle.layout_range.cpu().numpy(), ref["layout_range"])
    landed = np.minimum(cnt, R * T)
    rx, rs = recv if fp8 else (recv, None)
    gx = u8(rx) if fp8 else u16(rx)
    src = handle.recv_src.cpu().numpy()
    for e in range(E):
        n = landed[e]
        assert np.array_equal(gx[e, :n], ref["recv_x"][e, :n]), e
        assert np.array_equal(src[e, :n], ref["recv_src"][e, :n]), e
        if fp8:
            assert np.array_equal(rs[e, :n].cpu().numpy(), ref["recv_scales"][e, :n]), e
    y = _expert_outputs(E * R * T, H, seed=E).reshape(E, R * T, H)
    st = _status()
    out = ep.low_latency_combine(to_dev_bf16(y), to_dev(w), handle, status=st)
    ref_out, _ = oracle.ll_combine(y, ref["slot_map"], w)
    assert np.array_equal(u16(out), ref_out)
    assert status_value(st) == 0


def test_ll_receive_without_send_and_mismatch():
    cfg = ei.WORKLOADS[1].scaled(H=256)
    N, K, E, R, T = cfg.N, cfg.K, cfg.E, cfg.R, cfg.T
    ws = torch.zeros(ep.ep_ll_workspace_bytes(N, K, E, R, T), dtype=torch.uint8, device="cuda")
    cnt = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    st = _status()
    ep.ep_ll_dispatch_recv(ws, N, K, E, R, T, cnt, None, st)
    assert status_value(st) & ep.EP_ST_NOT_SENT
    assert torch.all(cnt == -7)
    # a proper send, then two receives: the second has no matching send
    d = ei.make_inputs(cfg, seed=1)
    recv, cnt2, handle, hook = ep.low_latency_dispatch(to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), T, E, R,
                                                       use_fp8=False, workspace=ws)
    st = _status()
    hook()
    assert status_value(st) == 0
    hook_st = _status()
    ep.ep_ll_dispatch_recv(ws, N, K, E, R, T, cnt, None, hook_st)
    assert status_value(hook_st) & ep.EP_ST_NOT_SENT
    # mismatched shapes against the workspace of that send
    st = _status()
    ep.ep_ll_combine(recv, to_dev(d["topk_weights"]), ws, N, K, 256, E, R, 64,
                     torch.empty((N, 256), dtype=torch.bfloat16, device="cuda"), st)
    assert status_value(st) & ep.EP_ST_MISMATCH


def test_ll_capacity_is_a_host_error():
    cfg = ei.WORKLOADS[1].scaled(H=256, N=8 * 20)
    d = ei.make_inputs(cfg, seed=1)
    with pytest.raises(ep.EPError) as ei_:
        ep.low_latency_dispatch(to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), 16, cfg.E, cfg.R, use_fp8=False)
    assert ei_.value.code == ep.EP_ERR_LL_CAPACITY


def test_ll_hook_on_another_stream_ordered_by_event():
    cfg = ei.WORKLOADS[1].scaled(H=512)
    d = ei.make_inputs(cfg, seed=6)
    x = to_dev_bf16(d["x"])
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        recv, cnt, handle, hook = ep.low_latency_dispatch(x, to_dev(d["topk_idx"]), cfg.T, cfg.E, cfg.R,
                                                          use_fp8=False)
        ev = torch.cuda.Event()
        ev.record(s1)
    s2.wait_event(ev)
    with torch.cuda.stream(s2):
        hook()
    torch.cuda.synchronize()
    ref = oracle.layout(d["topk_idx"], cfg.E, cfg.R)
    assert np.array_equal(cnt.cpu().numpy(), ref["num_tokens_per_expert"])


# -------------------------------------------------------------- encoders ----
def test_e4m3_encoder_exhaustive():
    """Every fp32 bit pattern through the device encoder vs the oracle's encoder."""
    chunk = 1 << 28
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    for c in range((1 << 32) // chunk):
        start = c * chunk - ((1 << 32) if c * chunk >= (1 << 31) else 0)  # as signed int32
        f = torch.arange(start, start + chunk, dtype=torch.int32, device="cuda").view(torch.float32)
        ep.ep_fp8_e4m3_encode(f, out)
        got = out.cpu().numpy()
        fh = f.cpu().numpy()
        ref = oracle.e4m3_from_f32(fh)
        nan = np.isnan(fh)
        assert np.array_equal(got[~nan], ref[~nan]), c
        assert np.all((got[nan] & 0x7F) == 0x7F), c
