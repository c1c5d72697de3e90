"""GPU parity of the rows built after the hot path: the two-phase low-latency
combine and CUDA-graph capture of the low-latency and the normal paths."""
import numpy as np
import pytest
import torch

import combine_ep_get_dispatch_gb300 as ep
import epinputs as ei
import oracle
from helpers import status_value, to_dev, to_dev_bf16, u16, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _expert_outputs(shape, seed):
    n = int(np.prod(shape))
    z = ei.normal(ei.stream_key(seed, 600), n).astype(np.float32) * 2.0
    return ei.bf16_bits_from_f32(z).reshape(shape)


@pytest.mark.parametrize("c,n_s,H", [(1, 16, 7168), (2, 16, 1024)])
def test_two_phase_ll_combine(c, n_s, H):
    # T = 32 only sizes the fixed regions (rows are packed from 0), and keeps
    # the host copy of the [E, R*T, H] expert outputs small.
    cfg = ei.WORKLOADS[c].scaled(N=ei.WORKLOADS[c].R * n_s, H=H, T=32)
    d = ei.make_inputs(cfg, seed=c + 20)
    st = _status()
    recv, cnt, handle, hook = ep.low_latency_dispatch(to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), cfg.T, cfg.E,
                                                      cfg.R, use_fp8=cfg.fp8, status=st)
    hook()
    ref = oracle.ll_dispatch(d["x"], d["topk_idx"], cfg.E, cfg.R, cfg.T, False)
    y = _expert_outputs((cfg.E, cfg.R * cfg.T, H), seed=c)
    w = to_dev(d["topk_weights"])
    out, chook = ep.low_latency_combine(to_dev_bf16(y), w, handle, status=st, return_recv_hook=True)
    chook()
    one = ep.low_latency_combine(to_dev_bf16(y), w, handle, status=st)
    want = oracle.ll_combine_recv(oracle.ll_combine_send(y, ref["slot_map"])[0], ref["slot_map"],
                                  d["topk_weights"])
    assert np.array_equal(u16(out), want)
    assert np.array_equal(u16(one), want)
    assert status_value(st) == 0


def test_ll_path_in_a_cuda_graph():
    """send + receive + combine captured once, replayed on two batches."""
    cfg = ei.WORKLOADS[1].scaled(H=2048)
    N, H, K, E, R, T = cfg.N, cfg.H, cfg.K, cfg.E, cfg.R, cfg.T
    x = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((N, K), dtype=torch.int32, device="cuda")
    w = torch.empty((N, K), dtype=torch.float32, device="cuda")
    ws = torch.zeros(ep.ep_ll_workspace_bytes(N, K, E, R, T), dtype=torch.uint8, device="cuda")
    recv_x = torch.empty((E, R * T, H), dtype=torch.bfloat16, device="cuda")
    recv_src = torch.empty((E, R * T), dtype=torch.int32, device="cuda")
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    rng = torch.empty((E, R), dtype=torch.int64, device="cuda")
    out = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    st = _status()

    def step():
        ep.ep_ll_dispatch_send(x, idx, H, E, R, T, False, recv_x, None, recv_src, ws, st)
        ep.ep_ll_dispatch_recv(ws, N, K, E, R, T, cnt, rng, st)
        ep.ep_ll_combine(recv_x, w, ws, N, K, H, E, R, T, out, st)

    d0 = ei.make_inputs(cfg, seed=30)
    x.copy_(to_dev_bf16(d0["x"])); idx.copy_(to_dev(d0["topk_idx"])); w.copy_(to_dev(d0["topk_weights"]))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (31, 32):
        d = ei.make_inputs(cfg, seed=seed)
        x.copy_(to_dev_bf16(d["x"])); idx.copy_(to_dev(d["topk_idx"])); w.copy_(to_dev(d["topk_weights"]))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.ll_dispatch(d["x"], d["topk_idx"], E, R, T, False)
        assert np.array_equal(cnt.cpu().numpy(), ref["recv_count"])
        ref_out, _ = oracle.ll_combine(ref["recv_x"], ref["slot_map"], d["topk_weights"])
        assert np.array_equal(u16(out), ref_out)
    assert status_value(st) == 0


def test_normal_path_in_a_cuda_graph():
    """layout + dispatch (worst-case capacities) + combine captured once, replayed on two batches."""
    cfg = ei.WORKLOADS[3].scaled(N=512, H=1024)
    N, H, K, E, R = cfg.N, cfg.H, cfg.K, cfg.E, cfg.R
    x = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((N, K), dtype=torch.int32, device="cuda")
    w = torch.empty((N, K), dtype=torch.float32, device="cuda")
    lay = ep.new_layout(idx, E, R)
    ws = torch.zeros(ep.ep_layout_workspace_bytes(N, K, E, R), dtype=torch.uint8, device="cuda")
    ex = torch.empty((N * K, H), dtype=torch.uint8, device="cuda")
    es = torch.empty((N * K, H // 128), dtype=torch.float32, device="cuda")
    ysrc = torch.empty((N * K, H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    st = _status()

    def step():
        ep.ep_get_dispatch_layout(lay, ws, st)
        ep.ep_dispatch(lay, x, True, w, None, ep._recv_struct(ex, es, None), st)
        ep.ep_dispatch(lay, x, False, w, None, ep._recv_struct(ysrc, None, None), st)
        ep.ep_combine(lay, ysrc, w, out, st)

    d0 = ei.make_inputs(cfg, seed=40)
    x.copy_(to_dev_bf16(d0["x"])); idx.copy_(to_dev(d0["topk_idx"])); w.copy_(to_dev(d0["topk_weights"]))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (41, 42):
        d = ei.make_inputs(cfg, seed=seed)
        x.copy_(to_dev_bf16(d["x"])); idx.copy_(to_dev(d["topk_idx"])); w.copy_(to_dev(d["topk_weights"]))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], E, R, True, with_rank=False)
        D_e = ref["exp_x"].shape[0]
        assert np.array_equal(u8(ex[:D_e]), ref["exp_x"])
        assert np.array_equal(es[:D_e].cpu().numpy(), ref["exp_scales"])
        ref_out, _ = oracle.combine(u16(ysrc[:D_e]), ref["layout"]["expert_slot"], d["topk_weights"])
        assert np.array_equal(u16(out), ref_out)
        assert np.array_equal(lay.expert_slot.cpu().numpy(), ref["layout"]["expert_slot"])
    assert status_value(st) == 0


def test_layout_dispatch_pair_in_a_cuda_graph():
    """ep_layout_dispatch (a programmatic-dependent pair of launches) + combine
    captured once, replayed on two batches."""
    cfg = ei.WORKLOADS[5].scaled(N=700, H=1024)
    N, H, K, E, R = cfg.N, cfg.H, cfg.K, cfg.E, cfg.R
    x = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((N, K), dtype=torch.int32, device="cuda")
    w = torch.empty((N, K), dtype=torch.float32, device="cuda")
    lay = ep.new_layout(idx, E, R)
    ws = torch.zeros(ep.ep_layout_workspace_bytes(N, K, E, R), dtype=torch.uint8, device="cuda")
    rx = torch.empty((N * min(K, R), H), dtype=torch.uint8, device="cuda")
    rs = torch.empty((N * min(K, R), H // 128), dtype=torch.float32, device="cuda")
    rsrc = torch.empty(N * min(K, R), dtype=torch.int32, device="cuda")
    ex = torch.empty((N * K, H), dtype=torch.uint8, device="cuda")
    es = torch.empty((N * K, H // 128), dtype=torch.float32, device="cuda")
    y = torch.empty((N * K, H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    st = _status()

    def step():
        ep.ep_layout_dispatch(lay, ws, x, True, w, ep._recv_struct(rx, rs, rsrc), ep._recv_struct(ex, es, None), st)
        ep.ep_combine(lay, y, w, out, st)

    y.copy_(to_dev_bf16(_expert_outputs((N * K, H), 7)))
    d0 = ei.make_inputs(cfg, seed=50)
    x.copy_(to_dev_bf16(d0["x"])); idx.copy_(to_dev(d0["topk_idx"])); w.copy_(to_dev(d0["topk_weights"]))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (51, 52):
        d = ei.make_inputs(cfg, seed=seed)
        x.copy_(to_dev_bf16(d["x"])); idx.copy_(to_dev(d["topk_idx"])); w.copy_(to_dev(d["topk_weights"]))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], E, R, True)
        D_e, D_r = ref["exp_x"].shape[0], ref["rank_x"].shape[0]
        assert np.array_equal(u8(ex[:D_e]), ref["exp_x"])
        assert np.array_equal(es[:D_e].cpu().numpy(), ref["exp_scales"])
        assert np.array_equal(u8(rx[:D_r]), ref["rank_x"])
        assert np.array_equal(rs[:D_r].cpu().numpy(), ref["rank_scales"])
        assert np.array_equal(rsrc[:D_r].cpu().numpy(), ref["rank_src"])
        ref_out, _ = oracle.combine(u16(y), ref["layout"]["expert_slot"], d["topk_weights"])
        assert np.array_equal(u16(out), ref_out)
    assert status_value(st) == 0


def test_overlapped_launches_back_to_back():
    """Ten low-latency steps and ten one-call layout + dispatch + combine steps
    enqueued back to back on one stream (new inputs and outputs each step, no
    host synchronisation between them): every step matches the oracle. Each
    step's layout starts behind the previous step's combine, and its dispatch
    starts early behind the layout (programmatic dependent launch)."""
    steps = 10
    st = _status()
    # low latency
    cfg = ei.WORKLOADS[1].scaled(H=1024)
    N, H, K, E, R, T = cfg.N, cfg.H, cfg.K, cfg.E, cfg.R, cfg.T
    ins = [ei.make_inputs(cfg, seed=70 + i) for i in range(steps)]
    xs = [to_dev_bf16(d["x"]) for d in ins]
    ids = [to_dev(d["topk_idx"]) for d in ins]
    ws_ = [to_dev(d["topk_weights"]) for d in ins]
    ws = torch.zeros(ep.ep_ll_workspace_bytes(N, K, E, R, T), dtype=torch.uint8, device="cuda")
    recv = [torch.empty((E, R * T, H), dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    src = torch.empty((E, R * T), dtype=torch.int32, device="cuda")
    cnt = [torch.empty(E, dtype=torch.int32, device="cuda") for _ in range(steps)]
    outs = [torch.empty((N, H), dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    for i in range(steps):
        ep.ep_ll_dispatch_send(xs[i], ids[i], H, E, R, T, False, recv[i], None, src, ws, st)
        ep.ep_ll_dispatch_recv(ws, N, K, E, R, T, cnt[i], None, st)
        ep.ep_ll_combine(recv[i], ws_[i], ws, N, K, H, E, R, T, outs[i], st)
    torch.cuda.synchronize()
    for i, d in enumerate(ins):
        ref = oracle.ll_dispatch(d["x"], d["topk_idx"], E, R, T, False)
        c = cnt[i].cpu().numpy()
        assert np.array_equal(c, ref["recv_count"])
        got = u16(recv[i])
        for e in range(E):
            assert np.array_equal(got[e, :c[e]], ref["recv_x"][e, :c[e]])
        ref_out, _ = oracle.ll_combine(ref["recv_x"], ref["slot_map"], d["topk_weights"])
        assert np.array_equal(u16(outs[i]), ref_out)
    # normal mode, layout + FP8 dispatch in one call, then combine of the BF16 rows
    cfg = ei.WORKLOADS[3].scaled(N=300, H=512)
    N, H, K, E, R = cfg.N, cfg.H, cfg.K, cfg.E, cfg.R
    ins = [ei.make_inputs(cfg, seed=80 + i) for i in range(steps)]
    ws = torch.zeros(ep.ep_layout_workspace_bytes(N, K, E, R), dtype=torch.uint8, device="cuda")
    y = torch.empty((N * K, H), dtype=torch.bfloat16, device="cuda")
    y.copy_(to_dev_bf16(_expert_outputs((N * K, H), 9)))
    res = []
    for d in ins:
        idx = to_dev(d["topk_idx"])
        lay = ep.new_layout(idx, E, R)
        ex = torch.empty((N * K, H), dtype=torch.uint8, device="cuda")
        es = torch.empty((N * K, H // 128), dtype=torch.float32, device="cuda")
        out = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
        ep.ep_layout_dispatch(lay, ws, to_dev_bf16(d["x"]), True, to_dev(d["topk_weights"]), None,
                              ep._recv_struct(ex, es, None), st)
        ep.ep_combine(lay, y, to_dev(d["topk_weights"]), out, st)
        res.append((lay, ex, es, out))
    torch.cuda.synchronize()
    for d, (lay, ex, es, out) in zip(ins, res):
        ref = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], E, R, True, with_rank=False)
        D_e = ref["exp_x"].shape[0]
        assert np.array_equal(u8(ex[:D_e]), ref["exp_x"])
        assert np.array_equal(es[:D_e].cpu().numpy(), ref["exp_scales"])
        ref_out, _ = oracle.combine(u16(y), ref["layout"]["expert_slot"], d["topk_weights"])
        assert np.array_equal(u16(out), ref_out)
    assert status_value(st) == 0


@pytest.mark.parametrize("round_scale,ue8m0", [(True, False), (False, True)])
def test_dispatch_power_of_two_and_ue8m0_scales(round_scale, ue8m0):
    cfg = ei.WORKLOADS[5].scaled(N=700, H=4096)
    d = ei.make_inputs(cfg, seed=50)
    # a few tokens with tiny magnitudes exercise the UE8M0 floor of 2^-127
    x = d["x"].copy()
    x[3, :128] = 0x0001
    x[4, :] = 0
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(d["topk_idx"]), cfg.E, cfg.R, status=st)
    res = ep.dispatch(to_dev_bf16(x), lay, to_dev(d["topk_weights"]), use_fp8=True, exact=True, status=st,
                      round_scale=round_scale, use_ue8m0=ue8m0)
    ref = oracle.dispatch(x, d["topk_idx"], d["topk_weights"], cfg.E, cfg.R, True, round_scale=round_scale,
                          ue8m0=ue8m0)
    assert np.array_equal(u8(res.expert_x), ref["exp_x"]) and np.array_equal(u8(res.rank_x), ref["rank_x"])
    got_s = res.expert_scales.cpu().numpy()
    assert got_s.dtype == (np.uint8 if ue8m0 else np.float32)
    assert np.array_equal(got_s, ref["exp_scales"]) and np.array_equal(res.rank_scales.cpu().numpy(),
                                                                         ref["rank_scales"])
    assert status_value(st) == 0


def test_ll_ue8m0_and_cumulative_receive_stats():
    cfg = ei.WORKLOADS[2].scaled(N=32 * 16, H=1024)
    stats = torch.zeros(cfg.E, dtype=torch.int32, device="cuda")
    total = np.zeros(cfg.E, np.int64)
    for seed in (60, 61):
        d = ei.make_inputs(cfg, seed=seed)
        st = _status()
        (rx, rs), cnt, handle, hook = ep.low_latency_dispatch(
            to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), cfg.T, cfg.E, cfg.R, use_fp8=True, use_ue8m0=True,
            status=st, cumulative_local_expert_recv_stats=stats)
        hook()
        ref = oracle.ll_dispatch(d["x"], d["topk_idx"], cfg.E, cfg.R, cfg.T, True, ue8m0=True)
        c = cnt.cpu().numpy()
        assert np.array_equal(c, ref["recv_count"])
        gx, gs = u8(rx), rs.cpu().numpy()
        for e in range(cfg.E):
            assert np.array_equal(gx[e, :c[e]], ref["recv_x"][e, :c[e]])
            assert np.array_equal(gs[e, :c[e]], ref["recv_scales"][e, :c[e]])
        total += c
        assert np.array_equal(stats.cpu().numpy(), total)
        assert status_value(st) == 0


def test_combine_with_shared_expert_bias():
    cfg = ei.WORKLOADS[3].scaled(N=600, H=2048)
    idx, w = ei.make_routing(cfg, seed=70)
    lay_ref = oracle.layout(idx, cfg.E, cfg.R)
    D_e = int(lay_ref["expert_offset"][-1])
    y = _expert_outputs((D_e, cfg.H), seed=70)
    bias = _expert_outputs((cfg.N, cfg.H), seed=71)
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(idx), cfg.E, cfg.R, status=st)
    out = ep.combine(to_dev_bf16(y), lay, to_dev(w), status=st, bias=to_dev_bf16(bias))
    ref, _ = oracle.combine(y, lay_ref["expert_slot"], w, bias)
    assert np.array_equal(u16(out), ref)
    # low latency, one launch and two phases
    lcfg = ei.WORKLOADS[1].scaled(H=1024)
    d = ei.make_inputs(lcfg, seed=72)
    recv, cnt, handle, hook = ep.low_latency_dispatch(to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), lcfg.T, lcfg.E,
                                                      lcfg.R, use_fp8=False, status=st)
    hook()
    lref = oracle.ll_dispatch(d["x"], d["topk_idx"], lcfg.E, lcfg.R, lcfg.T, False)
    b2 = _expert_outputs((lcfg.N, lcfg.H), seed=73)
    one = ep.low_latency_combine(recv, to_dev(d["topk_weights"]), handle, status=st, bias=to_dev_bf16(b2))
    two, h2 = ep.low_latency_combine(recv, to_dev(d["topk_weights"]), handle, status=st, bias=to_dev_bf16(b2),
                                     return_recv_hook=True)
    h2()
    want, _ = oracle.combine(lref["recv_x"].reshape(-1, lcfg.H), lref["slot_map"], d["topk_weights"], b2)
    assert np.array_equal(u16(one), want) and np.array_equal(u16(two), want)
    assert status_value(st) == 0


@pytest.mark.parametrize("A,fp8,ue8m0", [(128, False, False), (128, True, False), (2, True, True)])
def test_aligned_expert_layout_and_zero_padding(A, fp8, ue8m0):
    cfg = ei.WORKLOADS[5].scaled(N=900, H=1024)
    d = ei.make_inputs(cfg, seed=80)
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(d["topk_idx"]), cfg.E, cfg.R, status=st, expert_alignment=A)
    ref_lay = oracle.layout(d["topk_idx"], cfg.E, cfg.R, expert_alignment=A)
    for k in ("num_tokens_per_expert", "expert_offset", "expert_slot", "rank_slot", "rank_offset"):
        assert np.array_equal(getattr(lay, k).cpu().numpy(), ref_lay[k]), k
    D_e = int(ref_lay["expert_offset"][-1])
    # poison the buffers so the zero padding is visible
    res = ep.dispatch(to_dev_bf16(d["x"]), lay, to_dev(d["topk_weights"]), use_fp8=fp8, with_rank=False,
                      status=st, use_ue8m0=ue8m0)
    ref = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], cfg.E, cfg.R, fp8, lay=ref_lay,
                          with_rank=False, ue8m0=ue8m0)
    conv = u8 if fp8 else u16
    assert np.array_equal(conv(res.expert_x[:D_e]), ref["exp_x"])
    assert np.array_equal(res.expert_src[:D_e].cpu().numpy(), ref["exp_src"])
    if fp8:
        assert np.array_equal(res.expert_scales[:D_e].cpu().numpy(), ref["exp_scales"])
    # combine still reads the real rows
    y = _expert_outputs((D_e, cfg.H), seed=81)
    out = ep.combine(to_dev_bf16(y), lay, to_dev(d["topk_weights"]), status=st)
    want, _ = oracle.combine(y, ref_lay["expert_slot"], d["topk_weights"])
    assert np.array_equal(u16(out), want)
    assert status_value(st) == 0


def test_two_level_combine_matches_oracle():
    cfg = ei.WORKLOADS[3].scaled(N=800, H=1024)
    idx, w = ei.make_routing(cfg, seed=90)
    lay_ref = oracle.layout(idx, cfg.E, cfg.R)
    D_e = int(lay_ref["expert_offset"][-1])
    y = _expert_outputs((D_e, cfg.H), seed=90)
    bias = _expert_outputs((cfg.N, cfg.H), seed=91)
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(idx), cfg.E, cfg.R, status=st)
    out, rank_rows = ep.combine_two_level(to_dev_bf16(y), lay, to_dev(w), bias=to_dev_bf16(bias), status=st)
    part, _ = oracle.combine_to_ranks(y, idx, lay_ref, w, cfg.E, cfg.R)
    assert np.array_equal(u16(rank_rows), part)
    want, _ = oracle.combine(part, lay_ref["rank_slot"], None, bias)
    assert np.array_equal(u16(out), want)
    assert status_value(st) == 0


def test_dispatch_and_combine_backward():
    cfg = ei.WORKLOADS[4].scaled(N=700, H=2048)
    d = ei.make_inputs(cfg, seed=100)
    idx, w = d["topk_idx"], d["topk_weights"]
    lay_ref = oracle.layout(idx, cfg.E, cfg.R)
    es = lay_ref["expert_slot"]
    D_e = int(lay_ref["expert_offset"][-1])
    st = _status()
    lay = ep.get_dispatch_layout(to_dev(idx), cfg.E, cfg.R, status=st)
    # dispatch backward: unit-weight sum of the row gradients
    g_rows = _expert_outputs((D_e, cfg.H), seed=101)
    gx = ep.dispatch_backward(to_dev_bf16(g_rows), lay, status=st)
    want, _ = oracle.combine(g_rows, es, None)
    assert np.array_equal(u16(gx), want)
    # combine backward
    y = _expert_outputs((D_e, cfg.H), seed=102)
    g = _expert_outputs((cfg.N, cfg.H), seed=103)
    gy, gw = ep.combine_backward(to_dev_bf16(g), lay, to_dev_bf16(y), to_dev(w), status=st)
    ref_gy, ref_gw, _ = oracle.combine_backward(g, y, es, w)
    assert np.array_equal(u16(gy), ref_gy)
    gw = gw.cpu().numpy().astype(np.float64)
    gf = oracle.f32_from_bf16(g).astype(np.float64)
    yf = oracle.f32_from_bf16(y).astype(np.float64)
    bound = np.zeros_like(ref_gw)
    ok = es >= 0
    for t, k in zip(*np.nonzero(ok)):
        bound[t, k] = cfg.H * 2.0 ** -24 * np.abs(gf[t] * yf[es[t, k]]).sum()
    assert np.all(np.abs(gw - ref_gw) <= bound + 1e-30)
    assert np.all(gw[~ok] == 0)
    # deterministic: the same bits on a second run
    gy2, gw2 = ep.combine_backward(to_dev_bf16(g), lay, to_dev_bf16(y), to_dev(w), status=st)
    assert torch.equal(gy, gy2) and np.array_equal(gw, gw2.cpu().numpy().astype(np.float64))
    assert status_value(st) == 0


# ------------------------------------------------- shrink mode (rank masks) ----
def test_shrink_mask_buffer_update_query_clean():
    R = 8
    ws = torch.zeros(ep.ep_ll_workspace_bytes(64, 8, 64, R, 16), dtype=torch.uint8, device="cuda")
    assert ep.low_latency_query_mask_buffer(ws, num_ranks=R).tolist() == [0] * R
    ep.low_latency_update_mask_buffer(ws, 3, num_ranks=R)
    ep.low_latency_update_mask_buffer(ws, 5, num_ranks=R)
    assert ep.low_latency_query_mask_buffer(ws, num_ranks=R).tolist() == [0, 0, 0, 1, 0, 1, 0, 0]
    ep.low_latency_update_mask_buffer(ws, 3, mask=False, num_ranks=R)
    assert ep.low_latency_query_mask_buffer(ws, num_ranks=R).tolist() == [0, 0, 0, 0, 0, 1, 0, 0]
    ep.low_latency_clean_mask_buffer(ws, num_ranks=R)
    assert ep.low_latency_query_mask_buffer(ws, num_ranks=R).tolist() == [0] * R
    with pytest.raises(ep.EPError):
        ep.low_latency_update_mask_buffer(ws, R, num_ranks=R)


@pytest.mark.parametrize("c,n_s,H,T", [(1, 16, 2048, 32), (2, 16, 512, 16)])
def test_shrink_send_and_combine(c, n_s, H, T):
    """Ranks masked before the send drop out of the receive buffers; a rank lost
    between send and combine is skipped by the one- and the two-phase combine."""
    cfg = ei.WORKLOADS[c].scaled(N=ei.WORKLOADS[c].R * n_s, H=H, T=T)
    N, K, E, R, T = cfg.N, cfg.K, cfg.E, cfg.R, cfg.T
    d = ei.make_inputs(cfg, seed=c + 70)
    st = _status()
    ws = torch.zeros(ep.ep_ll_workspace_bytes(N, K, E, R, T), dtype=torch.uint8, device="cuda")
    m_send = np.zeros(R, np.int32)
    m_send[[1, R - 2]] = 1
    for r in np.nonzero(m_send)[0]:
        ep.low_latency_update_mask_buffer(ws, int(r), num_ranks=R)
    recv, cnt, handle, hook = ep.low_latency_dispatch(to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), T, E, R,
                                                      use_fp8=cfg.fp8, status=st, workspace=ws)
    hook()
    ref = oracle.ll_dispatch(d["x"], d["topk_idx"], E, R, T, cfg.fp8, rank_mask=m_send)
    cnt = cnt.cpu().numpy()
    assert np.array_equal(cnt, ref["recv_count"])
    assert cnt.sum() < np.count_nonzero(d["topk_idx"] >= 0)          # something was dropped
    assert np.array_equal(handle.layout_range.cpu().numpy(), ref["layout_range"])
    rx, rs = recv if cfg.fp8 else (recv, None)
    gx = u8(rx) if cfg.fp8 else u16(rx)
    src = handle.recv_src.cpu().numpy()
    for e in range(E):
        n = cnt[e]
        assert np.array_equal(gx[e, :n], ref["recv_x"][e, :n])
        assert np.array_equal(src[e, :n], ref["recv_src"][e, :n])
        if cfg.fp8:
            assert np.array_equal(rs[e, :n].cpu().numpy(), ref["recv_scales"][e, :n])
    # the mask changes before the combine: rank 2 is lost, rank R-2 is back
    m_comb = m_send.copy()
    m_comb[2], m_comb[R - 2] = 1, 0
    ep.low_latency_update_mask_buffer(handle, 2)
    ep.low_latency_update_mask_buffer(handle, R - 2, mask=False)
    assert ep.low_latency_query_mask_buffer(handle).cpu().numpy().tolist() == m_comb.tolist()
    y = _expert_outputs((E, R * T, H), seed=c + 71)
    w = to_dev(d["topk_weights"])
    ref_out, _ = oracle.ll_combine(y, ref["slot_map"], d["topk_weights"], rank_mask=m_comb, R=R)
    out = ep.low_latency_combine(to_dev_bf16(y), w, handle, status=st)
    assert np.array_equal(u16(out), ref_out)
    out2, hook2 = ep.low_latency_combine(to_dev_bf16(y), w, handle, status=st, return_recv_hook=True)
    hook2()
    assert np.array_equal(u16(out2), ref_out)
    # tokens of a masked source rank combine to +0
    toks = np.arange(N).reshape(R, n_s)[[1, 2]].reshape(-1)
    assert np.all(u16(out)[toks] == 0)
    assert status_value(st) == 0
