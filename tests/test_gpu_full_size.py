"""Whole-array parity at the full sizes of the five workloads, through the C ABI.

Every output array of every step is compared with the CPU oracle on the same
seeded inputs, in the launch configuration bench.py times (worst-case receive
capacities, the low-latency path's fixed [E, R*T, H] buffers):

* layout: counts, offsets, the per-rank mask, rank and expert slots;
* dispatch: per-rank rows, scales, source tokens, local top-k ids and
  weights; expert-major rows, scales and source slots;
* combine: the [N, H] output, against the oracle's fp32 fused multiply-add
  chain (bar: 1 BF16 step; asserted bit-exact);
* low latency: receive counts, the per-(expert, source rank) ranges, every
  received row (j < count) of every expert with its scales and source
  token, and the combine output against the oracle's low-latency combine.

Expert outputs fed to combine are rows of x picked by a seeded draw (input
generation only), so each routed slot carries a different row.
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


def _picked_rows(x: np.ndarray, n_rows: int, seed: int) -> np.ndarray:
    """n_rows BF16 rows of x chosen by a seeded draw: stand-in expert outputs."""
    pick = ei.splitmix64(ei.stream_key(seed, 700), n_rows) % np.uint64(x.shape[0])
    return x[pick.astype(np.int64)]


def _check_layout(lay, ref):
    for k in LAYOUT_KEYS:
        assert np.array_equal(getattr(lay, k).cpu().numpy(), ref[k]), k


def _check_dispatch_whole(res, ref, fp8):
    conv = u8 if fp8 else u16
    D_e, D_r = ref["exp_x"].shape[0], ref["rank_x"].shape[0]
    assert np.array_equal(conv(res.expert_x[:D_e]), ref["exp_x"]), "expert rows"
    assert np.array_equal(res.expert_src[:D_e].cpu().numpy(), ref["exp_src"]), "expert src"
    assert np.array_equal(conv(res.rank_x[:D_r]), ref["rank_x"]), "rank rows"
    assert np.array_equal(res.rank_src[:D_r].cpu().numpy(), ref["rank_src"]), "rank src"
    assert np.array_equal(res.rank_topk_idx[:D_r].cpu().numpy(), ref["rank_topk_idx"]), "rank top-k ids"
    assert np.array_equal(res.rank_topk_weights[:D_r].cpu().numpy(), ref["rank_topk_weights"]), "rank weights"
    if fp8:
        assert np.array_equal(res.expert_scales[:D_e].cpu().numpy(), ref["exp_scales"]), "expert scales"
        assert np.array_equal(res.rank_scales[:D_r].cpu().numpy(), ref["rank_scales"]), "rank scales"


@pytest.mark.parametrize("c", [3, 4, 5])
def test_full_size_normal_whole_arrays(c):
    cfg = ei.WORKLOADS[c]
    d = ei.make_inputs(cfg, seed=0)
    x, idx, w = to_dev_bf16(d["x"]), to_dev(d["topk_idx"]), to_dev(d["topk_weights"])
    ref_lay = oracle.layout(d["topk_idx"], cfg.E, cfg.R)
    ref = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], cfg.E, cfg.R, cfg.fp8, lay=ref_lay)
    assert ref["status"] == 0

    # Two calls: layout, then dispatch into worst-case buffers.
    st = _status()
    lay = ep.get_dispatch_layout(idx, cfg.E, cfg.R, status=st)
    _check_layout(lay, ref_lay)
    res = ep.dispatch(x, lay, w, use_fp8=cfg.fp8, status=st)
    _check_dispatch_whole(res, ref, cfg.fp8)
    assert status_value(st) == 0
    del res

    # One call: the dispatch as the layout's programmatic dependent.
    st = _status()
    lay2, res2 = ep.get_layout_and_dispatch(x, idx, cfg.E, cfg.R, w, use_fp8=cfg.fp8, status=st)
    _check_layout(lay2, ref_lay)
    _check_dispatch_whole(res2, ref, cfg.fp8)
    assert status_value(st) == 0
    del res2, lay2
    D_e = ref["exp_x"].shape[0]
    del ref
    torch.cuda.empty_cache()

    # Combine of D_e stand-in expert rows in the expert-major layout.
    y = _picked_rows(d["x"], D_e, seed=c)
    st = _status()
    out = ep.combine(to_dev_bf16(y), lay, w, status=st)
    ref_out, ref_st = oracle.combine(y, ref_lay["expert_slot"], d["topk_weights"])
    got = u16(out)
    assert ref_st == 0 and status_value(st) == 0
    assert bf16_ulp_diff(got, ref_out).max() <= 1
    assert np.array_equal(got, ref_out)


@pytest.mark.parametrize("c", [1, 2])
def test_full_size_low_latency_whole_arrays(c):
    cfg = ei.WORKLOADS[c]
    N, H, K, E, R, T = cfg.N, cfg.H, cfg.K, cfg.E, cfg.R, cfg.T
    RT = R * T
    d = ei.make_inputs(cfg, seed=0)
    # The oracle's fixed-shape buffers are zero-filled lazily by the OS; only
    # the received rows are ever written or read.
    ref = oracle.ll_dispatch(d["x"], d["topk_idx"], E, R, T, cfg.fp8)
    assert ref["status"] == 0

    st = _status()
    x, w = to_dev_bf16(d["x"]), to_dev(d["topk_weights"])
    recv, cnt, handle, hook = ep.low_latency_dispatch(x, to_dev(d["topk_idx"]), T, E, R, use_fp8=cfg.fp8,
                                                      status=st)
    hook()
    cnt_h = cnt.cpu().numpy()
    assert np.array_equal(cnt_h, ref["recv_count"])
    assert np.array_equal(handle.layout_range.cpu().numpy(), ref["layout_range"])
    rows = np.concatenate([e * RT + np.arange(cnt_h[e], dtype=np.int64) for e in range(E)])
    assert rows.size == int(cnt_h.sum())
    rows_d = torch.from_numpy(rows).cuda()
    rx, rs = recv if cfg.fp8 else (recv, None)
    got_x = rx.view(E * RT, H).index_select(0, rows_d)
    ref_x = ref["recv_x"].reshape(E * RT, H)[rows]
    assert np.array_equal(u8(got_x) if cfg.fp8 else u16(got_x), ref_x), "received rows"
    assert np.array_equal(handle.recv_src.view(-1).index_select(0, rows_d).cpu().numpy(),
                          ref["recv_src"].reshape(-1)[rows]), "received source tokens"
    if cfg.fp8:
        got_s = rs.view(E * RT, H // 128).index_select(0, rows_d).cpu().numpy()
        assert np.array_equal(got_s, ref["recv_scales"].reshape(E * RT, H // 128)[rows]), "received scales"
    assert status_value(st) == 0
    del got_x, recv, rx, rs
    torch.cuda.empty_cache()

    # Combine of BF16 stand-in expert outputs placed at the received rows.
    yv = _picked_rows(d["x"], rows.size, seed=10 + c)
    y = torch.zeros((E, RT, H), dtype=torch.bfloat16, device="cuda")
    y.view(E * RT, H).index_copy_(0, rows_d, to_dev_bf16(yv))
    out = ep.low_latency_combine(y, w, handle, status=st)
    ref_y = np.zeros((E, RT, H), np.uint16)
    ref_y.reshape(E * RT, H)[rows] = yv
    ref_out, ref_st = oracle.ll_combine(ref_y, ref["slot_map"], d["topk_weights"])
    got = u16(out)
    assert ref_st == 0 and status_value(st) == 0
    assert bf16_ulp_diff(got, ref_out).max() <= 1
    assert np.array_equal(got, ref_out)
