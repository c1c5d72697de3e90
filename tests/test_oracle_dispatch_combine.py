"""Pins of the oracle's dispatch, combine and low-latency paths.

* Dispatch moves whole rows: every written BF16 row is bit-identical to the
  source token's row, every routed (t, k) and (t, rank) pair is written once
  ("DeepEP Ascend deep dive", "Two Transfers" and "Dispatch's Three Phases").
* The pages' volume example: 16,384 x 7,168 x 2 B x 6 copies, halved by FP8.
* Combine: dispatch -> identity experts -> combine reproduces x (exactly for a
  single expert of weight 1; within one BF16 step when the weights sum to 1);
  with linear experts it matches the dense sum of w * x W_e (the lesson-14
  exercise's check) within the fp32 accumulation bound; a hand-derived case
  fixes the summation order and the fused multiply-add.
* Low-latency: per-expert receive counts equal the layout's counts and the
  packed rows equal the expert-major rows (DeepEP V1 guide 6.1 / 6.3).
"""
import json
import os

import numpy as np
import pytest

import epinputs as ei
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(c, N=None, H=None, **kw):
    cfg = ei.WORKLOADS[c]
    return cfg.scaled(N=N or cfg.N, H=H or cfg.H, **kw)


def _inputs(cfg, seed=0):
    d = ei.make_inputs(cfg, seed)
    return d["x"], d["topk_idx"], d["topk_weights"]


@pytest.mark.parametrize("c,N,H", [(3, 300, 256), (4, 257, 384), (5, 500, 512)])
def test_dispatch_rows_are_source_rows(c, N, H):
    cfg = _small(c, N, H, fp8=False)
    x, idx, w = _inputs(cfg)
    o = oracle.dispatch(x, idx, w, cfg.E, cfg.R, use_fp8=False)
    lay = o["layout"]
    assert o["status"] == 0
    D_e, D_r = int(lay["expert_offset"][-1]), int(lay["rank_offset"][-1])
    assert o["exp_x"].shape == (D_e, H) and o["rank_x"].shape == (D_r, H)
    # each expert row is x[t] with t*K + k its source
    src = o["exp_src"]
    assert np.array_equal(np.sort(src), np.sort(np.nonzero(idx.reshape(-1) >= 0)[0]))
    assert np.array_equal(o["exp_x"], x[src // cfg.K])
    assert np.array_equal(idx.reshape(-1)[src], np.repeat(np.arange(cfg.E), lay["num_tokens_per_expert"]))
    # each rank row is x[t], once per (t, r) in the mask, rank-major then token order
    rsrc = o["rank_src"]
    assert np.array_equal(o["rank_x"], x[rsrc])
    L = cfg.E // cfg.R
    r_of_row = np.repeat(np.arange(cfg.R), lay["num_tokens_per_rank"])
    for r in range(cfg.R):
        toks = rsrc[r_of_row == r]
        assert np.all(np.diff(toks) > 0)
        assert np.array_equal(toks, np.nonzero(lay["is_token_in_rank"][:, r])[0])
    # received top-k: local ids of the experts on that rank, weights carried along
    ti, tw = o["rank_topk_idx"], o["rank_topk_weights"]
    for row in range(0, D_r, 7):
        t, r = rsrc[row], r_of_row[row]
        for k in range(cfg.K):
            e = idx[t, k]
            if e >= 0 and e // L == r:
                assert ti[row, k] == e - r * L and tw[row, k] == w[t, k]
            else:
                assert ti[row, k] == -1 and tw[row, k] == 0


def test_dispatch_fp8_rows_are_quantised_source_rows():
    cfg = _small(3, 200, 512)
    x, idx, w = _inputs(cfg)
    o = oracle.dispatch(x, idx, w, cfg.E, cfg.R, use_fp8=True)
    q, s = oracle.quantize_rows(x)
    t = o["exp_src"] // cfg.K
    assert np.array_equal(o["exp_x"], q[t]) and np.array_equal(o["exp_scales"], s[t])
    assert np.array_equal(o["rank_x"], q[o["rank_src"]])
    assert np.array_equal(o["rank_scales"], s[o["rank_src"]])
    assert o["exp_x"].nbytes * 2 == o["exp_x"].shape[0] * 512 * 2


def test_volume_example():
    g = json.load(open(os.path.join(GOLDEN, "volume_example.json")))
    cfg = ei.WORKLOADS[4]
    assert (cfg.N, cfg.H, cfg.K) == (g["num_tokens"], g["hidden"], g["copies"])
    idx, w = ei.make_routing(cfg, 0)
    lay = oracle.layout(idx, cfg.E, cfg.R)
    D_e = int(lay["expert_offset"][-1])
    assert D_e == cfg.N * cfg.K
    assert D_e * cfg.H * 2 == g["expert_major_bytes_bf16"]
    assert D_e * cfg.H == g["expert_major_bytes_fp8_payload"]
    assert D_e * (cfg.H // 128) * 4 == g["fp8_scale_bytes"]
    # the same rows through the oracle's dispatch (on a 128-wide slice of H)
    o = oracle.dispatch(np.zeros((cfg.N, 128), np.uint16), idx, w, cfg.E, cfg.R, use_fp8=True,
                        lay=lay, with_rank=False)
    assert o["exp_x"].shape[0] * cfg.H == g["expert_major_bytes_fp8_payload"]


def test_dispatch_capacity_overflow_flagged():
    cfg = _small(4, 64, 128)
    x, idx, w = _inputs(cfg)
    lay = oracle.layout(idx, cfg.E, cfg.R)
    D_e = int(lay["expert_offset"][-1])
    o = oracle.dispatch(x, idx, w, cfg.E, cfg.R, False, lay=lay, exp_cap=D_e - 5, rank_cap=10)
    assert o["status"] & oracle.CAPACITY
    assert np.array_equal(o["exp_x"], x[o["exp_src"] // cfg.K])


def test_identity_single_expert_is_exact():
    cfg = _small(4, 300, 512, K=1)
    x, idx, _ = _inputs(cfg)
    w = np.ones_like(idx, dtype=np.float32)
    o = oracle.dispatch(x, idx, w, cfg.E, cfg.R, False, with_rank=False)
    out, st = oracle.combine(o["exp_x"], o["layout"]["expert_slot"], w)
    assert st == 0 and np.array_equal(out, x)


@pytest.mark.parametrize("c", [3, 4])
def test_identity_experts_reproduce_x(c):
    cfg = _small(c, 400, 768)
    x, idx, w = _inputs(cfg)
    o = oracle.dispatch(x, idx, w, cfg.E, cfg.R, False, with_rank=False)
    out, _ = oracle.combine(o["exp_x"], o["layout"]["expert_slot"], w)
    xf = oracle.f32_from_bf16(x).astype(np.float64)
    of = oracle.f32_from_bf16(out).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(xf), 2.0 ** -126))) - 7)
    assert np.all(np.abs(of - xf) <= ulp)


def test_linear_experts_match_dense_reference():
    # The lesson-14 exercise: N=4, H=4, K=2, E=4 with its routing table, then
    # a larger random case. Experts are y = x W_e; the combine must equal the
    # dense sum_k w_k y_k up to the fp32 accumulation and the final BF16 rounding.
    def run(N, H, K, E, idx, seed):
        key = ei.stream_key(seed, 40)
        x = ei.bf16_bits_from_f32(ei.normal(key, N * H).astype(np.float32)).reshape(N, H)
        raw = 0.1 + 0.9 * ei.uniform01(ei.stream_key(seed, 41), N * K).reshape(N, K)
        w = (raw / raw.sum(1, keepdims=True)).astype(np.float32)
        W = ei.normal(ei.stream_key(seed, 42), E * H * H).reshape(E, H, H) / np.sqrt(H)
        lay = oracle.layout(idx, E, 1)
        o = oracle.dispatch(x, idx, w, E, 1, False, lay=lay, with_rank=False)
        e_of_row = idx.reshape(-1)[o["exp_src"]]
        xin = oracle.f32_from_bf16(o["exp_x"]).astype(np.float64)
        y = ei.bf16_bits_from_f32(np.einsum("rh,rhg->rg", xin, W[e_of_row]).astype(np.float32))
        out, _ = oracle.combine(y, lay["expert_slot"], w)
        yf = oracle.f32_from_bf16(y).astype(np.float64)
        terms = np.where((idx >= 0)[:, :, None],
                         w[:, :, None].astype(np.float64) * yf[np.maximum(lay["expert_slot"], 0)], 0.0)
        ref = terms.sum(1)
        of = oracle.f32_from_bf16(out).astype(np.float64)
        bound = K * 2.0 ** -24 * np.abs(terms).sum(1) + \
            2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 8)
        assert np.all(np.abs(of - ref) <= bound * 1.0001)
        # the page's own tolerance on the unrounded sum, scaled to BF16 output
        assert np.allclose(of, ref, rtol=2 ** -7, atol=1e-5)

    run(4, 4, 2, 4, np.array([[0, 2], [1, 3], [0, 3], [1, 2]], np.int32), 42)
    N, H, K, E = 64, 64, 8, 16
    idx = np.argsort(ei.uniform01(ei.stream_key(5, 43), N * E).reshape(N, E), axis=1)[:, :K].astype(np.int32)
    run(N, H, K, E, idx, 5)


def test_summation_order_and_fused_multiply_add():
    # Hand-derived: acc0 = -(1 + 2^-7 + 2^-17) * 1; the second term
    # (1 + 2^-17) * (1 + 2^-7) = 1 + 2^-7 + 2^-17 + 2^-24 exactly, so one fused
    # multiply-add leaves exactly 2^-24 (a separate fp32 product would round
    # the 2^-24 away and leave 0; the reversed order also leaves 0).
    a = np.float32(1 + 2 ** -7 + 2 ** -17)
    b = np.float32(1 + 2 ** -17)
    y = ei.bf16_bits_from_f32(np.array([[1.0], [1 + 2 ** -7]], np.float32))
    slot = np.array([[0, 1]], np.int32)
    out, _ = oracle.combine(y, slot, np.array([[-a, b]], np.float32))
    assert oracle.f32_from_bf16(out)[0, 0] == np.float32(2 ** -24)
    out, _ = oracle.combine(y, slot[:, ::-1].copy(), np.array([[b, -a]], np.float32))
    assert oracle.f32_from_bf16(out)[0, 0] == 0.0


def test_masked_slots_skipped_and_all_masked_is_positive_zero():
    y = ei.bf16_bits_from_f32(np.array([[1.0, -2.0], [3.0, 4.0]], np.float32))
    slot = np.array([[-1, 1], [-1, -1]], np.int32)
    w = np.array([[5.0, 0.5], [7.0, 7.0]], np.float32)
    out, _ = oracle.combine(y, slot, w)
    assert oracle.f32_from_bf16(out).tolist() == [[1.5, 2.0], [0.0, 0.0]]
    assert out[1].tolist() == [0, 0]  # +0, not -0


@pytest.mark.parametrize("c,use_fp8", [(1, False), (2, True)])
def test_ll_matches_layout_and_expert_major(c, use_fp8):
    cfg = ei.WORKLOADS[c]
    n_s = 16 if c == 1 else 8
    cfg = cfg.scaled(N=cfg.R * n_s, H=256)
    x, idx, w = _inputs(cfg)
    ll = oracle.ll_dispatch(x, idx, cfg.E, cfg.R, cfg.T, use_fp8)
    assert ll["status"] == 0
    lay = oracle.layout(idx, cfg.E, cfg.R)
    assert np.array_equal(ll["recv_count"], lay["num_tokens_per_expert"])
    o = oracle.dispatch(x, idx, w, cfg.E, cfg.R, use_fp8, lay=lay, with_rank=False)
    cap = cfg.R * cfg.T
    for e in range(cfg.E):
        n = ll["recv_count"][e]
        a, b = lay["expert_offset"][e], lay["expert_offset"][e + 1]
        assert np.array_equal(ll["recv_x"][e, :n], o["exp_x"][a:b])
        assert np.array_equal(ll["recv_src"][e, :n], o["exp_src"][a:b] // cfg.K)
        assert np.all(ll["recv_src"][e, n:] == -1)
        if use_fp8:
            assert np.array_equal(ll["recv_scales"][e, :n], o["exp_scales"][a:b])
        # ranges: counts per source rank, offsets are their exclusive scan
        rng = ll["layout_range"][e]
        cnt, off = rng & 0xFFFFFFFF, rng >> 32
        src_rank = ll["recv_src"][e, :n] // n_s
        assert np.array_equal(cnt, np.bincount(src_rank, minlength=cfg.R))
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(cnt)[:-1]]))
    # slot map: row e*R*T + j
    sm = ll["slot_map"]
    ok = idx >= 0
    assert np.array_equal(sm[ok] // cap, idx[ok]) and np.all(sm[~ok] == -1)
    assert np.array_equal(sm[ok] % cap, lay["expert_slot"][ok] - lay["expert_offset"][idx[ok]])
    # per-rank view has the pages' shape [num_local_experts, num_ranks * T, hidden]
    L = cfg.E // cfg.R
    assert ll["recv_x"].reshape(cfg.R, L, cap, cfg.H).shape[1:] == (L, cfg.R * cfg.T, cfg.H)


def test_ll_combine_identity():
    cfg = ei.WORKLOADS[1].scaled(H=512)
    x, idx, w = _inputs(cfg)
    ll = oracle.ll_dispatch(x, idx, cfg.E, cfg.R, cfg.T, False)
    out, st = oracle.ll_combine(ll["recv_x"], ll["slot_map"], w)
    xf = oracle.f32_from_bf16(x).astype(np.float64)
    of = oracle.f32_from_bf16(out).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(xf), 2.0 ** -126))) - 7)
    assert st == 0 and np.all(np.abs(of - xf) <= ulp)


def test_ll_overflow_flagged():
    cfg = ei.WORKLOADS[1].scaled(H=128, N=8 * 20)
    x, idx, w = _inputs(cfg)
    ll = oracle.ll_dispatch(x, idx, cfg.E, cfg.R, 16, False)
    assert ll["status"] & oracle.LL_OVERFLOW


def test_two_phase_ll_combine_equals_single_phase():
    # Send half: every routed (t, k) row lands at staging row t*K + k, a copy
    # of y's row; receive half: the same weighted sum as the one-launch combine
    # ("DeepEP V1 guide" 6.1: low_latency_combine with a receive hook).
    # T = 8 fits the 8 tokens per rank; the packed rows do not depend on T.
    cfg = ei.WORKLOADS[2].scaled(N=32 * 8, H=256, T=8)
    x, idx, w = _inputs(cfg, seed=4)
    ll = oracle.ll_dispatch(x, idx, cfg.E, cfg.R, cfg.T, False)
    y = ei.bf16_bits_from_f32(ei.normal(ei.stream_key(9, 3), ll["recv_x"].size).astype(np.float32))
    y = y.reshape(ll["recv_x"].shape)
    staging, st = oracle.ll_combine_send(y, ll["slot_map"])
    assert st == 0
    sm = ll["slot_map"].reshape(-1)
    ok = sm >= 0
    assert np.array_equal(staging[ok], y.reshape(-1, cfg.H)[sm[ok]])
    assert np.all(staging[~ok] == 0)
    two = oracle.ll_combine_recv(staging, ll["slot_map"], w)
    one, _ = oracle.ll_combine(y, ll["slot_map"], w)
    assert np.array_equal(two, one)


def test_shrink_mask_hand_example():
    # "DeepEP V1 (legacy) guide" 6.4 (shrink mode): a masked rank neither sends
    # nor receives, so its experts' slots and its own tokens' slots drop out.
    # 4 tokens, 2 ranks of 2 experts, tokens 0-1 from rank 0 and 2-3 from rank 1.
    N, K, E, R, T, H = 4, 2, 4, 2, 2, 8
    idx = np.array([[0, 2], [3, 1], [2, -1], [1, 3]], np.int32)
    x = ei.bf16_bits_from_f32(np.arange(N * H, dtype=np.float32).reshape(N, H) + 1)
    # rank 1 masked at the send: only (t0 -> e0) and (t1 -> e1) remain
    ll = oracle.ll_dispatch(x, idx, E, R, T, False, rank_mask=np.array([0, 1], np.int32))
    assert ll["status"] == 0
    assert ll["recv_count"].tolist() == [1, 1, 0, 0]
    assert ll["slot_map"].tolist() == [[0, -1], [-1, 4], [-1, -1], [-1, -1]]
    assert np.array_equal(ll["recv_x"][0, 0], x[0]) and np.array_equal(ll["recv_x"][1, 0], x[1])
    assert ll["recv_src"][0].tolist() == [0, -1, -1, -1] and ll["recv_src"][1].tolist() == [1, -1, -1, -1]
    assert ll["layout_range"].tolist() == [[1, 1 << 32], [1, 1 << 32], [0, 0], [0, 0]]
    # nothing masked at the send; rank 0 is lost before the combine
    full = oracle.ll_dispatch(x, idx, E, R, T, False)
    assert full["slot_map"].tolist() == [[0, 8], [12, 4], [9, -1], [5, 13]]
    y = np.repeat(np.arange(1, E * R * T + 1, dtype=np.float32)[:, None], H, axis=1)   # row r holds r + 1
    y = ei.bf16_bits_from_f32(y).reshape(E, R * T, H)
    w = np.array([[1, 1], [1, 1], [0.5, 1], [1, 0.25]], np.float32)
    out, st = oracle.ll_combine(y, full["slot_map"], w, rank_mask=np.array([1, 0], np.int32), R=R)
    of = oracle.f32_from_bf16(out)
    assert st == 0
    assert out[0].tolist() == [0] * H and out[1].tolist() == [0] * H   # rank 0's tokens: +0
    assert np.all(of[2] == 0.5 * 10) and np.all(of[3] == 0.25 * 14)    # only rank 1's experts count


def test_shrink_mask_degenerate_cases():
    cfg = ei.WORKLOADS[2].scaled(N=32 * 8, H=256, T=8)
    x, idx, w = _inputs(cfg, seed=6)
    R, E, T = cfg.R, cfg.E, cfg.T
    plain = oracle.ll_dispatch(x, idx, E, R, T, True)
    none = oracle.ll_dispatch(x, idx, E, R, T, True, rank_mask=np.zeros(R, np.int32))
    for k in ("recv_x", "recv_scales", "recv_src", "recv_count", "layout_range", "slot_map"):
        assert np.array_equal(plain[k], none[k]), k
    every = oracle.ll_dispatch(x, idx, E, R, T, True, rank_mask=np.ones(R, np.int32))
    assert every["recv_count"].sum() == 0 and np.all(every["slot_map"] == -1)
    # masking ranks = the unmasked dispatch of the routing with their slots set to -1
    m = np.zeros(R, np.int32)
    m[[3, 17]] = 1
    L, n_s = E // R, cfg.N // R
    idx_m = idx.copy()
    for t in range(cfg.N):
        for k in range(cfg.K):
            if idx[t, k] >= 0 and (m[idx[t, k] // L] or m[t // n_s]):
                idx_m[t, k] = -1
    a = oracle.ll_dispatch(x, idx, E, R, T, True, rank_mask=m)
    b = oracle.ll_dispatch(x, idx_m, E, R, T, True)
    for k in ("recv_x", "recv_scales", "recv_src", "recv_count", "layout_range", "slot_map"):
        assert np.array_equal(a[k], b[k]), k
    y = ei.bf16_bits_from_f32(ei.normal(ei.stream_key(9, 4), plain["recv_x"].size).astype(np.float32))
    y = y.reshape(plain["recv_x"].shape)
    out, _ = oracle.ll_combine(y, plain["slot_map"], w, rank_mask=np.ones(R, np.int32), R=R)
    assert np.all(out == 0)
    same, _ = oracle.ll_combine(y, plain["slot_map"], w, rank_mask=np.zeros(R, np.int32), R=R)
    ref, _ = oracle.ll_combine(y, plain["slot_map"], w)
    assert np.array_equal(same, ref)


def test_bias_is_added_after_the_weighted_sum():
    # "DeepEP Ascend deep dive", "Combine: More Output, Same Cost": the shared
    # expert's output is added as a bias in the epilogue. Hand-derived: terms
    # 2^24 and 1 first give 2^24 in fp32 (2^24 + 1 rounds to even), then the
    # bias -2^24 leaves 0; adding the bias first would leave 1.
    y = ei.bf16_bits_from_f32(np.array([[1.0], [1.0]], np.float32))
    slot = np.array([[0, 1]], np.int32)
    w = np.array([[2.0 ** 24, 1.0]], np.float32)
    bias = ei.bf16_bits_from_f32(np.array([[-(2.0 ** 24)]], np.float32))
    out, _ = oracle.combine(y, slot, w, bias)
    assert oracle.f32_from_bf16(out)[0, 0] == 0.0
    # zero bias changes nothing; masked tokens give the bias itself
    cfg = _small(4, 200, 256)
    x, idx, w = _inputs(cfg)
    lay = oracle.layout(idx, cfg.E, cfg.R)
    y = ei.bf16_bits_from_f32(ei.normal(ei.stream_key(3, 5), int(lay["expert_offset"][-1]) * 256)
                              .astype(np.float32)).reshape(-1, 256)
    a, _ = oracle.combine(y, lay["expert_slot"], w)
    b, _ = oracle.combine(y, lay["expert_slot"], w, np.zeros_like(x))
    assert np.array_equal(a, b)
    none = np.full_like(lay["expert_slot"], -1)
    c, _ = oracle.combine(y, none, w, x)
    assert np.array_equal(c, x)


@pytest.mark.parametrize("A", [2, 128])
def test_expert_alignment_pads_each_segment(A):
    cfg = _small(5, 600, 256)
    x, idx, w = _inputs(cfg)
    plain = oracle.layout(idx, cfg.E, cfg.R)
    al = oracle.layout(idx, cfg.E, cfg.R, expert_alignment=A)
    cnt = plain["num_tokens_per_expert"]
    assert np.array_equal(al["num_tokens_per_expert"], cnt)
    seg = np.diff(al["expert_offset"])
    assert np.array_equal(seg, (cnt + A - 1) // A * A) and np.all(al["expert_offset"] % A == 0)
    es, ep_ = al["expert_slot"], plain["expert_slot"]
    ok = idx >= 0
    e = np.where(ok, idx, 0)
    assert np.array_equal(es[ok] - al["expert_offset"][e[ok]], ep_[ok] - plain["expert_offset"][e[ok]])
    assert np.array_equal(al["rank_slot"], plain["rank_slot"])
    o = oracle.dispatch(x, idx, w, cfg.E, cfg.R, True, lay=al, with_rank=False)
    used = np.zeros(o["exp_x"].shape[0], bool)
    used[es[ok]] = True
    assert np.all(o["exp_x"][~used] == 0) and np.all(o["exp_scales"][~used] == 0)
    assert np.all(o["exp_src"][~used] == -1)
    q, s = oracle.quantize_rows(x)
    assert np.array_equal(o["exp_x"][used], q[o["exp_src"][used] // cfg.K])


def test_two_level_combine():
    # Level 1: each rank sums its own experts' weighted outputs (one row per
    # (token, rank)); level 2: the ranks' rows are summed back per token.
    cfg = _small(3, 300, 256)
    x, idx, w = _inputs(cfg)
    lay = oracle.layout(idx, cfg.E, cfg.R)
    D_e = int(lay["expert_offset"][-1])
    y = ei.bf16_bits_from_f32(ei.normal(ei.stream_key(8, 1), D_e * 256).astype(np.float32)).reshape(D_e, 256)
    part, st = oracle.combine_to_ranks(y, idx, lay, w, cfg.E, cfg.R)
    assert st == 0 and part.shape[0] == int(lay["rank_offset"][-1])
    # each rank row: the f64 sum of that rank's terms, within the fp32 bound and one BF16 rounding
    L = cfg.E // cfg.R
    yf = oracle.f32_from_bf16(y).astype(np.float64)
    pf = oracle.f32_from_bf16(part).astype(np.float64)
    for t in range(0, cfg.N, 13):
        for r in range(cfg.R):
            row = lay["rank_slot"][t, r]
            if row < 0:
                continue
            ks = [k for k in range(cfg.K) if idx[t, k] >= 0 and idx[t, k] // L == r]
            terms = np.array([w[t, k] * yf[lay["expert_slot"][t, k]] for k in ks])
            ref = terms.sum(0)
            bound = len(ks) * 2.0 ** -24 * np.abs(terms).sum(0) + 2.0 ** (
                np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 8)
            assert np.all(np.abs(pf[row] - ref) <= bound * 1.0001)
    out, _ = oracle.combine(part, lay["rank_slot"], None)
    # with one expert per token the two levels equal the flat combine exactly
    idx1 = idx[:, :1].copy()
    lay1 = oracle.layout(idx1, cfg.E, cfg.R)
    y1 = y[: int(lay1["expert_offset"][-1])]
    p1, _ = oracle.combine_to_ranks(y1, idx1, lay1, w[:, :1].copy(), cfg.E, cfg.R)
    o2, _ = oracle.combine(p1, lay1["rank_slot"], None)
    o1, _ = oracle.combine(y1, lay1["expert_slot"], w[:, :1].copy())
    assert np.array_equal(o1, o2)
    # identity experts with weights summing to 1: within two BF16 steps of x
    o = oracle.dispatch(x, idx, w, cfg.E, cfg.R, False, lay=lay, with_rank=False)
    part, _ = oracle.combine_to_ranks(o["exp_x"], idx, lay, w, cfg.E, cfg.R)
    out, _ = oracle.combine(part, lay["rank_slot"], None)
    xf = oracle.f32_from_bf16(x).astype(np.float64)
    of = oracle.f32_from_bf16(out).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(xf), 2.0 ** -126))) - 7)
    assert np.all(np.abs(of - xf) <= 2 * ulp)


def test_backward_adjoint_identities():
    # Training reuse ("DeepEP V1 guide" 5.1): dispatch backward is a combine
    # with unit weights, combine backward is a dispatch (of the weighted
    # gradient). Both pinned by adjoint identities and a finite difference,
    # computed in float64 with numpy, independently of the oracle's code.
    cfg = _small(3, 120, 256)
    x, idx, w = _inputs(cfg, seed=6)
    lay = oracle.layout(idx, cfg.E, cfg.R)
    es = lay["expert_slot"]
    D_e = int(lay["expert_offset"][-1])
    o = oracle.dispatch(x, idx, w, cfg.E, cfg.R, False, lay=lay, with_rank=False)
    g_rows = ei.bf16_bits_from_f32(ei.normal(ei.stream_key(6, 1), D_e * 256).astype(np.float32)).reshape(D_e, 256)
    # <dispatch(x), g> == <x, dispatch_backward(g)>: dispatch_backward = unit-weight combine
    gx, _ = oracle.combine(g_rows, es, None)
    f = lambda a: oracle.f32_from_bf16(a).astype(np.float64)
    lhs = (f(o["exp_x"]) * f(g_rows)).sum()
    ref_gx = np.zeros((cfg.N, 256))
    ok = es >= 0
    for t, k in zip(*np.nonzero(ok)):
        ref_gx[t] += f(g_rows)[es[t, k]]
    assert abs(lhs - (f(x) * ref_gx).sum()) <= 1e-9 * np.abs(f(x) * ref_gx).sum()
    assert np.all(np.abs(f(gx) - ref_gx) <= np.abs(ref_gx) * 2.0 ** -7 + 1e-30 + cfg.K * 2.0 ** -24 * np.abs(ref_gx))
    # combine backward: grad_y rows are bf16(w * g); grad_w is the finite difference of <g, combine(y, w)>
    y = ei.bf16_bits_from_f32(ei.normal(ei.stream_key(6, 2), D_e * 256).astype(np.float32)).reshape(D_e, 256)
    g = ei.bf16_bits_from_f32(ei.normal(ei.stream_key(6, 3), cfg.N * 256).astype(np.float32)).reshape(cfg.N, 256)
    gy, gw, st = oracle.combine_backward(g, y, es, w)
    assert st == 0
    for t, k in list(zip(*np.nonzero(ok)))[::17]:
        want = ei.bf16_bits_from_f32((w[t, k] * oracle.f32_from_bf16(g[t])).astype(np.float32))
        assert np.array_equal(gy[es[t, k]], want)

        def loss(wtk):
            out = np.zeros(256)
            for kk in range(cfg.K):
                if es[t, kk] >= 0:
                    out += (wtk if kk == k else float(w[t, kk])) * f(y)[es[t, kk]]
            return (f(g)[t] * out).sum()
        d = 0.25
        fd = (loss(float(w[t, k]) + d) - loss(float(w[t, k]) - d)) / (2 * d)   # exact: loss is linear in w
        assert abs(gw[t, k] - fd) <= 1e-9 * (1 + abs(fd))
    assert np.all(gw[~ok] == 0)
