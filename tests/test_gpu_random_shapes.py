"""Seeded random shapes through the whole path, against the oracle.

Each case draws its shape (tokens, top-k, experts, ranks, hidden, share of
masked slots, BF16 or FP8 with one of the three scale formats) from a fixed
seed, and its routing and rows from the seeded input generators. Layout,
both receive buffers and combine (normal path), and send, receive and
combine (low-latency path) must equal the oracle bit for bit. The shapes
reach what the fixed cases do not: layouts of one to a few hundred CTAs with
column counts that are and are not multiples of four, combines whose last
partial wave is split into spans of every width, low-latency sends of every
form.
"""
import numpy as np
import pytest
import torch

import combine_ep_get_dispatch_gb300 as ep
import epinputs as ei
import oracle
from helpers import status_value, to_dev, to_dev_bf16, u16, u8

pytestmark = pytest.mark.gpu

LAYOUT_KEYS = ("num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "expert_offset",
               "rank_offset", "expert_slot", "rank_slot")
MAX_ELEMS = 96 << 20          # rows x hidden of the largest buffer a case holds


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available()


def _idx(N, K, E, seed, p_mask):
    """Distinct experts per token (uniform), a share p_mask of slots masked."""
    u = ei.uniform01(ei.stream_key(seed, 910), N * E).reshape(N, E)
    idx = np.argsort(u, axis=1)[:, :K].astype(np.int32)
    if p_mask:
        m = ei.uniform01(ei.stream_key(seed, 911), N * K).reshape(N, K) < p_mask
        idx[m] = -1
    return idx


def _weights(N, K, seed):
    return ei.uniform01(ei.stream_key(seed, 912), N * K).reshape(N, K).astype(np.float32)


def _rows(n, H, seed):
    z = ei.normal(ei.stream_key(seed, 913), n * H).astype(np.float32) * 2.0
    return ei.bf16_bits_from_f32(z).reshape(n, H)


def _flags(rng):
    """(fp8, round_scale, ue8m0) for a case."""
    kind = int(rng.integers(0, 4))
    return kind > 0, kind == 2, kind == 3


def _normal_shape(seed):
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.choice([1, 2, 4, 8, 16, 32]))
    L = int(rng.integers(1, max(2, 1024 // R)))
    E = R * L
    K = int(rng.integers(1, min(E, 16) + 1))
    entries = int(rng.choice([2000, 20000, 120000]))     # one CTA to ~120 layout CTAs
    N = int(rng.integers(0, entries // K + 1))
    fp8, rs, ue = _flags(rng)
    unit = 128 if fp8 else 8
    h_max = max(unit, min(4096, MAX_ELEMS // max(1, N * K)) // unit * unit)
    H = unit * int(rng.integers(1, h_max // unit + 1))
    p_mask = float(rng.choice([0.0, 0.05, 0.4]))
    return N, K, E, R, H, fp8, rs, ue, p_mask


@pytest.mark.parametrize("seed", range(24))
def test_random_normal_path(seed):
    N, K, E, R, H, fp8, rs, ue, p_mask = _normal_shape(seed)
    idx = _idx(N, K, E, seed, p_mask) if N else np.zeros((0, K), np.int32)
    w = _weights(N, K, seed) if N else np.zeros((0, K), np.float32)
    x = _rows(N, H, seed) if N else np.zeros((0, H), np.uint16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = ep.get_dispatch_layout(to_dev(idx), E, R, status=st)
    ref_lay = oracle.layout(idx, E, R)
    for k in LAYOUT_KEYS:
        assert np.array_equal(getattr(lay, k).cpu().numpy(), ref_lay[k]), (k, (N, K, E, R))
    res = ep.dispatch(to_dev_bf16(x), lay, to_dev(w), use_fp8=fp8, status=st, exact=True,
                      round_scale=rs, use_ue8m0=ue)
    ref = oracle.dispatch(x, idx, w, E, R, fp8, lay=ref_lay, round_scale=rs, ue8m0=ue)
    conv = u8 if fp8 else u16
    D_e, D_r = ref["exp_x"].shape[0], ref["rank_x"].shape[0]
    assert np.array_equal(conv(res.expert_x[:D_e]), ref["exp_x"])
    assert np.array_equal(res.expert_src[:D_e].cpu().numpy(), ref["exp_src"])
    assert np.array_equal(conv(res.rank_x[:D_r]), ref["rank_x"])
    assert np.array_equal(res.rank_src[:D_r].cpu().numpy(), ref["rank_src"])
    assert np.array_equal(res.rank_topk_idx[:D_r].cpu().numpy(), ref["rank_topk_idx"])
    assert np.array_equal(res.rank_topk_weights[:D_r].cpu().numpy(), ref["rank_topk_weights"])
    if fp8:
        assert np.array_equal(res.expert_scales[:D_e].cpu().numpy(), ref["exp_scales"])
        assert np.array_equal(res.rank_scales[:D_r].cpu().numpy(), ref["rank_scales"])
    y = _rows(max(D_e, 1), H, seed + 500)
    out = ep.combine(to_dev_bf16(y), lay, to_dev(w), status=st)
    ref_out, _ = oracle.combine(y, ref_lay["expert_slot"], w)
    assert np.array_equal(u16(out), ref_out)
    assert status_value(st) == 0


def _ll_shape(seed):
    rng = np.random.default_rng(2000 + seed)
    R = int(rng.choice([1, 2, 4, 8, 16, 32]))
    L = int(rng.integers(1, max(2, 512 // R // 4)))
    E = R * L
    K = int(rng.integers(1, min(E, 16) + 1))
    ns = int(rng.integers(1, int(rng.choice([4096, 16384, 40000])) // (R * K) + 2))
    if seed % 4 == 3:
        # a source rank of more than 8192 entries: the send takes the layout kernel
        R = int(rng.choice([1, 2]))
        E = R * L
        K = int(rng.integers(1, min(E, 2) + 1))
        ns = int(rng.integers(8192 // K + 1, 12000 // K + 1))
    fp8, rs, ue = _flags(rng)
    unit = 128 if fp8 else 8
    T = ns + int(rng.integers(0, 9))
    while E * R * T * unit > MAX_ELEMS and ns > 1:        # the fixed [E, R*T, H] receive buffer
        ns = max(1, ns // 2)
        T = ns + int(rng.integers(0, 9))
    h_max = max(unit, min(2048, MAX_ELEMS // (E * R * T)) // unit * unit)
    H = unit * int(rng.integers(1, h_max // unit + 1))
    p_mask = float(rng.choice([0.0, 0.05, 0.4]))
    return R * ns, K, E, R, T, H, fp8, rs, ue, p_mask


@pytest.mark.parametrize("seed", range(20))
def test_random_low_latency_path(seed):
    N, K, E, R, T, H, fp8, rs, ue, p_mask = _ll_shape(seed)
    idx = _idx(N, K, E, seed, p_mask)
    w = _weights(N, K, seed)
    x = _rows(N, H, seed)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    recv, cnt, handle, hook = ep.low_latency_dispatch(to_dev_bf16(x), to_dev(idx), T, E, R, use_fp8=fp8,
                                                      status=st, round_scale=rs, use_ue8m0=ue)
    hook()
    ref = oracle.ll_dispatch(x, idx, E, R, T, fp8, round_scale=rs, ue8m0=ue)
    cnt = cnt.cpu().numpy()
    assert np.array_equal(cnt, ref["recv_count"]), (N, K, E, R, T)
    assert np.array_equal(handle.layout_range.cpu().numpy(), ref["layout_range"])
    rx, rscale = recv if fp8 else (recv, None)
    gx = u8(rx) if fp8 else u16(rx)
    src = handle.recv_src.cpu().numpy()
    gs = rscale.cpu().numpy() if fp8 else None
    for e in range(E):
        n = cnt[e]
        assert np.array_equal(gx[e, :n], ref["recv_x"][e, :n]), e
        assert np.array_equal(src[e, :n], ref["recv_src"][e, :n]), e
        if fp8:
            assert np.array_equal(gs[e, :n], ref["recv_scales"][e, :n]), e
    y = np.zeros((E, R * T, H), np.uint16)
    z = _rows(E * R * T, H, seed + 700).reshape(E, R * T, H)
    for e in range(E):
        y[e, :cnt[e]] = z[e, :cnt[e]]
    out = ep.low_latency_combine(to_dev_bf16(y), to_dev(w), handle, status=st)
    ref_out, _ = oracle.ll_combine(y, ref["slot_map"], w)
    assert np.array_equal(u16(out), ref_out)
    assert status_value(st) == 0
