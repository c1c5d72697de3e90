"""CPU oracle for MoE layout / dispatch / combine: TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package. The product path (the CUDA library and its Python
binding) never calls it and has no CPU fallback.

This module is argument marshalling (numpy <-> the plain C++ oracle in
ep_oracle.cpp). What each function computes, and the passage of the DeepEP
write-ups it follows, is stated in ep_oracle.cpp.

Parity pins: every function here is pinned by the CPU tests against values
the pages fix (the lesson-14 routing table, the 1.4 GB volume example),
closed forms, invariants, brute force on tiny inputs and independent
formulations (a stable sort for slots, a nearest-code search for E4M3, the
library BF16 cast). No function is parity unpinned.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

_libs = {}
_all_cores = False


def use_all_cores(on: bool = True) -> bool:
    """Route the oracle's calls to the all-core build (the same source
    compiled with OpenMP; identical results) or back to the plain
    single-threaded one. Returns False, and stays on the plain build, when no
    all-core build is available. Only the benchmark's CPU-baseline timing
    uses it."""
    global _all_cores
    if on and _build.build_omp() is None:
        _all_cores = False
        return False
    _all_cores = on
    return True


def threads() -> int:
    """Threads the loaded oracle's row loops use (1 for the plain build)."""
    return int(lib().oracle_threads())


def lib():
    key = "omp" if _all_cores else "plain"
    if key not in _libs:
        if key == "omp":
            path = _build.build_omp()
        else:
            # EP_ORACLE_LIB: a prebuilt oracle library to load instead (the
            # mutation test points it at deliberately broken copies).
            path = os.environ.get("EP_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        L.oracle_bf16_from_f32.restype = ctypes.c_uint16
        L.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
        L.oracle_e4m3_from_f32.restype = ctypes.c_uint8
        L.oracle_e4m3_from_f32.argtypes = [ctypes.c_float]
        L.oracle_e4m3_to_f64.restype = ctypes.c_double
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_bf16_from_f32_n.argtypes = [P, P, i64]
        L.oracle_bf16_from_f32_n.restype = None
        L.oracle_e4m3_from_f32_n.argtypes = [P, P, i64]
        L.oracle_e4m3_from_f32_n.restype = None
        L.oracle_quantize_rows.argtypes = [P, i64, i32, P, P, i32]
        L.oracle_ue8m0_from_scales.argtypes = [P, i64, P]
        L.oracle_ue8m0_from_scales.restype = None
        L.oracle_quantize_rows.restype = None
        L.oracle_layout.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
        L.oracle_layout.restype = i32
        L.oracle_dispatch.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P, P,
                                      P, P, P, P, P, i64, P, P, P, i64]
        L.oracle_dispatch.restype = i32
        L.oracle_combine.argtypes = [P, i64, P, P, P, i32, i32, i32, P]
        L.oracle_combine_to_ranks.argtypes = [P, i64, P, P, P, P, i32, i32, i32, i32, i32, P, i64]
        L.oracle_combine_to_ranks.restype = i32
        L.oracle_combine_backward.argtypes = [P, P, i64, P, P, i32, i32, i32, P, P]
        L.oracle_combine_backward.restype = i32
        L.oracle_combine.restype = i32
        L.oracle_ll_dispatch.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32,
                                         P, P, P, P, P, P]
        L.oracle_ll_dispatch.restype = i32
        L.oracle_gather_rows.argtypes = [P, i64, P, i32, i32, i32, P]
        L.oracle_gather_rows.restype = i32
        L.oracle_combine_staged.argtypes = [P, P, P, i32, i32, i32, P]
        L.oracle_combine_staged.restype = i32
        L.oracle_ll_mask_routing.argtypes = [P, i32, i32, i32, i32, P, P]
        L.oracle_ll_mask_routing.restype = i32
        L.oracle_ll_mask_slot_map.argtypes = [P, i32, i32, i32, i32, i32, P, P]
        L.oracle_ll_mask_slot_map.restype = i32
        L.oracle_threads.argtypes = []
        L.oracle_threads.restype = i32
        _libs[key] = L
    return _libs[key]


# Status bits returned by the oracle.
BAD_INDEX, CAPACITY, LL_OVERFLOW = 1, 2, 4
# FP8 flags (the library's dispatch flags): E4M3 payload, power-of-two scales, UE8M0 scale bytes.
FP8, ROUND_SCALE, UE8M0 = 1, 2, 4


def fp8_flags(use_fp8: bool, round_scale: bool = False, ue8m0: bool = False) -> int:
    return (FP8 if use_fp8 else 0) | (ROUND_SCALE if round_scale else 0) | (UE8M0 if ue8m0 else 0)


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def bf16_from_f32(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    lib().oracle_bf16_from_f32_n(_p(f), _p(out), f.size)
    return out


def f32_from_bf16(h: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 (exact widening; no rounding involved)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def e4m3_from_f32(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint8)
    lib().oracle_e4m3_from_f32_n(_p(f), _p(out), f.size)
    return out


def e4m3_to_f64(c: np.ndarray) -> np.ndarray:
    table = np.array([lib().oracle_e4m3_to_f64(i) for i in range(256)], dtype=np.float64)
    return table[np.asarray(c, dtype=np.uint8)]


def quantize_rows(x_bf16: np.ndarray, round_scale: bool = False, ue8m0: bool = False):
    """[rows, H] BF16 bits -> (E4M3 codes [rows, H], fp32 scales [rows, H/128])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, H = x.shape
    assert H % 128 == 0
    q = np.empty((rows, H), dtype=np.uint8)
    s = np.empty((rows, H // 128), dtype=np.float32)
    lib().oracle_quantize_rows(_p(x), rows, H, _p(q), _p(s), fp8_flags(True, round_scale, ue8m0))
    return q, s


def ue8m0_from_scales(s: np.ndarray) -> np.ndarray:
    """Power-of-two fp32 scales -> UE8M0 bytes (2^(b - 127)); 0 -> 0."""
    s = np.ascontiguousarray(s, dtype=np.float32)
    out = np.empty(s.shape, np.uint8)
    lib().oracle_ue8m0_from_scales(_p(s), s.size, _p(out))
    return out


def layout(topk_idx: np.ndarray, E: int, R: int, expert_alignment: int = 1) -> dict:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    N, K = idx.shape
    assert E % R == 0
    o = {
        "num_tokens_per_rank": np.empty(R, np.int32),
        "num_tokens_per_expert": np.empty(E, np.int32),
        "is_token_in_rank": np.empty((N, R), np.uint8),
        "rank_offset": np.empty(R + 1, np.int32),
        "expert_offset": np.empty(E + 1, np.int32),
        "rank_slot": np.empty((N, R), np.int32),
        "expert_slot": np.empty((N, K), np.int32),
    }
    st = lib().oracle_layout(_p(idx), N, K, E, R, expert_alignment, _p(o["num_tokens_per_rank"]),
                             _p(o["num_tokens_per_expert"]), _p(o["is_token_in_rank"]),
                             _p(o["rank_offset"]), _p(o["expert_offset"]),
                             _p(o["rank_slot"]), _p(o["expert_slot"]))
    o["status"] = int(st)
    return o


def dispatch(x_bf16: np.ndarray, topk_idx: np.ndarray, topk_weights: np.ndarray, E: int, R: int,
             use_fp8: bool, lay: Optional[dict] = None, rank_cap: Optional[int] = None,
             exp_cap: Optional[int] = None, with_rank: bool = True, with_expert: bool = True,
             round_scale: bool = False, ue8m0: bool = False) -> dict:
    """Per-rank and expert-major receive buffers, sized exactly unless caps are given."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    N, H = x.shape
    K = idx.shape[1]
    if lay is None:
        lay = layout(idx, E, R)
    D_r = int(lay["rank_offset"][-1])
    D_e = int(lay["expert_offset"][-1])
    rank_cap = D_r if rank_cap is None else rank_cap
    exp_cap = D_e if exp_cap is None else exp_cap
    xdt = np.uint8 if use_fp8 else np.uint16
    sdt = np.uint8 if ue8m0 else np.float32
    S = max(H // 128, 1)
    o = {}
    if with_rank:
        o.update(rank_x=np.zeros((rank_cap, H), xdt),
                 rank_scales=np.zeros((rank_cap, S), sdt) if use_fp8 else None,
                 rank_src=np.full(rank_cap, -1, np.int32),
                 rank_topk_idx=np.full((rank_cap, K), -1, np.int32),
                 rank_topk_weights=np.zeros((rank_cap, K), np.float32))
    if with_expert:
        o.update(exp_x=np.zeros((exp_cap, H), xdt),
                 exp_scales=np.zeros((exp_cap, S), sdt) if use_fp8 else None,
                 exp_src=np.full(exp_cap, -1, np.int32))
    g = o.get
    st = lib().oracle_dispatch(_p(x), _p(idx), _p(w), N, K, H, E, R, fp8_flags(use_fp8, round_scale, ue8m0),
                               _p(lay["rank_slot"]), _p(lay["expert_slot"]),
                               _p(g("rank_x")), _p(g("rank_scales")), _p(g("rank_src")),
                               _p(g("rank_topk_idx")), _p(g("rank_topk_weights")), rank_cap,
                               _p(g("exp_x")), _p(g("exp_scales")), _p(g("exp_src")), exp_cap)
    o["status"] = int(st)
    o["layout"] = lay
    return o


def combine(y_bf16: np.ndarray, slot: np.ndarray, topk_weights: Optional[np.ndarray],
            bias: Optional[np.ndarray] = None) -> tuple:
    """out [N, H] BF16 bits from expert outputs y [rows, H] and slot map [N, K].

    topk_weights None: every weight is 1. bias [N, H] BF16 is added after the sum.
    """
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16).reshape(-1, y_bf16.shape[-1])
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    w = None if topk_weights is None else np.ascontiguousarray(topk_weights, dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.uint16)
    N, K = slot.shape
    H = y.shape[1]
    out = np.empty((N, H), np.uint16)
    st = lib().oracle_combine(_p(y), y.shape[0], _p(slot), _p(w), _p(b), N, K, H, _p(out))
    return out, int(st)


def combine_to_ranks(y_bf16: np.ndarray, topk_idx: np.ndarray, lay: dict, topk_weights: np.ndarray,
                     E: int, R: int) -> tuple:
    """Per-rank weighted pre-sums [D_r, H]: row rank_slot[t, r] sums t's experts on rank r."""
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    N, K = idx.shape
    H = y.shape[1]
    D_r = int(lay["rank_offset"][-1])
    out = np.zeros((D_r, H), np.uint16)
    st = lib().oracle_combine_to_ranks(_p(y), y.shape[0], _p(idx), _p(lay["expert_slot"]), _p(lay["rank_slot"]),
                                       _p(w), N, K, E, R, H, _p(out), D_r)
    return out, int(st)


def ll_mask_routing(topk_idx: np.ndarray, E: int, R: int, rank_mask: np.ndarray) -> np.ndarray:
    """Shrink mode: the routing with every slot of a masked rank (the expert's
    rank, or the token's source rank) set to -1."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    m = np.ascontiguousarray(rank_mask, dtype=np.int32)
    assert m.shape == (R,)
    N, K = idx.shape
    out = np.empty_like(idx)
    lib().oracle_ll_mask_routing(_p(idx), N, K, E, R, _p(m), _p(out))
    return out


def ll_mask_slot_map(slot_map: np.ndarray, E: int, R: int, T: int, rank_mask: np.ndarray) -> np.ndarray:
    """Shrink mode at combine time: slot-map entries of masked ranks set to -1."""
    slot = np.ascontiguousarray(slot_map, dtype=np.int32)
    m = np.ascontiguousarray(rank_mask, dtype=np.int32)
    assert m.shape == (R,)
    N, K = slot.shape
    out = np.empty_like(slot)
    lib().oracle_ll_mask_slot_map(_p(slot), N, K, E, R, T, _p(m), _p(out))
    return out


def ll_dispatch(x_bf16: np.ndarray, topk_idx: np.ndarray, E: int, R: int, T: int,
                use_fp8: bool, round_scale: bool = False, ue8m0: bool = False,
                rank_mask: Optional[np.ndarray] = None) -> dict:
    """Low-latency dispatch into the fixed [E, R*T, H] buffer (global view).

    rank_mask [R] (shrink mode): slots of masked ranks are dropped first.
    """
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    if rank_mask is not None:
        idx = ll_mask_routing(idx, E, R, rank_mask)
    N, H = x.shape
    K = idx.shape[1]
    xdt = np.uint8 if use_fp8 else np.uint16
    o = {
        "recv_x": np.zeros((E, R * T, H), xdt),
        "recv_scales": np.zeros((E, R * T, max(H // 128, 1)), np.uint8 if ue8m0 else np.float32)
        if use_fp8 else None,
        "recv_src": np.full((E, R * T), -1, np.int32),
        "recv_count": np.empty(E, np.int32),
        "layout_range": np.empty((E, R), np.int64),
        "slot_map": np.empty((N, K), np.int32),
    }
    st = lib().oracle_ll_dispatch(_p(x), _p(idx), N, K, H, E, R, T, fp8_flags(use_fp8, round_scale, ue8m0),
                                  _p(o["recv_x"]), _p(o["recv_scales"]), _p(o["recv_src"]),
                                  _p(o["recv_count"]), _p(o["layout_range"]), _p(o["slot_map"]))
    o["status"] = int(st)
    return o


def ll_combine(y_bf16: np.ndarray, slot_map: np.ndarray, topk_weights: np.ndarray,
               rank_mask: Optional[np.ndarray] = None, R: Optional[int] = None) -> tuple:
    """Low-latency combine: y is [E, R*T, H]; slot_map rows index its flattened view.

    rank_mask [R] (shrink mode, R given): slots of ranks masked now are skipped.
    """
    if rank_mask is not None:
        E, RT = y_bf16.shape[0], y_bf16.shape[1]
        slot_map = ll_mask_slot_map(slot_map, E, R, RT // R, rank_mask)
    return combine(y_bf16.reshape(-1, y_bf16.shape[-1]), slot_map, topk_weights)


def ll_combine_send(y_bf16: np.ndarray, slot_map: np.ndarray) -> tuple:
    """Token-major staging [N*K, H]: row t*K + k is y's row slot_map[t, k] (unwritten rows stay 0)."""
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16).reshape(-1, y_bf16.shape[-1])
    slot = np.ascontiguousarray(slot_map, dtype=np.int32)
    N, K = slot.shape
    H = y.shape[1]
    staging = np.zeros((N * K, H), np.uint16)
    st = lib().oracle_gather_rows(_p(y), y.shape[0], _p(slot), N, K, H, _p(staging))
    return staging, int(st)


def ll_combine_recv(staging: np.ndarray, slot_map: np.ndarray, topk_weights: np.ndarray) -> np.ndarray:
    """Weighted sum of the staged rows of every routed slot."""
    st_ = np.ascontiguousarray(staging, dtype=np.uint16)
    slot = np.ascontiguousarray(slot_map, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    N, K = slot.shape
    H = st_.shape[1]
    out = np.empty((N, H), np.uint16)
    lib().oracle_combine_staged(_p(st_), _p(slot), _p(w), N, K, H, _p(out))
    return out


def combine_backward(grad_out: np.ndarray, y_bf16: np.ndarray, slot: np.ndarray,
                     topk_weights: np.ndarray) -> tuple:
    """(grad_y [rows, H] BF16 bits, grad_w [N, K] float64) of out = sum_k w * y[slot]."""
    g = np.ascontiguousarray(grad_out, dtype=np.uint16)
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    N, K = slot.shape
    H = g.shape[1]
    grad_y = np.zeros(y.shape, np.uint16)
    grad_w = np.empty((N, K), np.float64)
    st = lib().oracle_combine_backward(_p(g), _p(y), y.shape[0], _p(slot), _p(w), N, K, H, _p(grad_y), _p(grad_w))
    return grad_y, grad_w, int(st)
