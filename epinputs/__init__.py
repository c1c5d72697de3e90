"""Seeded synthetic inputs for MoE layout / dispatch / combine.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark. It holds no arithmetic of the method itself (no counts, slots,
quantisation or weighted sums): it only draws hidden states and router
decisions, with the shapes and value distributions of the workloads the
DeepEP write-ups describe:

* hidden states x ~ N(0, 1), stored as BF16 (round to nearest even);
* router logits ~ N(0, 1) in fp32, softmax, top-k, weights renormalised over
  the chosen experts (the simulator exercise of "DeepSeek DeepEP lesson 14",
  section "practice task", and the DeepSeek-V3 gating it describes);
* group-limited gating (DeepEP V1 guide, section 1 / 2.1: "top-4 groups");
* a Zipf-skewed popularity with a fraction of top-k slots masked to -1
  (DeepEP V1 guide, section 6.3: "-1 in topk_idx means no expert").

Random numbers come from one counter-based generator, SplitMix64 (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014),
evaluated at position i of a stream as mix(key + (i + 1) * gamma). Normals use
the Box-Muller transform in float64. Everything is vectorised numpy, so the
same seed gives the same inputs on any host (up to the last bit of libm's
log/cos/sin, which both sides of a parity test share because inputs are drawn
once per process and fed to both).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

__all__ = [
    "Config", "WORKLOADS", "splitmix64", "uniform01", "normal", "bf16_bits_from_f32",
    "make_x", "make_routing", "make_inputs", "stream_key",
]

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function, applied in place to a uint64 array."""
    t = np.empty_like(z)
    np.right_shift(z, 30, out=t)
    z ^= t
    z *= _M1
    np.right_shift(z, 27, out=t)
    z ^= t
    z *= _M2
    np.right_shift(z, 31, out=t)
    z ^= t
    return z


def stream_key(seed: int, stream: int) -> int:
    """Key of an independent stream (one per tensor) derived from a seed."""
    with np.errstate(over="ignore"):
        s = _mix(np.array([seed], dtype=np.uint64) * _GAMMA + np.uint64(stream))
        s ^= np.uint64(0x5DEECE66D)
        return int(_mix(s)[0])


def splitmix64(key: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 sequence seeded with key."""
    out = np.empty(n, dtype=np.uint64)
    k = np.uint64(key)
    with np.errstate(over="ignore"):
        for a in range(0, n, _CHUNK):
            b = min(n, a + _CHUNK)
            z = out[a:b]
            z.view(np.int64)[:] = np.arange(start + a + 1, start + b + 1, dtype=np.int64)
            z *= _GAMMA
            z += k
            _mix(z)
    return out


def uniform01(key: int, n: int, start: int = 0) -> np.ndarray:
    """Uniform doubles in the open interval (0, 1): (top 53 bits + 0.5) / 2^53."""
    u = splitmix64(key, n, start)
    u >>= 11
    return (u.view(np.int64).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal(key: int, n: int) -> np.ndarray:
    """n standard normals (float64) by Box-Muller on consecutive uniform pairs."""
    out = np.empty(n, dtype=np.float64)
    pairs = (n + 1) // 2
    for a in range(0, pairs, _CHUNK):
        b = min(pairs, a + _CHUNK)
        u = uniform01(key, 2 * (b - a), 2 * a)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        th = (2.0 * np.pi) * u[1::2]
        z = np.empty(2 * (b - a), dtype=np.float64)
        z[0::2] = r * np.cos(th)
        z[1::2] = r * np.sin(th)
        lo, hi = 2 * a, min(n, 2 * b)
        out[lo:hi] = z[: hi - lo]
    return out


def bf16_bits_from_f32(f: np.ndarray) -> np.ndarray:
    """Input encoding of the generator: fp32 -> BF16 bit patterns, nearest-even.

    Only used to store generated hidden states; inputs are finite by
    construction.
    """
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


@dataclasses.dataclass(frozen=True)
class Config:
    """One synthetic workload.

    N tokens, H hidden, E experts, K top-k, R logical ranks (experts split
    evenly, E/R per rank), T the low-latency per-rank token capacity (None for
    normal mode), fp8 whether dispatch quantises.
    """
    name: str
    N: int
    H: int
    E: int
    K: int
    R: int
    fp8: bool
    mode: str                   # "ll" or "normal"
    routing: str                # "softmax", "grouped" or "zipf"
    T: Optional[int] = None
    n_groups: int = 1
    topk_groups: int = 1
    zipf_s: float = 0.0
    mask_frac: float = 0.0

    def scaled(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[int, Config] = {
    # Low-latency decode, tiny: 8 ranks x 16 tokens, BF16.
    1: Config("ll_decode_tiny_n128_h7168_e256_k8_r8", N=128, H=7168, E=256, K=8, R=8,
              fp8=False, mode="ll", routing="softmax", T=128),
    # Low-latency decode, FP8: 32 ranks x 128 tokens.
    2: Config("ll_decode_fp8_n4096_h7168_e256_k8_r32", N=4096, H=7168, E=256, K=8, R=32,
              fp8=True, mode="ll", routing="softmax", T=128),
    # Prefill with group-limited gating: 8 groups of 32, top-4 groups, top-8 experts.
    3: Config("prefill_grouped_n4096_h7168_e256_k8_r16", N=4096, H=7168, E=256, K=8, R=16,
              fp8=True, mode="normal", routing="grouped", n_groups=8, topk_groups=4),
    # Large prefill: 16384 tokens, top-6 of 256, 8 ranks, BF16 (about 1.4 GB of copies).
    4: Config("prefill_large_n16384_h7168_e256_k6_r8", N=16384, H=7168, E=256, K=6, R=8,
              fp8=False, mode="normal", routing="softmax"),
    # Skewed: Zipf(1.2) popularity over 128 experts, top-8, 10 % of slots masked.
    5: Config("skewed_zipf_n8192_h4096_e128_k8_r8", N=8192, H=4096, E=128, K=8, R=8,
              fp8=True, mode="normal", routing="zipf", zipf_s=1.2, mask_frac=0.1),
}

# Stream tags: one independent stream per drawn tensor.
_S_X, _S_LOGITS, _S_GUMBEL, _S_SCORES, _S_MASK = 1, 2, 3, 4, 5


def make_x(N: int, H: int, seed: int = 0) -> np.ndarray:
    """Hidden states [N, H] as BF16 bit patterns (uint16), x ~ N(0, 1)."""
    z = normal(stream_key(seed, _S_X), N * H).astype(np.float32)
    return bf16_bits_from_f32(z).reshape(N, H)


def _topk_desc(scores: np.ndarray, K: int) -> np.ndarray:
    # Descending score, ties to the lower expert id (stable sort of -score).
    return np.argsort(-scores, axis=1, kind="stable")[:, :K].astype(np.int32)


def _renormalised_softmax(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    chosen = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    m = chosen.max(axis=1, keepdims=True)
    p = np.exp(chosen - m)
    return (p / p.sum(axis=1, keepdims=True)).astype(np.float32)


def make_routing(cfg: Config, seed: int = 0):
    """(topk_idx int32 [N, K], topk_weights float32 [N, K]) for a config."""
    N, E, K = cfg.N, cfg.E, cfg.K
    if cfg.routing in ("softmax", "grouped"):
        logits = normal(stream_key(seed, _S_LOGITS), N * E).astype(np.float32).reshape(N, E)
        masked_logits = logits
        if cfg.routing == "grouped":
            G = cfg.n_groups
            assert E % G == 0
            gs = logits.reshape(N, G, E // G).max(axis=2)
            keep = _topk_desc(gs, cfg.topk_groups)
            allowed = np.zeros((N, G), dtype=bool)
            np.put_along_axis(allowed, keep.astype(np.int64), True, axis=1)
            allowed = np.repeat(allowed, E // G, axis=1)
            masked_logits = np.where(allowed, logits, -np.inf).astype(np.float32)
        idx = _topk_desc(masked_logits, K)
        # softmax over all E then renormalised over the chosen K equals a
        # softmax over the chosen logits.
        w = _renormalised_softmax(logits, idx)
        return idx, w
    if cfg.routing == "zipf":
        logp = -cfg.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        u = uniform01(stream_key(seed, _S_GUMBEL), N * E).reshape(N, E)
        g = logp[None, :] - np.log(-np.log(u))
        idx = _topk_desc(g, K)
        scores = normal(stream_key(seed, _S_SCORES), N * K).astype(np.float32).reshape(N, K)
        m = scores.max(axis=1, keepdims=True)
        p = np.exp(scores - m)
        w = (p / p.sum(axis=1, keepdims=True)).astype(np.float32)
        n_mask = int(round(cfg.mask_frac * N * K))
        if n_mask:
            order = np.argsort(splitmix64(stream_key(seed, _S_MASK), N * K), kind="stable")
            flat = order[:n_mask]
            idx.reshape(-1)[flat] = -1
            w.reshape(-1)[flat] = 0.0
        return idx, w
    raise ValueError(cfg.routing)


def make_inputs(cfg: Config, seed: int = 0, with_x: bool = True) -> dict:
    idx, w = make_routing(cfg, seed)
    out = {"topk_idx": idx, "topk_weights": w}
    if with_x:
        out["x"] = make_x(cfg.N, cfg.H, seed)
    return out
