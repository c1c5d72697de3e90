"""The device FP8 quantiser (ep_fp8_quantize, the code the FP8 dispatch runs)
against the oracle's quantize_rows, exhaustively over the BF16 inputs a
128-channel block can present to it.

A block's result depends on its amax a (which sets s = fl(a / 448)) and on
each element x with |x| <= a. Every block here holds a at channel 0 and 127
values of x, so that every non-negative BF16 x <= a meets every finite
positive BF16 a (about 537 M elements in all). Negative x and the
power-of-two scale formats are covered on every 16th a. Codes and scales
must be identical: the device divides x / s with one correctly rounded
reciprocal per block and a fused multiply-add correction instead of a
division per element, and this is where that has to agree with IEEE
division.
"""
import numpy as np
import pytest
import torch

import combine_ep_get_dispatch_gb300 as ep
import oracle

pytestmark = pytest.mark.gpu

H = 128 * 64           # 64 blocks per row
A_MAX = 0x7F7F         # largest finite positive BF16


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    oracle.use_all_cores(True)     # same results, every host core
    yield
    oracle.use_all_cores(False)


def _blocks(a_bits: np.ndarray, negative: bool) -> torch.Tensor:
    """[blocks, 128] BF16 bit patterns (int16, on the device): channel 0 = a,
    then the x bits 0..a (sign set if negative) in runs of 127, the last run
    padded with zeros. Built on the device: it is input generation only."""
    a = torch.from_numpy(a_bits.astype(np.int64)).cuda()
    n_blk = (a + 127) // 127
    nb = int(n_blk.sum().item())
    blk_a = torch.repeat_interleave(a, n_blk)
    start = torch.repeat_interleave(torch.cumsum(n_blk, 0) - n_blk, n_blk)
    first = (torch.arange(nb, device="cuda", dtype=torch.int64) - start) * 127
    xb = first[:, None] + torch.arange(127, device="cuda", dtype=torch.int64)[None, :]
    xb = torch.where(xb <= blk_a[:, None], xb, torch.zeros_like(xb))
    out = torch.empty((nb, 128), dtype=torch.int64, device="cuda")
    out[:, 0] = blk_a
    out[:, 1:] = xb | (0x8000 if negative else 0)
    out = torch.where(out >= 0x8000, out - 0x10000, out)   # uint16 bit patterns as int16 values
    return out.to(torch.int16)


def _check(blocks: torch.Tensor, flags: int):
    nb = blocks.shape[0]
    pad = (-nb) % (H // 128)
    if pad:
        blocks = torch.cat([blocks, torch.zeros((pad, 128), dtype=torch.int16, device="cuda")])
    xd = blocks.reshape(-1, H).contiguous()
    ue8m0 = bool(flags & ep.EP_FP8_UE8M0)
    q = torch.empty(xd.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty((xd.shape[0], H // 128), dtype=torch.uint8 if ue8m0 else torch.float32, device="cuda")
    ep.ep_fp8_quantize(xd.view(torch.bfloat16), q, s, flags)
    x = xd.cpu().numpy().view(np.uint16)
    rq, rs = oracle.quantize_rows(x, round_scale=bool(flags & ep.EP_FP8_ROUND_SCALE), ue8m0=ue8m0)
    if ue8m0:
        rs = oracle.ue8m0_from_scales(rs)
    gq = q.cpu().numpy()
    bad = np.nonzero((gq != rq).any(axis=1))[0]
    assert bad.size == 0, f"codes differ in row {bad[:4]}"
    assert np.array_equal(s.cpu().numpy(), rs)
    return nb


def _expected_blocks(a_all: np.ndarray) -> int:
    return int(((a_all.astype(np.int64) + 127) // 127).sum())


def _chunks(a_all: np.ndarray, max_blocks: int = 1 << 18):
    n_blk = (a_all.astype(np.int64) + 1 + 126) // 127
    cum = np.cumsum(n_blk)
    lo = 0
    while lo < a_all.size:
        base = cum[lo - 1] if lo else 0
        hi = int(np.searchsorted(cum, base + max_blocks, side="right"))
        hi = max(hi, lo + 1)
        yield a_all[lo:hi]
        lo = hi


def test_every_nonnegative_x_against_every_amax():
    a_all = np.arange(1, A_MAX + 1, dtype=np.int64)
    done = sum(_check(_blocks(a, negative=False), ep.EP_FP8) for a in _chunks(a_all))
    assert done == _expected_blocks(a_all) > 4_000_000      # about 539 M elements


def test_negative_x_on_every_16th_amax():
    a_all = np.arange(1, A_MAX + 1, 16, dtype=np.int64)
    done = sum(_check(_blocks(a, negative=True), ep.EP_FP8) for a in _chunks(a_all))
    assert done == _expected_blocks(a_all) > 250_000


@pytest.mark.parametrize("flags", [ep.EP_FP8 | ep.EP_FP8_ROUND_SCALE, ep.EP_FP8 | ep.EP_FP8_UE8M0])
def test_power_of_two_scales_on_every_16th_amax(flags):
    a_all = np.arange(3, A_MAX + 1, 16, dtype=np.int64)
    done = sum(_check(_blocks(a, negative=False), flags) for a in _chunks(a_all))
    assert done == _expected_blocks(a_all) > 250_000


def test_all_zero_and_signed_zero_blocks():
    x = torch.zeros((2, H), dtype=torch.int16, device="cuda")
    x[1, ::2] = -0x8000                     # -0.0
    _check(x.reshape(-1, 128), ep.EP_FP8)
