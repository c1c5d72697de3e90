"""GB300 (sm_103a) MoE token layout, dispatch and combine.

A thin Python binding over the C ABI of libep_gb300.so (include/ep.h). It
only marshals arguments: PyTorch provides device memory and the current CUDA
stream, every step runs in the library's own CUDA kernels. There is no CPU
fallback: if the library is missing, importing the functions that need it
raises.

Two layers:

* ``ep_*`` functions with the C ABI's names and arguments (raw tensors);
* the page-level calls of the DeepEP API shape: ``get_dispatch_layout``,
  ``dispatch``, ``combine``, ``low_latency_dispatch(..., return_recv_hook=True)``
  (returning a hook that launches the receive phase) and
  ``low_latency_combine`` ("DeepEP V1 (legacy) guide", sections 5.1 and 6.1;
  "How DeepEP enables hook-based overlapping", "Implementing Hook-Based
  Overlap in Practice").
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Callable, Optional, Tuple

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libep_gb300.so")

EP_OK = 0
EP_ERR_INVALID_ARG = -1
EP_ERR_ALIGNMENT = -2
EP_ERR_WORKSPACE = -3
EP_ERR_LL_CAPACITY = -4
EP_ERR_CUDA = -5
EP_ERR_UNSUPPORTED = -6

EP_ST_BAD_INDEX = 0x1
EP_ST_CAPACITY = 0x2
EP_ST_LL_OVERFLOW = 0x4
EP_ST_TIMEOUT = 0x8
EP_ST_NOT_SENT = 0x10
EP_ST_MISMATCH = 0x20
EP_ST_WORKSPACE = 0x40

EP_FP8 = 0x1
EP_FP8_ROUND_SCALE = 0x2
EP_FP8_UE8M0 = 0x4

EP_MAX_EXPERTS = 1024
EP_MAX_TOPK = 32
EP_MAX_HIDDEN = 16384


class EPError(RuntimeError):
    """A non-zero return code of the C ABI."""

    def __init__(self, what: str, code: int):
        super().__init__(f"{what}: {ep_error_string(code)} (code {code})")
        self.code = code


class ep_layout_t(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int32),
        ("num_topk", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("num_ranks", ctypes.c_int32),
        ("topk_idx", ctypes.c_void_p),
        ("num_tokens_per_rank", ctypes.c_void_p),
        ("num_tokens_per_expert", ctypes.c_void_p),
        ("is_token_in_rank", ctypes.c_void_p),
        ("rank_offset", ctypes.c_void_p),
        ("expert_offset", ctypes.c_void_p),
        ("rank_slot", ctypes.c_void_p),
        ("expert_slot", ctypes.c_void_p),
        ("expert_alignment", ctypes.c_int32),
    ]


class ep_recv_buffer_t(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("src_idx", ctypes.c_void_p),
        ("topk_idx", ctypes.c_void_p),
        ("topk_weights", ctypes.c_void_p),
        ("capacity", ctypes.c_int64),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` or "
            "`python combine_ep_get_dispatch_gb300/build.py`")
    L = ctypes.CDLL(LIB_PATH)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "ep_version": (I, []),
        "ep_error_string": (ctypes.c_char_p, [I]),
        "ep_layout_workspace_bytes": (SZ, [I, I, I, I]),
        "ep_get_dispatch_layout": (I, [ctypes.POINTER(ep_layout_t), P, SZ, P, P]),
        "ep_dispatch": (I, [ctypes.POINTER(ep_layout_t), P, I, I, P, ctypes.POINTER(ep_recv_buffer_t),
                            ctypes.POINTER(ep_recv_buffer_t), P, P]),
        "ep_layout_dispatch": (I, [ctypes.POINTER(ep_layout_t), P, SZ, P, I, I, P, ctypes.POINTER(ep_recv_buffer_t),
                                   ctypes.POINTER(ep_recv_buffer_t), P, P]),
        "ep_combine": (I, [ctypes.POINTER(ep_layout_t), P, I64, I, P, P, P, P, P]),
        "ep_combine_to_ranks": (I, [ctypes.POINTER(ep_layout_t), P, I64, I, P, P, I64, P, P]),
        "ep_combine_ranks": (I, [ctypes.POINTER(ep_layout_t), P, I64, I, P, P, P, P]),
        "ep_combine_backward": (I, [ctypes.POINTER(ep_layout_t), P, P, I64, I, P, P, P, P, P]),
        "ep_ll_workspace_bytes": (SZ, [I, I, I, I, I]),
        "ep_ll_dispatch_send": (I, [P, P, I, I, I, I, I, I, I, P, P, P, P, SZ, P, P]),
        "ep_ll_dispatch_recv": (I, [P, SZ, I, I, I, I, I, P, P, P, P, P]),
        "ep_ll_combine": (I, [P, P, P, P, SZ, I, I, I, I, I, I, P, P, P]),
        "ep_fp8_e4m3_encode": (I, [P, P, I64, P]),
        "ep_fp8_quantize": (I, [P, I64, I, I, P, P, P]),
        "ep_ll_combine_send": (I, [P, P, SZ, I, I, I, I, I, I, P, P, P]),
        "ep_ll_combine_recv": (I, [P, P, P, P, SZ, I, I, I, I, I, I, P, P, P]),
        "ep_ll_update_mask": (I, [P, SZ, I, I, I, P]),
        "ep_ll_query_mask": (I, [P, SZ, I, P, P]),
        "ep_ll_clean_mask": (I, [P, SZ, I, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def ep_error_string(code: int) -> str:
    try:
        return lib().ep_error_string(int(code)).decode()
    except RuntimeError:
        return f"code {code}"


def _check(rc: int, what: str) -> None:
    if rc != EP_OK:
        raise EPError(what, rc)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        if _raw_stream is not None:   # the current stream's handle without building a Stream object
            return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ---------------------------------------------------------------- handles ----
@dataclasses.dataclass
class Layout:
    """Routing layout of one batch (the handle of dispatch and combine)."""
    topk_idx: torch.Tensor
    num_experts: int
    num_ranks: int
    num_tokens_per_rank: torch.Tensor
    num_tokens_per_expert: torch.Tensor
    is_token_in_rank: torch.Tensor
    rank_offset: torch.Tensor
    expert_offset: torch.Tensor
    rank_slot: torch.Tensor
    expert_slot: torch.Tensor
    expert_alignment: int = 1
    _c: Optional[ep_layout_t] = dataclasses.field(default=None, init=False, repr=False, compare=False)

    def c_struct(self) -> ep_layout_t:
        """The C handle, built once: a Layout's arrays are fixed when it is made."""
        if self._c is None:
            N, K = self.topk_idx.shape
            self._c = ep_layout_t(N, K, self.num_experts, self.num_ranks, _p(self.topk_idx),
                                  _p(self.num_tokens_per_rank), _p(self.num_tokens_per_expert),
                                  _p(self.is_token_in_rank), _p(self.rank_offset), _p(self.expert_offset),
                                  _p(self.rank_slot), _p(self.expert_slot), int(self.expert_alignment))
        return self._c

    @property
    def num_recv_tokens_per_expert_list(self) -> torch.Tensor:
        """Per-rank view of the expert counts: [num_ranks, num_local_experts]."""
        return self.num_tokens_per_expert.view(self.num_ranks, -1)


def new_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int, expert_alignment: int = 1) -> Layout:
    N, K = topk_idx.shape
    dev = topk_idx.device
    i32 = dict(dtype=torch.int32, device=dev)
    return Layout(topk_idx, num_experts, num_ranks,
                  torch.empty(num_ranks, **i32), torch.empty(num_experts, **i32),
                  torch.empty((N, num_ranks), dtype=torch.uint8, device=dev),
                  torch.empty(num_ranks + 1, **i32), torch.empty(num_experts + 1, **i32),
                  torch.empty((N, num_ranks), **i32), torch.empty((N, K), **i32), expert_alignment)


def fp8_flags(use_fp8: bool, round_scale: bool = False, use_ue8m0: bool = False) -> int:
    """The `fp8_flags` argument of ep_dispatch / ep_ll_dispatch_send."""
    if not use_fp8:
        return 0
    return EP_FP8 | (EP_FP8_ROUND_SCALE if round_scale else 0) | (EP_FP8_UE8M0 if use_ue8m0 else 0)


def _recv_struct(x, scales=None, src=None, topk_idx=None, topk_w=None) -> ep_recv_buffer_t:
    return ep_recv_buffer_t(_p(x), _p(scales), _p(src), _p(topk_idx), _p(topk_w),
                            x.shape[0] if x is not None else 0)


# ------------------------------------------------------------- C ABI names ----
def ep_layout_workspace_bytes(N: int, K: int, E: int, R: int) -> int:
    return int(lib().ep_layout_workspace_bytes(N, K, E, R))


def ep_ll_workspace_bytes(N: int, K: int, E: int, R: int, T: int) -> int:
    return int(lib().ep_ll_workspace_bytes(N, K, E, R, T))


def ep_get_dispatch_layout(layout: Layout, workspace: torch.Tensor, status: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    c = layout.c_struct()
    _check(lib().ep_get_dispatch_layout(ctypes.byref(c), _p(workspace), workspace.numel(),
                                         _p(status), _stream(stream)), "ep_get_dispatch_layout")


def ep_dispatch(layout: Layout, x: torch.Tensor, fp8: int, topk_weights: Optional[torch.Tensor],
                rank_buf: Optional[ep_recv_buffer_t], expert_buf: Optional[ep_recv_buffer_t],
                status: Optional[torch.Tensor] = None, stream=None) -> None:
    """fp8: 0 / False (BF16), 1 / True (EP_FP8) or an EP_FP8 | ... flags word."""
    c = layout.c_struct()
    rb = ctypes.byref(rank_buf) if rank_buf is not None else None
    eb = ctypes.byref(expert_buf) if expert_buf is not None else None
    _check(lib().ep_dispatch(ctypes.byref(c), _p(x), x.shape[1], int(fp8), _p(topk_weights), rb, eb,
                             _p(status), _stream(stream)), "ep_dispatch")


def ep_layout_dispatch(layout: Layout, workspace: torch.Tensor, x: torch.Tensor, fp8: int,
                       topk_weights: Optional[torch.Tensor], rank_buf: Optional[ep_recv_buffer_t],
                       expert_buf: Optional[ep_recv_buffer_t], status: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """ep_get_dispatch_layout then ep_dispatch in one call (the dispatch overlaps the layout)."""
    c = layout.c_struct()
    rb = ctypes.byref(rank_buf) if rank_buf is not None else None
    eb = ctypes.byref(expert_buf) if expert_buf is not None else None
    _check(lib().ep_layout_dispatch(ctypes.byref(c), _p(workspace), workspace.numel(), _p(x), x.shape[1],
                                    int(fp8), _p(topk_weights), rb, eb, _p(status), _stream(stream)),
           "ep_layout_dispatch")


def ep_combine(layout: Layout, expert_y: torch.Tensor, topk_weights: torch.Tensor, out: torch.Tensor,
               status: Optional[torch.Tensor] = None, stream=None, bias: Optional[torch.Tensor] = None) -> None:
    c = layout.c_struct()
    _check(lib().ep_combine(ctypes.byref(c), _p(expert_y), expert_y.shape[0], expert_y.shape[1],
                            _p(topk_weights), _p(bias), _p(out), _p(status), _stream(stream)), "ep_combine")


def ep_combine_to_ranks(layout: Layout, expert_y: torch.Tensor, topk_weights: torch.Tensor,
                        rank_out: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None) -> None:
    c = layout.c_struct()
    _check(lib().ep_combine_to_ranks(ctypes.byref(c), _p(expert_y), expert_y.shape[0], expert_y.shape[1],
                                     _p(topk_weights), _p(rank_out), rank_out.shape[0], _p(status),
                                     _stream(stream)), "ep_combine_to_ranks")


def ep_combine_backward(layout: Layout, grad_out: torch.Tensor, expert_y: Optional[torch.Tensor],
                        topk_weights: torch.Tensor, grad_y: Optional[torch.Tensor], grad_w: Optional[torch.Tensor],
                        status: Optional[torch.Tensor] = None, stream=None) -> None:
    c = layout.c_struct()
    ref = expert_y if expert_y is not None else grad_y
    rows = ref.shape[0] if ref is not None else 0
    _check(lib().ep_combine_backward(ctypes.byref(c), _p(grad_out), _p(expert_y), rows, grad_out.shape[1],
                                     _p(topk_weights), _p(grad_y), _p(grad_w), _p(status), _stream(stream)),
           "ep_combine_backward")


def ep_combine_ranks(layout: Layout, rank_y: torch.Tensor, out: torch.Tensor, status: Optional[torch.Tensor] = None,
                     stream=None, bias: Optional[torch.Tensor] = None) -> None:
    c = layout.c_struct()
    _check(lib().ep_combine_ranks(ctypes.byref(c), _p(rank_y), rank_y.shape[0], rank_y.shape[1], _p(bias),
                                  _p(out), _p(status), _stream(stream)), "ep_combine_ranks")


def ep_ll_dispatch_send(x, topk_idx, H, E, R, T, fp8, recv_x, recv_scales, recv_src, workspace,
                        status=None, stream=None) -> None:
    N, K = topk_idx.shape
    _check(lib().ep_ll_dispatch_send(_p(x), _p(topk_idx), N, K, H, E, R, T, int(fp8), _p(recv_x),
                                     _p(recv_scales), _p(recv_src), _p(workspace), workspace.numel(),
                                     _p(status), _stream(stream)), "ep_ll_dispatch_send")


def ep_ll_dispatch_recv(workspace, N, K, E, R, T, recv_count, layout_range=None, status=None,
                        stream=None, cumulative_recv_stats=None) -> None:
    _check(lib().ep_ll_dispatch_recv(_p(workspace), workspace.numel(), N, K, E, R, T, _p(recv_count),
                                     _p(layout_range), _p(cumulative_recv_stats), _p(status), _stream(stream)),
           "ep_ll_dispatch_recv")


def ep_ll_combine(expert_y, topk_weights, workspace, N, K, H, E, R, T, out, status=None,
                  stream=None, bias=None) -> None:
    _check(lib().ep_ll_combine(_p(expert_y), _p(topk_weights), _p(bias), _p(workspace), workspace.numel(), N, K,
                               H, E, R, T, _p(out), _p(status), _stream(stream)), "ep_ll_combine")


def ep_ll_combine_send(expert_y, workspace, N, K, H, E, R, T, staging, status=None, stream=None) -> None:
    _check(lib().ep_ll_combine_send(_p(expert_y), _p(workspace), workspace.numel(), N, K, H, E, R, T,
                                    _p(staging), _p(status), _stream(stream)), "ep_ll_combine_send")


def ep_ll_combine_recv(staging, topk_weights, workspace, N, K, H, E, R, T, out, status=None,
                       stream=None, bias=None) -> None:
    _check(lib().ep_ll_combine_recv(_p(staging), _p(topk_weights), _p(bias), _p(workspace), workspace.numel(), N,
                                    K, H, E, R, T, _p(out), _p(status), _stream(stream)), "ep_ll_combine_recv")


def ep_ll_update_mask(workspace, R, rank, masked=True, stream=None) -> None:
    _check(lib().ep_ll_update_mask(_p(workspace), workspace.numel(), R, rank, int(bool(masked)),
                                   _stream(stream)), "ep_ll_update_mask")


def ep_ll_query_mask(workspace, R, out=None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(R, dtype=torch.int32, device=workspace.device)
    _check(lib().ep_ll_query_mask(_p(workspace), workspace.numel(), R, _p(out), _stream(stream)),
           "ep_ll_query_mask")
    return out


def ep_ll_clean_mask(workspace, R, stream=None) -> None:
    _check(lib().ep_ll_clean_mask(_p(workspace), workspace.numel(), R, _stream(stream)), "ep_ll_clean_mask")


def ep_fp8_e4m3_encode(x: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _check(lib().ep_fp8_e4m3_encode(_p(x), _p(out), x.numel(), _stream(stream)), "ep_fp8_e4m3_encode")


def ep_fp8_quantize(x: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, fp8: int = EP_FP8, stream=None) -> None:
    """x [rows, H] bf16 -> q [rows, H] uint8 (E4M3) and scales [rows, H/128] (fp32, or uint8 UE8M0)."""
    _check(lib().ep_fp8_quantize(_p(x), x.shape[0], x.shape[1], int(fp8), _p(q), _p(scales), _stream(stream)),
           "ep_fp8_quantize")


# -------------------------------------------------------------- page-level ----
def _status(dev) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=dev)


def get_dispatch_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int,
                        status: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None, expert_alignment: int = 1) -> Layout:
    """Counts, is_token_in_rank mask and slots for a [N, K] int32 topk_idx.

    expert_alignment A > 1 pads each expert's expert-major segment to a
    multiple of A rows (dispatch zero-fills the padding rows). A workspace
    passed in must have been zero-filled once when it was allocated (each
    call leaves it ready for the next); without one, a zeroed one is made.
    """
    topk_idx = topk_idx.to(torch.int32).contiguous()
    N, K = topk_idx.shape
    layout = new_layout(topk_idx, num_experts, num_ranks, expert_alignment)
    need = ep_layout_workspace_bytes(N, K, num_experts, num_ranks)
    if need == 0:
        raise EPError("get_dispatch_layout", EP_ERR_INVALID_ARG)
    if workspace is None or workspace.numel() < need:
        workspace = torch.zeros(need, dtype=torch.uint8, device=topk_idx.device)
    ep_get_dispatch_layout(layout, workspace, status, stream)
    return layout


@dataclasses.dataclass
class DispatchResult:
    rank_x: Optional[torch.Tensor] = None        # [cap_r, H] bf16 or uint8 (E4M3)
    rank_scales: Optional[torch.Tensor] = None   # [cap_r, H/128] fp32
    rank_src: Optional[torch.Tensor] = None      # [cap_r] int32 token index
    rank_topk_idx: Optional[torch.Tensor] = None  # [cap_r, K] local expert id or -1
    rank_topk_weights: Optional[torch.Tensor] = None
    expert_x: Optional[torch.Tensor] = None      # [cap_e, H]
    expert_scales: Optional[torch.Tensor] = None
    expert_src: Optional[torch.Tensor] = None    # [cap_e] int32 t*K + k


def _recv_buffers(x: torch.Tensor, layout: Layout, topk_weights: Optional[torch.Tensor], use_fp8: bool,
                  use_ue8m0: bool, with_rank: bool, with_expert: bool, cap_r: int, cap_e: int):
    """Receive buffers of a dispatch (capacities cap_r, cap_e rows) and their C structs."""
    H = x.shape[1]
    K = layout.topk_idx.shape[1]
    dev = x.device
    xdt = torch.uint8 if use_fp8 else torch.bfloat16
    sdt = torch.uint8 if use_ue8m0 else torch.float32
    S = H // 128
    res = DispatchResult()
    rb = eb = None
    if with_rank:
        res.rank_x = torch.empty((cap_r, H), dtype=xdt, device=dev)
        res.rank_scales = torch.empty((cap_r, S), dtype=sdt, device=dev) if use_fp8 else None
        res.rank_src = torch.empty(cap_r, dtype=torch.int32, device=dev)
        res.rank_topk_idx = torch.empty((cap_r, K), dtype=torch.int32, device=dev)
        res.rank_topk_weights = torch.empty((cap_r, K), dtype=torch.float32, device=dev) \
            if topk_weights is not None else None
        rb = _recv_struct(res.rank_x, res.rank_scales, res.rank_src, res.rank_topk_idx,
                          res.rank_topk_weights)
    if with_expert:
        res.expert_x = torch.empty((cap_e, H), dtype=xdt, device=dev)
        res.expert_scales = torch.empty((cap_e, S), dtype=sdt, device=dev) if use_fp8 else None
        res.expert_src = torch.empty(cap_e, dtype=torch.int32, device=dev)
        eb = _recv_struct(res.expert_x, res.expert_scales, res.expert_src)
    return res, rb, eb


def _worst_case_caps(N: int, layout: Layout):
    K = layout.topk_idx.shape[1]
    A = max(1, layout.expert_alignment)
    return N * min(K, layout.num_ranks), N * K + layout.num_experts * (A - 1)


def dispatch(x: torch.Tensor, layout: Layout, topk_weights: Optional[torch.Tensor] = None,
             use_fp8: bool = False, with_rank: bool = True, with_expert: bool = True,
             exact: bool = False, status: Optional[torch.Tensor] = None, stream=None,
             round_scale: bool = False, use_ue8m0: bool = False) -> DispatchResult:
    """Scatter x [N, H] bf16 into per-rank and expert-major receive buffers.

    exact=False sizes the buffers for the worst case (N*min(K,R) and N*K
    rows), with no host synchronisation; exact=True reads the counts first
    (one device->host copy) and sizes them exactly.
    """
    if exact:
        cap_r = int(layout.rank_offset[-1].item())
        cap_e = int(layout.expert_offset[-1].item())
    else:
        cap_r, cap_e = _worst_case_caps(x.shape[0], layout)
    res, rb, eb = _recv_buffers(x, layout, topk_weights, use_fp8, use_ue8m0, with_rank, with_expert, cap_r, cap_e)
    tw = topk_weights.contiguous() if topk_weights is not None else None
    ep_dispatch(layout, x.contiguous(), fp8_flags(use_fp8, round_scale, use_ue8m0), tw, rb, eb, status, stream)
    return res


def get_layout_and_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, num_experts: int, num_ranks: int,
                            topk_weights: Optional[torch.Tensor] = None, use_fp8: bool = False,
                            with_rank: bool = True, with_expert: bool = True,
                            status: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                            stream=None, expert_alignment: int = 1, round_scale: bool = False,
                            use_ue8m0: bool = False):
    """get_dispatch_layout and dispatch in one library call (ep_layout_dispatch).

    Returns (layout, DispatchResult). The dispatch overlaps the layout on the
    GPU; the receive buffers are sized for the worst case, since the counts
    are not known before the call.
    """
    topk_idx = topk_idx.to(torch.int32).contiguous()
    N, K = topk_idx.shape
    layout = new_layout(topk_idx, num_experts, num_ranks, expert_alignment)
    need = ep_layout_workspace_bytes(N, K, num_experts, num_ranks)
    if need == 0:
        raise EPError("get_layout_and_dispatch", EP_ERR_INVALID_ARG)
    if workspace is None or workspace.numel() < need:
        workspace = torch.zeros(need, dtype=torch.uint8, device=topk_idx.device)
    cap_r, cap_e = _worst_case_caps(N, layout)
    res, rb, eb = _recv_buffers(x, layout, topk_weights, use_fp8, use_ue8m0, with_rank, with_expert, cap_r, cap_e)
    tw = topk_weights.contiguous() if topk_weights is not None else None
    ep_layout_dispatch(layout, workspace, x.contiguous(), fp8_flags(use_fp8, round_scale, use_ue8m0), tw, rb, eb,
                       status, stream)
    return layout, res


def combine(expert_y: torch.Tensor, layout: Layout, topk_weights: torch.Tensor,
            out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
            stream=None, bias: Optional[torch.Tensor] = None) -> torch.Tensor:
    """out [N, H] bf16 = sum_k w[t,k] * expert_y[expert_slot[t,k]] (+ bias), fp32 accumulation."""
    N = layout.topk_idx.shape[0]
    if out is None:
        out = torch.empty((N, expert_y.shape[1]), dtype=torch.bfloat16, device=expert_y.device)
    b = bias.contiguous() if bias is not None else None
    ep_combine(layout, expert_y.contiguous(), topk_weights.contiguous(), out, status, stream, bias=b)
    return out


def dispatch_backward(grad_expert_x: torch.Tensor, layout: Layout, status: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """grad_x [N, H] bf16: the unit-weight sum of each token's expert-major row gradients."""
    N = layout.topk_idx.shape[0]
    out = torch.empty((N, grad_expert_x.shape[1]), dtype=torch.bfloat16, device=grad_expert_x.device)
    c = layout.c_struct()
    g = grad_expert_x.contiguous()
    _check(lib().ep_combine(ctypes.byref(c), _p(g), g.shape[0], g.shape[1], None, None, _p(out), _p(status),
                            _stream(stream)), "ep_combine")
    return out


def combine_backward(grad_out: torch.Tensor, layout: Layout, expert_y: torch.Tensor, topk_weights: torch.Tensor,
                     status: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """(grad_y [rows, H] bf16, grad_w [N, K] fp32) of out = sum_k w * expert_y[expert_slot]."""
    grad_y = torch.zeros_like(expert_y)
    grad_w = torch.empty_like(topk_weights, dtype=torch.float32)
    ep_combine_backward(layout, grad_out.contiguous(), expert_y.contiguous(), topk_weights.contiguous(), grad_y,
                        grad_w, status, stream)
    return grad_y, grad_w


def combine_two_level(expert_y: torch.Tensor, layout: Layout, topk_weights: torch.Tensor,
                      bias: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                      stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-rank pre-sums (one row per (token, rank)) then the cross-rank sum.

    Returns (out [N, H], rank_rows [D_r, H]); reads the per-rank row count
    from the layout (one device->host copy).
    """
    N = layout.topk_idx.shape[0]
    H = expert_y.shape[1]
    D_r = int(layout.rank_offset[-1].item())
    rank_rows = torch.empty((D_r, H), dtype=torch.bfloat16, device=expert_y.device)
    ep_combine_to_ranks(layout, expert_y.contiguous(), topk_weights.contiguous(), rank_rows, status, stream)
    out = torch.empty((N, H), dtype=torch.bfloat16, device=expert_y.device)
    b = bias.contiguous() if bias is not None else None
    ep_combine_ranks(layout, rank_rows, out, status, stream, bias=b)
    return out, rank_rows


@dataclasses.dataclass
class LLHandle:
    """Routing of one low-latency batch: the workspace the send filled."""
    workspace: torch.Tensor
    N: int
    K: int
    H: int
    E: int
    R: int
    T: int
    recv_src: torch.Tensor
    layout_range: torch.Tensor


def low_latency_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, num_max_dispatch_tokens_per_rank: int,
                         num_experts: int, num_ranks: int, use_fp8: bool = True,
                         return_recv_hook: bool = True, status: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, stream=None,
                         round_scale: bool = False, use_ue8m0: bool = False,
                         cumulative_local_expert_recv_stats: Optional[torch.Tensor] = None):
    """Fixed-shape low-latency dispatch.

    Returns (recv_x, recv_count, handle, hook): recv_x is a [E, R*T, H] bf16
    tensor, or a (E4M3 uint8 [E, R*T, H], fp32 scales [E, R*T, H/128]) tuple;
    recv_count [E] int32 is valid once the hook has run. With
    return_recv_hook=False the receive phase is launched at once and hook is
    None.
    """
    N, H = x.shape
    K = topk_idx.shape[1]
    E, R, T = num_experts, num_ranks, num_max_dispatch_tokens_per_rank
    dev = x.device
    need = ep_ll_workspace_bytes(N, K, E, R, T)
    if need == 0:
        raise EPError("low_latency_dispatch", EP_ERR_INVALID_ARG)
    if workspace is None or workspace.numel() < need:
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    recv_x = torch.empty((E, R * T, H), dtype=torch.uint8 if use_fp8 else torch.bfloat16, device=dev)
    recv_scales = torch.empty((E, R * T, H // 128), dtype=torch.uint8 if use_ue8m0 else torch.float32,
                              device=dev) if use_fp8 else None
    recv_src = torch.empty((E, R * T), dtype=torch.int32, device=dev)
    recv_count = torch.empty(E, dtype=torch.int32, device=dev)
    layout_range = torch.empty((E, R), dtype=torch.int64, device=dev)
    idx = topk_idx.to(torch.int32).contiguous()
    ep_ll_dispatch_send(x.contiguous(), idx, H, E, R, T, fp8_flags(use_fp8, round_scale, use_ue8m0), recv_x,
                        recv_scales, recv_src, workspace, status, stream)
    handle = LLHandle(workspace, N, K, H, E, R, T, recv_src, layout_range)

    def hook() -> None:
        ep_ll_dispatch_recv(workspace, N, K, E, R, T, recv_count, layout_range, status, stream,
                            cumulative_local_expert_recv_stats)

    out_x = (recv_x, recv_scales) if use_fp8 else recv_x
    if not return_recv_hook:
        hook()
        return out_x, recv_count, handle, None
    return out_x, recv_count, handle, hook


def low_latency_combine(expert_y: torch.Tensor, topk_weights: torch.Tensor, handle: LLHandle,
                        out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                        return_recv_hook: bool = False, stream=None, bias: Optional[torch.Tensor] = None):
    """out [N, H] bf16 from expert outputs in the [E, R*T, H] receive layout.

    return_recv_hook=False: one launch, returns out. True: the send phase
    gathers the rows back into a token-major staging buffer now and the
    returned hook runs the weighted sum; returns (out, hook), out valid after
    hook() ("DeepEP V1 (legacy) guide", section 6.1).
    """
    h = handle
    if out is None:
        out = torch.empty((h.N, h.H), dtype=torch.bfloat16, device=expert_y.device)
    y = expert_y.contiguous()
    w = topk_weights.contiguous()
    b = bias.contiguous() if bias is not None else None
    if not return_recv_hook:
        ep_ll_combine(y, w, h.workspace, h.N, h.K, h.H, h.E, h.R, h.T, out, status, stream, bias=b)
        return out
    staging = torch.empty((h.N * h.K, h.H), dtype=torch.bfloat16, device=y.device)
    ep_ll_combine_send(y, h.workspace, h.N, h.K, h.H, h.E, h.R, h.T, staging, status, stream)

    def hook() -> None:
        ep_ll_combine_recv(staging, w, h.workspace, h.N, h.K, h.H, h.E, h.R, h.T, out, status, stream, bias=b)

    return out, hook


# ------------------------------------------------- shrink mode (rank masks) ----
def _ws_ranks(handle, num_ranks):
    if isinstance(handle, LLHandle):
        return handle.workspace, handle.R
    if num_ranks is None:
        raise ValueError("num_ranks is needed with a bare workspace tensor")
    return handle, num_ranks


def low_latency_update_mask_buffer(handle, rank: int, mask: bool = True, num_ranks: Optional[int] = None,
                                   stream=None) -> None:
    """Shrink mode ("DeepEP V1 (legacy) guide", section 6.4): mask (or, with
    mask=False, restore) rank `rank` in the low-latency workspace. handle is
    an LLHandle or the workspace tensor itself (then num_ranks is needed).
    Sends on that workspace drop every slot whose expert lives on a masked
    rank or whose token comes from one; combines skip them as well."""
    ws, R = _ws_ranks(handle, num_ranks)
    ep_ll_update_mask(ws, R, rank, mask, stream)


def low_latency_query_mask_buffer(handle, num_ranks: Optional[int] = None, stream=None) -> torch.Tensor:
    """The current rank mask, [R] int32 on the device (non-zero = masked)."""
    ws, R = _ws_ranks(handle, num_ranks)
    return ep_ll_query_mask(ws, R, stream=stream)


def low_latency_clean_mask_buffer(handle, num_ranks: Optional[int] = None, stream=None) -> None:
    """Restore every rank."""
    ws, R = _ws_ranks(handle, num_ranks)
    ep_ll_clean_mask(ws, R, stream)
