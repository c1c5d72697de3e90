"""Benchmark: MoE layout -> dispatch -> combine on one GB300 (or N replicas).

One step is one pass of the whole hot path over one batch of a workload.
The default workload is the large prefill (16384 tokens, hidden 7168 BF16,
256 experts top-6, 8 logical ranks): the routing layout, dispatch into the
per-rank and the expert-major receive buffers (BF16), and combine of
identity expert outputs (the expert-major rows) back into [16384, 7168] BF16.

--workload 1..5 selects the other synthetic workloads (same JSON line):
  3, 5  prefill with FP8 dispatch: layout, FP8 dispatch (per-rank and
        expert-major, E4M3 + per-128-channel scales), combine of BF16 expert
        outputs (a fixed BF16 buffer in the expert-major layout);
  1, 2  low latency: send, receive (the hook), combine of BF16 expert outputs
        in the fixed [E, R*T, H] layout.

Prints one JSON line (rank 0). `value` is tokens/s of the whole job with
inputs resident in HBM; `e2e` is the same through the C ABI from pinned host
buffers, with the host->device copy of x / topk_idx / topk_weights and the
device->host copy of the combined output of every step inside the timed
region (pipelined: a step's copies overlap its neighbours' compute).

--impl reference times the CPU oracle (plain single-threaded C++) on the same
workload, each step a bounded sample of tokens.

The default run (the large prefill workload, no variant flags) also measures
workloads 1, 2, 3 and 5 the same way and reports them under `workloads`.
`cpu_baseline` is the oracle on every host core, with its single-core figure
beside it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import epinputs as ei  # noqa: E402

METRIC = "dispatch+combine tokens/s and HBM GB/s (% of GB300 peak) at 1 GPU"
DEFAULT_WORKLOAD = 4          # the 16384-token large prefill workload
L2_FLUSH_BYTES = 256 << 20
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "dispatch_traffic.json")
NOMINAL_HBM_GBS = 8000.0      # GB300's ~8 TB/s nominal HBM3e bandwidth (context beside the measured peak)
EXTRA_WORKLOADS = (1, 2, 3, 5)  # measured in the default run beside the headline workload
KERNEL_SOURCES = [os.path.join(ROOT, "combine_ep_get_dispatch_gb300", "csrc", f)
                  for f in ("dispatch.cu", "common.cuh", "kernels.cuh")]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(ei.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=None, help="override the token count (profiling runs)")
    ap.add_argument("--fp8-scales", default="fp32", choices=["fp32", "pow2", "ue8m0"],
                    help="FP8 workloads: fp32 scales, power-of-two fp32 scales, or UE8M0 bytes")
    ap.add_argument("--expert-alignment", type=int, default=1,
                    help="normal workloads: pad each expert's segment to a multiple of this many rows")
    ap.add_argument("--combine-bias", action="store_true", help="add a shared-expert BF16 row in combine")
    ap.add_argument("--combine", default="flat", choices=["flat", "two-level"],
                    help="normal workloads: one weighted sum, or per-rank pre-sums then the cross-rank sum")
    ap.add_argument("--training", action="store_true",
                    help="normal workloads: also the backward passes (combine backward, then dispatch backward)")
    ap.add_argument("--ll-combine", default="one-phase", choices=["one-phase", "two-phase"],
                    help="low-latency workloads: combine in one launch, or send + receive hook")
    ap.add_argument("--mask-ranks", default="",
                    help="low-latency workloads: comma-separated ranks masked in the workspace (shrink mode)")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured once in a CUDA graph and replayed (reported as `graph`)")
    ap.add_argument("--fused-layout", action="store_true",
                    help="normal workloads: layout and dispatch through one call (ep_layout_dispatch), timed as one phase")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=None,
                    help="tokens of the workload the oracle baseline runs on (default: all of them); its time "
                         "is bounded by repetitions, about 10 s on every core and 5 s on one")
    ap.add_argument("--l2-flush", default="write", choices=["write", "write-read"],
                    help="between steps: write 256 MiB (default), or write it and read it back so that no "
                         "dirty line of the flush is left in L2 when the step starts")
    ap.add_argument("--extra-workloads", default="auto",
                    help="workloads measured beside the headline one and reported under `workloads` "
                         "(comma-separated, 'none', or 'auto': 1,2,3,5 for the default run)")
    return ap.parse_args()


def extra_workloads(args):
    """The other workloads measured in this run (the default run: all four)."""
    if args.extra_workloads == "none":
        return []
    if args.extra_workloads != "auto":
        return [int(v) for v in args.extra_workloads.split(",") if v]
    default_variant = (args.fp8_scales == "fp32" and args.expert_alignment == 1 and not args.combine_bias
                       and args.combine == "flat" and not args.training and args.ll_combine == "one-phase"
                       and not args.mask_ranks and not args.fused_layout and not args.graph)
    if args.workload == DEFAULT_WORKLOAD and args.tokens is None and default_variant:
        return list(EXTRA_WORKLOADS)
    return []


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def profile_traffic():
    """(DRAM bytes per full-size dispatch launch, source hash) from the committed
    ncu figures (profiles/dispatch_traffic.json), or (None, None)."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None, None
    d = json.load(open(PROFILE_TRAFFIC))
    return d.get("dram_bytes_per_full_launch"), d.get("kernel_source_sha256_16")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed work runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        """Median SM clock, maximum clock and throttle reasons seen between t0 and t1 (host time)."""
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if t0 and t1 and t0 - 0.06 <= r[0] <= t1 + 0.06] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for name, v in zip(names, r[3][1:5]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def max_over_ranks(values, device, world):
    """Element-wise maximum of per-rank timings (every rank gets the result)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(tokens_per_rank, world, ms_per_step):
    """Whole-job tokens/s: the tokens of all replicas over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


# ------------------------------------------------------------------ workloads ----
def fp8_flag_word(ep, cfg, scales: str) -> int:
    return ep.fp8_flags(cfg.fp8, round_scale=scales == "pow2", use_ue8m0=scales == "ue8m0")


class NormalWorkload:
    """Layout, dispatch (per-rank + expert-major, BF16 or FP8), combine."""

    def __init__(self, cfg, dev, inp, scales="fp32", align=1, bias=False, two_level=False, training=False,
                 fused=False):
        import torch
        import combine_ep_get_dispatch_gb300 as ep
        self.ep, self.cfg = ep, cfg
        self.flags = fp8_flag_word(ep, cfg, scales)
        self.align, self.two_level = max(1, align), two_level
        sdt = torch.uint8 if scales == "ue8m0" else torch.float32
        N, H, K, E, R = cfg.N, cfg.H, cfg.K, cfg.E, cfg.R
        self.inp = inp   # the host inputs (the oracle baseline reuses them)
        self.x_host = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16)
        self.idx_host = torch.from_numpy(inp["topk_idx"])
        self.w_host = torch.from_numpy(inp["topk_weights"])
        self.x, self.idx, self.w = self.x_host.to(dev), self.idx_host.to(dev), self.w_host.to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # Buffers allocated once (worst-case capacities: no host sync in a step).
        self.lay = ep.new_layout(self.idx, E, R, self.align)
        self.ws = torch.zeros(ep.ep_layout_workspace_bytes(N, K, E, R), dtype=torch.uint8, device=dev)
        cap_r, cap_e = N * min(K, R), N * K + E * (self.align - 1)
        xdt = torch.uint8 if cfg.fp8 else torch.bfloat16
        S = H // 128
        self.rank_x = torch.empty((cap_r, H), dtype=xdt, device=dev)
        self.rank_s = torch.empty((cap_r, S), dtype=sdt, device=dev) if cfg.fp8 else None
        self.rank_src = torch.empty(cap_r, dtype=torch.int32, device=dev)
        self.rank_ti = torch.empty((cap_r, K), dtype=torch.int32, device=dev)
        self.rank_tw = torch.empty((cap_r, K), dtype=torch.float32, device=dev)
        self.exp_x = torch.empty((cap_e, H), dtype=xdt, device=dev)
        self.exp_s = torch.empty((cap_e, S), dtype=sdt, device=dev) if cfg.fp8 else None
        self.exp_src = torch.empty(cap_e, dtype=torch.int32, device=dev)
        self.out = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        self.bias = torch.empty((N, H), dtype=torch.bfloat16, device=dev).normal_() if bias else None
        self.rank_y = torch.empty((cap_r, H), dtype=torch.bfloat16, device=dev) if two_level else None
        self.rb = ep._recv_struct(self.rank_x, self.rank_s, self.rank_src, self.rank_ti, self.rank_tw)
        self.eb = ep._recv_struct(self.exp_x, self.exp_s, self.exp_src)
        # Expert outputs fed to combine: the BF16 rows themselves (identity
        # experts) for BF16 dispatch; for FP8 dispatch a BF16 buffer in the
        # same expert-major layout (what an expert GEMM would write).
        if cfg.fp8:
            self.y = torch.empty((cap_e, H), dtype=torch.bfloat16, device=dev)
            lay0 = ep.get_dispatch_layout(self.idx, E, R, expert_alignment=self.align)
            ep.ep_dispatch(lay0, self.x, False, None, None, ep._recv_struct(self.y, None, None))
        else:
            self.y = self.exp_x
        # fused: layout and dispatch through one call (ep_layout_dispatch), the
        # dispatch launched as the layout's programmatic dependent: one phase.
        self.fused = fused
        self.phases = (["layout+dispatch"] if fused else ["layout", "dispatch"]) + \
            (["combine_to_ranks", "combine_ranks"] if two_level else ["combine"])
        self.training = training
        if training:
            # Backward: a gradient of the combined output flows back through
            # combine (to the expert rows and the weights), then through dispatch.
            self.grad_out = torch.empty((N, H), dtype=torch.bfloat16, device=dev).normal_()
            self.grad_y = torch.empty((cap_e, H), dtype=torch.bfloat16, device=dev)
            self.grad_w = torch.empty((N, K), dtype=torch.float32, device=dev)
            self.grad_x = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
            self.phases += ["combine_backward", "dispatch_backward"]
        self.dominant = "layout+dispatch" if fused else "dispatch"
        dk = f"dispatch_kernel<{'fp8' if cfg.fp8 else 'bf16'}>"
        self.kernel_names = {"layout": "layout_kernel", "dispatch": dk,
                             "layout+dispatch": f"layout_kernel + {dk} (programmatic dependent pair)",
                             "combine": "combine_kernel", "combine_to_ranks": "combine_to_ranks_kernel",
                             "combine_ranks": "combine_kernel"}

    def launches_per_step(self):
        """This library's kernel launches in one step."""
        n = 2                                    # layout, dispatch (one call or two)
        n += 1 if self.align > 1 else 0          # zero fill of the padding rows
        n += 2 if self.two_level else 1          # combine
        n += 2 if self.training else 0           # combine backward, dispatch backward
        return n

    def layout_for(self, idx):
        L = self.lay
        return self.ep.Layout(idx, L.num_experts, L.num_ranks, L.num_tokens_per_rank, L.num_tokens_per_expert,
                              L.is_token_in_rank, L.rank_offset, L.expert_offset, L.rank_slot, L.expert_slot,
                              L.expert_alignment)

    def run(self, stream, x, idx_layout, w, ev=None, out=None):
        ep = self.ep
        out = self.out if out is None else out
        mark = iter(ev) if ev else None

        def tick():
            if mark is not None:
                next(mark).record(stream)

        tick()
        if self.fused:
            ep.ep_layout_dispatch(idx_layout, self.ws, x, self.flags, w, self.rb, self.eb, self.status, stream)
            tick()
        else:
            ep.ep_get_dispatch_layout(idx_layout, self.ws, self.status, stream)
            tick()
            ep.ep_dispatch(idx_layout, x, self.flags, w, self.rb, self.eb, self.status, stream)
            tick()
        if self.two_level:
            ep.ep_combine_to_ranks(idx_layout, self.y, w, self.rank_y, self.status, stream)
            tick()
            ep.ep_combine_ranks(idx_layout, self.rank_y, out, self.status, stream, bias=self.bias)
            tick()
            return
        ep.ep_combine(idx_layout, self.y, w, out, self.status, stream, bias=self.bias)
        tick()
        if self.training:
            ep.ep_combine_backward(idx_layout, self.grad_out, self.y, w, self.grad_y, self.grad_w, self.status, stream)
            tick()
            ep.ep_combine(idx_layout, self.grad_y, None, self.grad_x, self.status, stream)
            tick()

    def rows(self):
        r = {"per_rank": int(self.lay.rank_offset[-1].item()),
             "expert_major": int(self.lay.num_tokens_per_expert.sum().item())}
        if self.align > 1:
            r["padded_expert_major"] = int(self.lay.expert_offset[-1].item())
        return r

    def algorithmic_bytes(self):
        cfg = self.cfg
        N, H, K, R, E = cfg.N, cfg.H, cfg.K, cfg.R, cfg.E
        rows = self.rows()
        D_r, D_e = rows["per_rank"], rows["expert_major"]
        out_row = H + (H // 128) * self.rank_s.element_size() if cfg.fp8 else 2 * H
        layout = N * K * 4 + (N * K * 4 + N * R * 4 + N * R + 4 * (2 * E + 2 * R + 2))
        dispatch = (N * 2 * H                                 # x read once
                    + N * K * 4 * 3 + N * R * 4               # idx, w, expert_slot, rank_slot read
                    + (D_r + D_e) * out_row                   # every output row (and its scales) written once
                    + D_e * 4 + D_r * 4 + D_r * K * 8)        # src indices, per-rank top-k idx / weights
        rows = self.rows()
        D_pad = rows.get("padded_expert_major", D_e)
        dispatch += (D_pad - D_e) * out_row                   # zeroed padding rows (aligned layouts)
        bias_b = N * 2 * H if self.bias is not None else 0
        first = {"layout+dispatch": layout + dispatch} if self.fused else {"layout": layout, "dispatch": dispatch}
        if self.two_level:
            return {**first,
                    "combine_to_ranks": D_e * 2 * H + N * K * 12 + N * R * 4 + D_r * 2 * H,
                    "combine_ranks": D_r * 2 * H + N * R * 4 + N * 2 * H + bias_b}
        combine = D_e * 2 * H + N * K * 8 + N * 2 * H + bias_b  # rows + slots/weights read, out written
        out = {**first, "combine": combine}
        if self.training:
            # grad_out and the forward rows read, grad rows and grad_w written
            out["combine_backward"] = N * 2 * H + D_e * 2 * H * 2 + N * K * 12
            out["dispatch_backward"] = D_e * 2 * H + N * K * 4 + N * 2 * H
        return out


class LLWorkload:
    """Low-latency send, receive (the hook) and combine on the fixed [E, R*T, H] layout."""

    def __init__(self, cfg, dev, inp, two_phase=False, scales="fp32", bias=False):
        import torch
        import combine_ep_get_dispatch_gb300 as ep
        self.ep, self.cfg = ep, cfg
        self.flags = fp8_flag_word(ep, cfg, scales)
        self.scale_bytes = 1 if scales == "ue8m0" else 4
        N, H, K, E, R, T = cfg.N, cfg.H, cfg.K, cfg.E, cfg.R, cfg.T
        self.inp = inp   # the host inputs (the oracle baseline reuses them)
        self.x_host = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16)
        self.idx_host = torch.from_numpy(inp["topk_idx"])
        self.w_host = torch.from_numpy(inp["topk_weights"])
        self.x, self.idx, self.w = self.x_host.to(dev), self.idx_host.to(dev), self.w_host.to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = torch.zeros(ep.ep_ll_workspace_bytes(N, K, E, R, T), dtype=torch.uint8, device=dev)
        xdt = torch.uint8 if cfg.fp8 else torch.bfloat16
        self.recv_x = torch.empty((E, R * T, H), dtype=xdt, device=dev)
        self.recv_s = torch.empty((E, R * T, H // 128), dtype=torch.uint8 if scales == "ue8m0" else torch.float32,
                                  device=dev) if cfg.fp8 else None
        self.recv_src = torch.empty((E, R * T), dtype=torch.int32, device=dev)
        self.recv_count = torch.empty(E, dtype=torch.int32, device=dev)
        self.layout_range = torch.empty((E, R), dtype=torch.int64, device=dev)
        self.out = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        self.bias = torch.empty((N, H), dtype=torch.bfloat16, device=dev).normal_() if bias else None
        if cfg.fp8:
            # BF16 expert outputs in the receive layout (what an expert GEMM would write).
            self.y = torch.empty((E, R * T, H), dtype=torch.bfloat16, device=dev)
            ep.ep_ll_dispatch_send(self.x, self.idx, H, E, R, T, False, self.y, None, self.recv_src, self.ws)
        else:
            self.y = self.recv_x
        self.two_phase = two_phase
        if two_phase:
            self.staging = torch.empty((N * K, H), dtype=torch.bfloat16, device=dev)
            self.phases = ["send", "recv", "combine_send", "combine_recv"]
        else:
            self.phases = ["send", "recv", "combine"]
        self.dominant = "send"
        small = cfg.N > 0 and cfg.N * cfg.K <= 4096 and cfg.E * cfg.R <= 16384
        self.kernel_names = {"send": "ll_send_small_kernel" if small else "layout_kernel<ll> + dispatch_kernel",
                             "recv": "ll_recv_kernel",
                             "combine": "combine_kernel", "combine_send": "combine_kernel<gather>",
                             "combine_recv": "combine_kernel"}

    def launches_per_step(self):
        """This library's kernel launches in one step: the send is one launch
        for a batch of at most 4096 (token, slot) entries with E * R <= 16384
        (the library's one-launch send), else two; then the receive and the
        combine (two launches when two-phase)."""
        c = self.cfg
        send = 1 if (c.N > 0 and c.N * c.K <= 4096 and c.E * c.R <= 16384) else 2
        return send + 1 + (2 if self.two_phase else 1)

    def layout_for(self, idx):
        return idx

    def run(self, stream, x, idx, w, ev=None, out=None):
        ep, c = self.ep, self.cfg
        out = self.out if out is None else out
        if ev:
            ev[0].record(stream)
        ep.ep_ll_dispatch_send(x, idx, c.H, c.E, c.R, c.T, self.flags, self.recv_x, self.recv_s, self.recv_src,
                               self.ws, self.status, stream)
        if ev:
            ev[1].record(stream)
        ep.ep_ll_dispatch_recv(self.ws, c.N, c.K, c.E, c.R, c.T, self.recv_count, self.layout_range,
                               self.status, stream)
        if ev:
            ev[2].record(stream)
        if self.two_phase:
            ep.ep_ll_combine_send(self.y, self.ws, c.N, c.K, c.H, c.E, c.R, c.T, self.staging, self.status, stream)
            if ev:
                ev[3].record(stream)
            ep.ep_ll_combine_recv(self.staging, w, self.ws, c.N, c.K, c.H, c.E, c.R, c.T, out, self.status,
                                  stream, bias=self.bias)
            if ev:
                ev[4].record(stream)
            return
        ep.ep_ll_combine(self.y, w, self.ws, c.N, c.K, c.H, c.E, c.R, c.T, out, self.status, stream,
                         bias=self.bias)
        if ev:
            ev[3].record(stream)

    def rows(self):
        return {"received": int(self.recv_count.sum().item())}

    def algorithmic_bytes(self):
        c = self.cfg
        N, H, K, R, E = c.N, c.H, c.K, c.R, c.E
        D = self.rows()["received"]
        row = H + (H // 128) * self.scale_bytes if c.fp8 else 2 * H
        send = N * 2 * H + N * K * 4 + D * row + D * 4 + N * K * 4 + E * R * 8 + E * 4
        recv = 2 * (E * 4 + E * R * 8)
        bias_b = N * 2 * H if self.bias is not None else 0
        combine = D * 2 * H + N * K * 8 + N * 2 * H + bias_b
        if self.two_phase:
            return {"send": send, "recv": recv, "combine_send": D * 2 * H * 2 + N * K * 4,
                    "combine_recv": D * 2 * H + N * K * 8 + N * 2 * H + bias_b}
        return {"send": send, "recv": recv, "combine": combine}


def workload_config(cfg, args, world, rows):
    """The line's `config`: the workload, its variant flags and its row counts (both arms print the same)."""
    return {"workload": cfg.name, "tokens": cfg.N, "hidden": cfg.H, "experts": cfg.E, "topk": cfg.K,
            "ranks": cfg.R, "max_tokens_per_rank": cfg.T,
            "dispatch_dtype": (f"fp8_e4m3 + {args.fp8_scales} scales / 128 ch" if cfg.fp8 else "bf16"),
            "combine_dtype": "bf16 (fp32 accumulation)",
            "l2": ("flushed between steps (256 MiB write)" if args.l2_flush == "write" else
                   "flushed between steps (256 MiB write, then read back: no dirty flush lines left)"),
            "variant": {"expert_alignment": args.expert_alignment, "combine_bias": args.combine_bias,
                        "combine": args.combine, "ll_combine": args.ll_combine,
                        "fp8_scales": args.fp8_scales, "training": args.training,
                        "mask_ranks": args.mask_ranks, "fused_layout": args.fused_layout},
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "rows": rows}


def oracle_rows(cfg, args):
    """Row counts of the full workload from the oracle's layout (the reference arm's copy of wl.rows())."""
    import oracle
    idx = ei.make_inputs(cfg, seed=0, with_x=False)["topk_idx"]
    if cfg.mode == "ll":
        mask = np.zeros(cfg.R, np.int32)
        for r in (int(v) for v in args.mask_ranks.split(",") if v):
            mask[r] = 1
        if mask.any():
            idx = oracle.ll_mask_routing(idx, cfg.E, cfg.R, mask)
        return {"received": int(oracle.layout(idx, cfg.E, cfg.R)["num_tokens_per_expert"].sum())}
    lay = oracle.layout(idx, cfg.E, cfg.R, max(1, args.expert_alignment))
    r = {"per_rank": int(lay["rank_offset"][-1]), "expert_major": int(lay["num_tokens_per_expert"].sum())}
    if args.expert_alignment > 1:
        r["padded_expert_major"] = int(lay["expert_offset"][-1])
    return r


def build_workload(cfg, args, dev, headline):
    """The workload object of cfg; variant flags apply to the headline workload only."""
    import combine_ep_get_dispatch_gb300 as ep
    inp = ei.make_inputs(cfg, seed=0)
    if cfg.mode == "ll":
        if not headline:
            return LLWorkload(cfg, dev, inp)
        wl = LLWorkload(cfg, dev, inp, two_phase=args.ll_combine == "two-phase", scales=args.fp8_scales,
                        bias=args.combine_bias)
        for r in (int(v) for v in args.mask_ranks.split(",") if v):
            ep.low_latency_update_mask_buffer(wl.ws, r, num_ranks=cfg.R)   # shrink mode: rank r is out
        return wl
    if not headline:
        return NormalWorkload(cfg, dev, inp)
    return NormalWorkload(cfg, dev, inp, scales=args.fp8_scales, align=args.expert_alignment,
                          bias=args.combine_bias, two_level=args.combine == "two-level", training=args.training,
                          fused=args.fused_layout)


def flush_l2(flush, i, mode):
    """Evict the last step's data from L2: write 256 MiB (twice L2); with
    mode write-read, also read it back so the dirty lines of the fill are
    written back before the step starts."""
    import torch
    flush.fill_(i & 0xFF)
    if mode == "write-read":
        flush.view(torch.int64).max()


def time_workload(wl, cfg, args, dev, world, stream, flush, sampler, with_e2e, with_graph):
    """Warm-up, then `steps` timed steps (L2 flushed before each, CUDA events
    around every phase on the launching stream); optionally the graph replay
    and the pipelined end-to-end run. Returns the raw timings."""
    import torch
    import combine_ep_get_dispatch_gb300 as ep
    lay = wl.layout_for(wl.idx)
    for _ in range(args.warmup):
        flush_l2(flush, 1, args.l2_flush)
        wl.run(stream, wl.x, lay, wl.w)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    nph = len(wl.phases)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    t_begin = time.time()
    for i in range(args.steps):
        flush_l2(flush, i, args.l2_flush)   # nothing of the last step stays in L2
        wl.run(stream, wl.x, lay, wl.w, evs[i])
    torch.cuda.synchronize()
    t_end = time.time()
    if world > 1:
        torch.distributed.barrier()
    phase_ms = {ph: np.array([e[j].elapsed_time(e[j + 1]) for e in evs]) for j, ph in enumerate(wl.phases)}
    step_ms = np.array([e[0].elapsed_time(e[nph]) for e in evs])
    st = int(wl.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st}: {ep.ep_error_string(st)}")
    out = {"phase_ms": phase_ms, "total_ms": float(step_ms.sum()), "window": (t_begin, t_end), "graph_ms": None,
           "e2e": None}

    # The same step captured once in a CUDA graph and replayed K times (the
    # launches of a step then cost one graph launch); L2 flushed before each
    # replay, CUDA events around it. Reported beside the eager numbers.
    if with_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            wl.run(side, wl.x, lay, wl.w)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            wl.run(torch.cuda.current_stream(dev), wl.x, lay, wl.w)
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2(flush, i, args.l2_flush)
            gev[i][0].record(stream)
            g.replay()
            gev[i][1].record(stream)
        torch.cuda.synchronize()
        out["graph_ms"] = float(np.mean([a.elapsed_time(b) for a, b in gev]))
        st = int(wl.status.item())
        if st != 0:
            raise RuntimeError(f"device status {st}: {ep.ep_error_string(st)}")

    # End to end through the C ABI from pinned host memory, pipelined as a
    # serving loop runs it: while step i computes, step i+1's inputs go up on
    # one stream and step i-1's output comes down on another (two sets of
    # device inputs and outputs; events order the reuse of each set).
    if with_e2e:
        xp, ip, wp = wl.x_host.pin_memory(), wl.idx_host.pin_memory(), wl.w_host.pin_memory()
        outp = [torch.empty(wl.out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        xd = [torch.empty_like(wl.x) for _ in range(2)]
        idd = [torch.empty_like(wl.idx) for _ in range(2)]
        wd = [torch.empty_like(wl.w) for _ in range(2)]
        outd = [torch.empty_like(wl.out) for _ in range(2)]
        lay_d = [wl.layout_for(t) for t in idd]
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        e2e_steps = max(3, min(args.steps, 50))
        n_all = 2 + e2e_steps
        up_done = [torch.cuda.Event() for _ in range(n_all)]
        comp_done = [torch.cuda.Event() for _ in range(n_all)]
        down_done = [torch.cuda.Event() for _ in range(n_all)]

        def e2e_step(i):
            j = i & 1
            if i >= 2:
                s_up.wait_event(comp_done[i - 2])      # step i-2 has consumed input set j
            with torch.cuda.stream(s_up):
                xd[j].copy_(xp, non_blocking=True)
                idd[j].copy_(ip, non_blocking=True)
                wd[j].copy_(wp, non_blocking=True)
            up_done[i].record(s_up)
            stream.wait_event(up_done[i])
            if i >= 2:
                stream.wait_event(down_done[i - 2])    # output set j has been read back
            wl.run(stream, xd[j], lay_d[j], wd[j], out=outd[j])
            comp_done[i].record(stream)
            s_down.wait_event(comp_done[i])
            with torch.cuda.stream(s_down):
                outp[j].copy_(outd[j], non_blocking=True)
            down_done[i].record(s_down)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_up)
        for i in range(2, n_all):
            e2e_step(i)
        stream.wait_event(down_done[n_all - 1])
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
        if not torch.equal(outp[(n_all - 1) & 1], wl.out.cpu()):
            raise RuntimeError("e2e output differs from the device-resident run")
        out["e2e"] = (e2e_ms, xp.numel() * 2 + ip.numel() * 4 + wp.numel() * 4, outp[0].numel() * 2)
    return out


def phase_report(wl, timing, ms_per_step, peak, peak_kind):
    """Per-phase µs, algorithmic GB/s and fractions of the measured and the nominal HBM peak."""
    nbytes = wl.algorithmic_bytes()
    mean_s = {ph: float(v.mean()) / 1e3 for ph, v in timing["phase_ms"].items()}
    phases = {}
    for ph in wl.phases:
        gbs = nbytes[ph] / mean_s[ph] / 1e9
        phases[f"{ph}_us"] = round(mean_s[ph] * 1e6, 2)
        phases[f"{ph}_gbs"] = round(gbs, 1)
        phases[f"{ph}_frac"] = round(gbs / peak, 4)
        phases[f"{ph}_frac_nominal"] = round(gbs / NOMINAL_HBM_GBS, 4)
    phases["step_gbs"] = round(sum(nbytes.values()) / (ms_per_step / 1e3) / 1e9, 1)
    phases["peak_note"] = (f"*_frac: fractions of the {peak_kind} HBM copy peak {peak} GB/s; "
                           f"*_frac_nominal: of the {NOMINAL_HBM_GBS:.0f} GB/s nominal peak")
    return phases, nbytes, mean_s


def run_ours(args):
    import torch
    import combine_ep_get_dispatch_gb300 as ep  # noqa: F401  (fails loudly if the library is missing)

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    cfg = ei.WORKLOADS[args.workload]
    if args.tokens:
        cfg = cfg.scaled(N=args.tokens)
    wl = build_workload(cfg, args, dev, headline=True)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    time.sleep(0.3)
    timing = time_workload(wl, cfg, args, dev, world, stream, flush, sampler, not args.no_e2e, args.graph)

    # The other workloads, measured the same way (same steps, warm-up, L2
    # flush and events), reported under `workloads`.
    extras = {}
    for w in extra_workloads(args):
        if w == args.workload:
            continue
        c2 = ei.WORKLOADS[w]
        wl2 = build_workload(c2, args, dev, headline=False)
        t2 = time_workload(wl2, c2, args, dev, world, stream, flush, sampler, not args.no_e2e, False)
        extras[w] = (c2, wl2.rows(), wl2, t2)
        del wl2
        torch.cuda.empty_cache()
    sampler.stop()

    total_ms = timing["total_ms"]
    e2e = timing["e2e"]
    vals = max_over_ranks([total_ms, e2e[0] if e2e else 0.0, timing["graph_ms"] or 0.0]
                          + [t[3]["total_ms"] for t in extras.values()]
                          + [t[3]["e2e"][0] if t[3]["e2e"] else 0.0 for t in extras.values()], dev, world)
    total_ms, e2e_ms_max, graph_ms = vals[0], vals[1], vals[2]
    extra_tot = dict(zip(extras, vals[3:3 + len(extras)]))
    extra_e2e = dict(zip(extras, vals[3 + len(extras):]))
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peak, peak_kind = peaks()
    ms_per_step = total_ms / args.steps
    N = cfg.N
    value = job_throughput(N, world, ms_per_step)
    phases, nbytes, mean_s = phase_report(wl, timing, ms_per_step, peak, peak_kind)
    dom = wl.dominant
    achieved = nbytes[dom] / mean_s[dom] / 1e9
    traffic = None
    if dom == "dispatch" and not cfg.fp8 and args.workload == DEFAULT_WORKLOAD:
        traffic_full, src_hash = profile_traffic()
        if traffic_full is not None and src_hash == kernel_hash():
            traffic = traffic_full * (N / ei.WORKLOADS[DEFAULT_WORKLOAD].N)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded: x ~ N(0,1) BF16, router logits N(0,1) softmax top-k renormalised; "
                "see epinputs for the grouped and Zipf recipes)",
        "config": workload_config(cfg, args, world, wl.rows()),
        "phases": phases,
        "roofline": {"bound": "hbm", "kernel": wl.kernel_names[dom], "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": nbytes[dom], "peak_kind": peak_kind,
                     "peak_nominal": NOMINAL_HBM_GBS, "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4)},
        "gpu_launches": wl.launches_per_step() * args.steps,
        "clocks": sampler.summary(*timing["window"]),
    }
    if timing["graph_ms"] is not None:
        line["graph"] = {"ms_per_step": round(graph_ms, 4), "value": round(job_throughput(N, world, graph_ms), 1),
                         "unit": "tokens/s"}
    if e2e:
        line["e2e"] = {"value": round(job_throughput(N, world, e2e_ms_max), 1), "unit": "tokens/s",
                       "h2d_bytes_per_step": e2e[1], "d2h_bytes_per_step": e2e[2],
                       "ms_per_step": round(e2e_ms_max, 4)}
    if extras:
        line["workloads"] = {}
        for w, (c2, rows2, wl2, t2) in extras.items():
            ms2 = extra_tot[w] / args.steps
            ph2, nb2, ms_s2 = phase_report(wl2, t2, ms2, peak, peak_kind)
            d2 = wl2.dominant
            ach2 = nb2[d2] / ms_s2[d2] / 1e9
            entry = {"workload": c2.name, "value": round(job_throughput(c2.N, world, ms2), 1), "unit": "tokens/s",
                     "ms_per_step": round(ms2, 4), "phases": ph2,
                     "dominant": {"phase": d2, "kernel": wl2.kernel_names[d2], "achieved": round(ach2, 1),
                                  "frac": round(ach2 / peak, 4), "frac_nominal": round(ach2 / NOMINAL_HBM_GBS, 4)},
                     "rows": rows2, "gpu_launches": wl2.launches_per_step() * args.steps,
                     "clocks": sampler.summary(*t2["window"])}
            if t2["e2e"]:
                entry["e2e"] = {"value": round(job_throughput(c2.N, world, extra_e2e[w]), 1), "unit": "tokens/s",
                                "h2d_bytes_per_step": t2["e2e"][1], "d2h_bytes_per_step": t2["e2e"][2],
                                "ms_per_step": round(extra_e2e[w], 4)}
            line["workloads"][c2.name] = entry
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_sample_tokens, wl.inp)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# --------------------------------------------------------------- CPU oracle ----
def _oracle_step(sub):
    import oracle
    if sub["mode"] == "ll":
        ll = oracle.ll_dispatch(sub["x"], sub["topk_idx"], sub["E"], sub["R"], sub["T"], sub["fp8"])
        y = ll["recv_x"] if not sub["fp8"] else np.zeros(ll["recv_x"].shape, np.uint16)
        oracle.ll_combine(y, ll["slot_map"], sub["topk_weights"])
        return
    lay = oracle.layout(sub["topk_idx"], sub["E"], sub["R"])
    o = oracle.dispatch(sub["x"], sub["topk_idx"], sub["topk_weights"], sub["E"], sub["R"], sub["fp8"], lay=lay)
    y = o["exp_x"] if not sub["fp8"] else o["exp_x"].astype(np.uint16)
    oracle.combine(y, lay["expert_slot"], sub["topk_weights"])


def _sample(cfg, n_tok, inp=None):
    """The first n_tok tokens' inputs (all of them for None); `inp`, the whole
    workload's inputs when already made, is reused for the whole workload."""
    if n_tok is None:
        n_tok = cfg.N
    if cfg.mode == "ll":
        n_tok = max(cfg.R, (min(n_tok, cfg.N) // cfg.R) * cfg.R)
    else:
        n_tok = min(n_tok, cfg.N)
    d = dict(inp) if (inp is not None and n_tok == cfg.N) else ei.make_inputs(cfg.scaled(N=n_tok), seed=0)
    # Low latency: the sample's own per-rank capacity (rows do not depend on T).
    T = max(1, n_tok // cfg.R) if cfg.mode == "ll" else None
    d.update(E=cfg.E, R=cfg.R, T=T, fp8=cfg.fp8, mode=cfg.mode, n_tok=n_tok)
    return d


def _time_oracle(sub, budget_s, max_reps=1000):
    _oracle_step(sub)  # warm the library and the page cache
    reps, t = 0, 0.0
    while t < budget_s and reps < max_reps:
        t0 = time.perf_counter()
        _oracle_step(sub)
        t += time.perf_counter() - t0
        reps += 1
    return reps, t


def cpu_baseline(cfg, n_tok, inp=None):
    """The oracle on the first n_tok tokens of the workload (the whole step on
    those tokens), on every host core (its OpenMP build: the row loops of
    dispatch and combine in parallel, the layout sequential, identical
    results), with the plain single-threaded build's figure beside it."""
    import oracle
    sub = _sample(cfg, n_tok, inp)
    n_tok = sub["n_tok"]
    oracle.use_all_cores(False)
    reps1, t1 = _time_oracle(sub, budget_s=5.0)
    one = {"value": round(n_tok * reps1 / t1, 1), "unit": "tokens/s", "cores": 1,
           "sample": f"{n_tok} of {cfg.N} tokens, {reps1} reps, {t1:.1f} s"}
    if not oracle.use_all_cores(True):
        return {**one, "kind": "oracle", "sample": f"{n_tok} of {cfg.N} tokens of {cfg.name} (the whole step on "
                                                     f"those tokens), {reps1} reps, {t1:.1f} s; no OpenMP build"}
    try:
        cores = oracle.threads()
        reps, t = _time_oracle(sub, budget_s=10.0)
    finally:
        oracle.use_all_cores(False)
    return {"value": round(n_tok * reps / t, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_tok} of {cfg.N} tokens of {cfg.name} (the whole step on those tokens: layout "
                      f"sequential, row loops of dispatch and combine on {cores} threads), {reps} reps, {t:.1f} s",
            "single_core": one}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    cfg = ei.WORKLOADS[args.workload]
    sub = _sample(cfg, 256)
    n_tok = sub["n_tok"]
    for _ in range(args.warmup):
        _oracle_step(sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(sub)
    t = time.perf_counter() - t0
    v = n_tok * args.steps / t
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(cfg, args, world, oracle_rows(cfg, args)),
            "cpu_baseline": {"value": round(v, 1), "unit": "tokens/s", "kind": "oracle", "cores": 1,
                             "sample": f"{n_tok} tokens of {cfg.name} per step (the whole step: layout, "
                                       f"dispatch and combine on those tokens)"},
            "e2e": {"value": round(v, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
