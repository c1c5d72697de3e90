"""Benchmark: MoE layout -> dispatch -> combine on one GB300 (or N replicas).

One step is one pass of the whole hot path over one batch of the large
prefill workload (16384 tokens, hidden 7168 BF16, 256 experts top-6, 8
logical ranks): the routing layout, dispatch into the per-rank and the
expert-major receive buffers (BF16), and combine of identity expert outputs
(the expert-major rows) back into [16384, 7168] BF16.

Prints one JSON line (rank 0). `value` is tokens/s of the whole job with
inputs resident in HBM; `e2e` is the same through the C ABI from pinned host
buffers, with the host->device copy of x / topk_idx / topk_weights and the
device->host copy of the combined output inside the timed region.

--impl reference times the CPU oracle (plain single-threaded C++) on the same
workload, each step a bounded sample of tokens.
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
WORKLOAD = 4          # the 16384-token large prefill workload
L2_FLUSH_BYTES = 256 << 20
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "dispatch_kernel_prefill_large.md")
KERNEL_SOURCES = [os.path.join(ROOT, "combine_ep_get_dispatch_gb300", "csrc", f)
                  for f in ("dispatch.cu", "common.cuh", "kernels.cuh")]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=None, help="override the token count (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=2048)
    return ap.parse_args()


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
    """(bytes per full-size dispatch launch, source hash) from the committed ncu summary."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None, None
    traffic = src = None
    for line in open(PROFILE_TRAFFIC):
        if line.startswith("traffic_bytes_per_full_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
        if line.startswith("kernel_source_sha256_16:"):
            src = line.split(":", 1)[1].strip()
    return traffic, src


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed work runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

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

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
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
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 - 0.06 <= r[0] <= self.t1 + 0.06] or rows
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


def algorithmic_bytes(cfg, D_r, D_e):
    N, H, K, R, E = cfg.N, cfg.H, cfg.K, cfg.R, cfg.E
    row = H * 2
    layout = N * K * 4 + (N * K * 4 + N * R * 4 + N * R + 4 * (2 * E + 2 * R + 2))
    dispatch = (N * row                                   # x read once
                + N * K * 4 * 3 + N * R * 4               # idx, w, expert_slot, rank_slot read
                + (D_r + D_e) * row                       # every output row written once
                + D_e * 4 + D_r * 4 + D_r * K * 8)        # src indices, per-rank top-k idx / weights
    combine = D_e * row + N * K * 8 + N * row             # rows + slots/weights read, out written
    return layout, dispatch, combine


def run_ours(args):
    import torch
    import combine_ep_get_dispatch_gb300 as ep

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    cfg = ei.CONFIGS[WORKLOAD]
    if args.tokens:
        cfg = cfg.scaled(N=args.tokens)
    N, H, K, E, R = cfg.N, cfg.H, cfg.K, cfg.E, cfg.R
    inp = ei.make_inputs(cfg, seed=0)
    x_host = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16)
    idx_host = torch.from_numpy(inp["topk_idx"])
    w_host = torch.from_numpy(inp["topk_weights"])
    x = x_host.to(dev)
    idx = idx_host.to(dev)
    w = w_host.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    # Buffers allocated once (worst-case capacities: no host sync in a step).
    lay = ep.new_layout(idx, E, R)
    ws = torch.empty(ep.ep_layout_workspace_bytes(N, K, E, R), dtype=torch.uint8, device=dev)
    cap_r, cap_e = N * min(K, R), N * K
    rank_x = torch.empty((cap_r, H), dtype=torch.bfloat16, device=dev)
    rank_src = torch.empty(cap_r, dtype=torch.int32, device=dev)
    rank_ti = torch.empty((cap_r, K), dtype=torch.int32, device=dev)
    rank_tw = torch.empty((cap_r, K), dtype=torch.float32, device=dev)
    exp_x = torch.empty((cap_e, H), dtype=torch.bfloat16, device=dev)
    exp_src = torch.empty(cap_e, dtype=torch.int32, device=dev)
    out = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    rb = ep._recv_struct(rank_x, None, rank_src, rank_ti, rank_tw)
    eb = ep._recv_struct(exp_x, None, exp_src)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def layout_for(idxi):
        # Same output arrays, a different topk_idx buffer.
        return ep.Layout(idxi, E, R, lay.num_tokens_per_rank, lay.num_tokens_per_expert, lay.is_token_in_rank,
                         lay.rank_offset, lay.expert_offset, lay.rank_slot, lay.expert_slot)

    def step(li, xi, wi, ev=None):
        if ev:
            ev[0].record(stream)
        ep.ep_get_dispatch_layout(li, ws, status, stream)
        if ev:
            ev[1].record(stream)
        ep.ep_dispatch(li, xi, False, wi, rb, eb, status, stream)
        if ev:
            ev[2].record(stream)
        ep.ep_combine(li, exp_x, wi, out, status, stream)
        if ev:
            ev[3].record(stream)

    sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        flush.fill_(1)
        step(lay, x, w)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    sampler.mark(True)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)   # write 256 MiB between steps: nothing of the last step stays in L2
        step(lay, x, w, evs[i])
    torch.cuda.synchronize()
    sampler.mark(False)
    if world > 1:
        torch.distributed.barrier()
    lay_ms = np.array([e[0].elapsed_time(e[1]) for e in evs])
    dis_ms = np.array([e[1].elapsed_time(e[2]) for e in evs])
    com_ms = np.array([e[2].elapsed_time(e[3]) for e in evs])
    step_ms = np.array([e[0].elapsed_time(e[3]) for e in evs])
    total_ms = float(step_ms.sum())
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st}: {ep.ep_error_string(st)}")

    D_r = int(lay.rank_offset[-1].item())
    D_e = int(lay.expert_offset[-1].item())

    # End to end through the C ABI from pinned host memory.
    e2e = None
    if not args.no_e2e:
        xp, ip, wp = x_host.pin_memory(), idx_host.pin_memory(), w_host.pin_memory()
        outp = torch.empty((N, H), dtype=torch.bfloat16).pin_memory()
        xd, idd, wd = torch.empty_like(x), torch.empty_like(idx), torch.empty_like(w)
        lay_d = layout_for(idd)
        e2e_steps = max(3, min(args.steps, 50))
        for _ in range(2):
            xd.copy_(xp, non_blocking=True); idd.copy_(ip, non_blocking=True); wd.copy_(wp, non_blocking=True)
            step(lay_d, xd, wd)
            outp.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            xd.copy_(xp, non_blocking=True); idd.copy_(ip, non_blocking=True); wd.copy_(wp, non_blocking=True)
            step(lay_d, xd, wd)
            outp.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
        if not torch.equal(outp, out.cpu()):
            raise RuntimeError("e2e output differs from the device-resident run")
        e2e = (e2e_ms, xp.numel() * 2 + ip.numel() * 4 + wp.numel() * 4, outp.numel() * 2)
    sampler.stop()

    # max over ranks
    times = torch.tensor([total_ms, e2e[0] if e2e else 0.0], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(times, op=torch.distributed.ReduceOp.MAX)
    total_ms, e2e_ms_max = float(times[0]), float(times[1])
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peak, peak_kind = peaks()
    b_lay, b_dis, b_com = algorithmic_bytes(cfg, D_r, D_e)
    dis_s, com_s, lay_s = dis_ms.mean() / 1e3, com_ms.mean() / 1e3, lay_ms.mean() / 1e3
    ms_per_step = total_ms / args.steps
    value = N * world / (ms_per_step / 1e3)
    traffic_full, src_hash = profile_traffic()
    traffic = None
    if traffic_full is not None and src_hash == kernel_hash():
        traffic = traffic_full * (N / ei.CONFIGS[WORKLOAD].N)
    clocks = sampler.summary()
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
        "data": "synthetic (seeded: x ~ N(0,1) BF16, router logits N(0,1), softmax top-6 renormalised)",
        "config": {"workload": cfg.name, "tokens": N, "hidden": H, "experts": E, "topk": K, "ranks": R,
                   "dispatch_dtype": "bf16", "combine_dtype": "bf16 (fp32 accumulation)",
                   "l2": "flushed between steps (256 MiB write); inputs and outputs larger than L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "rows": {"per_rank": D_r, "expert_major": D_e}},
        "phases": {
            "layout_us": round(lay_s * 1e6, 2),
            "dispatch_us": round(dis_s * 1e6, 2),
            "combine_us": round(com_s * 1e6, 2),
            "dispatch_gbs": round(b_dis / dis_s / 1e9, 1),
            "combine_gbs": round(b_com / com_s / 1e9, 1),
            "dispatch_frac": round(b_dis / dis_s / 1e9 / peak, 4),
            "combine_frac": round(b_com / com_s / 1e9 / peak, 4),
            "step_gbs": round((b_lay + b_dis + b_com) / (ms_per_step / 1e3) / 1e9, 1),
            "peak_note": f"fractions of the {peak_kind} HBM copy peak {peak} GB/s",
        },
        "roofline": {"bound": "hbm", "kernel": "dispatch_kernel<bf16>", "achieved": round(b_dis / dis_s / 1e9, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(b_dis / dis_s / 1e9 / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": b_dis, "peak_kind": peak_kind},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if e2e:
        line["e2e"] = {"value": round(N * world / (e2e_ms_max / 1e3), 1), "unit": "tokens/s",
                       "h2d_bytes_per_step": e2e[1], "d2h_bytes_per_step": e2e[2],
                       "ms_per_step": round(e2e_ms_max, 4)}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_sample_tokens)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _oracle_step(sub):
    import oracle
    lay = oracle.layout(sub["topk_idx"], sub["E"], sub["R"])
    o = oracle.dispatch(sub["x"], sub["topk_idx"], sub["topk_weights"], sub["E"], sub["R"], False, lay=lay)
    oracle.combine(o["exp_x"], lay["expert_slot"], sub["topk_weights"])


def _sample(cfg, n_tok):
    d = ei.make_inputs(cfg.scaled(N=n_tok), seed=0)
    d.update(E=cfg.E, R=cfg.R)
    return d


def cpu_baseline(cfg, n_tok):
    """The oracle as written (single thread) on the first n_tok tokens of the workload."""
    sub = _sample(cfg, n_tok)
    _oracle_step(sub)  # warm the library and the page cache
    reps, t = 0, 0.0
    while t < 10.0 and reps < 20:
        t0 = time.perf_counter()
        _oracle_step(sub)
        t += time.perf_counter() - t0
        reps += 1
    return {"value": round(n_tok * reps / t, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_tok} of {cfg.N} tokens of {cfg.name} (layout + BF16 dispatch + combine), "
                      f"{reps} reps, {t:.1f} s"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    cfg = ei.CONFIGS[WORKLOAD]
    n_tok = 256
    sub = _sample(cfg, n_tok)
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
            "data": "synthetic", "config": {"workload": cfg.name, "tokens_per_step_sample": n_tok},
            "cpu_baseline": {"value": round(v, 1), "unit": "tokens/s", "kind": "oracle", "cores": 1,
                             "sample": f"{n_tok} tokens of {cfg.name} per step"},
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
