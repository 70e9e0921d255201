"""Benchmark of the GB300 MoE expert block.

One step = one pass of the whole forward hot path (counts, offsets, row map,
permute, grouped fc1 + SwiGLU, grouped fc2, unpermute) over one batch of the
Mixtral-8x7B-shaped workload (T=4096 tokens, H=4096, F=14336, 8 experts,
top-2), seeded synthetic inputs resident in HBM. L2 is flushed (a 512 MB
write, untimed) before every timed step; each step is bracketed by CUDA
events on the launching stream.

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

# DRAM bytes (read + write) of one fc1 launch on the default workload, from
# the ncu capture summarised in profiles/; null once the kernel source changes.
FC1_TRAFFIC = {"bytes": None, "src_sha": None}


def _sha_of_kernel_sources():
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm_bf16.cu", "common.cuh"):
        with open(os.path.join(ROOT, "moe_expert_dispatch_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                      "--format=csv,noheader,nounits"], capture_output=True,
                                     text=True, timeout=5).stdout.strip()
                if out:
                    self.samples.append([v.strip() for v in out.split(",")])
            except Exception:
                pass
            self._stop.wait(0.1)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if len(s) > 3 + i and s[3 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(v: float, ws: int, device):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_oracle_sample(w, inp, n_tokens: int):
    """Time the oracle (as it stands) on n_tokens sampled tokens of the workload."""
    import oracle as orc
    toks = list(range(n_tokens))
    t0 = time.perf_counter()
    orc.sampled_forward(inp["x"].float().numpy(), synth.F32Slices(inp["w_gate"]),
                        synth.F32Slices(inp["w_up"]), synth.F32Slices(inp["w_down"]),
                        inp["expert_ids"].numpy(), inp["probs"].numpy(), toks)
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": os.cpu_count(),
            "kind": "oracle", "seconds": dt,
            "sample": f"{n_tokens} tokens of {w.name} (T={w.T}), per-token float64 loop, "
                      "NumPy BLAS threads"}


def run_reference(args, w):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    inp = synth.make_inputs(w, 0)
    times = []
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state worth discarding beyond the first call
    for _ in range(args.steps):
        r = cpu_oracle_sample(w, inp, args.ref_tokens)
        times.append(r["seconds"])
    sec_per_token = float(np.mean(times)) / args.ref_tokens
    value = 1.0 / sec_per_token
    line = {"impl": "reference", "metric": "MoE expert-block tokens/s", "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec_per_token * w.T * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{args.ref_tokens} tokens per step of {w.name}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_ours(args, w):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import moe_expert_dispatch_gb300 as m

    inp = synth.make_inputs(w, 0)
    x = inp["x"].to(device)
    wg, wu, wd = (inp[k].to(device) for k in ("w_gate", "w_up", "w_down"))
    ids, probs = inp["expert_ids"].to(device), inp["probs"].to(device)
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(m.STEP_EVENTS)]
    for e in evs:
        e.record(stream)
    cfg = m.config()
    cfg_ev = m.config(step_events=evs)
    nbytes = m.moe_workspace_size(w.T, w.H, w.F, w.E, w.k, cfg)
    work = torch.empty(nbytes, dtype=torch.uint8, device=device)
    y = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=device)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)

    def step(c):
        m.moe_expert_forward(x, wg, wu, wd, ids, probs, y=y, workspace=work, cfg=c)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step(cfg)
    torch.cuda.synchronize()
    st = m.moe_get_error()
    if st != 0:
        raise RuntimeError(f"device error {st}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    parts = np.zeros(m.STEP_EVENTS - 1)
    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step(cfg_ev)
            ends[i].record(stream)
            evs[-1].synchronize()
            parts += [evs[j].elapsed_time(evs[j + 1]) for j in range(m.STEP_EVENTS - 1)]
        torch.cuda.synchronize()
    _barrier(ws)
    ms = float(np.mean([s.elapsed_time(e) for s, e in zip(starts, ends)]))
    ms = _max_over_ranks(ms, ws, device)
    parts /= args.steps
    if m.moe_get_error() != 0:
        raise RuntimeError("device error during the timed region")

    # end to end through the public call, host buffers: H2D of x/ids/probs,
    # the block, D2H of y, every step
    hx = inp["x"].pin_memory()
    hids = inp["expert_ids"].pin_memory()
    hprobs = inp["probs"].pin_memory()
    hy = torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory()
    dx = torch.empty_like(x)
    dids = torch.empty_like(ids)
    dprobs = torch.empty_like(probs)
    h2d = hx.numel() * 2 + hids.numel() * 4 + hprobs.numel() * 4
    d2h = hy.numel() * 2
    e2e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e2e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps + 2):
        flush.zero_()
        if i >= 2:
            e2e_s[i - 2].record(stream)
        dx.copy_(hx, non_blocking=True)
        dids.copy_(hids, non_blocking=True)
        dprobs.copy_(hprobs, non_blocking=True)
        m.moe_expert_forward(dx, wg, wu, wd, dids, dprobs, y=y, workspace=work, cfg=cfg)
        hy.copy_(y, non_blocking=True)
        if i >= 2:
            e2e_e[i - 2].record(stream)
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(float(np.mean([s.elapsed_time(e) for s, e in zip(e2e_s, e2e_e)])),
                             ws, device)

    hbm, bf16_burst, bf16_sus, peak_src = _peaks()
    R = w.T * w.k
    fc1_flop = 4.0 * R * w.H * w.F
    fc2_flop = 2.0 * R * w.F * w.H
    fc1_tflops = fc1_flop / (parts[1] * 1e-3) / 1e12
    traffic = FC1_TRAFFIC["bytes"] if FC1_TRAFFIC["src_sha"] == _sha_of_kernel_sources() else None
    line = {
        "metric": "MoE expert-block tokens/s", "value": ws * w.T / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k,
                   "l2": "flushed before every step (512 MB write)",
                   "parallelism": "replicas" if ws > 1 else "single"},
        "roofline": {"bound": "tensor", "kernel": "fc1_swiglu (grouped GEMM)",
                     "achieved": fc1_tflops, "peak": bf16_burst, "unit": "TFLOP/s",
                     "frac": fc1_tflops / bf16_burst, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16 burst"},
        "steps_ms": {"routing": parts[0], "fc1_swiglu": parts[1], "fc2": parts[2],
                     "unpermute": parts[3]},
        "grouped_gemm_tflops": (fc1_flop + fc2_flop) / ((parts[1] + parts[2]) * 1e-3) / 1e12,
        "e2e": {"value": ws * w.T / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 7 * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(w, inp, args.ref_tokens)
        line["cpu_baseline"].pop("seconds", None)
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral_bf16", choices=list(synth.WORKLOADS))
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
