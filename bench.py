"""Benchmark of the GB300 MoE expert block.

One step = one pass of the whole hot path over one batch of a workload, with
seeded synthetic inputs resident in HBM:
  * BF16 forward (default: the Mixtral-8x7B-shaped layer, T=4096 tokens,
    H=4096, F=14336, 8 experts, top-2): counts, offsets, row map, permute,
    grouped fc1 + SwiGLU, grouped fc2, unpermute;
  * MXFP8 forward (--workload mxfp8): the same with x quantised while it is
    permuted, block-scaled GEMMs and h quantised in fc1's epilogue (weights
    quantised once, outside the timed region, as a deployment would);
  * BF16 training step (--workload train_bf16): forward (saving what the
    backward needs) + backward (dX, dW1gate, dW1up, dW2, dprobs).
L2 is flushed (a 512 MB write, untimed) before every timed step; each step
is bracketed by CUDA events on the launching stream, and the library records
events at its own step boundaries on the same stream (moe_config.step_events)
for the per-kernel times and the roofline.

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

# DRAM bytes (read + write) per launch of the dominant kernel on a workload,
# from the ncu captures summarised in profiles/, with the kernel's source
# files and their hash when the counters were taken; reported as null once
# any of those files changes.
BF16_GEMM_SOURCES = ("gemm_bf16.cu", "common.cuh", "internal.h")
MXFP8_GEMM_SOURCES = ("gemm_mxfp8.cu", "mx.cuh", "common.cuh", "internal.h")
TRAFFIC = {
    # DRAM bytes per launch of each workload's dominant GEMM, from counters of
    # small cases (dram__bytes_read.sum + dram__bytes_write.sum) scaled to the
    # full launch by the algorithmic bytes; the captures and the arithmetic are
    # summarised under profiles/
    ("mixtral_bf16", "fc1_swiglu"): {"bytes": 2170e6, "sources": BF16_GEMM_SOURCES,
                                     "src_sha": "c08da4619780dca4"},
    ("skewed_bf16", "fc1_swiglu"): {"bytes": 1177.7e6, "sources": BF16_GEMM_SOURCES,
                                    "src_sha": "c08da4619780dca4"},
    ("train_bf16", "dW1"): {"bytes": 5685e6, "sources": BF16_GEMM_SOURCES,
                            "src_sha": "c08da4619780dca4"},
    ("mxfp8", "fc1_swiglu"): {"bytes": 2908e6, "sources": MXFP8_GEMM_SOURCES,
                              "src_sha": "ea8876c85818a3f2"},
    ("train_mxfp8", "fc1_swiglu"): {"bytes": 4102e6, "sources": MXFP8_GEMM_SOURCES,
                                    "src_sha": "ea8876c85818a3f2"},
    ("train_mxfp8", "dW1"): {"bytes": 4603e6, "sources": MXFP8_GEMM_SOURCES,
                             "src_sha": "ea8876c85818a3f2"},
}
FP8_OVER_BF16 = 2.0   # nominal dense FP8 / BF16 tensor rate (4.5 / 2.25 PFLOP/s)


def _sha_of_sources(files):
    """Hash of the kernel sources' code: comments and whitespace are left
    out, so that only a change to the code itself retires a capture."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "moe_expert_dispatch_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def _peaks(sustained: bool = False):
    """(HBM GB/s, dense bf16 TFLOP/s, source). The bf16 figure is the burst
    one for kernels of a short step; a long step under the power cap (the
    training steps) is held to the sustained one."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        if sustained and "bf16_tflops_sustained" in p:
            return p["hbm_gbs"], p["bf16_tflops_sustained"], "measured bf16 sustained"
        return p["hbm_gbs"], p["bf16_tflops"], "measured bf16 burst"
    except Exception:
        if sustained:
            return 6800.0, 1700.0, "fallback bf16 sustained"
        return 6800.0, 1900.0, "fallback bf16 burst"


class ClockSampler:
    """SM clock, power and throttle reasons sampled every 20 ms by one
    nvidia-smi process in loop mode while the GPU runs the settle pass and the
    timed region; each sample carries its host time, so that the summary can
    count the samples inside the timed region itself."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []          # (host time, fields)
        self.timed = None          # (start, end) host times of the timed region
        self._p = None
        self._t = None

    def _read(self):
        for line in self._p.stdout:
            line = line.strip()
            if line:
                self.samples.append((time.monotonic(), [v.strip() for v in line.split(",")]))

    def __enter__(self):
        try:
            self._p = subprocess.Popen(["nvidia-smi", "-i", str(self.index),
                                        "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                        "-lms", "20"], stdout=subprocess.PIPE,
                                       stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.1)        # the first sample precedes the load
        except Exception:
            self._p = None
        return self

    def __exit__(self, *a):
        if self._p is not None:
            self._p.terminate()
            try:
                self._p.wait(timeout=10)
            except Exception:
                self._p.kill()
            self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        num = lambda v: v.replace(".", "", 1).isdigit()  # noqa: E731
        rows = [f for _, f in self.samples]
        sm = [float(f[0]) for f in rows if num(f[0])]
        mx = [float(f[1]) for f in rows if num(f[1])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for f in rows for i in range(4)
                          if len(f) > 3 + i and f[3 + i].lower() == "active"})
        out = {"sm_mhz": float(np.median(sm)) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
               "samples": len(rows)}
        if self.timed is not None:
            t0, t1 = self.timed
            tsm = [float(f[0]) for t, f in self.samples if t0 <= t <= t1 and num(f[0])]
            out["samples_timed"] = len(tsm)
            out["sm_mhz_timed"] = float(np.median(tsm)) if tsm else None
        return out


def _dist():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


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


# ---------------------------------------------------------------- CPU oracle sample

def _cpu_threads() -> int:
    """Threads the oracle's NumPy BLAS calls run on: the BLAS pool's size
    where threadpoolctl can read it, else the cores this process may use."""
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:   # not installed, or a BLAS it cannot query
        pass
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_oracle_sample(w, inp, n_tokens: int):
    """Time the oracle (as it stands) on n_tokens sampled tokens of the workload."""
    import oracle as orc
    toks = list(range(n_tokens))
    f32 = synth.F32Slices
    t0 = time.perf_counter()
    if w.mxfp8 and w.backward:
        orc.backward_rows_mxfp8(inp["dy"].float().numpy(), inp["x"].float().numpy(),
                                f32(inp["w_gate_t"]), f32(inp["w_up_t"]), f32(inp["w_down_t"]),
                                inp["expert_ids"].numpy(), inp["probs"].numpy(), toks)
        what = "MXFP8 forward + backward (dX, dprobs)"
    elif w.mxfp8:
        orc.sampled_forward_mxfp8(inp["x"].float().numpy(), f32(inp["w_gate_t"]),
                                  f32(inp["w_up_t"]), f32(inp["w_down_t"]),
                                  inp["expert_ids"].numpy(), inp["probs"].numpy(), toks)
        what = "MXFP8 forward"
    elif w.backward:
        orc.backward_rows(inp["dy"].float().numpy(), inp["x"].float().numpy(),
                          f32(inp["w_gate"]), f32(inp["w_up"]), f32(inp["w_down"]),
                          inp["expert_ids"].numpy(), inp["probs"].numpy(), toks)
        what = "forward + backward (dX, dprobs)"
    else:
        orc.sampled_forward(inp["x"].float().numpy(), f32(inp["w_gate"]), f32(inp["w_up"]),
                            f32(inp["w_down"]), inp["expert_ids"].numpy(), inp["probs"].numpy(),
                            toks)
        what = "forward"
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": _cpu_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"{what} of {n_tokens} tokens of {w.name} (T={w.T}), float64, "
                      "one expert's weights converted at a time, NumPy BLAS threads"}


def run_reference(args, w):
    _, rank, _ = _dist()
    if rank != 0:
        return 0
    inp = synth.make_inputs(w, 0)
    steps = args.steps if args.steps > 0 else 3
    for _ in range(args.warmup):          # untimed, as the GPU arm's warm-up steps
        cpu_oracle_sample(w, inp, args.ref_tokens)
    times = [cpu_oracle_sample(w, inp, args.ref_tokens)["seconds"] for _ in range(steps)]
    sec_per_token = float(np.mean(times)) / args.ref_tokens
    value = 1.0 / sec_per_token
    # a step of this arm is one sampled step of ref_tokens tokens; its
    # ms_per_step is that step's measured time. The full batch's time at the
    # same rate is an extrapolation, reported under its own name.
    line = {"impl": "reference", "metric": "MoE expert-block tokens/s", "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "ms_per_step": float(np.mean(times)) * 1e3,
            "tokens_per_step": args.ref_tokens,
            "extrapolated_ms_per_full_batch": sec_per_token * w.T * 1e3,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _cpu_threads(),
                             "kind": "oracle",
                             "sample": f"{args.ref_tokens} tokens per step of {w.name}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU runs

class Runner:
    """The timed step of one workload kind, its per-kernel events and FLOPs."""

    def __init__(self, m, w, inp, device, fuse_gather=False, mx_tile_n=0, gate=False, chunks=0,
                 gemm_sms=0, cta_pairs=0):
        import torch
        self.m, self.w, self.dev = m, w, device
        self.gate = gate
        self.chunks = chunks
        if chunks and (w.mxfp8 or gate):
            raise SystemExit("--chunks runs the BF16 block from given ids only")
        if chunks and w.T % chunks:
            raise SystemExit(f"--chunks {chunks} does not divide T = {w.T}")
        if gate:
            if w.mxfp8 or w.routing not in ("router", "gaussian"):
                raise SystemExit(f"--gate needs a BF16 workload routed from logits, not {w.name}")
            # router logits in, routing out: the fused gate replaces the counting step
            self.logits = synth.router_logits(w, 0, inp["x"]).to(device)
        T, H, F, E, k = w.T, w.H, w.F, w.E, w.k
        R = T * k
        self.x = inp["x"].to(device)
        self.ids, self.probs = inp["expert_ids"].to(device), inp["probs"].to(device)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        self.stream = torch.cuda.current_stream()
        mk = lambda n: [torch.cuda.Event(enable_timing=True) for _ in range(n)]  # noqa: E731
        self.fev = mk(m.STEP_EVENTS)
        self.bev = (mk(m.MX_BWD_STEP_EVENTS if w.mxfp8 else m.BWD_STEP_EVENTS) if w.backward
                    else [])
        self.qev = mk(1)
        for e in self.fev + self.bev + self.qev:
            e.record(self.stream)
        if w.mxfp8:
            self.wq = []
            self.w_bf16 = [inp[key].to(device) for key in ("w_gate_t", "w_up_t", "w_down_t")]
            for wt in self.w_bf16:
                q, s = m.moe_quantize_mxfp8(wt)
                self.wq += [q, s]
            save = bool(w.backward)
            # forward only: the weights are held in MXFP8 across steps, their
            # scales laid out once for the block-scaled MMAs
            pretiled = not w.backward
            if pretiled:
                self.wq[1], self.wq[5] = m.moe_tile_weight_scales_mxfp8(
                    self.wq[1], self.wq[3], self.wq[5], cfg=m.config(mxfp8_tile_n=mx_tile_n))
                self.wq[3] = None
            self.pretiled = pretiled
            self.launches = 8 if pretiled else 10
            self.cfg = m.config(mxfp8_tile_n=mx_tile_n, save_for_backward=save,
                                cta_pairs=cta_pairs, mx_scales_pretiled=pretiled)
            self.cfg_ev = m.config(step_events=self.fev, mxfp8_tile_n=mx_tile_n,
                                   save_for_backward=save, cta_pairs=cta_pairs,
                                   mx_scales_pretiled=pretiled)
            nbytes = m.moe_workspace_size_mxfp8(T, H, F, E, k, self.cfg)
            self.dtype = "mxfp8 (e4m3 + e8m0 per 32; bf16 out)"
            if w.backward:
                # training re-quantises its weights every step, in the forward's
                # orientation and in the backward's (along the other axis)
                self.wq_b = [None] * 6
                for i, wt in enumerate(self.w_bf16):
                    self.wq_b[2 * i], self.wq_b[2 * i + 1] = m.moe_quantize_mxfp8_t(wt)
                self.dy = inp["dy"].to(device)
                self.cfg_bev = m.config(save_for_backward=True, step_events=self.bev,
                                        mxfp8_tile_n=mx_tile_n, cta_pairs=cta_pairs)
                self.bws = torch.empty(m.moe_workspace_size_mxfp8_backward(T, H, F, E, k),
                                       dtype=torch.uint8, device=device)
                self.grads = dict(
                    dx=torch.empty_like(self.x),
                    dw_gate_t=torch.empty((E, F, H), dtype=torch.float32, device=device),
                    dw_up_t=torch.empty((E, F, H), dtype=torch.float32, device=device),
                    dw_down_t=torch.empty((E, H, F), dtype=torch.float32, device=device),
                    dprobs=torch.empty((T, k), dtype=torch.float32, device=device))
                # weights 3 (both orientations each), forward 10 + zero padding,
                # backward 14
                self.launches = 3 + 11 + 14
        else:
            self.wg, self.wu, self.wd = (inp[key].to(device) for key in ("w_gate", "w_up", "w_down"))
            save = bool(w.backward)
            self.cfg = m.config(save_for_backward=save, fuse_gather=fuse_gather, num_sms=gemm_sms,
                                cta_pairs=cta_pairs)
            self.cfg_ev = m.config(save_for_backward=save, fuse_gather=fuse_gather,
                                   num_sms=gemm_sms, step_events=self.fev, cta_pairs=cta_pairs)
            nbytes = m.moe_workspace_size(T, H, F, E, k, self.cfg)
            if chunks and not w.backward:
                nbytes = max(nbytes, m._lib.moe_workspace_size_pipelined(T, H, F, E, k, chunks))
            self.dtype = "bf16"
            self.launches = 6 if (fuse_gather and not save) else 7
            if gate:
                self.launches -= 1          # one gate kernel for the histogram and scan pair
            if chunks:
                self.launches = 7 * min(chunks, T)   # the whole forward once per chunk
            if w.backward:
                self.dy = inp["dy"].to(device)
                self.cfg_bev = m.config(save_for_backward=True, step_events=self.bev,
                                        cta_pairs=cta_pairs)
                self.bws = torch.empty(m.moe_workspace_size(T, H, F, E, k, self.cfg, True),
                                       dtype=torch.uint8, device=device)
                self.grads = dict(
                    dx=torch.empty_like(self.x),
                    dw_gate=torch.empty((E, H, F), dtype=torch.float32, device=device),
                    dw_up=torch.empty((E, H, F), dtype=torch.float32, device=device),
                    dw_down=torch.empty((E, F, H), dtype=torch.float32, device=device),
                    dprobs=torch.empty((T, k), dtype=torch.float32, device=device))
                self.launches = (7 if gate else 8) + 7
                if chunks:
                    # micro-batches: the whole step once per chunk, one chunk's
                    # workspaces reused by every chunk
                    tc = T // chunks
                    self.launches = 15 * chunks
                    self.cwork = torch.empty(m.moe_workspace_size(tc, H, F, E, k, self.cfg),
                                             dtype=torch.uint8, device=device)
                    self.cbws = torch.empty(m.moe_workspace_size(tc, H, F, E, k, self.cfg, True),
                                            dtype=torch.uint8, device=device)
        self.work = torch.empty(nbytes, dtype=torch.uint8, device=device)
        # per-kernel FLOPs of the grouped GEMMs (algorithmic: routed rows only)
        self.flops = {"fc1_swiglu": 4.0 * R * H * F, "fc2": 2.0 * R * F * H}
        if w.backward:
            self.flops.update({"dH_swiglu_bwd": 2.0 * R * H * F, "dXp": 4.0 * R * H * F,
                               "dW1": 4.0 * R * H * F, "dW2": 2.0 * R * F * H})

    def step(self, events: bool, x=None, ids=None, probs=None, dy=None, logits=None,
             plain=False):
        """One step; with --chunks the pipelined forward unless plain (the
        single-stream forward that records the per-kernel events)."""
        m = self.m
        x = self.x if x is None else x
        ids = self.ids if ids is None else ids
        probs = self.probs if probs is None else probs
        if self.w.mxfp8:
            if self.w.backward:
                if events:
                    self.qev[0].record(self.stream)
                for i, wt in enumerate(self.w_bf16):
                    m.moe_quantize_mxfp8_dual(wt, out=(self.wq[2 * i], self.wq[2 * i + 1],
                                                       self.wq_b[2 * i], self.wq_b[2 * i + 1]))
            m.moe_expert_forward_mxfp8(x, *self.wq, ids, probs, y=self.y, workspace=self.work,
                                       cfg=self.cfg_ev if events else self.cfg)
            if self.w.backward:
                g = self.grads
                m.moe_expert_backward_mxfp8(self.dy if dy is None else dy, x, *self.wq_b, ids,
                                            probs, self.work, dx=g["dx"],
                                            dw_gate_t=g["dw_gate_t"], dw_up_t=g["dw_up_t"],
                                            dw_down_t=g["dw_down_t"], dprobs=g["dprobs"],
                                            workspace=self.bws,
                                            cfg=self.cfg_bev if events else self.cfg)
            return
        if self.chunks and self.w.backward and not plain:
            # the training step over micro-batches of T / chunks tokens: each
            # chunk's forward and backward, dX, dprobs and y into the chunk's
            # rows, the weight gradients accumulated over the chunks
            g, tc = self.grads, self.w.T // self.chunks
            dy = self.dy if dy is None else dy
            for c in range(self.chunks):
                sl = slice(c * tc, (c + 1) * tc)
                m.moe_expert_forward(x[sl], self.wg, self.wu, self.wd, ids[sl], probs[sl],
                                     y=self.y[sl], workspace=self.cwork, cfg=self.cfg)
                m.moe_expert_backward(dy[sl], x[sl], self.wg, self.wu, self.wd, ids[sl],
                                      probs[sl], self.cwork, dx=g["dx"][sl], dw_gate=g["dw_gate"],
                                      dw_up=g["dw_up"], dw_down=g["dw_down"],
                                      dprobs=g["dprobs"][sl], accumulate_dw=c > 0,
                                      workspace=self.cbws, cfg=self.cfg)
            return
        if self.chunks and not plain:
            m.moe_expert_forward_pipelined(x, self.wg, self.wu, self.wd, ids, probs, self.chunks,
                                           y=self.y, workspace=self.work, cfg=self.cfg)
        elif self.gate:                     # ids and probs are the gate's outputs
            m.moe_expert_forward_from_logits(x, self.wg, self.wu, self.wd,
                                             self.logits if logits is None else logits, self.w.k,
                                             y=self.y, expert_ids=ids, probs=probs,
                                             workspace=self.work,
                                             cfg=self.cfg_ev if events else self.cfg)
        else:
            m.moe_expert_forward(x, self.wg, self.wu, self.wd, ids, probs, y=self.y,
                                 workspace=self.work, cfg=self.cfg_ev if events else self.cfg)
        if self.w.backward:
            g = self.grads
            m.moe_expert_backward(self.dy if dy is None else dy, x, self.wg, self.wu, self.wd,
                                  ids, probs, self.work, dx=g["dx"], dw_gate=g["dw_gate"],
                                  dw_up=g["dw_up"], dw_down=g["dw_down"], dprobs=g["dprobs"],
                                  workspace=self.bws,
                                  cfg=self.cfg_bev if events else self.cfg)

    def parts(self):
        """Per-kernel milliseconds of the last event-recorded step."""
        f = self.fev
        out = {"routing": f[0].elapsed_time(f[1]), "fc1_swiglu": f[1].elapsed_time(f[2]),
               "fc2": f[2].elapsed_time(f[3]), "unpermute": f[3].elapsed_time(f[4])}
        if self.bev and self.w.mxfp8:
            out["quantise_weights"] = self.qev[0].elapsed_time(f[0])
            b = self.bev
            names = ["dO_dprobs_quantise", "dH_swiglu_bwd", "quantise_dA", "dXp", "dX",
                     "quantise_x_h", "dW1", "dW2"]
            for i, n in enumerate(names):
                out[n] = b[i].elapsed_time(b[i + 1])
        elif self.bev:
            b = self.bev
            names = ["dO_dprobs", "dH_swiglu_bwd", "dXp", "dX", "dW1", "dW2"]
            for i, n in enumerate(names):
                out[n] = b[i].elapsed_time(b[i + 1])
        return out


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
    run = Runner(m, w, inp, device, fuse_gather=args.fuse_gather, mx_tile_n=args.mxfp8_tile_n,
                 gate=args.gate, chunks=args.chunks, gemm_sms=args.gemm_sms,
                 cta_pairs=args.cta_pairs)
    stream = run.stream
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    warm = max(3, args.warmup)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(warm):
        flush.zero_()
        if i == warm - 1:
            w0.record(stream)
        run.step(False)
        if i == warm - 1:
            w1.record(stream)
    torch.cuda.synchronize()
    st = m.moe_get_error()
    if st != 0:
        raise RuntimeError(f"device error {st}")
    step_s = _max_over_ranks(max(w0.elapsed_time(w1), 1e-3) * 1e-3, ws, device)
    # steps: as asked, else enough for about a second of timed work; a
    # timed region shorter than that is preceded by untimed settle steps, so
    # that the clocks are sampled, and the timed steps run, under a load
    # that has lasted about a second
    if args.steps <= 0:
        args.steps = int(min(2000, max(20, np.ceil(1.0 / step_s))))
    settle = int(max(0, np.ceil((1.0 - args.steps * step_s) / step_s)))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    parts = {}
    graph = None
    if args.graph:
        # the whole step (every kernel of the block, launched through the C
        # ABI) captured once into a CUDA graph and replayed; step times come
        # from events on the launching stream around each replay, per-kernel
        # times from the ordinary stream launches below (events recorded
        # inside a graph cannot be timed)
        gstream = torch.cuda.Stream()
        gstream.wait_stream(stream)
        with torch.cuda.stream(gstream):
            run.step(False)                   # warm the capture stream
            torch.cuda.current_stream().synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gstream):
                run.step(False)
        stream.wait_stream(gstream)
        torch.cuda.synchronize()
    separate_parts = graph is not None or run.chunks > 0
    if separate_parts:
        for _ in range(args.steps):
            flush.zero_()
            run.step(True, plain=True)
            run.fev[-1].synchronize()
            if run.bev:
                run.bev[-1].synchronize()
            for key, v in run.parts().items():
                parts[key] = parts.get(key, 0.0) + v
        torch.cuda.synchronize()
    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for _ in range(settle):
            flush.zero_()
            if graph is not None:
                graph.replay()
            else:
                run.step(False)
        torch.cuda.synchronize()
        t_timed0 = time.monotonic()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            if graph is not None:
                graph.replay()
            else:
                run.step(True)
            ends[i].record(stream)
            ends[i].synchronize()
            if not separate_parts:
                for key, v in run.parts().items():
                    parts[key] = parts.get(key, 0.0) + v
        torch.cuda.synchronize()
        clk.timed = (t_timed0, time.monotonic())
    _barrier(ws)
    ms = _max_over_ranks(float(np.mean([s.elapsed_time(e) for s, e in zip(starts, ends)])), ws,
                         device)
    parts = {key: v / args.steps for key, v in parts.items()}
    if m.moe_get_error() != 0:
        raise RuntimeError("device error during the timed region")

    # end to end through the public calls with host buffers: every step copies
    # its own inputs from pinned host memory and reads its result back. Two
    # copy streams double-buffer them, so that step i+1's inputs and step
    # i-1's result move while step i computes, as a serving loop would run;
    # E = steps x tokens over the whole span, first copy to last read back.
    pin = lambda t: t.pin_memory()  # noqa: E731
    nb = 2
    hx, hids, hprobs = pin(inp["x"]), pin(inp["expert_ids"]), pin(inp["probs"])
    dx_ = [torch.empty_like(run.x) for _ in range(nb)]
    dids = [torch.empty_like(run.ids) for _ in range(nb)]
    dprobs = [torch.empty_like(run.probs) for _ in range(nb)]
    h2d = hx.numel() * 2 + hids.numel() * 4 + hprobs.numel() * 4
    if run.gate:                            # logits in; ids and probs come from the gate
        hlogits = pin(run.logits.cpu())
        dlogits = [torch.empty_like(run.logits) for _ in range(nb)]
        h2d = hx.numel() * 2 + hlogits.numel() * 4
    if w.backward:
        hdy = pin(inp["dy"])
        ddy = [torch.empty_like(run.dy) for _ in range(nb)]
        h2d += hdy.numel() * 2
        dres = [[run.grads["dx"], run.grads["dprobs"]]]
        dres += [[torch.empty_like(t) for t in dres[0]] for _ in range(nb - 1)]
    else:
        dres = [[run.y]] + [[torch.empty_like(run.y)] for _ in range(nb - 1)]
    hres = [[torch.empty_like(t, device="cpu").pin_memory() for t in ds] for ds in dres]
    d2h = sum(t.numel() * t.element_size() for t in hres[0])
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nb)]
    ev_done = [torch.cuda.Event() for _ in range(nb)]
    ev_out = [torch.cuda.Event() for _ in range(nb)]

    def e2e_step(i):
        b = i % nb
        with torch.cuda.stream(up):
            if i >= nb:
                up.wait_event(ev_done[b])    # step i - nb has read slot b's inputs
            dx_[b].copy_(hx, non_blocking=True)
            if run.gate:
                dlogits[b].copy_(hlogits, non_blocking=True)
            else:
                dids[b].copy_(hids, non_blocking=True)
                dprobs[b].copy_(hprobs, non_blocking=True)
            if w.backward:
                ddy[b].copy_(hdy, non_blocking=True)
            ev_in[b].record(up)
        stream.wait_event(ev_in[b])
        if i >= nb:
            stream.wait_event(ev_out[b])     # slot b's previous result has been read back
        if w.backward:
            run.grads["dx"], run.grads["dprobs"] = dres[b]
        else:
            run.y = dres[b][0]
        run.step(False, x=dx_[b], ids=dids[b], probs=dprobs[b],
                 dy=ddy[b] if w.backward else None, logits=dlogits[b] if run.gate else None)
        ev_done[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[b])
            for h, d in zip(hres[b], dres[b]):
                h.copy_(d, non_blocking=True)
            ev_out[b].record(down)

    for i in range(nb):                      # warm-up through both slots
        e2e_step(i)
    torch.cuda.synchronize()
    _barrier(ws)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(up)
    for i in range(nb, nb + args.steps):
        e2e_step(i)
    t1.record(down)
    torch.cuda.synchronize()
    piped_ms = t0.elapsed_time(t1) / args.steps

    # the same steps one after another on the compute stream (copy in, block,
    # read back), each timed alone after an L2 flush: for launch-bound
    # shapes the pipeline's extra stream and event calls cost more host time
    # than the copies it hides
    seq_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    seq_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps + 2):
        flush.zero_()
        if i >= 2:
            seq_s[i - 2].record(stream)
        dx_[0].copy_(hx, non_blocking=True)
        if run.gate:
            dlogits[0].copy_(hlogits, non_blocking=True)
        else:
            dids[0].copy_(hids, non_blocking=True)
            dprobs[0].copy_(hprobs, non_blocking=True)
        if w.backward:
            ddy[0].copy_(hdy, non_blocking=True)
        if w.backward:
            run.grads["dx"], run.grads["dprobs"] = dres[0]
        else:
            run.y = dres[0][0]
        run.step(False, x=dx_[0], ids=dids[0], probs=dprobs[0],
                 dy=ddy[0] if w.backward else None, logits=dlogits[0] if run.gate else None)
        for h, d in zip(hres[0], dres[0]):
            h.copy_(d, non_blocking=True)
        if i >= 2:
            seq_e[i - 2].record(stream)
    torch.cuda.synchronize()
    seq_ms = float(np.mean([a.elapsed_time(b) for a, b in zip(seq_s, seq_e)]))
    e2e_loop = "pipelined" if piped_ms <= seq_ms else "sequential"
    e2e_ms = _max_over_ranks(min(piped_ms, seq_ms), ws, device)

    # every timed step follows about a second of load (the settle pass, or the
    # timed region itself): the kernels run at the clocks of sustained work,
    # under the power cap, so they are held to the sustained peak
    hbm, bf16_peak, peak_src = _peaks(sustained=True)
    peak = bf16_peak * (FP8_OVER_BF16 if w.mxfp8 else 1.0)
    tflops = {key: run.flops[key] / (parts[key] * 1e-3) / 1e12 for key in run.flops}
    dominant = max(run.flops, key=lambda key: parts[key])
    tr = TRAFFIC.get((w.name, dominant))
    traffic = tr["bytes"] if tr and tr["src_sha"] == _sha_of_sources(tr["sources"]) else None
    gemm_ms = sum(parts[key] for key in run.flops)
    line = {
        "metric": "MoE expert-block tokens/s", "value": ws * w.T / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": warm,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": run.dtype, "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k,
                   "step": "forward + backward" if w.backward else "forward",
                   "dispatch": "gathered by fc1's cp.async warps" if (args.fuse_gather and not
                                                                   w.backward and not w.mxfp8)
                   else "materialised permute",
                   "l2": "flushed before every step (512 MB write)",
                   "e2e": {"loop": e2e_loop,
                           "pipelined": ("host buffers double-buffered on two copy streams: "
                                         "step i+1's inputs and step i-1's result move while "
                                         "step i computes; no L2 flush in that loop"),
                           "sequential": "copy in, block, read back; L2 flushed before each",
                           "tokens_per_s": {"pipelined": ws * w.T / (piped_ms * 1e-3),
                                            "sequential": ws * w.T / (seq_ms * 1e-3)}},
                   "launch": "one CUDA graph per step" if args.graph else "stream launches",
                   "settle_steps": settle,
                   "settle": ("untimed steps run right before the timed region, after the "
                              "warm-up, when the timed region alone is shorter than a second: "
                              "the clocks are sampled, and the timed steps run, under a load "
                              "that has lasted about a second"),
                   "pipeline": (("micro-batch split of the training step into "
                                 f"{run.chunks} chunks of {w.T // run.chunks} tokens, dW "
                                 "accumulated (per-kernel times from unsplit steps)")
                                if run.chunks and w.backward else
                                (f"{run.chunks} token chunks, routing and combine on a second "
                                 "stream (per-kernel times from unpipelined steps)")
                                if run.chunks else "none"),
                   "gemm_ctas": args.gemm_sms or "one per SM",
                   "cta_pairs": {0: "automatic", 1: "off", 2: "on"}[args.cta_pairs],
                   **({"mx_weight_scales": ("laid out once for the block-scaled MMAs "
                                            "(weights held in MXFP8 across steps)"
                                            if run.pretiled else
                                            "quantised and laid out in every step")}
                      if w.mxfp8 else {}),
                   "routing": ("fused top-k gate from float32 router logits [T, E]" if run.gate
                               else "expert ids and weights given"),
                   "parallelism": "replicas" if ws > 1 else "single"},
        "roofline": {"bound": "tensor", "kernel": f"{dominant} (grouped GEMM)",
                     "achieved": tflops[dominant], "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops[dominant] / peak, "traffic": traffic,
                     "peak_source": peak_src + (" x 2 (nominal FP8/BF16)" if w.mxfp8 else "")},
        "steps_ms": parts,
        "gemm_tflops": tflops,
        "grouped_gemm_tflops": sum(run.flops.values()) / (gemm_ms * 1e-3) / 1e12,
        "e2e": {"value": ws * w.T / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": run.launches * args.steps,
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


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (default: enough for about a second of timed work; "
                         "3 sampled steps for --impl reference)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral_bf16", choices=list(synth.WORKLOADS))
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mxfp8-tile-n", type=int, default=0, choices=[0, 128, 256])
    ap.add_argument("--gate", action="store_true",
                    help="BF16 forward from router logits: the fused top-k gate replaces the "
                         "counting step")
    ap.add_argument("--chunks", type=int, default=0,
                    help="BF16 forward: micro-batch pipeline over this many token chunks; "
                         "BF16 training step: run it as this many micro-batches")
    ap.add_argument("--gemm-sms", type=int, default=0,
                    help="persistent GEMM grid size (default: one CTA per SM)")
    ap.add_argument("--cta-pairs", type=int, default=0, choices=[0, 1, 2],
                    help="GEMMs over routed rows: 2 = CTA pairs share M = 256 tiles, "
                         "1 = one CTA per tile, 0 = automatic")
    ap.add_argument("--graph", action="store_true",
                    help="capture each step once into a CUDA graph and replay it")
    ap.add_argument("--fuse-gather", action=argparse.BooleanOptionalAction, default=False,
                    help="BF16 forward: fc1 gathers the routed rows itself (no permuted copy)")
    return ap


def main():
    args = build_parser().parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
