#!/usr/bin/env python
"""Throughput of one MoE layer's forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config qwen3|dsv2lite|skew|drafter|tiny]

A step is one pass of the whole hot path over one batch of synthetic input:
route top-k, histogram/offsets/permutation, the simulated expert-parallel
layout (with its one device-to-host copy), dispatch, grouped SwiGLU experts,
combine, and the backward of each. Rank 0 prints one JSON line.

* value: tokens/s over all ranks, inputs resident in HBM, per-step CUDA events
  on the launching stream; before every timed step, outside its events, L2 is
  flushed by writing a 256 MiB buffer and then reading another 256 MiB one (so
  no dirty flush lines are left for the step's first kernel to write back).
* step_ms_median, step_ms_min_max, aa: the spread of the timed steps and the
  same K steps timed again back to back (A/A noise floor).
* e2e: the same metric through the layer API with pinned host buffers
  (MoELayer.run_from_host over the timed steps): each step copies logits, x
  and dout in and the output and input gradient out; step i+1's upload and
  step i's download overlap compute on two copy streams, and the first upload
  and the last download fall inside the timed region.
* roofline: the dominant kernel's algorithmic flops (or bytes) per launch over
  its average launch duration, from per-launch events the library records on
  the launching stream during a second pass of the same timed steps (the
  first pass, which gives `value`, has no events between launches, so each
  kernel can be launched while its predecessor finishes).
* cpu_baseline: the CPU oracle timed on a bounded sample of the same workload.
* --impl reference: the CPU oracle as the reference arm (rank 0 only).

Multi-GPU runs (torchrun) are independent replicas with no data-path
collective: every rank runs the same layer on its own GPU.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd tokens/s on 1 GB300; % of bf16 TC / HBM roofline per kernel"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the MXFP8 forward comparison")
    ap.add_argument("--no-side-configs", action="store_true",
                    help="report only the headline workload (no configs sub-object)")
    ap.add_argument("--cpu-sample-tokens", type=int, default=0)
    ap.add_argument("--profile-case", choices=["gemm", "gemm_ragged", "gemm_l2", "gemm_drafter",
                                               "gemm_drafter64", "layer", "hbm", "routing",
                                               "combine_side", "fp8"],
                    default=None,
                    help="run a small fixed case twice for an ncu capture and exit")
    return ap.parse_args()


def profile_case(which: str):
    """Small cases for ncu captures (inputs above the 129 MB L2, a few GB on the device).

    gemm:    the grouped-GEMM entry points, forward and backward, on E=64 experts x 512 rows
             (d=2048, I=768; the qwen3 workload's rows per expert), run twice.
    gemm_ragged: as gemm, with seeded expert sizes 512 + round(N(0, 21)) (the spread of the
             qwen3 workload's routed rows; most experts end inside a K16 step), run twice.
    gemm_drafter: the grouped-GEMM entry points on the drafter workload's expert shape (d=4096,
             I=2048) with E=8 experts of 4096 + round(N(0, 64)) rows (~3.2 GB on the device),
             run twice: the tensor-bound regime of the headline workload.
    gemm_drafter64: the same with all 64 of the drafter's experts (~21 GB on the device).
    gemm_l2: the same entry points on one expert of 16384 rows (d=2048, I=768): weights
             and activations mostly resident in L2, which isolates the kernels' own
             pipeline from DRAM streaming.
    layer:   one qwen3-shaped layer at T=2048 tokens (forward + backward), run twice.
    routing: the forward's front on the qwen3 workload at full size (the fused route +
             permutation + EP layout with its host copy, token-major dispatch), run twice;
             ~0.4 GB on the device.
    fp8:     the MXFP8 forward (weight quantization, then moe_grouped_ffn_fp8) on E=64 experts
             x 512 rows (d=2048, I=768), run twice; ~1.5 GB on the device.
    combine_side: the combine, its backward and the dispatch backward at the qwen3 workload's
             full size (T=8192, d=2048, K=8; the routing of the qwen3 inputs), on synthetic
             expert outputs and gradients (~1.1 GB on the device), run twice, with 256 MiB
             of L2-flushing writes before each kernel.
    hbm:     HBM bandwidth by access pattern on 2 GiB fp32 buffers (torch's fill, sum and
             copy; CUDA events, 20 launches after 3 warm-ups): the ceilings that write-only,
             read-only and copy-like kernels are compared with.
    Prints each kernel's launch time (CUDA events on the launching stream) and rate for
    the last run.
    """
    import torch
    if which == "hbm":
        dev = torch.device("cuda:0")
        n = 1 << 29
        a = torch.full((n,), 1.0, device=dev)
        b = torch.full((n,), 2.0, device=dev)

        def rate(fn, nbytes, reps=20):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(reps):
                fn()
            e.record()
            torch.cuda.synchronize()
            return nbytes / (s.elapsed_time(e) / reps * 1e-3) / 1e9

        print(json.dumps({"write_gbs": rate(lambda: a.fill_(3.0), 4 * n),
                          "read_gbs": rate(lambda: torch.sum(a), 4 * n),
                          "copy_gbs": rate(lambda: b.copy_(a), 8 * n)}))
        return
    from grouped_gemm_moe_gb300 import binding as B
    from grouped_gemm_moe_gb300 import build as build_mod
    from grouped_gemm_moe_gb300 import layer as L
    from grouped_gemm_moe_gb300 import workloads as W
    if not os.path.exists(B.LIB_PATH):
        build_mod.build()
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(0)
    flops = {}
    if which in ("gemm", "gemm_ragged", "gemm_l2", "gemm_drafter", "gemm_drafter64"):
        E, d, I, rows = {"gemm_l2": (1, 2048, 768, 16384),
                         "gemm_drafter": (8, 4096, 2048, 4096),
                         "gemm_drafter64": (64, 4096, 2048, 4096)}.get(which, (64, 2048, 768, 512))
        if which in ("gemm_ragged", "gemm_drafter", "gemm_drafter64"):
            gc = torch.Generator().manual_seed(3)
            spread = 21 if which == "gemm_ragged" else 64
            sizes = (rows + torch.randn(E, generator=gc) * spread).round().clamp(min=1).to(torch.int64)
        else:
            sizes = torch.full((E,), rows, dtype=torch.int64)
        M = int(sizes.sum())
        flops = {"gemm_gate_up": 4 * M * d * I, "gemm_down": 2 * M * d * I, "gemm_dh": 2 * M * d * I,
                 "gemm_dx": 4 * M * d * I, "gemm_wgrad_gate_up": 4 * M * d * I,
                 "gemm_wgrad_down": 2 * M * d * I}
        bf = torch.bfloat16
        rnd = lambda *s, sc=1.0: (torch.randn(*s, device=dev, generator=g) * sc).to(bf)  # noqa: E731
        off = torch.cat([torch.zeros(1, dtype=torch.int64), sizes.cumsum(0)]).to(torch.int32).to(dev)
        xp, dy, gu, h = rnd(M, d), rnd(M, d, sc=0.1), rnd(M, 2 * I), rnd(M, I, sc=0.5)
        wg, wu, wd = rnd(E, d, I, sc=0.02), rnd(E, d, I, sc=0.02), rnd(E, I, d, sc=0.02)
        for it in range(2):
            if it == 1:
                torch.cuda.synchronize()
                B.moe_profile_start(64)
            B.moe_grouped_ffn_backward(dy, xp, gu, h, off, wg, wu, wd)
            B.moe_grouped_ffn(xp, off, wg, wu, wd)
    elif which == "fp8":
        E, d, I, rows = 64, 2048, 768, 512
        M = E * rows
        bf = torch.bfloat16
        rnd = lambda *s, sc=1.0: (torch.randn(*s, device=dev, generator=g) * sc).to(bf)  # noqa: E731
        off = (torch.arange(E + 1, dtype=torch.int32) * rows).to(dev)
        xp = rnd(M, d)
        wg, wu, wd = rnd(E, d, I, sc=0.02), rnd(E, d, I, sc=0.02), rnd(E, I, d, sc=0.02)
        flops = {"gemm_gate_up_fp8": 4 * M * d * I, "gemm_down_fp8": 2 * M * d * I}
        for it in range(2):
            if it == 1:
                torch.cuda.synchronize()
                B.moe_profile_start(64)
            wgu = B.moe_mxfp8_quantize_weights(wg, wu)
            wdq = B.moe_mxfp8_quantize_weights(wd)
            B.moe_grouped_ffn_fp8(xp, off, wgu, wdq)
    elif which == "combine_side":
        cfg = W.CONFIGS["qwen3"]
        inp = W.make_inputs(cfg, with_backward=False)
        idx, w = B.moe_route_topk(inp["logits"].to(dev), cfg.K, cfg.renorm)
        _, _, _, inv = B.moe_build_permutation(idx, cfg.E)
        TK, d = cfg.T * cfg.K, cfg.d
        y = (torch.randn(TK, d, device=dev, generator=g) * 0.1).to(torch.bfloat16)
        dxp = (torch.randn(TK, d, device=dev, generator=g) * 0.1).to(torch.bfloat16)
        dout = torch.randn(cfg.T, d, device=dev, generator=g).to(torch.bfloat16)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        for it in range(2):
            if it == 1:
                torch.cuda.synchronize()
                B.moe_profile_start(64)
            flush.zero_()
            B.moe_combine(y, w, inv)
            flush.zero_()
            B.moe_combine_backward(dout, y, w, inv)
            flush.zero_()
            B.moe_dispatch_backward(dxp, inv, cfg.T, cfg.K)
        torch.cuda.synchronize()
        for name, ms in B.moe_profile_stop():
            print(f"  {name:22s} {ms * 1e3:9.1f} us")
    elif which == "routing":
        cfg = W.CONFIGS["qwen3"]
        inp = W.make_inputs(cfg, with_backward=False)
        logits, x = inp["logits"].to(dev), inp["x"].to(dev)
        host = torch.empty(cfg.R * cfg.E + cfg.R * cfg.R, dtype=torch.int32).pin_memory()
        for it in range(2):
            if it == 1:
                torch.cuda.synchronize()
                B.moe_profile_start(64)
            res = B.moe_route_permute_ep(logits, cfg.K, cfg.R, cfg.renorm, host_splits=host)
            B.moe_dispatch_scatter(x, res[5], cfg.K)
        torch.cuda.synchronize()
        for name, ms in B.moe_profile_stop():
            print(f"  {name:22s} {ms * 1e3:9.1f} us")
    else:
        cfg = W.MoEConfig("qwen3-2k", T=2048, d=2048, E=128, K=8, I=768, R=8)
        inp = W.make_inputs(cfg)
        layer = L.layer_from_config(cfg, inp, dev)
        logits, x, dout = (inp[k].to(dev) for k in ("logits", "x", "dout"))
        for _ in range(2):
            layer.forward(logits, x)
            layer.backward(dout)
    torch.cuda.synchronize()
    if flops:
        for name, ms in B.moe_profile_stop():
            print(f"  {name:22s} {ms * 1e3:9.1f} us  {flops.get(name, 0) / (ms * 1e-3) / 1e12:8.1f} TFLOP/s")
    print(f"profile case {which} ok, peak {torch.cuda.max_memory_allocated() / 2**30:.2f} GiB")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's figure (replicas run the same work; the job is done
    when the last one is)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(ms_per_step: float, tokens_per_rank: int, world: int) -> float:
    """Whole-job tokens/s: every rank processes its own batch in ms_per_step."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ------------------------------------------------------------------ work model
def kernel_work(name: str, cfg, shared: bool):
    """Algorithmic work of one launch: (flops, bytes). Bytes count each input
    read once and each output written once (bf16 activations and weights,
    fp32 weight gradients, int32 indices), i.e. no re-reads."""
    T, d, E, K, I = cfg.T, cfg.d, cfg.E, cfg.K, cfg.I
    TK = T * K
    if shared:
        M, Ie, Ee = T, cfg.shared_I, 1
    else:
        M, Ie, Ee = TK, I, E
    w1 = 2 * Ee * d * Ie * 2          # W_gate + W_up, bf16
    wd = Ee * Ie * d * 2              # W_down, bf16
    gemm = {
        "gemm_gate_up": (4 * M * d * Ie, M * d * 2 + w1 + M * Ie * 2 + M * 2 * Ie * 2),
        "gemm_down": (2 * M * Ie * d, M * Ie * 2 + wd + M * d * 2),
        "gemm_dh": (2 * M * d * Ie, M * d * 2 + wd + 2 * (M * 2 * Ie * 2)),
        "gemm_dx": (4 * M * d * Ie, M * 2 * Ie * 2 + w1 + M * d * 2),
        "gemm_wgrad_gate_up": (4 * M * d * Ie, M * d * 2 + M * 2 * Ie * 2 + 2 * Ee * d * Ie * 4),
        "gemm_wgrad_down": (2 * M * Ie * d, M * Ie * 2 + M * d * 2 + Ee * Ie * d * 4),
    }
    if name in gemm:
        return gemm[name]
    hbm = {
        "route_topk": T * (4 * E + 8 * K),
        # the fused front: logits read and top-k written (route_hist), then the ids
        # read and five index arrays written (place_ep)
        "route_hist": T * (4 * E + 8 * K),
        "place_ep": 24 * TK,
        "route_topk_backward": T * (12 * K + 4 * E),
        "perm_hist": 4 * TK, "perm_scatter": 12 * TK, "ep_hist": 4 * TK,
        # the layer's fused call also writes perm and inv_perm from the EP scatter
        "ep_scatter": 24 * TK,
        "dispatch": T * (2 * d * (1 + K) + 4 * K),
        "combine": T * (2 * d * K + 8 * K + 2 * d + (2 * d if cfg.shared_I else 0)),
        "combine_backward": T * (2 * d + 4 * d * K + 12 * K),
        "dispatch_backward": T * (2 * d * K + 4 * K + 2 * d + (2 * d if cfg.shared_I else 0)),
    }
    return 0, hbm.get(name, 0)


# nominal GB300 figures (context beside the measured peaks): HBM3e and dense bf16
NOMINAL_GBS = 7900.0
NOMINAL_TFLOPS = 2250.0

KERNEL_SOURCE = {"route_hist": "front.cu", "place": "front.cu", "route": "route.cu",
                 "perm": "permute.cu",
                 "ep_": "permute.cu",
                 "dispatch": "gather.cu", "combine": "gather.cu", "gemm": "grouped_gemm.cu"}


def code_digest(path: str) -> str:
    """sha256 of a C++/CUDA source with its comments and blank lines removed
    (line comments outside string literals, block comments), so that an edit
    of the comments keeps a measured figure while any change of code drops it."""
    import hashlib
    import re
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = []
    for line in text.splitlines():
        code, in_str, i = [], False, 0
        while i < len(line):
            ch = line[i]
            if ch == '"' and (i == 0 or line[i - 1] != "\\"):
                in_str = not in_str
            if not in_str and line.startswith("//", i):
                break
            code.append(ch)
            i += 1
        stripped = "".join(code).rstrip()
        if stripped.strip():
            out.append(stripped)
    return hashlib.sha256("\n".join(out).encode()).hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu
    summary under profiles/: a line 'traffic-record: kernel=<name>
    workload=<name> bytes_per_launch=<B> source=<file> code-sha256=<hex>'. The
    figure counts only while the kernel's source file still has the recorded
    code digest (code_digest; None otherwise)."""
    import glob
    here = os.path.dirname(os.path.abspath(__file__))
    src = next((f for pre, f in KERNEL_SOURCE.items() if kernel.startswith(pre)), None)
    if src is None:
        return None
    path = os.path.join(here, "grouped_gemm_moe_gb300", "csrc", src)
    if not os.path.exists(path):
        return None
    digest = code_digest(path)
    for md in sorted(glob.glob(os.path.join(here, "profiles", "*.md"))):
        for line in open(md):
            if not line.startswith("traffic-record:"):
                continue
            kv = dict(f.split("=", 1) for f in line.split()[1:] if "=" in f)
            if (kv.get("kernel") == kernel and kv.get("workload") == workload
                    and kv.get("source") == src and kv.get("code-sha256") == digest):
                return float(kv["bytes_per_launch"])
    return None


def roofline_of(flops: float, nbytes: float, ms: float, pk) -> dict:
    """The bound of one launch is whichever of its flops at the bf16 tensor peak
    or its bytes at HBM bandwidth takes longer; achieved is in that unit."""
    t_tc = flops / (pk["bf16_tflops_sustained"] * 1e12)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    if t_tc >= t_hbm and flops > 0:
        ach = flops / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops_sustained"],
                "roofline_ms": t_tc * 1e3}
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": ach / pk["hbm_gbs"], "roofline_ms": t_hbm * 1e3}


def label_records(records, steps):
    """Splits the launch records into steps and tags the second occurrence of a
    GEMM name within a step as the shared-expert launch."""
    if not records or len(records) % steps:
        return [(n, ms, False) for n, ms in records]
    per = len(records) // steps
    out = []
    for s in range(steps):
        seen = {}
        for n, ms in records[s * per:(s + 1) * per]:
            k = seen.get(n, 0)
            seen[n] = k + 1
            out.append((n, ms, n.startswith("gemm_") and k == 1))
    return out


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file if ln.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle
class OracleSample:
    """The CPU oracle on a bounded token sample of a workload. A step runs the
    oracle's forward and backward on the first T tokens, restricted to the
    experts those tokens select (relabelled in ascending order; with
    renormalised weights the selection and its weights are the same among them
    as among all E, and every other expert's work is zero); only that is timed.
    Token inputs are converted to float64 once; expert weights stay as
    bf16-exact float32 arrays, which the oracle converts one expert at a time,
    so a large workload's weights are never held in float64 all at once."""

    WEIGHTS = ("w_gate", "w_up", "w_down")
    SHARED = ("ws_gate", "ws_up", "ws_down")

    def __init__(self, cfg, inputs=None, t_max: int = 512):
        from grouped_gemm_moe_gb300 import workloads as W
        self.cfg = cfg
        t_max -= t_max % cfg.R
        if inputs is None:
            inputs = W.make_inputs(cfg, T=t_max, with_backward=True)
        t_max = min(t_max, inputs["logits"].shape[0])
        self.tok = {k: W.to_f64(inputs[k][:t_max]) for k in ("logits", "x", "dout")}
        self.wts = {k: inputs[k].float().numpy() for k in self.WEIGHTS + self.SHARED
                    if k in inputs}
        self.t_max = t_max
        self._cached = (None, None)

    def inputs(self, T: int):
        if self._cached[0] == T:
            return self._cached[1]
        import numpy as np
        from oracle import moe_oracle as O
        lg = self.tok["logits"][:T]
        idx, _ = O.route_topk(lg, self.cfg.K, self.cfg.renorm)
        used = np.unique(idx)
        whole = len(used) == self.cfg.E
        sub = {"logits": lg if whole else lg[:, used], "x": self.tok["x"][:T],
               "dout": self.tok["dout"][:T]}
        for k in self.WEIGHTS:
            sub[k] = self.wts[k] if whole else self.wts[k][used]
        for k in self.SHARED:
            if k in self.wts:
                sub[k] = self.wts[k]
        self._cached = (T, sub)
        return sub

    def step(self, T: int) -> float:
        from oracle import moe_oracle as O
        cfg = self.cfg
        inp = self.inputs(T)
        t0 = time.perf_counter()
        fwd = O.layer_forward(inp, cfg.K, 1, cfg.renorm)
        O.layer_backward(inp, fwd, inp["dout"], cfg.K, cfg.renorm)
        return time.perf_counter() - t0

    def tokens_for(self, seconds: float) -> int:
        """Token count whose step takes about ``seconds`` (linear fit through two
        probe sizes: the oracle has a fixed per-step cost of its own)."""
        R = self.cfg.R
        a, b = 2 * R, 8 * R
        self.step(a)                       # first call: page faults of the fp64 gradient arrays
        ta, tb = self.step(a), self.step(b)
        per_tok = max((tb - ta) / (b - a), 1e-9)
        fixed = max(ta - per_tok * a, 0.0)
        T = int((seconds - fixed) / per_tok) if seconds > fixed else R
        T = max(R, min(self.t_max, T))
        return T - T % R


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(cfg, tokens, inputs=None):
    smp = OracleSample(cfg, inputs)
    if tokens <= 0:
        tokens = smp.tokens_for(15.0)
    dt = smp.step(tokens)
    return {"value": tokens / dt, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"the first {tokens} of {cfg.T} tokens of the same workload, fwd+bwd, "
                      f"restricted to the experts they select (full-size expert weights), "
                      f"float64 NumPy, one run of {dt:.2f} s"}


def run_reference(args, cfg, world, rank):
    if rank != 0:
        return
    from grouped_gemm_moe_gb300 import workloads as W
    smp = OracleSample(cfg)
    n_steps = args.steps + args.warmup
    tokens = smp.tokens_for(max(90.0 / n_steps, 0.2))
    for _ in range(args.warmup):
        smp.step(tokens)
    times = [smp.step(tokens) for _ in range(args.steps)]
    ms = statistics.mean(times) * 1e3
    value = tokens / (ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) logits/activations, N(0,0.02) weights)",
        "config": {"workload": f"{cfg.name}: {W.describe(cfg)}, fwd+bwd",
                   "sample_tokens_per_step": tokens},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"the first {tokens} of {cfg.T} tokens per step, restricted to "
                                   f"the experts they select (full-size expert weights), "
                                   f"float64 NumPy oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
class Runner:
    """Times one workload's layer forward + backward on one GPU: K steps with
    per-step events (L2 flushed before each, outside the events), the same K
    steps again (A/A), and a third pass with the library's per-launch events
    for the per-kernel table."""

    def __init__(self, cfg, inputs, dev, flush_l2, world):
        import torch
        from grouped_gemm_moe_gb300 import layer as L
        self.cfg, self.dev, self.flush_l2, self.world = cfg, dev, flush_l2, world
        self.layer = L.layer_from_config(cfg, inputs, dev)
        self.logits, self.x, self.dout = (inputs[k].to(dev) for k in ("logits", "x", "dout"))
        self.stream = torch.cuda.current_stream(dev)

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def step(self):
        self.layer.forward(self.logits, self.x)
        self.layer.backward(self.dout)

    def warm(self, n: int, min_seconds: float = 0.0):
        import torch
        t0 = time.time()
        for _ in range(max(n, 3)):
            self.flush_l2()
            self.step()
        torch.cuda.synchronize()
        # keep the GPU busy long enough for the clock sampler to see it under load
        while time.time() - t0 < min_seconds:
            self.step()
            torch.cuda.synchronize()
        if self.layer.device_status() != 0:
            raise SystemExit("device status word reports an error")

    def timed(self, steps: int):
        import torch
        self.barrier()
        torch.cuda.synchronize()
        evs = []
        for _ in range(steps):
            self.flush_l2()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(self.stream)
            self.step()
            e.record(self.stream)
            evs.append((s, e))
        torch.cuda.synchronize()
        self.barrier()
        return [s.elapsed_time(e) for s, e in evs]

    def per_launch(self, steps: int):
        import torch
        from grouped_gemm_moe_gb300 import binding as B
        B.moe_profile_start(64 * steps + 64)
        for _ in range(steps):
            self.flush_l2()
            self.step()
        torch.cuda.synchronize()
        self.barrier()
        return B.moe_profile_stop()


def kernel_table(cfg, records, steps, pk):
    """Per-kernel launches, average duration, share and roofline, and the
    per-step algorithmic totals."""
    per = {}
    for n, kms, sh in label_records(records, steps):
        key = n + ("[shared]" if sh else "")
        c = per.setdefault(key, {"launches": 0, "total_ms": 0.0, "shared": sh, "name": n})
        c["launches"] += 1
        c["total_ms"] += kms
    tot = sum(c["total_ms"] for c in per.values()) or 1.0
    kernels = {}
    for k, c in per.items():
        fl, nb = kernel_work(c["name"], cfg, c["shared"])
        avg = c["total_ms"] / c["launches"]
        rf = roofline_of(fl, nb, avg, pk)
        kernels[k] = {"launches": c["launches"], "avg_ms": round(avg, 5),
                      "share": round(c["total_ms"] / tot, 4), "bound": rf["bound"],
                      "achieved": round(rf["achieved"], 1), "unit": rf["unit"],
                      "frac": round(rf["frac"], 4), "roofline_ms": round(rf["roofline_ms"], 5)}
    flops_step = sum(kernel_work(c["name"], cfg, c["shared"])[0] * c["launches"]
                     for c in per.values()) / steps
    bytes_step = sum(kernel_work(c["name"], cfg, c["shared"])[1] * c["launches"]
                     for c in per.values()) / steps
    layer_roof_ms = max(flops_step / (pk["bf16_tflops_sustained"] * 1e12),
                        bytes_step / (pk["hbm_gbs"] * 1e9)) * 1e3
    sum_roof_ms = sum(v["roofline_ms"] * v["launches"] for v in kernels.values()) / steps
    return per, kernels, flops_step, bytes_step, layer_roof_ms, sum_roof_ms


def side_config(name, args, dev, flush_l2, world, rank, pk):
    """One of the other forward + backward workloads: its step time, tokens/s,
    layer fraction of roofline and kernel table (fewer steps than the headline)."""
    import torch
    from grouped_gemm_moe_gb300 import workloads as W
    cfg = W.CONFIGS[name]
    inp = W.make_inputs(cfg, seed=cfg.seed + rank)
    run = Runner(cfg, inp, dev, flush_l2, world)
    steps = max(5, min(args.steps, 10))
    run.warm(3)
    step_ms = run.timed(steps)
    records = run.per_launch(steps)
    _, kernels, fl, nb, roof_ms, sum_ms = kernel_table(cfg, records, steps, pk)
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    out = {"workload": f"{cfg.name}: {W.describe(cfg)}, fwd+bwd", "steps": steps,
           "ms_per_step": ms, "step_ms_median": statistics.median(step_ms),
           "tokens_per_s": aggregate_value(ms, cfg.T, world),
           "step_tflop": fl / 1e12, "step_gbytes_algorithmic": nb / 1e9,
           "layer_roofline_ms": roof_ms, "layer_frac_of_roofline": roof_ms / ms,
           "sum_of_kernel_rooflines_ms": sum_ms, "gpu_launches": len(records),
           "kernels": kernels}
    del run, inp
    torch.cuda.empty_cache()
    return out


def load_balance_block(cfg, layer, logits, dev, flush_l2, steps, pk):
    """Load-balance metrics, loss and gradient on the headline routing (not part
    of the headline step): K timed iterations with per-launch events, L2
    flushed before each."""
    import torch
    from grouped_gemm_moe_gb300 import binding as B
    from grouped_gemm_moe_gb300 import workloads as W
    lb_frac, lb_pmean, lb_stats = (torch.empty(cfg.E, device=dev), torch.empty(cfg.E, device=dev),
                                   torch.empty(4, device=dev))
    lb_ws = B.new_workspace(B.workspace_size(B.MOE_OP_LOAD_BALANCE, cfg.T, cfg.E, cfg.K), dev)
    lb_dl = torch.zeros(cfg.T, cfg.E, device=dev)
    for _ in range(3):
        B.moe_load_balance(logits, layer.counts, cfg.K, ws=lb_ws, out=(lb_frac, lb_pmean, lb_stats))
        B.moe_load_balance_backward(logits, lb_frac, 0.01, dlogits=lb_dl, accumulate=True)
    torch.cuda.synchronize()
    B.moe_profile_start(16 * steps + 16)
    for _ in range(steps):
        flush_l2()
        B.moe_load_balance(logits, layer.counts, cfg.K, ws=lb_ws, out=(lb_frac, lb_pmean, lb_stats))
        B.moe_load_balance_backward(logits, lb_frac, 0.01, dlogits=lb_dl, accumulate=True)
    torch.cuda.synchronize()
    lb_rec = {}
    for n, kms in B.moe_profile_stop():
        lb_rec.setdefault(n, []).append(kms)
    TE = cfg.T * cfg.E
    lb_bytes = {"load_balance": 4 * TE, "load_balance_final": 4 * 256 * cfg.E + 12 * cfg.E,
                "load_balance_backward": 12 * TE + 4 * cfg.E}
    out = {"workload": f"{cfg.name} routing, logits [{cfg.T},{cfg.E}] fp32", "kernels": {}}
    for n, v in lb_rec.items():
        avg = statistics.mean(v)
        bw = lb_bytes.get(n, 0) / (avg * 1e-3) / 1e9
        out["kernels"][n] = {"launches": len(v), "avg_us": round(avg * 1e3, 2),
                             "bytes": lb_bytes.get(n, 0), "achieved_gbs": round(bw, 1),
                             "frac_hbm": round(bw / pk["hbm_gbs"], 4)}
    out["loss"] = float(lb_stats[0])
    out["max_over_uniform"] = float(lb_stats[1])
    del lb_dl
    return out


def fp8_block(cfg, layer, dev, flush_l2, steps, pk):
    """The MXFP8 grouped-expert forward beside the bf16 one on the headline
    workload's dispatched rows (the layer's own xp and offsets after its last
    forward): per-launch events on the launching stream, L2 flushed before each
    forward. The FP8 tensor peak is the measured bf16 one times the nominal
    FP8 / bf16 ratio of 2."""
    import torch
    from grouped_gemm_moe_gb300 import binding as B
    w = layer.w
    TK, d, I, E = cfg.T * cfg.K, cfg.d, cfg.I, cfg.E
    wgu = B.moe_mxfp8_quantize_weights(w["w_gate"], w["w_up"])
    wdq = B.moe_mxfp8_quantize_weights(w["w_down"])
    ws = B.new_workspace(B.workspace_size(B.MOE_OP_GROUPED_FFN_FP8, TK, E, 1, 1, d, I), dev)
    out8 = (torch.empty(TK, d, dtype=torch.bfloat16, device=dev),
            torch.empty(TK, I, dtype=torch.bfloat16, device=dev),
            torch.empty(TK, 2 * I, dtype=torch.bfloat16, device=dev))
    out16 = (layer.y, layer.h, layer.gu)

    def both():
        flush_l2()
        B.moe_grouped_ffn(layer.xp, layer.offsets, w["w_gate"], w["w_up"], w["w_down"],
                          ws=layer.ws_ffn, out=out16)
        flush_l2()
        B.moe_grouped_ffn_fp8(layer.xp, layer.offsets, wgu, wdq, ws=ws, out=out8)
        flush_l2()
        B.moe_mxfp8_quantize_weights(w["w_gate"], w["w_up"], out=wgu)
        B.moe_mxfp8_quantize_weights(w["w_down"], out=wdq)

    for _ in range(3):
        both()
    torch.cuda.synchronize()
    B.moe_profile_start(16 * steps + 16)
    for _ in range(steps):
        both()
    torch.cuda.synchronize()
    rec = {}
    for n, ms in B.moe_profile_stop():
        rec.setdefault(n, []).append(ms)
    avg = {n: statistics.mean(v) for n, v in rec.items()}
    per_fwd = {n: sum(v) / steps for n, v in rec.items()}   # all of a kernel's launches per forward
    fl = {"gemm_gate_up": 4 * TK * d * I, "gemm_down": 2 * TK * d * I,
          "gemm_gate_up_fp8": 4 * TK * d * I, "gemm_down_fp8": 2 * TK * d * I}
    peak8 = 2 * pk["bf16_tflops"]
    kern = {}
    for n, ms in avg.items():
        k = {"launches": len(rec[n]), "avg_us": round(ms * 1e3, 1)}
        if n in fl:
            tf = fl[n] / (ms * 1e-3) / 1e12
            k["tflops"] = round(tf, 1)
            k["frac"] = round(tf / (peak8 if n.endswith("_fp8") else pk["bf16_tflops"]), 4)
        kern[n] = k
    f16 = avg.get("gemm_gate_up", 0) + avg.get("gemm_down", 0)
    # the call quantizes xp (H's E4M3 copy comes from the gate/up epilogue)
    f8 = (per_fwd.get("gemm_gate_up_fp8", 0) + per_fwd.get("gemm_down_fp8", 0) +
          per_fwd.get("mxfp8_quantize_rows", 0))
    out = {"workload": f"{cfg.name} experts' forward on its dispatched rows (M={TK}, d={d}, I={I}, E={E})",
           "format": "MXFP8: E4M3 elements, one UE8M0 scale per 32 K",
           "peaks_tflops": {"bf16_measured_burst": pk["bf16_tflops"], "fp8_derived_burst": peak8},
           "bf16_forward_ms": round(f16, 4),
           "fp8_forward_ms": round(f8, 4),
           "fp8_forward_ms_note": "both GEMMs plus the quantization of xp inside the call (H is "
                                  "quantized in the gate/up epilogue)",
           "speedup": round(f16 / f8, 3) if f8 else None,
           "weight_quantization_ms": round(2 * avg.get("mxfp8_quantize_weights", 0), 4),
           "kernels": kern}
    del out8, ws, wgu, wdq
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    if args.profile_case:
        profile_case(args.profile_case)
        return
    world, rank, local = dist_env()
    from grouped_gemm_moe_gb300 import workloads as W
    cfg = W.CONFIGS[args.config or W.BENCH_CONFIG]
    if args.impl == "reference":
        run_reference(args, cfg, world, rank)
        return
    import torch
    import torch.distributed as dist
    from grouped_gemm_moe_gb300 import binding as B
    from grouped_gemm_moe_gb300 import build as build_mod

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not os.path.exists(B.LIB_PATH):
        build_mod.build()
    B.load()
    if not cfg.backward:
        raise SystemExit("the benchmark workload must include the backward pass")

    inp = W.make_inputs(cfg, seed=cfg.seed + rank)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one: the step starts with
        # L2 holding none of its data and no dirty lines left to write back
        flush.zero_()
        flush_rd.sum()

    run = Runner(cfg, inp, dev, flush_l2, world)
    layer, stream = run.layer, run.stream

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id) if rank == 0 else None

    run.warm(args.warmup, min_seconds=1.5)
    step_ms = run.timed(args.steps)
    # A/A: the same K steps again, back to back, for the run-to-run noise floor
    step_ms_aa = run.timed(args.steps)
    # per-kernel durations: the same K steps again, each library launch bracketed by
    # events on its stream (kept out of the passes above, where events between launches
    # would hold back each kernel's early launch behind its predecessor)
    records = run.per_launch(args.steps)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    value = aggregate_value(ms, cfg.T, world)

    # per-kernel table and the dominant kernel's roofline
    pk = peaks()
    per, kernels, flops_step, bytes_step, layer_roof_ms, sum_roof_ms = kernel_table(
        cfg, records, args.steps, pk)
    dom = max(per, key=lambda k: per[k]["total_ms"])
    dfl, dnb = kernel_work(per[dom]["name"], cfg, per[dom]["shared"])
    davg = per[dom]["total_ms"] / per[dom]["launches"]
    rf = roofline_of(dfl, dnb, davg, pk)
    roof = {"bound": rf["bound"], "kernel": dom, "achieved": rf["achieved"], "peak": rf["peak"],
            "unit": rf["unit"], "frac": rf["frac"],
            "peak_source": pk["source"] + (" bf16 sustained" if rf["bound"] == "tensor"
                                           else " HBM copy (read+write)"),
            "traffic": measured_traffic(dom, cfg.name),
            "frac_of_nominal": rf["achieved"] / (NOMINAL_TFLOPS if rf["bound"] == "tensor"
                                                 else NOMINAL_GBS),
            "work_per_launch": {"flop": dfl, "bytes": dnb},
            "avg_launch_ms": davg}

    load_balance = load_balance_block(cfg, layer, run.logits, dev, flush_l2, args.steps, pk)
    fp8 = None if args.no_fp8 else fp8_block(cfg, layer, dev, flush_l2, min(args.steps, 10), pk)

    # end to end through the layer API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.pin_memory()  # noqa: E731
        lh, xh, dh = pin(inp["logits"]), pin(inp["x"]), pin(inp["dout"])
        out_h = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory()
        dx_h = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory()
        layer.run_from_host([(lh, xh, dh, out_h, dx_h)] * 2)
        torch.cuda.synchronize()
        run.barrier()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        h2d, d2h = layer.run_from_host([(lh, xh, dh, out_h, dx_h)] * args.steps)
        e.record(stream)
        torch.cuda.synchronize()
        run.barrier()
        ems = max_over_ranks(s.elapsed_time(e) / args.steps, world, dev)
        e2e = {"value": aggregate_value(ems, cfg.T, world), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems,
               "l2": (f"not flushed between steps: the steps run back to back, each step's "
                      f"uploads and downloads overlapping its neighbours' compute; one step "
                      f"moves {bytes_step / 1e9:.1f} GB of algorithmic traffic, "
                      f"{bytes_step / (129 << 20):.0f}x the 129 MB L2")}
        del lh, xh, dh, out_h, dx_h

    # the other forward + backward workloads (shorter runs), after the headline
    del run, layer
    torch.cuda.empty_cache()
    configs = {}
    if not args.no_side_configs and args.config is None:
        for name in W.SIDE_CONFIGS:
            configs[name] = side_config(name, args, dev, flush_l2, world, rank, pk)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, args.cpu_sample_tokens, inp)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) logits/activations, N(0,0.02) weights)",
            "config": {"workload": f"{cfg.name}: {W.describe(cfg)}, fwd+bwd",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "flushed before every timed step (256 MiB written, then 256 MiB read; outside its events)",
                       "step_tflop": flops_step / 1e12,
                       "step_gbytes_algorithmic": bytes_step / 1e9,
                       "layer_tflops_achieved": flops_step / (ms / 1e3) / 1e12,
                       "layer_roofline_ms": layer_roof_ms,
                       "layer_frac_of_roofline": layer_roof_ms / ms,
                       "sum_of_kernel_rooflines_ms": sum_roof_ms},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": len(records), "clocks": clocks,
            "step_ms_min_max": [min(step_ms), max(step_ms)],
            "step_ms_median": statistics.median(step_ms),
            "aa": {"ms_per_step": statistics.mean(step_ms_aa),
                   "rel_diff": abs(statistics.mean(step_ms_aa) - statistics.mean(step_ms))
                   / statistics.mean(step_ms)},
            "kernels": kernels, "configs": configs, "load_balance": load_balance, "fp8": fp8,
            "device": torch.cuda.get_device_name(dev),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
