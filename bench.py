#!/usr/bin/env python3
"""Benchmark of the routed-expert NVFP4 MoE block on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config decode1|decode2..decode64|prefill4096|skew16384|tiny]

A step is one forward of the whole MoE block (router, top-k, grouping, routed
gate/up + SiLU*up, shared gate/up, routed and shared down, weighted combine and
shared add) over one batch of synthetic tokens.  The default workload is
single-token decode (M=1, H=2048, E=128, top_k=8, I=768, shared I=768).

Weights of `layers` independent synthetic layers stay resident in HBM and the
steps rotate through them (step i runs layer i mod layers), so every step
streams its experts from HBM rather than L2 (the rotation's working set is far
larger than the 129 MB L2).  The timed region replays CUDA graphs of the steps.

The default command reports the whole metric in one JSON line: the headline
(single-token decode, tokens/s with its HBM roofline and the end-to-end figure)
and, under "records", the decode batch sweep (M = 2 .. 64, HBM roofline), the
M = 4096 prefill and the Zipf-skewed M = 16384 workload (tensor roofline, total
and routed-only TFLOP/s, per-expert load histogram), each timed the same way
with its own SM-clock record.  cpu_baseline times the oracle on all host cores
and on one thread, with the CPU model.

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica on
its own tokens (the block has no cross-token exchange), so scaling is weak and
no collective touches the data path.  Rank 0 prints one JSON line.

--impl reference times the CPU oracle (the plain C implementation the parity
tests use) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from nvfp4_w4a16_mixture_gb300 import synth  # noqa: E402

METRIC = "MoE-layer tokens/s & weight HBM GB/s (decode M<=64); TFLOP/s at M=4096"
DECODE_MAX_TOKENS = 64


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=0, help="0 = 10000 (decode) / 40 (large batches)")
    p.add_argument("--warmup", type=int, default=0, help="0 = 200 (decode) / 5 (large batches)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default="decode1", choices=sorted(synth.CONFIGS))
    p.add_argument("--layers", type=int, default=0, help="weight sets rotated (0 = auto)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-sweep", dest="sweep", action="store_false",
                   help="time the headline configuration only (the default also times the decode "
                        "sweep, prefill4096 and skew16384 as records of the same line)")
    p.add_argument("--profile", action="store_true",
                   help="run --warmup then --steps plain (eager) forwards and exit, for ncu launch lists")
    return p.parse_args()


def workload_name(cfg: str) -> str:
    M, H, E, k, I, SI = synth.CONFIGS[cfg]
    extra = ", Zipf(1.2)-skewed router" if cfg.startswith("skew") else ""
    return f"{cfg}: M={M} H={H} E={E} top_k={k} I={I} SI={SI} (NVFP4 experts, BF16 shared{extra})"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(vals, device="cpu"):
    """Element-wise maximum of per-rank timings over all ranks (a no-op on
    one process): the job is as slow as its slowest replica."""
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist = torch.distributed
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_tokens_per_s(tokens_per_rank_step: int, steps: int, world: int, ms_total_max: float) -> float:
    """Whole-job throughput: every rank runs its own replica on its own
    tokens (weak scaling), so all ranks' tokens count over the slowest rank's
    time."""
    return tokens_per_rank_step * steps * world / (ms_total_max / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples (the JSON line carries their summary); FLINT_BENCH_CLOCKS_DIR
        # keeps them somewhere else than the temporary directory
        out_dir = os.environ.get("FLINT_BENCH_CLOCKS_DIR", tempfile.gettempdir())
        self.path = os.path.join(out_dir, f"flint_clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            return summarize_clocks(parse_clock_lines(f), t0, t1)


def parse_clock_lines(lines):
    """Rows (unix time, SM MHz, max SM MHz, [reason fields]) of nvidia-smi's
    csv,noheader,nounits output for ClockSampler.FIELDS; other lines skipped."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
            rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[5:]))
        except Exception:
            continue
    return rows


def summarize_clocks(rows, t0: float, t1: float):
    """The JSON line's clocks object: median SM clock and the throttle reasons
    seen in [t0, t1] (the nearest three samples if none fell inside)."""
    if not rows:
        return None
    inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
    use = inside or sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
    reasons = set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in use:
        for name, v in zip(names, r[3][1:5]):
            if v.strip().lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
            "reasons": sorted(reasons), "samples": len(use),
            "samples_inside_timed_region": len(inside)}


# --------------------------------------------------------------- workload
def make_layers(cfg: str, n_layers: int, device: str, seed: int):
    M, H, E, k, I, SI = synth.CONFIGS[cfg]
    scale = synth.zipf_router_scale(E) if cfg.startswith("skew") else None
    layers, xs = [], []
    for li in range(n_layers):
        gen = torch.Generator(device=device).manual_seed(seed * 1000 + li)
        xs.append(synth.make_x(M, H, gen, device))
        layers.append(synth.make_layer(H, E, I, SI, gen, device, router_row_scale=scale))
    return xs, layers


LAUNCHES_PER_PATH = {1: 1, 2: 3, 3: 3, 4: 9}  # FLINT_PATH_* -> kernels per forward


def launches_per_step(M: int, path: int = 0) -> int:
    """Kernels of one forward: the single launch (1); decode router, gate/up,
    down+combine (3); grouped path router, group count/scan/scatter, plan,
    gather, GEMM1, GEMM2, combine (9).  Without a path: the default for M."""
    if path:
        return LAUNCHES_PER_PATH[path]
    return 3 if M <= DECODE_MAX_TOKENS else 9


def traffic_record(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (hash match), else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    from nvfp4_w4a16_mixture_gb300 import build as b
    h = hashlib.sha256()
    for p in sorted(b.sources()):
        h.update(open(p, "rb").read())
    entry = rec.get(kernel)
    if entry and entry.get("csrc_sha256") == h.hexdigest():
        return entry.get("dram_bytes_per_step")
    return None


# ----------------------------------------------------------------- profile
def run_profile(args, local):
    """Eager forwards only (no graphs, no timing): `warmup` steps, then `steps`
    steps, each a fixed sequence of launches_per_step(M) kernels, so an ncu
    launch list can skip the first and capture the rest."""
    import nvfp4_w4a16_mixture_gb300 as fm

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    M, H, E, k, I, SI = synth.CONFIGS[args.config]
    n_layers = args.layers or (16 if M <= DECODE_MAX_TOKENS else 2)
    fm.load()
    xs, layers = make_layers(args.config, n_layers, dev, seed=1)
    ws = fm.alloc_workspace(M, H, E, k, I, SI, dev)
    outs = [torch.empty_like(x) for x in xs]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            li = i % n_layers
            fm.forward_layer(xs[li], layers[li], k, workspace=ws, out=outs[li], stream=stream)
    stream.synchronize()
    assert fm.flint_moe_status(ws, stream) == fm.FLINT_OK
    print(f"profile: {args.config}, {args.warmup} + {args.steps} steps of "
          f"{launches_per_step(M)} launches, {n_layers} layers rotated", file=sys.stderr)


# -------------------------------------------------------------------- ours
SWEEP = ("decode2", "decode4", "decode8", "decode16", "decode32", "decode64", "prefill4096",
         "skew16384")


class Workload:
    """Resident weights and inputs of one configuration (several layers
    rotated) and the graphs of its steps.  kind: "forward" (the block),
    "add_norm" (the block with its add-RMSNorm prologue), "bf16" (BF16 routed
    experts, shared output given), "nvfp4_shared" (NVFP4 shared expert)."""

    def __init__(self, cfg, dev, rank, n_layers, layers=None, kind="forward"):
        import nvfp4_w4a16_mixture_gb300 as fm
        self.fm = fm
        self.cfg = cfg
        self.kind = kind
        self.M, self.H, self.E, self.k, self.I, self.SI = synth.CONFIGS[cfg]
        self.n_layers = n_layers
        if layers is None:
            _, layers = make_layers(cfg, n_layers, dev, seed=1 + rank)
        self.layers = layers
        self.xs = [synth.make_x(self.M, self.H, torch.Generator(device=dev).manual_seed(9000 + 97 * rank + li), dev)
                   for li in range(n_layers)]
        self.ws = fm.alloc_workspace(self.M, self.H, self.E, self.k, self.I, self.SI, dev)
        self.outs = [torch.empty_like(x) for x in self.xs]
        self.ids = [torch.empty(self.M, self.k, dtype=torch.int32, device=dev) for _ in self.xs]
        self.stream = torch.cuda.Stream(device=dev)
        self.path = fm.flint_moe_plan(self.M, self.H, self.E, self.k, self.I,
                                      0 if kind in ("bf16", "nvfp4_shared") else self.SI)
        M, H, E, I, SI = self.M, self.H, self.E, self.I, self.SI
        g = torch.Generator(device=dev).manual_seed(4242 + rank)
        if kind == "add_norm":
            self.res = [synth.make_x(M, H, g, dev) for _ in range(n_layers)]
            self.res_out = [torch.empty_like(r) for r in self.res]
            self.lnw = (1 + 0.1 * torch.randn(H, generator=g, device=dev)).to(torch.bfloat16)
        elif kind == "bf16":
            # BF16 routed experts of the same shapes (one set per rotated layer)
            self.w13 = [(torch.randn(E, 2 * I, H, generator=g, device=dev) * 0.02).to(torch.bfloat16)
                        for _ in range(n_layers)]
            self.w2 = [(torch.randn(E, H, I, generator=g, device=dev) * 0.02).to(torch.bfloat16)
                       for _ in range(n_layers)]
            self.shared = [(torch.randn(M, H, generator=g, device=dev) * 0.05).to(torch.bfloat16)
                           for _ in range(n_layers)]
            self.ws = fm.alloc_workspace(M, H, E, self.k, I, 0, dev)
        elif kind == "nvfp4_shared":
            self.sh = []
            for _ in range(n_layers):
                gc, gf, gg = synth.quantize_nvfp4(torch.randn(2 * SI, H, generator=g, device=dev) * 0.02)
                dc, df, dg = synth.quantize_nvfp4(torch.randn(H, SI, generator=g, device=dev) * 0.02)
                self.sh.append((gc, gf, gg.reshape(1).contiguous(), dc, df, dg.reshape(1).contiguous()))

    def bytes_per_step(self, unique_experts: float) -> float:
        """Algorithmic weight bytes of one step."""
        M, H, E, I, SI = self.M, self.H, self.E, self.I, self.SI
        if self.kind == "bf16":
            return unique_experts * 3 * I * H * 2 + E * H * 2 + M * H * 2
        wb = synth.weight_bytes(H, E, I, SI, int(round(unique_experts)))
        if self.kind == "nvfp4_shared":
            return wb["total"] - wb["shared"] + 3 * SI * H // 2 + 3 * SI * H // 16
        return wb["total"]

    def step(self, i, s):
        li = i % self.n_layers
        fm, L = self.fm, self.layers[li] if self.layers else None
        if self.kind == "forward":
            fm.forward_layer(self.xs[li], L, self.k, workspace=self.ws, out=self.outs[li], ids_out=self.ids[li],
                             stream=s)
        elif self.kind == "add_norm":
            fm.forward_add_norm_layer(self.xs[li], self.res[li], self.lnw, 1e-6, L, self.k, workspace=self.ws,
                                      out=self.outs[li], residual_out=self.res_out[li], ids_out=self.ids[li],
                                      stream=s)
        elif self.kind == "bf16":
            fm.flint_moe_forward_bf16(self.xs[li], L.router_w, self.w13[li], self.w2[li], self.k, self.outs[li],
                                      self.ws, shared_out=self.shared[li], ids_out=self.ids[li], stream=s)
        else:
            gc, gf, gg, dc, df, dg = self.sh[li]
            fm.flint_moe_forward_nvfp4_shared(self.xs[li], L.router_w, L.w13, L.w13_sf, L.w13_gs, L.w2, L.w2_sf,
                                              L.w2_gs, gc, gf, gg, dc, df, dg, self.k, self.outs[li], self.ws,
                                              ids_out=self.ids[li], stream=s)


def time_workload(w: Workload, steps: int, warmup: int, world: int, local: int):
    """Device time of `steps` steps replayed from CUDA graphs (max over
    ranks), with the SM clocks sampled during the timed region."""
    fm, stream = w.fm, w.stream
    with torch.cuda.stream(stream):
        for i in range(max(warmup, w.n_layers)):
            w.step(i, stream)
    stream.synchronize()
    assert fm.flint_moe_status(w.ws, stream) == fm.FLINT_OK
    full, rem = divmod(steps, w.n_layers)
    g_full = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full, stream=stream):
        for i in range(w.n_layers):
            w.step(i, stream)
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            for i in range(rem):
                w.step(i, stream)
    with torch.cuda.stream(stream):
        g_full.replay()
    stream.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    stream.synchronize()
    t1 = time.time()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_total = ev0.elapsed_time(ev1)
    clk = clocks.stop(t0, t1)
    assert fm.flint_moe_status(w.ws, stream) == fm.FLINT_OK
    del g_full, g_rem
    (ms_total,) = max_over_ranks([ms_total], device=f"cuda:{local}")
    return ms_total, clk


class QkvWorkload:
    """The fused decode qkv (flint_qkv_fused) of one token: H = 2048, 32 q
    heads, 4 kv heads of 128 (N = 5120 rows), NVFP4 weights, a residual,
    RoPE from a 4096-position table and a paged cache of 256 blocks of 16
    slots; `n_layers` weight sets rotated (5.9 MB each, more than L2 in all)."""

    def __init__(self, dev, rank, n_layers=32, M=1, H=2048, nq=32, nkv=4):
        import nvfp4_w4a16_mixture_gb300 as fm
        self.fm, self.M, self.H, self.nq, self.nkv, self.n_layers = fm, M, H, nq, nkv, n_layers
        N = (nq + 2 * nkv) * 128
        g = torch.Generator(device=dev).manual_seed(777 + rank)
        self.x = [synth.make_x(M, H, g, dev) for _ in range(n_layers)]
        self.res = [synth.make_x(M, H, g, dev) for _ in range(n_layers)]
        self.nw = (1 + 0.1 * torch.randn(H, generator=g, device=dev)).to(torch.bfloat16)
        self.w = []
        for _ in range(n_layers):
            c, sf, gs = synth.quantize_nvfp4(torch.randn(N, H, generator=g, device=dev) * 0.03)
            self.w.append((c, sf, gs.reshape(1).contiguous()))
        self.qn = (1 + 0.1 * torch.randn(128, generator=g, device=dev)).to(torch.bfloat16)
        self.kn = (1 + 0.1 * torch.randn(128, generator=g, device=dev)).to(torch.bfloat16)
        ang = torch.arange(4096, dtype=torch.float64, device=dev)[:, None] * \
            (1e6 ** (-torch.arange(64, device=dev) / 64.0))[None, :]
        self.cs = torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).float().contiguous()
        self.pos = torch.randint(0, 4096, (M,), generator=g, device=dev, dtype=torch.int64)
        self.kc = torch.zeros(256, 16, nkv, 128, dtype=torch.bfloat16, device=dev)
        self.vc = torch.zeros_like(self.kc)
        self.slots = torch.randint(0, 256 * 16, (M,), generator=g, device=dev, dtype=torch.int64)
        self.q = torch.empty(M, nq * 128, dtype=torch.bfloat16, device=dev)
        self.r_out = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
        self.ws = torch.zeros(fm.flint_qkv_workspace_bytes(M, H, nq, nkv), dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.bytes = N * H // 2 + N * H // 16 + 4

    def step(self, i, s):
        li = i % self.n_layers
        c, sf, gs = self.w[li]
        self.fm.flint_qkv_fused(self.x[li], self.res[li], self.nw, 1e-6, c, sf, gs, self.qn, self.kn, 1e-6,
                                self.cs, self.pos, self.kc, self.vc, self.slots, self.nq, self.nkv,
                                q_out=self.q, residual_out=self.r_out, workspace=self.ws, stream=s)


def expert_load(w: Workload) -> dict:
    """Pairs per expert over the resident batches (one step per layer)."""
    cnt = torch.zeros(w.E, dtype=torch.int64)
    for t in w.ids:
        cnt += torch.bincount(t.reshape(-1).cpu().long(), minlength=w.E)
    n = int(cnt.sum())
    top = torch.sort(cnt, descending=True).values
    return {"pairs": n, "steps": len(w.ids), "per_expert": cnt.tolist(),
            "max_over_mean": round(float(top[0]) * w.E / max(n, 1), 3),
            "top8_share": round(float(top[:8].sum()) / max(n, 1), 4),
            "experts_unused": int((cnt == 0).sum())}


def record_of(w: Workload, ms_total: float, steps: int, world: int, clk, peaks) -> dict:
    """One configuration's timing with its roofline."""
    M, H, E, k, I, SI = w.M, w.H, w.E, w.k, w.I, w.SI
    ms_step = ms_total / steps
    step_s = ms_step / 1e3
    uniq = [int(torch.unique(t).numel()) for t in w.ids]
    wb = [synth.weight_bytes(H, E, I, SI, u) for u in uniq]
    mean_bytes = sum(w.bytes_per_step(u) for u in uniq) / len(uniq)
    mean_expert_bytes = sum(x["experts"] for x in wb) / len(wb)
    if w.kind == "bf16":
        mean_expert_bytes = sum(u * 3 * I * H * 2 for u in uniq) / len(uniq)
    flops = synth.flops_of(M, H, E, k, I, SI)
    rec = {"workload": workload_name(w.cfg), "tokens_per_step": M, "steps": steps,
           "ms_per_step": round(ms_step, 6),
           "tokens_per_s": round(job_tokens_per_s(M, steps, world, ms_total), 2),
           "path": ({"forward": "", "add_norm": "add-RMSNorm kernel + ", "bf16": "",
                     "nvfp4_shared": ""}[w.kind] +
                    ({1: "single launch", 2: "decode (3 kernels)", 3: "decode fallback (3 kernels)",
                      4: "grouped (9 kernels)"}.get(w.path, str(w.path)) if w.kind != "bf16" else
                     "BF16 experts (router, gate/up, down, combine)") +
                    (" + NVFP4 shared expert (gate/up, down, add)" if w.kind == "nvfp4_shared" else "")),
           "gpu_launches_per_step": (4 if w.kind == "bf16" else launches_per_step(M, w.path) +
                                     {"forward": 0, "add_norm": 1, "nvfp4_shared": 3}[w.kind]),
           "weight_gbs": round(mean_bytes / step_s / 1e9, 1),
           "expert_weight_gbs": round(mean_expert_bytes / step_s / 1e9, 1),
           "tflops": round(flops["total"] / step_s / 1e12, 3),
           "clocks": clk, "traffic": traffic_record(w.cfg)}
    if M <= DECODE_MAX_TOKENS:
        achieved = mean_bytes / step_s / 1e9
        rec["roofline"] = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                           "traffic": rec["traffic"], "algorithmic_bytes_per_step": int(mean_bytes),
                           "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)"}
    else:
        peak = peaks["bf16_tflops"]
        total = flops["total"] / step_s / 1e12
        routed = flops["routed"] / step_s / 1e12
        rec["roofline"] = {"bound": "tensor", "achieved": round(total, 1), "peak": peak, "unit": "TFLOP/s",
                           "frac": round(total / peak, 4), "routed_only_tflops": round(routed, 1),
                           "routed_only_frac": round(routed / peak, 4), "traffic": rec["traffic"],
                           "algorithmic_flops_per_step": flops["total"],
                           "routed_flops_per_step": flops["routed"],
                           "peak_source": peaks["source"] + " (bf16_tflops burst)"}
    return rec


def e2e_of(w: Workload, steps: int, local: int, world: int) -> dict:
    """End to end through the C ABI from pinned host buffers: every step
    copies its tokens in and its outputs back inside the timed region."""
    stream = w.stream
    x_host = [x.cpu().pin_memory() for x in w.xs]
    out_host = [torch.empty(w.M, w.H, dtype=torch.bfloat16).pin_memory() for _ in w.xs]

    def run(n):
        for i in range(n):
            li = i % w.n_layers
            w.xs[li].copy_(x_host[li], non_blocking=True)
            w.step(i, stream)
            out_host[li].copy_(w.outs[li], non_blocking=True)

    with torch.cuda.stream(stream):
        run(min(50, steps))
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run(steps)
        e1.record(stream)
    stream.synchronize()
    (ms,) = max_over_ranks([e0.elapsed_time(e1) / steps], device=f"cuda:{local}")
    return {"value": round(w.M * world / (ms / 1e3), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": w.M * w.H * 2, "d2h_bytes_per_step": w.M * w.H * 2,
            "ms_per_step": round(ms, 6), "steps": steps}


def kernel_spans(w: Workload, steps: int = 40) -> dict:
    """Per-kernel spans of `steps` eager steps (each timed alone: the buffer
    is zeroed, the step runs, its spans are read): mean ns per kernel from its
    first CTA's start to its last warp's exit, the step's span, and each
    kernel's share of the sum of spans."""
    fm = w.fm
    buf = torch.zeros(fm._lib.SPAN_KERNELS * fm._lib.SPAN_CTAS * 2, dtype=torch.int64, device=w.ws.device)
    acc, step_ns = {}, []
    fm.flint_moe_record_spans(buf)
    try:
        for i in range(steps):
            buf.zero_()
            with torch.cuda.stream(w.stream):
                w.step(i, w.stream)
            w.stream.synchronize()
            sp = fm.spans_of(buf)
            if not sp:
                continue
            t0 = min(v[0] for v in sp.values())
            step_ns.append(max(v[1] for v in sp.values()) - t0)
            for name, (a, b) in sp.items():
                acc.setdefault(name, []).append((b - a, a - t0))
    finally:
        fm.flint_moe_record_spans(None)
    tot = sum(sum(d for d, _ in v) / len(v) for v in acc.values()) or 1
    out = {name: {"us": round(sum(d for d, _ in v) / len(v) / 1e3, 3),
                  "start_us": round(sum(o for _, o in v) / len(v) / 1e3, 3),
                  "share": round(sum(d for d, _ in v) / len(v) / tot, 4)} for name, v in acc.items()}
    return {"steps": len(step_ns), "step_span_us": round(sum(step_ns) / max(len(step_ns), 1) / 1e3, 3),
            "kernels": out,
            "how": "globaltimer at each CTA's start and each warp's exit (flint_moe_record_spans), "
                   "eager steps each timed alone"}


def dominant_roofline(w: Workload, spans: dict, peaks) -> dict | None:
    """The dominant kernel against its own roofline, from its measured span:
    the decode gate/up kernel's weight bytes (routed w13 + scales of the
    step's experts, shared gate/up) over its span; the grouped GEMM1's flops
    over its span."""
    ks = spans.get("kernels", {})
    if not ks:
        return None
    name = max(ks, key=lambda n: ks[n]["us"])
    M, H, E, k, I, SI = w.M, w.H, w.E, w.k, w.I, w.SI
    us = ks[name]["us"]
    if name in ("gate_up", "single_launch", "down") and M <= DECODE_MAX_TOKENS:
        uniq = sum(int(torch.unique(t).numel()) for t in w.ids) / len(w.ids)
        if name == "gate_up":
            b = uniq * (2 * I * H // 2 + 2 * I * H // 16) + 2 * SI * H * 2
        elif name == "down":
            b = uniq * (H * I // 2 + H * I // 16) + SI * H * 2
        else:
            b = synth.weight_bytes(H, E, I, SI, int(round(uniq)))["total"]
        ach = b / (us * 1e-6) / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4), "span_us": us,
                "algorithmic_bytes": int(b)}
    if name in ("gemm1", "gemm2"):
        f = 2 * M * k * (2 * I * H if name == "gemm1" else H * I) + 2 * M * (2 * SI * H if name == "gemm1" else SI * H)
        ach = f / (us * 1e-6) / 1e12
        return {"kernel": name, "bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4), "span_us": us,
                "algorithmic_flops": int(f)}
    return {"kernel": name, "span_us": us}


def run_ours(args, rank, world, local):
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    peaks = load_peaks()
    cfg = args.config
    M = synth.CONFIGS[cfg][0]
    n_layers = args.layers or (16 if M <= DECODE_MAX_TOKENS else 2)
    w = Workload(cfg, dev, rank, n_layers)
    K = args.steps
    ms_total, clk = time_workload(w, K, args.warmup, world, local)
    head = record_of(w, ms_total, K, world, clk, peaks)
    e2e = e2e_of(w, min(K, 2000), local, world)
    spans = kernel_spans(w)
    rl = head["roofline"]
    rl["dominant_kernel"] = dominant_roofline(w, spans, peaks)
    rl["kernel"] = ("whole step: " + head["path"] + " (the kernels of a step overlap through "
                    "programmatic dependent launch, so the step is timed whole)")
    res = {
        "metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; NVFP4-quantised N(0,0.02) experts, N(0,1) tokens)",
        "config": {"workload": head["workload"], "global_batch": M * world, "tokens_per_step": M,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "layers_rotated": n_layers,
                   "l2": f"weights of {n_layers} layers rotate "
                         f"({sum(l.expert_bytes() * w.E for l in w.layers) / 1e9:.1f} GB resident), "
                         "each step's working set streams from HBM"},
        "weight_gbs": head["weight_gbs"], "expert_weight_gbs": head["expert_weight_gbs"],
        "tflops": head["tflops"], "path": head["path"],
        "roofline": rl, "e2e": e2e,
        "gpu_launches": K * head["gpu_launches_per_step"],
        "clocks": clk,
        "kernel_spans": spans,
    }
    if args.sweep:
        # the rest of the metric: the decode batch sweep and the large-batch
        # workloads, each timed the same way (decode shapes share the
        # headline's resident layers)
        recs = {}
        for c in SWEEP:
            Mc = synth.CONFIGS[c][0]
            if Mc <= DECODE_MAX_TOKENS:
                wc = Workload(c, dev, rank, n_layers, layers=w.layers)
                steps_c, warm_c = 2000, 50
            else:
                wc = Workload(c, dev, rank, 2)
                steps_c, warm_c = (20, 3) if Mc <= 4096 else (10, 3)
            ms_c, clk_c = time_workload(wc, steps_c, warm_c, world, local)
            r = record_of(wc, ms_c, steps_c, world, clk_c, peaks)
            if c.startswith("skew") or c.startswith("prefill"):
                r["expert_load"] = expert_load(wc)
            r["kernel_spans"] = kernel_spans(wc, steps=10 if Mc > DECODE_MAX_TOKENS else 40)
            r["roofline"]["dominant_kernel"] = dominant_roofline(wc, r["kernel_spans"], peaks)
            r["gpu_launches"] = steps_c * r["gpu_launches_per_step"]
            recs[c] = r
            del wc
            torch.cuda.empty_cache()
        # the widened rows at the headline's shape: add-RMSNorm prologue, BF16
        # routed experts, NVFP4 shared expert
        wide = (("decode1_add_norm", "add_norm", n_layers,
                 "NVFP4 experts, BF16 shared, residual add + RMSNorm before the router"),
                ("decode1_bf16_experts", "bf16", 8, "BF16 routed experts, shared output given"),
                ("decode1_nvfp4_shared", "nvfp4_shared", n_layers, "NVFP4 experts, NVFP4 shared"))
        for c, kind, nl, what in (wide if synth.CONFIGS[cfg][1:] == synth.CONFIGS["decode1"][1:] else ()):
            nl = min(nl, len(w.layers))
            wc = Workload("decode1", dev, rank, nl, layers=w.layers[:nl], kind=kind)
            ms_c, clk_c = time_workload(wc, 2000, 50, world, local)
            r = record_of(wc, ms_c, 2000, world, clk_c, peaks)
            r["workload"] = f"{c}: M=1 H={wc.H} E={wc.E} top_k={wc.k} I={wc.I} SI={wc.SI} ({what})"
            r["traffic"] = None
            r["roofline"]["traffic"] = None
            r["gpu_launches"] = 2000 * r["gpu_launches_per_step"]
            recs[c] = r
            del wc
            torch.cuda.empty_cache()
        # the fused decode qkv of one token (the attention-side widened row)
        wq = QkvWorkload(dev, rank)
        ms_q, clk_q = time_workload(wq, 2000, 50, world, local)
        step_s = ms_q / 2000 / 1e3
        ach = wq.bytes / step_s / 1e9
        recs["qkv_decode1"] = {
            "workload": "qkv_decode1: M=1 H=2048 32 q heads, 4 kv heads of 128 (N=5120), NVFP4 weights, "
                        "residual add-RMSNorm, q/k RMSNorm, NeoX RoPE, paged KV write",
            "tokens_per_step": 1, "steps": 2000, "ms_per_step": round(ms_q / 2000, 6),
            "tokens_per_s": round(job_tokens_per_s(1, 2000, world, ms_q), 2),
            "path": "input RMSNorm, qkv GEMV, heads (3 kernels)", "gpu_launches_per_step": 3,
            "gpu_launches": 3 * 2000, "weight_gbs": round(ach, 1), "clocks": clk_q, "traffic": None,
            "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": None,
                         "algorithmic_bytes_per_step": wq.bytes,
                         "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)"}}
        del wq
        torch.cuda.empty_cache()
        res["records"] = recs
    return res


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    architecture)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                v = line.split(":", 1)[1].strip()
                if v and not v.isdigit():
                    return v
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def cpu_baseline(cfg: str, n_tokens: int = 384, n_tokens_1t: int = 32, seed: int = 5):
    """The oracle on a bounded sample of the configuration's layer shape (one
    layer; its per-token work does not depend on M): n_tokens tokens on all
    host cores (OpenMP over tokens), and n_tokens_1t tokens on one thread."""
    import oracle
    M, H, E, k, I, SI = synth.CONFIGS[cfg]
    scale = synth.zipf_router_scale(E) if cfg.startswith("skew") else None
    gen = torch.Generator().manual_seed(seed)
    x = synth.make_x(n_tokens, H, gen)
    layer = synth.make_layer(H, E, I, SI, gen, router_row_scale=scale)
    oracle.build()
    oracle.forward(x[:1], layer, k)  # warm
    cores = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.forward(x, layer, k, nthreads=cores)
    dt = time.perf_counter() - t0
    t1 = time.perf_counter()
    oracle.forward(x[:n_tokens_1t], layer, k, nthreads=1)
    dt1 = time.perf_counter() - t1
    return {"value": round(n_tokens / dt, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{n_tokens} tokens of one {cfg} layer, {dt:.1f} s wall on {cores} threads",
            "one_thread": {"value": round(n_tokens_1t / dt1, 3), "unit": "tokens/s", "cores": 1,
                           "sample": f"{n_tokens_1t} tokens of the same layer, {dt1:.1f} s on 1 thread"}}


def run_reference(args):
    """--impl reference: the CPU oracle, timed over K steps of the workload."""
    import oracle
    cfg = args.config
    M, H, E, k, I, SI = synth.CONFIGS[cfg]
    scale = synth.zipf_router_scale(E) if cfg.startswith("skew") else None
    oracle.build()
    gen = torch.Generator().manual_seed(11)
    layer = synth.make_layer(H, E, I, SI, gen, router_row_scale=scale)
    # bounded sample: a decode step is its M tokens; a large-batch step is
    # sampled down to 32 of its tokens (the per-token work does not depend on
    # M) and throughput counts the tokens computed.  The token total is capped
    # so that the run stays within a few minutes.
    K = args.steps
    per_step = M if M <= DECODE_MAX_TOKENS else 32
    per_step_eff = max(1, min(per_step, 12000 // max(K, 1)))
    K_eff = K
    W = min(args.warmup, 8)
    x = synth.make_x(per_step_eff * (K_eff + W), H, gen)
    if W:
        oracle.forward(x[: per_step_eff * W], layer, k)
    t0 = time.perf_counter()
    oracle.forward(x[per_step_eff * W:], layer, k)
    dt = time.perf_counter() - t0
    tokens_per_s = per_step_eff * K_eff / dt
    cores = oracle.max_threads()
    ms_step = dt / K_eff * 1e3 * (M / per_step_eff)
    value = round(tokens_per_s, 3)
    sample = (f"{K_eff} steps x {per_step_eff} tokens of one {cfg} layer on {cores} threads "
              f"(OpenMP over tokens), {dt:.1f} s")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": K_eff, "warmup": W, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name(cfg), "global_batch": M},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    M = synth.CONFIGS[args.config][0]
    if args.steps <= 0:
        args.steps = 10000 if M <= DECODE_MAX_TOKENS else 40
    if args.warmup <= 0:
        args.warmup = 200 if M <= DECODE_MAX_TOKENS else 5
    rank, world, local = dist_env()
    if args.profile:
        run_profile(args, local)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    if args.config != "decode1":
        args.sweep = False  # the records belong to the headline line
    res = run_ours(args, rank, world, local)
    if world > 1:
        torch.distributed.barrier()
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:  # the host baseline is an N = 1 figure
            res["cpu_baseline"] = cpu_baseline(args.config)
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
