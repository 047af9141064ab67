#!/usr/bin/env python3
"""Benchmark of the MoE expert-layer forward pass on B300.

One step = the whole hot path on one batch of seeded synthetic input already resident in
HBM: route -> permute -> grouped GEMM1 + scaled SwiGLU -> grouped GEMM2 -> combine, each a
call through the C ABI (libmoe.so), with CUDA events between the calls so that every
kernel's duration is measured live inside the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  ``value`` = tokens/s of the whole job (all ranks).  Under
torchrun (N > 1) every rank runs an independent replica on its own token batch (the layer
shards by tokens with no exchange), time = max over ranks.

``--impl reference`` times the CPU oracle (fp64, OpenMP on the host cores) on a bounded
sample of tokens of the same workload instead; it is a deliberately slow baseline.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import WORKLOADS, gen_logits, gen_weights, gen_x  # noqa: E402

METRIC = "MoE-layer tokens/s; grouped-GEMM TFLOP/s as % of B300 BF16/MXFP8 peak"
DEFAULT_WORKLOAD = "bf16_e64"
L2_BYTES = 126 * 1024 * 1024


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU-oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    p.add_argument("--rows-hint", type=int, default=None,
                   help="expected rows per local expert passed to the grouped GEMMs (default T*k/E); "
                        "it selects the GEMM kernel shape (>= 2048: CTA pairs, bf16)")
    p.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward"],
                   help="backward: time moe_layer_backward (bf16 workloads) instead of the forward step")
    p.add_argument("--no-gather", action="store_true",
                   help="feed GEMM1 from a permuted copy of x instead of reading the token rows (row gather)")
    p.add_argument("--no-sweep", action="store_true",
                   help="time the headline workload only (default: also every other configuration, "
                        "reported under 'workloads')")
    p.add_argument("--sweep-cpu-seconds", type=float, default=3.0,
                   help="budget of the CPU-oracle sample of each swept configuration")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh), "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def max_over_ranks(value: float, device) -> float:
    """Max of a per-rank number over all ranks (the job time is the slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own batch of tokens per step."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


# ----------------------------------------------------------------------------- CPU oracle
def oracle_inputs(w):
    import oracle
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    if w.dtype == "mxfp8":
        cg, sg = oracle.mx_quantize(Wg, "bf16", (w.E_loc, w.d, w.f))
        cu, su = oracle.mx_quantize(Wu, "bf16", (w.E_loc, w.d, w.f))
        cd, sd = oracle.mx_quantize(Wd, "bf16", (w.E_loc, w.f, w.d))
        wts = (cg, cu, cd, "e4m3", (sg, su, sd))
    else:
        wts = (Wg, Wu, Wd, w.act_dtype, (None, None, None))
    return x, lg, wts


def oracle_time(w, x, lg, wts, tokens, threads):
    import oracle
    Wg, Wu, Wd, wdt, scales = wts
    t0 = time.perf_counter()
    if w.dtype == "fp8":  # per-tensor FP8: h's one scale needs every local row, whatever the sample
        oracle.moe_forward_fp8(x, lg, w.k, w.e0, w.E_loc, Wg, Wu, Wd, tokens=tokens)
        return time.perf_counter() - t0
    oracle.moe_forward(x, w.act_dtype, lg, w.d, w.f, w.E, w.k, w.e0, w.E_loc, Wg, Wu, Wd, wdt, scales,
                       mx_act=(w.dtype == "mxfp8"), tokens=tokens, nthreads=threads)
    return time.perf_counter() - t0


def calibrate_sample(w, x, lg, wts, threads, budget_s):
    """Number of tokens whose oracle run takes about budget_s (tokens drawn round-robin)."""
    n = max(threads, 8)
    rng = np.random.default_rng(123)
    order = rng.permutation(w.T)
    if w.dtype == "fp8":  # the oracle's cost does not depend on the sample: time all tokens
        return np.arange(w.T)
    while True:
        dt = oracle_time(w, x, lg, wts, np.sort(order[:n]), threads)
        if dt > budget_s / 4 or n >= w.T:
            break
        n = min(w.T, n * 4)
    n = int(min(w.T, max(1, n * budget_s / max(dt, 1e-6))))
    return np.sort(order[:n])


def cpu_baseline(w, budget_s):
    threads = host_cores()
    x, lg, wts = oracle_inputs(w)
    tok = calibrate_sample(w, x, lg, wts, threads, budget_s)
    dt = oracle_time(w, x, lg, wts, tok, threads)
    return {"value": tok.size / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{tok.size} of {w.T} tokens of {w.name} (seeded uniform sample), fp64 "
                      f"{'numpy oracle (per-tensor FP8)' if w.dtype == 'fp8' else 'C++ oracle'}, {dt:.1f} s"}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    threads = host_cores()
    x, lg, wts = oracle_inputs(w)
    per_step = max(1.0, 150.0 / (args.steps + args.warmup))
    tok = calibrate_sample(w, x, lg, wts, threads, per_step)
    for _ in range(args.warmup):
        oracle_time(w, x, lg, wts, tok, threads)
    times = [oracle_time(w, x, lg, wts, tok, threads) for _ in range(args.steps)]
    total = sum(times)
    value = tok.size * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{tok.size} of {w.T} tokens per step (seeded sample), fp64 C++ oracle"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,clocks.mem,clocks.max.mem,pstate")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.perf_counter(), ln.strip()))

    def mark(self, which):
        setattr(self, which, time.perf_counter())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power, mem, mmax, pstates = [], [], set(), [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t_begin", 0.0), getattr(self, "t_end", 1e30) + 0.05
        for ts, ln in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            try:
                power.append(float(parts[2]))
            except ValueError:
                pass
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
            if len(parts) >= 11:
                try:
                    mem.append(float(parts[8]))
                    mmax.append(float(parts[9]))
                except ValueError:
                    pass
                pstates.add(parts[10])
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "mem_mhz": statistics.median(mem) if mem else None, "mem_max_mhz": max(mmax) if mmax else None,
                "pstates": sorted(pstates), "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- ours
def workload_config(w):
    wbytes = 3 * w.d * w.f * w.E_loc * (4 if w.dtype == "f32" else 2 if w.dtype == "bf16" else 1)
    return {"workload": w.name, "T": w.T, "d": w.d, "f": w.f, "E": w.E, "k": w.k, "e0": w.e0, "E_loc": w.E_loc,
            "bias": list(w.bias) if w.bias else None, "seed": w.seed,
            "l2": ("inputs larger than L2 (local expert weights %.0f MB)" % (wbytes / 1e6)) if wbytes > L2_BYTES
            else "L2 flushed between timed steps (256 MB write)",
            "parallelism": "token-sharded replicas (no exchange)"}


def recorded_traffic(kernel: str, workload: str):
    """dram bytes per launch from a committed ncu capture, if the kernel sources are unchanged."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel, {}).get(workload)
    if not ent:
        return None
    h = hashlib.sha256()
    for f in ent["sources"]:
        path = os.path.join(ROOT, "mixture_experts_layer_103_b300", "csrc", f)
        if not os.path.exists(path):
            return None
        with open(path, "rb") as fh:
            h.update(fh.read())
    if h.hexdigest()[:16] != ent["sources_sha"]:
        return None
    return ent["dram_bytes_per_launch"]


def to_dev(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def layer_bytes_flops(w, N, nonempty, n_tok_local):
    """Algorithmic FLOPs and bytes of the layer and of each grouped GEMM for one step."""
    wb = 4 if w.dtype == "f32" else 2 if w.dtype == "bf16" else 1 + 1 / 32
    ab = 4 if w.dtype == "f32" else 2          # x / y element bytes
    pb = 4 if w.dtype == "f32" else 2 if w.dtype == "bf16" else 1 + 1 / 32  # permuted x and h
    out = {
        "layer_flops": 6.0 * N * w.d * w.f,
        "layer_bytes": 3.0 * w.d * w.f * wb * nonempty + n_tok_local * w.d * ab + w.T * w.d * ab + w.T * w.E * 4,
        "gemm1_flops": 4.0 * N * w.d * w.f,
        "gemm1_bytes": 2.0 * w.d * w.f * wb * nonempty + N * w.d * pb + N * w.f * pb,
        "gemm2_flops": 2.0 * N * w.d * w.f,
        "gemm2_bytes": 1.0 * w.d * w.f * wb * nonempty + N * w.f * pb + N * w.d * 2,
    }
    return out


def backward_floor(w, N, nonempty, pk):
    """Per-kernel roofline of the bf16 backward: sum over its kernels of max(FLOPs / tensor
    peak, algorithmic bytes / HBM bandwidth), in seconds, with the per-kernel terms."""
    d, f, T, E = w.d, w.f, w.T, nonempty
    tf, bw = pk["bf16_tflops"] * 1e12, pk["hbm_gbs"] * 1e9
    parts = {  # name: (FLOPs, bytes)
        "row_copies": (0.0, 2 * (N * d * 2 + T * d * 2)),
        "dh_dswiglu": (2.0 * N * d * f, E * d * f * 2 + N * d * 2 + N * 2 * f * 2 + N * 2 * f * 2 + N * f * 2),
        "dx_gemm": (4.0 * N * d * f, N * 2 * f * 2 + E * d * 2 * f * 2 + N * d * 2),
        "slot_sum": (0.0, N * d * 2 + T * d * 2),
        "wgrad_down": (2.0 * N * d * f, N * f * 2 + N * d * 2 + w.E_loc * f * d * 4),
        "wgrad_gate_up": (4.0 * N * d * f, N * d * 2 + N * 2 * f * 2 + w.E_loc * d * 2 * f * 4),
    }
    terms = {k: max(fl / tf, by / bw) for k, (fl, by) in parts.items()}
    return sum(terms.values()), terms


SWEEP = ["tiny_fp32", "ep8_zipf_T512", "ep64_T2048", "ep64_T8192", "ep64_T32768", "mxfp8_ep8_zipf_T8192",
         "mxfp8_ep64_T8192", "fp8_ep64_T8192"]


def measure(moe, args, w, pk, pk_kind, rank, world, local, headline: bool):
    """Time K steps of one workload (one CUDA-graph replay) and compute its rooflines.

    headline: also the eager and end-to-end legs.  Returns a dict of results."""
    import torch

    wr = w.replace(seed=w.seed + rank)  # each rank its own token batch; same expert weights
    x, lg = gen_x(wr), gen_logits(wr)
    Wg, Wu, Wd = gen_weights(w)
    xd, lgd = to_dev(x), to_dev(lg)
    del x, lg
    wg_d, wu_d, wd_d = to_dev(Wg), to_dev(Wu), to_dev(Wd)
    del Wg, Wu, Wd
    pw = moe.moe_pack_weights(wg_d, wu_d, wd_d, w.dtype)
    torch.cuda.synchronize()
    del wg_d, wu_d, wd_d
    torch.cuda.empty_cache()

    T, d, k, E_loc, e0 = w.T, w.d, w.k, w.E_loc, w.e0
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    probs = torch.empty(T, k, dtype=torch.float32, device="cuda")
    hint = args.rows_hint if args.rows_hint is not None else moe.moe_rows_hint(T, k, w.E)
    # the library's own kernel choice per GEMM (a forced rows_hint names its kernel directly)
    forced = {-1: "cta", -2: "pair", -3: "swap"}
    kinds = {g: (forced.get(args.rows_hint, "cta") if args.rows_hint is not None and args.rows_hint < 0 else
                 moe.moe_layer_gemm_kernel(T, d, w.f, k, w.E, E_loc, w.dtype, g)) for g in (1, 2)}
    gather = not args.no_gather and w.dtype == "bf16"
    mx = w.dtype == "mxfp8"
    P = moe.alloc_permute(T, d, k, E_loc, xd.dtype, w.dtype, maps_only=gather)
    xq, xs = (torch.empty(T, d, dtype=torch.uint8, device="cuda"),
              torch.empty(T, d // 32, dtype=torch.uint8, device="cuda")) if gather and mx else (None, None)
    ws_perm = moe.workspace(moe.moe_permute_workspace_size(T, k, E_loc))
    h, hs = moe.alloc_h(moe.n_cap(T, k, E_loc), pw)
    Y2 = torch.empty(moe.n_cap(T, k, E_loc), d, dtype=moe.torch_dtype(w.dtype), device="cuda")
    y = torch.empty(T, d, dtype=moe.torch_dtype(w.dtype), device="cuda")
    ws_g = moe.workspace(256)
    # GEMM1's own workspace (per-tensor FP8: + bf16 h and its amax)
    ws_g1 = moe.workspace(moe.lib().moe_expert_gemm1_workspace_size(moe.n_cap(T, k, E_loc), w.f, moe._dt(w.dtype)))
    wbytes = 3 * w.d * w.f * w.E_loc * (4 if w.dtype == "f32" else 2 if w.dtype == "bf16" else 1)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda") if wbytes <= L2_BYTES else None

    # the layer's own choice: GEMM2 with the combine folded in on expert slices with under
    # one local slot per token (the standalone entry adds a small per-token set-up kernel
    # that moe_layer_forward folds into its permute), else GEMM2 and the combine kernel
    fused = moe.moe_layer_fused_combine(k, w.E, E_loc, w.dtype)
    names = ["route_topk", "permute", "gemm1_swiglu"] + (["gemm2_combine"] if fused else ["gemm2", "combine"])
    nc = len(names)
    ws_c = moe.workspace(moe.lib().moe_expert_gemm2_combine_workspace_size(moe.n_cap(T, k, E_loc), T, d)) \
        if fused else None

    def call(i):
        if i == 0:
            moe.moe_route_topk(lgd, k, ids, probs)
        elif i == 1:
            moe.moe_permute(xd, ids, probs, e0, E_loc, w.dtype, ws=ws_perm, out=P)
            if gather and mx:
                moe.moe_quantize_mx_rows(xd, xq, xs, pair_to_row=P["pair_to_row"])
        elif i == 2:
            if gather:
                moe.moe_expert_gemm1_swiglu_gather(xq if mx else xd, xs, P["row_src_token"], P["offsets"],
                                                   P["row_prob"], pw, h=h, h_scale=hs, ws=ws_g, rows_hint=hint)
            else:
                moe.moe_expert_gemm1_swiglu(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw, h=h,
                                            h_scale=hs, ws=ws_g1, rows_hint=hint)
        elif i == 3 and fused:
            moe.moe_expert_gemm2_combine(h, hs, P["offsets"], P["row_src_token"], P["pair_to_row"], pw, y=y,
                                         ws=ws_c, rows_hint=hint)
        elif i == 3:
            moe.moe_expert_gemm2(h, hs, P["offsets"], pw, Y2=Y2, ws=ws_g, rows_hint=hint)
        else:
            moe.moe_unpermute_combine(Y2, P["pair_to_row"], w.dtype, y=y)

    def step(marks):
        """One step; marks[i] (an event or None) is recorded before call i, marks[nc] after the last."""
        for i in range(nc):
            if marks[i] is not None:
                marks[i].record()
            call(i)
        if marks[nc] is not None:
            marks[nc].record()

    for _ in range(args.warmup):
        if flush is not None:
            flush.zero_()
        step([None] * (nc + 1))
    torch.cuda.synchronize()
    err = moe.moe_get_device_error(ws_g) or (moe.moe_get_device_error(ws_c) if fused else 0)
    if err != 0:
        raise RuntimeError(f"{w.name}: device error {err} during warm-up")
    offs = P["offsets"].cpu().numpy().astype(np.int64)
    N = int(offs[-1])
    nonempty = int((np.diff(offs) > 0).sum())
    p2r = P["pair_to_row"].cpu().numpy()
    n_tok_local = int((p2r >= 0).any(axis=1).sum())

    def ev():
        return torch.cuda.Event(enable_timing=True, external=True)

    def capture(n_steps, mark_all):
        """CUDA graph of n_steps steps.  Only GEMM1 (the dominant kernel) is bracketed by
        event nodes unless mark_all: event nodes between kernels cut the programmatic
        dependent-launch overlap, so the timed graph keeps them to that one kernel."""
        # with an L2 flush between steps the step itself is bracketed too (the flush is
        # excluded from the step time)
        keep = (0, 2, 3, nc) if flush is not None else (2, 3)
        marks = [[ev() if (mark_all or j in keep) else None for j in range(nc + 1)] for _ in range(n_steps)]
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cs):
            for i in range(n_steps):
                if flush is not None:
                    flush.zero_()
                step(marks[i])
        torch.cuda.synchronize()
        return g, marks

    # The K timed steps are one CUDA graph (the library launches nothing else and
    # allocates nothing, so the calls capture as they are).
    graph, marks = capture(args.steps, mark_all=False)
    graph.replay()  # warm replay of the captured steps
    torch.cuda.synchronize()
    region0, region1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    if rank == 0:
        clocks.start()
    clocks.mark("t_begin")
    region0.record()
    graph.replay()
    region1.record()
    torch.cuda.synchronize()
    clocks.mark("t_end")
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if rank == 0 else None
    err = moe.moe_get_device_error(ws_g) or (moe.moe_get_device_error(ws_c) if fused else 0)
    if err != 0:
        raise RuntimeError(f"{w.name}: device error {err} in the timed region")
    del graph
    region_ms = region0.elapsed_time(region1)
    gemm1_ms = statistics.mean(marks[i][2].elapsed_time(marks[i][3]) for i in range(args.steps))
    total_ms = (sum(marks[i][0].elapsed_time(marks[i][nc]) for i in range(args.steps)) if flush is not None
                else region_ms)
    # per-kernel breakdown: a separate (untimed for `value`) graph with events between all kernels
    nb = min(args.steps, 50)
    bgraph, bmarks = capture(nb, mark_all=True)
    bgraph.replay()
    torch.cuda.synchronize()
    kern_ms = {nm: statistics.mean(bmarks[i][j].elapsed_time(bmarks[i][j + 1]) for i in range(nb))
               for j, nm in enumerate(names)}
    kern_ms["gemm1_swiglu_timed_region"] = gemm1_ms
    del bgraph
    eager_ms = None
    if headline:
        # eager (one Python call per step), for reference only: includes host launch overhead
        n_eager = min(args.steps, 50)
        ev_e = [[torch.cuda.Event(enable_timing=True) for _ in range(nc + 1)] for _ in range(n_eager)]
        for i in range(n_eager):
            step(ev_e[i])
        torch.cuda.synchronize()
        eager_ms = statistics.mean(ev_e[i][0].elapsed_time(ev_e[i][-1]) for i in range(n_eager))

    total_ms = max_over_ranks(total_ms, "cuda")
    ms_per_step = total_ms / args.steps

    # ---- roofline of the dominant kernel and of the whole layer
    bf = layer_bytes_flops(w, N, nonempty, n_tok_local)
    hbm = pk["hbm_gbs"]
    tpeak = pk["bf16_tflops"] * (2.0 if w.dtype in ("mxfp8", "fp8") else 1.0)
    g2name = "gemm2_combine" if fused else "gemm2"
    dom = max(("gemm1_swiglu", g2name), key=lambda n: kern_ms[n])
    key = "gemm1" if dom == "gemm1_swiglu" else "gemm2"
    fl, by = bf[key + "_flops"], bf[key + "_bytes"]
    # the dominant kernel's duration: live, from the events around it in the timed region
    t_s = (gemm1_ms if dom == "gemm1_swiglu" else kern_ms[dom]) / 1e3
    tensor_bound = (fl / (tpeak * 1e12)) >= (by / (hbm * 1e9))
    if w.dtype == "f32":
        roof = {"bound": "alu", "achieved": fl / t_s / 1e12, "peak": None, "unit": "TFLOP/s", "frac": None}
    elif tensor_bound:
        roof = {"bound": "tensor", "achieved": fl / t_s / 1e12, "peak": tpeak, "unit": "TFLOP/s",
                "frac": fl / t_s / 1e12 / tpeak}
    else:
        roof = {"bound": "hbm", "achieved": by / t_s / 1e9, "peak": hbm, "unit": "GB/s",
                "frac": by / t_s / 1e9 / hbm}
    kname = ("simt_grouped_gemm_kernel" if w.dtype == "f32" else
             {"cta": "tc_grouped_gemm_kernel", "pair": "tc_grouped_gemm_pair_kernel",
              "swap": "tc_swap_gemm_kernel"}[kinds[1 if dom == "gemm1_swiglu" else 2]])
    roof.update({"kernel": f"{kname} ({dom})", "traffic": recorded_traffic(dom, w.name),
                 "peak_kind": pk_kind + (" (bf16 x2 nominal fp8 ratio)" if w.dtype in ("mxfp8", "fp8") else "")})
    t_roof = max(bf["layer_flops"] / (tpeak * 1e12), bf["layer_bytes"] / (hbm * 1e9))
    gemm_s = (gemm1_ms + kern_ms[g2name]) / 1e3
    layer = {"roofline_us": t_roof * 1e6, "measured_us": ms_per_step * 1e3, "frac": t_roof / (ms_per_step / 1e3),
             "algorithmic_bytes": bf["layer_bytes"], "flops": bf["layer_flops"], "N_pairs": N,
             "nonempty_experts": nonempty, "tokens_with_local_expert": n_tok_local,
             "grouped_gemm_tflops": bf["layer_flops"] / gemm_s / 1e12,
             "grouped_gemm_pct_of_peak": 100 * bf["layer_flops"] / gemm_s / 1e12 / tpeak}

    # ---- end to end through moe_layer_forward with host buffers
    e2e = None
    if headline and not args.no_e2e:
        e2e = e2e_leg(moe, args, w, xd, lgd, y, pw, flush, world)
    # route 1, permute 3 (+1 copy or MXFP8 per-token quantisation), GEMM1, then GEMM2 +
    # combine (set-up kernel + fused GEMM2) or GEMM2 and the combine kernel
    launches_per_step = 1 + 3 + (0 if gather and not mx else 1) + 3
    return dict(value=job_tokens_per_s(T, world, ms_per_step), ms_per_step=ms_per_step, roof=roof, layer=layer,
                kern_ms=kern_ms, region_ms=region_ms, gather=gather, eager_ms=eager_ms, e2e=e2e, clocks=clk,
                launches_per_step=launches_per_step)


def e2e_leg(moe, args, w, xd, lgd, y, pw, flush, world):
    """The same metric end to end through moe_layer_forward with pinned host buffers."""
    import torch
    T, d, k, E_loc, e0 = w.T, w.d, w.k, w.E_loc, w.e0
    # Steps are pipelined over three streams with triple-buffered device inputs and
    # outputs: step i's host->device copy and step i-1's device->host read overlap
    # step i-1's / i's compute.  Every step still copies its own inputs in and its
    # result out inside the timed region.
    x_pin = torch.empty(xd.shape, dtype=xd.dtype).pin_memory()
    x_pin.copy_(xd.cpu())
    lg_pin = torch.empty(lgd.shape, dtype=lgd.dtype).pin_memory()
    lg_pin.copy_(lgd.cpu())
    nbuf = 3
    y_pin = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(nbuf)]
    xb = [torch.empty_like(xd) for _ in range(nbuf)]
    lgb = [torch.empty_like(lgd) for _ in range(nbuf)]
    yb = [torch.empty_like(y) for _ in range(nbuf)]
    ws_layer = moe.workspace(moe.moe_layer_workspace_size(T, d, w.f, w.E, k, E_loc, w.dtype))
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    for b_ in range(nbuf):  # start with every buffer free
        ev_comp[b_].record(s_comp)
        ev_out[b_].record(s_out)

    def e2e_step(i):
        b_ = i % nbuf
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[b_])   # step i-nbuf has finished reading this input buffer
            xb[b_].copy_(x_pin, non_blocking=True)
            lgb[b_].copy_(lg_pin, non_blocking=True)
            ev_in[b_].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[b_])
            s_comp.wait_event(ev_out[b_])  # step i-nbuf's result has left this output buffer
            if flush is not None:
                flush.zero_()
            moe.moe_layer_forward(xb[b_], lgb[b_], w.E, k, e0, pw, y=yb[b_], ws=ws_layer)
            ev_comp[b_].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b_])
            y_pin[b_].copy_(yb[b_], non_blocking=True)
            ev_out[b_].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    # as many steps as the device-timed region (at least 10): the pipeline's first copy in
    # and last copy out are not overlapped, so few steps would mostly time its fill
    n2 = args.e2e_steps or max(10, args.steps)
    # the n2 steps (copies, layer calls, event dependencies on three streams) are captured
    # once as a CUDA graph and replayed inside the timed region, like the device-only steps
    ge = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(ge, stream=cap):
        for st_ in (s_in, s_comp, s_out):
            st_.wait_stream(cap)
        for b_ in range(nbuf):
            ev_comp[b_].record(s_comp)
            ev_out[b_].record(s_out)
        for i in range(n2):
            e2e_step(i)
        for st_ in (s_in, s_comp, s_out):
            cap.wait_stream(st_)
    ge.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    ge.replay()
    b.record()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws_layer) == 0
    ms = a.elapsed_time(b) / n2
    x_pin_bytes = x_pin.numel() * x_pin.element_size()

    # the copies alone (same buffers, 5 each, after the timed region): the host link's
    # rates, which bound the end-to-end step from below
    def copy_ms(fn):
        e0_, e1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize()
        e0_.record()
        for _ in range(5):
            fn()
        e1_.record()
        torch.cuda.synchronize()
        return e0_.elapsed_time(e1_) / 5

    h2d_bytes = x_pin_bytes + lg_pin.numel() * 4
    d2h_bytes = y_pin[0].numel() * y_pin[0].element_size()
    h2d_ms = copy_ms(lambda: (xb[0].copy_(x_pin, non_blocking=True), lgb[0].copy_(lg_pin, non_blocking=True)))
    d2h_ms = copy_ms(lambda: y_pin[0].copy_(yb[0], non_blocking=True))

    def both():  # a step's copies in both directions at once, as the pipeline runs them
        s_in.wait_stream(torch.cuda.current_stream())
        s_out.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_in):
            xb[0].copy_(x_pin, non_blocking=True)
            lgb[0].copy_(lg_pin, non_blocking=True)
        with torch.cuda.stream(s_out):
            y_pin[1].copy_(yb[1], non_blocking=True)
        torch.cuda.current_stream().wait_stream(s_in)
        torch.cuda.current_stream().wait_stream(s_out)
    both_ms = copy_ms(both)
    return {"value": T * world / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_gbs": h2d_bytes / (h2d_ms / 1e3) / 1e9, "d2h_gbs": d2h_bytes / (d2h_ms / 1e3) / 1e9,
            "copy_bound_ms_per_step": max(h2d_ms, d2h_ms),
            "copies_both_directions_ms_per_step": both_ms,
            "h2d_bytes_per_step": int(x_pin_bytes + lg_pin.numel() * 4),
            "d2h_bytes_per_step": int(y_pin[0].numel() * y_pin[0].element_size()), "steps": n2,
            "entry_point": "moe_layer_forward",
            "pipelining": "copies of neighbouring steps overlap compute (3 streams, 3 buffers), "
                          "the steps replayed as one CUDA graph"}


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import mixture_experts_layer_103_b300 as moe

    pk, pk_kind = peaks()
    R = measure(moe, args, w, pk, pk_kind, rank, world, local, headline=True)
    torch.cuda.empty_cache()
    # every other configuration of the pages' workloads, timed the same way in this process
    # (one rank: the sweep documents per-config kernel quality, the headline line scales)
    sweep = {}
    if not args.no_sweep and world == 1:
        for name in SWEEP:
            if name == w.name:
                continue
            ws_ = WORKLOADS[name]
            r = measure(moe, args, ws_, pk, pk_kind, rank, world, local, headline=False)
            torch.cuda.empty_cache()
            cpu_ws = None if args.no_cpu_baseline else cpu_baseline(ws_, args.sweep_cpu_seconds)
            sweep[name] = {"value": r["value"], "unit": "tokens/s", "ms_per_step": r["ms_per_step"],
                           "dtype": ws_.dtype, "config": workload_config(ws_), "roofline": r["roof"],
                           "layer": r["layer"], "kernels_us": {n: 1e3 * v for n, v in r["kern_ms"].items()},
                           "gemm1_operand": "token rows gathered in the kernel" if r["gather"]
                           else "permuted copy of x", "gpu_launches": r["launches_per_step"] * args.steps,
                           "clocks": r["clocks"], "cpu_baseline": cpu_ws}

    if world > 1:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return
    cpu = None if args.no_cpu_baseline else cpu_baseline(w, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": R["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": R["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"f32": "f32", "bf16": "bf16", "mxfp8": "e4m3+e8m0 (mxfp8)",
                                       "fp8": "e4m3, one power-of-two scale per tensor (fp8)"}[w.dtype],
        "data": "synthetic (seeded; shapes of the pages' workloads)", "config": workload_config(w),
        "roofline": R["roof"], "layer": R["layer"], "kernels_us": {n: 1e3 * v for n, v in R["kern_ms"].items()},
        "timed_region_ms": R["region_ms"],
        "gemm1_operand": "token rows gathered in the kernel" if R["gather"] else "permuted copy of x",
        "timing": ("one CUDA-graph replay of the K steps (region events; with an L2 flush, the sum of the steps' "
                   "own event intervals); GEMM1 bracketed by event nodes in the timed graph; kernels_us from a "
                   "separate graph with events between all kernels"),
        "eager_ms_per_step": R["eager_ms"], "e2e": R["e2e"], "cpu_baseline": cpu,
        "gpu_launches": R["launches_per_step"] * args.steps, "clocks": R["clocks"],
        "workloads": sweep,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_backward(args, w):
    """One step = moe_layer_backward (maps, dy and x rows copied into routed order, dh +
    ScaledSwiGLU backward, dx, router-logit and weight gradients; the gate/up
    pre-activations come from moe_layer_forward_train) on inputs resident in HBM; K steps
    captured as one CUDA graph and replayed inside the timed region."""
    import torch
    import torch.distributed as dist

    if w.dtype not in ("bf16", "mxfp8", "fp8"):
        raise SystemExit("the backward is bf16, MXFP8 or per-tensor FP8")
    mx = w.dtype in ("mxfp8", "fp8")
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import mixture_experts_layer_103_b300 as moe
    from synthetic import gen_dy

    pk, pk_kind = peaks()
    wr = w.replace(seed=w.seed + rank)
    xd, lgd, dyd = to_dev(gen_x(wr)), to_dev(gen_logits(wr)), to_dev(gen_dy(wr))
    Wg, Wu, Wd = (to_dev(a) for a in gen_weights(w))
    if mx:
        # MXFP8: g, u recomputed on the block-scaled tensor cores inside the backward
        pw = moe.moe_pack_weights(Wg, Wu, Wd, w.dtype)
        bw = moe.moe_pack_weights_backward_mx(Wg, Wu, Wd, w_exp=pw.w_exp)
        del Wg, Wu, Wd
        ids, probs = moe.moe_route_topk(lgd, w.k)

        def bwd(ws=None, out=None):
            return moe.moe_layer_backward_mx(xd, dyd, ids, probs, w.E, w.e0, pw, bw, ws=ws, out=out)
    else:
        pw = moe.moe_pack_weights(Wg, Wu, Wd, "bf16")
        WguT = moe.moe_pack_weights_backward(Wg, Wu)
        del Wg, Wu
        # the training forward keeps the routing and the gate/up pre-activations for the backward
        _, ids, probs, gu, _ = moe.moe_layer_forward_train(xd, lgd, w.E, w.k, w.e0, pw)

        def bwd(ws=None, out=None):
            return moe.moe_layer_backward(xd, dyd, ids, probs, w.E, w.e0, pw, Wd, WguT, ws=ws, out=out, gu_saved=gu)
    out, ws = bwd()
    for _ in range(args.warmup):
        bwd(ws=ws, out=out)
    torch.cuda.synchronize()
    if moe.moe_get_device_error(ws) != 0:
        raise RuntimeError("device error during warm-up")
    P = moe.moe_permute(xd, ids, probs, w.e0, w.E_loc, "bf16", maps_only=True)
    N = int(P["offsets"][-1].item())
    nonempty = int((P["counts"] > 0).sum().item())
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cs):
        for _ in range(args.steps):
            bwd(ws=ws, out=out)
    g.replay()
    torch.cuda.synchronize()
    e0_, e1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]))
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark("t_begin")
    e0_.record()
    g.replay()
    e1_.record()
    torch.cuda.synchronize()
    clocks.mark("t_end")
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(e0_.elapsed_time(e1_) / args.steps, torch.device("cuda", local))
    value = job_tokens_per_s(w.T, world, ms)
    # the backward's GEMM work (g, u saved by the training forward): dh 2NDF, dx 4NDF,
    # weight gradients 6NDF (MXFP8: + the 4NDF recompute of g, u)
    flops = 12.0 * N * w.d * w.f
    floor_s, floor_terms = backward_floor(w, N, nonempty, pk)
    line = {
        "metric": "MoE-layer backward tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"mxfp8": "e4m3+e8m0 (mxfp8)", "fp8": "e4m3, one power-of-two scale per tensor (fp8)"}.get(w.dtype, "bf16"),
        "data": "synthetic (seeded)",
        "config": workload_config(w), "pass": "backward",
        "roofline": {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"],
                     "kernel": "whole backward (12 N d f FLOP)", "traffic": None, "peak_kind": pk_kind},
        "N_pairs": N, "gpu_launches": ({"mxfp8": 15, "fp8": 23}.get(w.dtype, 11)) * args.steps, "clocks": clk,
        "per_kernel_floor": {"roofline_us": floor_s * 1e6, "measured_us": ms * 1e3, "frac": floor_s / (ms * 1e-3),
                             "terms_us": {k: v * 1e6 for k, v in floor_terms.items()},
                             "note": "sum over the backward's kernels of max(FLOPs / bf16 peak, bytes / HBM)"},
        "saved_preactivations": ("recomputed on the block-scaled tensor cores (4 N d f more FLOP, not counted "
                                 "above)" if mx else "from moe_layer_forward_train (no recompute)"),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    elif args.which == "backward":
        run_backward(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
