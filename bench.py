"""Benchmark of the routed block-scaled FP4 MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step is one fp4moe_forward over one batch: routing, permutation,
activation quantisation, gate/up GEMM + SwiGLU + requantisation, down GEMM +
combine.  The default workload is the Kimi-shaped decode layer (T=8, H=7168,
I=2048, E=384, top-8, MXFP4 A4W4).  Weights (~9 GB) are drawn on the device
from the seeded generator; inputs are resident in HBM when timing starts.
Between timed steps a 256 MiB buffer is written to flush L2 (untimed).  Each
step is timed with CUDA events on the launching stream; the dominant kernel
(gate/up GEMM) is timed by events recorded around its launch.

--emulate times an NVFP4 workload in emulation mode (BF16 dequantised experts,
NVFP4 QDQ activations, BF16 GEMMs).  --w8a8 times the W8A8 layer instead: the same synthetic MXFP4 experts after the
exact per-channel FP8 conversion, per-token dynamic E4M3 activations
(fp4moe_forward_w8a8).

With torchrun (N > 1) each rank runs an independent replica on its own batch
(no collective on the data path); the line reports the max over ranks.

--impl reference times the FP64 CPU oracle (the only other implementation of
this layer) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "MoE-layer tokens/s; FP4 TFLOP/s (prefill), weight-stream HBM GB/s (decode)"
L2_FLUSH_BYTES = 256 << 20


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def code_text(src: str) -> str:
    """C++/CUDA source without comments and blank space: a comment-only edit
    leaves the kernel, and so this text, unchanged.  String literals (inline
    PTX) are kept as they are."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"':  # string literal, escapes included
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_sha(paths) -> str:
    """Hash of the code (comments and spacing excluded) of the given files."""
    h = hashlib.sha256()
    for p in paths:
        h.update(code_text((ROOT / p).read_text()).encode())
    return h.hexdigest()[:16]


GEMM_SOURCES = ["block_scaled_fp4_sigmoid_gb300/csrc/gemm.cuh", "block_scaled_fp4_sigmoid_gb300/csrc/common.cuh",
                "block_scaled_fp4_sigmoid_gb300/csrc/gemm_launch.cuh"]
# the committed ncu summary names the kernel it measured
PROFILED_KERNEL = "moe_gemm_kernel"


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the gate/up kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    f = ROOT / "profiles" / f"ncu_gateup_{workload}.md"
    if not f.exists():
        return None
    text = f.read_text()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != source_sha(GEMM_SOURCES):
        return None
    return float(m.group(1))


def profiled_ratios(workload: str):
    """DRAM bytes over algorithmic bytes of the two expert GEMMs, from the
    committed ncu summary of a smaller case of the workload (its file names
    the case), if it was taken on the current kernel source; else None.  A
    launch's traffic grows with the bytes it must move (touched experts and
    routes), so the ratio carries over to the full workload."""
    for f in sorted((ROOT / "profiles").glob(f"ncu_gemm_{workload}*.md")):
        text = f.read_text()
        s = re.search(r"source_sha:\s*([0-9a-f]+)", text)
        g = re.search(r"dram_ratio_gateup:\s*([0-9.]+)", text)
        d = re.search(r"dram_ratio_down:\s*([0-9.]+)", text)
        if s and g and d and s.group(1) == source_sha(GEMM_SOURCES):
            return {"gateup": float(g.group(1)), "down": float(d.group(1)), "from": f.name}
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle timing
def oracle_route_sample(cfg_name: str, n_routes: int, frac: float = 1.0, start_token: int = 0, w8a8: bool = False,
                        emulate: bool = False):
    """Times the FP64 oracle on n_routes (token, expert) routes of the
    workload: each token's routing and x quantisation, then its expert MLPs.
    frac < 1 evaluates each MLP on the first frac * I intermediate channels
    only (a sub-problem of the same form: whole 32-blocks of h).  Weight
    generation is input preparation and stays outside the timing.
    Returns (seconds, tokens processed)."""
    from dataclasses import replace
    import numpy as np
    import synth
    from oracle import inputs as OI
    from oracle import moe as M
    from oracle import quant as Q
    from oracle import emulation as EM
    from oracle import w8a8 as W8
    from oracle.router import route, router_logits
    cfg = synth.configs()[cfg_name]
    Ip = cfg.I if frac >= 1 else max(32, int(cfg.I * frac) // 32 * 32)
    sub = replace(cfg, I=Ip)
    ws = W8.fp8_weight_source(cfg) if w8a8 else OI.oracle_weights(cfg)
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    bias = synth.gen_bias_f32(cfg)
    done, t_total, t = 0, 0.0, start_token
    while done < n_routes:
        x = synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg, t % cfg.T, t % cfg.T + 1))
        t0 = time.perf_counter()
        logits, _ = router_logits(x, wr)
        idx, w = route(logits, bias, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.routed_scaling, cfg.renormalize)
        if w8a8:
            a = W8.fp8_dequant(*W8.fp8_quantize(x))
        elif emulate:
            a = EM.nv_dequant_bf16(*Q.nv_quantize(x))
        else:
            xc, xs, gx = Q.quantize(x, cfg.fmt)
            a = Q.dequant(xc, xs, cfg.fmt, gx)
        t_total += time.perf_counter() - t0
        experts = [int(e) for e in idx[0]] + list(range(cfg.E, cfg.E + cfg.n_shared))
        for j, e in enumerate(experts):
            if done >= n_routes:
                break
            wt = w[0, j] if j < cfg.top_k else 1.0
            names = ("w13", "w2") if e < cfg.E else ("sh13", "sh2")
            ee = e if e < cfg.E else e - cfg.E
            w13 = ws.get(names[0], ee)
            w2 = ws.get(names[1], ee)
            blk = 16 if cfg.fmt == "nvfp4" else 32
            keep = np.r_[0:Ip, cfg.I:cfg.I + Ip]
            if w8a8:  # value matrices
                s13, s2 = w13[keep], np.ascontiguousarray(w2[:, :Ip])
            else:
                s13 = (w13[0][keep], w13[1][keep], w13[2])
                s2 = (np.ascontiguousarray(w2[0][:, :Ip]), np.ascontiguousarray(w2[1][:, :Ip // blk]), w2[2])
            sub_ws = M.WeightSource(lambda which, _e, _a=s13, _b=s2: _a if which in ("w13", "sh13") else _b)
            t0 = time.perf_counter()
            if w8a8:
                W8.expert_rows_fp8(sub, e, a, np.array([wt]), sub_ws, with_ambiguity=False)
            elif emulate:
                EM.emulated_expert_rows(sub, e, a, np.array([wt]), sub_ws, with_ambiguity=False)
            else:
                M.expert_rows(sub, e, a, np.array([wt]), sub_ws, with_ambiguity=False)
            t_total += time.perf_counter() - t0
            ws.drop(names[0], ee)
            ws.drop(names[1], ee)
            done += 1
        t += 1
    rpt = cfg.top_k + cfg.n_shared
    return t_total, n_routes / rpt * (Ip / cfg.I)


def oracle_full_layer(cfg_name: str, max_experts: int | None = None, conv_rows: int = 0):
    """The FP64 oracle over a whole workload on the host cores: routing of
    every token, activation quantisation, the permutation, then every
    touched expert's MLP on all of its routed rows (oracle.moe.expert_rows,
    the combine included).  Weight generation is input preparation and stays
    outside the timing.  max_experts bounds the run to the first experts of
    the permutation (None: all); conv_rows > 0 also times the MXFP4 -> FP8
    conversion oracle on that many expert rows.  Returns a dict of seconds
    and counts."""
    import numpy as np
    import synth
    from oracle import inputs as OI
    from oracle import moe as M
    from oracle import quant as Q
    from oracle.convert import mxfp4_to_fp8_rowscale
    from oracle.permute import permute
    from oracle.router import route, router_logits
    cfg = synth.configs()[cfg_name]
    x = synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg))
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    bias = synth.gen_bias_f32(cfg)
    ws = OI.oracle_weights(cfg)
    t0 = time.perf_counter()
    logits, _ = router_logits(x, wr)
    idx, w = route(logits, bias, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.routed_scaling, cfg.renormalize)
    xc, xs, gx = Q.quantize(x, cfg.fmt)
    counts, offsets, ptok, pslot = permute(idx, cfg.E, cfg.n_shared)
    t_route = time.perf_counter() - t0
    experts = [e for e in range(cfg.E + cfg.n_shared) if counts[e] > 0]
    done = experts if max_experts is None else experts[:max_experts]
    out = np.zeros((cfg.T, cfg.H))
    t_experts, routes, flops = 0.0, 0, 0.0
    for e in done:
        rows = np.arange(offsets[e], offsets[e + 1])
        toks, slots = ptok[rows], pslot[rows]
        wts = w[toks, np.minimum(slots, cfg.top_k - 1)] if e < cfg.E else np.ones(len(rows))
        names = ("w13", "w2") if e < cfg.E else ("sh13", "sh2")
        ee = e if e < cfg.E else e - cfg.E
        ws.get(names[0], ee), ws.get(names[1], ee)  # generated outside the timing
        t0 = time.perf_counter()
        a = Q.dequant(xc[toks], xs[toks], cfg.fmt, gx)
        info = M.expert_rows(cfg, e, a, wts, ws, with_ambiguity=False)
        np.add.at(out, toks, wts[:, None] * info["y"])
        t_experts += time.perf_counter() - t0
        routes += len(rows)
        flops += 2.0 * 3 * cfg.I * cfg.H * len(rows)
        ws.drop(names[0], ee)
        ws.drop(names[1], ee)
    res = {"config": cfg_name, "tokens": cfg.T, "experts_done": len(done), "experts_touched": len(experts),
           "routes_done": routes, "routes_total": int(counts.sum()), "route_s": t_route, "expert_s": t_experts,
           "expert_gflops": flops / max(t_experts, 1e-9) / 1e9, "cores": cpu_cores()}
    if conv_rows:  # w13 rows (K = H) of consecutive experts, generation outside the timing
        rows, _ = synth.weight_shape(cfg, "w13")
        t_conv, done_rows, e = 0.0, 0, 0
        while done_rows < conv_rows:
            codes, scales = synth.gen_mx_weight(cfg, "w13", e)
            take = min(rows, conv_rows - done_rows)
            t1 = time.perf_counter()
            mxfp4_to_fp8_rowscale(codes[:take], scales[:take])
            t_conv += time.perf_counter() - t1
            done_rows += take
            e += 1
        res["conversion_rows"] = done_rows
        res["conversion_s"] = t_conv
    return res


def _conversion_task(args):
    """One expert matrix through the conversion oracle, in row blocks (worker
    process of oracle_full_conversion): (rows, seconds in the oracle)."""
    import synth
    from oracle.convert import mxfp4_to_fp8_rowscale
    cfg_name, which, e = args
    cfg = synth.configs()[cfg_name]
    codes, scales = synth.gen_mx_weight(cfg, which, e)
    secs = 0.0
    for r0 in range(0, codes.shape[0], 1024):
        t0 = time.perf_counter()
        mxfp4_to_fp8_rowscale(codes[r0:r0 + 1024], scales[r0:r0 + 1024])
        secs += time.perf_counter() - t0
    return codes.shape[0], secs


def oracle_full_conversion(cfg_name: str = "skewed_shared") -> dict:
    """The MXFP4 -> FP8 conversion oracle over every routed expert row of a
    layer (gate/up rows with K = H and down rows with K = I), one worker
    process per host core.  Weight generation happens in the workers and is
    not counted: each worker times its oracle calls only."""
    import multiprocessing as mp
    import synth
    cfg = synth.configs()[cfg_name]
    procs = cpu_cores()
    tasks = [(cfg_name, w, e) for e in range(cfg.E) for w in ("w13", "w2")]
    t0 = time.perf_counter()
    with mp.get_context("spawn").Pool(procs) as pool:
        res = pool.map(_conversion_task, tasks, chunksize=1)
    wall = time.perf_counter() - t0
    rows = sum(r for r, _ in res)
    secs = sum(s for _, s in res)
    return {"config": cfg_name, "conversion_rows": rows, "oracle_core_s": secs, "procs": procs,
            "oracle_s_per_proc": secs / procs, "rows_per_s": rows / (secs / procs), "wall_s_with_generation": wall,
            "cores": procs}


def algorithmic_bytes(H: int, I: int, fmt: str, mode: str, touched: int, routes: int,
                      tokens: int) -> tuple[float, float]:
    """Bytes the gate/up and the down GEMM of one layer call must move at
    least: the touched experts' weights (with their scales), the activation
    rows each reads and what each writes, for R routes of T tokens.
      a4w4:    FP4 values at 0.5 B plus one scale byte per block (MXFP4 32,
               NVFP4 16); gate/up reads x, writes the quantised h; down
               reads it and leaves one fp32 output row per token (the
               weighted sum of the token's routes, written once).
      w8a8:    E4M3 bytes plus fp32 scales per weight row and per activation
               row; gate/up writes fp32 h, down reads its E4M3 form.
      emulate: BF16 weights and activation rows; gate/up writes fp32 h."""
    if mode == "emulate":
        gu = touched * (2 * I * H * 2) + routes * H * 2 + routes * I * 4
        dn = touched * (H * I * 2) + routes * I * 2 + tokens * H * 4
    elif mode == "w8a8":
        gu = touched * (2 * I * H + 2 * I * 4) + routes * (H + 4) + routes * I * 4
        dn = touched * (H * I + H * 4) + routes * (I + 4) + tokens * H * 4
    elif mode == "a4w4":
        act = 0.5 + 1.0 / (16 if fmt == "nvfp4" else 32)  # bytes per FP4 value incl. scale
        gu = touched * (2 * I * H * act) + routes * H * act + routes * I * act
        dn = touched * (H * I * act) + routes * I * act + tokens * H * 4
    else:
        raise ValueError(mode)
    return gu, dn


def rank_token_range(rank: int, T: int) -> tuple[int, int]:
    """Weak scaling: every rank runs its own batch of T tokens, tokens
    rank*T .. (rank+1)*T of the seeded stream."""
    return rank * T, (rank + 1) * T


def max_over_ranks(vals, world: int, device) -> list:
    """Element-wise maximum over the ranks (the slowest rank's times); the
    identity for one rank."""
    import torch
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Units all ranks processed per second, over the slowest rank's time."""
    return units_per_rank * world / (ms_max * 1e-3)


def reference_arm(args, cfg, rank, world):
    if rank != 0:
        return
    # size each step so that warm-up + steps take about two minutes
    t_one, _ = oracle_route_sample(args.config, 1, w8a8=args.w8a8, emulate=args.emulate)
    budget = 120.0 / (args.steps + args.warmup)
    frac = min(1.0, budget / max(t_one, 1e-3))
    secs, toks = [], 0.0
    for i in range(args.warmup + args.steps):
        sec, n = oracle_route_sample(args.config, 1, frac, start_token=i, w8a8=args.w8a8, emulate=args.emulate)
        if i >= args.warmup:
            secs.append(sec)
            toks += n
    total = sum(secs)
    value = toks / total
    cores = cpu_cores()
    Ip = cfg.I if frac >= 1 else max(32, int(cfg.I * frac) // 32 * 32)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": cfg_label(cfg, args.w8a8, args.emulate),
                                            "step": f"one (token, expert) route on {Ip} of {cfg.I} channels"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} routes of the {cfg.name} workload, {Ip}/{cfg.I} "
                                       f"intermediate channels each"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cfg_label(cfg, w8a8: bool = False, emulate: bool = False) -> str:
    fmt = ("FP8 W8A8 (experts exactly converted from MXFP4)" if w8a8 else
           "NVFP4 emulation (BF16 dequantised experts, NVFP4 QDQ activations)" if emulate else
           f"{cfg.fmt.upper()} A4W4")
    return (f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} top-{cfg.top_k}"
            f"{f' groups {cfg.n_group}/{cfg.topk_group}' if cfg.n_group > 1 else ''}"
            f"{' +1 shared' if cfg.n_shared else ''} {fmt}")


# ------------------------------------------------------------------ MXFP4 -> FP8 conversion
def time_conversion(layer, peaks, stream, reps: int = 5):
    """fp4moe_mxfp4_to_fp8_rowscale over every routed expert row of the layer
    (w13 rows of K = H, then w2 rows of K = I), timed with CUDA events.
    Algorithmic bytes: codes + scales in, E4M3 bytes + row scale + status out."""
    import torch
    import block_scaled_fp4_sigmoid_gb300 as fm
    d = layer.dims
    s = stream.cuda_stream
    ws = torch.zeros(256, dtype=torch.uint8, device=layer.device)
    w13s, w2s = layer.raw_scales
    parts = [(layer.w13, w13s, d.E * 2 * d.I, d.H), (layer.w2, w2s, d.E * d.H, d.I)]
    total_ms, total_bytes, rows_all = 0.0, 0, 0
    for codes, scales, rows, K in parts:
        out = torch.empty((rows, K), dtype=torch.uint8, device=layer.device)
        rs = torch.empty(rows, dtype=torch.float32, device=layer.device)
        st = torch.empty(rows, dtype=torch.uint8, device=layer.device)
        args = (codes.data_ptr(), scales.data_ptr(), rows, K, out.data_ptr(), rs.data_ptr(), st.data_ptr(),
                ws.data_ptr(), 256, s)
        fm.mxfp4_to_fp8_rowscale(*args)  # warm-up
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
        for i in range(reps):
            ev[2 * i].record(stream)
            fm.mxfp4_to_fp8_rowscale(*args)
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        total_ms += statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(reps))
        total_bytes += rows * (K // 2 + K // 32 + K + 4 + 1)
        rows_all += rows
        del out, rs, st
    st_code, n_bad = fm.get_status(ws.data_ptr(), s)
    gbs = total_bytes / (total_ms * 1e-3) / 1e9
    return {"rows": rows_all, "ms": total_ms, "achieved": gbs, "unit": "GB/s", "peak": peaks["hbm_gbs"],
            "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": total_bytes, "rows_flagged": n_bad,
            "bound": "hbm", "l2": "inputs and outputs (25.9 GB) far exceed L2"}


# ------------------------------------------------------------------ dense linear
def linear_arm(args, rank, world, local_rank):
    """fp4moe_linear on one dense shape: out[T, N] = quantize(x)[T, K] . W^T,
    MXFP4 weights of the synthetic recipe, bf16 x ~ N(0, 1), drawn on the
    device.  FLOPs 2 T K N per call; the roofline is the dense FP4 tensor
    peak (6 x the measured bf16 peak, the nominal 13.5 / 2.25 ratio)."""
    import numpy as np
    import torch
    import block_scaled_fp4_sigmoid_gb300 as fm
    import synth
    import __graft_entry__

    __graft_entry__.build()
    T, K, N = (int(v) for v in args.linear.split(","))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    seed = 0
    x = torch.empty((T, K), dtype=torch.int16, device=dev)
    synth.dev_normal_bf16(seed, synth.S_X, rank * T * K, x, 1.0)
    x = x.view(torch.bfloat16)
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    cs, ss = synth._mx_streams("w2")
    synth.dev_uniform_bytes(seed, cs, 0, codes)
    raw = torch.empty((N, K // 32), dtype=torch.uint8, device=dev)
    synth.dev_e8m0_scales(seed, ss, 0, N, K // 32, raw)
    sf = torch.empty(fm.packed_scales_bytes(1, N, K // 32, fm.MXFP4), dtype=torch.uint8, device=dev)
    fm.pack_scales(raw.data_ptr(), sf.data_ptr(), 1, N, K // 32, fm.MXFP4, s)
    out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    n = fm.linear_workspace_size(fm.MXFP4, T, K, N)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def call(xp=None):
        fm.linear(fm.MXFP4, T, K, N, (xp if xp is not None else x).data_ptr(), codes.data_ptr(), sf.data_ptr(),
                  None, out.data_ptr(), ws.data_ptr(), n, s)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        call()
    torch.cuda.synchronize()
    assert fm.get_status(ws.data_ptr(), s) == (0, 0)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        time.sleep(0.3)
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        time.sleep(0.3)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    # end to end: host x in, host out back, every step
    xh = x.cpu().pin_memory()
    oh = torch.empty((T, N), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(x)
    e2e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for i in range(20):
        flush.fill_(float(i))
        e2e[i][0].record(stream)
        xd.copy_(xh, non_blocking=True)
        call(xd)
        oh.copy_(out, non_blocking=True)
        e2e[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in e2e)
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], world, dev)
    if rank != 0:
        return
    flops = 2.0 * T * K * N
    peaks = measured_peaks()
    fp4_peak = 6 * peaks["bf16_tflops"]
    tflops = whole_job_rate(flops, world, ms) / 1e12
    # CPU baseline: the oracle on a bounded sample of rows
    from oracle import linear as LIN
    from oracle.formats import unpack_nibbles
    rows = 4
    xs = x[:rows].float().cpu().numpy().astype(np.float64)
    wc, wsc = unpack_nibbles(codes.cpu().numpy()), raw.cpu().numpy()
    t0 = time.perf_counter()
    LIN.linear_forward(xs, wc, wsc, "mxfp4")
    cpu_s = time.perf_counter() - t0
    line = {
        "metric": "dense block-scaled FP4 linear TFLOP/s", "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp4", "data": "synthetic (seeded; drawn on the device)",
        "config": {"workload": f"dense MXFP4 linear T={T} K={K} N={N} (bf16 in, on-the-fly activation quantisation, "
                               f"bf16 out)", "l2": "flushed between steps (256 MiB write, untimed)"},
        "clocks": clk.summary(),
        "e2e": {"value": whole_job_rate(flops, world, e2e_ms) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": T * K * 2, "d2h_bytes_per_step": T * N * 2},
        "gpu_launches": 5 * args.steps,
        "roofline": {"bound": "tensor", "kernel": "moe_gemm_kernel<down> (one expert)", "achieved": tflops / world,
                     "peak": fp4_peak, "unit": "TFLOP/s", "frac": tflops / world / fp4_peak, "traffic": None,
                     "peak_source": peaks["source"] + " bf16 x 6 (nominal dense FP4 / bf16)"},
        "cpu_baseline": {"value": 2.0 * rows * K * N / cpu_s / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": f"{rows} rows of the same shape, FP64 numpy"},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ roofline
def fp4_peak_tflops(peaks: dict) -> float:
    """Dense FP4 tensor peak: the measured bf16 peak times the nominal dense
    FP4 / bf16 ratio 13.5 / 2.25 = 6."""
    return 6.0 * peaks["bf16_tflops"]


def roofline(nbytes: float, flops: float, ms: float, peaks: dict) -> dict:
    """The slower of the two rooflines for work that moves `nbytes` and does
    `flops` in `ms`: time at the measured HBM bandwidth against time at the
    dense FP4 tensor peak; the bound is the larger, and the fraction is that
    time over the measured one (achieved over peak in the bound's unit)."""
    t_b = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    t_f = flops / (fp4_peak_tflops(peaks) * 1e12) * 1e3
    if t_b >= t_f:
        rec = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        rec = {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": fp4_peak_tflops(peaks),
               "unit": "TFLOP/s"}
    rec.update({"frac": rec["achieved"] / rec["peak"], "ms": ms, "roofline_ms": max(t_b, t_f), "bytes_ms": t_b,
                "flops_ms": t_f, "algorithmic_bytes": nbytes, "flops": flops})
    return rec


def layer_work(H: int, I: int, E: int, T: int, fmt: str, mode: str, touched: int, routes: int) -> dict:
    """Algorithmic bytes and FLOPs of one layer call and of its two expert
    GEMMs: the GEMMs' bytes as algorithmic_bytes gives them, plus the router
    (its weights and x, bf16) and the bf16 output for the layer.  FLOPs: 2 *
    3 * I * H per route (gate, up, down)."""
    gu, dn = algorithmic_bytes(H, I, fmt, mode, touched, routes, T)
    return {"gateup": (gu, 2.0 * 2 * I * H * routes), "down": (dn, 2.0 * H * I * routes),
            "layer": (gu + dn + E * H * 2 + 2 * T * H * 2, 2.0 * 3 * I * H * routes)}


# ------------------------------------------------------------------ GPU arm
def _events(torch, stream, n):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record(stream)
    return evs


def measure_layer(torch, fm, layer, x, fwd, steps: int, warmup: int, stream, flush, stage_runs: int = 50,
                  clock_gpu: int | None = None, bracket=None):
    """Times one layer configuration: warm-up calls, `steps` replays of one
    forward captured in a CUDA graph (L2 flushed before each, untimed), and
    eager forwards with events between the stages.  `bracket` (nullable) runs
    right before and right after the timed replays (the ranks' barrier).
    Returns per-step times, stage times, the GEMMs' times, touched experts
    and routes."""
    d = layer.dims
    out = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=x.device)
    s = stream.cuda_stream
    for _ in range(warmup):
        flush.fill_(1.0)
        fwd(x, out)
    torch.cuda.synchronize()
    wsbuf = layer.emu_ws if getattr(layer, "emu_ws", None) is not None and fwd == getattr(layer, "forward_emulated",
                                                                                          None) else layer.ws
    st, _ = fm.get_status(wsbuf.data_ptr(), s)
    if st != 0:
        raise RuntimeError(f"device status {fm.STATUS.get(st, st)}")
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        fwd(x, out)
    torch.cuda.synchronize()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    ev = [_events(torch, stream, 2) for _ in range(steps)]
    torch.cuda.synchronize()
    if bracket:
        bracket()
    sampler = ClockSampler(clock_gpu) if clock_gpu is not None else None
    if sampler:
        sampler.__enter__()
        time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if bracket:
        bracket()
    if sampler:
        time.sleep(0.3)
        sampler.__exit__(None, None, None)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    gev = _events(torch, stream, 8)
    dbg = fm.Debug()
    for i, e in enumerate(gev):
        dbg.events[i] = e.cuda_event
    runs, gu_ms, dn_ms = [], [], []
    for i in range(min(steps, stage_runs)):
        flush.fill_(float(i))
        torch.cuda.synchronize()
        fwd(x, out, debug=dbg)
        torch.cuda.synchronize()
        runs.append([gev[j].elapsed_time(gev[j + 1]) for j in range(7)])
        gu_ms.append(gev[4].elapsed_time(gev[5]))
        dn_ms.append(gev[5].elapsed_time(gev[6]))
    ne = d.E + d.n_shared
    off = layer.layout.expert_count
    count = wsbuf[off:off + 4 * ne].view(torch.int32).cpu().numpy()
    return {"step_ms": step_ms, "ms": statistics.mean(step_ms), "wall_s": wall, "graph": graph, "out": out,
            "stages_ms": {fm.STAGES[j]: statistics.mean(r[j] for r in runs) for j in range(7)},
            "gu_ms": statistics.mean(gu_ms), "dn_ms": statistics.mean(dn_ms),
            "touched": int((count > 0).sum()), "routes": int(count.sum()),
            "clocks": sampler.summary() if sampler else None}


def config_record(cfg, layer, m: dict, peaks: dict, mode: str = "a4w4", w8a8: bool = False,
                  emulate: bool = False) -> dict:
    """One workload's sub-record: throughput, stage times and the rooflines
    of the layer and of its two expert GEMMs."""
    d = layer.dims
    work = layer_work(d.H, d.I, d.E, d.T, cfg.fmt, mode, m["touched"], m["routes"])
    kern = {"gateup": roofline(*work["gateup"], m["gu_ms"], peaks), "down": roofline(*work["down"], m["dn_ms"], peaks)}
    ratios = profiled_ratios(cfg.name)
    for k, r in kern.items():
        r["traffic"] = r["algorithmic_bytes"] * ratios[k] if ratios else None
        if ratios:
            r["traffic_source"] = f"ncu DRAM bytes / algorithmic bytes of {ratios['from']}, times this launch's"
    dominant = max(kern, key=lambda k: kern[k]["ms"])
    return {"workload": cfg_label(cfg, w8a8, emulate), "ms_per_step": m["ms"], "tokens_per_s": d.T / (m["ms"] * 1e-3),
            "tflops": work["layer"][1] / (m["ms"] * 1e-3) / 1e12, "touched_experts": m["touched"],
            "routes": m["routes"], "stages_ms": m["stages_ms"], "roofline": roofline(*work["layer"], m["ms"], peaks),
            "kernels": kern, "dominant_kernel": dominant, "clocks": m["clocks"],
            "launch": "one forward captured in a CUDA graph, replayed per step; L2 flushed between steps"}


# the workloads measured beside the headline one, in this order
OTHER_CONFIGS = ("kimi_prefill", "deepseek_nvfp4", "skewed_shared", "tiny")


def other_configs(args, torch, fm, dev, stream, flush, peaks, local_rank):
    """Every other workload of the layer (and the MXFP4 -> FP8 conversion of
    the skewed workload's experts), one after another on this GPU.  The
    384-expert MXFP4 layers share one set of expert tensors."""
    import synth
    from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
    cfgs = synth.configs()
    steps = max(5, min(args.steps, 30))
    recs = {}
    base = MoELayer.synthetic(cfgs["skewed_shared"], device=dev)  # 384 experts + the shared one
    for name in OTHER_CONFIGS:
        cfg = cfgs[name]
        if cfg.fmt == "mxfp4" and (cfg.E, cfg.H, cfg.I) == (base.dims.E, base.dims.H, base.dims.I):
            layer = base.variant(cfg)
        else:
            layer = MoELayer.synthetic(cfg, device=dev)
        x = layer.synthetic_x()
        m = measure_layer(torch, fm, layer, x, layer.forward, steps, args.warmup, stream, flush, stage_runs=20,
                          clock_gpu=local_rank)
        recs[name] = config_record(cfg, layer, m, peaks)
        if name == "tiny":
            recs[name]["us_per_step"] = m["ms"] * 1e3
        del layer, x, m
        torch.cuda.synchronize()
    recs["conversion"] = time_conversion(base, peaks, stream)
    del base
    torch.cuda.empty_cache()
    return recs


def gpu_arm(args, cfg, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import block_scaled_fp4_sigmoid_gb300 as fm
    from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    layer = MoELayer.synthetic(cfg, device=dev)
    if args.w8a8:
        from block_scaled_fp4_sigmoid_gb300.layer import W8A8Layer
        if cfg.fmt != "mxfp4":
            raise SystemExit("--w8a8 converts MXFP4 experts")
        mx = layer
        layer = W8A8Layer(mx)
        del mx.w13, mx.w2, mx.w13_t, mx.w2_t  # the converted copies are what the W8A8 layer reads
        torch.cuda.empty_cache()
    # each rank runs its own batch: tokens rank*T .. (rank+1)*T of the stream
    x = layer.synthetic_x(*rank_token_range(rank, cfg.T))
    if args.emulate and cfg.fmt != "nvfp4":
        raise SystemExit("--emulate runs NVFP4 layers")
    fwd = layer.forward_emulated if args.emulate else layer.forward
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    steps = args.steps

    # eager calls (host launch overhead included), for context
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup):
        flush.fill_(1.0)
        fwd(x, out)
    eager_n = min(steps, 100)
    eager_ev = [_events(torch, stream, 2) for _ in range(eager_n)]
    torch.cuda.synchronize()
    for i in range(eager_n):
        flush.fill_(float(i))
        eager_ev[i][0].record(stream)
        fwd(x, out)
        eager_ev[i][1].record(stream)
    torch.cuda.synchronize()
    eager_ms = statistics.mean(a.elapsed_time(b) for a, b in eager_ev)

    # the timed steps: graph replays bracketed by a barrier on every rank
    def bracket():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    m = measure_layer(torch, fm, layer, x, fwd, steps, args.warmup, stream, flush, clock_gpu=local_rank,
                      bracket=bracket)
    ms = m["ms"]

    # end to end through the public API with host buffers
    x_host = x.cpu().pin_memory()
    out_host = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    e2e_steps = max(10, min(steps, 200))
    for _ in range(3):
        x_dev.copy_(x_host, non_blocking=True)
        fwd(x_dev, out)
        out_host.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e2e_ev = [_events(torch, stream, 2) for _ in range(e2e_steps)]
    torch.cuda.synchronize()
    for i in range(e2e_steps):
        flush.fill_(float(i))
        e2e_ev[i][0].record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        fwd(x_dev, out)
        out_host.copy_(out, non_blocking=True)
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in e2e_ev)

    touched, routes = m["touched"], m["routes"]
    wpe = layer.weight_bytes_per_expert()
    d = layer.dims
    mode = "emulate" if args.emulate else "w8a8" if args.w8a8 else "a4w4"
    work = layer_work(d.H, d.I, d.E, d.T, cfg.fmt, mode, touched, routes)
    ms_max, e2e_max, gu_max, dn_max = max_over_ranks([ms, e2e_ms, m["gu_ms"], m["dn_ms"]], world, dev)
    head = {"clocks": m["clocks"], "stages_ms": m["stages_ms"], "wall_s": m["wall_s"]}
    del m
    peaks = measured_peaks()
    # the remaining workloads (default run, one GPU): measured after the headline
    others = None
    if world == 1 and not (args.w8a8 or args.emulate or args.no_configs or args.experts or args.tokens):
        others = other_configs(args, torch, fm, dev, stream, flush, peaks, local_rank)
    if rank != 0:
        return
    gu = roofline(*work["gateup"], gu_max, peaks)
    dn = roofline(*work["down"], dn_max, peaks)
    dom_name, dom = ("gate/up grouped GEMM", gu) if gu["ms"] >= dn["ms"] else ("down grouped GEMM", dn)
    traffic = profiled_traffic(cfg.name + ("_w8a8" if args.w8a8 else "")) if dom is gu else None
    # few tokens: front end (routing, plan, x quantisation), gate/up, down,
    # finalise; else router, top-k, plan, scatter, gather, gate/up, down, finalise
    if args.w8a8:  # router, top-k, plan, scatter, x quantisation, gate/up, h quantisation, down, finalise
        launches_per_step = 9
    elif args.emulate:  # + weight dequantisation (w13, w2, shared), amax, x and h QDQ
        launches_per_step = 11 + 2 * cfg.n_shared
    elif cfg.fmt == "mxfp4":
        launches_per_step = 4 if cfg.T <= 16 else 8
    else:
        launches_per_step = 10
    conversion = None
    if args.conversion and not args.w8a8:
        conversion = time_conversion(layer, peaks, stream)
    elif others is not None:
        conversion = others.pop("conversion")
    # CPU baseline: the oracle on the whole step when that is a bounded
    # amount of work (a decode-sized A4W4 layer: ~15 s on 16 cores), else on
    # a bounded sample of routes
    whole = (args.cpu_routes is None and cfg.T <= 16 and not (args.w8a8 or args.emulate)
             and cfg.name == args.config)
    if whole:
        full = oracle_full_layer(cfg.name)
        cpu_s, cpu_tok = full["route_s"] + full["expert_s"], float(cfg.T)
        cpu_sample = (f"the whole step: {cfg.T} tokens, {full['routes_done']} routes over all "
                      f"{full['experts_done']} touched experts, FP64 numpy")
    else:
        n_routes = 16 if args.cpu_routes is None else args.cpu_routes
        cpu_s, cpu_tok = (oracle_route_sample(args.config, n_routes, w8a8=args.w8a8, emulate=args.emulate)
                          if n_routes > 0 else (float("nan"), 0.0))
        cpu_sample = f"{n_routes} routes ({cpu_tok:g} tokens) of the same workload, FP64 numpy"
    line = {
        "metric": METRIC,
        "value": whole_job_rate(cfg.T, world, ms_max),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if args.w8a8 else "bf16" if args.emulate else ("mxfp4" if cfg.fmt == "mxfp4" else "nvfp4"),
        "data": "synthetic (seeded; weights drawn on the device)",
        "config": {"workload": cfg_label(cfg, args.w8a8, args.emulate), "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "launch": "one fp4moe_forward captured in a CUDA graph, replayed per step",
                   "l2": "flushed between steps (256 MiB write, untimed)", "touched_experts": touched,
                   "routes": routes},
        "clocks": head["clocks"],
        "e2e": {"value": whole_job_rate(cfg.T, world, e2e_max), "unit": "tokens/s",
                "h2d_bytes_per_step": int(x.numel() * 2), "d2h_bytes_per_step": int(out.numel() * 2)},
        "gpu_launches": launches_per_step * steps,
        "roofline": {"bound": dom["bound"], "kernel": dom_name, "achieved": dom["achieved"], "peak": dom["peak"],
                     "unit": dom["unit"], "frac": dom["frac"], "traffic": traffic,
                     "algorithmic_bytes": dom["algorithmic_bytes"], "flops": dom["flops"],
                     "peak_source": peaks["source"] + ("" if dom["bound"] == "hbm" else
                                                       " bf16 x 6 (nominal dense FP4 / bf16)")},
        "step": {"weight_stream_gbs": (touched * wpe) / (ms_max * 1e-3) / 1e9,
                 "weight_stream_frac": (touched * wpe) / (ms_max * 1e-3) / 1e9 / peaks["hbm_gbs"],
                 "tflops": work["layer"][1] / (ms_max * 1e-3) / 1e12, "stages_ms": head["stages_ms"],
                 "layer_roofline": roofline(*work["layer"], ms_max, peaks), "kernels": {"gateup": gu, "down": dn},
                 "wall_s": head["wall_s"], "eager_ms_per_step": eager_ms},
        "cpu_baseline": {"value": cpu_tok / cpu_s, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": cpu_sample},
        "context": "pages: 1.43 ms per MoE layer call at T=8 on one Gaudi 2 card holding 48 of 384 experts",
        "conversion": conversion,
        "configs": others,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="kimi_decode")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-routes", type=int, default=None)
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (smaller device footprint for profiler captures)")
    ap.add_argument("--tokens", type=int, default=None, help="override T")
    ap.add_argument("--linear", default=None, metavar="T,K,N",
                    help="time the dense block-scaled FP4 linear (fp4moe_linear) on this shape instead")
    ap.add_argument("--emulate", action="store_true",
                    help="NVFP4 workloads: the emulation mode (fp4moe_forward_nvfp4_emulated)")
    ap.add_argument("--w8a8", action="store_true",
                    help="the W8A8 layer: experts exactly converted to FP8 per channel, FP8 per-token activations")
    ap.add_argument("--conversion", action="store_true",
                    help="also time the MXFP4 -> FP8 conversion of all routed expert rows")
    ap.add_argument("--cpu-full", default=None, metavar="CONFIG[,MAX_EXPERTS]",
                    help="time the FP64 oracle over a whole workload on the host cores (no GPU) and print a JSON line")
    ap.add_argument("--cpu-conv-rows", type=int, default=0,
                    help="with --cpu-full: also time the conversion oracle on this many expert rows")
    ap.add_argument("--cpu-conv-full", action="store_true",
                    help="time the conversion oracle over every routed expert row of the skewed layer on all host "
                         "cores (no GPU) and print a JSON line")
    ap.add_argument("--no-configs", action="store_true",
                    help="time the chosen workload only (by default a one-GPU run also measures every other "
                         "workload and the conversion, in the line's configs object)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.cpu_conv_full:
        print(json.dumps(oracle_full_conversion()), flush=True)
        return
    if args.cpu_full:
        name, _, mx = args.cpu_full.partition(",")
        print(json.dumps(oracle_full_layer(name, int(mx) if mx else None, args.cpu_conv_rows)), flush=True)
        return
    import synth
    from dataclasses import replace
    cfg = synth.configs()[args.config]
    if args.experts:
        cfg = replace(cfg, E=args.experts, name=f"{cfg.name}_e{args.experts}")
    if args.tokens:
        cfg = replace(cfg, T=args.tokens, name=f"{cfg.name}_t{args.tokens}")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, cfg, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        if args.linear:
            linear_arm(args, rank, world, local_rank)
        else:
            gpu_arm(args, cfg, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
