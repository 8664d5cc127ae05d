"""Benchmark: MoE expert-layer backward on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one full backward pass (routing metadata, gathers / quantisation, the four grouped GEMMs,
dx scatter-sum, ds, bias sums) over one synthetic batch of the named workload.  `value` is useful
tensor FLOP/s (12*T*K*H*I per MoE step, 4*M*N*K per dense step; padding rows and quantisation
excluded) with inputs resident in HBM; `e2e` is the same metric with the step's activations copied
from pinned host memory and dx/ds copied back inside the timed region.  With N > 1 (torchrun), every
rank runs an independent replica (the pass has no exchange step), value = sum over ranks / max time.
`--impl reference` times the CPU float64 oracle on a bounded sample of the same workload.
The headline timed region records nothing but its two events; the per-stage times (stage_ms, the
roofline's dominant kernel) come from a second pass of the same steps.  The default run then times
the other workloads with a throughput bar (fine-grained BF16, many-expert MXFP8, the dense 4096^3
MXFP8 linear backward) the same way, under `workloads`.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "imbalanced_mxfp8"
METRIC_MOE = "MoE-backward TFLOP/s (BF16, MXFP8) & % of tensor peak; tokens/s"
METRIC_LINEAR = "dense MXFP8 linear-backward TFLOP/s & % of tensor peak"
FALLBACK_PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)
L2_BYTES_GB300 = 126 * 2 ** 20 + 2 ** 19   # without a device to ask (the timed arm asks its own)
FP8_OVER_BF16 = 2.0   # nominal dense ratio 4.5 / 2.25 PFLOP/s


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha():
    """Hash of the kernel sources' code (comments and whitespace dropped, so that an edit of a comment
    does not retire the ncu counters recorded for that code)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_expert_layer_routing_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            h.update(name.encode() + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_mxfp8_peak():
    """MXFP8 dense GEMM peak measured through cuBLAS on this machine (`bench.py --measure-peaks`),
    from a committed summary line `mxfp8_peak burst_tflops=.. sustained_tflops=..`."""
    pdir = os.path.join(ROOT, "profiles")
    pat = re.compile(r"mxfp8_peak burst_tflops=([0-9.]+) sustained_tflops=([0-9.]+)")
    if os.path.isdir(pdir):
        for name in sorted(os.listdir(pdir)):
            if name.endswith((".md", ".txt")):
                for line in open(os.path.join(pdir, name)):
                    m = pat.search(line)
                    if m:
                        return float(m.group(1)), float(m.group(2))
    return None


def measure_peaks():
    """Dense 8192^3 GEMMs through the vendor library: bf16 (torch.matmul) and MXFP8
    (torch._scaled_mm, e4m3 operands, E8M0 scales per 32 K-elements), burst and ~3 s sustained."""
    import torch
    M = N = K = 8192
    dev = "cuda"
    res = {}

    def timed(f, secs):
        for _ in range(5):
            f()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = 1e30
        for _ in range(10):
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        n, t0 = 0, time.time()
        e0.record()
        while time.time() - t0 < secs:
            f()
            n += 1
        e1.record()
        torch.cuda.synchronize()
        return 2.0 * M * N * K / (best * 1e-3) / 1e12, 2.0 * M * N * K * n / (e0.elapsed_time(e1) * 1e-3) / 1e12

    a = torch.randn(M, K, device=dev, dtype=torch.bfloat16)
    b = torch.randn(N, K, device=dev, dtype=torch.bfloat16)
    res["bf16_tflops_burst"], res["bf16_tflops_sustained"] = timed(lambda: a @ b.t(), 3.0)
    try:
        a8, b8 = a.to(torch.float8_e4m3fn), b.to(torch.float8_e4m3fn)
        ns = ((M + 127) // 128 * 128) * ((K // 32 + 3) // 4 * 4)
        sa = torch.full((ns,), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
        sb = torch.full((ns,), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
        f = lambda: torch._scaled_mm(a8, b8.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)  # noqa: E731
        res["mxfp8_tflops_burst"], res["mxfp8_tflops_sustained"] = timed(f, 3.0)
    except Exception as ex:  # library without block-scaled FP8 support
        res["mxfp8_error"] = repr(ex)[:300]
    res["how"] = "8192^3 GEMMs, CUDA events, best of 10 (burst) and back to back for 3 s (sustained)"
    print(json.dumps(res), flush=True)
    if "mxfp8_tflops_burst" in res:
        print(f"mxfp8_peak burst_tflops={res['mxfp8_tflops_burst']:.1f} "
              f"sustained_tflops={res['mxfp8_tflops_sustained']:.1f}", flush=True)


def recorded_traffic(workload: str, stage: str):
    """DRAM bytes per launch of a stage from a committed ncu summary, only if it was captured on
    the current kernel sources (a line `traffic workload=.. stage=.. bytes_per_launch=.. source_sha=..`)."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    sha = source_sha()
    pat = re.compile(r"traffic workload=(\S+) stage=(\S+) bytes_per_launch=(\d+) source_sha=(\w+)")
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        for line in open(os.path.join(pdir, name)):
            m = pat.search(line)
            if m and m.group(1) == workload and m.group(2) == stage and m.group(4) == sha:
                return int(m.group(3))
    return None


def workload_config(cfg, is_linear, world):
    if is_linear:
        return dict(workload=cfg.name, M=cfg.M, N=cfg.N, K=cfg.K, precision="mxfp8 e5m2",
                    parallelism=f"replicas x{world}")
    return dict(workload=cfg.name, T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, top_k=cfg.K, block_size=cfg.block_size,
                precision="mxfp8 (e4m3 weights, e5m2 activations, E8M0 scales)" if cfg.precision == 1 else "bf16",
                affinity="on_I" if cfg.affinity == 1 else "on_H", bias=cfg.bias, parallelism=f"replicas x{world}")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        if not sm:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["unsampled"], samples=0)
        sm_sorted = sorted(sm)
        busy = [v for v in sm_sorted if v > 0.5 * max(sm_sorted)] or sm_sorted
        return dict(sm_mhz=busy[len(busy) // 2], sm_max_mhz=max(mx), reasons=sorted(reasons), samples=len(sm))


# ---------------------------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------------------------
def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v: float, world: int) -> float:
    """Max over ranks (the slowest rank's time defines a step)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------------
# CPU oracle sample (the baseline, never the product path)
# ---------------------------------------------------------------------------------------------
def oracle_sample_moe(inp, target_rows: int):
    """The non-empty expert whose load is closest to target_rows, with all its tokens (the oracle's
    cost is dominated per expert by its weight quantisation and per row by the four contractions)."""
    import numpy as np
    from oracle import moe as om
    from oracle import sample as osm
    cfg = inp.cfg
    ids = inp.ids.cpu().numpy()
    counts = np.bincount(ids.reshape(-1)[(ids.reshape(-1) >= 0) & (ids.reshape(-1) < cfg.E)], minlength=cfg.E)
    nz = np.nonzero(counts)[0]
    e = int(nz[np.argmin(np.abs(counts[nz] - target_rows))])
    rows = int(counts[e])
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    sub = osm.subproblem(cpu(inp.x), cpu(inp.dout), cpu(inp.W1), cpu(inp.W2), inp.s.cpu().numpy(), ids,
                         cpu(inp.ckpt), cfg.block_size, experts=[e], b2=cpu(inp.b2))

    def run():
        if cfg.precision == 1:
            om.moe_backward_mxfp8(sub["x"], sub["dout"], sub["W1"], sub["W2"], sub["s"], sub["ids"], sub["h"],
                                  affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w)
        else:
            om.moe_backward(sub["x"], sub["dout"], sub["W1"], sub["W2"], sub["s"], sub["ids"], sub["h"],
                            b2=sub["b2"], with_bias=cfg.bias)

    flops = 12.0 * rows * cfg.H * cfg.I
    desc = f"expert {e} with {rows} routed rows (all its tokens), all of its outputs"
    return run, flops, desc


def oracle_sample_linear(inp, rows: int):
    import torch
    from oracle import linear as ol
    dY = inp.dY[:rows].cpu()
    X = inp.X[:rows].cpu()
    W = inp.W.cpu()

    def run():
        ol.linear_backward_mxfp8(dY, W, X)

    flops = 4.0 * rows * inp.cfg.N * inp.cfg.K
    desc = f"first {rows} of {inp.cfg.M} rows of dY and X (dX rows and a dW partial over them)"
    return run, flops, desc


def time_oracle(run, flops, max_s):
    t0 = time.perf_counter()
    n = 0
    while True:
        run()
        n += 1
        if time.perf_counter() - t0 > max_s or n >= 50:
            break
    dt = (time.perf_counter() - t0) / n
    return flops / dt / 1e12, n


# ---------------------------------------------------------------------------------------------
def recompute_row(mb, cfg, inp, kw, steps, stream, peak_tf, dev):
    """The whole backward with the gate/up pre-activations recomputed by the forward grouped GEMM G0
    (act_src RECOMPUTE) instead of read from the checkpoint: G0's own rate against the tensor peak
    (4*T*K*H*I FLOPs, not counted as useful) and the step time."""
    import torch
    op = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size, precision=cfg.precision,
                   affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w, has_bias=cfg.bias,
                   act_src=mb.ACT_RECOMPUTE, device=dev)
    kw = {k: v for k, v in kw.items() if k != "ckpt"}
    W1t = inp.W1.transpose(1, 2).contiguous()
    if cfg.precision == mb.PREC_MXFP8:
        kw["W1t_q"], kw["W1t_sf"] = mb.quantize_weights(W1t, cfg.fp8_w)
        del W1t
    else:
        kw["W1t"] = W1t
    kw["b1"] = inp.b1 if cfg.bias else None
    op.bind(**kw)
    for _ in range(3):
        op.run()
    torch.cuda.synchronize()
    if int(op.status.item()) != 0:
        raise SystemExit(f"device status {int(op.status.item())} (recompute)")
    mb.profile_enable(True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        op.run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    st, n = mb.profile_read()
    mb.profile_enable(False)
    g0 = st["G0_recompute_h"] / max(n, 1)
    g0_flops = 4.0 * cfg.T * cfg.K * cfg.H * cfg.I
    return dict(ms_per_step=ms, useful_tflops=cfg.useful_flops() / (ms * 1e-3) / 1e12,
                g0_ms=g0, g0_tflops=g0_flops / (g0 * 1e-3) / 1e12, g0_frac=g0_flops / (g0 * 1e-3) / 1e12 / peak_tf,
                g0_flops_per_launch=g0_flops, bound="tensor",
                note="G0 recomputes h = x_g W1_e (+ b1_e) into the block checkpoint layout; its FLOPs are "
                     "excluded from useful_tflops")


def resident_input_bytes(cfg) -> int:
    """Bytes of the inputs a step reads from HBM as the timed step holds them: dY, W, X (bf16) for the
    dense case; x, dout, s, ids, the [N,2,I,B] checkpoint, b2 and the weights (bf16, or MXFP8 codes
    with one scale byte per 32) for the MoE backward."""
    from moe_expert_layer_routing_gb300.inputs import LinearConfig, num_blocks_bound
    if isinstance(cfg, LinearConfig):
        return 2 * (cfg.M * cfg.N + cfg.N * cfg.K + cfg.M * cfg.K)
    T, H, I, E, K, B = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.block_size
    w = E * H * 2 * I + E * I * H
    wbytes = w + w // 32 if cfg.precision == 1 else 2 * w
    return (2 * 2 * T * H + 2 * 4 * T * K + 2 * num_blocks_bound(T, K, E, B) * 2 * I * B
            + (2 * E * H if cfg.bias else 0) + wbytes)


def l2_note(in_bytes: int, l2_bytes: int) -> str:
    """How the timed steps keep L2 from serving the inputs (recorded in the JSON line's config)."""
    if in_bytes <= l2_bytes:
        return (f"L2 flushed before each timed step ({in_bytes / 1e9:.2f} GB resident inputs <= "
                f"{l2_bytes / 1e9:.2f} GB L2: a {2 * l2_bytes / 1e9:.2f} GB buffer written between steps, "
                f"each step timed by its own events)")
    return f"inputs larger than L2 ({in_bytes / 1e9:.2f} GB resident inputs > {l2_bytes / 1e9:.2f} GB L2)"


def device_l2_bytes() -> int:
    import torch
    if torch.cuda.is_available():
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    return L2_BYTES_GB300


def setup_problem(mb, cfg, dev):
    """Inputs, device buffers and the step of one workload (untimed); MXFP8 weights are quantised
    once here, outside any timed region."""
    from moe_expert_layer_routing_gb300.inputs import LinearConfig, make_linear_inputs, make_moe_inputs
    if isinstance(cfg, LinearConfig):
        inp = make_linear_inputs(cfg, device=dev)
        op = mb.LinearBwd(cfg.M, cfg.N, cfg.K, mb.PREC_MXFP8, cfg.fp8, dev)
        return dict(is_linear=True, inp=inp, op=op, kw=None, step=lambda: op.run(inp.dY, inp.W, inp.X),
                    flops=float(cfg.useful_flops()), tokens=cfg.M, prec=mb.PREC_MXFP8,
                    in_bytes=resident_input_bytes(cfg))
    inp = make_moe_inputs(cfg, device=dev)
    op = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size,
                   precision=cfg.precision, affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w,
                   has_bias=cfg.bias, device=dev)
    kw = dict(x=inp.x, dout=inp.dout, s=inp.s, ids=inp.ids, ckpt=inp.ckpt, b2=inp.b2 if cfg.bias else None)
    if cfg.precision == mb.PREC_MXFP8:
        W1_q, W1_sf = mb.quantize_weights(inp.W1, cfg.fp8_w)
        W2_q, W2_sf = mb.quantize_weights(inp.W2, cfg.fp8_w)
        kw.update(W1_q=W1_q, W1_sf=W1_sf, W2_q=W2_q, W2_sf=W2_sf)
    else:
        kw.update(W1=inp.W1, W2=inp.W2)
    op.bind(**kw)
    return dict(is_linear=False, inp=inp, op=op, kw=kw, step=lambda: op.run(), flops=float(cfg.useful_flops()),
                tokens=cfg.T, prec=cfg.precision, in_bytes=resident_input_bytes(cfg))


def time_problem(mb, P, steps, warmup, world, local, stream):
    """Warm-up, then `steps` timed steps with nothing else recorded on the stream (the headline time,
    CUDA events, max over ranks, clocks sampled meanwhile), then -- for the MoE backward -- a second
    pass of the same steps with the library's per-stage events on (stage_ms, and that pass's own
    time to show the events cost nothing measurable)."""
    import torch
    step = P["step"]
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if not P["is_linear"]:
        st0 = int(P["op"].status.item())
        if st0 != 0:
            raise SystemExit(f"device status {st0} after warm-up")
    # resident inputs larger than L2: back-to-back steps; otherwise L2 is flushed before every step (a
    # buffer of twice its size written on the stream) and each step is timed by its own pair of events
    l2_bytes = device_l2_bytes()
    flush = None
    if P["in_bytes"] <= l2_bytes:
        flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=torch.cuda.current_device())
    launches0 = mb.kernel_launches()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        if flush is None:
            ev0.record(stream)
            for _ in range(steps):
                step()
            ev1.record(stream)
        else:
            for i in range(steps):
                flush.fill_(i & 255)
                evs[i][0].record(stream)
                step()
                evs[i][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    local_ms = (ev0.elapsed_time(ev1) if flush is None else sum(a.elapsed_time(b) for a, b in evs)) / steps
    ms = allreduce_max(local_ms, world)
    launches = mb.kernel_launches() - launches0
    del flush
    out = dict(ms=ms, launches=launches, clocks=clk.summary(), stages=None, profiled_ms=None,
               l2=l2_note(P["in_bytes"], l2_bytes))
    if not P["is_linear"]:
        mb.profile_enable(True)
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        stages, ncalls = mb.profile_read()
        mb.profile_enable(False)
        out["stages"] = {k: v / max(ncalls, 1) for k, v in stages.items()}
        out["profiled_ms"] = ev0.elapsed_time(ev1) / steps
        if int(P["op"].status.item()) != 0:
            raise SystemExit(f"device status {int(P['op'].status.item())} after the timed steps")
    return out


def dominant_roofline(cfg, stages, per_gpu_value, prec, peak_tf, peak_src):
    """Roofline line of the dominant kernel: the grouped-GEMM stage with the largest time (its
    useful FLOPs over its average duration from the stage events), or the whole dense step."""
    if stages is None:
        return dict(bound="tensor", kernel="linear_bwd (dX and dW GEMMs + quantisation)", achieved=per_gpu_value,
                    peak=peak_tf, unit="TFLOP/s", frac=per_gpu_value / peak_tf, traffic=None,
                    peak_source=f"{peak_src} bf16 burst x2 (nominal fp8/bf16)")
    H, I, TK = cfg.H, cfg.I, cfg.T * cfg.K
    stage_flops = {"G1_dA_dswiglu": 2.0 * TK * H * I, "G3_dW2": 2.0 * TK * H * I,
                   "G2_dx_expanded": 4.0 * TK * H * I, "G4_dW1": 4.0 * TK * H * I}
    dom = max(stage_flops, key=lambda k: stages[k])
    achieved = stage_flops[dom] / (stages[dom] * 1e-3) / 1e12
    return dict(bound="tensor", kernel=dom, achieved=achieved, peak=peak_tf, unit="TFLOP/s",
                frac=achieved / peak_tf, traffic=recorded_traffic(cfg.name, dom),
                algorithmic_flops_per_launch=stage_flops[dom],
                per_stage_frac={k: stage_flops[k] / (stages[k] * 1e-3) / 1e12 / peak_tf for k in stage_flops},
                peak_source=f"{peak_src} bf16 burst" + (" x2 (nominal fp8/bf16)" if prec == 1 else ""),
                timing="stage events of a second pass of the same steps (profiled_ms_per_step)")


EXTRA_WORKLOADS = ("finegrained_bf16", "manyexpert_mxfp8", "dense_mxfp8_4096")


def extra_workloads(mb, args, world, local, stream, peaks, peak_src, dev):
    """The other configurations with a throughput bar, each timed like the headline (device-resident,
    unprofiled timed region, stage events in a second pass, own clock record)."""
    import torch
    from moe_expert_layer_routing_gb300.inputs import CONFIGS
    lib_peak = recorded_mxfp8_peak()
    out = {}
    for name in EXTRA_WORKLOADS:
        if name == args.workload:
            continue
        cfg = CONFIGS[name]
        P = setup_problem(mb, cfg, dev)
        T = time_problem(mb, P, args.steps, args.warmup, world, local, stream)
        value = P["flops"] * world / (T["ms"] * 1e-3) / 1e12
        peak_tf = peaks["bf16_tflops"] * (FP8_OVER_BF16 if P["prec"] == 1 else 1.0)
        rl = dominant_roofline(cfg, T["stages"], value / world, P["prec"], peak_tf, peak_src)
        if P["prec"] == 1 and lib_peak:
            rl["frac_of_mxfp8_library"] = rl["achieved"] / lib_peak[0]
        out[name] = dict(value=value, unit="TFLOP/s", ms_per_step=T["ms"], profiled_ms_per_step=T["profiled_ms"],
                         dtype="mxfp8" if P["prec"] == 1 else "bf16",
                         pct_of_tensor_peak=100.0 * value / world / peak_tf,
                         pct_of_mxfp8_library_peak=(100.0 * value / world / lib_peak[0])
                         if (P["prec"] == 1 and lib_peak) else None,
                         tokens_per_s=P["tokens"] * world / (T["ms"] * 1e-3), gpu_launches=T["launches"],
                         roofline=dict(kernel=rl["kernel"], achieved=rl["achieved"], frac=rl["frac"],
                                       peak=rl["peak"], per_stage_frac=rl.get("per_stage_frac")),
                         stage_ms=T["stages"], clocks=T["clocks"],
                         config=dict(workload_config(cfg, P["is_linear"], world), l2=T["l2"]))
        del P
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other bar workloads after the headline")
    ap.add_argument("--measure-peaks", action="store_true", help="library GEMM peaks only")
    args = ap.parse_args()
    if args.measure_peaks:
        measure_peaks()
        return
    args.warmup = max(args.warmup, 3)

    import torch

    from moe_expert_layer_routing_gb300.inputs import CONFIGS, LinearConfig, make_linear_inputs, make_moe_inputs

    world, rank, local = dist_setup(args.gpus)
    cfg = CONFIGS[args.workload]
    is_linear = isinstance(cfg, LinearConfig)
    cores = len(os.sched_getaffinity(0))

    if args.impl == "reference":
        if rank != 0:
            return
        inp = make_linear_inputs(cfg) if is_linear else make_moe_inputs(cfg, device="cuda" if torch.cuda.is_available() else "cpu")
        run, flops, desc = oracle_sample_linear(inp, 128) if is_linear else oracle_sample_moe(inp, 128)
        for _ in range(args.warmup):
            run()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            run()
        dt = (time.perf_counter() - t0) / args.steps
        value = flops / dt / 1e12
        line = dict(metric=METRIC_LINEAR if is_linear else METRIC_MOE, value=value,
                    unit="TFLOP/s", n_gpus=world, steps=args.steps, warmup=args.warmup, ms_per_step=dt * 1e3,
                    higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                    impl="reference",
                    config=dict(workload_config(cfg, is_linear, world),
                                l2=l2_note(resident_input_bytes(cfg), device_l2_bytes())),
                    cpu_baseline=dict(value=value, unit="TFLOP/s", cores=cores, kind="oracle", sample=desc),
                    e2e=dict(value=value, unit="TFLOP/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
        print(json.dumps(line), flush=True)
        return

    import moe_expert_layer_routing_gb300 as mb
    from __graft_entry__ import build
    if rank == 0:
        build()
    barrier(world)
    mb.lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()

    P = setup_problem(mb, cfg, dev)
    op, inp, kw, flops, tokens, prec = (P[k] for k in ("op", "inp", "kw", "flops", "tokens", "prec"))
    T = time_problem(mb, P, args.steps, args.warmup, world, local, stream)
    ms, launches, clocks, stages = T["ms"], T["launches"], T["clocks"], T["stages"]
    value = flops * world / (ms * 1e-3) / 1e12
    peak_tf = peaks["bf16_tflops"] * (FP8_OVER_BF16 if prec == 1 else 1.0)
    roofline = dominant_roofline(cfg, stages, value / world, prec, peak_tf, peak_src)

    # ---------------------------------------------------------------- router backward (consumes ds)
    next_rows = None
    if not is_linear:
        logits = inp.extra["logits"]
        dl = mb.router_bwd(mb.ROUTER_TOPK_OVER_SOFTMAX, inp.ids, op.ds, cfg.E, logits=logits, scores=inp.s, renorm=True)
        for _ in range(3):
            mb.router_bwd(mb.ROUTER_TOPK_OVER_SOFTMAX, inp.ids, op.ds, cfg.E, logits=logits, scores=inp.s, renorm=True)
        # its inputs fit in L2: flushed before each call, each call timed by its own events
        flush = torch.empty(2 * device_l2_bytes(), dtype=torch.uint8, device=dev)
        revs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 255)
            revs[i][0].record(stream)
            mb.router_bwd(mb.ROUTER_TOPK_OVER_SOFTMAX, inp.ids, op.ds, cfg.E, logits=logits, scores=inp.s, renorm=True)
            revs[i][1].record(stream)
        torch.cuda.synchronize()
        rms = sum(a.elapsed_time(b) for a, b in revs) / args.steps
        del flush
        rbytes = cfg.T * cfg.E * 4 * 2 + cfg.T * cfg.K * 4 * 3   # logits in, dlogits out; ds, scores, ids in
        gbs = rbytes / (rms * 1e-3) / 1e9
        next_rows = dict(router_bwd=dict(form="top-K over softmax, renormalised", ms=rms, bound="hbm",
                                         algorithmic_bytes=rbytes, achieved_gbs=gbs, peak_gbs=peaks["hbm_gbs"],
                                         frac=gbs / peaks["hbm_gbs"], l2="flushed before each call"))
        del dl
        next_rows["recompute_h"] = recompute_row(mb, cfg, inp, kw, args.steps, stream, peak_tf, dev)

    lib_peak = recorded_mxfp8_peak()
    if prec == 1 and lib_peak:
        roofline["frac_of_mxfp8_library"] = roofline["achieved"] / lib_peak[0]
        roofline["mxfp8_library_peak"] = lib_peak[0]

    # ---------------------------------------------------------------- end to end through host buffers
    # Each step copies its activations from pinned host memory and reads dx/ds (or dX/dW) back.
    # Two bound problems alternate so that step i+1's host->device copy (copy stream) overlaps
    # step i's backward (compute stream); events order every buffer reuse.
    e2e = None
    if not args.no_e2e:
        if is_linear:
            names, onames = ["dY", "W", "X"], ["dX", "dW"]
            ops = [op, mb.LinearBwd(cfg.M, cfg.N, cfg.K, mb.PREC_MXFP8, cfg.fp8, dev)]
            dev_in = [{k: getattr(inp, k) for k in names}, {k: torch.empty_like(getattr(inp, k)) for k in names}]
            runs = [lambda b: ops[b].run(dev_in[b]["dY"], dev_in[b]["W"], dev_in[b]["X"])] * 2
        else:
            names, onames = ["x", "dout", "s", "ids", "ckpt"], ["dx", "ds"]
            op2 = mb.MoeBwd(T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, block_size=cfg.block_size,
                            precision=cfg.precision, affinity=cfg.affinity, fp8_act=cfg.fp8_act, fp8_w=cfg.fp8_w,
                            has_bias=cfg.bias, device=dev)
            ops = [op, op2]
            dev_in = [{k: getattr(inp, k) for k in names}, {k: torch.empty_like(getattr(inp, k)) for k in names}]
            kw2 = dict(kw)
            kw2.update(dev_in[1])
            op2.bind(**kw2)
            runs = [lambda b: ops[b].run()] * 2
        host_in = {k: getattr(inp, k).cpu().pin_memory() for k in names}
        host_out = [{k: torch.empty_like(getattr(o, k), device="cpu").pin_memory() for k in onames} for o in ops]
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
        copy = torch.cuda.Stream()      # host -> device
        back = torch.cuda.Stream()      # device -> host
        comp = stream
        in_ready = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        out_read = [torch.cuda.Event(), torch.cuda.Event()]

        def e2e_steps(n):
            for i in range(n):
                b = i & 1
                with torch.cuda.stream(copy):
                    copy.wait_event(done[b])       # buffer b's previous backward has consumed its inputs
                    for k, t in host_in.items():
                        dev_in[b][k].copy_(t, non_blocking=True)
                    in_ready[b].record(copy)
                comp.wait_event(in_ready[b])
                comp.wait_event(out_read[b])       # buffer b's previous outputs have been read back
                runs[b](b)
                done[b].record(comp)
                with torch.cuda.stream(back):
                    back.wait_event(done[b])
                    for k, t in host_out[b].items():
                        t.copy_(getattr(ops[b], k), non_blocking=True)
                    out_read[b].record(back)

        e2e_steps(2)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(copy)
        comp.wait_event(e0)
        e2e_steps(args.steps)
        comp.wait_stream(back)
        e1.record(comp)
        torch.cuda.synchronize()
        ems = allreduce_max(e0.elapsed_time(e1) / args.steps, world)
        e2e = dict(value=flops * world / (ems * 1e-3) / 1e12, unit="TFLOP/s", ms_per_step=ems,
                   h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                   note=("activations (x, dout, s, ids, checkpoint) in, dx and ds out; weights and weight "
                         "gradients stay resident; copies overlap the previous step's backward" if not is_linear
                         else "dY, W, X in; dX, dW out; copies overlap the previous step"))
        del ops, dev_in

    # ---------------------------------------------------------------- the other bar workloads (N=1)
    extra = None
    if world == 1 and not args.no_extra and args.workload == DEFAULT_WORKLOAD:
        extra = extra_workloads(mb, args, world, local, stream, peaks, peak_src, dev)

    if rank != 0:
        barrier(world)
        return
    # ---------------------------------------------------------------- CPU oracle baseline (rank 0, N=1)
    cpu_baseline = None
    if world == 1 and not args.no_cpu:
        if is_linear:
            run, cflops, desc = oracle_sample_linear(inp, 512)
        else:
            run, cflops, desc = oracle_sample_moe(inp, 512)
        cval, n = time_oracle(run, cflops, 15.0)
        cpu_baseline = dict(value=cval, unit="TFLOP/s", cores=cores, kind="oracle", sample=desc + f"; {n} run(s)")

    conf = workload_config(cfg, is_linear, world)
    conf["l2"] = T["l2"]
    line = dict(
        metric=METRIC_LINEAR if is_linear else METRIC_MOE,
        value=value, unit="TFLOP/s", n_gpus=world, steps=args.steps, warmup=args.warmup, ms_per_step=ms,
        higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="mxfp8" if prec == 1 else "bf16", data="synthetic (seeded; shapes and routing of the workload)",
        config=conf, tokens_per_s=tokens * world / (ms * 1e-3), pct_of_tensor_peak=100.0 * value / world / peak_tf,
        pct_of_mxfp8_library_peak=(100.0 * value / world / lib_peak[0]) if (prec == 1 and lib_peak) else None,
        roofline=roofline, cpu_baseline=cpu_baseline, e2e=e2e, clocks=clocks, gpu_launches=launches,
        next_rows=next_rows, stage_ms=stages, profiled_ms_per_step=T["profiled_ms"], workloads=extra,
        source_sha=source_sha())
    print(json.dumps(line), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
