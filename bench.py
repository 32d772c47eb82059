"""Benchmark of the selective scan (S6 forward) and the decode step on B300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2] [--impl ours|reference]

One step = one ssm_scan_fwd over one batch of the workload (all of: loads, Delta, discretise,
recurrence, readout + D skip + silu gate, final state). Inputs are synthetic (seeded) and
resident in HBM before the timed region; L2 is flushed (256 MiB write) before every step,
outside the per-step CUDA events. The same JSON line also carries the decode sweep
(64 layers x ssm_state_update per generated token, replayed from CUDA graphs), the
end-to-end number through host buffers, the roofline of the dominant kernel, the SM clocks
sampled during the run and the fp64 CPU oracle timed on a bounded sample.

Under torchrun (N > 1) every rank runs the same workload on its own GPU (independent
batches: weak scaling, no collective on the data path); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import DECODE_CONFIG, make_decode_layer_params, make_decode_state  # noqa: E402
from workloads import make_decode_tokens, make_scan_inputs, scan_config, ssd_config  # noqa: E402

METRIC = "selective-scan B·D·L elem/s & achieved HBM GB/s (% of peak); decode steps/s"
SM_PER_GPU_FALLBACK = 148
ALU_ELEM_PER_CLK_PER_SM = 2.0  # 16 SFU exp2 (32/clk/SM) and 64 FP32 lane-ops (128/clk/SM) per element
BWD_ELEM_PER_CLK_PER_SM = 32.0 / 48.0  # backward: 48 SFU exp2 per element at 32/clk/SM
BWD_CKPT_ELEM_PER_CLK_PER_SM = 32.0 / 32.0  # backward given the forward's checkpoints: 32 exp2
L2_FLUSH_BYTES = 256 << 20
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the scan kernel on this workload,
# from one ncu capture of the same kernel code (summarised under profiles/, the file named in
# SCAN_TRAFFIC_SOURCE); re-taken whenever the kernel changes.
SCAN_KERNEL_NAME = "scan_kernel: the launches of one scan (local-end pass, whole blocks, segments)"
SCAN_TRAFFIC_BYTES = {"c2_mamba2p8b": 312_334_336}
SCAN_TRAFFIC_SOURCE = {"c2_mamba2p8b": "ncu capture in profiles/scan_fwd_c2_mamba2p8b.md: 12.10 + "
                                       "280.02 + 20.21 MB over the three launches of one scan"}


# ------------------------------------------------------------------------------------------
# helpers

def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


def scan_algorithmic_bytes(cfg) -> int:
    """Compulsory HBM bytes of one scan: every input read once, y and the final state
    written once (the per-token state is never stored)."""
    ein = 2 if cfg.in_dtype == "bf16" else 4
    eout = 2 if cfg.out_dtype == "bf16" else 4
    act = cfg.batch * cfg.dim * cfg.seqlen
    bc = cfg.batch * cfg.dstate * cfg.seqlen
    nact_in = 2 + (1 if cfg.has_z else 0)
    per_ch = cfg.dim * cfg.dstate * 4 + cfg.dim * 4 * ((1 if cfg.has_D else 0) + (1 if cfg.has_bias else 0))
    return act * (nact_in * ein + eout) + 2 * bc * ein + per_ch + cfg.batch * cfg.dim * cfg.dstate * 4


def decode_algorithmic_bytes(batch, dim, dstate, conv=False) -> int:
    """Per layer-step: state read + write (fp32), x/dt/z read + out write (bf16), B and C
    (bf16), A (fp32) and D, dt_bias (fp32); with the convolution also its bf16 window of 4
    read + write and its fp32 taps and bias."""
    n = (batch * dim * dstate * 4 * 2 + batch * dim * 2 * 4 + batch * dstate * 2 * 2
         + dim * dstate * 4 + dim * 4 * 2)
    if conv:
        n += batch * dim * 4 * 2 * 2 + dim * 4 * 4 + dim * 4
    return n


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampling in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        rows = []
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                rows.append(dict(sm=float(p[0]), smax=float(p[1]), util=float(p[2]),
                                 hw=p[5], hwt=p[6], swt=p[7], swp=p[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["smax"] for r in busy), "reasons": sorted(reasons),
                "samples": len(busy)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Max of a per-rank float over all ranks (the slowest rank sets the job time)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# our arm

def time_scan(cfg, steps, warmup, x, flush, stream, soak_s=1.0):
    from selective_state_space_110_b300 import ssm_scan_fwd, workspace_size
    out_dtype = torch.bfloat16 if cfg.out_dtype == "bf16" else torch.float32
    out = torch.empty(cfg.batch, cfg.dim, cfg.seqlen, dtype=out_dtype, device="cuda")
    fin = torch.empty(cfg.batch, cfg.dim, cfg.dstate, dtype=torch.float32, device="cuda")
    ws_n = workspace_size(cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda") if ws_n else None

    def call():
        ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                     x["delta_bias"], x["delta_softplus"], out=out, final_state=fin,
                     workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.fill_(1)
            call()
        # untimed soak so the clock samples see the kernel at steady state
        t_end = time.time() + soak_s
        while time.time() < t_end:
            for _ in range(20):
                call()
            stream.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(steps):
            flush.fill_(1)
            ev[s][0].record(stream)
            call()
            ev[s][1].record(stream)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in ev]
    return times, scan_launches(cfg)


def scan_launches(cfg) -> int:
    """Kernel launches of one ssm_scan_fwd of this workload: one for whole blocks, plus a
    local-end pass when blocks are cut into segments, plus the segments' own launch when whole
    and cut blocks are mixed (the balanced plan)."""
    from selective_state_space_110_b300 import scan_plan
    p = scan_plan(cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen,
                  in_dtype=torch.bfloat16 if cfg.in_dtype == "bf16" else torch.float32)
    if p["split_blocks"] == 0 or p["segments"] == 1:
        return 1
    return 3 if p["whole_blocks"] > 0 else 2


def time_segments(cfg) -> int:
    """Time segments per cut block of the library's launch plan on this device (1 = none)."""
    from selective_state_space_110_b300 import scan_plan
    return scan_plan(cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen)["segments"]


def plan_summary(cfg) -> dict:
    """The launch plan of the scan on this device, and the exps it runs per element: every cut
    block's first segments-1 segments are scanned twice (the local-end pass, then the full pass
    after the fold)."""
    from selective_state_space_110_b300 import scan_plan
    p = scan_plan(cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen,
                  in_dtype=torch.bfloat16 if cfg.in_dtype == "bf16" else torch.float32)
    blocks = p["whole_blocks"] + p["split_blocks"]
    seg, L = p["segments"], max(cfg.seqlen, 1)
    twice = p["split_blocks"] * min(L, (seg - 1) * p["segment_tokens"]) / (blocks * L) if seg > 1 else 0.0
    return {"plan": {"whole_blocks": p["whole_blocks"], "split_blocks": p["split_blocks"],
                     "time_segments": seg, "segment_tokens": p["segment_tokens"],
                     "channels_per_block": p["channels_per_block"], "rows_per_lane": p["rows_per_lane"]},
            "exp_passes": round(1 + twice, 3)}


def other_scan_summary(name, args, flush, stream, sms, sm_mhz, hbm_peak):
    """Another scan workload timed like the main one (L2 flushed, CUDA events per step):
    median ms, elements/s, compulsory GB/s against the HBM and arithmetic ceilings, and the
    time split the plan takes (each extra segment runs its exps a second time)."""
    cfg = scan_config(name)
    x = make_scan_inputs(cfg, "cuda")
    steps = 3 if cfg.elements > (1 << 30) else max(3, min(args.steps, 10))
    times, launches = time_scan(cfg, steps, 3, x, flush, stream, soak_s=0.2)
    del x
    ms = statistics.median(times)
    alg = scan_algorithmic_bytes(cfg)
    elem_s = cfg.elements / (ms * 1e-3)
    alu_elem_s = ALU_ELEM_PER_CLK_PER_SM * sms * sm_mhz * 1e6
    return {"shape": {"batch": cfg.batch, "dim": cfg.dim, "dstate": cfg.dstate, "seqlen": cfg.seqlen},
            "steps": steps, "ms_per_step": round(ms, 4), "elem_per_s": round(elem_s, 1),
            "achieved_gbs": round(alg / (ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(alg / (ms * 1e-3) / 1e9 / hbm_peak, 4),
            "alu_frac": round(elem_s / alu_elem_s, 4),
            **plan_summary(cfg),
            "launches_per_step": launches}


def time_bwd(cfg, steps, warmup, x, flush, stream, checkpoints=False):
    """ssm_scan_bwd on the same workload (gradients of every input for a random bf16 dout),
    L2 flushed before every step. Returns per-step times (ms) and launches per step.
    checkpoints=True times the pair a training step runs when the forward keeps its states:
    ssm_scan_fwd_ckpt, then ssm_scan_bwd given those checkpoints; it returns the times of
    the pair and of the backward alone."""
    from selective_state_space_110_b300 import bwd_workspace_size, ssm_scan_bwd, ssm_scan_fwd_ckpt
    gen = torch.Generator("cuda").manual_seed(cfg.seed + 7)
    dout = torch.randn(cfg.batch, cfg.dim, cfg.seqlen, generator=gen, device="cuda").to(torch.bfloat16)
    ws = torch.empty(bwd_workspace_size(cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen, checkpoints),
                     dtype=torch.uint8, device="cuda")
    args = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
            x["delta_softplus"])
    if checkpoints:
        out = torch.empty(cfg.batch, cfg.dim, cfg.seqlen, dtype=torch.bfloat16, device="cuda")
        ck = torch.empty(cfg.batch, cfg.dim, (cfg.seqlen + 15) // 16, cfg.dstate, device="cuda")
        mid = [(torch.cuda.Event(enable_timing=True)) for _ in range(steps)]

    def call(s=None):
        if checkpoints:
            ssm_scan_fwd_ckpt(*args, out=out, checkpoints=ck, stream=stream)
            if s is not None:
                mid[s].record(stream)
        ssm_scan_bwd(*args, dout=dout, workspace=ws, stream=stream,
                     checkpoints=ck if checkpoints else None)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.fill_(1)
            call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(steps):
            flush.fill_(1)
            ev[s][0].record(stream)
            call(s)
            ev[s][1].record(stream)
    torch.cuda.synchronize()
    if checkpoints:
        return [a.elapsed_time(b) for a, b in ev], [m.elapsed_time(b) for m, (_, b) in zip(mid, ev)], 3
    return [a.elapsed_time(b) for a, b in ev], 2


def ssd_work(cfg):
    """Algorithmic tensor FLOPs (the four chunk products once each, no hi/lo split), FLOPs the
    tensor cores execute (C S, M X and B^T (w X) twice: bf16 hi and lo parts), and compulsory
    HBM bytes (x, z read and y written once, bf16; B, C, dt read once) of one SSD call."""
    Q, N, P = 128, cfg.dstate, cfg.headdim
    chunks = cfg.batch * cfg.nheads * ((cfg.seqlen + Q - 1) // Q)
    g1, g2, g3, g4 = 2 * Q * Q * N, 2 * Q * Q * P, 2 * Q * N * P, 2 * Q * N * P
    alg = chunks * (g1 + g2 + g3 + g4)
    executed = chunks * (g1 + 2 * (g2 + g3 + g4))
    byts = (cfg.elements * 2 * 3 + cfg.batch * cfg.seqlen * cfg.ngroups * N * 2 * 2 +
            cfg.batch * cfg.seqlen * cfg.nheads * 2 + cfg.batch * cfg.nheads * P * N * 4)
    return alg, executed, byts


def time_ssd(cfg, steps, warmup, flush, stream):
    """ssd_chunk_scan_fwd on the Mamba-2 layer workload, L2 flushed before every step."""
    from selective_state_space_110_b300 import ssd_chunk_scan_fwd, ssd_workspace_size
    from workloads import make_ssd_inputs
    x = make_ssd_inputs(cfg, "cuda")
    y = torch.empty(x["x"].shape, dtype=torch.bfloat16, device="cuda")
    fin = torch.empty(cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate, device="cuda")
    need = ssd_workspace_size(cfg.batch, cfg.seqlen, cfg.nheads)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda") if need else None

    def call():
        ssd_chunk_scan_fwd(x["x"], x["dt"], x["A"], x["B"], x["C"], x["D"], x["z"], x["dt_bias"],
                           x["dt_softplus"], y=y, final_state=fin, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.fill_(1)
            call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(steps):
            flush.fill_(1)
            ev[s][0].record(stream)
            call()
            ev[s][1].record(stream)
    torch.cuda.synchronize()
    # launches of one call: unsplit one; balanced the state-only pass, the whole chains, the
    # fold and the segments
    launches = 4 if ws is not None else 1
    return [a.elapsed_time(b) for a, b in ev], launches


def time_scan_e2e(cfg, steps, warmup, x, stream):
    """The same scan through the host-buffer entry point ssm_scan_fwd_host: every step uploads
    the step's inputs from pinned host memory, scans, and downloads y and the final state (the
    library pipelines the copies with the scan, one sequence at a time)."""
    from selective_state_space_110_b300 import host_workspace_size, ssm_scan_fwd_host
    names = ["u", "delta", "A", "B", "C", "D", "z", "delta_bias"]
    host = {k: (x[k].cpu().pin_memory() if x[k] is not None else None) for k in names}
    out_dtype = torch.bfloat16 if cfg.out_dtype == "bf16" else torch.float32
    out_h = torch.empty(cfg.batch, cfg.dim, cfg.seqlen, dtype=out_dtype).pin_memory()
    fin_h = torch.empty(cfg.batch, cfg.dim, cfg.dstate, dtype=torch.float32).pin_memory()
    ws = torch.empty(host_workspace_size(cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen,
                                         x["u"].dtype, out_dtype), dtype=torch.uint8, device="cuda")
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = out_h.numel() * out_h.element_size() + fin_h.numel() * fin_h.element_size()

    def step():
        ssm_scan_fwd_host(host["u"], host["delta"], host["A"], host["B"], host["C"], host["D"],
                          host["z"], host["delta_bias"], x["delta_softplus"], out=out_h,
                          final_state=fin_h, workspace=ws, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


def time_decode(batch, steps, warmup, stream, conv=False):
    """Decode sweep: per generated token, ssm_state_update on each of 64 layers (own state,
    A, D, dt_bias per layer); the 64 calls of a token are one CUDA graph, one graph per slot
    of the ring of 8 token-input sets. conv=True: the fused step of the short convolution
    (own bf16 window of 4 inputs and fp32 taps per layer) and the state update,
    ssm_conv_state_update."""
    from selective_state_space_110_b300 import ssm_conv_state_update, ssm_state_update
    cfg = DECODE_CONFIG
    p = make_decode_layer_params(cfg, "cuda")
    gen = torch.Generator("cuda").manual_seed(cfg.seed + 17)
    layers = []
    for l in range(cfg.layers):
        layers.append(dict(A=p["A"].clone(), D=p["D"].clone(), bias=p["dt_bias"].clone(),
                           state=make_decode_state(cfg, batch, l, "cuda"),
                           out=torch.empty(batch, cfg.dim, dtype=torch.bfloat16, device="cuda"),
                           toks=[make_decode_tokens(cfg, batch, l, s, "cuda") for s in range(cfg.ring)]))
        if conv:
            layers[-1].update(
                cs=torch.randn(batch, cfg.dim, 4, generator=gen, device="cuda").to(torch.bfloat16),
                w=torch.randn(cfg.dim, 4, generator=gen, device="cuda") * 0.5,
                cb=torch.randn(cfg.dim, generator=gen, device="cuda") * 0.1)

    def token_step(slot):
        for L in layers:
            t = L["toks"][slot]
            if conv:
                ssm_conv_state_update(L["cs"], t["x"], L["w"], L["cb"], True, L["state"], t["dt"],
                                      L["A"], t["B"], t["C"], L["D"], t["z"], out=L["out"],
                                      dt_bias=L["bias"], stream=stream)
            else:
                ssm_state_update(L["state"], t["x"], t["dt"], L["A"], t["B"], t["C"], L["D"],
                                 t["z"], out=L["out"], dt_bias=L["bias"], stream=stream)

    with torch.cuda.stream(stream):
        for s in range(3):
            token_step(s % cfg.ring)
    torch.cuda.synchronize()
    graphs = []
    for slot in range(cfg.ring):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            token_step(slot)
        graphs.append(g)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(warmup):
            graphs[s % cfg.ring].replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for s in range(steps):
            graphs[s % cfg.ring].replay()
        b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return ms, cfg.layers


def cpu_baseline(cfg, x, target_s=12.0):
    """The fp64 oracle as it stands, on the host cores, on a bounded sample of rows of the
    same workload (all tokens of each sampled row)."""
    import oracle
    R = cfg.batch * cfg.dim
    rng = torch.Generator().manual_seed(0)
    perm = torch.randperm(R, generator=rng)

    def run(nrows):
        rows = perm[:nrows].sort().values
        rd = rows.to("cuda")
        flat = lambda t: t.view(R, -1)[rd].cpu()
        args = (rows.numpy(), flat(x["u"]), flat(x["delta"]), x["A"].cpu(), x["B"].cpu(),
                x["C"].cpu(), None if x["D"] is None else x["D"].cpu(),
                None if x["z"] is None else flat(x["z"]),
                None if x["delta_bias"] is None else x["delta_bias"].cpu(), x["delta_softplus"])
        import oracle as o
        prepared = [o._f64(a) if hasattr(a, "detach") else a for a in args]
        t0 = time.perf_counter()
        oracle.scan_fwd_rows(*prepared)
        return time.perf_counter() - t0

    n0 = min(R, 64)
    t0 = run(n0)
    n = int(min(R, max(n0, n0 * target_s / max(t0, 1e-3))))
    t = run(n) if n > n0 else t0
    elems = n * cfg.seqlen
    return {"value": elems / t, "unit": "elem/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{n} of {R} (batch, channel) rows x all {cfg.seqlen} tokens of {cfg.name} "
                      f"({elems} elements, {t:.1f} s)"}


def ssd_summary(scfg, ms, launches, world, scan_ms, scan_cfg):
    alg, executed, byts = ssd_work(scfg)
    _, _, tflops_peak = read_tensor_peak()
    hbm_peak, _ = read_peaks()
    sec = ms * 1e-3
    from selective_state_space_110_b300 import ssd_plan
    plan = ssd_plan(scfg.batch, scfg.seqlen, scfg.nheads)
    out = {"what": "ssd_chunk_scan_fwd: Mamba-2 SSD layer, 128-token chunks on tcgen05, "
                   "state in tensor memory (ssd_fwd_kernel)",
           "plan": plan,
           "workload": scfg.name,
           "shape": {"batch": scfg.batch, "seqlen": scfg.seqlen, "nheads": scfg.nheads,
                     "headdim": scfg.headdim, "ngroups": scfg.ngroups, "dstate": scfg.dstate},
           "ms_per_step": round(ms, 4),
           "elem_per_s": round(world * scfg.elements / sec, 1),
           "tensor_tflops_algorithmic": round(alg / sec / 1e12, 1),
           "tensor_tflops_executed": round(executed / sec / 1e12, 1),
           "tensor_frac": round(executed / sec / 1e12 / tflops_peak, 4),
           "tensor_peak_tflops": tflops_peak,
           "achieved_gbs": round(byts / sec / 1e9, 1),
           "hbm_frac": round(byts / sec / 1e9 / hbm_peak, 4),
           "launches_per_step": launches}
    if scfg.elements == scan_cfg.elements:
        out["vs_s6_scan_same_elements"] = round(scan_ms / ms, 3)
    return out


def read_tensor_peak():
    """(sustained, source, burst) dense bf16 TFLOP/s: measured, else the fallback figures."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d.get("bf16_tflops_sustained"), "measured", float(d["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1400.0, "fallback", 1800.0


def run_ours(args):
    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    from selective_state_space_110_b300 import LIB_PATH  # noqa: F401  (fails loudly if missing)
    cfg = scan_config(args.workload)
    hbm_peak, peak_src = read_peaks()
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    x = make_scan_inputs(cfg, "cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    barrier(world)
    with ClockSampler(local) as clk:
        times, launches = time_scan(cfg, args.steps, args.warmup, x, flush, stream, args.soak_s)
    barrier(world)
    ms_total = max_over_ranks(sum(times), world)
    ms_step = ms_total / args.steps
    elems = cfg.elements * world
    value = elems / (ms_step * 1e-3)
    clocks = clk.summary()

    ssd_cfg = ssd_config(args.ssd_workload)
    ssd_times, ssd_launches = time_ssd(ssd_cfg, max(3, min(args.steps, 10)), 3, flush, stream)
    ssd_ms = max_over_ranks(statistics.median(ssd_times), world)
    bwd_times, bwd_launches = time_bwd(cfg, max(3, min(args.steps, 10)), 3, x, flush, stream)
    bwd_ms = max_over_ranks(statistics.median(bwd_times), world)
    pair_times, bwdc_times, pair_launches = time_bwd(cfg, max(3, min(args.steps, 10)), 3, x, flush,
                                                     stream, checkpoints=True)
    pair_ms = max_over_ranks(statistics.median(pair_times), world)
    bwdc_ms = max_over_ranks(statistics.median(bwdc_times), world)
    e2e_ms, h2d, d2h = time_scan_e2e(cfg, max(2, min(args.steps, 10)), 2, x, stream)
    e2e_ms = max_over_ranks(e2e_ms, world)
    dec, dec_conv = {}, {}
    for conv, sink in ((False, dec), (True, dec_conv)):
        for b in (args.decode_batches if not conv else args.decode_conv_batches):
            dms, nl = time_decode(b, args.decode_steps, 8, stream, conv=conv)
            dms = max_over_ranks(dms, world)
            dbytes = decode_algorithmic_bytes(b, DECODE_CONFIG.dim, DECODE_CONFIG.dstate, conv) * nl
            sink[f"batch{b}"] = {"steps_per_s": round(world * 1e3 / dms, 1),
                                 "tokens_per_s": round(world * b * 1e3 / dms, 1),
                                 "ms_per_step": round(dms, 4),
                                 "achieved_gbs": round(dbytes / (dms * 1e-3) / 1e9, 1),
                                 "hbm_frac": round(dbytes / (dms * 1e-3) / 1e9 / hbm_peak, 3),
                                 "launches_per_step": nl}

    sm_mhz = clocks["sm_mhz"] or 1900.0
    others = {}
    for name in args.other_workloads:
        o = other_scan_summary(name, args, flush, stream, sms, sm_mhz, hbm_peak)
        o["ms_per_step"] = round(max_over_ranks(o["ms_per_step"], world), 4)
        others[scan_config(name).name] = o

    if rank != 0:
        return
    alg = scan_algorithmic_bytes(cfg)
    kern_ms = statistics.mean(times)
    achieved = alg / (kern_ms * 1e-3) / 1e9
    alu_peak_elem = ALU_ELEM_PER_CLK_PER_SM * sms * sm_mhz * 1e6
    alu_peak_gbs = alu_peak_elem * alg / cfg.elements / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "elem/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in/out, fp32 compute",
        "data": "synthetic (seeded N(0,1)/N(0,0.25) activations, A=-(n+1), log-uniform dt)",
        "config": {"workload": cfg.name, "batch": cfg.batch, "dim": cfg.dim, "dstate": cfg.dstate,
                   "seqlen": cfg.seqlen, "elements_per_step": cfg.elements * world,
                   "l2": "256 MiB write before every step, outside the per-step events",
                   "parallelism": f"{world} independent replica(s), no collective"},
        "achieved_gbs": round(achieved, 1),
        "hbm_frac": round(achieved / hbm_peak, 4),
        "roofline": {"bound": "alu", "achieved": round(achieved, 1), "peak": round(alu_peak_gbs, 1),
                     "unit": "GB/s", "frac": round(achieved / alu_peak_gbs, 4),
                     "traffic": SCAN_TRAFFIC_BYTES.get(cfg.name),
                     "traffic_source": SCAN_TRAFFIC_SOURCE.get(cfg.name),
                     "kernel": SCAN_KERNEL_NAME,
                     "peak_note": f"ALU ceiling {ALU_ELEM_PER_CLK_PER_SM} elem/clk/SM x {sms} SMs x "
                                  f"{sm_mhz:.0f} MHz, as GB/s of compulsory bytes; the rates behind "
                                  "it (ex2 32/clk/SM, fp32 FMA 128 lanes/clk/SM) are measured by "
                                  "bench.py --pipe-rates, profiles/pipe_rates_b300.md",
                     "hbm_peak": hbm_peak, "hbm_peak_source": peak_src,
                     "hbm_frac": round(achieved / hbm_peak, 4)},
        "plan": plan_summary(cfg),
        "e2e": {"value": round(elems / (e2e_ms * 1e-3), 1), "unit": "elem/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "backward": {"what": "ssm_scan_bwd: all input gradients, state every 16 tokens, "
                             "chunks recomputed (scan_bwd_kernel + scan_bwd_reduce_kernel)",
                     "ms_per_step": round(bwd_ms, 4),
                     "elem_per_s": round(elems / (bwd_ms * 1e-3), 1),
                     "vs_forward_time": round(bwd_ms / kern_ms, 2),
                     "alu_frac": round(elems / (bwd_ms * 1e-3) /
                                       (BWD_ELEM_PER_CLK_PER_SM * sms * sm_mhz * 1e6), 4),
                     "alu_note": f"ceiling {BWD_ELEM_PER_CLK_PER_SM:.3f} elem/clk/SM: 48 SFU exp2 "
                                 "per element (3 passes x 16 states) at 32 per clock per SM",
                     "launches_per_step": bwd_launches,
                     "with_forward_checkpoints": {
                         "what": "ssm_scan_fwd_ckpt (the forward keeping the state before every "
                                 "16th token) then ssm_scan_bwd given them: no recomputing pass",
                         "fwd_ckpt_ms": round(pair_ms - bwdc_ms, 4),
                         "bwd_ms": round(bwdc_ms, 4),
                         "fwd_plus_bwd_ms": round(pair_ms, 4),
                         "plain_fwd_plus_bwd_ms": round(kern_ms + bwd_ms, 4),
                         "bwd_alu_frac": round(elems / (bwdc_ms * 1e-3) /
                                               (BWD_CKPT_ELEM_PER_CLK_PER_SM * sms * sm_mhz * 1e6), 4),
                         "alu_note": f"ceiling {BWD_CKPT_ELEM_PER_CLK_PER_SM:.3f} elem/clk/SM: 32 "
                                     "SFU exp2 per element (2 passes x 16 states)",
                         "launches_per_step": pair_launches}},
        "other_workloads": others,
        "ssd": ssd_summary(ssd_cfg, ssd_ms, ssd_launches, world, kern_ms, cfg),
        "decode": {"layers": DECODE_CONFIG.layers, "dim": DECODE_CONFIG.dim, **dec},
        "decode_conv": {"layers": DECODE_CONFIG.layers, "dim": DECODE_CONFIG.dim,
                        "what": "ssm_conv_state_update: width-4 convolution step + state update",
                        **dec_conv},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, x)
    print(json.dumps(line), flush=True)


def run_profile(args):
    """One scan of the workload (plus one decode layer-step at batch 64 and one at 16), or with
    --profile-op bwd two backward calls: a small, bounded program for ncu captures."""
    from selective_state_space_110_b300 import ssm_scan_fwd, ssm_state_update
    cfg = scan_config(args.workload)
    x = make_scan_inputs(cfg, "cuda")
    if args.profile_op == "ssd":
        from selective_state_space_110_b300 import ssd_chunk_scan_fwd
        from workloads import make_ssd_inputs
        scfg = ssd_config(args.ssd_workload)
        xs = make_ssd_inputs(scfg, "cuda")
        for _ in range(2):
            y, _ = ssd_chunk_scan_fwd(xs["x"], xs["dt"], xs["A"], xs["B"], xs["C"], xs["D"], xs["z"],
                                      xs["dt_bias"], xs["dt_softplus"])
        torch.cuda.synchronize()
        print(json.dumps({"profile": scfg.name, "op": "ssd", "finite": bool(torch.isfinite(y).all().item())}))
        return
    if args.profile_op == "bwd":
        from selective_state_space_110_b300 import ssm_scan_bwd
        gen = torch.Generator("cuda").manual_seed(cfg.seed + 7)
        dout = torch.randn(cfg.batch, cfg.dim, cfg.seqlen, generator=gen, device="cuda").to(torch.bfloat16)
        for _ in range(2):
            g = ssm_scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                             x["delta_bias"], x["delta_softplus"], dout=dout)
        torch.cuda.synchronize()
        print(json.dumps({"profile": cfg.name, "op": "bwd",
                          "finite": bool(torch.isfinite(g["du"]).all().item())}))
        return
    out, fin = ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                            x["delta_bias"], x["delta_softplus"])
    p = make_decode_layer_params(DECODE_CONFIG, "cuda")
    for batch in (64, 16):
        st = make_decode_state(DECODE_CONFIG, batch, 0, "cuda")
        t = make_decode_tokens(DECODE_CONFIG, batch, 0, 0, "cuda")
        ssm_state_update(st, t["x"], t["dt"], p["A"], t["B"], t["C"], p["D"], t["z"],
                         dt_bias=p["dt_bias"])
    torch.cuda.synchronize()
    print(json.dumps({"profile": cfg.name, "finite": bool(torch.isfinite(out).all().item())}))


# ------------------------------------------------------------------------------------------
# reference arm: the fp64 oracle, as it stands, on the host cores

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    cfg = scan_config(args.workload)
    x = make_scan_inputs(cfg.replace(batch=1), "cpu")
    # a bounded sample: up to 2,048 rows x all tokens per step (enough work that the oracle's
    # thread start-up does not set its rate)
    rows_per_step = min(2048, cfg.dim)
    rows = torch.arange(rows_per_step)
    flat = lambda t: t.view(cfg.dim, -1)[rows]
    args_ = [rows.numpy(), flat(x["u"]), flat(x["delta"]), x["A"], x["B"], x["C"], x["D"],
             flat(x["z"]), x["delta_bias"], True]
    prepared = [oracle._f64(a) if hasattr(a, "detach") else a for a in args_]
    for _ in range(args.warmup):
        oracle.scan_fwd_rows(*prepared)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan_fwd_rows(*prepared)
    dt = (time.perf_counter() - t0) / args.steps
    elems = rows_per_step * cfg.seqlen
    v = elems / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "elem/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "batch": cfg.batch, "dim": cfg.dim, "dstate": cfg.dstate,
                   "seqlen": cfg.seqlen},
        "cpu_baseline": {"value": round(v, 1), "unit": "elem/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"{rows_per_step} (batch, channel) rows x all {cfg.seqlen} tokens per step"},
        "e2e": {"value": round(v, 1), "unit": "elem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_pipe_rates(args):
    """Pipe rates of this GPU that the scan's arithmetic ceiling rests on (one CTA of 1,024
    threads per SM, clock64 around a fixed loop; see csrc/pipe_probe.cu), one JSON line."""
    import ctypes
    from selective_state_space_110_b300 import build as b
    lib = ctypes.CDLL(b.build_probe())
    lib.selscan_probe_rate.restype = ctypes.c_double
    lib.selscan_probe_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.c_void_p]
    torch.cuda.set_device(0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device="cuda")
    sink = torch.zeros(sms * 1024, dtype=torch.float32, device="cuda")
    names = ["ex2_per_clk_per_sm", "ffma_lanes_per_clk_per_sm", "lg2_per_clk_per_sm",
             "rcp_per_clk_per_sm", "ffma2_lanes_per_clk_per_sm", "shfl_per_clk_per_sm",
             "lds32_words_per_clk_per_sm", "lds128_words_per_clk_per_sm"]
    iters = {0: 4096, 1: 16384, 2: 4096, 3: 4096, 4: 16384, 5: 4096, 6: 4096, 7: 2048}
    out = {"pipe_rates": torch.cuda.get_device_name(0), "sms": sms,
           "method": "1 CTA x 1024 threads per SM, 16 independent chains (8 loads) per thread, "
                     "clock64 around the loop; best of 3 runs"}
    for which, name in enumerate(names):
        best = 0.0
        for _ in range(3):
            r = lib.selscan_probe_rate(which, sms, iters[which], cycles.data_ptr(), sink.data_ptr())
            if r < 0:
                raise RuntimeError(f"probe {name} failed ({r})")
            best = max(best, r)
        out[name] = round(best, 2)
    with ClockSampler(0) as clk:
        for _ in range(20):
            lib.selscan_probe_rate(0, sms, 16384, cycles.data_ptr(), sink.data_ptr())
    out["clocks"] = clk.summary()
    print(json.dumps(out), flush=True)


def run_oracle_timings(args):
    """The fp64 oracle as it stands, on the host cores, over whole workloads (a baseline only):
    C0-C3 in full (rows in batches; only the oracle calls are timed) and decode at batch 64 on
    8 of the 64 layers for 8 steps, scaled to a 64-layer step. One JSON line per workload."""
    import numpy as np
    import oracle
    from workloads import (DECODE_CONFIG, make_decode_layer_params, make_decode_state,
                           make_decode_tokens)
    cores = oracle.max_threads()
    f64 = oracle._f64
    for name in ("c0_tiny_f32", "c1_mamba130m", "c2_mamba2p8b", "c3_long_1m"):
        cfg = scan_config(name)
        x = make_scan_inputs(cfg, "cpu")
        R = cfg.batch * cfg.dim
        per_call = max(1, min(R, (1 << 26) // cfg.seqlen))  # about 64 M elements a call
        A, B, C = f64(x["A"]), f64(x["B"]), f64(x["C"])
        D = None if x["D"] is None else f64(x["D"])
        bias = None if x["delta_bias"] is None else f64(x["delta_bias"])
        total = 0.0
        for r0 in range(0, R, per_call):
            rows = np.arange(r0, min(R, r0 + per_call), dtype=np.int64)
            sl = lambda t: None if t is None else f64(t.reshape(R, -1)[r0:r0 + len(rows)])
            u, dl, z = sl(x["u"]), sl(x["delta"]), sl(x["z"])
            t0 = time.perf_counter()
            oracle.scan_fwd_rows(rows, u, dl, A, B, C, D, z, bias, x["delta_softplus"])
            total += time.perf_counter() - t0
        elems = R * cfg.seqlen
        print(json.dumps({"oracle_timing": name, "value": round(elems / total, 1), "unit": "elem/s",
                          "seconds": round(total, 3), "elements": elems, "cores": cores,
                          "kind": "oracle", "sample": "all rows and tokens"}), flush=True)
        del x
    dc = DECODE_CONFIG
    batch, layers, steps = 64, 8, 8
    p = {k: f64(v) for k, v in make_decode_layer_params(dc, "cpu").items()}
    total = 0.0
    for layer in range(layers):
        state = f64(make_decode_state(dc, batch, layer, "cpu"))
        for step in range(steps):
            t = {k: f64(v) for k, v in make_decode_tokens(dc, batch, layer, step % dc.ring, "cpu").items()}
            t0 = time.perf_counter()
            state, _ = oracle.state_update(state, t["x"], t["dt"], p["A"], t["B"], t["C"], p["D"],
                                           t["z"], p["dt_bias"], True)
            total += time.perf_counter() - t0
    per_call = total / (layers * steps)
    print(json.dumps({"oracle_timing": f"{dc.name}_batch{batch}",
                      "value": round(1.0 / (per_call * dc.layers), 2), "unit": "steps/s",
                      "seconds_per_layer_call": round(per_call, 6), "cores": cores,
                      "kind": "oracle",
                      "sample": f"{layers} of {dc.layers} layers x {steps} steps, scaled to "
                                f"{dc.layers} layers"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="c2_mamba2p8b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-batches", type=int, nargs="*", default=[1, 16, 64])
    ap.add_argument("--decode-steps", type=int, default=256)
    ap.add_argument("--decode-conv-batches", type=int, nargs="*", default=[1, 64])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="untimed back-to-back scans before the timed steps (clock sampling)")
    ap.add_argument("--profile", action="store_true",
                    help="run one scan of the workload and exit (for ncu captures)")
    ap.add_argument("--profile-op", default="fwd", choices=["fwd", "bwd", "ssd"],
                    help="with --profile: the forward scan (default), the backward, or the SSD "
                         "layer (--ssd-workload)")
    ap.add_argument("--ssd-workload", default="ssd1_mamba2_2p7b")
    ap.add_argument("--oracle-timings", action="store_true",
                    help="time the fp64 oracle on the host cores over C0-C3 and decode, and exit")
    ap.add_argument("--pipe-rates", action="store_true",
                    help="measure the SFU / FMA / shared-memory / shuffle rates and exit")
    ap.add_argument("--other-workloads", nargs="*", default=["c1_mamba130m", "c3_long_1m"],
                    help="scan workloads timed after the main one and reported beside it")
    args = ap.parse_args()
    if args.pipe_rates:
        run_pipe_rates(args)
        return
    if args.oracle_timings:
        run_oracle_timings(args)
        return
    if args.profile:
        run_profile(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
