"""Throughput of the RankMixer block-stack forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config rankmixer_1b|rankmixer_100m|moe_1b] [--batch B]

Prints ONE JSON line on rank 0.  A step is one forward pass of the whole hot
path (L x [token mixing + LN1, per-token FFN GEMM1 + GELU, GEMM2 + residual +
LN2 statistics], LN2 finalisation + mean pooling) over one batch of
synthetic input resident in HBM.  `value` = samples/s of the whole job
(weak scaling: every rank processes its own batch of B samples).  `e2e` is
the same metric through the pipelined host entry rm_stack_forward_host_async
(pinned host input, H2D copy, forward, D2H of the pooled output of every step
inside the timed region; the copy of step i + 1 overlaps step i's compute).

--impl reference times the CPU oracle (the plain float64 restatement used by
the tests) on the host cores, on a bounded sample of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# dominant kernel, from one ncu capture of this bench's own command line, keyed
# by (config, batch per GPU, layers, kernel kind), with the SHA-256 of the
# kernel sources the capture ran on.  Reported only while those sources are
# unchanged; otherwise the traffic is unknown (null).
# embedding coordinates per token for --pass score (the tokenizer's slice length d)
SCORE_SLICE = {"rankmixer_1b": 512, "rankmixer_100m": 256}
# --pass unimix: UniMixing in every layer at block size D / T (the TokenMixing
# granularity), the pages' final temperature and a fixed Sinkhorn-Knopp round count
UNIMIX_TAU = 0.05
UNIMIX_ITERS = 20

KERNEL_SOURCES = ("rankmixer_feature_interaction_gb300/csrc/rm_gemm_tc.cu",
                  "rankmixer_feature_interaction_gb300/csrc/rm_common.cuh")
TRAFFIC = {
    # ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum on
    # "bench.py --steps 3 --warmup 3 --no-cpu-baseline", averaged over two launches of the
    # fused layer kernel (both FFN GEMMs of a layer per launch); between boxes the figure for
    # the same kernel code has ranged from 6.3 to 8.8 GB
    ("rankmixer_1b", 4096, 2, "pffn"): (6337070080, "51a917a84a212143feb9652766e6d06d29948d804904d2fc1e6e56f11462e771"),
    # the expert GEMMs of "bench.py --config moe_1b --steps 3 --warmup 3 --no-cpu-baseline"
    ("moe_1b", 4096, 1, "moe_gemm1"): (4679440384, "51a917a84a212143feb9652766e6d06d29948d804904d2fc1e6e56f11462e771"),
    ("moe_1b", 4096, 1, "moe_gemm2"): (4784491776, "51a917a84a212143feb9652766e6d06d29948d804904d2fc1e6e56f11462e771"),
}


def kernel_source_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def captured_traffic(config: str, batch: int, layers: int, kind: str):
    rec = TRAFFIC.get((config, batch, layers, kind))
    if rec is None or rec[1] != kernel_source_digest():
        return None
    return rec[0]


def load_peaks():
    try:
        with open(PEAKS_PATH) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# A timed region shorter than this runs as a burst before the power cap pulls
# the clock down (the dense-GEMM peak measured back to back for seconds is the
# lower, sustained figure).
BURST_SECONDS = 1.0


def pick_tensor_peak(peaks: dict, src: str, timed_s: float, clk: dict) -> tuple[float, str]:
    """The dense bf16 peak the timed region ran against: the burst figure when the region
    lasted under BURST_SECONDS or its median SM clock sat at the maximum, otherwise the
    sustained (power-capped) figure."""
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    at_max = sm is not None and smax and sm >= 0.97 * smax
    if timed_s < BURST_SECONDS or at_max:
        why = f"timed region {timed_s:.2f} s" if timed_s < BURST_SECONDS else f"median SM clock {sm:.0f} MHz (max)"
        return float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])), f"{src} bf16_tflops (burst: {why})"
    why = f"timed region {timed_s:.1f} s at median SM clock {sm if sm is not None else 'unknown'} MHz"
    return (float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])),
            f"{src} bf16_tflops_sustained ({why})")


# ----------------------------------------------------------------------------
# Clock sampling during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0: float, t1: float):
        """Host wall-clock bounds of the timed region; samples outside it are dropped."""
        self.window = (t0, t1)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "window", (0.0, float("inf")))
        for ts, ln in self.lines:
            if not (t0 <= ts <= t1 + 0.15):
                continue
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------
# Distributed helpers (one process per GPU; weak scaling, no data-path collective)
# ----------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def shard_batch(global_batch: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of the samples rank `rank` owns when `global_batch` samples are split
    as evenly as possible over `world` ranks (first ranks take the remainder)."""
    base, rem = divmod(global_batch, world)
    start = rank * base + min(rank, rem)
    return start, start + base + (1 if rank < rem else 0)


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest of the ranks' values of x (each rank passes its own); x itself
    when no process group is running."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def allreduce_grads(flat) -> None:
    """Data-parallel training's one exchange: sum every rank's parameter gradients
    (one flat float32 buffer) over the ranks, in place; nothing without a process group."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(flat, op=dist.ReduceOp.SUM)


def job_rate(samples_per_rank: int, world: int, steps: int, seconds_max: float) -> float:
    """Whole-job throughput: the samples all ranks processed over the slowest rank's time."""
    return world * samples_per_rank * steps / seconds_max


# ----------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    from rankmixer_feature_interaction_gb300 import _lib, synth
    from rankmixer_feature_interaction_gb300.api import RankMixer

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    c = dict(synth.CONFIGS[args.config])
    B = args.batch or c["B"]
    T, D, k = c["T"], c["D"], c["k"]
    moe = args.config == "moe_1b"
    train = args.pass_ == "train"
    score = args.pass_ == "score"
    unimix = args.pass_ == "unimix"
    if moe and (score or unimix):
        raise SystemExit("--pass score / unimix run the dense stack (rankmixer_1b / rankmixer_100m)")
    L = args.layers or c["L"]
    E, Fe = c.get("E", 0), c.get("Fe", 0)
    # weak scaling: the job's batch is world * B samples, rank r owns shard r
    start, stop = shard_batch(world * B, world, rank)
    layers = synth.make_stack(T, D, k, L, 4242, "bf16", dev, E=E, Fe=Fe, active=c.get("active", 2.0))
    if moe and train:    # the dense-training router: about 6 of 8 experts open
        layers[0].update(synth.make_train_router(T, D, E, 4243, "bf16", dev, active=0.75 * E))
    m = RankMixer(T, D, k, layers, dtype="bf16", max_batch=B, n_experts=E, expert_hidden=Fe,
                  training=train and not moe)
    del layers
    bs_um = D // T
    if unimix:
        for n in range(L):
            WG, WB = synth.make_unimix_weights(T, D, bs_um, 4245 + n, dev)
            m.set_unimixing(n, WG, WB, tau=UNIMIX_TAU, iters=UNIMIX_ITERS)
            del WG, WB
    torch.cuda.empty_cache()
    X0 = synth.make_input_shard(world * B, start, stop, T, D, 20260101, "bf16", dev)
    pooled = torch.empty((B, D), dtype=torch.float32, device=dev)
    S_in = X0  # MoE PFFN input (an LN1 output in the model; same distribution class for timing)
    V = torch.empty((B, T, D), dtype=torch.float32, device=dev) if moe else None
    if train and not moe:
        # the gradient of a batch-mean loss at the pooled output
        dP = synth.make_output_grad((B, D), 20260102 + rank, scale=1.0 / (B * world), device=dev)
        dX0 = torch.empty((B, T, D), dtype=torch.float32, device=dev)
        gflat = torch.empty(m.flat_grad_numel(), dtype=torch.float32, device=dev)
        grads = m.alloc_grads(dev, flat=gflat)
    if moe and train:
        Gt = torch.empty((B, T, E), dtype=torch.float32, device=dev)
        Gi = torch.empty_like(Gt)
        lreg = torch.empty(B, dtype=torch.float32, device=dev)
        Aexp = torch.empty(E, dtype=torch.float32, device=dev)
    d_tok = SCORE_SLICE[args.config] if score else 0
    if score:
        # tokenizer (token t projects its d-coordinate slice) and head, random-init; embeddings N(0, 1)
        gtok = torch.Generator(device=dev).manual_seed(4244)
        Wtok = (torch.randn((T, d_tok, D), generator=gtok, device=dev) / d_tok ** 0.5).to(torch.bfloat16)
        btok = (0.1 * torch.randn((T, D), generator=gtok, device=dev)).to(torch.bfloat16)
        m.set_tokenizer(Wtok, btok)
        del Wtok, btok
        Emb = synth.make_input_shard(world * B, start, stop, T, d_tok, 20260103, "bf16", dev).reshape(B, T * d_tok)
        hw = torch.randn(D, generator=gtok, device=dev) / D ** 0.5
        p_out = torch.empty(B, dtype=torch.float32, device=dev)

    def step():
        if moe and train:
            _lib.rm_moe_pffn_forward_train(m.ctx, 0, S_in.data_ptr(), V.data_ptr(), Gt.data_ptr(), Gi.data_ptr(),
                                           lreg.data_ptr(), Aexp.data_ptr(), B, stream.cuda_stream)
        elif moe:
            m.moe_pffn_forward(0, S_in, V)
        elif score:
            m.score(Emb, hw, 0.1, p_out)
        elif train:
            m.stack_forward_train(X0, pooled)
            m.stack_backward_saved(dP, dX0, grads)
            allreduce_grads(gflat)          # the replicas' gradient sum (N > 1)
        else:
            m.stack_forward(X0, pooled)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)                  # let nvidia-smi come up

    def timed(profiled: bool):
        """K steps between two CUDA events on the launching stream (barrier and synchronize
        on both sides); profiled: with the library's per-kernel events around every launch."""
        m.profile(profiled)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        h0 = time.time()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        h1 = time.time()
        if world > 1:
            dist.barrier()
        ks = m.profile_read() if profiled else None
        m.profile(False)
        return ev0.elapsed_time(ev1), (h0, h1), ks

    # The timed region runs without per-kernel events: the kernels are launched with
    # programmatic stream serialization, and an event between two launches would hold
    # the second back until the first ends.  The same K steps then run again with the
    # per-kernel events, for the kernel split and the dominant kernel's launch time.
    ms_total, window, _ = timed(False)
    clocks.mark(*window)
    ms_total_prof, _, kstats = timed(True)
    clk = clocks.stop()
    status = m.sync_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    ms_max = max_over_ranks(ms_total, dev)
    ms_step = ms_max / args.steps
    samples_per_s = job_rate(B, world, args.steps, ms_max / 1e3)

    # ---- e2e through the host-buffer entry point -----------------------------------
    e2e = None
    if score:
        Eh = Emb.cpu().pin_memory()
        ph_ = torch.empty(B, dtype=torch.float32).pin_memory()

        def step_host():
            Emb.copy_(Eh, non_blocking=True)
            m.score(Emb, hw, 0.1, p_out)
            ph_.copy_(p_out, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        for _ in range(2):
            step_host()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step_host()
        t1 = time.perf_counter()
        e2e = {"value": round(job_rate(B, world, args.steps, max_over_ranks(t1 - t0, dev)), 2), "unit": "samples/s",
               "h2d_bytes_per_step": int(Eh.numel() * Eh.element_size()),
               "d2h_bytes_per_step": int(ph_.numel() * ph_.element_size())}
    elif train and not moe:
        # host X0 and pooled-output gradient in, pooled output back: copies on the
        # compute stream around the same forward + backward calls
        Xh = X0.cpu().pin_memory()
        dPh = dP.cpu().pin_memory()
        ph = torch.empty((B, D), dtype=torch.float32).pin_memory()

        def step_host():
            X0.copy_(Xh, non_blocking=True)
            dP.copy_(dPh, non_blocking=True)
            m.stack_forward_train(X0, pooled)
            m.stack_backward_saved(dP, dX0, grads)
            allreduce_grads(gflat)
            ph.copy_(pooled, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        for _ in range(2):
            step_host()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step_host()
        t1 = time.perf_counter()
        e2e = {"value": round(job_rate(B, world, args.steps, max_over_ranks(t1 - t0, dev)), 2), "unit": "samples/s",
               "h2d_bytes_per_step": int(Xh.numel() * Xh.element_size() + dPh.numel() * dPh.element_size()),
               "d2h_bytes_per_step": int(ph.numel() * ph.element_size())}
    elif not moe:
        # the serving loop through the pipelined host entry: batch i + 1 is enqueued (its
        # copy in overlaps batch i's compute) before batch i's pooled output is waited for;
        # every step's H2D copy of X0 and D2H copy of pooled lie inside the timed region
        Xh = X0.cpu().pin_memory()
        ph = [torch.empty((B, D), dtype=torch.float32).pin_memory() for _ in range(2)]

        def serve(n):
            prev = None
            for i in range(n):
                t = m.stack_forward_host_async(Xh, ph[i % 2])
                if prev is not None:
                    m.host_wait(prev)
                prev = t
            m.host_wait(prev)

        serve(3)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        serve(args.steps)
        t1 = time.perf_counter()
        ph = ph[0]
        e2e = {"value": round(job_rate(B, world, args.steps, max_over_ranks(t1 - t0, dev)), 2), "unit": "samples/s",
               "h2d_bytes_per_step": int(Xh.numel() * Xh.element_size()),
               "d2h_bytes_per_step": int(ph.numel() * ph.element_size())}

    # ---- roofline of the dominant kernel ------------------------------------------
    peaks, peak_src = load_peaks()
    peak, peak_why = pick_tensor_peak(peaks, peak_src, ms_max / 1e3, clk)
    flops_gemm = 2.0 * B * T * D * (k * D)          # one GEMM launch of the dense PFFN (either layer)
    gemm_kinds = ["moe_gemm1", "moe_gemm2"] if moe else ["gemm1", "gemm2", "pffn"]
    # flops per timed scope: one GEMM, or two (both FFN GEMMs of a layer in one launch, the
    # backward's data-gradient pair and recompute pair)
    scope_flops = {"gemm1": flops_gemm, "gemm2": flops_gemm, "pffn": 2 * flops_gemm, "bwd_wgrad": flops_gemm,
                   "bwd_dgrad": 2 * flops_gemm, "bwd_recompute": 2 * flops_gemm}
    # (bwd_recompute times the training forward of a layer: LN1 and both FFN layers)
    if train and not moe:
        gemm_kinds = ["gemm1", "gemm2", "bwd_wgrad", "bwd_dgrad", "bwd_recompute"]
    dom = max(gemm_kinds, key=lambda kk: kstats[kk][1])
    launches, tot_ms = kstats[dom]
    active = None
    if moe:
        # algorithmic flops: every open (sample, token, expert) runs 2 D Fe flops in each
        # expert layer, each layer one launch over all (token, expert) groups
        if train:
            active = int((Gt > 0).sum().item())
        else:
            _, G = m.moe_pffn_forward(0, S_in, V, return_gates=True)
            active = int((G > 0).sum().item())
        per_layer = 2.0 * active * D * Fe
        flops_launch = per_layer
        flops_step = 2 * per_layer + 2.0 * B * T * D * E * (2 if train else 1)      # + router(s)
    else:
        flops_launch = scope_flops[dom]
    roofline = None
    if launches > 0 and flops_launch:
        avg_ms = tot_ms / launches
        achieved = flops_launch / (avg_ms / 1e3) / 1e12
        kname = {"bwd_wgrad": "train_gemm_wgrad_tcgen05", "bwd_dgrad": "train_gemm_dgrad_tcgen05 (x2 per scope)",
                 "bwd_recompute": "train_gemm_forward_tcgen05 (x2 per scope)",
                 "pffn": "pffn_layer_tcgen05 (both FFN GEMMs of a layer)"}.get(dom, f"pffn_{dom}_tcgen05")
        roofline = {"kernel": kname, "bound": "tensor", "achieved": round(achieved, 1),
                    "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "traffic": captured_traffic(args.config, B, L, dom) if not (moe and train) else None,
                    "peak_source": peak_why,
                    "sm_mhz": clk.get("sm_mhz"),
                    "avg_launch_ms": round(avg_ms, 4)}
    flops_executed = None
    unimix_info = None
    if not moe:
        flops_step = 4.0 * k * L * T * D * D * B
        if unimix:
            # per layer and sample: the global product 2 nb^2 bs = 2 (T D)^2 / bs and the
            # local products 2 (T D) bs
            um_sample = 2.0 * (T * D) ** 2 / bs_um + 2.0 * T * D * bs_um
            flops_step += L * B * um_sample
            n_um, t_um = kstats["unimix"]
            if n_um:
                um_ms = t_um / n_um
                unimix_info = {"bs": bs_um, "nb": T * D // bs_um, "tau": UNIMIX_TAU, "iters": UNIMIX_ITERS,
                               "ms_per_layer": round(um_ms, 4),
                               "global_product_gflop_per_layer": round(2.0 * (T * D) ** 2 / bs_um * B / 1e9, 1),
                               "tflops_scope": round(B * um_sample / (um_ms / 1e3) / 1e12, 1),
                               "scope": "local block products + global product (tcgen05) + residual + LN1"}
        if score:
            flops_step += 2.0 * T * d_tok * D * B + 2.0 * D * B      # tokenizer + head
        if train:
            # forward + backward = 3 x the forward GEMM flops (the training forward keeps the
            # activations, so no GEMM runs twice)
            flops_executed = 3.0 * flops_step
            flops_step = 3.0 * flops_step
    gpu_launches = int(sum(v[0] for kk, v in kstats.items() if kk != "misc"))
    what = ("DTSI train forward" if moe else "train step: fwd + bwd") if train else (
        "score: tokenize + fwd + head" if score else ("fwd with UniMixing" if unimix else "fwd"))

    out = {
        "metric": f"samples/s (RankMixer-1B-shape block stack {what})" if args.config == "rankmixer_1b"
        else f"samples/s ({args.config} {'MoE PFFN' if moe else 'block stack'} {what})",
        "value": round(samples_per_s, 2),
        "unit": "samples/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs, N(0,1/fan_in) weights; random-init)",
        "config": {"workload": f"{args.config} B={B} T={T} D={D} k={k} L={L}" + (f" E={E} Fe={Fe}" if moe else "")
                   + (f" d={d_tok}" if score else "")
                   + (f" unimixing bs={bs_um} tau={UNIMIX_TAU}" if unimix else ""),
                   "batch_per_gpu": B, "global_batch": B * world,
                   "parallelism": f"replicas x{world} (batch sharded"
                   + (", gradients all-reduced)" if train and not moe and world > 1 else ")"),
                   "l2": "inputs larger than L2 (X0 %.0f MB, weights %.0f MB > 129 MB)" % (
                       X0.numel() * 2 / 1e6, m.info.weight_bytes / 1e6)},
        "tflops": round(flops_step * args.steps * world / (ms_max / 1e3) / 1e12, 1),
        "tflops_executed": round(flops_executed * args.steps * world / (ms_max / 1e3) / 1e12, 1)
        if flops_executed else None,
        "frac_of_peak_step": round(flops_step * args.steps / (ms_max / 1e3) / 1e12 / peak, 4),
        "roofline": roofline,
        "kernels_ms_per_step": {kk: round(v[1] / args.steps, 4) for kk, v in kstats.items() if v[0]},
        "ms_per_step_profiled": round(max_over_ranks(ms_total_prof, dev) / args.steps, 4),
        "gpu_launches": gpu_launches,
        "moe_mean_active_experts": round(active / (B * T), 3) if moe else None,
        "unimix": unimix_info,
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.config, B, args.cpu_seconds, train=train, score=score,
                                           unimix=unimix)
    if rank == 0:
        print(json.dumps(out), flush=True)
    m.close()
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ----------------------------------------------------------------------------
def cpu_baseline(config: str, B_full: int, seconds: float, n_steps: int = 1, train: bool = False,
                 score: bool = False, unimix: bool = False) -> dict:
    import numpy as np

    import oracle
    from rankmixer_feature_interaction_gb300 import synth

    c = synth.CONFIGS[config]
    T, D, k, L = c["T"], c["D"], c["k"], c["L"]
    moe = config == "moe_1b"
    layers = synth.to_f64(synth.make_stack(T, D, k, L, 4242, "bf16", "cpu", E=c.get("E", 0), Fe=c.get("Fe", 0),
                                           active=c.get("active", 2.0)))
    if moe and train:
        layers[0].update(synth.to_f64(synth.make_train_router(T, D, c["E"], 4243, "bf16", "cpu", active=0.75 * c["E"])))
    d_tok = SCORE_SLICE.get(config, 0)
    if score:
        r = np.random.default_rng(4244)
        Wtok = r.standard_normal((T, d_tok, D)) / d_tok ** 0.5
        btok = 0.1 * r.standard_normal((T, D))
        hw = r.standard_normal(D) / D ** 0.5
    if unimix:
        for n, p in enumerate(layers):
            WG, WB = synth.make_unimix_weights(T, D, D // T, 4245 + n, "cpu")
            p["WG"] = oracle.sinkhorn(synth.to_f64(WG), UNIMIX_TAU, UNIMIX_ITERS)
            p["WB"] = oracle.sinkhorn(synth.to_f64(WB), UNIMIX_TAU, UNIMIX_ITERS)
    cores = oracle.num_threads()

    def run(nb):
        X = synth.to_f64(synth.make_input(nb, T, D, 99, "bf16", "cpu"))
        t0 = time.perf_counter()
        if moe and train:
            p = layers[0]
            oracle.moe_pffn_train(X, p["Wg_train"], p["bg_train"], p["Wg"], p["bg"], p["eW1"], p["eb1"], p["eW2"],
                                  p["eb2"])
        elif moe:
            p = layers[0]
            oracle.moe_pffn(X, p["Wg"], p["bg"], p["eW1"], p["eb1"], p["eW2"], p["eb2"])
        elif score:
            E_ = np.random.default_rng(99).standard_normal((nb, T * d_tok))
            oracle.head(oracle.stack_forward(oracle.tokenize(E_, Wtok, btok), layers), hw, 0.1)
        elif train:
            oracle.stack_forward(X, layers)
            oracle.stack_backward(X, np.full((nb, D), 1.0 / nb), layers)
        elif unimix:
            oracle.stack_forward_unimix(X, layers)
        else:
            oracle.stack_forward(X, layers)
        return time.perf_counter() - t0

    probe_n = max(1, cores)
    run(probe_n)                     # first touch of the weights
    dt = run(probe_n)
    per_sample = dt / probe_n
    nb = int(max(probe_n, min(4096, seconds / max(per_sample, 1e-9))))
    nb = max(probe_n, (nb // probe_n) * probe_n)
    total_t, total_n = 0.0, 0
    for _ in range(n_steps):
        total_t += run(nb)
        total_n += nb
    return {"value": round(total_n / total_t, 3), "unit": "samples/s", "cores": cores, "kind": "oracle",
            "sample": f"{nb} samples of the {config} workload per step (of B={B_full}), float64 oracle"
                      f"{' forward + backward' if train else ''}{' with UniMixing' if unimix else ''}, "
                      f"OpenMP over samples on {cores} host threads, {n_steps} step(s), {total_t:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from rankmixer_feature_interaction_gb300 import synth
    c = synth.CONFIGS[args.config]
    B = args.batch or c["B"]
    steps = max(1, args.steps)
    # each step is a bounded sample; the whole run is kept to a few minutes
    per_step_s = min(args.cpu_seconds, 150.0 / (steps + args.warmup))
    train = args.pass_ == "train"
    score = args.pass_ == "score"
    unimix = args.pass_ == "unimix"
    moe = args.config == "moe_1b"
    cb = cpu_baseline(args.config, B, per_step_s, n_steps=steps, train=train, score=score, unimix=unimix)
    what = ("DTSI train forward" if moe else "train step: fwd + bwd") if train else (
        "score: tokenize + fwd + head" if score else ("fwd with UniMixing" if unimix else "fwd"))
    out = {
        "impl": "reference",
        "metric": f"samples/s (RankMixer-1B-shape block stack {what})" if args.config == "rankmixer_1b"
        else f"samples/s ({args.config}{' ' + what if (train or score or unimix) else ''})",
        "value": cb["value"], "unit": "samples/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": f"{args.config} B={B} T={c['T']} D={c['D']} k={c['k']} L={c['L']}"},
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": "samples/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def launch_ranks(n: int, argv: list[str]) -> int:
    """Run this script as n ranks on this node (one process per GPU) under
    torch.distributed.run, rendezvous on 127.0.0.1; returns its exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=["rankmixer_1b", "rankmixer_100m", "moe_1b"], default="rankmixer_1b")
    ap.add_argument("--batch", type=int, default=0, help="override the batch per GPU")
    ap.add_argument("--layers", type=int, default=0, help="override the number of layers (profiling captures)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU oracle budget per measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "train", "score", "unimix"], default="fwd",
                    help="fwd: the forward stack (the headline); train: forward + backward of the stack (with "
                         "moe_1b: the dense-training MoE forward); score: tokenization + stack + head; unimix: "
                         "the forward stack with UniMixing in place of TokenMixing in every layer")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ:
        if args.gpus > 1:               # N ranks, one per GPU, launched here
            raise SystemExit(launch_ranks(args.gpus, argv))
    elif int(os.environ["WORLD_SIZE"]) != args.gpus:
        ap.error(f"--gpus {args.gpus} disagrees with WORLD_SIZE={os.environ['WORLD_SIZE']} of the launcher")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
