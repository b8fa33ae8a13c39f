"""Benchmark of the hot path: one step = AdaLN modulate + dense attention (head
groups) + gated residual over one synthetic batch of the 10 s clip at
1344x768 (72,576 tokens, 56 heads x 128, hidden 5,376).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fv|reference]

Prints one JSON line.  ``value`` is attention TFLOP/s (4 N^2 d H per step over
the whole step time, all ranks); ``roofline`` is the attention kernel's own
rate against the measured bf16 peak; ``e2e`` times the same step through the
C ABI with inputs copied from pinned host memory and results read back;
``cpu_baseline`` times the fp64 oracle on a bounded sample of the step.
``--impl reference`` times only that oracle (the slow reference arm).
Under torchrun every rank runs its own copy of the workload (independent
problems, no collective on the data path) and rank 0 prints.
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "attention TFLOP/s (4*N^2*d*H) at N=72,576, 56x128 heads; % of GB300 BF16 peak"
UNIT = "TFLOP/s"
EPS = 1e-6
DATA = ("synthetic: seeded N(0,1) bf16 Q/K/V, residual x and branch output a; N(0,0.1^2) fp32 AdaLN tables "
        "(8 steps, step 3); no trained weights")


# The pages' own figures, each on its own hardware and for its own scope:
# context for the numbers above, not a target and not comparable with them.
PAGES_CONTEXT = {
    "attention_share_of_denoiser_runtime": {"value": ">85%", "kind": "reported", "model": "dense MiniMax H3"},
    "seconds_per_sampling_step_72576_tokens": {
        "values": {"32 GiB VRAM cap": 8.93, "8 GiB VRAM cap": 12.7, "8 GiB VRAM + 8 GiB RAM": 15.1},
        "hardware": "1x H200 (capped)", "scope": "whole DiT step at 1344x768, 243 frames, weight streaming included"},
    "end_to_end_10s_clip_1344x768_s": {"value": 122, "hardware": "GeForce RTX 5090 32 GB + 64 GB RAM",
                                       "scope": "full two-pass pipeline (8 half- + 3 full-resolution steps)"},
}

def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16_tflops": d.get("bf16_tflops"), "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d.get("hbm_gbs"), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def attn_source_hash() -> str:
    """Hash of the attention kernel's sources; ties recorded ncu traffic to them."""
    import hashlib
    h = hashlib.sha256()
    for f in ("attn_fwd.cu", "sm103_ptx.cuh"):
        with open(os.path.join(ROOT, "video_diffusion_transformer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value across ranks (the job's wall time is its slowest rank)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

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
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------- CPU oracle
def oracle_sample(w: W.Workload, q, k, v, x_mod, shift, scale, x_res, a, gate, rows_per_head: int):
    """Run the fp64 oracle over a bounded sample of one step: the same
    rows_per_head query rows of every head, and that many rows of the two
    elementwise ops.  Returns (seconds, attention FLOPs of the sample)."""
    import numpy as np

    import oracle
    sc = 1.0 / math.sqrt(W.HEAD_DIM)
    t0 = time.perf_counter()
    rows_e = np.arange(rows_per_head, dtype=np.int64) * max(1, w.n // max(1, rows_per_head))
    oracle.modulate(x_mod, shift[W.ADALN_STEP].numpy(), scale[W.ADALN_STEP].numpy(), EPS, rows=rows_e)
    outs = []
    for h in range(w.heads):
        rows = W.sampled_rows(w.n, h, rows_per_head).numpy()[:rows_per_head]
        outs.append((h, rows, oracle.attn_rows(q, k, v, h, rows, sc)[0]))
    oracle.gated_residual(x_res, a, gate[W.ADALN_STEP].numpy(), rows=rows_e)
    dt = time.perf_counter() - t0
    return dt, 4.0 * w.n * W.HEAD_DIM * rows_per_head * w.heads, outs


def oracle_elementwise(x_mod, shift, scale, x_res, a, gate, rows: int) -> dict:
    """The oracle's modulate and gated residual timed on their own over
    ``rows`` rows spread through the tensors, in GB/s of the ops' algorithmic
    bytes (bf16 in and out: 4 B per element for modulate, 6 for the gated
    residual; the oracle itself computes in float64), and extrapolated to the
    14.4 s clip's 102,816 x 5,376 tensors."""
    import numpy as np

    import oracle
    n = x_mod.shape[0]
    idx = np.arange(rows, dtype=np.int64) * max(1, n // rows)
    full_rows = W.video_tokens(1344, 768, 345)
    out = {}
    for name, per_elem, fn in (
            ("adaln_modulate", 4, lambda: oracle.modulate(x_mod, shift[W.ADALN_STEP].numpy(),
                                                          scale[W.ADALN_STEP].numpy(), EPS, rows=idx)),
            ("gated_residual", 6, lambda: oracle.gated_residual(x_res, a, gate[W.ADALN_STEP].numpy(), rows=idx))):
        t0 = time.perf_counter()
        fn()
        dt = time.perf_counter() - t0
        nbytes = rows * W.HIDDEN * per_elem
        out[name] = {"gbs": nbytes / dt / 1e9, "rows": rows, "s": dt,
                     "extrapolated_full_s": dt * full_rows / rows,
                     "extrapolated_to": f"{full_rows} x {W.HIDDEN}"}
    return out


def sample_errors(o_gpu: torch.Tensor, outs) -> dict:
    """max-abs / mean-abs of the GPU output on the oracle's sampled rows."""
    o_cpu = o_gpu.detach().cpu()
    worst, tot, cnt = 0.0, 0.0, 0
    for h, rows, ref in outs:
        got = o_cpu[rows, h * W.HEAD_DIM:(h + 1) * W.HEAD_DIM].to(torch.float64).numpy()
        d = abs(got - ref)
        worst = max(worst, float(d.max()))
        tot += float(d.sum())
        cnt += d.size
    return {"max_abs": worst, "mean_abs": tot / max(1, cnt), "rows": cnt // W.HEAD_DIM,
            "pass": worst <= 2e-2 and tot / max(1, cnt) <= 2e-3}


def cpu_inputs(w: W.Workload):
    q, k, v = W.qkv(w)
    x_mod, shift, scale = W.modulate_inputs(w, rows=w.n)
    x_res, a, gate = W.gated_residual_inputs(w, rows=w.n)
    return q, k, v, x_mod, shift, scale, x_res, a, gate


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores, each step a
    bounded sample of the workload, scaled to attention TFLOP/s."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = workload_of(args)
    inputs = cpu_inputs(w)
    rows = args.ref_rows
    times = []
    flops = 0.0
    for i in range(args.warmup + args.steps):
        dt, flops, _ = oracle_sample(w, *inputs, rows_per_head=rows)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = flops * len(times) / total / 1e12
    cores = os.cpu_count()
    sample = f"{rows} query rows of each of the {w.heads} heads (of {w.n}) + {rows} rows of modulate and gated residual"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_of(args) -> W.Workload:
    """The named workload, or (--heads) the same workload with fewer heads: a
    small case of the same kernels for profiling."""
    w = W.WORKLOADS[args.workload]
    if args.heads is None:
        return w
    import dataclasses
    return dataclasses.replace(w, heads=args.heads, head_group=min(w.head_group, args.heads))


def config_of(w: W.Workload) -> dict:
    groups = [min(w.head_group, w.heads - h0) for h0 in range(0, w.heads, w.head_group)]
    return {"workload": w.name, "tokens": w.n, "heads": w.heads, "head_dim": W.HEAD_DIM,
            "head_groups": groups, "hidden": W.HIDDEN, "adaln_step": W.ADALN_STEP,
            "step": "adaln_modulate -> attention (head groups) -> gated_residual",
            "l2": l2_note(w)}


def l2_note(w: W.Workload) -> str:
    """How the timed step stands to L2: its resident working set (Q, K, V, O
    and the elementwise operands) against the 126 MB L2."""
    # the bench runs both elementwise ops on all N rows (bf16 x, y; x, a, out)
    ws = 4 * w.n * w.heads * W.HEAD_DIM * 2 + w.n * W.HIDDEN * 4 + w.n * W.HIDDEN * 6
    if ws > 126e6:
        return f"inputs larger than L2 ({ws / 1e9:.1f} GB resident working set vs 126 MB L2); no flush"
    return f"working set {ws / 1e6:.0f} MB fits in L2 (126 MB); L2-resident timing, not a bench workload"


# ---------------------------------------------------------------- GPU arm
def run_fv(args):
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        from video_diffusion_transformer_gb300 import build as fbuild
        fbuild.build()
    barrier(world)
    import video_diffusion_transformer_gb300 as fv
    fv.load_library()

    w = workload_of(args)
    cpu = cpu_inputs(w)
    q_h, k_h, v_h, xm_h, shift_h, scale_h, xr_h, a_h, gate_h = cpu
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    xm, xr, a = xm_h.to(dev), xr_h.to(dev), a_h.to(dev)
    shift, scale, gate = shift_h.to(dev), scale_h.to(dev), gate_h.to(dev)
    o = torch.empty_like(q)
    y = torch.empty((w.n, W.HIDDEN), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(xr)
    stream = torch.cuda.Stream(device=dev)
    launches_per_step = 1 + len(range(0, w.heads, w.head_group)) + 1

    def step(ev0=None, ev1=None):
        fv.adaln_modulate(xm, shift, scale, W.ADALN_STEP, eps=EPS, out=y, stream=stream)
        if ev0 is not None:
            ev0.record(stream)
        fv.attn_fwd(q, k, v, o, head_group=w.head_group, stream=stream)
        if ev1 is not None:
            ev1.record(stream)
        fv.gated_residual(xr, a, gate, W.ADALN_STEP, out=out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
        fv.sync_status(stream)

        # ---- device-resident timing
        ev_a = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        barrier(world)
        torch.cuda.synchronize(dev)
        start.record(stream)
        for i in range(args.steps):
            step(*ev_a[i])
        end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        clocks = sampler.stop()
        fv.sync_status(stream)
        ms_total = start.elapsed_time(end)
        attn_ms = [e0.elapsed_time(e1) for e0, e1 in ev_a]

        # ---- windowed attention (the Video DeltaNet softmax branch) on the same Q, K, V
        window = None
        if not args.no_window and w.n % W.tokens_per_latent_frame(1344, 768) == 0:
            t_f = W.tokens_per_latent_frame(1344, 768)
            ow = torch.empty_like(q)
            for _ in range(2):
                fv.attn_fwd_window(q, k, v, ow, frame_tokens=t_f, chunk_frames=5, window_chunks=1,
                                   head_group=w.head_group, stream=stream)
            reps = 5
            w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            w0.record(stream)
            for _ in range(reps):
                fv.attn_fwd_window(q, k, v, ow, frame_tokens=t_f, chunk_frames=5, window_chunks=1,
                                   head_group=w.head_group, stream=stream)
            w1.record(stream)
            torch.cuda.synchronize(dev)
            fv.sync_status(stream)
            wms = w0.elapsed_time(w1) / reps
            pairs = W.window_pairs(w.n, t_f, 5, 1)
            window = {"kernel": "attn_fwd_kernel (window)", "frame_tokens": t_f, "chunk_frames": 5,
                      "window_chunks": 1, "density": pairs / float(w.n) ** 2, "ms": wms,
                      "effective_tflops": 4.0 * W.HEAD_DIM * w.heads * pairs / (wms / 1e3) / 1e12,
                      "speedup_vs_dense": (sum(attn_ms) / len(attn_ms)) / wms}

        # ---- Video Delta Attention (the VDN linear branch) on the same Q, K, V
        delta = None
        if not args.no_window and w.n % W.tokens_per_latent_frame(1344, 768) == 0:
            t_f = W.tokens_per_latent_frame(1344, 768)
            frames = w.n // t_f
            gd = torch.Generator(device="cpu").manual_seed(77)
            beta = torch.sigmoid(torch.randn((w.heads, w.n), generator=gd)).to(dev)
            alpha = (0.9 + 0.1 * torch.rand((w.heads, frames, W.HEAD_DIM), generator=gd)).to(dev)
            tstate = (torch.randn((w.heads, W.HEAD_DIM, W.HEAD_DIM), generator=gd) * 0.1).to(dev)
            od = torch.empty_like(q)
            st_shape = (2, w.heads, frames, W.HEAD_DIM, W.HEAD_DIM)
            states = torch.empty(st_shape, dtype=torch.float32, device=dev)
            wsp = torch.empty(st_shape, dtype=torch.float32, device=dev)

            def run_delta():
                fv.delta_attn(q, k, v, beta, alpha, frame_tokens=t_f, chunk_frames=5, window_chunks=1,
                              text_state=tstate, out=od, states=states, workspace=wsp, stream=stream)

            run_delta()
            reps = 5
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            d0.record(stream)
            for _ in range(reps):
                run_delta()
            d1.record(stream)
            torch.cuda.synchronize(dev)
            fv.sync_status(stream)
            dms = d0.elapsed_time(d1) / reps
            dd = W.HEAD_DIM
            written = max(0, frames - 2)
            flops = w.heads * (written * (4.0 * t_f * dd * dd + 4.3 * dd ** 3 + 2 * 2.0 * dd ** 3)
                               + frames * 2.0 * t_f * dd * dd)
            delta = {"kernels": "vda_stats_tc, vda_solve, vda_scan_tc, vda_wsplit, vda_readout_tc", "ms": dms,
                     "gflop": flops / 1e9, "tflops": flops / (dms / 1e3) / 1e12,
                     "vdn_hybrid_ms": (window["ms"] + dms) if window else None}

        # ---- VSA-style block-sparse attention: (4, 4, 4) tiles of the latent
        # grid, 90% sparsity, on the same Q, K, V
        vsa = None
        if not args.no_window and w.n % W.tokens_per_latent_frame(1344, 768) == 0:
            lat_h, lat_w = 768 // 32, 1344 // 32
            frames = w.n // (lat_h * lat_w)
            nt = fv.vsa_num_tiles(frames, lat_h, lat_w)
            topk = fv.vsa_topk(nt, 0.9)
            ov = torch.empty_like(q)
            sel = torch.empty((w.heads, nt, topk), dtype=torch.int32, device=dev)
            wsv = torch.empty(fv.load_library().fv_vsa_workspace_bytes(w.heads, frames, lat_h, lat_w, topk),
                              dtype=torch.uint8, device=dev)

            def run_vsa():
                fv.vsa_attn(q, k, v, frames=frames, height=lat_h, width=lat_w, topk=topk, out=ov, selected=sel,
                            workspace=wsv, stream=stream)

            for _ in range(2):
                run_vsa()
            reps = 5
            v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            v0.record(stream)
            for _ in range(reps):
                run_vsa()
            v1.record(stream)
            torch.cuda.synchronize(dev)
            fv.sync_status(stream)
            vms = v0.elapsed_time(v1) / reps
            # useful work: every query against the real tokens of its kept tiles
            tw, th = (lat_w + 3) // 4, (lat_h + 3) // 4
            b = np.arange(nt)
            sizes = (np.minimum(4, lat_w - 4 * (b % tw)) * np.minimum(4, lat_h - 4 * ((b // tw) % th))
                     * np.minimum(4, frames - 4 * (b // (tw * th))))
            kept = sizes[sel.cpu().numpy()].sum(axis=2)
            flops = 4.0 * W.HEAD_DIM * float((kept * sizes[None, :]).sum())
            vsa = {"kernels": "vsa_pool, vsa_select, vsa_fine", "grid": [frames, lat_h, lat_w], "tiles": nt,
                   "topk": topk, "sparsity": 0.9, "ms": vms, "useful_tflop": flops / 1e12,
                   "effective_tflops": flops / (vms / 1e3) / 1e12,
                   "speedup_vs_dense": (sum(attn_ms) / len(attn_ms)) / vms}

        # ---- the elementwise kernels alone, on the 14.4 s clip's 102,816 rows:
        # L2 flushed (512 MB written) before every rep, 20 reps, median and best
        elementwise = None
        if not args.no_window and args.heads is None:
            rows = W.video_tokens(1344, 768, 345)
            ge = torch.Generator(device=dev)
            ge.manual_seed(4)
            ex = torch.randn((rows, W.HIDDEN), generator=ge, device=dev).to(torch.bfloat16)
            ea = torch.randn((rows, W.HIDDEN), generator=ge, device=dev).to(torch.bfloat16)
            ey, eo = torch.empty_like(ex), torch.empty_like(ex)
            flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
            hbm = peaks()["hbm_gbs"]

            def time_reps(fn, reps=20):
                fn()
                times = []
                for _ in range(reps):
                    flush.fill_(1)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                    e1.synchronize()
                    times.append(e0.elapsed_time(e1))
                return statistics.median(times), min(times)

            # per-token modality rows: three modalities (row step * 3 + tag),
            # tags drawn per token (the most mixed packing)
            nmod = 3
            tags = torch.randint(0, nmod, (rows,), generator=ge, device=dev, dtype=torch.int64).to(torch.uint8)
            shift_t, scale_t, gate_t = (t.repeat_interleave(nmod, dim=0).contiguous() for t in (shift, scale, gate))
            with torch.cuda.stream(stream):
                mod = time_reps(lambda: fv.adaln_modulate(ex, shift, scale, W.ADALN_STEP, eps=EPS, out=ey,
                                                          stream=stream))
                gre = time_reps(lambda: fv.gated_residual(ex, ea, gate, W.ADALN_STEP, out=eo, stream=stream))
                mod_t = time_reps(lambda: fv.adaln_modulate_tagged(ex, shift_t, scale_t, W.ADALN_STEP, tags, nmod,
                                                                   eps=EPS, out=ey, stream=stream))
                gre_t = time_reps(lambda: fv.gated_residual_tagged(ex, ea, gate_t, W.ADALN_STEP, tags, nmod, out=eo,
                                                                   stream=stream))
            fv.sync_status(stream)
            mod_bytes = rows * W.HIDDEN * 4 + 2 * W.HIDDEN * 4
            gre_bytes = rows * W.HIDDEN * 6 + W.HIDDEN * 4

            def entry(t, nbytes):
                med, best = t
                return {"median_ms": med, "best_ms": best, "bytes": nbytes, "gbs_median": nbytes / med / 1e6,
                        "gbs_best": nbytes / best / 1e6,
                        "frac_of_hbm_median": (nbytes / med / 1e6) / hbm if hbm else None}

            # the small configurations' operands (1,008 rows of modulate, 5,040 of
            # the gated residual, <= 163 MB) stay in L2 between reps: timed
            # without the flush and labelled so
            def time_resident(fn, reps=20):
                fn()
                times = []
                for _ in range(reps):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                    e1.synchronize()
                    times.append(e0.elapsed_time(e1))
                return statistics.median(times), min(times)

            rm = W.tokens_per_latent_frame(1344, 768)   # 1,008 rows: one latent frame
            rg = 5 * rm                                  # 5,040 rows: one 17-frame VAE chunk
            with torch.cuda.stream(stream):
                mod_s = time_resident(lambda: fv.adaln_modulate(ex[:rm], shift, scale, W.ADALN_STEP, eps=EPS,
                                                                out=ey[:rm], stream=stream))
                gre_s = time_resident(lambda: fv.gated_residual(ex[:rg], ea[:rg], gate, W.ADALN_STEP, out=eo[:rg],
                                                                stream=stream))
            fv.sync_status(stream)
            resident = {"flush": "none: the operands stay in L2 (labelled L2-resident)", "reps": 20,
                        "adaln_modulate_bf16": dict(entry(mod_s, rm * W.HIDDEN * 4 + 2 * W.HIDDEN * 4), rows=rm),
                        "gated_residual": dict(entry(gre_s, rg * W.HIDDEN * 6 + W.HIDDEN * 4), rows=rg)}
            elementwise = {"rows": rows, "hidden": W.HIDDEN, "flush": "512 MB written before every rep",
                           "reps": 20, "peak_gbs": hbm, "adaln_modulate_bf16": entry(mod, mod_bytes),
                           "l2_resident_small": resident,
                           "gated_residual": entry(gre, gre_bytes),
                           "tagged": {"modalities": nmod, "tags": "one per token, seeded uniform",
                                      "adaln_modulate_bf16": entry(mod_t, rows * W.HIDDEN * 4 + rows
                                                                   + nmod * 2 * W.HIDDEN * 4),
                                      "gated_residual": entry(gre_t, rows * W.HIDDEN * 6 + rows
                                                              + nmod * W.HIDDEN * 4)}}
            del ex, ea, ey, eo, flush, tags

        # ---- end to end through the C ABI: pinned host inputs in, results out.
        # Every step copies its own inputs host->device and reads its results
        # back; copies run on their own streams, double-buffered, so step i's
        # copies overlap the compute of its neighbours.  Each kernel waits only
        # for its own inputs (modulate for x, attention for Q, K, V, the gated
        # residual for x and the branch output), and each result is read back
        # as soon as its kernel is done.
        e2e = None
        if not args.no_e2e:
            # input groups in copy order: modulate's, attention's, gated residual's
            groups_h = [[xm_h], [q_h, k_h, v_h], [xr_h, a_h]]
            pin = [[t.pin_memory() for t in g] for g in groups_h]
            outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (y, o, out)]
            h2d = sum(t.numel() * t.element_size() for g in pin for t in g)
            d2h = sum(t.numel() * t.element_size() for t in outs_h)
            ins = [[[xm], [q, k, v], [xr, a]],
                   [[torch.empty_like(xm)], [torch.empty_like(t) for t in (q, k, v)],
                    [torch.empty_like(t) for t in (xr, a)]]]
            outs = [[y, o, out], [torch.empty_like(t) for t in (y, o, out)]]
            s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
            ev = {name: [torch.cuda.Event(), torch.cuda.Event()] for name in ("in_free", "read")}
            ev_in = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]    # group g of buffer b landed
            ev_out = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]   # result r of buffer b ready

            def run_pipelined(nsteps):
                for i in range(nsteps):
                    b = i % 2
                    if i >= 2:
                        s_h2d.wait_event(ev["in_free"][b])
                    with torch.cuda.stream(s_h2d):
                        for g, (dsts, srcs) in enumerate(zip(ins[b], pin)):
                            for d, src in zip(dsts, srcs):
                                d.copy_(src, non_blocking=True)
                            ev_in[b][g].record(s_h2d)
                    if i >= 2:
                        stream.wait_event(ev["read"][b])
                    (xmm,), (qq, kk, vv), (xrr, aa) = ins[b]
                    yy, oo, oout = outs[b]
                    with torch.cuda.stream(stream):
                        stream.wait_event(ev_in[b][0])
                        fv.adaln_modulate(xmm, shift, scale, W.ADALN_STEP, eps=EPS, out=yy, stream=stream)
                        ev_out[b][0].record(stream)
                        stream.wait_event(ev_in[b][1])
                        fv.attn_fwd(qq, kk, vv, oo, head_group=w.head_group, stream=stream)
                        ev_out[b][1].record(stream)
                        stream.wait_event(ev_in[b][2])
                        fv.gated_residual(xrr, aa, gate, W.ADALN_STEP, out=oout, stream=stream)
                        ev_out[b][2].record(stream)
                        ev["in_free"][b].record(stream)
                    with torch.cuda.stream(s_d2h):
                        for r, (hdst, dsrc) in enumerate(zip(outs_h, outs[b])):
                            s_d2h.wait_event(ev_out[b][r])
                            hdst.copy_(dsrc, non_blocking=True)
                        ev["read"][b].record(s_d2h)

            run_pipelined(max(2, args.warmup // 2))
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(world)
            torch.cuda.synchronize(dev)
            t_wall = time.perf_counter()
            e0.record(s_h2d)
            run_pipelined(args.steps)
            s_h2d.wait_stream(s_d2h)
            e1.record(s_h2d)
            torch.cuda.synchronize(dev)
            t_wall = time.perf_counter() - t_wall
            barrier(world)
            fv.sync_status(stream)
            e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
            e2e = {"value": world * w.flops * args.steps / (e2e_ms / 1e3) / 1e12, "unit": UNIT,
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "ms_per_step": e2e_ms / args.steps, "wall_ms_per_step": 1e3 * t_wall / args.steps,
                   "copies": "own streams, double-buffered, overlapped with neighbouring steps' compute; "
                             "each kernel waits for its own inputs, each result is read back when its kernel is done"}

    ms_total = max_over_ranks(ms_total, world, dev)

    # CPU baseline: the oracle on a bounded sample of the step (rank 0, one GPU).
    # Its attention rows double as a parity check of the output just timed.
    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, fl, outs = oracle_sample(w, q_h, k_h, v_h, xm_h, shift_h, scale_h, xr_h, a_h, gate_h,
                                     rows_per_head=args.cpu_rows)
        cpu_baseline = {"value": fl / dt / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                        "sample": f"{args.cpu_rows} query rows of each of the {w.heads} heads (of {w.n}) + "
                                  f"{args.cpu_rows} rows of modulate and gated residual; {dt:.1f} s",
                        "parity_of_timed_output": sample_errors(o, outs),
                        "extrapolated_full_attention_s": w.flops / (fl / dt),
                        "elementwise": oracle_elementwise(xm_h, shift_h, scale_h, xr_h, a_h, gate_h,
                                                          rows=args.cpu_ew_rows)}

    if rank != 0:
        return 0
    pk = peaks()
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    achieved = w.flops / (attn_avg_ms / 1e3) / 1e12
    # Each attention launch is timed alone (CUDA events around it) at the
    # clock it runs at, far above the clock of the sustained matmul loop: the
    # burst figure is the denominator, the sustained ratio a second field.
    peak = pk["bf16_tflops"]
    sustained = pk["bf16_tflops_sustained"]
    # DRAM bytes of the step's attention launches, from one ncu capture of a
    # single 16-head launch of this workload (a step's 16-head launches are the
    # same launch), scaled by heads; null once the kernel source has changed.
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof):
        rec = json.load(open(prof)).get(w.name)
        if rec and rec.get("kernel_source") == attn_source_hash():
            traffic = rec["attn_fwd_kernel_bytes"] * w.heads / rec["heads_captured"]
    value = world * w.flops * args.steps / (ms_total / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": DATA, "config": config_of(w),
        "pct_of_bf16_peak": {"burst": 100.0 * value / pk["bf16_tflops"] if pk["bf16_tflops"] else None,
                             "sustained": 100.0 * value / peak if peak else None, "peaks": pk["source"]},
        "roofline": {"kernel": "attn_fwd_kernel", "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak if peak else None, "traffic": traffic,
                     "peak_kind": f"bf16_tflops, burst ({pk['source']})",
                     "frac_of_sustained": achieved / sustained if sustained else None,
                     "per": f"one step's {len(range(0, w.heads, w.head_group))} head-group launches, "
                            f"{w.flops / 1e12:.2f} TFLOP, avg {attn_avg_ms:.2f} ms"},
        "e2e": e2e, "cpu_baseline": cpu_baseline, "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "elementwise_ms_per_step": (ms_total / args.steps) - attn_avg_ms,
        "vdn_window_attention": window,
        "vdn_delta_attention": delta,
        "vsa_block_sparse_attention": vsa,
        "elementwise_alone": elementwise,
        "context": PAGES_CONTEXT,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("fv", "reference"), default="fv")
    ap.add_argument("--workload", default=W.HEADLINE, choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-rows", type=int, default=256, help="oracle query rows per head for cpu_baseline")
    ap.add_argument("--ref-rows", type=int, default=16, help="oracle query rows per head per reference step")
    ap.add_argument("--cpu-ew-rows", type=int, default=8192,
                    help="rows of the oracle's modulate and gated residual timed alone for cpu_baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-window", action="store_true",
                    help="skip the side measurements (windowed, delta and VSA attention, elementwise kernels alone)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=None,
                    help="run the workload with this many heads (a small case of the same kernels, for "
                         "profiling); the elementwise kernels are then not timed alone")
    args = ap.parse_args(argv)
    if args.heads is not None and not 1 <= args.heads <= W.WORKLOADS[args.workload].heads:
        ap.error("--heads must be between 1 and the workload's head count")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


def main(argv=None):
    args = parse(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_fv(args)


if __name__ == "__main__":
    sys.exit(main())
