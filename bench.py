"""Benchmark of the attention hot path on GB300.

One step = one pass of every stage of the path over the long-context workload
B=2, H=16, N=8192, d=128 (16K tokens, the 8K/128 shape):
  1. BF16 forward              (attn_fwd)
  2. BF16 backward             (attn_bwd: row-dot pre-pass, main kernel, dQ conversion)
  3. FP8 pre-pass              (attn_fp8_quantize_bf16: block scales + Hadamard on Q, K,
                                read from the same bfloat16 Q, K, V as the BF16 stages)
  4. FP8 forward               (attn_fwd_fp8)
Inputs are seeded synthetic N(0,1) tensors (bfloat16) resident in HBM before
timing; together they are larger than the 129 MB L2, so no explicit flush is done.

value = algorithmic TFLOP per step / step time, with forward FLOP =
4*B*H*N^2*d (halved if causal), backward = 2.5x forward, FP8 forward = forward.
The pre-pass does no tensor-core work and is reported in GB/s.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--causal] [--impl reference]
Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas, weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B, H, N, D = 2, 16, 8192, 128
METRIC = "Attn fwd/bwd TFLOP/s (BF16, FP8) & % of GB300 dense tensor peak, N=8K d=128"
WORKLOAD = "attention step (bf16 fwd + bf16 bwd + fp8 pre-pass + fp8 fwd), B=2 H=16 N=8192 d=128"

# DRAM bytes (read + write) per launch of each stage's main kernel, measured by
# ncu (dram__bytes_read.sum + dram__bytes_write.sum of one launch on this
# workload, non-causal).  "src" is the digest (see kernel_source_digest) of the
# kernel's source files when the capture was taken; once they change, the
# figure no longer describes the kernel and the line reports traffic as null.
NCU_TRAFFIC = {
    "fwd_bf16": {"bytes": 247_944_960, "src": "4556e39afb1bcd95"},      # 201.4 MB read + 46.5 MB write
    "bwd_bf16": {"bytes": 622_878_976, "src": "b46ee46459be4a33"},      # 404.9 MB read + 217.9 MB write
    "fwd_fp8": {"bytes": 129_437_184, "src": "e467db4535cb85c2"},       # 100.7 MB read + 28.7 MB write
    "fp8_prepass": {"bytes": 270_651_136, "src": "e467db4535cb85c2"},   # 201.4 MB read + 69.3 MB write
}
KERNEL_SOURCES = {"fwd_bf16": "fwd.cu", "bwd_bf16": "bwd.cu", "fwd_fp8": "fp8.cu",
                  "fp8_prepass": "fp8.cu"}
KERNEL_OF = {"fwd_bf16": "fwd_kernel", "bwd_bf16": "bwd_main_kernel (timed as the whole attn_bwd call)",
             "fwd_fp8": "fwd_fp8_kernel", "fp8_prepass": "fp8_quant_kernel"}


def kernel_source_digest(stage):
    """First 16 hex digits of the SHA-256 of the stage's kernel source file and
    the device primitives it includes."""
    import hashlib
    csrc = os.path.join(ROOT, "exact_tiled_attention_25_gb300", "csrc")
    h = hashlib.sha256()
    for name in (KERNEL_SOURCES[stage], "sm103_prims.cuh", "common.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def fwd_flop(causal):
    f = 4.0 * B * H * N * N * D
    return f / 2 if causal else f


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].strip() not in ("", "[N/A]"))}


def max_over_ranks(value, device):
    """Largest value over all ranks (the slowest rank's time defines the job)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(step_flop, ms_per_step, world):
    """Whole-job throughput: every rank runs one replica of the step (weak
    scaling), so the job does world * step_flop in the slowest rank's time."""
    return world * step_flop / (ms_per_step * 1e-3) / 1e12


def make_inputs(torch, dev, seed=3):
    g = torch.Generator(device=dev).manual_seed(seed)
    shape = (B, H, N, D)
    q, k, v, do = (torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
                   for _ in range(4))
    signs = torch.where(torch.rand(D, generator=g, device=dev) < 0.5, -1.0, 1.0).float()
    return q, k, v, do, signs


def run_ours(args, rank, world):
    import torch
    import exact_tiled_attention_25_gb300 as attn

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    attn.load_library()
    stream = torch.cuda.current_stream()
    causal = args.causal
    scale = 1.0 / math.sqrt(D)
    q32, k32, v32, do32, signs = make_inputs(torch, dev)
    q, k, v, do = (t.to(torch.bfloat16) for t in (q32, k32, v32, do32))
    del q32, k32, v32, do32
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, D), dtype=torch.uint8, device=dev)
    nblk = (N + 127) // 128
    q8, k8, v8 = (torch.empty((B, H, N, D), dtype=torch.uint8, device=dev) for _ in range(3))
    qs, ks, vs = (torch.empty((B, H, nblk), dtype=torch.float32, device=dev) for _ in range(3))
    o8 = torch.empty_like(q)
    lse8 = torch.empty_like(lse)
    rope = None
    if args.rope:
        # rotary tables: model constants, resident on the device like weights
        import workloads
        rope = tuple(torch.from_numpy(t).to(dev) for t in workloads.rope_tables(N, D))

    parts = {}

    def part_fwd():
        attn.attn_fwd(q, k, v, causal=causal, softmax_scale=scale, o=o, lse=lse)

    def part_bwd():
        attn.attn_bwd(q, k, v, o, do, lse, causal=causal, softmax_scale=scale,
                      dq=dq, dk=dk, dv=dv, workspace=ws)

    def part_quant():
        lib = attn.load_library()
        if rope is not None:
            code = lib.attn_fp8_quantize_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), 1,
                                            rope[0].data_ptr(), rope[1].data_ptr(), signs.data_ptr(),
                                            q8.data_ptr(), k8.data_ptr(), v8.data_ptr(),
                                            qs.data_ptr(), ks.data_ptr(), vs.data_ptr(), None,
                                            B, N, 0, H, H, D, 0, stream.cuda_stream)
            if code:
                raise attn.AttnError(code, "attn_fp8_quantize_ex")
            return
        code = lib.attn_fp8_quantize_bf16(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                          signs.data_ptr(), q8.data_ptr(), k8.data_ptr(),
                                          v8.data_ptr(), qs.data_ptr(), ks.data_ptr(), vs.data_ptr(),
                                          B, H, H, N, D, 0, stream.cuda_stream)
        if code:
            raise attn.AttnError(code, "attn_fp8_quantize_bf16")

    def part_fp8():
        attn.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=causal, softmax_scale=scale,
                          o=o8, lse=lse8)

    candidates = [("fwd_bf16", part_fwd, fwd_flop(causal), 1),
                  ("bwd_bf16", part_bwd, 2.5 * fwd_flop(causal), 3),
                  ("fp8_prepass", part_quant, 0.0, 1),
                  ("fwd_fp8", part_fp8, fwd_flop(causal), 1)]
    step_parts = []
    skipped = []
    for name, fn, flop, launches in candidates:
        try:
            fn()
            torch.cuda.synchronize()
            step_parts.append((name, fn, flop, launches))
        except attn.AttnError as e:
            if e.code != attn.ATTN_ERR_UNSUPPORTED:
                raise
            skipped.append(name)
    assert attn.attn_get_device_status() == 0, attn.attn_last_error()

    # prepass algorithmic bytes: read 3 bf16 tensors, write 3 e4m3 tensors + descales
    prepass_bytes = 3 * B * H * N * D * (2 + 1) + 3 * B * H * nblk * 4
    if rope is not None:
        prepass_bytes += 2 * N * (D // 2) * 4

    for _ in range(args.warmup):
        for _, fn, _, _ in step_parts:
            fn()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ev = {name: [] for name, *_ in step_parts}
    step_start = torch.cuda.Event(enable_timing=True)
    step_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        time.sleep(0.3)
        torch.cuda.synchronize()
        step_start.record(stream)
        for _ in range(args.steps):
            for name, fn, _, _ in step_parts:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ev[name].append((a, b))
        step_end.record(stream)
        torch.cuda.synchronize()
    total_ms = step_start.elapsed_time(step_end)
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
    assert attn.attn_get_device_status() == 0, attn.attn_last_error()
    ms_per_step = total_ms / args.steps
    step_flop = sum(f for _, _, f, _ in step_parts)
    value = aggregate_tflops(step_flop, ms_per_step, world)

    pk = peaks()
    # Each kernel is timed in isolation for well under a second at full clocks,
    # so the denominator is the measured burst figure (not the power-capped
    # seconds-long one); e4m3 takes 2x it, the nominal dense e4m3:bf16 ratio.
    bf16_peak = pk["bf16_tflops"]
    fp8_peak = 2.0 * bf16_peak
    breakdown = {}
    for name, _, flop, _ in step_parts:
        times = [a.elapsed_time(b) for a, b in ev[name]]
        avg = sum(times) / len(times)
        entry = {"ms": round(avg, 4), "share": round(sum(times) / total_ms, 4)}
        if flop:
            tf = flop / (avg * 1e-3) / 1e12
            peak = fp8_peak if name == "fwd_fp8" else bf16_peak
            entry.update(tflops=round(tf, 1), frac_of_peak=round(tf / peak, 4))
        else:
            gbs = prepass_bytes / (avg * 1e-3) / 1e9
            entry.update(gbs=round(gbs, 1), frac_of_hbm=round(gbs / pk["hbm_gbs"], 4))
        breakdown[name] = entry

    dominant = max(breakdown, key=lambda n: breakdown[n]["ms"])
    dflop = dict((n, f) for n, _, f, _ in step_parts)[dominant]
    if dflop:
        roof = {"bound": "tensor", "achieved": breakdown[dominant]["tflops"],
                "peak": fp8_peak if dominant == "fwd_fp8" else bf16_peak, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": breakdown[dominant]["gbs"], "peak": pk["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["kernel"] = KERNEL_OF[dominant]
    cap = NCU_TRAFFIC.get(dominant, {})
    fresh = cap.get("bytes") is not None and cap.get("src") == kernel_source_digest(dominant)
    roof["traffic"] = cap["bytes"] if (fresh and not causal) else None
    roof["traffic_unit"] = "bytes per launch (ncu dram read + write)"
    roof["traffic_capture"] = {
        "kernel_src_digest": kernel_source_digest(dominant), "captured_src_digest": cap.get("src"),
        "status": ("current" if fresh else "stale: kernel source changed since the capture"
                   if cap.get("bytes") is not None else "not captured for this source")
                  + ("" if not causal else "; captured non-causal only")}
    roof["peak_source"] = (f"{pk['source']} MEASURED_PEAKS.json bf16_tflops (burst: the kernel is "
                           "timed alone, well under a second, at full clocks); fp8 = 2x bf16")

    e2e = run_e2e(args, torch, attn, dev, stream, step_parts, causal, scale, q, k, v, do, signs, rope)
    ablation = (run_ablation(torch, attn, stream, causal, scale, q, k, v, args.exp2_eighths)
                if args.sweep else None)
    sweep = run_sweep(torch, attn, dev, stream, causal) if args.sweep else None
    fp8_acc = run_fp8_accuracy(torch, attn, dev) if args.sweep else None
    launches = sum(l for _, _, _, l in step_parts) * args.steps
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16+e4m3 (fp32 accumulate)", "data": "synthetic N(0,1), seeded",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "d": D, "causal": causal,
                   "global_batch": B * world, "seq_len": N, "parallelism": f"replicas{world}",
                   "step": [n for n, *_ in step_parts], "not_built": skipped,
                   "fp8_prepass_rotary": bool(args.rope),
                   "l2": "no flush: Q/K/V/dO/O (bf16, 67 MB each) exceed the 129 MB L2"},
        "breakdown": breakdown,
        "roofline": roof,
        "clocks": clocks.summary(),
        "e2e": e2e,
        "gpu_launches": launches,
    }
    if ablation is not None:
        line["ablation"] = ablation
    if fp8_acc is not None:
        line["fp8_rmse"] = fp8_acc
    if sweep is not None:
        line["headdim_sweep"] = sweep
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(line), flush=True)


def run_e2e(args, torch, attn, dev, stream, step_parts, causal, scale, q, k, v, do, signs, rope=None):
    """The same step through the public API with inputs in pinned host memory:
    host-to-device copies of every step's inputs and device-to-host copies of
    every output are inside the timed region.

    Two measurements.  `serial`: one stream, each step uploads, computes and
    downloads in turn.  `value` (pipelined, as a caller streaming batches would
    run it): uploads on a copy stream, compute on the launching stream and
    downloads on a third stream, with two device buffer sets, so step k+1's
    upload and step k-1's download overlap step k's kernels.  Every step still
    moves the same bytes; the timed region runs from the first upload to the
    end of the last download."""
    names = [n for n, *_ in step_parts]
    pin = lambda t: t.cpu().pin_memory()
    h_in = {"q": pin(q), "k": pin(k), "v": pin(v), "do": pin(do)}
    if "fp8_prepass" in names:
        h_in.update(signs=pin(signs))
    bf = torch.bfloat16
    shp = tuple(h_in["q"].shape)
    B_, H_, N_, _ = shp

    def new_slot():
        d_in = {k_: torch.empty_like(t, device=dev) for k_, t in h_in.items()}
        outs = {"o": torch.empty(shp, dtype=bf, device=dev),
                "lse": torch.empty((B_, H_, N_), dtype=torch.float32, device=dev)}
        if "bwd_bf16" in names:
            outs.update(dq=torch.empty(shp, dtype=bf, device=dev),
                        dk=torch.empty(shp, dtype=bf, device=dev),
                        dv=torch.empty(shp, dtype=bf, device=dev),
                        ws=torch.empty(attn.attn_bwd_workspace_size(B_, H_, N_, shp[3]),
                                       dtype=torch.uint8, device=dev))
        if "fwd_fp8" in names:
            outs.update(o8=torch.empty(shp, dtype=bf, device=dev),
                        lse8=torch.empty((B_, H_, N_), dtype=torch.float32, device=dev))
        return d_in, outs

    slots = [new_slot(), new_slot()]
    result_keys = [k_ for k_ in ("o", "lse", "dq", "dk", "dv", "o8", "lse8") if k_ in slots[0][1]]
    h_out = [{k_: torch.empty(slots[0][1][k_].shape, dtype=slots[0][1][k_].dtype, pin_memory=True)
              for k_ in result_keys} for _ in range(2)]

    def compute(d_in, outs, s):
        attn.attn_fwd(d_in["q"], d_in["k"], d_in["v"], causal=causal, softmax_scale=scale,
                      o=outs["o"], lse=outs["lse"], stream=s)
        if "bwd_bf16" in names:
            attn.attn_bwd(d_in["q"], d_in["k"], d_in["v"], outs["o"], d_in["do"], outs["lse"],
                          causal=causal, softmax_scale=scale, dq=outs["dq"], dk=outs["dk"],
                          dv=outs["dv"], workspace=outs["ws"], stream=s)
        if "fp8_prepass" in names:
            if rope is not None:
                (q8, k8, v8), (qs, ks, vs) = attn.attn_fp8_quantize_ex(
                    d_in["q"], d_in["k"], d_in["v"], rope[0], rope[1], d_in["signs"], stream=s)
            else:
                (q8, k8, v8), (qs, ks, vs) = attn.attn_fp8_quantize_bf16(
                    d_in["q"], d_in["k"], d_in["v"], d_in["signs"], stream=s)
            if "fwd_fp8" in names:
                attn.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=causal, softmax_scale=scale,
                                  o=outs["o8"], lse=outs["lse8"], stream=s)

    def upload(d_in):
        for k_, t in h_in.items():
            d_in[k_].copy_(t, non_blocking=True)

    def download(outs, hb):
        for k_ in result_keys:
            hb[k_].copy_(outs[k_], non_blocking=True)

    # serial: one stream
    def serial_step():
        d_in, outs = slots[0]
        upload(d_in)
        compute(d_in, outs, stream)
        download(outs, h_out[0])

    def timed(run, steps, s_first, s_last):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(s_first)
        run(steps)
        b.record(s_last)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    def serial(steps):
        with torch.cuda.stream(stream):
            for _ in range(steps):
                serial_step()

    # (two upload streams measured no faster: the host link is the limit)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def pipelined(steps):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def start_upload(slot):
            with torch.cuda.stream(s_in):
                if used[slot]:
                    s_in.wait_event(comp_done[slot])       # the step before is done reading them
                upload(slots[slot][0])
                in_ready[slot].record(s_in)

        start_upload(0)
        for k in range(steps):
            cur, nxt = k % 2, (k + 1) % 2
            if k + 1 < steps:
                start_upload(nxt)
            stream.wait_event(in_ready[cur])
            if used[cur]:
                stream.wait_event(out_done[cur])           # step k-2's results are downloaded
            with torch.cuda.stream(stream):
                compute(slots[cur][0], slots[cur][1], stream)
                comp_done[cur].record(stream)
            used[cur] = True
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[cur])
                download(slots[cur][1], h_out[cur])
                out_done[cur].record(s_out)

    for _ in range(max(1, args.warmup)):
        serial(1)
    pipelined(max(2, args.warmup))
    ms_serial = timed(serial, args.steps, stream, stream)
    ms = timed(pipelined, args.steps, s_in, s_out)
    flop = sum(f for _, _, f, _ in step_parts)
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())
    return {"value": round(flop / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": True,
            "serial_value": round(flop / (ms_serial * 1e-3) / 1e12, 2),
            "serial_ms_per_step": round(ms_serial, 4)}


def time_call(torch, stream, fn, steps=20, warmup=3):
    """Mean milliseconds per call over `steps` calls (CUDA events on `stream`)."""
    for _ in range(warmup):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def run_ablation(torch, attn, stream, causal, scale, q, k, v, exp2_eighths=(2,)):
    """The forward pipeline ablation on the timed workload: the default schedule
    (two query tiles per CTA alternating on the tensor core, lazy rescaling)
    against one query tile per CTA (nothing fills the tensor core while a
    tile's softmax runs) and eager rescaling (the output accumulator rescaled
    whenever the row max grows); and the FP8 forward with a quarter of its
    exponentials evaluated on the FMA pipe.  TFLOP/s of the same algorithmic FLOP."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    flop = fwd_flop(causal)
    out = {}
    for name, sched in (("default", 0), ("one_tile", 1), ("eager_rescale", 2),
                        ("one_tile_eager_rescale", 3)):
        fn = lambda: attn.attn_fwd_schedule(q, k, v, sched, causal=causal, softmax_scale=scale,
                                            o=o, lse=lse, stream=stream)
        ms = time_call(torch, stream, fn)
        out[name] = {"ms": round(ms, 4), "tflops": round(flop / (ms * 1e-3) / 1e12, 1)}
    # FP8 forward: the library's default (one sixteenth of the exponentials on the
    # FMA pipe for non-causal batches), all on the MUFU unit, and k eighths (--exp2-eighths)
    signs = torch.where(torch.arange(q.shape[-1], device=q.device) % 3 == 0, -1.0, 1.0).float()
    (q8, k8, v8), (qs, ks, vs) = attn.attn_fp8_quantize_bf16(q, k, v, signs, stream=stream)
    o8 = torch.empty_like(q)
    names = {1: "eighth", 2: "quarter", 3: "three_eighths", 4: "half"}
    variants = ([("fp8_default", 0), ("fp8_exp2_none", attn.ATTN_SCHED_EXP2_NONE)] +
                [(f"fp8_exp2_poly_{names[e]}", attn.ATTN_SCHED_EXP2_EIGHTHS(e)) for e in exp2_eighths])
    for name, sched in variants:
        fn = lambda: attn.attn_fwd_fp8_schedule(q8, k8, v8, qs, ks, vs, sched, causal=causal,
                                                softmax_scale=scale, o=o8, lse=lse, stream=stream)
        ms = time_call(torch, stream, fn)
        out[name] = {"ms": round(ms, 4), "tflops": round(flop / (ms * 1e-3) / 1e12, 1)}
    assert attn.attn_get_device_status() == 0, attn.attn_last_error()
    return out


def run_fp8_accuracy(torch, attn, dev):
    """RMSE of the FP8 forward against exact attention on the outlier-stress
    workload (B=2, H=16, N=4096, d=128; float32 N(0,1) plus N(0, 10^2) on a
    random 0.1 % of entries), for the per-tensor comparator, block scales, and
    block scales + Hadamard.  The exact reference is float64 softmax(Q K^T s) V
    of the float32 inputs, computed by torch on the device for three heads."""
    import workloads
    w = workloads.FP8_FWD
    q, k, v = (torch.from_numpy(x).to(dev) for x in
               workloads.normal_with_outliers(w.seed, (w.B, w.H, w.N, w.d), 3))
    signs = torch.from_numpy(workloads.random_signs(workloads.FP8_HADAMARD_SIGN_SEED, w.d)).to(dev)
    heads = [(0, 0), (1, 9), (0, 15)]
    ref = {}
    for b, h in heads:
        s64 = (q[b, h].double() @ k[b, h].double().T) * w.scale
        ref[(b, h)] = torch.softmax(s64, dim=-1) @ v[b, h].double()
    out = {"workload": f"{w.name} (seeded outliers), heads {heads}",
           "pages_reference": "9.1e-3 block+Hadamard vs 2.4e-2 per-tensor (their workload unstated)"}
    for name, sg, pt in (("per_tensor", None, True), ("block", None, False),
                         ("block_hadamard", signs, False)):
        (q8, k8, v8), (qd, kd, vd) = attn.attn_fp8_quantize(q, k, v, hadamard_signs=sg,
                                                            per_tensor=pt)
        o, _ = attn.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=w.causal, softmax_scale=w.scale)
        err = torch.cat([(o[b, h].double() - ref[(b, h)]).flatten() for b, h in heads])
        out[name] = float(f"{err.pow(2).mean().sqrt().item():.4g}")
    assert attn.attn_get_device_status() == 0, attn.attn_last_error()
    return out


def run_sweep(torch, attn, dev, stream, causal, steps=20, warmup=3):
    """Head-dimension sweep of the long-context workload at 16K tokens and
    H*d = 2048: BF16 forward at d = 64, 128, 256 and backward at d = 64, 128
    (TFLOP/s, CUDA events, inputs resident in HBM)."""
    out = {}
    for d, h in ((64, 32), (128, 16), (256, 8)):
        g = torch.Generator(device=dev).manual_seed(7)
        q, k, v, do = (torch.randn((B, h, N, d), generator=g, device=dev).to(torch.bfloat16)
                       for _ in range(4))
        o = torch.empty_like(q)
        lse = torch.empty((B, h, N), dtype=torch.float32, device=dev)
        flop = 4.0 * B * h * N * N * d / (2 if causal else 1)
        fns = [("fwd", lambda: attn.attn_fwd(q, k, v, causal=causal, o=o, lse=lse), flop)]
        if d <= 128:
            ws = torch.empty(attn.attn_bwd_workspace_size(B, h, N, d), dtype=torch.uint8, device=dev)
            dq, dk, dv = (torch.empty_like(q) for _ in range(3))
            fns.append(("bwd", lambda: attn.attn_bwd(q, k, v, o, do, lse, causal=causal, dq=dq,
                                                     dk=dk, dv=dv, workspace=ws), 2.5 * flop))
        for name, fn, fl in fns:
            for _ in range(warmup):
                fn()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / steps
            out[f"{name}_d{d}_h{h}"] = {"ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 1)}
        del q, k, v, do, o, lse
    out.update(run_varlen_gqa(torch, attn, dev, stream, causal, steps, warmup))
    out.update(run_fp8_gqa(torch, attn, dev, stream, causal, steps, warmup))
    out.update(run_prepass_rope(torch, attn, dev, stream, steps, warmup))
    out.update(run_prepass_rope_bf16(torch, attn, dev, stream, steps, warmup))
    out.update(run_decode(torch, attn, dev, stream, steps, warmup))
    out.update(run_decode_fp8(torch, attn, dev, stream, steps, warmup))
    assert attn.attn_get_device_status() == 0, attn.attn_last_error()
    return out


def run_decode(torch, attn, dev, stream, steps=20, warmup=3):
    """Paged decode: 16 sequences of 8192 cached tokens, H = 32 query heads
    sharing H_kv = 8 key/value heads, d = 128, pages of 256 tokens (the block
    size of the paged cache the sources describe) in a shuffled order, n_q = 1
    and 4 new tokens (causal).  GB/s of algorithmic bytes: the cached keys and
    values read once, plus Q and O."""
    Bq, L, h, hkv, d, ps = 16, 8192, 32, 8, 128, 256
    npg = Bq * L // ps
    g = torch.Generator(device=dev).manual_seed(10)
    kc, vc = (torch.randn((npg, ps, hkv, d), generator=g, device=dev).to(torch.bfloat16)
              for _ in range(2))
    table = torch.randperm(npg, generator=g, device=dev).to(torch.int32).view(Bq, L // ps)
    lens = torch.full((Bq,), L, dtype=torch.int32, device=dev)
    out = {}
    for n_q in (1, 4):
        q = torch.randn((Bq, h, n_q, d), generator=g, device=dev).to(torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty((Bq, h, n_q), dtype=torch.float32, device=dev)
        ws = torch.empty(attn.attn_decode_workspace_size(Bq, h, hkv, n_q, d, L), dtype=torch.uint8,
                         device=dev)
        fn = lambda: attn.attn_decode_paged(q, kc, vc, table, lens, L, causal=True, o=o, lse=lse,
                                            workspace=ws, stream=stream)
        for _ in range(warmup):
            fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        nbytes = 2 * Bq * L * hkv * d * 2 + 2 * Bq * h * n_q * d * 2
        out[f"decode_b{Bq}_len{L}_h{h}kv{hkv}_d{d}_nq{n_q}_page{ps}"] = {
            "ms": round(ms, 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    return out


def run_decode_fp8(torch, attn, dev, stream, steps=20, warmup=3):
    """Paged decode over an e4m3 cache at the shape of run_decode: random codes
    with a random descale per (page, head); n_q = 1, 2, 4 and 8, and n_q = 1
    with the key transform.  GB/s of algorithmic bytes: the cached codes read once, the
    descales, Q and O."""
    Bq, L, h, hkv, d, ps = 16, 8192, 32, 8, 128, 256
    npg = Bq * L // ps
    g = torch.Generator(device=dev).manual_seed(11)
    kc, vc = (torch.randn((npg, ps, hkv, d), generator=g, device=dev).to(torch.float8_e4m3fn)
              .view(torch.uint8) for _ in range(2))
    kd, vd = (torch.rand((npg, hkv), generator=g, device=dev) * 0.02 + 0.01 for _ in range(2))
    table = torch.randperm(npg, generator=g, device=dev).to(torch.int32).view(Bq, L // ps)
    lens = torch.full((Bq,), L, dtype=torch.int32, device=dev)
    signs = torch.where(torch.rand(d, generator=g, device=dev) < 0.5, -1.0, 1.0).float()
    out = {}
    for n_q, sg in ((1, None), (2, None), (4, None), (8, None), (1, signs)):
        q = torch.randn((Bq, h, n_q, d), generator=g, device=dev).to(torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty((Bq, h, n_q), dtype=torch.float32, device=dev)
        ws = torch.empty(attn.attn_decode_workspace_size(Bq, h, hkv, n_q, d, L), dtype=torch.uint8,
                         device=dev)
        fn = lambda: attn.attn_decode_paged_fp8(q, kc, vc, kd, vd, table, lens, L, causal=True,
                                                hadamard_signs=sg, o=o, lse=lse, workspace=ws,
                                                stream=stream)
        for _ in range(warmup):
            fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        nbytes = 2 * Bq * L * hkv * d + 2 * npg * hkv * 4 + 2 * Bq * h * n_q * d * 2
        tag = "_hadamard" if sg is not None else ""
        out[f"decode_fp8_b{Bq}_len{L}_h{h}kv{hkv}_d{d}_nq{n_q}_page{ps}{tag}"] = {
            "ms": round(ms, 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    return out


def run_prepass_rope(torch, attn, dev, stream, steps=20, warmup=3):
    """The FP8 pre-pass with the rotary embedding fused in (block mode,
    Hadamard on Q and K) at the timed shape: GB/s of algorithmic bytes (read 3
    float32 tensors and the two [N, d/2] tables, write 3 e4m3 tensors and the
    descales)."""
    import workloads
    g = torch.Generator(device=dev).manual_seed(9)
    q, k, v = (torch.randn((B, H, N, D), generator=g, device=dev) for _ in range(3))
    cos, sin = (torch.from_numpy(t).to(dev) for t in workloads.rope_tables(N, D))
    signs = torch.where(torch.rand(D, generator=g, device=dev) < 0.5, -1.0, 1.0).float()
    fn = lambda: attn.attn_fp8_quantize_rope(q, k, v, cos, sin, hadamard_signs=signs, stream=stream)
    for _ in range(warmup):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    nblk = (N + 127) // 128
    nbytes = 3 * B * H * N * D * (4 + 1) + 3 * B * H * nblk * 4 + 2 * N * (D // 2) * 4
    return {f"fp8_prepass_rope_b{B}h{H}n{N}d{D}": {"ms": round(ms, 4),
                                                    "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}}


def run_prepass_rope_bf16(torch, attn, dev, stream, steps=20, warmup=3):
    """The FP8 pre-pass on bfloat16 inputs with rotary embedding and the
    Hadamard transform (attn_fp8_quantize_ex) at the timed shape: GB/s of
    algorithmic bytes (read 3 bfloat16 tensors and the two [N, d/2] tables,
    write 3 e4m3 tensors and the descales)."""
    import workloads
    g = torch.Generator(device=dev).manual_seed(13)
    q, k, v = (torch.randn((B, H, N, D), generator=g, device=dev).to(torch.bfloat16) for _ in range(3))
    cos, sin = (torch.from_numpy(t).to(dev) for t in workloads.rope_tables(N, D))
    signs = torch.where(torch.rand(D, generator=g, device=dev) < 0.5, -1.0, 1.0).float()
    fn = lambda: attn.attn_fp8_quantize_ex(q, k, v, cos, sin, hadamard_signs=signs, stream=stream)
    ms = time_call(torch, stream, fn, steps, warmup)
    nblk = (N + 127) // 128
    nbytes = 3 * B * H * N * D * (2 + 1) + 3 * B * H * nblk * 4 + 2 * N * (D // 2) * 4
    return {f"fp8_prepass_rope_bf16_b{B}h{H}n{N}d{D}": {"ms": round(ms, 4),
                                                         "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}}


def run_fp8_gqa(torch, attn, dev, stream, causal, steps=20, warmup=3):
    """FP8 forward with grouped-query heads at the timed shape: B = 2, N = 8192,
    H = 16 query heads sharing H_kv = 4 key/value heads, d = 128 (block scales
    and the Hadamard transform from the pre-pass, which runs once untimed).
    FLOP = 4*B*H*N^2*d, halved causal."""
    g = torch.Generator(device=dev).manual_seed(12)
    hkv = 4
    q = torch.randn((B, H, N, D), generator=g, device=dev)
    k, v = (torch.randn((B, hkv, N, D), generator=g, device=dev) for _ in range(2))
    signs = torch.where(torch.rand(D, generator=g, device=dev) < 0.5, -1.0, 1.0).float()
    (q8, k8, v8), (qd, kd, vd) = attn.attn_fp8_quantize_gqa(q, k, v, hadamard_signs=signs,
                                                            stream=stream)
    del q, k, v
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fn = lambda: attn.attn_fwd_fp8_gqa(q8, k8, v8, qd, kd, vd, causal=causal, o=o, lse=lse,
                                       stream=stream)
    for _ in range(warmup):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    flop = 4.0 * B * H * N * N * D / (2 if causal else 1)
    return {f"fp8_gqa_fwd_b{B}h{H}kv{hkv}n{N}d{D}": {"ms": round(ms, 4),
                                                     "tflops": round(flop / (ms * 1e-3) / 1e12, 1)}}


def run_varlen_gqa(torch, attn, dev, stream, causal, steps=20, warmup=3):
    """A packed batch of 8 sequences of mixed length (seeded, 256..4096 tokens,
    ~18K in all) with grouped-query heads: H = 16 query heads sharing H_kv = 4
    key/value heads, d = 128.  FLOP = sum over sequences of 4*len^2*d*H (halved
    causal); backward 2.5x."""
    import workloads
    cu_np, lens = workloads.varlen_lengths(8, 8, 4096, 256)
    total, maxlen, h, hkv, d = int(cu_np[-1]), int(lens.max()), 16, 4, 128
    g = torch.Generator(device=dev).manual_seed(8)
    q, do = (torch.randn((total, h, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn((total, hkv, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(2))
    cu = torch.from_numpy(cu_np).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((h, total), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(attn.attn_bwd_varlen_workspace_size(len(lens), maxlen, total, h, d),
                     dtype=torch.uint8, device=dev)
    flop = sum(4.0 * float(n) * float(n) * d * h for n in lens) / (2 if causal else 1)
    fns = [("fwd", lambda: attn.attn_fwd_varlen(q, k, v, cu, maxlen, causal=causal, o=o, lse=lse),
            flop),
           ("bwd", lambda: attn.attn_bwd_varlen(q, k, v, o, do, lse, cu, maxlen, causal=causal,
                                                dq=dq, dk=dk, dv=dv, workspace=ws), 2.5 * flop)]
    out = {}
    for name, fn, fl in fns:
        for _ in range(warmup):
            fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        out[f"varlen_gqa_{name}_b{len(lens)}_t{total}_h{h}kv{hkv}_d{d}"] = {
            "ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 1)}
    return out


def cpu_sample_problem(seed=3):
    """One head of the timed workload (N=8192, d=128), float64 on the host."""
    import numpy as np
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((N, D)) for _ in range(4)]


def cpu_baseline(args, heads=8):
    """The CPU oracle as it stands, on a bounded sample of the workload: the
    forward and backward of `heads` head(s) at N=8192, d=128."""
    import oracle
    q, k, v, do = cpu_sample_problem()
    scale = 1.0 / math.sqrt(D)
    t0 = time.perf_counter()
    for _ in range(heads):
        oracle.attention_forward_head(q, k, v, scale, args.causal)
        oracle.attention_backward_head(q, k, v, do, scale, args.causal)
    dt = time.perf_counter() - t0
    flop = heads * 3.5 * 4.0 * N * N * D / (2 if args.causal else 1)
    threads = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        threads = max(i.get("num_threads", 0) for i in threadpool_info()) or threads
    except Exception:
        pass
    return {"value": round(flop / dt / 1e12, 5), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{heads} head(s) of the workload, forward + backward, float64 NumPy"}


def run_reference(args, rank):
    """The CPU oracle timed as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    q, k, v, do = cpu_sample_problem()
    scale = 1.0 / math.sqrt(D)
    for _ in range(args.warmup):
        oracle.attention_forward_head(q[:256], k, v, scale, args.causal)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_forward_head(q, k, v, scale, args.causal)
        oracle.attention_backward_head(q, k, v, do, scale, args.causal)
    dt = time.perf_counter() - t0
    flop = args.steps * 3.5 * 4.0 * N * N * D / (2 if args.causal else 1)
    value = flop / dt / 1e12
    threads = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic N(0,1), seeded",
            "config": {"workload": WORKLOAD + " -- oracle sample: one head fwd+bwd per step",
                       "B": B, "H": H, "N": N, "d": D, "causal": args.causal},
            "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle",
                             "sample": "one head (N=8192, d=128) forward + backward per step"},
            "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_decode_only(args):
    """The paged decode lines alone, as one JSON line (not the bench contract's
    line: no step is timed)."""
    import torch
    import exact_tiled_attention_25_gb300 as attn
    attn.load_library()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    out = run_decode(torch, attn, dev, stream, args.steps, args.warmup)
    out.update(run_decode_fp8(torch, attn, dev, stream, args.steps, args.warmup))
    assert attn.attn_get_device_status() == 0, attn.attn_last_error()
    hbm = peaks()["hbm_gbs"]
    for v in out.values():
        v["frac_hbm"] = round(v["gbs"] / hbm, 3)
    print(json.dumps({"decode": out, "hbm_peak_gbs": hbm}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--rope", action="store_true",
                    help="the step's FP8 pre-pass also applies rotary embedding to Q and K")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false",
                    help="skip the head-dimension sweep")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--exp2-eighths", type=int, nargs="+", default=[2], choices=[1, 2, 3, 4],
                    help="shares (in eighths) of the FP8 forward's exponentials evaluated on the FMA "
                         "pipe in the ablation entries (default: a quarter)")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the paged decode lines (BF16 and e4m3 caches) and print them; "
                         "the profiling captures of the decode kernels use this")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if args.steps < 1:
            raise SystemExit("--steps must be >= 1")
        run_reference(args, rank)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.decode_only:
        run_decode_only(args)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    run_ours(args, rank, world)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
