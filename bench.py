#!/usr/bin/env python3
"""Benchmark of the GB300 loss-scaled AdamW optimizer step.

One step is one attempted logical update over k micro-batches, the whole hot
path: k-1 accumulations, the fused last-micro-batch + unscale + overflow check
+ squared-norm pass, the global norm / clip coefficient, clip + AdamW + recast,
and the scaler update.  The default workload is the ~1.24B-parameter Llama
tensor list (146 tensors, bf16 parameters and gradients, fp32 master/m/v and
accumulation buffer, k = 8 micro-batches, synthetic seeded inputs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  ``value`` is whole-job Gparams/s (parameters
updated per second, all ranks) with inputs resident in HBM; ``e2e`` is the same
metric through the Python binding with the micro-batch gradients copied from
pinned host memory inside the timed region and the step's status read back.
With N > 1 (torchrun) each rank runs an independent replica on its own GPU: the
optimizer step has no exchange of its own, so there is no collective.
``--impl reference`` times the CPU oracle (the reference statement of the step)
on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused optimizer-step Gparams/s and achieved HBM GB/s as % of GB300 peak"
UNIT = "Gparams/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama_1b")
    ap.add_argument("--path", choices=["resident", "per_microbatch", "remat"], default="resident",
                    help="resident: the k micro-batch gradient lists are read in one pass (tl_accumulate_many); "
                         "per_microbatch: one tl_accumulate per micro-batch; remat (k <= 4): the lists are "
                         "checked without storing u (tl_unscale_check_many) and the AdamW pass recomputes u "
                         "from them")
    ap.add_argument("--layout", choices=["aligned", "packed", "misaligned"], default="aligned",
                    help="tensor placement inside the flat buffers (see GpuWorkload)")
    ap.add_argument("--graph", action="store_true", help="also time every sequence replayed from a CUDA graph")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed helpers (replicas; used with gloo on CPU in the tests)
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, device="cpu") -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def whole_job_rate(params_per_step: int, steps: int, world: int, seconds_max: float) -> float:
    """Gparams/s of the whole job: every rank updates params_per_step per step; the job
    takes the slowest rank's time."""
    return params_per_step * steps * world / seconds_max / 1e9


# ---------------------------------------------------------------------------
# peaks, traffic summary, clocks
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            v = float(json.load(fh)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest() -> str:
    """Digest of the kernel sources' code: comments, indentation and blank lines do not
    count, so recorded counters stay valid across edits that cannot change a kernel."""
    import hashlib
    h = hashlib.sha256()
    for f in ("tl_kernels.cu", "tl_kernels_split.cu", "tl_internal.cuh"):
        with open(os.path.join(ROOT, "loss_scaled_adamw_gb300", "csrc", f)) as fh:
            for line in fh:
                cut = line.find("//")
                if cut >= 0 and '"' not in line[:cut]:
                    line = line[:cut]
                line = line.strip()
                if line:
                    h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str, workload: str, layout: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary, if it was taken
    from the current kernel source on this workload and layout (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        line = line.strip()
        if "=" in line and not line.startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_digest") != kernel_source_digest():
        return None
    if kv.get("workload") != workload or kv.get("layout") != layout:
        return None
    v = kv.get(kernel_key + ".dram_bytes_per_launch")
    return float(v) if v else None


def gpu_id(local_rank: int) -> str:
    """nvidia-smi's id of this process's GPU (its UUID, whatever CUDA_VISIBLE_DEVICES says)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local_rank)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu_index)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, a in enumerate(r[3]) if a.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

class GpuWorkload:
    """Device-resident tensor lists of a workload, packed into flat buffers."""

    def __init__(self, wl, device, layout="aligned"):
        import torch
        import loss_scaled_adamw_gb300 as tl
        from loss_scaled_adamw_gb300 import workloads as W
        self.wl = wl
        P = wl.P
        self.P = P
        self.device = device
        # tensor offsets inside each flat buffer: "aligned" starts every tensor on a
        # 32-byte boundary (packed when the sizes allow), "packed" puts tensors back to
        # back (same element phase in every list), "misaligned" puts a seeded 0-3
        # element gap before every tensor (many start off any 16-byte boundary)
        # with "misaligned" every list gets its own gaps (no common element phase)
        self.layout = layout
        self.offs_of = {}

        def offsets(key):
            if key not in self.offs_of:
                self.offs_of[key] = W.layout_offsets(wl.numel, layout == "misaligned", 1 if layout == "packed" else 8,
                                                     key if layout == "misaligned" else 0)
            return self.offs_of[key]

        gscale = wl.init_scale if wl.grads_prescaled else 1.0

        def spread(flat, dtype, key):
            offs, total = offsets(key)
            if offs == np.cumsum([0] + wl.numel[:-1]).tolist():
                return flat
            buf = torch.zeros(total + 16, dtype=dtype, device=device)
            n = torch.tensor(wl.numel, dtype=torch.int64)
            shift = torch.tensor(offs, dtype=torch.int64) - (torch.cumsum(n, 0) - n)
            idx = torch.arange(P, dtype=torch.int64, device=device) + torch.repeat_interleave(shift.to(device), n.to(device))
            buf[idx] = flat
            return buf

        keys = {"param": 1, "master": 2, "m": 3, "v": 4, "acc": 5}
        master = W.master_init(wl, device)
        self.master = spread(master, torch.float32, keys["master"])
        self.param = spread(W.to_16bit(master, wl.param_dtype), W.to_16bit(master[:1], wl.param_dtype).dtype, keys["param"])
        del master
        self.m = torch.zeros(offsets(keys["m"])[1] + 16, dtype=torch.float32, device=device)
        self.v = torch.zeros(offsets(keys["v"])[1] + 16, dtype=torch.float32, device=device)
        self.acc = torch.empty(offsets(keys["acc"])[1] + 16, dtype=torch.float32, device=device)
        fp8 = wl.grad_dtype == "e4m3b16"

        def e4m3_buffer(pair, key):
            # every tensor on a 16-byte boundary: codes padded to 16 bytes, then block scales
            offs, soffs, total = W.e4m3_layout(wl.numel, layout == "misaligned", key)
            codes, scales = pair
            buf = torch.zeros(total + 16, dtype=torch.uint8, device=device)
            n = torch.tensor(wl.numel, dtype=torch.int64)
            nb = (n + 15) // 16
            ci = torch.arange(P, dtype=torch.int64) + torch.repeat_interleave(
                torch.tensor(offs, dtype=torch.int64) - (torch.cumsum(n, 0) - n), n)
            si = torch.arange(int(nb.sum()), dtype=torch.int64) + torch.repeat_interleave(
                torch.tensor(soffs, dtype=torch.int64) // 4 - (torch.cumsum(nb, 0) - nb), nb)
            buf[ci.to(device)] = codes.to(device)
            buf.view(torch.float32)[si.to(device)] = scales.to(device)
            return buf

        self.grads = []
        for i in range(wl.k):
            g = W.grad_input(wl, 1, i, scale=gscale, device=device)
            self.grads.append(e4m3_buffer(g, 10 + i) if fp8 else spread(g, g.dtype, 10 + i))
            del g

        def plist(t, key):
            es, base = t.element_size(), t.data_ptr()
            if fp8 and key >= 10:   # a gradient list of 8-bit tensors: byte offsets of the layout above
                p = tl.PtrList([base + o for o in W.e4m3_layout(wl.numel, layout == "misaligned", key)[0]])
            else:
                p = tl.PtrList([base + o * es for o in offsets(key)[0]])
            p.keep = t
            return p

        self.plist = plist
        self.plists = {n: plist(getattr(self, n), keys[n]) for n in keys}
        self.gplists = [plist(g, 10 + i) for i, g in enumerate(self.grads)]
        # element offset of the first gradient element of tensor 0 in grads[0]
        first = int(self.gplists[0].array[0]) - self.grads[0].data_ptr()
        self.plists_first_offset = first // self.grads[0].element_size()
        self.many = tl.ManyLists(self.gplists)
        dt = {"bf16": tl.TL_BF16, "f16": tl.TL_F16, "f32": tl.TL_F32, "e4m3b16": tl.TL_E4M3B16}
        cfg = tl.make_config(dt[wl.param_dtype], dt[wl.grad_dtype], wl.scaler_enabled,
                             wl.init_scale if wl.scaler_enabled else 1.0, interval=wl.interval)
        L = self.plists
        self.ctx = tl.tl_create(wl.numel, L["param"], L["master"], L["m"], L["v"], L["acc"], cfg)
        self.counts = wl.counts(1)
        self.N = sum(self.counts)
        self.hp = tl.tl_adamw_hp(1e-3, 0.9, 0.95, 1e-8, 0.1)
        # gradient bytes per parameter (8-bit: the code and a quarter of a 4-byte scale)
        sg = {"bf16": 2, "f16": 2, "f32": 4, "e4m3b16": 1.25}[wl.grad_dtype]
        sp = {"bf16": 2, "f16": 2}[wl.param_dtype]
        self.adam_bytes = 16 + 12 + sp

        k = wl.k
        # (kernel name, algorithmic bytes per parameter, call) for each path
        per = []
        for i in range(k - 1):
            per.append(("accumulate_first" if i == 0 else "accumulate", sg + 4 if i == 0 else sg + 8,
                        lambda i=i: tl.tl_accumulate(self.ctx, self.gplists[i], self.counts[i], self.N, 1 if i == 0 else 0)))
        per.append(("unscale_check", sg + (8 if k > 1 else 4),
                    lambda: tl.tl_unscale_check(self.ctx, self.gplists[k - 1], self.counts[k - 1], self.N)))
        tail = [("grad_norm", None, lambda: tl.tl_grad_norm(self.ctx, self.wl.max_norm)),
                ("clip_adamw_step", self.adam_bytes, lambda: tl.tl_clip_adamw_step(self.ctx, self.hp)),
                ("scaler_update", None, lambda: tl.tl_scaler_update(self.ctx))]
        # the resident pass reads 8 lists per launch, writes acc once per launch
        launches = (k + 7) // 8
        many_bytes = k * sg + 4 * launches + 4 * (launches - 1)
        res = [("accumulate_many", many_bytes,
                lambda: tl.tl_accumulate_many(self.ctx, self.many, self.counts, self.N, 1))]
        self.paths = {"resident": res + tail, "per_microbatch": per + tail}
        if k <= 4:
            # re-materialising: the lists are read twice (check, then AdamW), u never stored
            self.paths["remat"] = [
                ("unscale_check_many", k * sg,
                 lambda: tl.tl_unscale_check_many(self.ctx, self.many, self.counts, self.N)),
                tail[0],
                ("clip_adamw_step_remat", 12 + 12 + sp + k * sg, lambda: tl.tl_clip_adamw_step(self.ctx, self.hp)),
                tail[2]]

    def step_bytes(self, path):
        return self.P * sum(b for _, b, _ in self.paths[path] if b)

    def step(self, path, events=None):
        """One logical update; with `events`, a pair of CUDA events around every call."""
        import torch
        for name, _, fn in self.paths[path]:
            if events is None:
                fn()
            else:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                events.append((name, a, b))


def time_graph(args, gw, path, world):
    """K steps of one path replayed from a CUDA graph captured once (the update has no
    host synchronisation, so the whole step captures): no per-call host overhead."""
    import torch
    import loss_scaled_adamw_gb300 as tl
    for _ in range(max(args.warmup, 1)):
        gw.step(path)  # also uploads any device pointer tables before capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    launches0 = tl.tl_launch_count(gw.ctx)
    with torch.cuda.graph(g, stream=s):
        gw.step(path)
    per_step = tl.tl_launch_count(gw.ctx) - launches0
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier()
    el = max_over_ranks(t0.elapsed_time(t1) / 1e3, gw.device)
    return {"value": whole_job_rate(gw.P, args.steps, world, el), "ms_per_step": el / args.steps * 1e3,
            "launches_per_step": per_step}


def time_path(args, gw, path, world):
    """K timed steps of one path (after W warm-up steps), then the same K steps again with
    a pair of CUDA events around every call for the per-kernel attribution (those events
    and their host calls are kept out of the headline timing, where on short steps their
    host time would show up as idle device time)."""
    import torch
    import loss_scaled_adamw_gb300 as tl
    for _ in range(args.warmup):
        gw.step(path)
    torch.cuda.synchronize()
    barrier()
    launches0 = tl.tl_launch_count(gw.ctx)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        gw.step(path)
    t1.record()
    torch.cuda.synchronize()
    barrier()
    elapsed = t0.elapsed_time(t1) / 1e3
    launches = tl.tl_launch_count(gw.ctx) - launches0
    elapsed_max = max_over_ranks(elapsed, gw.device)
    events = []
    i0, i1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    i0.record()
    for _ in range(args.steps):
        gw.step(path, events)
    i1.record()
    torch.cuda.synchronize()
    barrier()
    elapsed_instr = i0.elapsed_time(i1) / 1e3
    peak, peak_kind = hbm_peak()
    per = {}
    for name, a, b in events:
        per.setdefault(name, []).append(a.elapsed_time(b) / 1e3)
    bytes_of = {n: b for n, b, _ in gw.paths[path]}
    kernels = {}
    for name, ts in per.items():
        avg = sum(ts) / len(ts)
        entry = {"launches": len(ts), "avg_ms": avg * 1e3, "share": sum(ts) / elapsed_instr}
        if bytes_of.get(name):
            gbs = bytes_of[name] * gw.P / avg / 1e9
            entry.update({"bytes_per_param": bytes_of[name], "bytes_per_launch": bytes_of[name] * gw.P,
                          "achieved_gbs": gbs, "frac": gbs / peak})
        kernels[name] = entry
    sb = gw.step_bytes(path)
    return {"elapsed_max": elapsed_max, "launches": launches, "kernels": kernels,
            "instrumented_ms_per_step": elapsed_instr / args.steps * 1e3,
            "value": whole_job_rate(gw.P, args.steps, world, elapsed_max),
            "ms_per_step": elapsed_max / args.steps * 1e3,
            "hbm": {"algorithmic_bytes_per_step": sb, "bytes_per_param": sb / gw.P,
                    "achieved_gbs_per_gpu": sb * args.steps / elapsed_max / 1e9, "peak_gbs": peak,
                    "peak_kind": peak_kind, "frac": sb * args.steps / elapsed_max / 1e9 / peak}}


TRAFFIC_KEYS = {"accumulate": "k_accumulate_bf16", "clip_adamw_step": "k_adamw_bf16",
                "unscale_check": "k_unscale_bf16_acc_grad", "accumulate_first": "k_accumulate_first_bf16",
                "accumulate_many": "k_accum_many_bf16_first_last"}


def table_plan(tl, numel, local_rank):
    """The chunk table the context lays this list out in on this device (tl_plan, host
    only): chunk counts, segment length, squared-norm runs, split forms, fused norm."""
    import torch
    try:
        sm = torch.cuda.get_device_properties(local_rank).multi_processor_count
        return tl.tl_plan(list(numel), sm)
    except Exception as exc:   # a note on the layout must never cost the measurement
        return {"error": str(exc)[:200]}


def run_gpu(args, rank, world, local_rank):
    import torch
    import loss_scaled_adamw_gb300 as tl
    from loss_scaled_adamw_gb300 import workloads as W
    from loss_scaled_adamw_gb300 import _build
    _build.build()
    tl.load_library()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    wl = W.make(args.workload)
    gw = GpuWorkload(wl, device, args.layout)
    P, k = wl.P, wl.k
    with ClockSampler(gpu_id(local_rank)) as clk:
        if args.path not in gw.paths:
            raise SystemExit(f"--path {args.path} needs k <= 4 micro-batches ({wl.name} has k = {k})")
        names = [args.path] + [p for p in gw.paths if p != args.path]
        timed = {p: time_path(args, gw, p, world) for p in names}
        head = timed[args.path]
        graphs = {p: time_graph(args, gw, p, world) for p in names} if args.graph else None
        e2e = None if args.no_e2e else run_e2e(args, gw, world)
        st = tl.tl_read_status(gw.ctx)
        skipped = time_skipped(args, gw, args.path, world)
    kernels = head["kernels"]
    dom = max((n for n in kernels if "achieved_gbs" in kernels[n]), key=lambda n: kernels[n]["share"])
    peak, peak_kind = hbm_peak()
    out = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": f"synthetic (seeded; random-init masters, N(0,{wl.grad_std:g}) {wl.grad_dtype} grads)",
        "config": {"workload": f"{wl.name}: ~1.24B-param Llama tensor list, {len(wl.numel)} tensors, P={P}, "
                               f"bf16 params/grads, fp32 master/m/v/acc, k={k} micro-batches"
                               if wl.name == "llama_1b" else
                               f"{wl.name}: {len(wl.numel)} tensors, P={P}, {wl.param_dtype} params, "
                               f"{wl.grad_dtype} grads, k={k}",
                   "P": P, "k": k, "tensors": len(wl.numel), "counts": gw.counts, "path": args.path,
                   "layout": args.layout,
                   "l2": (f"no flush: every launch streams >= {P * 6 / 1e9:.1f} GB, far above the 129 MB L2"
                          if P * 6 > 10 * 129e6 else "small case: the working set fits in L2 (launch-latency bound)"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "table": table_plan(tl, wl.numel, local_rank)},
        "hbm": head["hbm"],
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["achieved_gbs"], "peak": peak,
                     "unit": "GB/s", "frac": kernels[dom]["frac"], "peak_kind": peak_kind,
                     "traffic": recorded_traffic(TRAFFIC_KEYS.get(dom, dom), wl.name, args.layout)},
        "kernels": kernels,
        "kernel_timing": "per-call CUDA events on the launching stream, from a second run of the same K steps "
                         "(the headline timing has no per-call events)",
        "gpu_launches": head["launches"],
        "paths": {p: {k2: timed[p][k2] for k2 in (("value", "ms_per_step", "hbm") if p == args.path else
                                                   ("value", "ms_per_step", "hbm", "kernels"))} for p in names},
        "clocks": clk.summary(),
        **({"cuda_graph": graphs} if graphs else {}),
        "status": {"S": st.S, "t": st.t, "skipped": st.skipped, "norm": st.norm},
    }
    out["skipped_step"] = skipped
    if e2e is not None:
        out["e2e"] = e2e
    return out


def time_skipped(args, gw, path, world):
    """The same path timed while every step overflows (a non-finite value planted in
    the first element of the first micro-batch's gradients): the overflow check still
    reads every gradient, the AdamW kernel exits on the device flag.  The element is
    restored afterwards."""
    import torch
    import loss_scaled_adamw_gb300 as tl
    g = gw.grads[0]
    pos = int(gw.plists_first_offset)
    saved = g[pos].clone()
    if g.dtype == torch.uint8:
        g[pos] = 0x7F                       # an E4M3 NaN code
    else:
        g[pos] = float("inf")
    for _ in range(max(args.warmup, 1)):
        gw.step(path)
    torch.cuda.synchronize()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        gw.step(path)
    t1.record()
    torch.cuda.synchronize()
    barrier()
    st = tl.tl_read_status(gw.ctx)
    g[pos] = saved
    torch.cuda.synchronize()
    el = max_over_ranks(t0.elapsed_time(t1) / 1e3, gw.device)
    return {"path": path, "ms_per_step": el / args.steps * 1e3, "value": whole_job_rate(gw.P, args.steps, world, el),
            "unit": UNIT, "skipped": int(st.skipped)}


def run_e2e(args, gw, world):
    """Same metric through the binding with every step's k micro-batch gradients copied
    from pinned host memory inside the timed region, and the step's status read back to
    the host.  Two device sets of gradient buffers alternate between steps, so the copies
    of step s+1 stream over the host link while step s computes (the link, ~211 GB/s on
    this box, is the bound: 19.8 GB per step at 1.24B parameters and k = 8)."""
    import torch
    import loss_scaled_adamw_gb300 as tl
    k = gw.wl.k
    why = ""
    try:
        host = [torch.empty(g.numel(), dtype=g.dtype, pin_memory=True) for g in gw.grads]
        for h, g in zip(host, gw.grads):
            h.copy_(g)
        sets = [gw.grads, [torch.empty_like(g) for g in gw.grads]]
    except RuntimeError as ex:      # pinned host memory or a second device set unavailable
        host = sets = None
        torch.cuda.empty_cache()
        why = str(ex).splitlines()[0]
    # every rank runs the leg or none does (its barriers and reductions are collective)
    if max_over_ranks(1.0 if why else 0.0, gw.device) > 0.0:
        return {"unavailable": "buffers of the end-to-end leg could not be allocated"
                               + (f": {why}" if why else " on another rank")}
    many = [gw.many, tl.ManyLists([gw.plist(g, 10 + i) for i, g in enumerate(sets[1])])]
    torch.cuda.synchronize()
    copy_stream = torch.cuda.Stream()
    compute = torch.cuda.current_stream()
    h2d = sum(h.numel() * h.element_size() for h in host)
    status_bytes = ctypes_sizeof_status()
    landed = [None, None]      # copy-done event of each set
    released = [None, None]    # compute-done-reading event of each set

    def enqueue_copies(step):
        b = step % 2
        with torch.cuda.stream(copy_stream):
            if released[b] is not None:
                copy_stream.wait_event(released[b])
            for i in range(k):
                sets[b][i].copy_(host[i], non_blocking=True)
            e = torch.cuda.Event()
            e.record(copy_stream)
            landed[b] = e

    remat = args.path == "remat"

    def compute_step(step):
        b = step % 2
        compute.wait_event(landed[b])
        e = torch.cuda.Event()
        if remat:
            tl.tl_unscale_check_many(gw.ctx, many[b], gw.counts, gw.N)
            tl.tl_grad_norm(gw.ctx, gw.wl.max_norm)
            tl.tl_clip_adamw_step(gw.ctx, gw.hp)   # the last reader of the lists
            e.record(compute)
        else:
            tl.tl_accumulate_many(gw.ctx, many[b], gw.counts, gw.N, 1)
            e.record(compute)
            tl.tl_grad_norm(gw.ctx, gw.wl.max_norm)
            tl.tl_clip_adamw_step(gw.ctx, gw.hp)
        released[b] = e
        tl.tl_scaler_update(gw.ctx)

    def run(nsteps):
        enqueue_copies(0)
        for step in range(nsteps):
            if step + 1 < nsteps:
                enqueue_copies(step + 1)
            compute_step(step)
            tl.tl_read_status(gw.ctx)  # device -> host read of the step's result
        torch.cuda.synchronize()

    run(2)
    barrier()
    t = time.perf_counter()
    run(args.steps)
    el = max_over_ranks(time.perf_counter() - t, gw.device)
    return {"value": whole_job_rate(gw.P, args.steps, world, el), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": status_bytes, "ms_per_step": el / args.steps * 1e3,
            "h2d_gbs": h2d * args.steps / el / 1e9,
            "how": "every step: the k gradient lists copied from pinned host memory (copy stream, into one of "
                   "two device buffer sets, overlapping the previous step's compute), the resident pass, "
                   "norm, clip+AdamW, scaler, and a blocking read of the step's status"}


def ctypes_sizeof_status() -> int:
    import ctypes
    import loss_scaled_adamw_gb300 as tl
    return ctypes.sizeof(tl.tl_status)


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(wl, n_params: int):
    """A contiguous slice of the workload's flat tensor list: masters and k gradients."""
    import torch
    from loss_scaled_adamw_gb300 import workloads as W
    n = min(n_params, wl.P)
    g = torch.Generator().manual_seed(W.SEED)
    master = (torch.randn(n, generator=g) * wl.master_std).numpy().astype(np.float32)
    grads = []
    for _ in range(wl.k):
        x = torch.randn(n, generator=g) * wl.grad_std
        if wl.grad_dtype == "e4m3b16":      # the slice taken as one tensor of n elements
            codes, scales = W.quantize_e4m3b16(x, [n])
            grads.append((codes.numpy(), scales.numpy()))
        elif wl.grad_dtype == "f32":
            grads.append(x.numpy().astype(np.float32))
        else:
            grads.append(W.to_16bit(x, wl.grad_dtype).view(torch.int16).numpy().view(np.uint16))
    p0 = W.to_16bit(torch.from_numpy(master), wl.param_dtype).view(torch.int16).numpy().view(np.uint16)
    return master, p0, grads


def host_cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


class SlicedOracle:
    """The oracle's element-wise functions (tlo_accumulate, tlo_unscale_check, tlo_sumsq,
    tlo_adamw_recast), unchanged, run on `threads` disjoint contiguous slices of one flat
    list from host threads (ctypes releases the GIL during each call); the slices'
    squared norms are added in slice order, and the per-update scalars are the oracle's
    own (tlo_adamw_prepare, tlo_scaler_update).  A timing baseline on all host cores, not
    a parity reference."""

    def __init__(self, master, p0, wl, threads: int):
        import ctypes
        import oracle
        self.ct = ctypes
        self.lib = oracle.load()
        self.oracle = oracle
        self.w = np.ascontiguousarray(master, np.float32).copy()
        self.m = np.zeros_like(self.w)
        self.v = np.zeros_like(self.w)
        self.p = np.ascontiguousarray(p0, np.uint16).copy()
        self.acc = np.empty_like(self.w)
        self.n = self.w.size
        self.wl = wl
        self.pdt = oracle.dtype_code(wl.param_dtype)
        self.threads = max(1, int(threads))
        step = (self.n + self.threads - 1) // self.threads
        self.slices = [(lo, min(self.n, lo + step)) for lo in range(0, self.n, step)]
        self.state = oracle.State(1.0, 0, 0, 1.0, 1.0)
        self.cfg = oracle.ScalerCfg(0, 2.0, 0.5, 2000, 1.0, 2.0 ** 127)
        self.hp = oracle.AdamWHP(1e-3, 0.9, 0.95, 1e-8, 0.1)
        from concurrent.futures import ThreadPoolExecutor
        self.pool = ThreadPoolExecutor(self.threads)

    def _at(self, a, lo):
        return self.ct.c_void_p(a.ctypes.data + a.itemsize * lo)

    def _par(self, fn):
        return list(self.pool.map(lambda s: fn(*s), self.slices))

    def step(self, grads, counts, max_norm):
        lib, ct, orc = self.lib, self.ct, self.oracle
        N = sum(counts)
        for i, g in enumerate(grads):
            if isinstance(g, tuple):            # 8-bit: the oracle's dequantization of the sample first
                g = orc.dequant_e4m3b16(g[0], g[1], [g[0].size])
                dt = orc.DT_F32
            else:
                dt = orc.DT_F32 if g.dtype == np.float32 else orc.dtype_code(self.wl.grad_dtype)
            wi = lib.tlo_microbatch_weight(counts[i], N)
            self._par(lambda lo, hi: lib.tlo_accumulate(self._at(self.acc, lo), self._at(g, lo), dt, hi - lo, wi,
                                                        1 if i == 0 else 0))
        found = any(self._par(lambda lo, hi: lib.tlo_unscale_check(self._at(self.acc, lo), hi - lo, self.state.S)))
        sums = self._par(lambda lo, hi: lib.tlo_sumsq(self._at(self.acc, lo), hi - lo))
        sumsq = 0.0
        for x in sums:
            sumsq += x
        st = self.state
        b1n = st.b1p * float(np.float32(self.hp.beta1))
        b2n = st.b2p * float(np.float32(self.hp.beta2))
        if not found and np.isfinite(sumsq):
            coef = lib.tlo_clip_coef(lib.tlo_norm_from_sumsq(sumsq), max_norm)
            sc = lib.tlo_adamw_prepare(ct.byref(self.hp), b1n, b2n)
            self._par(lambda lo, hi: lib.tlo_adamw_recast(self._at(self.w, lo), self._at(self.m, lo),
                                                          self._at(self.v, lo), self._at(self.p, lo), self.pdt,
                                                          self._at(self.acc, lo), hi - lo, coef, ct.byref(sc)))
        else:
            found = True
        lib.tlo_scaler_update(ct.byref(st), ct.byref(self.cfg), 1 if found else 0, b1n, b2n)


def time_oracle(wl, seconds: float, steps=None, threads: int = 1):
    """Time the oracle's logical update on a contiguous sample of the workload sized for
    about `seconds` of CPU time (at most 2^27 parameters, repeated over several logical
    updates when the cap binds, unless `steps` is given).
    threads = 1: the plain single-threaded oracle (tlo_step); threads > 1: its element
    functions on disjoint slices on that many host cores (SlicedOracle)."""
    import oracle

    def make(n):
        master, p0, grads = oracle_sample(wl, n)
        if threads == 1:
            return oracle.Oracle(master, p0, wl.param_dtype, wl.grad_dtype, numel=[master.size]), grads
        return SlicedOracle(master, p0, wl, threads), grads

    n = 1 << 20
    o, grads = make(n)
    t = time.perf_counter()
    o.step(grads, wl.counts(1), wl.max_norm)
    per_param = (time.perf_counter() - t) / n
    # at most 2^27 parameters: drawing the sample's inputs costs more than stepping them
    n = int(min(max(seconds / per_param / (steps or 1), 1 << 20), 1 << 27, wl.P))
    if steps is None:
        steps = max(1, int(round(seconds / (per_param * n))))
    o, grads = make(n)
    t = time.perf_counter()
    for s in range(steps):
        o.step(grads, wl.counts(s + 1), wl.max_norm)
    el = time.perf_counter() - t
    how = "single-threaded C oracle (tlo_step)" if threads == 1 else \
        f"the C oracle's element functions on {threads} disjoint slices, one host thread each"
    return {"value": n * steps / el / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} parameters (a contiguous slice of the {wl.name} tensor list), k={wl.k}, "
                      f"{steps} logical update(s), {el:.1f} s, {how}"}


def run_reference(args, rank, world):
    from loss_scaled_adamw_gb300 import workloads as W
    import oracle
    oracle.build()
    wl = W.make(args.workload)
    per_step = max(args.cpu_seconds / max(args.steps, 1), 1.0)
    cores = host_cores()
    for _ in range(min(args.warmup, 1)):
        time_oracle(wl, 0.5, threads=cores)
    t = time.perf_counter()
    res = time_oracle(wl, per_step * args.steps, steps=args.steps, threads=cores)
    el = time.perf_counter() - t
    return {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": f"{wl.name}: sample of the tensor list on the host cores", "P": wl.P, "k": wl.k},
            "cpu_baseline": res, "e2e": {"value": res["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                                          "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        # rank 0 alone times the oracle on the host cores; other ranks exit without work
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
    out = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        # the oracle's CPU baseline: rank 0 of a single-GPU run only
        if not args.no_cpu_baseline and world == 1:
            from loss_scaled_adamw_gb300 import workloads as W
            import oracle
            oracle.build()
            wl = W.make(args.workload)
            # the oracle on every host core (its element functions on disjoint slices),
            # and the plain single-threaded oracle beside it
            out["cpu_baseline"] = time_oracle(wl, args.cpu_seconds, threads=host_cores())
            out["cpu_baseline_single_core"] = time_oracle(wl, args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
