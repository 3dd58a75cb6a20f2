#!/usr/bin/env python
"""Benchmark: Gpixel/s labelled (device-timed) and % of the HBM roofline.

Default workload: the 806.4-Mpixel construction-sheet analogue (24000 rows x
33600 columns, RGBA, 8-connectivity, every pixel labelled) -- the workload the
headline target is quoted on.  One step is one ccl_label call over the whole
sheet (all four stages: Start, Connect, Collapse, Number).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload c0|c1|c2|c3:<structure>:<conn>:<mode>|c4|c4i|c4rgb|c4:HxW|flat:HxW]

Prints ONE JSON line (rank 0).  Device time: CUDA events on the launching
stream around exactly K steps, inputs resident in HBM.  Per-stage times come
from CUDA events the library records on the same stream (option
CCL_OPT_STAGE_EVENTS).  e2e: the same metric through ccl_label_host with
page-locked host buffers, host<->device copies inside the timed region, with
the same copies timed alone beside it (the link's floor).  cpu_baseline: the
oracle (single-threaded BFS) over the whole workload on this machine's host
cores; its labels and counts are compared with the device run's, every pixel
("parity").  --impl reference: the oracle on a band of the sheet.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Gpixel/s labelled (device-timed) and % of HBM roofline, 1 GB300"
UNIT = "Gpixel/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0          # the GB300's nominal HBM3e bandwidth, for the second fraction
L2_BYTES = 129 * 1024 * 1024
REF_ROWS = 1200           # rows of the sheet one reference step labels


# ------------------------------------------------------------------ workloads

def make_workload(name, device):
    """Returns (config dict, device tensor [B,H,W] or [H,W], pb, conn, mode)."""
    import workloads as wl
    if name == "c4":
        img = wl.c4_sheet(device=device)
        return (dict(workload="c4_sheet_24000x33600_rgba", batch=1, H=wl.C4_H, W=wl.C4_W,
                     pixel_bytes=4, connectivity=8, mode="all"), img, 4, 8, 0)
    if name == "c4i":               # the sheet with its white paper ignored
        img = wl.c4_sheet(device=device)
        return (dict(workload="c4_sheet_24000x33600_rgba_paper_ignored", batch=1, H=wl.C4_H,
                     W=wl.C4_W, pixel_bytes=4, connectivity=8, mode="ignore",
                     ignore_value="0xFFFFFFFF"), img, 4, 8, -1)
    if name == "c4rgb":             # the sheet as packed 24-bit RGB (2.4 GB)
        img = wl.c4_sheet_rgb(device=device)
        return (dict(workload="c4_sheet_24000x33600_rgb24", batch=1, H=wl.C4_H, W=wl.C4_W,
                     pixel_bytes=3, connectivity=8, mode="all"), img, 3, 8, 0)
    if name.startswith("c4:"):      # the sheet generator at another size, e.g. c4:6000x8400
        H, W = (int(v) for v in name[3:].split("x"))
        img = wl.c4_sheet(device=device, H=H, W=W)
        return (dict(workload="c4_sheet_%dx%d_rgba" % (H, W), batch=1, H=H, W=W,
                     pixel_bytes=4, connectivity=8, mode="all"), img, 4, 8, 0)
    if name.startswith("flat:"):    # one colour everywhere, e.g. flat:6000x8400: the fixed cost
        H, W = (int(v) for v in name[5:].split("x"))
        import torch
        img = torch.full((H, W), -1, dtype=torch.int32, device=device)
        return (dict(workload="flat_%dx%d_rgba" % (H, W), batch=1, H=H, W=W,
                     pixel_bytes=4, connectivity=8, mode="all"), img, 4, 8, 0)
    if name == "c0":
        img = wl.c0_drawing(device=device)
        return (dict(workload="c0_drawing_1024_rgba", batch=1, H=1024, W=1024, pixel_bytes=4,
                     connectivity=8, mode="all"), img, 4, 8, 0)
    if name == "c1":
        img = wl.c1_masks(device=device)
        return (dict(workload="c1_masks_64x1024x1024_u8", batch=64, H=1024, W=1024,
                     pixel_bytes=1, connectivity=8, mode="binary"), img, 1, 8, 1)
    if name == "c2":
        img = wl.c2_slide(device=device)
        return (dict(workload="c2_slide_20000x20000_u8", batch=1, H=20000, W=20000,
                     pixel_bytes=1, connectivity=4, mode="binary"), img, 1, 4, 1)
    if name.startswith("c3"):
        _, structure, conn, mode = name.split(":")
        img = wl.c3_structures(device=device)[structure]
        m = 1 if mode == "binary" else 0
        return (dict(workload="c3_%s_8192x8192_u8" % structure, batch=1, H=8192, W=8192,
                     pixel_bytes=1, connectivity=int(conn), mode=mode), img, 1, int(conn), m)
    raise SystemExit("unknown workload %r" % name)


def sheet_band(rows, device="cpu"):
    import workloads as wl
    return wl.c4_sheet(device=device, rows=(0, rows))


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_sha():
    """Hash of the CUDA sources without their comments and whitespace: a
    committed ncu traffic figure is only used while the code it was measured
    on is unchanged (a comment edit does not change a kernel)."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "connected_component_labelling_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh")):
            continue
        with open(os.path.join(csrc, name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", " ", text)                 # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def traffic_per_px(kernel, workload):
    """DRAM bytes per pixel of `kernel` from the committed ncu summary, or
    None when the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("source_sha") != source_sha():
        return None
    ent = t.get("kernels", {}).get(workload, {}).get(kernel)
    return None if ent is None else float(ent)


class ClockSampler:
    """nvidia-smi samples (every 200 ms) of the GPU this rank uses; keeps
    the arrival time of every line so samples can be matched to a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [s.strip() for s in line.split(",")]))

    def wait_first(self, timeout=10.0):
        t0 = time.time()
        while self.proc and not self.rows and time.time() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [r for (t, r) in self.rows if t0 <= t <= t1 + 0.2]
        note = "inside the timed region"
        if not inside:   # region shorter than the sampling period: nearest samples
            inside = [r for (t, r) in self.rows if t0 - 0.5 <= t <= t1 + 0.5]
            note = "within 0.5 s of the timed region (region shorter than the 200 ms period)"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            try:
                sm.append(float(r[1])); mx.append(float(r[2]))
            except Exception:
                continue
            for k, nm in enumerate(names):
                if len(r) > 5 + k and r[5 + k].lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": note}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (torch.cuda.is_available() and args.impl != "reference") else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ oracle legs

def time_oracle(img_np, conn, mode):
    import oracle
    t0 = time.perf_counter()
    oracle.label(img_np, conn, mode)
    return time.perf_counter() - t0


def host_info():
    """The host the oracle is timed on: logical cores and the CPU model as
    /proc/cpuinfo names it (x86: model name; Arm: implementer and part)."""
    import platform
    info = {"nproc": os.cpu_count(), "machine": platform.machine()}
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        if "model name" in fields:
            info["cpu"] = fields["model name"]
        elif "CPU part" in fields:
            info["cpu"] = "implementer %s part %s" % (fields.get("CPU implementer", "?"),
                                                      fields["CPU part"])
    except OSError:
        pass
    return info


def run_reference(args, world, rank):
    """The oracle as it stands, timed on this machine's host cores, one step =
    one labelling of a REF_ROWS-row band of the sheet."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    oracle.build()
    rows = args.ref_rows
    band = sheet_band(rows).numpy().view(np.uint32)
    px = band.size
    for _ in range(args.warmup):
        time_oracle(band, 8, oracle.MODE_ALL)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle(band, 8, oracle.MODE_ALL)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    gpxs = px / dt / 1e9
    sample = "rows 0-%d of the 24000 x 33600 sheet (%d px) per step, single thread" % (rows, px)
    line = {"impl": "reference", "metric": METRIC, "value": gpxs, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": "c4_sheet_24000x33600_rgba", "batch": 1, "H": 24000,
                       "W": 33600, "pixel_bytes": 4, "connectivity": 8, "mode": "all",
                       "sample_rows": rows},
            "cpu_baseline": {"value": gpxs, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample, "host": host_info()},
            "e2e": {"value": gpxs, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ccl", choices=["ccl", "reference"])
    ap.add_argument("--workload", default="c4")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stats", action="store_true",
                    help="skip timing ccl_region_stats on the labels")
    ap.add_argument("--counters", action="store_true",
                    help="also label the workload once with the counters build of the library "
                         "and report walks, steps per walk and links (not timed)")
    ap.add_argument("--ref-rows", type=int, default=REF_ROWS,
                    help="rows of the sheet one reference (oracle) step labels")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import numpy as np
    import torch
    import connected_component_labelling_gb300 as ccl

    ccl.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg, img, pb, conn, mode = make_workload(args.workload, dev)
    img = img.contiguous()
    B, H, W = cfg["batch"], cfg["H"], cfg["W"]
    px = B * H * W
    labels = torch.empty(px, dtype=torch.int32, device=dev)
    nreg = torch.empty(B, dtype=torch.int32, device=dev)
    # (ignoring one value is the binary mode's pipeline: its workspace size)
    wsb = ccl.ccl_workspace_bytes(B, H, W, pb, conn, 1 if mode != 0 else 0)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def step():
        if mode < 0:   # one value ignored
            rc = ccl.ccl_label_ignore(img.data_ptr(), B, H, W, pb, conn,
                                      int(cfg["ignore_value"], 16), labels.data_ptr(),
                                      nreg.data_ptr(), ws.data_ptr(), wsb, sp)
        else:
            rc = ccl.ccl_label_ws(img.data_ptr(), B, H, W, pb, conn, mode, labels.data_ptr(),
                                  nreg.data_ptr(), ws.data_ptr(), wsb, sp)
        if rc != ccl.CCL_OK:
            raise ccl.CCLError(rc, "labelling call")

    for _ in range(args.warmup):
        step()
    ccl.check_status(stream)

    small = (px * (pb + 4)) < 2 * L2_BYTES
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev) if small else None
    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [s for s in vis.split(",") if s.strip()]
        if local < len(ids):
            gpu_index = ids[local]
    sampler = ClockSampler(gpu_index)
    sampler.wait_first()

    ccl.ccl_stage_times()                       # forget anything recorded before
    ccl.ccl_set_option(ccl.CCL_OPT_STAGE_EVENTS, 1)
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = ccl.ccl_kernel_launches()
    t_wall0 = time.time()
    if not small:
        # one event after each step as well, for the per-step median and minimum
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e0.record(stream)
        for k in range(args.steps):
            step()
            marks[k].record(stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        total_ms = e0.elapsed_time(e1)
        step_ms = [(marks[k - 1] if k else e0).elapsed_time(marks[k]) for k in range(args.steps)]
    else:
        # inputs fit in L2: flush it between steps, outside the timed events
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        step_ms = [a.elapsed_time(b) for a, b in evs]
        total_ms = sum(step_ms)
    t_wall1 = time.time()
    launches = ccl.ccl_kernel_launches() - launches0
    barrier(world)
    ccl.ccl_set_option(ccl.CCL_OPT_STAGE_EVENTS, 0)
    sampler.stop()
    ccl.check_status(stream)
    stage_ms, ncalls = ccl.ccl_stage_times()
    ms = total_ms / args.steps
    ms_max = max_over_ranks(ms, world)
    value = world * px / (ms_max * 1e-3) / 1e9
    clocks = sampler.summary(t_wall0, t_wall1)
    n_regions = nreg.cpu().tolist()

    # ---- roofline
    peak, peak_kind = load_peaks()
    names = [ccl.ccl_stage_name(k) for k in range(len(stage_ms))]
    per_call = [s / max(1, ncalls) for s in stage_ms]
    # bytes per pixel charged to the stages that stream whole images:
    # tile_local carries the method's figure (image read once + int32 labels
    # written), the per-unit figure of the roofline when it dominates; number
    # its own least traffic (labels written, 4 B)
    alg = {"tile_local": pb + 4, "number": 4}
    dom = max(range(len(per_call)), key=lambda k: per_call[k]) if per_call else 0
    dom_name = names[dom] if names else "tile_local"
    dom_alg = alg.get(dom_name)
    stages = {}
    for k, nm in enumerate(names):
        ent = {"ms": per_call[k], "share": per_call[k] / sum(per_call) if sum(per_call) else None}
        if nm in alg:
            gbs = alg[nm] * px / (per_call[k] * 1e-3) / 1e9 if per_call[k] > 0 else None
            ent.update({"alg_bytes_per_px": alg[nm], "achieved_gbs": gbs,
                        "frac": gbs / peak if gbs else None})
        stages[nm] = ent
    if dom_alg is None:
        dom_alg = 0
    achieved = dom_alg * px / (per_call[dom] * 1e-3) / 1e9 if per_call and per_call[dom] > 0 else None
    tpp = traffic_per_px(dom_name, cfg["workload"])
    roofline = {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
                "traffic": (tpp * px) if tpp is not None else None,
                "alg_bytes": dom_alg * px, "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s"}
    path_gbs = (pb + 4) * px / (ms * 1e-3) / 1e9
    roofline_path = {"bound": "hbm", "alg_bytes_per_px": pb + 4, "achieved": path_gbs,
                     "peak": peak, "unit": "GB/s", "frac": path_gbs / peak,
                     "frac_of_nominal": path_gbs / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "note": "whole ccl_label call: image read once + int32 label write; "
                             "frac against the measured copy bandwidth, frac_of_nominal "
                             "against the GB300's nominal 8 TB/s"}

    # ---- region statistics of the labels just made (the step after
    # labelling), timed on their own: labels read once, one 40-byte entry
    # written per region
    region_stats = None
    if not args.no_stats:
        total = int(nreg.to(torch.int64).sum().item())
        sraw = torch.empty(max(total, 1) * ccl.STAT_BYTES, dtype=torch.uint8, device=dev)
        swb = ccl.ccl_region_stats_workspace_bytes(B)
        sws = torch.empty(swb, dtype=torch.uint8, device=dev)

        def sstep():
            rc = ccl.ccl_region_stats(labels.data_ptr(), B, H, W, nreg.data_ptr(), sraw.data_ptr(),
                                      total, sws.data_ptr(), swb, sp)
            if rc != ccl.CCL_OK:
                raise ccl.CCLError(rc, "ccl_region_stats")

        for _ in range(3):
            sstep()
        ccl.check_status(stream)
        ksteps = max(3, min(args.steps, 20))
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(ksteps)]
        barrier(world)
        torch.cuda.synchronize(dev)
        for a, b in sev:
            if flush is not None:
                flush.fill_(1)
            a.record(stream)
            sstep()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ccl.check_status(stream)
        sms = max_over_ranks(sum(a.elapsed_time(b) for a, b in sev) / ksteps, world)
        salg = 4 * px + ccl.STAT_BYTES * total
        sgbs = salg / (sms * 1e-3) / 1e9
        region_stats = {"api": "ccl_region_stats", "ms": sms, "value": world * px / (sms * 1e-3) / 1e9,
                        "unit": UNIT, "steps": ksteps, "regions": total, "alg_bytes": salg,
                        "achieved_gbs": sgbs, "peak": peak, "frac": sgbs / peak,
                        "note": "labels read once (4 B/px) + one 40-byte entry per region; "
                                "3 kernel launches per call"}
        del sraw, sws

    # ---- event counters: one untimed call through the counters build
    counters = None
    if args.counters and rank == 0:
        CL = ccl.counters_library()
        ccl.read_counters(CL, reset=True)
        if mode < 0:
            rc = CL.ccl_label_ignore(img.data_ptr(), B, H, W, pb, conn, int(cfg["ignore_value"], 16),
                                     labels.data_ptr(), nreg.data_ptr(), ws.data_ptr(), wsb, sp)
        else:
            rc = CL.ccl_label_ws(img.data_ptr(), B, H, W, pb, conn, mode, labels.data_ptr(),
                                 nreg.data_ptr(), ws.data_ptr(), wsb, sp)
        if rc != ccl.CCL_OK:
            raise ccl.CCLError(rc, "counters build")
        c = ccl.read_counters(CL, reset=True)
        counters = dict(c)
        counters["tile_steps_per_walk"] = c["tile_steps"] / max(1, c["tile_walks"])
        counters["global_steps_per_walk"] = c["global_steps"] / max(1, c["global_walks"])
        counters["tile_links_per_px"] = c["tile_links"] / px
        counters["build"] = "libccl_counters.so (-DCCL_COUNTERS), one call, not timed"

    # ---- e2e through the host entry point, and the copies alone (the link's
    # floor for the same bytes: the image up, the labels down)
    e2e = None
    if not args.no_e2e and mode >= 0:
        himg = img.cpu().contiguous().pin_memory()
        hlab = torch.empty(px, dtype=torch.int32).pin_memory()
        hn = torch.empty(B, dtype=torch.int32).pin_memory()
        rc = ccl.ccl_label_host(himg.data_ptr(), B, H, W, pb, conn, mode, hlab.data_ptr(),
                                hn.data_ptr(), sp)      # warm the pool
        if rc != ccl.CCL_OK:
            raise ccl.CCLError(rc, "ccl_label_host")
        torch.cuda.synchronize(dev)
        dimg = torch.empty_like(img)
        up_ms, down_ms = [], []
        for _ in range(args.e2e_steps):
            a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            a.record(stream)
            dimg.copy_(himg.view(dimg.shape), non_blocking=True)
            b.record(stream)
            hlab.copy_(labels, non_blocking=True)
            c.record(stream)
            torch.cuda.synchronize(dev)
            up_ms.append(a.elapsed_time(b))
            down_ms.append(b.elapsed_time(c))
        del dimg
        floor_ms = statistics.median(up_ms) + statistics.median(down_ms)
        floor_mean_ms = statistics.mean(up_ms) + statistics.mean(down_ms)
        barrier(world)
        t0 = time.perf_counter()
        call_ms = []   # each call returns after its own synchronisation
        for _ in range(args.e2e_steps):
            tc = time.perf_counter()
            rc = ccl.ccl_label_host(himg.data_ptr(), B, H, W, pb, conn, mode, hlab.data_ptr(),
                                    hn.data_ptr(), sp)
            call_ms.append((time.perf_counter() - tc) * 1e3)
            if rc != ccl.CCL_OK:
                raise ccl.CCLError(rc, "ccl_label_host")
        dt = (time.perf_counter() - t0) / args.e2e_steps
        dt = max_over_ranks(dt, world)
        same = bool(torch.equal(hlab, labels.cpu()))
        e2e = {"value": world * px / dt / 1e9, "unit": UNIT, "ms_per_step": dt * 1e3,
               "h2d_bytes_per_step": px * pb, "d2h_bytes_per_step": px * 4 + B * 4,
               "steps": args.e2e_steps, "api": "ccl_label_host (pinned host buffers)",
               "labels_match_device_run": same,
               "ms_per_call_median": statistics.median(call_ms), "ms_per_call_min": min(call_ms),
               "ms_per_call_max": max(call_ms), "ms_per_call": [round(c, 3) for c in call_ms],
               "copy_floor_ms": floor_ms, "copy_floor_mean_ms": floor_mean_ms,
               "frac_of_floor_median": floor_ms / statistics.median(call_ms),
               "h2d_ms": statistics.median(up_ms),
               "d2h_ms": statistics.median(down_ms), "frac_of_floor": floor_ms / (dt * 1e3),
               "floor_note": "the same pinned buffers copied alone in this process (image up, "
                             "then labels down, median of the e2e steps); frac_of_floor = "
                             "copy_floor_ms / ms_per_step; frac_of_floor_median = copy_floor_ms / "
                             "ms_per_call_median; copy_floor_mean_ms: the mean copies, which stall "
                             "like the calls (the host side is shared)"}
        del himg, hlab

    # ---- cpu baseline and parity: the oracle over the whole workload on this
    # host (1 thread), its labels and counts compared with the device run's
    cpu_baseline = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        if pb == 3:   # [B, H, W, 3] bytes
            himg_np = img.cpu().numpy().reshape(B, H, W, 3)
        else:
            himg_np = img.cpu().numpy().view({1: np.uint8, 2: np.uint16, 4: np.uint32}[pb])
            himg_np = himg_np.reshape(B, H, W)
        t0 = time.perf_counter()
        if mode < 0:
            olab, on = oracle.label_ignore(himg_np, int(cfg["ignore_value"], 16), conn)
        else:
            olab, on = oracle.label(himg_np, conn, oracle.MODE_BINARY if mode == 1 else oracle.MODE_ALL)
        dt = time.perf_counter() - t0
        del himg_np
        dlab = labels.cpu().numpy()
        labels_equal = bool(np.array_equal(olab.reshape(-1), dlab))
        counts_equal = bool(np.array_equal(np.asarray(on).reshape(-1), np.asarray(n_regions)))
        parity = {"labels_equal": labels_equal, "counts_equal": counts_equal, "pixels": px,
                  "against": "oracle (plain BFS, CPU), every pixel of the last timed call's labels"}
        del olab, dlab
        cpu_baseline = {"value": px / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
                        "sample": "the whole workload (%d px), one single-threaded BFS pass, %.1f s"
                                  % (px, dt),
                        "host": host_info()}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                "ms_per_step_median": statistics.median(step_ms), "ms_per_step_min": min(step_ms),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "int32", "data": "synthetic",
                "config": dict(cfg, l2=("L2 flushed between steps (outside the events)" if small
                                        else "inputs larger than L2 (%.2f GB moved per step)"
                                        % (px * (pb + 4) / 1e9)),
                               parallelism="replicas" if world > 1 else "single"),
                "roofline": roofline, "roofline_path": roofline_path, "stages": stages,
                "parity": (parity["labels_equal"] and parity["counts_equal"]) if parity else None,
                "parity_detail": parity, "cpu_baseline": cpu_baseline, "e2e": e2e, "gpu_launches": launches,
                "region_stats": region_stats, "counters": counters,
                "clocks": clocks, "n_regions": n_regions[:8],
                "kernel_source_sha": source_sha()}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
