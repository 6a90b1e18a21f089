"""Benchmark: fwd+bwd effective TFLOP/s of tile-top-k block-sparse attention
on the video-DiT workload (latent 20x48x80 tiled 4x8x8 -> 300 tiles, 76,800
tokens; B=1, 40 heads, D=128, bf16, BSHD; top-30 KV tiles per Q tile).

One step = the whole hot path on one batch: block map (pool + coarse top-k
+ both indices), forward (O, LSE) and backward (dQ, dK, dV), through the
C ABI. FLOPs are counted on selected tile pairs only:
2*D*M*N*(2 fwd + 5 bwd) per pair, M = query rows of the tile, N = valid
keys of the KV tile.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 1|3|4|5|6] [--shard heads|replicas]

Under torchrun the problem's heads are split over the ranks (vsa_head_slice:
whole GQA groups per rank, no exchange between ranks; strong scaling), or,
with --shard replicas, every rank runs its own copy (weak scaling); timing is
the max over ranks. --impl reference times the CPU oracle on a bounded
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd effective TFLOP/s (selected blocks) on 1 GB300; % of bf16 TC peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Per-launch DRAM bytes of the attention kernels come from an ncu capture of
# this workload cut to a few heads (every head is an independent problem, so
# a launch's traffic scales with the heads). The capture records the hash of
# the source file that defines each kernel; a kernel whose source changed
# since then reports no traffic.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_bytes_video_dit_4heads.json")
KERNEL_SOURCE = {"fwd_attn": "fwd_kernel.cu", "fwd_redo": "fwd_kernel.cu", "bwd_dkdv": "bwd_kernels.cu",
                 "bwd_dq": "bwd_kernels.cu", "bwd_prep": "bwd_kernels.cu", "dkdv_order": "bwd_kernels.cu",
                 "pool": "index_kernels.cu", "select_topk": "index_kernels.cu",
                 "transpose_index": "index_kernels.cu"}
# CUDA kernel function -> the name the library's launch records use
KERNEL_FUNCTION = {"k_fwd2": "fwd_attn", "k_fwd": "fwd_redo", "k_dkdv": "bwd_dkdv", "k_dq": "bwd_dq",
                   "k_bwd_prep": "bwd_prep", "k_dk_order": "dkdv_order", "k_pool": "pool",
                   "k_select": "select_topk", "k_transpose": "transpose_index"}
CPU_SAMPLE_TILES = 2   # query tiles (forward, dQ) and KV tiles (dK, dV) of the oracle sample


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(kernel):
    """Hash (first 16 hex digits of SHA-256) of the source file defining a kernel."""
    path = os.path.join(ROOT, "bwd_tile_mean_gb300", "csrc", KERNEL_SOURCE[kernel])
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_traffic(kernel, heads):
    """(bytes per launch at `heads` heads, note) from the committed capture,
    or (None, why not)."""
    if kernel not in KERNEL_SOURCE or not os.path.exists(TRAFFIC_FILE):
        return None, "no ncu capture of this kernel"
    with open(TRAFFIC_FILE) as f:
        cap = json.load(f)
    k = cap.get("kernels", {}).get(kernel)
    if k is None:
        return None, "no ncu capture of this kernel"
    if k.get("source_sha256") != source_sha(kernel):
        return None, f"kernel source changed since the capture ({cap.get('captured', '?')})"
    return (k["dram_bytes_read"] + k["dram_bytes_write"]) * heads / cap["heads"], \
        f"ncu capture {cap.get('captured', '?')} on {cap['heads']} heads, scaled to {heads}"


def write_traffic(csv_path, heads, command):
    """Per-launch DRAM bytes of each kernel from an ncu CSV (--metrics
    dram__bytes_read.sum,dram__bytes_write.sum --csv --log-file) of one step
    at `heads` heads, written to TRAFFIC_FILE with the source hashes."""
    import csv
    import re
    scale = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12}
    launches = {}  # (ncu launch id, kernel) -> {metric: bytes}
    with open(csv_path, newline="") as fh:
        lines = [ln for ln in fh if ln.startswith('"')]
    for row in csv.DictReader(lines):
        name = row.get("Kernel Name", "")
        kern = next((v for k, v in KERNEL_FUNCTION.items() if re.search(rf"\b{k}\b", name)), None)
        metric = row.get("Metric Name", "")
        if kern is None or metric not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        val = float(row["Metric Value"].replace(",", "")) * scale[row["Metric Unit"].strip().lower()]
        launches.setdefault((row["ID"], kern), {})[metric] = val
    out = {}
    for (_, kern), m in launches.items():
        k = out.setdefault(kern, {"launches": 0, "dram_bytes_read": 0.0, "dram_bytes_write": 0.0})
        k["launches"] += 1
        k["dram_bytes_read"] += m.get("dram__bytes_read.sum", 0.0)
        k["dram_bytes_write"] += m.get("dram__bytes_write.sum", 0.0)
    for kern, k in out.items():
        n = k["launches"]
        k["dram_bytes_read"] = round(k["dram_bytes_read"] / n)
        k["dram_bytes_write"] = round(k["dram_bytes_write"] / n)
        k["source_sha256"] = source_sha(kern)
    cap = {"heads": heads, "captured": time.strftime("%Y-%m-%d"), "command": command,
           "note": "bytes per launch, averaged over the captured launches of each kernel", "kernels": out}
    with open(TRAFFIC_FILE, "w") as fh:
        json.dump(cap, fh, indent=1, sort_keys=True)
        fh.write("\n")
    print(json.dumps(cap, indent=1, sort_keys=True))


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x, world_size, device):
    """Max of a per-rank float over all ranks (identity on one rank)."""
    return _reduce(x, world_size, device, "max")


def reduce_sum(x, world_size, device):
    """Sum of a per-rank float over all ranks (identity on one rank)."""
    return _reduce(x, world_size, device, "sum")


def _reduce(x, world_size, device, op):
    if world_size == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, bus_id=None):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits", "-lms", "50"]
        if bus_id:
            cmd.insert(1, f"--id={bus_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < len(self.FIELDS):
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- CPU oracle

def oracle_sample(n_tiles=CPU_SAMPLE_TILES, seed=42):
    """Time the CPU oracle (block map + forward + backward) on a bounded
    sample of the workload: one head of the same shape (300 tiles, topk 30),
    its whole block map, the forward and dQ rows of n_tiles query tiles and
    dK/dV of n_tiles KV tiles. Credited with the effective FLOPs (14 D M N)
    of the selected pairs of those query tiles. Returns a dict: tflops,
    seconds, the seconds of each part, the sample and the threads used."""
    import numpy as np
    from bwd_tile_mean_gb300.inputs import Problem, make_tensors
    from oracle import oracle as orc

    nt = 300
    p = Problem("video-dit-1head", "bshd", 1, 1, 1, 128, 256, 256, nt, nt, q_var=[256] * nt, kv_var=[256] * nt,
                topk=30, seed=seed)
    t = make_tensors(p)
    q, k, v, dO = (orc._f64(t[n]) for n in ("q", "k", "v", "dO"))
    orc.lib()
    parts = {}
    t0 = time.perf_counter()
    m, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    t1 = time.perf_counter()
    rows = np.asarray([(0, 0, i * 256 + r) for i in range(n_tiles) for r in range(256)], dtype=np.int32)
    orc.forward_rows(p, q, k, v, qi, qc, p.cap, rows=rows)
    t2 = time.perf_counter()
    orc.backward_dq_rows(p, dO, q, k, v, qi, qc, p.cap, rows=rows)
    t3 = time.perf_counter()
    tiles = np.asarray([(0, 0, j) for j in range(n_tiles)], dtype=np.int32)
    orc.backward_dkdv_tiles(p, dO, q, k, v, qi, qc, p.cap, tiles=tiles)
    t4 = time.perf_counter()
    parts = {"block_map_s": t1 - t0, "forward_s": t2 - t1, "dq_s": t3 - t2, "dkdv_s": t4 - t3}
    dt = t4 - t0
    pairs = int(qc[0, 0, :n_tiles].sum())
    flops = pairs * 2.0 * 128 * 256 * 256 * 7
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    desc = (f"oracle block map of one 300-tile head + forward and dQ of {n_tiles} query tiles' rows + dK/dV of "
            f"{n_tiles} KV tiles ({pairs} selected pairs credited, 14*D*M*N flops each)")
    return {"tflops": flops / dt / 1e12, "seconds": dt, "parts": parts, "sample": desc, "threads": threads}


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    vals, secs, parts = [], [], {}
    r = None
    for it in range(args.warmup + args.steps):
        r = oracle_sample()
        if it >= args.warmup:
            vals.append(r["tflops"])
            secs.append(r["seconds"])
            for n, x in r["parts"].items():
                parts.setdefault(n, []).append(x)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "video-dit-76800 (one-head sample, see cpu_baseline.sample)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": r["threads"], "kind": "oracle",
                             "sample": r["sample"],
                             "seconds_by_part": {n: statistics.mean(x) for n, x in parts.items()}},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ layout step

def layout_step(q, p, dev, stream, e0, e1):
    """Times the 3D tiling of the latent [1, 20, 48, 80, heads, 128] into the
    attention's token order (tile_3d) and back (untile_3d): HBM-bound copies
    that move every token row once each way."""
    import torch

    from bwd_tile_mean_gb300 import vsa

    latent = q.view(1, 20, 48, 80, p.Hq, p.D)
    tiled_buf, back_buf = torch.empty_like(q), torch.empty_like(latent)
    var_buf = torch.empty(300, dtype=torch.int32, device=dev)
    res = {}
    for name, fn in (("tile_3d", lambda: vsa.tile_3d(latent, out=tiled_buf, tile_var=var_buf, stream=stream)),
                     ("untile_3d", lambda: vsa.untile_3d(tiled_buf, (20, 48, 80), out=back_buf, stream=stream))):
        for _ in range(3):
            fn()
        reps = 10
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t_ms = e0.elapsed_time(e1) / reps
        moved = 2 * q.numel() * q.element_size()  # every token row read once and written once
        res[name] = {"ms": t_ms, "GB_per_s": moved / (t_ms * 1e-3) / 1e9, "bytes": moved}
    return res


# ------------------------------------------------------------------ ours

def workload(args):
    from bwd_tile_mean_gb300 import inputs
    p = inputs.config(args.config)
    if args.heads is not None and args.heads != p.Hq:  # smaller copy of the same workload (profiling captures)
        if p.Hq != p.Hkv:
            raise SystemExit("--heads applies to workloads with as many KV heads as query heads")
        p = dataclasses.replace(p, Hq=args.heads, Hkv=args.heads)
    return p


def head_shard(p, t, ws, rank, dev):
    """This rank's slice of the problem's heads (vsa_head_slice): the slice
    problem and its tensors, cut from the whole problem's seeded tensors."""
    from bwd_tile_mean_gb300 import inputs, vsa
    full = vsa.describe(p.layout, inputs.DTYPES[p.dtype], p.B, p.Hq, p.Hkv, p.D, p.Sq, p.Skv, p.tile_q, p.tile_kv,
                        p.nQ, p.nKV)
    sd, q0, kv0 = vsa.vsa_head_slice(full, ws, rank)
    ps = inputs.Problem(p.name, p.layout, p.B, sd.Hq, sd.Hkv, p.D, p.tile_q, p.tile_kv, p.nQ, p.nKV, dtype=p.dtype,
                        q_var=p.q_var, kv_var=p.kv_var, topk=p.topk, gate=p.gate, seed=p.seed, backward=p.backward)
    hd = 1 if p.layout == "bhsd" else 2
    ts = {n: x.narrow(hd, q0 if n in ("q", "dO", "gate") else kv0,
                      sd.Hq if n in ("q", "dO", "gate") else sd.Hkv).contiguous() for n, x in t.items()}
    return ps, ts, (q0, sd.Hq)


def l2_note(q, k):
    """How the step's inputs compare with the 126 MB L2 (no flush between steps)."""
    qb, kb = q.numel() * q.element_size(), k.numel() * k.element_size()
    if min(qb, kb) > 126e6:
        size = "each input larger than L2"
    elif 2 * (qb + kb) > 126e6:
        size = "inputs larger than L2 together, not each"
    else:
        size = "inputs fit in L2"
    return f"{size} (q, dO {qb / 1e6:.1f} MB each; k, v {kb / 1e6:.1f} MB each; L2 126 MB); no flush"


def host_link(h_in, d_in, h_out, d_out, dev, stream, e0, e1, reps=3):
    """Host<->device copy rates (GB/s) of this machine for one contiguous tensor
    from / to pinned memory: each direction alone and both at once (the
    host-buffer step moves its inputs and outputs through this link)."""
    import torch
    nb = h_in.numel() * h_in.element_size()
    side = torch.cuda.Stream(dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    def both():
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            h_out.copy_(d_out, non_blocking=True)
        d_in.copy_(h_in, non_blocking=True)
        stream.wait_stream(side)

    scratch = torch.empty_like(d_in)
    h2d = timed(lambda: scratch.copy_(h_in, non_blocking=True))
    d2h = timed(lambda: h_out.copy_(d_out, non_blocking=True))
    d_in, scratch = scratch, d_in  # both(): write the scratch copy, leave the input tensor as it is
    bi = timed(both)
    return {"h2d": round(nb / h2d / 1e6, 1), "d2h": round(nb / d2h / 1e6, 1),
            "both_each_way": round(nb / bi / 1e6, 1), "bytes_per_copy": nb}


def ours(args):
    import torch

    from bwd_tile_mean_gb300 import inputs, vsa

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shard = ws > 1 and args.shard == "heads"
    p_full = workload(args)
    t = inputs.make_tensors(p_full, device=dev)
    heads = (0, p_full.Hq)
    if shard:
        p, t, heads = head_shard(p_full, t, ws, rank, dev)
    else:
        p = p_full
    gated = p.gate is not None
    train = p.backward
    T = inputs.DTYPES[p.dtype]
    q, k, v, dO = t["q"], t["k"], t["v"], t["dO"]
    i32 = dict(dtype=torch.int32, device=dev)
    plan = vsa.Plan(p.layout, T, p.B, p.Hq, p.Hkv, p.D, p.tile_q, p.tile_kv, p.nQ, p.nKV, p.Sq, p.Skv, p.cap,
                    gate=gated, q_var=torch.as_tensor(p.q_var, **i32), kv_var=torch.as_tensor(p.kv_var, **i32),
                    scale=p.scale, device=dev)
    gate = t.get("gate")
    out = torch.empty_like(q)
    osp = torch.empty_like(q) if gated else None
    lse = torch.empty(plan.lse_shape(), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)

    def step(qq, kk, vv, dd):
        plan.build_block_map(qq, kk, p.topk, need_bwd_index=train)
        plan.forward(qq, kk, vv, gate=gate, out=out, lse=lse, o_sparse=osp)
        if train:
            plan.backward(dd, qq, kk, vv, osp if gated else out, lse, gate=gate, dq=dq, dk=dk, dv=dv)

    def barrier():
        torch.cuda.synchronize(dev)
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step(q, k, v, dO)
    barrier()
    # effective FLOPs from the selection actually made (this rank's heads)
    qc = plan.q_cnt.long()
    qidx = plan.q_idx.long().clamp(min=0)
    kvv = torch.as_tensor(p.kv_var, device=dev).long()
    valid_keys = float(torch.where(plan.q_idx >= 0, kvv[qidx], torch.zeros_like(qidx)).sum().item())
    pairs = int(qc.sum().item())
    flop_unit = 2.0 * p.D * p.tile_q  # x N x 7 per pair
    fwd_flops = flop_unit * valid_keys * 2
    step_flops = flop_unit * valid_keys * (7 if train else 2)
    # whole-job work: every rank's own heads (sharded) or copies (replicas)
    job_flops = reduce_sum(step_flops, ws, dev)
    job_pairs = int(reduce_sum(pairs, ws, dev))

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        bus = None
    sampler = ClockSampler(bus) if rank == 0 else None
    n0 = vsa.vsa_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step(q, k, v, dO)
    e1.record(stream)
    barrier()
    launches = vsa.vsa_launch_count() - n0
    ms = reduce_max(e0.elapsed_time(e1) / args.steps, ws, dev)
    clocks = sampler.stop() if sampler else None

    # per-kernel times over a second, instrumented pass of the same steps
    with vsa.profile() as prof:
        for _ in range(args.steps):
            step(q, k, v, dO)
        torch.cuda.synchronize(dev)
    per = {}
    for name, t_ms in prof.records:
        per.setdefault(name, []).append(t_ms)
    kern = {n: {"launches": len(x), "avg_ms": statistics.mean(x), "total_ms_per_step": sum(x) / args.steps}
            for n, x in per.items()}

    # end to end through the public API with host buffers (pinned), copies timed
    # (training: q, k, v, dO [, gate] in, O, dq, dk, dv out; inference: q, k, v [, gate] in, O out)
    ins = (("q", q), ("k", k), ("v", v)) + ((("dO", dO),) if train else ()) + ((("gate", gate),) if gated else ())
    outs = (("out", out),) + ((("dq", dq), ("dk", dk), ("dv", dv)) if train else ())
    # A throwaway allocation of twice their size is taken (and written)
    # first and released once the buffers exist. On a Grace host, copies
    # from the first host memory a process took right after another
    # process had released its own were measured to stall 60-250 ms in
    # about one copy in five, pinned by cudaHostAlloc or by cudaHostRegister
    # alike, while buffers allocated after it stalled in 1 of 576 calls.
    nbytes = sum(x.numel() * x.element_size() for _, x in list(ins) + list(outs))
    throwaway = torch.empty(2 * nbytes, dtype=torch.uint8, pin_memory=True)
    throwaway.fill_(0)
    host_in = {n: x.to("cpu").pin_memory() for n, x in ins}
    host_out = {n: torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for n, x in outs}
    del throwaway
    groups = max(g for g in range(1, 9) if p.Hkv % g == 0)
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in host_out.values())
    e_steps = max(2, min(args.steps, 10))

    def e2e_step():
        # the library's host-buffer step: head slices, copies overlapped with the kernels
        if train:
            plan.train_step_host(host_in["q"], host_in["k"], host_in["v"], host_in["dO"], p.topk, groups,
                                 gate=host_in.get("gate"), out=host_out["out"], dq=host_out["dq"],
                                 dk=host_out["dk"], dv=host_out["dv"], stream=stream)
        else:
            plan.fwd_step_host(host_in["q"], host_in["k"], host_in["v"], p.topk, groups, gate=host_in.get("gate"),
                               out=host_out["out"], stream=stream)

    link = host_link(host_in["q"], q, host_out["out"], out, dev, stream, e0, e1)
    for _ in range(args.warmup):
        e2e_step()
    barrier()
    # one event per call as well, so that a call stalled by the host link
    # shows up in the line (the value stays the mean over all calls)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps + 1)]
    e0.record(stream)
    marks[0].record(stream)
    for i in range(e_steps):
        e2e_step()
        marks[i + 1].record(stream)
    e1.record(stream)
    barrier()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e_steps, ws, dev)
    per_call = [marks[i].elapsed_time(marks[i + 1]) for i in range(e_steps)]
    job_h2d, job_d2h = int(reduce_sum(h2d, ws, dev)), int(reduce_sum(d2h, ws, dev))

    # the layout step on either side of the attention: 3D tiling of the
    # latent [1, 20, 48, 80, heads, 128] into the attention's token order and
    # back (HBM-bound copies; reported beside the step, not inside it)
    layout = {}
    if args.config == 3:
        layout = layout_step(q, p, dev, stream, e0, e1)

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    pk, pk_kind = peaks()
    for v_ in layout.values():
        v_["frac_of_hbm"] = v_["GB_per_s"] / pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tensor_peak = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    value = job_flops / (ms * 1e-3) / 1e12
    dominant = max(kern.items(), key=lambda kv_: kv_[1]["total_ms_per_step"]) if kern else None
    roof = None
    if dominant:
        name, info = dominant
        unit_flops = {"bwd_dkdv": 8.0, "bwd_dq": 6.0, "fwd_attn": 4.0}.get(name)
        if unit_flops is not None:
            launch_flops = 2.0 * p.D * p.tile_q * valid_keys * unit_flops / 2.0
            achieved = launch_flops / (info["avg_ms"] * 1e-3) / 1e12
            traffic, note = measured_traffic(name, p.Hq) if args.config == 3 else \
                (None, "no ncu capture of this workload")
            roof = {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": tensor_peak,
                    "unit": "TFLOP/s", "frac": achieved / tensor_peak, "traffic": traffic,
                    "traffic_unit": "bytes per launch", "traffic_source": note,
                    "peak_kind": f"bf16_tflops_sustained ({pk_kind})", "flops_per_launch": launch_flops}
    cpu = None
    if not args.no_cpu_baseline and args.config == 3:
        r = oracle_sample()
        cpu = {"value": r["tflops"], "unit": "TFLOP/s", "cores": r["threads"], "kind": "oracle",
               "sample": r["sample"], "seconds": r["seconds"], "seconds_by_part": r["parts"]}
    if args.config == 3 and not shard:
        wl = ("video-dit-76800: latent 20x48x80 tiled 4x8x8 -> 300 tiles, 76,800 tokens; "
              f"B=1, H={p.Hq}, D=128, bf16, BSHD; topk 30 (10% density)")
    else:
        wl = (f"{p_full.name}: B={p_full.B}, H={p_full.Hq}/{p_full.Hkv}, D=128, {p_full.dtype}, {p_full.layout}, "
              f"{p_full.nQ} Q x {p_full.nKV} KV tiles of {p_full.tile_q}/{p_full.tile_kv}, topk {p_full.topk}"
              + (", gated" if gated else "") + ("" if train else ", forward only"))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong" if shard else "weak", "vs_baseline": None, "dtype": p.dtype, "data": "synthetic",
        "config": {"workload": wl, "selected_pairs": job_pairs, "tflop_per_step": job_flops / 1e12,
                   "fwd_tflop_per_step": fwd_flops * (job_flops / step_flops) / 1e12,
                   "l2": l2_note(q, k),
                   "parallelism": (f"heads split over {ws} GPUs ({heads[1]} query heads each, no exchange)" if shard
                                   else f"replicas x{ws}")},
        "pct_of_peak": {"bf16_burst": value / ws / pk.get("bf16_tflops", 1900.0),
                        "bf16_sustained": value / ws / tensor_peak, "peaks": pk_kind},
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": job_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": job_h2d, "d2h_bytes_per_step": job_d2h,
                "path": f"{'vsa_train_step_host' if train else 'vsa_fwd_step_host'}: {groups} head slices, "
                        "copies overlapped with the kernels",
                "host_memory": "torch pinned (cudaHostAlloc), taken after a same-sized throwaway allocation",
                "host_link_GB_per_s": link, "calls": e_steps,
                "call_ms": {"median": round(statistics.median(per_call), 3), "min": round(min(per_call), 3),
                            "max": round(max(per_call), 3)}},
        "gpu_launches": launches, "clocks": clocks,
        "layout_step": {"bound": "hbm", "peak_GB_per_s": pk.get("hbm_gbs"), **layout},
        "kernels": {n: {"avg_ms": round(x["avg_ms"], 4), "launches_per_step": x["launches"] // args.steps,
                        "ms_per_step": round(x["total_ms_per_step"], 4)} for n, x in kern.items()},
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=None,
                    help="heads of the workload (its own count by default; fewer only for profiling captures)")
    ap.add_argument("--config", type=int, default=3, choices=[1, 3, 4, 5, 6],
                    help="workload: 3 = video DiT 76,800 tokens (the headline); 1 tiny, 4 gated ragged, "
                         "5 long-video forward only, 6 the long-video grid taken literally (1,024 tiles)")
    ap.add_argument("--shard", choices=["heads", "replicas"], default="heads",
                    help="with several GPUs: split the problem's heads over them (default) or run copies")
    ap.add_argument("--write-traffic", metavar="CSV",
                    help="write the committed per-kernel DRAM-bytes file from this ncu CSV and exit")
    ap.add_argument("--traffic-command", default="", help="the capture command, recorded with --write-traffic")
    args = ap.parse_args()
    if args.write_traffic:
        write_traffic(args.write_traffic, args.heads if args.heads is not None else 40, args.traffic_command)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
