"""Benchmark: fwd+bwd effective TFLOP/s of tile-top-k block-sparse attention
on the video-DiT workload (latent 20x48x80 tiled 4x8x8 -> 300 tiles, 76,800
tokens; B=1, 40 heads, D=128, bf16, BSHD; top-30 KV tiles per Q tile).

One step = the whole hot path on one batch: block map (pool + coarse top-k
+ both indices), forward (O, LSE) and backward (dQ, dK, dV), through the
C ABI. FLOPs are counted on selected tile pairs only:
2*D*M*N*(2 fwd + 5 bwd) per pair, M = query rows of the tile, N = valid
keys of the KV tile.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica of the workload on its own
GPU (weak scaling); timing is the max over ranks. --impl reference times
the CPU oracle on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd effective TFLOP/s (selected blocks) on 1 GB300; % of bf16 TC peak"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of each
# attention kernel, from one `ncu --set full` capture of the current kernels
# on this workload cut to 4 heads; every head is an independent problem, so
# the traffic of a launch scales with the heads. Set an entry to None when its
# kernel changes after the capture.
DRAM_BYTES_PER_4_HEADS = {
    "bwd_dkdv": 397.200128e6 + 141.905152e6,
    "bwd_dq": 406.098432e6 + 73.191424e6,
    "fwd_attn": 306.897408e6 + 67.292672e6,
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x, world_size, device):
    """Max of a per-rank float over all ranks (identity on one rank)."""
    if world_size == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
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

def oracle_sample(n_tiles=2, seed=42):
    """Time the CPU oracle (block map + forward + backward) on a bounded
    sample of the workload: one head of the same shape (300 tiles, topk 30),
    forward and dQ for the rows of n_tiles query tiles and dK/dV of n_tiles
    KV tiles. Credited with the effective FLOPs of the selected pairs of
    those query tiles. Returns (tflops, seconds, description, threads)."""
    import numpy as np
    import torch
    from bwd_tile_mean_gb300.inputs import Problem, make_tensors
    from oracle import oracle as orc

    nt = 300
    p = Problem("video-dit-1head", "bshd", 1, 1, 1, 128, 256, 256, nt, nt, q_var=[256] * nt, kv_var=[256] * nt,
                topk=30, seed=seed)
    t = make_tensors(p)
    q, k, v, dO = (orc._f64(t[n]) for n in ("q", "k", "v", "dO"))
    orc.lib()
    t0 = time.perf_counter()
    m, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    rows = np.asarray([(0, 0, i * 256 + r) for i in range(n_tiles) for r in range(256)], dtype=np.int32)
    orc.forward_rows(p, q, k, v, qi, qc, p.cap, rows=rows)
    orc.backward_dq_rows(p, dO, q, k, v, qi, qc, p.cap, rows=rows)
    tiles = np.asarray([(0, 0, j) for j in range(n_tiles)], dtype=np.int32)
    orc.backward_dkdv_tiles(p, dO, q, k, v, qi, qc, p.cap, tiles=tiles)
    dt = time.perf_counter() - t0
    pairs = int(qc[0, 0, :n_tiles].sum())
    flops = pairs * 2.0 * 128 * 256 * 256 * 7
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    desc = (f"oracle block map of one 300-tile head + forward and dQ of {n_tiles} query tiles' rows + dK/dV of "
            f"{n_tiles} KV tiles ({pairs} selected pairs credited, 14*D*M*N flops each)")
    del torch
    return flops / dt / 1e12, dt, desc, threads


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    vals, secs = [], []
    desc, threads = "", 1
    for it in range(args.warmup + args.steps):
        v, dt, desc, threads = oracle_sample(n_tiles=1)
        if it >= args.warmup:
            vals.append(v)
            secs.append(dt)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "video-dit-76800 (one-head sample, see cpu_baseline.sample)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc},
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

def ours(args):
    import torch

    from bwd_tile_mean_gb300 import inputs, vsa

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    p = inputs.config(args.config)
    if args.config == 3 and args.heads != p.Hq:  # smaller replica of the same workload (profiling captures)
        p = inputs.Problem(p.name, p.layout, p.B, args.heads, args.heads, p.D, p.tile_q, p.tile_kv, p.nQ, p.nKV,
                           q_var=p.q_var, kv_var=p.kv_var, topk=p.topk, seed=p.seed)
    gated = p.gate is not None
    train = p.backward
    T = inputs.DTYPES[p.dtype]
    t = inputs.make_tensors(p, device=dev)
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

    def max_over_ranks(x):
        return reduce_max(x, ws, dev)

    for _ in range(args.warmup):
        step(q, k, v, dO)
    barrier()
    # effective FLOPs from the selection actually made
    qc = plan.q_cnt.long()
    qidx = plan.q_idx.long().clamp(min=0)
    kvv = torch.as_tensor(p.kv_var, device=dev).long()
    valid_keys = torch.where(plan.q_idx >= 0, kvv[qidx], torch.zeros_like(qidx)).sum()
    pairs = int(qc.sum().item())
    flop_unit = 2.0 * p.D * p.tile_q  # x N x 7 per pair
    fwd_flops = flop_unit * float(valid_keys.item()) * 2
    step_flops = flop_unit * float(valid_keys.item()) * (7 if train else 2)

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
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms)
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
    host_in = {n: x.to("cpu").pin_memory() for n, x in ins}
    host_out = {n: torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for n, x in outs}
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

    e2e_step()
    barrier()
    e0.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps)

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
    value = step_flops * ws / (ms * 1e-3) / 1e12
    dominant = max(kern.items(), key=lambda kv_: kv_[1]["total_ms_per_step"]) if kern else None
    roof = None
    if dominant:
        name, info = dominant
        unit_flops = {"bwd_dkdv": 8.0, "bwd_dq": 6.0, "fwd_attn": 4.0}.get(name)
        if unit_flops is not None:
            launch_flops = 2.0 * p.D * p.tile_q * float(valid_keys.item()) * unit_flops / 2.0
            achieved = launch_flops / (info["avg_ms"] * 1e-3) / 1e12
            dram = DRAM_BYTES_PER_4_HEADS.get(name)
            traffic = dram * p.Hq / 4.0 if dram is not None else None
            roof = {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": tensor_peak,
                    "unit": "TFLOP/s", "frac": achieved / tensor_peak, "traffic": traffic,
                    "traffic_unit": "bytes per launch (ncu, 4-head capture scaled to the heads)",
                    "peak_kind": f"bf16_tflops_sustained ({pk_kind})",
                    "flops_per_launch": launch_flops}
    cpu = None
    if not args.no_cpu_baseline and args.config == 3:
        v_cpu, dt, desc, threads = oracle_sample(n_tiles=2)
        cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc,
               "seconds": dt}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": ("video-dit-76800: latent 20x48x80 tiled 4x8x8 -> 300 tiles, 76,800 tokens; "
                                f"B=1, H={p.Hq}, D=128, bf16, BSHD; topk 30 (10% density)") if args.config == 3 else
                               (f"{p.name}: B={p.B}, H={p.Hq}/{p.Hkv}, D=128, {p.dtype}, {p.layout}, "
                                f"{p.nQ} Q x {p.nKV} KV tiles of {p.tile_q}/{p.tile_kv}, topk {p.topk}"
                                + (", gated" if gated else "") + ("" if train else ", forward only")),
                   "selected_pairs": pairs, "tflop_per_step": step_flops / 1e12,
                   "fwd_tflop_per_step": fwd_flops / 1e12,
                   "l2": "inputs larger than L2 (each of q, k, v, dO is 786 MB vs 126 MB L2); no flush",
                   "parallelism": f"replicas x{ws}"},
        "pct_of_peak": {"bf16_burst": value / ws / pk.get("bf16_tflops", 1900.0),
                        "bf16_sustained": value / ws / tensor_peak, "peaks": pk_kind},
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": step_flops * ws / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": f"{'vsa_train_step_host' if train else 'vsa_fwd_step_host'}: {groups} head slices, "
                        "copies overlapped with the kernels"},
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
    ap.add_argument("--heads", type=int, default=40, help="heads of the workload (40; fewer only for profiling)")
    ap.add_argument("--config", type=int, default=3, choices=[1, 3, 4, 5],
                    help="workload: 3 = video DiT 76,800 tokens (the headline); 1 tiny, 4 gated ragged, "
                         "5 long-video forward only")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
