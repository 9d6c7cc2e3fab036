"""Benchmark of the sparse-convolution hot path on one or more GPUs.

One step = one pass of the submanifold path over the LiDAR-like scene (batch 2,
41 x 1600 x 1408 grid, 120,000 voxels, fp16 features 16 -> 16):
  spc_build_indice_map (validate + key + hash build + probe of all 27 offsets),
  then spc_conv_fwd over the map.
The headline value is conv TFLOP/s over active pairs (2 * P * Cin * Cout per
step) divided by the whole step time; the indice-map rate (Mvoxel/s) and the
conv-only rate are reported beside it.  Inputs are resident in HBM when the
timed region starts; L2 is flushed (256 MiB write) between timed steps,
outside the timed events.  `e2e` times the same step through the C ABI from
pinned host buffers, host->device copies of the inputs and the device->host
copy of the output inside the timed region.

--impl reference runs the CPU oracle (the slow fp64 restatement of the method
used by the tests) on the host cores, on a bounded sample of the same workload.

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica of
the workload (voxels of different scenes never interact, so the path shards by
scene with no data exchange); value = work of all ranks / max time over ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import scenes  # noqa: E402

METRIC = "SubM3d conv TFLOP/s over active pairs (and % roofline); indice-map Mvoxel/s"
WORKLOAD = "lidar_subm_f16"
SHAPE = (41, 1600, 1408)
BATCH = 2
L2_FLUSH_BYTES = 256 << 20
# kernels of ours per step: build = hash clear + insert + probe; fwd = 1
LAUNCHES_PER_STEP = 4


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = max(smax, float(parts[2]))
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        except OSError:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def reduce_max(v: float, dist, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def algorithmic_bytes(n, K, cin, cout, s, pairs):
    build = 16 * n + 4 * K * n + 4 * n + 4 * K
    fwd = s * n * cin + s * n * cout + s * K * cin * cout + 4 * pairs
    return build, fwd


def run_ours(args, rank, world, local, dist):
    import sparse_convolution_hash_gb300 as spc
    from sparse_convolution_hash_gb300 import binding

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = scenes.workload(WORKLOAD)
    coords_h = torch.from_numpy(w["coords"])
    n = coords_h.shape[0]
    cin, cout, K = w["cin"], w["cout"], 27
    coords = coords_h.to(dev)
    x = w["x"].to(dev)
    wt = w["w"].to(dev)
    ws = torch.empty(max(binding.spc_indice_map_workspace_size(n), 256), dtype=torch.uint8,
                     device=dev)
    status = binding.new_status(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    m = spc.spc_build_indice_map(coords, BATCH, SHAPE, ksize=3, subm=True, status=status, ws=ws)
    y = spc.spc_conv_fwd(x, wt, None, m["imap"], m["mask"])
    torch.cuda.synchronize()
    binding.check_status(status, "bench build")
    pairs = int(m["pair_count"].sum().item())

    def build():
        spc.spc_build_indice_map(coords, BATCH, SHAPE, ksize=3, subm=True, out=m)

    def fwd():
        spc.spc_conv_fwd(x, wt, None, m["imap"], m["mask"], out=y)

    # The step's launches are captured once as CUDA graphs (the C ABI allocates
    # nothing and only enqueues on the current stream), so the timed replays
    # measure GPU work, not the host's Python and ctypes overhead.
    g_build, g_fwd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_build):
        build()
    with torch.cuda.graph(g_fwd):
        fwd()
    for _ in range(args.warmup):
        g_build.replay()
        g_fwd.replay()
    torch.cuda.synchronize()
    binding.check_status(status, "bench warmup")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        # keep the device busy while the host enqueues all steps, so that no
        # host gap falls inside a timed step
        torch.cuda._sleep(int(4e6) * args.steps // 10 + int(2e6))
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            g_build.replay()
            ev[i][1].record(stream)
            g_fwd.replay()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
    barrier(dist)
    binding.check_status(status, "bench timed")
    build_ms = [e[0].elapsed_time(e[1]) for e in ev]
    fwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    total_ms = sum(b + f for b, f in zip(build_ms, fwd_ms))
    total_ms = reduce_max(total_ms, dist, dev)
    ms_step = total_ms / args.steps
    flops = 2.0 * pairs * cin * cout
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12

    # end to end through the C ABI from pinned host buffers
    coords_p = coords_h.pin_memory()
    x_p = w["x"].pin_memory()
    w_p = w["w"].pin_memory()
    y_p = torch.empty((n, cout), dtype=x.dtype).pin_memory()
    e2e_steps = max(1, min(args.steps, 20))
    c_d, x_d, w_d = torch.empty_like(coords), torch.empty_like(x), torch.empty_like(wt)
    y_d = torch.empty_like(y)

    def e2e_step():
        # the calls a user makes: copy in, build the map, convolve, copy out
        c_d.copy_(coords_p, non_blocking=True)
        x_d.copy_(x_p, non_blocking=True)
        w_d.copy_(w_p, non_blocking=True)
        spc.spc_build_indice_map(c_d, BATCH, SHAPE, ksize=3, subm=True, out=m)
        spc.spc_conv_fwd(x_d, w_d, None, m["imap"], m["mask"], out=y_d)
        y_p.copy_(y_d, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), dist, dev) / e2e_steps
    h2d = coords_h.numel() * 4 + w["x"].numel() * w["x"].element_size() + w["w"].numel() * w["w"].element_size()
    d2h = n * cout * x.element_size()

    hbm, bf16_tf, peak_src = peaks()
    s = x.element_size()
    b_build, b_fwd = algorithmic_bytes(n, K, cin, cout, s, pairs)
    build_avg = sum(build_ms) / len(build_ms)
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    if build_avg >= fwd_avg:
        dom, dom_bytes, dom_ms = "spc_build_indice_map (hash clear + insert + probe)", b_build, build_avg
    else:
        dom, dom_bytes, dom_ms = "spc_conv_fwd", b_fwd, fwd_avg
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    clocks = clk.summary()

    line = {
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded LiDAR-like scene, random-init weights)",
        "config": {
            "workload": "lidar_subm_f16: SubMConv3d k3 indice build + forward, batch 2, "
                        "41x1600x1408 grid, 120000 voxels, fp16 16->16, no bias",
            "n_voxels": n, "pairs": pairs, "cin": cin, "cout": cout, "K": K,
            "l2": "flushed between timed steps (256 MiB write, outside the events)",
            "parallelism": f"replicas x{world}",
        },
        "indice_map_mvoxel_s": round(world * n / (build_avg * 1e-3) / 1e6, 2),
        "conv_fwd_tflops": round(world * flops / (fwd_avg * 1e-3) / 1e12, 4),
        "build_ms": round(build_avg, 5),
        "fwd_ms": round(fwd_avg, 5),
        "roofline": {
            "kernel": dom,
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": hbm,
            "unit": "GB/s",
            "frac": round(achieved / hbm, 4),
            "traffic": None,
            "peak_source": f"{peak_src} hbm_gbs (burst copy)",
            "alg_bytes_per_launch": dom_bytes,
        },
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, pairs, budget_s=args.cpu_seconds)
    return line


def cpu_baseline(w, pairs, budget_s=10.0):
    """The oracle as it stands, timed on the host: whole-workload steps until the budget."""
    import oracle

    oracle.build()
    coords = w["coords"]
    x64, w64 = oracle.f64(w["x"]), oracle.f64(w["w"])
    flops = 2.0 * pairs * w["cin"] * w["cout"]
    reps, t0 = 0, time.perf_counter()
    while True:
        imap, _ = oracle.subm_map(coords, BATCH, SHAPE, 3)
        oracle.conv_fwd(x64, w64, None, imap)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(reps * flops / dt / 1e12, 8), "unit": "TFLOP/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{reps} whole steps (indice map + fp64 forward over all {coords.shape[0]} "
                      f"voxels) in {dt:.1f} s, single thread",
            "ms_per_step": round(1e3 * dt / reps, 2)}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = scenes.workload(WORKLOAD)
    import oracle

    oracle.build()
    coords = w["coords"]
    x64, w64 = oracle.f64(w["x"]), oracle.f64(w["w"])
    imap, cnt = oracle.subm_map(coords, BATCH, SHAPE, 3)
    pairs = int(cnt.sum())
    flops = 2.0 * pairs * w["cin"] * w["cout"]
    for _ in range(args.warmup):
        pass  # the oracle has no warm state; warm-up steps would only repeat the work
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        imap, _ = oracle.subm_map(coords, BATCH, SHAPE, 3)
        oracle.conv_fwd(x64, w64, None, imap)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = args.steps * flops / tot / 1e12
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 8), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded LiDAR-like scene, random-init weights)",
        "config": {"workload": "lidar_subm_f16: SubMConv3d k3 indice build + forward, batch 2, "
                               "41x1600x1408 grid, 120000 voxels, fp16 16->16, no bias",
                   "n_voxels": int(coords.shape[0]), "pairs": pairs},
        "cpu_baseline": {"value": round(value, 8), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} whole steps, single thread"},
        "e2e": {"value": round(value, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local, dist = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        import __graft_entry__

        if rank == 0:
            __graft_entry__.build()
        barrier(dist)
        __graft_entry__.build()
        line = run_ours(args, rank, world, local, dist)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
