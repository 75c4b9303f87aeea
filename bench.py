"""Benchmark of the hash-blocked TSDF integrate path (allocate + update).

One step = integrate a whole trajectory into a freshly reset volume: reset,
then for every frame the allocate kernel and the update kernel.  The default
workload is the 300-frame 1280x720 room walk (400 primitives in an 8 m room,
voxel 4 mm, truncation 16 mm, pool 2^20 blocks, table 2^21 slots), with
inputs resident in device memory; the frames (4.4 GB) and the pool (10.7 GB)
are far larger than L2, so no flush is needed between steps.

Prints one JSON line (rank 0):
  value   = valid depth points integrated per second (all ranks),
  e2e     = the same metric through tsdf_integrate_batch_host, with the
            frames copied from pinned host memory every step and the
            counters read back,
  roofline for the update kernel (HBM bytes the algorithm must move) and the
  L2 atomic throughput it sustains,
  cpu_baseline = the CPU oracle on a bounded sample of the same workload.

--impl reference times the CPU oracle itself as the reference arm.
Multi-GPU (torchrun): every rank integrates its own copy of the workload
(weak scaling, no collective on the data path); timing is the maximum over
ranks, bracketed by barriers.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import subprocess
import sys
import time

import numpy as np

REPO = os.path.dirname(os.path.abspath(__file__))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

METRIC = "depth points integrated/sec and voxel-updates/sec (alloc+update) vs roofline"

WORKLOADS = {
    "room_walk": ("room_random_walk", {"n_frames": 300}),
    "orbit": ("orbit_trajectory", {"n_frames": 100}),
    "vga": ("vga_sphere_plane", {}),
    "tiny": ("tiny_sphere_plane", {}),
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="room_walk")
    ap.add_argument("--frames", type=int, default=0, help="override the trajectory length")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def make_frames(workload: str, n_frames: int):
    from hash_blocked_tsdf_gb300 import scenes
    fn, kw = WORKLOADS[workload]
    kw = dict(kw)
    if n_frames and "n_frames" in kw:
        kw["n_frames"] = n_frames
    return getattr(scenes, fn)(**kw)


def workload_config(frames, args) -> dict:
    return {
        "workload": frames.name,
        "frames_per_step": frames.n_frames,
        "width": frames.width,
        "height": frames.height,
        "voxel_size_m": frames.voxel_size,
        "trunc_m": frames.trunc,
        "pool_capacity": frames.pool_capacity,
        "table_capacity": frames.table_capacity or "default",
        "seed": frames.seed,
        "l2": "inputs larger than L2 (frames and pool exceed 129 MB)",
        "step": "reset + (allocate, update) per frame",
    }


# ----------------------------------------------------------------------------
# Clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.path = os.path.join(REPO, "gpurun_out", f"clocks_rank{device_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# Distributed helpers (one process per GPU under torchrun)
# ----------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if _cuda_ok() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def _cuda_ok():
    import torch
    return torch.cuda.is_available()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if _cuda_ok() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if _cuda_ok() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle arm
# ----------------------------------------------------------------------------

def oracle_sample(frames, seconds_target: float):
    """Time the oracle on the first frames of the workload until about
    `seconds_target` seconds of CPU work; returns (points/s, voxel-updates/s,
    description)."""
    import oracle
    o = oracle.OracleVolume(frames.voxel_size, frames.trunc)
    t0 = time.perf_counter()
    n = 0
    while n < frames.n_frames:
        o.integrate(frames.depth[n], frames.rgb[n], frames.K, frames.poses[n])
        n += 1
        if time.perf_counter() - t0 >= seconds_target:
            break
    dt = time.perf_counter() - t0
    c = o.counters()
    return (c["valid_points"] / dt, c["passing_samples"] / dt,
            f"first {n} of {frames.n_frames} frames of {frames.name} ({dt:.1f} s, 1 thread)")


def run_reference(args):
    rank, local, world = dist_setup()
    if rank != 0:
        return
    frames = make_frames(args.workload, args.frames)
    per_step = max(1, min(frames.n_frames, 2))
    import oracle
    oracle.build()

    def step(i):
        o = oracle.OracleVolume(frames.voxel_size, frames.trunc)
        for f in range(per_step):
            g = (i * per_step + f) % frames.n_frames
            o.integrate(frames.depth[g], frames.rgb[g], frames.K, frames.poses[g])
        return o.counters()

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    pts = 0
    for i in range(args.steps):
        pts += step(args.warmup + i)["valid_points"]
    dt = time.perf_counter() - t0
    value = pts / dt
    sample = f"{per_step} frames of {frames.name} per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "points/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(frames, args), frames_per_step=per_step),
        "cpu_baseline": {"value": value, "unit": "points/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "cpu": platform.machine()},
        "e2e": {"value": value, "unit": "points/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def _peaks():
    try:
        with open(os.path.join(REPO, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def run_ours(args):
    import torch

    rank, local, world = dist_setup()
    torch.cuda.set_device(local)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    if rank != 0:
        __graft_entry__.build()
    from hash_blocked_tsdf_gb300 import TsdfVolume, binding

    frames = make_frames(args.workload, args.frames)
    n = frames.n_frames
    stream = torch.cuda.current_stream()
    d_dev = torch.from_numpy(frames.depth).cuda()
    c_dev = torch.from_numpy(frames.rgb).cuda()
    vol = TsdfVolume(frames.pool_capacity, frames.voxel_size, frames.trunc,
                     frames.table_capacity)
    h = vol.handle
    lib = binding.load_library()
    K = np.ascontiguousarray(frames.K, dtype=np.float32)
    poses = np.ascontiguousarray(frames.poses, dtype=np.float32).reshape(n, 16)
    import ctypes
    kp = K.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
    pps = [poses[f].ctypes.data_as(ctypes.POINTER(ctypes.c_float)) for f in range(n)]
    px = frames.width * frames.height
    sptr = stream.cuda_stream
    dptr, cptr = d_dev.data_ptr(), c_dev.data_ptr()

    def one_step(events=None):
        rc = lib.tsdf_reset(h, sptr)
        assert rc == 0
        for f in range(n):
            if events is not None:
                events[2 * f].record(stream)
            rc = lib.tsdf_allocate(h, dptr + 4 * f * px, frames.width, frames.height, kp,
                                   pps[f], sptr)
            assert rc == 0, binding.load_library().tsdf_last_error()
            if events is not None:
                events[2 * f + 1].record(stream)
            rc = lib.tsdf_update(h, dptr + 4 * f * px, cptr + 12 * f * px, frames.width,
                                 frames.height, kp, pps[f], sptr)
            assert rc == 0, binding.load_library().tsdf_last_error()
        if events is not None:
            events[2 * n].record(stream)

    # warm-up, and the per-step counts from the first warm-up step
    for i in range(max(args.warmup, 1)):
        one_step()
        if i == 0:
            torch.cuda.synchronize()
            st = vol.stats()
            blocks = vol.block_count()
    points_per_step = st["valid_points"]
    updates_per_step = st["voxel_updates"]

    # census of distinct voxels per frame (untimed): the algorithmic bytes
    # of the update kernel are counted per distinct voxel it must modify
    distinct = census_distinct_voxels(torch, vol, frames, d_dev, c_dev)

    # timed region
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n + 1)]
    stage_alloc = 0.0
    stage_update = 0.0
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    per_step_events = []
    for k in range(args.steps):
        evk = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n + 1)]
        one_step(evk)
        per_step_events.append(evk)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    for evk in per_step_events:
        for f in range(n):
            stage_alloc += evk[2 * f].elapsed_time(evk[2 * f + 1])
            stage_update += evk[2 * f + 1].elapsed_time(evk[2 * f + 2] if f + 1 < n
                                                        else evk[2 * n])
    max_ms = max_over_ranks(elapsed_ms, world)
    total_points = sum_over_ranks(points_per_step * args.steps, world)
    value = total_points / (max_ms / 1000.0)
    upd_rate = sum_over_ranks(updates_per_step * args.steps, world) / (max_ms / 1000.0)

    # roofline of the update kernel
    hbm_peak, peak_kind = _peaks()
    n_update_launches = n * args.steps
    upd_ms_avg = stage_update / n_update_launches
    alloc_ms_avg = stage_alloc / n_update_launches
    bytes_per_launch = (16.0 * points_per_step + 40.0 * distinct["total"]) / n
    achieved = bytes_per_launch / (upd_ms_avg / 1000.0) / 1e9
    roofline = {
        "bound": "hbm", "kernel": "update_kernel", "achieved": achieved, "peak": hbm_peak,
        "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": None,
        "peak_source": f"{peak_kind} hbm_gbs", "bytes_per_launch_alg": bytes_per_launch,
        "avg_launch_ms": upd_ms_avg,
        "atomics": {
            "issued_per_launch": 5.0 * updates_per_step / n,
            "algorithmic_per_launch": 5.0 * distinct["total"] / n,
            "achieved_issued_per_s": 5.0 * updates_per_step / n / (upd_ms_avg / 1000.0),
        },
    }
    result = {
        "metric": METRIC, "value": value, "unit": "points/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": dict(workload_config(frames, args), parallelism=f"replicas{world}"),
        "voxel_updates_per_s": upd_rate,
        "stages_ms_per_frame": {"allocate": alloc_ms_avg, "update": upd_ms_avg},
        "blocks": blocks, "points_per_step": points_per_step,
        "voxel_updates_per_step": updates_per_step,
        "distinct_voxels_per_step": distinct["total"],
        "clocks": clk,
        "gpu_launches": args.steps * (1 + 2 * n),
        "roofline": roofline,
    }

    if not args.no_e2e:
        result["e2e"] = e2e_host(torch, vol, frames, args)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, u, sample = oracle_sample(frames, args.cpu_baseline_seconds)
        result["cpu_baseline"] = {"value": v, "unit": "points/s", "cores": 1, "kind": "oracle",
                                  "sample": sample, "voxel_updates_per_s": u,
                                  "cpu": platform.machine()}
    vol.close()
    if rank == 0:
        print(json.dumps(result), flush=True)


def census_distinct_voxels(torch, vol, frames, d_dev, c_dev) -> dict:
    """Distinct voxels the update kernel modifies in each frame, counted by
    comparing the weight array before and after each frame."""
    from hash_blocked_tsdf_gb300 import binding
    vol.reset()
    ptrs = binding.tsdf_pool_arrays(vol.handle)
    cap = vol.info["pool_capacity"]
    weight = _as_tensor(torch, ptrs["weight"], cap * 512)
    prev = torch.empty_like(weight)
    per_frame = []
    for f in range(frames.n_frames):
        used = vol.block_count() * 512
        prev[:used].copy_(weight[:used])
        vol.integrate(d_dev[f], c_dev[f], frames.K, frames.poses[f])
        used = vol.block_count() * 512
        per_frame.append(int((weight[:used] != prev[:used]).sum().item()))
    vol.reset()
    torch.cuda.synchronize()
    return {"total": int(sum(per_frame)), "per_frame_mean": float(np.mean(per_frame))}


def _as_tensor(torch, ptr: int, n: int):
    class _Arr:
        __cuda_array_interface__ = {"shape": (n,), "typestr": "<f4", "data": (ptr, False),
                                    "version": 3, "strides": None}
    return torch.as_tensor(_Arr(), device="cuda")


def e2e_host(torch, vol, frames, args) -> dict:
    """Same metric through tsdf_integrate_batch_host: frames copied from
    pinned host memory inside the timed region, counters read back."""
    d_host = torch.from_numpy(frames.depth).pin_memory()
    c_host = torch.from_numpy(frames.rgb).pin_memory()
    stream = torch.cuda.current_stream()
    for _ in range(max(1, args.warmup)):
        vol.reset()
        vol.integrate_batch_host(d_host, c_host, frames.K, frames.poses)
        st = vol.stats()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    pts = 0
    for _ in range(args.steps):
        vol.reset()
        vol.integrate_batch_host(d_host, c_host, frames.K, frames.poses)
        st = vol.stats()                     # device -> host read of the step's result
        pts += st["valid_points"]
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    from hash_blocked_tsdf_gb300 import binding
    return {"value": pts / (ms / 1000.0), "unit": "points/s",
            "h2d_bytes_per_step": int(frames.depth.nbytes + frames.rgb.nbytes),
            "d2h_bytes_per_step": int(__import__("ctypes").sizeof(binding.tsdf_stats)),
            "ms_per_step": ms / args.steps}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
