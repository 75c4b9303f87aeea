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
import tempfile
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
    # the orbit seen through 4 cm voxels: nearly every pixel sees a voxel edge
    # 5+ pixels wide, so many samples share a voxel (the dense regime)
    "orbit_coarse": ("orbit_trajectory", {"n_frames": 100, "voxel_size": 0.04, "trunc": 0.16,
                                          "pool_capacity": 1 << 16}),
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="room_walk")
    ap.add_argument("--frames", type=int, default=0, help="override the trajectory length")
    ap.add_argument("--group", type=int, default=0,
                    help="frames per batch call (default: the library's frames per launch)")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=15.0)
    ap.add_argument("--clock-log", default="",
                    help="also write the nvidia-smi clock samples of the timed region here")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gate", choices=["full", "sample"], default="full",
                    help="what the parity gate compares with the oracle: the whole trajectory "
                         "(default; the oracle in parallel on the host cores) or its first "
                         "frames only (quick runs, profiling)")
    ap.add_argument("--sweep", action="store_true",
                    help="run the measurement matrix (one JSON line per cell) instead of the "
                         "headline workload")
    ap.add_argument("--probe-report", action="store_true",
                    help="print the probe-depth histogram at table occupancy 0.1 .. 0.5 "
                         "(untimed) instead of the headline workload")
    ap.add_argument("--probe-atomics", action="store_true",
                    help="print the shared-memory atomic and 32-byte record reduction rates "
                         "(untimed by the driver) instead of the headline workload")
    ap.add_argument("--pool", type=int, default=0,
                    help="override the workload's pool capacity in blocks (small profiling runs)")
    ap.add_argument("--update-kernel",
                    choices=["auto", "adaptive", "per_sample", "pre_reduced", "fused"],
                    default="auto",
                    help="how the library's update reaches the pool (auto, the library's "
                         "default, times like per_sample here: the stages are timed as "
                         "separate calls)")
    ap.add_argument("--layout", choices=["interleaved", "planar"], default="interleaved",
                    help="pool layout: tsdf, weight, r, g interleaved per voxel (default) or "
                         "five separate arrays")
    ap.add_argument("--occlusion", choices=["ray", "reproject"], default="ray",
                    help="occlusion test: the ray pixel's depth (default) or the depth where "
                         "the voxel centre projects")
    return ap.parse_args()


def make_frames(workload: str, n_frames: int, pool: int = 0):
    import dataclasses
    from hash_blocked_tsdf_gb300 import scenes
    fn, kw = WORKLOADS[workload]
    kw = dict(kw)
    if n_frames and "n_frames" in kw:
        kw["n_frames"] = n_frames
    frames = getattr(scenes, fn)(**kw)
    if "voxel_size" in kw:
        frames = dataclasses.replace(frames, name=f"{frames.name}_voxel{round(kw['voxel_size'] * 1000)}mm")
    if pool:
        frames = dataclasses.replace(frames, pool_capacity=pool)
    return frames


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
        "l2": _l2_note(frames),
        "step": "reset + (allocate, update) per group of frames",
    }


def _l2_note(frames) -> str:
    step_bytes = frames.depth.nbytes + frames.rgb.nbytes + 20 * 512 * frames.pool_capacity
    if frames.depth.nbytes + frames.rgb.nbytes > (129 << 20):
        return (f"inputs larger than L2: {frames.depth.nbytes + frames.rgb.nbytes >> 20} MB of "
                f"frames per step, {20 * 512 * frames.pool_capacity >> 20} MB pool; no flush")
    return (f"not flushed: step inputs {step_bytes >> 20} MB (frames + pool) may stay in the "
            f"129 MB L2 between steps")


# ----------------------------------------------------------------------------
# Clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "temperature.gpu")

    def __init__(self, device_index: int, keep_path: str = ""):
        self.device_index = device_index
        self.keep_path = keep_path
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"tsdf_bench_clocks_{device_index}_",
                                         suffix=".csv")
        os.close(fd)

    def start(self):
        try:
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
        sm, smax, temp, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            lines = fh.readlines()
        if self.keep_path:
            with open(self.keep_path, "w") as fh:
                fh.writelines(lines)
        os.remove(self.path)
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            try:
                temp.append(float(parts[9]))
            except (ValueError, IndexError):
                pass
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        out = {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
               "reasons": sorted(reasons), "samples": len(sm)}
        if temp:
            out["temp_c_median"] = float(np.median(temp))
            out["temp_c_max"] = float(max(temp))
        return out


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

def oracle_sample(frames, seconds_target: float, min_frames: int = 1, occlusion: str = "ray"):
    """Time the oracle on the first frames of the workload until about
    `seconds_target` seconds of CPU work (at least `min_frames` frames);
    returns (points/s, voxel-updates/s, description, the oracle volume,
    frames integrated)."""
    import oracle
    o = oracle.OracleVolume(frames.voxel_size, frames.trunc)
    o.set_occlusion(occlusion)
    t0 = time.perf_counter()
    n = 0
    while n < frames.n_frames:
        o.integrate(frames.depth[n], frames.rgb[n], frames.K, frames.poses[n])
        n += 1
        if n >= min_frames and time.perf_counter() - t0 >= seconds_target:
            break
    dt = time.perf_counter() - t0
    c = o.counters()
    return (c["valid_points"] / dt, c["passing_samples"] / dt,
            f"first {n} of {frames.n_frames} frames of {frames.name} ({dt:.1f} s, 1 thread)",
            o, n)


def gate_reference(frames, scope: str, occlusion: str, sampled=None):
    """The oracle's volume the gate compares with: the whole trajectory the
    steps integrate (scope "full": the oracle run in parallel on the host
    cores, frames cut into chunks and blocks into partitions), or the first
    frames only (scope "sample": the CPU-baseline sample's volume when there
    is one, else two frames).  Returns (frames covered, export, counters,
    description)."""
    t0 = time.perf_counter()
    if scope == "full":
        from oracle.parallel import full_volume_oracle, worker_count
        o, oc = full_volume_oracle(frames, occlusion=occlusion)
        n = frames.n_frames
        how = (f"whole trajectory: all {n} frames, oracle in {worker_count()} processes "
               f"({time.perf_counter() - t0:.0f} s)")
        return n, o, oc, how
    if sampled is None:
        _, _, _, ovol, n = oracle_sample(frames, 0.0, min_frames=min(2, frames.n_frames),
                                         occlusion=occlusion)
    else:
        ovol, n = sampled
    how = f"first {n} of {frames.n_frames} frames (oracle sample)"
    return n, ovol.export(), ovol.counters(), how


def compare_volumes(g: dict, st: dict, o: dict, oc: dict) -> dict:
    """The GPU export `g` and statistics `st` against the oracle's export `o`
    (coords sorted) and counters `oc`: exact block set, weights and counters;
    sums within the stated bound max(1e-5 |x|, 1e-6), widened by the float32
    summation bound gamma(w - 1) sum |t| where a voxel's terms cancel.
    Reports, per sum, how many voxels needed the widening and the worst error
    against each bound."""
    out = {"blocks": int(len(o["coords"])), "voxels": int(len(o["coords"])) * 512}
    order = np.lexsort((g["coords"][:, 2], g["coords"][:, 1], g["coords"][:, 0]))
    out["block_set_equal"] = bool(g["coords"].shape == o["coords"].shape and
                                  np.array_equal(g["coords"][order], o["coords"]))
    out["weights_equal"] = bool(out["block_set_equal"] and
                                np.array_equal(g["weight"][order], o["weight"]))
    out["counters_equal"] = bool(st["valid_points"] == oc["valid_points"] and
                                 st["voxel_updates"] == oc["accumulated"] and
                                 st["missed_contributions"] == oc["missed_contributions"] and
                                 st["out_of_range_samples"] == oc["out_of_range_samples"] and
                                 st["pool_exhausted"] == 0 and st["probe_overflow"] == 0)
    worst = float("inf")
    sums = {}
    if out["weights_equal"]:
        u = 2.0 ** -24
        m = np.maximum(o["weight"] - 1.0, 0.0)
        gamma = m * u / (1.0 - m * u)
        worst = 0.0
        for k, absum in (("tsdf", o["tsdf_abs"]), ("r", None), ("g", None), ("b", None)):
            x = o[k]
            err = np.abs(g[k][order].astype(np.float64) - x)
            stated = np.maximum(1e-5 * np.abs(x), 1e-6)
            widened = np.maximum(stated, gamma * (np.abs(x) if absum is None else absum))
            over = err > stated
            sums[k] = {"voxels_over_stated_bound": int(over.sum()),
                       "worst_error_over_stated_bound": float(np.max(err / stated)),
                       "worst_error_over_widened_bound": float(np.max(err / widened))}
            worst = max(worst, sums[k]["worst_error_over_widened_bound"])
    out["sums"] = sums
    out["sums_worst_error_over_bound"] = worst
    out["pass"] = bool(out["weights_equal"] and out["counters_equal"] and worst <= 1.0)
    return out


def parity_gate(torch, vol, frames, d_dev, c_dev, scope: str, occlusion: str,
                sampled=None) -> dict:
    """The frames the oracle integrated (by default the whole trajectory one
    timed step integrates), integrated again on the GPU into a fresh volume
    with the bench's settings, and compared with the oracle's volume.  The
    headline is withheld when this check fails."""
    n, o, oc, how = gate_reference(frames, scope, occlusion, sampled)
    vol.reset()
    vol.integrate_batch(d_dev[:n], c_dev[:n], frames.K, frames.poses[:n])
    torch.cuda.synchronize()
    st = vol.stats()
    g = vol.export_blocks()
    out = {"scope": scope, "frames": n, "oracle": how}
    out.update(compare_volumes(g, st, o, oc))
    return out


def apply_gate(result: dict, gate: dict) -> None:
    """Record the parity gate in the bench line; when it failed, withhold
    the headline and end-to-end values (kept under "withheld" for the
    record), as a measurement cell whose check failed is discarded."""
    result["parity_gate"] = gate
    result["gated"] = bool(gate["pass"])
    if gate["pass"]:
        return
    result["withheld"] = {"value": result.get("value"),
                          "e2e_value": (result.get("e2e") or {}).get("value"),
                          "reason": "the GPU volume did not match the oracle on the "
                                    "parity-gate frames"}
    result["value"] = None
    if result.get("e2e"):
        result["e2e"]["value"] = None


def measure_extraction(torch, vol, blocks: int, hbm_peak: float) -> dict:
    """Marching tetrahedra over the volume as the timed steps left it (the
    whole trajectory): device time of tsdf_extract_triangles (block
    coordinates, the kernel, the count) and, separately, the copy of the
    triangles to pinned host memory.  Algorithmic bytes: each block's tsdf
    and weight arrays read once (8 B x 512) plus 36 B per triangle written."""
    import ctypes
    from hash_blocked_tsdf_gb300 import binding
    lib = binding.load_library()
    stream = torch.cuda.current_stream()
    n = ctypes.c_uint64()
    rc = lib.tsdf_extract_triangles(vol.handle, stream.cuda_stream, None, 0, ctypes.byref(n))
    assert rc == 0, lib.tsdf_last_error()
    n_tris = int(n.value)
    buf = torch.empty((max(n_tris, 1), 3, 3), dtype=torch.float32, device="cuda")
    best = None
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        rc = lib.tsdf_extract_triangles(vol.handle, stream.cuda_stream, buf.data_ptr(), n_tris,
                                        ctypes.byref(n))
        b.record(stream)
        assert rc == 0, lib.tsdf_last_error()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    host = torch.empty(buf.shape, dtype=torch.float32, pin_memory=True)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    host.copy_(buf, non_blocking=True)
    b.record(stream)
    torch.cuda.synchronize()
    d2h = a.elapsed_time(b)
    alg = 8.0 * 512 * blocks + 36.0 * n_tris
    return {"triangles": n_tris, "blocks": blocks, "ms_device": best, "ms_d2h": d2h,
            "d2h_bytes": 36 * n_tris,
            "roofline": {"bound": "hbm", "achieved": alg / (best / 1e3) / 1e9, "peak": hbm_peak,
                         "unit": "GB/s", "frac": alg / (best / 1e3) / 1e9 / hbm_peak,
                         "bytes_alg": alg}}


# ----------------------------------------------------------------------------
# Measurement matrix (the pages time every arm over a matrix of cells, not one
# scene: point count at fixed geometry, extent at fixed angular resolution,
# hash load factor, scene shape; per stage p50/p95/p99 with the count, clocks
# and temperature per cell, and a cell counts only if its block count equals
# the reference's: every cell's parity with the oracle is asserted by
# tests/test_gpu_sweep.py on the same cell definitions)
# ----------------------------------------------------------------------------

def _sweep_cell_specs():
    """(axis, name, build) for every cell; build() renders its frames."""
    from hash_blocked_tsdf_gb300 import scenes

    def sp(name, W, H, fx, scale=1.0, voxel=0.01, table=0, pool=1 << 16):
        def build():
            d, c, pose, K = scenes.sphere_plane(
                W, H, fx, fx, noise_sigma=0.002, invalid_frac=0.1, seed=7,
                sphere_centre=(0.0, 0.0, 1.5 * scale), sphere_radius=0.5 * scale,
                plane_z=2.5 * scale)
            return scenes.Frames(name, d[None], c[None], pose[None], K, voxel, 4 * voxel, pool,
                                 table, 7)
        return name, build

    specs = []
    for W, H, fx in ((160, 120, 131.25), (320, 240, 262.5), (640, 480, 525.0),
                     (1280, 960, 1050.0), (2560, 1920, 2100.0)):
        specs.append(("points_at_fixed_geometry",) + sp(f"sphere_plane_{W}x{H}", W, H, fx))
    for sc in (0.5, 1.0, 2.0, 4.0):
        specs.append(("extent_at_fixed_angular_resolution",) +
                     sp(f"sphere_plane_640x480_scale{sc}", 640, 480, 525.0, scale=sc,
                        pool=1 << 17))
    # the scale-2 scene holds 6,854 blocks: tables of 2^14 .. 2^17 slots give
    # load factors 0.42 .. 0.05 (the pool, half the table, still holds them)
    for t in (1 << 14, 1 << 15, 1 << 16, 1 << 17):
        specs.append(("hash_load_factor",) +
                     sp(f"sphere_plane_640x480_scale2_table{t}", 640, 480, 525.0, scale=2.0,
                        table=t, pool=t // 2))
    specs.append(("scene_shape", "tiny_sphere_plane_160x120", scenes.tiny_sphere_plane))
    specs.append(("scene_shape", "vga_sphere_plane_640x480", scenes.vga_sphere_plane))
    specs.append(("scene_shape", "orbit_100x640x480[0:8]",
                  lambda: scenes.orbit_trajectory(n_frames=100, frames=(0, 8))))
    specs.append(("scene_shape", "room_walk_300x1280x720[0:8]",
                  lambda: scenes.room_random_walk(n_frames=300, frames=(0, 8))))
    return specs


def _sweep_cells():
    return [(axis, build()) for axis, _, build in _sweep_cell_specs()]


def run_sweep(args):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from hash_blocked_tsdf_gb300 import TsdfVolume
    dev = torch.cuda.current_device()
    stream = torch.cuda.current_stream()
    reps = 30
    for axis, fr in _sweep_cells():
        d = torch.from_numpy(fr.depth).cuda()
        c = torch.from_numpy(fr.rgb).cuda()
        vol = TsdfVolume(fr.pool_capacity, fr.voxel_size, fr.trunc, fr.table_capacity)
        clocks = ClockSampler(dev)
        clocks.start()
        times = {"allocate": [], "update": [], "fused": [], "auto": []}
        for r in range(reps + 3):
            for mode in ("per_sample", "fused", "auto"):
                vol.set_update_kernel(mode)
                vol.reset()
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                ev[0].record(stream)
                if mode in ("fused", "auto"):
                    vol.integrate_batch(d, c, fr.K, fr.poses)
                    ev[1].record(stream)
                else:
                    vol.allocate_batch(d, fr.K, fr.poses)
                    ev[1].record(stream)
                    vol.update_batch(d, c, fr.K, fr.poses)
                ev[2].record(stream)
                torch.cuda.synchronize()
                if r >= 3:
                    if mode in ("fused", "auto"):
                        times[mode].append(ev[0].elapsed_time(ev[1]))
                    else:
                        times["allocate"].append(ev[0].elapsed_time(ev[1]))
                        times["update"].append(ev[1].elapsed_time(ev[2]))
        clk = clocks.stop()
        st = vol.stats()
        blocks = vol.block_count()
        table = vol.info["table_capacity"]
        vol.close()
        total = [a + u for a, u in zip(times["allocate"], times["update"])]
        pts = st["valid_points"]
        print(json.dumps({
            "sweep": axis, "cell": fr.name, "frames": fr.n_frames,
            "points": pts, "voxel_updates": st["voxel_updates"], "blocks": blocks,
            "table_capacity": table, "load_factor": blocks / table,
            "pool_exhausted": st["pool_exhausted"], "probe_overflow": st["probe_overflow"],
            "parity": "tests/test_gpu_sweep.py (same cells)",
            "allocate_ms": _percentiles(times["allocate"]),
            "update_ms": _percentiles(times["update"]),
            "allocate_update_ms": _percentiles(total),
            "fused_ms": _percentiles(times["fused"]),
            "points_per_s": pts / (float(np.median(total)) / 1e3),
            "points_per_s_fused": pts / (float(np.median(times["fused"])) / 1e3),
            "points_per_s_integrate_default": pts / (float(np.median(times["auto"])) / 1e3),
            "integrate_default_ms": _percentiles(times["auto"]),
            "clocks": clk}), flush=True)
    for rec in probe_depth_report(torch):
        print(json.dumps({"sweep": "probe_depth", **rec}), flush=True)


def probe_depth_report(torch, targets=(0.1, 0.2, 0.3, 0.4, 0.5), n_frames: int = 100):
    """Probe depth against table occupancy (the load-factor configuration:
    the orbit scene into fixed tables).  For each target occupancy the orbit
    is integrated frame by frame into a fixed table (2^17 slots below 0.25,
    2^16 above) until the block count reaches it; 0.5, beyond what the
    orbit allocates in 2^16 slots, is reached by topping the table up with
    blocks far from the scene through the same insert path.  Then every
    stored key is looked up again through the insert path with the probe
    instrumentation on: each probe is a successful search, and its length is
    the key's displacement + 1.  Reports the probe-length histogram, mean and
    maximum beside Knuth's expected successful-search cost for random keys,
    (1 + 1 / (1 - alpha)) / 2 (TAOCP vol. 3, 6.4), and the counters that
    show nothing was dropped.  Untimed."""
    from hash_blocked_tsdf_gb300 import TsdfVolume, scenes
    frames = scenes.orbit_trajectory(n_frames=n_frames)
    d = torch.from_numpy(frames.depth).cuda()
    c = torch.from_numpy(frames.rgb).cuda()
    out = []
    for target in targets:
        T = 1 << 17 if target < 0.25 else 1 << 16
        vol = TsdfVolume(T // 2, frames.voxel_size, frames.trunc, T)
        vol.set_update_kernel("per_sample")     # the allocate and update kernels
        f = 0
        while f < frames.n_frames and vol.block_count() < target * T:
            vol.integrate(d[f], c[f], frames.K, frames.poses[f])
            f += 1
        B = vol.block_count()
        topped = 0
        if B < target * T:
            want = int(round(target * T)) - B
            g = np.stack(np.meshgrid(np.arange(1000, 1064), np.arange(0, 64),
                                     np.arange(0, 64), indexing="ij"), -1).reshape(-1, 3)[:want]
            vol.allocate_blocks(torch.from_numpy(np.ascontiguousarray(g, np.int32)).cuda())
            topped = int(g.shape[0])
            B = vol.block_count()
        st_build = vol.stats()
        coords = vol.export_blocks(fields=("coords",))["coords"]
        vol.clear_stats()
        vol.set_instrumentation(True)
        vol.allocate_blocks(torch.from_numpy(np.ascontiguousarray(coords)).cuda())
        torch.cuda.synchronize()
        st = vol.stats()
        vol.close()
        alpha = B / T
        hist = [int(x) for x in st["probe_hist"]]
        while len(hist) > 1 and hist[-1] == 0:
            hist.pop()
        out.append({
            "target_occupancy": target, "table_capacity": T, "frames_integrated": f,
            "blocks_from_far_topping": topped, "blocks": B, "occupancy": alpha,
            "probes": st["probe_inserts"], "probe_mean": st["probe_steps"] / max(1, st["probe_inserts"]),
            "probe_max": st["probe_max"],
            "knuth_successful_search_mean": 0.5 * (1.0 + 1.0 / (1.0 - alpha)),
            "probe_hist_len1_up": hist,
            "pool_exhausted": st_build["pool_exhausted"], "probe_overflow": st_build["probe_overflow"],
            "blocks_added_by_the_lookup_pass": st["blocks_allocated"] - B,
        })
    return out


def _percentiles(xs) -> dict:
    a = np.asarray(xs, dtype=np.float64)
    return {"p50": float(np.percentile(a, 50)), "p95": float(np.percentile(a, 95)),
            "p99": float(np.percentile(a, 99)), "n": int(a.size)}


def _update_kernels(args, frames, n_frames: int) -> int:
    """Kernels one update launch runs: the adaptive mode runs the per-sample
    and the pre-reducing kernel when the launch holds 2^18 pixels or more;
    the fused mode runs one kernel for both stages (counted here, with the
    allocate counted as none); the others one."""
    if getattr(args, "occlusion", "ray") == "reproject":
        return 1                 # per-sample update, allocate and update as two kernels
    if args.update_kernel == "fused":
        return 0
    if args.update_kernel == "adaptive" and frames.width * frames.height * n_frames >= 1 << 18:
        return 2
    return 1


def other_processes_mib(device_index: int):
    """Device memory held by other processes, from nvidia-smi (None if it
    cannot tell)."""
    try:
        out = subprocess.run(["nvidia-smi", f"--id={device_index}",
                              "--query-compute-apps=pid,used_memory",
                              "--format=csv,noheader,nounits"],
                             capture_output=True, text=True, timeout=20).stdout
    except (OSError, subprocess.TimeoutExpired):
        return None
    total = 0
    for line in out.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) == 2 and parts[0].isdigit() and int(parts[0]) != os.getpid():
            try:
                total += int(parts[1])
            except ValueError:
                pass
    return total


def run_reference(args):
    rank, local, world = dist_setup()
    if rank != 0:
        return
    frames = make_frames(args.workload, args.frames, args.pool)
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
        "config": dict(workload_config(frames, args), frames_per_step=per_step,
                       l2="not applicable: the oracle runs on the host CPU"),
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

    frames = make_frames(args.workload, args.frames, args.pool)
    n = frames.n_frames
    stream = torch.cuda.current_stream()
    d_dev = torch.from_numpy(frames.depth).cuda()
    c_dev = torch.from_numpy(frames.rgb).cuda()
    vol = TsdfVolume(frames.pool_capacity, frames.voxel_size, frames.trunc,
                     frames.table_capacity)
    vol.set_pool_layout(args.layout)
    vol.set_update_kernel(args.update_kernel)
    vol.set_occlusion(args.occlusion)
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

    group = args.group or vol.info["max_frames_per_launch"]
    groups = [(a, min(n, a + group)) for a in range(0, n, group)]

    fused = args.update_kernel == "fused" and args.occlusion == "ray"

    def one_fused_step():
        rc = lib.tsdf_reset(h, sptr)
        assert rc == 0
        for a, b in groups:
            rc = lib.tsdf_integrate_batch(h, b - a, dptr + 4 * a * px, cptr + 12 * a * px,
                                          frames.width, frames.height, kp, pps[a], sptr)
            assert rc == 0, lib.tsdf_last_error()

    def one_step(events=None):
        rc = lib.tsdf_reset(h, sptr)
        assert rc == 0
        for g, (a, b) in enumerate(groups):
            if fused:
                # one call, one kernel: its time is booked as the update stage
                if events is not None:
                    events[2 * g].record(stream)
                    events[2 * g + 1].record(stream)
                rc = lib.tsdf_integrate_batch(h, b - a, dptr + 4 * a * px, cptr + 12 * a * px,
                                              frames.width, frames.height, kp, pps[a], sptr)
                assert rc == 0, lib.tsdf_last_error()
                continue
            if events is not None:
                events[2 * g].record(stream)
            rc = lib.tsdf_allocate_batch(h, b - a, dptr + 4 * a * px, frames.width,
                                         frames.height, kp, pps[a], sptr)
            assert rc == 0, lib.tsdf_last_error()
            if events is not None:
                events[2 * g + 1].record(stream)
            rc = lib.tsdf_update_batch(h, b - a, dptr + 4 * a * px, cptr + 12 * a * px,
                                       frames.width, frames.height, kp, pps[a], sptr)
            assert rc == 0, lib.tsdf_last_error()
        if events is not None:
            events[2 * len(groups)].record(stream)

    # warm-up, and the per-step counts from the first warm-up step
    for i in range(max(args.warmup, 1)):
        one_step()
        if i == 0:
            torch.cuda.synchronize()
            st = vol.stats()
            blocks = vol.block_count()
    points_per_step = st["valid_points"]
    updates_per_step = st["voxel_updates"]

    # census of distinct voxels each update launch modifies (untimed): the
    # algorithmic bytes of a launch count each such voxel once
    distinct = census_distinct_voxels(torch, vol, frames, d_dev, c_dev, groups)

    # timed region
    ng = len(groups)
    other_mib = other_processes_mib(torch.cuda.current_device())
    clocks = ClockSampler(torch.cuda.current_device(), args.clock_log)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    per_step_events = []
    for k in range(args.steps):
        evk = [torch.cuda.Event(enable_timing=True) for _ in range(2 * ng + 1)]
        one_step(evk)
        per_step_events.append(evk)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    launch_alloc, launch_update, step_ms = [], [], []
    for evk in per_step_events:
        for g in range(ng):
            launch_alloc.append(evk[2 * g].elapsed_time(evk[2 * g + 1]))
            launch_update.append(evk[2 * g + 1].elapsed_time(evk[2 * g + 2]))
        step_ms.append(evk[0].elapsed_time(evk[2 * ng]))
    stage_alloc = float(sum(launch_alloc))
    stage_update = float(sum(launch_update))
    max_ms = max_over_ranks(elapsed_ms, world)
    total_points = sum_over_ranks(points_per_step * args.steps, world)
    value = total_points / (max_ms / 1000.0)
    upd_rate = sum_over_ranks(updates_per_step * args.steps, world) / (max_ms / 1000.0)

    # rooflines.  Units as defined for the integrate path: per frame, the
    # update kernel must read 16 B per valid point and read-modify-write the
    # five 4-byte sums of every distinct voxel the frame touches (40 B), and
    # issue 5 float additions per such voxel; a launch covers `group` frames.
    red_peaks, cas_peaks = measure_red_peaks(torch)
    red_peak = max(v["adds_per_s"] for v in red_peaks["hbm_4GB"].values())
    hbm_peak, peak_kind = _peaks()
    n_update_launches = ng * args.steps
    upd_ms_avg = stage_update / n_update_launches
    alloc_ms_avg = stage_alloc / n_update_launches
    u_frames = distinct["frame_by_frame"]
    bytes_per_launch = (16.0 * points_per_step + 40.0 * u_frames) / ng
    achieved = bytes_per_launch / (upd_ms_avg / 1000.0) / 1e9
    # the kernels the update stage launches in the selected mode
    upd_kernel = {"per_sample": "update_kernel", "auto": "update_kernel",
                  "pre_reduced": "update_rows_kernel",
                  "adaptive": "update_kernel+update_rows_kernel",
                  "fused": "integrate_fused_kernel"}[args.update_kernel]
    if args.occlusion == "reproject":
        upd_kernel = "update_kernel (reprojection test)"
    mode = args.update_kernel if args.occlusion == "ray" else "reproject"
    if mode == "auto":
        mode = "per_sample"         # the stage calls run the per-sample update
    if args.layout == "planar":
        mode += "_planar"
    prof_upd = _profile_record(f"update_{mode}_room_walk_1280x720.md",
                               ["tsdf_update.cu", "tsdf_device.cuh", "tsdf_internal.h"])
    prof_alloc = _profile_record("allocate_kernel_room_walk_1280x720.md"
                                 if args.occlusion == "ray" else
                                 "allocate_kernel_reproject_room_walk_1280x720.md",
                                 ["tsdf_alloc.cu", "tsdf_device.cuh", "tsdf_internal.h"])
    same_shape = (args.workload == "room_walk" and frames.width == 1280 and frames.height == 720
                  and group == vol.info["max_frames_per_launch"])
    roofline = {
        "bound": "hbm", "kernel": upd_kernel, "achieved": achieved, "peak": hbm_peak,
        "unit": "GB/s", "frac": achieved / hbm_peak,
        "traffic": (_per_launch(prof_upd, "traffic_bytes_per_launch", n / ng)
                    if same_shape else None),
        "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS)",
        "bytes_per_launch_alg": bytes_per_launch, "avg_launch_ms": upd_ms_avg,
        "units": "per frame: 16 B per valid point + 40 B per distinct voxel of the frame",
    }
    adds_alg = 5.0 * u_frames / ng
    red_peak_l2 = max(v["adds_per_s"] for v in red_peaks["l2_32MB"].values())
    add_rate = adds_alg / (upd_ms_avg / 1000.0)
    red_roof = {
        "bound": "l2_red", "kernel": upd_kernel, "unit": "float adds/s",
        "achieved": add_rate, "peak": red_peak, "frac": add_rate / red_peak,
        "peak_l2_resident": red_peak_l2, "frac_l2_resident": add_rate / red_peak_l2,
        "algorithmic_adds_per_launch": adds_alg,
        "issued_adds_per_launch": 5.0 * updates_per_step / ng,
        "peak_source": "measured live: best red.global.add pattern, 4 GB footprint "
                       "(peak_l2_resident: best pattern, 32 MB footprint)",
        "probe": red_peaks,
    }
    # the closest memory-side ceiling: L2 reduction sectors the kernel sends
    # (ncu, per launch, while the source matches the capture) per second of
    # the live launch time, against the measured rate of scattered 4-wide
    # reductions into L2-resident lines (one sector each)
    req_peak = red_peaks["l2_32MB"]["v4_scattered"]["ops_per_s"]
    sectors = (_per_launch(prof_upd, "l2_red_sectors_per_launch", n / ng)
               if same_shape else None)
    red_requests = {
        "bound": "l2_red_requests", "kernel": upd_kernel, "unit": "sectors/s",
        "peak": req_peak,
        "peak_source": "measured live: scattered red.global.add.v4.f32, 32 MB footprint",
        "sectors_per_launch": sectors,
        "achieved": None if sectors is None else sectors / (upd_ms_avg / 1000.0),
        "frac": None if sectors is None else sectors / (upd_ms_avg / 1000.0) / req_peak,
    }
    t_hbm = bytes_per_launch / (hbm_peak * 1e9)
    t_red = adds_alg / red_peak
    combined = {"roofline_ms_per_launch": 1000.0 * max(t_hbm, t_red),
                "binding_term": "hbm" if t_hbm >= t_red else "l2_red",
                "frac": 1000.0 * max(t_hbm, t_red) / upd_ms_avg}
    # stricter: a launch's voxels counted once for all of its frames
    u_union = distinct["total"] / ng
    b_union = (16.0 * points_per_step / ng + 40.0 * u_union)
    union = {"bytes_per_launch_alg": b_union,
             "frac_hbm": b_union / (upd_ms_avg / 1000.0) / 1e9 / hbm_peak,
             "frac_l2_red": 5.0 * u_union / (upd_ms_avg / 1000.0) / red_peak}
    # the allocate kernel is bound by instruction issue: warp instructions per
    # launch (ncu count for this kernel source) against 4 issue slots per SM
    # per cycle at the SM clock sampled over the timed region
    alloc_roof = None
    sm_mhz = (clk or {}).get("sm_mhz") or 2070.0
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    if same_shape and prof_alloc.get("warp_instructions_per_launch"):
        ipl = _per_launch(prof_alloc, "warp_instructions_per_launch", n / ng)
        peak_issue = sms * 4 * sm_mhz * 1e6
        ach = ipl / (alloc_ms_avg / 1000.0)
        alloc_roof = {"bound": "alu", "kernel": "allocate_kernel", "unit": "warp instructions/s",
                      "achieved": ach, "peak": peak_issue, "frac": ach / peak_issue,
                      "warp_instructions_per_launch": ipl,
                      "peak_source": f"{sms} SMs x 4 issue slots x sampled {sm_mhz:.0f} MHz",
                      "traffic": _per_launch(prof_alloc, "traffic_bytes_per_launch", n / ng)}
    # its memory terms, for the record (far from binding): HBM bytes it must
    # read (4 B of depth per pixel of the launch) and the L2 atomic sectors
    # ncu counted (compare-and-swaps and pool-counter adds) against the
    # measured compare-and-swap rate
    px_launch = frames.width * frames.height * n / ng
    alloc_mem = {"hbm_bytes_per_launch_alg": 4.0 * px_launch,
                 "frac_hbm": 4.0 * px_launch / (alloc_ms_avg / 1000.0) / 1e9 / hbm_peak,
                 "cas_peak_ops_per_s": cas_peaks["hbm_4GB"]["ops_per_s"],
                 "cas_peak_ops_per_s_l2": cas_peaks["l2_32MB"]["ops_per_s"]}
    if same_shape and prof_alloc.get("l2_atomic_sectors_per_launch"):
        at = _per_launch(prof_alloc, "l2_atomic_sectors_per_launch", n / ng)
        alloc_mem["l2_atomic_sectors_per_launch"] = at
        alloc_mem["frac_l2_atomics"] = at / (alloc_ms_avg / 1000.0) / cas_peaks["l2_32MB"]["ops_per_s"]

    result = {
        "metric": METRIC, "value": value, "unit": "points/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": dict(workload_config(frames, args), parallelism=f"replicas{world}"),
        "voxel_updates_per_s": upd_rate,
        "frames_per_launch": group,
        "update_kernel": args.update_kernel,
        "occlusion": args.occlusion,
        "pool_layout": args.layout,
        "stages_ms_per_launch": {"allocate": alloc_ms_avg, "update": upd_ms_avg},
        "stages_note": ("fused: one kernel per group, booked as the update stage" if fused
                        else "allocate launch, then update launch(es), per group"),
        # each launch is its own timing window (CUDA events around it); steps
        # in timed order, split in halves to show drift across the run
        "stage_percentiles_ms": {"allocate": _percentiles(launch_alloc),
                                 "update": _percentiles(launch_update),
                                 "step_without_reset": _percentiles(step_ms)},
        "step_halves_median_ms": [float(np.median(step_ms[:len(step_ms) // 2] or step_ms)),
                                  float(np.median(step_ms[len(step_ms) // 2:]))],
        "other_processes_mib": other_mib,
        "stages_ms_per_frame": {"allocate": stage_alloc / (n * args.steps),
                                "update": stage_update / (n * args.steps)},
        "blocks": blocks, "points_per_step": points_per_step,
        "voxel_updates_per_step": updates_per_step,
        "distinct_voxels_per_step": distinct["total"],
        "distinct_voxels_per_step_frame_by_frame": distinct["frame_by_frame"],
        "fixed_divisor_fast_path": vol.info["fixed_divisor_fast_path"],
        "clocks": clk,
        "gpu_launches": args.steps * (1 + sum(1 + _update_kernels(args, frames, b - a)
                                              for a, b in groups)),
        "roofline": roofline,
        "roofline_l2_red": red_roof,
        "roofline_l2_red_requests": red_requests,
        "roofline_update_combined": combined,
        "roofline_update_launch_union": union,
        "roofline_allocate": alloc_roof,
        "allocate_memory_terms": alloc_mem,
    }

    if not args.no_e2e:
        result["e2e"] = e2e_host(torch, vol, frames, args)
    result["extraction"] = measure_extraction(torch, vol, blocks, hbm_peak)
    if not fused:
        # the fused allocate+update variant on the same frames, same protocol
        # (not the headline: integration as specified runs two kernels)
        vol.set_update_kernel("fused")
        for _ in range(max(args.warmup, 1)):
            one_fused_step()
        torch.cuda.synchronize()
        fa = torch.cuda.Event(enable_timing=True)
        fb_ = torch.cuda.Event(enable_timing=True)
        fa.record(stream)
        for _ in range(args.steps):
            one_fused_step()
        fb_.record(stream)
        torch.cuda.synchronize()
        fused_ms = max_over_ranks(fa.elapsed_time(fb_), world)
        result["variant_fused"] = {
            "value": sum_over_ranks(points_per_step * args.steps, world) / (fused_ms / 1000.0),
            "unit": "points/s", "ms_per_step": fused_ms / args.steps,
            "note": "tsdf_integrate_batch per group with TSDF_UPDATE_FUSED: one kernel "
                    "allocates and updates (dense tiles pre-reduced by a second)"}
        vol.set_update_kernel(args.update_kernel)
    if not fused and args.occlusion == "ray" and args.layout == "interleaved":
        result["variant_planar"] = variant_planar(torch, vol, frames, groups, one_step, stream,
                                                  args, world)
    if not fused and args.occlusion == "ray":
        result["variant_reproject"] = variant_reproject(
            torch, vol, frames, d_dev, c_dev, groups, one_step, stream, args, world,
            hbm_peak, red_peak)
    if rank == 0:
        # the single-thread CPU baseline: the oracle as it stands on a
        # bounded sample of the workload
        sampled = None
        if world == 1 and not args.no_cpu_baseline:
            v, u, sample, ovol, n_sample = oracle_sample(frames, args.cpu_baseline_seconds,
                                                         occlusion=args.occlusion)
            result["cpu_baseline"] = {"value": v, "unit": "points/s", "cores": 1,
                                      "kind": "oracle", "sample": sample,
                                      "voxel_updates_per_s": u, "cpu": platform.machine()}
            sampled = (ovol, n_sample)
        # the timing counts only if the GPU's volume matches the oracle's
        # (over the whole trajectory by default); otherwise the headline is
        # withheld
        gate = parity_gate(torch, vol, frames, d_dev, c_dev, args.gate, args.occlusion,
                           sampled)
        apply_gate(result, gate)
    vol.close()
    if rank == 0:
        print(json.dumps(result), flush=True)


def variant_planar(torch, vol, frames, groups, one_step, stream, args, world) -> dict:
    """The same step with the pool as five separate arrays (the pages' own
    layout), same protocol: what the interleaved records gain."""
    vol.reset()
    torch.cuda.synchronize()
    vol.set_pool_layout("planar")
    for _ in range(max(args.warmup, 1)):
        one_step()
    ng = len(groups)
    torch.cuda.synchronize()
    ta = torch.cuda.Event(enable_timing=True)
    tb = torch.cuda.Event(enable_timing=True)
    ta.record(stream)
    evs = []
    for _ in range(args.steps):
        evk = [torch.cuda.Event(enable_timing=True) for _ in range(2 * ng + 1)]
        one_step(evk)
        evs.append(evk)
    tb.record(stream)
    torch.cuda.synchronize()
    st = vol.stats()
    ms = max_over_ranks(ta.elapsed_time(tb), world)
    alloc = [e[2 * g].elapsed_time(e[2 * g + 1]) for e in evs for g in range(ng)]
    upd = [e[2 * g + 1].elapsed_time(e[2 * g + 2]) for e in evs for g in range(ng)]
    vol.reset()
    torch.cuda.synchronize()
    vol.set_pool_layout(args.layout)
    return {
        "value": sum_over_ranks(st["valid_points"] * args.steps, world) / (ms / 1000.0),
        "unit": "points/s", "ms_per_step": ms / args.steps,
        "stages_ms_per_launch": {"allocate": float(np.mean(alloc)), "update": float(np.mean(upd))},
        "note": "TSDF_LAYOUT_PLANAR: the five sums as separate arrays, five scalar reductions "
                "per merged sample",
    }


def variant_reproject(torch, vol, frames, d_dev, c_dev, groups, one_step, stream, args, world,
                      hbm_peak, red_peak) -> dict:
    """The reprojection occlusion test on the same frames and protocol: the
    same step (reset, then allocate and update per group), timed as a whole
    and per launch; the update's rooflines with the same units as the
    headline's (16 B per valid point and 40 B / 5 adds per distinct voxel of
    each frame)."""
    vol.set_occlusion("reproject")
    for i in range(max(args.warmup, 1)):
        one_step()
        if i == 0:
            torch.cuda.synchronize()
            st = vol.stats()
    distinct = census_distinct_voxels(torch, vol, frames, d_dev, c_dev, groups)
    ng = len(groups)
    torch.cuda.synchronize()
    ta = torch.cuda.Event(enable_timing=True)
    tb = torch.cuda.Event(enable_timing=True)
    ta.record(stream)
    evs = []
    for _ in range(args.steps):
        evk = [torch.cuda.Event(enable_timing=True) for _ in range(2 * ng + 1)]
        one_step(evk)
        evs.append(evk)
    tb.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(ta.elapsed_time(tb), world)
    alloc = [e[2 * g].elapsed_time(e[2 * g + 1]) for e in evs for g in range(ng)]
    upd = [e[2 * g + 1].elapsed_time(e[2 * g + 2]) for e in evs for g in range(ng)]
    vol.set_occlusion(args.occlusion)
    upd_avg = float(np.mean(upd))
    pts = st["valid_points"]
    u_frames = distinct["frame_by_frame"]
    b_launch = (16.0 * pts + 40.0 * u_frames) / ng
    adds = 5.0 * u_frames / ng
    return {
        "value": sum_over_ranks(pts * args.steps, world) / (ms / 1000.0), "unit": "points/s",
        "ms_per_step": ms / args.steps,
        "voxel_updates_per_step": st["voxel_updates"],
        "stages_ms_per_launch": {"allocate": float(np.mean(alloc)), "update": upd_avg},
        "stage_percentiles_ms": {"allocate": _percentiles(alloc), "update": _percentiles(upd)},
        "roofline_update": {"bound": "hbm", "achieved": b_launch / (upd_avg / 1000.0) / 1e9,
                            "peak": hbm_peak, "unit": "GB/s",
                            "frac": b_launch / (upd_avg / 1000.0) / 1e9 / hbm_peak,
                            "bytes_per_launch_alg": b_launch},
        "roofline_update_l2_red": {"achieved": adds / (upd_avg / 1000.0), "peak": red_peak,
                                   "unit": "float adds/s",
                                   "frac": adds / (upd_avg / 1000.0) / red_peak},
        "note": "TSDF_OCCLUSION_REPROJECT: allocate and per-sample update kernels, the depth "
                "and colour read where each voxel centre projects",
    }


RED_MODES = ((0, "scalar_coalesced", 1), (1, "scalar_scattered", 1), (2, "v4_coalesced", 4),
             (3, "v4_scattered", 4), (4, "scalar_sector_grouped", 1))
CAS_MODE = 5


def measure_red_peaks(torch) -> dict:
    """L2 float-reduction throughput (red.global.add), float additions per
    second, for scalar / 4-wide operands and coalesced / scattered addresses,
    over an L2-resident (32 MB) and an HBM-resident (4 GB) footprint, and the
    rate of 64-bit compare-and-swaps on scattered 16-byte entries; best of 6
    launches each.  Returns (reductions, compare-and-swaps)."""
    import ctypes
    from hash_blocked_tsdf_gb300 import _build
    lib = ctypes.CDLL(_build.peaks_library_path())
    lib.peak_red.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                             ctypes.c_int, ctypes.c_void_p]
    lib.peak_red.restype = ctypes.c_int
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    stream = torch.cuda.current_stream()
    out = {}
    cas_out = {}
    for foot, nbytes in (("l2_32MB", 32 << 20), ("hbm_4GB", 4 << 30)):
        buf = torch.zeros(nbytes // 4, dtype=torch.float32, device="cuda")
        res = {}
        for mode, name, width in RED_MODES:
            blocks, reps = sms * 8, 64
            best = None
            for _ in range(6):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                rc = lib.peak_red(buf.data_ptr(), buf.numel(), mode, reps, blocks,
                                  stream.cuda_stream)
                b.record(stream)
                assert rc == 0, rc
                torch.cuda.synchronize()
                ms = a.elapsed_time(b)
                best = ms if best is None else min(best, ms)
            ops = blocks * 256 * reps
            res[name] = {"ops_per_s": ops / (best / 1e3), "adds_per_s": width * ops / (best / 1e3)}
        out[foot] = res
        buf.zero_()
        best = None
        for _ in range(6):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            rc = lib.peak_red(buf.data_ptr(), buf.numel(), CAS_MODE, 64, sms * 8,
                              stream.cuda_stream)
            b.record(stream)
            assert rc == 0, rc
            torch.cuda.synchronize()
            best = a.elapsed_time(b) if best is None else min(best, a.elapsed_time(b))
        cas_out[foot] = {"ops_per_s": sms * 8 * 256 * 64 / (best / 1e3)}
        del buf
    torch.cuda.empty_cache()
    return out, cas_out


def measure_atomic_probes(torch) -> dict:
    """What two alternative update designs would pay, measured: atomic adds
    to shared memory at random addresses of a 64 KB array (float and 32-bit
    integer; lane operations per second and per SM per clock at the sampled
    clock), and random 32-byte records (all five sums of a voxel in one
    sector) reduced as a 4-wide plus a scalar reduction or as one 32-byte
    bulk reduction from shared memory, into an L2-resident 32 MB footprint
    (records per second).  Best of 5 launches each, CUDA events."""
    import ctypes
    from hash_blocked_tsdf_gb300 import _build
    lib = ctypes.CDLL(_build.peaks_library_path())
    lib.peak_smem_atomic.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_void_p]
    lib.peak_smem_atomic.restype = ctypes.c_int
    lib.peak_record_red.argtypes = [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_void_p]
    lib.peak_record_red.restype = ctypes.c_int
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sms = props.multi_processor_count
    stream = torch.cuda.current_stream()

    def best_ms(launch):
        best = None
        for _ in range(6):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            rc = launch()
            b.record(stream)
            assert rc == 0, rc
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        return best

    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    out = {}
    blocks, reps = sms * 2, 4096
    col = torch.zeros(blocks * 256, dtype=torch.float32, device="cuda")
    smem = {}
    for mode, name in ((0, "f32_atomic_add"), (1, "u32_atomic_add")):
        ms = best_ms(lambda: lib.peak_smem_atomic(col.data_ptr(), mode, reps, blocks,
                                                  stream.cuda_stream))
        smem[name] = {"lane_ops_per_s": blocks * 256 * reps / (ms / 1e3)}
    rec = {}
    buf = torch.zeros((32 << 20) // 4, dtype=torch.float32, device="cuda")
    n_records = buf.numel() // 8
    for mode, name in ((0, "v4_plus_scalar"), (1, "bulk_32B_from_shared")):
        rb, rr = sms * 8, 256
        ms = best_ms(lambda: lib.peak_record_red(buf.data_ptr(), n_records, mode, rr, rb,
                                                 stream.cuda_stream))
        rec[name] = {"records_per_s": rb * 256 * rr / (ms / 1e3)}
    c = clk.stop() or {}
    mhz = c.get("sm_mhz") or 2070.0
    for v in smem.values():
        v["per_sm_per_clock"] = v["lane_ops_per_s"] / sms / (mhz * 1e6)
    out["shared_memory_64KB"] = smem
    out["records_32B_l2_32MB"] = rec
    out["sm_mhz"] = mhz
    out["sms"] = sms
    del buf, col
    torch.cuda.empty_cache()
    return out


def _profile_record(name: str, sources) -> dict:
    """Figures recorded in a committed ncu summary under profiles/, used only
    while the kernel's source is unchanged since the capture (matching hash)."""
    import hashlib
    path = os.path.join(REPO, "profiles", name)
    try:
        text = open(path).read()
    except OSError:
        return {}
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(REPO, "hash_blocked_tsdf_gb300", "csrc", src), "rb") as fh:
            h.update(fh.read())
    rec = {}
    for line in text.splitlines():
        if ":" in line and not line.startswith(("|", " ", "#")):
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip()
    if rec.get("kernel_source_sha256_16") != h.hexdigest()[:16]:
        return {}
    out = {}
    for k in ("traffic_bytes_per_launch", "warp_instructions_per_launch",
              "l2_atomic_sectors_per_launch", "l2_red_sectors_per_launch",
              "frames_per_captured_launch"):
        if k in rec:
            out[k] = float(rec[k])
    return out


def _per_launch(rec: dict, key: str, frames_per_launch: float):
    """A captured per-launch figure scaled to the timed launches' average
    frame count (the last group of a trajectory is shorter), in proportion
    to the frames processed."""
    if key not in rec:
        return None
    return rec[key] * frames_per_launch / rec.get("frames_per_captured_launch", frames_per_launch)


def census_distinct_voxels(torch, vol, frames, d_dev, c_dev, groups) -> dict:
    """Distinct voxels each update launch modifies (a launch covers a group of
    frames), and for reference the sum over single frames, counted by
    comparing the weight array before and after."""
    from hash_blocked_tsdf_gb300 import binding
    ptrs = binding.tsdf_get_pool(vol.handle)
    cap = vol.info["pool_capacity"]
    # the weight sums (every 4th float in the interleaved layout)
    weight = _as_tensor(torch, ptrs["weight"], cap * 512, stride=ptrs["stride"])
    prev = torch.empty(weight.shape, dtype=weight.dtype, device=weight.device)
    out = {}
    for name, grp in (("total", groups), ("frame_by_frame",
                                          [(f, f + 1) for f in range(frames.n_frames)])):
        vol.reset()
        counts = []
        for a, b in grp:
            used = vol.block_count() * 512
            prev[:used].copy_(weight[:used])
            vol.allocate_batch(d_dev[a:b], frames.K, frames.poses[a:b])
            vol.update_batch(d_dev[a:b], c_dev[a:b], frames.K, frames.poses[a:b])
            used = vol.block_count() * 512
            counts.append(int((weight[:used] != prev[:used]).sum().item()))
        out[name] = int(sum(counts))
    vol.reset()
    torch.cuda.synchronize()
    del prev
    return out


def _as_tensor(torch, ptr: int, n: int, stride: int = 1):
    class _Arr:
        __cuda_array_interface__ = {"shape": (n,), "typestr": "<f4", "data": (ptr, False),
                                    "version": 3,
                                    "strides": None if stride == 1 else (4 * stride,)}
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
    if args.sweep:
        run_sweep(args)
        return
    if args.probe_report:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        for rec in probe_depth_report(torch):
            print(json.dumps({"probe_depth": rec}), flush=True)
        return
    if args.probe_atomics:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        print(json.dumps({"probe_atomics": measure_atomic_probes(torch)}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
