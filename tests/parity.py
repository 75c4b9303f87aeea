"""Comparison of the CUDA path's read-out with the CPU oracle, and a
frame-parallel driver for the oracle on large trajectories.

Tolerance.  Block coordinates, block count and weight sums must match
exactly (unit weights make every weight sum an integer below 2^24).  TSDF
and colour sums are float32 sums accumulated by atomics in an unspecified
order; the oracle holds the exact sum x of the same float32 terms (double
accumulation).  The stated bound is max(1e-5 |x|, 1e-6).  Any float32
summation of n terms t_i, in any order or tree, errs by at most
gamma(n-1) * sum |t_i| with gamma(m) = m u / (1 - m u), u = 2^-24 (Higham,
Accuracy and Stability of Numerical Algorithms, 2nd ed., section 4.2).  For a
voxel observed in many frames whose TSDF terms cancel, that a-priori bound
can exceed 1e-6, so multi-frame comparisons accept
max(1e-5 |x|, 1e-6, gamma(n-1) * sum |t_i|) and report how many voxels needed
the last term; single-frame comparisons use the stated bound alone.
"""
from __future__ import annotations

import os

import numpy as np

U = 2.0 ** -24


def gamma(m):
    m = np.asarray(m, dtype=np.float64)
    return m * U / (1.0 - m * U)


def sort_by_coords(coords):
    return np.lexsort((coords[:, 2], coords[:, 1], coords[:, 0]))


def compare_sums(gpu: dict, ref: dict, strict: bool, rows=None) -> dict:
    """gpu: float32 arrays [n, 512] already aligned with ref's rows.  Returns a
    report; raises AssertionError on any violation."""
    report = {}
    w_ref = ref["weight"] if rows is None else ref["weight"][rows]
    w_gpu = gpu["weight"].astype(np.float64)
    bad_w = int(np.sum(w_gpu != w_ref))
    assert bad_w == 0, f"{bad_w} voxel weights differ"
    for k in ("tsdf", "r", "g", "b"):
        x = ref[k] if rows is None else ref[k][rows]
        y = gpu[k].astype(np.float64)
        err = np.abs(y - x)
        base = np.maximum(1e-5 * np.abs(x), 1e-6)
        if k == "tsdf":
            s_abs = ref["tsdf_abs"] if rows is None else ref["tsdf_abs"][rows]
        else:
            s_abs = np.abs(x)
        bound = gamma(np.maximum(w_ref - 1.0, 0.0)) * s_abs
        over_base = int(np.sum(err > base))
        tol = base if strict else np.maximum(base, bound)
        over = int(np.sum(err > tol))
        report[k] = {"max_err": float(err.max()) if err.size else 0.0,
                     "max_err_over_base": float((err / base).max()) if err.size else 0.0,
                     "voxels_over_base": over_base}
        assert over == 0, (f"{k}: {over} voxels outside tolerance "
                           f"(max error {err.max():.3g}, strict={strict})")
    return report


def compare_volume(gpu_export: dict, ref_export: dict, strict: bool) -> dict:
    """Full comparison of a GPU export (any pool order) with an oracle export
    (sorted by coordinate)."""
    gc = gpu_export["coords"]
    order = sort_by_coords(gc)
    gc = gc[order]
    rc = ref_export["coords"]
    assert gc.shape == rc.shape, f"block count {gc.shape[0]} != oracle {rc.shape[0]}"
    assert np.array_equal(gc, rc), "block coordinate sets differ"
    aligned = {k: gpu_export[k][order] for k in ("tsdf", "weight", "r", "g", "b")}
    rep = compare_sums(aligned, ref_export, strict)
    rep["blocks"] = int(gc.shape[0])
    return rep


def check_counters(stats: dict, oracle_counters: dict):
    assert stats["valid_points"] == oracle_counters["valid_points"], (stats, oracle_counters)
    assert stats["voxel_updates"] == oracle_counters["accumulated"], (stats, oracle_counters)
    assert stats["missed_contributions"] == oracle_counters["missed_contributions"]
    assert stats["out_of_range_samples"] == oracle_counters["out_of_range_samples"]
    assert stats["probe_overflow"] == 0


# ----------------------------------------------------------------------------
# Full-volume oracle for long trajectories, run in parallel
# ----------------------------------------------------------------------------

def _cpu_count() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_piece(args):
    """One worker: frames [start, stop) of the memory-mapped trajectory,
    sums kept for block partition `part` of `parts`.  Returns the block set
    and counters (partition 0 only: the other partitions walk the same
    frames) and the kept blocks' sums."""
    folder, start, stop, parts, part, occlusion, voxel, trunc = args
    os.environ["OMP_NUM_THREADS"] = "1"
    import oracle
    depth = np.load(os.path.join(folder, "depth.npy"), mmap_mode="r")
    rgb = np.load(os.path.join(folder, "rgb.npy"), mmap_mode="r")
    poses = np.load(os.path.join(folder, "poses.npy"))
    K = np.load(os.path.join(folder, "K.npy"))
    o = oracle.OracleVolume(voxel, trunc)
    o.set_occlusion(occlusion)
    o.keep_partition(parts, part)
    for f in range(start, stop):
        o.integrate(depth[f], rgb[f], K, poses[f])
    e = o.export()
    if part == 0:
        return o.coords(), o.counters(), e
    return None, None, e


SUM_FIELDS = ("tsdf", "weight", "r", "g", "b", "tsdf_abs")


def full_volume_oracle(frames, occlusion: str = "ray", workers: int = 0, parts: int = 4):
    """The oracle's whole volume for a long trajectory, computed in parallel.

    The frames are cut into chunks and the blocks into `parts` partitions
    ((bx + by + bz) mod parts); one worker integrates one chunk of frames and
    keeps the sums of one partition.  Sums commute, so adding the chunks'
    sums block by block gives one sequential run's sums up to double
    rounding; the block set is the union of the chunks' block sets, and the
    counters add.  Frames reach the workers through memory-mapped files.

    Returns the export of one sequential oracle run: coords sorted by
    (x, y, z) and float64 [n, 512] arrays tsdf, weight, r, g, b, tsdf_abs,
    plus the summed counters."""
    import multiprocessing as mp
    import shutil
    import tempfile

    workers = workers or max(2, min(16, _cpu_count()))
    parts = max(1, min(parts, workers))
    chunks = max(1, min(frames.n_frames, workers // parts))
    folder = tempfile.mkdtemp(prefix="tsdf_oracle_frames_")
    try:
        np.save(os.path.join(folder, "depth.npy"), np.ascontiguousarray(frames.depth))
        np.save(os.path.join(folder, "rgb.npy"), np.ascontiguousarray(frames.rgb))
        np.save(os.path.join(folder, "poses.npy"), np.ascontiguousarray(frames.poses))
        np.save(os.path.join(folder, "K.npy"), np.ascontiguousarray(frames.K))
        bounds = np.linspace(0, frames.n_frames, chunks + 1).round().astype(int)
        jobs = [(folder, int(a), int(b), parts, p, occlusion, frames.voxel_size, frames.trunc)
                for a, b in zip(bounds[:-1], bounds[1:]) if b > a for p in range(parts)]
        rows = {}
        cap = 1 << 14
        acc = {k: np.zeros((cap, 512), np.float64) for k in SUM_FIELDS}
        block_sets = []
        counters = {}
        ctx = mp.get_context("spawn")
        with ctx.Pool(min(len(jobs), workers)) as pool:
            for coords, cnt, e in pool.imap_unordered(_oracle_piece, jobs):
                if coords is not None:
                    block_sets.append(coords)
                    for k, v in cnt.items():
                        counters[k] = counters.get(k, 0) + v
                idx = np.fromiter((rows.setdefault(c, len(rows))
                                   for c in map(tuple, e["coords"].tolist())),
                                  dtype=np.int64, count=e["coords"].shape[0])
                if len(rows) > cap:
                    while cap < len(rows):
                        cap *= 2
                    for k in SUM_FIELDS:
                        grown = np.zeros((cap, 512), np.float64)
                        grown[:acc[k].shape[0]] = acc[k]
                        acc[k] = grown
                for k in SUM_FIELDS:
                    acc[k][idx] += e[k]          # rows of one piece are distinct
                del e
    finally:
        shutil.rmtree(folder, ignore_errors=True)
    all_coords = np.unique(np.concatenate(block_sets), axis=0)
    kept = np.array(list(rows.keys()), dtype=np.int32).reshape(-1, 3)
    order = sort_by_coords(kept)
    out = {"coords": kept[order]}
    for k in SUM_FIELDS:
        out[k] = acc[k][:kept.shape[0]][order]      # row i holds the i-th key of `rows`
        acc[k] = None
    assert np.array_equal(out["coords"], all_coords), "partitions do not cover the block set"
    return out, counters
