"""The CPU oracle's whole volume for a long trajectory, computed in parallel
on the host cores -- TEST INFRASTRUCTURE ONLY, like the rest of this package
(used by the GPU parity tests and by the benchmark's parity gate).

The frames are cut into chunks and the blocks into partitions
((bx + by + bz) mod parts, the oracle's keep_partition filter, which changes
none of its arithmetic); one worker process integrates one chunk of frames
with the plain sequential oracle and keeps the sums of one partition.  Sums
commute ("What Irregularity Costs", design section, accumulation), so adding
the chunks' sums block by block gives one sequential run's sums up to
double rounding; the block set is the union of the chunks' block sets and
the counters add.  Workers start with the spawn method, so a process that
already uses CUDA can call this.
"""
from __future__ import annotations

import os

import numpy as np


def _sort_by_coords(coords):
    return np.lexsort((coords[:, 2], coords[:, 1], coords[:, 0]))


def _cpu_count() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def worker_count() -> int:
    """Worker processes full_volume_oracle starts by default: the host's
    cores, at least 2 and at most 16."""
    return max(2, min(16, _cpu_count()))


def _oracle_piece(args):
    """One worker: frames [start, stop) of the memory-mapped trajectory,
    sums kept for block partition `part` of `parts`.  Returns the block set
    and counters (partition 0 only: the other partitions walk the same
    frames) and the kept blocks' sums."""
    folder, start, stop, parts, part, occlusion, voxel, trunc = args
    os.environ["OMP_NUM_THREADS"] = "1"
    from oracle import OracleVolume
    depth = np.load(os.path.join(folder, "depth.npy"), mmap_mode="r")
    rgb = np.load(os.path.join(folder, "rgb.npy"), mmap_mode="r")
    poses = np.load(os.path.join(folder, "poses.npy"))
    K = np.load(os.path.join(folder, "K.npy"))
    o = OracleVolume(voxel, trunc)
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

    workers = workers or worker_count()
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
    order = _sort_by_coords(kept)
    out = {"coords": kept[order]}
    for k in SUM_FIELDS:
        out[k] = acc[k][:kept.shape[0]][order]      # row i holds the i-th key of `rows`
        acc[k] = None
    assert np.array_equal(out["coords"], all_coords), "partitions do not cover the block set"
    return out, counters
