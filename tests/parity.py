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


# The oracle's whole volume for a long trajectory, computed in parallel
# (oracle/parallel.py).
from oracle.parallel import full_volume_oracle  # noqa: E402,F401
