"""Host-side logic of bench.py that needs no GPU: launch-time percentiles,
the count of update kernels per launch, and the parity gate's comparison
(fed with the oracle's own result, then with planted mistakes)."""
import types

import numpy as np
import pytest

import bench
from hash_blocked_tsdf_gb300 import scenes


def test_percentiles_of_known_values():
    p = bench._percentiles(list(range(1, 101)))
    assert p["n"] == 100
    assert p["p50"] == pytest.approx(50.5)
    assert p["p95"] == pytest.approx(95.05)
    assert p["p99"] == pytest.approx(99.01)


def test_update_kernel_count_per_launch():
    big = types.SimpleNamespace(width=640, height=480)
    small = types.SimpleNamespace(width=160, height=120)
    adaptive = types.SimpleNamespace(update_kernel="adaptive")
    per_sample = types.SimpleNamespace(update_kernel="per_sample")
    assert bench._update_kernels(adaptive, big, 1) == 2          # 307,200 px >= 2^18
    assert bench._update_kernels(adaptive, small, 8) == 1        # 153,600 px < 2^18
    assert bench._update_kernels(adaptive, small, 16) == 2
    assert bench._update_kernels(per_sample, big, 8) == 1
    # the reprojection test always runs the per-sample update as its own kernel
    for kind in ("adaptive", "pre_reduced", "fused"):
        reproject = types.SimpleNamespace(update_kernel=kind, occlusion="reproject")
        assert bench._update_kernels(reproject, big, 8) == 1


class _FakeVolume:
    """Stands in for a GPU volume: returns a prepared export and counters."""

    def __init__(self, export, stats):
        self._export, self._stats = export, stats

    def reset(self):
        pass

    def integrate_batch(self, *args):
        pass

    def stats(self):
        return dict(self._stats)

    def export_blocks(self):
        return {k: v.copy() for k, v in self._export.items()}


def _gate(oracle_mod, mutate=None, scope="sample"):
    frames = scenes.tiny_sphere_plane()
    o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    o.integrate_frames(frames)
    e = o.export()
    c = o.counters()
    rng = np.random.default_rng(0)
    perm = rng.permutation(len(e["coords"]))             # pool order, not coordinate order
    g = {k: np.asarray(e[k])[perm].astype(np.int32 if k == "coords" else np.float32)
         for k in ("coords", "tsdf", "weight", "r", "g", "b")}
    if mutate:
        mutate(g)
    stats = {"valid_points": c["valid_points"], "voxel_updates": c["accumulated"],
             "missed_contributions": c["missed_contributions"],
             "out_of_range_samples": c["out_of_range_samples"], "pool_exhausted": 0,
             "probe_overflow": 0}
    fake_torch = types.SimpleNamespace(cuda=types.SimpleNamespace(synchronize=lambda: None))
    return bench.parity_gate(fake_torch, _FakeVolume(g, stats), frames, frames.depth,
                             frames.rgb, scope, "ray", sampled=(o, frames.n_frames))


def test_parity_gate_passes_on_the_oracle_itself(oracle_mod):
    out = _gate(oracle_mod)
    assert out["pass"] and out["block_set_equal"] and out["weights_equal"]
    assert out["sums_worst_error_over_bound"] <= 1.0


def test_parity_gate_over_the_whole_trajectory_uses_the_parallel_oracle(oracle_mod):
    # scope "full" recomputes the oracle's volume in worker processes (frame
    # chunks x block partitions) instead of taking the sample's volume
    out = _gate(oracle_mod, scope="full")
    assert out["scope"] == "full" and "processes" in out["oracle"]
    assert out["pass"] and out["block_set_equal"] and out["weights_equal"]
    assert out["sums_worst_error_over_bound"] <= 1.0
    out = _gate(oracle_mod, lambda g: g["weight"].__setitem__((0, 0), 7.0), scope="full")
    assert not out["pass"]


def test_parity_gate_rejects_a_wrong_weight(oracle_mod):
    def bump(g):
        i = np.argwhere(g["weight"] > 0)[0]
        g["weight"][tuple(i)] += 1.0
    out = _gate(oracle_mod, bump)
    assert not out["weights_equal"] and not out["pass"]


def test_parity_gate_rejects_a_missing_block(oracle_mod):
    def drop(g):
        for k in g:
            g[k] = g[k][1:]
    out = _gate(oracle_mod, drop)
    assert not out["block_set_equal"] and not out["pass"]


def test_parity_gate_rejects_a_sum_outside_the_bound(oracle_mod):
    def shift(g):
        i = np.argwhere(g["weight"] > 0)[0]
        g["tsdf"][tuple(i)] += 1e-3
    out = _gate(oracle_mod, shift)
    assert out["sums_worst_error_over_bound"] > 1.0 and not out["pass"]
    assert out["sums"]["tsdf"]["voxels_over_stated_bound"] == 1
    assert out["sums"]["r"]["voxels_over_stated_bound"] == 0


def test_a_failed_gate_withholds_the_headline(oracle_mod):
    line = {"value": 5.0, "e2e": {"value": 4.0, "unit": "points/s"}}
    bench.apply_gate(line, {"pass": True})
    assert line["value"] == 5.0 and line["gated"] is True and "withheld" not in line
    line = {"value": 5.0, "e2e": {"value": 4.0, "unit": "points/s"}}
    bench.apply_gate(line, _gate(oracle_mod, lambda g: g["weight"].__setitem__((0, 0), 7.0)))
    assert line["value"] is None and line["e2e"]["value"] is None and line["gated"] is False
    assert line["withheld"]["value"] == 5.0 and line["withheld"]["e2e_value"] == 4.0


def test_captured_figures_scale_to_the_timed_launches():
    # a 32-frame capture stands for launches that average 30 frames
    rec = {"traffic_bytes_per_launch": 3200.0, "frames_per_captured_launch": 32.0}
    assert bench._per_launch(rec, "traffic_bytes_per_launch", 30.0) == pytest.approx(3000.0)
    assert bench._per_launch(rec, "warp_instructions_per_launch", 30.0) is None
    # a record without the captured frame count is taken as it stands
    assert bench._per_launch({"traffic_bytes_per_launch": 5.0}, "traffic_bytes_per_launch",
                             8.0) == 5.0
