"""Pins of the oracle's alternative occlusion test, by reprojection of the
voxel centre (the design section's occlusion test, read the other way: the
depth compared against is the one where the centre projects, not the one of
the pixel whose ray selected the voxel).  Checked against geometry computed
here in float64, not against the oracle itself:

- values: on a slanted surface with a step and holes, seen from a rotated
  pose, every voxel that received samples has the mean tsdf
  min(1, (d' - z_c) / trunc) of its own centre, where d' is the depth of the
  pixel nearest to the centre's projection, and the mean colour of that pixel
  (the colours encode the pixel coordinates); and that pixel passes the test;
- completeness: on a constant-depth plane seen head on, the test agrees with
  the ray-depth test (already pinned) for every voxel that projects inside
  the image, so no passing sample is dropped; voxels that project outside
  receive nothing.

Planted mistakes in the reprojection are compiled and each must be rejected.
"""
import os

import numpy as np
import pytest

VOXEL = 0.02
TRUNC = 0.06
W, H = 64, 48


def _rotation(ay, ax):
    cy, sy, cx, sx = np.cos(ay), np.sin(ay), np.cos(ax), np.sin(ax)
    ry = np.array([[cy, 0, sy], [0, 1, 0], [-sy, 0, cy]])
    rx = np.array([[1, 0, 0], [0, cx, -sx], [0, sx, cx]])
    return ry @ rx


def _slanted_step_frame():
    """A slanted surface with a nearer rectangle and a sprinkling of holes;
    colours r = u / W, g = v / H."""
    v, u = np.mgrid[0:H, 0:W].astype(np.float64)
    depth = 1.0 + 0.004 * u + 0.002 * v
    depth[14:30, 20:36] = 0.7 + 0.003 * u[14:30, 20:36]
    depth.reshape(-1)[::17] = 0.0
    rgb = np.stack([u / W, v / H, np.full_like(u, 0.25)], axis=-1)
    K = np.array([60.0, 52.0, 31.3, 23.6])
    pose = np.eye(4)
    pose[:3, :3] = _rotation(0.15, -0.1)
    pose[:3, 3] = [0.1, -0.05, 0.2]
    return depth.astype(np.float32), rgb.astype(np.float32), K.astype(np.float32), \
        pose.astype(np.float32)


def _voxel_centres(e):
    j = np.arange(512)
    local = np.stack([j % 8, (j // 8) % 8, j // 64], axis=1)
    idx = e["coords"][:, None, :].astype(np.int64) * 8 + local[None]
    return (idx + 0.5) * VOXEL


def _project(centres, K, pose):
    """Camera-frame centre and (u, v) projection, float64."""
    R = pose[:3, :3].astype(np.float64)
    t = pose[:3, 3].astype(np.float64)
    c = (centres - t) @ R          # rows: R^T (centre - t)
    u = K[0] * (c[..., 0] / c[..., 2]) + K[2]
    v = K[1] * (c[..., 1] / c[..., 2]) + K[3]
    return c, u, v


def _integrate(oracle_mod, mutant, mode, depth, rgb, K, pose):
    o = oracle_mod.OracleVolume(VOXEL, TRUNC, mutant=mutant)
    o.set_occlusion(mode)
    o.integrate(depth, rgb, K, pose)
    return o.export()


def _near_boundary(x, eps=1e-3):
    """x + 1/2 within eps of an integer: the nearest pixel is not decided in
    float64 with margin to spare."""
    f = x + 0.5 - np.floor(x + 0.5)
    return (f < eps) | (f > 1 - eps)


def pin_values(oracle_mod, mutant=0):
    depth, rgb, K, pose = _slanted_step_frame()
    e = _integrate(oracle_mod, mutant, "reproject", depth, rgb, K, pose)
    w = e["weight"]
    seen = w > 0
    if seen.sum() < 2000:
        return [f"only {int(seen.sum())} voxels received samples"]
    c, u, v = _project(_voxel_centres(e), K, pose)
    fails = []
    decided = seen & ~_near_boundary(u) & ~_near_boundary(v)
    pu = np.floor(u + 0.5).astype(np.int64)
    pv = np.floor(v + 0.5).astype(np.int64)
    inside = (pu >= 0) & (pu < W) & (pv >= 0) & (pv < H)
    if np.any(decided & ~inside):
        fails.append(f"{int(np.sum(decided & ~inside))} voxels with samples project outside")
    ok = decided & inside
    d = np.where(ok, depth[np.clip(pv, 0, H - 1), np.clip(pu, 0, W - 1)], np.nan).astype(np.float64)
    if np.any(ok & ~(d > 0)):
        fails.append(f"{int(np.sum(ok & ~(d > 0)))} voxels with samples project onto holes")
    ok &= d > 0
    sdf = d - c[..., 2]
    if np.any(ok & (sdf < -TRUNC - 1e-5)):
        fails.append(f"{int(np.sum(ok & (sdf < -TRUNC - 1e-5)))} voxels with samples lie more "
                     "than trunc behind the depth where they project")
    ok &= sdf >= -TRUNC + 1e-5
    mean = e["tsdf"][ok] / w[ok]
    want = np.minimum(1.0, sdf[ok] / TRUNC)
    if np.abs(mean - want).max() > 2e-5:
        fails.append(f"mean tsdf off the reprojected value by {np.abs(mean - want).max():.3g}")
    r = e["r"][ok] / w[ok]
    g = e["g"][ok] / w[ok]
    if np.abs(r - pu[ok] / W).max() > 1e-6 or np.abs(g - pv[ok] / H).max() > 1e-6:
        fails.append("mean colour is not the colour of the reprojected pixel")
    if ok.sum() < 1000:
        fails.append(f"only {int(ok.sum())} voxels checked")
    return fails


def pin_agrees_with_the_ray_test_on_a_plane(oracle_mod, mutant=0):
    D = 1.2031
    depth = np.full((H, W), D, np.float32)
    rgb = np.full((H, W, 3), 0.5, np.float32)
    K = np.array([60.0, 60.0, 31.5, 23.5], np.float32)
    pose = np.eye(4, dtype=np.float32)
    e_ray = _integrate(oracle_mod, 0, "ray", depth, rgb, K, pose)
    e_rep = _integrate(oracle_mod, mutant, "reproject", depth, rgb, K, pose)
    # compare voxel by voxel over the union of both block sets
    keys = {tuple(c): i for i, c in enumerate(e_ray["coords"])}
    fails = []
    n_inside = 0
    for i, cc in enumerate(e_rep["coords"]):
        if tuple(cc) not in keys:
            keys[tuple(cc)] = None
    for cc in keys:
        one = {"coords": np.array([cc], np.int32)}
        _, u, v = _project(_voxel_centres(one), K, pose)
        u, v = u[0], v[0]
        edge = (np.abs(u + 0.5) < 1e-3) | (np.abs(u + 0.5 - W) < 1e-3) | \
            (np.abs(v + 0.5) < 1e-3) | (np.abs(v + 0.5 - H) < 1e-3)
        inside = (u + 0.5 >= 0) & (u + 0.5 < W) & (v + 0.5 >= 0) & (v + 0.5 < H) & ~edge
        w_ray = np.zeros(512)
        w_rep = np.zeros(512)
        if keys[cc] is not None:
            w_ray = e_ray["weight"][keys[cc]]
        hit = np.flatnonzero(np.all(e_rep["coords"] == np.array(cc), axis=1))
        if len(hit):
            w_rep = e_rep["weight"][hit[0]]
        n_inside += int(np.sum(inside & (w_ray > 0)))
        if np.any(inside & (w_ray != w_rep)):
            fails.append(f"block {cc}: weights differ from the ray test inside the image")
        if np.any(~inside & ~edge & (w_rep > 0)):
            fails.append(f"block {cc}: samples added at voxels projecting outside the image")
        if len(fails) > 3:
            break
    if n_inside < 5000:
        fails.append(f"only {n_inside} voxels compared")
    return fails


PINS = [pin_values, pin_agrees_with_the_ray_test_on_a_plane]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_reprojection_passes_pin(oracle_mod, pin):
    assert pin(oracle_mod) == []


PLANTED_REPROJECT = {
    19: "projection rounded down instead of to the nearest pixel",
    20: "x and y of the projection swapped",
    21: "tested against the ray pixel's depth",
    22: "centre taken to the camera frame with R instead of R^T",
    23: "colour of the ray pixel instead of the reprojected one",
}


@pytest.mark.parametrize("mutant", sorted(PLANTED_REPROJECT), ids=lambda m: f"m{m}")
def test_planted_reprojection_mistakes_are_caught(oracle_mod, mutant):
    caught = []
    try:
        for pin in PINS:
            caught = pin(oracle_mod, mutant)
            if caught:
                break
    finally:
        path = oracle_mod.library_path(mutant)
        if os.path.exists(path):
            os.remove(path)
    assert caught, f"no pin rejects the planted mistake: {PLANTED_REPROJECT[mutant]}"


def test_ray_mode_is_unchanged_by_the_switch(oracle_mod):
    # selecting "ray" explicitly is the default test, sum for sum
    depth, rgb, K, pose = _slanted_step_frame()
    a = oracle_mod.OracleVolume(VOXEL, TRUNC)
    a.integrate(depth, rgb, K, pose)
    b = oracle_mod.OracleVolume(VOXEL, TRUNC)
    b.set_occlusion("ray")
    b.integrate(depth, rgb, K, pose)
    ea, eb = a.export(), b.export()
    for k in ("coords", "tsdf", "weight", "r", "g", "b"):
        np.testing.assert_array_equal(ea[k], eb[k])
    with pytest.raises(KeyError):
        b.set_occlusion("nearest")
