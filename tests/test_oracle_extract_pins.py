"""Pins of the oracle's surface extraction (marching tetrahedra over the mean
TSDF), checked against what geometry fixes, not against the oracle itself:

- a linear field: every vertex lies on its zero plane, and the triangles'
  total area equals the plane's cross-section of the cells, computed by
  brute force (polygon of the plane cut by each cube's 12 edges);
- a signed-distance sphere written into blocks: a closed, watertight,
  manifold mesh (every edge in exactly two triangles, Euler characteristic
  2) whose vertices lie on the sphere to within the interpolation error;
- a fronto-parallel plane integrated from a constant-depth frame: every
  vertex at the plane's depth (the mean tsdf is linear across the surface);
- the analytic sphere scene (design section; correctness section, analytic
  tier): the visible cap within a quarter voxel of the true sphere.

Planted mistakes in the extraction are compiled and each must be rejected.
"""
import os

import numpy as np
import pytest

from hash_blocked_tsdf_gb300 import scenes

VOXEL = 0.01


def _region_field(oracle_mod, mutant, fn, blocks, weights):
    """An oracle volume whose blocks [0, blocks)^3 hold sums w * fn(centre)."""
    o = oracle_mod.OracleVolume(VOXEL, 4 * VOXEL, mutant=mutant)
    j = np.arange(512)
    local = np.stack([j % 8, (j // 8) % 8, j // 64], axis=1)
    for bx in range(blocks):
        for by in range(blocks):
            for bz in range(blocks):
                idx = local + 8 * np.array([bx, by, bz])
                centres = (idx + 0.5) * VOXEL
                w = weights(idx)
                o.set_block((bx, by, bz), w * fn(centres), w)
    return o


def _area(tris):
    a = tris[:, 1].astype(np.float64) - tris[:, 0]
    b = tris[:, 2].astype(np.float64) - tris[:, 0]
    return 0.5 * np.linalg.norm(np.cross(a, b), axis=1)


def _section_area(n, d, lo, hi):
    """Area of {x : n.x = d} inside the box [lo, hi] (brute force)."""
    corners = np.array([[lo[0] if (k & 1) == 0 else hi[0], lo[1] if (k & 2) == 0 else hi[1],
                         lo[2] if (k & 4) == 0 else hi[2]] for k in range(8)])
    g = corners @ n - d
    pts = []
    for a in range(8):
        for ax in range(3):
            b = a | (1 << ax)
            if b == a:
                continue
            if (g[a] < 0) != (g[b] < 0):
                t = g[a] / (g[a] - g[b])
                pts.append(corners[a] + t * (corners[b] - corners[a]))
    if len(pts) < 3:
        return 0.0
    pts = np.array(pts)
    c = pts.mean(axis=0)
    u = np.cross(n, [1.0, 0.0, 0.0] if abs(n[0]) < 0.9 else [0.0, 1.0, 0.0])
    u /= np.linalg.norm(u)
    w = np.cross(n, u)
    ang = np.arctan2((pts - c) @ w, (pts - c) @ u)
    p2 = np.stack([(pts - c) @ u, (pts - c) @ w], axis=1)[np.argsort(ang)]
    return 0.5 * abs(np.sum(p2[:, 0] * np.roll(p2[:, 1], -1) - np.roll(p2[:, 0], -1) * p2[:, 1]))


def pin_linear_field(oracle_mod, mutant=0):
    rng = np.random.default_rng(11)
    n = rng.normal(size=3)
    n /= np.linalg.norm(n)
    x0 = np.array([0.081, 0.077, 0.085]) + rng.uniform(-0.002, 0.002, 3)
    o = _region_field(oracle_mod, mutant, lambda p: (p - x0) @ n, 2,
                      lambda idx: rng.integers(1, 6, size=len(idx)).astype(np.float64))
    tris = o.extract()
    fails = []
    if len(tris) == 0:
        return ["no triangles from a plane through the region"]
    off = np.abs((tris.reshape(-1, 3).astype(np.float64) - x0) @ n)
    if off.max() > 1e-5:
        fails.append(f"vertex {off.max():.3g} m off the zero plane")
    want = 0.0
    for i in range(15):
        for j in range(15):
            for k in range(15):
                lo = (np.array([i, j, k]) + 0.5) * VOXEL
                want += _section_area(n, n @ x0, lo, lo + VOXEL)
    got = _area(tris).sum()
    if abs(got - want) > 1e-4 * want:
        fails.append(f"triangle area {got:.6g} against the plane's cross-section {want:.6g}")
    return fails


def pin_closed_sphere(oracle_mod, mutant=0):
    # (centre and radius chosen so that no voxel centre lies on the sphere:
    # a corner value of exactly 0 collapses edges into that corner)
    c = np.array([12.31, 11.83, 12.07]) * VOXEL
    R = 7.29 * VOXEL
    rng = np.random.default_rng(12)
    o = _region_field(oracle_mod, mutant, lambda p: np.linalg.norm(p - c, axis=1) - R, 3,
                      lambda idx: rng.integers(1, 4, size=len(idx)).astype(np.float64))
    tris = o.extract()
    fails = []
    if len(tris) == 0:
        return ["no triangles from a sphere inside the region"]
    v = tris.reshape(-1, 3).astype(np.float64)
    err = np.abs(np.linalg.norm(v - c, axis=1) - R)
    # linear interpolation of a distance field along an edge of length L
    # errs by at most L^2 / (8 R); the longest tetrahedron edge is sqrt(3) voxels
    if err.max() > 3 * VOXEL ** 2 / (8 * R) * 1.05:
        fails.append(f"vertex {err.max() / VOXEL:.3f} voxels off the sphere")
    # merge identical vertices; a closed manifold has every edge in exactly
    # two triangles and Euler characteristic V - E + F = 2
    keys, inv = np.unique(tris.reshape(-1, 3), axis=0, return_inverse=True)
    ids = inv.reshape(-1, 3)
    edges = np.sort(np.concatenate([ids[:, [0, 1]], ids[:, [1, 2]], ids[:, [2, 0]]]), axis=1)
    ue, counts = np.unique(edges, axis=0, return_counts=True)
    if not np.all(counts == 2):
        fails.append(f"{int(np.sum(counts != 2))} edges not shared by exactly two triangles")
    chi = len(keys) - len(ue) + len(tris)
    if chi != 2:
        fails.append(f"Euler characteristic {chi}, not 2")
    return fails


def pin_flat_plane(oracle_mod, mutant=0):
    D = 1.2031
    depth = np.full((48, 64), D, np.float32)
    rgb = np.full((48, 64, 3), 0.5, np.float32)
    K = np.array([400.0, 400.0, 31.5, 23.5], np.float32)    # 3 mm pixels: every voxel seen
    o = oracle_mod.OracleVolume(VOXEL, 4 * VOXEL, mutant=mutant)
    o.integrate(depth, rgb, K, np.eye(4, dtype=np.float32))
    tris = o.extract()
    if len(tris) < 100:
        return [f"only {len(tris)} triangles from a plane filling the view"]
    dz = np.abs(tris[..., 2].astype(np.float64) - D)
    return [f"vertex {dz.max():.3g} m off the plane"] if dz.max() > 1e-5 else []


def pin_sphere_scene(oracle_mod, mutant=0):
    f = scenes.tiny_sphere_plane()
    o = oracle_mod.OracleVolume(f.voxel_size, f.trunc, mutant=mutant)
    o.integrate_frames(f)
    v = o.extract().reshape(-1, 3).astype(np.float64)
    fails = []
    c = np.array([0.0, 0.0, 1.5])
    rel = v - c
    nr = np.linalg.norm(rel, axis=1)
    cap = (-rel[:, 2] / nr > 0.7) & (np.abs(nr - 0.5) < 0.1)      # within ~45 degrees of the view
    if cap.sum() < 1000:
        fails.append(f"only {int(cap.sum())} vertices on the visible cap")
    elif np.abs(nr[cap] - 0.5).max() > f.voxel_size / 4:
        fails.append(f"cap vertex {np.abs(nr[cap] - 0.5).max():.4f} m off the sphere")
    far = (np.abs(v[:, 2] - 2.5) < 0.1) & (np.linalg.norm(v[:, :2], axis=1) > 1.2)
    if far.sum() < 1000 or np.abs(v[far, 2] - 2.5).max() > 1e-5:
        fails.append("plane vertices away from the sphere are not at z = 2.5")
    return fails


PINS = [pin_linear_field, pin_closed_sphere, pin_flat_plane, pin_sphere_scene]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_extraction_passes_pin(oracle_mod, pin):
    assert pin(oracle_mod) == []


PLANTED_EXTRACT = {
    15: "interpolation measured from the wrong end of the edge",
    16: "a tetrahedron set that does not tile the cube",
    17: "sums not divided by the weight",
    18: "corner values fetched with x and y swapped",
}


@pytest.mark.parametrize("mutant", sorted(PLANTED_EXTRACT), ids=lambda m: f"m{m}")
def test_planted_extraction_mistakes_are_caught(oracle_mod, mutant):
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
    assert caught, f"no pin rejects the planted mistake: {PLANTED_EXTRACT[mutant]}"
