"""Pins for the CPU oracle: checks that do not trust the oracle itself.

Each pin is a function returning a list of failure messages, so the same
checks run (a) against the real oracle, where they must all pass, and
(b) against throw-away builds of the oracle with one planted mistake each,
where at least one pin must fail (test_planted_mistakes_are_caught).

Pins used:
* worked examples with closed-form answers, derived by hand from the
  geometry (a fronto-parallel plane seen along the optical axis, and an
  oblique 3-4-5 ray), under an identity pose and under an axis-permuting
  rotation with a translation into negative coordinates;
* the analytic sphere of the correctness section of "What Irregularity
  Costs" (surface recovered within a quarter voxel), plus the plane behind
  it, under an identity and an oblique camera pose;
* dense-grid brute force (tests/helpers.py): the same per-sample walk
  accumulated straight into a dense array with numpy, no blocks, no map;
* invariants: every block receives a contribution; the weight sum equals the
  number of passing samples; the valid-point count equals the number of
  finite positive depths;
* pool-limit accounting.
"""
import math

import numpy as np
import pytest

import helpers
from hash_blocked_tsdf_gb300 import scenes

VOXEL = 0.02
TRUNC = 0.08


# ----------------------------------------------------------------------------
# Worked examples (closed form)
# ----------------------------------------------------------------------------

# A 5x1 image with fx = fy = 4, cx = 1, cy = 0.  Pixel u = 1 looks straight
# down the optical axis (xn = 0).  Pixel u = 4 has xn = (4 - 1) / 4 = 0.75,
# so its ray (0.75, 0, 1) has length 1.25 and unit direction (0.6, 0, 0.8):
# a 3-4-5 triangle.  The other pixels are invalid (depth 0).  Voxel 2 cm,
# truncation 8 cm: 9 samples at offsets -8, -6, ..., +8 cm along the unit ray.
WE_K = np.array([4.0, 4.0, 1.0, 0.0], dtype=np.float32)
WE_RGB = np.array([[[0.9, 0.9, 0.9], [0.25, 0.5, 0.75], [0.9, 0.9, 0.9], [0.9, 0.9, 0.9],
                    [0.125, 0.375, 0.625]]], dtype=np.float32)
RGB_AXIS = (0.25, 0.5, 0.75)
RGB_OBLIQUE = (0.125, 0.375, 0.625)

# Identity pose, axis depth 1.015 m, oblique depth 1.005 m.
#
# Axis pixel: samples at z = 1.015 + 0.02 (i - 4), i = 0..8, i.e. at
# 46.75 + i voxels -> voxels (0, 0, 46 + i).  Centres z_c = 0.93 + 0.02 i, so
# sdf = 1.015 - z_c = 0.085 - 0.02 i and tsdf = sdf / 0.08:
# 1.0625 (clamped to 1), 0.8125, 0.5625, 0.3125, 0.0625, -0.1875, -0.4375,
# -0.6875, -0.9375 (the last, sdf = -0.075, still passes sdf >= -0.08).
#
# Oblique pixel: p = (0.75 * 1.005, 0, 1.005); sample j = i - 4 sits at
# x = 37.6875 + 0.6 j and z = 50.25 + 0.8 j voxels:
#   j  : -4     -3     -2     -1     0      1      2      3      4
#   ix : 35     35     36     37     37     38     38     39     40
#   iz : 47     47     48     49     50     51     51     52     53
# so samples j = -4, -3 share a voxel, as do j = 1, 2 (weight 2 each).
# sdf = 1.005 - (iz + 0.5) * 0.02 depends only on iz:
#   iz 47: 0.055 -> 0.6875   48: 0.035 -> 0.4375   49: 0.015 -> 0.1875
#   iz 50: -0.005 -> -0.0625 51: -0.025 -> -0.3125 52: -0.045 -> -0.5625
#   iz 53: -0.065 -> -0.8125
WE_IDENTITY_DEPTH = np.array([[0.0, 1.015, 0.0, 0.0, 1.005]], dtype=np.float32)
WE_IDENTITY_POSE = np.eye(4, dtype=np.float32)
WE_IDENTITY_EXPECT = {}
for _i, _t in enumerate([1.0, 0.8125, 0.5625, 0.3125, 0.0625, -0.1875, -0.4375, -0.6875,
                         -0.9375]):
    WE_IDENTITY_EXPECT[(0, 0, 46 + _i)] = (1, _t, RGB_AXIS)
for _v, _w, _t in [((35, 0, 47), 2, 2 * 0.6875), ((36, 0, 48), 1, 0.4375),
                   ((37, 0, 49), 1, 0.1875), ((37, 0, 50), 1, -0.0625),
                   ((38, 0, 51), 2, 2 * -0.3125), ((39, 0, 52), 1, -0.5625),
                   ((40, 0, 53), 1, -0.8125)]:
    WE_IDENTITY_EXPECT[_v] = (_w, _t, RGB_OBLIQUE)
WE_IDENTITY_BLOCKS = {(0, 0, 5), (0, 0, 6), (4, 0, 5), (4, 0, 6), (5, 0, 6)}

# Rotated pose: R maps camera x -> world y, camera y -> world z, camera
# z -> world x (R = [[0,0,1],[1,0,0],[0,1,0]], not symmetric), and
# t = (-1.0, 0.25, -0.13).  A camera point s lands at world
# (s_z - 1.0, s_x + 0.25, s_y - 0.13), so world x crosses zero inside the
# band (negative voxel and block indices).  The centre's camera depth is its
# world x + 1.0.  Both depths are 1.005 m.
#
# Axis pixel: world x = 0.005 + 0.02 j -> ix = j (0.25 voxel past each
# boundary), iy = floor(12.5) = 12, iz = floor(-6.5) = -7.  z_c = 1.01 + 0.02 j,
# sdf = -0.005 - 0.02 j: j = -4..3 give 0.9375, 0.6875, 0.4375, 0.1875,
# -0.0625, -0.3125, -0.5625, -0.8125; j = 4 has sdf = -0.085 < -0.08 and is
# dropped by the occlusion test.
#
# Oblique pixel: world x = 0.005 + 0.016 j -> 0.25 + 0.8 j voxels, world
# y = 0.75375 + 0.012 j + 0.25 -> 50.1875 + 0.6 j voxels:
#   j  : -4     -3     -2     -1     0      1      2      3      4
#   ix : -3     -3     -2     -1     0      1      1      2      3
#   iy : 47     48     48     49     50     50     51     51     52
# all nine voxels distinct; sdf = 1.005 - ((ix + 0.5) * 0.02 + 1.0).
WE_ROT_DEPTH = np.array([[0.0, 1.005, 0.0, 0.0, 1.005]], dtype=np.float32)
WE_ROT_POSE = np.array([[0, 0, 1, -1.0], [1, 0, 0, 0.25], [0, 1, 0, -0.13], [0, 0, 0, 1]],
                       dtype=np.float32)
WE_ROT_EXPECT = {}
for _j, _t in zip(range(-4, 4), [0.9375, 0.6875, 0.4375, 0.1875, -0.0625, -0.3125, -0.5625,
                                 -0.8125]):
    WE_ROT_EXPECT[(_j, 12, -7)] = (1, _t, RGB_AXIS)
_SDF_OF_IX = {-3: 0.6875, -2: 0.4375, -1: 0.1875, 0: -0.0625, 1: -0.3125, 2: -0.5625, 3: -0.8125}
for _ix, _iy in [(-3, 47), (-3, 48), (-2, 48), (-1, 49), (0, 50), (1, 50), (1, 51), (2, 51),
                 (3, 52)]:
    WE_ROT_EXPECT[(_ix, _iy, -7)] = (1, _SDF_OF_IX[_ix], RGB_OBLIQUE)
WE_ROT_BLOCKS = {(-1, 1, -1), (0, 1, -1), (-1, 5, -1), (-1, 6, -1), (0, 6, -1)}


def _voxel_dict(export):
    """{voxel index: (weight, tsdf sum, (r, g, b) sums)} of observed voxels."""
    vox = helpers.voxel_indices_of_blocks(export["coords"])
    out = {}
    w = export["weight"]
    for bi in range(vox.shape[0]):
        for j in np.nonzero(w[bi])[0]:
            key = tuple(int(c) for c in vox[bi, j])
            out[key] = (w[bi, j], export["tsdf"][bi, j],
                        (export["r"][bi, j], export["g"][bi, j], export["b"][bi, j]))
    return out


def _check_worked(oracle_mod, mutant, depth, pose, expect, blocks):
    fails = []
    o = oracle_mod.OracleVolume(VOXEL, TRUNC, mutant=mutant)
    o.integrate(depth, WE_RGB, WE_K, pose)
    e = o.export()
    got_blocks = {tuple(int(v) for v in c) for c in e["coords"]}
    if got_blocks != blocks:
        fails.append(f"blocks {sorted(got_blocks)} != {sorted(blocks)}")
    got = _voxel_dict(e)
    if set(got) != set(expect):
        fails.append(f"voxels differ: missing {sorted(set(expect) - set(got))}, "
                     f"extra {sorted(set(got) - set(expect))}")
    for k in set(got) & set(expect):
        w, t, rgb = got[k]
        ew, et, ergb = expect[k]
        if w != ew:
            fails.append(f"weight at {k}: {w} != {ew}")
        if abs(t - et) > 1e-5:
            fails.append(f"tsdf at {k}: {t} != {et}")
        for c in range(3):
            if abs(rgb[c] - ew * ergb[c]) > 1e-6:
                fails.append(f"colour {c} at {k}: {rgb[c]} != {ew * ergb[c]}")
    return fails


def pin_worked_identity(oracle_mod, mutant=0):
    return _check_worked(oracle_mod, mutant, WE_IDENTITY_DEPTH, WE_IDENTITY_POSE,
                         WE_IDENTITY_EXPECT, WE_IDENTITY_BLOCKS)


def pin_worked_rotated(oracle_mod, mutant=0):
    return _check_worked(oracle_mod, mutant, WE_ROT_DEPTH, WE_ROT_POSE, WE_ROT_EXPECT,
                         WE_ROT_BLOCKS)


# ----------------------------------------------------------------------------
# Analytic sphere and plane
# ----------------------------------------------------------------------------

SPHERE_C = np.array([0.0, 0.0, 1.5])
SPHERE_R = 0.5


def oblique_sphere_frames():
    """The sphere seen from 1.6 m along an oblique direction, 160x120."""
    a = np.array([0.35, -0.25, 1.0])
    a /= np.linalg.norm(a)
    pose = scenes.look_at(SPHERE_C - 1.6 * a, SPHERE_C)
    depth, rgb, pose32, K = scenes.sphere_plane(160, 120, 131.25, 131.25, 79.5, 59.5,
                                                seed=3, pose=pose)
    return scenes.Frames("oblique_sphere", depth[None], rgb[None], pose32[None], K,
                         VOXEL, TRUNC, 4096, 16384, 3)


def _sphere_and_plane_errors(export, pose, voxel, plane=True):
    mean, lo = helpers.mean_tsdf_grid(export["coords"], export["tsdf"], export["weight"])
    view = pose[:3, 2].astype(np.float64)
    axis = int(np.argmax(np.abs(view)))
    pts = helpers.zero_crossings(mean, lo, voxel, axis, int(np.sign(view[axis])))
    q = pts - SPHERE_C
    dist = np.linalg.norm(q, axis=1)
    cam = pose[:3, 3].astype(np.float64)
    to_c = (SPHERE_C - cam) / np.linalg.norm(SPHERE_C - cam)
    front = (q / dist[:, None]) @ (-to_c) > math.cos(math.radians(45.0))
    sel = (np.abs(dist - SPHERE_R) < 0.1) & front
    s_err = dist[sel] - SPHERE_R
    p_err = np.array([])
    if plane:
        lateral = np.linalg.norm(pts[:, :2], axis=1)
        psel = (np.abs(pts[:, 2] - 2.5) < 0.1) & (lateral > 0.95)
        p_err = pts[psel, 2] - 2.5
    return s_err, p_err


def pin_sphere(oracle_mod, mutant=0):
    fails = []
    for frames, plane in ((scenes.tiny_sphere_plane(), True), (oblique_sphere_frames(), False)):
        o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc, mutant=mutant)
        o.integrate_frames(frames)
        e = o.export()
        if e["coords"].shape[0] == 0:
            fails.append(f"{frames.name}: no blocks")
            continue
        s_err, p_err = _sphere_and_plane_errors(e, frames.poses[0], frames.voxel_size, plane)
        quarter = frames.voxel_size / 4.0
        if s_err.size < 300:
            fails.append(f"{frames.name}: only {s_err.size} sphere crossings")
        elif np.abs(s_err).max() > quarter:
            fails.append(f"{frames.name}: sphere radius error {np.abs(s_err).max():.5f} m "
                         f"> v/4")
        if plane:
            if p_err.size < 3000:
                fails.append(f"{frames.name}: only {p_err.size} plane crossings")
            elif np.abs(p_err).max() > quarter:
                fails.append(f"{frames.name}: plane error {np.abs(p_err).max():.5f} m > v/4")
    return fails


# ----------------------------------------------------------------------------
# Dense-grid brute force and invariants
# ----------------------------------------------------------------------------

def _frames_for_dense():
    return [scenes.tiny_sphere_plane(), oblique_sphere_frames(), scenes.vga_sphere_plane()]


def pin_dense(oracle_mod, mutant=0):
    fails = []
    for frames in _frames_for_dense():
        o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc, mutant=mutant)
        o.integrate_frames(frames)
        e = o.export()
        lo, dense, n_pass = helpers.dense_bruteforce(frames.depth[0], frames.rgb[0], frames.K,
                                                     frames.poses[0], frames.voxel_size,
                                                     frames.trunc)
        shape = dense["weight"].shape
        try:
            mine = helpers.blocks_to_dense(e["coords"], {k: e[k] for k in
                                                         ("weight", "tsdf", "r", "g", "b")},
                                           lo, shape)
        except ValueError as exc:
            fails.append(f"{frames.name}: {exc}")
            continue
        if not np.array_equal(mine["weight"], dense["weight"]):
            fails.append(f"{frames.name}: weights differ in "
                         f"{int((mine['weight'] != dense['weight']).sum())} voxels")
            continue
        for k in ("tsdf", "r", "g", "b"):
            diff = np.abs(mine[k] - dense[k]).max()
            if diff > 1e-9:
                fails.append(f"{frames.name}: {k} differs by {diff}")
        # every block touched by a passing sample, and no other block
        vox = np.argwhere(dense["weight"] > 0) + lo
        want = {tuple(int(c) for c in b) for b in np.unique(np.floor_divide(vox, 8), axis=0)}
        got = {tuple(int(c) for c in b) for b in o.coords()}
        if want != got:
            fails.append(f"{frames.name}: block set differs ({len(got)} vs {len(want)})")
    return fails


def pin_invariants(oracle_mod, mutant=0):
    fails = []
    for frames in (scenes.tiny_sphere_plane(), scenes.vga_sphere_plane()):
        o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc, mutant=mutant)
        o.integrate_frames(frames)
        e = o.export()
        c = o.counters()
        wsum = e["weight"].sum()
        per_block = e["weight"].sum(axis=1)
        n_valid = int(np.sum(np.isfinite(frames.depth) & (frames.depth > 0)))
        if c["valid_points"] != n_valid:
            fails.append(f"{frames.name}: valid points {c['valid_points']} != {n_valid}")
        if wsum != c["passing_samples"] or c["accumulated"] != c["passing_samples"]:
            fails.append(f"{frames.name}: weight sum {wsum} vs passing {c['passing_samples']}")
        if np.any(per_block <= 0):
            fails.append(f"{frames.name}: {int(np.sum(per_block <= 0))} blocks never observed")
        for k in ("missed_contributions", "out_of_range_samples", "dropped_blocks",
                  "bad_local_index"):
            if c[k] != 0:
                fails.append(f"{frames.name}: {k} = {c[k]}")
        if c["passing_samples"] > 9 * c["valid_points"]:
            fails.append(f"{frames.name}: more than 9 samples per point")
        if np.any(np.abs(e["tsdf"]) > e["weight"] + 1e-9):
            fails.append(f"{frames.name}: |tsdf mean| > 1")
    return fails


# ----------------------------------------------------------------------------
# The walk against a float64 evaluation in another operation order
# ----------------------------------------------------------------------------

def _walk_float64(depth, K, pose, voxel, trunc, pixels):
    """Band samples of the given pixels evaluated in float64, in the
    camera-then-world order of the plain reading of the walk: sample
    i = 0 .. 2k at p + (i voxel - trunc) dir in camera coordinates, moved to
    the world with [R | t], divided by the voxel edge and floored; the
    occlusion test at the voxel centre, z_c = (R^T (centre - t))_z,
    sdf = d - z_c, pass iff z_c > 0 and sdf >= -trunc.  Returns the voxels
    [n, S, 3], pass flags [n, S], each coordinate's distance (in voxels)
    from the nearest voxel boundary [n, S, 3], and the distance (in voxels)
    of the test's quantities from their thresholds [n, S]."""
    fx, fy, cx, cy = (float(x) for x in K)
    R = pose[:3, :3].astype(np.float64)
    t = pose[:3, 3].astype(np.float64)
    v = float(np.float32(voxel))
    tau = float(np.float32(trunc))
    k = int(round(tau / v))
    u = pixels[:, 0].astype(np.float64)
    vv = pixels[:, 1].astype(np.float64)
    d = depth[pixels[:, 1], pixels[:, 0]].astype(np.float64)
    ray = np.stack([(u - cx) / fx, (vv - cy) / fy, np.ones_like(u)], axis=1)
    p = ray * d[:, None]
    dirn = ray / np.linalg.norm(ray, axis=1, keepdims=True)
    off = np.arange(2 * k + 1, dtype=np.float64) * v - tau
    cam = p[:, None, :] + off[None, :, None] * dirn[:, None, :]
    world = cam @ R.T + t
    q = world / v
    vox = np.floor(q)
    edge = np.abs(q - np.round(q))
    centre = (vox + 0.5) * v
    zc = (centre - t) @ R[:, 2]
    sdf = d[:, None] - zc
    passes = (zc > 0) & (sdf >= -tau)
    test_margin = np.minimum(np.abs(sdf + tau), np.abs(zc)) / v
    return vox.astype(np.int64), passes, edge, test_margin


def _walk_frames():
    """(name, depth, K, pose, voxel, trunc, pixel step) cases: the worked
    examples, the sphere frames, and subsamples of the noisy 640x480 frame
    and of a room-walk frame (a general rotation)."""
    cases = []
    for name, depth, pose in (("worked identity", WE_IDENTITY_DEPTH, WE_IDENTITY_POSE),
                              ("worked rotated", WE_ROT_DEPTH, WE_ROT_POSE)):
        cases.append((name, depth, WE_K, pose, VOXEL, TRUNC, 0))
    for frames, step in ((scenes.tiny_sphere_plane(), 1), (oblique_sphere_frames(), 1),
                         (scenes.vga_sphere_plane(), 7),
                         (scenes.room_random_walk(n_frames=300, frames=(0, 1)), 41)):
        cases.append((frames.name, frames.depth[0], frames.K, frames.poses[0],
                      frames.voxel_size, frames.trunc, step))
    return cases


def pin_walk_float64(oracle_mod, mutant=0):
    """Every band sample of the oracle against the float64 evaluation above.
    Per axis, where the float64 coordinate lies more than 1e-4 voxel from a
    voxel boundary, the oracle's voxel index must equal its floor; where all
    three do and the occlusion test's quantities are 1e-4 voxel clear of
    their thresholds, the oracle must take the same decision; every pixel
    must have 2k + 1 samples.  The oracle evaluates the walk in voxel units
    with float32 operations in another order, so this does not share its
    arithmetic; float32 rounding moves a sample by far less than 1e-4 voxel
    at these coordinates.  (Coordinates on a boundary, such as the zero x of
    a ray along the optical axis, are skipped on that axis.)"""
    fails = []
    margin = 1e-4
    for name, depth, K, pose, voxel, trunc, step in _walk_frames():
        vv, uu = np.nonzero(np.isfinite(depth) & (depth > 0))
        pix = np.stack([uu, vv], axis=1)
        if step:
            pix = pix[::step]
        vox64, pass64, edge, tmargin = _walk_float64(depth, K, pose, voxel, trunc, pix)
        o = oracle_mod.OracleVolume(voxel, trunc, mutant=mutant)
        S = vox64.shape[1]
        clear = edge > margin
        axes = whole = decided = 0
        bad = []
        for n, (u, v) in enumerate(pix):
            ix, st = o.walk(K, pose, int(u), int(v), float(depth[v, u]))
            if ix.shape[0] != S:
                bad.append(f"pixel ({u}, {v}): {ix.shape[0]} samples, not {S}")
                continue
            for i in range(S):
                if st[i] == 2:
                    bad.append(f"pixel ({u}, {v}) sample {i}: out of range")
                    continue
                for a in range(3):
                    if clear[n, i, a]:
                        axes += 1
                        if ix[i, a] != vox64[n, i, a]:
                            bad.append(f"pixel ({u}, {v}) sample {i} axis {a}: voxel "
                                       f"{ix[i, a]} != {vox64[n, i, a]}")
                if clear[n, i].all():
                    whole += 1
                    if tmargin[n, i] > margin:
                        decided += 1
                        if (st[i] == 0) != bool(pass64[n, i]):
                            bad.append(f"pixel ({u}, {v}) sample {i}: test {st[i]} != "
                                       f"{'pass' if pass64[n, i] else 'occluded'}")
            if len(bad) > 5:
                break
        o.close()
        total = pix.shape[0] * S
        if bad:
            fails.append(f"{name}: " + "; ".join(bad[:3]))
        elif axes < total:
            fails.append(f"{name}: only {axes} coordinates of {total} samples clear of "
                         f"voxel boundaries")
        elif step and (whole < 0.8 * total or decided < 0.8 * total):
            fails.append(f"{name}: only {whole} / {decided} of {total} samples compared "
                         f"whole / decided")
    return fails


# cheapest first: the planted-mistake test stops at the first pin that fails
ALL_PINS = [pin_worked_identity, pin_worked_rotated, pin_invariants, pin_walk_float64,
            pin_sphere, pin_dense]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(oracle_mod, pin):
    assert pin(oracle_mod) == []


PLANTED = {
    1: "signed distance taken at the ray sample instead of the voxel centre",
    2: "signed distance with its sign flipped",
    3: "voxel corner used instead of the centre",
    4: "world-to-camera rotation not transposed",
    5: "voxel order inside a block x-slowest",
    6: "occlusion test without the truncation side",
    7: "tsdf not clamped at +1",
    8: "voxel index truncated toward zero instead of floored",
    9: "block index truncated toward zero instead of floored",
    10: "red and blue channels swapped",
    11: "weight 2 per observation",
    12: "allocate pass ignores the occlusion test",
    13: "band one voxel too wide",
    14: "ray direction not normalised",
    25: "ray direction moved to the world by R^T instead of R",
    26: "camera position added after the division by the voxel edge",
}


@pytest.mark.parametrize("mutant", sorted(PLANTED), ids=lambda m: f"m{m}")
def test_planted_mistakes_are_caught(oracle_mod, mutant):
    import os
    caught = {}
    try:
        for pin in ALL_PINS:
            f = pin(oracle_mod, mutant)
            if f:
                caught[pin.__name__] = f[0]
                break
    finally:
        path = oracle_mod.library_path(mutant)
        if os.path.exists(path):
            os.remove(path)
    assert caught, f"no pin rejects the planted mistake: {PLANTED[mutant]}"


# ----------------------------------------------------------------------------
# Counter semantics
# ----------------------------------------------------------------------------

def test_pool_limit_accounting(oracle_mod):
    frames = scenes.vga_sphere_plane()
    full = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    full.integrate_frames(frames)
    B = full.block_count()
    limit = B // 2
    o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc, block_limit=limit)
    o.integrate_frames(frames)
    c = o.counters()
    e = o.export()
    assert o.block_count() == limit
    assert c["dropped_blocks"] == B - limit
    assert c["missed_contributions"] > 0
    assert c["accumulated"] + c["missed_contributions"] == c["passing_samples"]
    assert e["weight"].sum() == c["accumulated"]
    assert c["passing_samples"] == full.counters()["passing_samples"]


def test_out_of_range_samples_are_counted_and_skipped(oracle_mod):
    frames = scenes.tiny_sphere_plane()
    far = np.eye(4, dtype=np.float32)
    far[0, 3] = 1.0e6            # 5e7 voxels of 2 cm: beyond the 2^23-voxel key range
    o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    o.integrate(frames.depth[0], frames.rgb[0], frames.K, far)
    c = o.counters()
    assert o.block_count() == 0
    assert c["passing_samples"] == 0
    assert c["out_of_range_samples"] == 9 * c["valid_points"] > 0


def test_invalid_depths_are_skipped(oracle_mod):
    frames = scenes.tiny_sphere_plane()
    d = frames.depth[0].copy()
    d[0, :10] = np.nan
    d[1, :10] = np.inf
    d[2, :10] = -1.0
    d[3, :10] = 0.0
    o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    o.integrate(d, frames.rgb[0], frames.K, frames.poses[0])
    assert o.counters()["valid_points"] == d.size - 40


def test_empty_frame(oracle_mod):
    o = oracle_mod.OracleVolume(VOXEL, TRUNC)
    o.integrate(np.zeros((7, 9), np.float32), np.zeros((7, 9, 3), np.float32), WE_K,
                np.eye(4, dtype=np.float32))
    assert o.block_count() == 0 and o.counters()["valid_points"] == 0


def test_keep_only_restricts_sums_not_the_block_set(oracle_mod):
    frames = scenes.vga_sphere_plane()
    full = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    full.integrate_frames(frames)
    ef = full.export()
    pick = ef["coords"][::97]
    part = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    part.keep_only(pick)
    part.integrate_frames(frames)
    ep = part.export()
    assert part.block_count() == full.block_count()
    assert np.array_equal(ep["coords"], pick)
    rows = np.arange(0, ef["coords"].shape[0], 97)
    for k in ("tsdf", "weight", "r", "g", "b", "tsdf_abs"):
        assert np.array_equal(ep[k], ef[k][rows])


def test_keep_partition_splits_the_volume_into_disjoint_parts(oracle_mod):
    """keep_partition(parts, part) keeps the sums of the blocks with
    (bx + by + bz) mod parts == part: the parts are disjoint, together they
    are the whole volume, and each part's sums equal the unrestricted run's
    (the filter only selects blocks; the arithmetic is the same)."""
    frames = scenes.tiny_sphere_plane()
    full = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    full.integrate_frames(frames)
    ef = full.export()
    parts = 3
    seen = []
    for p in range(parts):
        o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
        o.keep_partition(parts, p)
        o.integrate_frames(frames)
        e = o.export()
        assert o.block_count() == full.block_count()
        assert o.counters() == full.counters()
        assert np.all(np.mod(e["coords"].astype(np.int64).sum(axis=1), parts) == p)
        rows = np.nonzero(np.mod(ef["coords"].astype(np.int64).sum(axis=1), parts) == p)[0]
        assert np.array_equal(e["coords"], ef["coords"][rows])
        for k in ("tsdf", "weight", "r", "g", "b", "tsdf_abs"):
            assert np.array_equal(e[k], ef[k][rows])
        seen.append(e["coords"])
    assert sum(s.shape[0] for s in seen) == ef["coords"].shape[0]
    assert min(s.shape[0] for s in seen) > 0
    with pytest.raises(RuntimeError):
        oracle_mod.OracleVolume(frames.voxel_size, frames.trunc).keep_partition(3, 3)
