"""Independent checks used to pin the CPU oracle (and, on the GPU, the CUDA
path): a dense-grid brute-force integrator written with numpy, and analytic
surface-crossing extraction for closed-form scenes."""
from __future__ import annotations

import os

import numpy as np

F32 = np.float32


def voxel_indices_of_blocks(coords: np.ndarray) -> np.ndarray:
    """Voxel indices [n, 512, 3] of the voxels of each block, x fastest
    inside a block (j = lx + 8 ly + 64 lz)."""
    j = np.arange(512)
    local = np.stack([j % 8, (j // 8) % 8, j // 64], axis=1)
    return coords[:, None, :].astype(np.int64) * 8 + local[None, :, :]


def dense_bruteforce(depth, rgb, K, pose, voxel, trunc):
    """Dense-grid integration of one frame, vectorised over pixels.

    Walks the same band samples as the method (float32, one rounding per
    operation, in the same order: per pixel the observed point in voxel
    units and the world direction, per sample their combination) but
    accumulates straight into a dense
    voxel grid with np.add.at in float64, with no blocks and no hash map.
    Returns (origin[3] int, dict of dense float64 arrays weight/tsdf/r/g/b,
    n_passing).
    """
    H, W = depth.shape
    fx, fy, cx, cy = (F32(k) for k in K)
    pose = np.asarray(pose, dtype=F32)
    R = pose[:3, :3]
    t = pose[:3, 3]
    v = F32(voxel)
    tau = F32(trunc)
    k = int(round(float(trunc) / float(voxel)))
    uu, vv = np.meshgrid(np.arange(W, dtype=F32), np.arange(H, dtype=F32))
    d = np.asarray(depth, dtype=F32)
    valid = np.isfinite(d) & (d > F32(0))
    u = uu[valid]
    vy = vv[valid]
    d = d[valid]
    col = np.asarray(rgb, dtype=F32).reshape(H, W, 3)[valid]
    xn = (u - cx) / fx
    yn = (vy - cy) / fy
    px, py, pz = xn * d, yn * d, d
    ln = np.sqrt((xn * xn + yn * yn) + F32(1))
    dx, dy, dz = xn / ln, yn / ln, F32(1) / ln
    # the observed point in voxel units and the world direction, per pixel
    pv = [(((R[a, 0] * px + R[a, 1] * py) + R[a, 2] * pz) + t[a]) / v for a in range(3)]
    e = [(R[a, 0] * dx + R[a, 1] * dy) + R[a, 2] * dz for a in range(3)]
    idx_l, val_l, col_l = [], [], []
    for i in range(-k, k + 1):
        q = [np.floor(pv[a] + F32(i) * e[a]) for a in range(3)]
        ok = np.ones(q[0].shape, dtype=bool)
        for qa in q:
            ok &= (qa >= F32(-8388608.0)) & (qa <= F32(8388607.0))
        q = [np.where(ok, qa, F32(0)) for qa in q]
        ii = [qa.astype(np.int64) for qa in q]
        c = [(ii[a].astype(F32) + F32(0.5)) * v - t[a] for a in range(3)]
        zc = (R[0, 2] * c[0] + R[1, 2] * c[1]) + R[2, 2] * c[2]
        sdf = d - zc
        ok &= (zc > F32(0)) & (sdf >= -tau)
        tsdf = np.minimum(F32(1), sdf / tau)
        idx_l.append(np.stack([a[ok] for a in ii], axis=1))
        val_l.append(tsdf[ok])
        col_l.append(col[ok])
    idx = np.concatenate(idx_l)
    val = np.concatenate(val_l).astype(np.float64)
    colr = np.concatenate(col_l).astype(np.float64)
    if idx.shape[0] == 0:
        return np.zeros(3, dtype=np.int64), {}, 0
    lo = idx.min(axis=0)
    hi = idx.max(axis=0)
    shape = tuple((hi - lo + 1).tolist())
    rel = tuple((idx - lo).T)
    out = {}
    for name, vals in (("weight", np.ones_like(val)), ("tsdf", val), ("r", colr[:, 0]),
                       ("g", colr[:, 1]), ("b", colr[:, 2])):
        a = np.zeros(shape, dtype=np.float64)
        np.add.at(a, rel, vals)
        out[name] = a
    return lo, out, int(idx.shape[0])


def blocks_to_dense(coords, arrays: dict, lo, shape):
    """Scatter block arrays ([n, 512] each) into dense grids of `shape`
    starting at voxel index `lo`; voxels outside the grid must be empty
    (weight 0), else ValueError."""
    vox = voxel_indices_of_blocks(np.asarray(coords)).reshape(-1, 3) - np.asarray(lo)[None, :]
    inside = np.all((vox >= 0) & (vox < np.asarray(shape)[None, :]), axis=1)
    w = np.asarray(arrays["weight"]).reshape(-1)
    if np.any(w[~inside] != 0):
        raise ValueError("weight outside the brute-force grid")
    out = {}
    for name, a in arrays.items():
        g = np.zeros(shape, dtype=np.float64)
        flat = np.asarray(a, dtype=np.float64).reshape(-1)
        g[tuple(vox[inside].T)] = flat[inside]
        out[name] = g
    return out


def mean_tsdf_grid(coords, tsdf, weight):
    """Dense mean-tsdf grid (nan where weight is 0) and its voxel origin."""
    vox = voxel_indices_of_blocks(np.asarray(coords)).reshape(-1, 3)
    lo = vox.min(axis=0)
    shape = tuple((vox.max(axis=0) - lo + 1).tolist())
    T = np.zeros(shape)
    Wt = np.zeros(shape)
    rel = tuple((vox - lo).T)
    T[rel] = np.asarray(tsdf, dtype=np.float64).reshape(-1)
    Wt[rel] = np.asarray(weight, dtype=np.float64).reshape(-1)
    with np.errstate(invalid="ignore", divide="ignore"):
        mean = np.where(Wt > 0, T / np.where(Wt > 0, Wt, 1), np.nan)
    return mean, lo


def zero_crossings(mean, lo, voxel, axis, direction):
    """World points where the mean tsdf changes from > 0 to <= 0 between two
    observed voxels adjacent along `axis`, stepping in `direction` (+1/-1),
    by linear interpolation between the voxel centres."""
    m = np.moveaxis(mean, axis, 0)
    if direction < 0:
        m = m[::-1]
    a, b = m[:-1], m[1:]
    hit = np.isfinite(a) & np.isfinite(b) & (a > 0) & (b <= 0)
    k, *rest = np.nonzero(hit)
    frac = a[hit] / (a[hit] - b[hit])
    n_along = mean.shape[axis]
    if direction < 0:
        pos_along = (n_along - 1 - k) - frac          # index along axis, moving down
    else:
        pos_along = k + frac
    other = [r.astype(np.float64) for r in rest]
    idx = [None, None, None]
    oth_axes = [ax for ax in range(3) if ax != axis]
    idx[axis] = pos_along
    for ax, r in zip(oth_axes, other):
        idx[ax] = r
    pts = np.stack(idx, axis=1) + np.asarray(lo)[None, :] + 0.5
    return pts * voxel


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SPLITMIX64_GAMMA = 0x9E3779B97F4A7C15


def splitmix64_vectors():
    """(input, output) pairs of the SplitMix64 output mix from its published
    output sequence (tests/golden/splitmix64_seed1234567.txt): output k of
    seed s is the mix of the state s + k * gamma (mod 2^64)."""
    out = []
    with open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            seed, k, value = (int(v) for v in line.split())
            out.append(((seed + k * SPLITMIX64_GAMMA) % (1 << 64), value))
    return out
