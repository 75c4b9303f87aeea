"""Seeded synthetic depth + colour frames for hash-blocked TSDF integration.

This module only makes inputs: analytic ray casting of spheres, axis-aligned
boxes, a plane and the inner walls of a room, camera trajectories, depth
noise, invalid pixels and colour.  It holds none of the integrate path's own
arithmetic (no band walk, no voxel or block indexing, no hashing).  Both the
CUDA path and the CPU oracle consume what it produces, so the two always see
bit-identical inputs.

Conventions shared by every frame:

* depth is float32 ``[H][W]`` in metres, the camera-frame z of the first
  surface hit along the pixel's ray; 0 marks an invalid pixel (no hit, or
  dropped on purpose);
* colour is float32 ``[H][W][3]`` in [0, 1);
* intrinsics are ``(fx, fy, cx, cy)`` with pixel centres at integer (u, v)
  and the camera looking down +z, x right, y down;
* a pose is a float32 4x4 row-major camera-to-world matrix [R | t].

The workloads are those of the scene families described for the hash-blocked
TSDF benchmark: a single sphere-before-plane frame at 160x120 and at 640x480,
a 100-frame orbit around 40 random primitives, and a 300-frame random walk in
a room with 400 primitives at 1280x720.  Every random draw comes from one
``numpy.random.Generator(PCG64(seed))`` per scene, in a fixed order.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
from typing import Optional

import numpy as np

SPHERE = 0
BOX = 1


@dataclasses.dataclass
class Frames:
    """A batch of frames plus the volume parameters the workload asks for."""

    name: str
    depth: np.ndarray            # float32 [n, H, W]
    rgb: np.ndarray              # float32 [n, H, W, 3]
    poses: np.ndarray            # float32 [n, 4, 4] camera -> world, row-major
    K: np.ndarray                # float32 [4]: fx, fy, cx, cy
    voxel_size: float
    trunc: float
    pool_capacity: int
    table_capacity: int          # 0 = library default (next power of two above 2x pool)
    seed: int

    @property
    def n_frames(self) -> int:
        return int(self.depth.shape[0])

    @property
    def height(self) -> int:
        return int(self.depth.shape[1])

    @property
    def width(self) -> int:
        return int(self.depth.shape[2])

    def subset(self, start: int, stop: int) -> "Frames":
        return dataclasses.replace(
            self, name=f"{self.name}[{start}:{stop}]",
            depth=self.depth[start:stop], rgb=self.rgb[start:stop],
            poses=self.poses[start:stop])


# ----------------------------------------------------------------------------
# Ray casting (the C helper in scene_raycast.c; double precision, rounded to
# float32 once, after noise).
# ----------------------------------------------------------------------------

_RAYCAST_LIB = None


def _raycast_lib():
    global _RAYCAST_LIB
    if _RAYCAST_LIB is None:
        from . import _build
        path = _build.scene_library_path()
        if not os.path.exists(path):
            _build.build_scene_library()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        lib.scene_raycast_frames.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, ctypes.c_int, ip, dp, dp,
            ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_double, dp]
        lib.scene_raycast_frames.restype = None
        _RAYCAST_LIB = lib
    return _RAYCAST_LIB


def raycast(prims, poses, K, width, height, plane_z: Optional[float] = None,
            room_half: Optional[float] = None) -> np.ndarray:
    """Camera-frame depth, float64 [n, H, W]; 0 where nothing is hit.

    ``prims`` is a list of (kind, centre[3], size[3]); for a sphere size[0] is
    the diameter, for a box size holds the edge lengths along x, y, z.
    ``plane_z`` adds the world plane z = plane_z; ``room_half`` adds the six
    inner walls of the cube [-room_half, room_half]^3.
    """
    lib = _raycast_lib()
    poses = np.ascontiguousarray(np.asarray(poses, dtype=np.float64).reshape(-1, 16))
    n = poses.shape[0]
    kinds = np.ascontiguousarray([p[0] for p in prims], dtype=np.int32)
    centres = np.ascontiguousarray([p[1] for p in prims], dtype=np.float64).reshape(-1, 3)
    sizes = np.ascontiguousarray([p[2] for p in prims], dtype=np.float64).reshape(-1, 3)
    Kd = np.ascontiguousarray(np.asarray(K, dtype=np.float64))
    out = np.empty((n, height, width), dtype=np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.scene_raycast_frames(
        n, width, height, Kd.ctypes.data_as(dp), poses.ctypes.data_as(dp), len(prims),
        kinds.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), centres.ctypes.data_as(dp),
        sizes.ctypes.data_as(dp), int(plane_z is not None), float(plane_z or 0.0),
        int(room_half is not None), float(room_half or 0.0), out.ctypes.data_as(dp))
    return out


# ----------------------------------------------------------------------------
# Poses
# ----------------------------------------------------------------------------

def look_at(position, target, up=(0.0, 1.0, 0.0)) -> np.ndarray:
    """Camera-to-world pose at ``position`` looking at ``target`` (y down)."""
    p = np.asarray(position, dtype=np.float64)
    f = np.asarray(target, dtype=np.float64) - p
    f /= np.linalg.norm(f)
    x = np.cross(f, np.asarray(up, dtype=np.float64))
    x /= np.linalg.norm(x)
    y = np.cross(f, x)
    T = np.eye(4)
    T[:3, 0], T[:3, 1], T[:3, 2], T[:3, 3] = x, y, f, p
    return T


def axis_angle(axis, angle) -> np.ndarray:
    """3x3 rotation by ``angle`` radians about the unit vector ``axis``."""
    a = np.asarray(axis, dtype=np.float64)
    a = a / np.linalg.norm(a)
    k = np.array([[0.0, -a[2], a[1]], [a[2], 0.0, -a[0]], [-a[1], a[0], 0.0]])
    return np.eye(3) + math.sin(angle) * k + (1.0 - math.cos(angle)) * (k @ k)


# ----------------------------------------------------------------------------
# Scene families
# ----------------------------------------------------------------------------

def _finish_depth(rng, depth64, noise_sigma, invalid_frac):
    d = depth64.copy()
    valid = d > 0.0
    if noise_sigma > 0.0:
        d = d + np.where(valid, rng.normal(0.0, noise_sigma, size=d.shape), 0.0)
        d = np.where(valid & (d > 0.0), d, 0.0)
    if invalid_frac > 0.0:
        n = d.size
        k = int(round(invalid_frac * n))
        drop = rng.choice(n, size=k, replace=False)
        d.reshape(-1)[drop] = 0.0
    return d.astype(np.float32)


def _render(rng, prims, poses, K, width, height, noise_sigma, invalid_frac=0.0,
            plane_z=None, room_half=None, frame_seeds=None):
    """Ray cast every pose, then draw colour and noise frame by frame: from
    ``rng`` in frame order, or, when ``frame_seeds`` is given, from a fresh
    generator per frame seeded with that frame's entry (so any range of frames
    can be rendered on its own)."""
    d64 = raycast(prims, poses, K, width, height, plane_z=plane_z, room_half=room_half)
    n = len(poses)
    depth = np.empty((n, height, width), dtype=np.float32)
    rgb = np.empty((n, height, width, 3), dtype=np.float32)
    for f in range(n):
        g = rng if frame_seeds is None else np.random.Generator(np.random.PCG64(frame_seeds[f]))
        rgb[f] = g.random((height, width, 3), dtype=np.float32)
        depth[f] = _finish_depth(g, d64[f], noise_sigma, invalid_frac)
    return depth, rgb


def _frame_range(n_frames, frames):
    if frames is None:
        return 0, n_frames
    start, stop = frames
    if not (0 <= start <= stop <= n_frames):
        raise ValueError(f"frame range {frames} outside [0, {n_frames}]")
    return start, stop


def sphere_plane(width=160, height=120, fx=131.25, fy=131.25, cx=None, cy=None,
                 noise_sigma=0.0, invalid_frac=0.0, seed=0, pose=None,
                 sphere_centre=(0.0, 0.0, 1.5), sphere_radius=0.5, plane_z=2.5):
    """One frame of a sphere in front of the world plane z = plane_z.

    Returns (depth float32 [H, W], rgb float32 [H, W, 3], pose float32 [4, 4],
    K float32 [4]).
    """
    cx = (width - 1) / 2.0 if cx is None else cx
    cy = (height - 1) / 2.0 if cy is None else cy
    K = np.array([fx, fy, cx, cy], dtype=np.float32)
    pose = np.eye(4) if pose is None else np.asarray(pose, dtype=np.float64)
    rng = np.random.Generator(np.random.PCG64(seed))
    prims = [(SPHERE, np.asarray(sphere_centre, dtype=np.float64),
              np.array([2.0 * sphere_radius] * 3))]
    depth, rgb = _render(rng, prims, [pose], K, width, height, noise_sigma,
                         invalid_frac, plane_z=plane_z)
    return depth[0], rgb[0], pose.astype(np.float32), K


def tiny_sphere_plane(seed=0) -> Frames:
    """160x120 noise-free sphere (r 0.5 m at z 1.5 m) before the plane z = 2.5 m.

    Voxel 2 cm, truncation 8 cm, pool 4096 blocks, table 16384 entries.
    """
    depth, rgb, pose, K = sphere_plane(160, 120, 131.25, 131.25, 79.5, 59.5, seed=seed)
    return Frames("tiny_sphere_plane_160x120", depth[None], rgb[None], pose[None], K,
                  0.02, 0.08, 4096, 16384, seed)


def vga_sphere_plane(seed=0) -> Frames:
    """640x480 sphere + plane, depth noise 2 mm, 10% of pixels invalid.

    Voxel 1 cm, truncation 4 cm, pool 2^16 blocks, default table size.
    """
    depth, rgb, pose, K = sphere_plane(640, 480, 525.0, 525.0, 319.5, 239.5,
                                       noise_sigma=0.002, invalid_frac=0.10, seed=seed)
    return Frames("vga_sphere_plane_640x480", depth[None], rgb[None], pose[None], K,
                  0.01, 0.04, 1 << 16, 0, seed)


def random_primitives(rng, n, lo, hi, size_lo=0.1, size_hi=0.8):
    """``n`` primitives, half spheres and half boxes, centres U[lo, hi]^3.

    A sphere's diameter and each box edge are U[size_lo, size_hi].
    """
    prims = []
    for i in range(n):
        kind = SPHERE if rng.random() < 0.5 else BOX
        centre = rng.uniform(lo, hi, size=3)
        if kind == SPHERE:
            s = rng.uniform(size_lo, size_hi)
            size = np.array([s, s, s])
        else:
            size = rng.uniform(size_lo, size_hi, size=3)
        prims.append((kind, centre, size))
    return prims


def orbit_trajectory(n_frames=100, seed=0, width=640, height=480,
                     voxel_size=0.005, trunc=0.02, pool_capacity=1 << 18,
                     table_capacity=0, frames=None) -> Frames:
    """40 random boxes/spheres in a 4 m cube, camera orbiting at 2.5 m.

    The camera circles the origin in the y = 0 plane, 3.6 degrees per frame,
    always looking at the origin.  Depth noise 2 mm; rays that hit nothing
    read 0.  ``frames=(start, stop)`` renders only that range of the
    trajectory (identical to the same frames of the full render).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    prims = random_primitives(rng, 40, -2.0, 2.0)
    K = np.array([525.0, 525.0, 319.5, 239.5], dtype=np.float32)
    start, stop = _frame_range(n_frames, frames)
    poses = []
    for f in range(start, stop):
        a = math.radians(3.6 * f)
        pos = (2.5 * math.sin(a), 0.0, 2.5 * math.cos(a))
        poses.append(look_at(pos, (0.0, 0.0, 0.0)))
    seeds = [[seed, 1, f] for f in range(start, stop)]
    depth, rgb = _render(rng, prims, poses, K, width, height, 0.002, frame_seeds=seeds)
    name = f"orbit_{n_frames}x{width}x{height}"
    if frames is not None:
        name += f"[{start}:{stop}]"
    return Frames(name, depth, rgb, np.asarray(poses, dtype=np.float32).reshape(-1, 4, 4), K,
                  voxel_size, trunc, pool_capacity, table_capacity, seed)


def _prim_bounds(kind, centre, size):
    """Bounding sphere (centre, radius) of a primitive."""
    if kind == SPHERE:
        return centre, 0.5 * size[0]
    return centre, 0.5 * float(np.linalg.norm(size))


def _inside_any(p, prims, clearance):
    for kind, centre, size in prims:
        bc, rho = _prim_bounds(kind, np.asarray(centre), np.asarray(size))
        if np.linalg.norm(p - bc) < rho + clearance:
            return True
    return False


def room_walk_poses(rng, prims, n_frames, room_half=4.0, margin=0.5,
                    step=0.02, turn_deg=1.0, clearance=0.1):
    """Random walk: each frame moves ``step`` m along a fresh random unit
    direction and turns ``turn_deg`` degrees about a fresh random unit axis.
    A move that would come within ``margin`` of a wall is reflected off it;
    a move into a primitive's bounding sphere is redrawn (at most 16 times,
    then the camera stays put for that frame)."""
    pos = np.zeros(3)
    for _ in range(1000):
        if not _inside_any(pos, prims, 0.3):
            break
        pos = rng.uniform(-room_half + margin, room_half - margin, size=3)
    R = axis_angle(rng.normal(size=3), rng.uniform(0.0, 2.0 * math.pi))
    poses = []
    lim = room_half - margin
    for f in range(n_frames):
        T = np.eye(4)
        T[:3, :3], T[:3, 3] = R, pos
        poses.append(T)
        for _ in range(16):
            dvec = rng.normal(size=3)
            dvec /= np.linalg.norm(dvec)
            cand = pos + step * dvec
            for a in range(3):
                if cand[a] > lim or cand[a] < -lim:
                    dvec[a] = -dvec[a]
            cand = pos + step * dvec
            if not _inside_any(cand, prims, clearance):
                pos = cand
                break
        R = R @ axis_angle(rng.normal(size=3), math.radians(turn_deg))
    return poses


def room_random_walk(n_frames=300, seed=0, width=1280, height=720,
                     voxel_size=0.004, trunc=0.016, pool_capacity=1 << 20,
                     table_capacity=1 << 21, n_prims=400, frames=None) -> Frames:
    """400 random boxes/spheres inside an 8 m room whose six inner walls are
    part of the scene; 1280x720 random-walk trajectory, depth noise 3 mm.
    ``frames=(start, stop)`` renders only that range of the trajectory
    (identical to the same frames of the full render)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    prims = random_primitives(rng, n_prims, -3.6, 3.6)
    K = np.array([920.0, 920.0, 639.5, 359.5], dtype=np.float32)
    poses = room_walk_poses(rng, prims, n_frames)
    start, stop = _frame_range(n_frames, frames)
    poses = poses[start:stop]
    seeds = [[seed, 2, f] for f in range(start, stop)]
    depth, rgb = _render(rng, prims, poses, K, width, height, 0.003, room_half=4.0,
                         frame_seeds=seeds)
    name = f"room_walk_{n_frames}x{width}x{height}"
    if frames is not None:
        name += f"[{start}:{stop}]"
    return Frames(name, depth, rgb, np.asarray(poses, dtype=np.float32).reshape(-1, 4, 4), K,
                  voxel_size, trunc, pool_capacity, table_capacity, seed)
