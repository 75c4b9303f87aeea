"""CPU oracle for hash-blocked TSDF integration -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the C-ABI library
and its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``tsdf_oracle.cpp`` (plain single-threaded C++,
``std::unordered_map`` keyed by block coordinate, double-precision sums); this
module compiles it with gcc (``-O2 -ffp-contract=off``, no fast-math) and wraps
it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

ORACLE_DIR = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(ORACLE_DIR, "tsdf_oracle.cpp")
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

COUNTER_NAMES = ("valid_points", "passing_samples", "accumulated", "missed_contributions",
                 "out_of_range_samples", "dropped_blocks", "bad_local_index")


def library_path(mutant: int = 0) -> str:
    if mutant == 0:
        return os.path.join(ORACLE_DIR, "liboracle.so")
    return os.path.join(tempfile.gettempdir(), f"tsdf_oracle_mutant_{mutant}_{os.getpid()}.so")


def build(force: bool = False, mutant: int = 0) -> str:
    """Compile the oracle (or a planted-mistake variant) and return its path."""
    out = library_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SOURCE)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++"] + CXXFLAGS + [f"-DORACLE_MUTANT={mutant}", "-o", tmp, SOURCE]
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if proc.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + " ".join(cmd) + "\n" + proc.stdout)
    os.replace(tmp, out)
    return out


_LIBS = {}


def _p(t):
    return ctypes.POINTER(t)


def load(mutant: int = 0):
    if mutant in _LIBS:
        return _LIBS[mutant]
    lib = ctypes.CDLL(build(mutant=mutant))
    f32p, f64p, i32p, u64p, i64p = (_p(ctypes.c_float), _p(ctypes.c_double), _p(ctypes.c_int32),
                                    _p(ctypes.c_uint64), _p(ctypes.c_longlong))
    sig = {
        "oracle_create": ([ctypes.c_float, ctypes.c_float, ctypes.c_longlong], ctypes.c_void_p),
        "oracle_destroy": ([ctypes.c_void_p], None),
        "oracle_keep_only": ([ctypes.c_void_p, i32p, ctypes.c_longlong], ctypes.c_int),
        "oracle_keep_partition": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int], ctypes.c_int),
        "oracle_walk": ([ctypes.c_void_p, f32p, f32p, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                         i32p, i32p], ctypes.c_int),
        "oracle_integrate": ([ctypes.c_void_p, f32p, f32p, ctypes.c_int, ctypes.c_int, f32p, f32p],
                             ctypes.c_int),
        "oracle_set_occlusion": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
        "oracle_block_count": ([ctypes.c_void_p], ctypes.c_longlong),
        "oracle_kept_count": ([ctypes.c_void_p], ctypes.c_longlong),
        "oracle_counters": ([ctypes.c_void_p, _p(ctypes.c_ulonglong)], None),
        "oracle_export_coords": ([ctypes.c_void_p, ctypes.c_longlong, i32p], ctypes.c_longlong),
        "oracle_export_sums": ([ctypes.c_void_p, ctypes.c_longlong, i32p, f64p, f64p, f64p, f64p,
                                f64p, f64p], ctypes.c_longlong),
        "oracle_pack_key": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, u64p], ctypes.c_int),
        "oracle_unpack_key": ([ctypes.c_uint64, i32p], ctypes.c_int),
        "oracle_hash_slot": ([ctypes.c_uint64, ctypes.c_uint64], ctypes.c_uint64),
        "oracle_probe_build": ([u64p, ctypes.c_longlong, ctypes.c_uint64, u64p, i64p, i64p],
                               ctypes.c_longlong),
        "oracle_clustered_coords": ([ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, i32p,
                                     ctypes.c_int32, ctypes.c_longlong, i32p], ctypes.c_longlong),
        "oracle_extract": ([ctypes.c_void_p, ctypes.c_longlong, f32p], ctypes.c_longlong),
        "oracle_set_block": ([ctypes.c_void_p, i32p, f64p, f64p, f64p, f64p, f64p], ctypes.c_int),
        "oracle_mutant_id": ([], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _LIBS[mutant] = lib
    return lib


def _ptr(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


class OracleVolume:
    """Plain CPU integrator: blocks in a hash map, sums in double.

    ``block_limit`` caps the number of blocks (pool exhaustion); negative means
    unlimited.  ``keep_only(coords)`` restricts the kept sums to a block subset
    (the block set and counters still cover every block).
    """

    def __init__(self, voxel_size: float, trunc: float, block_limit: int = -1, mutant: int = 0):
        self._lib = load(mutant)
        self._h = self._lib.oracle_create(float(voxel_size), float(trunc), int(block_limit))
        if not self._h:
            raise ValueError("invalid voxel size or truncation")
        self.voxel_size = float(voxel_size)
        self.trunc = float(trunc)

    def close(self):
        if self._h:
            self._lib.oracle_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def keep_only(self, coords) -> None:
        c = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 3))
        if self._lib.oracle_keep_only(self._h, _ptr(c, ctypes.c_int32), c.shape[0]) != 0:
            raise RuntimeError("keep_only must be called before the first integrate")

    def keep_partition(self, parts: int, part: int) -> None:
        """Keep sums only for blocks with (bx + by + bz) mod parts == part; the
        ``parts`` partitions are disjoint and cover every block."""
        if self._lib.oracle_keep_partition(self._h, int(parts), int(part)) != 0:
            raise RuntimeError("keep_partition must be called before the first integrate, "
                               "with 0 <= part < parts")

    def walk(self, K, pose, u: int, v: int, d: float):
        """The band walk of pixel (u, v) at depth d under the ray-depth test:
        (voxel indices int32 [S, 3], status int32 [S]: 0 pass, 1 occluded,
        2 out of range); empty arrays for an invalid depth."""
        K = np.ascontiguousarray(K, dtype=np.float32).reshape(4)
        pose = np.ascontiguousarray(pose, dtype=np.float32).reshape(16)
        S = 2 * int(round(self.trunc / self.voxel_size)) + 3
        ix = np.zeros((S, 3), np.int32)
        st = np.zeros(S, np.int32)
        n = self._lib.oracle_walk(self._h, _ptr(K, ctypes.c_float), _ptr(pose, ctypes.c_float),
                                  int(u), int(v), float(d), _ptr(ix, ctypes.c_int32),
                                  _ptr(st, ctypes.c_int32))
        return ix[:n], st[:n]

    def set_occlusion(self, mode: str) -> None:
        """Occlusion test of later integrations: "ray" (the ray pixel's depth,
        the default) or "reproject" (the depth where the voxel centre
        projects)."""
        if self._lib.oracle_set_occlusion(self._h, {"ray": 0, "reproject": 1}[mode]) != 0:
            raise ValueError(mode)

    def integrate(self, depth, rgb, K, pose) -> None:
        depth = np.ascontiguousarray(depth, dtype=np.float32)
        H, W = depth.shape
        rgb = np.ascontiguousarray(rgb, dtype=np.float32).reshape(H, W, 3)
        K = np.ascontiguousarray(K, dtype=np.float32).reshape(4)
        pose = np.ascontiguousarray(pose, dtype=np.float32).reshape(16)
        rc = self._lib.oracle_integrate(self._h, _ptr(depth, ctypes.c_float),
                                        _ptr(rgb, ctypes.c_float), W, H,
                                        _ptr(K, ctypes.c_float), _ptr(pose, ctypes.c_float))
        if rc != 0:
            raise ValueError("oracle_integrate rejected its arguments")

    def integrate_frames(self, frames, start: int = 0, stop=None) -> None:
        stop = frames.n_frames if stop is None else stop
        for f in range(start, stop):
            self.integrate(frames.depth[f], frames.rgb[f], frames.K, frames.poses[f])

    def block_count(self) -> int:
        return int(self._lib.oracle_block_count(self._h))

    def counters(self) -> dict:
        out = (ctypes.c_ulonglong * len(COUNTER_NAMES))()
        self._lib.oracle_counters(self._h, out)
        return {k: int(out[i]) for i, k in enumerate(COUNTER_NAMES)}

    def coords(self) -> np.ndarray:
        n = self.block_count()
        c = np.zeros((n, 3), dtype=np.int32)
        got = self._lib.oracle_export_coords(self._h, n, _ptr(c, ctypes.c_int32))
        return c[:got]

    def export(self) -> dict:
        """Kept blocks sorted by (x, y, z): coords int32 [n, 3] and float64
        [n, 512] arrays tsdf, weight, r, g, b, tsdf_abs."""
        n = int(self._lib.oracle_kept_count(self._h))
        c = np.zeros((n, 3), dtype=np.int32)
        arrs = {k: np.zeros((n, 512), dtype=np.float64)
                for k in ("tsdf", "weight", "r", "g", "b", "tsdf_abs")}
        got = self._lib.oracle_export_sums(
            self._h, n, _ptr(c, ctypes.c_int32),
            *[_ptr(arrs[k], ctypes.c_double) for k in ("tsdf", "weight", "r", "g", "b", "tsdf_abs")])
        assert got == n
        out = {"coords": c}
        out.update(arrs)
        return out

    def extract(self) -> np.ndarray:
        """Marching-tetrahedra triangles of the mean TSDF's zero level set,
        float32 [n, 3, 3] (triangle, vertex, xyz), in the oracle's cell order."""
        n = int(self._lib.oracle_extract(self._h, 0, None))
        out = np.zeros((n, 3, 3), dtype=np.float32)
        if n:
            got = self._lib.oracle_extract(self._h, n, _ptr(out, ctypes.c_float))
            assert got == n
        return out

    def set_block(self, coord, tsdf, weight, r=None, g=None, b=None) -> None:
        """Create or overwrite block `coord` with the given [512] sums."""
        c = np.ascontiguousarray(np.asarray(coord, dtype=np.int32).reshape(3))
        arrs = [None if a is None else np.ascontiguousarray(np.asarray(a, np.float64).reshape(512))
                for a in (tsdf, weight, r, g, b)]
        ptrs = [None if a is None else _ptr(a, ctypes.c_double) for a in arrs]
        self._lib.oracle_set_block(self._h, _ptr(c, ctypes.c_int32), *ptrs)


# ----------------------------------------------------------------------------
# Key packing, slot hash, sequential linear probing (table-structure reference)
# ----------------------------------------------------------------------------

def pack_key(x: int, y: int, z: int, mutant: int = 0):
    """Packed 64-bit key of a block coordinate, or None when out of range."""
    k = ctypes.c_uint64()
    rc = load(mutant).oracle_pack_key(int(x), int(y), int(z), ctypes.byref(k))
    return None if rc != 0 else int(k.value)


def unpack_key(key: int, mutant: int = 0):
    out = (ctypes.c_int32 * 3)()
    rc = load(mutant).oracle_unpack_key(ctypes.c_uint64(key), out)
    return None if rc != 0 else (out[0], out[1], out[2])


def hash_slot(key: int, table_size: int, mutant: int = 0) -> int:
    return int(load(mutant).oracle_hash_slot(ctypes.c_uint64(key), ctypes.c_uint64(table_size)))


def pack_keys(coords) -> np.ndarray:
    """Vectorised pack_key (raises on an out-of-range coordinate)."""
    c = np.asarray(coords, dtype=np.int32).reshape(-1, 3)
    lib = load()
    out = np.empty(c.shape[0], dtype=np.uint64)
    k = ctypes.c_uint64()
    for i in range(c.shape[0]):
        if lib.oracle_pack_key(int(c[i, 0]), int(c[i, 1]), int(c[i, 2]), ctypes.byref(k)) != 0:
            raise ValueError(f"coordinate {tuple(c[i])} out of range")
        out[i] = k.value
    return out


def probe_build(keys, table_size: int):
    """Sequential linear-probing inserts.  Returns (table[T] uint64 with
    all-ones for empty, probe_len[n] int64, total_displacement, distinct)."""
    k = np.ascontiguousarray(np.asarray(keys, dtype=np.uint64))
    table = np.empty(table_size, dtype=np.uint64)
    plen = np.empty(k.size, dtype=np.int64)
    disp = ctypes.c_longlong()
    distinct = load().oracle_probe_build(_ptr(k, ctypes.c_uint64), k.size, table_size,
                                         _ptr(table, ctypes.c_uint64),
                                         _ptr(plen, ctypes.c_longlong), ctypes.byref(disp))
    if distinct < 0:
        raise RuntimeError("table full")
    return table, plen, int(disp.value), int(distinct)


def clustered_coords(table_size: int, window_start: int, window_len: int, origin, side: int,
                     want: int) -> np.ndarray:
    """Block coordinates whose home slot falls in a window of the table."""
    o = np.ascontiguousarray(np.asarray(origin, dtype=np.int32).reshape(3))
    out = np.zeros((want, 3), dtype=np.int32)
    n = load().oracle_clustered_coords(table_size, window_start, window_len,
                                       _ptr(o, ctypes.c_int32), side, want,
                                       _ptr(out, ctypes.c_int32))
    return out[:n]
