"""Python binding of libtsdf.so (the C ABI in include/tsdf.h).

Argument marshalling only: every step of the integrate path runs in the
library's CUDA kernels.  Tensors are passed by device pointer
(``tensor.data_ptr()``) together with the caller's current CUDA stream;
PyTorch provides the device memory and the streams, nothing else.  There is
no fallback: if the library is missing, loading it raises.

Functions carry the C names (``tsdf_create``, ``tsdf_integrate``, ...);
``TsdfVolume`` wraps them for convenience.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import _build

PROBE_HIST_BINS = 32
EMPTY_KEY = 0xFFFFFFFFFFFFFFFF
INDEX_PENDING = 0xFFFFFFFF
INDEX_FAILED = 0xFFFFFFFE

ERROR_NAMES = {0: "TSDF_OK", -1: "TSDF_ERR_ARG", -2: "TSDF_ERR_CUDA", -3: "TSDF_ERR_OOM"}


class TsdfError(RuntimeError):
    def __init__(self, code: int, fn: str, msg: str):
        super().__init__(f"{fn} failed with {ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class tsdf_info(ctypes.Structure):
    _fields_ = [("pool_capacity", ctypes.c_uint32), ("table_capacity", ctypes.c_uint32),
                ("voxel_size", ctypes.c_float), ("trunc", ctypes.c_float),
                ("band_samples", ctypes.c_int32), ("device", ctypes.c_int32),
                ("fixed_divisor_fast_path", ctypes.c_int32),
                ("max_frames_per_launch", ctypes.c_int32), ("pool_layout", ctypes.c_int32),
                ("voxel_division_fast_path", ctypes.c_int32)]


class tsdf_pool_view(ctypes.Structure):
    _fields_ = [("tsdf", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("r", ctypes.c_void_p),
                ("g", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("pool_capacity", ctypes.c_uint32), ("stride", ctypes.c_uint32)]


class tsdf_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "blocks_allocated", "pool_exhausted", "probe_overflow", "missed_contributions",
        "out_of_range_samples", "valid_points", "voxel_updates", "probe_inserts",
        "probe_steps", "probe_max")] + [("probe_hist", ctypes.c_uint64 * PROBE_HIST_BINS),
                                         ("publish_timeouts", ctypes.c_uint64)]


_VP = ctypes.c_void_p
_I = ctypes.c_int
_U32 = ctypes.c_uint32
_F = ctypes.c_float
_FP = ctypes.POINTER(ctypes.c_float)

SIGNATURES = {
    "tsdf_create": ([_U32, _F, _F, ctypes.POINTER(_VP)], _I),
    "tsdf_create_ex": ([_U32, _U32, _F, _F, ctypes.POINTER(_VP)], _I),
    "tsdf_destroy": ([_VP], _I),
    "tsdf_get_info": ([_VP, ctypes.POINTER(tsdf_info)], _I),
    "tsdf_get_pool": ([_VP, ctypes.POINTER(tsdf_pool_view)], _I),
    "tsdf_reset": ([_VP, _VP], _I),
    "tsdf_integrate": ([_VP, _VP, _VP, _I, _I, _FP, _FP, _VP], _I),
    "tsdf_allocate": ([_VP, _VP, _I, _I, _FP, _FP, _VP], _I),
    "tsdf_update": ([_VP, _VP, _VP, _I, _I, _FP, _FP, _VP], _I),
    "tsdf_integrate_batch": ([_VP, _I, _VP, _VP, _I, _I, _FP, _FP, _VP], _I),
    "tsdf_integrate_batch_host": ([_VP, _I, _VP, _VP, _I, _I, _FP, _FP, _VP], _I),
    "tsdf_allocate_batch": ([_VP, _I, _VP, _I, _I, _FP, _FP, _VP], _I),
    "tsdf_update_batch": ([_VP, _I, _VP, _VP, _I, _I, _FP, _FP, _VP], _I),
    "tsdf_allocate_blocks": ([_VP, _VP, _U32, _VP], _I),
    "tsdf_block_count": ([_VP, _VP, ctypes.POINTER(_U32)], _I),
    "tsdf_export_blocks": ([_VP, _VP, _U32, _U32, _VP, _VP, _VP, _VP, _VP, _VP], _I),
    "tsdf_export_table": ([_VP, _VP, _U32, _VP, _VP], _I),
    "tsdf_extract_triangles": ([_VP, _VP, _VP, ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64)],
                               _I),
    "tsdf_import_blocks": ([_VP, _VP, _U32, _VP, _VP, _VP, _VP, _VP, _VP], _I),
    "tsdf_export_block_coords_noalloc": ([_VP, _VP, _U32, _U32, _VP], _I),
    "tsdf_get_stats": ([_VP, _VP, ctypes.POINTER(tsdf_stats)], _I),
    "tsdf_clear_stats": ([_VP, _VP], _I),
    "tsdf_set_instrumentation": ([_VP, _I], _I),
    "tsdf_set_update_kernel": ([_VP, _I], _I),
    "tsdf_set_occlusion": ([_VP, _I], _I),
    "tsdf_set_pool_layout": ([_VP, _I], _I),
    "tsdf_last_error": ([], ctypes.c_char_p),
}

_LIB = None


def library_path() -> str:
    return _build.tsdf_library_path()


def load_library():
    """Load libtsdf.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libtsdf.so not found at {path}: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = lib
    return lib


def _check(rc: int, fn: str):
    if rc != 0:
        msg = load_library().tsdf_last_error().decode("utf-8", "replace")
        raise TsdfError(rc, fn, msg)


def _floats(values, n: int):
    a = np.ascontiguousarray(np.asarray(values, dtype=np.float32).reshape(-1))
    if a.size != n:
        raise ValueError(f"expected {n} floats, got {a.size}")
    return a, a.ctypes.data_as(_FP)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t, dtype, name, shape_tail=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape_tail is not None and tuple(t.shape[-len(shape_tail):]) != tuple(shape_tail):
        raise ValueError(f"{name} has shape {tuple(t.shape)}")
    return t.data_ptr()


# ----------------------------------------------------------------------------
# C-named functions
# ----------------------------------------------------------------------------

def tsdf_create(pool_capacity: int, voxel_size: float, trunc: float, table_capacity: int = 0):
    h = _VP()
    lib = load_library()
    if table_capacity:
        rc = lib.tsdf_create_ex(pool_capacity, table_capacity, voxel_size, trunc, ctypes.byref(h))
    else:
        rc = lib.tsdf_create(pool_capacity, voxel_size, trunc, ctypes.byref(h))
    _check(rc, "tsdf_create")
    return h


def tsdf_destroy(h) -> None:
    _check(load_library().tsdf_destroy(h), "tsdf_destroy")


def tsdf_get_info(h) -> dict:
    info = tsdf_info()
    _check(load_library().tsdf_get_info(h, ctypes.byref(info)), "tsdf_get_info")
    return {k: getattr(info, k) for k, _ in tsdf_info._fields_}


def tsdf_get_pool(h) -> dict:
    """Device pointers (ints) of the five pool sums.  Voxel v = 512 b + j
    (block b, voxel j) has its tsdf, weight, r and g sums at float index
    stride * v from the respective pointer (interleaved records, stride 4)
    and its blue sum at float index v from b."""
    v = tsdf_pool_view()
    _check(load_library().tsdf_get_pool(h, ctypes.byref(v)), "tsdf_get_pool")
    return {"tsdf": v.tsdf, "weight": v.weight, "r": v.r, "g": v.g, "b": v.b,
            "pool_capacity": v.pool_capacity, "stride": v.stride}


tsdf_pool_arrays = tsdf_get_pool


def tsdf_reset(h, stream=None) -> None:
    _check(load_library().tsdf_reset(h, _stream_ptr(stream)), "tsdf_reset")


def tsdf_integrate(h, depth, rgb, K, pose, stream=None) -> None:
    import torch
    H, W = depth.shape[-2], depth.shape[-1]
    d = _dev(depth, torch.float32, "depth")
    c = _dev(rgb, torch.float32, "rgb", (H, W, 3))
    k, kp = _floats(K, 4)
    p, pp = _floats(pose, 16)
    _check(load_library().tsdf_integrate(h, d, c, W, H, kp, pp, _stream_ptr(stream)),
           "tsdf_integrate")


def tsdf_allocate(h, depth, K, pose, stream=None) -> None:
    import torch
    H, W = depth.shape[-2], depth.shape[-1]
    d = _dev(depth, torch.float32, "depth")
    k, kp = _floats(K, 4)
    p, pp = _floats(pose, 16)
    _check(load_library().tsdf_allocate(h, d, W, H, kp, pp, _stream_ptr(stream)),
           "tsdf_allocate")


def tsdf_update(h, depth, rgb, K, pose, stream=None) -> None:
    import torch
    H, W = depth.shape[-2], depth.shape[-1]
    d = _dev(depth, torch.float32, "depth")
    c = _dev(rgb, torch.float32, "rgb", (H, W, 3))
    k, kp = _floats(K, 4)
    p, pp = _floats(pose, 16)
    _check(load_library().tsdf_update(h, d, c, W, H, kp, pp, _stream_ptr(stream)),
           "tsdf_update")


def tsdf_integrate_batch(h, depth, rgb, K, poses, stream=None) -> None:
    import torch
    n, H, W = depth.shape
    d = _dev(depth, torch.float32, "depth")
    c = _dev(rgb, torch.float32, "rgb", (n, H, W, 3))
    k, kp = _floats(K, 4)
    p, pp = _floats(poses, 16 * n)
    _check(load_library().tsdf_integrate_batch(h, n, d, c, W, H, kp, pp, _stream_ptr(stream)),
           "tsdf_integrate_batch")


def tsdf_allocate_batch(h, depth, K, poses, stream=None) -> None:
    import torch
    n, H, W = depth.shape
    d = _dev(depth, torch.float32, "depth")
    k, kp = _floats(K, 4)
    p, pp = _floats(poses, 16 * n)
    _check(load_library().tsdf_allocate_batch(h, n, d, W, H, kp, pp, _stream_ptr(stream)),
           "tsdf_allocate_batch")


def tsdf_update_batch(h, depth, rgb, K, poses, stream=None) -> None:
    import torch
    n, H, W = depth.shape
    d = _dev(depth, torch.float32, "depth")
    c = _dev(rgb, torch.float32, "rgb", (n, H, W, 3))
    k, kp = _floats(K, 4)
    p, pp = _floats(poses, 16 * n)
    _check(load_library().tsdf_update_batch(h, n, d, c, W, H, kp, pp, _stream_ptr(stream)),
           "tsdf_update_batch")


def tsdf_integrate_batch_host(h, depth, rgb, K, poses, stream=None) -> None:
    """depth / rgb: host arrays (numpy, or CPU torch tensors, ideally pinned)."""
    n, H, W = depth.shape
    dp = _host_ptr(depth, (n, H, W), "depth")
    cp = _host_ptr(rgb, (n, H, W, 3), "rgb")
    k, kp = _floats(K, 4)
    p, pp = _floats(poses, 16 * n)
    _check(load_library().tsdf_integrate_batch_host(h, n, dp, cp, W, H, kp, pp,
                                                    _stream_ptr(stream)),
           "tsdf_integrate_batch_host")


def _host_ptr(a, shape, name) -> int:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            if a.is_cuda or a.dtype != torch.float32 or not a.is_contiguous():
                raise TypeError(f"{name} must be a contiguous float32 CPU tensor")
            if tuple(a.shape) != tuple(shape):
                raise ValueError(f"{name} has shape {tuple(a.shape)}")
            return a.data_ptr()
    except ImportError:
        pass
    if not (isinstance(a, np.ndarray) and a.dtype == np.float32 and a.flags.c_contiguous):
        raise TypeError(f"{name} must be a contiguous float32 array")
    if a.shape != tuple(shape):
        raise ValueError(f"{name} has shape {a.shape}")
    return a.ctypes.data


def tsdf_allocate_blocks(h, coords, stream=None) -> None:
    import torch
    c = _dev(coords, torch.int32, "coords", (3,))
    _check(load_library().tsdf_allocate_blocks(h, c, coords.shape[0], _stream_ptr(stream)),
           "tsdf_allocate_blocks")


def tsdf_block_count(h, stream=None) -> int:
    out = _U32()
    _check(load_library().tsdf_block_count(h, _stream_ptr(stream), ctypes.byref(out)),
           "tsdf_block_count")
    return int(out.value)


def tsdf_export_blocks(h, first: int = 0, count: Optional[int] = None, stream=None,
                       fields=("coords", "tsdf", "weight", "r", "g", "b")) -> dict:
    if count is None:
        count = tsdf_block_count(h, stream) - first
    out = {}
    ptrs = []
    for f in ("coords", "tsdf", "weight", "r", "g", "b"):
        if f in fields:
            a = (np.zeros((count, 3), np.int32) if f == "coords"
                 else np.zeros((count, 512), np.float32))
            out[f] = a
            ptrs.append(a.ctypes.data)
        else:
            ptrs.append(None)
    _check(load_library().tsdf_export_blocks(h, _stream_ptr(stream), first, count, *ptrs),
           "tsdf_export_blocks")
    return out


NOALLOC_MAX_BLOCKS = 65536


def tsdf_export_block_coords_noalloc(h, first: int, count: int, stream=None) -> np.ndarray:
    """Block coordinates of pool blocks [first, first + count), int32 [count, 3],
    through the library's built-in scratch array: no device memory is
    allocated (for callers whose device memory is spoken for).  count must not
    exceed NOALLOC_MAX_BLOCKS."""
    out = np.zeros((count, 3), np.int32)
    _check(load_library().tsdf_export_block_coords_noalloc(h, _stream_ptr(stream), first, count,
                                                           out.ctypes.data),
           "tsdf_export_block_coords_noalloc")
    return out


def tsdf_extract_triangles(h, stream=None, capacity=None):
    """Marching-tetrahedra triangles of the mean TSDF's zero level set, as a
    CUDA float32 tensor [n, 3, 3] (triangle, vertex, xyz; order unspecified).
    Without `capacity` the library counts first and the buffer is sized to
    fit; with it, at most `capacity` are returned."""
    import torch
    lib = load_library()
    n = ctypes.c_uint64()
    sp = _stream_ptr(stream)
    if capacity is None:
        _check(lib.tsdf_extract_triangles(h, sp, None, 0, ctypes.byref(n)), "tsdf_extract_triangles")
        capacity = int(n.value)
    out = torch.empty((max(capacity, 1), 3, 3), dtype=torch.float32, device="cuda")
    _check(lib.tsdf_extract_triangles(h, sp, out.data_ptr(), capacity, ctypes.byref(n)),
           "tsdf_extract_triangles")
    return out[:min(capacity, int(n.value))]


def tsdf_import_blocks(h, coords, tsdf, weight, r, g, b, stream=None) -> None:
    """Set blocks from host arrays: coords int32 [n, 3] (distinct), and the
    five float32 [n, 512] arrays."""
    c = np.ascontiguousarray(np.asarray(coords, np.int32).reshape(-1, 3))
    n = c.shape[0]
    arrs = [np.ascontiguousarray(np.asarray(a, np.float32).reshape(n, 512))
            for a in (tsdf, weight, r, g, b)]
    _check(load_library().tsdf_import_blocks(h, _stream_ptr(stream), n, c.ctypes.data,
                                             *[a.ctypes.data for a in arrs]),
           "tsdf_import_blocks")


def tsdf_export_table(h, stream=None):
    T = tsdf_get_info(h)["table_capacity"]
    keys = np.zeros(T, np.uint64)
    idx = np.zeros(T, np.uint32)
    _check(load_library().tsdf_export_table(h, _stream_ptr(stream), T, keys.ctypes.data,
                                            idx.ctypes.data), "tsdf_export_table")
    return keys, idx


def tsdf_get_stats(h, stream=None) -> dict:
    st = tsdf_stats()
    _check(load_library().tsdf_get_stats(h, _stream_ptr(stream), ctypes.byref(st)),
           "tsdf_get_stats")
    out = {k: int(getattr(st, k)) for k, _ in tsdf_stats._fields_ if k != "probe_hist"}
    out["probe_hist"] = [int(v) for v in st.probe_hist]
    return out


def tsdf_clear_stats(h, stream=None) -> None:
    _check(load_library().tsdf_clear_stats(h, _stream_ptr(stream)), "tsdf_clear_stats")


def tsdf_set_instrumentation(h, on: bool) -> None:
    _check(load_library().tsdf_set_instrumentation(h, 1 if on else 0), "tsdf_set_instrumentation")


UPDATE_ADAPTIVE = 0
UPDATE_PER_SAMPLE = 1
UPDATE_PRE_REDUCED = 2
UPDATE_FUSED = 3
UPDATE_AUTO = 4
UPDATE_KERNELS = {"adaptive": UPDATE_ADAPTIVE, "per_sample": UPDATE_PER_SAMPLE,
                  "pre_reduced": UPDATE_PRE_REDUCED, "fused": UPDATE_FUSED,
                  "auto": UPDATE_AUTO}


def tsdf_set_update_kernel(h, kind) -> None:
    """Select how updates reach the pool: "auto" (default: "per_sample", with
    integrate launches under 2^19 pixels run as "fused"), "per_sample" (each
    warp merges its lanes' samples of one voxel, then reduces into the pool),
    "adaptive" (tiles whose samples crowd into voxels pre-reduce in shared
    memory), "pre_reduced" (every tile does), or "fused" (integrate calls run
    allocate and update as one kernel); or the header's integer constants."""
    k = UPDATE_KERNELS[kind] if isinstance(kind, str) else int(kind)
    _check(load_library().tsdf_set_update_kernel(h, k), "tsdf_set_update_kernel")


OCCLUSION_RAY = 0
OCCLUSION_REPROJECT = 1
OCCLUSION_TESTS = {"ray": OCCLUSION_RAY, "reproject": OCCLUSION_REPROJECT}


POOL_LAYOUTS = {"interleaved": 0, "planar": 1}


def tsdf_set_pool_layout(h, layout) -> None:
    """Store the five sums "interleaved" (default: tsdf, weight, r, g in one
    16-byte record per voxel, blue apart) or "planar" (five separate arrays);
    only while the volume holds no block."""
    k = POOL_LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    _check(load_library().tsdf_set_pool_layout(h, k), "tsdf_set_pool_layout")


def tsdf_set_occlusion(h, mode) -> None:
    """Select the occlusion test of later launches: "ray" (default: the depth
    of the pixel whose ray selected the voxel) or "reproject" (the depth of
    the pixel nearest to the voxel centre's projection); or the header's
    integer constants."""
    m = OCCLUSION_TESTS[mode] if isinstance(mode, str) else int(mode)
    _check(load_library().tsdf_set_occlusion(h, m), "tsdf_set_occlusion")


# ----------------------------------------------------------------------------
# Convenience wrapper
# ----------------------------------------------------------------------------

class TsdfVolume:
    """Owns one tsdf_volume handle; methods forward to the C functions."""

    def __init__(self, pool_capacity: int, voxel_size: float, trunc: float,
                 table_capacity: int = 0):
        self.handle = tsdf_create(pool_capacity, voxel_size, trunc, table_capacity)
        self.info = tsdf_get_info(self.handle)

    def close(self):
        if self.handle:
            tsdf_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self, stream=None):
        tsdf_reset(self.handle, stream)

    def integrate(self, depth, rgb, K, pose, stream=None):
        tsdf_integrate(self.handle, depth, rgb, K, pose, stream)

    def allocate(self, depth, K, pose, stream=None):
        tsdf_allocate(self.handle, depth, K, pose, stream)

    def update(self, depth, rgb, K, pose, stream=None):
        tsdf_update(self.handle, depth, rgb, K, pose, stream)

    def integrate_batch(self, depth, rgb, K, poses, stream=None):
        tsdf_integrate_batch(self.handle, depth, rgb, K, poses, stream)

    def allocate_batch(self, depth, K, poses, stream=None):
        tsdf_allocate_batch(self.handle, depth, K, poses, stream)

    def update_batch(self, depth, rgb, K, poses, stream=None):
        tsdf_update_batch(self.handle, depth, rgb, K, poses, stream)

    def integrate_batch_host(self, depth, rgb, K, poses, stream=None):
        tsdf_integrate_batch_host(self.handle, depth, rgb, K, poses, stream)

    def allocate_blocks(self, coords, stream=None):
        tsdf_allocate_blocks(self.handle, coords, stream)

    def block_count(self, stream=None) -> int:
        return tsdf_block_count(self.handle, stream)

    def export_blocks(self, first=0, count=None, stream=None, **kw) -> dict:
        return tsdf_export_blocks(self.handle, first, count, stream, **kw)

    def extract_triangles(self, stream=None, capacity=None):
        return tsdf_extract_triangles(self.handle, stream, capacity)

    def import_blocks(self, coords, tsdf, weight, r, g, b, stream=None):
        tsdf_import_blocks(self.handle, coords, tsdf, weight, r, g, b, stream)

    def export_table(self, stream=None):
        return tsdf_export_table(self.handle, stream)

    def stats(self, stream=None) -> dict:
        return tsdf_get_stats(self.handle, stream)

    def clear_stats(self, stream=None):
        tsdf_clear_stats(self.handle, stream)

    def set_instrumentation(self, on: bool):
        tsdf_set_instrumentation(self.handle, on)

    def set_update_kernel(self, kind):
        tsdf_set_update_kernel(self.handle, kind)

    def set_occlusion(self, mode):
        tsdf_set_occlusion(self.handle, mode)

    def set_pool_layout(self, layout):
        tsdf_set_pool_layout(self.handle, layout)
        self.info = tsdf_get_info(self.handle)
