"""The block-coordinate export that allocates no memory.

Some callers cannot let the library allocate device memory: their device
memory belongs to a caching allocator that has reserved nearly all of it, or
they live under a fixed device-memory budget, or they run on threads that
must not stall in cudaMalloc.  tsdf_export_block_coords_noalloc serves them
from a scratch array compiled into the library.  This test calls it through
the C ABI on a fresh volume, first (before the ordinary export has run) and
then again with the device's free memory unchanged across the call, and
checks that it returns exactly what the ordinary export (tsdf_export_blocks,
which allocates its own buffer) returns, on two calls in a row and after a
call on a different range (the scratch array is shared and keeps the last
call's contents).  Block coordinates are integers, so the
comparison is exact.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_noalloc_coordinate_export_matches_the_allocating_export():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    from hash_blocked_tsdf_gb300 import TsdfVolume, binding, scenes

    lib = binding.load_library()
    frames = scenes.vga_sphere_plane()
    vol = TsdfVolume(frames.pool_capacity, frames.voxel_size, frames.trunc,
                     frames.table_capacity)
    vol.integrate(torch.from_numpy(frames.depth[0]).cuda(),
                  torch.from_numpy(frames.rgb[0]).cuda(), frames.K, frames.poses[0])
    n = vol.block_count()
    assert 0 < n <= binding.NOALLOC_MAX_BLOCKS
    stream = torch.cuda.current_stream().cuda_stream

    def call(first, count):
        out = np.full((count, 3), -7, np.int32)
        rc = lib.tsdf_export_block_coords_noalloc(vol.handle, stream, first, count,
                                                  out.ctypes.data)
        assert rc == 0, lib.tsdf_last_error()
        return out

    # on a fresh volume, before the allocating export has ever run: the first
    # call, then a second one across which the device's free memory must not
    # move (the allocating export would take a coordinate buffer here)
    first_call = call(0, n)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    second_call = call(0, n)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, (free_before, free_after)
    np.testing.assert_array_equal(first_call, second_call)

    expected = vol.export_blocks(fields=("coords",))["coords"]
    np.testing.assert_array_equal(first_call, expected)
    np.testing.assert_array_equal(call(0, n), expected)
    np.testing.assert_array_equal(call(17, 100), expected[17:117])
    np.testing.assert_array_equal(call(0, n), expected)

    # sizes beyond the built-in array are refused, with a message
    big = np.zeros((binding.NOALLOC_MAX_BLOCKS + 1, 3), np.int32)
    rc = lib.tsdf_export_block_coords_noalloc(vol.handle, stream, 0,
                                              binding.NOALLOC_MAX_BLOCKS + 1, big.ctypes.data)
    assert rc == -1 and b"65536" in lib.tsdf_last_error()
    # so are ranges past the allocated blocks
    rc = lib.tsdf_export_block_coords_noalloc(vol.handle, stream, n, 1, big.ctypes.data)
    assert rc == -1
    vol.close()
