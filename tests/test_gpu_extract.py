"""Surface extraction and block import on the GPU, through the C ABI.

Exact parity: the oracle integrates a scene (or holds a known field), its
sums rounded to float32 are imported into a GPU volume, and the GPU's
marching-tetrahedra triangles must equal the oracle's extraction of the
same sums triangle for triangle (both evaluate the same float32 operations
in the same order; the triangle order is unspecified, so both sides are
sorted).  Cross-arm: the GPU's own integration and extraction against the
oracle's, by mean and maximum vertex distance (the correctness section
compares arms this way), plus the analytic sphere to within a quarter voxel.
"""
import numpy as np
import pytest

from hash_blocked_tsdf_gb300 import scenes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    return torch


def _sorted_rows(tris):
    a = np.asarray(tris, dtype=np.float32).reshape(-1, 9)
    return a[np.lexsort(a.T[::-1])]


def _import_oracle(torch, o, voxel, trunc, pool=None, layout=None):
    from hash_blocked_tsdf_gb300 import TsdfVolume
    e = o.export()
    n = len(e["coords"])
    vol = TsdfVolume(pool or max(4096, 2 * n), voxel, trunc)
    if layout is not None:
        vol.set_pool_layout(layout)
    vol.import_blocks(e["coords"], *(e[k].astype(np.float32) for k in ("tsdf", "weight", "r",
                                                                          "g", "b")))
    return vol, e


def _assert_same_triangles(gpu, oracle_tris):
    g = _sorted_rows(gpu.cpu().numpy())
    o = _sorted_rows(oracle_tris)
    assert g.shape == o.shape, (g.shape, o.shape)
    np.testing.assert_array_equal(g, o)


@pytest.mark.parametrize("layout", ["interleaved", "planar"])
def test_import_round_trip(torch_cuda, oracle_mod, layout):
    f = scenes.tiny_sphere_plane()
    o = oracle_mod.OracleVolume(f.voxel_size, f.trunc)
    o.integrate_frames(f)
    vol, e = _import_oracle(torch_cuda, o, f.voxel_size, f.trunc, layout=layout)
    g = vol.export_blocks()
    order = np.lexsort((g["coords"][:, 2], g["coords"][:, 1], g["coords"][:, 0]))
    np.testing.assert_array_equal(g["coords"][order], e["coords"])
    for k in ("tsdf", "weight", "r", "g", "b"):
        np.testing.assert_array_equal(g[k][order], e[k].astype(np.float32))
    vol.close()


@pytest.mark.parametrize("layout", ["interleaved", "planar"])
def test_extract_equals_oracle_on_the_sphere_scene(torch_cuda, oracle_mod, layout):
    f = scenes.tiny_sphere_plane()
    o = oracle_mod.OracleVolume(f.voxel_size, f.trunc)
    o.integrate_frames(f)
    vol, _ = _import_oracle(torch_cuda, o, f.voxel_size, f.trunc, layout=layout)
    tris = vol.extract_triangles()
    assert len(tris) > 50000
    _assert_same_triangles(tris, o.extract())
    vol.close()


def test_extract_equals_oracle_on_a_closed_sphere(torch_cuda, oracle_mod):
    # a signed-distance sphere written straight into 27 blocks, with uneven
    # weights (sums = w * value): a closed mesh crossing every block face
    voxel = 0.01
    c = np.array([12.31, 11.83, 12.07]) * voxel
    R = 7.29 * voxel
    rng = np.random.default_rng(12)
    o = oracle_mod.OracleVolume(voxel, 4 * voxel)
    j = np.arange(512)
    local = np.stack([j % 8, (j // 8) % 8, j // 64], axis=1)
    for bx in range(3):
        for by in range(3):
            for bz in range(3):
                idx = local + 8 * np.array([bx, by, bz])
                w = rng.integers(1, 4, size=512).astype(np.float64)
                o.set_block((bx, by, bz), w * (np.linalg.norm((idx + 0.5) * voxel - c, axis=1) - R),
                            w, w * 0.25, w * 0.5, w * 0.75)
    vol, _ = _import_oracle(torch_cuda, o, voxel, 4 * voxel)
    _assert_same_triangles(vol.extract_triangles(), o.extract())
    vol.close()


def test_extract_block_with_thousands_of_triangles(torch_cuda, oracle_mod):
    # an alternating-sign field: every cell crossed, up to 12 triangles per
    # cell, thousands per block (many emission rounds per warp, with both
    # halves of a round full), in full and with an output capacity that cuts
    # through a block's range
    voxel = 0.01
    o = oracle_mod.OracleVolume(voxel, 4 * voxel)
    j = np.arange(512)
    local = np.stack([j % 8, (j // 8) % 8, j // 64], axis=1)
    rng = np.random.default_rng(5)
    for bx in range(2):
        for bz in range(2):
            idx = local + 8 * np.array([bx, 0, bz])
            sign = np.where(idx.sum(axis=1) % 2 == 0, 1.0, -1.0)
            val = sign * (0.25 + rng.random(512))
            w = rng.integers(1, 5, size=512).astype(np.float64)
            o.set_block((bx, 0, bz), w * val, w, w * 0.1, w * 0.2, w * 0.3)
    vol, _ = _import_oracle(torch_cuda, o, voxel, 4 * voxel)
    ref = o.extract()
    assert len(ref) > 4 * 2000
    full = vol.extract_triangles()
    _assert_same_triangles(full, ref)
    for cap in (len(ref) // 2 + 7, 31, 33):
        part = vol.extract_triangles(capacity=cap)
        assert len(part) == cap
        full_rows = {tuple(r) for r in _sorted_rows(full.cpu().numpy())}
        assert all(tuple(r) in full_rows for r in _sorted_rows(part.cpu().numpy()))
    vol.close()


def test_extract_after_gpu_integration_against_the_oracle(torch_cuda, oracle_mod):
    from hash_blocked_tsdf_gb300 import TsdfVolume
    torch = torch_cuda
    f = scenes.vga_sphere_plane()
    vol = TsdfVolume(f.pool_capacity, f.voxel_size, f.trunc, f.table_capacity)
    vol.integrate(torch.from_numpy(f.depth[0]).cuda(), torch.from_numpy(f.rgb[0]).cuda(), f.K,
                  f.poses[0])
    g = vol.extract_triangles().cpu().numpy().reshape(-1, 3).astype(np.float64)
    o = oracle_mod.OracleVolume(f.voxel_size, f.trunc)
    o.integrate_frames(f)
    r = o.extract().reshape(-1, 3).astype(np.float64)
    # the same surface up to the float rounding of the sums: the triangle
    # counts agree closely and every vertex has a twin within a small distance
    assert abs(len(g) - len(r)) <= 0.001 * len(r)
    cKDTree = pytest.importorskip("scipy.spatial").cKDTree
    d_g, _ = cKDTree(r).query(g)
    d_r, _ = cKDTree(g).query(r)
    print("GPU vs oracle vertices: mean", d_g.mean(), "max", max(d_g.max(), d_r.max()))
    assert d_g.mean() < 1e-6 and d_r.mean() < 1e-6
    assert max(d_g.max(), d_r.max()) < f.voxel_size / 4
    # the analytic sphere (radius 0.5 m at z = 1.5 m), its visible cap
    rel = g - np.array([0.0, 0.0, 1.5])
    nr = np.linalg.norm(rel, axis=1)
    cap = (-rel[:, 2] / nr > 0.7) & (np.abs(nr - 0.5) < 0.1)
    assert cap.sum() > 10000
    assert np.abs(nr[cap] - 0.5).max() < f.voxel_size / 4
    vol.close()


def test_extract_count_capacity_and_empty(torch_cuda, oracle_mod):
    import ctypes
    from hash_blocked_tsdf_gb300 import TsdfVolume, binding
    torch = torch_cuda
    f = scenes.tiny_sphere_plane()
    vol = TsdfVolume(f.pool_capacity, f.voxel_size, f.trunc, f.table_capacity)
    assert len(vol.extract_triangles()) == 0                     # empty volume
    vol.integrate(torch.from_numpy(f.depth[0]).cuda(), torch.from_numpy(f.rgb[0]).cuda(), f.K,
                  f.poses[0])
    full = vol.extract_triangles()
    n = len(full)
    part = vol.extract_triangles(capacity=n // 2)
    assert len(part) == n // 2
    full_rows = {tuple(r) for r in _sorted_rows(full.cpu().numpy())}
    assert all(tuple(r) in full_rows for r in _sorted_rows(part.cpu().numpy()))
    lib = binding.load_library()
    total = ctypes.c_uint64()
    assert lib.tsdf_extract_triangles(vol.handle, None, None, 5, ctypes.byref(total)) == -1
    assert lib.tsdf_extract_triangles(vol.handle, None, None, 0, ctypes.byref(total)) == 0
    assert total.value == n
    vol.close()


def test_import_rejects_duplicates_and_counts_pool_exhaustion(torch_cuda):
    from hash_blocked_tsdf_gb300 import TsdfVolume, TsdfError
    vol = TsdfVolume(4, 0.01, 0.04)
    z = np.zeros((2, 512), np.float32)
    with pytest.raises(TsdfError):
        vol.import_blocks([[0, 0, 0], [0, 0, 0]], z, z, z, z, z)
    coords = np.array([[i, 0, 0] for i in range(6)], np.int32)
    vals = np.ones((6, 512), np.float32)
    vol.import_blocks(coords, vals, vals, vals, vals, vals)
    st = vol.stats()
    assert vol.block_count() == 4 and st["pool_exhausted"] == 2
    g = vol.export_blocks()
    assert np.all(g["weight"] == 1.0)
    vol.close()
