"""Parity of the CUDA integrate path (through the C ABI) with the CPU oracle.

Exact: block coordinate set, block count, every weight sum, the counters.
Float: TSDF and colour sums within max(1e-5 |x|, 1e-6) for single frames;
for trajectories the float32 summation bound is admitted as well (see
tests/parity.py).
"""
import numpy as np
import pytest

import parity
from hash_blocked_tsdf_gb300 import scenes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    return torch


def _gpu_volume(torch, frames, **kw):
    from hash_blocked_tsdf_gb300 import TsdfVolume
    cap = kw.get("pool_capacity", frames.pool_capacity)
    table = kw.get("table_capacity", frames.table_capacity)
    return TsdfVolume(cap, frames.voxel_size, frames.trunc, table)


def _integrate_gpu(torch, frames, vol, batch=True):
    d = torch.from_numpy(frames.depth).cuda()
    c = torch.from_numpy(frames.rgb).cuda()
    if batch:
        vol.integrate_batch(d, c, frames.K, frames.poses)
    else:
        for f in range(frames.n_frames):
            vol.integrate(d[f], c[f], frames.K, frames.poses[f])
    torch.cuda.synchronize()


def _oracle(oracle_mod, frames, block_limit=-1):
    o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc, block_limit=block_limit)
    o.integrate_frames(frames)
    return o


def _full_parity(torch, oracle_mod, frames, strict, batch=True, kernel=None, layout=None):
    vol = _gpu_volume(torch, frames)
    if layout is not None:
        vol.set_pool_layout(layout)
    if kernel is not None:
        vol.set_update_kernel(kernel)
    _integrate_gpu(torch, frames, vol, batch)
    g = vol.export_blocks()
    st = vol.stats()
    o = _oracle(oracle_mod, frames)
    rep = parity.compare_volume(g, o.export(), strict)
    parity.check_counters(st, o.counters())
    assert st["pool_exhausted"] == 0
    assert vol.block_count() == o.block_count()
    # every allocated block received a contribution (same occlusion test in both passes)
    assert np.all(g["weight"].sum(axis=1) > 0)
    vol.close()
    return rep


def test_smoke_entry(torch_cuda):
    import __graft_entry__
    __graft_entry__.smoke()


KERNELS = ["adaptive", "pre_reduced", "per_sample", "fused", "auto"]


@pytest.mark.parametrize("kernel", KERNELS)
def test_parity_tiny_sphere_plane(torch_cuda, oracle_mod, kernel):
    rep = _full_parity(torch_cuda, oracle_mod, scenes.tiny_sphere_plane(), strict=True,
                       kernel=kernel)
    assert rep["blocks"] > 500


@pytest.mark.parametrize("kernel", KERNELS)
def test_parity_vga_sphere_plane(torch_cuda, oracle_mod, kernel):
    _full_parity(torch_cuda, oracle_mod, scenes.vga_sphere_plane(), strict=True, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_parity_oblique_pose(torch_cuda, oracle_mod, kernel):
    from test_oracle_pins import oblique_sphere_frames
    _full_parity(torch_cuda, oracle_mod, oblique_sphere_frames(), strict=True, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("wh", [(1, 1), (7, 3), (33, 17), (161, 121), (257, 1), (1, 300)])
def test_parity_ragged_sizes(torch_cuda, oracle_mod, wh, kernel):
    W, H = wh
    depth, rgb, pose, K = scenes.sphere_plane(W, H, fx=0.8 * max(W, H), fy=0.8 * max(W, H),
                                              noise_sigma=0.002, invalid_frac=0.1, seed=W * H)
    frames = scenes.Frames(f"ragged_{W}x{H}", depth[None], rgb[None], pose[None], K,
                           0.01, 0.04, 4096, 0, 0)
    _full_parity(torch_cuda, oracle_mod, frames, strict=True, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_parity_long_band_single_frame(torch_cuda, oracle_mod, kernel):
    """Voxel 5 mm, truncation 5 cm: 21 samples per ray under the ray-depth
    test.  Bands longer than 9 samples take the allocate kernel's step-by-step
    insert path, the pre-reducing kernel's three-way band split with 7
    samples per part, and (fused mode) the two-kernel fallback."""
    f = scenes.tiny_sphere_plane()
    frames = scenes.Frames("long_band_160x120", f.depth, f.rgb, f.poses, f.K, 0.005, 0.05,
                           1 << 15, 0, 0)
    rep = _full_parity(torch_cuda, oracle_mod, frames, strict=True, kernel=kernel)
    assert rep["blocks"] > 1000


@pytest.mark.parametrize("kernel", KERNELS)
def test_parity_long_band_orbit_batch(torch_cuda, oracle_mod, kernel):
    """Eight orbit frames in one launch through 2 cm voxels with a 20 cm
    truncation (21 samples per ray): near tiles see voxel edges 5+ pixels
    wide, so the adaptive mode sends them to the pre-reducing kernel with the
    long band."""
    frames = scenes.orbit_trajectory(n_frames=100, frames=(0, 8), voxel_size=0.02, trunc=0.2,
                                     pool_capacity=1 << 16)
    _full_parity(torch_cuda, oracle_mod, frames, strict=False, kernel=kernel)


def _flat_frame(name, W, H, f, depth_m, pose, voxel, trunc, pool, rgb_scale=1.0, rgb_shift=0.0,
                seed=0):
    """One frame of a surface at constant camera depth, colours uniform."""
    rng = np.random.default_rng(seed)
    depth = np.full((1, H, W), depth_m, np.float32)
    rgb = (rng.random((1, H, W, 3)) * rgb_scale + rgb_shift).astype(np.float32)
    K = np.array([f, f, (W - 1) / 2, (H - 1) / 2], np.float32)
    return scenes.Frames(name, depth, rgb, pose[None].astype(np.float32), K, voxel, trunc, pool,
                         0, seed)


# The allocate kernel skips the ray-depth occlusion test on band steps it
# proves pass (a margin argument on the voxel-centre depth, tsdf_device.cuh
# sure_pass).  These cases sit at the proof's edges; the block set must stay
# exactly the oracle's.

@pytest.mark.parametrize("ratio", [3.6, 4.4])
@pytest.mark.parametrize("kernel", ["per_sample", "auto"])
def test_parity_truncation_not_a_multiple_of_the_voxel(torch_cuda, oracle_mod, ratio, kernel):
    f = scenes.vga_sphere_plane()
    frames = scenes.Frames(f"vga_trunc{ratio}", f.depth, f.rgb, f.poses, f.K, 0.01,
                           float(np.float32(0.01 * ratio)), 1 << 16, 0, 0)
    _full_parity(torch_cuda, oracle_mod, frames, strict=True, kernel=kernel)


@pytest.mark.parametrize("scale", [1.00001, 1.05])
def test_parity_pose_not_exactly_a_rotation(torch_cuda, oracle_mod, scale):
    # 1.00001: R^T R - I ~ 2e-5, the proof allows for it; 1.05: far from a
    # rotation, the proof is not attempted and every step is tested
    from test_oracle_pins import oblique_sphere_frames
    f = oblique_sphere_frames()
    poses = f.poses.copy()
    poses[:, :3, :3] *= np.float32(scale)
    frames = scenes.Frames(f"oblique_scaled{scale}", f.depth, f.rgb, poses, f.K, f.voxel_size,
                           f.trunc, f.pool_capacity, f.table_capacity, 0)
    _full_parity(torch_cuda, oracle_mod, frames, strict=True, kernel="per_sample")


# For most rays the allocate kernel finds the band steps that start a block
# from where the band crosses block boundaries (an estimate per axis,
# confirmed by evaluating the steps on both sides exactly) instead of
# visiting every step.  These frames put rays along the world axes and
# nearly so (a direction component of a few 1e-5 makes the estimate
# unreliable; the kernel then walks step by step), band samples exactly on
# voxel and block boundaries (a voxel edge of 1/16 m and depths that are
# exact in binary), and every band length from 1 to 9 steps.
_AXIS_POSES = {
    "identity": (np.eye(3), (0.0, 0.0, 0.0)),
    "z_to_x": (np.array([[0.0, 0.0, 1.0], [1.0, 0.0, 0.0], [0.0, 1.0, 0.0]]), (0.5, -0.5, 1.0)),
    "z_to_minus_y": (np.array([[1.0, 0.0, 0.0], [0.0, 0.0, -1.0], [0.0, 1.0, 0.0]]),
                     (-1.0, 0.25, 0.0)),
    "nearly_identity": (scenes.axis_angle(np.array([1.0, 2.0, 3.0]) / np.sqrt(14.0), 3e-5),
                        (0.5, 0.5, -0.5)),
}


@pytest.mark.parametrize("ratio", [0.4, 1.0, 2.0, 3.0, 4.0])
@pytest.mark.parametrize("pose_name", sorted(_AXIS_POSES))
@pytest.mark.parametrize("depth_m", [2.0, 2.03125])
def test_parity_axis_rays_on_block_boundaries(torch_cuda, oracle_mod, ratio, pose_name, depth_m):
    R, t = _AXIS_POSES[pose_name]
    pose = np.eye(4)
    pose[:3, :3] = R
    pose[:3, 3] = t
    voxel = 0.0625
    frames = _flat_frame(f"axis_{pose_name}_{ratio}_{depth_m}", 33, 33, 16.0, depth_m, pose,
                         voxel, ratio * voxel, 4096, seed=5)
    _full_parity(torch_cuda, oracle_mod, frames, strict=True, kernel="per_sample")


@pytest.mark.parametrize("depth_m", [0.03, 0.045, 0.0488, 0.05, 0.06])
def test_parity_surface_at_the_near_limit(torch_cuda, oracle_mod, depth_m):
    # voxel 1 cm, truncation 4 cm: the proof needs depth / voxel above about
    # 4.9; nearer surfaces have band samples behind the camera
    a = np.array([0.3, -0.2, 1.0]) / np.linalg.norm([0.3, -0.2, 1.0])
    pose = scenes.look_at(-0.37 * a + np.array([0.011, -0.007, 0.003]),
                          np.array([0.011, -0.007, 0.003]))
    frames = _flat_frame(f"near_{depth_m}", 96, 64, 60.0, depth_m, pose, 0.01, 0.04, 4096,
                         seed=11)
    _full_parity(torch_cuda, oracle_mod, frames, strict=True, kernel="per_sample")


def test_pre_reduced_colours_outside_unit_range(torch_cuda, oracle_mod):
    # colours in [-50, 205): those pixels take the per-sample path; the sums
    # must still match the oracle exactly as before
    frames = _flat_frame("colours_wide", 96, 64, 80.0, 1.2031, np.eye(4), 0.01, 0.04, 4096,
                         rgb_scale=255.0, rgb_shift=-50.0, seed=3)
    _full_parity(torch_cuda, oracle_mod, frames, strict=True, kernel="pre_reduced")


def test_pre_reduced_dense_close_range(torch_cuda, oracle_mod):
    # 0.25 mm pixels against 1 cm voxels, seen at 40 degrees: every 8 x 8 tile
    # sends all 64 rays through the same few voxels, up to two samples per ray
    # and voxel, the most a cell can receive from one tile
    pose = np.eye(4)
    pose[:3, :3] = scenes.axis_angle([0.0, 1.0, 0.0], np.deg2rad(40.0))
    frames = _flat_frame("dense_close", 64, 64, 2000.0, 0.5037, pose, 0.01, 0.04, 4096, seed=4)
    rep = _full_parity(torch_cuda, oracle_mod, frames, strict=True, kernel="pre_reduced")
    o = _oracle(oracle_mod, frames)
    assert o.export()["weight"].max() >= 64, "the case must put many samples in one voxel"
    print("dense close range:", rep)


@pytest.mark.parametrize("kernel", ["per_sample", "adaptive", "fused"])
def test_adaptive_mixes_dense_and_sparse_tiles(torch_cuda, oracle_mod, kernel):
    # one 640 x 480 frame, 3 cm voxels at fx = 525: the sphere's front
    # (depth < 1.575 m) sees a voxel edge 10+ pixels wide (the one-frame
    # rule) and is pre-reduced, the plane at 2.5 m is not; each tile is
    # integrated exactly once
    f = scenes.vga_sphere_plane()
    frames = scenes.Frames("vga_mixed", f.depth, f.rgb, f.poses, f.K, 0.03, 0.12, 8192, 0, 0)
    d = frames.depth[0]
    near = (d > 0) & (0.03 * frames.K[0] >= 10 * d)
    assert 0.05 < near.mean() < 0.6, "the frame must hold both kinds of pixel"
    # the near tiles put 100+ samples of one frame in a voxel; their float32
    # sums, merged in registers in any grouping, are held to the a-priori
    # summation bound (tests/parity.py), as in the trajectories
    _full_parity(torch_cuda, oracle_mod, frames, strict=False, kernel=kernel)


@pytest.mark.parametrize("kernel", ["per_sample", "adaptive", "fused"])
def test_adaptive_eight_frame_batch(torch_cuda, oracle_mod, kernel):
    # eight orbit frames in one launch with 2 cm voxels: objects nearer than
    # 2.1 m see a voxel edge 5+ pixels wide (the several-frame rule)
    f = scenes.orbit_trajectory(n_frames=100, frames=(0, 8))
    frames = scenes.Frames("orbit_mixed", f.depth, f.rgb, f.poses, f.K, 0.02, 0.08, 1 << 16, 0, 0)
    d = frames.depth
    near = (d > 0) & (0.02 * frames.K[0] >= 5 * d)
    assert 0.02 < near.sum() / (d > 0).sum() < 0.9, "the batch must hold both kinds of pixel"
    _full_parity(torch_cuda, oracle_mod, frames, strict=False, kernel=kernel)


@pytest.mark.parametrize("kernel", ["per_sample", "adaptive", "fused"])
def test_adaptive_dense_frame(torch_cuda, oracle_mod, kernel):
    # 512 x 512 pixels of 1.5 mm against 2 cm voxels: every tile is dense and
    # hundreds of samples reach each voxel (summation tolerance)
    pose = np.eye(4)
    pose[:3, :3] = scenes.axis_angle([0.0, 1.0, 0.0], np.deg2rad(35.0))
    frames = _flat_frame("dense_frame", 512, 512, 600.0, 0.9037, pose, 0.02, 0.08, 4096, seed=6)
    rep = _full_parity(torch_cuda, oracle_mod, frames, strict=False, kernel=kernel)
    print("dense frame:", rep)


def test_fused_room_walk_batch(torch_cuda, oracle_mod):
    # allocate and update in one kernel, on the first 16 frames of the room
    # walk: exact blocks and weights, no wait for a published index gave up
    frames = scenes.room_random_walk(n_frames=300, frames=(0, 16))
    vol = _gpu_volume(torch_cuda, frames)
    vol.set_update_kernel("fused")
    _integrate_gpu(torch_cuda, frames, vol)
    st = vol.stats()
    o = _oracle(oracle_mod, frames)
    parity.compare_volume(vol.export_blocks(), o.export(), strict=False)
    parity.check_counters(st, o.counters())
    assert st["publish_timeouts"] == 0
    vol.close()


def test_pre_reduced_row_table_overflow(torch_cuda, oracle_mod):
    # 15 cm pixels against 5 mm voxels: each ray's 9 samples lie in 9 different
    # voxel rows, so an 8 x 8 tile touches ~576 rows, more than the shared
    # table holds; the rows that find no slot go straight to the pool
    frames = _flat_frame("wide_rows", 32, 32, 20.0, 3.0011, np.eye(4), 0.005, 0.02, 8192,
                         seed=5)
    _full_parity(torch_cuda, oracle_mod, frames, strict=True, kernel="pre_reduced")


def test_parity_orbit_prefix_per_frame_vs_batch(torch_cuda, oracle_mod):
    frames = scenes.orbit_trajectory(n_frames=100, frames=(0, 8))
    _full_parity(torch_cuda, oracle_mod, frames, strict=False, batch=False)
    _full_parity(torch_cuda, oracle_mod, frames, strict=False, batch=True)


@pytest.mark.slow
def test_parity_orbit_trajectory_full(torch_cuda, oracle_mod):
    rep = _full_parity(torch_cuda, oracle_mod, scenes.orbit_trajectory(), strict=False)
    print("orbit trajectory parity:", rep)


def test_host_batch_matches_device_batch(torch_cuda, oracle_mod):
    torch = torch_cuda
    frames = scenes.orbit_trajectory(n_frames=100, frames=(10, 15))
    a = _gpu_volume(torch, frames)
    _integrate_gpu(torch, frames, a)
    b = _gpu_volume(torch, frames)
    d = torch.from_numpy(frames.depth).pin_memory()
    c = torch.from_numpy(frames.rgb).pin_memory()
    b.integrate_batch_host(d, c, frames.K, frames.poses)
    torch.cuda.synchronize()
    ga, gb = a.export_blocks(), b.export_blocks()
    oa, ob = parity.sort_by_coords(ga["coords"]), parity.sort_by_coords(gb["coords"])
    assert np.array_equal(ga["coords"][oa], gb["coords"][ob])
    assert np.array_equal(ga["weight"][oa], gb["weight"][ob])
    o = _oracle(oracle_mod, frames)
    parity.compare_volume(gb, o.export(), strict=False)
    a.close()
    b.close()


def test_host_batch_over_many_groups_matches_device_batch(torch_cuda):
    """A host batch long enough for several staging groups: the groups grow
    from 16 frames (16, 21, 28, 15 for 80 frames), and the double-buffered
    staging area is reused twice.  The result must be the device batch's:
    the same blocks, weights and counters, sums equal up to the order of
    the float additions."""
    torch = torch_cuda
    frames = scenes.orbit_trajectory(n_frames=100, frames=(0, 80))
    a = _gpu_volume(torch, frames)
    _integrate_gpu(torch, frames, a)
    b = _gpu_volume(torch, frames)
    d = torch.from_numpy(frames.depth).pin_memory()
    c = torch.from_numpy(frames.rgb).pin_memory()
    b.integrate_batch_host(d, c, frames.K, frames.poses)
    torch.cuda.synchronize()
    ga, gb = a.export_blocks(), b.export_blocks()
    oa, ob = parity.sort_by_coords(ga["coords"]), parity.sort_by_coords(gb["coords"])
    assert np.array_equal(ga["coords"][oa], gb["coords"][ob])
    assert np.array_equal(ga["weight"][oa], gb["weight"][ob])
    # two float32 summations of the same w terms, |tsdf term| <= 1 and colour
    # terms >= 0: each within gamma(w) of the exact sum of |terms|
    w = ga["weight"][oa].astype(np.float64)
    u = 2.0 ** -24
    for k in ("tsdf", "r", "g", "b"):
        x, y = ga[k][oa].astype(np.float64), gb[k][ob].astype(np.float64)
        mag = w if k == "tsdf" else np.abs(x)
        bound = 2.0 * w * u * mag + 1e-5 * np.abs(x) + 1e-6
        assert np.all(np.abs(x - y) <= bound), k
    sa, sb = a.stats(), b.stats()
    for k in ("valid_points", "voxel_updates", "missed_contributions", "out_of_range_samples"):
        assert sa[k] == sb[k], k
    a.close()
    b.close()


def test_integrate_batch_replayed_from_a_cuda_graph(torch_cuda):
    """A reset and a batch integration captured into a CUDA graph (after one
    call with the same frame size has allocated the ray table) and replayed
    twice give the volume a direct call gives: the same blocks and weights,
    sums equal up to the order of the float additions."""
    torch = torch_cuda
    frames = scenes.orbit_trajectory(n_frames=100, frames=(0, 8))
    d = torch.from_numpy(frames.depth).cuda()
    c = torch.from_numpy(frames.rgb).cuda()
    ref = _gpu_volume(torch, frames)
    ref.integrate_batch(d, c, frames.K, frames.poses)
    vol = _gpu_volume(torch, frames)
    vol.integrate_batch(d[:1], c[:1], frames.K, frames.poses[:1])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        vol.reset()
        vol.integrate_batch(d, c, frames.K, frames.poses)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    ga, gb = ref.export_blocks(), vol.export_blocks()
    oa, ob = parity.sort_by_coords(ga["coords"]), parity.sort_by_coords(gb["coords"])
    assert np.array_equal(ga["coords"][oa], gb["coords"][ob])
    assert np.array_equal(ga["weight"][oa], gb["weight"][ob])
    w = ga["weight"][oa].astype(np.float64)
    u = 2.0 ** -24
    for k in ("tsdf", "r", "g", "b"):
        x, y = ga[k][oa].astype(np.float64), gb[k][ob].astype(np.float64)
        mag = w if k == "tsdf" else np.abs(x)
        assert np.all(np.abs(x - y) <= 2.0 * w * u * mag + 1e-5 * np.abs(x) + 1e-6), k
    ref.close()
    vol.close()


@pytest.mark.parametrize("layout", ["interleaved", "planar"])
def test_pool_view_matches_export(torch_cuda, layout):
    """The zero-copy pool view: tsdf, weight, r and g interleaved per voxel
    (stride 4, voxels in 2 x 2 x 2 bricks) or planar (stride 1, x fastest),
    blue plain in the same order; the same numbers as the export's separate
    x-fastest arrays."""
    from hash_blocked_tsdf_gb300 import binding
    torch = torch_cuda
    frames = scenes.tiny_sphere_plane()
    vol = _gpu_volume(torch, frames)
    vol.set_pool_layout(layout)
    assert vol.info["pool_layout"] == binding.POOL_LAYOUTS[layout]
    _integrate_gpu(torch, frames, vol)
    n = vol.block_count()
    g = vol.export_blocks()
    p = binding.tsdf_get_pool(vol.handle)
    cap = p["pool_capacity"]
    step = 4 if layout == "interleaved" else 4 * cap * 512    # bytes between fields
    assert p["stride"] == (4 if layout == "interleaved" else 1)
    assert (p["weight"] - p["tsdf"], p["r"] - p["tsdf"], p["g"] - p["tsdf"]) == \
        (step, 2 * step, 3 * step)

    class _View:
        def __init__(self, ptr, count):
            self.__cuda_array_interface__ = {"shape": (count,), "typestr": "<f4",
                                             "data": (ptr, False), "version": 3,
                                             "strides": None}
    if layout == "interleaved":
        rec = torch.as_tensor(_View(p["tsdf"], cap * 512 * 4), device="cuda").view(cap, 512, 4)
    else:
        rec = torch.as_tensor(_View(p["tsdf"], 4 * cap * 512), device="cuda").view(
            4, cap, 512).permute(1, 2, 0)
    blue = torch.as_tensor(_View(p["b"], cap * 512), device="cuda").view(cap, 512)
    # position of x-fastest voxel j in the pool: 2 x 2 x 2 bricks in the
    # interleaved layout (include/tsdf.h), x fastest in the planar one
    j = np.arange(512)
    lx, ly, lz = j & 7, (j >> 3) & 7, j >> 6
    if layout == "interleaved":
        pos = 8 * ((lx >> 1) + 4 * (ly >> 1) + 16 * (lz >> 1)) + (lx & 1) + 2 * (ly & 1) + 4 * (lz & 1)
        assert np.array_equal(np.sort(pos), j)
    else:
        pos = j
    for k, key in enumerate(("tsdf", "weight", "r", "g")):
        np.testing.assert_array_equal(rec[:n, :, k].cpu().numpy()[:, pos], g[key])
    np.testing.assert_array_equal(blue[:n].cpu().numpy()[:, pos], g["b"])
    assert float(rec[n:].abs().sum()) == 0.0 and float(blue[n:].abs().sum()) == 0.0
    # export of a sub-range (offset into the records)
    part = vol.export_blocks(first=n // 3, count=n // 2)
    for key in ("tsdf", "weight", "r", "g", "b"):
        np.testing.assert_array_equal(part[key], g[key][n // 3:n // 3 + n // 2])
    vol.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_planar_layout_parity(torch_cuda, oracle_mod, kernel):
    # the pages' five separate arrays, under every update mode: same sums
    _full_parity(torch_cuda, oracle_mod, scenes.tiny_sphere_plane(), strict=True, kernel=kernel,
                 layout="planar")
    _full_parity(torch_cuda, oracle_mod, scenes.orbit_trajectory(n_frames=100, frames=(0, 8)),
                 strict=False, kernel=kernel, layout="planar")


def test_pool_layout_changes_only_while_empty(torch_cuda, oracle_mod):
    from hash_blocked_tsdf_gb300 import TsdfError
    torch = torch_cuda
    frames = scenes.tiny_sphere_plane()
    vol = _gpu_volume(torch, frames)
    _integrate_gpu(torch, frames, vol)
    with pytest.raises(TsdfError):
        vol.set_pool_layout("planar")
    with pytest.raises(KeyError):
        vol.set_pool_layout("tiled")
    vol.reset()
    vol.set_pool_layout("planar")             # empty again: allowed
    _integrate_gpu(torch, frames, vol)
    o = _oracle(oracle_mod, frames)
    parity.compare_volume(vol.export_blocks(), o.export(), strict=True)
    vol.close()


def test_reset_gives_a_fresh_volume(torch_cuda, oracle_mod):
    torch = torch_cuda
    frames = scenes.vga_sphere_plane()
    vol = _gpu_volume(torch, frames)
    other = scenes.orbit_trajectory(n_frames=100, frames=(0, 2))
    _integrate_gpu(torch, other.subset(0, 2), vol)  # different scene first
    vol.reset()
    _integrate_gpu(torch, frames, vol)
    o = _oracle(oracle_mod, frames)
    parity.compare_volume(vol.export_blocks(), o.export(), strict=True)
    parity.check_counters(vol.stats(), o.counters())
    vol.close()


def test_empty_and_invalid_frames(torch_cuda, oracle_mod):
    torch = torch_cuda
    frames = scenes.tiny_sphere_plane()
    d = frames.depth[0].copy()
    d[:, :] = 0.0
    vol = _gpu_volume(torch, frames)
    vol.integrate(torch.from_numpy(d).cuda(), torch.from_numpy(frames.rgb[0]).cuda(), frames.K,
                  frames.poses[0])
    assert vol.block_count() == 0
    st = vol.stats()
    assert st["valid_points"] == 0 and st["voxel_updates"] == 0
    d = frames.depth[0].copy()
    d[0, :] = np.nan
    d[1, :] = np.inf
    d[2, :] = -np.inf
    d[3, :] = -0.5
    vol.reset()
    vol.integrate(torch.from_numpy(d).cuda(), torch.from_numpy(frames.rgb[0]).cuda(), frames.K,
                  frames.poses[0])
    o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    o.integrate(d, frames.rgb[0], frames.K, frames.poses[0])
    parity.compare_volume(vol.export_blocks(), o.export(), strict=True)
    parity.check_counters(vol.stats(), o.counters())
    vol.close()


def test_out_of_range_pose_counts_and_skips(torch_cuda, oracle_mod):
    torch = torch_cuda
    frames = scenes.tiny_sphere_plane()
    far = np.eye(4, dtype=np.float32)
    far[0, 3] = 1.0e6
    vol = _gpu_volume(torch, frames)
    vol.integrate(torch.from_numpy(frames.depth[0]).cuda(),
                  torch.from_numpy(frames.rgb[0]).cuda(), frames.K, far)
    st = vol.stats()
    assert vol.block_count() == 0
    assert st["out_of_range_samples"] == 9 * st["valid_points"] > 0
    vol.close()


def test_pool_exhaustion_is_counted_not_hidden(torch_cuda, oracle_mod):
    torch = torch_cuda
    frames = scenes.vga_sphere_plane()
    full = _oracle(oracle_mod, frames)
    B = full.block_count()
    cap = B // 2
    vol = _gpu_volume(torch, frames, pool_capacity=cap, table_capacity=0)
    _integrate_gpu(torch, frames, vol)
    st = vol.stats()
    assert vol.block_count() == cap
    assert st["pool_exhausted"] == B - cap
    assert st["probe_overflow"] == 0
    assert st["missed_contributions"] > 0
    assert st["voxel_updates"] + st["missed_contributions"] == full.counters()["passing_samples"]
    g = vol.export_blocks()
    assert g["weight"].sum() == st["voxel_updates"]
    # a block that won a pool slot received every one of its contributions
    ref = full.export()
    rows = np.searchsorted(
        np.ravel_multi_index((ref["coords"] + 4096).T, (8192, 8192, 8192)),
        np.ravel_multi_index((g["coords"] + 4096).T, (8192, 8192, 8192)))
    assert np.array_equal(ref["coords"][rows], g["coords"])
    parity.compare_sums({k: g[k] for k in ("tsdf", "weight", "r", "g", "b")}, ref, strict=True,
                        rows=rows)
    vol.close()


def _check_table_structure(oracle_mod, vol, expected_coords):
    keys, idx = vol.export_table()
    empty = np.uint64(0xFFFFFFFFFFFFFFFF)
    occ = keys != empty
    T = keys.size
    want = oracle_mod.pack_keys(expected_coords)
    assert np.array_equal(np.sort(keys[occ]), np.sort(want)), "table keys differ"
    n = int(occ.sum())
    assert np.array_equal(np.sort(idx[occ]), np.arange(n, dtype=np.uint32)), \
        "pool indices are not a permutation of [0, B)"
    # linear probing with insertions only: the occupied slots and the total
    # displacement do not depend on the insertion order, so the concurrent
    # table must equal the sequential reference exactly in both
    ref_table, _, ref_disp, _ = oracle_mod.probe_build(want, T)
    assert np.array_equal(occ, ref_table != empty), "occupied slot sets differ"
    slots = np.nonzero(occ)[0]
    home = np.array([oracle_mod.hash_slot(int(k), T) for k in keys[occ]], dtype=np.int64)
    disp = int(((slots - home) % T).sum())
    assert disp == ref_disp
    return disp / max(n, 1)


@pytest.mark.parametrize("T", [1 << 16, 1 << 21])
def test_home_slot_known_answers_from_the_published_splitmix64_sequence(torch_cuda, T):
    """The kernels' slot hash against SplitMix64's published outputs: the
    generator states with bit 63 clear are valid packed keys, so their
    block coordinates are inserted one at a time into an empty table; each
    key must land in the slot given by the published output, masked to the
    table (and the stored key must be the state: the packing agrees)."""
    import helpers
    from hash_blocked_tsdf_gb300 import TsdfVolume
    torch = torch_cuda
    planted = [(k, v) for k, v in helpers.splitmix64_vectors() if k >> 63 == 0]
    assert len(planted) == 3
    for key, value in planted:
        coord = np.array([[(key >> (21 * a) & 0x1FFFFF) - (1 << 20) for a in range(3)]],
                         dtype=np.int32)
        vol = TsdfVolume(64, 0.01, 0.04, T)
        vol.allocate_blocks(torch.from_numpy(coord).cuda())
        torch.cuda.synchronize()
        keys, idx = vol.export_table()
        occ = np.nonzero(keys != np.uint64(0xFFFFFFFFFFFFFFFF))[0]
        assert occ.tolist() == [value % T], (hex(key), occ, value % T)
        assert int(keys[occ[0]]) == key and int(idx[occ[0]]) == 0
        vol.close()


def test_table_structure_matches_sequential_linear_probing(torch_cuda, oracle_mod):
    torch = torch_cuda
    frames = scenes.orbit_trajectory(n_frames=100, frames=(0, 4))
    vol = _gpu_volume(torch, frames, pool_capacity=1 << 15, table_capacity=1 << 16)
    _integrate_gpu(torch, frames, vol)
    o = _oracle(oracle_mod, frames)
    _check_table_structure(oracle_mod, vol, o.coords())
    vol.close()


def test_adversarial_clustered_keys(torch_cuda, oracle_mod):
    """Keys whose home slots all fall in a window of T/64 slots, filling the
    table to load 0.5: one long cluster; nothing may be dropped."""
    from hash_blocked_tsdf_gb300 import TsdfVolume
    torch = torch_cuda
    T = 1 << 16
    want = T // 2
    coords = oracle_mod.clustered_coords(T, 12345, T // 64, (-100, 50, -20), 160, want)
    assert coords.shape[0] == want
    vol = TsdfVolume(T // 2, 0.01, 0.04, T)
    vol.set_instrumentation(True)
    dup = np.concatenate([coords, coords[::3]])            # repeated keys are found, not re-added
    perm = np.random.Generator(np.random.PCG64(1)).permutation(dup.shape[0])
    vol.allocate_blocks(torch.from_numpy(np.ascontiguousarray(dup[perm])).cuda())
    torch.cuda.synchronize()
    st = vol.stats()
    assert vol.block_count() == want
    assert st["pool_exhausted"] == 0 and st["probe_overflow"] == 0
    mean_disp = _check_table_structure(oracle_mod, vol, coords)
    assert mean_disp > want / 2 - T // 64
    assert st["probe_inserts"] > 0 and st["probe_max"] > 1000
    hist = list(st["probe_hist"])
    print("adversarial: mean displacement", mean_disp, "probe max", st["probe_max"],
          "mean probe", st["probe_steps"] / st["probe_inserts"], "probes", st["probe_inserts"],
          "histogram (lengths 1..31, 32+)", hist)
    vol.close()


@pytest.mark.slow
def test_load_factor_sweep(torch_cuda, oracle_mod):
    """Table occupancy 0.1 ... 0.5 on the orbit scene.  Two fixed tables
    follow the trajectory (2^17 slots for the low loads, 2^16 for the high
    ones); at the first frame that crosses each target the GPU state is
    compared with the oracle's (blocks, sums, counters, and the table against
    sequential linear probing).  The last target, exactly 0.5, is reached by
    topping the 2^16 table up with extra blocks far from the scene."""
    torch = torch_cuda
    full = scenes.orbit_trajectory(n_frames=100)
    small = _gpu_volume(torch, full, pool_capacity=1 << 15, table_capacity=1 << 16)
    large = _gpu_volume(torch, full, pool_capacity=1 << 16, table_capacity=1 << 17)
    plan = [(0.1, large, 1 << 17), (0.2, large, 1 << 17), (0.3, small, 1 << 16),
            (0.4, small, 1 << 16)]
    o = oracle_mod.OracleVolume(full.voxel_size, full.trunc)
    d = torch.from_numpy(full.depth).cuda()
    c = torch.from_numpy(full.rgb).cuda()
    reached = []
    for f in range(full.n_frames):
        o.integrate(full.depth[f], full.rgb[f], full.K, full.poses[f])
        for vol in (small, large):
            vol.integrate(d[f], c[f], full.K, full.poses[f])
        while plan and o.block_count() / plan[0][2] >= plan[0][0]:
            target, vol, T = plan.pop(0)
            rep = parity.compare_volume(vol.export_blocks(), o.export(), strict=False)
            parity.check_counters(vol.stats(), o.counters())
            _check_table_structure(oracle_mod, vol, o.coords())
            reached.append((target, f + 1, round(o.block_count() / T, 3), rep["blocks"]))
    assert not plan, f"targets not reached: {plan}"
    # top up to exactly half full with blocks far outside the scene
    B = o.block_count()
    extra = np.stack(np.meshgrid(np.arange(1000, 1064), np.arange(0, 64), np.arange(0, 16),
                                 indexing="ij"), axis=-1).reshape(-1, 3)[: (1 << 15) - B]
    small.allocate_blocks(torch.from_numpy(np.ascontiguousarray(extra, dtype=np.int32)).cuda())
    torch.cuda.synchronize()
    st = small.stats()
    assert small.block_count() == 1 << 15
    assert st["pool_exhausted"] == 0 and st["probe_overflow"] == 0
    _check_table_structure(oracle_mod, small, np.concatenate([o.coords(), extra]))
    reached.append((0.5, full.n_frames, 0.5, 1 << 15))
    print("load sweep (target, frames, load, blocks):", reached)
    small.close()
    large.close()


@pytest.mark.slow
def test_room_walk_full_volume(torch_cuda, oracle_mod):
    """The 300-frame 1280x720 room walk (pool 2^20, table 2^21) in the batch
    call the benchmark times, compared with the oracle's whole volume
    (computed in parallel over frame chunks and block partitions): the exact
    block set, every weight of every block, the counters, and every TSDF
    and colour sum within max(1e-5 |x|, 1e-6), or the float32 summation
    bound where a voxel's terms cancel (the test prints how many voxels
    needed it, and by how much they exceeded the stated bound)."""
    torch = torch_cuda
    frames = scenes.room_random_walk(n_frames=300)
    vol = _gpu_volume(torch, frames)
    _integrate_gpu(torch, frames, vol)
    st = vol.stats()
    g = vol.export_blocks()
    vol.close()
    torch.cuda.empty_cache()
    ref, counters = parity.full_volume_oracle(frames)
    del frames
    assert st["pool_exhausted"] == 0 and st["probe_overflow"] == 0
    assert st["valid_points"] == counters["valid_points"]
    assert st["voxel_updates"] == counters["accumulated"] == counters["passing_samples"]
    assert st["missed_contributions"] == counters["missed_contributions"] == 0
    assert st["out_of_range_samples"] == counters["out_of_range_samples"]
    rep = parity.compare_volume(g, ref, strict=False)
    assert rep["blocks"] == st["blocks_allocated"]
    assert np.all(g["weight"].sum(axis=1) > 0)
    print(f"room walk full volume: {rep['blocks']} blocks, {rep['blocks'] * 512} voxels, "
          f"{st['voxel_updates']} voxel updates; "
          + "; ".join(f"{k}: max error {rep[k]['max_err']:.3g}, "
                      f"{rep[k]['voxels_over_base']} voxels over max(1e-5|x|, 1e-6) "
                      f"(worst {rep[k]['max_err_over_base']:.3g}x)"
                      for k in ("tsdf", "r", "g", "b")))


@pytest.mark.parametrize("voxel,trunc", [(0.02, 0.08), (0.01, 0.04), (0.005, 0.02),
                                         (0.004, 0.016)])
def test_fixed_divisor_fast_path_verified(torch_cuda, voxel, trunc):
    """At create the library checks, over all 2^32 float32 dividends, that the
    reciprocal-and-correction division by the truncation distance gives the
    walk the same tsdf values as IEEE division; for the workloads' divisors
    that check must pass (the parity tests then run on that path)."""
    from hash_blocked_tsdf_gb300 import TsdfVolume
    vol = TsdfVolume(64, voxel, trunc)
    assert vol.info["fixed_divisor_fast_path"] == 1
    # the back-projection's division by the voxel edge, checked bit for bit
    assert vol.info["voxel_division_fast_path"] == 1
    vol.close()


def test_ray_table_follows_frame_size_and_intrinsics(torch_cuda, oracle_mod):
    """The back-projection reads each pixel's ray from a table the volume
    builds for the call's frame size and intrinsics.  One volume takes frames
    of two sizes and three intrinsics, back and forth (the table is rebuilt,
    grown, and reused); the result must be the oracle's for the same
    sequence."""
    torch = torch_cuda
    from hash_blocked_tsdf_gb300 import TsdfVolume
    voxel, trunc = 0.01, 0.04
    seq = []
    for n, (W, H, scale) in enumerate([(161, 121, 0.8), (161, 121, 0.9), (320, 240, 0.8),
                                       (161, 121, 0.8), (320, 240, 0.7)]):
        depth, rgb, pose, K = scenes.sphere_plane(W, H, fx=scale * max(W, H),
                                                  fy=scale * max(W, H) * 1.01,
                                                  noise_sigma=0.002, invalid_frac=0.05, seed=n)
        seq.append((depth, rgb, pose, np.asarray(K, np.float32)))
    vol = TsdfVolume(8192, voxel, trunc)
    o = oracle_mod.OracleVolume(voxel, trunc)
    for n, (depth, rgb, pose, K) in enumerate(seq):
        d = torch.from_numpy(depth).cuda()
        c = torch.from_numpy(rgb).cuda()
        if n % 2:
            vol.integrate(d, c, K, pose)
        else:
            vol.integrate_batch(d[None], c[None], K, pose[None])
        o.integrate(depth, rgb, K, pose)
    torch.cuda.synchronize()
    rep = parity.compare_volume(vol.export_blocks(), o.export(), strict=False)
    parity.check_counters(vol.stats(), o.counters())
    assert rep["blocks"] > 0
    vol.close()
