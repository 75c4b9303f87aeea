"""Parity of the reprojection occlusion test (the alternative reading of the
design section's occlusion test) on the GPU, through the C ABI, with the
oracle run under the same test.

Exact: block coordinate set, every weight sum, the counters.  Float: TSDF and
colour sums within max(1e-5 |x|, 1e-6) for single frames, plus the float32
summation bound for trajectories (tests/parity.py).
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


def _run(torch, oracle_mod, frames, strict, kernel=None, batch=True, modes=None, layout=None):
    """Integrate `frames` on the GPU and in the oracle; modes[f] is the
    occlusion test of frame f (default: reprojection for every frame)."""
    from hash_blocked_tsdf_gb300 import TsdfVolume
    modes = modes or ["reproject"] * frames.n_frames
    vol = TsdfVolume(frames.pool_capacity, frames.voxel_size, frames.trunc,
                     frames.table_capacity)
    if layout is not None:
        vol.set_pool_layout(layout)
    if kernel is not None:
        vol.set_update_kernel(kernel)
    d = torch.from_numpy(frames.depth).cuda()
    c = torch.from_numpy(frames.rgb).cuda()
    o = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    f = 0
    while f < frames.n_frames:
        g = f
        while g < frames.n_frames and modes[g] == modes[f]:
            g += 1
        vol.set_occlusion(modes[f])
        if batch:
            vol.integrate_batch(d[f:g], c[f:g], frames.K, frames.poses[f:g])
        else:
            for k in range(f, g):
                vol.integrate(d[k], c[k], frames.K, frames.poses[k])
        o.set_occlusion(modes[f])
        o.integrate_frames(frames, f, g)
        f = g
    torch.cuda.synchronize()
    g = vol.export_blocks()
    st = vol.stats()
    rep = parity.compare_volume(g, o.export(), strict)
    parity.check_counters(st, o.counters())
    assert st["pool_exhausted"] == 0
    # both passes apply the same test: every allocated block got a sample
    assert np.all(g["weight"].sum(axis=1) > 0)
    vol.close()
    return rep, o


def _slanted_step(W=64, H=48):
    """The oracle pins' slanted surface with a nearer rectangle and holes,
    seen from a rotated pose; colours encode the pixel."""
    from test_oracle_reproject_pins import _slanted_step_frame
    depth, rgb, K, pose = _slanted_step_frame()
    return scenes.Frames("slanted_step", depth[None], rgb[None], pose[None], K, 0.02, 0.06, 4096,
                         0, 0)


KERNELS = ["adaptive", "pre_reduced", "per_sample", "fused"]


@pytest.mark.parametrize("kernel", KERNELS)
def test_reproject_tiny_sphere_plane(torch_cuda, oracle_mod, kernel):
    # every update mode runs the per-sample kernels under this test
    rep, _ = _run(torch_cuda, oracle_mod, scenes.tiny_sphere_plane(), strict=True, kernel=kernel)
    assert rep["blocks"] > 500


@pytest.mark.parametrize("layout", ["interleaved", "planar"])
def test_reproject_slanted_step_rotated(torch_cuda, oracle_mod, layout):
    _run(torch_cuda, oracle_mod, _slanted_step(), strict=True, layout=layout)


def test_reproject_vga_sphere_plane(torch_cuda, oracle_mod):
    _run(torch_cuda, oracle_mod, scenes.vga_sphere_plane(), strict=True)


def test_reproject_oblique_pose(torch_cuda, oracle_mod):
    from test_oracle_pins import oblique_sphere_frames
    _run(torch_cuda, oracle_mod, oblique_sphere_frames(), strict=True)


@pytest.mark.parametrize("wh", [(1, 1), (7, 3), (33, 17), (161, 121), (257, 1), (1, 300)])
def test_reproject_ragged_sizes(torch_cuda, oracle_mod, wh):
    W, H = wh
    depth, rgb, pose, K = scenes.sphere_plane(W, H, fx=0.8 * max(W, H), fy=0.8 * max(W, H),
                                              noise_sigma=0.002, invalid_frac=0.1, seed=W * H)
    frames = scenes.Frames(f"ragged_{W}x{H}", depth[None], rgb[None], pose[None], K,
                           0.01, 0.04, 4096, 0, 0)
    _run(torch_cuda, oracle_mod, frames, strict=True)


def test_reproject_long_band(torch_cuda, oracle_mod):
    # 21 samples per ray: the allocate kernel's step-by-step insert path
    f = scenes.tiny_sphere_plane()
    frames = scenes.Frames("long_band", f.depth, f.rgb, f.poses, f.K, 0.005, 0.05, 1 << 15, 0, 0)
    _run(torch_cuda, oracle_mod, frames, strict=True)


def test_reproject_orbit_batch_per_frame_and_batched(torch_cuda, oracle_mod):
    frames = scenes.orbit_trajectory(n_frames=100, frames=(0, 8))
    _run(torch_cuda, oracle_mod, frames, strict=False, batch=False)
    _run(torch_cuda, oracle_mod, frames, strict=False, batch=True)


def test_switching_tests_between_launches(torch_cuda, oracle_mod):
    # frames 0-2 under the ray test, 3-5 reprojected, 6-7 the ray test again
    frames = scenes.orbit_trajectory(n_frames=100, frames=(0, 8))
    modes = ["ray"] * 3 + ["reproject"] * 3 + ["ray"] * 2
    _run(torch_cuda, oracle_mod, frames, strict=False, modes=modes)


def test_the_two_tests_differ_at_depth_edges(torch_cuda, oracle_mod):
    # the slanted step has a depth discontinuity: the two readings must not
    # coincide there (so the parity above exercises the reprojected depth)
    frames = _slanted_step()
    _, o_rep = _run(torch_cuda, oracle_mod, frames, strict=True)
    o_ray = oracle_mod.OracleVolume(frames.voxel_size, frames.trunc)
    o_ray.integrate_frames(frames)
    a, b = o_ray.counters(), o_rep.counters()
    assert a["passing_samples"] != b["passing_samples"]


def test_room_walk_batch_reprojected(torch_cuda, oracle_mod):
    # the first 16 frames of the 1280 x 720 room walk in one launch
    frames = scenes.room_random_walk(n_frames=300, frames=(0, 16))
    _run(torch_cuda, oracle_mod, frames, strict=False)


def test_invalid_occlusion_mode_rejected(torch_cuda):
    from hash_blocked_tsdf_gb300 import TsdfVolume, TsdfError, binding
    vol = TsdfVolume(64, 0.01, 0.04)
    with pytest.raises(TsdfError):
        binding.tsdf_set_occlusion(vol.handle, 2)
    vol.close()


@pytest.mark.slow
def test_room_walk_full_volume_reprojected(torch_cuda, oracle_mod):
    """The 300-frame 1280x720 room walk in batch launches under the
    reprojection test, compared with the oracle's whole volume: exact block
    set, every weight, the counters, every sum within the stated bound (or
    the float32 summation bound where a voxel's terms cancel)."""
    torch = torch_cuda
    from hash_blocked_tsdf_gb300 import TsdfVolume
    frames = scenes.room_random_walk(n_frames=300)
    vol = TsdfVolume(frames.pool_capacity, frames.voxel_size, frames.trunc,
                     frames.table_capacity)
    vol.set_occlusion("reproject")
    vol.integrate_batch(torch.from_numpy(frames.depth).cuda(), torch.from_numpy(frames.rgb).cuda(),
                        frames.K, frames.poses)
    torch.cuda.synchronize()
    st = vol.stats()
    g = vol.export_blocks()
    vol.close()
    torch.cuda.empty_cache()
    ref, counters = parity.full_volume_oracle(frames, occlusion="reproject")
    del frames
    assert st["pool_exhausted"] == 0 and st["probe_overflow"] == 0
    assert st["valid_points"] == counters["valid_points"]
    assert st["voxel_updates"] == counters["accumulated"] == counters["passing_samples"]
    assert st["missed_contributions"] == counters["missed_contributions"] == 0
    assert st["out_of_range_samples"] == counters["out_of_range_samples"]
    rep = parity.compare_volume(g, ref, strict=False)
    print(f"room walk full volume (reprojection): {rep['blocks']} blocks; "
          + "; ".join(f"{k}: {rep[k]['voxels_over_base']} voxels over the stated bound "
                      f"(worst {rep[k]['max_err_over_base']:.3g}x)"
                      for k in ("tsdf", "r", "g", "b")))
