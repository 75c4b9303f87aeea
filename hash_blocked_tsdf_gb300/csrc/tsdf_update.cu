// Update kernel ("What Irregularity Costs", design section, integration:
// the regular stage; accumulation: sums, not running means).  Every thread
// walks one pixel's truncation band with the same band_sample() as the
// allocate kernel, looks up each passing sample's block (almost always at
// the first probe) and adds (tsdf, 1, r, g, b) into the five SoA arrays.
#include "tsdf_device.cuh"

namespace tsdf {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void red_add(float* addr, float v)
{
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__global__ void __launch_bounds__(kThreads) update_kernel(VolumeView vol, FrameView fr)
{
    const int n_pix = fr.width * fr.height;
    const int pix = blockIdx.x * kThreads + threadIdx.x;
    RayPoint p;
    bool valid = false;
    float cr = 0.0f, cg = 0.0f, cb = 0.0f;
    if (pix < n_pix) {
        const int v = pix / fr.width;
        const int u = pix - v * fr.width;
        valid = back_project(fr.cam, u, v, __ldg(fr.depth + pix), p);
        if (valid) {
            cr = __ldg(fr.rgb + 3 * (size_t)pix);
            cg = __ldg(fr.rgb + 3 * (size_t)pix + 1);
            cb = __ldg(fr.rgb + 3 * (size_t)pix + 2);
        }
    }
    uint32_t updates = 0, missed = 0;
    if (valid) {
        unsigned long long last = kEmptyKey;
        uint32_t idx = kIndexFailed;
        for (int i = -vol.band_half; i <= vol.band_half; ++i) {
            VoxelSample s;
            if (band_sample(fr.cam, vol.voxel, vol.trunc, p, i, s) != kSamplePass) continue;
            const unsigned long long key = block_key(s.ix, s.iy, s.iz);
            if (key != last) {
                idx = lookup(vol.table, vol.table_mask, key);
                last = key;
            }
            if (idx >= vol.pool_capacity) {     // absent, FAILED or never published
                ++missed;
                continue;
            }
            const size_t e = (size_t)idx * kBlockVoxels + (size_t)local_voxel(s.ix, s.iy, s.iz);
            red_add(vol.tsdf + e, s.tsdf);
            red_add(vol.weight + e, 1.0f);
            red_add(vol.red + e, cr);
            red_add(vol.green + e, cg);
            red_add(vol.blue + e, cb);
            ++updates;
        }
    }
    const uint32_t w_valid = __reduce_add_sync(0xFFFFFFFFu, valid ? 1u : 0u);
    const uint32_t w_updates = __reduce_add_sync(0xFFFFFFFFu, updates);
    const uint32_t w_missed = __reduce_add_sync(0xFFFFFFFFu, missed);
    if (lane_id() == 0) {
        const int stripe = blockIdx.x % kCounterStripes;
        if (w_valid) atomicAdd(&vol.counters->valid_points[stripe], (unsigned long long)w_valid);
        if (w_updates)
            atomicAdd(&vol.counters->voxel_updates[stripe], (unsigned long long)w_updates);
        if (w_missed) atomicAdd(&vol.counters->missed[stripe], (unsigned long long)w_missed);
    }
}

}  // namespace

cudaError_t launch_update(const VolumeView& vol, const FrameView& fr, cudaStream_t stream)
{
    const int n_pix = fr.width * fr.height;
    const unsigned grid = (unsigned)((n_pix + kThreads - 1) / kThreads);
    update_kernel<<<grid, kThreads, 0, stream>>>(vol, fr);
    return cudaGetLastError();
}

}  // namespace tsdf
