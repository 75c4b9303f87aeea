// Update kernel ("What Irregularity Costs", design section, integration:
// the regular stage; accumulation: sums, not running means).
//
// A block of 256 threads owns a 16 x 16 pixel tile of one frame of the batch,
// each warp an 8 x 4 patch of it.  The grid runs tile-major, frame-minor: the
// batch's frames update the same region of the scene (mostly the same
// voxels, since consecutive views overlap) within a short window, so those
// voxels' lines take all of the batch's reductions in L2 and go back to HBM
// once, not once per frame.  Every thread walks its pixel's truncation band
// with the same band_sample() as the allocate kernel, finds each passing
// sample's block with one lookup per new key (almost always a first-probe
// hit), and adds (tsdf, 1, r, g, b) into the five SoA arrays with
// red.global.add.f32.
//
// Reductions are issued per sample.  Pre-summing rows of voxels in shared
// memory before the reductions cuts the L2 requests about three-fold, but on
// this workload it costs more issue slots than it saves L2 time (measured on
// GB300: 0.21-0.25 ms against 0.15 ms per 1280x720 frame).
#include "tsdf_device.cuh"

namespace tsdf {
namespace {

constexpr int kTileW = 16;
constexpr int kTileH = 16;
constexpr int kThreads = kTileW * kTileH;

__device__ __forceinline__ void red_add(float* addr, float v)
{
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

template <bool kFast>
__global__ void __launch_bounds__(kThreads) update_kernel(VolumeView vol,
                                                         const __grid_constant__ FrameBatch fb)
{
    const int f = blockIdx.x % fb.n;
    const int tile = blockIdx.x / fb.n;
    const int tiles_x = (fb.width + kTileW - 1) / kTileW;
    const Camera cam = fb.frame[f].cam;
    // each warp takes an 8 x 4 pixel patch of the tile (8 warps: 2 across,
    // 4 down): a squarer footprint puts more of a warp's samples in common
    // voxel rows (one 32-byte sector per array) than a 16 x 2 strip
    const int w = (int)(threadIdx.x >> 5), l = (int)(threadIdx.x & 31u);
    const int u = (tile % tiles_x) * kTileW + (w & 1) * 8 + (l & 7);
    const int v = (tile / tiles_x) * kTileH + (w >> 1) * 4 + (l >> 3);

    RayPoint p;
    bool valid = false;
    float cr = 0.0f, cg = 0.0f, cb = 0.0f;
    if (u < fb.width && v < fb.height) {
        const size_t pix = (size_t)v * fb.width + u;
        valid = back_project(cam, u, v, __ldg(fb.frame[f].depth + pix), p);
        if (valid) {
            const float* rgb = fb.frame[f].rgb;
            cr = __ldg(rgb + 3 * pix);
            cg = __ldg(rgb + 3 * pix + 1);
            cb = __ldg(rgb + 3 * pix + 2);
        }
    }
    uint32_t updates = 0, missed = 0;
    if (valid) {
        unsigned long long last = kEmptyKey;
        uint32_t idx = kIndexFailed;
        for (int i = -vol.band_half; i <= vol.band_half; ++i) {
            VoxelSample s;
            if (band_sample<kFast>(cam, vol.div, p, i, s) != kSamplePass) continue;
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
    if (l == 0) {
        const int stripe = blockIdx.x % kCounterStripes;
        if (w_valid) atomicAdd(&vol.counters->valid_points[stripe], (unsigned long long)w_valid);
        if (w_updates)
            atomicAdd(&vol.counters->voxel_updates[stripe], (unsigned long long)w_updates);
        if (w_missed) atomicAdd(&vol.counters->missed[stripe], (unsigned long long)w_missed);
    }
}

}  // namespace

cudaError_t launch_update(const VolumeView& vol, const FrameBatch& fb, cudaStream_t stream)
{
    const unsigned tiles = (unsigned)(((fb.width + kTileW - 1) / kTileW) *
                                      ((fb.height + kTileH - 1) / kTileH));
    const unsigned grid = tiles * (unsigned)fb.n;
    if (vol.fast_div)
        update_kernel<true><<<grid, kThreads, 0, stream>>>(vol, fb);
    else
        update_kernel<false><<<grid, kThreads, 0, stream>>>(vol, fb);
    return cudaGetLastError();
}

}  // namespace tsdf
