// Volume maintenance kernels: clearing the used prefix of the pool,
// recovering each pool block's coordinate from the table for read-out, the
// per-batch table of pixel rays, and the check of the fixed-divisor
// divisions.
#include "tsdf_device.cuh"

namespace tsdf {
namespace {

constexpr int kThreads = 256;

// Zero blocks [0, min(*pool_counter, capacity)) of the pool, in either
// layout.  The count is read on the device, so a reset needs no host round
// trip.
__global__ void __launch_bounds__(kThreads) zero_used_blocks_kernel(VolumeView vol)
{
    const uint32_t used = min(*vol.pool_counter, vol.pool_capacity);
    const size_t n = (size_t)used * (kBlockVoxels / 4);     // float4s per field in use
    const size_t plane4 = vol.plane / 4;                     // float4s per planar array
    float4* base = vol.voxel4;
    float4* blue4 = reinterpret_cast<float4*>(vol.blue);
    const float4 z = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const size_t stride = (size_t)gridDim.x * kThreads;
    for (size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x; e < n; e += stride) {
        if (vol.planar) {
#pragma unroll
            for (int a = 0; a < 4; ++a) base[(size_t)a * plane4 + e] = z;
        } else {
            // the interleaved records of the used blocks: 4 n float4s
#pragma unroll
            for (int a = 0; a < 4; ++a) base[4 * e + a] = z;
        }
        blue4[e] = z;
    }
}

// Interleaved layout: voxels [first, first + n) of the pool, in the C ABI's
// x-fastest numbering (first and n multiples of 512), split into five
// planes: out[k * n + i] = sum k (tsdf, weight, red, green, blue) of voxel
// first + i, read from the brick-ordered records and blue sums.
__global__ void __launch_bounds__(kThreads) split_records_kernel(VolumeView vol, size_t first,
                                                                 size_t n, float* out)
{
    const size_t stride = (size_t)gridDim.x * kThreads;
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride) {
        const size_t v = first + i;
        const size_t src = (v & ~(size_t)(kBlockVoxels - 1)) + voxel_slot_of(vol, (int)(v & 511));
        const float4 r = vol.voxel4[src];
        out[i] = r.x;
        out[n + i] = r.y;
        out[2 * n + i] = r.z;
        out[3 * n + i] = r.w;
        out[4 * n + i] = vol.blue[src];
    }
}

// coords[idx] = coordinate of the block whose table entry holds pool index idx.
__global__ void __launch_bounds__(kThreads) export_coords_kernel(VolumeView vol, int32_t* coords)
{
    const uint32_t slot = blockIdx.x * kThreads + threadIdx.x;
    if (slot > vol.table_mask) return;
    const Entry e = vol.table[slot];
    if (e.key == kEmptyKey || e.idx >= vol.pool_capacity) return;
    unpack_block(e.key, coords + 3 * (size_t)e.idx);
}

// Every float32 bit pattern x: does the fixed-divisor quotient come out as
// IEEE division gives it?  kDivideTrunc: for x >= -y, compared as
// min(1, x / y) (y the truncation distance); kDivideVoxel: for every
// non-NaN x, bit for bit (y the voxel edge, div_voxel's ranges).
template <int kCheck>
__global__ void __launch_bounds__(kThreads) verify_fixed_divisor_kernel(
    float y, float r, unsigned long long* mismatches)
{
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    uint32_t bad = 0;
    DivisorPair dv = {y, r, y, r};
    for (uint64_t b = (uint64_t)blockIdx.x * kThreads + threadIdx.x; b < (1ull << 32);
         b += stride) {
        const float x = __uint_as_float((uint32_t)b);
        const float ieee = __fdiv_rn(x, y);
        bool same;
        if (kCheck == kDivideTrunc) {
            const float fast = div_trunc<true>(x, y, r);
            same = !(x >= -y) || fminf(1.0f, fast) == fminf(1.0f, ieee);
        } else {
            same = isnan(x) || __float_as_uint(div_voxel(dv, true, x)) == __float_as_uint(ieee);
        }
        bad += same ? 0u : 1u;
    }
    bad = __reduce_add_sync(0xFFFFFFFFu, bad);
    if (lane_id() == 0 && bad) atomicAdd(mismatches, (unsigned long long)bad);
}

// The ray table of a width x height image (FrameBatch::rays, ray_yn).
__global__ void __launch_bounds__(kThreads) build_rays_kernel(float fx, float fy, float cx,
                                                              float cy, int width, int height,
                                                              float4* rays, float* ray_yn)
{
    const size_t n = (size_t)width * (size_t)height;
    const size_t stride = (size_t)gridDim.x * kThreads;
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride) {
        const int u = (int)(i % (size_t)width);
        const int v = (int)(i / (size_t)width);
        float yn;
        rays[i] = pixel_ray(fx, fy, cx, cy, u, v, yn);
        if (u == 0) ray_yn[v] = yn;
    }
}

}  // namespace

cudaError_t launch_verify_fixed_divisor(float y, float inv_y, int check,
                                        unsigned long long* mismatches, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    const unsigned grid = (unsigned)(sms * 16);
    if (check == kDivideVoxel)
        verify_fixed_divisor_kernel<kDivideVoxel><<<grid, kThreads, 0, stream>>>(y, inv_y,
                                                                                 mismatches);
    else
        verify_fixed_divisor_kernel<kDivideTrunc><<<grid, kThreads, 0, stream>>>(y, inv_y,
                                                                                 mismatches);
    return cudaGetLastError();
}

cudaError_t launch_build_rays(float fx, float fy, float cx, float cy, int width, int height,
                              float4* rays, float* ray_yn, cudaStream_t stream)
{
    const size_t n = (size_t)width * (size_t)height;
    const size_t want = (n + kThreads - 1) / kThreads;
    const unsigned grid = (unsigned)(want < 8192 ? want : 8192);
    build_rays_kernel<<<grid, kThreads, 0, stream>>>(fx, fy, cx, cy, width, height, rays,
                                                     ray_yn);
    return cudaGetLastError();
}

cudaError_t launch_zero_used_blocks(const VolumeView& vol, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    zero_used_blocks_kernel<<<(unsigned)(sms * 8), kThreads, 0, stream>>>(vol);
    return cudaGetLastError();
}

cudaError_t launch_split_records(const VolumeView& vol, size_t first, size_t n, float* out,
                                 cudaStream_t stream)
{
    if (n == 0) return cudaSuccess;
    const size_t want = (n + kThreads - 1) / kThreads;
    const unsigned grid = (unsigned)(want < 4096 ? want : 4096);
    split_records_kernel<<<grid, kThreads, 0, stream>>>(vol, first, n, out);
    return cudaGetLastError();
}

cudaError_t launch_export_coords(const VolumeView& vol, int32_t* coords, cudaStream_t stream)
{
    const uint64_t slots = (uint64_t)vol.table_mask + 1;
    const unsigned grid = (unsigned)((slots + kThreads - 1) / kThreads);
    export_coords_kernel<<<grid, kThreads, 0, stream>>>(vol, coords);
    return cudaGetLastError();
}

}  // namespace tsdf
