// Volume maintenance kernels: clearing the used prefix of the pool, and
// recovering each pool block's coordinate from the table for read-out.
#include "tsdf_device.cuh"

namespace tsdf {
namespace {

constexpr int kThreads = 256;

// Zero blocks [0, min(*pool_counter, capacity)) of all five arrays.  The
// count is read on the device, so a reset needs no host round trip.
__global__ void __launch_bounds__(kThreads) zero_used_blocks_kernel(VolumeView vol)
{
    const uint32_t used = min(*vol.pool_counter, vol.pool_capacity);
    const size_t n4 = (size_t)used * (kBlockVoxels / 4);
    float4* arrays[5] = {reinterpret_cast<float4*>(vol.tsdf), reinterpret_cast<float4*>(vol.weight),
                         reinterpret_cast<float4*>(vol.red), reinterpret_cast<float4*>(vol.green),
                         reinterpret_cast<float4*>(vol.blue)};
    const float4 z = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const size_t stride = (size_t)gridDim.x * kThreads;
    for (size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x; e < n4; e += stride) {
#pragma unroll
        for (int a = 0; a < 5; ++a) arrays[a][e] = z;
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

}  // namespace

cudaError_t launch_zero_used_blocks(const VolumeView& vol, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    zero_used_blocks_kernel<<<(unsigned)(sms * 8), kThreads, 0, stream>>>(vol);
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
