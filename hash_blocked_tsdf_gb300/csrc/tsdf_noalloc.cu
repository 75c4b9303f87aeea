// Block-coordinate export that allocates no memory.
//
// tsdf_export_blocks recovers block coordinates into a device buffer that it
// allocates with cudaMalloc on first use.  Some callers cannot let a library
// allocate device memory: processes whose device memory belongs to a caching
// allocator such as PyTorch's, which has already reserved nearly all of it
// (a raw cudaMalloc of a large buffer then fails, or fragments the pool);
// processes held to a fixed device-memory budget after they set up their own
// arena; and latency-critical threads that must not stall in cudaMalloc,
// which may synchronise the device.  This variant uses a fixed scratch array
// that lives in the library image instead.
//
// The scratch is a file-scope __device__ array of kNoAllocMaxBlocks block
// coordinates (768 KB); every GPU that loads the library holds one copy until
// the process exits.  Host code may not hand the array's name to a kernel
// (on the host it names a stand-in, not device memory), so its device address
// is looked up with cudaGetSymbolAddress when a volume is created, with the
// volume's device current, and kept in the volume.  Looking it up there also
// loads the module that holds the array and its export kernel (CUDA loads
// modules and kernels lazily, on first use), so the array's memory is set
// aside by tsdf_create, which allocates anyway, and never by the export
// call.  A volume created after a
// cudaDeviceReset looks the address up again in the new context.  All calls
// share the one array, and it keeps the previous call's contents: each call
// clears the part it uses, and two calls whose work overlaps on the GPU race
// on it.
#include "tsdf_device.cuh"

namespace tsdf {
namespace {

constexpr uint32_t kNoAllocMaxBlocks = TSDF_NOALLOC_MAX_BLOCKS;
constexpr int kThreads = 256;

__device__ __align__(256) int32_t g_coord_scratch[3 * kNoAllocMaxBlocks];

// coords[idx - first] = coordinate of the block whose table entry holds pool
// index idx, for idx in [first, first + count).
__global__ void __launch_bounds__(kThreads) export_coords_range_kernel(VolumeView vol,
                                                                       int32_t* coords,
                                                                       uint32_t first,
                                                                       uint32_t count)
{
    const uint32_t slot = blockIdx.x * kThreads + threadIdx.x;
    if (slot > vol.table_mask) return;
    const Entry e = vol.table[slot];
    if (e.key == kEmptyKey || e.idx < first || e.idx - first >= count) return;
    unpack_block(e.key, coords + 3 * (size_t)(e.idx - first));
}

}  // namespace

int resolve_noalloc_scratch(int32_t** out)
{
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_coord_scratch);
    if (e != cudaSuccess || !p)
        return record_error(TSDF_ERR_CUDA, "cudaGetSymbolAddress(g_coord_scratch) failed");
    // load the export kernel as well (kernels too are loaded on first use)
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, export_coords_range_kernel);
    if (e != cudaSuccess)
        return record_error(TSDF_ERR_CUDA, "cudaFuncGetAttributes(export kernel) failed");
    *out = static_cast<int32_t*>(p);
    return TSDF_OK;
}

}  // namespace tsdf

using namespace tsdf;

extern "C" int tsdf_export_block_coords_noalloc(tsdf_volume* vol, void* stream, uint32_t first,
                                                uint32_t count, int32_t* coords)
{
    if (!vol || !coords) return record_error(TSDF_ERR_ARG, "volume and coords must be non-null");
    if (count > kNoAllocMaxBlocks)
        return record_error(TSDF_ERR_ARG,
                            "count exceeds the no-allocation export limit of 65536 blocks");
    uint32_t n = 0;
    int rc = tsdf_block_count(vol, stream, &n);     // (checks the current device too)
    if (rc) return rc;
    if ((uint64_t)first + count > n)
        return record_error(TSDF_ERR_ARG, "first + count exceeds the number of allocated blocks");
    if (count == 0) return TSDF_OK;
    int32_t* scratch = noalloc_scratch_of(vol);
    if (!scratch) return record_error(TSDF_ERR_CUDA, "the volume has no scratch address");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const VolumeView view = volume_view(vol);
    const size_t bytes = (size_t)count * 3 * sizeof(int32_t);
    // the array keeps the previous call's contents: clear the part this call uses
    cudaError_t e = cudaMemsetAsync(scratch, 0, bytes, s);
    if (e == cudaSuccess) {
        const uint64_t slots = (uint64_t)view.table_mask + 1;
        export_coords_range_kernel<<<(unsigned)((slots + kThreads - 1) / kThreads), kThreads, 0,
                                     s>>>(view, scratch, first, count);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(coords, scratch, bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return record_error(TSDF_ERR_CUDA, cudaGetErrorString(e));
    return TSDF_OK;
}
