// Internal declarations shared by the libtsdf translation units: the device
// view of a volume, the per-frame launch parameters, the device counters and
// the kernel launchers.  Nothing here is part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tsdf.h"

namespace tsdf {

constexpr int kBlockEdge = 8;
constexpr int kBlockVoxels = 512;
constexpr int kCounterStripes = 32;     // high-rate counters are spread over 32 words
constexpr unsigned long long kEmptyKey = TSDF_EMPTY_KEY;
constexpr uint32_t kIndexPending = TSDF_INDEX_PENDING;
constexpr uint32_t kIndexFailed = TSDF_INDEX_FAILED;

// One hash-table slot: the packed block key, the block's pool index, padding.
struct __align__(16) Entry {
    unsigned long long key;
    uint32_t idx;
    uint32_t pad;
};
static_assert(sizeof(Entry) == 16, "table entries are 16 bytes");

struct DeviceCounters {
    unsigned long long pool_exhausted;
    unsigned long long probe_overflow;
    unsigned long long probe_inserts;
    unsigned long long probe_steps;
    unsigned long long probe_max;
    unsigned long long reserved[2];
    unsigned long long publish_timeouts;    // fused integrate: waits for an index that gave up
    unsigned long long probe_hist[TSDF_PROBE_HIST_BINS];
    unsigned long long missed[kCounterStripes];
    unsigned long long out_of_range[kCounterStripes];
    unsigned long long valid_points[kCounterStripes];
    unsigned long long voxel_updates[kCounterStripes];
};

// Camera intrinsics and camera-to-world pose, by value in every launch.
struct Camera {
    float fx, fy, cx, cy;
    float r00, r01, r02, r10, r11, r12, r20, r21, r22;   // R, row-major
    float tx, ty, tz;                                   // t
    // Bounds with which the allocate kernel proves, before testing, that a
    // band sample passes the ray-depth occlusion test (sure_pass in
    // tsdf_device.cuh; computed on the host from the pose, the voxel edge
    // and the truncation, each rounded towards the safe side):
    float sure_tau;     // trunc / voxel - (sqrt(3) / 2) |R column 2| - 1e-3; -inf: never
    float sure_near;    // (sqrt(3) / 2) |R column 2| + 1e-2
    float sure_err;     // 64 * 2^-24 + 4 * max |R^T R - I|: rounding per voxel of magnitude
    float sure_tmag;    // (|tx| + |ty| + |tz|) / voxel
};

// The two divisors of the walk with their float reciprocals.
struct DivisorPair {
    float voxel, inv_voxel;
    float trunc, inv_trunc;
};

// Everything a kernel needs to reach a volume.
struct VolumeView {
    Entry* table;
    uint32_t table_mask;        // table_capacity - 1
    uint32_t pool_capacity;
    // The pool's five sums per voxel; voxel j of block b is v = b * 512 + j.
    // Interleaved layout (the default): tsdf, weight, red and green of voxel
    // v in one 16-byte record voxel4[v] (a sample reaches them with one
    // 4-wide reduction).  Planar layout (five separate arrays): field k
    // (tsdf, weight, red, green) of voxel v at float k * plane + v from
    // voxel4.  Blue is blue[v] in both.
    float4* voxel4;             // [pool_capacity][512] records, or the planar arrays' base
    float* blue;                // [pool_capacity][512]
    size_t plane;               // voxels per array: pool_capacity * 512
    bool planar;                // TSDF_LAYOUT_PLANAR
    uint32_t* pool_counter;     // bump allocator for pool indices
    DeviceCounters* counters;
    DivisorPair div;            // voxel size and truncation, with reciprocals
    bool fast_div;              // the fixed-divisor division was verified exact
    bool fast_voxel;            // ... and the one by the voxel edge (back-projection)
    int band_half;              // samples at offsets -band_half .. band_half voxels
    int occlusion;              // TSDF_OCCLUSION_RAY or TSDF_OCCLUSION_REPROJECT
    // Adaptive update: the dense 16 x 16 pixel tiles of the current update
    // launch, (frame << 24 | tile), listed by the per-sample kernel for the
    // pre-reducing one; dense_next is the latter's work counter.
    uint32_t* dense_list;       // [dense_capacity]
    uint32_t dense_capacity;
    uint32_t* dense_count;
    uint32_t* dense_next;
    uint32_t* dense_done;       // blocks of the pre-reducing kernel that have finished;
                                // the last one sets all three back to zero
};

struct FrameView {
    const float* depth;         // [height][width]
    const float* rgb;           // [height][width][3] (update only)
    Camera cam;
};

// Up to kMaxBatch frames of one size, processed by one launch of each kernel;
// blocks of threads are ordered region-major, frame-minor, so the frames'
// work on the same part of the scene runs close together in time and their
// reductions on a voxel meet in L2.  Measured on the room walk: 8, 16, 32 and
// 64 frames per launch gave 7.6, 8.2, 8.7 and 8.9 G points/s with the first
// kernels, and 64 against 32 saves 1.9 % of the two stages with the current
// ones (allocate 4.5 %, update 1.0 %); the launch parameters are then 6 KB
// and the host-batch staging two buffers of 64 frames.
constexpr int kMaxBatch = 64;
constexpr uint32_t kDenseListCapacity = 1u << 20;

// Division of an index x < 2^31 by a divisor 1 <= d < 2^31 that is fixed for
// a launch, by one multiply-high and a shift (T. Granlund and P. Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994).  With
// l = ceil(log2 d) and m = ceil(2^(31+l) / d) (below 2^32: d > 2^(l-1)),
//     x / d = floor(x m / 2^(31+l)) = umulhi(2x, m) >> l,
// since x m / 2^(31+l) - x / d = x (m d - 2^(31+l)) / (d 2^(31+l)) lies in
// [0, 1/d) for x < 2^31, too little to reach the next integer.  The kernels'
// indices (grid positions, pixel and tile indices) stay below 2^31: frames
// hold at most 2^30 pixels.
struct IndexDivisor {
    uint32_t d;
    uint32_t m;
    uint32_t l;
};

inline IndexDivisor make_index_divisor(uint32_t d)
{
    uint32_t l = 0;
    while (l < 31 && (1u << l) < d) ++l;
    const uint64_t p = 1ull << (31 + l);
    return {d, (uint32_t)((p + d - 1) / d), l};
}

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t divide_index(const IndexDivisor& q, uint32_t x)
{
    return __umulhi(x << 1, q.m) >> q.l;
}
#endif

struct FrameBatch {
    int n;
    int width;
    int height;
    // n, width and the frame's widths in 16- and 8-pixel tiles, as divisors
    IndexDivisor by_n, by_width, by_tiles16_x, by_tiles8_x;
    // The pixels' rays for the batch's intrinsics (build_rays): for pixel
    // (u, v), rays[v * width + u] = (dx, dy, dz, xn), the unit viewing ray
    // (xn, yn, 1) / |(xn, yn, 1)| and xn = (u - cx) / fx; ray_yn[v] =
    // (v - cy) / fy.
    const float4* rays;
    const float* ray_yn;
    FrameView frame[kMaxBatch];
};

cudaError_t launch_allocate(const VolumeView& vol, const FrameBatch& fb, bool instrument,
                            cudaStream_t stream);
// Allocate and update in one kernel (bands of at most 9 samples, the ray
// occlusion test).
cudaError_t launch_integrate_fused(const VolumeView& vol, const FrameBatch& fb, bool instrument,
                                   cudaStream_t stream);
cudaError_t launch_allocate_blocks(const VolumeView& vol, const int32_t* coords, uint32_t n,
                                   bool instrument, cudaStream_t stream);
// kind: TSDF_UPDATE_ADAPTIVE, TSDF_UPDATE_PER_SAMPLE or TSDF_UPDATE_PRE_REDUCED.
// With the reprojection occlusion test every kind runs the per-sample kernel.
cudaError_t launch_update(const VolumeView& vol, const FrameBatch& fb, int kind,
                          cudaStream_t stream);
// All 2^32 float32 bit patterns x tried against IEEE division by y, the
// count of mismatches added to *mismatches.  kDivideTrunc: x >= -y, compared
// as min(1, x / y) (the truncated distance); kDivideVoxel: every x, compared
// bit for bit (the back-projection's division by the voxel edge).
enum DivisorCheck { kDivideTrunc = 0, kDivideVoxel = 1 };
cudaError_t launch_verify_fixed_divisor(float y, float inv_y, int check,
                                        unsigned long long* mismatches, cudaStream_t stream);
// The rays of every pixel of a width x height image for intrinsics
// (fx, fy, cx, cy), written to rays and ray_yn as FrameBatch describes.
cudaError_t launch_build_rays(float fx, float fy, float cx, float cy, int width, int height,
                              float4* rays, float* ray_yn, cudaStream_t stream);
cudaError_t launch_zero_used_blocks(const VolumeView& vol, cudaStream_t stream);
// Marching tetrahedra over blocks [0, n_blocks) (coords[idx] = coordinate of
// pool index idx); triangles past `capacity` are counted, not written.
cudaError_t launch_extract(const VolumeView& vol, const int32_t* coords, uint32_t n_blocks,
                           uint32_t* neighbours, float* out, uint64_t capacity,
                           unsigned long long* count, cudaStream_t stream);
// Copy block i's five sums (src: [5][n][512], the order tsdf, weight, red,
// green, blue) to the pool slot the table gives its coordinate (inserted
// beforehand).
cudaError_t launch_import(const VolumeView& vol, const int32_t* coords, uint32_t n,
                          const float* src, cudaStream_t stream);
cudaError_t launch_export_coords(const VolumeView& vol, int32_t* coords, cudaStream_t stream);
// Split voxel records [first, first + n) into four planes of n floats each
// (tsdf, weight, red, green) at out.
cudaError_t launch_split_records(const VolumeView& vol, size_t first, size_t n, float* out,
                                 cudaStream_t stream);

}  // namespace tsdf

// Internal accessors for translation units other than the volume's own.
struct tsdf_volume;
namespace tsdf {
VolumeView volume_view(const tsdf_volume* vol);
int record_error(int code, const char* message);   // sets tsdf_last_error, returns code
// Device address of the no-allocation export's scratch array on the current
// device (looked up at volume creation; tsdf_noalloc.cu).
int resolve_noalloc_scratch(int32_t** out);
int32_t* noalloc_scratch_of(const tsdf_volume* vol);
}  // namespace tsdf
