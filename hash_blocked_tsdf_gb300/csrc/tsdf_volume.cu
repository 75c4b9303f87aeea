// Host side of libtsdf.so: the C ABI declared in include/tsdf.h.  It owns
// the volume's device memory, validates every argument before enqueueing
// anything, and launches the kernels on the caller's stream.
#include <algorithm>
#include <array>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <limits>
#include <new>
#include <string>
#include <vector>

#include "tsdf_internal.h"

using namespace tsdf;

namespace {

// Blocks per chunk when export splits the interleaved layout's voxel records
// and blue sums into planes (16,384 blocks: a 160 MB scratch buffer).
// In the default update mode, integrate launches of fewer pixels than this
// (frames x width x height) run the fused kernel: measured on GB300, one
// fused launch took 0.039 / 0.046 / 0.077 ms against 0.054 / 0.061 / 0.079 ms
// for allocate + update at 160x120 / 320x240 / 640x480, and 0.205 against
// 0.194 ms at 1280x960, where the two kernels fill the GPU.
constexpr uint64_t kAutoFusedPixels = 1ull << 19;
constexpr uint32_t kExportChunkBlocks = 1u << 14;
// tsdf_integrate_batch_host: frames in its first group (later groups grow
// to kMaxBatch).  On GB300 with 1280x720 frames, a 64-frame group's copy
// takes ~4.5 ms, all of it before the first kernel when the first group is a
// full one.
constexpr int kHostFirstGroup = 16;

// Device-resident mutable state: the pool's bump counter and the counters.
struct DeviceState {
    uint32_t pool_counter;
    uint32_t dense_count;       // adaptive update: dense tiles listed in this launch,
    uint32_t dense_next;        // ... taken by the pre-reducing kernel,
    uint32_t dense_done;        // ... whose blocks count out here (all three are zero
                                //     between launches)
    unsigned long long triangles;   // extraction: triangles found
    uint32_t pad[2];
    DeviceCounters counters;
};

}  // namespace

struct tsdf_volume {
    int device = 0;
    uint32_t pool_capacity = 0;
    uint32_t table_capacity = 0;
    float voxel = 0.0f;
    float trunc = 0.0f;
    int band_half = 0;
    bool instrument = false;
    int update_kind = TSDF_UPDATE_AUTO;
    int occlusion = TSDF_OCCLUSION_RAY;
    int layout = TSDF_LAYOUT_INTERLEAVED;
    DivisorPair div = {};
    bool fast_div = false;          // the fixed-divisor division by trunc was verified
    bool fast_voxel = false;        // ... and the one by the voxel edge

    Entry* table = nullptr;
    uint32_t* dense_list = nullptr;  // [kDenseListCapacity] adaptive update's dense tiles
    float* pool = nullptr;          // pool_capacity * 512 voxel records of 4 floats, then
                                    // pool_capacity * 512 blue sums
    DeviceState* state = nullptr;
    int32_t* coords = nullptr;      // [pool_capacity][3], allocated on first export
    uint32_t* neighbours = nullptr; // [pool_capacity][8], allocated on first extraction
    int32_t* noalloc_scratch = nullptr;  // device address of the no-allocation export's
                                         // scratch array, looked up at create
    float* export_scratch = nullptr;  // [5][kExportChunkBlocks][512], allocated on first export

    // the pixels' rays for the last batch's intrinsics and frame size
    // (FrameBatch::rays), allocated on first use and grown for larger frames
    float4* rays = nullptr;
    float* ray_yn = nullptr;
    size_t ray_pixels = 0;          // capacity of rays, in pixels
    int ray_rows = 0;               // capacity of ray_yn
    bool rays_built = false;        // rays hold ray_size / ray_k
    int ray_size[2] = {0, 0};
    float ray_k[4] = {0.0f, 0.0f, 0.0f, 0.0f};

    // host-batch staging: two buffers of (depth, rgb) frames
    float* stage[2] = {nullptr, nullptr};
    size_t stage_pixels = 0;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t copied[2] = {nullptr, nullptr};
    cudaEvent_t consumed[2] = {nullptr, nullptr};
};

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg)
{
    g_last_error = msg;
    return code;
}

int cuda_fail(cudaError_t e, const char* what)
{
    g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
    // take a non-sticky error (a failed allocation, a bad launch argument)
    // off the runtime's last-error slot, so that the launch check of a later
    // call does not report it again
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? TSDF_ERR_OOM : TSDF_ERR_CUDA;
}

#define TSDF_CUDA(call, what)                         \
    do {                                              \
        cudaError_t e_ = (call);                      \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

size_t array_floats(const tsdf_volume* v) { return (size_t)v->pool_capacity * kBlockVoxels; }

VolumeView view_of(const tsdf_volume* v)
{
    VolumeView w;
    w.table = v->table;
    w.table_mask = v->table_capacity - 1;
    w.pool_capacity = v->pool_capacity;
    const size_t n = array_floats(v);
    w.voxel4 = reinterpret_cast<float4*>(v->pool);      // n records, or 4 planar arrays
    w.blue = v->pool + 4 * n;
    w.plane = n;
    w.planar = v->layout == TSDF_LAYOUT_PLANAR;
    w.pool_counter = &v->state->pool_counter;
    w.counters = &v->state->counters;
    w.div = v->div;
    w.fast_div = v->fast_div;
    w.fast_voxel = v->fast_voxel;
    w.occlusion = v->occlusion;
    w.band_half = v->band_half;
    w.dense_list = v->dense_list;
    w.dense_capacity = kDenseListCapacity;
    w.dense_count = &v->state->dense_count;
    w.dense_next = &v->state->dense_next;
    w.dense_done = &v->state->dense_done;
    return w;
}

bool is_pow2(uint64_t x) { return x && !(x & (x - 1)); }

int make_camera(const float* K, const float* pose, Camera* c)
{
    if (!K || !pose) return fail(TSDF_ERR_ARG, "K and pose must be non-null host arrays");
    for (int i = 0; i < 4; ++i)
        if (!std::isfinite(K[i])) return fail(TSDF_ERR_ARG, "K has a non-finite entry");
    if (K[0] == 0.0f || K[1] == 0.0f) return fail(TSDF_ERR_ARG, "fx and fy must be non-zero");
    for (int i = 0; i < 12; ++i)
        if (!std::isfinite(pose[i])) return fail(TSDF_ERR_ARG, "pose has a non-finite entry");
    c->fx = K[0];
    c->fy = K[1];
    c->cx = K[2];
    c->cy = K[3];
    c->r00 = pose[0]; c->r01 = pose[1]; c->r02 = pose[2];  c->tx = pose[3];
    c->r10 = pose[4]; c->r11 = pose[5]; c->r12 = pose[6];  c->ty = pose[7];
    c->r20 = pose[8]; c->r21 = pose[9]; c->r22 = pose[10]; c->tz = pose[11];
    return TSDF_OK;
}

// The bounds of Camera::sure_* for a volume of voxel edge `voxel` and
// truncation `trunc`.  Where the pose is far from a rotation (an entry of
// R^T R - I above 1e-3) the proof is not attempted (sure_tau = -inf).
void sure_pass_bounds(float voxel, float trunc, Camera* c)
{
    const double R[3][3] = {{c->r00, c->r01, c->r02}, {c->r10, c->r11, c->r12},
                            {c->r20, c->r21, c->r22}};
    double defect = 0.0;
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) {
            double g = 0.0;
            for (int k = 0; k < 3; ++k) g += R[k][i] * R[k][j];
            defect = std::max(defect, std::fabs(g - (i == j ? 1.0 : 0.0)));
        }
    const double s3n2 = 0.5 * std::sqrt(3.0) *
                        std::sqrt(R[0][2] * R[0][2] + R[1][2] * R[1][2] + R[2][2] * R[2][2]);
    const double tau = (double)trunc / (double)voxel - s3n2 - 1e-3;
    const double tmag = (std::fabs((double)c->tx) + std::fabs((double)c->ty) +
                         std::fabs((double)c->tz)) / (double)voxel;
    const float inf = std::numeric_limits<float>::infinity();
    if (!(defect <= 1e-3) || !std::isfinite(tmag)) {
        c->sure_tau = -inf;
        c->sure_near = inf;
        c->sure_err = inf;
        c->sure_tmag = inf;
        return;
    }
    c->sure_tau = std::nextafter((float)tau, -inf);
    c->sure_near = std::nextafter((float)(s3n2 + 1e-2), inf);
    c->sure_err = std::nextafter((float)(64.0 * 0x1p-24 + 4.0 * defect), inf);
    c->sure_tmag = std::nextafter((float)tmag, inf);
}

int check_size(int width, int height)
{
    if (width <= 0 || height <= 0) return fail(TSDF_ERR_ARG, "width and height must be positive");
    if ((int64_t)width * (int64_t)height > (int64_t)1 << 30)
        return fail(TSDF_ERR_ARG, "width * height exceeds 2^30 pixels");
    return TSDF_OK;
}

// Every call that touches the volume's device memory runs with the volume's
// device current; a call from another device would hand that device's
// kernels pointers into the wrong GPU's memory.
int check_volume(const tsdf_volume* v)
{
    if (!v) return fail(TSDF_ERR_ARG, "volume is null");
    int dev = -1;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != v->device)
        return fail(TSDF_ERR_ARG, "the current CUDA device is " + std::to_string(dev) +
                                      " but the volume lives on device " +
                                      std::to_string(v->device) +
                                      ": call cudaSetDevice with the volume's device first");
    return TSDF_OK;
}

int ensure_staging(tsdf_volume* v, size_t pixels)
{
    if (!v->copy_stream) {
        TSDF_CUDA(cudaStreamCreateWithFlags(&v->copy_stream, cudaStreamNonBlocking),
                  "cudaStreamCreateWithFlags");
        for (int b = 0; b < 2; ++b) {
            TSDF_CUDA(cudaEventCreateWithFlags(&v->copied[b], cudaEventDisableTiming),
                      "cudaEventCreateWithFlags");
            TSDF_CUDA(cudaEventCreateWithFlags(&v->consumed[b], cudaEventDisableTiming),
                      "cudaEventCreateWithFlags");
        }
    }
    if (v->stage_pixels >= pixels) return TSDF_OK;
    for (int b = 0; b < 2; ++b) {
        if (v->stage[b]) {
            TSDF_CUDA(cudaEventSynchronize(v->consumed[b]), "cudaEventSynchronize");
            TSDF_CUDA(cudaFree(v->stage[b]), "cudaFree");
            v->stage[b] = nullptr;
        }
    }
    v->stage_pixels = 0;
    for (int b = 0; b < 2; ++b)
        TSDF_CUDA(cudaMalloc(&v->stage[b], pixels * 4 * sizeof(float)), "cudaMalloc(staging)");
    v->stage_pixels = pixels;
    return TSDF_OK;
}

void release(tsdf_volume* v)
{
    if (v->table) cudaFree(v->table);
    if (v->dense_list) cudaFree(v->dense_list);
    if (v->pool) cudaFree(v->pool);
    if (v->export_scratch) cudaFree(v->export_scratch);
    if (v->state) cudaFree(v->state);
    if (v->coords) cudaFree(v->coords);
    if (v->neighbours) cudaFree(v->neighbours);
    if (v->rays) cudaFree(v->rays);
    if (v->ray_yn) cudaFree(v->ray_yn);
    for (int b = 0; b < 2; ++b) {
        if (v->stage[b]) cudaFree(v->stage[b]);
        if (v->copied[b]) cudaEventDestroy(v->copied[b]);
        if (v->consumed[b]) cudaEventDestroy(v->consumed[b]);
    }
    if (v->copy_stream) cudaStreamDestroy(v->copy_stream);
    delete v;
}

// Make the volume's ray table hold the rays of a width x height image for
// the intrinsics of camera c, building it on `stream` unless it already
// does.  Under stream capture the build is always recorded (a replay must
// not depend on the table's state outside the graph), and the table must
// already be large enough: allocating synchronises the device.
int ensure_rays(tsdf_volume* v, int width, int height, const Camera& c, cudaStream_t stream)
{
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    TSDF_CUDA(cudaStreamIsCapturing(stream, &cap), "cudaStreamIsCapturing");
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    const size_t px = (size_t)width * (size_t)height;
    if (v->ray_pixels < px || v->ray_rows < height) {
        if (capturing)
            return fail(TSDF_ERR_ARG, "the first integrate call for a frame size allocates the "
                                      "ray table and must not be made during stream capture");
        if (v->rays) cudaFree(v->rays);
        if (v->ray_yn) cudaFree(v->ray_yn);
        v->rays = nullptr;
        v->ray_yn = nullptr;
        v->ray_pixels = 0;
        v->ray_rows = 0;
        v->rays_built = false;
        TSDF_CUDA(cudaMalloc(&v->rays, px * sizeof(float4)), "cudaMalloc(rays)");
        TSDF_CUDA(cudaMalloc(&v->ray_yn, (size_t)height * sizeof(float)), "cudaMalloc(rays)");
        v->ray_pixels = px;
        v->ray_rows = height;
    }
    const bool same = v->rays_built && v->ray_size[0] == width && v->ray_size[1] == height &&
                      v->ray_k[0] == c.fx && v->ray_k[1] == c.fy && v->ray_k[2] == c.cx &&
                      v->ray_k[3] == c.cy;
    if (same && !capturing) return TSDF_OK;
    v->rays_built = false;
    TSDF_CUDA(launch_build_rays(c.fx, c.fy, c.cx, c.cy, width, height, v->rays, v->ray_yn,
                                stream), "build_rays kernel");
    v->rays_built = true;
    v->ray_size[0] = width;
    v->ray_size[1] = height;
    v->ray_k[0] = c.fx;
    v->ray_k[1] = c.fy;
    v->ray_k[2] = c.cx;
    v->ray_k[3] = c.cy;
    return TSDF_OK;
}

// Launch the allocate and/or update kernels over n_frames frames laid out
// back to back (depth [n][H][W], rgb [n][H][W][3]), at most kMaxBatch frames
// per launch.  With `interleave`, each group's update follows its allocate;
// otherwise every allocate launch precedes every update launch.
int batch_kernels(tsdf_volume* v, int n_frames, const float* depth, const float* rgb,
                  int width, int height, const Camera* cams, bool do_allocate, bool do_update,
                  cudaStream_t stream)
{
    const VolumeView vol = view_of(v);
    const size_t px = (size_t)width * (size_t)height;
    if (n_frames > 0) {
        // one intrinsics matrix per call: every frame's camera has the same
        const int rc = ensure_rays(v, width, height, cams[0], stream);
        if (rc) return rc;
    }
    for (int first = 0; first < n_frames; first += kMaxBatch) {
        FrameBatch fb;
        fb.n = n_frames - first < kMaxBatch ? n_frames - first : kMaxBatch;
        fb.width = width;
        fb.height = height;
        fb.by_n = make_index_divisor((uint32_t)fb.n);
        fb.by_width = make_index_divisor((uint32_t)width);
        fb.by_tiles16_x = make_index_divisor((uint32_t)((width + 15) / 16));
        fb.by_tiles8_x = make_index_divisor((uint32_t)((width + 7) / 8));
        fb.rays = v->rays;
        fb.ray_yn = v->ray_yn;
        for (int f = 0; f < fb.n; ++f) {
            fb.frame[f].depth = depth + (first + f) * px;
            fb.frame[f].rgb = rgb ? rgb + 3 * (first + f) * px : nullptr;
            fb.frame[f].cam = cams[first + f];
        }
        // one fused kernel instead of allocate + update: always in the fused
        // mode, and in the default mode for launches too small to fill the
        // GPU, where the two kernels' latencies add up
        const bool small = (uint64_t)px * (uint64_t)fb.n < kAutoFusedPixels;
        const bool fuse = v->update_kind == TSDF_UPDATE_FUSED ||
                          (v->update_kind == TSDF_UPDATE_AUTO && small);
        if (do_allocate && do_update && fuse && v->occlusion == TSDF_OCCLUSION_RAY &&
            2 * v->band_half + 1 <= 9) {
            TSDF_CUDA(launch_integrate_fused(vol, fb, v->instrument, stream), "fused kernel");
            continue;
        }
        if (do_allocate)
            TSDF_CUDA(launch_allocate(vol, fb, v->instrument, stream), "allocate kernel");
        if (do_update) {
            const int kind = (v->update_kind == TSDF_UPDATE_FUSED ||
                              v->update_kind == TSDF_UPDATE_AUTO) ? TSDF_UPDATE_PER_SAMPLE
                                                                  : v->update_kind;
            TSDF_CUDA(launch_update(vol, fb, kind, stream), "update kernel");
        }
    }
    return TSDF_OK;
}

int check_batch(tsdf_volume* v, int n_frames, const float* depth, const float* rgb, int width,
                int height, const float* K, const float* poses, bool need_rgb,
                std::vector<Camera>* cams)
{
    int rc = check_volume(v);
    if (rc) return rc;
    if (n_frames < 0) return fail(TSDF_ERR_ARG, "n_frames must be >= 0");
    if ((rc = check_size(width, height))) return rc;
    if (n_frames > 0 && (!depth || !poses || (need_rgb && !rgb)))
        return fail(TSDF_ERR_ARG, "null frame pointer");
    cams->resize((size_t)n_frames);
    for (int f = 0; f < n_frames; ++f)
        if ((rc = make_camera(K, poses + 16 * (size_t)f, &(*cams)[f]))) return rc;
    for (int f = 0; f < n_frames; ++f) sure_pass_bounds(v->voxel, v->trunc, &(*cams)[f]);
    return TSDF_OK;
}

int one_frame(tsdf_volume* v, const float* depth, const float* rgb, int width, int height,
              const float K[4], const float pose[16], void* stream, bool do_allocate,
              bool do_update)
{
    std::vector<Camera> cams;
    int rc = check_batch(v, 1, depth, rgb, width, height, K, pose, do_update, &cams);
    if (rc) return rc;
    return batch_kernels(v, 1, depth, rgb, width, height, cams.data(), do_allocate, do_update,
                         as_stream(stream));
}

// Check, for every float32 dividend, that the walk's truncated distances
// and the back-projection's divisions by the voxel edge come out the same
// with the fixed-divisor division as with IEEE division; each is used only
// where its check passed.
int verify_divisors(tsdf_volume* v)
{
    unsigned long long* bad = &v->state->counters.reserved[0];
    unsigned long long h[2] = {1, 1};
    const float y[2] = {v->div.trunc, v->div.voxel};
    const float r[2] = {v->div.inv_trunc, v->div.inv_voxel};
    const int check[2] = {kDivideTrunc, kDivideVoxel};
    for (int k = 0; k < 2; ++k) {
        TSDF_CUDA(cudaMemsetAsync(bad, 0, sizeof(unsigned long long), 0), "cudaMemsetAsync");
        TSDF_CUDA(launch_verify_fixed_divisor(y[k], r[k], check[k], bad, 0), "verify kernel");
        TSDF_CUDA(cudaMemcpyAsync(&h[k], bad, sizeof(h[k]), cudaMemcpyDeviceToHost, 0),
                  "cudaMemcpyAsync");
        TSDF_CUDA(cudaStreamSynchronize(0), "cudaStreamSynchronize");
    }
    TSDF_CUDA(cudaMemsetAsync(bad, 0, sizeof(unsigned long long), 0), "cudaMemsetAsync");
    TSDF_CUDA(cudaStreamSynchronize(0), "cudaStreamSynchronize");
    v->fast_div = h[0] == 0;
    v->fast_voxel = h[1] == 0;
    return TSDF_OK;
}

}  // namespace

namespace tsdf {
VolumeView volume_view(const tsdf_volume* vol) { return view_of(vol); }
int32_t* noalloc_scratch_of(const tsdf_volume* vol) { return vol->noalloc_scratch; }
int record_error(int code, const char* message) { return fail(code, message); }
}  // namespace tsdf

extern "C" {

const char* tsdf_last_error(void) { return g_last_error.c_str(); }

int tsdf_create_ex(uint32_t pool_capacity, uint32_t table_capacity, float voxel_size, float trunc,
                   tsdf_volume** out)
{
    if (!out) return fail(TSDF_ERR_ARG, "out is null");
    *out = nullptr;
    if (pool_capacity < 1 || pool_capacity > TSDF_MAX_POOL_CAPACITY)
        return fail(TSDF_ERR_ARG, "pool_capacity must be in [1, 2^23]");
    if (!std::isfinite(voxel_size) || !(voxel_size > 0.0f) || !std::isfinite(trunc) ||
        !(trunc > 0.0f))
        return fail(TSDF_ERR_ARG, "voxel_size and trunc must be finite and positive");
    const double ratio = std::round((double)trunc / (double)voxel_size);
    if (2.0 * ratio + 1.0 > TSDF_MAX_BAND_SAMPLES)
        return fail(TSDF_ERR_ARG, "trunc / voxel_size is too large");
    uint64_t T = table_capacity;
    if (T == 0) {
        T = 1;
        while (T <= 2ull * pool_capacity) T <<= 1;     // strictly above twice the pool
    } else if (!is_pow2(T) || T < 2ull * pool_capacity) {
        return fail(TSDF_ERR_ARG, "table_capacity must be a power of two >= 2 * pool_capacity");
    }
    if (T > TSDF_MAX_TABLE_CAPACITY) return fail(TSDF_ERR_ARG, "table_capacity exceeds 2^30");

    tsdf_volume* v = new (std::nothrow) tsdf_volume();
    if (!v) return fail(TSDF_ERR_OOM, "host allocation failed");
    v->pool_capacity = pool_capacity;
    v->table_capacity = (uint32_t)T;
    v->voxel = voxel_size;
    v->trunc = trunc;
    v->band_half = (int)ratio;
    v->div.voxel = voxel_size;
    v->div.inv_voxel = 1.0f / voxel_size;     // IEEE reciprocal, correctly rounded
    v->div.trunc = trunc;
    v->div.inv_trunc = 1.0f / trunc;
    cudaError_t e = cudaGetDevice(&v->device);
    const size_t pool_bytes = 5 * array_floats(v) * sizeof(float);
    if (e == cudaSuccess) e = cudaMalloc(&v->table, T * sizeof(Entry));
    if (e == cudaSuccess) e = cudaMalloc(&v->dense_list, kDenseListCapacity * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMalloc(&v->pool, pool_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&v->state, sizeof(DeviceState));
    if (e == cudaSuccess) e = cudaMemsetAsync(v->pool, 0, pool_bytes, 0);
    if (e == cudaSuccess) e = cudaMemsetAsync(v->table, 0xFF, T * sizeof(Entry), 0);
    if (e == cudaSuccess) e = cudaMemsetAsync(v->state, 0, sizeof(DeviceState), 0);
    if (e == cudaSuccess) e = cudaStreamSynchronize(0);
    if (e != cudaSuccess) {
        int rc = cuda_fail(e, "tsdf_create");
        release(v);
        cudaGetLastError();
        return rc;
    }
    int rc = verify_divisors(v);
    // the no-allocation export's scratch address, looked up now so that the
    // module holding the array is loaded here and not in that call
    if (!rc) rc = resolve_noalloc_scratch(&v->noalloc_scratch);
    if (rc) {
        release(v);
        return rc;
    }
    *out = v;
    return TSDF_OK;
}

int tsdf_create(uint32_t pool_capacity, float voxel_size, float trunc, tsdf_volume** out)
{
    return tsdf_create_ex(pool_capacity, 0, voxel_size, trunc, out);
}

int tsdf_destroy(tsdf_volume* vol)
{
    if (!vol) return fail(TSDF_ERR_ARG, "volume is null");
    // free on the volume's own device, then restore the caller's; the copy
    // stream of the host-batch call is the only stream the volume owns
    const int dev = vol->device;
    int prev = -1;
    cudaError_t e = cudaGetDevice(&prev);
    if (e == cudaSuccess && prev != dev) e = cudaSetDevice(dev);
    if (e == cudaSuccess && vol->copy_stream) e = cudaStreamSynchronize(vol->copy_stream);
    release(vol);
    if (prev >= 0 && prev != dev) cudaSetDevice(prev);
    if (e != cudaSuccess) return cuda_fail(e, "tsdf_destroy");
    return TSDF_OK;
}

int tsdf_get_info(const tsdf_volume* vol, tsdf_info* out)
{
    if (!vol || !out) return fail(TSDF_ERR_ARG, "null argument");
    out->pool_capacity = vol->pool_capacity;
    out->table_capacity = vol->table_capacity;
    out->voxel_size = vol->voxel;
    out->trunc = vol->trunc;
    out->band_samples = 2 * vol->band_half + 1;
    out->device = vol->device;
    out->fixed_divisor_fast_path = vol->fast_div ? 1 : 0;
    out->voxel_division_fast_path = vol->fast_voxel ? 1 : 0;
    out->max_frames_per_launch = kMaxBatch;
    out->pool_layout = vol->layout;
    return TSDF_OK;
}

int tsdf_get_pool(const tsdf_volume* vol, tsdf_pool_view* out)
{
    if (!vol || !out) return fail(TSDF_ERR_ARG, "null argument");
    const VolumeView w = view_of(vol);
    float* base = reinterpret_cast<float*>(w.voxel4);
    // interleaved: field k of voxel v at base + 4 v + k; planar: base + k n + v
    const size_t step = w.planar ? w.plane : 1;
    out->tsdf = base;
    out->weight = base + step;
    out->r = base + 2 * step;
    out->g = base + 3 * step;
    out->b = w.blue;
    out->pool_capacity = vol->pool_capacity;
    out->stride = w.planar ? 1 : 4;
    return TSDF_OK;
}

int tsdf_reset(tsdf_volume* vol, void* stream)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    cudaStream_t s = as_stream(stream);
    TSDF_CUDA(launch_zero_used_blocks(view_of(vol), s), "zero kernel");
    TSDF_CUDA(cudaMemsetAsync(vol->table, 0xFF, (size_t)vol->table_capacity * sizeof(Entry), s),
              "cudaMemsetAsync(table)");
    TSDF_CUDA(cudaMemsetAsync(vol->state, 0, sizeof(DeviceState), s), "cudaMemsetAsync(state)");
    return TSDF_OK;
}

int tsdf_integrate(tsdf_volume* vol, const float* depth, const float* rgb, int width, int height,
                   const float K[4], const float pose[16], void* stream)
{
    return one_frame(vol, depth, rgb, width, height, K, pose, stream, true, true);
}

int tsdf_allocate(tsdf_volume* vol, const float* depth, int width, int height, const float K[4],
                  const float pose[16], void* stream)
{
    return one_frame(vol, depth, nullptr, width, height, K, pose, stream, true, false);
}

int tsdf_update(tsdf_volume* vol, const float* depth, const float* rgb, int width, int height,
                const float K[4], const float pose[16], void* stream)
{
    return one_frame(vol, depth, rgb, width, height, K, pose, stream, false, true);
}

int tsdf_integrate_batch(tsdf_volume* vol, int n_frames, const float* depth, const float* rgb,
                         int width, int height, const float K[4], const float* poses,
                         void* stream)
{
    std::vector<Camera> cams;
    int rc = check_batch(vol, n_frames, depth, rgb, width, height, K, poses, true, &cams);
    if (rc || n_frames == 0) return rc;
    return batch_kernels(vol, n_frames, depth, rgb, width, height, cams.data(), true, true,
                         as_stream(stream));
}

int tsdf_allocate_batch(tsdf_volume* vol, int n_frames, const float* depth, int width,
                        int height, const float K[4], const float* poses, void* stream)
{
    std::vector<Camera> cams;
    int rc = check_batch(vol, n_frames, depth, nullptr, width, height, K, poses, false, &cams);
    if (rc || n_frames == 0) return rc;
    return batch_kernels(vol, n_frames, depth, nullptr, width, height, cams.data(), true, false,
                         as_stream(stream));
}

int tsdf_update_batch(tsdf_volume* vol, int n_frames, const float* depth, const float* rgb,
                      int width, int height, const float K[4], const float* poses, void* stream)
{
    std::vector<Camera> cams;
    int rc = check_batch(vol, n_frames, depth, rgb, width, height, K, poses, true, &cams);
    if (rc || n_frames == 0) return rc;
    return batch_kernels(vol, n_frames, depth, rgb, width, height, cams.data(), false, true,
                         as_stream(stream));
}

int tsdf_integrate_batch_host(tsdf_volume* vol, int n_frames, const float* depth_host,
                              const float* rgb_host, int width, int height, const float K[4],
                              const float* poses, void* stream)
{
    std::vector<Camera> cams;
    int rc = check_batch(vol, n_frames, depth_host, rgb_host, width, height, K, poses, true,
                         &cams);
    if (rc || n_frames == 0) return rc;
    const size_t px = (size_t)width * (size_t)height;
    if ((rc = ensure_staging(vol, px * kMaxBatch))) return rc;
    cudaStream_t s = as_stream(stream);
    // The kernels of a group wait for its copy, and nothing hides the first
    // copy; so the groups start small and grow by about a third each, which
    // the copies (faster per frame than the kernels) keep up with, up to
    // full launches.
    int size = kHostFirstGroup;
    int n = 0;
    int group = 0;
    for (int first = 0; first < n_frames; first += n, ++group) {
        n = std::min(std::min(size, kMaxBatch), n_frames - first);
        size = std::min(kMaxBatch, size + std::max(1, size / 3));
        const int b = group & 1;
        float* d_dev = vol->stage[b];
        float* c_dev = vol->stage[b] + px * kMaxBatch;
        // the copy into buffer b waits for the kernels that last read it
        TSDF_CUDA(cudaStreamWaitEvent(vol->copy_stream, vol->consumed[b], 0), "cudaStreamWaitEvent");
        TSDF_CUDA(cudaMemcpyAsync(d_dev, depth_host + first * px, n * px * sizeof(float),
                                  cudaMemcpyHostToDevice, vol->copy_stream), "cudaMemcpyAsync(depth)");
        TSDF_CUDA(cudaMemcpyAsync(c_dev, rgb_host + 3 * first * px, 3 * n * px * sizeof(float),
                                  cudaMemcpyHostToDevice, vol->copy_stream), "cudaMemcpyAsync(rgb)");
        TSDF_CUDA(cudaEventRecord(vol->copied[b], vol->copy_stream), "cudaEventRecord");
        TSDF_CUDA(cudaStreamWaitEvent(s, vol->copied[b], 0), "cudaStreamWaitEvent");
        rc = batch_kernels(vol, n, d_dev, c_dev, width, height, cams.data() + first, true, true, s);
        if (rc) return rc;
        TSDF_CUDA(cudaEventRecord(vol->consumed[b], s), "cudaEventRecord");
    }
    return TSDF_OK;
}

int tsdf_allocate_blocks(tsdf_volume* vol, const int32_t* coords, uint32_t n, void* stream)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    if (n == 0) return TSDF_OK;
    if (!coords) return fail(TSDF_ERR_ARG, "coords is null");
    if (n > (1u << 30)) return fail(TSDF_ERR_ARG, "n exceeds 2^30");
    TSDF_CUDA(launch_allocate_blocks(view_of(vol), coords, n, vol->instrument, as_stream(stream)),
              "allocate_blocks kernel");
    return TSDF_OK;
}

int tsdf_block_count(tsdf_volume* vol, void* stream, uint32_t* out)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    if (!out) return fail(TSDF_ERR_ARG, "out is null");
    uint32_t counter = 0;
    cudaStream_t s = as_stream(stream);
    TSDF_CUDA(cudaMemcpyAsync(&counter, &vol->state->pool_counter, sizeof(uint32_t),
                              cudaMemcpyDeviceToHost, s), "cudaMemcpyAsync(count)");
    TSDF_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    *out = counter < vol->pool_capacity ? counter : vol->pool_capacity;
    return TSDF_OK;
}

int tsdf_export_blocks(tsdf_volume* vol, void* stream, uint32_t first, uint32_t count,
                       int32_t* coords, float* tsdf_out, float* weight, float* r, float* g,
                       float* b)
{
    uint32_t n = 0;
    int rc = tsdf_block_count(vol, stream, &n);
    if (rc) return rc;
    if ((uint64_t)first + count > n)
        return fail(TSDF_ERR_ARG, "first + count exceeds the number of allocated blocks");
    if (count == 0) return TSDF_OK;
    cudaStream_t s = as_stream(stream);
    if (coords) {
        if (!vol->coords)
            TSDF_CUDA(cudaMalloc(&vol->coords, (size_t)vol->pool_capacity * 3 * sizeof(int32_t)),
                      "cudaMalloc(coords)");
        TSDF_CUDA(launch_export_coords(view_of(vol), vol->coords, s), "export_coords kernel");
        TSDF_CUDA(cudaMemcpyAsync(coords, vol->coords + 3 * (size_t)first,
                                  (size_t)count * 3 * sizeof(int32_t), cudaMemcpyDeviceToHost, s),
                  "cudaMemcpyAsync(coords)");
    }
    const VolumeView w = view_of(vol);
    float* dst[5] = {tsdf_out, weight, r, g, b};
    if (w.planar) {
        // five x-fastest arrays: copied out directly
        for (int a = 0; a < 5; ++a) {
            if (!dst[a]) continue;
            const float* src = a < 4 ? reinterpret_cast<float*>(w.voxel4) + a * w.plane : w.blue;
            TSDF_CUDA(cudaMemcpyAsync(dst[a], src + (size_t)first * kBlockVoxels,
                                      (size_t)count * kBlockVoxels * sizeof(float),
                                      cudaMemcpyDeviceToHost, s), "cudaMemcpyAsync(sums)");
        }
    } else if (tsdf_out || weight || r || g || b) {
        // the brick-ordered records and blue sums are split into x-fastest
        // planes on the device, a chunk of blocks at a time, and each plane is
        // copied out whole
        if (!vol->export_scratch)
            TSDF_CUDA(cudaMalloc(&vol->export_scratch,
                                 (size_t)kExportChunkBlocks * kBlockVoxels * 5 * sizeof(float)),
                      "cudaMalloc(export scratch)");
        for (uint32_t c0 = 0; c0 < count; c0 += kExportChunkBlocks) {
            const uint32_t nb = count - c0 < kExportChunkBlocks ? count - c0 : kExportChunkBlocks;
            const size_t nv = (size_t)nb * kBlockVoxels;
            TSDF_CUDA(launch_split_records(w, ((size_t)first + c0) * kBlockVoxels, nv,
                                           vol->export_scratch, s), "split_records kernel");
            for (int a = 0; a < 5; ++a) {
                if (!dst[a]) continue;
                TSDF_CUDA(cudaMemcpyAsync(dst[a] + (size_t)c0 * kBlockVoxels,
                                          vol->export_scratch + (size_t)a * nv,
                                          nv * sizeof(float), cudaMemcpyDeviceToHost, s),
                          "cudaMemcpyAsync(sums)");
            }
        }
    }
    TSDF_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    return TSDF_OK;
}

int tsdf_extract_triangles(tsdf_volume* vol, void* stream, float* triangles, uint64_t capacity,
                           uint64_t* n_out)
{
    uint32_t n = 0;
    int rc = tsdf_block_count(vol, stream, &n);
    if (rc) return rc;
    if (!n_out) return fail(TSDF_ERR_ARG, "n_out is null");
    if (!triangles && capacity) return fail(TSDF_ERR_ARG, "triangles is null but capacity > 0");
    cudaStream_t s = as_stream(stream);
    if (!vol->coords)
        TSDF_CUDA(cudaMalloc(&vol->coords, (size_t)vol->pool_capacity * 3 * sizeof(int32_t)),
                  "cudaMalloc(coords)");
    const VolumeView w = view_of(vol);
    TSDF_CUDA(launch_export_coords(w, vol->coords, s), "export_coords kernel");
    TSDF_CUDA(cudaMemsetAsync(&vol->state->triangles, 0, sizeof(unsigned long long), s),
              "cudaMemsetAsync(triangles)");
    if (!vol->neighbours)
        TSDF_CUDA(cudaMalloc(&vol->neighbours, (size_t)vol->pool_capacity * 8 * sizeof(uint32_t)),
                  "cudaMalloc(neighbours)");
    TSDF_CUDA(launch_extract(w, vol->coords, n, vol->neighbours, triangles, capacity,
                             &vol->state->triangles, s), "extract kernel");
    unsigned long long total = 0;
    TSDF_CUDA(cudaMemcpyAsync(&total, &vol->state->triangles, sizeof(total),
                              cudaMemcpyDeviceToHost, s), "cudaMemcpyAsync(triangles)");
    TSDF_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    *n_out = total;
    return TSDF_OK;
}

int tsdf_import_blocks(tsdf_volume* vol, void* stream, uint32_t n, const int32_t* coords,
                       const float* tsdf_in, const float* weight, const float* r, const float* g,
                       const float* b)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    if (n == 0) return TSDF_OK;
    if (!coords || !tsdf_in || !weight || !r || !g || !b)
        return fail(TSDF_ERR_ARG, "null host array");
    {
        std::vector<std::array<int32_t, 3>> c(n);
        for (uint32_t i = 0; i < n; ++i) c[i] = {coords[3 * i], coords[3 * i + 1], coords[3 * i + 2]};
        std::sort(c.begin(), c.end());
        for (uint32_t i = 1; i < n; ++i)
            if (c[i] == c[i - 1]) return fail(TSDF_ERR_ARG, "duplicate block coordinate");
    }
    cudaStream_t s = as_stream(stream);
    const size_t n_vals = (size_t)n * kBlockVoxels;
    int32_t* d_coords = nullptr;
    float* d_vals = nullptr;
    cudaError_t e = cudaMalloc(&d_coords, (size_t)n * 3 * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&d_vals, 5 * n_vals * sizeof(float));
    const float* src[5] = {tsdf_in, weight, r, g, b};
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(d_coords, coords, (size_t)n * 3 * sizeof(int32_t),
                            cudaMemcpyHostToDevice, s);
    for (int a = 0; a < 5 && e == cudaSuccess; ++a)
        e = cudaMemcpyAsync(d_vals + a * n_vals, src[a], n_vals * sizeof(float),
                            cudaMemcpyHostToDevice, s);
    const VolumeView w = view_of(vol);
    if (e == cudaSuccess) e = launch_allocate_blocks(w, d_coords, n, vol->instrument, s);
    if (e == cudaSuccess) e = launch_import(w, d_coords, n, d_vals, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (d_coords) cudaFree(d_coords);
    if (d_vals) cudaFree(d_vals);
    if (e != cudaSuccess) return cuda_fail(e, "tsdf_import_blocks");
    return TSDF_OK;
}

int tsdf_export_table(tsdf_volume* vol, void* stream, uint32_t capacity, uint64_t* keys,
                      uint32_t* indices)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    if (capacity != vol->table_capacity)
        return fail(TSDF_ERR_ARG, "capacity must equal the table capacity");
    std::vector<Entry> host(capacity);
    cudaStream_t s = as_stream(stream);
    TSDF_CUDA(cudaMemcpyAsync(host.data(), vol->table, (size_t)capacity * sizeof(Entry),
                              cudaMemcpyDeviceToHost, s), "cudaMemcpyAsync(table)");
    TSDF_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    for (uint32_t i = 0; i < capacity; ++i) {
        if (keys) keys[i] = host[i].key;
        if (indices) indices[i] = host[i].idx;
    }
    return TSDF_OK;
}

int tsdf_get_stats(tsdf_volume* vol, void* stream, tsdf_stats* out)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    if (!out) return fail(TSDF_ERR_ARG, "out is null");
    DeviceState h;
    cudaStream_t s = as_stream(stream);
    TSDF_CUDA(cudaMemcpyAsync(&h, vol->state, sizeof(DeviceState), cudaMemcpyDeviceToHost, s),
              "cudaMemcpyAsync(stats)");
    TSDF_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    std::memset(out, 0, sizeof(*out));
    const DeviceCounters& c = h.counters;
    out->blocks_allocated = h.pool_counter;
    out->pool_exhausted = c.pool_exhausted;
    out->probe_overflow = c.probe_overflow;
    for (int i = 0; i < kCounterStripes; ++i) {
        out->missed_contributions += c.missed[i];
        out->out_of_range_samples += c.out_of_range[i];
        out->valid_points += c.valid_points[i];
        out->voxel_updates += c.voxel_updates[i];
    }
    out->probe_inserts = c.probe_inserts;
    out->probe_steps = c.probe_steps;
    out->probe_max = c.probe_max;
    for (int i = 0; i < TSDF_PROBE_HIST_BINS; ++i) out->probe_hist[i] = c.probe_hist[i];
    out->publish_timeouts = c.publish_timeouts;
    return TSDF_OK;
}

int tsdf_clear_stats(tsdf_volume* vol, void* stream)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    TSDF_CUDA(cudaMemsetAsync(&vol->state->counters, 0, sizeof(DeviceCounters), as_stream(stream)),
              "cudaMemsetAsync(counters)");
    return TSDF_OK;
}

int tsdf_set_instrumentation(tsdf_volume* vol, int on)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    vol->instrument = on != 0;
    return TSDF_OK;
}

int tsdf_set_update_kernel(tsdf_volume* vol, int kind)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    if (kind != TSDF_UPDATE_ADAPTIVE && kind != TSDF_UPDATE_PER_SAMPLE &&
        kind != TSDF_UPDATE_PRE_REDUCED && kind != TSDF_UPDATE_FUSED &&
        kind != TSDF_UPDATE_AUTO)
        return fail(TSDF_ERR_ARG, "update mode must be TSDF_UPDATE_ADAPTIVE, "
                                  "TSDF_UPDATE_PER_SAMPLE, TSDF_UPDATE_PRE_REDUCED, "
                                  "TSDF_UPDATE_FUSED or TSDF_UPDATE_AUTO");
    vol->update_kind = kind;
    return TSDF_OK;
}

int tsdf_set_occlusion(tsdf_volume* vol, int mode)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    if (mode != TSDF_OCCLUSION_RAY && mode != TSDF_OCCLUSION_REPROJECT)
        return fail(TSDF_ERR_ARG, "occlusion must be TSDF_OCCLUSION_RAY or "
                                  "TSDF_OCCLUSION_REPROJECT");
    vol->occlusion = mode;
    return TSDF_OK;
}

int tsdf_set_pool_layout(tsdf_volume* vol, int layout)
{
    int rc = check_volume(vol);
    if (rc) return rc;
    if (layout != TSDF_LAYOUT_INTERLEAVED && layout != TSDF_LAYOUT_PLANAR)
        return fail(TSDF_ERR_ARG, "layout must be TSDF_LAYOUT_INTERLEAVED or TSDF_LAYOUT_PLANAR");
    uint32_t n = 0;
    if ((rc = tsdf_block_count(vol, nullptr, &n))) return rc;
    if (n != 0) return fail(TSDF_ERR_ARG, "the pool layout can only change while the volume is empty");
    vol->layout = layout;
    return TSDF_OK;
}

}  // extern "C"
