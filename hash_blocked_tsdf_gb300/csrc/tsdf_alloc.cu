// Allocate kernel ("What Irregularity Costs", design section, integration:
// the irregular stage).  Every thread walks one pixel's truncation band; the
// block keys of passing samples are de-duplicated, first against the
// thread's previous key, then across the warp with __match_any_sync, and one
// leader per distinct key probes the table and claims an empty slot with a
// single 64-bit compare-and-swap.  Winners of one step take consecutive pool
// indices from one atomicAdd per warp and publish them into their slots.
#include "tsdf_device.cuh"

namespace tsdf {
namespace {

constexpr int kThreads = 256;

// Per-block probe statistics, flushed once per block.
struct ProbeStats {
    unsigned long long hist[TSDF_PROBE_HIST_BINS];
    unsigned long long inserts;
    unsigned long long steps;
    unsigned long long max;
};

__device__ __forceinline__ void record_probe(ProbeStats* st, uint32_t steps)
{
    const int bin = steps > TSDF_PROBE_HIST_BINS ? TSDF_PROBE_HIST_BINS - 1 : (int)steps - 1;
    atomicAdd(&st->hist[bin], 1ull);
    atomicAdd(&st->inserts, 1ull);
    atomicAdd(&st->steps, (unsigned long long)steps);
    atomicMax(&st->max, (unsigned long long)steps);
}

__device__ __forceinline__ void flush_probe_stats(ProbeStats* st, DeviceCounters* c)
{
    __syncthreads();
    const int t = threadIdx.x;
    if (t < TSDF_PROBE_HIST_BINS && st->hist[t]) atomicAdd(&c->probe_hist[t], st->hist[t]);
    if (t == 0) {
        if (st->inserts) atomicAdd(&c->probe_inserts, st->inserts);
        if (st->steps) atomicAdd(&c->probe_steps, st->steps);
        if (st->max) atomicMax(&c->probe_max, st->max);
    }
}

__device__ __forceinline__ void init_probe_stats(ProbeStats* st)
{
    const int t = threadIdx.x;
    if (t < TSDF_PROBE_HIST_BINS) st->hist[t] = 0;
    if (t == 0) st->inserts = st->steps = st->max = 0;
    __syncthreads();
}

// One warp-wide insert step: lanes with `fresh` set offer `key`; equal keys
// are merged, one leader per key probes, and the warp's winners take pool
// indices together.  Must be called by all 32 lanes.
template <bool kInstrument>
__device__ __forceinline__ void warp_insert_step(const VolumeView& vol, bool fresh,
                                                 unsigned long long key, ProbeStats* st)
{
    const unsigned lane = lane_id();
    const unsigned fresh_mask = __ballot_sync(0xFFFFFFFFu, fresh);
    if (fresh_mask == 0) return;
    bool leader = false;
    if (fresh) {
        const unsigned group = __match_any_sync(fresh_mask, key);
        leader = lane == (unsigned)(__ffs(group) - 1);
    }
    int res = kProbeFound;
    uint32_t slot = 0, steps = 0;
    if (leader) {
        res = probe_insert(vol.table, vol.table_mask, key, &slot, &steps);
        if (kInstrument) record_probe(st, steps);
        if (res == kProbeOverflow) atomicAdd(&vol.counters->probe_overflow, 1ull);
    }
    const bool won = leader && res == kProbeWon;
    const unsigned won_mask = __ballot_sync(0xFFFFFFFFu, won);
    if (won_mask == 0) return;
    const int first = __ffs(won_mask) - 1;
    uint32_t base = 0;
    if ((int)lane == first) base = atomicAdd(vol.pool_counter, (uint32_t)__popc(won_mask));
    base = __shfl_sync(0xFFFFFFFFu, base, first);
    if (won) {
        const uint32_t idx = base + (uint32_t)__popc(won_mask & ((1u << lane) - 1u));
        if (idx < vol.pool_capacity) {
            vol.table[slot].idx = idx;
        } else {
            vol.table[slot].idx = kIndexFailed;
            atomicAdd(&vol.counters->pool_exhausted, 1ull);
        }
    }
}

// Longest band for which a thread keeps its distinct keys in registers.
constexpr int kShortBand = 9;

// Block b of the grid covers 256 consecutive pixels (chunk b / n) of frame
// b % n: the batch's frames are interleaved chunk by chunk.
//
// With kShort (bands of at most kShortBand samples) a thread first walks its
// whole band and keeps the distinct block keys of its passing samples in a
// small register list; the warp then runs one insert round per list entry
// (usually two or three) instead of one per band sample.  Longer bands insert
// step by step.
template <bool kInstrument, bool kFast, bool kShort>
__global__ void __launch_bounds__(kThreads) allocate_kernel(VolumeView vol,
                                                           const __grid_constant__ FrameBatch fb)
{
    __shared__ ProbeStats st;
    if (kInstrument) init_probe_stats(&st);

    const int f = blockIdx.x % fb.n;
    const int chunk = blockIdx.x / fb.n;
    const Camera cam = fb.frame[f].cam;
    const float* depth = fb.frame[f].depth;
    const int n_pix = fb.width * fb.height;
    const int pix = chunk * kThreads + threadIdx.x;
    RayPoint p;
    bool valid = false;
    if (pix < n_pix) {
        const int v = pix / fb.width;
        const int u = pix - v * fb.width;
        valid = back_project(cam, u, v, __ldg(depth + pix), p);
    }
    const int steps = 2 * vol.band_half + 1;
    unsigned long long last = kEmptyKey;
    uint32_t out_of_range = 0;
    if (kShort) {
        unsigned long long keys[kShortBand];
        int n_keys = 0;
#pragma unroll
        for (int j = 0; j < kShortBand; ++j) {
            keys[j] = kEmptyKey;
            if (valid && j < steps) {
                VoxelSample s;
                const int status = band_sample<kFast, false>(cam, vol.div, p, j - vol.band_half, s);
                if (status == kSamplePass) {
                    const unsigned long long key = block_key(s.ix, s.iy, s.iz);
                    if (key != last) {          // newest key first; static indices only
#pragma unroll
                        for (int m = kShortBand - 1; m > 0; --m) keys[m] = keys[m - 1];
                        keys[0] = key;
                        ++n_keys;
                        last = key;
                    }
                } else if (status == kSampleOutOfRange) {
                    ++out_of_range;
                }
            }
        }
        const int rounds = (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)n_keys);
        for (int r = 0; r < rounds; ++r) {
            warp_insert_step<kInstrument>(vol, r < n_keys, keys[0], &st);
#pragma unroll
            for (int m = 0; m < kShortBand - 1; ++m) keys[m] = keys[m + 1];
        }
    } else {
        for (int i = -vol.band_half; i <= vol.band_half; ++i) {
            unsigned long long key = kEmptyKey;
            if (valid) {
                VoxelSample s;
                const int status = band_sample<kFast, false>(cam, vol.div, p, i, s);
                if (status == kSamplePass)
                    key = block_key(s.ix, s.iy, s.iz);
                else if (status == kSampleOutOfRange)
                    ++out_of_range;
            }
            const bool fresh = key != kEmptyKey && key != last;
            if (key != kEmptyKey) last = key;
            warp_insert_step<kInstrument>(vol, fresh, key, &st);
        }
    }
    // one atomic per warp for the out-of-range count
    const uint32_t oor = __reduce_add_sync(0xFFFFFFFFu, out_of_range);
    if (lane_id() == 0 && oor)
        atomicAdd(&vol.counters->out_of_range[blockIdx.x % kCounterStripes],
                  (unsigned long long)oor);
    if (kInstrument) flush_probe_stats(&st, vol.counters);
}

template <bool kInstrument>
__global__ void __launch_bounds__(kThreads) allocate_blocks_kernel(VolumeView vol,
                                                                   const int32_t* coords,
                                                                   uint32_t n)
{
    __shared__ ProbeStats st;
    if (kInstrument) init_probe_stats(&st);
    const uint32_t i = blockIdx.x * kThreads + threadIdx.x;
    unsigned long long key = kEmptyKey;
    uint32_t out_of_range = 0;
    if (i < n) {
        const int bx = coords[3 * i], by = coords[3 * i + 1], bz = coords[3 * i + 2];
        const int lo = -(1 << 20), hi = (1 << 20) - 1;
        if (bx >= lo && bx <= hi && by >= lo && by <= hi && bz >= lo && bz <= hi)
            key = pack_block(bx, by, bz);
        else
            out_of_range = 1;
    }
    warp_insert_step<kInstrument>(vol, key != kEmptyKey, key, &st);
    const uint32_t oor = __reduce_add_sync(0xFFFFFFFFu, out_of_range);
    if (lane_id() == 0 && oor)
        atomicAdd(&vol.counters->out_of_range[blockIdx.x % kCounterStripes],
                  (unsigned long long)oor);
    if (kInstrument) flush_probe_stats(&st, vol.counters);
}

}  // namespace

template <bool kInstrument, bool kFast>
void launch_allocate_t(const VolumeView& vol, const FrameBatch& fb, unsigned grid,
                       cudaStream_t stream)
{
    if (2 * vol.band_half + 1 <= kShortBand)
        allocate_kernel<kInstrument, kFast, true><<<grid, kThreads, 0, stream>>>(vol, fb);
    else
        allocate_kernel<kInstrument, kFast, false><<<grid, kThreads, 0, stream>>>(vol, fb);
}

cudaError_t launch_allocate(const VolumeView& vol, const FrameBatch& fb, bool instrument,
                            cudaStream_t stream)
{
    const int n_pix = fb.width * fb.height;
    const unsigned grid = (unsigned)((n_pix + kThreads - 1) / kThreads) * (unsigned)fb.n;
    if (instrument) {
        if (vol.fast_div)
            launch_allocate_t<true, true>(vol, fb, grid, stream);
        else
            launch_allocate_t<true, false>(vol, fb, grid, stream);
    } else {
        if (vol.fast_div)
            launch_allocate_t<false, true>(vol, fb, grid, stream);
        else
            launch_allocate_t<false, false>(vol, fb, grid, stream);
    }
    return cudaGetLastError();
}

cudaError_t launch_allocate_blocks(const VolumeView& vol, const int32_t* coords, uint32_t n,
                                   bool instrument, cudaStream_t stream)
{
    if (n == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((n + kThreads - 1) / kThreads);
    if (instrument)
        allocate_blocks_kernel<true><<<grid, kThreads, 0, stream>>>(vol, coords, n);
    else
        allocate_blocks_kernel<false><<<grid, kThreads, 0, stream>>>(vol, coords, n);
    return cudaGetLastError();
}

}  // namespace tsdf
