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

// What an offering lane learns from an insert step: the outcome for its key
// (found, won or overflow) and the key's slot.
struct InsertResult {
    int res;
    uint32_t slot;
};

// One warp-wide insert step: lanes with `fresh` set offer `key`; equal keys
// are merged, one leader per key probes, and the warp's winners take pool
// indices together and publish them before the step returns.  Every offering
// lane gets its key's outcome and slot.  Must be called by all 32 lanes.
// Most keys a frame offers are already in the table, and almost all of those
// sit in their home slot: each offering lane first reads its key's home
// slot, and only the lanes that do not find their key there go on to the
// warp's de-duplication and the probe (keys are never removed, so a key seen
// there is in the table).  With kInstrument every offered key is probed, so
// that the probe statistics count every key.
template <bool kInstrument, bool kResult = true>
__device__ __forceinline__ InsertResult warp_insert_step(const VolumeView& vol, bool fresh,
                                                         unsigned long long key, ProbeStats* st)
{
    const unsigned lane = lane_id();
    InsertResult out = {kProbeOverflow, 0u};
    bool at_home = false;
    if (!kInstrument && fresh) {
        const uint32_t home = home_slot(key, vol.table_mask);
        at_home = vol.table[home].key == key;
        if (at_home) {
            out.res = kProbeFound;
            out.slot = home;
            fresh = false;
        }
    }
    const unsigned fresh_mask = __ballot_sync(0xFFFFFFFFu, fresh);
    if (fresh_mask == 0) return out;
    bool leader = false;
    int leader_lane = (int)lane;
    if (fresh) {
        const unsigned group = __match_any_sync(fresh_mask, key);
        leader_lane = __ffs(group) - 1;
        leader = (int)lane == leader_lane;
    }
    int res = kProbeFound;
    uint32_t slot = 0, steps = 0;
    if (leader) {
        res = probe_insert(vol.table, vol.table_mask, key, &slot, &steps);
        if (kInstrument) record_probe(st, steps);
        if (res == kProbeOverflow) atomicAdd(&vol.counters->probe_overflow, 1ull);
    }
    if (kResult) {                          // (the allocate kernel does not need it)
        const int r = __shfl_sync(0xFFFFFFFFu, res, leader_lane);
        const uint32_t sl = __shfl_sync(0xFFFFFFFFu, slot, leader_lane);
        if (!at_home) {
            out.res = r;
            out.slot = sl;
        }
    }
    const bool won = leader && res == kProbeWon;
    const unsigned won_mask = __ballot_sync(0xFFFFFFFFu, won);
    if (won_mask == 0) return out;
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
    return out;
}

// Longest band for which a thread keeps its distinct keys in registers.
constexpr int kShortBand = 9;

// Whether the sample in voxel s passes the volume's occlusion test (the
// allocate kernel needs only the decision, not the value).
template <bool kFast, bool kReproject>
__device__ __forceinline__ bool allocate_visible(const VolumeView& vol, const Camera& cam,
                                                 const RayPoint& p, const float* depth,
                                                 int width, int height, VoxelSample s)
{
    if (kReproject) {
        size_t pix;
        return reprojected_visible<kFast, false>(cam, vol.div, depth, width, height, s, pix);
    }
    float zc;
    return ray_visible(cam, vol.div, p, s, zc);
}

// (float)j for 0 <= j < 2^23, exactly and without a conversion: the float
// whose significand holds j above 2^23, less 2^23.
__device__ __forceinline__ float small_int_to_float(int j)
{
    return __fsub_rn(__int_as_float(0x4B000000 + j), 8388608.0f);
}

// The block index along one axis (origin o and direction e in voxel units)
// of band step j, evaluated as band_voxel_unchecked evaluates the step's
// voxel.
__device__ __forceinline__ int axis_block(float o, float e, int j, float fhalf)
{
    const float fi = __fsub_rn(small_int_to_float(j), fhalf);
    return __float2int_rd(__fadd_rn(o, __fmul_rn(fi, e))) >> 3;
}

// The band step at which the block index along one axis moves from a0 (at
// step 0) to a1 = a0 +- 1 (at step `last`).  Each rounding of o + fi e is
// monotone in fi, so the index is monotone in the step and moves exactly
// once.  The step is estimated from where the ray meets the block boundary
// and confirmed by evaluating the two steps around it exactly; -1 where the
// estimate misses (an axis the ray barely moves along).
__device__ __forceinline__ int axis_crossing(float o, float e, int a0, int a1, int last,
                                             float fhalf)
{
    const bool up = a1 > a0;
    const float boundary = (float)(8 * (up ? a1 : a0));   // |8 a| <= 2^23: exact
    const float q = __fadd_rn(__fdividef(__fsub_rn(boundary, o), e), fhalf);
    int t = up ? __float2int_ru(q) : min(__float2int_rd(q), last) + 1;
    t = min(max(t, 1), last);
    return axis_block(o, e, t - 1, fhalf) == a0 && axis_block(o, e, t, fhalf) == a1 ? t : -1;
}

// The allocate kernel's start mask for a short band (see allocate_kernel)
// from the steps at which the ray's block changes, without visiting every
// step: for rays whose band steps are all proven to pass the occlusion test
// except perhaps the last, and whose block moves by at most one along each
// axis over the band.  Then every proven step passes, so the proven steps
// that start a block are step 0 and the steps where the block changes, and
// the last step, when unproven, starts one if it enters another block and
// passes the test.  Returns false (mask untouched) where the conditions fail
// or a crossing estimate misses; the caller then walks step by step.
template <bool kFast>
__device__ __forceinline__ bool starts_from_crossings(const VolumeView& vol, const Camera& cam,
                                                      const RayPoint& p, int steps, int j_proven,
                                                      float fhalf, uint32_t& starts)
{
    const int last = steps - 1;
    VoxelSample a, b;
    band_voxel_unchecked(p, __fsub_rn(0.0f, fhalf), a);
    band_voxel_unchecked(p, __fsub_rn(small_int_to_float(last), fhalf), b);
    const int ax = a.ix >> 3, ay = a.iy >> 3, az = a.iz >> 3;
    const int bx = b.ix >> 3, by = b.iy >> 3, bz = b.iz >> 3;
    if (abs(bx - ax) > 1 || abs(by - ay) > 1 || abs(bz - az) > 1) return false;
    uint32_t changes = 1u;                  // step 0 and the steps entering another block
    if (bx != ax) {
        const int t = axis_crossing(p.vx, p.ex, ax, bx, last, fhalf);
        if (t < 0) return false;
        changes |= 1u << t;
    }
    if (by != ay) {
        const int t = axis_crossing(p.vy, p.ey, ay, by, last, fhalf);
        if (t < 0) return false;
        changes |= 1u << t;
    }
    if (bz != az) {
        const int t = axis_crossing(p.vz, p.ez, az, bz, last, fhalf);
        if (t < 0) return false;
        changes |= 1u << t;
    }
    const uint32_t proven = j_proven >= 0 ? (2u << j_proven) - 1u : 0u;
    uint32_t m = changes & proven;
    if ((changes & ~proven) != 0u && allocate_visible<kFast, false>(vol, cam, p, nullptr, 0, 0, b))
        m |= 1u << last;
    starts = m;
    return true;
}

// Block b of the grid covers 256 consecutive pixels (chunk b / n) of frame
// b % n: the batch's frames are interleaved chunk by chunk.
//
// With kShort (bands of at most kShortBand samples) a thread first walks its
// whole band and marks, in a bit mask, each band step whose sample passes
// the occlusion test and lies in another block than the last passing sample
// (a sample in the block of the last passing one is not tested: it cannot
// add a block).  The samples of a ray move monotonically along each axis,
// so a block once left never comes back and the marked steps are exactly
// the first passing samples of the ray's distinct blocks.  The warp then
// runs one insert round per marked step (usually two or three): each lane
// recomputes the voxel of its next marked step (the same float operations,
// hence the same voxel) and offers its block.  Longer bands insert step by
// step.  With kReproject the occlusion test is the reprojection of the voxel
// centre (reprojected_visible), as in the update it pairs with.
template <bool kInstrument, bool kFast, bool kShort, bool kReproject>
__global__ void __launch_bounds__(kThreads) allocate_kernel(VolumeView vol,
                                                           const __grid_constant__ FrameBatch fb)
{
    __shared__ ProbeStats st;
    if (kInstrument) init_probe_stats(&st);

    const uint32_t chunk = divide_index(fb.by_n, blockIdx.x);
    const int f = (int)(blockIdx.x - chunk * (uint32_t)fb.n);
    const Camera cam = fb.frame[f].cam;
    const float* depth = fb.frame[f].depth;
    const int n_pix = fb.width * fb.height;
    const int pix = (int)chunk * kThreads + (int)threadIdx.x;
    RayPoint p;
    bool valid = false;
    if (pix < n_pix) {
        const int v = (int)divide_index(fb.by_width, (uint32_t)pix);
        valid = back_project_pixel(vol, fb, cam, v, (size_t)pix, __ldg(depth + pix), p);
    }
    const int half = vol.band_half;
    const int steps = 2 * half + 1;
    uint32_t out_of_range = 0;
    if (kShort) {
        uint32_t starts = 0;                // band steps that start a new block
        int lbx = 0, lby = 0, lbz = 0;      // block of the last passing sample
        bool any = false;
        // band steps whose ray-depth test provably passes are not tested
        SurePass sure = {-INFINITY, false};
        if (!kReproject && valid) sure = sure_pass(cam, vol.div, p, half);
        const float fhalf = (float)half;
        // when every lane's whole band lies in the key range (always, in
        // practice) the per-sample range check is left out
        const bool all_in = __all_sync(0xFFFFFFFFu, !valid || ray_in_range(p, fhalf));
        // the proven steps as one bound on j: step j (at fi = j - half, an
        // integer) is proven when max(fi, 0) <= i_max, i.e. when
        // j <= half + floor(i_max) and i_max >= 0
        int j_proven = -1;
        if (!kReproject && sure.near && sure.i_max >= 0.0f)
            j_proven = half + (int)floorf(fminf(sure.i_max, fhalf));
        // most rays: the mask from the band's block crossings; the others
        // walk the band step by step
        bool walked = !valid;
        if (!kReproject && valid && all_in && j_proven >= steps - 2)
            walked = starts_from_crossings<kFast>(vol, cam, p, steps, j_proven, fhalf, starts);
#pragma unroll
        for (int j = 0; j < kShortBand; ++j) {
            if (!walked && j < steps) {
                VoxelSample s;
                // the step j - half as a float: exact, with no integer
                // conversion per step
                const float fi = __fsub_rn((float)j, fhalf);
                bool in_range = true;
                if (all_in) band_voxel_unchecked(p, fi, s);
                else in_range = band_voxel_f<kFast>(p, fi, s);
                if (!in_range) {
                    ++out_of_range;
                } else {
                    const int bx = s.ix >> 3, by = s.iy >> 3, bz = s.iz >> 3;
                    const bool proven = j <= j_proven;
                    if ((!any || bx != lbx || by != lby || bz != lbz) &&
                        (proven || allocate_visible<kFast, kReproject>(vol, cam, p, depth,
                                                                       fb.width, fb.height, s))) {
                        starts |= 1u << j;
                        lbx = bx;
                        lby = by;
                        lbz = bz;
                        any = true;
                    }
                }
            }
        }
        const int rounds = (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)__popc(starts));
        for (int r = 0; r < rounds; ++r) {
            unsigned long long key = kEmptyKey;
            const bool offer = starts != 0u;
            if (offer) {
                const int j = __ffs(starts) - 1;
                starts &= starts - 1u;
                VoxelSample s;
                band_voxel_unchecked(p, __fsub_rn((float)j, fhalf), s);    // a passing step: in range
                key = block_key(s.ix, s.iy, s.iz);
            }
            warp_insert_step<kInstrument, false>(vol, offer, key, &st);
        }
    } else {
        unsigned long long last = kEmptyKey;
        for (int i = -half; i <= half; ++i) {
            unsigned long long key = kEmptyKey;
            if (valid) {
                VoxelSample s;
                if (!band_voxel<kFast>(cam, vol.div, p, i, s)) {
                    ++out_of_range;
                } else {
                    const unsigned long long k = block_key(s.ix, s.iy, s.iz);
                    // (the block of the last passing sample needs no test)
                    if (k == last || allocate_visible<kFast, kReproject>(vol, cam, p, depth,
                                                                         fb.width, fb.height, s))
                        key = k;
                }
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

// ---------------------------------------------------------------------------
// Fused integrate: allocate and update in one kernel.
// ---------------------------------------------------------------------------

// Waits for a published index are bounded by this many polls (~64 ns apart).
constexpr uint32_t kPublishSpinLimit = 1u << 20;

// The pool index published in `slot`.  The lane that claimed the slot takes
// the index from the pool counter and stores it in the same insert step,
// waiting on nothing, so this wait is short; it is bounded all the same: a
// wait that gives up reports PENDING and the caller counts it.
__device__ __forceinline__ uint32_t published_index(const VolumeView& vol, uint32_t slot)
{
    const volatile uint32_t* p = &vol.table[slot].idx;
    uint32_t idx = *p;
    for (uint32_t n = 0; idx == kIndexPending && n < kPublishSpinLimit; ++n) {
        __nanosleep(64);
        idx = *p;
    }
    return idx;
}

// One walk per pixel does both stages: the band's samples (voxel, tsdf) are
// kept in registers while the distinct block keys go through the allocate
// kernel's warp insert rounds; each round's result (the key's slot, hence
// its pool index) gives the pool index of that key's samples, with no second
// walk and no lookup.  The samples are then added band step by band step,
// the warp merging the samples of one step that fall in the same voxel, as
// in the per-sample update kernel (here through shared-memory slots).
// Tiles and warp patches as in that kernel (16 x 16, 8 x 4), grid
// tile-major, frame-minor.
template <bool kInstrument, bool kFast>
__global__ void __launch_bounds__(kThreads) integrate_fused_kernel(
    VolumeView vol, const __grid_constant__ FrameBatch fb)
{
    __shared__ ProbeStats st;
    __shared__ float4 s_stage[kThreads];    // each warp's merge slots
    if (kInstrument) init_probe_stats(&st);

    const TilePos tp = tile_of_block(fb, fb.by_tiles16_x, blockIdx.x);
    const int f = tp.f;
    const Camera cam = fb.frame[f].cam;
    const int w = (int)(threadIdx.x >> 5), l = (int)(threadIdx.x & 31u);
    const int u = tp.tx * 16 + (w & 1) * 8 + (l & 7);
    const int v = tp.ty * 16 + (w >> 1) * 4 + (l >> 3);
    const bool inside = u < fb.width && v < fb.height;
    const float depth = inside ? __ldg(fb.frame[f].depth + (size_t)v * fb.width + u) : 0.0f;
    RayPoint p;
    bool valid = false;
    float cr = 0.0f, cg = 0.0f, cb = 0.0f;
    if (inside) {
        const size_t pix = (size_t)v * fb.width + u;
        valid = back_project_pixel(vol, fb, cam, v, pix, depth, p);
        if (valid) {
            const float* rgb = fb.frame[f].rgb;
            cr = __ldg(rgb + 3 * pix);
            cg = __ldg(rgb + 3 * pix + 1);
            cb = __ldg(rgb + 3 * pix + 2);
        }
    }
    const int half = vol.band_half;
    const int steps = 2 * half + 1;
    const float fhalf = (float)half;
    // per band step: the sample's voxel in its block, its tsdf and (after the
    // insert rounds) its block's pool index; `passed` marks the steps whose
    // sample passed, `starts` those that begin a new block (the samples of a
    // ray move monotonically along each axis, so a block's passing samples
    // are the passing steps from its start to the next start)
    int lv[kShortBand];
    float tv[kShortBand];
    uint32_t sidx[kShortBand];
    uint32_t passed = 0, starts = 0;
    int lbx = 0, lby = 0, lbz = 0;
    uint32_t out_of_range = 0;
#pragma unroll
    for (int j = 0; j < kShortBand; ++j) {
        lv[j] = 0;
        tv[j] = 0.0f;
        sidx[j] = kIndexFailed;
        if (valid && j < steps) {
            VoxelSample s;
            const int status = band_sample<kFast>(cam, vol.div, p, __fsub_rn((float)j, fhalf), s);
            if (status == kSamplePass) {
                lv[j] = (int)voxel_slot(vol, s.ix & 7, s.iy & 7, s.iz & 7);
                tv[j] = s.tsdf;
                const int bx = s.ix >> 3, by = s.iy >> 3, bz = s.iz >> 3;
                if (passed == 0u || bx != lbx || by != lby || bz != lbz) {
                    starts |= 1u << j;
                    lbx = bx;
                    lby = by;
                    lbz = bz;
                }
                passed |= 1u << j;
            } else if (status == kSampleOutOfRange) {
                ++out_of_range;
            }
        }
    }
    uint32_t updates = 0, timeouts = 0;
    const int rounds = (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)__popc(starts));
    uint32_t rest = starts;
    for (int r = 0; r < rounds; ++r) {
        const bool offered = rest != 0u;
        unsigned long long key = kEmptyKey;
        uint32_t mine = 0;                  // this key's passing steps
        if (offered) {
            const int j = __ffs(rest) - 1;
            rest &= rest - 1u;
            const uint32_t from = 1u << j;
            mine = passed & (rest ? (rest & (0u - rest)) - from : 0u - from);
            VoxelSample s;
            band_voxel<kFast>(cam, vol.div, p, j - half, s);
            key = block_key(s.ix, s.iy, s.iz);
        }
        const InsertResult ins = warp_insert_step<kInstrument>(vol, offered, key, &st);
        __syncwarp();                       // this warp's winners have published
        if (offered) {
            uint32_t idx = kIndexFailed;
            if (ins.res != kProbeOverflow) {
                idx = published_index(vol, ins.slot);
                if (idx == kIndexPending) ++timeouts;
            }
#pragma unroll
            for (int j = 0; j < kShortBand; ++j)
                if (mine & (1u << j)) sidx[j] = idx;
        }
    }
    // the update, one band step at a time for the whole warp
#pragma unroll
    for (int j = 0; j < kShortBand; ++j) {
        // (pool indices are below 2^23, so e fits in 32 bits)
        const bool add = (passed >> j & 1u) && sidx[j] < vol.pool_capacity;
        const uint32_t e = add ? sidx[j] * (uint32_t)kBlockVoxels + (uint32_t)lv[j] : 0u;
        warp_add_samples<true>(vol, s_stage + (threadIdx.x & ~31u), add, e, tv[j], cr, cg, cb);
        updates += add ? 1u : 0u;
    }
    // absent (overflow), FAILED or timed out
    const uint32_t missed = (uint32_t)__popc(passed) - updates;
    const uint32_t w_valid = __reduce_add_sync(0xFFFFFFFFu, valid ? 1u : 0u);
    const uint32_t w_updates = __reduce_add_sync(0xFFFFFFFFu, updates);
    const uint32_t w_missed = __reduce_add_sync(0xFFFFFFFFu, missed);
    const uint32_t w_oor = __reduce_add_sync(0xFFFFFFFFu, out_of_range);
    const uint32_t w_timeouts = __reduce_add_sync(0xFFFFFFFFu, timeouts);
    if (l == 0) {
        const int stripe = blockIdx.x % kCounterStripes;
        if (w_valid) atomicAdd(&vol.counters->valid_points[stripe], (unsigned long long)w_valid);
        if (w_updates)
            atomicAdd(&vol.counters->voxel_updates[stripe], (unsigned long long)w_updates);
        if (w_missed) atomicAdd(&vol.counters->missed[stripe], (unsigned long long)w_missed);
        if (w_oor) atomicAdd(&vol.counters->out_of_range[stripe], (unsigned long long)w_oor);
        if (w_timeouts) atomicAdd(&vol.counters->publish_timeouts, (unsigned long long)w_timeouts);
    }
    if (kInstrument) flush_probe_stats(&st, vol.counters);
}

}  // namespace

template <bool kInstrument, bool kFast, bool kReproject>
void launch_allocate_r(const VolumeView& vol, const FrameBatch& fb, unsigned grid,
                       cudaStream_t stream)
{
    if (2 * vol.band_half + 1 <= kShortBand)
        allocate_kernel<kInstrument, kFast, true, kReproject><<<grid, kThreads, 0, stream>>>(vol,
                                                                                           fb);
    else
        allocate_kernel<kInstrument, kFast, false, kReproject><<<grid, kThreads, 0, stream>>>(vol,
                                                                                            fb);
}

template <bool kInstrument, bool kFast>
void launch_allocate_t(const VolumeView& vol, const FrameBatch& fb, unsigned grid,
                       cudaStream_t stream)
{
    if (vol.occlusion == TSDF_OCCLUSION_REPROJECT)
        launch_allocate_r<kInstrument, kFast, true>(vol, fb, grid, stream);
    else
        launch_allocate_r<kInstrument, kFast, false>(vol, fb, grid, stream);
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

cudaError_t launch_integrate_fused(const VolumeView& vol, const FrameBatch& fb, bool instrument,
                                   cudaStream_t stream)
{
    // (the fused kernel applies the ray-depth occlusion test only)
    if (2 * vol.band_half + 1 > kShortBand || vol.occlusion != TSDF_OCCLUSION_RAY)
        return cudaErrorInvalidValue;
    const unsigned tiles = (unsigned)(((fb.width + 15) / 16) * ((fb.height + 15) / 16));
    const unsigned grid = tiles * (unsigned)fb.n;
    if (instrument) {
        if (vol.fast_div) integrate_fused_kernel<true, true><<<grid, kThreads, 0, stream>>>(vol, fb);
        else integrate_fused_kernel<true, false><<<grid, kThreads, 0, stream>>>(vol, fb);
    } else {
        if (vol.fast_div) integrate_fused_kernel<false, true><<<grid, kThreads, 0, stream>>>(vol, fb);
        else integrate_fused_kernel<false, false><<<grid, kThreads, 0, stream>>>(vol, fb);
    }
    return cudaGetLastError();
}

}  // namespace tsdf
