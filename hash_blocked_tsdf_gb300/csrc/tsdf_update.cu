// Update kernels ("What Irregularity Costs", design section, integration:
// the regular stage; accumulation: sums, not running means).
//
// By default (TSDF_UPDATE_PER_SAMPLE) update_kernel alone adds every
// sample, merging a warp's samples of the same voxel first.  In the
// adaptive mode both kernels run on every batch and split the frame by
// 16 x 16 pixel tiles: a tile whose pixels are small against the voxels (the
// density rule in tsdf_device.cuh: at least half of them see a voxel edge 5
// or more pixels wide, 10 for launches of fewer than 4 frames) has its
// samples crowd into few voxels; update_kernel lists it and the persistent
// update_rows_kernel pre-reduces it in shared memory; update_kernel adds
// every other tile's samples itself.  In the pre-reduced mode
// update_rows_kernel takes every tile.
//
// update_kernel (per sample): every thread walks one pixel's band, looks
// up each passing sample's block (one lookup per new key, almost always a
// first-probe hit) and adds (tsdf, 1, r, g, b) with two reductions: one
// 4-wide into the voxel's (tsdf, weight, red, green) record, one scalar into
// the blue array.  The lanes of a warp take the band steps together, and the
// samples of one step that fall in the same voxel are summed in registers
// first (warp_add_samples, by shuffles), so such a group costs one pair of
// reductions.
// Blocks of 256 threads own 16 x 16 pixel tiles of one frame, each warp an
// 8 x 4 patch.  On GB300 no unit saturates: the walk is issue-bound, the
// merge waits on its matches and shuffles, and the L2's atomic units run
// about a third busy.
//
// update_rows_kernel (pre-reducing): a block of 192 threads takes an 8 x 8
// pixel tile of one frame at a time (a listed 16 x 16 tile is four of them;
// with TSDF_UPDATE_PRE_REDUCED every tile, one per block), three threads per pixel, each walking one third
// of the pixel's truncation band (a warp covers an 8 x 4 pixel patch).  The
// block keeps a shared table of the voxel rows its samples fall in (a row is
// the 8 voxels of a block that share ly and lz: in the planar layout one
// 32-byte sector of each array, in the interleaved one four 2 x 2 x 2
// bricks' records), and for every
// voxel of a row two 64-bit masks: which of
// the tile's pixels put a sample in it, and which put a second one (a ray
// puts at most two samples in a voxel: samples are one voxel edge apart and a
// voxel is sqrt(3) edges across).  That takes one shared atomicOr per sample.
// Afterwards every touched voxel recomputes its samples' truncated distances
// from the pixel depths and its own centre -- the walk's arithmetic, so the
// same values -- sums them with the pixels' colours in pixel order, and adds
// its five sums to the pool; the voxels of a row are flushed by adjacent
// lanes, so each row reaches L2 as a few sectors instead of two reductions per
// sample.  Rows that find no slot in the shared table add their samples
// directly.
//
// Both grids run tile-major, frame-minor, so the frames' updates of the same
// voxels meet in L2.
#include <atomic>

#include "tsdf_device.cuh"

namespace tsdf {
namespace {

constexpr int kTileW = 16;
constexpr int kTileH = 16;
constexpr int kThreads = kTileW * kTileH;

// kSparseOnly: leave dense tiles to update_rows_kernel (adaptive mode).
// kReproject: the occlusion test by reprojection of the voxel centre; each
// passing sample adds the colour of the pixel it was tested against.
template <bool kFast, bool kSparseOnly, bool kReproject>
__global__ void __launch_bounds__(kThreads) update_kernel(VolumeView vol,
                                                         const __grid_constant__ FrameBatch fb)
{
    const TilePos tp = tile_of_block(fb, fb.by_tiles16_x, blockIdx.x);
    const int f = tp.f;
    const Camera cam = fb.frame[f].cam;
    // each warp takes an 8 x 4 pixel patch of the tile (8 warps: 2 across,
    // 4 down): a squarer footprint puts more of a warp's samples in common
    // voxel rows than a 16 x 2 strip
    const int w = (int)(threadIdx.x >> 5), l = (int)(threadIdx.x & 31u);
    const int u = tp.tx * kTileW + (w & 1) * 8 + (l & 7);
    const int v = tp.ty * kTileH + (w >> 1) * 4 + (l >> 3);

    const bool inside = u < fb.width && v < fb.height;
    const float depth = inside ? __ldg(fb.frame[f].depth + (size_t)v * fb.width + u) : 0.0f;
    if (kSparseOnly) {
        const uint32_t n_valid = (uint32_t)__syncthreads_count(valid_depth(depth));
        const uint32_t n_dense =
            (uint32_t)__syncthreads_count(dense_pixel(depth, vol.div.voxel, cam.fx, fb.n));
        if (dense_tile(n_valid, n_dense)) {             // uniform over the block
            // list the tile for update_rows_kernel; if the list is full,
            // integrate it here after all
            __shared__ uint32_t s_listed;
            if (threadIdx.x == 0) {
                const uint32_t pos = atomicAdd(vol.dense_count, 1u);
                s_listed = pos < vol.dense_capacity ? 1u : 0u;
                if (s_listed)
                    vol.dense_list[pos] = (uint32_t)f << 24 | divide_index(fb.by_n, blockIdx.x);
            }
            __syncthreads();
            if (s_listed) return;
        }
    }
    RayPoint p;
    bool valid = false;
    float cr = 0.0f, cg = 0.0f, cb = 0.0f;
    if (inside) {
        const size_t pix = (size_t)v * fb.width + u;
        valid = back_project_pixel(vol, fb, cam, v, pix, depth, p);
        if (valid && !kReproject) {
            const float* rgb = fb.frame[f].rgb;
            cr = __ldg(rgb + 3 * pix);
            cg = __ldg(rgb + 3 * pix + 1);
            cb = __ldg(rgb + 3 * pix + 2);
        }
    }
    uint32_t updates = 0, missed = 0;
    int lbx = 0, lby = 0, lbz = 0;          // block of the last lookup
    bool looked_up = false;
    uint32_t idx = kIndexFailed;
    // every lane runs every band step (the warp merges each step's samples);
    // the step also counts as a float, exactly, to spare a conversion per step;
    // when every lane's whole band lies in the key range (always, in
    // practice) the per-sample range check is left out
    const bool all_in =
        __all_sync(0xFFFFFFFFu, !valid || ray_in_range(p, (float)vol.band_half));
    float fi = -(float)vol.band_half;
    for (int i = -vol.band_half; i <= vol.band_half; ++i, fi = __fadd_rn(fi, 1.0f)) {
        VoxelSample s;
        s.tsdf = 0.0f;
        bool add = false;
        uint32_t e = 0;
        if (valid) {
            int status;
            if (kReproject) {
                size_t q;
                status = band_sample_reprojected<kFast>(cam, vol.div, p, i, fb.frame[f].depth,
                                                        fb.width, fb.height, s, q);
                if (status == kSamplePass) {
                    const float* rgb = fb.frame[f].rgb;
                    cr = __ldg(rgb + 3 * q);
                    cg = __ldg(rgb + 3 * q + 1);
                    cb = __ldg(rgb + 3 * q + 2);
                }
            } else {
                status = all_in ? band_sample<kFast, false>(cam, vol.div, p, fi, s)
                                : band_sample<kFast, true>(cam, vol.div, p, fi, s);
            }
            if (status == kSamplePass) {
                const int bx = s.ix >> 3, by = s.iy >> 3, bz = s.iz >> 3;
                if (!looked_up || bx != lbx || by != lby || bz != lbz) {
                    idx = lookup(vol.table, vol.table_mask, pack_block(bx, by, bz));
                    lbx = bx;
                    lby = by;
                    lbz = bz;
                    looked_up = true;
                }
                if (idx < vol.pool_capacity) {
                    // (pool indices are below 2^23, so e fits in 32 bits)
                    e = idx * (uint32_t)kBlockVoxels + voxel_slot(vol, s.ix & 7, s.iy & 7, s.iz & 7);
                    add = true;
                    ++updates;
                } else {
                    ++missed;                   // absent, FAILED or never published
                }
            }
        }
        warp_add_samples<false>(vol, nullptr, add, e, s.tsdf, cr, cg, cb);
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


// ---------------------------------------------------------------------------
// Pre-reduced update.
// ---------------------------------------------------------------------------
constexpr int kRowTile = 8;                           // 8 x 8 pixel tiles
static_assert(kTileW == 16 && kTileH == 16 && kRowTile == 8,
              "the batch's tile divisors (by_tiles16_x, by_tiles8_x) assume these tiles");
constexpr int kRowPix = kRowTile * kRowTile;          // 64
constexpr int kRowParts = 3;                          // threads per pixel
constexpr int kRowThreads = kRowPix * kRowParts;      // 192
constexpr int kRowBlocksPerSM = 5;
constexpr int kRows = 224;                            // shared row slots
constexpr int kCellWords = 4;                         // once-mask (2 words), twice-mask (2)
constexpr int kRowWords = 8 * kCellWords + 4;         // + 4 words to spread the banks
constexpr int kRowMaxProbe = 32;
constexpr uint32_t kNoRow = 0xFFFFFFFFu;
// Per-pixel fields in shared memory, [field][64].
enum PixField { kPxValid = 0, kPxD, kPxVx, kPxVy, kPxVz, kPxEx, kPxEy, kPxEz, kPxR, kPxG, kPxB,
                kPxFields };
// Shared layout in 32-bit words (offsets keep the 64-bit block keys 8-byte
// aligned and the sums 16-byte aligned).
constexpr int kOffKey = 0;                                   // [kRows] row key or kNoRow
constexpr int kOffList = kOffKey + kRows;                    // [kRows] claimed slots
constexpr int kOffCount = kOffList + kRows;                  // [8] rows, cells, vote per warp
constexpr int kOffBlock = kOffCount + 8;                     // [kRows] u64 block key of the row
constexpr int kOffCells = kOffBlock + 2 * kRows;             // [kRows][kRowWords]
constexpr int kOffPix = kOffCells + kRows * kRowWords;       // [kPxFields][64]
constexpr int kOffCellList = kOffPix + kPxFields * kRowPix;  // [8 * kRows] u16 (slot << 3 | lx)
constexpr int kRowSmemWords = kOffCellList + 8 * kRows / 2;
constexpr size_t kRowSmemBytes = (size_t)kRowSmemWords * sizeof(uint32_t);
static_assert(kOffBlock % 2 == 0 && kOffCells % 4 == 0, "shared layout alignment");

// Find or claim the shared slot of each lane's row (row_key = pool index << 6
// | row), or -1 for lanes that do not want one or find no slot within
// kRowMaxProbe probes.  The loop runs the same number of times on every lane
// (it ends when no lane is still probing), so the warp leaves it converged.
// The lane that claims a slot records the row's block key and lists the slot.
__device__ __forceinline__ int claim_row(uint32_t* sm, bool want, uint32_t row_key,
                                         unsigned long long block)
{
    uint32_t* s_key = sm + kOffKey;
    uint32_t slot = __umulhi(row_key * 0x9E3779B1u, (uint32_t)kRows);
    int found = -1;
    bool probing = want;
    for (int n = 0; n < kRowMaxProbe; ++n) {
        if (!__any_sync(0xFFFFFFFFu, probing)) break;
        if (probing) {
            uint32_t k = s_key[slot];
            if (k == kNoRow) {
                k = atomicCAS(&s_key[slot], kNoRow, row_key);
                if (k == kNoRow) {
                    reinterpret_cast<unsigned long long*>(sm + kOffBlock)[slot] = block;
                    sm[kOffList + atomicAdd(sm + kOffCount, 1u)] = slot;
                    k = row_key;
                }
            }
            if (k == row_key) {
                found = (int)slot;
                probing = false;
            } else {
                slot = slot + 1 == (uint32_t)kRows ? 0u : slot + 1;
            }
        }
    }
    return found;
}

template <bool kFast>
__device__ __forceinline__ void flush_rows(const VolumeView& vol, const Camera& cam, uint32_t* sm);

// One 8 x 8 pixel tile (origin u0, v0) of frame f, pre-reduced; called by
// the whole block.  Adds the tile's counts to the caller's.
template <bool kFast>
__device__ __forceinline__ void rows_tile(const VolumeView& vol, const FrameBatch& fb, int f,
                                          int u0, int v0, uint32_t* sm, uint32_t& n_valid,
                                          uint32_t& updates, uint32_t& missed)
{
    uint32_t* s_key = sm + kOffKey;
    uint32_t* s_cells = sm + kOffCells;
    uint32_t* s_pix = sm + kOffPix;
    float* s_pixf = reinterpret_cast<float*>(s_pix);
    const int t = threadIdx.x;
    const Camera cam = fb.frame[f].cam;

    if (t < kRowPix) {
        const int u = u0 + (t & (kRowTile - 1)), v = v0 + t / kRowTile;
        RayPoint p = {};
        bool valid = false;
        float c[3] = {0.0f, 0.0f, 0.0f};
        if (u < fb.width && v < fb.height) {
            const size_t pix = (size_t)v * fb.width + u;
            valid = back_project_pixel(vol, fb, cam, v, pix, __ldg(fb.frame[f].depth + pix), p);
            if (valid) {
                const float* rgb = fb.frame[f].rgb;
                c[0] = __ldg(rgb + 3 * pix);
                c[1] = __ldg(rgb + 3 * pix + 1);
                c[2] = __ldg(rgb + 3 * pix + 2);
            }
        }
        s_pix[kPxValid * kRowPix + t] = valid ? 1u : 0u;
        s_pixf[kPxD * kRowPix + t] = p.d;
        s_pixf[kPxVx * kRowPix + t] = p.vx;
        s_pixf[kPxVy * kRowPix + t] = p.vy;
        s_pixf[kPxVz * kRowPix + t] = p.vz;
        s_pixf[kPxEx * kRowPix + t] = p.ex;
        s_pixf[kPxEy * kRowPix + t] = p.ey;
        s_pixf[kPxEz * kRowPix + t] = p.ez;
        s_pixf[kPxR * kRowPix + t] = c[0];
        s_pixf[kPxG * kRowPix + t] = c[1];
        s_pixf[kPxB * kRowPix + t] = c[2];
    }
    for (int i = t; i < kRows; i += kRowThreads) s_key[i] = kNoRow;
    if (t < 2) sm[kOffCount + t] = 0;
    uint4* cells4 = reinterpret_cast<uint4*>(s_cells);
    for (int i = t; i < kRows * kRowWords / 4; i += kRowThreads) cells4[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    // walk: thread (pixel q, part) takes band steps [part * per, (part + 1) * per);
    // a warp holds 32 pixels of one part, so the trip count is warp-uniform
    const int q = t % kRowPix;
    const int part = t / kRowPix;
    const int steps = 2 * vol.band_half + 1;
    const int per = (steps + kRowParts - 1) / kRowParts;
    const int i0 = part * per;
    const int i1 = min(steps, i0 + per);
    const bool valid = s_pix[kPxValid * kRowPix + q] != 0;
    RayPoint p;
    p.d = s_pixf[kPxD * kRowPix + q];
    p.vx = s_pixf[kPxVx * kRowPix + q];
    p.vy = s_pixf[kPxVy * kRowPix + q];
    p.vz = s_pixf[kPxVz * kRowPix + q];
    p.ex = s_pixf[kPxEx * kRowPix + q];
    p.ey = s_pixf[kPxEy * kRowPix + q];
    p.ez = s_pixf[kPxEz * kRowPix + q];
    const uint32_t bit = 1u << (q & 31);
    const int half_word = q >> 5;
    unsigned long long last = kEmptyKey;
    uint32_t idx = kIndexFailed;
    for (int i = i0; i < i1; ++i) {
        VoxelSample s;      // (invalid pixels walk a zero ray: finite values, never used)
        const int status = band_sample<kFast>(cam, vol.div, p, i - vol.band_half, s);
        const bool pass = valid && status == kSamplePass;
        const unsigned long long key = pass ? block_key(s.ix, s.iy, s.iz) : kEmptyKey;
        if (pass && key != last) {
            idx = lookup(vol.table, vol.table_mask, key);
            last = key;
        }
        const bool add = pass && idx < vol.pool_capacity;   // else absent, FAILED or unpublished
        missed += (pass && !add) ? 1u : 0u;
        updates += add ? 1u : 0u;
        const uint32_t row = (uint32_t)((s.iy & 7) | ((s.iz & 7) << 3));
        const int lx = s.ix & 7;
        const int slot = claim_row(sm, add, (idx << 6) | row, key);
        bool direct = add && slot < 0;
        if (slot >= 0) {
            uint32_t* cell = s_cells + slot * kRowWords + lx * kCellWords;
            const uint32_t once = atomicOr(cell + half_word, bit);
            if (once & bit) {
                // a ray puts at most two samples in a voxel (samples are one
                // voxel edge apart, a voxel is sqrt(3) edges across); a third
                // would still be added, directly
                const uint32_t twice = atomicOr(cell + 2 + half_word, bit);
                direct = (twice & bit) != 0;
            }
        }
        if (direct) {
            const size_t e = (size_t)idx * kBlockVoxels + voxel_slot(vol, lx, row & 7, row >> 3);
            add_to_voxel(vol, e, s.tsdf, 1.0f, s_pixf[kPxR * kRowPix + q],
                         s_pixf[kPxG * kRowPix + q], s_pixf[kPxB * kRowPix + q]);
        }
    }
    flush_rows<kFast>(vol, cam, sm);
    n_valid += (valid && part == 0) ? 1u : 0u;
}

// kAlways: block b pre-reduces 8 x 8 tile b / n of frame b % n.  Otherwise
// the blocks are persistent and take the dense 16 x 16 tiles that
// update_kernel listed, each as four 8 x 8 tiles.
template <bool kFast, bool kAlways>
__global__ void __launch_bounds__(kRowThreads, kRowBlocksPerSM) update_rows_kernel(
    VolumeView vol, const __grid_constant__ FrameBatch fb)
{
    extern __shared__ __align__(16) uint32_t sm[];
    const int t = threadIdx.x;
    uint32_t n_valid = 0, updates = 0, missed = 0;
    if (kAlways) {
        const TilePos tp = tile_of_block(fb, fb.by_tiles8_x, blockIdx.x);
        rows_tile<kFast>(vol, fb, tp.f, tp.tx * kRowTile, tp.ty * kRowTile, sm, n_valid, updates,
                         missed);
    } else {
        const uint32_t n_listed = *vol.dense_count;
        if (n_listed == 0) return;          // nothing listed: nothing taken, nothing to reset
        const uint32_t n_items = 4u * min(n_listed, vol.dense_capacity);
        uint32_t* s_item = sm + kOffCount + 2;
        for (;;) {
            if (t == 0) *s_item = atomicAdd(vol.dense_next, 1u);
            __syncthreads();
            const uint32_t j = *s_item;
            __syncthreads();                // all have read the item before it is replaced
            if (j >= n_items) break;        // uniform over the block
            const uint32_t entry = vol.dense_list[j >> 2];
            const int f = (int)(entry >> 24);
            const uint32_t tile16 = entry & 0xFFFFFFu;
            const uint32_t ty = divide_index(fb.by_tiles16_x, tile16);
            const int u0 = (int)(tile16 - ty * fb.by_tiles16_x.d) * 16 + (int)(j & 1u) * kRowTile;
            const int v0 = (int)ty * 16 + (int)((j >> 1) & 1u) * kRowTile;
            if (u0 < fb.width && v0 < fb.height)
                rows_tile<kFast>(vol, fb, f, u0, v0, sm, n_valid, updates, missed);
        }
        // the last block to finish leaves the list empty for the next launch
        // (stream order makes the reset visible to it)
        if (t == 0 && atomicAdd(vol.dense_done, 1u) == gridDim.x - 1) {
            *vol.dense_count = 0;
            *vol.dense_next = 0;
            *vol.dense_done = 0;
        }
    }
    const unsigned lane = lane_id();
    const uint32_t w_valid = __reduce_add_sync(0xFFFFFFFFu, n_valid);
    const uint32_t w_updates = __reduce_add_sync(0xFFFFFFFFu, updates);
    const uint32_t w_missed = __reduce_add_sync(0xFFFFFFFFu, missed);
    if (lane == 0) {
        const int stripe = blockIdx.x % kCounterStripes;
        if (w_valid) atomicAdd(&vol.counters->valid_points[stripe], (unsigned long long)w_valid);
        if (w_updates)
            atomicAdd(&vol.counters->voxel_updates[stripe], (unsigned long long)w_updates);
        if (w_missed) atomicAdd(&vol.counters->missed[stripe], (unsigned long long)w_missed);
    }
}

// The pre-reducing tile's second half (called by the whole block): list the
// non-empty voxels of the claimed rows, then flush them.
template <bool kFast>
__device__ __forceinline__ void flush_rows(const VolumeView& vol, const Camera& cam, uint32_t* sm)
{
    __syncthreads();
    const uint32_t* s_key = sm + kOffKey;
    const uint32_t* s_cells = sm + kOffCells;
    const float* s_pixf = reinterpret_cast<const float*>(sm + kOffPix);
    uint16_t* s_cell_list = reinterpret_cast<uint16_t*>(sm + kOffCellList);
    const int t = threadIdx.x;
    const unsigned lane = lane_id();

    // list the non-empty cells of the claimed rows, row by row, lx ascending
    const int n_rows = (int)sm[kOffCount];
    for (int base = t & ~31; base < 8 * n_rows; base += kRowThreads) {   // warp-uniform
        const int j = base + (int)lane;
        bool used = false;
        uint32_t code = 0;
        if (j < 8 * n_rows) {
            const uint32_t slot = sm[kOffList + (j >> 3)];
            const uint32_t* cell = s_cells + slot * kRowWords + (j & 7) * kCellWords;
            used = (cell[0] | cell[1]) != 0;
            code = slot << 3 | (uint32_t)(j & 7);
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, used);
        uint32_t pos = 0;
        if (lane == 0 && m) pos = atomicAdd(sm + kOffCount + 1, (uint32_t)__popc(m));
        pos = __shfl_sync(0xFFFFFFFFu, pos, 0);
        if (used) s_cell_list[pos + __popc(m & ((1u << lane) - 1u))] = (uint16_t)code;
    }
    __syncthreads();

    // flush: each listed cell recomputes its samples' tsdf from the pixel
    // depths and its voxel centre (the walk's own arithmetic), sums them with
    // the colours in pixel order, and adds the five sums to the pool; cells of
    // one row sit next to each other, so a row reaches L2 as a few sectors
    const int n_cells = (int)sm[kOffCount + 1];
    for (int k = t; k < n_cells; k += kRowThreads) {
        const uint32_t code = s_cell_list[k];
        const uint32_t slot = code >> 3;
        const int lx = (int)(code & 7u);
        const uint32_t row_key = s_key[slot];
        const unsigned long long block = reinterpret_cast<const unsigned long long*>(sm + kOffBlock)[slot];
        const uint4 cw = *reinterpret_cast<const uint4*>(s_cells + slot * kRowWords + lx * kCellWords);
        const int row = (int)(row_key & 63u);
        int bc[3];
        unpack_block(block, bc);
        const float zc = centre_depth(cam, vol.div.voxel, bc[0] * kBlockEdge + lx,
                                      bc[1] * kBlockEdge + (row & 7), bc[2] * kBlockEdge + (row >> 3));
        float sum[5] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t once = h == 0 ? cw.x : cw.y;
            const uint32_t twice = h == 0 ? cw.z : cw.w;
            while (once) {
                const int b = __ffs(once) - 1;
                once &= once - 1;
                const int px = h * 32 + b;
                const float tv = truncated_sdf<kFast>(vol.div, s_pixf[kPxD * kRowPix + px], zc);
                const int reps = (twice >> b & 1u) ? 2 : 1;
                for (int r = 0; r < reps; ++r) {
                    sum[0] = __fadd_rn(sum[0], tv);
                    sum[1] = __fadd_rn(sum[1], 1.0f);
                    sum[2] = __fadd_rn(sum[2], s_pixf[kPxR * kRowPix + px]);
                    sum[3] = __fadd_rn(sum[3], s_pixf[kPxG * kRowPix + px]);
                    sum[4] = __fadd_rn(sum[4], s_pixf[kPxB * kRowPix + px]);
                }
            }
        }
        const size_t e = (size_t)(row_key >> 6) * kBlockVoxels + voxel_slot(vol, lx, row & 7, row >> 3);
        add_to_voxel(vol, e, sum[0], sum[1], sum[2], sum[3], sum[4]);
    }
}

}  // namespace

// Opt in to the pre-reducing kernel's shared memory, once per device and
// instance.
template <bool kFast, bool kAlways>
cudaError_t launch_rows(const VolumeView& vol, const FrameBatch& fb, unsigned grid,
                        cudaStream_t stream)
{
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(update_rows_kernel<kFast, kAlways>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRowSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    update_rows_kernel<kFast, kAlways><<<grid, kRowThreads, kRowSmemBytes, stream>>>(vol, fb);
    return cudaGetLastError();
}

cudaError_t launch_update(const VolumeView& vol, const FrameBatch& fb, int kind,
                          cudaStream_t stream)
{
    // adaptive: the per-sample kernel takes the sparse 16 x 16 tiles and
    // lists the dense ones, which the persistent pre-reducing kernel takes
    if (kind == TSDF_UPDATE_ADAPTIVE &&
        (uint64_t)fb.width * (uint64_t)fb.height * (uint64_t)fb.n < kAdaptiveMinPixels)
        kind = TSDF_UPDATE_PER_SAMPLE;
    // the pre-reducing kernel recomputes a sample's value from its ray pixel's
    // depth, which the reprojection test does not use
    const bool reproject = vol.occlusion == TSDF_OCCLUSION_REPROJECT;
    if (reproject) kind = TSDF_UPDATE_PER_SAMPLE;
    if (kind != TSDF_UPDATE_PRE_REDUCED) {
        const unsigned tiles = (unsigned)(((fb.width + kTileW - 1) / kTileW) *
                                          ((fb.height + kTileH - 1) / kTileH));
        const unsigned grid = tiles * (unsigned)fb.n;
        const bool sparse_only = kind == TSDF_UPDATE_ADAPTIVE;
        if (reproject) {
            if (vol.fast_div) update_kernel<true, false, true><<<grid, kThreads, 0, stream>>>(vol, fb);
            else update_kernel<false, false, true><<<grid, kThreads, 0, stream>>>(vol, fb);
        } else if (vol.fast_div) {
            if (sparse_only) update_kernel<true, true, false><<<grid, kThreads, 0, stream>>>(vol, fb);
            else update_kernel<true, false, false><<<grid, kThreads, 0, stream>>>(vol, fb);
        } else {
            if (sparse_only) update_kernel<false, true, false><<<grid, kThreads, 0, stream>>>(vol, fb);
            else update_kernel<false, false, false><<<grid, kThreads, 0, stream>>>(vol, fb);
        }
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess || kind == TSDF_UPDATE_PER_SAMPLE) return e;
    }
    const bool always = kind == TSDF_UPDATE_PRE_REDUCED;
    unsigned grid;
    if (always) {
        grid = (unsigned)(((fb.width + kRowTile - 1) / kRowTile) *
                          ((fb.height + kRowTile - 1) / kRowTile)) * (unsigned)fb.n;
    } else {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        grid = (unsigned)(sms > 0 ? sms : 1) * kRowBlocksPerSM;
    }
    if (vol.fast_div)
        return always ? launch_rows<true, true>(vol, fb, grid, stream)
                      : launch_rows<true, false>(vol, fb, grid, stream);
    return always ? launch_rows<false, true>(vol, fb, grid, stream)
                  : launch_rows<false, false>(vol, fb, grid, stream);
}

}  // namespace tsdf
