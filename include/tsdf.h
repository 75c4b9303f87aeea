/*
 * tsdf.h -- C ABI of libtsdf.so: hash-blocked TSDF integration on one GPU.
 *
 * The operation is the integrate path of "What Irregularity Costs: CUDA C++,
 * Rust, and Triton on a Hash-Blocked GPU Workload" (arXiv 2608.08287):
 *
 *   design section, data structure: the volume is cut into blocks of
 *     8^3 = 512 voxels.  An open-addressed, linear-probing hash table of
 *     16-byte entries (a packed 64-bit block key, a 32-bit pool index, 4 bytes
 *     of padding), sized to a power of two at least twice the pool capacity,
 *     maps a block coordinate to an index into a flat pool holding five
 *     float sums per voxel: TSDF, weight, red, green and blue.
 *   design section, integration: two kernels run over the same
 *     back-projected depth points.  ALLOCATE walks each point's truncation
 *     band and inserts every missing block with a single 64-bit
 *     compare-exchange.  UPDATE walks the same band and adds each passing
 *     sample into its voxel with atomic additions.  Both apply the same
 *     occlusion test.
 *   design section, accumulation: the arrays hold sums, so the mean of a
 *     voxel is sum / weight, formed only at read-out.
 *
 * Per sample (band offsets (i - k) * voxel, i = 0..2k, k = round(trunc /
 * voxel), along the unit ray through the pixel's back-projected point):
 * voxel = floor(world / voxel); signed distance at the voxel CENTRE
 * sdf = depth - z_centre (camera frame); the sample passes iff
 * z_centre > 0 and sdf >= -trunc; it adds (min(1, sdf / trunc), 1, r, g, b).
 * The walk is computed in IEEE float32 with one rounding per operation
 * (no fused multiply-add), so the voxel each sample selects is reproducible
 * bit for bit by any IEEE implementation that evaluates the same operations
 * in the same order.
 *
 * Conventions
 *   - depth: float32 [height][width], metres, camera-frame z; a pixel is
 *     valid iff its depth is finite and > 0.
 *   - rgb: float32 [height][width][3] (any range; [0, 1] by convention).
 *   - K: host float[4] = {fx, fy, cx, cy}; pixel centres at integer (u, v).
 *   - pose: host float[16], row-major 4x4 camera-to-world [R | t] (the last
 *     row is ignored).
 *   - block coordinates must lie in [-2^20, 2^20 - 1] per axis (the 21-bit
 *     key fields); samples outside are counted (out_of_range_samples) and
 *     skipped.
 *   - voxel numbering in a block, at every call of this ABI (export,
 *     import, extraction): j = lx + 8 * ly + 64 * lz, x fastest.
 *   - pool layout: voxel (lx, ly, lz) of block b is record v = b * 512 + s.
 *     By default its TSDF, weight, red and green sums are interleaved in one
 *     16-byte record, floats 4v .. 4v + 3 of the record array, and its blue
 *     sum is element v of a separate blue array, with the block stored as
 *     64 bricks of 2 x 2 x 2 voxels: s = 8 * (lx/2 + 4 (ly/2) + 16 (lz/2)) +
 *     (lx%2) + 2 (ly%2) + 4 (lz%2) (a brick's records fill one 128-byte
 *     line); the pages' five separate arrays, x fastest (s = j), are
 *     available as TSDF_LAYOUT_PLANAR (tsdf_set_pool_layout).  The record lets a sample's update reach four
 *     of its five sums with one 4-wide reduction, and L2 executes reduction
 *     requests at about the same rate whether they carry one float or four.
 *     tsdf_export_blocks returns the five sums as separate arrays in both.
 *
 * Ownership and synchronisation
 *   - A tsdf_volume owns its device memory (table, pool, counters), allocated
 *     at create and released at destroy, on the device that was current at
 *     create.  Call every function with that device current: a call that
 *     touches the volume's memory from another current device returns
 *     TSDF_ERR_ARG and enqueues nothing (tsdf_destroy switches to the
 *     volume's device by itself).
 *   - Device pointers passed in (depth, rgb, coords) are borrowed: they must
 *     stay valid until the work enqueued on `stream` has finished.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     that enqueue work return without synchronising, except the read-out
 *     calls (block_count, export_*, get_stats), which synchronise `stream`.
 *   - A volume is not thread-safe; concurrent calls on one volume race.
 *     Work enqueued on one volume must also run in order on the device: use
 *     one stream per volume, or order different streams with events (the
 *     update keeps a per-launch work list in the volume's device state).
 *
 * Errors: every call returns TSDF_OK or a negative code.  On TSDF_ERR_ARG
 * nothing was enqueued.  tsdf_last_error() returns a message describing the
 * last failure on the calling thread.
 */
#ifndef TSDF_H
#define TSDF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TSDF_OK 0
#define TSDF_ERR_ARG (-1)      /* invalid argument; nothing enqueued */
#define TSDF_ERR_CUDA (-2)     /* a CUDA runtime call failed */
#define TSDF_ERR_OOM (-3)      /* a device or pinned allocation failed */

#define TSDF_BLOCK_VOXELS 512
#define TSDF_PROBE_HIST_BINS 32
#define TSDF_MAX_POOL_CAPACITY (1u << 23)
#define TSDF_MAX_TABLE_CAPACITY (1u << 30)
#define TSDF_MAX_BAND_SAMPLES 255
#define TSDF_EMPTY_KEY 0xFFFFFFFFFFFFFFFFull   /* key of an empty table slot */
#define TSDF_INDEX_PENDING 0xFFFFFFFFu         /* slot claimed, index not yet published */
#define TSDF_INDEX_FAILED 0xFFFFFFFEu          /* key inserted but the pool was full */

typedef struct tsdf_volume tsdf_volume;

typedef struct tsdf_info {
    uint32_t pool_capacity;     /* blocks in the pool */
    uint32_t table_capacity;    /* table slots (a power of two) */
    float voxel_size;           /* metres */
    float trunc;                /* metres */
    int32_t band_samples;       /* samples per point, 2k + 1 */
    int32_t device;             /* CUDA device ordinal that owns the memory */
    int32_t fixed_divisor_fast_path;  /* 1: the per-sample division by trunc uses a
                                          reciprocal-and-correction sequence that was
                                          checked at create to give the same truncated
                                          distance as IEEE division for every float32
                                          dividend; 0: IEEE division */
    int32_t max_frames_per_launch;    /* frames a batch call packs into one launch */
    int32_t pool_layout;              /* TSDF_LAYOUT_INTERLEAVED or TSDF_LAYOUT_PLANAR */
    int32_t voxel_division_fast_path; /* 1: the back-projection's division by the voxel
                                          edge uses the same sequence, checked at create
                                          to equal IEEE division bit for bit for every
                                          float32 dividend; 0: IEEE division */
} tsdf_info;

/* Device pointers to the pool's five sums.  Record v = b * 512 + s (block b,
 * voxel at position s of the pool layout: the brick order above in the
 * interleaved layout, s = j in the planar one) holds tsdf[stride * v],
 * weight[stride * v], r[stride * v] and g[stride * v], and b[v]: stride 4 in
 * the interleaved layout (weight = tsdf + 1, r = tsdf + 2, g = tsdf + 3),
 * stride 1 in the planar one (five separate arrays).  Each field spans pool_capacity * 512 voxels.  They stay valid until tsdf_destroy; reading them races with
 * kernels still running. */
typedef struct tsdf_pool_view {
    float* tsdf;
    float* weight;
    float* r;
    float* g;
    float* b;
    uint32_t pool_capacity;
    uint32_t stride;            /* floats between voxels in tsdf, weight, r, g: 4 or 1 */
} tsdf_pool_view;

/* Counters accumulated since create / reset / tsdf_clear_stats. */
typedef struct tsdf_stats {
    uint64_t blocks_allocated;      /* pool counter; may exceed capacity when exhausted */
    uint64_t pool_exhausted;        /* distinct keys inserted with no pool slot left */
    uint64_t probe_overflow;        /* inserts that examined every slot without success */
    uint64_t missed_contributions;  /* passing samples whose block was absent or FAILED */
    uint64_t out_of_range_samples;  /* samples outside the key range (allocate pass) */
    uint64_t valid_points;          /* valid pixels seen by the update pass */
    uint64_t voxel_updates;         /* samples accumulated by the update pass */
    /* probe statistics, collected only while instrumentation is on: */
    uint64_t probe_inserts;         /* insert probes issued (after de-duplication) */
    uint64_t probe_steps;           /* slots examined by those probes */
    uint64_t probe_max;             /* longest probe */
    uint64_t probe_hist[TSDF_PROBE_HIST_BINS];  /* bin b: probes of length b + 1; last bin: longer */
    uint64_t publish_timeouts;      /* fused integrate: waits for a published index that gave up
                                       (their samples count as missed); 0 in normal operation */
} tsdf_stats;

/* Create a volume of `pool_capacity` blocks, voxel edge `voxel_size` metres,
 * truncation `trunc` metres, with the default table size: the smallest power
 * of two strictly greater than 2 * pool_capacity ("What Irregularity Costs",
 * design section, data structure: blocks of 8^3 voxels, a flat pool of five
 * float sums per voxel, an open-addressed linear-probing table of 16-byte
 * entries sized to the next power of two above twice the pool capacity, so
 * that an occupied table is at most half full; "above" is read as strictly
 * above).  Requires
 * 1 <= pool_capacity <= TSDF_MAX_POOL_CAPACITY, finite voxel_size > 0 and
 * trunc > 0, and 2 * round(trunc / voxel_size) + 1 <= TSDF_MAX_BAND_SAMPLES.
 * Zeroes the pool and empties the table (synchronously).  *out receives the
 * handle, or NULL on failure. */
int tsdf_create(uint32_t pool_capacity, float voxel_size, float trunc, tsdf_volume** out);

/* As tsdf_create with an explicit table size: table_capacity must be a power
 * of two with 2 * pool_capacity <= table_capacity <= TSDF_MAX_TABLE_CAPACITY,
 * or 0 for the default (design section, data structure: any such table keeps
 * the load at or below one half; the load-factor sweep of the expressiveness
 * section varies the occupancy with the table fixed). */
int tsdf_create_ex(uint32_t pool_capacity, uint32_t table_capacity, float voxel_size,
                   float trunc, tsdf_volume** out);

/* (design section, layout shared by the arms: the volume's memory is
 * allocated once and handed to the kernels as pointers; this releases it.)
 * Release the volume's device memory, on the volume's device (the caller's
 * current device is restored).  It waits for the volume's own copy stream
 * (tsdf_integrate_batch_host); cudaFree itself waits for work already
 * enqueued on the device.  No other call may use the volume afterwards. */
int tsdf_destroy(tsdf_volume* vol);

/* The volume's parameters (design section, data structure: pool and table
 * capacities; integration: the band's sample count). */
int tsdf_get_info(const tsdf_volume* vol, tsdf_info* out);

/* Zero-copy access to the pool arrays, for read-out kernels of the caller
 * (design section, accumulation: the arrays hold sums, and a reader forms the
 * mean sum / weight itself). */
int tsdf_get_pool(const tsdf_volume* vol, tsdf_pool_view* out);

/* Empty the volume on `stream`: zero the used prefix of the pool (the first
 * min(blocks_allocated, pool_capacity) blocks' records and blue sums), empty the
 * table and zero every counter.  This is the fresh volume each timed allocate
 * starts from (measurement section: allocate is timed from an empty table;
 * design section, data structure: an empty slot holds the all-ones key). */
int tsdf_reset(tsdf_volume* vol, void* stream);

/* Integrate one frame: tsdf_allocate followed by tsdf_update on `stream`
 * (design section, integration: two kernels over the same points). */
int tsdf_integrate(tsdf_volume* vol, const float* depth, const float* rgb, int width,
                   int height, const float K[4], const float pose[16], void* stream);

/* The allocate kernel alone (design section, integration: the irregular
 * stage; the insert publishes a whole packed key with one compare-exchange):
 * make sure every block touched by a passing sample of this frame exists in
 * the table (keys are de-duplicated within a
 * warp before probing; a new key is claimed with one 64-bit compare-and-swap
 * and receives the next pool index).  Probing is unbounded up to the table
 * size; an insert that finds no slot counts probe_overflow, a key that finds
 * the pool full is published as TSDF_INDEX_FAILED and counts
 * pool_exhausted. */
int tsdf_allocate(tsdf_volume* vol, const float* depth, int width, int height,
                  const float K[4], const float pose[16], void* stream);

/* The update kernel alone (design section, integration: the regular stage,
 * a lookup that almost always hits at the first probe and atomic additions
 * into the five sums; accumulation: sums, not running means): add
 * (tsdf, 1, r, g, b) of every passing sample into its voxel.  A sample whose block is absent or FAILED counts
 * missed_contributions.  Call it after tsdf_allocate of the same frame (on
 * the same stream) for the full integrate semantics. */
int tsdf_update(tsdf_volume* vol, const float* depth, const float* rgb, int width,
                int height, const float K[4], const float pose[16], void* stream);

/* Integrate n_frames frames (design section, integration, applied to each
 * frame in turn; sums commute, accumulation).  depth: device float32
 * [n_frames][height][width];
 * rgb: device float32 [n_frames][height][width][3]; K: host float[4] shared by
 * all frames; poses: host float[n_frames][16].  Frames are taken in groups of
 * up to max_frames_per_launch (tsdf_info): one allocate launch over the group,
 * then one update launch over the group, whose blocks of threads run image
 * region by image region, frame-minor, so updates of the same voxels from
 * neighbouring frames meet in L2.  The result equals integrating the frames
 * one by one (same blocks, same weights; sums up to float summation order),
 * except under pool exhaustion, where which blocks are refused depends on the
 * order in which inserts win pool indices, which is unspecified.
 *
 * Every batch and single-frame call back-projects through a per-pixel ray
 * table the volume keeps for the last frame size and K (16 bytes per pixel
 * plus 4 per row), rebuilt on `stream` when either changes.  The first call
 * with a larger frame than any before allocates it (cudaMalloc, which
 * synchronises the device), so that call must not be made during stream
 * capture (TSDF_ERR_ARG); under capture the rebuild is always recorded. */
int tsdf_integrate_batch(tsdf_volume* vol, int n_frames, const float* depth, const float* rgb,
                         int width, int height, const float K[4], const float* poses,
                         void* stream);

/* The two stages of tsdf_integrate_batch separately, each over all n_frames
 * frames in launches of up to max_frames_per_launch frames: every allocate
 * launch of tsdf_allocate_batch, then (when called next on the same stream)
 * every update launch of tsdf_update_batch.  For timing the stages
 * (measurement section: stages timed on their own; results section: the
 * allocate stage's share of integrate). */
int tsdf_allocate_batch(tsdf_volume* vol, int n_frames, const float* depth, int width,
                        int height, const float K[4], const float* poses, void* stream);
int tsdf_update_batch(tsdf_volume* vol, int n_frames, const float* depth, const float* rgb,
                      int width, int height, const float K[4], const float* poses, void* stream);

/* As tsdf_integrate_batch, but depth and rgb are HOST arrays (design
 * section, extraction: host transfers are kept apart from kernel time; this
 * call overlaps them with the kernels instead).  Each group of
 * frames is copied into a double-buffered device staging area owned by the
 * volume on a separate copy stream, overlapping the copy of group g + 1 with
 * the kernels of group g.  The first group has 16 frames and each next one
 * about a third more, up to max_frames_per_launch, so that the kernels start
 * after a short copy instead of a full group's.  For the copies to be asynchronous the host arrays must be
 * page-locked (cudaHostAlloc / cudaHostRegister); pageable memory works but
 * serialises.  The host arrays must stay valid and unchanged until the work on
 * `stream` has finished.  The staging area is allocated on first use (and
 * grown for larger frames); that first call must not be made during stream
 * capture. */
int tsdf_integrate_batch_host(tsdf_volume* vol, int n_frames, const float* depth_host,
                              const float* rgb_host, int width, int height, const float K[4],
                              const float* poses, void* stream);

/* Insert explicit block coordinates (device int32 [n][3]) through the same
 * de-duplicate / probe / compare-and-swap / pool-index path as the allocate
 * kernel (design section, integration: the insert; expressiveness section:
 * the load-factor table, whose occupancies and clustered probe chains this
 * reaches without a scene).  Coordinates outside the key range count out_of_range_samples. */
int tsdf_allocate_blocks(tsdf_volume* vol, const int32_t* coords, uint32_t n, void* stream);

/* Synchronise `stream` and return min(blocks_allocated, pool_capacity): the
 * number of allocated blocks, which the correctness section checks exactly
 * against the reference (design section, occlusion: applying the test in
 * both passes keeps this count consistent). */
int tsdf_block_count(tsdf_volume* vol, void* stream, uint32_t* out);

/* Copy pool blocks [first, first + count) to the host, after synchronising
 * `stream` (design section, accumulation: the sums are read out and the mean
 * is formed only then; extraction: the device-to-host copy is a separate
 * step, not part of integrate): coords int32 [count][3] (block coordinates, recovered from the
 * table) and the five sums as separate arrays float32 [count][512] each.  Any
 * output pointer may be NULL to skip it.  first + count must not exceed
 * tsdf_block_count.  In the interleaved layout the first call that asks for
 * a sum allocates a 160 MB device scratch buffer (kept until tsdf_destroy)
 * in which the brick-ordered records are split into x-fastest arrays,
 * 16,384 blocks at a time.  Pool
 * order is the order in which blocks won their pool index, which is not
 * deterministic: compare by coordinate. */
int tsdf_export_blocks(tsdf_volume* vol, void* stream, uint32_t first, uint32_t count,
                       int32_t* coords, float* tsdf, float* weight, float* r, float* g,
                       float* b);

/* Block coordinates of pool blocks [first, first + count) into coords
 * (host int32 [count][3]), like the coords output of tsdf_export_blocks, but
 * without allocating any memory: for callers that cannot let the library
 * call cudaMalloc (device memory owned by a caching allocator that has
 * reserved nearly all of it, a fixed device-memory budget, threads that must
 * not stall in the allocator).  The paper has no counterpart; it is a
 * service of this library.  The coordinates pass through a scratch array
 * compiled into the library (TSDF_NOALLOC_MAX_BLOCKS blocks, 768 KB, held by
 * every GPU that loads the library until exit), so count must not exceed
 * TSDF_NOALLOC_MAX_BLOCKS (else TSDF_ERR_ARG, nothing done); first + count
 * must not exceed tsdf_block_count.  tsdf_create looks up the array's device
 * address (cudaGetSymbolAddress) with the volume's device current and loads
 * the export kernel, so that this call only uses them; a volume does not
 * survive cudaDeviceReset (create a new one afterwards).  Every call shares
 * the array and it keeps the last call's contents (each call clears the part
 * it uses): calls whose work overlaps on the GPU (other streams, other
 * threads) race.  Synchronises `stream`. */
#define TSDF_NOALLOC_MAX_BLOCKS 65536u
int tsdf_export_block_coords_noalloc(tsdf_volume* vol, void* stream, uint32_t first,
                                     uint32_t count, int32_t* coords);

/* Extract the surface: the zero level set of the mean TSDF (tsdf sum /
 * weight; "What Irregularity Costs", design section: sums are stored and the
 * mean is recovered at extraction, by marching tetrahedra).  Readings, as the
 * page gives no detail:
 *   - lattice points are voxel centres, world ((float)i + 0.5) * voxel_size
 *     per axis; a voxel is observed iff its weight > 0; its value is the
 *     float32 quotient tsdf / weight;
 *   - cell (i, j, k) spans voxels (i..i+1, j..j+1, k..k+1) and is used only if
 *     all 8 are observed; corner c has offset (c & 1, c >> 1 & 1, c >> 2 & 1);
 *   - each cell is cut into the 6 tetrahedra {0,1,3,7} {0,1,5,7} {0,2,3,7}
 *     {0,2,6,7} {0,4,5,7} {0,4,6,7} (watertight across cells);
 *   - a corner is inside when its value is < 0; a vertex lies on every
 *     tetrahedron edge whose ends differ, at t = fA / (fA - fB) from the
 *     lower-numbered end A: p = pA + t (pB - pA), float32;
 *   - one odd corner o (others a, b, c in tetrahedron order): triangle
 *     (E(o,a), E(o,b), E(o,c)); two inside i1 < i2, two outside o1 < o2:
 *     (E(i1,o1), E(i1,o2), E(i2,o2)) and (E(i1,o1), E(i2,o2), E(i2,o1)).
 * `triangles` is device memory, float32 [capacity][3][3] (triangle, vertex,
 * xyz), borrowed; the triangle order is unspecified.  *n_out receives the
 * total number of triangles, which may exceed `capacity`: then only
 * `capacity` of them are written (call again with a larger buffer).
 * `triangles` may be NULL with capacity 0 to count only.  The first call
 * allocates two device buffers kept until tsdf_destroy: the block
 * coordinates (12 B per pool block, shared with tsdf_export_blocks) and the
 * pool indices of each block's upper neighbours (32 B per pool block).
 * Synchronises
 * `stream`.  TSDF_ERR_ARG for a null n_out, or a null buffer with
 * capacity > 0. */
int tsdf_extract_triangles(tsdf_volume* vol, void* stream, float* triangles, uint64_t capacity,
                           uint64_t* n_out);

/* Set blocks from host arrays (restoring a saved volume, or loading a known
 * field; design section, accumulation: a volume's whole state is its block
 * set and the five sums of each voxel): for each of the n block coordinates (int32 [n][3], all distinct),
 * ensure the block exists through the allocate kernel's insert path, then
 * overwrite its five sums with tsdf, weight, r, g, b (float32 [n][512]
 * each, voxel j = lx + 8 ly + 64 lz, the layout tsdf_export_blocks
 * returns).  Blocks that find the pool full are counted (pool_exhausted) and
 * left unwritten; coordinates outside [-2^20, 2^20 - 1] are counted as out of
 * range.  The host arrays are copied before the call returns; the call
 * allocates and frees device staging and synchronises `stream`.
 * TSDF_ERR_ARG for a null array or a repeated coordinate (nothing is
 * enqueued), TSDF_ERR_OOM if staging cannot be allocated. */
int tsdf_import_blocks(tsdf_volume* vol, void* stream, uint32_t n, const int32_t* coords,
                       const float* tsdf, const float* weight, const float* r, const float* g,
                       const float* b);

/* Copy the raw hash table to the host after synchronising `stream` (design
 * section, data structure: the 16-byte entries with their packed keys and
 * pool indices; for checking the table's structure and probe chains): keys
 * uint64 [table_capacity] (TSDF_EMPTY_KEY for an empty slot) and indices
 * uint32 [table_capacity].  `capacity` must equal the table capacity. Either
 * output may be NULL. */
int tsdf_export_table(tsdf_volume* vol, void* stream, uint32_t capacity, uint64_t* keys,
                      uint32_t* indices);

/* Synchronise `stream` and read the counters (correctness section: no point
 * dropped and pool exhaustion reported; expressiveness section: dropped
 * blocks counted rather than lost, probe depth). */
int tsdf_get_stats(tsdf_volume* vol, void* stream, tsdf_stats* out);

/* Zero the counters (not the pool counter, the table or the pool), as
 * tsdf_get_stats reads them. */
int tsdf_clear_stats(tsdf_volume* vol, void* stream);

/* Turn probe instrumentation (probe_* statistics) on or off for later
 * launches (expressiveness section: probe depth under load).  It costs a shared-memory histogram per block of threads; keep it
 * off when timing. */
int tsdf_set_instrumentation(tsdf_volume* vol, int on);

/* How later update launches (integrate, update and their batch forms) add
 * the samples to the pool.  Every mode computes the same sums ("What
 * Irregularity Costs", design section, integration: the update adds tsdf, 1
 * and the pixel colour into the five sums for every passing sample); they
 * differ in how the additions reach memory:
 *   TSDF_UPDATE_AUTO (the default): TSDF_UPDATE_PER_SAMPLE, except that
 *     calls which both allocate and update (tsdf_integrate and its batch
 *     forms) run TSDF_UPDATE_FUSED's single kernel for launches of fewer than
 *     2^19 pixels (frames x width x height), where the two kernels would not
 *     fill the GPU and their latencies add up (same conditions as the fused
 *     mode: ray-depth test, bands of at most 9 samples).
 *   TSDF_UPDATE_PER_SAMPLE: each thread walks one pixel's band
 *     (16 x 16 pixel tiles, 8 x 4 per warp); at every band step the warp sums
 *     in registers the samples of its lanes that fall in the same voxel, and
 *     one lane adds them with two reductions (a 4-wide one into the voxel's
 *     tsdf, weight, red, green record, a scalar one into blue).
 *   TSDF_UPDATE_ADAPTIVE: each 16 x 16 pixel tile of a frame chooses between
 *     the per-sample path and the pre-reduction below.  Where at least half of
 *     its valid pixels see a voxel edge w or more pixels wide
 *     (voxel_size * fx >= w * depth; w = 5 when a launch holds 4 or more
 *     frames, else 10), the tile pre-reduces; launches of fewer than 2^18
 *     pixels in all never do.  (On GB300 the per-sample path with its warp
 *     merge is faster in every regime measured, dense ones included.)
 *   TSDF_UPDATE_PRE_REDUCED: every tile pre-reduces: it records in shared
 *     memory which of its pixels reached each voxel (once or twice), then sums
 *     every touched voxel's contributions in pixel order and adds the five
 *     sums to the pool once, a row of 8 voxels at a time.
 *   TSDF_UPDATE_FUSED: calls that both allocate and update (tsdf_integrate and
 *     its batch forms) run one fused kernel instead of the two: each pixel's
 *     band is walked once, its samples kept in registers while its block keys
 *     go through the allocate kernel's insert rounds, and each key's pool
 *     index then serves the update's additions (merged per warp and band step
 *     as in the per-sample path).  A key claimed by another thread of the
 *     launch is used once that thread has published its index (the wait on
 *     PENDING, bounded: a wait that gives up is counted in publish_timeouts
 *     and its samples in missed_contributions).  Bands longer than 9 samples,
 *     update-only calls and the reprojection occlusion test use the
 *     two-kernel path (per sample).
 * Returns TSDF_ERR_ARG for any other value. */
#define TSDF_UPDATE_ADAPTIVE 0
#define TSDF_UPDATE_PER_SAMPLE 1
#define TSDF_UPDATE_PRE_REDUCED 2
#define TSDF_UPDATE_FUSED 3
#define TSDF_UPDATE_AUTO 4
int tsdf_set_update_kernel(tsdf_volume* vol, int kind);

/* The occlusion test of later allocate and update launches.  The design
 * section (occlusion) fixes that both passes apply the same test but not its
 * formula; two readings are offered, and both passes always use the same one:
 *   TSDF_OCCLUSION_RAY (the default): the test above, against the depth of
 *     the pixel whose ray selected the voxel.
 *   TSDF_OCCLUSION_REPROJECT: the centre of the sample's voxel, in camera
 *     coordinates c = R^T (centre - t), is projected through the pinhole,
 *     u = fx (c_x / c_z) + cx, v = fy (c_y / c_z) + cy (IEEE float32, one
 *     rounding per operation), and rounded to the nearest pixel centre
 *     (floor(u + 1/2), floor(v + 1/2)).  The sample passes iff c_z > 0, that
 *     pixel lies inside the image with a valid depth d', and
 *     d' - c_z >= -trunc; it then adds (min(1, (d' - c_z) / trunc), 1, and
 *     that pixel's colour).  The band walk and its voxels are unchanged.
 *     Updates under this test always add their samples one by one
 *     (TSDF_UPDATE_PER_SAMPLE) whatever the update mode, and allocate and
 *     update run as two kernels.
 * Switching between launches is allowed; each sample is added under the test
 * in force when its update ran.  Returns TSDF_ERR_ARG for any other value. */
#define TSDF_OCCLUSION_RAY 0
#define TSDF_OCCLUSION_REPROJECT 1
int tsdf_set_occlusion(tsdf_volume* vol, int mode);

/* How the pool stores the five sums of a voxel (record v = b * 512 + s):
 *   TSDF_LAYOUT_INTERLEAVED (the default): TSDF, weight, red and green sums
 *     in one 16-byte record per voxel, blue in an array of its own, voxels
 *     in 2 x 2 x 2 bricks (s as above); an update adds a sample with one
 *     4-wide and one scalar reduction.
 *   TSDF_LAYOUT_PLANAR: five separate float arrays [pool_capacity][512]
 *     (the pages' own layout, "design section, data structure"); an update
 *     adds a sample with five scalar reductions, a row of 8 voxels being one
 *     32-byte sector of each array.
 * Every mode and kernel works in both; the sums are the same.  The layout can
 * only change while the volume holds no block (after create, or after
 * tsdf_reset; the call synchronises the legacy default stream to check),
 * else TSDF_ERR_ARG.  tsdf_get_pool reports the layout through its stride. */
#define TSDF_LAYOUT_INTERLEAVED 0
#define TSDF_LAYOUT_PLANAR 1
int tsdf_set_pool_layout(tsdf_volume* vol, int layout);

/* Message of the last failure on the calling thread ("" if none); every
 * call of this C ABI (design section, layout shared by the arms: a C ABI
 * handing pointers across) reports failures by code and message. */
const char* tsdf_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TSDF_H */
