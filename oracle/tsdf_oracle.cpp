/*
 * CPU oracle for hash-blocked TSDF integration.  TEST INFRASTRUCTURE ONLY:
 * the tests, the smoke check and the benchmark's CPU-baseline leg may call
 * it; the product path never does.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * What it restates (from "What Irregularity Costs: CUDA C++, Rust, and
 * Triton on a Hash-Blocked GPU Workload", arXiv 2608.08287):
 *
 *   - design section, data structure: the volume is cut into blocks of
 *     8^3 = 512 voxels; each block holds five per-voxel quantities (signed
 *     distance, weight, three colour channels);
 *   - design section, integration: two passes over the same back-projected
 *     points.  The first (allocate) walks each point's truncation band and
 *     makes sure every block it touches exists; the second (update) walks the
 *     same band and adds each observation into its voxel;
 *   - design section, accumulation: the arrays hold weighted SUMS, not
 *     running means, so the mean is only formed at read-out;
 *   - design section, occlusion: one occlusion test, applied identically in
 *     both passes;
 *   - correctness section (analytic tier): the signed distance is evaluated
 *     at the voxel centre, not at the ray sample that selected the voxel.
 *
 * Where the page is silent this file takes the following readings (they are
 * listed with their reasons in the design notes of the repository):
 *   - pinhole camera, pixel centres at integer (u, v), x right, y down,
 *     z forward; pose = camera-to-world [R | t], R row-major;
 *   - the band is walked along the unit ray through the observed point, in
 *     steps of one voxel, S = 2k + 1 samples at offsets (i - k) * voxel with
 *     k = round(trunc / voxel); evaluated in voxel units: per pixel the
 *     observed point p' = (R p + t) / voxel and the world direction e = R dir,
 *     per sample p' + j e (j = i - k), whose floor is the voxel;
 *   - projective signed distance at the voxel centre: sdf = d - z_c, where z_c
 *     is the camera-frame depth of the centre and d the pixel's depth;
 *   - occlusion test: z_c > 0 and sdf >= -trunc;
 *   - alternative occlusion test (selected per volume): the voxel centre is
 *     projected into the frame and tested against the depth of the nearest
 *     pixel, floor(u + 1/2), floor(v + 1/2); the sample passes when that
 *     pixel lies inside the image with a valid depth d' and d' - z_c >=
 *     -trunc; it then adds min(1, (d' - z_c) / trunc) and that pixel's
 *     colour (the walk and its voxels are unchanged);
 *   - value added: tsdf = min(1, sdf / trunc), weight 1, the pixel's colour;
 *   - voxel order inside a block: x fastest, j = lx + 8 ly + 64 lz;
 *   - block coordinates must lie in [-2^20, 2^20 - 1] on every axis (the
 *     range of the packed 21-bit key); samples outside are counted, skipped.
 *
 * Arithmetic: the walk is float32 with one rounding per written operation,
 * evaluated in the order written (the library is compiled with
 * -ffp-contract=off and without fast-math), so that the voxel each sample
 * selects is defined to the bit.  The sums are accumulated in double, i.e.
 * they are the exact sums of the float32 terms up to double rounding.
 *
 * The blocks live in a std::unordered_map keyed by block coordinate; the
 * oracle never uses the packed key or the hash table.  The key packing, the
 * multiply-xor slot hash and a sequential linear-probing table are restated
 * separately at the end of this file, as a reference for the table's
 * structure (occupied slots, displacement), not as part of integration.
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <memory>
#include <unordered_map>
#include <unordered_set>
#include <vector>

/* Planted mistakes for the self-test of the pins.  Every normal build has
 * ORACLE_MUTANT == 0; the test suite compiles throw-away variants with one
 * mistake each and checks that some pin rejects every one of them. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

namespace {

const int kEdge = 8;                 // voxels per block edge
const int kBlockVoxels = 512;        // 8^3
const int32_t kCoordMin = -(1 << 20);
const int32_t kCoordMax = (1 << 20) - 1;

struct BlockCoord {
    int32_t x, y, z;
};

bool operator==(const BlockCoord& a, const BlockCoord& b)
{
    return a.x == b.x && a.y == b.y && a.z == b.z;
}

bool operator<(const BlockCoord& a, const BlockCoord& b)
{
    if (a.x != b.x) return a.x < b.x;
    if (a.y != b.y) return a.y < b.y;
    return a.z < b.z;
}

struct BlockCoordHash {
    size_t operator()(const BlockCoord& c) const noexcept
    {
        size_t h = std::hash<int32_t>()(c.x);
        h = h * 1000003u + std::hash<int32_t>()(c.y);
        h = h * 1000003u + std::hash<int32_t>()(c.z);
        return h;
    }
};

/* Exact-as-possible per-voxel sums of one block.  tsdf_abs is the sum of
 * |tsdf| over the same terms, kept so a test can bound the float32 rounding
 * error of any summation order. */
struct BlockSums {
    double tsdf[kBlockVoxels];
    double weight[kBlockVoxels];
    double r[kBlockVoxels];
    double g[kBlockVoxels];
    double b[kBlockVoxels];
    double tsdf_abs[kBlockVoxels];
};

struct Camera {
    float fx, fy, cx, cy;
    float R[3][3];   // camera-to-world rotation, row-major
    float t[3];      // camera position in the world
};

enum SampleStatus { SAMPLE_PASS = 0, SAMPLE_OCCLUDED = 1, SAMPLE_OUT_OF_RANGE = 2 };

struct Sample {
    int32_t ix, iy, iz;   // voxel index
    float tsdf;
};

/* floor(a / 8) for any int32 a, written without shifts. */
int32_t floor_div8(int32_t a)
{
#if ORACLE_MUTANT == 9
    return a / kEdge;                       // planted: truncates toward zero
#else
    int32_t q = a / kEdge;
    if (a % kEdge != 0 && a < 0) q -= 1;
    return q;
#endif
}

/* The part of the band walk shared by a pixel's samples: the observed point
 * in world coordinates divided by the voxel edge, p' = (R p + t) / voxel, and
 * the unit ray direction in world coordinates, e = R dir.  Sample i lies at
 * p + i voxel dir, i.e. at p' + i e in voxel units. */
struct WalkRay {
    float d;              // the pixel's depth
    float vx, vy, vz;     // p'
    float ex, ey, ez;     // e
    float pz, dz;         // camera-frame z of p and of dir (planted mistake 1 only)
};

/* One sample of the truncation band: band step i (offset i voxels from the
 * observed point along the unit ray), its voxel, and the truncated signed
 * distance at that voxel's centre. */
SampleStatus band_sample(const Camera& cam, float voxel, float trunc, const WalkRay& r, int i,
                         Sample* s)
{
    const float d = r.d;
    // the sample in voxel units: p' + i e
    float fi = (float)i;
    float wx = r.vx + fi * r.ex;
    float wy = r.vy + fi * r.ey;
    float wz = r.vz + fi * r.ez;
    // voxel index = floor of the sample in voxel units, kept inside the
    // packable block range
#if ORACLE_MUTANT == 8
    float qx = std::trunc(wx), qy = std::trunc(wy), qz = std::trunc(wz);   // planted
#else
    float qx = std::floor(wx), qy = std::floor(wy), qz = std::floor(wz);
#endif
    const float lo = (float)kCoordMin * kEdge;           // -2^23
    const float hi = (float)(kCoordMax * kEdge + (kEdge - 1));  // 2^23 - 1
    if (!(qx >= lo && qx <= hi && qy >= lo && qy <= hi && qz >= lo && qz <= hi))
        return SAMPLE_OUT_OF_RANGE;
    s->ix = (int32_t)qx;
    s->iy = (int32_t)qy;
    s->iz = (int32_t)qz;
    // the voxel centre, moved to the camera origin ...
#if ORACLE_MUTANT == 3
    float cxw = ((float)s->ix) * voxel - cam.t[0];      // planted: corner, not centre
    float cyw = ((float)s->iy) * voxel - cam.t[1];
    float czw = ((float)s->iz) * voxel - cam.t[2];
#else
    float cxw = ((float)s->ix + 0.5f) * voxel - cam.t[0];
    float cyw = ((float)s->iy + 0.5f) * voxel - cam.t[1];
    float czw = ((float)s->iz + 0.5f) * voxel - cam.t[2];
#endif
    // ... and its camera-frame depth z_c = (R^T c)_z = column 2 of R dotted with c
#if ORACLE_MUTANT == 4
    float zc = (cam.R[2][0] * cxw + cam.R[2][1] * cyw) + cam.R[2][2] * czw;  // planted: R not transposed
#else
    float zc = (cam.R[0][2] * cxw + cam.R[1][2] * cyw) + cam.R[2][2] * czw;
#endif
    // projective signed distance at the centre (positive in front of the surface)
#if ORACLE_MUTANT == 1
    float sdf = d - (r.pz + ((float)i * voxel) * r.dz);   // planted: at the sample, not the centre
#elif ORACLE_MUTANT == 2
    float sdf = zc - d;                     // planted: sign flipped
#else
    float sdf = d - zc;
#endif
    // occlusion test
#if ORACLE_MUTANT == 6
    if (!(zc > 0.0f)) return SAMPLE_OCCLUDED;            // planted: no truncation side test
#else
    if (!(zc > 0.0f && sdf >= -trunc)) return SAMPLE_OCCLUDED;
#endif
#if ORACLE_MUTANT == 7
    s->tsdf = sdf / trunc;                  // planted: no clamp at +1
#else
    s->tsdf = std::fmin(1.0f, sdf / trunc);
#endif
    return SAMPLE_PASS;
}

/* The alternative occlusion test, by reprojection.  The centre of the
 * sample's voxel, in camera coordinates c = R^T (centre - t), is projected
 * through the pinhole, u = fx (c_x / c_z) + cx, v = fy (c_y / c_z) + cy, and
 * rounded to the nearest pixel centre.  The sample passes when the centre is
 * in front of the camera, the pixel lies inside the image and holds a valid
 * depth d', and the centre is no more than one truncation distance behind
 * it; the value is then min(1, (d' - c_z) / trunc) and *pix is the pixel
 * whose colour the sample adds.  `d_ray` is the depth of the pixel whose ray
 * selected the voxel; the test itself does not use it. */
SampleStatus reprojected_sample(const Camera& cam, float voxel, float trunc, const float* depth,
                                int W, int H, float d_ray, Sample* s, long long* pix)
{
    (void)d_ray;
    float cxw = ((float)s->ix + 0.5f) * voxel - cam.t[0];
    float cyw = ((float)s->iy + 0.5f) * voxel - cam.t[1];
    float czw = ((float)s->iz + 0.5f) * voxel - cam.t[2];
    // c = R^T (centre - t): component k is column k of R dotted with the centre
#if ORACLE_MUTANT == 22
    float x = (cam.R[0][0] * cxw + cam.R[0][1] * cyw) + cam.R[0][2] * czw;  // planted: R, not R^T
    float y = (cam.R[1][0] * cxw + cam.R[1][1] * cyw) + cam.R[1][2] * czw;
#else
    float x = (cam.R[0][0] * cxw + cam.R[1][0] * cyw) + cam.R[2][0] * czw;
    float y = (cam.R[0][1] * cxw + cam.R[1][1] * cyw) + cam.R[2][1] * czw;
#endif
    float z = (cam.R[0][2] * cxw + cam.R[1][2] * cyw) + cam.R[2][2] * czw;
    if (!(z > 0.0f)) return SAMPLE_OCCLUDED;
#if ORACLE_MUTANT == 20
    float u = cam.fx * (y / z) + cam.cx;          // planted: x and y swapped
    float v = cam.fy * (x / z) + cam.cy;
#else
    float u = cam.fx * (x / z) + cam.cx;
    float v = cam.fy * (y / z) + cam.cy;
#endif
    // nearest pixel centre: floor(u + 1/2), inside [0, W) x [0, H)
#if ORACLE_MUTANT == 19
    float uh = u, vh = v;                          // planted: rounds down, not to nearest
#else
    float uh = u + 0.5f, vh = v + 0.5f;
#endif
    if (!(uh >= 0.0f && uh < (float)W && vh >= 0.0f && vh < (float)H)) return SAMPLE_OCCLUDED;
    long long pu = (long long)std::floor(uh), pv = (long long)std::floor(vh);
    long long p = pv * W + pu;
#if ORACLE_MUTANT == 21
    float d = d_ray;                               // planted: the ray pixel's depth
#else
    float d = depth[p];
#endif
    if (!(std::isfinite(d) && d > 0.0f)) return SAMPLE_OCCLUDED;
    float sdf = d - z;
    if (!(sdf >= -trunc)) return SAMPLE_OCCLUDED;
    s->tsdf = std::fmin(1.0f, sdf / trunc);
    *pix = p;
    return SAMPLE_PASS;
}

/* Walk the truncation band of pixel (u, v) with depth d, calling
 * visit(status, sample) once per band sample.  Returns false (and visits
 * nothing) for an invalid pixel. */
template <class Visit>
bool walk_pixel(const Camera& cam, float voxel, float trunc, int band_half,
                int u, int v, float d, Visit visit)
{
    if (!(std::isfinite(d) && d > 0.0f)) return false;
    // back-project the pixel: p = d * ((u - cx) / fx, (v - cy) / fy, 1)
    float xn = ((float)u - cam.cx) / cam.fx;
    float yn = ((float)v - cam.cy) / cam.fy;
    float px = xn * d, py = yn * d, pz = d;
    // unit ray direction through the pixel
    float len = std::sqrt((xn * xn + yn * yn) + 1.0f);
#if ORACLE_MUTANT == 14
    float dx = xn, dy = yn, dz = 1.0f;      // planted: ray not normalised
    (void)len;
#else
    float dx = xn / len, dy = yn / len, dz = 1.0f / len;
#endif
    // the observed point and the direction in world coordinates, the point
    // in voxel units: p' = (R p + t) / voxel, e = R dir (rows of R summed
    // left to right)
    WalkRay r;
    r.d = d;
#if ORACLE_MUTANT == 26
    r.vx = ((cam.R[0][0] * px + cam.R[0][1] * py) + cam.R[0][2] * pz) / voxel + cam.t[0];  // planted:
    r.vy = ((cam.R[1][0] * px + cam.R[1][1] * py) + cam.R[1][2] * pz) / voxel + cam.t[1];  // t not in
    r.vz = ((cam.R[2][0] * px + cam.R[2][1] * py) + cam.R[2][2] * pz) / voxel + cam.t[2];  // voxels
#else
    r.vx = (((cam.R[0][0] * px + cam.R[0][1] * py) + cam.R[0][2] * pz) + cam.t[0]) / voxel;
    r.vy = (((cam.R[1][0] * px + cam.R[1][1] * py) + cam.R[1][2] * pz) + cam.t[1]) / voxel;
    r.vz = (((cam.R[2][0] * px + cam.R[2][1] * py) + cam.R[2][2] * pz) + cam.t[2]) / voxel;
#endif
#if ORACLE_MUTANT == 25
    r.ex = (cam.R[0][0] * dx + cam.R[1][0] * dy) + cam.R[2][0] * dz;   // planted: R^T dir
    r.ey = (cam.R[0][1] * dx + cam.R[1][1] * dy) + cam.R[2][1] * dz;
    r.ez = (cam.R[0][2] * dx + cam.R[1][2] * dy) + cam.R[2][2] * dz;
#else
    r.ex = (cam.R[0][0] * dx + cam.R[0][1] * dy) + cam.R[0][2] * dz;
    r.ey = (cam.R[1][0] * dx + cam.R[1][1] * dy) + cam.R[1][2] * dz;
    r.ez = (cam.R[2][0] * dx + cam.R[2][1] * dy) + cam.R[2][2] * dz;
#endif
    r.pz = pz;
    r.dz = dz;
#if ORACLE_MUTANT == 13
    int steps_half = band_half + 1;         // planted: band one voxel too wide
#else
    int steps_half = band_half;
#endif
    for (int i = -steps_half; i <= steps_half; ++i) {
        Sample s;
        SampleStatus st = band_sample(cam, voxel, trunc, r, i, &s);
        visit(st, s);
    }
    return true;
}

struct Volume {
    float voxel;
    float trunc;
    int band_half;           // k: samples at offsets -k..k voxels
    long long block_limit;   // < 0: no pool limit
    bool reproject = false;  // occlusion test by reprojection instead of the ray's depth

    bool keep_all = true;    // false: sums are kept only for blocks in `keep`
    std::unordered_set<BlockCoord, BlockCoordHash> keep;
    int keep_parts = 0;      // > 0: sums are kept only for blocks of partition keep_part
    int keep_part = 0;

    // every allocated block; the sums pointer is null when not kept
    std::unordered_map<BlockCoord, std::unique_ptr<BlockSums>, BlockCoordHash> blocks;
    // keys that found the pool full (each counted once)
    std::unordered_set<BlockCoord, BlockCoordHash> dropped;

    unsigned long long valid_points = 0;          // pixels with finite depth > 0
    unsigned long long passing_samples = 0;       // samples that pass the occlusion test
    unsigned long long accumulated = 0;           // passing samples added into a block
    unsigned long long missed_contributions = 0;  // passing samples whose block is absent
    unsigned long long out_of_range_samples = 0;  // samples outside the key range
    unsigned long long dropped_blocks = 0;        // distinct keys refused for lack of pool
    unsigned long long bad_local_index = 0;       // self-check: local index outside [0, 512)
};

/* Partition of a block for keep_partition: (bx + by + bz) mod parts, taken
 * non-negative.  It only selects which blocks' sums are kept. */
bool in_partition(const Volume& v, const BlockCoord& b)
{
    if (v.keep_parts <= 0) return false;
    const long long s = (long long)b.x + (long long)b.y + (long long)b.z;
    const long long m = ((s % v.keep_parts) + v.keep_parts) % v.keep_parts;
    return m == v.keep_part;
}

BlockCoord block_of(const Sample& s)
{
    return BlockCoord{floor_div8(s.ix), floor_div8(s.iy), floor_div8(s.iz)};
}

int local_index(const Sample& s, const BlockCoord& b)
{
    int lx = s.ix - kEdge * b.x, ly = s.iy - kEdge * b.y, lz = s.iz - kEdge * b.z;
#if ORACLE_MUTANT == 5
    return lz + kEdge * ly + kEdge * kEdge * lx;   // planted: x slowest
#else
    return lx + kEdge * ly + kEdge * kEdge * lz;
#endif
}

Camera make_camera(const float K[4], const float pose[16])
{
    Camera c;
    c.fx = K[0];
    c.fy = K[1];
    c.cx = K[2];
    c.cy = K[3];
    for (int r = 0; r < 3; ++r) {
        for (int k = 0; k < 3; ++k) c.R[r][k] = pose[4 * r + k];
        c.t[r] = pose[4 * r + 3];
    }
    return c;
}

}  // namespace

extern "C" {

/* ------------------------------------------------------------------------
 * Integration
 * --------------------------------------------------------------------- */

void* oracle_create(float voxel_size, float trunc, long long block_limit)
{
    if (!(voxel_size > 0.0f) || !(trunc > 0.0f) || !std::isfinite(voxel_size) ||
        !std::isfinite(trunc))
        return nullptr;
    Volume* v = new Volume();
    v->voxel = voxel_size;
    v->trunc = trunc;
    v->band_half = (int)std::lround((double)trunc / (double)voxel_size);
    v->block_limit = block_limit;
    return v;
}

void oracle_destroy(void* h) { delete static_cast<Volume*>(h); }

/* Keep sums only for the listed blocks (coords: n x 3).  The block set and
 * all counters are still tracked for every block. */
int oracle_keep_only(void* h, const int32_t* coords, long long n)
{
    Volume* v = static_cast<Volume*>(h);
    if (!v->blocks.empty()) return -1;
    v->keep_all = false;
    for (long long i = 0; i < n; ++i)
        v->keep.insert(BlockCoord{coords[3 * i], coords[3 * i + 1], coords[3 * i + 2]});
    return 0;
}

/* The band walk of one pixel (u, v) with depth d, as the integrator walks
 * it under the ray-depth test: for band sample i = 0 .. 2k, its voxel index
 * (ix_out[3 i .. 3 i + 2], left unset when out of range) and status
 * (status_out[i]: 0 passes, 1 occluded, 2 out of range).  Returns the number
 * of samples, or 0 for an invalid depth.  For checking the walk on its own;
 * it changes nothing in the volume. */
int oracle_walk(void* h, const float K[4], const float pose[16], int u, int v, float d,
                int32_t* ix_out, int32_t* status_out)
{
    Volume* vol = static_cast<Volume*>(h);
    const Camera cam = make_camera(K, pose);
    int n = 0;
    walk_pixel(cam, vol->voxel, vol->trunc, vol->band_half, u, v, d,
               [&](SampleStatus st, const Sample& s) {
        status_out[n] = (int32_t)st;
        if (st != SAMPLE_OUT_OF_RANGE) {
            ix_out[3 * n] = s.ix;
            ix_out[3 * n + 1] = s.iy;
            ix_out[3 * n + 2] = s.iz;
        }
        ++n;
    });
    return n;
}

/* Keep sums only for the blocks whose (bx + by + bz) mod parts equals part
 * (taken non-negative): `parts` calls with part = 0 .. parts - 1 split the
 * volume into disjoint pieces that together hold every block.  The block set
 * and all counters are still tracked for every block. */
int oracle_keep_partition(void* h, int parts, int part)
{
    Volume* v = static_cast<Volume*>(h);
    if (!v->blocks.empty() || parts < 1 || part < 0 || part >= parts) return -1;
    v->keep_all = false;
    v->keep_parts = parts;
    v->keep_part = part;
    return 0;
}

/* Integrate one frame: depth float32 [H][W] (metres, 0 = invalid),
 * rgb float32 [H][W][3], K = {fx, fy, cx, cy}, pose = row-major 4x4
 * camera-to-world. */
int oracle_integrate(void* h, const float* depth, const float* rgb, int W, int H,
                     const float K[4], const float pose[16])
{
    Volume* v = static_cast<Volume*>(h);
    if (W <= 0 || H <= 0) return -1;
    const Camera cam = make_camera(K, pose);

    // Pass 1, allocate: every block touched by a passing sample exists
    // afterwards (unless the pool limit refuses it).
    for (int py = 0; py < H; ++py) {
        for (int px = 0; px < W; ++px) {
            float d = depth[(size_t)py * W + px];
            walk_pixel(cam, v->voxel, v->trunc, v->band_half, px, py, d,
                       [&](SampleStatus st, const Sample& s0) {
                if (st == SAMPLE_OUT_OF_RANGE) {
                    v->out_of_range_samples++;
                    return;
                }
                Sample s = s0;
                long long pix = 0;
                if (v->reproject) st = reprojected_sample(cam, v->voxel, v->trunc, depth, W, H, d,
                                                          &s, &pix);
                bool allocate = (st == SAMPLE_PASS);
#if ORACLE_MUTANT == 12
                allocate = true;                   // planted: allocate ignores occlusion
#endif
                if (!allocate) return;
                BlockCoord b = block_of(s);
                if (v->blocks.count(b) || v->dropped.count(b)) return;
                if (v->block_limit >= 0 && (long long)v->blocks.size() >= v->block_limit) {
                    v->dropped.insert(b);
                    v->dropped_blocks++;
                    return;
                }
                std::unique_ptr<BlockSums> sums;
                if (v->keep_all || v->keep.count(b) || in_partition(*v, b)) {
                    sums.reset(new BlockSums);
                    std::memset(sums.get(), 0, sizeof(BlockSums));
                }
                v->blocks.emplace(b, std::move(sums));
            });
        }
    }

    // Pass 2, update: add (tsdf, 1, r, g, b) of every passing sample into
    // its voxel's sums.
    for (int py = 0; py < H; ++py) {
        for (int px = 0; px < W; ++px) {
            size_t pix = (size_t)py * W + px;
            float d = depth[pix];
            float cr = rgb[3 * pix + 0], cg = rgb[3 * pix + 1], cb = rgb[3 * pix + 2];
#if ORACLE_MUTANT == 10
            std::swap(cr, cb);                     // planted: red and blue swapped
#endif
            bool valid = walk_pixel(cam, v->voxel, v->trunc, v->band_half, px, py, d,
                                    [&](SampleStatus st, const Sample& s0) {
                Sample s = s0;
                float sr = cr, sg = cg, sb = cb;
                if (v->reproject && st != SAMPLE_OUT_OF_RANGE) {
                    long long q = 0;
                    st = reprojected_sample(cam, v->voxel, v->trunc, depth, W, H, d, &s, &q);
#if ORACLE_MUTANT != 23
                    if (st == SAMPLE_PASS) {       // the colour of the pixel tested against
                        sr = rgb[3 * q + 0];
                        sg = rgb[3 * q + 1];
                        sb = rgb[3 * q + 2];
                    }
#endif                                             // (planted 23: the ray pixel's colour)
                }
                if (st != SAMPLE_PASS) return;
                v->passing_samples++;
                BlockCoord b = block_of(s);
                auto it = v->blocks.find(b);
                if (it == v->blocks.end()) {
                    v->missed_contributions++;
                    return;
                }
                v->accumulated++;
                BlockSums* sums = it->second.get();
                if (!sums) return;
                int j = local_index(s, b);
                if (j < 0 || j >= kBlockVoxels) {          // cannot happen in a correct build
                    v->bad_local_index++;
                    return;
                }
                sums->tsdf[j] += (double)s.tsdf;
                sums->tsdf_abs[j] += std::fabs((double)s.tsdf);
#if ORACLE_MUTANT == 11
                sums->weight[j] += 2.0;            // planted: weight 2 per observation
#else
                sums->weight[j] += 1.0;
#endif
                sums->r[j] += (double)sr;
                sums->g[j] += (double)sg;
                sums->b[j] += (double)sb;
            });
            if (valid) v->valid_points++;
        }
    }
    return 0;
}

/* Occlusion test of later integrations: 0 = the ray pixel's depth (default),
 * 1 = reprojection of the voxel centre.  Returns -1 for any other mode. */
int oracle_set_occlusion(void* h, int mode)
{
    if (mode != 0 && mode != 1) return -1;
    static_cast<Volume*>(h)->reproject = mode == 1;
    return 0;
}

long long oracle_block_count(void* h) { return (long long)static_cast<Volume*>(h)->blocks.size(); }

/* Counters, in this order: valid_points, passing_samples, accumulated,
 * missed_contributions, out_of_range_samples, dropped_blocks,
 * bad_local_index. */
void oracle_counters(void* h, unsigned long long out[7])
{
    Volume* v = static_cast<Volume*>(h);
    out[0] = v->valid_points;
    out[1] = v->passing_samples;
    out[2] = v->accumulated;
    out[3] = v->missed_contributions;
    out[4] = v->out_of_range_samples;
    out[5] = v->dropped_blocks;
    out[6] = v->bad_local_index;
}

/* Every allocated block coordinate, sorted by (x, y, z).  Returns the count
 * written (at most max_n). */
long long oracle_export_coords(void* h, long long max_n, int32_t* coords)
{
    Volume* v = static_cast<Volume*>(h);
    std::vector<BlockCoord> all;
    all.reserve(v->blocks.size());
    for (const auto& kv : v->blocks) all.push_back(kv.first);
    std::sort(all.begin(), all.end());
    long long n = std::min<long long>(max_n, (long long)all.size());
    for (long long i = 0; i < n; ++i) {
        coords[3 * i] = all[i].x;
        coords[3 * i + 1] = all[i].y;
        coords[3 * i + 2] = all[i].z;
    }
    return n;
}

/* Blocks whose sums are kept, sorted by (x, y, z), with their six per-voxel
 * arrays ([n][512] each; any pointer may be null to skip that array). */
long long oracle_export_sums(void* h, long long max_n, int32_t* coords, double* tsdf,
                             double* weight, double* r, double* g, double* b,
                             double* tsdf_abs)
{
    Volume* v = static_cast<Volume*>(h);
    std::vector<std::pair<BlockCoord, const BlockSums*>> kept;
    for (const auto& kv : v->blocks)
        if (kv.second) kept.emplace_back(kv.first, kv.second.get());
    std::sort(kept.begin(), kept.end(),
              [](const std::pair<BlockCoord, const BlockSums*>& a,
                 const std::pair<BlockCoord, const BlockSums*>& c) { return a.first < c.first; });
    long long n = std::min<long long>(max_n, (long long)kept.size());
    const size_t bytes = sizeof(double) * kBlockVoxels;
    for (long long i = 0; i < n; ++i) {
        const BlockSums* s = kept[i].second;
        coords[3 * i] = kept[i].first.x;
        coords[3 * i + 1] = kept[i].first.y;
        coords[3 * i + 2] = kept[i].first.z;
        if (tsdf) std::memcpy(tsdf + i * kBlockVoxels, s->tsdf, bytes);
        if (weight) std::memcpy(weight + i * kBlockVoxels, s->weight, bytes);
        if (r) std::memcpy(r + i * kBlockVoxels, s->r, bytes);
        if (g) std::memcpy(g + i * kBlockVoxels, s->g, bytes);
        if (b) std::memcpy(b + i * kBlockVoxels, s->b, bytes);
        if (tsdf_abs) std::memcpy(tsdf_abs + i * kBlockVoxels, s->tsdf_abs, bytes);
    }
    return n;
}

long long oracle_kept_count(void* h)
{
    Volume* v = static_cast<Volume*>(h);
    long long n = 0;
    for (const auto& kv : v->blocks)
        if (kv.second) ++n;
    return n;
}

/* ------------------------------------------------------------------------
 * Packed key, slot hash and a sequential linear-probing table: a reference
 * for the hash table's structure ("What Irregularity Costs", design section,
 * data structure: 64-bit key with each block axis biased by 2^20 into 21
 * bits; open addressing, linear probing; multiply-xor hash).
 * --------------------------------------------------------------------- */

/* Key layout (a reading; the page's formula did not survive): x in bits
 * 0-20, y in bits 21-41, z in bits 42-62, each stored as coordinate + 2^20.
 * Bit 63 is always zero, so the all-ones word can mark an empty slot.
 * Returns 0 and writes *key for an in-range coordinate, -1 otherwise. */
int oracle_pack_key(int32_t x, int32_t y, int32_t z, uint64_t* key)
{
    const int64_t bias = (int64_t)1 << 20;
    int64_t c[3] = {x, y, z};
    uint64_t out = 0;
    for (int a = 0; a < 3; ++a) {
        int64_t biased = c[a] + bias;
        if (biased < 0 || biased >= ((int64_t)1 << 21)) return -1;
        out += (uint64_t)biased * ((uint64_t)1 << (21 * a));
    }
    *key = out;
    return 0;
}

/* Inverse of oracle_pack_key; -1 if bit 63 is set. */
int oracle_unpack_key(uint64_t key, int32_t out[3])
{
    if (key >> 63) return -1;
    const int64_t bias = (int64_t)1 << 20;
    for (int a = 0; a < 3; ++a) {
        uint64_t field = (key / ((uint64_t)1 << (21 * a))) % ((uint64_t)1 << 21);
        out[a] = (int32_t)((int64_t)field - bias);
    }
    return 0;
}

/* Home slot of a key in a table of T = 2^m slots (a reading; the page names
 * a multiply-xor hash but not its constants): the 64-bit finalizer of
 * SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014) -- xor-shift, multiply, xor-shift, multiply,
 * xor-shift -- then the low m bits.  Every step is a bijection on 64-bit
 * words, and every output bit depends on every key bit, so neighbouring
 * block coordinates spread over the whole table. */
uint64_t oracle_hash_slot(uint64_t key, uint64_t table_size)
{
    uint64_t z = key;
    z = z ^ (z >> 30);
    z = z * 0xBF58476D1CE4E5B9ull;        // modulo 2^64
    z = z ^ (z >> 27);
#if ORACLE_MUTANT == 24
    z = z * 0xBF58476D1CE4E5B9ull;        // planted: the first multiplier used twice
#else
    z = z * 0x94D049BB133111EBull;
#endif
#if ORACLE_MUTANT == 23
    z = z ^ (z >> 32);                    // planted: last shift 32 instead of 31
#else
    z = z ^ (z >> 31);
#endif
    return z % table_size;                // table_size is a power of two
}

/* Insert keys[0..n) one after another into an empty table of T slots with
 * linear probing.  A key already present is found, not inserted again.
 * table_out[T]: the key in each slot, or all-ones for an empty slot.
 * probe_len[i]: slots examined by the i-th insert (1 = its home slot).
 * *total_displacement: sum over distinct keys of (final slot - home) mod T.
 * Returns the number of distinct keys, or -1 if the table filled up. */
long long oracle_probe_build(const uint64_t* keys, long long n, uint64_t table_size,
                             uint64_t* table_out, long long* probe_len,
                             long long* total_displacement)
{
    const uint64_t empty = ~(uint64_t)0;
    for (uint64_t s = 0; s < table_size; ++s) table_out[s] = empty;
    long long distinct = 0;
    long long disp = 0;
    for (long long i = 0; i < n; ++i) {
        uint64_t home = oracle_hash_slot(keys[i], table_size);
        uint64_t slot = home;
        long long examined = 1;
        while (table_out[slot] != empty && table_out[slot] != keys[i]) {
            slot = (slot + 1) % table_size;
            ++examined;
            if ((uint64_t)examined > table_size) return -1;
        }
        if (table_out[slot] == empty) {
            table_out[slot] = keys[i];
            ++distinct;
            disp += (long long)((slot + table_size - home) % table_size);
        }
        if (probe_len) probe_len[i] = examined;
    }
    if (total_displacement) *total_displacement = disp;
    return distinct;
}

/* Block coordinates whose home slot lies in [window_start, window_start +
 * window_len) of a T-slot table: scans the cube origin + [0, side)^3 in
 * x-fastest raster order and keeps the first `want` hits (coords_out: want
 * x 3).  Returns the number found. */
long long oracle_clustered_coords(uint64_t table_size, uint64_t window_start,
                                  uint64_t window_len, const int32_t origin[3], int32_t side,
                                  long long want, int32_t* coords_out)
{
    long long found = 0;
    for (int32_t z = 0; z < side && found < want; ++z)
        for (int32_t y = 0; y < side && found < want; ++y)
            for (int32_t x = 0; x < side && found < want; ++x) {
                uint64_t key;
                int32_t c[3] = {origin[0] + x, origin[1] + y, origin[2] + z};
                if (oracle_pack_key(c[0], c[1], c[2], &key) != 0) continue;
                uint64_t slot = oracle_hash_slot(key, table_size);
                uint64_t rel = (slot + table_size - window_start) % table_size;
                if (rel < window_len) {
                    coords_out[3 * found] = c[0];
                    coords_out[3 * found + 1] = c[1];
                    coords_out[3 * found + 2] = c[2];
                    ++found;
                }
            }
    return found;
}

/* ------------------------------------------------------------------------
 * Extraction (read-out): the zero level set of the mean TSDF
 *
 * The page recovers means only at extraction (design section,
 * accumulation: sums, divided by the weight when read) and extracts the
 * surface by marching tetrahedra (design section; its details are not on the
 * page).  Readings:
 *   - lattice points are voxel centres, world position ((float)i + 0.5) * voxel
 *     per axis; the value there is the mean RN(float(tsdf sum) / float(weight)),
 *     and a voxel is observed iff its weight is > 0;
 *   - cell (i, j, k) spans the 8 voxels (i..i+1, j..j+1, k..k+1); corner c has
 *     offset (c & 1, c >> 1 & 1, c >> 2 & 1); a cell is used only when all 8
 *     corners are observed;
 *   - the cube is cut into the 6 tetrahedra that share its diagonal 0-7, one
 *     per order of the axes (x,y,z), (x,z,y), (y,x,z), (y,z,x), (z,x,y),
 *     (z,y,x): {0, 1, 3, 7}, {0, 1, 5, 7}, {0, 2, 3, 7}, {0, 2, 6, 7},
 *     {0, 4, 5, 7}, {0, 4, 6, 7} (neighbouring cells then cut their shared
 *     faces along the same diagonals, so the surface has no cracks);
 *   - a corner is inside when its value is < 0;
 *   - a surface vertex sits on every tetrahedron edge whose ends differ, at
 *     the zero of the linear interpolation, t = fA / (fA - fB) from the lower
 *     end A (all coordinates <= B's) towards B: p = pA + t * (pB - pA), in
 *     float32, one rounding per operation;
 *   - one inside (or one outside) corner o with the others a, b, c in the
 *     tetrahedron's order: triangle (E(o,a), E(o,b), E(o,c)); two inside
 *     corners i1, i2 and two outside o1, o2: triangles (E(i1,o1), E(i1,o2),
 *     E(i2,o2)) and (E(i1,o1), E(i2,o2), E(i2,o1)).
 * Triangles are written cell by cell, blocks in (x, y, z) order, voxels in
 * storage order, tetrahedra in the order above.
 * --------------------------------------------------------------------- */

}  // extern "C"

namespace {

#if ORACLE_MUTANT == 16
const int kTets[6][4] = {{0, 1, 2, 7}, {0, 1, 5, 7}, {0, 2, 3, 7},   // planted: not a tiling
                         {0, 2, 6, 7}, {0, 4, 5, 7}, {0, 4, 6, 7}};
#else
const int kTets[6][4] = {{0, 1, 3, 7}, {0, 1, 5, 7}, {0, 2, 3, 7},
                         {0, 2, 6, 7}, {0, 4, 5, 7}, {0, 4, 6, 7}};
#endif

/* Offset of cell corner c along axis ax (0 = x). */
int corner_offset(int c, int ax) { return (c >> ax) & 1; }

/* The offset used to fetch a corner's value (the same one). */
int value_offset(int c, int ax)
{
#if ORACLE_MUTANT == 18
    return (c >> (ax == 0 ? 1 : ax == 1 ? 0 : 2)) & 1;     // planted: x and y swapped
#else
    return corner_offset(c, ax);
#endif
}

/* Mean TSDF of voxel (ix, iy, iz); false when the voxel is not observed. */
bool mean_tsdf(const Volume* v, int32_t ix, int32_t iy, int32_t iz, float* f)
{
    const BlockCoord b{floor_div8(ix), floor_div8(iy), floor_div8(iz)};
    auto it = v->blocks.find(b);
    if (it == v->blocks.end() || !it->second) return false;
    const int j = (ix - b.x * kEdge) + kEdge * (iy - b.y * kEdge) +
                  kEdge * kEdge * (iz - b.z * kEdge);
    const double w = it->second->weight[j];
    if (!(w > 0.0)) return false;
    const float sum = (float)it->second->tsdf[j];
    const float wf = (float)w;
#if ORACLE_MUTANT == 17
    *f = sum;                                               // planted: not divided
    (void)wf;
#else
    *f = sum / wf;
#endif
    return true;
}

float centre(int32_t i, float voxel) { return ((float)i + 0.5f) * voxel; }

struct Cell {
    int32_t i[3];      // corner 0
    float f[8];        // corner values
};

/* Surface vertex on the edge between corners a < b of the cell. */
void edge_vertex(const Cell& c, int a, int b, float voxel, float out[3])
{
    const float fa = c.f[a], fb = c.f[b];
#if ORACLE_MUTANT == 15
    const float t = fb / (fb - fa);                         // planted: from the wrong end
#else
    const float t = fa / (fa - fb);
#endif
    for (int ax = 0; ax < 3; ++ax) {
        const float pa = centre(c.i[ax] + corner_offset(a, ax), voxel);
        const float pb = centre(c.i[ax] + corner_offset(b, ax), voxel);
        out[ax] = pa + t * (pb - pa);
    }
}

void put_triangle(const Cell& c, const int e[3][2], float voxel, std::vector<float>* out)
{
    for (int k = 0; k < 3; ++k) {
        const int a = std::min(e[k][0], e[k][1]), b = std::max(e[k][0], e[k][1]);
        float p[3];
        edge_vertex(c, a, b, voxel, p);
        out->insert(out->end(), p, p + 3);
    }
}

void march_tetrahedron(const Cell& c, const int* t, float voxel, std::vector<float>* out)
{
    int in[4], out_[4], n_in = 0, n_out = 0;
    for (int k = 0; k < 4; ++k) {
        if (c.f[t[k]] < 0.0f)
            in[n_in++] = t[k];
        else
            out_[n_out++] = t[k];
    }
    if (n_in == 1 || n_in == 3) {
        const int o = n_in == 1 ? in[0] : out_[0];
        const int* rest = n_in == 1 ? out_ : in;
        const int e[3][2] = {{o, rest[0]}, {o, rest[1]}, {o, rest[2]}};
        put_triangle(c, e, voxel, out);
    } else if (n_in == 2) {
        const int e1[3][2] = {{in[0], out_[0]}, {in[0], out_[1]}, {in[1], out_[1]}};
        const int e2[3][2] = {{in[0], out_[0]}, {in[1], out_[1]}, {in[1], out_[0]}};
        put_triangle(c, e1, voxel, out);
        put_triangle(c, e2, voxel, out);
    }
}

}  // namespace

extern "C" {

/* Triangles of the zero level set, 9 floats each (three vertices x, y, z);
 * writes at most max_tris and returns the total number. */
long long oracle_extract(void* h, long long max_tris, float* out)
{
    const Volume* v = static_cast<const Volume*>(h);
    std::vector<BlockCoord> order;
    for (const auto& kv : v->blocks)
        if (kv.second) order.push_back(kv.first);
    std::sort(order.begin(), order.end());
    std::vector<float> tris;
    for (const BlockCoord& b : order) {
        for (int j = 0; j < kBlockVoxels; ++j) {
            Cell c;
            c.i[0] = b.x * kEdge + j % kEdge;
            c.i[1] = b.y * kEdge + (j / kEdge) % kEdge;
            c.i[2] = b.z * kEdge + j / (kEdge * kEdge);
            bool all = true;
            for (int k = 0; k < 8 && all; ++k)
                all = mean_tsdf(v, c.i[0] + value_offset(k, 0), c.i[1] + value_offset(k, 1),
                                c.i[2] + value_offset(k, 2), &c.f[k]);
            if (!all) continue;
            for (int t = 0; t < 6; ++t) march_tetrahedron(c, kTets[t], v->voxel, &tris);
        }
    }
    const long long n = (long long)(tris.size() / 9);
    const long long w = std::min(n, max_tris);
    if (out && w > 0) std::memcpy(out, tris.data(), sizeof(float) * 9 * (size_t)w);
    return n;
}

/* Set (create or overwrite) a block's five sums directly, for building
 * volumes from a known field in the pins; tsdf_abs becomes |tsdf|. */
int oracle_set_block(void* h, const int32_t coord[3], const double* tsdf, const double* weight,
                     const double* r, const double* g, const double* b)
{
    Volume* v = static_cast<Volume*>(h);
    const BlockCoord c{coord[0], coord[1], coord[2]};
    std::unique_ptr<BlockSums>& s = v->blocks[c];
    if (!s) s.reset(new BlockSums());
    for (int j = 0; j < kBlockVoxels; ++j) {
        s->tsdf[j] = tsdf[j];
        s->weight[j] = weight[j];
        s->r[j] = r ? r[j] : 0.0;
        s->g[j] = g ? g[j] : 0.0;
        s->b[j] = b ? b[j] : 0.0;
        s->tsdf_abs[j] = std::fabs(tsdf[j]);
    }
    return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }

}  // extern "C"
