// Device building blocks of the integrate path: back-projection, the
// truncation-band walk with its occlusion test, the packed block key, the
// slot hash, and the table probe / insert / lookup.
//
// Arithmetic of the walk ("What Irregularity Costs", design section,
// integration; correctness section, analytic tier for the voxel-centre
// distance): every float operation is spelled with a round-to-nearest
// intrinsic, so no multiply-add is ever fused and divisions and square
// roots are IEEE-exact.  The voxel a sample selects is therefore the one any
// IEEE float32 evaluation of the same operations in the same order selects.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tsdf_internal.h"

namespace tsdf {

enum SampleStatus { kSamplePass = 0, kSampleOccluded = 1, kSampleOutOfRange = 2 };

// What the band walk of a valid pixel needs: its depth d, the back-projected
// point p = d (xn, yn, 1) moved to the world and divided by the voxel edge,
// p' = (R p + t) / voxel, and the unit ray direction in world coordinates,
// e = R dir.  Band step j lies at p' + j e in voxel units.
struct RayPoint {
    float d;
    float vx, vy, vz;       // p'
    float ex, ey, ez;       // e
};

struct VoxelSample {
    int ix, iy, iz;     // voxel index
    float tsdf;         // min(1, sdf / trunc)
};

// Division by a divisor y that is fixed for the whole volume (the
// truncation distance or the voxel edge), given r = RN(1 / y): Markstein's
// reciprocal-and-correction scheme (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990): q0 = RN(x r) is within an ulp of x / y, the residual x - q0 y is
// exact in one fused multiply-add, and one more fused multiply-add rounds
// q0 + r (x - q0 y) to the correctly rounded quotient.  At volume creation the
// host has the GPU check, for every one of the 2^32 float32 bit patterns x,
// that min(1, x / trunc) comes out the same as with IEEE division for every
// x >= -trunc (the only dividends the walk divides by trunc), and that
// x / voxel comes out bit for bit the same for every x (div_voxel).  Only
// where its check passed is the scheme used.
__device__ __forceinline__ float div_fixed(float x, float y, float r)
{
    const float q0 = __fmul_rn(x, r);
    const float e = __fmaf_rn(-q0, y, x);
    return __fmaf_rn(e, r, q0);
}

// x / trunc as the walk uses it (checked exhaustively for x >= -trunc).  The
// residual of the correction step is only exact while it stays a normal
// number, i.e. for |x| well above the subnormal range; smaller dividends
// (which real depths never produce) take the IEEE division.
template <bool kFast>
__device__ __forceinline__ float div_trunc(float x, float y, float r)
{
    if (kFast && fabsf(x) >= 0x1p-96f) return div_fixed(x, y, r);
    return __fdiv_rn(x, y);
}

// Division of a world coordinate by the voxel edge in the back-projection:
// the reciprocal-and-correction quotient where `fast` (the volume checked
// it, at create, against IEEE division for every float32 dividend) and
// the magnitude lies in [2^-96, 2^100), where the residual stays a normal
// number and x r cannot overflow; IEEE division otherwise.
__device__ __forceinline__ float div_voxel(const DivisorPair& dv, bool fast, float x)
{
    const float a = fabsf(x);
    if (fast && a >= 0x1p-96f && a < 0x1p100f) return div_fixed(x, dv.voxel, dv.inv_voxel);
    return __fdiv_rn(x, dv.voxel);
}

// The viewing ray of pixel (u, v): xn = (u - cx) / fx, yn = (v - cy) / fy,
// and the unit direction (xn, yn, 1) / sqrt(xn^2 + yn^2 + 1), returned as
// (dx, dy, dz, xn).  It depends only on the pixel and the intrinsics, so a
// batch computes it once per pixel into a table (build_rays) that every
// frame's back-projection reads: the two divisions of the normalised
// coordinates, the square root and the three divisions of the direction are
// the expensive part of back-projecting a pixel, and the table holds their
// IEEE results unchanged.
__device__ __forceinline__ float4 pixel_ray(float fx, float fy, float cx, float cy, int u, int v,
                                            float& yn)
{
    const float xn = __fdiv_rn(__fsub_rn((float)u, cx), fx);
    yn = __fdiv_rn(__fsub_rn((float)v, cy), fy);
    const float len = __fsqrt_rn(__fadd_rn(__fadd_rn(__fmul_rn(xn, xn), __fmul_rn(yn, yn)), 1.0f));
    return make_float4(__fdiv_rn(xn, len), __fdiv_rn(yn, len), __fdiv_rn(1.0f, len), xn);
}

// Back-project a pixel of depth d whose ray (pixel_ray) is `ray`, with yn
// its row's normalised coordinate: p = d (xn, yn, 1) moved to the world and
// divided by the voxel edge, and the world direction of the ray.
__device__ __forceinline__ bool back_project(const Camera& c, const DivisorPair& dv,
                                             bool fast_voxel, const float4& ray, float yn,
                                             float d, RayPoint& p)
{
    if (!(isfinite(d) && d > 0.0f)) return false;
    const float px = __fmul_rn(ray.w, d);
    const float py = __fmul_rn(yn, d);
    const float pz = d;
    const float dx = ray.x, dy = ray.y, dz = ray.z;
    // rows of R summed left to right, then t; one division per axis
    p.d = d;
    p.vx = div_voxel(dv, fast_voxel,
                     __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(c.r00, px), __fmul_rn(c.r01, py)),
                                         __fmul_rn(c.r02, pz)), c.tx));
    p.vy = div_voxel(dv, fast_voxel,
                     __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(c.r10, px), __fmul_rn(c.r11, py)),
                                         __fmul_rn(c.r12, pz)), c.ty));
    p.vz = div_voxel(dv, fast_voxel,
                     __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(c.r20, px), __fmul_rn(c.r21, py)),
                                         __fmul_rn(c.r22, pz)), c.tz));
    p.ex = __fadd_rn(__fadd_rn(__fmul_rn(c.r00, dx), __fmul_rn(c.r01, dy)), __fmul_rn(c.r02, dz));
    p.ey = __fadd_rn(__fadd_rn(__fmul_rn(c.r10, dx), __fmul_rn(c.r11, dy)), __fmul_rn(c.r12, dz));
    p.ez = __fadd_rn(__fadd_rn(__fmul_rn(c.r20, dx), __fmul_rn(c.r21, dy)), __fmul_rn(c.r22, dz));
    // If any of p' and e is not finite (absurd depths or poses), every band
    // sample has a non-finite coordinate on some axis (a non-finite p'
    // component stays non-finite after adding a step; a non-finite e
    // component gives 0 * inf = NaN at the middle step and +-inf or NaN at
    // the others), so every sample is out of range.  The ray is replaced by
    // one whose samples all lie at +inf in x, which band_voxel's integer
    // range check rejects like the non-finite originals.
    if (!(isfinite(p.vx) && isfinite(p.vy) && isfinite(p.vz) && isfinite(p.ex) &&
          isfinite(p.ey) && isfinite(p.ez))) {
        p.vx = INFINITY;
        p.vy = p.vz = p.ex = p.ey = p.ez = 0.0f;
    }
    return true;
}

// Back-project pixel index pix = v * width + u of a batch's frame, its depth
// d, reading the pixel's ray from the batch's table.
__device__ __forceinline__ bool back_project_pixel(const VolumeView& vol, const FrameBatch& fb,
                                                   const Camera& cam, int v, size_t pix, float d,
                                                   RayPoint& p)
{
    const float4 ray = __ldg(fb.rays + pix);
    const float yn = __ldg(fb.ray_yn + v);
    return back_project(cam, vol.div, vol.fast_voxel, ray, yn, d, p);
}

// A pixel holds an observation when its depth is finite and positive.
__device__ __forceinline__ bool valid_depth(float d) { return isfinite(d) && d > 0.0f; }

// Frame f and tile (tx, ty) of block b of a tiled grid ordered tile-major,
// frame-minor (b = tile * n + f, tile = ty * tiles_x + tx), by_tiles_x the
// frame's width in tiles.
struct TilePos {
    int f, tx, ty;
};

__device__ __forceinline__ TilePos tile_of_block(const FrameBatch& fb,
                                                 const IndexDivisor& by_tiles_x, uint32_t b)
{
    const uint32_t tile = divide_index(fb.by_n, b);
    const uint32_t ty = divide_index(by_tiles_x, tile);
    return {(int)(b - tile * (uint32_t)fb.n), (int)(tile - ty * by_tiles_x.d), (int)ty};
}

// Voxel indices in [-2^23, 2^23 - 1] <=> block indices in [-2^20, 2^20 - 1].
constexpr unsigned kVoxelIndexBias = 1u << 23;
constexpr unsigned kVoxelIndexSpan = 1u << 24;

// Camera-frame depth of the centre of voxel (ix, iy, iz):
// z_c = (R^T (centre - t))_z = r02 * cx + r12 * cy + r22 * cz, with the
// centre taken relative to the camera position.
__device__ __forceinline__ float centre_depth(const Camera& c, float voxel, int ix, int iy, int iz)
{
    const float cxr = __fsub_rn(__fmul_rn(__fadd_rn((float)ix, 0.5f), voxel), c.tx);
    const float cyr = __fsub_rn(__fmul_rn(__fadd_rn((float)iy, 0.5f), voxel), c.ty);
    const float czr = __fsub_rn(__fmul_rn(__fadd_rn((float)iz, 0.5f), voxel), c.tz);
    return __fadd_rn(__fadd_rn(__fmul_rn(c.r02, cxr), __fmul_rn(c.r12, cyr)),
                     __fmul_rn(c.r22, czr));
}

// The truncated signed distance min(1, sdf / trunc) of a sample whose pixel
// depth is d and whose voxel centre lies at camera depth zc.
template <bool kFast>
__device__ __forceinline__ float truncated_sdf(const DivisorPair& dv, float d, float zc)
{
    return fminf(1.0f, div_trunc<kFast>(__fsub_rn(d, zc), dv.trunc, dv.inv_trunc));
}

// The voxel of band sample `i` (offset i voxels along the unit ray, i in
// -k..k): the floor of p' + i e, and whether it lies in the packable range.
// The floor and the conversion to an integer are one round-toward-minus-
// infinity conversion, which saturates values beyond the int32 range, so the
// range test is an integer comparison; back_project guarantees finite p' and
// e (or a ray whose every sample is rejected), so no coordinate is NaN.
template <bool kFast>
__device__ __forceinline__ bool band_voxel_f(const RayPoint& p, float fi, VoxelSample& s)
{
    s.ix = __float2int_rd(__fadd_rn(p.vx, __fmul_rn(fi, p.ex)));
    s.iy = __float2int_rd(__fadd_rn(p.vy, __fmul_rn(fi, p.ey)));
    s.iz = __float2int_rd(__fadd_rn(p.vz, __fmul_rn(fi, p.ez)));
    return ((unsigned)s.ix + kVoxelIndexBias < kVoxelIndexSpan) &
           ((unsigned)s.iy + kVoxelIndexBias < kVoxelIndexSpan) &
           ((unsigned)s.iz + kVoxelIndexBias < kVoxelIndexSpan);
}

// The voxel of band step fi without the range check, for rays whose whole
// band ray_in_range has proven to lie in the packable range.
__device__ __forceinline__ void band_voxel_unchecked(const RayPoint& p, float fi, VoxelSample& s)
{
    s.ix = __float2int_rd(__fadd_rn(p.vx, __fmul_rn(fi, p.ex)));
    s.iy = __float2int_rd(__fadd_rn(p.vy, __fmul_rn(fi, p.ey)));
    s.iz = __float2int_rd(__fadd_rn(p.vz, __fmul_rn(fi, p.ez)));
}

// Whether every band step -half .. half of the ray lies in the packable
// voxel range: per axis |p'| + half |e| stays 4 below 2^23 - 1, which covers
// the floor and the rounding of p' + i e (at most one unit at these
// magnitudes).  Non-finite rays fail it.
__device__ __forceinline__ bool ray_in_range(const RayPoint& p, float fhalf)
{
    const float lim = 8388603.0f;
    return fabsf(p.vx) + fhalf * fabsf(p.ex) <= lim && fabsf(p.vy) + fhalf * fabsf(p.ey) <= lim &&
           fabsf(p.vz) + fhalf * fabsf(p.ez) <= lim;
}

// The same with the step as an int (i converts exactly: |i| <= 127).
template <bool kFast>
__device__ __forceinline__ bool band_voxel(const Camera& c, const DivisorPair& dv,
                                           const RayPoint& p, int i, VoxelSample& s)
{
    return band_voxel_f<kFast>(p, (float)i, s);
}

// Which band steps of a ray provably pass the ray-depth occlusion test,
// before it is evaluated (the allocate kernel skips it there).  In exact
// arithmetic, with R a rotation, sample i of the ray lies at camera depth
// d + i voxel dz (dz <= 1 the ray's z direction), and the centre of its voxel
// lies within half a voxel diagonal, (sqrt(3) / 2) voxel, of it; so the
// centre's depth is at most d + (max(i, 0) + sqrt(3) / 2) voxel and at least
// d - (k + sqrt(3) / 2) voxel.  The test (centre depth > 0 and
// d - centre depth >= -trunc) therefore passes when
//     max(i, 0) + sqrt(3) / 2 + e <= trunc / voxel   and
//     d / voxel > k + sqrt(3) / 2 + e,
// where e bounds, in voxels, every rounding of the float32 walk and test:
// each of the ~20 operations from the pose to the centre's depth errs by at
// most 2^-24 of its operands, whose magnitudes are at most
// m = |p'|_1 + 2k + 2 (the ray in voxel units) plus the camera position
// |t|_1 / voxel, so e = (64 * 2^-24 + 4 * defect) (m + |t|_1 / voxel), with
// defect = max |R^T R - I| covering a pose that is not exactly a rotation
// (above 1e-3 no band step is proven).  Returns the largest provably passing
// max(i, 0) (in voxels; -inf when none) and whether the near side holds.
struct SurePass {
    float i_max;
    bool near;
};

__device__ __forceinline__ SurePass sure_pass(const Camera& c, const DivisorPair& dv,
                                              const RayPoint& p, int half)
{
    const float m = fabsf(p.vx) + fabsf(p.vy) + fabsf(p.vz) + (float)(2 * half + 2);
    const float e = c.sure_err * (m + c.sure_tmag);
    SurePass r;
    r.i_max = c.sure_tau - e;
    // d / voxel through the reciprocal (relative error 2^-23 at most), with
    // margin for it
    r.near = __fmul_rn(p.d, dv.inv_voxel) * 0.999999f > (float)half + c.sure_near + e;
    return r;
}

// The occlusion test of the sample in voxel s against its own ray's depth:
// the centre lies in front of the camera and not more than one truncation
// distance behind the observed surface.  zc is the centre's camera depth.
__device__ __forceinline__ bool ray_visible(const Camera& c, const DivisorPair& dv,
                                            const RayPoint& p, const VoxelSample& s, float& zc)
{
    zc = centre_depth(c, dv.voxel, s.ix, s.iy, s.iz);
    return zc > 0.0f && __fsub_rn(p.d, zc) >= -dv.trunc;
}

// Band sample `i`: its voxel and truncated signed distance at the voxel
// centre, or the reason it is skipped.  The update kernels use it; the
// allocate kernel, which only needs the voxel and the test, calls
// band_voxel and ray_visible itself.  Written without early exits: every
// quantity is computed and the status is selected at the end.
template <bool kFast, bool kCheckRange = true>
__device__ __forceinline__ int band_sample(const Camera& c, const DivisorPair& dv,
                                           const RayPoint& p, float fi, VoxelSample& s)
{
    bool in_range = true;
    if (kCheckRange) in_range = band_voxel_f<kFast>(p, fi, s);
    else band_voxel_unchecked(p, fi, s);
    float zc;
    const bool visible = ray_visible(c, dv, p, s, zc);
    s.tsdf = truncated_sdf<kFast>(dv, p.d, zc);
    return !in_range ? kSampleOutOfRange : (visible ? kSamplePass : kSampleOccluded);
}

// The same with the step as an int (converted exactly: |i| <= 127).
template <bool kFast>
__device__ __forceinline__ int band_sample(const Camera& c, const DivisorPair& dv,
                                           const RayPoint& p, int i, VoxelSample& s)
{
    return band_sample<kFast>(c, dv, p, (float)i, s);
}

// The occlusion test by reprojection (selected per volume; the alternative
// reading of the design section's occlusion test).  The centre of voxel s,
// in camera coordinates c = R^T (centre - t), is projected through the
// pinhole, u = fx (c_x / c_z) + cx, v = fy (c_y / c_z) + cy, and rounded to
// the nearest pixel centre, floor(u + 1/2), floor(v + 1/2).  The sample
// passes when the centre is in front of the camera, that pixel lies inside
// the image and holds a valid depth d', and d' - c_z >= -trunc; then (with
// kWantTsdf) s.tsdf = min(1, (d' - c_z) / trunc), and `pix` is the pixel
// whose colour the sample adds.
template <bool kFast, bool kWantTsdf>
__device__ __forceinline__ bool reprojected_visible(const Camera& c, const DivisorPair& dv,
                                                    const float* __restrict__ depth, int width,
                                                    int height, VoxelSample& s, size_t& pix)
{
    const float voxel = dv.voxel;
    const float cxr = __fsub_rn(__fmul_rn(__fadd_rn((float)s.ix, 0.5f), voxel), c.tx);
    const float cyr = __fsub_rn(__fmul_rn(__fadd_rn((float)s.iy, 0.5f), voxel), c.ty);
    const float czr = __fsub_rn(__fmul_rn(__fadd_rn((float)s.iz, 0.5f), voxel), c.tz);
    // component k of R^T (centre - t) is column k of R dotted with the centre
    const float x = __fadd_rn(__fadd_rn(__fmul_rn(c.r00, cxr), __fmul_rn(c.r10, cyr)),
                              __fmul_rn(c.r20, czr));
    const float y = __fadd_rn(__fadd_rn(__fmul_rn(c.r01, cxr), __fmul_rn(c.r11, cyr)),
                              __fmul_rn(c.r21, czr));
    const float z = __fadd_rn(__fadd_rn(__fmul_rn(c.r02, cxr), __fmul_rn(c.r12, cyr)),
                              __fmul_rn(c.r22, czr));
    if (!(z > 0.0f)) return false;
    const float uh = __fadd_rn(__fadd_rn(__fmul_rn(c.fx, __fdiv_rn(x, z)), c.cx), 0.5f);
    const float vh = __fadd_rn(__fadd_rn(__fmul_rn(c.fy, __fdiv_rn(y, z)), c.cy), 0.5f);
    // (NaN fails every comparison)
    if (!(uh >= 0.0f && uh < (float)width && vh >= 0.0f && vh < (float)height)) return false;
    pix = (size_t)floorf(vh) * (size_t)width + (size_t)floorf(uh);
    const float d = __ldg(depth + pix);
    if (!valid_depth(d)) return false;
    if (!(__fsub_rn(d, z) >= -dv.trunc)) return false;
    if (kWantTsdf) s.tsdf = truncated_sdf<kFast>(dv, d, z);
    return true;
}

// Band sample `i` under the reprojection test: its voxel (the walk is the
// ray test's) and, when it passes, its value and the pixel of its colour.
template <bool kFast>
__device__ __forceinline__ int band_sample_reprojected(const Camera& c, const DivisorPair& dv,
                                                       const RayPoint& p, int i,
                                                       const float* __restrict__ depth,
                                                       int width, int height, VoxelSample& s,
                                                       size_t& pix)
{
    if (!band_voxel<kFast>(c, dv, p, i, s)) return kSampleOutOfRange;
    return reprojected_visible<kFast, true>(c, dv, depth, width, height, s, pix)
               ? kSamplePass : kSampleOccluded;
}

// Packed key: block coordinate (voxel index >> 3, an arithmetic shift, i.e.
// floor division) biased by 2^20 into 21 bits per axis; x in bits 0-20,
// y in 21-41, z in 42-62.  Bit 63 stays clear, so no key equals kEmptyKey.
__device__ __forceinline__ unsigned long long block_key(int ix, int iy, int iz)
{
    const unsigned long long bx = (unsigned long long)((ix >> 3) + (1 << 20));
    const unsigned long long by = (unsigned long long)((iy >> 3) + (1 << 20));
    const unsigned long long bz = (unsigned long long)((iz >> 3) + (1 << 20));
    return bx | (by << 21) | (bz << 42);
}

__device__ __forceinline__ unsigned long long pack_block(int bx, int by, int bz)
{
    return (unsigned long long)(bx + (1 << 20)) |
           ((unsigned long long)(by + (1 << 20)) << 21) |
           ((unsigned long long)(bz + (1 << 20)) << 42);
}

__device__ __forceinline__ void unpack_block(unsigned long long key, int32_t* out)
{
    out[0] = (int32_t)(key & 0x1FFFFFull) - (1 << 20);
    out[1] = (int32_t)((key >> 21) & 0x1FFFFFull) - (1 << 20);
    out[2] = (int32_t)((key >> 42) & 0x1FFFFFull) - (1 << 20);
}

// Where the pool stores voxel (lx, ly, lz) of a block (0..511).  The planar
// layout keeps the x-fastest order.  The interleaved layout stores the block
// as 64 bricks of 2 x 2 x 2 voxels, bricks x-fastest, voxels in a brick
// x-fastest: a brick's eight 16-byte records are one 128-byte line and its
// eight blue sums one 32-byte sector.  The samples a warp adds at one band
// step lie on a sheet across the surface; whatever its orientation, a brick
// holds several of them, where an x-row of 8 voxels holds one when the sheet
// runs across x.  (Measured by simulation on the room walk: 12 % fewer L2
// requests than x-rows.)
__device__ __forceinline__ uint32_t brick_slot(int lx, int ly, int lz)
{
    return (uint32_t)((((lx >> 1) | ((ly >> 1) << 2) | ((lz >> 1) << 4)) << 3) |
                      (lx & 1) | ((ly & 1) << 1) | ((lz & 1) << 2));
}

__device__ __forceinline__ uint32_t voxel_slot(const VolumeView& vol, int lx, int ly, int lz)
{
    return vol.planar ? (uint32_t)(lx | (ly << 3) | (lz << 6)) : brick_slot(lx, ly, lz);
}

// The pool position of x-fastest voxel offset j.
__device__ __forceinline__ uint32_t voxel_slot_of(const VolumeView& vol, int j)
{
    return voxel_slot(vol, j & 7, (j >> 3) & 7, j >> 6);
}

// Slot hash: the SplitMix64 output mix (xor-shift / multiply, twice, then a
// final xor-shift; Steele, Lea and Flood, OOPSLA 2014), masked to the table.
__device__ __forceinline__ uint32_t home_slot(unsigned long long key, uint32_t mask)
{
    unsigned long long z = key;
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return (uint32_t)z & mask;
}

enum ProbeResult { kProbeFound = 0, kProbeWon = 1, kProbeOverflow = 2 };

// Find or claim `key` by linear probing from its home slot.  Slots are read
// with plain (L1-cacheable) loads: a stale EMPTY only costs a failed
// compare-and-swap that returns the slot's real key, after which the probe
// carries on; keys are never removed while a kernel runs, so a stale
// non-empty key is never wrong.  The probe is unbounded up to the table size.
__device__ __forceinline__ int probe_insert(Entry* table, uint32_t mask, unsigned long long key,
                                            uint32_t* slot_out, uint32_t* steps_out)
{
    uint32_t slot = home_slot(key, mask);
    uint32_t steps = 1;
    int res;
    for (;;) {
        const unsigned long long k = table[slot].key;
        if (k == key) {
            res = kProbeFound;
            break;
        }
        if (k == kEmptyKey) {
            const unsigned long long old = atomicCAS(&table[slot].key, kEmptyKey, key);
            if (old == kEmptyKey) {
                res = kProbeWon;
                break;
            }
            if (old == key) {
                res = kProbeFound;
                break;
            }
        }
        if (steps > mask) {           // examined all table_capacity slots
            res = kProbeOverflow;
            break;
        }
        slot = (slot + 1) & mask;
        ++steps;
    }
    *slot_out = slot;
    *steps_out = steps;
    return res;
}

// Pool index of `key`, or kIndexFailed when the key is absent.  The table is
// read-only during the update kernel, so whole entries are read through the
// non-coherent path in one 16-byte load.
__device__ __forceinline__ uint32_t lookup(const Entry* __restrict__ table, uint32_t mask,
                                           unsigned long long key)
{
    uint32_t slot = home_slot(key, mask);
    for (uint32_t n = 0; n <= mask; ++n) {
        const uint4 e = __ldg(reinterpret_cast<const uint4*>(table) + slot);
        const unsigned long long k = (unsigned long long)e.x | ((unsigned long long)e.y << 32);
        if (k == key) return e.z;
        if (k == kEmptyKey) return kIndexFailed;
        slot = (slot + 1) & mask;
    }
    return kIndexFailed;
}

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

// Field k (0 tsdf, 1 weight, 2 red, 3 green) of the planar layout.
__device__ __forceinline__ float* planar_field(const VolumeView& vol, int k)
{
    return reinterpret_cast<float*>(vol.voxel4) + (size_t)k * vol.plane;
}

// The tsdf and weight sums of voxel e (the first half of its record).
__device__ __forceinline__ float2 tsdf_and_weight(const VolumeView& vol, size_t e)
{
    if (vol.planar) return make_float2(__ldg(planar_field(vol, 0) + e), __ldg(planar_field(vol, 1) + e));
    return __ldg(reinterpret_cast<const float2*>(vol.voxel4 + e));
}

__device__ __forceinline__ void red_add_f32(float* addr, float v)
{
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// Add one observation's terms to voxel e of the pool.  Interleaved layout:
// (tsdf, weight, red, green) with one 4-wide float reduction into the
// voxel's 16-byte record, blue with one scalar reduction; L2 executes a
// reduction request at about the same rate whether it carries one float or
// four, so this takes two requests where the planar layout takes five.
__device__ __forceinline__ void add_to_voxel(const VolumeView& vol, size_t e, float tsdf,
                                             float weight, float r, float g, float b)
{
    if (vol.planar) {
        red_add_f32(planar_field(vol, 0) + e, tsdf);
        red_add_f32(planar_field(vol, 1) + e, weight);
        red_add_f32(planar_field(vol, 2) + e, r);
        red_add_f32(planar_field(vol, 3) + e, g);
    } else {
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(vol.voxel4 + e),
                     "f"(tsdf), "f"(weight), "f"(r), "f"(g)
                     : "memory");
    }
    red_add_f32(vol.blue + e, b);
}

// Add one band step's samples of a warp (lane: add, voxel e, its terms).
// Lanes whose samples fall in the same voxel are summed on the lowest of
// them first (the rays of a tile's neighbouring pixels often meet in a
// voxel), and that lane adds the group's sums with one pair of reductions;
// the leader adds its members' terms in lane order.  The members' terms
// reach the leader either by shuffles, four per member and round, the rounds
// running to the largest group of the warp (kStaged false), or through
// `stage`, the warp's 32 float4 slots in shared memory: one 16-byte store per
// lane and one 16-byte load per member (kStaged true).  Measured on GB300:
// shuffles are faster in the per-sample update kernel on sparse scenes,
// the slots in the fused kernel, whose registers are scarcer.  Must be
// called by all 32 lanes.
template <bool kStaged>
__device__ __forceinline__ void warp_add_samples(const VolumeView& vol, float4* stage, bool add,
                                                 uint32_t e, float tsdf, float r, float g,
                                                 float b)
{
    const unsigned act = __ballot_sync(0xFFFFFFFFu, add);
    if (act == 0) return;
    const int lane = (int)(threadIdx.x & 31u);
    unsigned grp = 0;
    if (add) grp = __match_any_sync(act, e);
    const bool leader = add && __ffs(grp) - 1 == lane;
    unsigned rest = leader ? grp & (grp - 1u) : 0u;       // the group's other lanes
    float st = tsdf, sr = r, sg = g, sb = b;
    if (kStaged) {
        if (__any_sync(0xFFFFFFFFu, rest != 0u)) {
            stage[lane] = make_float4(tsdf, r, g, b);
            __syncwarp();
            for (; rest != 0u; rest &= rest - 1u) {
                const float4 m = stage[__ffs(rest) - 1];
                st = __fadd_rn(st, m.x);
                sr = __fadd_rn(sr, m.y);
                sg = __fadd_rn(sg, m.z);
                sb = __fadd_rn(sb, m.w);
            }
            __syncwarp();                   // the slots are rewritten at the next step
        }
    } else {
        const int rounds = (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)__popc(rest));
        for (int k = 0; k < rounds; ++k) {
            const int src = rest ? __ffs(rest) - 1 : lane;
            rest &= rest - 1u;
            const float a_t = __shfl_sync(0xFFFFFFFFu, tsdf, src);
            const float a_r = __shfl_sync(0xFFFFFFFFu, r, src);
            const float a_g = __shfl_sync(0xFFFFFFFFu, g, src);
            const float a_b = __shfl_sync(0xFFFFFFFFu, b, src);
            if (src != lane) {
                st = __fadd_rn(st, a_t);
                sr = __fadd_rn(sr, a_r);
                sg = __fadd_rn(sg, a_g);
                sb = __fadd_rn(sb, a_b);
            }
        }
    }
    if (leader) add_to_voxel(vol, e, st, (float)__popc(grp), sr, sg, sb);
}


// Where to pre-reduce in shared memory (adaptive mode).  A 16 x 16 pixel
// tile is dense when at least half of its valid pixels (finite depth > 0) see
// a voxel edge at least w pixels wide (voxel * fx >= w * depth): there
// samples crowd into few voxels.  The widths are where the shared-memory
// pre-reduction overtook five direct reductions per sample on GB300: near 5
// pixels for launches of several frames (the frames' samples of a voxel meet
// in L2 as well) and near 10 for a single frame; against the warp-merged
// per-sample kernel it no longer wins anywhere measured, which is why the
// mode is not the default.  The per-sample kernel applies this rule to its
// 16 x 16 tiles and lists the dense ones for the pre-reducing kernel, so
// every tile is integrated exactly once.  Launches below kAdaptiveMinPixels
// pixels add every sample directly (there launch latency dominates).
constexpr uint32_t kAdaptiveMinPixels = 1u << 18;

__device__ __forceinline__ float dense_width(int n_frames) { return n_frames >= 4 ? 5.0f : 10.0f; }

__device__ __forceinline__ bool dense_pixel(float d, float voxel, float fx, int n_frames)
{
    return valid_depth(d) && __fmul_rn(voxel, fx) >= __fmul_rn(dense_width(n_frames), d);
}

__device__ __forceinline__ bool dense_tile(uint32_t n_valid, uint32_t n_dense)
{
    return n_valid != 0 && 2 * n_dense >= n_valid;
}


}  // namespace tsdf
