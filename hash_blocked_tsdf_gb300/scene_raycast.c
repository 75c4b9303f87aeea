/*
 * Analytic ray caster for the synthetic depth frames (input synthesis only).
 *
 * Casts one ray per pixel through a pinhole camera (pixel centres at integer
 * (u, v), camera looking down +z, x right, y down) against spheres,
 * axis-aligned boxes, an optional world plane z = plane_z and the optional
 * six inner walls of the cube [-room_half, room_half]^3.  It writes the
 * camera-frame z of the nearest hit in front of the camera, or 0 when the ray
 * hits nothing.  Everything is double precision; the caller rounds to float32.
 *
 * This file holds no part of the TSDF integrate path: no band walk, no voxel
 * or block indexing, no hashing.  Frames are independent, so they are split
 * across OpenMP threads; each frame's result does not depend on the split.
 */
#include <math.h>
#include <stddef.h>

#define KIND_SPHERE 0
#define KIND_BOX 1

static double hit_sphere(const double o[3], const double d[3], const double c[3], double r)
{
    double oc[3] = {o[0] - c[0], o[1] - c[1], o[2] - c[2]};
    double a = d[0] * d[0] + d[1] * d[1] + d[2] * d[2];
    double b = 2.0 * (d[0] * oc[0] + d[1] * oc[1] + d[2] * oc[2]);
    double cc = oc[0] * oc[0] + oc[1] * oc[1] + oc[2] * oc[2] - r * r;
    double disc = b * b - 4.0 * a * cc;
    if (disc < 0.0) return INFINITY;
    double sq = sqrt(disc);
    double t0 = (-b - sq) / (2.0 * a);
    double t1 = (-b + sq) / (2.0 * a);
    if (t0 > 0.0) return t0;
    if (t1 > 0.0) return t1;
    return INFINITY;
}

static double hit_box(const double o[3], const double d[3], const double lo[3], const double hi[3])
{
    double tn = -INFINITY, tf = INFINITY;
    for (int a = 0; a < 3; ++a) {
        if (d[a] == 0.0) {
            if (o[a] < lo[a] || o[a] > hi[a]) return INFINITY;
            continue;
        }
        double ta = (lo[a] - o[a]) / d[a];
        double tb = (hi[a] - o[a]) / d[a];
        double t_lo = ta < tb ? ta : tb;
        double t_hi = ta < tb ? tb : ta;
        if (t_lo > tn) tn = t_lo;
        if (t_hi < tf) tf = t_hi;
    }
    if (!(tn <= tf) || !(tf > 0.0)) return INFINITY;
    return tn > 0.0 ? tn : tf;
}

/* Pixel rectangle [u0,u1) x [v0,v1) that holds the projection of the box
 * with the given camera-frame corners.  Returns 0 if off-screen, 1 for a
 * rectangle, 2 when the box reaches the camera plane (use the whole image). */
static int project_rect(const double corners_cam[8][3], const double K[4], int W, int H,
                        int* u0, int* u1, int* v0, int* v1)
{
    double zmin = INFINITY, zmax = -INFINITY;
    for (int i = 0; i < 8; ++i) {
        if (corners_cam[i][2] < zmin) zmin = corners_cam[i][2];
        if (corners_cam[i][2] > zmax) zmax = corners_cam[i][2];
    }
    if (zmax <= 1e-3) return 0;
    if (zmin <= 1e-2) {
        *u0 = 0; *u1 = W; *v0 = 0; *v1 = H;
        return 2;
    }
    double umin = INFINITY, umax = -INFINITY, vmin = INFINITY, vmax = -INFINITY;
    for (int i = 0; i < 8; ++i) {
        double u = K[0] * corners_cam[i][0] / corners_cam[i][2] + K[2];
        double v = K[1] * corners_cam[i][1] / corners_cam[i][2] + K[3];
        if (u < umin) umin = u;
        if (u > umax) umax = u;
        if (v < vmin) vmin = v;
        if (v > vmax) vmax = v;
    }
    int a0 = (int)floor(umin) - 1, a1 = (int)ceil(umax) + 2;
    int b0 = (int)floor(vmin) - 1, b1 = (int)ceil(vmax) + 2;
    if (a0 < 0) a0 = 0;
    if (b0 < 0) b0 = 0;
    if (a1 > W) a1 = W;
    if (b1 > H) b1 = H;
    if (a0 >= a1 || b0 >= b1) return 0;
    *u0 = a0; *u1 = a1; *v0 = b0; *v1 = b1;
    return 1;
}

static void raycast_frame(int W, int H, const double K[4], const double pose[16],
                          int n_prims, const int* kinds, const double* centres,
                          const double* sizes, int has_plane, double plane_z,
                          int has_room, double room_half, double* out)
{
    const double R[9] = {pose[0], pose[1], pose[2], pose[4], pose[5], pose[6],
                         pose[8], pose[9], pose[10]};
    const double o[3] = {pose[3], pose[7], pose[11]};
    for (int v = 0; v < H; ++v) {
        for (int u = 0; u < W; ++u) {
            double xc = ((double)u - K[2]) / K[0];
            double yc = ((double)v - K[3]) / K[1];
            double d[3] = {R[0] * xc + R[1] * yc + R[2], R[3] * xc + R[4] * yc + R[5],
                           R[6] * xc + R[7] * yc + R[8]};
            double best = INFINITY;
            if (has_plane && d[2] != 0.0) {
                double t = (plane_z - o[2]) / d[2];
                if (t > 0.0 && t < best) best = t;
            }
            if (has_room) {
                for (int a = 0; a < 3; ++a) {
                    if (d[a] == 0.0) continue;
                    double wall = d[a] > 0.0 ? room_half : -room_half;
                    double t = (wall - o[a]) / d[a];
                    if (t > 0.0 && t < best) best = t;
                }
            }
            out[(size_t)v * W + u] = best;
        }
    }
    for (int p = 0; p < n_prims; ++p) {
        const double* c = centres + 3 * p;
        const double* s = sizes + 3 * p;
        double corners[8][3];
        int k = 0;
        for (int sx = 0; sx < 2; ++sx)
            for (int sy = 0; sy < 2; ++sy)
                for (int sz = 0; sz < 2; ++sz, ++k) {
                    double w[3] = {c[0] + (sx ? 0.5 : -0.5) * s[0] - o[0],
                                   c[1] + (sy ? 0.5 : -0.5) * s[1] - o[1],
                                   c[2] + (sz ? 0.5 : -0.5) * s[2] - o[2]};
                    /* camera = R^T (world - o) */
                    corners[k][0] = R[0] * w[0] + R[3] * w[1] + R[6] * w[2];
                    corners[k][1] = R[1] * w[0] + R[4] * w[1] + R[7] * w[2];
                    corners[k][2] = R[2] * w[0] + R[5] * w[1] + R[8] * w[2];
                }
        int u0, u1, v0, v1;
        if (!project_rect(corners, K, W, H, &u0, &u1, &v0, &v1)) continue;
        double lo[3] = {c[0] - 0.5 * s[0], c[1] - 0.5 * s[1], c[2] - 0.5 * s[2]};
        double hi[3] = {c[0] + 0.5 * s[0], c[1] + 0.5 * s[1], c[2] + 0.5 * s[2]};
        for (int v = v0; v < v1; ++v) {
            for (int u = u0; u < u1; ++u) {
                double xc = ((double)u - K[2]) / K[0];
                double yc = ((double)v - K[3]) / K[1];
                double d[3] = {R[0] * xc + R[1] * yc + R[2], R[3] * xc + R[4] * yc + R[5],
                               R[6] * xc + R[7] * yc + R[8]};
                double t = kinds[p] == KIND_SPHERE ? hit_sphere(o, d, c, 0.5 * s[0])
                                                   : hit_box(o, d, lo, hi);
                double* px = out + (size_t)v * W + u;
                if (t < *px) *px = t;
            }
        }
    }
    for (size_t i = 0; i < (size_t)W * H; ++i)
        if (!isfinite(out[i])) out[i] = 0.0;
}

/* Render n_frames depth images (camera-frame z, 0 = no hit) into out
 * (double [n_frames][H][W]).  poses: n_frames row-major 4x4 camera-to-world.
 * kinds/centres/sizes: n_prims primitives (size = box edges, or the sphere
 * diameter in size[0]). */
void scene_raycast_frames(int n_frames, int W, int H, const double K[4], const double* poses,
                          int n_prims, const int* kinds, const double* centres,
                          const double* sizes, int has_plane, double plane_z, int has_room,
                          double room_half, double* out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int f = 0; f < n_frames; ++f)
        raycast_frame(W, H, K, poses + 16 * (size_t)f, n_prims, kinds, centres, sizes,
                      has_plane, plane_z, has_room, room_half, out + (size_t)f * W * H);
}
