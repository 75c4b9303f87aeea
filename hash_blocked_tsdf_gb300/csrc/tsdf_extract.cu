// Read-out kernels: surface extraction and block import.
//
// Extraction ("What Irregularity Costs", design section: the arrays hold
// sums and the mean is recovered at extraction; the surface is extracted by
// marching tetrahedra, once, in CUDA).  The page gives no further detail;
// the readings, written out here and in the header:
//   - lattice points are voxel centres, world position ((float)i + 0.5) *
//     voxel per axis; the value there is the mean RN(tsdf sum / weight), and
//     a voxel is observed iff its weight is > 0;
//   - cell (i, j, k) spans voxels (i..i+1, j..j+1, k..k+1), corner c at offset
//     (c & 1, c >> 1 & 1, c >> 2 & 1); only cells with 8 observed corners;
//   - the cube is cut into the 6 tetrahedra around its diagonal 0-7, one per
//     order of the axes: {0,1,3,7} {0,1,5,7} {0,2,3,7} {0,2,6,7} {0,4,5,7}
//     {0,4,6,7}, so neighbouring cells cut shared faces alike;
//   - inside means value < 0; a vertex sits on each tetrahedron edge whose
//     ends differ, at t = fA / (fA - fB) from the lower end A towards B,
//     p = pA + t (pB - pA), float32, one rounding per operation;
//   - one odd corner o, others a, b, c in tetrahedron order: triangle
//     (E(o,a), E(o,b), E(o,c)); two inside i1, i2 and two outside o1, o2:
//     (E(i1,o1), E(i1,o2), E(i2,o2)) and (E(i1,o1), E(i2,o2), E(i2,o1)).
//
// One block of 256 threads per allocated block.  A first pass looks up every
// block's seven upper neighbours (+x, +y, +z and their combinations) in the
// table, all in parallel; the block's 512 means and the 217 lattice points its cells take from those
// neighbours go to shared memory (9 x 9 x 9, NaN where unobserved); each
// thread classifies two cells by the sign mask of their corners (one lookup
// in a table built at compile time gives the crossed tetrahedra); the
// tetrahedra the surface crosses become one task list for the block, those
// with two triangles first (scans of both counts; one atomic takes the
// block's range of the output), and all 256 threads emit the list's
// triangles.
#include "tsdf_device.cuh"

namespace tsdf {
namespace {

constexpr int kThreads = 256;

// Corner k (0..3) of tetrahedron `tet`: the path 0, e_p, e_p + e_q, 7 through
// the cube, with p = tet / 2 the first axis and q the lower (tet even) or
// higher (tet odd) of the other two -- the sets {0,1,3,7} {0,1,5,7}
// {0,2,3,7} {0,2,6,7} {0,4,5,7} {0,4,6,7}, corners in ascending order.
__device__ __forceinline__ int tet_corner(int tet, int k)
{
    const int p = tet >> 1;
    const int lo = p == 0 ? 1 : 0, hi = p == 2 ? 1 : 2;
    const int q = (tet & 1) ? hi : lo;
    const int c1 = 1 << p, c2 = c1 | (1 << q);
    return k == 0 ? 0 : k == 1 ? c1 : k == 2 ? c2 : 7;
}

__device__ __forceinline__ float lattice(int i, float voxel)
{
    return __fmul_rn(__fadd_rn((float)i, 0.5f), voxel);
}

// Element k (0..3, known only at run time) of four values held in registers.
template <typename T>
__device__ __forceinline__ T pick(T a, T b, T c, T d, int k)
{
    return k == 0 ? a : k == 1 ? b : k == 2 ? c : d;
}

// The tetrahedron's four corners: ids (0..7) and values, in its own order.
struct Tet {
    int id[4];
    float v[4];
};

// Vertex on the edge between tetrahedron corners p and q (0..3): from the
// lower-numbered cell corner A towards B.
__device__ __forceinline__ void edge_vertex(const Tet& T, const int cell[3], int p, int q,
                                            float voxel, float* out)
{
    int a = pick(T.id[0], T.id[1], T.id[2], T.id[3], p);
    int b = pick(T.id[0], T.id[1], T.id[2], T.id[3], q);
    float fa = pick(T.v[0], T.v[1], T.v[2], T.v[3], p);
    float fb = pick(T.v[0], T.v[1], T.v[2], T.v[3], q);
    if (a > b) {
        const int ti = a; a = b; b = ti;
        const float tf = fa; fa = fb; fb = tf;
    }
    const float t = __fdiv_rn(fa, __fsub_rn(fa, fb));
#pragma unroll
    for (int ax = 0; ax < 3; ++ax) {
        const float pa = lattice(cell[ax] + ((a >> ax) & 1), voxel);
        const float pb = lattice(cell[ax] + ((b >> ax) & 1), voxel);
        out[ax] = __fadd_rn(pa, __fmul_rn(t, __fsub_rn(pb, pa)));
    }
}

__device__ __forceinline__ void write_triangle(const Tet& T, const int cell[3], int p0, int q0,
                                               int p1, int q1, int p2, int q2, float voxel,
                                               float* tri)
{
    edge_vertex(T, cell, p0, q0, voxel, tri);
    edge_vertex(T, cell, p1, q1, voxel, tri + 3);
    edge_vertex(T, cell, p2, q2, voxel, tri + 6);
}

// Bit mask of the tetrahedron's inside corners (bit k = its corner k).
__device__ __forceinline__ int inside_mask(const Tet& T)
{
    return (T.v[0] < 0.0f ? 1 : 0) | (T.v[1] < 0.0f ? 2 : 0) | (T.v[2] < 0.0f ? 4 : 0) |
           (T.v[3] < 0.0f ? 8 : 0);
}

// Triangle `which` of the tetrahedron (which = 1 only when two of its
// corners are inside and it holds two): its three edges are chosen by case,
// then one write_triangle computes them, so that lanes in different cases
// share the vertex arithmetic.
__device__ __forceinline__ void tet_triangle(const Tet& T, const int cell[3], float voxel,
                                             int which, float* tri)
{
    const int in = inside_mask(T);
    const int ot = ~in & 0xF;
    const int n_in = __popc(in);
    int p0, q0, p1, q1, p2, q2;
    if (n_in == 2) {
        const int i0 = __ffs(in) - 1;
        const int i1 = __ffs(in & (in - 1)) - 1;
        const int o0 = __ffs(ot) - 1;
        const int o1 = __ffs(ot & (ot - 1)) - 1;
        p0 = i0; q0 = o0;
        p1 = which ? i1 : i0; q1 = o1;
        p2 = i1; q2 = which ? o0 : o1;
    } else {
        // the odd corner, then the other three in tetrahedron order
        const int odd_set = n_in == 1 ? in : ot;
        int rest = n_in == 1 ? ot : in;
        const int o = __ffs(odd_set) - 1;
        p0 = p1 = p2 = o;
        q0 = __ffs(rest) - 1;
        rest &= rest - 1;
        q1 = __ffs(rest) - 1;
        rest &= rest - 1;
        q2 = __ffs(rest) - 1;
    }
    write_triangle(T, cell, p0, q0, p1, q1, p2, q2, voxel, tri);
}

// A warp's staged triangles (n of them, 9 floats each) to output triangles
// [at, at + n), in contiguous stores; those at or past `capacity` are
// dropped.
__device__ __forceinline__ void flush_triangles(const float* stage, float* out, uint64_t at,
                                                uint32_t n, uint64_t capacity, unsigned lane)
{
    const uint32_t kept = at >= capacity ? 0u : (uint32_t)min((uint64_t)n, capacity - at);
    for (uint32_t i = lane; i < 9u * kept; i += 32u) out[9 * at + i] = stage[i];
}

// The block's lattice with its upper neighbours' first layer: 9 x 9 x 9
// points, x fastest (index lx + 9 ly + 81 lz); a point's value is the mean
// tsdf / weight, and NaN marks an unobserved point.
constexpr int kLat = 9;
constexpr int kLatPoints = kLat * kLat * kLat;          // 729
constexpr int kHaloPoints = kLatPoints - kBlockVoxels;  // 217

// For every inside mask m of a cell's eight corners (bit k = corner k), the
// cell's crossed tetrahedra: bits 0-5 mark the tetrahedra that have both
// inside and outside corners, bits 8-13 those among them with two corners
// inside (two triangles; one or three inside give one).  Built at compile
// time from tet_corner's sets, so a cell is classified with one lookup.
struct CellTable {
    uint32_t v[256];
};

constexpr uint32_t tet_mask_c(int tet)
{
    const int p = tet >> 1;
    const int lo = p == 0 ? 1 : 0, hi = p == 2 ? 1 : 2;
    const int q = (tet & 1) ? hi : lo;
    return 1u | (1u << (1 << p)) | (1u << ((1 << p) | (1 << q))) | (1u << 7);
}
// the sets {0,1,3,7} {0,1,5,7} {0,2,3,7} {0,2,6,7} {0,4,5,7} {0,4,6,7}
static_assert(tet_mask_c(0) == 0x8Bu && tet_mask_c(1) == 0xA3u && tet_mask_c(2) == 0x8Du &&
                  tet_mask_c(3) == 0xC5u && tet_mask_c(4) == 0xB1u && tet_mask_c(5) == 0xD1u,
              "tetrahedron corner sets");

constexpr int popcount_c(uint32_t x)
{
    int n = 0;
    for (; x; x &= x - 1) ++n;
    return n;
}

constexpr CellTable make_cell_table()
{
    CellTable t{};
    for (int m = 0; m < 256; ++m) {
        uint32_t e = 0;
        for (int tet = 0; tet < 6; ++tet) {
            const int k = popcount_c((uint32_t)m & tet_mask_c(tet));
            if (k != 0 && k != 4) e |= 1u << tet;
            if (k == 2) e |= 1u << (8 + tet);
        }
        t.v[m] = e;
    }
    return t;
}

__device__ const CellTable kCellTable = make_cell_table();

// Lattice index of corner k of the cell at (lx, ly, lz).
__device__ __forceinline__ int corner_point(int base, int k)
{
    return base + (k & 1) + ((k >> 1) & 1) * kLat + ((k >> 2) & 1) * kLat * kLat;
}

// nb[8 b + d] = pool index of block b's neighbour (bx + (d & 1), by + (d >> 1
// & 1), bz + (d >> 2 & 1)), kIndexFailed when absent (d = 0: b itself): all
// lookups of all blocks in parallel, so no extraction block waits on one.
__global__ void __launch_bounds__(kThreads) neighbour_kernel(VolumeView vol,
                                                            const int32_t* coords,
                                                            uint32_t n_blocks, uint32_t* nb)
{
    const uint32_t i = blockIdx.x * kThreads + threadIdx.x;
    if (i >= 8u * n_blocks) return;
    const uint32_t b = i >> 3;
    const int d = (int)(i & 7u);
    uint32_t idx = b;
    if (d != 0) {
        const int nx = coords[3 * b] + (d & 1), ny = coords[3 * b + 1] + ((d >> 1) & 1),
                  nz = coords[3 * b + 2] + ((d >> 2) & 1);
        const int hi = (1 << 20) - 1;
        idx = kIndexFailed;
        if (nx <= hi && ny <= hi && nz <= hi)
            idx = lookup(vol.table, vol.table_mask, pack_block(nx, ny, nz));
    }
    nb[i] = idx;
}

// Eight blocks per SM (registers capped at 32): the kernel waits on loads
// more than it computes, so resident blocks count (measured: 1.7 % faster
// than the six that 40 registers allow).
__global__ void __launch_bounds__(kThreads, 8) extract_kernel(VolumeView vol, const int32_t* coords,
                                                          const uint32_t* nb, float* out,
                                                          uint64_t capacity,
                                                          unsigned long long* count)
{
    __shared__ float s_lat[kLatPoints];
    // crossed tetrahedra of the block: cell (9 bits) | tetrahedron (3) << 9
    __shared__ uint32_t s_task[6 * kBlockVoxels];
    __shared__ uint32_t s_warp_tasks[kThreads / 32], s_warp_tris[kThreads / 32];
    __shared__ uint32_t s_total_tasks, s_total_twos;
    __shared__ float s_stage[kThreads / 32 * 32 * 9];    // each warp's 32 staged triangles
    __shared__ unsigned long long s_first;
    const uint32_t b = blockIdx.x;
    const int t = threadIdx.x;
    const int bc[3] = {coords[3 * b], coords[3 * b + 1], coords[3 * b + 2]};
    // the block's own 512 means (two per thread) and the upper neighbours'
    // first layers: +x face, +y face, +z face (64 points each), the three
    // edges (8 each) and the corner.  The neighbour's index is loaded first,
    // so that its dependent load overlaps the thread's own two.
    static_assert(kBlockVoxels == 2 * kThreads, "two voxels per thread");
    const bool halo = t < kHaloPoints;
    int d = 0, lx = 0, ly = 0, lz = 0;      // neighbour, and the lattice point (0..8)
    if (t < 64) {
        d = 1; lx = 8; ly = t & 7; lz = t >> 3;
    } else if (t < 128) {
        d = 2; lx = (t - 64) & 7; ly = 8; lz = (t - 64) >> 3;
    } else if (t < 192) {
        d = 4; lx = (t - 128) & 7; ly = (t - 128) >> 3; lz = 8;
    } else if (t < 200) {
        d = 3; lx = 8; ly = 8; lz = t - 192;
    } else if (t < 208) {
        d = 5; lx = 8; ly = t - 200; lz = 8;
    } else if (t < 216) {
        d = 6; lx = t - 208; ly = 8; lz = 8;
    } else {
        d = 7; lx = 8; ly = 8; lz = 8;
    }
    const uint32_t n_idx = halo ? __ldg(nb + 8 * (size_t)b + d) : kIndexFailed;
    const float2 own0 = tsdf_and_weight(vol, (size_t)b * kBlockVoxels + voxel_slot_of(vol, t));
    const float2 own1 =
        tsdf_and_weight(vol, (size_t)b * kBlockVoxels + voxel_slot_of(vol, t + kThreads));
    float2 tw_h = make_float2(0.0f, 0.0f);
    if (n_idx < vol.pool_capacity) {
        const int jj = (lx & 7) | ((ly & 7) << 3) | ((lz & 7) << 6);
        tw_h = tsdf_and_weight(vol, (size_t)n_idx * kBlockVoxels + voxel_slot_of(vol, jj));
    }
    const float nan = __int_as_float(0x7FFFFFFF);
    {
        const int j0 = t, j1 = t + kThreads;
        s_lat[(j0 & 7) + ((j0 >> 3) & 7) * kLat + (j0 >> 6) * kLat * kLat] =
            own0.y > 0.0f ? __fdiv_rn(own0.x, own0.y) : nan;
        s_lat[(j1 & 7) + ((j1 >> 3) & 7) * kLat + (j1 >> 6) * kLat * kLat] =
            own1.y > 0.0f ? __fdiv_rn(own1.x, own1.y) : nan;
    }
    if (halo) s_lat[lx + ly * kLat + lz * kLat * kLat] = tw_h.y > 0.0f ? __fdiv_rn(tw_h.x, tw_h.y) : nan;
    __syncthreads();

    // the two cells of this thread: the sign mask of their corners (a cell
    // counts when all 8 corners are observed), and from it the tetrahedra
    // the surface crosses (bits 0-5 for cell 0, 8-13 for cell 1) and those
    // of them holding two triangles
    uint32_t tets = 0, twos = 0;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int j = t + c * kThreads;
        const int base = (j & 7) + ((j >> 3) & 7) * kLat + (j >> 6) * kLat * kLat;
        uint32_t m = 0;
        bool seen = true;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float v = s_lat[corner_point(base, k)];
            seen = seen && !isnan(v);
            m |= (v < 0.0f ? 1u : 0u) << k;
        }
        if (seen) {
            const uint32_t e = __ldg(&kCellTable.v[m]);
            tets |= (e & 0x3Fu) << (8 * c);
            twos |= ((e >> 8) & 0x3Fu) << (8 * c);
        }
    }

    // the block's crossed tetrahedra become one task list: those with two
    // triangles first, then those with one, so that the warps emitting
    // them take the same path (block-wide scans of both counts)
    const unsigned lane = lane_id();
    const int warp = t >> 5;
    const uint32_t n2 = (uint32_t)__popc(twos), n1 = (uint32_t)__popc(tets) - n2;
    uint32_t incl2 = n2, incl1 = n1;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t a2 = __shfl_up_sync(0xFFFFFFFFu, incl2, d);
        const uint32_t a1 = __shfl_up_sync(0xFFFFFFFFu, incl1, d);
        if ((int)lane >= d) {
            incl2 += a2;
            incl1 += a1;
        }
    }
    if (lane == 31) {
        s_warp_tasks[warp] = incl2;
        s_warp_tris[warp] = incl1;
    }
    __syncthreads();
    if (t == 0) {
        uint32_t c2 = 0, c1 = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            const uint32_t a2 = s_warp_tasks[w], a1 = s_warp_tris[w];
            s_warp_tasks[w] = c2;
            s_warp_tris[w] = c1;
            c2 += a2;
            c1 += a1;
        }
        s_total_twos = c2;
        s_total_tasks = c2 + c1;
        const uint32_t tris = 2 * c2 + c1;
        s_first = tris ? atomicAdd(count, (unsigned long long)tris) : 0ull;
    }
    __syncthreads();
    const uint32_t total_twos = s_total_twos;
    uint32_t r2 = s_warp_tasks[warp] + incl2 - n2;          // this thread's first ranks
    uint32_t r1 = s_warp_tris[warp] + incl1 - n1;
    while (tets) {
        const int bit = __ffs(tets) - 1;
        tets &= tets - 1u;
        const uint32_t cell_tet = (uint32_t)(t + (bit >> 3) * kThreads) | ((uint32_t)(bit & 7) << 9);
        if ((twos >> bit) & 1u)
            s_task[r2++] = cell_tet;
        else
            s_task[total_twos + r1++] = cell_tet;
    }
    __syncthreads();

    // Emission, 32 tasks per warp round (task k0 + lane).  A round's
    // triangles fill one contiguous range of the block's output: the first
    // triangles of its two-triangle tasks, then their second triangles and
    // the one-triangle tasks' triangles.  Each half is staged in the warp's
    // shared slots and leaves in contiguous stores.
    const float voxel = vol.div.voxel;
    const unsigned long long first = s_first;
    const uint32_t total = s_total_tasks;
    float* stage = s_stage + warp * 32 * 9;
    for (uint32_t k0 = (uint32_t)warp * 32u; k0 < total; k0 += kThreads) {
        const uint32_t k = k0 + lane;
        const bool active = k < total;
        const uint32_t n_a = total_twos > k0 ? min(total_twos - k0, 32u) : 0u;
        const uint32_t n_act = min(total - k0, 32u);
        const uint64_t at = first + 2ull * min(k0, total_twos) + (k0 > total_twos ? k0 - total_twos : 0u);
        Tet T;
        int cell[3] = {0, 0, 0};
        if (active) {
            const uint32_t code = s_task[k];
            const int j = (int)(code & 511u);
            const int tet = (int)((code >> 9) & 7u);
            const int base = (j & 7) + ((j >> 3) & 7) * kLat + (j >> 6) * kLat * kLat;
            cell[0] = bc[0] * kBlockEdge + (j & 7);
            cell[1] = bc[1] * kBlockEdge + ((j >> 3) & 7);
            cell[2] = bc[2] * kBlockEdge + (j >> 6);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                T.id[q] = tet_corner(tet, q);
                T.v[q] = s_lat[corner_point(base, T.id[q])];
            }
        }
        if (n_a) {
            if (lane < n_a && at + lane < capacity) tet_triangle(T, cell, voxel, 0, stage + 9 * lane);
            __syncwarp();
            flush_triangles(stage, out, at, n_a, capacity, lane);
            __syncwarp();
        }
        if (active && at + n_a + lane < capacity)
            tet_triangle(T, cell, voxel, lane < n_a ? 1 : 0, stage + 9 * lane);
        __syncwarp();
        flush_triangles(stage, out, at + n_a, n_act, capacity, lane);
        __syncwarp();
    }
}

// Block b of the input: find its pool index (inserted just before) and copy
// its five sums there.
__global__ void __launch_bounds__(kThreads) import_kernel(VolumeView vol, const int32_t* coords,
                                                         const float* src)
{
    __shared__ uint32_t s_idx;
    const uint32_t b = blockIdx.x;
    const uint32_t n = gridDim.x;
    if (threadIdx.x == 0) {
        const int x = coords[3 * b], y = coords[3 * b + 1], z = coords[3 * b + 2];
        const int lo = -(1 << 20), hi = (1 << 20) - 1;
        uint32_t idx = kIndexFailed;
        if (x >= lo && x <= hi && y >= lo && y <= hi && z >= lo && z <= hi)
            idx = lookup(vol.table, vol.table_mask, pack_block(x, y, z));
        s_idx = idx;
    }
    __syncthreads();
    const uint32_t idx = s_idx;
    if (idx >= vol.pool_capacity) return;           // refused (pool full) or out of range
    for (int j = threadIdx.x; j < kBlockVoxels; j += kThreads) {
        const size_t e = (size_t)idx * kBlockVoxels + voxel_slot_of(vol, j);
        float v[5];
#pragma unroll
        for (int a = 0; a < 5; ++a) v[a] = src[((size_t)a * n + b) * kBlockVoxels + j];
        if (vol.planar) {
#pragma unroll
            for (int a = 0; a < 4; ++a) planar_field(vol, a)[e] = v[a];
        } else {
            vol.voxel4[e] = make_float4(v[0], v[1], v[2], v[3]);
        }
        vol.blue[e] = v[4];
    }
}

}  // namespace

cudaError_t launch_extract(const VolumeView& vol, const int32_t* coords, uint32_t n_blocks,
                           uint32_t* neighbours, float* out, uint64_t capacity,
                           unsigned long long* count, cudaStream_t stream)
{
    if (n_blocks == 0) return cudaSuccess;
    neighbour_kernel<<<(8 * n_blocks + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
        vol, coords, n_blocks, neighbours);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    extract_kernel<<<n_blocks, kThreads, 0, stream>>>(vol, coords, neighbours, out, capacity,
                                                      count);
    return cudaGetLastError();
}

cudaError_t launch_import(const VolumeView& vol, const int32_t* coords, uint32_t n,
                          const float* src, cudaStream_t stream)
{
    if (n == 0) return cudaSuccess;
    import_kernel<<<n, kThreads, 0, stream>>>(vol, coords, src);
    return cudaGetLastError();
}

}  // namespace tsdf
