// Throughput probes for the ceilings that bound the integrate kernels and
// that no library figure gives: the rate at which L2 executes global float
// reductions (red.global.add) for scalar and 4-wide vector operands, with
// coalesced or scattered addresses, and 64-bit compare-and-swaps on
// scattered 16-byte entries (the hash table's insert operation), over an
// L2-resident or an HBM-resident footprint.  Built into libtsdf_peaks.so,
// used only by the benchmark.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t mix32(uint32_t x)
{
    // integer finaliser (xor-shift-multiply), to scatter addresses
    x ^= x >> 16;
    x *= 0x7FEB352Du;
    x ^= x >> 15;
    x *= 0x846CA68Bu;
    x ^= x >> 16;
    return x;
}

__device__ __forceinline__ void red_f32(float* p, float v)
{
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ void red_v4_f32(float* p, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

// mode 0: scalar, a warp covers 32 consecutive floats (4 sectors)
// mode 1: scalar, every lane in its own random 32-byte sector
// mode 2: float4, a warp covers 512 consecutive bytes (16 sectors)
// mode 3: float4, every lane in its own random 32-byte sector
// mode 4: scalar, 8 lanes share a random sector (4 sectors per warp, scattered)
// mode 5: 64-bit compare-and-swap on the first word of a random 16-byte entry
//         (0 -> a nonzero value: the first one succeeds, later ones fail;
//         both kinds are counted, as in a table insert)
__global__ void __launch_bounds__(kThreads) red_kernel(float* buf, uint64_t n_floats, int mode,
                                                       int reps)
{
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint64_t nthreads = (uint64_t)gridDim.x * kThreads;
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t n_sectors = n_floats / 8;
    unsigned long long seen = 0;
    for (int r = 0; r < reps; ++r) {
        const uint64_t g = tid + (uint64_t)r * nthreads;
        switch (mode) {
        case 0:
            red_f32(buf + (g % n_floats), 1.0f);
            break;
        case 1: {
            const uint64_t s = mix32((uint32_t)g) % n_sectors;
            red_f32(buf + s * 8 + (lane & 7u), 1.0f);
            break;
        }
        case 2:
            red_v4_f32(buf + (4 * g) % n_floats, 1.0f, 1.0f, 1.0f, 1.0f);
            break;
        case 3: {
            const uint64_t s = mix32((uint32_t)g) % n_sectors;
            red_v4_f32(buf + s * 8 + 4 * (lane & 1u), 1.0f, 1.0f, 1.0f, 1.0f);
            break;
        }
        case 4: {
            const uint64_t s = mix32((uint32_t)(g >> 3)) % n_sectors;
            red_f32(buf + s * 8 + (lane & 7u), 1.0f);
            break;
        }
        default: {
            const uint64_t e = mix32((uint32_t)g) % (n_floats / 4);
            seen ^= atomicCAS(reinterpret_cast<unsigned long long*>(buf + 4 * e), 0ull, g + 1);
            break;
        }
        }
    }
    if (seen == 0x5A5A5A5A5A5A5A5Aull) buf[0] = 1.0f;   // keeps the returned words live
}

}  // namespace

extern "C" {

// Launch `blocks` x 256 threads, each issuing `reps` operations of the given
// mode into buf (n_floats floats, a multiple of 8, 16-byte aligned).  Returns
// a cudaError_t as int.
int peak_red(float* buf, uint64_t n_floats, int mode, int reps, int blocks, void* stream)
{
    if (!buf || n_floats < 8 || (n_floats & 7) || reps < 1 || blocks < 1 || mode < 0 || mode > 5)
        return (int)cudaErrorInvalidValue;
    red_kernel<<<blocks, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(buf, n_floats,
                                                                                 mode, reps);
    return (int)cudaGetLastError();
}

}  // extern "C"
