// Throughput probes for the ceilings that bound the integrate kernels and
// that no library figure gives: the rate at which L2 executes global float
// reductions (red.global.add) for scalar and 4-wide vector operands, with
// coalesced or scattered addresses, and 64-bit compare-and-swaps on
// scattered 16-byte entries (the hash table's insert operation), over an
// L2-resident or an HBM-resident footprint; float and integer atomic adds to
// shared memory (what a block-wide accumulation in shared memory would pay);
// and scattered 32-byte records reduced either as a 4-wide plus a scalar
// reduction or as one 32-byte bulk reduction from shared memory.  Built
// into libtsdf_peaks.so, used only by the benchmark.
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

// Shared-memory atomic adds at random addresses of a 64 KB array: mode 0
// float, mode 1 32-bit integer.  out receives each thread's column sum (keeps
// the work live).
constexpr int kSmemWords = 16384;

__global__ void __launch_bounds__(kThreads) smem_atomic_kernel(float* out, int mode, int reps)
{
    extern __shared__ float words[];
    for (int i = threadIdx.x; i < kSmemWords; i += kThreads) words[i] = 0.0f;
    __syncthreads();
    uint32_t x = blockIdx.x * kThreads + threadIdx.x + 12345u;
    for (int r = 0; r < reps; ++r) {
        x = x * 1664525u + 1013904223u;              // a linear congruential step
        const uint32_t i = (x >> 8) & (uint32_t)(kSmemWords - 1);
        if (mode == 0) atomicAdd(&words[i], 1.0f);
        else atomicAdd(reinterpret_cast<uint32_t*>(words) + i, 1u);
    }
    __syncthreads();
    float acc = 0.0f;
    for (int i = threadIdx.x; i < kSmemWords; i += kThreads) acc += words[i];
    out[blockIdx.x * kThreads + threadIdx.x] = acc;
}

// Scattered 32-byte records (n_records of them, buf 32-byte aligned), all
// five sums of a voxel in one record: mode 0 adds them with a 4-wide and a
// scalar reduction (two requests to the same sector), mode 1 with one
// 32-byte bulk reduction from the thread's slot in shared memory (four slots
// per thread in flight).
constexpr int kBulkSlots = 4;

__global__ void __launch_bounds__(kThreads) record_red_kernel(float* buf, uint32_t n_records,
                                                              int mode, int reps)
{
    __shared__ __align__(128) float slots[kThreads][kBulkSlots][8];
    const uint32_t tid = blockIdx.x * kThreads + threadIdx.x;
    for (int r = 0; r < reps; ++r) {
        const uint32_t rec = mix32(tid * 7919u + (uint32_t)r) % n_records;
        float* dst = buf + (size_t)rec * 8;
        if (mode == 0) {
            red_v4_f32(dst, 1.0f, 1.0f, 1.0f, 1.0f);
            red_f32(dst + 4, 1.0f);
        } else {
            const int k = r % kBulkSlots;
            if (r >= kBulkSlots)
                asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kBulkSlots - 1) : "memory");
            float* src = slots[threadIdx.x][k];
#pragma unroll
            for (int q = 0; q < 8; ++q) src[q] = q < 5 ? 1.0f : 0.0f;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const uint32_t saddr = (uint32_t)__cvta_generic_to_shared(src);
            asm volatile(
                "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], 32;" ::"l"(
                    dst),
                "r"(saddr)
                : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
    }
    if (mode != 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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

// Launch `blocks` x 256 threads of shared-memory atomic adds (mode 0 float,
// 1 integer), `reps` each; out holds blocks x 256 floats.
int peak_smem_atomic(float* out, int mode, int reps, int blocks, void* stream)
{
    if (!out || reps < 1 || blocks < 1 || mode < 0 || mode > 1) return (int)cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(smem_atomic_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemWords * (int)sizeof(float));
    if (e != cudaSuccess) return (int)e;
    smem_atomic_kernel<<<blocks, kThreads, kSmemWords * sizeof(float),
                         reinterpret_cast<cudaStream_t>(stream)>>>(out, mode, reps);
    return (int)cudaGetLastError();
}

// Launch `blocks` x 256 threads reducing into random 32-byte records of buf
// (n_records records, buf 32-byte aligned), `reps` each, by mode (0: a 4-wide
// and a scalar reduction; 1: one 32-byte bulk reduction from shared memory).
int peak_record_red(float* buf, uint32_t n_records, int mode, int reps, int blocks, void* stream)
{
    if (!buf || n_records < 1 || ((uintptr_t)buf & 31) || reps < 1 || blocks < 1 || mode < 0 ||
        mode > 1)
        return (int)cudaErrorInvalidValue;
    record_red_kernel<<<blocks, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        buf, n_records, mode, reps);
    return (int)cudaGetLastError();
}

}  // extern "C"
