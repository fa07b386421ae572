// Bandwidth probes for bench.py --probe: the ceilings the Engram kernels are
// measured against on this GPU.  Not part of libengram.
//  - random_rows: one warp reads 2 random 256-byte rows per load instruction
//    (the gather's access pattern, 12 loads in flight per lane) from a buffer
//    of n_rows rows, optionally with one 4-byte scale per row from a second
//    array, and reduces them so the loads cannot be dropped.  The rows may sit
//    in device memory (read-only cache path) or in pinned host memory reached
//    over unified addressing (plain loads, as the staging kernel does).
#include <cuda_runtime.h>
#include <stdint.h>

__device__ __forceinline__ uint64_t mix64(uint64_t x) {  // SplitMix64 finaliser
    x ^= x >> 30; x *= 0xBF58476D1CE4E5B9ull;
    x ^= x >> 27; x *= 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

// The 4-byte scale read with different cache operators: 0 the read-only
// path (ld.global.nc), 1 L2 only (ld.global.cg), 2 read-only without L1
// allocation, 3 the coherent path without L1 allocation.  Which one fetches
// the fewest DRAM bytes per scattered 4-byte read decides the gather's.
template <int kFlavor>
__device__ __forceinline__ float load_scale(const float *p) {
    float v;
    if (kFlavor == 0)
        v = __ldg(p);
    else if (kFlavor == 1)
        asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    else if (kFlavor == 2)
        asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    else
        asm volatile("ld.global.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

template <bool kPlain, int kFlavor = 0>
__global__ void random_rows_kernel(const uint8_t *rows, const float *scales, int64_t n_rows, int64_t n_warps,
                                   uint64_t seed, float *sink) {
    const int lane = threadIdx.x & 31;
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (w >= n_warps) return;
    const int half = lane >> 4, c16 = lane & 15;
    uint4 v[12];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 12; ++i) {
        const uint64_t r = mix64(seed ^ (uint64_t)(w * 24 + 2 * i + half)) & (uint64_t)(n_rows - 1);  // n_rows: power of 2
        const uint4 *src = reinterpret_cast<const uint4 *>(rows + r * 256) + c16;
        v[i] = kPlain ? *src : __ldg(src);
        if (scales && c16 == 0) s += load_scale<kFlavor>(scales + r);
    }
    uint32_t x = 0;
#pragma unroll
    for (int i = 0; i < 12; ++i) x ^= v[i].x ^ v[i].y ^ v[i].z ^ v[i].w;
    if (x == 0x12345678u && s == 1.2345f) sink[0] = (float)x;  // keeps the loads alive
}

extern "C" int probe_random_rows(const uint8_t *rows, const float *scales, int64_t n_rows, int64_t n_warps,
                                 uint64_t seed, float *sink, void *stream) {
    const int64_t threads = n_warps * 32;
    random_rows_kernel<false><<<(unsigned)((threads + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
        rows, scales, n_rows, n_warps, seed, sink);
    return (int)cudaGetLastError();
}

// rows + scales with scale-load flavour 0..3 (see load_scale)
extern "C" int probe_random_rows_flavor(const uint8_t *rows, const float *scales, int64_t n_rows, int64_t n_warps,
                                        uint64_t seed, float *sink, int flavor, void *stream) {
    const unsigned grid = (unsigned)((n_warps * 32 + 255) / 256);
    cudaStream_t st = (cudaStream_t)stream;
    switch (flavor) {
        case 0: random_rows_kernel<false, 0><<<grid, 256, 0, st>>>(rows, scales, n_rows, n_warps, seed, sink); break;
        case 1: random_rows_kernel<false, 1><<<grid, 256, 0, st>>>(rows, scales, n_rows, n_warps, seed, sink); break;
        case 2: random_rows_kernel<false, 2><<<grid, 256, 0, st>>>(rows, scales, n_rows, n_warps, seed, sink); break;
        default: random_rows_kernel<false, 3><<<grid, 256, 0, st>>>(rows, scales, n_rows, n_warps, seed, sink); break;
    }
    return (int)cudaGetLastError();
}

// rows in pinned host memory (plain loads); no scales
extern "C" int probe_random_host_rows(const uint8_t *rows, int64_t n_rows, int64_t n_warps, uint64_t seed, float *sink,
                                      void *stream) {
    const int64_t threads = n_warps * 32;
    random_rows_kernel<true><<<(unsigned)((threads + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
        rows, nullptr, n_rows, n_warps, seed, sink);
    return (int)cudaGetLastError();
}
