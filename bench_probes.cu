// Bandwidth probes for bench.py --probe: the ceilings the Engram kernels are
// measured against on this GPU.  Not part of libengram.
//  - random_rows: one warp reads 2 random 256-byte rows per load instruction
//    (the gather's access pattern, 12 loads in flight per lane) from a buffer
//    of n_rows rows, optionally with one 4-byte scale per row from a second
//    array, and reduces them so the loads cannot be dropped.
#include <cuda_runtime.h>
#include <stdint.h>

__device__ __forceinline__ uint64_t mix64(uint64_t x) {  // SplitMix64 finaliser
    x ^= x >> 30; x *= 0xBF58476D1CE4E5B9ull;
    x ^= x >> 27; x *= 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

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
        v[i] = __ldg(reinterpret_cast<const uint4 *>(rows + r * 256) + c16);
        if (scales && c16 == 0) s += __ldg(scales + r);
    }
    uint32_t x = 0;
#pragma unroll
    for (int i = 0; i < 12; ++i) x ^= v[i].x ^ v[i].y ^ v[i].z ^ v[i].w;
    if (x == 0x12345678u && s == 1.2345f) sink[0] = (float)x;  // keeps the loads alive
}

extern "C" int probe_random_rows(const uint8_t *rows, const float *scales, int64_t n_rows, int64_t n_warps,
                                 uint64_t seed, float *sink, void *stream) {
    const int64_t threads = n_warps * 32;
    random_rows_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, (cudaStream_t)stream>>>(rows, scales, n_rows,
                                                                                          n_warps, seed, sink);
    return (int)cudaGetLastError();
}
