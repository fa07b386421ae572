// Device twin of the seeded generators in synth/ (philox.py, sampler.py,
// host.py): Philox4x64-10 (Salmon et al., SC'11) and the discrete
// inverse-CDF sampler, bit-identical to the numpy versions, so tables of tens
// of GB can be filled in HBM (or in pinned host memory through unified
// addressing) while any row can still be redrawn on the host.
//
// Holds no Engram arithmetic.  Stream ids and word layouts match
// synth/configs.py and synth/host.py.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
constexpr uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;

__device__ __forceinline__ void philox(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3, uint64_t k0, uint64_t k1,
                                       uint64_t out[4]) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
        const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += W0;
        k1 += W1;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

// number of thresholds <= u  (thresholds strictly increasing)
__device__ __forceinline__ int cdf_index(const uint32_t *thr, int n_thr, uint32_t u) {
    int lo = 0, hi = n_thr;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (thr[mid] <= u) lo = mid + 1; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ uint32_t word_of(const uint64_t out[4], int i) {
    return (uint32_t)(out[i >> 1] >> (32 * (i & 1)));
}

// e4m3 codes: table j0+jj, row r, code c <- u32 word r*256 + c of stream (seed, 0x100 + j);
// rows are row_stride bytes apart (256, or 272 for rows that carry their scale)
__global__ void fill_tables_kernel(uint8_t *dst, uint64_t seed, int j0, int nj, int64_t R, int64_t row_stride,
                                   const uint32_t *thr_g, const uint16_t *codes_g, int n_codes) {
    extern __shared__ uint32_t sm[];
    uint32_t *thr = sm;
    uint16_t *codes = reinterpret_cast<uint16_t *>(sm + n_codes);
    for (int i = threadIdx.x; i < n_codes; i += blockDim.x) {
        if (i < n_codes - 1) thr[i] = thr_g[i];
        codes[i] = codes_g[i];
    }
    __syncthreads();
    const int64_t total = (int64_t)nj * R * 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t jj = i / (R * 32);
        const int64_t rem = i - jj * R * 32;
        const uint64_t row = (uint64_t)(rem >> 5), b = (uint64_t)(rem & 31);
        uint64_t out[4];
        philox(row * 32 + b, 0, 0, 0, seed, 0x100 + (uint64_t)(j0 + jj), out);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t code = codes[cdf_index(thr, n_codes - 1, word_of(out, k))] & 0xFFu;
            if (k < 4) lo |= code << (8 * k); else hi |= code << (8 * (k - 4));
        }
        *reinterpret_cast<uint2 *>(dst + ((int64_t)jj * R + (int64_t)row) * row_stride + b * 8) = make_uint2(lo, hi);
    }
}

// per-row scales of tables j0.. : word = row of stream (seed, 0x200 + j); the
// scale of row (jj, row) goes to dst + (jj*R + row)*stride + offset bytes
__global__ void fill_scales_kernel(uint8_t *dst, uint64_t seed, int j0, int nj, int64_t R, int64_t stride,
                                   int64_t offset) {
    const int64_t blocks_per_table = (R + 7) / 8;
    const int64_t total = (int64_t)nj * blocks_per_table;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t jj = i / blocks_per_table;
        const int64_t blk = i - jj * blocks_per_table;
        uint64_t out[4];
        philox((uint64_t)blk, 0, 0, 0, seed, 0x200 + (uint64_t)(j0 + jj), out);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t row = blk * 8 + k;
            if (row < R) {
                const uint32_t u = word_of(out, k);
                const long long x = (1ll << 24) + 3ll * (long long)(u >> 8);
                *reinterpret_cast<float *>(dst + (jj * R + row) * stride + offset) =
                    __ll2float_rn(x) * 0x1p-25f;  // exact power-of-two scaling
            }
        }
    }
}

// E8M0 block-scale bytes of tables j0.. : byte b of row (jj, row) is
// 125 + floor(5 u / 2^32), u = word row*8 + b of stream (seed, 0x400 + j); the
// eight bytes go to dst + (jj*R + row)*stride + offset
__global__ void fill_mx_scales_kernel(uint8_t *dst, uint64_t seed, int j0, int nj, int64_t R, int64_t stride,
                                      int64_t offset) {
    const int64_t total = (int64_t)nj * R;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t jj = i / R;
        const int64_t row = i - jj * R;
        uint64_t out[4];
        philox((uint64_t)row, 0, 0, 0, seed, 0x400 + (uint64_t)(j0 + jj), out);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t e = 125u + (uint32_t)(((uint64_t)word_of(out, k) * 5ull) >> 32);
            if (k < 4) lo |= e << (8 * k); else hi |= e << (8 * (k - 4));
        }
        *reinterpret_cast<uint2 *>(dst + i * stride + offset) = make_uint2(lo, hi);
    }
}

// bf16 bit patterns, words word0 .. word0+count-1 of stream (seed, stream)
__global__ void fill_bf16_kernel(uint16_t *dst, uint64_t seed, uint64_t stream, uint64_t word0, int64_t count,
                                 const uint32_t *thr_g, const uint16_t *codes_g, int n_codes) {
    extern __shared__ uint32_t sm[];
    uint32_t *thr = sm;
    uint16_t *codes = reinterpret_cast<uint16_t *>(sm + n_codes);
    for (int i = threadIdx.x; i < n_codes; i += blockDim.x) {
        if (i < n_codes - 1) thr[i] = thr_g[i];
        codes[i] = codes_g[i];
    }
    __syncthreads();
    const int64_t first_blk = (int64_t)(word0 >> 3);
    const int64_t last_blk = (int64_t)((word0 + count + 7) >> 3);
    for (int64_t i = first_blk + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < last_blk;
         i += (int64_t)gridDim.x * blockDim.x) {
        uint64_t out[4];
        philox((uint64_t)i, 0, 0, 0, seed, stream, out);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t w = i * 8 + k;
            if (w >= (int64_t)word0 && w < (int64_t)(word0 + count))
                dst[w - (int64_t)word0] = codes[cdf_index(thr, n_codes - 1, word_of(out, k))];
        }
    }
}

int grid_for(int64_t work) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (work + 255) / 256;
    const int64_t cap = (int64_t)sms * 16;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

extern "C" int synth_fill_tables(uint8_t *dst, uint64_t seed, int j0, int nj, int64_t R, int64_t row_stride,
                                 const uint32_t *thr, const uint16_t *codes, int n_codes, void *stream) {
    const size_t sm = (size_t)n_codes * 4 + (size_t)n_codes * 2;
    fill_tables_kernel<<<grid_for((int64_t)nj * R * 32), 256, sm, (cudaStream_t)stream>>>(dst, seed, j0, nj, R,
                                                                                        row_stride, thr, codes,
                                                                                        n_codes);
    return (int)cudaGetLastError();
}

extern "C" int synth_fill_scales(uint8_t *dst, uint64_t seed, int j0, int nj, int64_t R, int64_t stride,
                                 int64_t offset, void *stream) {
    fill_scales_kernel<<<grid_for((int64_t)nj * ((R + 7) / 8)), 256, 0, (cudaStream_t)stream>>>(dst, seed, j0, nj, R,
                                                                                            stride, offset);
    return (int)cudaGetLastError();
}

extern "C" int synth_fill_mx_scales(uint8_t *dst, uint64_t seed, int j0, int nj, int64_t R, int64_t stride,
                                    int64_t offset, void *stream) {
    if ((stride % 8) != 0 || (offset % 8) != 0 || (reinterpret_cast<uintptr_t>(dst) % 8) != 0)
        return (int)cudaErrorInvalidValue;
    fill_mx_scales_kernel<<<grid_for((int64_t)nj * R), 256, 0, (cudaStream_t)stream>>>(dst, seed, j0, nj, R, stride,
                                                                                      offset);
    return (int)cudaGetLastError();
}

extern "C" int synth_fill_bf16(uint16_t *dst, uint64_t seed, uint64_t stream_id, uint64_t word0, int64_t count,
                               const uint32_t *thr, const uint16_t *codes, int n_codes, void *stream) {
    const size_t sm = (size_t)n_codes * 4 + (size_t)n_codes * 2;
    if (sm > 48 * 1024) return (int)cudaErrorInvalidValue;
    fill_bf16_kernel<<<grid_for(count / 8 + 1), 256, sm, (cudaStream_t)stream>>>(dst, seed, stream_id, word0, count,
                                                                                 thr, codes, n_codes);
    return (int)cudaGetLastError();
}
