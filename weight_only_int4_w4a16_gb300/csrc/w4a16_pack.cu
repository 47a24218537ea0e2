// Load-time kernels: pack 4-bit values into 32-bit words, unpack them again,
// and restore the fp32 / fp16 weights (q - z) * s.
//
// Layout: element k of a row is nibble k % 8 (bits 4*(k%8)..+3) of word k / 8;
// zeros use the same rule along the group axis with ceil(G/8) words per row.
// The thread "vLLM on Hygon Z100" (forum.sourcefind.cn), section 四, stores
// INT4 weights as "[N,K/8] int32" and builds its packed weights once after
// loading, with a 2-D repack kernel instead of a per-chunk host loop; these
// kernels are that load-time step for this library's layout.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kThreads = 256;

// One thread per 32-bit word of qweight: 8 input bytes -> 8 nibbles.
__global__ void pack_q_kernel(const uint8_t *__restrict__ q, uint32_t *__restrict__ qw,
                              long long n_words) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_words;
         i += (long long)gridDim.x * blockDim.x) {
        uint2 b = *reinterpret_cast<const uint2 *>(q + 8 * i);
        // bytes b0..b7 (little endian) -> nibble j = low 4 bits of byte j
        uint32_t lo = b.x & 0x0f0f0f0fu;  // bytes 0..3
        uint32_t hi = b.y & 0x0f0f0f0fu;  // bytes 4..7
        // gather the low nibble of each byte: byte j lands at nibble j
        uint32_t w = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            w |= ((lo >> (8 * j)) & 0xfu) << (4 * j);
            w |= ((hi >> (8 * j)) & 0xfu) << (4 * (j + 4));
        }
        qw[i] = w;
    }
}

__global__ void pack_z_kernel(const uint8_t *__restrict__ z, uint32_t *__restrict__ zeros, int N,
                              int G, int ZW) {
    long long total = (long long)N * ZW;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        long long n = i / ZW;
        int w = (int)(i - n * ZW);
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int g = 8 * w + j;
            if (g < G) word |= (uint32_t)(z[n * G + g] & 0xfu) << (4 * j);
        }
        zeros[i] = word;
    }
}

__global__ void unpack_q_kernel(const uint32_t *__restrict__ qw, uint8_t *__restrict__ q,
                                long long n_words) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_words;
         i += (long long)gridDim.x * blockDim.x) {
        uint32_t w = qw[i];
        uint2 b;
        b.x = (w & 0xfu) | ((w >> 4) & 0xfu) << 8 | ((w >> 8) & 0xfu) << 16 |
              ((w >> 12) & 0xfu) << 24;
        b.y = ((w >> 16) & 0xfu) | ((w >> 20) & 0xfu) << 8 | ((w >> 24) & 0xfu) << 16 |
              ((w >> 28) & 0xfu) << 24;
        *reinterpret_cast<uint2 *>(q + 8 * i) = b;
    }
}

__global__ void unpack_z_kernel(const uint32_t *__restrict__ zeros, uint8_t *__restrict__ z, int N,
                                int G, int ZW) {
    long long total = (long long)N * G;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        long long n = i / G;
        int g = (int)(i - n * G);
        z[i] = (uint8_t)((zeros[n * ZW + g / 8] >> (4 * (g % 8))) & 0xfu);
    }
}

// One thread per word: 8 weights of one group.  The fp32 product of a 4-bit
// difference and an fp16 scale needs at most 15 significant bits, so it is
// exact; the fp16 output is that exact value rounded once (nearest-even).
__global__ void dequant_kernel(const uint32_t *__restrict__ qw, const __half *__restrict__ scales,
                               const uint32_t *__restrict__ zeros, int N, int K, int G, int ZW,
                               float *__restrict__ w32, __half *__restrict__ w16) {
    const int KW = K / 8;
    long long total = (long long)N * KW;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        long long n = i / KW;
        int kw = (int)(i - n * KW);
        int g = (8 * kw) / kGroup;
        uint32_t w = qw[i];
        int zv = (int)((zeros[n * ZW + g / 8] >> (4 * (g % 8))) & 0xfu);
        float s = __half2float(scales[n * G + g]);
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (float)((int)((w >> (4 * j)) & 0xfu) - zv) * s;
        if (w32) {
            float4 *o = reinterpret_cast<float4 *>(w32 + 8 * i);
            o[0] = make_float4(v[0], v[1], v[2], v[3]);
            o[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
        if (w16) {
            __half2 h[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                h[j] = __halves2half2(__float2half_rn(v[2 * j]), __float2half_rn(v[2 * j + 1]));
            *reinterpret_cast<uint4 *>(w16 + 8 * i) = *reinterpret_cast<uint4 *>(h);
        }
    }
}

// ---- checkpoint repack: transpose a packed 4-bit matrix at nibble level ----
// The Z100 thread (section 四) transposes and repacks INT4 checkpoint layouts
// at load time in 8 x 8 nibble blocks, without unpacking the whole matrix to
// int32.  Here a CTA moves a tile of 32 x 32 blocks (256 source rows x 256
// source columns): each thread loads the 8 words of a block (8 source rows,
// coalesced across the warp), brings their nibbles into sequential order,
// transposes the block in registers (three exchange stages: 4 x 4 quadrants
// between words e and e + 4, 2 x 2 within them between e and e + 2, single
// nibbles between e and e + 1) and parks the 8 result words in shared memory;
// the CTA then writes whole destination rows, coalesced.
constexpr int kTile = 32;  // blocks per tile side

__device__ __forceinline__ void swap_bits(uint32_t &lo, uint32_t &hi, int shift, uint32_t mask) {
    const uint32_t t = ((lo >> shift) ^ hi) & mask;
    lo ^= t << shift;
    hi ^= t;
}

__global__ void __launch_bounds__(kThreads)
    transpose_u4_kernel(const uint32_t *__restrict__ src, int rows, int SW, uint32_t order,
                        int sequential, uint32_t *__restrict__ dst, int cols, int DW) {
    // [nibble j][column word in tile][row block in tile], padded against bank conflicts
    __shared__ uint32_t tile[8][kTile][kTile + 1];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int cw0 = blockIdx.x * kTile, rb0 = blockIdx.y * kTile;
    const int cw = cw0 + tx;
    for (int i = 0; i < kTile / 8; ++i) {
        const int rbl = ty + 8 * i;
        const long long r0 = 8LL * (rb0 + rbl);
        uint32_t a[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const long long r = r0 + e;
            a[e] = (cw < SW && r < rows) ? src[r * SW + cw] : 0u;
        }
        if (!sequential) {  // element j of a word sits at nibble (order >> 4j) & 7
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                uint32_t w = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t pos = (order >> (4 * j)) & 7u;
                    w |= ((a[e] >> (4 * pos)) & 0xfu) << (4 * j);
                }
                a[e] = w;
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) swap_bits(a[e], a[e + 4], 16, 0x0000ffffu);
        swap_bits(a[0], a[2], 8, 0x00ff00ffu);
        swap_bits(a[1], a[3], 8, 0x00ff00ffu);
        swap_bits(a[4], a[6], 8, 0x00ff00ffu);
        swap_bits(a[5], a[7], 8, 0x00ff00ffu);
#pragma unroll
        for (int e = 0; e < 8; e += 2) swap_bits(a[e], a[e + 1], 4, 0x0f0f0f0fu);
        // a[j] is now column 8 * cw + j of the source over the block's 8 rows
#pragma unroll
        for (int j = 0; j < 8; ++j) tile[j][tx][rbl] = a[j];
    }
    __syncthreads();
    // destination row 8 * (cw0 + c) + j, words rb0 .. rb0 + 31 (one per lane)
    for (int d = ty; d < 8 * kTile; d += kThreads / 32) {
        const int c = d >> 3, j = d & 7;
        const long long row = 8LL * (cw0 + c) + j;
        if (row < cols && rb0 + tx < DW) dst[row * DW + rb0 + tx] = tile[j][c][tx];
    }
}

// Transpose of a 16-bit matrix by 32 x 32 tiles (the scales of a checkpoint
// stored [G, N] into this layout's [N, G]).
__global__ void __launch_bounds__(kThreads)
    transpose_u16_kernel(const uint16_t *__restrict__ src, int rows, int cols,
                         uint16_t *__restrict__ dst) {
    __shared__ uint16_t tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int i = ty; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + tx;
        if (r < rows && c < cols) tile[i][tx] = src[(long long)r * cols + c];
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, r = r0 + tx;
        if (c < cols && r < rows) dst[(long long)c * rows + r] = tile[tx][i];
    }
}

int grid_for(long long items) {
    long long b = (items + kThreads - 1) / kThreads;
    if (b < 1) b = 1;
    if (b > 65535LL * 8) b = 65535LL * 8;
    return (int)b;
}

}  // namespace

cudaError_t launch_pack(const uint8_t *q, const uint8_t *z, int N, int K, uint32_t *qw,
                        uint32_t *zeros, cudaStream_t stream) {
    int G = K / kGroup, ZW = (G + 7) / 8;
    long long n_words = (long long)N * (K / 8);
    pack_q_kernel<<<grid_for(n_words), kThreads, 0, stream>>>(q, qw, n_words);
    pack_z_kernel<<<grid_for((long long)N * ZW), kThreads, 0, stream>>>(z, zeros, N, G, ZW);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t *qw, const uint32_t *zeros, int N, int K, uint8_t *q,
                          uint8_t *z, cudaStream_t stream) {
    int G = K / kGroup, ZW = (G + 7) / 8;
    long long n_words = (long long)N * (K / 8);
    unpack_q_kernel<<<grid_for(n_words), kThreads, 0, stream>>>(qw, q, n_words);
    unpack_z_kernel<<<grid_for((long long)N * G), kThreads, 0, stream>>>(zeros, z, N, G, ZW);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t *qw, const __half *scales, const uint32_t *zeros,
                           int N, int K, float *w_f32, __half *w_f16, cudaStream_t stream) {
    int G = K / kGroup, ZW = (G + 7) / 8;
    long long n_words = (long long)N * (K / 8);
    dequant_kernel<<<grid_for(n_words), kThreads, 0, stream>>>(qw, scales, zeros, N, K, G, ZW,
                                                               w_f32, w_f16);
    return cudaGetLastError();
}

cudaError_t launch_transpose_u4(const uint32_t *src, int rows, int cols, uint32_t order,
                                uint32_t *dst, cudaStream_t stream) {
    const int SW = cols / 8, DW = (rows + 7) / 8;
    const dim3 grid((SW + kTile - 1) / kTile, (DW + kTile - 1) / kTile);
    transpose_u4_kernel<<<grid, kThreads, 0, stream>>>(src, rows, SW, order,
                                                       order == 0x76543210u, dst, cols, DW);
    return cudaGetLastError();
}

cudaError_t launch_transpose_u16(const uint16_t *src, int rows, int cols, uint16_t *dst,
                                 cudaStream_t stream) {
    const dim3 grid((cols + 31) / 32, (rows + 31) / 32);
    transpose_u16_kernel<<<grid, kThreads, 0, stream>>>(src, rows, cols, dst);
    return cudaGetLastError();
}

}  // namespace w4a16
