// CUDA-core W4A16 GEMV for M = 1..8 tokens (rungs "gemv" and "gemv_splitk").
//
// The method: forum.sourcefind.cn thread "vLLM on Hygon Z100", sections 四 and
// 五.  Section 四's M = 1 kernel stages the activation on chip, streams the
// packed INT4 weights with non-temporal loads, gives each wavefront some output
// rows, multiplies paired fp16 values and accumulates in fp32; section 五's
// small-M kernel streams the weights once and serves every activation row from
// them.  The same structure on sm_103a:
//
//   * a CTA (8 warps) stages x[:, K-slice] in shared memory once, converted to
//     the pair order the unpack below produces (convert the input once, before
//     the inner loop: haowenji.com V100 decode article, the fix that took two
//     projections from 350 GB/s to full speed);
//   * each warp streams its own sequence of output rows: lane 0 keeps the
//     next kRing row slices in flight with cp.async.bulk copies into a
//     per-warp shared-memory ring (completion on an mbarrier), so the bytes in
//     flight do not depend on registers; lane j then works on 16-byte chunks
//     j, j+32, ... of the row slice (32 k values, always inside one 128-wide
//     group), and the next row's scales and zeros are fetched while the
//     current row is computed;
//   * unpack: a nibble OR-ed into the mantissa of the fp16 constant 1024 (or 64
//     for the odd nibble positions, which sit 4 bits higher) is the fp16 value
//     1024 + q (64 + q), two lanes of a 32-bit register at once; subtracting
//     (1024 + z) is exact and leaves q - z as an fp16 integer.  This is the
//     "splice the integer into the fp16 bit pattern, subtract a fixed offset"
//     conversion of the V100 article's attention kernel, applied to nibbles;
//   * dot product: fma.rn.f32.f16 multiplies two fp16 values exactly and adds
//     in fp32, per token; each chunk's sum is scaled by its group's fp32 scale
//     once (scale hoisted out of the inner loop);
//   * the 32 lane sums of a row are combined with xor-shuffles.
//
// Split-K (ninfer-perf-tuning notes, rule 21 and the per-shape knob table:
// split K only when the row grid cannot fill the GPU, keep several K steps per
// slice; reduce in fp32): each (row block, slice) CTA writes fp32 partials,
// bumps the row block's arrival counter, and the CTA that arrives last sums the
// S partials in slice order 0..S-1 and writes y.  No CTA ever waits for
// another, and the sum order does not depend on arrival order, so results are
// bit-identical from run to run.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 8;                // each warp streams its own rows
constexpr int kThreads = kWarps * 32;
constexpr int kRing = 4;                 // row slices in flight per warp
constexpr int kChunkK = 32;              // k values per 16-byte chunk
constexpr int kMaxSliceGroups = 64;      // 4 KB of packed weights per row slice
constexpr int kXBudget = 64 * 1024;      // staged activations per CTA
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;

struct GemvParams {
    const __half *x;
    const uint32_t *qw;
    const __half *scales;
    const uint32_t *zeros;
    __half *y;
    float *partials;
    unsigned *counters;
    int *status;
    int N, K, G, ZW, KW;
    int S, slice_groups;
    int rows_per_cta;
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;  // (a & b) | c
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// a0 += lo(w) * lo(x), a1 += hi(w) * hi(x): fp16 x fp16 products (exact) added in fp32.
__device__ __forceinline__ void fma_pair(float &a0, float &a1, uint32_t w, uint32_t x) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w), "r"(x));
}

// 8 consecutive fp16 (h0..h7) -> pairs (h0,h4) (h1,h5) (h2,h6) (h3,h7): the
// order in which the unpack below yields the nibbles of one word.
__device__ __forceinline__ uint4 pair_order(uint4 v) {
    uint4 o;
    o.x = prmt(v.x, v.z, 0x5410);
    o.y = prmt(v.x, v.z, 0x7632);
    o.z = prmt(v.y, v.w, 0x5410);
    o.w = prmt(v.y, v.w, 0x7632);
    return o;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase (false after kWaitNs).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kWaitNs) return false;
    return true;
}

// One row slice: `bytes` contiguous bytes from global memory into shared
// memory, completion counted on the mbarrier.
__device__ __forceinline__ void bulk_row(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

template <int M>
__global__ void __launch_bounds__(kThreads) gemv_kernel(GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_last;
    __shared__ __align__(8) uint64_t bars[kWarps][kRing];

    const int s = blockIdx.y;
    const int g0 = s * p.slice_groups;
    const int g1 = min(p.G, g0 + p.slice_groups);
    const int k0 = g0 * kGroup;
    const int nchunks = (g1 - g0) * (kGroup / kChunkK);
    const int nCB = (nchunks + 31) / 32;  // lane chunks per row (<= kMaxLaneChunks)
    const uint32_t slice_bytes = (uint32_t)nchunks * 16u;
    const uint32_t ring_stride = (slice_bytes + 127u) & ~127u;  // bytes per ring slot

    uint4 *xs = reinterpret_cast<uint4 *>(smem);  // [M][nCB][4][32] uint4
    uint8_t *ring = smem + (size_t)M * nCB * 4 * 32 * sizeof(uint4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * p.rows_per_cta;
    const int row_end = min(p.N, row0 + p.rows_per_cta);
    // this warp's rows: row0 + warp + 8 i
    const int my_rows = row_end > row0 + warp ? (row_end - row0 - warp + kWarps - 1) / kWarps : 0;
    uint8_t *my_ring = ring + (size_t)warp * kRing * ring_stride;

    if (lane == 0)
        for (int i = 0; i < kRing; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[warp][i]))
                         : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();
    // Start the weight stream before staging x: the first row slices are in
    // flight while x is converted.
    int issued = 0;  // row slices whose copy lane 0 has issued
    if (lane == 0)
        for (int i = 0; i < kRing && i < my_rows; ++i, ++issued) {
            const int n = row0 + warp + kWarps * i;
            bulk_row(smem_u32(my_ring + i * ring_stride), p.qw + (size_t)n * p.KW + k0 / 8,
                     slice_bytes, smem_u32(&bars[warp][i]));
        }

    // Stage x[:, k0 : k0 + 32*nchunks] in pair order.  Piece (m, c, t) holds
    // the 8 values of word t of chunk c; lane c%32 reads it with one LDS.128.
    for (int i = threadIdx.x; i < M * nchunks * 4; i += kThreads) {
        int m = i / (nchunks * 4);
        int rem = i - m * nchunks * 4;
        int c = rem >> 2, t = rem & 3;
        uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)m * p.K + k0 + kChunkK * c +
                                                        8 * t));
        xs[((m * nCB + (c >> 5)) * 4 + t) * 32 + (c & 31)] = pair_order(v);
    }
    __syncthreads();

    // Per-row metadata, one row ahead: lane l holds the scales of slice groups
    // l and l + 32, and the zeros word g0/8 + l; the chunk loop fetches the
    // values it needs from the owning lane with shuffles.
    const int zw0 = g0 >> 3;
    const int nzw = ((g1 - 1) >> 3) - zw0 + 1;  // zeros words touched by the slice
    float s_lo_next = 0.f, s_hi_next = 0.f;
    uint32_t z_next = 0;
    auto fetch_meta = [&](int i) {
        if (i < my_rows) {
            const int n = row0 + warp + kWarps * i;
            const __half *srow = p.scales + (size_t)n * p.G + g0;
            if (lane < g1 - g0) s_lo_next = __half2float(srow[lane]);
            if (lane + 32 < g1 - g0) s_hi_next = __half2float(srow[lane + 32]);
            if (lane < nzw) z_next = __ldg(p.zeros + (size_t)n * p.ZW + zw0 + lane);
        }
    };
    fetch_meta(0);
    bool ok = true;

    for (int i = 0; i < my_rows; ++i) {
        const int n = row0 + warp + kWarps * i;
        const int slot = i % kRing;
        const float s_lo = s_lo_next, s_hi = s_hi_next;
        const uint32_t zrow = z_next;
        fetch_meta(i + 1);
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp][slot]), (i / kRing) & 1))) {
            if (lane == 0) atomicOr(p.status, 1);
            ok = false;
            break;
        }
        const uint4 *wrow = reinterpret_cast<const uint4 *>(my_ring + slot * ring_stride);
        float acc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = 0.f;
        for (int j = 0; j < nCB; ++j) {
            // chunk c = lane + 32 j lies in slice group gl = 8 j + lane / 4
            const int c = lane + 32 * j;
            const int gl = 8 * j + (lane >> 2);
            const float sc = __shfl_sync(0xffffffffu, (j >> 2) ? s_hi : s_lo, gl & 31);
            const int zg = g0 + gl;
            const uint32_t zword = __shfl_sync(0xffffffffu, zrow, ((zg >> 3) - zw0) & 31);
            if (c < nchunks) {
                const uint4 wv = wrow[c];
                const uint32_t z = (zword >> (4 * (zg & 7))) & 0xfu;
                const uint32_t zz_hi = 0x64006400u | z | (z << 16);         // 1024 + z
                const uint32_t zz_lo = 0x54005400u | (z << 4) | (z << 20);  // 64 + z
                float part0[M], part1[M];
#pragma unroll
                for (int m = 0; m < M; ++m) part0[m] = part1[m] = 0.f;
                const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t w = words[t];
                    const uint32_t w8 = w >> 8;
                    const uint32_t d0 = hsub2(lop3_and_or(w, 0x000f000fu, 0x64006400u), zz_hi);
                    const uint32_t d1 = hsub2(lop3_and_or(w, 0x00f000f0u, 0x54005400u), zz_lo);
                    const uint32_t d2 = hsub2(lop3_and_or(w8, 0x000f000fu, 0x64006400u), zz_hi);
                    const uint32_t d3 = hsub2(lop3_and_or(w8, 0x00f000f0u, 0x54005400u), zz_lo);
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const uint4 xv = xs[((m * nCB + j) * 4 + t) * 32 + lane];
                        fma_pair(part0[m], part1[m], d0, xv.x);
                        fma_pair(part0[m], part1[m], d1, xv.y);
                        fma_pair(part0[m], part1[m], d2, xv.z);
                        fma_pair(part0[m], part1[m], d3, xv.w);
                    }
                }
#pragma unroll
                for (int m = 0; m < M; ++m) acc[m] = fmaf(sc, part0[m] + part1[m], acc[m]);
            }
        }
        // the slot is consumed: refill it with the row kRing ahead
        __syncwarp();
        if (lane == 0 && i + kRing < my_rows) {
            const int nn = row0 + warp + kWarps * (i + kRing);
            bulk_row(smem_u32(my_ring + slot * ring_stride), p.qw + (size_t)nn * p.KW + k0 / 8,
                     slice_bytes, smem_u32(&bars[warp][slot]));
            ++issued;
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
        }
        if (lane == 0) {
            if (p.S == 1) {
#pragma unroll
                for (int m = 0; m < M; ++m) p.y[(size_t)m * p.N + n] = __float2half_rn(acc[m]);
            } else {
#pragma unroll
                for (int m = 0; m < M; ++m) p.partials[((size_t)s * M + m) * p.N + n] = acc[m];
            }
        }
    }
    // Every copy this warp issued must have landed before the block exits
    // (only a warp that gave up a wait can still have copies in flight).
    if (!ok && lane == 0) {
        for (int i = issued > kRing ? issued - kRing : 0; i < issued; ++i)
            if (!mbar_wait(smem_u32(&bars[warp][i % kRing]), (i / kRing) & 1)) atomicOr(p.status, 2);
    }
    __syncwarp();

    if (p.S > 1) {
        // Publish this slice's partials, count the arrival; the last CTA of
        // the row range sums all slices in fixed order.
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned prev = atomicAdd(p.counters + blockIdx.x, 1u);
            s_last = (prev == (unsigned)(p.S - 1));
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            const int nrows = row_end - row0;
            for (int idx = threadIdx.x; idx < M * nrows; idx += kThreads) {
                const int m = idx / nrows;
                const int n = row0 + (idx - m * nrows);
                float sum = 0.f;
                for (int s2 = 0; s2 < p.S; ++s2)
                    sum += __ldcg(p.partials + ((size_t)s2 * M + m) * p.N + n);
                p.y[(size_t)m * p.N + n] = __float2half_rn(sum);
            }
            if (threadIdx.x == 0) p.counters[blockIdx.x] = 0u;  // ready for the next launch
        }
    }
}

template <int M>
cudaError_t launch_m(const GemvParams &p, const GemvPlan &plan, cudaStream_t stream) {
    dim3 grid(plan.grid_x, plan.S);
    gemv_kernel<M><<<grid, kThreads, plan.smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

int smem_for(int M, int slice_groups) {
    const int nchunks = slice_groups * (kGroup / kChunkK);
    const int nCB = (nchunks + 31) / 32;
    const int ring_stride = (nchunks * 16 + 127) & ~127;
    return M * nCB * 4 * 32 * (int)sizeof(uint4) + kWarps * kRing * ring_stride;
}

int occupancy_cache[kGemvMaxTokens + 1][8];  // [M][smem bucket] resident CTAs per SM

int resident_ctas(int M, int smem) {
    int bucket = smem / (32 * 1024);
    if (bucket > 7) bucket = 7;
    int &slot = occupancy_cache[M][bucket];
    if (slot > 0) return slot;
    int probe = (bucket + 1) * 32 * 1024;
    if (probe > 226 * 1024) probe = 226 * 1024;
    if (probe < smem) probe = smem;
    int n = 0;
    cudaError_t e = cudaSuccess;
    switch (M) {
#define W4A16_OCC(MM)                                                                           \
    case MM:                                                                                    \
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_kernel<MM>, kThreads, probe); \
        break;
        W4A16_OCC(1) W4A16_OCC(2) W4A16_OCC(3) W4A16_OCC(4)
        W4A16_OCC(5) W4A16_OCC(6) W4A16_OCC(7) W4A16_OCC(8)
#undef W4A16_OCC
    }
    if (e != cudaSuccess || n < 1) n = 1;
    slot = n;
    return n;
}

}  // namespace

GemvPlan plan_gemv(int M, int N, int K, int split, const DeviceInfo &dev) {
    GemvPlan pl{};
    pl.M = M;
    const int G = K / kGroup;
    // Largest slice: 4 KB of packed weights per row (the ring slot) and the
    // staged activations (2 KB per token per 32 chunks) within kXBudget.
    int max_groups = kMaxSliceGroups;
    const int x_groups = (kXBudget / (M * 32 * 4 * (int)sizeof(uint4))) * 32 / (kGroup / kChunkK);
    if (x_groups < max_groups) max_groups = x_groups;
    int S = (G + max_groups - 1) / max_groups;
    if (split == 0 && S > 1) {
        pl.ok = false;
        return pl;
    }
    const int min_rows = kWarps;  // at least one row per warp
    int ctas_for_rows = (N + min_rows - 1) / min_rows;
    int per_sm = resident_ctas(M, smem_for(M, (G + S - 1) / S));
    int slots = dev.sm_count * per_sm;
    if (split != 0) {
        // Fill the GPU when the rows alone cannot: at least 4 groups per slice
        // (ninfer-perf-tuning rule 21: each slice keeps several K steps).
        if (ctas_for_rows * S < slots) {
            int s_fill = slots / (ctas_for_rows < slots ? ctas_for_rows : slots);
            int s_cap = G / 4 > 0 ? G / 4 : 1;
            if (s_fill > s_cap) s_fill = s_cap;
            if (s_fill > S) S = s_fill;
        }
        if (split == 1 && S < 2 && G >= 2) S = 2;
    }
    pl.slice_groups = (G + S - 1) / S;
    S = (G + pl.slice_groups - 1) / pl.slice_groups;
    pl.S = S;
    pl.smem_bytes = smem_for(M, pl.slice_groups);
    per_sm = resident_ctas(M, pl.smem_bytes);
    slots = dev.sm_count * per_sm;
    // Row ranges: one per CTA column, balanced to within one row; enough
    // CTA columns for one resident wave across all slices.
    int cols = slots / S;
    if (cols < 1) cols = 1;
    if (cols > ctas_for_rows) cols = ctas_for_rows;
    pl.rows_per_cta = (N + cols - 1) / cols;
    pl.grid_x = (N + pl.rows_per_cta - 1) / pl.rows_per_cta;
    pl.n_row_blocks = pl.grid_x;
    pl.ws_bytes = S > 1 ? (size_t)S * M * N * sizeof(float) : 0;
    pl.threads = kThreads;
    pl.ok = true;
    return pl;
}

cudaError_t launch_gemv(const LinearArgs &a, const GemvPlan &plan, const Workspace &ws,
                        cudaStream_t stream) {
    GemvParams p;
    p.x = a.x;
    p.qw = a.qw;
    p.scales = a.scales;
    p.zeros = a.zeros;
    p.y = a.y;
    p.partials = ws.partials;
    p.counters = ws.counters;
    p.status = ws.status;
    p.N = a.N;
    p.K = a.K;
    p.G = a.K / kGroup;
    p.ZW = (p.G + 7) / 8;
    p.KW = a.K / 8;
    p.S = plan.S;
    p.slice_groups = plan.slice_groups;
    p.rows_per_cta = plan.rows_per_cta;
    switch (plan.M) {
        case 1: return launch_m<1>(p, plan, stream);
        case 2: return launch_m<2>(p, plan, stream);
        case 3: return launch_m<3>(p, plan, stream);
        case 4: return launch_m<4>(p, plan, stream);
        case 5: return launch_m<5>(p, plan, stream);
        case 6: return launch_m<6>(p, plan, stream);
        case 7: return launch_m<7>(p, plan, stream);
        case 8: return launch_m<8>(p, plan, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t gemv_init_attributes(const DeviceInfo &dev) {
    // leave room for the kernel's static shared memory (barriers, flags)
    const int dyn = dev.max_smem_optin - 1024;
    cudaError_t e = cudaSuccess;
#define W4A16_ATTR(MM)                                                                        \
    if (e == cudaSuccess)                                                                     \
        e = cudaFuncSetAttribute(gemv_kernel<MM>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 dyn);
    W4A16_ATTR(1) W4A16_ATTR(2) W4A16_ATTR(3) W4A16_ATTR(4)
    W4A16_ATTR(5) W4A16_ATTR(6) W4A16_ATTR(7) W4A16_ATTR(8)
#undef W4A16_ATTR
    for (auto &row : occupancy_cache)
        for (int &v : row) v = 0;
    return e;
}

}  // namespace w4a16
