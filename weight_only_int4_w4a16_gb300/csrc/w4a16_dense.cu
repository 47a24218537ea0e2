// Dense 16-bit linear y = x @ W^T for small M on the warp-level tensor-core
// MMA: W [N, K] holds fp16 or bf16 weights that were dequantised once at load
// time (forum.sourcefind.cn thread "vLLM on Hygon Z100", section 六: FP8
// weights dequantised at load to FP16/BF16 exposed the need for a large-K,
// small-M GEMV that streams K in chunks, keeps only a slice of the activations
// per work group, handles several output rows at once and multiplies and adds
// in fp32).
//
// The same skeleton as the 4-bit mma rung, without the unpack:
//   * a warp owns 16-row strips; MMA rows are weight rows, MMA columns the
//     M <= 8 tokens.  Lane (g = lane/4, c = lane%4) reads, per 32-wide chunk
//     of k, 16 bytes (8 consecutive k) of rows g and g + 8 and the same 16
//     bytes of token g's staged x: the MMA's k slots stand for a permutation
//     of k that A and B share, so neither needs reordering;
//   * weights move by TMA, per warp and stage one box of 16 rows x 128 k
//     (4 KB, laid out [chunk][row][64 B]) into a two-slot ring per warp, with a
//     proxy fence before a slot is refilled; rows past N arrive as zeros;
//   * a CTA stages its unit's K slice of x once by bulk copy; units (a K slice
//     x a block of strips) go round-robin over persistent CTAs;
//   * split K: fp32 partials per slice, the CTA that brings a block's last
//     slice sums them in slice order (deterministic) and writes y;
//   * every wait is bounded (200 ms); an expired wait sets a status bit and
//     the CTA drains its copies and leaves.
#include <cuda.h>
#include <string.h>

#include "../../include/w4a16.h"
#include "w4a16_device.cuh"
#include "w4a16_internal.h"
#include "w4a16_mma_common.cuh"

namespace w4a16 {
namespace {

using namespace warp_mma;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCtasPerSm = 2;
constexpr int kStageK = 128;                        // k per stage: 4 chunks of 32
constexpr int kStageBytes = 16 * kStageK * 2;       // 4 KB
constexpr int kDepth = 2;                           // ring slots per warp
constexpr int kRingBytes = kWarps * kDepth * kStageBytes;  // 64 KB
constexpr int kBarBytes = 256;  // ring barriers, the x barrier, flags
constexpr int kSmemPerCta = 228 * 1024 / kCtasPerSm - 1024;
constexpr int kMaxSplit = 32;
constexpr int kErrDenseWait = 512;  // device status bit: a wait of the dense kernel expired

struct DenseParams {
    CUtensorMap tmap;  // W as (element in chunk, row, chunk of 32 k)
    const __half *x;   // 16-bit storage, fp16 or bf16
    __half *y;
    float *partials;
    unsigned *counters;
    int *status;
    int M, N, K, S, slice_stages, n_strips, strips_per_warp, n_blocks, units, xstride;
};

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// weights: boxes {32 elements, 16 rows, 4 chunks} at (0, row, chunk) (tma_box)

// y = the sum of the S partial slices of block sb, in slice order
template <bool kBf16>
__device__ __noinline__ void dense_reduce(const DenseParams &P, int sb) {
    const int rows_per_block = kWarps * P.strips_per_warp * 16;
    const int row0 = sb * rows_per_block;
    const int nrows = min(P.N - row0, rows_per_block);
    for (int i = threadIdx.x; i < P.M * nrows; i += kThreads) {
        const int t = i / nrows, row = row0 + i - t * nrows;
        float sum = 0.f;
        for (int s = 0; s < P.S; ++s) sum += __ldcg(P.partials + ((size_t)s * P.M + t) * P.N + row);
        P.y[(size_t)t * P.N + row] = from_float<kBf16>(sum);
    }
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    dense_kernel(const __grid_constant__ DenseParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    uint8_t *ring = smem + (size_t)warp * kDepth * kStageBytes;
    const uint32_t ring0 = dev::smem_u32(ring);
    const uint32_t bar0 = dev::smem_u32(smem + kRingBytes) + 16 * warp;  // this warp's 2 slots
    const uint32_t x_bar = dev::smem_u32(smem + kRingBytes + 128);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + kRingBytes + 136);
    uint8_t *xs = smem + kRingBytes + kBarBytes;
    const int total_stages = P.K / kStageK;
    const int grid = gridDim.x;
    if (lane == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        if (warp == 0) mbar_init(x_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        flags[0] = 0;  // a wait expired: every warp stops at its next unit
        flags[1] = 0;  // this CTA reduces the block of its unit
    }
    __syncthreads();

    // ---- this warp's copy stream: (unit, strip, stage) in consumption order,
    // up to kDepth stages ahead of the consumer
    int iu = blockIdx.x, ir = 0, ij = 0, i_strip = 0, i_nst = 0, i_chunk0 = 0;
    bool i_done = false;
    unsigned t_iss = 0, t_cons = 0;
    auto i_enter = [&]() {  // the first unit from iu on in which this warp has a strip
        for (; iu < P.units; iu += grid) {
            const int slice = iu / P.n_blocks, sb = iu - slice * P.n_blocks;
            const int strip0 = sb * kWarps * P.strips_per_warp + warp;
            if (strip0 >= P.n_strips) continue;
            ir = 0;
            ij = 0;
            i_strip = strip0;
            i_nst = min(P.slice_stages, total_stages - slice * P.slice_stages);
            i_chunk0 = slice * P.slice_stages * (kStageK / 32);
            return;
        }
        i_done = true;
    };
    auto issue_next = [&]() {
        if (i_done) return;
        const uint32_t slot = t_iss & 1u;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar0 + 8 * slot, kStageBytes);
            tma_box(ring0 + slot * kStageBytes, &P.tmap, i_strip * 16,
                    i_chunk0 + (kStageK / 32) * ij, bar0 + 8 * slot);
        }
        ++t_iss;
        if (++ij == i_nst) {
            ij = 0;
            if (++ir < P.strips_per_warp && i_strip + kWarps < P.n_strips) {
                i_strip += kWarps;
            } else {
                iu += grid;
                i_enter();
            }
        }
    };
    static_assert(kDepth == 2, "the slot and parity arithmetic assumes two slots");
    i_enter();
    issue_next();
    issue_next();

    uint32_t x_par = 0;
    bool x_pending = false, dead = false;
    const int tok = g < P.M ? g : 0;  // lanes of tokens >= M compute a column nobody stores
    for (int u = blockIdx.x; u < P.units; u += grid) {
        const int slice = u / P.n_blocks, sb = u - slice * P.n_blocks;
        const int nst = min(P.slice_stages, total_stages - slice * P.slice_stages);
        __syncthreads();  // the previous unit's x reads and reduction are done
        if (flags[0]) {
            dead = true;
            break;
        }
        // ---- stage x[:, slice] (one bulk copy per token row)
        if (threadIdx.x == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const uint32_t bytes = (uint32_t)nst * kStageK * 2;
            mbar_arrive_expect_tx(x_bar, bytes * P.M);
            for (int t = 0; t < P.M; ++t)
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1], %2, [%3];" ::"r"(dev::smem_u32(xs) + t * P.xstride),
                    "l"(P.x + (size_t)t * P.K + (size_t)slice * P.slice_stages * kStageK),
                    "r"(bytes), "r"(x_bar)
                    : "memory");
        }
        x_pending = true;
        if (!__all_sync(0xffffffffu, mbar_wait(x_bar, x_par))) {
            if (lane == 0) {
                atomicOr(P.status, kErrDenseWait);
                flags[0] = 1;
            }
            dead = true;
            break;
        }
        x_par ^= 1u;
        x_pending = false;
        const uint8_t *xrow = xs + (size_t)tok * P.xstride + 16 * c;
        for (int r = 0, strip = sb * kWarps * P.strips_per_warp + warp;
             r < P.strips_per_warp && strip < P.n_strips; ++r, strip += kWarps) {
            float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
            for (int j = 0; j < nst; ++j) {
                const uint32_t slot = t_cons & 1u, par = (t_cons >> 1) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * slot, par))) {
                    if (lane == 0) {
                        atomicOr(P.status, kErrDenseWait);
                        flags[0] = 1;
                    }
                    dead = true;
                    break;
                }
                // rows g and g + 8 (512 bytes further) of each 32-k chunk
                const uint8_t *st = ring + slot * kStageBytes + g * 64 + 16 * c;
                const uint8_t *xj = xrow + (size_t)j * kStageK * 2;
#pragma unroll
                for (int q = 0; q < kStageK / 32; ++q) {
                    const uint4 wa = *reinterpret_cast<const uint4 *>(st + q * 1024);
                    const uint4 wb = *reinterpret_cast<const uint4 *>(st + q * 1024 + 512);
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xj + q * 64);
                    const uint32_t a0[4] = {wa.x, wb.x, wa.y, wb.y};
                    const uint32_t a1[4] = {wa.z, wb.z, wa.w, wb.w};
                    if constexpr (kBf16) {
                        mma16816_bf16(acc0, a0, xv.x, xv.y);
                        mma16816_bf16(acc1, a1, xv.z, xv.w);
                    } else {
                        mma16816(acc0, a0, xv.x, xv.y);
                        mma16816(acc1, a1, xv.z, xv.w);
                    }
                }
                // the lanes' reads of the slot before the TMA refills it
                __syncwarp();
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                ++t_cons;
                issue_next();
            }
            if (dead) break;
            // acc[0..1]: row ra, tokens 2c, 2c + 1; acc[2..3]: row rb
            const int ra = strip * 16 + g, rb = ra + 8, t0 = 2 * c, t1 = 2 * c + 1;
            const bool va = ra < P.N, vb = rb < P.N;
            float acc[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = acc0[e] + acc1[e];
            if (P.S == 1) {
                if (va && t0 < P.M) P.y[(size_t)t0 * P.N + ra] = from_float<kBf16>(acc[0]);
                if (va && t1 < P.M) P.y[(size_t)t1 * P.N + ra] = from_float<kBf16>(acc[1]);
                if (vb && t0 < P.M) P.y[(size_t)t0 * P.N + rb] = from_float<kBf16>(acc[2]);
                if (vb && t1 < P.M) P.y[(size_t)t1 * P.N + rb] = from_float<kBf16>(acc[3]);
            } else {
                float *ps = P.partials + (size_t)slice * P.M * P.N;
                if (va && t0 < P.M) ps[(size_t)t0 * P.N + ra] = acc[0];
                if (va && t1 < P.M) ps[(size_t)t1 * P.N + ra] = acc[1];
                if (vb && t0 < P.M) ps[(size_t)t0 * P.N + rb] = acc[2];
                if (vb && t1 < P.M) ps[(size_t)t1 * P.N + rb] = acc[3];
            }
        }
        if (dead) break;
        if (P.S > 1) {
            // the CTA whose arrival completes the block sums its slices
            __syncthreads();
            if (threadIdx.x == 0) {
                unsigned prev;
                asm volatile("fence.acq_rel.gpu;\n\tatom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                             : "=r"(prev)
                             : "l"(P.counters + sb)
                             : "memory");
                flags[1] = prev == (unsigned)(P.S - 1);
            }
            __syncthreads();
            if (flags[1]) {
                dense_reduce<kBf16>(P, sb);
                if (threadIdx.x == 0) P.counters[sb] = 0u;  // ready for the next launch
            }
        }
    }
    if (dead) {
        // let this warp's copies in flight land (bounded) before the shared
        // memory goes away
        for (; t_cons < t_iss; ++t_cons) mbar_wait(bar0 + 8 * (t_cons & 1u), (t_cons >> 1) & 1u);
        if (x_pending) mbar_wait(x_bar, x_par);
    }
}


int dense_xstride(int slice_stages) { return slice_stages * kStageK * 2 + 64; }

}  // namespace

DensePlan plan_dense(int M, int N, int K, const DeviceInfo &dev) {
    DensePlan pl{};
    pl.M = M;
    const int total = K / kStageK;
    pl.n_strips = (N + 15) / 16;
    // largest slice whose staged x fits (row stride = slice bytes + 64: the
    // rows of two tokens fall on different 64-byte halves of a bank line)
    const int budget = kSmemPerCta - kRingBytes - kBarBytes;
    int max_stages = (budget / M - 64) / (kStageK * 2);
    if (max_stages < 1) max_stages = 1;
    const int grid_max = kCtasPerSm * dev.sm_count;
    const int s_min = (total + max_stages - 1) / max_stages;
    int s_hi = total < kMaxSplit ? total : kMaxSplit;
    if (s_hi < s_min) s_hi = s_min;
    // the cost model of the 4-bit rung's one-linear planner: a dense 4 KB
    // stage moves the same bytes as a 4-bit one
    double best = 1e30;
    for (int spw = 1; spw <= 8; spw *= 2) {
        const int nb = (pl.n_strips + kWarps * spw - 1) / (kWarps * spw);
        for (int S = s_min; S <= s_hi; ++S) {
            const int ss = (total + S - 1) / S;
            if (ss > max_stages) continue;
            const int S_eff = (total + ss - 1) / ss;
            const long long units = (long long)nb * S_eff;
            const long long per_cta = (units + grid_max - 1) / grid_max;
            const double load = (double)(units < grid_max ? units : grid_max) / grid_max;
            const double cost = (double)per_cta * (2.2 + (double)spw * ss * (0.85 + 0.45 * load)) +
                                (S_eff > 1 ? 4.5 + 2.0 * S_eff : 0.0);
            if (cost < best - 1e-9) {
                best = cost;
                pl.slice_stages = ss;
                pl.S = S_eff;
                pl.strips_per_warp = spw;
                pl.n_blocks = nb;
            }
        }
    }
    if (pl.slice_stages == 0) return pl;  // ok = false
    pl.units = pl.S * pl.n_blocks;
    pl.grid = pl.units < grid_max ? pl.units : grid_max;
    pl.smem_bytes = kRingBytes + kBarBytes + M * dense_xstride(pl.slice_stages);
    pl.ws_bytes = pl.S > 1 ? (size_t)pl.S * M * N * sizeof(float) : 0;
    pl.ok = true;
    return pl;
}

cudaError_t launch_dense(const __half *x, const __half *w, __half *y, int M, int N, int K,
                         bool bf16, const DensePlan &plan, const Workspace &ws,
                         cudaStream_t stream) {
    const EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorInitializationError;
    DenseParams P;
    memset(&P, 0, sizeof(P));
    // W as a 3-D tensor of 16-bit elements: (element in a 32-k chunk, row,
    // chunk); a box brings 16 rows x 4 chunks, chunk-major
    const cuuint64_t dims[3] = {32, (cuuint64_t)N, (cuuint64_t)K / 32};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 64};
    const cuuint32_t box[3] = {32, 16, (cuuint32_t)(kStageK / 32)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(&P.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, (void *)w, dims,
                                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    P.x = x;
    P.y = y;
    P.partials = ws.partials;
    P.counters = ws.counters;
    P.status = ws.status;
    P.M = M;
    P.N = N;
    P.K = K;
    P.S = plan.S;
    P.slice_stages = plan.slice_stages;
    P.n_strips = plan.n_strips;
    P.strips_per_warp = plan.strips_per_warp;
    P.n_blocks = plan.n_blocks;
    P.units = plan.units;
    P.xstride = dense_xstride(plan.slice_stages);
    if (bf16) {
        dense_kernel<true><<<plan.grid, kThreads, plan.smem_bytes, stream>>>(P);
    } else {
        dense_kernel<false><<<plan.grid, kThreads, plan.smem_bytes, stream>>>(P);
    }
    return cudaGetLastError();
}

cudaError_t dense_init(const DeviceInfo &dev) {
    if (!tensor_map_encoder()) return cudaErrorSymbolNotFound;
    int dyn = kSmemPerCta;
    if (dyn > dev.max_smem_optin - 1024) dyn = dev.max_smem_optin - 1024;
    cudaError_t e = cudaSuccess;
    const void *fns[2] = {(const void *)dense_kernel<false>, (const void *)dense_kernel<true>};
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
        e = cudaFuncSetAttribute(fns[k], cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fns[k], cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
    }
    return e;
}

}  // namespace w4a16
