// W4A16 small-M rung on the warp-level tensor-core MMA ("mma", "mma_splitk").
//
// Why this rung exists: at M = 2..8 tokens the CUDA-core GEMV needs M fp32
// FMAs per weight and runs out of issue slots well below HBM speed (an SM
// issues 128 lane-instructions per clock; streaming at HBM speed delivers
// about 45 weights per clock per SM), and a tcgen05.mma of M = 128 rows and
// N <= 64 tokens costs a fixed ~46 cycles per 2048 weights whatever N is,
// which is the HBM rate itself with no slack.  mma.sync.m16n8k16 takes its A
// operand from registers: the dequantised weights never touch shared or
// tensor memory, one instruction consumes 256 weights for up to 8 tokens,
// and the SM sustains ~0.47 of them per clock (4x what HBM speed needs).
//
// The method is unchanged (forum.sourcefind.cn thread "vLLM on Hygon Z100",
// sections 四 and 五: stream the packed INT4 weights once for all M rows,
// unpack, subtract the zero, multiply with the fp16 activations, scale per
// group, accumulate in fp32):
//
//   * MMA rows are weight rows n (a warp owns a 16-row tile, a CTA 128 rows),
//     MMA columns are the M <= 8 tokens, MMA k runs along K;
//   * lane (g = lane/4, c = lane%4) loads 16 bytes of row g and of row g + 8:
//     the 32 k values 32c .. 32c+31 of a 128-wide group, so one warp load
//     instruction reads 8 rows x 64 contiguous bytes, kDepth groups ahead;
//   * the unpack (exponent-bias trick, exact) turns each word into four fp16
//     pairs (q0-z, q4-z) (q1-z, q5-z) (q2-z, q6-z) (q3-z, q7-z), which are the
//     A fragment registers as they come: the MMA's k slots 2c, 2c+1, 2c+8,
//     2c+9 stand for the actual k values k0, k4, k1, k5 (and k2, k6, k3, k7
//     for the second MMA of the word).  The B fragment must use the same
//     order, so x is staged once per CTA in pair order (x0,x4,x1,x5,...) and
//     each lane reads its two MMAs' B registers with one 16-byte load;
//   * the 8 MMAs of a group accumulate (q - z) * x exactly into a fresh fp32
//     accumulator, which is then scaled by the group's fp32 scale into the
//     running fp32 sums (scale hoisted out of the k loop);
//   * split K: fp32 partials and a last-arriving-CTA reduction in slice order,
//     as on the other rungs (deterministic, no CTA waits for another).
#include "w4a16_device.cuh"
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTileRows = 16 * kWarps;  // 128 output rows per CTA
constexpr int kDepth = 4;               // groups in flight per warp
constexpr int kXBudget = 96 * 1024;     // staged activations per CTA
constexpr int kMinSliceGroups = 4;

struct MmaParams {
    const __half *x;
    const uint32_t *qw;
    const __half *scales;
    const uint32_t *zeros;
    __half *y;
    float *partials;
    unsigned *counters;
    int N, K, G, ZW, KW;
    int M;  // tokens, 1..8
    int S, slice_groups;
    int xstride;  // bytes per staged token row
};

// Staged x: 16-byte unit J of a token row (8 activations, pair order) lives
// at unit J ^ (bit 3 of J moved to bit 1).  Together with a row stride of
// 16 (mod 128) bytes this keeps the 16-byte reads of a quarter warp (two
// tokens x four lanes) on distinct banks.
__device__ __forceinline__ int x_unit(int J) { return J ^ (((J >> 3) & 1) << 1); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kThreads, 2) mma_kernel(MmaParams p) {
    extern __shared__ __align__(128) uint8_t xs[];
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int tile = blockIdx.x, slice = blockIdx.y;
    const int g0 = slice * p.slice_groups;
    const int g1 = min(p.G, g0 + p.slice_groups);
    const int ng = g1 - g0;

    const int ra = tile * kTileRows + warp * 16 + g;  // rows of this lane
    const int rb = ra + 8;
    const bool va = ra < p.N, vb = rb < p.N;
    const uint32_t *wa_row = p.qw + (size_t)(va ? ra : 0) * p.KW + 4 * c;
    const uint32_t *wb_row = p.qw + (size_t)(vb ? rb : 0) * p.KW + 4 * c;
    const __half *sa_row = p.scales + (size_t)(va ? ra : 0) * p.G;
    const __half *sb_row = p.scales + (size_t)(vb ? rb : 0) * p.G;
    const uint32_t *za_row = p.zeros + (size_t)(va ? ra : 0) * p.ZW;
    const uint32_t *zb_row = p.zeros + (size_t)(vb ? rb : 0) * p.ZW;

    // ---- weights, scales, zeros of the first kDepth groups: in flight while
    // x is staged
    uint4 wa[kDepth], wb[kDepth];
    float sa[kDepth], sb[kDepth];
    uint32_t za[kDepth], zb[kDepth];
    auto load = [&](int d, int i) {
        const int gg = g0 + i;
        wa[d] = va ? dev::ld_stream(wa_row + (size_t)gg * 16) : make_uint4(0, 0, 0, 0);
        wb[d] = vb ? dev::ld_stream(wb_row + (size_t)gg * 16) : make_uint4(0, 0, 0, 0);
        sa[d] = va ? __half2float(sa_row[gg]) : 0.f;
        sb[d] = vb ? __half2float(sb_row[gg]) : 0.f;
        za[d] = va ? __ldg(za_row + (gg >> 3)) : 0u;
        zb[d] = vb ? __ldg(zb_row + (gg >> 3)) : 0u;
    };
#pragma unroll
    for (int d = 0; d < kDepth; ++d)
        if (d < ng) load(d, d);

    // ---- stage x[:, slice] in pair order
    {
        const int nunits = ng * (kGroup / 8);
        const int k0 = g0 * kGroup;
        for (int i = threadIdx.x; i < p.M * nunits; i += kThreads) {
            const int t = i / nunits, J = i - t * nunits;
            const uint4 v =
                __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)t * p.K + k0 + 8 * J));
            *reinterpret_cast<uint4 *>(xs + (size_t)t * p.xstride + 16 * x_unit(J)) =
                dev::pair_order(v);
        }
    }
    __syncthreads();

    const bool has_x = g < p.M;
    const uint8_t *xrow = xs + (size_t)(has_x ? g : 0) * p.xstride;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};

    for (int i0 = 0; i0 < ng; i0 += kDepth) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int i = i0 + d;
            if (i < ng) {
                const int gg = g0 + i;
                const dev::ZeroPair zA = dev::zero_pair((za[d] >> (4 * (gg & 7))) & 0xfu);
                const dev::ZeroPair zB = dev::zero_pair((zb[d] >> (4 * (gg & 7))) & 0xfu);
                const uint32_t wA[4] = {wa[d].x, wa[d].y, wa[d].z, wa[d].w};
                const uint32_t wB[4] = {wb[d].x, wb[d].y, wb[d].z, wb[d].w};
                const float sA = sa[d], sB = sb[d];
                if (i + kDepth < ng) load(d, i + kDepth);
                float dacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint32_t qa[4], qb[4];
                    dev::unpack_word(wA[u], zA, qa);
                    dev::unpack_word(wB[u], zB, qb);
                    uint4 xv = make_uint4(0, 0, 0, 0);
                    if (has_x)
                        xv = *reinterpret_cast<const uint4 *>(xrow + 16 * x_unit(16 * i + 4 * c + u));
                    const uint32_t a0[4] = {qa[0], qb[0], qa[1], qb[1]};
                    const uint32_t a1[4] = {qa[2], qb[2], qa[3], qb[3]};
                    mma16816(dacc, a0, xv.x, xv.y);
                    mma16816(dacc, a1, xv.z, xv.w);
                }
                acc[0] = fmaf(sA, dacc[0], acc[0]);
                acc[1] = fmaf(sA, dacc[1], acc[1]);
                acc[2] = fmaf(sB, dacc[2], acc[2]);
                acc[3] = fmaf(sB, dacc[3], acc[3]);
            }
        }
    }

    // acc[0..1]: row ra, tokens 2c, 2c+1; acc[2..3]: row rb, tokens 2c, 2c+1
    const int t0 = 2 * c, t1 = 2 * c + 1;
    if (p.S == 1) {
        if (va && t0 < p.M) p.y[(size_t)t0 * p.N + ra] = __float2half_rn(acc[0]);
        if (va && t1 < p.M) p.y[(size_t)t1 * p.N + ra] = __float2half_rn(acc[1]);
        if (vb && t0 < p.M) p.y[(size_t)t0 * p.N + rb] = __float2half_rn(acc[2]);
        if (vb && t1 < p.M) p.y[(size_t)t1 * p.N + rb] = __float2half_rn(acc[3]);
        return;
    }
    float *part = p.partials + (size_t)slice * p.M * p.N;
    if (va && t0 < p.M) part[(size_t)t0 * p.N + ra] = acc[0];
    if (va && t1 < p.M) part[(size_t)t1 * p.N + ra] = acc[1];
    if (vb && t0 < p.M) part[(size_t)t0 * p.N + rb] = acc[2];
    if (vb && t1 < p.M) part[(size_t)t1 * p.N + rb] = acc[3];
    // publish the partials, count the arrival; the last CTA of the tile sums
    // all slices in slice order
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(p.counters + tile, 1u);
        s_last = (prev == (unsigned)(p.S - 1));
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        const int row0 = tile * kTileRows;
        const int nrows = min(kTileRows, p.N - row0);
        for (int idx = threadIdx.x; idx < p.M * nrows; idx += kThreads) {
            const int t = idx / nrows;
            const int n = row0 + (idx - t * nrows);
            float sum = 0.f;
            for (int s2 = 0; s2 < p.S; ++s2)
                sum += __ldcg(p.partials + ((size_t)s2 * p.M + t) * p.N + n);
            p.y[(size_t)t * p.N + n] = __float2half_rn(sum);
        }
        if (threadIdx.x == 0) p.counters[tile] = 0u;  // ready for the next launch
    }
}

int xstride_for(int slice_groups) { return slice_groups * kGroup * 2 + 16; }

}  // namespace

MmaPlan plan_mma(int M, int N, int K, int split, const DeviceInfo &dev) {
    MmaPlan pl{};
    pl.M = M;
    const int G = K / kGroup;
    pl.n_tiles = (N + kTileRows - 1) / kTileRows;
    // largest slice whose staged x fits the budget
    int max_groups = (kXBudget / M - 16) / (kGroup * 2);
    if (max_groups < 1) max_groups = 1;
    int S = (G + max_groups - 1) / max_groups;
    if (split == 0 && S > 1) {
        pl.ok = false;
        return pl;
    }
    if (split != 0) {
        // two resident CTAs per SM; split K until the tiles cover two waves,
        // keeping at least kMinSliceGroups groups per slice
        const int want = 4 * dev.sm_count;
        if (pl.n_tiles * S < want) {
            int s_fill = (want + pl.n_tiles - 1) / pl.n_tiles;
            int s_cap = G / kMinSliceGroups > 0 ? G / kMinSliceGroups : 1;
            if (s_fill > s_cap) s_fill = s_cap;
            if (s_fill > S) S = s_fill;
        }
        if (split == 1 && S < 2 && G >= 2) S = 2;
    }
    pl.slice_groups = (G + S - 1) / S;
    pl.S = (G + pl.slice_groups - 1) / pl.slice_groups;
    pl.smem_bytes = M * xstride_for(pl.slice_groups);
    pl.ws_bytes = pl.S > 1 ? (size_t)pl.S * M * N * sizeof(float) : 0;
    pl.ok = true;
    return pl;
}

cudaError_t launch_mma(const LinearArgs &a, const MmaPlan &plan, const Workspace &ws,
                       cudaStream_t stream) {
    MmaParams p;
    p.x = a.x;
    p.qw = a.qw;
    p.scales = a.scales;
    p.zeros = a.zeros;
    p.y = a.y;
    p.partials = ws.partials;
    p.counters = ws.counters;
    p.N = a.N;
    p.K = a.K;
    p.G = a.K / kGroup;
    p.ZW = (p.G + 7) / 8;
    p.KW = a.K / 8;
    p.M = a.M;
    p.S = plan.S;
    p.slice_groups = plan.slice_groups;
    p.xstride = xstride_for(plan.slice_groups);
    dim3 grid(plan.n_tiles, plan.S);
    mma_kernel<<<grid, kThreads, plan.smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t mma_init(const DeviceInfo &dev) {
    int dyn = kXBudget + 1024;
    if (dyn > dev.max_smem_optin - 1024) dyn = dev.max_smem_optin - 1024;
    return cudaFuncSetAttribute(mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

}  // namespace w4a16
