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
//   * lane (g = lane/4, c = lane%4) works on row g and row g + 8 of its
//     warp's tile: the 32 k values 32c .. 32c+31 of each 128-wide group.  The
//     lane copies its 2 x 16 bytes of weights of a group with cp.async into
//     its own slot of a kDepth-deep ring in shared memory (a warp's copy
//     instruction reads 8 rows x 64 contiguous bytes, with a 256-byte L2
//     fetch), and one of the four 32-bit words holding the scales and zeros of
//     its row pair (the four lanes of a row pair share them), so kDepth groups
//     are in flight per lane without holding registers;
//   * CTAs are persistent: a CTA owns one K slice, stages that slice of x
//     once, then walks its tiles with one continuous copy stream;
//   * the unpack is one lop3 per pair of nibbles: a nibble OR-ed into the
//     fp16 constant 1024 (even k) or, four bits higher, 64 (odd k) gives the
//     exact fp16 values (1024 + q) and (64 + q), in the pairs (q0,q4) (q1,q5)
//     (q2,q6) (q3,q7).  These are the A fragment registers as they come: the
//     MMA's k slots 2c, 2c+1, 2c+8, 2c+9 stand for the actual k values k0,
//     k4, k1, k5 (and k2, k6, k3, k7 for the second MMA of the word).  The B
//     fragment must use the same order, so x is staged once per CTA in pair
//     order (x0,x4,x1,x5,...) and a lane reads its two MMAs' B registers with
//     one 16-byte load;
//   * the 8 MMAs of a group accumulate D = sum (bias_k + q) * x into a fresh
//     fp32 accumulator (products exact); the zero point and the biases are
//     removed per group with the token's sums of x over even and odd k,
//     computed once per CTA:
//         sum_k (q - z) x = D - (1024 + z) * S_even - (64 + z) * S_odd,
//     and the group's fp32 scale multiplies that into the running sums.  This
//     takes the zero subtraction out of the per-weight work (the unpack costs
//     5 instructions per 8 weights); integer-valued cases stay exact;
//   * split K: fp32 partials and a last-arriving-CTA reduction in slice order,
//     as on the other rungs (deterministic, no CTA waits for another).
#include "w4a16_device.cuh"
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kDepth = 4;               // groups in flight per lane
// one ring stage of one warp: 32 lanes x 32 bytes of weights, then 8 row
// pairs x 4 words of metadata (scale word of row g, of row g+8, zeros word of
// row g, of row g+8)
constexpr int kStageW = 32 * 32;
constexpr int kStageBytes = kStageW + 8 * 16;
constexpr int kRingBytes = kWarps * kDepth * kStageBytes;  // 36 KB
constexpr int kXBudget = 32 * 1024;     // staged activations per CTA
constexpr int kMinSliceGroups = 4;
constexpr int kMaxSliceGroups = 256;

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
    int n_strips, ctas_per_slice;  // 16-row strips; persistent CTAs per slice
    int xstride;  // bytes per staged token row
};

// Optional section timers (build with -DW4A16_TRACE): warp 0 of CTA 0 records
// the SM cycle counter at each step of its first kTraceSteps groups.
#ifdef W4A16_TRACE
constexpr int kTraceSteps = 64;
__device__ long long g_trace_mma[4 * kTraceSteps + 4];
#define W4A16_MMA_TR(ev, j)                                                          \
    do {                                                                             \
        if (blockIdx.x == 0 && threadIdx.x == 0 && (j) < kTraceSteps)                \
            g_trace_mma[(ev) * kTraceSteps + (j)] = clock64();                       \
    } while (0)
#define W4A16_MMA_TR_AT(slot)                                                        \
    do {                                                                             \
        if (blockIdx.x == 0 && threadIdx.x == 0) g_trace_mma[slot] = clock64();      \
    } while (0)
#else
#define W4A16_MMA_TR(ev, j) \
    do {                    \
    } while (0)
#define W4A16_MMA_TR_AT(slot) \
    do {                      \
    } while (0)
#endif

// Staged x: 16-byte unit J of a token row (8 activations, pair order) lives
// at unit J ^ (bit 3 of J moved to bit 1).  With a row stride of 16 (mod 128)
// bytes the 16-byte reads of a quarter warp (two tokens x four lanes) fall on
// distinct banks.
__device__ __forceinline__ int x_unit(int J) { return J ^ (((J >> 3) & 1) << 1); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// global -> shared copies that bypass registers; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Unpack one word with the biases left in: four fp16 pairs
// (1024+q0, 1024+q4) (64+q1, 64+q5) (1024+q2, 1024+q6) (64+q3, 64+q7).
__device__ __forceinline__ void unpack_biased(uint32_t w, uint32_t (&d)[4]) {
    const uint32_t w8 = w >> 8;
    d[0] = dev::lop3_and_or(w, 0x000f000fu, 0x64006400u);
    d[1] = dev::lop3_and_or(w, 0x00f000f0u, 0x54005400u);
    d[2] = dev::lop3_and_or(w8, 0x000f000fu, 0x64006400u);
    d[3] = dev::lop3_and_or(w8, 0x00f000f0u, 0x54005400u);
}

// One lane's copy sources for one 16-row strip: its two weight rows, and the
// one metadata item it copies for its row pair (c = 0: scale of row g, 1:
// scale of row g+8, 2: zeros word of row g, 3: zeros word of row g+8).
struct StripSrc {
    const uint32_t *qa, *qb;  // weights at group g0 (lane's 16 bytes)
    const uint8_t *meta;      // scale element at group g0, or the zeros row
    uint32_t bytes_a, bytes_b, bytes_m;
};

__device__ __forceinline__ StripSrc strip_src(const MmaParams &p, int strip, int g, int c, int g0) {
    StripSrc t;
    const int ra = strip * 16 + g, rb = ra + 8;
    const bool va = ra < p.N, vb = rb < p.N;
    const size_t ia = (size_t)(va ? ra : 0), ib = (size_t)(vb ? rb : 0);
    t.qa = p.qw + ia * p.KW + (size_t)g0 * 16 + 4 * c;
    t.qb = p.qw + ib * p.KW + (size_t)g0 * 16 + 4 * c;
    const size_t im = (c & 1) ? ib : ia;
    t.meta = (c < 2) ? reinterpret_cast<const uint8_t *>(p.scales + im * p.G + g0)
                     : reinterpret_cast<const uint8_t *>(p.zeros + im * p.ZW);
    t.bytes_a = va ? 16u : 0u;
    t.bytes_b = vb ? 16u : 0u;
    t.bytes_m = ((c & 1) ? vb : va) ? 4u : 0u;
    return t;
}

__global__ void __launch_bounds__(kThreads, 3) mma_kernel(MmaParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;                   // [warp][stage][kStageBytes]
    uint8_t *xs = smem + kRingBytes;        // staged x
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    W4A16_MMA_TR_AT(4 * kTraceSteps + 1);  // kernel start
    const int slice = blockIdx.x % p.S;
    const int q = blockIdx.x / p.S;         // index among the CTAs of this slice
    const int g0 = slice * p.slice_groups;
    const int ng = min(p.G, g0 + p.slice_groups) - g0;
    // this warp's strips: first, first + stride, ...
    const int first = q * kWarps + warp;
    const int stride = p.ctas_per_slice * kWarps;
    const int my_strips = first < p.n_strips ? (p.n_strips - 1 - first) / stride + 1 : 0;
    float *sums = reinterpret_cast<float *>(xs + (size_t)p.M * p.xstride);  // [ng][8][2]
    uint8_t *wring = ring + (size_t)warp * kDepth * kStageBytes;
    const uint32_t wring_u32 = dev::smem_u32(wring);

    // ---- the first pieces of x this thread stages are requested before the
    // weight stream starts, so they are not queued behind it
    const int nunits = ng * (kGroup / 8);
    const int xtotal = p.M * nunits;  // a multiple of 16
    const int k0 = g0 * kGroup;
    uint4 xfirst = make_uint4(0, 0, 0, 0);
    {
        const int i = warp * 32 + lane;
        if (i < xtotal) {
            const int t = i / nunits, J = i - t * nunits;
            xfirst = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)t * p.K + k0 + 8 * J));
        }
    }

    // ---- copy stream: one step = one group of one strip; the issue cursor
    // runs kDepth steps ahead of the consume cursor
    int is_k = 0, is_i = 0, is_slot = 0;
    StripSrc src = strip_src(p, first, g, c, g0);
    auto issue_next = [&]() {
        if (is_k < my_strips) {
            const uint32_t st = wring_u32 + is_slot * kStageBytes;
            cp16(st + lane * 32, src.qa + is_i * 16, src.bytes_a);
            cp16(st + lane * 32 + 16, src.qb + is_i * 16, src.bytes_b);
            // c < 2: the aligned word holding the scale (scales are 2-byte
            // aligned); c >= 2: the zeros word of the group
            const uint8_t *m = c < 2 ? (const uint8_t *)((uintptr_t)(src.meta + 2 * is_i) &
                                                         ~(uintptr_t)3)
                                     : src.meta + 4 * ((g0 + is_i) >> 3);
            cp4(st + kStageW + g * 16 + 4 * c, m, src.bytes_m);
            is_slot = is_slot + 1 == kDepth ? 0 : is_slot + 1;
            if (++is_i == ng) {
                is_i = 0;
                if (++is_k < my_strips) src = strip_src(p, first + is_k * stride, g, c, g0);
            }
        }
        cp_commit();
    };
#pragma unroll
    for (int j = 0; j < kDepth; ++j) issue_next();

    // ---- stage x[:, slice] in pair order, and each (group, token)'s sums of
    // x over even and over odd k: the 16 lanes of a half warp hold the 16
    // units of one group of one token and add theirs with shuffles
    for (int base = warp * 32; base < xtotal; base += kThreads) {
        const int i = base + lane;
        const bool valid = i < xtotal;
        const int t = i / nunits, J = i - t * nunits;
        uint4 v = xfirst;
        if (base != warp * 32)
            v = valid ? __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)t * p.K + k0 + 8 * J))
                      : make_uint4(0, 0, 0, 0);
        if (valid)
            *reinterpret_cast<uint4 *>(xs + (size_t)t * p.xstride + 16 * x_unit(J)) =
                dev::pair_order(v);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
        const float2 e = __half22float2(*reinterpret_cast<const __half2 *>(&v.z));
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&v.w));
        float se = (a.x + b.x) + (e.x + f.x);  // k % 8 = 0, 2, 4, 6
        float so = (a.y + b.y) + (e.y + f.y);  // k % 8 = 1, 3, 5, 7
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {
            se += __shfl_xor_sync(0xffffffffu, se, off);
            so += __shfl_xor_sync(0xffffffffu, so, off);
        }
        if (valid && (J & 15) == 0) {
            sums[((J >> 4) * 8 + t) * 2] = se;
            sums[((J >> 4) * 8 + t) * 2 + 1] = so;
        }
    }
    // tokens M..7 have no x: their sums are zero
    for (int i = threadIdx.x; i < ng * (8 - p.M); i += kThreads) {
        const int gi = i / (8 - p.M), t = p.M + i % (8 - p.M);
        sums[(gi * 8 + t) * 2] = 0.f;
        sums[(gi * 8 + t) * 2 + 1] = 0.f;
    }
    __syncthreads();

    W4A16_MMA_TR_AT(4 * kTraceSteps);  // prologue done (x staged, sums computed)
    const bool has_x = g < p.M;
    const uint8_t *xrow = xs + (size_t)(has_x ? g : 0) * p.xstride;
    int jstep = 0;
    const int xo0 = 16 * x_unit(4 * c + 0), xo1 = 16 * x_unit(4 * c + 1);
    const int xo2 = 16 * x_unit(4 * c + 2), xo3 = 16 * x_unit(4 * c + 3);
    int cs_slot = 0;

    for (int k = 0; k < my_strips; ++k) {
        const int strip = first + k * stride;
        const int ra = strip * 16 + g, rb = ra + 8;
        const bool va = ra < p.N, vb = rb < p.N;
        // byte offset (0 or 2) of group g0's scale inside its aligned word
        const uint32_t spa =
            (uint32_t)((uintptr_t)(p.scales + (size_t)(va ? ra : 0) * p.G + g0) & 2);
        const uint32_t spb =
            (uint32_t)((uintptr_t)(p.scales + (size_t)(vb ? rb : 0) * p.G + g0) & 2);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < ng; ++i) {
            const int gg = g0 + i;
            W4A16_MMA_TR(0, jstep);
            cp_wait<kDepth - 1>();  // this lane's copies of the step have landed
            __syncwarp();           // ... and those of the other lanes of the warp
            W4A16_MMA_TR(1, jstep);
            const uint8_t *st = wring + cs_slot * kStageBytes;
            cs_slot = cs_slot + 1 == kDepth ? 0 : cs_slot + 1;
            const uint4 wa = *reinterpret_cast<const uint4 *>(st + lane * 32);
            const uint4 wb = *reinterpret_cast<const uint4 *>(st + lane * 32 + 16);
            const uint4 meta = *reinterpret_cast<const uint4 *>(st + kStageW + g * 16);
            // unpack all eight words and decode the metadata: once every lane
            // has its values in registers the slot can be refilled
            uint32_t qa[4][4], qb[4][4];
            unpack_biased(wa.x, qa[0]);
            unpack_biased(wa.y, qa[1]);
            unpack_biased(wa.z, qa[2]);
            unpack_biased(wa.w, qa[3]);
            unpack_biased(wb.x, qb[0]);
            unpack_biased(wb.y, qb[1]);
            unpack_biased(wb.z, qb[2]);
            unpack_biased(wb.w, qb[3]);
            const float sA = __half2float(__ushort_as_half(
                (unsigned short)(meta.x >> (8 * ((spa + 2 * (uint32_t)i) & 2)))));
            const float sB = __half2float(__ushort_as_half(
                (unsigned short)(meta.y >> (8 * ((spb + 2 * (uint32_t)i) & 2)))));
            const float zA = (float)((meta.z >> (4 * (gg & 7))) & 0xfu);
            const float zB = (float)((meta.w >> (4 * (gg & 7))) & 0xfu);
            __syncwarp();
            issue_next();
            const float4 sx = *reinterpret_cast<const float4 *>(sums + (i * 8 + 2 * c) * 2);
            const uint8_t *xg = xrow + 256 * i;
            uint4 xv[4];
            xv[0] = has_x ? *reinterpret_cast<const uint4 *>(xg + xo0) : make_uint4(0, 0, 0, 0);
            xv[1] = has_x ? *reinterpret_cast<const uint4 *>(xg + xo1) : make_uint4(0, 0, 0, 0);
            xv[2] = has_x ? *reinterpret_cast<const uint4 *>(xg + xo2) : make_uint4(0, 0, 0, 0);
            xv[3] = has_x ? *reinterpret_cast<const uint4 *>(xg + xo3) : make_uint4(0, 0, 0, 0);
            // two independent accumulator chains (words 0,1 and 2,3)
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint32_t a0[4] = {qa[u][0], qb[u][0], qa[u][1], qb[u][1]};
                const uint32_t a1[4] = {qa[u][2], qb[u][2], qa[u][3], qb[u][3]};
                const uint32_t a2[4] = {qa[u + 2][0], qb[u + 2][0], qa[u + 2][1], qb[u + 2][1]};
                const uint32_t a3[4] = {qa[u + 2][2], qb[u + 2][2], qa[u + 2][3], qb[u + 2][3]};
                mma16816(d0, a0, xv[u].x, xv[u].y);
                mma16816(d1, a2, xv[u + 2].x, xv[u + 2].y);
                mma16816(d0, a1, xv[u].z, xv[u].w);
                mma16816(d1, a3, xv[u + 2].z, xv[u + 2].w);
            }
            W4A16_MMA_TR(2, jstep);
            const float dacc[4] = {d0[0] + d1[0], d0[1] + d1[1], d0[2] + d1[2], d0[3] + d1[3]};
            // sum (q - z) x = D - (1024 + z) S_even - (64 + z) S_odd, per token
            // (sx = S_even(t0), S_odd(t0), S_even(t1), S_odd(t1))
            float v;
            v = fmaf(-(1024.f + zA), sx.x, dacc[0]);
            v = fmaf(-(64.f + zA), sx.y, v);
            acc[0] = fmaf(sA, v, acc[0]);
            v = fmaf(-(1024.f + zA), sx.z, dacc[1]);
            v = fmaf(-(64.f + zA), sx.w, v);
            acc[1] = fmaf(sA, v, acc[1]);
            v = fmaf(-(1024.f + zB), sx.x, dacc[2]);
            v = fmaf(-(64.f + zB), sx.y, v);
            acc[2] = fmaf(sB, v, acc[2]);
            v = fmaf(-(1024.f + zB), sx.z, dacc[3]);
            v = fmaf(-(64.f + zB), sx.w, v);
            acc[3] = fmaf(sB, v, acc[3]);
            W4A16_MMA_TR(3, jstep);
            ++jstep;
        }

        // ---- end of strip: acc[0..1] row ra, tokens 2c, 2c+1; acc[2..3] row rb
        const int t0 = 2 * c, t1 = 2 * c + 1;
        if (p.S == 1) {
            if (va && t0 < p.M) p.y[(size_t)t0 * p.N + ra] = __float2half_rn(acc[0]);
            if (va && t1 < p.M) p.y[(size_t)t1 * p.N + ra] = __float2half_rn(acc[1]);
            if (vb && t0 < p.M) p.y[(size_t)t0 * p.N + rb] = __float2half_rn(acc[2]);
            if (vb && t1 < p.M) p.y[(size_t)t1 * p.N + rb] = __float2half_rn(acc[3]);
            continue;
        }
        float *part = p.partials + (size_t)slice * p.M * p.N;
        if (va && t0 < p.M) part[(size_t)t0 * p.N + ra] = acc[0];
        if (va && t1 < p.M) part[(size_t)t1 * p.N + ra] = acc[1];
        if (vb && t0 < p.M) part[(size_t)t0 * p.N + rb] = acc[2];
        if (vb && t1 < p.M) part[(size_t)t1 * p.N + rb] = acc[3];
        // publish this slice of the strip and count the arrival; the warp that
        // arrives last sums the slices in slice order (no warp waits)
        __threadfence();
        __syncwarp();
        unsigned prev = 0;
        if (lane == 0) prev = atomicAdd(p.counters + strip, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == (unsigned)(p.S - 1)) {
            __threadfence();
            const int rows[2] = {ra, rb};
            const bool ok[2] = {va, vb};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 2 * c + e;
                    if (ok[h] && t < p.M) {
                        float sum = 0.f;
                        for (int s2 = 0; s2 < p.S; ++s2)
                            sum += __ldcg(p.partials + ((size_t)s2 * p.M + t) * p.N + rows[h]);
                        p.y[(size_t)t * p.N + rows[h]] = __float2half_rn(sum);
                    }
                }
            }
            if (lane == 0) p.counters[strip] = 0u;  // ready for the next launch
        }
    }
    cp_wait<0>();
}

int xstride_for(int slice_groups) { return slice_groups * kGroup * 2 + 16; }

int smem_for(int M, int slice_groups) {
    return kRingBytes + M * xstride_for(slice_groups) + slice_groups * 8 * 2 * (int)sizeof(float);
}

}  // namespace

MmaPlan plan_mma(int M, int N, int K, int split, const DeviceInfo &dev) {
    MmaPlan pl{};
    pl.M = M;
    const int G = K / kGroup;
    pl.n_strips = (N + 15) / 16;
    // largest slice whose staged x fits the budget
    int max_groups = (kXBudget / M - 16) / (kGroup * 2);
    if (max_groups > kMaxSliceGroups) max_groups = kMaxSliceGroups;
    if (max_groups < 1) max_groups = 1;
    const int s_min = (G + max_groups - 1) / max_groups;
    if (split == 0 && s_min > 1) {
        pl.ok = false;
        return pl;
    }
    const int warps = 3 * dev.sm_count * kWarps;  // three persistent CTAs per SM
    // Pick the number of K slices that minimises the steps of the busiest warp
    // (strips per warp x groups per slice), plus a small charge per extra
    // slice for the partial-sum traffic; at least kMinSliceGroups groups per
    // slice.
    int best_S = s_min;
    double best_cost = 1e30;
    int s_hi = split == 0 ? 1 : (G / kMinSliceGroups > s_min ? G / kMinSliceGroups : s_min);
    int s_lo = s_min;
    if (split == 1 && s_lo < 2 && G >= 2) s_lo = 2;
    if (s_hi < s_lo) s_hi = s_lo;
    for (int S = s_lo; S <= s_hi; ++S) {
        const int sg = (G + S - 1) / S;
        const int S_eff = (G + sg - 1) / sg;
        const long long units = (long long)pl.n_strips * S_eff;
        const long long per_warp = (units + warps - 1) / warps;
        const double cost = (double)per_warp * sg + (S_eff > 1 ? 2.0 + 0.5 * S_eff : 0.0);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best_S = S_eff;
        }
    }
    pl.slice_groups = (G + best_S - 1) / best_S;
    pl.S = (G + pl.slice_groups - 1) / pl.slice_groups;
    int per_slice = 3 * dev.sm_count / pl.S;
    const int need = (pl.n_strips + kWarps - 1) / kWarps;  // CTAs to give every strip a warp
    if (per_slice > need) per_slice = need;
    if (per_slice < 1) per_slice = 1;
    pl.ctas_per_slice = per_slice;
    pl.grid = per_slice * pl.S;
    pl.smem_bytes = smem_for(M, pl.slice_groups);
    pl.ws_bytes = pl.S > 1 ? (size_t)pl.S * M * N * sizeof(float) : 0;
    pl.ok = true;
    return pl;
}

#ifdef W4A16_TRACE
extern "C" int w4a16_debug_trace_mma(long long *out, int n) {
    if (n > 4 * kTraceSteps + 4) n = 4 * kTraceSteps + 4;
    return (int)cudaMemcpyFromSymbol(out, g_trace_mma, n * sizeof(long long));
}
#endif

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
    p.n_strips = plan.n_strips;
    p.ctas_per_slice = plan.ctas_per_slice;
    p.xstride = xstride_for(plan.slice_groups);
    mma_kernel<<<plan.grid, kThreads, plan.smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t mma_init(const DeviceInfo &dev) {
    int dyn = smem_for(1, kMaxSliceGroups);
    const int dyn8 = kRingBytes + kXBudget + kMaxSliceGroups * 64;
    if (dyn8 > dyn) dyn = dyn8;
    if (dyn > dev.max_smem_optin - 1024) dyn = dev.max_smem_optin - 1024;
    return cudaFuncSetAttribute(mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

}  // namespace w4a16
