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
    const uint32_t *qa, *qb;  // weights of the next group to copy (lane's 16 bytes)
    uintptr_t meta;           // byte address: scale element, or zeros word, of that group
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
    t.meta = (c < 2) ? (uintptr_t)(p.scales + im * p.G + g0)
                     : (uintptr_t)(p.zeros + im * p.ZW + (g0 >> 3));
    t.bytes_a = va ? 16u : 0u;
    t.bytes_b = vb ? 16u : 0u;
    t.bytes_m = ((c & 1) ? vb : va) ? 4u : 0u;
    return t;
}

__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 3) mma_kernel(MmaParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;                   // [warp][stage][kStageBytes]
    uint8_t *xs = smem + kRingBytes;        // staged x, then 256 zero bytes
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    W4A16_MMA_TR_AT(4 * kTraceSteps + 1);  // kernel start
    // the next kernel in the stream may be scheduled as SMs free up; it waits
    // for this grid to finish before it touches anything this grid writes
    grid_dependents_launch();
    const int slice = blockIdx.x % p.S;
    const int q = blockIdx.x / p.S;         // index among the CTAs of this slice
    const int g0 = slice * p.slice_groups;
    const int ng = min(p.G, g0 + p.slice_groups) - g0;
    // this warp's strips: first, first + stride, ...
    const int first = q * kWarps + warp;
    const int stride = p.ctas_per_slice * kWarps;
    const int my_strips = first < p.n_strips ? (p.n_strips - 1 - first) / stride + 1 : 0;
    uint8_t *zero_x = xs + (size_t)p.M * p.xstride;                     // 256 zero bytes
    float *sums = reinterpret_cast<float *>(zero_x + 256);              // [ng][8][2]
    uint8_t *wring = ring + (size_t)warp * kDepth * kStageBytes;
    const uint32_t wring_u32 = dev::smem_u32(wring);

    // ---- copy stream: one step = one group of one strip; the issue cursor
    // runs kDepth steps ahead of the consume cursor.  Weights, scales and
    // zeros are parameters (never written by a preceding kernel), so the
    // stream starts before the grid-dependency wait.
    int is_k = 0, is_i = 0, is_slot = 0;
    StripSrc src = strip_src(p, first, g, c, g0);
    const uint32_t dst_w = wring_u32 + lane * 32;
    const uint32_t dst_m = wring_u32 + kStageW + g * 16 + 4 * c;
    auto issue_next = [&]() {
        if (is_k < my_strips) {
            const uint32_t so = is_slot * kStageBytes;
            cp16(dst_w + so, src.qa, src.bytes_a);
            cp16(dst_w + so + 16, src.qb, src.bytes_b);
            // c < 2: the aligned word holding the scale (scales are 2-byte
            // aligned); c >= 2: the zeros word of the group
            cp4(dst_m + so, (const void *)(c < 2 ? (src.meta & ~(uintptr_t)3) : src.meta),
                src.bytes_m);
            src.qa += 16;
            src.qb += 16;
            src.meta += c < 2 ? 2 : (((g0 + is_i + 1) & 7) == 0 ? 4 : 0);
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

    // ---- from here on: x, y and the split-K workspace may belong to the
    // preceding kernel
    grid_dependency_wait();

    // ---- stage x[:, slice] in pair order, and each (group, token)'s sums of
    // x over even and over odd k: the 16 lanes of a half warp hold the 16
    // units of one group of one token and add theirs with shuffles
    {
        const int nunits = ng * (kGroup / 8);
        const int xtotal = p.M * nunits;  // a multiple of 16
        const int k0 = g0 * kGroup;
        for (int base = warp * 32; base < xtotal; base += kThreads) {
            const int i = base + lane;
            const bool valid = i < xtotal;
            const int t = i / nunits, J = i - t * nunits;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (valid) {
                v = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)t * p.K + k0 + 8 * J));
                *reinterpret_cast<uint4 *>(xs + (size_t)t * p.xstride + 16 * x_unit(J)) =
                    dev::pair_order(v);
            }
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
        // tokens M..7 have no x: their sums are zero; so is the zero block
        for (int i = threadIdx.x; i < ng * (8 - p.M); i += kThreads) {
            const int gi = i / (8 - p.M), t = p.M + i % (8 - p.M);
            sums[(gi * 8 + t) * 2] = 0.f;
            sums[(gi * 8 + t) * 2 + 1] = 0.f;
        }
        if (threadIdx.x < 16) reinterpret_cast<uint4 *>(zero_x)[threadIdx.x] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();

    W4A16_MMA_TR_AT(4 * kTraceSteps);  // prologue done (x staged, sums computed)
    const bool has_x = g < p.M;
    const uint8_t *xrow = xs + (size_t)(has_x ? g : 0) * p.xstride;
    // unit of word u of this lane's chunk in a group: x_unit(4c + u)
    const int xo0 = 16 * x_unit(4 * c + 0), xo1 = 16 * x_unit(4 * c + 1);
    const int xo2 = 16 * x_unit(4 * c + 2), xo3 = 16 * x_unit(4 * c + 3);
    const uint8_t *cs_base = wring + lane * 32;
    const uint8_t *cs_meta = wring + kStageW + g * 16;
    int cs_slot = 0;
    int jstep = 0;

    for (int k = 0; k < my_strips; ++k) {
        const int strip = first + k * stride;
        const int ra = strip * 16 + g, rb = ra + 8;
        const bool va = ra < p.N, vb = rb < p.N;
        // shift that brings group g0's scale to the low half of its word; it
        // flips by 16 bits from one group to the next
        uint32_t sha = 8u * (uint32_t)((uintptr_t)(p.scales + (size_t)(va ? ra : 0) * p.G + g0) & 2);
        uint32_t shb = 8u * (uint32_t)((uintptr_t)(p.scales + (size_t)(vb ? rb : 0) * p.G + g0) & 2);
        uint32_t zsh = 4u * (uint32_t)(g0 & 7);  // nibble of the group in its zeros word
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < ng; ++i) {
            W4A16_MMA_TR(0, jstep);
            cp_wait<kDepth - 1>();  // this lane's copies of the step have landed
            __syncwarp();           // ... and those of the other lanes of the warp
            W4A16_MMA_TR(1, jstep);
            const uint32_t so = cs_slot * kStageBytes;
            cs_slot = cs_slot + 1 == kDepth ? 0 : cs_slot + 1;
            const uint4 wa = *reinterpret_cast<const uint4 *>(cs_base + so);
            const uint4 wb = *reinterpret_cast<const uint4 *>(cs_base + so + 16);
            const uint4 meta = *reinterpret_cast<const uint4 *>(cs_meta + so);
            // A fragments straight from the unpack: MMA 2u takes the pairs
            // (q0,q4) (q1,q5) of word u, MMA 2u+1 the pairs (q2,q6) (q3,q7);
            // rows g and g + 8 interleave as the fragment layout wants
            uint32_t a[8][4];
            const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
            const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t xa = wA[u], xb = wB[u], xa8 = xa >> 8, xb8 = xb >> 8;
                a[2 * u][0] = dev::lop3_and_or(xa, 0x000f000fu, 0x64006400u);
                a[2 * u][1] = dev::lop3_and_or(xb, 0x000f000fu, 0x64006400u);
                a[2 * u][2] = dev::lop3_and_or(xa, 0x00f000f0u, 0x54005400u);
                a[2 * u][3] = dev::lop3_and_or(xb, 0x00f000f0u, 0x54005400u);
                a[2 * u + 1][0] = dev::lop3_and_or(xa8, 0x000f000fu, 0x64006400u);
                a[2 * u + 1][1] = dev::lop3_and_or(xb8, 0x000f000fu, 0x64006400u);
                a[2 * u + 1][2] = dev::lop3_and_or(xa8, 0x00f000f0u, 0x54005400u);
                a[2 * u + 1][3] = dev::lop3_and_or(xb8, 0x00f000f0u, 0x54005400u);
            }
            // scale halves and zero nibbles of the two rows, decoded before
            // the slot is released
            const float sA = __half2float(__ushort_as_half((unsigned short)(meta.x >> sha)));
            const float sB = __half2float(__ushort_as_half((unsigned short)(meta.y >> shb)));
            const uint32_t zA = (meta.z >> zsh) & 0xfu, zB = (meta.w >> zsh) & 0xfu;
            sha ^= 16u;
            shb ^= 16u;
            zsh = (zsh + 4u) & 31u;
            // the slot's values are in registers in every lane: refill it
            __syncwarp();
            issue_next();
            // 1024 + z and 64 + z as exact fp32 (z in the mantissa)
            const float hA = __uint_as_float(0x44800000u | (zA << 13));
            const float lA = __uint_as_float(0x42800000u | (zA << 17));
            const float hB = __uint_as_float(0x44800000u | (zB << 13));
            const float lB = __uint_as_float(0x42800000u | (zB << 17));
            const float4 sx = *reinterpret_cast<const float4 *>(sums + (i * 8 + 2 * c) * 2);
            const uint8_t *xg = has_x ? xrow + 256 * i : zero_x;
            const uint4 x0 = *reinterpret_cast<const uint4 *>(xg + (has_x ? xo0 : 0));
            const uint4 x1 = *reinterpret_cast<const uint4 *>(xg + (has_x ? xo1 : 0));
            const uint4 x2 = *reinterpret_cast<const uint4 *>(xg + (has_x ? xo2 : 0));
            const uint4 x3 = *reinterpret_cast<const uint4 *>(xg + (has_x ? xo3 : 0));
            // two independent accumulator chains (words 0,1 and words 2,3)
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(d0, a[0], x0.x, x0.y);
            mma16816(d1, a[4], x2.x, x2.y);
            mma16816(d0, a[1], x0.z, x0.w);
            mma16816(d1, a[5], x2.z, x2.w);
            mma16816(d0, a[2], x1.x, x1.y);
            mma16816(d1, a[6], x3.x, x3.y);
            mma16816(d0, a[3], x1.z, x1.w);
            mma16816(d1, a[7], x3.z, x3.w);
            W4A16_MMA_TR(2, jstep);
            // sum (q - z) x = D - (1024 + z) S_even - (64 + z) S_odd, per token
            // (sx = S_even(t0), S_odd(t0), S_even(t1), S_odd(t1))
            float v;
            v = fmaf(-hA, sx.x, d0[0] + d1[0]);
            v = fmaf(-lA, sx.y, v);
            acc[0] = fmaf(sA, v, acc[0]);
            v = fmaf(-hA, sx.z, d0[1] + d1[1]);
            v = fmaf(-lA, sx.w, v);
            acc[1] = fmaf(sA, v, acc[1]);
            v = fmaf(-hB, sx.x, d0[2] + d1[2]);
            v = fmaf(-lB, sx.y, v);
            acc[2] = fmaf(sB, v, acc[2]);
            v = fmaf(-hB, sx.z, d0[3] + d1[3]);
            v = fmaf(-lB, sx.w, v);
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
        // count this slice's arrival for the strip with one release-acquire
        // atomic after a warp barrier (the barrier orders the other lanes'
        // partial writes before it); the warp that arrives last sums the
        // slices in slice order.  No warp waits for another.
        __syncwarp();
        unsigned prev = 0;
        if (lane == 0)
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                         : "=r"(prev)
                         : "l"(p.counters + strip)
                         : "memory");
        prev = __shfl_sync(0xffffffffu, prev, 0);
        __syncwarp();  // the other lanes' reads below come after lane 0's acquire
        if (prev == (unsigned)(p.S - 1)) {
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
            __syncwarp();
            if (lane == 0) p.counters[strip] = 0u;  // ready for the next launch
        }
    }
    cp_wait<0>();
}

int xstride_for(int slice_groups) { return slice_groups * kGroup * 2 + 16; }

int smem_for(int M, int slice_groups) {
    return kRingBytes + M * xstride_for(slice_groups) + 256 +
           slice_groups * 8 * 2 * (int)sizeof(float);
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
    // programmatic dependent launch: the grid may start while the previous
    // kernel in the stream drains; the kernel waits for it (griddepcontrol)
    // before touching x, y or the workspace
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mma_kernel, p);
}

cudaError_t mma_init(const DeviceInfo &dev) {
    int dyn = smem_for(1, kMaxSliceGroups);
    const int dyn8 = kRingBytes + kXBudget + 256 + kMaxSliceGroups * 64;
    if (dyn8 > dyn) dyn = dyn8;
    if (dyn > dev.max_smem_optin - 1024) dyn = dev.max_smem_optin - 1024;
    return cudaFuncSetAttribute(mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

}  // namespace w4a16
