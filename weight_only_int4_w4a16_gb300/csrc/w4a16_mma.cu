// W4A16 small-M rung on the warp-level tensor-core MMA ("mma", "mma_splitk").
//
// Why this rung exists: at M = 2..8 tokens the CUDA-core GEMV needs M fp32
// FMAs per weight and runs out of issue slots well below HBM speed, and a
// tcgen05.mma of M = 128 rows and N <= 64 tokens costs a fixed ~46 cycles per
// 2048 weights whatever N is, which is the HBM rate itself with no slack.
// mma.sync.m16n8k16 takes its A operand from registers: the dequantised
// weights never touch shared or tensor memory, one instruction consumes 256
// weights for up to 8 tokens, and the SM sustains ~0.47 of them per clock.
//
// The method is unchanged (forum.sourcefind.cn thread "vLLM on Hygon Z100",
// sections 四 and 五: stream the packed INT4 weights once for all M rows,
// unpack, subtract the zero, multiply with the fp16 activations, scale per
// group, accumulate in fp32):
//
//   * MMA rows are weight rows n (a warp owns a 16-row strip), MMA columns
//     are the M <= 8 tokens, MMA k runs along K.  Lane (g = lane/4, c =
//     lane%4) works on rows g and g + 8 of the strip and on the 32 k values
//     32c .. 32c+31 of each 128-wide group;
//   * weights move by TMA, one box per warp and stage: 16 rows x 4 groups x
//     64 bytes (4 KB), laid out group-major in shared memory ([group][row][64
//     bytes], so the rows of a group sit 64 bytes apart and a quarter warp's
//     16-byte reads hit distinct banks).  Each row of a box is one 256-byte
//     run of global memory: on GB300 runs of 64 bytes per row (one group per
//     request) stream at well under half the rate of 256-byte runs when
//     thousands of rows are in flight.  The 16 rows' scale and zero words of
//     the stage follow the box (lanes copy them with cp.async); the copies and
//     the box complete on one mbarrier per ring slot;
//   * every warp runs its own two-slot ring: it waits for a slot, reads the
//     whole stage into registers, refills the slot two stages ahead and then
//     computes, so two stages per warp stay in flight;
//   * the unpack is one lop3 per pair of nibbles and adds no bias: a nibble at
//     bits 0..3 of an fp16 half is the subnormal q * 2^-24, at bits 4..7 it is
//     q * 2^-20, both exact.  The pairs (q0,q4) (q2,q6) of a word feed one
//     MMA chain (D_lo, scale 2^-24) and (q1,q5) (q3,q7) another (D_hi, scale
//     2^-20); the MMA k slots stand for k0,k4,k2,k6 and k1,k5,k3,k7, and x is
//     staged once per CTA in the same order;
//   * the zero point enters as one more MMA on the D_lo chain: sum_k (q - z) x
//     = sum_k q x - z * S with S the group's sum of x, given to the MMA as an
//     fp16 pair S_hi + S_lo (S_hi = fp16(S), S_lo = fp16(S - S_hi)) against
//     the fp16 subnormal -z * 2^-24.  Then per group
//         acc += s * (16 * D_lo + D_hi)
//     and y = 2^20 * acc, which is sum_g s_g * sum_k (q - z) x;
//   * CTAs are persistent: a CTA owns one K slice, stages that slice of x
//     once, then each warp walks its strips with one continuous copy stream;
//   * split K: fp32 partials and a last-arriving-warp reduction in slice
//     order (deterministic, no warp waits for another).
#include <cuda.h>

#include "w4a16_device.cuh"
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCtasPerSm = 2;
constexpr int kStageGroups = 4;                 // groups per box
constexpr int kDepth = 2;                       // ring slots per warp
constexpr int kStageW = kStageGroups * 16 * 64;  // 4 KB of weights
constexpr int kStageMeta = 16 * 16;             // per row: 3 scale words, 1 zeros word
constexpr int kStageBytes = kStageW + kStageMeta;
constexpr int kRingBytes = kWarps * kDepth * kStageBytes;  // 69632
constexpr int kBarBytes = kWarps * kDepth * 8;
constexpr int kSmemPerCta = 228 * 1024 / kCtasPerSm - 1024;  // leaves the per-CTA reserve
constexpr int kMaxSliceGroups = 128;
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // 200 ms per wait
constexpr int kErrMmaWait = 128;  // device status bit: a ring wait expired
constexpr float kTwo20 = 1048576.f;

struct MmaParams {
    const __half *x;
    const __half *scales;
    const uint32_t *zeros;
    __half *y;
    float *partials;
    unsigned *counters;
    int *status;
    uintptr_t scales_first;  // the aligned word holding the first scale
    uintptr_t scales_end;    // one past the last byte of the scales array
    int N, K, G, ZW;
    int M;  // tokens, 1..8
    int S, slice_groups;
    int n_strips, ctas_per_slice;  // 16-row strips; persistent CTAs per slice
    int xstride;                   // bytes per staged token row
};

// Staged x: 16-byte unit J of a token row lives at unit J ^ (bit 3 of J moved
// to bit 1).  With a row stride of 16 (mod 128) bytes the 16-byte reads of a
// quarter warp (two tokens x four lanes) fall on distinct banks.
__device__ __forceinline__ int x_unit(int J) { return J ^ (((J >> 3) & 1) << 1); }

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- copies and barriers ----------------------------------------------------
__device__ __forceinline__ void cp4(uint32_t dst, uintptr_t src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
// the barrier's pending count drops by one once this thread's earlier cp.async
// copies have landed
__device__ __forceinline__ void cp_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
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
// true once the phase with this parity has completed; false after kWaitNs
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = dev::globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 0 && dev::globaltimer() - t0 > kWaitNs) return false;
    }
}

// box {16 words, 16 rows, 4 groups} at (word 0, row, group) of the qweight
// tensor map (dims: word in group, row, group)
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap *map, int row, int grp,
                                        uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(grp), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// 8 consecutive fp16 activations (x0..x7) -> (x0,x4) (x2,x6) (x1,x5) (x3,x7):
// the B registers of the two MMAs that take one weight word.
__device__ __forceinline__ uint4 mma_pair_order(uint4 v) {
    uint4 o;
    o.x = dev::prmt(v.x, v.z, 0x5410);
    o.y = dev::prmt(v.y, v.w, 0x5410);
    o.z = dev::prmt(v.x, v.z, 0x7632);
    o.w = dev::prmt(v.y, v.w, 0x7632);
    return o;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    mma_kernel(const __grid_constant__ CUtensorMap tmap, const MmaParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    uint8_t *wring = smem + (size_t)warp * kDepth * kStageBytes;  // this warp's two slots
    uint8_t *xs = smem + kRingBytes + kBarBytes;                   // staged x, then the sums
    // the next kernel in the stream may be scheduled as SMs free up; it waits
    // for this grid to finish before it touches anything this grid writes
    grid_dependents_launch();

    const int slice = blockIdx.x % p.S;
    const int q = blockIdx.x / p.S;  // index among the CTAs of this slice
    const int g0 = slice * p.slice_groups;  // a multiple of kStageGroups
    const int ng = min(p.G, g0 + p.slice_groups) - g0;
    const int nst = (ng + kStageGroups - 1) / kStageGroups;  // stages per strip
    // this warp's strips: first, first + stride, ...
    const int first = q * kWarps + warp;
    const int stride = p.ctas_per_slice * kWarps;
    const int my_strips = first < p.n_strips ? (p.n_strips - 1 - first) / stride + 1 : 0;

    const uint32_t bar0 = dev::smem_u32(smem + kRingBytes) + 8 * kDepth * warp;
    const uint32_t ring0 = dev::smem_u32(wring);
    if (lane == 0) {
        // one arrival with the box's byte count, plus one per lane once its
        // metadata copies have landed
        for (int s = 0; s < kDepth; ++s) mbar_init(bar0 + 8 * s, 1 + 32);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    // ---- copy stream: the issue cursor runs kDepth stages ahead of the
    // consume cursor.  Weights, scales and zeros are parameters (never written
    // by a preceding kernel), so the stream starts before the grid-dependency
    // wait.  Metadata: lane (r = lane % 16, h = lane / 16) copies, for row r
    // of the strip, scale words 0 and 1 of the stage (h = 0) or scale word 2
    // and the zeros word (h = 1); the scale words are the three aligned words
    // that hold the stage's four (2-byte aligned) scales.
    int is_k = 0, is_j = 0, is_slot = 0;
    const int r = lane & 15, h = lane >> 4;
    auto issue_next = [&]() {
        if (is_k >= my_strips) return;
        const int strip = first + is_k * stride;
        const int grp = g0 + is_j * kStageGroups;
        const uint32_t bar = bar0 + 8 * is_slot;
        const uint32_t dst = ring0 + is_slot * kStageBytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, kStageW);
            tma_box(dst, &tmap, strip * 16, grp, bar);
        }
        const int row = strip * 16 + r;
        const bool vr = row < p.N;
        const size_t rr = (size_t)(vr ? row : 0);
        const uint32_t md = dst + kStageW + r * 16 + 8 * h;
        const uintptr_t sa =
            (((uintptr_t)(p.scales + rr * p.G + grp)) & ~(uintptr_t)3) + 8 * (uintptr_t)h;
        // copy the part of the word at a that lies inside the scales array
        // (a word past the end, or of a row past N, becomes zeros and reads
        // nothing; its source address is then the array's first word)
        auto copy_scale_word = [&](uint32_t d, uintptr_t a) {
            const uint32_t n = !vr || a >= p.scales_end
                                   ? 0u
                                   : (p.scales_end - a >= 4 ? 4u : (uint32_t)(p.scales_end - a));
            cp4(d, n ? a : p.scales_first, n);
        };
        copy_scale_word(md, sa);
        if (h == 0)
            copy_scale_word(md + 4, sa + 4);
        else
            cp4(md + 4, (uintptr_t)(p.zeros + rr * p.ZW + (grp >> 3)), vr ? 4u : 0u);
        cp_arrive_noinc(bar);
        is_slot ^= 1;  // kDepth == 2
        if (++is_j == nst) {
            is_j = 0;
            ++is_k;
        }
    };
    static_assert(kDepth == 2, "the slot and phase updates assume two slots");
#pragma unroll
    for (int s = 0; s < kDepth; ++s) issue_next();

    // ---- from here on: x, y and the split-K workspace may belong to the
    // preceding kernel
    grid_dependency_wait();

    // ---- stage x[:, slice] in MMA pair order, and each (group, token)'s sum
    // of x as an fp16 pair (S_hi, S_lo): the 16 lanes of a half warp hold the
    // 16 units of one group of one token and add theirs with shuffles
    const int M = p.M;
    uint32_t *sums = reinterpret_cast<uint32_t *>(xs + (size_t)M * p.xstride);  // [group][8]
    {
        const int nunits = ng * (kGroup / 8);
        const int xtotal = M * nunits;  // a multiple of 16
        const int k0 = g0 * kGroup;
        for (int base = warp * 32; base < xtotal; base += kThreads) {
            const int i = base + lane;
            const bool valid = i < xtotal;
            const int t = i / nunits, J = i - t * nunits;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (valid) {
                v = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)t * p.K + k0 + 8 * J));
                *reinterpret_cast<uint4 *>(xs + (size_t)t * p.xstride + 16 * x_unit(J)) =
                    mma_pair_order(v);
            }
            const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
            const float2 e = __half22float2(*reinterpret_cast<const __half2 *>(&v.z));
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&v.w));
            float sum = ((a.x + a.y) + (b.x + b.y)) + ((e.x + e.y) + (f.x + f.y));
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (valid && (J & 15) == 0) {
                const __half hi = __float2half_rn(sum);
                const __half lo = __float2half_rn(sum - __half2float(hi));
                sums[(J >> 4) * 8 + t] = (uint32_t)__half_as_ushort(hi) |
                                         ((uint32_t)__half_as_ushort(lo) << 16);
            }
        }
    }
    __syncthreads();

    // lanes of tokens >= M compute a column nobody stores: they read token 0
    const int tok = g < M ? g : 0;
    const uint8_t *xrow = xs + (size_t)tok * p.xstride;
    // unit of word u of this lane's chunk in a group: x_unit(4c + u)
    const int xo0 = 16 * x_unit(4 * c + 0), xo1 = 16 * x_unit(4 * c + 1);
    const int xo2 = 16 * x_unit(4 * c + 2), xo3 = 16 * x_unit(4 * c + 3);
    // -z * 2^-24 as an fp16 pair sits in k slots 0 and 1: lanes c == 0 only
    const uint32_t zmul = c == 0 ? 0x00010001u : 0u;
    const uint32_t zbase = c == 0 ? 0x80008000u : 0u;
    int cs_slot = 0;
    uint32_t cs_par = 0;

    for (int k = 0; k < my_strips; ++k) {
        const int strip = first + k * stride;
        const int ra = strip * 16 + g, rb = ra + 8;
        const bool va = ra < p.N, vb = rb < p.N;
        // where the slice's first scale of each row sits in its aligned word
        // (the same in every stage: a stage advances 8 bytes)
        const uint32_t offA =
            (uint32_t)(((uintptr_t)(p.scales + (size_t)(va ? ra : 0) * p.G + g0)) >> 1) & 1u;
        const uint32_t offB =
            (uint32_t)(((uintptr_t)(p.scales + (size_t)(vb ? rb : 0) * p.G + g0)) >> 1) & 1u;
        const uint32_t shA = 16u * offA, shB = 16u * offB;
        const uint32_t selA = offA ? 0x54u : 0x32u, selB = offB ? 0x54u : 0x32u;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < nst; ++j) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * cs_slot, cs_par))) {
                if (lane == 0) atomicOr(p.status, kErrMmaWait);
                cp_wait_all();
                return;
            }
            // the whole stage into registers: this lane's 16 bytes of rows g
            // and g + 8 of each group, and the metadata of both rows
            const uint8_t *st = wring + cs_slot * kStageBytes;
            uint4 wa[kStageGroups], wb[kStageGroups];
#pragma unroll
            for (int i = 0; i < kStageGroups; ++i) {
                wa[i] = *reinterpret_cast<const uint4 *>(st + i * 1024 + g * 64 + 16 * c);
                wb[i] = *reinterpret_cast<const uint4 *>(st + i * 1024 + (g + 8) * 64 + 16 * c);
            }
            const uint4 ma = *reinterpret_cast<const uint4 *>(st + kStageW + g * 16);
            const uint4 mb = *reinterpret_cast<const uint4 *>(st + kStageW + (g + 8) * 16);
            __syncwarp();  // every lane has read the slot: refill it
            issue_next();
            cs_slot ^= 1;
            if (cs_slot == 0) cs_par ^= 1;

            // zero nibbles of the stage's groups: the stage starts at group
            // g0 + 4j, nibble (g0 + 4j) % 8 of its zeros word
            const uint32_t zsh = ((g0 + j * kStageGroups) & 4) ? 16u : 0u;
            const uint32_t zwA = ma.w >> zsh, zwB = mb.w >> zsh;
            const uint32_t mA[3] = {ma.x, ma.y, ma.z}, mB[3] = {mb.x, mb.y, mb.z};
            const int n_in = min(kStageGroups, ng - j * kStageGroups);
            const uint8_t *xg = xrow + (size_t)j * (kStageGroups * 256);
            const uint32_t *sg = sums + (j * kStageGroups) * 8 + tok;
#pragma unroll
            for (int i = 0; i < kStageGroups; ++i) {
                if (i < n_in) {
                    // scales of rows ra and rb: half (off + i) of the words
                    uint32_t hA, hB;
                    if (i & 1) {
                        hA = dev::prmt(mA[i >> 1], mA[(i >> 1) + 1], selA);
                        hB = dev::prmt(mB[i >> 1], mB[(i >> 1) + 1], selB);
                    } else {
                        hA = mA[i >> 1] >> shA;
                        hB = mB[i >> 1] >> shB;
                    }
                    const float sA = __half2float(__ushort_as_half((unsigned short)hA));
                    const float sB = __half2float(__ushort_as_half((unsigned short)hB));
                    const uint32_t cA = ((zwA >> (4 * i)) & 0xfu) * zmul + zbase;
                    const uint32_t cB = ((zwB >> (4 * i)) & 0xfu) * zmul + zbase;
                    const uint32_t sx = sg[i * 8];  // (S_hi, S_lo) of token tok
                    const uint8_t *xi = xg + i * 256;
                    uint4 xv[4];
                    xv[0] = *reinterpret_cast<const uint4 *>(xi + xo0);
                    xv[1] = *reinterpret_cast<const uint4 *>(xi + xo1);
                    xv[2] = *reinterpret_cast<const uint4 *>(xi + xo2);
                    xv[3] = *reinterpret_cast<const uint4 *>(xi + xo3);
                    const uint32_t wA[4] = {wa[i].x, wa[i].y, wa[i].z, wa[i].w};
                    const uint32_t wB[4] = {wb[i].x, wb[i].y, wb[i].z, wb[i].w};
                    float dl[4] = {0.f, 0.f, 0.f, 0.f}, dh[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(dl, cA, cB, 0u, 0u, sx, sx);  // - z * S
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t a = wA[u], b = wB[u], a8 = a >> 8, b8 = b >> 8;
                        mma16816(dl, a & 0x000f000fu, b & 0x000f000fu, a8 & 0x000f000fu,
                                 b8 & 0x000f000fu, xv[u].x, xv[u].y);
                        mma16816(dh, a & 0x00f000f0u, b & 0x00f000f0u, a8 & 0x00f000f0u,
                                 b8 & 0x00f000f0u, xv[u].z, xv[u].w);
                    }
                    acc[0] = fmaf(sA, fmaf(16.f, dl[0], dh[0]), acc[0]);
                    acc[1] = fmaf(sA, fmaf(16.f, dl[1], dh[1]), acc[1]);
                    acc[2] = fmaf(sB, fmaf(16.f, dl[2], dh[2]), acc[2]);
                    acc[3] = fmaf(sB, fmaf(16.f, dl[3], dh[3]), acc[3]);
                }
            }
        }

        // ---- end of strip: acc[0..1] row ra, tokens 2c, 2c+1; acc[2..3] row rb
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] *= kTwo20;
        const int t0 = 2 * c, t1 = 2 * c + 1;
        if (p.S == 1) {
            if (va && t0 < M) p.y[(size_t)t0 * p.N + ra] = __float2half_rn(acc[0]);
            if (va && t1 < M) p.y[(size_t)t1 * p.N + ra] = __float2half_rn(acc[1]);
            if (vb && t0 < M) p.y[(size_t)t0 * p.N + rb] = __float2half_rn(acc[2]);
            if (vb && t1 < M) p.y[(size_t)t1 * p.N + rb] = __float2half_rn(acc[3]);
            continue;
        }
        float *part = p.partials + (size_t)slice * M * p.N;
        if (va && t0 < M) part[(size_t)t0 * p.N + ra] = acc[0];
        if (va && t1 < M) part[(size_t)t1 * p.N + ra] = acc[1];
        if (vb && t0 < M) part[(size_t)t0 * p.N + rb] = acc[2];
        if (vb && t1 < M) part[(size_t)t1 * p.N + rb] = acc[3];
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
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 2 * c + e;
                    if (ok[hh] && t < M) {
                        float sum = 0.f;
                        for (int s2 = 0; s2 < p.S; ++s2)
                            sum += __ldcg(p.partials + ((size_t)s2 * M + t) * p.N + rows[hh]);
                        p.y[(size_t)t * p.N + rows[hh]] = __float2half_rn(sum);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) p.counters[strip] = 0u;  // ready for the next launch
        }
    }
    cp_wait_all();
}

int xstride_for(int slice_groups) { return slice_groups * kGroup * 2 + 16; }

int smem_for(int M, int slice_groups) {
    return kRingBytes + kBarBytes + M * xstride_for(slice_groups) + slice_groups * 8 * 4;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode_mma = nullptr;

}  // namespace

MmaPlan plan_mma(int M, int N, int K, int split, const DeviceInfo &dev) {
    MmaPlan pl{};
    pl.M = M;
    const int G = K / kGroup;
    pl.n_strips = (N + 15) / 16;
    // largest slice (a whole number of stages) whose staged x and sums fit
    const int budget = kSmemPerCta - kRingBytes - kBarBytes;
    int max_groups = (budget - 16 * M) / (kGroup * 2 * M + 32);
    max_groups = max_groups / kStageGroups * kStageGroups;
    if (max_groups > kMaxSliceGroups) max_groups = kMaxSliceGroups;
    if (max_groups < kStageGroups) max_groups = kStageGroups;
    const int s_min = (G + max_groups - 1) / max_groups;
    if (split == 0 && s_min > 1) {
        pl.ok = false;
        return pl;
    }
    const int warps = kCtasPerSm * dev.sm_count * kWarps;
    // Pick the number of K slices that minimises the work of the busiest warp
    // (strips per warp x (groups per slice + a per-strip charge)), plus a
    // charge per extra slice for the partial sums; slices are whole stages.
    int s_lo = s_min;
    if (split == 1 && s_lo < 2 && G > kStageGroups) s_lo = 2;
    int s_hi = split == 0 ? 1 : (G + kStageGroups - 1) / kStageGroups;
    if (s_hi < s_lo) s_hi = s_lo;
    int best_sg = 0;
    double best_cost = 1e30;
    for (int S = s_lo; S <= s_hi; ++S) {
        int sg = (G + S - 1) / S;
        sg = (sg + kStageGroups - 1) / kStageGroups * kStageGroups;
        if (sg > max_groups) continue;
        const int S_eff = (G + sg - 1) / sg;
        if (split == 1 && S_eff < 2 && G > kStageGroups) continue;
        const long long units = (long long)pl.n_strips * S_eff;
        const long long per_warp = (units + warps - 1) / warps;
        const double cost = (double)per_warp * (sg + 2) + (S_eff > 1 ? 2.0 + 0.5 * S_eff : 0.0);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best_sg = sg;
        }
    }
    if (best_sg == 0) {  // split == 1 and too few groups to split along stage lines
        pl.ok = false;
        return pl;
    }
    pl.slice_groups = best_sg;
    pl.S = (G + best_sg - 1) / best_sg;
    int per_slice = kCtasPerSm * dev.sm_count / pl.S;
    const int need = (pl.n_strips + kWarps - 1) / kWarps;  // CTAs to give every strip a warp
    if (per_slice > need) per_slice = need;
    if (per_slice < 1) per_slice = 1;
    pl.ctas_per_slice = per_slice;
    pl.grid = per_slice * pl.S;
    pl.smem_bytes = smem_for(M, pl.slice_groups);
    pl.ws_bytes = pl.S > 1 ? (size_t)pl.S * M * N * sizeof(float) : 0;
    pl.ok = pl.S <= 65535;
    return pl;
}

cudaError_t launch_mma(const LinearArgs &a, const MmaPlan &plan, const Workspace &ws,
                       cudaStream_t stream) {
    if (!g_encode_mma) return cudaErrorInitializationError;
    const int G = a.K / kGroup;
    // qweight as a 3-D tensor of uint32: (word in group, row, group), so one
    // box brings a strip's 16 rows x 4 groups, group-major
    CUtensorMap tmap;
    const cuuint64_t dims[3] = {16, (cuuint64_t)a.N, (cuuint64_t)G};
    const cuuint64_t strides[2] = {(cuuint64_t)a.K / 2, 64};
    const cuuint32_t box[3] = {16, 16, (cuuint32_t)kStageGroups};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode_mma(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, (void *)a.qw, dims, strides,
                              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    MmaParams p;
    p.x = a.x;
    p.scales = a.scales;
    p.zeros = a.zeros;
    p.y = a.y;
    p.partials = ws.partials;
    p.counters = ws.counters;
    p.status = ws.status;
    p.scales_first = (uintptr_t)a.scales & ~(uintptr_t)3;
    p.scales_end = (uintptr_t)(a.scales + (size_t)a.N * G);
    p.N = a.N;
    p.K = a.K;
    p.G = G;
    p.ZW = (G + 7) / 8;
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
    return cudaLaunchKernelEx(&cfg, mma_kernel, tmap, p);
}

cudaError_t mma_init(const DeviceInfo &dev) {
    if (!g_encode_mma) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
        g_encode_mma = reinterpret_cast<EncodeTiledFn>(fn);
    }
    int dyn = kSmemPerCta;
    if (dyn > dev.max_smem_optin - 1024) dyn = dev.max_smem_optin - 1024;
    cudaError_t e = cudaFuncSetAttribute(mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mma_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

}  // namespace w4a16
