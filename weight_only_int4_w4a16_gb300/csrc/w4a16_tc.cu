// tcgen05 dequant-GEMM for W4A16 (rungs "tc" and "tc_splitk").
//
// The method is the same linear as the CUDA-core rungs (forum.sourcefind.cn
// thread "vLLM on Hygon Z100", section 四: unpack the INT4 words, restore
// (q - z) * s, multiply-accumulate with fp16 activations in fp32).  Section 七
// of the thread notes that once M grows the GEMV is no longer the right shape
// and the crossover to a GEMM path has to be measured; this is the GEMM path,
// written for the sm_103a tensor cores:
//
//   MMA shape (swap AB): the MMA's M = 128 weight rows n of one tile, its
//   N = T tokens (16, 32 or 64; M is padded up with zero rows of x), K = 16
//   per instruction, fp16 inputs, fp32 accumulation in tensor memory.
//
//   warp 20 (one thread) streams packed weights with TMA: one box of
//     128 rows x 64 bytes (one 128-wide group) per stage, 64-byte swizzle;
//   warps 4..19, two teams of 8 taking alternate groups, unpack a stage:
//     thread = one row (its TMEM lane), two warps per 32-lane quarter split
//     the group's 128 k in halves.  The nibble
//     unpack is the exponent-bias one of the CUDA-core rung ((1024 + q) and
//     (64 + q) spliced into fp16, minus (1024 + z) / (64 + z), exact), and
//     the exact fp16 (q - z) values go to tensor memory with tcgen05.st as
//     the MMA's A operand.  The same warps stage the group's slice of x in
//     shared memory (canonical K-major layout, no swizzle), in the pair order
//     the unpack produces, as the MMA's B operand;
//   warps 21 and 22 (one thread each) take alternate groups and issue a
//     group's 8 tcgen05.mma into a fresh fp32 accumulator in tensor memory
//     (one accumulator per group, ring of 4), then commit to mbarriers.  At
//     N = 16 one issuing thread spends ~85 cycles per instruction while the
//     tensor pipe idles most of the time; two issuers cut M = 16 from 63.5
//     to 49 us.  Each A buffer (ring of 4) and each accumulator belongs to
//     one team and one issuer, so every barrier's phases are consumed in
//     order by a single waiter;
//   warps 0..3 read each group's accumulator with tcgen05.ld and add
//     s[n, g] * acc into fp32 registers.  The scale is applied in fp32 per
//     group, so the tensor-core products (q - z) * x are exact and only the
//     fp32 sums round;
//   split K: slices of whole groups per CTA; the last CTA of a tile sums the
//     fp32 partials in slice order (same scheme as the CUDA-core rung).
//
// Every mbarrier wait is bounded by %globaltimer; on expiry the kernel records
// an error code in device memory, every role drains what it has in flight
// (again bounded), and the CTA frees its tensor memory and exits.
#include <cuda.h>

#include <cstring>

#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kTileN = 128;                      // weight rows per tile (MMA M)
constexpr int kChunkWords = kGroup / 8;          // 16 words = 64 bytes per row per group
constexpr int kStageBytes = kTileN * kChunkWords * 4;  // 8 KB per TMA stage
constexpr int kPStages = 12;                     // packed-weight stages in flight (96 KB)
constexpr int kAStages = 4;                      // A (dequantised group) buffers in TMEM
constexpr int kDStages = 4;                      // per-group accumulator sets in TMEM
constexpr int kDCols = 64;                       // TMEM columns per accumulator set
constexpr int kACols = kGroup / 2;               // TMEM columns per A buffer (2 fp16 / column)
constexpr int kXAhead = 2;                       // a team's groups of x fetched ahead (cp.async)
constexpr int kEpiWarps = 4;
constexpr int kDeqTeams = 2;                     // dequant teams take alternate groups
constexpr int kDeqWarps = 8;                     // warps per team (2 per TMEM lane quarter)
constexpr int kTmaWarp = kEpiWarps + kDeqTeams * kDeqWarps;  // 20
constexpr int kMmaWarp = kTmaWarp + 1;                       // 21
constexpr int kMmaWarps = 2;                                 // MMA issuers, alternate groups
constexpr int kThreads = (kMmaWarp + kMmaWarps) * 32;        // 736
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // 200 ms per wait

// error codes recorded in the device status word (bit flags)
constexpr int kErrWaitFull = 1, kErrWaitAFull = 2, kErrWaitDFull = 4, kErrWaitEmpty = 8,
              kErrWaitAEmpty = 16, kErrWaitDEmpty = 32, kErrDrain = 64;

struct TcParams {
    CUtensorMap tmap;  // qweight as a 2-D tensor of uint32: {K/8, N}
    const __half *x;
    const __half *scales;
    const uint32_t *zeros;
    __half *y;
    float *partials;
    unsigned *counters;
    int *status;
    int N, K, G, ZW;
    int M;             // real tokens in this launch (<= T)
    int S, slice_groups;
};

template <int T>
struct TcConfig {
    static constexpr int kXBytes = T * kGroup * 2;          // one group of x, T tokens
    // A group's 8 MMAs go round-robin into kChains independent accumulators
    // (T columns each) so that consecutive MMAs do not wait on one another;
    // the epilogue adds the chains.
    static constexpr int kChains = kDCols / T;               // 4, 2, 1
    static constexpr int kDBase = kAStages * kACols;         // 192
    static constexpr int kColsUsed = kDBase + kDStages * kDCols;
    static constexpr int kTmemCols = kColsUsed <= 256 ? 256 : 512;
    static constexpr int kSmemP = kPStages * kStageBytes;
    static constexpr int kSmemX = kAStages * kXBytes;
    static constexpr int kSmemXRaw = kDeqTeams * kXAhead * kXBytes;  // x copies in flight
    static constexpr int kSmemBar = 1024;
    static constexpr int kSmemBytes = 1024 /*align slack*/ + kSmemP + kSmemX + kSmemXRaw + kSmemBar;
    static constexpr int kPiecesPerThread = T * 16 / (kDeqWarps * 32);  // 16-byte x pieces
    // instruction descriptor: D f32, A f16, B f16, both K-major, N = T, M = 128
    static constexpr uint32_t kIdesc =
        (1u << 4) | ((uint32_t)(T >> 3) << 17) | ((uint32_t)(kTileN >> 4) << 24);
};

// Optional section timers (build with -DW4A16_TRACE): CTA (0, 0) records the
// SM cycle counter at each pipeline event of its first kTraceChunks groups.
#ifdef W4A16_TRACE
constexpr int kTraceChunks = 32;
constexpr int kTraceEvents = 9;
__device__ unsigned long long g_trace[kTraceEvents * kTraceChunks];
#define W4A16_TR(ev, c)                                                                   \
    do {                                                                                  \
        if (blockIdx.x == 0 && blockIdx.y == 0 && (c) < kTraceChunks)                     \
            g_trace[(ev) * kTraceChunks + (c)] = clock64();                               \
    } while (0)
#else
#define W4A16_TR(ev, c) \
    do {                \
    } while (0)
#endif

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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

// Bounded wait: true once the phase with this parity has completed; false if
// another role aborted or the time limit passed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > kWaitNs) return false;
        }
    }
}

__device__ __forceinline__ void fail(volatile int *abort, int *status, int code) {
    *abort = 1;
    atomicOr(status, code);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    // tcgen05 shared-memory matrix descriptor, no swizzle: start address,
    // leading byte offset (between core matrices along K), stride byte offset
    // (between 8-row groups along M/N), fixed version field 1 at bit 46.
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
           ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
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

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16-byte global -> shared copy that bypasses registers; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 8 consecutive fp16 x values -> (x0,x4) (x1,x5) (x2,x6) (x3,x7): the order in
// which the unpack yields the nibbles of one word.
__device__ __forceinline__ uint4 pair_order(uint4 v) {
    uint4 o;
    o.x = prmt(v.x, v.z, 0x5410);
    o.y = prmt(v.x, v.z, 0x7632);
    o.z = prmt(v.y, v.w, 0x5410);
    o.w = prmt(v.y, v.w, 0x7632);
    return o;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int T>
__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ TcParams p) {
    using C = TcConfig<T>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sm_p = smem;                   // packed stages
    uint8_t *sm_x = smem + C::kSmemP;       // x buffers (MMA operand layout)
    uint8_t *sm_xraw = sm_x + C::kSmemX;    // x copies in flight (row-major pieces)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm_xraw + C::kSmemXRaw);
    uint64_t *full = bars;                          // [kPStages]
    uint64_t *empty = full + kPStages;              // [kPStages]
    uint64_t *a_full = empty + kPStages;            // [kAStages]
    uint64_t *a_empty = a_full + kAStages;          // [kAStages]
    uint64_t *d_full = a_empty + kAStages;          // [kDStages]
    uint64_t *d_empty = d_full + kDStages;          // [kDStages]
    uint64_t *done = d_empty + kDStages;            // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_last = const_cast<int *>(abort + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, slice = blockIdx.y;
    const int g0 = slice * p.slice_groups;
    const int g1 = min(p.G, g0 + p.slice_groups);
    const int nchunks = g1 - g0;

    if (threadIdx.x == kTmaWarp * 32) {
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), kDeqWarps);
        }
        for (int i = 0; i < kAStages; ++i) {
            mbar_init(smem_u32(a_full + i), kDeqWarps);
            mbar_init(smem_u32(a_empty + i), 1);
        }
        for (int i = 0; i < kDStages; ++i) {
            mbar_init(smem_u32(d_full + i), 1);
            mbar_init(smem_u32(d_empty + i), kEpiWarps);
        }
        mbar_init(smem_u32(done), kMmaWarps);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap))
                     : "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kPStages;
                if (!mbar_wait(smem_u32(empty + s), ((c / kPStages) & 1) ^ 1, abort)) {
                    fail(abort, p.status, kErrWaitEmpty);
                    break;
                }
                W4A16_TR(0, c);
                mbar_arrive_expect_tx(smem_u32(full + s), kStageBytes);
                tma_load_2d(smem_u32(sm_p + s * kStageBytes), &p.tmap, (g0 + c) * kChunkWords,
                            tile * kTileN, smem_u32(full + s));
                issued = c + 1;
            }
            // drain: every issued copy must have landed before the CTA exits
            for (int c = issued - kPStages > 0 ? issued - kPStages : 0; c < issued; ++c) {
                if (!mbar_wait(smem_u32(full + c % kPStages), (c / kPStages) & 1, abort) &&
                    !mbar_try_wait(smem_u32(full + c % kPStages), (c / kPStages) & 1)) {
                    // bounded second chance independent of the abort flag
                    const unsigned long long t0 = globaltimer();
                    bool ok = false;
                    while (!ok && globaltimer() - t0 < kWaitNs)
                        ok = mbar_try_wait(smem_u32(full + c % kPStages), (c / kPStages) & 1);
                    if (!ok) atomicOr(p.status, kErrDrain);
                }
            }
        }
    } else if (warp >= kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            for (int c = warp - kMmaWarp; c < nchunks; c += kMmaWarps) {
                const int a = c % kAStages, d = c % kDStages;
                if (!mbar_wait(smem_u32(a_full + a), (c / kAStages) & 1, abort)) {
                    fail(abort, p.status, kErrWaitAFull);
                    break;
                }
                W4A16_TR(4, c);
                if (!mbar_wait(smem_u32(d_empty + d), ((c / kDStages) & 1) ^ 1, abort)) {
                    fail(abort, p.status, kErrWaitDEmpty);
                    break;
                }
                tc_fence_after();
                W4A16_TR(5, c);
                const uint32_t xb = smem_u32(sm_x + a * C::kXBytes);
                const uint32_t d_tmem = tmem + C::kDBase + d * kDCols;
                const uint64_t bdesc0 = smem_desc_kmajor(xb, 128, 2048);
#pragma unroll
                for (int j = 0; j < kGroup / 16; ++j) {
                    // k step j: B advances 256 bytes (two 8x8 core matrices);
                    // accumulator chain j % kChains starts fresh on its first step
                    mma_f16_ts(d_tmem + (j % C::kChains) * T, tmem + a * kACols + 8 * j,
                               bdesc0 + (uint64_t)(16 * j), C::kIdesc, j >= C::kChains);
                }
                mma_commit(smem_u32(a_empty + a));
                mma_commit(smem_u32(d_full + d));
                W4A16_TR(6, c);
            }
            // all MMAs of this CTA complete before the tensor memory is freed
            mma_commit(smem_u32(done));
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(done), 0)) {
                if (globaltimer() - t0 > kWaitNs) {
                    atomicOr(p.status, kErrDrain);
                    break;
                }
            }
        }
    } else if (warp >= kEpiWarps) {
        // ------------------------------------------------ dequantise + stage x
        const int team = (warp - kEpiWarps) / kDeqWarps;  // groups team, team+2, ...
        const int dw = (warp - kEpiWarps) % kDeqWarps;    // 0..7 within the team
        const int quarter = warp & 3;         // TMEM lanes 32*quarter ..
        const int half = dw >> 2;             // which 64 k of the group
        const int r = quarter * 32 + lane;    // row within the tile
        const int n = tile * kTileN + r;
        const uint32_t *zrow = p.zeros + (size_t)(n < p.N ? n : 0) * p.ZW;
        const int dt = dw * 32 + lane;        // 0..255 among dequant threads
        // x pieces this thread moves: piece pc = dt + 256 i is (token pc % T,
        // 8-block pc / T) of a group; copied kXAhead groups ahead with cp.async
        // into a raw ring, then re-ordered into the MMA layout when its group
        // comes up.
        uint8_t *team_raw = sm_xraw + team * kXAhead * C::kXBytes;
        // the team's li-th group is c = team + kDeqTeams * li
        auto issue_x = [&](int li) {
            const int c = team + kDeqTeams * li;
            if (c < nchunks) {
                const int g = g0 + c;
                uint8_t *raw = team_raw + (li % kXAhead) * C::kXBytes;
#pragma unroll
                for (int i = 0; i < C::kPiecesPerThread; ++i) {
                    const int pc = dt + i * kDeqWarps * 32;
                    const int t = pc % T, kb = pc / T;
                    const __half *src =
                        t < p.M ? p.x + (size_t)t * p.K + (size_t)g * kGroup + 8 * kb : p.x;
                    cp_async16(smem_u32(raw + pc * 16), src, t < p.M ? 16u : 0u);
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int li = 0; li < kXAhead; ++li) issue_x(li);
        const int c_first = team;
        uint32_t zw_cur = (n < p.N && c_first < nchunks) ? __ldg(zrow + ((g0 + c_first) >> 3)) : 0u;
        uint32_t zw_next = (n < p.N && c_first + kDeqTeams < nchunks)
                               ? __ldg(zrow + ((g0 + c_first + kDeqTeams) >> 3))
                               : 0u;
        int li = 0;
        for (int c = c_first; c < nchunks; c += kDeqTeams, ++li) {
            const int s = c % kPStages, a = c % kAStages;
            const int g = g0 + c;
            const uint32_t zw = zw_cur;
            zw_cur = zw_next;
            zw_next = (n < p.N && c + 2 * kDeqTeams < nchunks)
                          ? __ldg(zrow + ((g + 2 * kDeqTeams) >> 3))
                          : 0u;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(full + s), (c / kPStages) & 1, abort))) {
                fail(abort, p.status, kErrWaitFull);
                break;
            }
            if (dw == 0 && lane == 0) W4A16_TR(1, c);
            // this row's 32 bytes of the stage: 16-byte chunks 2*half, 2*half+1,
            // stored 64-byte swizzled (chunk ^= (row >> 1) & 3)
            const uint8_t *st = sm_p + s * kStageBytes + r * 64;
            const int sw = (r >> 1) & 3;
            const uint4 w0 = *reinterpret_cast<const uint4 *>(st + 16 * ((2 * half) ^ sw));
            const uint4 w1 = *reinterpret_cast<const uint4 *>(st + 16 * ((2 * half + 1) ^ sw));
            if (!__all_sync(0xffffffffu,
                            mbar_wait(smem_u32(a_empty + a), ((c / kAStages) & 1) ^ 1, abort))) {
                fail(abort, p.status, kErrWaitAEmpty);
                break;
            }
            // the MMAs that read A[a] and x[a] have completed (commit); order
            // this warp's tensor-memory stores after that observation
            tc_fence_after();
            if (dw == 0 && lane == 0) W4A16_TR(2, c);
            const uint32_t z = (zw >> (4 * (g & 7))) & 0xfu;
            const uint32_t zz_hi = 0x64006400u | z | (z << 16);
            const uint32_t zz_lo = 0x54005400u | (z << 4) | (z << 20);
            const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t w = words[u], w8 = w >> 8;
                v[4 * u + 0] = hsub2(lop3_and_or(w, 0x000f000fu, 0x64006400u), zz_hi);
                v[4 * u + 1] = hsub2(lop3_and_or(w, 0x00f000f0u, 0x54005400u), zz_lo);
                v[4 * u + 2] = hsub2(lop3_and_or(w8, 0x000f000fu, 0x64006400u), zz_hi);
                v[4 * u + 3] = hsub2(lop3_and_or(w8, 0x00f000f0u, 0x54005400u), zz_lo);
            }
            // every lane has consumed its words of the stage: release it
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(empty + s));
            tmem_st_x32(tmem + ((uint32_t)(quarter * 32) << 16) + a * kACols + 32 * half, v);
            // x of this group: this thread's pieces arrived (own cp.async group);
            // re-order to pair order at (t/8)*2048 + kb*128 + (t%8)*16
            cp_async_wait<kXAhead - 1>();
            {
                const uint8_t *raw = team_raw + (li % kXAhead) * C::kXBytes;
                uint8_t *xb = sm_x + a * C::kXBytes;
#pragma unroll
                for (int i = 0; i < C::kPiecesPerThread; ++i) {
                    const int pc = dt + i * kDeqWarps * 32;
                    const int t = pc % T, kb = pc / T;
                    const uint4 v4 = pair_order(*reinterpret_cast<const uint4 *>(raw + pc * 16));
                    *reinterpret_cast<uint4 *>(xb + (t >> 3) * 2048 + kb * 128 + (t & 7) * 16) = v4;
                }
            }
            issue_x(li + kXAhead);  // refills the raw slot just read
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(a_full + a));
            if (dw == 0 && lane == 0) W4A16_TR(3, c);
        }
        cp_async_wait<0>();
    } else {
        // ------------------------------------------------ epilogue (warps 0..3)
        const int quarter = warp;  // warp % 4 == warp here
        const int r = quarter * 32 + lane;
        const int n = tile * kTileN + r;
        const __half *srow = p.scales + (size_t)(n < p.N ? n : 0) * p.G;
        float acc[T];
#pragma unroll
        for (int t = 0; t < T; ++t) acc[t] = 0.f;
        // scales fetched four groups ahead (a rotating set of registers)
        auto ld_scale = [&](int c) {
            return (n < p.N && c < nchunks) ? __half2float(srow[g0 + c]) : 0.f;
        };
        float s0 = ld_scale(0), s1 = ld_scale(1), s2 = ld_scale(2), s3 = ld_scale(3);
        for (int c = 0; c < nchunks; ++c) {
            const int d = c % kDStages;
            const float sc = s0;
            s0 = s1;
            s1 = s2;
            s2 = s3;
            s3 = ld_scale(c + 4);
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(d_full + d), (c / kDStages) & 1, abort))) {
                fail(abort, p.status, kErrWaitDFull);
                break;
            }
            tc_fence_after();
            if (warp == 0 && lane == 0) W4A16_TR(7, c);
            const uint32_t taddr =
                tmem + ((uint32_t)(quarter * 32) << 16) + C::kDBase + d * kDCols;
            if constexpr (C::kChains == 1) {
#pragma unroll
                for (int t0 = 0; t0 < T; t0 += 32) {
                    float v[16], w[16];
                    tmem_ld_x16(taddr + t0, v);
                    tmem_ld_x16(taddr + t0 + 16, w);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[t0 + i] = fmaf(sc, v[i], acc[t0 + i]);
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[t0 + 16 + i] = fmaf(sc, w[i], acc[t0 + 16 + i]);
                }
            } else {
                float sum[T];
#pragma unroll
                for (int t = 0; t < T; ++t) sum[t] = 0.f;
#pragma unroll
                for (int b = 0; b < kDCols / 16; b += 2) {
                    float v[16], w[16];
                    tmem_ld_x16(taddr + 16 * b, v);
                    tmem_ld_x16(taddr + 16 * b + 16, w);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) sum[(16 * b + i) % T] += v[i];
#pragma unroll
                    for (int i = 0; i < 16; ++i) sum[(16 * b + 16 + i) % T] += w[i];
                }
#pragma unroll
                for (int t = 0; t < T; ++t) acc[t] = fmaf(sc, sum[t], acc[t]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(d_empty + d));
            if (warp == 0 && lane == 0) W4A16_TR(8, c);
        }
        // one reader decides for all four epilogue warps (named barrier 1)
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        if (threadIdx.x == 0) *s_last = *abort ? -1 : 0;
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        if (*s_last == 0) {
            if (p.S == 1) {
                if (n < p.N) {
#pragma unroll
                    for (int t = 0; t < T; ++t)
                        if (t < p.M) p.y[(size_t)t * p.N + n] = __float2half_rn(acc[t]);
                }
            } else {
                if (n < p.N) {
#pragma unroll
                    for (int t = 0; t < T; ++t)
                        if (t < p.M) p.partials[((size_t)slice * p.M + t) * p.N + n] = acc[t];
                }
                __threadfence();
                asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
                if (threadIdx.x == 0) {
                    const unsigned prev = atomicAdd(p.counters + tile, 1u);
                    *s_last = (prev == (unsigned)(p.S - 1)) ? 1 : 0;
                }
                asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
                if (*s_last == 1) {
                    __threadfence();
                    if (n < p.N) {
                        for (int t = 0; t < p.M; ++t) {
                            float sum = 0.f;
                            for (int s2 = 0; s2 < p.S; ++s2)
                                sum += __ldcg(p.partials + ((size_t)s2 * p.M + t) * p.N + n);
                            p.y[(size_t)t * p.N + n] = __float2half_rn(sum);
                        }
                    }
                    if (threadIdx.x == 0) p.counters[tile] = 0u;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(C::kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int T>
cudaError_t launch_t(const TcParams &p, dim3 grid, cudaStream_t stream) {
    tc_kernel<T><<<grid, kThreads, TcConfig<T>::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

TcPlan plan_tc(int M, int N, int K, int split, const DeviceInfo &dev) {
    TcPlan pl{};
    pl.M = M;
    pl.T = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    const int G = K / kGroup;
    pl.n_tiles = (N + kTileN - 1) / kTileN;
    const int slots = dev.sm_count;  // one CTA of 448 threads per SM
    int S = 1;
    if (split != 0) {
        // whole groups per slice, at least 4 groups each; fill the SMs
        if (pl.n_tiles < slots) {
            S = slots / pl.n_tiles;
            int cap = G / 4 > 0 ? G / 4 : 1;
            if (S > cap) S = cap;
        }
        if (split == 1 && S < 2 && G >= 2) S = 2;
        if (S < 1) S = 1;
    }
    pl.slice_groups = (G + S - 1) / S;
    pl.S = (G + pl.slice_groups - 1) / pl.slice_groups;
    pl.ws_bytes = pl.S > 1 ? (size_t)pl.S * M * N * sizeof(float) : 0;
    pl.ok = G >= 1 && pl.S <= 65535;
    return pl;
}

cudaError_t tc_init(const DeviceInfo &dev) {
    (void)dev;
    if (!tensor_map_encoder()) return cudaErrorSymbolNotFound;
    cudaError_t e = cudaFuncSetAttribute(tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcConfig<16>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcConfig<32>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcConfig<64>::kSmemBytes);
    return e;
}

#ifdef W4A16_TRACE
extern "C" int w4a16_debug_trace(unsigned long long *out, int n) {
    if (n > kTraceEvents * kTraceChunks) n = kTraceEvents * kTraceChunks;
    return (int)cudaMemcpyFromSymbol(out, g_trace, n * sizeof(unsigned long long));
}
#endif

cudaError_t launch_tc(const LinearArgs &a, const TcPlan &plan, const Workspace &ws, int *status,
                      cudaStream_t stream) {
    const EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorInitializationError;
    TcParams p;
    memset(&p, 0, sizeof(p));
    const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 8), (cuuint64_t)a.N};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 8) * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kChunkWords, (cuuint32_t)kTileN};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&p.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, (void *)a.qw, dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    p.x = a.x;
    p.scales = a.scales;
    p.zeros = a.zeros;
    p.y = a.y;
    p.partials = ws.partials;
    p.counters = ws.counters;
    p.status = status;
    p.N = a.N;
    p.K = a.K;
    p.G = a.K / kGroup;
    p.ZW = (p.G + 7) / 8;
    p.M = a.M;
    p.S = plan.S;
    p.slice_groups = plan.slice_groups;
    dim3 grid(plan.n_tiles, plan.S);
    switch (plan.T) {
        case 16: return launch_t<16>(p, grid, stream);
        case 32: return launch_t<32>(p, grid, stream);
        case 64: return launch_t<64>(p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace w4a16
