// tcgen05 dequant-GEMM for W4A16 (rungs "tc" and "tc_splitk"), 9..64 tokens.
//
// The method is the same linear as the other rungs (forum.sourcefind.cn
// thread "vLLM on Hygon Z100", section 四: unpack the INT4 words, restore
// (q - z) * s, multiply-accumulate with fp16 activations in fp32).  Section 七
// of the thread notes that once M grows the GEMV is no longer the right shape
// and the crossover to a GEMM path has to be measured; this is the GEMM path,
// written for the sm_103a tensor cores.
//
//   MMA shape (swap AB): the MMA's M = 128 weight rows of one tile, its N = T
//   tokens (16, 32 or 64; missing tokens are zero rows of x), K = 16 per
//   instruction, fp16 inputs, fp32 accumulation in tensor memory.
//
//   The restore step writes A = (q - z) * s as fp16, rounded once from the
//   exact product (the pages' "restore to fp16" before the multiply, and the
//   fp16 result w4a16_dequant defines): the scale is inside the MMA operand,
//   so one accumulator collects every group of a K range and is read once,
//   where a per-group fp32 scale would read the accumulator after every group.
//   The product fits fp16 while |s| < 4096; a row whose scales reach that
//   (or are Inf or NaN) has its outputs of the K range recomputed exactly on
//   the CUDA cores by its epilogue thread (w = (q - z) * s in fp32, exact), so
//   every finite scale gives the method's result.
//
//   Roles (one CTA per SM, 800 threads):
//   warp 20 streams, per stage, a TMA box of 128 rows x 4 groups of packed
//     weights (each row a 256-byte run of memory, 64-byte swizzle; L2
//     evict-first, read once), and its lanes copy the rows' scale and zeros
//     words (cp.async) next to it;
//   warps 4..19, four teams of 4 (team i takes the groups c with c % 4 == i),
//     restore a group: thread = one row (its TMEM lane) and its 128 inputs
//     (a team of 4 warps has more registers per thread and fewer handoffs
//     per group than two teams of 8 with 64 inputs a thread: 43.3 -> 41.1 us
//     at M = 16, 48.7 -> 45.3 at M = 32); it reads its words of the stage at
//     once (so the stage is free for the next box early), then
//     the nibble unpack splices (1024 + q) or (64 + q) into fp16, subtracts the
//     matching (1024 + z) / (64 + z) exactly, multiplies by s (one rounding)
//     and puts the pairs in k order; tcgen05.st puts the values in tensor
//     memory as the MMA's A operand (a ring of 4 buffers).  One lane of each
//     team loads the group's x for all T tokens by TMA straight from the
//     caller's x into the matching x slot: two boxes of T rows x 128 bytes
//     land in the MMA's 128-byte swizzled K-major layout;
//   warps 21..24 (one thread each) take groups c with c % 4 == their index and
//     issue a group's 8 tcgen05.mma into their own accumulator chains (so the
//     sums of each chain come in a fixed order), then commit;
//   warps 0..3 (thread = row) read the chains once per K range, add them in a
//     fixed order, and write y, or, for a K range that is part of a tile, fp32
//     partial sums that the last CTA of the tile adds in K order.
//
//   Work: CTAs take equal runs of the (tile, stage) sequence ("stream-K"), so
//   that every SM streams the same number of bytes however the tiles divide
//   among the SMs; a tile split between CTAs is summed by the last of them in
//   K order (deterministic).  Without the split, CTAs take whole tiles in turn.
//
// Every mbarrier wait is bounded by %globaltimer; on expiry the kernel records
// an error code in device memory, every role drains what it has in flight
// (again bounded), and the CTA frees its tensor memory and exits.
#include <cuda.h>

#include <cstring>

#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kTileN = 128;                    // weight rows per tile (MMA M)
constexpr int kSG = 4;                         // groups per stage (one TMA box)
constexpr int kGroupBytes = kTileN * 64;       // 8 KB of packed weights per group
constexpr int kStageW = kSG * kGroupBytes;     // 32 KB
constexpr int kAStages = 4;                    // A (restored group) buffers in TMEM
constexpr int kACols = kGroup / 2;             // 64 TMEM columns per A buffer
constexpr int kEpiWarps = 4;
constexpr int kDeqTeams = 4;                   // restore teams: group c to team c % 4
constexpr int kDeqWarps = 4;                   // warps per team (one per TMEM lane quarter)
constexpr int kHalves = 8 / kDeqWarps;         // 64-input halves of a group row per thread
constexpr int kPerTeam = kSG / kDeqTeams;      // a team's groups per stage
constexpr int kTmaWarp = kEpiWarps + kDeqTeams * kDeqWarps;  // 20
constexpr int kMmaWarp = kTmaWarp + 1;                       // 21 .. 24
constexpr int kMmaWarps = 4;                                 // MMA issuers: group c to c % 4
constexpr int kThreads = (kMmaWarp + kMmaWarps) * 32;        // 800
constexpr int kTmemCols = 512;
constexpr int kMaxStages = 6;
constexpr int kSmemBudget = 220 * 1024;        // weight stages and the x ring
static_assert(kMmaWarps == kAStages, "issuer i owns A buffer i (and x slot i)");
// the mbarriers (full, empty per stage; a_full, a_empty, x_full per A buffer;
// d_full, d_empty; done), then the tensor-memory address, abort and last flags
constexpr int kBarBytes = (2 * kMaxStages + 3 * kAStages + 5) * 8 + 16;
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // 200 ms per wait
// scales whose 16-bit restore may overflow: |s| >= 4096 in fp16, |s| >= 2^120
// in bf16 (bits of |s|; Inf and NaN included): those rows take the exact path
constexpr uint32_t kBigScale = 0x6C00u;
constexpr uint32_t kBigScaleBf16 = 0x7B80u;

// error codes recorded in the device status word (bit flags)
constexpr int kErrWaitFull = 1, kErrWaitAFull = 2, kErrWaitDFull = 4, kErrWaitEmpty = 8,
              kErrWaitAEmpty = 16, kErrWaitDEmpty = 32, kErrDrain = 64, kErrWaitLinear = 65536;

struct TcParams {
    TcLinDesc single;       // the linear of a one-linear launch (start 0, no wait)
    const TcLinDesc *lins;  // a fused round: device [n_lin] linears; null for one linear
    int n_lin;
    unsigned *done;         // a round with waits: [n_lin] tiles finished, then CTAs finished
    float *partials;        // stream-K: [2 * grid][M][128] fp32
    int *status;
    int M;
    int streamk;
    int n_stages;           // shared-memory stages
    long long total;        // stages of all linears
};

template <int T, bool kBf16 = false>
struct TcConfig {
    // x of one group for T tokens: a slot of the x ring (one per A buffer)
    static constexpr int kXSlot = T * kGroup * 2;
    static constexpr int kXRing = kAStages * kXSlot;
    // per row: the 3 aligned words holding its 4 scales of the stage, then the
    // zeros word holding its 4 zeros
    static constexpr int kMeta = kTileN * 16;
    static constexpr int kStageBytes = kStageW + kMeta;
    static constexpr int kDBase = kAStages * kACols;      // 256: accumulators after A
    // Each issuer spreads a group's 8 MMAs over kChains independent
    // accumulators (k step kk into chain kk % kChains), so that consecutive MMAs
    // do not wait on one another's sums; an accumulator set holds every
    // issuer's chains, [issuer][chain][T columns]: 128 columns for T <= 32
    // (two sets, so that a K range's sums are read while the next one's run),
    // 256 for T = 64 (one set)
    static constexpr int kChains = T == 16 ? 2 : 1;
    static constexpr int kDBuf = kMmaWarps * kChains * T;
    static constexpr int kDSets = T == 64 ? 1 : 2;
    static_assert(kDBase + kDSets * kDBuf <= kTmemCols, "tensor memory");
    // instruction descriptor: D f32, A and B f16 (or both bf16), both K-major,
    // N = T, M = 128
    static constexpr uint32_t kIdesc = (1u << 4) | (kBf16 ? (1u << 7) | (1u << 10) : 0u) |
                                       ((uint32_t)(T >> 3) << 17) | ((uint32_t)(kTileN >> 4) << 24);
};

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

// The same wait, bounded by time alone (draining after an abort).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kWaitNs) return false;
    return true;
}

__device__ __forceinline__ void fail(volatile int *abort, int *status, int code) {
    *abort = 1;
    atomicOr(status, code);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

// 4-byte global -> shared copy; src_bytes 0 writes zeros and reads nothing
__device__ __forceinline__ void cp4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
// the barrier's pending count drops by one once this thread's earlier cp.async
// copies have landed
__device__ __forceinline__ void cp_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ uint64_t smem_desc_kmajor_sw128(uint32_t addr) {
    // tcgen05 shared-memory matrix descriptor of a K-major operand in the
    // 128-byte swizzled layout (8-row atoms of 128-byte rows, the 16-byte
    // chunks of row r XOR-ed with r % 8, atoms 1024-byte aligned): start
    // address, leading byte offset 16 (unused: an MMA's K = 16 halves stay
    // within one 128-byte row), stride byte offset 1024 (between 8-row
    // groups along N), version 1 at bit 46, swizzle mode 2 (128 B) at bit 61.
    // Stepping K inside the atom moves the start address by 32 bytes.
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(16 >> 4) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
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
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t sub_bf2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t mul_bf2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// 16-bit activations, scales, residuals and outputs: IEEE binary16, or
// bfloat16 (the top half of a binary32); storage is 16-bit either way
template <bool kBf16>
__device__ __forceinline__ float f16_to_float(__half h) {
    if constexpr (kBf16) return __uint_as_float((uint32_t)__half_as_ushort(h) << 16);
    else return __half2float(h);
}
template <bool kBf16>
__device__ __forceinline__ __half float_to_f16(float v) {  // nearest, ties to even
    if constexpr (kBf16) return __ushort_as_half(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
    else return __float2half_rn(v);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
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
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// the CTA's work: segments (a tile and a run of its stages), in order
// ---------------------------------------------------------------------------
struct Walk {
    long long pos, end;  // stream-K: the CTA's stage range
    int tile;            // whole tiles: the current tile
    bool started;
    int l;               // the linear of the current segment
};

__device__ __forceinline__ long long range_begin(const TcParams &p, int b) {
    return (long long)b * p.total / gridDim.x;
}

__device__ __forceinline__ void walk_init(const TcParams &p, Walk &w) {
    w.pos = range_begin(p, blockIdx.x);
    w.end = range_begin(p, blockIdx.x + 1);
    w.tile = blockIdx.x;
    w.started = false;
    w.l = 0;
}

// next segment: linear l, its tile t, stages [j0, j1) of it; false when the
// CTA is done.  Stream-K runs over the round's sequence of (linear, tile,
// stage); whole tiles (one linear only) go to the CTAs in turn.
__device__ __forceinline__ bool walk_next(const TcParams &p, const TcLinDesc *lins, int n_lin,
                                          Walk &w, int &l, int &t, int &j0, int &j1) {
    if (p.streamk) {
        if (w.pos >= w.end) return false;
        while (w.l + 1 < n_lin && w.pos >= lins[w.l + 1].start) ++w.l;
        l = w.l;
        const long long base = lins[l].start;
        const int spt = lins[l].spt;
        t = (int)((w.pos - base) / spt);
        const long long t0 = base + (long long)t * spt;
        j0 = (int)(w.pos - t0);
        const long long e = t0 + spt < w.end ? t0 + spt : w.end;
        j1 = (int)(e - t0);
        w.pos = e;
        return true;
    }
    if (w.started) w.tile += gridDim.x;
    w.started = true;
    if (w.tile >= lins[0].n_tiles) return false;
    l = 0;
    t = w.tile;
    j0 = 0;
    j1 = lins[0].spt;
    return true;
}

// groups of stage j: [4j, min(4j + 4, G))
__device__ __forceinline__ int stage_groups(const TcLinDesc &L, int j) {
    return min(kSG, L.G - kSG * j);
}

// Weight row of tile row r (0..127): rows 0..63 and 64..127 of a tile come as
// two TMA boxes of 64 rows.  A plain tile is 128 consecutive rows; with
// SiLU-and-mul it is 64 gate rows and the matching up rows N/2 below, so that
// both halves of 64 outputs meet in one tile.
__device__ __forceinline__ int tile_row(const TcLinDesc &L, int t, int r) {
    if (L.silu) return (r < 64 ? 0 : L.N / 2) + 64 * t + (r & 63);
    return kTileN * t + r;
}
// whether tile row r of tile t is a row of the weight matrix
__device__ __forceinline__ bool tile_row_valid(const TcLinDesc &L, int t, int r) {
    if (L.silu) return 64 * t + (r & 63) < L.N / 2;
    return kTileN * t + r < L.N;
}

// The CTA whose range holds stage st (stream-K).
__device__ __forceinline__ int cta_of(const TcParams &p, long long st) {
    return (int)(((st + 1) * (long long)gridDim.x - 1) / p.total);
}

// y[t0 .. t0 + 15][n] = v (+ residual), one rounding each.  The residual may
// be y itself (in place), so every residual value is read before any output
// is written: sixteen independent loads, one round trip, where a load after
// each store would wait for the store (the compiler must assume they alias).
template <bool kBf16>
__device__ __forceinline__ void store_y16(const TcLinDesc &L, int M, int n, int t0,
                                          const float (&v)[16]) {
    float res[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        res[i] = L.residual && t0 + i < M
                     ? f16_to_float<kBf16>(L.residual[(size_t)(t0 + i) * L.N + n])
                     : 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (t0 + i < M) L.y[(size_t)(t0 + i) * L.N + n] = float_to_f16<kBf16>(v[i] + res[i]);
}

// Whether CTA b's range begins strictly inside the tile whose first stage is
// tile0: then its segment of that tile is its first one and uses partial-sum
// slot 2b; any other partial segment of CTA b (its last one, which starts at a
// tile's first stage) uses slot 2b + 1.
__device__ __forceinline__ bool starts_inside(const TcParams &p, int b, long long tile0, int spt) {
    const long long rb = range_begin(p, b);
    return rb > tile0 && rb < tile0 + spt;
}

// A fused round with waits: linear w has finished once every tile of it has
// its outputs written (p.done[w] counts them).  Bounded: false on expiry.
__device__ __forceinline__ bool wait_linear(const TcParams &p, const TcLinDesc *lins, int w,
                                            volatile int *abort) {
    const volatile unsigned *d = p.done + w;
    const unsigned need = (unsigned)lins[w].n_tiles;
    const unsigned long long t0 = globaltimer();
    for (uint32_t i = 1; *d < need; ++i) {
        __nanosleep(64);
        if ((i & 15) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > kWaitNs) return false;
        }
    }
    // the writers fenced before they counted; order this thread's later
    // reads (and its TMA copies, the async proxy) after the count
    __threadfence();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// ---------------------------------------------------------------------------
// The outputs of row n over groups [g0, g1) for every token, exactly: w =
// (q - z) * s in fp32 (at most 15 significant bits), summed in increasing k,
// 16 tokens at a time; to y (a whole tile: plus the residual, if any, then one
// rounding) or to the partial-sum slot `part` (row n's column of it).  For
// rows whose scales reach 4096 (or are Inf or NaN), where the fp16 restore of
// the tensor-core path may overflow.  Kept
// out of line: it is rare, and its registers stay out of the kernel's.
// ---------------------------------------------------------------------------
template <bool kBf16>
__device__ __noinline__ void exact_row(const TcLinDesc &L, int M, int n, int g0, int g1,
                                       bool whole, float *part) {
    const uint32_t *qrow = L.qw + (size_t)n * (L.K / 8);
    for (int t0 = 0; t0 < M; t0 += 16) {
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
        for (int g = g0; g < g1; ++g) {
            const float sc = f16_to_float<kBf16>(L.scales[(size_t)n * L.G + g]);
            const int z = (int)((L.zeros[(size_t)n * L.ZW + (g >> 3)] >> (4 * (g & 7))) & 0xfu);
            for (int wd = 0; wd < kGroup / 8; ++wd) {
                const uint32_t word = qrow[g * (kGroup / 8) + wd];
                for (int nb = 0; nb < 8; ++nb) {
                    const int k = g * kGroup + wd * 8 + nb;
                    const float wv = (float)((int)((word >> (4 * nb)) & 0xfu) - z) * sc;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (t0 + i < M)
                            acc[i] = fmaf(wv, f16_to_float<kBf16>(L.x[(size_t)(t0 + i) * L.K + k]),
                                          acc[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int tt = t0 + i;
            if (tt >= M) break;
            if (!whole) {
                part[(size_t)tt * kTileN] = acc[i];
            } else {
                const size_t o = (size_t)tt * L.N + n;
                const float res = L.residual ? f16_to_float<kBf16>(L.residual[o]) : 0.f;
                L.y[o] = float_to_f16<kBf16>(acc[i] + res);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// kRound: a fused round (the linears' descriptors in device memory); else one
// linear, whose descriptor the kernel reads from its parameters
template <int T, bool kBf16, bool kRound>
__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ TcParams p) {
    using C = TcConfig<T, kBf16>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int NS = p.n_stages;
    uint8_t *sm_x = smem;                   // the x ring: kAStages slots of one group
    uint8_t *sm_stage = smem + C::kXRing;   // NS weight stages (32 KB, then the metadata)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm_stage + (size_t)NS * C::kStageBytes);
    uint64_t *full = bars;                     // [kMaxStages] weight stage landed
    uint64_t *empty = full + kMaxStages;       // [kMaxStages] weight stage read
    uint64_t *a_full = empty + kMaxStages;     // [kAStages] A restored
    uint64_t *a_empty = a_full + kAStages;     // [kAStages] A and x slot free (MMAs done)
    uint64_t *x_full = a_empty + kAStages;     // [kAStages] x slot landed
    uint64_t *d_full = x_full + kAStages;      // [2]
    uint64_t *d_empty = d_full + 2;            // [2]
    uint64_t *done = d_empty + 2;              // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_last = const_cast<int *>(abort + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dependents_launch();

    if (threadIdx.x == kTmaWarp * 32) {
        for (int i = 0; i < NS; ++i) {
            // the TMA bytes (one arrival), then each producer lane's metadata copies
            mbar_init(smem_u32(full + i), 1 + 32);
            mbar_init(smem_u32(empty + i), kDeqTeams * kDeqWarps);  // every restore warp
        }
        for (int i = 0; i < kAStages; ++i) {
            mbar_init(smem_u32(a_full + i), kDeqWarps);
            mbar_init(smem_u32(a_empty + i), 1);
            mbar_init(smem_u32(x_full + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(d_full + i), kMmaWarps);
            mbar_init(smem_u32(d_empty + i), kEpiWarps);
        }
        mbar_init(smem_u32(done), kMmaWarps);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!p.lins) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(
                             reinterpret_cast<uint64_t>(&p.single.wmap))
                         : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(
                             reinterpret_cast<uint64_t>(&p.single.xmap))
                         : "memory");
        }
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // the linears: the round's, or the one of this launch
    const TcLinDesc *lins = kRound ? p.lins : &p.single;
    const int n_lin = kRound ? p.n_lin : 1;
    Walk wk;
    walk_init(p, wk);
    int l = 0, t = 0, j0 = 0, j1 = 0;

    if (warp == kTmaWarp) {
        // ------------------------------------------------ weight producer
        // Lane 0 issues the TMA boxes; every lane copies, for 4 rows of the
        // tile, the stage's scale and zeros words (cp.async, completing on the
        // stage's barrier like the boxes).  A scale word past the end of the
        // array, or of a row past N, becomes zeros and reads nothing.
        uint64_t pol = 0;
        if (lane == 0)  // the weights are read once
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
        int sc = 0;  // stages issued
        bool ok = true;
        while (ok && walk_next(p, lins, kRound ? n_lin : 1, wk, l, t, j0, j1)) {
            const TcLinDesc &L = kRound ? p.lins[l] : p.single;
            const uintptr_t s_end = (uintptr_t)(L.scales + (size_t)L.N * L.G);
            const void *s_any = L.scales;  // a valid source for zero-byte copies
            for (int j = j0; j < j1; ++j, ++sc) {
                const int s = sc % NS;
                if (sc >= NS &&
                    !__all_sync(0xffffffffu, mbar_wait(smem_u32(empty + s), ((sc / NS) - 1) & 1,
                                                       abort))) {
                    if (lane == 0) fail(abort, p.status, kErrWaitEmpty);
                    ok = false;
                    break;
                }
                const uint32_t bar = smem_u32(full + s);
                uint8_t *st = sm_stage + (size_t)s * C::kStageBytes;
                if (lane == 0) {
                    // tile rows 0..63, then 64..127: [half][group][64 rows][64 bytes]
                    mbar_arrive_expect_tx(bar, (uint32_t)kStageW);
                    tma_load_3d(smem_u32(st), &L.wmap, 0, tile_row(L, t, 0), kSG * j, bar, pol);
                    tma_load_3d(smem_u32(st + kStageW / 2), &L.wmap, 0, tile_row(L, t, 64), kSG * j,
                                bar, pol);
                }
                uint8_t *m = st + kStageW;
#pragma unroll
                for (int i = 0; i < kTileN / 32; ++i) {
                    const int r = lane + 32 * i, n = tile_row(L, t, r);
                    const uint32_t dst = smem_u32(m + r * 16);
                    if (tile_row_valid(L, t, r)) {
                        const uintptr_t a0 =
                            (uintptr_t)(L.scales + (size_t)n * L.G + kSG * j) & ~(uintptr_t)3;
#pragma unroll
                        for (int w = 0; w < 3; ++w) {
                            const uintptr_t a = a0 + 4 * w;
                            cp4(dst + 4 * w, a < s_end ? (const void *)a : s_any,
                                a < s_end ? 4u : 0u);
                        }
                        cp4(dst + 12, L.zeros + (size_t)n * L.ZW + (kSG * j) / 8, 4u);
                    } else {
#pragma unroll
                        for (int w = 0; w < 4; ++w) cp4(dst + 4 * w, s_any, 0u);
                    }
                }
                cp_arrive_noinc(bar);
            }
        }
        // drain: every issued copy must have landed before the CTA exits
        if (lane == 0)
            for (int c = sc - NS > 0 ? sc - NS : 0; c < sc; ++c)
                if (!mbar_wait_drain(smem_u32(full + c % NS), (c / NS) & 1))
                    atomicOr(p.status, kErrDrain);
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp >= kMmaWarp) {
        // ------------------------------------------------ MMA issuers
        if (lane == 0) {
            const int me = warp - kMmaWarp;  // groups c with c % 4 == me: A buffer and x slot me
            int c = 0, q = 0;                // groups, segments seen
            bool ok = true;
            const uint32_t xb = smem_u32(sm_x + me * C::kXSlot);
            while (ok && walk_next(p, lins, kRound ? n_lin : 1, wk, l, t, j0, j1)) {
            const TcLinDesc &L = kRound ? p.lins[l] : p.single;
                const int dset = q % C::kDSets, duse = q / C::kDSets;
                if (!mbar_wait(smem_u32(d_empty + dset), (duse & 1) ^ 1, abort)) {
                    fail(abort, p.status, kErrWaitDEmpty);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem =
                    tmem + C::kDBase + dset * C::kDBuf + me * C::kChains * T;
                bool first = true;  // this issuer's first MMAs of the segment start its chains
                const int ng = min(L.G, kSG * j1) - kSG * j0;
                for (int gi = 0; gi < ng; ++gi, ++c) {
                    if ((c & (kMmaWarps - 1)) != me) continue;
                    const uint32_t use = (uint32_t)(c / kAStages) & 1;
                    if (!mbar_wait(smem_u32(a_full + me), use, abort)) {
                        fail(abort, p.status, kErrWaitAFull);
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(smem_u32(x_full + me), use, abort)) {
                        fail(abort, p.status, kErrWaitFull);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kGroup / 16; ++kk) {
                        // k 16 kk .. 16 kk + 15 of x: half kk / 4 of the slot (T
                        // rows of 128 bytes, swizzled), 32 bytes per k step
                        const uint64_t bdesc = smem_desc_kmajor_sw128(
                            xb + (uint32_t)((kk >> 2) * (T * 128) + (kk & 3) * 32));
                        // chain kk % kChains starts fresh with this issuer's first
                        // MMA of it in the segment
                        mma_f16_ts(d_tmem + (kk % C::kChains) * T, tmem + me * kACols + 8 * kk,
                                   bdesc, C::kIdesc, first && kk < C::kChains ? 0u : 1u);
                    }
                    first = false;
                    // the A buffer and the x slot are free once these MMAs are done
                    mma_commit(smem_u32(a_empty + me));
                }
                if (!ok) break;
                mma_commit(smem_u32(d_full + dset));
                ++q;
            }
            // all MMAs of this issuer complete before the tensor memory is freed
            mma_commit(smem_u32(done));
            if (!mbar_wait_drain(smem_u32(done), 0)) atomicOr(p.status, kErrDrain);
        }
    } else if (warp >= kEpiWarps) {
        // ------------------------------------------------ restore teams
        const int team = (warp - kEpiWarps) / kDeqWarps;  // groups c with c % kDeqTeams == team
        const int dw = (warp - kEpiWarps) % kDeqWarps;    // warp within the team
        const int quarter = warp & 3;                     // TMEM lanes 32 * quarter ..
        const int half0 = (dw >> 2) * kHalves;            // its first 64 inputs of the group
        const int r = quarter * 32 + lane;                // row within the tile
        const bool x_issuer = dw == 0 && lane == 0;       // loads x of the team's groups
        uint64_t pol_x = 0;
        if (x_issuer)  // x is read by every CTA
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
        bool dep_waited = false;
        int x_waited = -1;  // the last linear whose wait_for this thread has waited for
        // x copies this thread issued, per slot: whether any (bit a of xused) and
        // the parity of their count (bit a of xpar); bit masks, not an array
        // indexed at run time, which would live in local memory
        uint32_t xused = 0, xpar = 0;
        int c = 0, sc = 0;
        bool ok = true;
        while (ok && walk_next(p, lins, kRound ? n_lin : 1, wk, l, t, j0, j1)) {
            const TcLinDesc &L = kRound ? p.lins[l] : p.single;
            const int n = tile_row(L, t, r);
            const __half *srow = L.scales + (size_t)(tile_row_valid(L, t, r) ? n : 0) * L.G;
            for (int j = j0; j < j1 && ok; ++j, ++sc) {
                const int s = sc % NS, ng = stage_groups(L, j);
                const uint8_t *st = sm_stage + (size_t)s * C::kStageBytes;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(full + s), (sc / NS) & 1, abort))) {
                    fail(abort, p.status, kErrWaitFull);
                    ok = false;
                    break;
                }
                // this row's words of the team's group of the stage (at most
                // kPerTeam: group gi of the stage is team (c + gi) % kDeqTeams's),
                // read at once so that the stage is free for the next box early;
                // 16-byte chunks 2 half and 2 half + 1 of a row, stored 64-byte
                // swizzled (chunk ^= (row >> 1) & 3)
                const int gfirst = ((team - c) % kDeqTeams + kDeqTeams) % kDeqTeams;
                const int sw = (r >> 1) & 3;
                uint4 w[kPerTeam][kHalves][2];
#pragma unroll
                for (int k2 = 0; k2 < kPerTeam; ++k2) {
                    const int gi = gfirst + kDeqTeams * k2;
                    if (gi < ng) {
                        const uint8_t *rowp =
                            st + (r >> 6) * (kStageW / 2) + gi * (kGroupBytes / 2) + (r & 63) * 64;
#pragma unroll
                        for (int hf = 0; hf < kHalves; ++hf) {
                            const int half = half0 + hf;
                            w[k2][hf][0] = *reinterpret_cast<const uint4 *>(rowp + 16 * ((2 * half) ^ sw));
                            w[k2][hf][1] =
                                *reinterpret_cast<const uint4 *>(rowp + 16 * ((2 * half + 1) ^ sw));
                        }
                    }
                }
                // its scale words and zeros word; its 4 scales start at byte
                // `off` of the words (rows past N: all zero)
                const uint4 md = *reinterpret_cast<const uint4 *>(st + kStageW + r * 16);
                // every read of the stage comes before the next copies into it
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(empty + s));
                const uint32_t off = (uint32_t)((uintptr_t)(srow + kSG * j) & 2);
                const uint32_t zsh = 4u * (uint32_t)((kSG * j) & 7);  // the stage's first nibble
                // the team's groups of the stage are restored one after the
                // other and their tensor-memory stores waited for once: the
                // store latency is paid once per stage, not per group
                int done_a[kPerTeam];
#pragma unroll
                for (int k2 = 0; k2 < kPerTeam; ++k2) done_a[k2] = -1;
#pragma unroll
                for (int k2 = 0; k2 < kPerTeam; ++k2) {
                    const int gi = gfirst + kDeqTeams * k2;
                    if (gi >= ng) break;
                    const int cg = c + gi;  // the group's number in the CTA's sequence
                    const int a = cg % kAStages;
                    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(a_empty + a),
                                                           ((cg / kAStages) & 1) ^ 1, abort))) {
                        fail(abort, p.status, kErrWaitAEmpty);
                        ok = false;
                        break;
                    }
                    // the MMAs that read A[a] and x slot a have completed (commit)
                    tc_fence_after();
                    if (x_issuer) {
                        // x of this group into slot a; x is written by the
                        // preceding kernel: wait for it once
                        if (!dep_waited) {
                            grid_dependency_wait();
                            dep_waited = true;
                        }
                        // a round with waits: x may be an earlier linear's output
                        if (kRound && p.done && L.wait_for >= 0 && l != x_waited) {
                            x_waited = l;
                            if (!wait_linear(p, lins, L.wait_for, abort))
                                fail(abort, p.status, kErrWaitLinear);
                        }
                        const uint32_t xbar = smem_u32(x_full + a);
                        mbar_arrive_expect_tx(xbar, (uint32_t)C::kXSlot);
                        const int k0 = (kSG * j + gi) * kGroup;
                        tma_load_2d(smem_u32(sm_x + a * C::kXSlot), &L.xmap, k0, 0, xbar, pol_x);
                        tma_load_2d(smem_u32(sm_x + a * C::kXSlot + T * 128), &L.xmap, k0 + 64, 0,
                                    xbar, pol_x);
                        xused |= 1u << a;
                        xpar ^= 1u << a;
                    }
                    const uint32_t bp = off + 2u * gi;  // byte of the scale in the words
                    // the word holding it (selected, not indexed: no local memory)
                    const uint32_t sw4 = bp >> 2;
                    const uint32_t sword = sw4 == 0 ? md.x : (sw4 == 1 ? md.y : md.z);
                    const uint32_t sbits = (sword >> (8u * (bp & 2u))) & 0xffffu;
                    const uint32_t z = (md.w >> (zsh + 4u * gi)) & 0xfu;
                    const uint32_t zz_hi = 0x64006400u | z | (z << 16);
                    const uint32_t zz_lo = 0x54005400u | (z << 4) | (z << 20);
                    const uint32_t zz_b = 0x43004300u | z | (z << 16);  // bf16 (128 + z) pair
                    const uint32_t ss = sbits | (sbits << 16);
                    // 16 columns (4 words) per store, so that few values are live
#pragma unroll
                    for (int hh = 0; hh < 2 * kHalves; ++hh) {
                        const int hf = hh >> 1, hw = hh & 1;
                        const uint32_t words[4] = {w[k2][hf][hw].x, w[k2][hf][hw].y,
                                                   w[k2][hf][hw].z, w[k2][hf][hw].w};
                        uint32_t v[16];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t wd = words[u], w8 = wd >> 8;
                            // (q - z) exact, then times s rounded once: the pairs
                            // (q0,q4) (q1,q5) (q2,q6) (q3,q7) of the word ...
                            uint32_t r0, r1, r2, r3;
                            if constexpr (kBf16) {
                                // a nibble at mantissa bits 0..3 of bf16 128.0 is
                                // 128 + q (bf16 has 7 mantissa bits); minus 128 + z
                                r0 = mul_bf2(sub_bf2(lop3_and_or(wd, 0x000f000fu, 0x43004300u), zz_b), ss);
                                r1 = mul_bf2(sub_bf2(lop3_and_or(wd >> 4, 0x000f000fu, 0x43004300u), zz_b), ss);
                                r2 = mul_bf2(sub_bf2(lop3_and_or(w8, 0x000f000fu, 0x43004300u), zz_b), ss);
                                r3 = mul_bf2(sub_bf2(lop3_and_or(wd >> 12, 0x000f000fu, 0x43004300u), zz_b), ss);
                            } else {
                                r0 = hmul2(hsub2(lop3_and_or(wd, 0x000f000fu, 0x64006400u), zz_hi), ss);
                                r1 = hmul2(hsub2(lop3_and_or(wd, 0x00f000f0u, 0x54005400u), zz_lo), ss);
                                r2 = hmul2(hsub2(lop3_and_or(w8, 0x000f000fu, 0x64006400u), zz_hi), ss);
                                r3 = hmul2(hsub2(lop3_and_or(w8, 0x00f000f0u, 0x54005400u), zz_lo), ss);
                            }
                            // ... in k order, (q0,q1) (q2,q3) (q4,q5) (q6,q7): the
                            // order of x in memory, which the TMA box keeps
                            v[4 * u + 0] = prmt(r0, r1, 0x5410);
                            v[4 * u + 1] = prmt(r2, r3, 0x5410);
                            v[4 * u + 2] = prmt(r0, r1, 0x7632);
                            v[4 * u + 3] = prmt(r2, r3, 0x7632);
                        }
                        tmem_st_x16(tmem + ((uint32_t)(quarter * 32) << 16) + a * kACols +
                                        32 * (half0 + hf) + 16 * hw, v);
                    }
                    done_a[k2] = a;
                }
                if (done_a[0] >= 0) {
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int k2 = 0; k2 < kPerTeam; ++k2)
                            if (done_a[k2] >= 0) mbar_arrive(smem_u32(a_full + done_a[k2]));
                    }
                }
                c += ng;
            }
        }
        // the x copies this thread issued land before the CTA exits: each is
        // waited for by its MMA issuer, or, after an abort, here (bounded)
        if (x_issuer && !ok)
            for (int a = 0; a < kAStages; ++a)
                if (((xused >> a) & 1u) &&
                    !mbar_wait_drain(smem_u32(x_full + a), ((xpar >> a) & 1u) ^ 1u))
                    atomicOr(p.status, kErrDrain);
    } else {
        // ------------------------------------------------ epilogue (warps 0..3)
        const int r = warp * 32 + lane;  // row within the tile; TMEM lanes of this warp
        // outputs, partial sums and counters may belong to the preceding kernel
        grid_dependency_wait();
        int c = 0, q = 0;
        int waited = -1;  // the last linear whose wait_for this role has waited for
        bool ok = true;
        while (ok && walk_next(p, lins, kRound ? n_lin : 1, wk, l, t, j0, j1)) {
            const TcLinDesc &L = kRound ? p.lins[l] : p.single;
            const int dset = q % C::kDSets, duse = q / C::kDSets;
            const int n = tile_row(L, t, r);
            const bool vrow = tile_row_valid(L, t, r);
            const int g0 = kSG * j0, g1 = min(L.G, kSG * j1);
            const int c0 = c;
            c += g1 - g0;
            // while the MMAs run: does a scale of this row in the range reach
            // 4096 (or Inf, NaN)?  Then the fp16 restore may overflow, and the
            // row is recomputed exactly below.
            bool big = false;
            if (vrow) {
                const unsigned short *sr =
                    reinterpret_cast<const unsigned short *>(L.scales) + (size_t)n * L.G;
                const uint32_t lim = kBf16 ? kBigScaleBf16 : kBigScale;
                for (int g = g0; g < g1; ++g) big |= (sr[g] & 0x7fffu) >= lim;
            }
            if (kRound && p.done && L.wait_for >= 0 && l != waited) {
                // a round with waits: what this linear writes (and its residual
                // and x, which the exact path reads) may belong to an earlier
                // linear: wait until it has finished
                waited = l;
                bool fine = true;
                if (threadIdx.x == 0) fine = wait_linear(p, lins, L.wait_for, abort);
                if (!fine) fail(abort, p.status, kErrWaitLinear);
                asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
                if (*abort) {
                    ok = false;
                    break;
                }
            }
            if (!__all_sync(0xffffffffu,
                            mbar_wait(smem_u32(d_full + dset), duse & 1, abort))) {
                fail(abort, p.status, kErrWaitDFull);
                ok = false;
                break;
            }
            tc_fence_after();
            const bool whole = j0 == 0 && j1 == L.spt;
            // y straight from the sums: a whole tile without SiLU-and-mul.  Else
            // the sums go to this CTA's partial-sum slot: part of a tile (the
            // last CTA of the tile adds the slots in K order, which is CTA
            // order), or a whole SiLU-and-mul tile, whose gate and up rows
            // meet there (slot 2b + 1 for it: this CTA's last partial segment,
            // which also uses it, comes after every whole one)
            const bool direct = whole && !L.silu;
            const long long tile0 = L.start + (long long)t * L.spt;  // its first stage
            const int slot =
                2 * (int)blockIdx.x +
                (whole || !starts_inside(p, blockIdx.x, tile0, L.spt) ? 1 : 0);
            float *part = p.partials + (size_t)slot * p.M * kTileN + r;
            // 16 tokens' outputs of this row: y = h (+ residual), one rounding,
            // or the partial sums
            auto put16 = [&](int t0, float (&v)[16]) {
                if (direct) {
                    if (vrow) store_y16<kBf16>(L, p.M, n, t0, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (t0 + i < p.M) part[(size_t)(t0 + i) * kTileN] = v[i];
                }
            };
            const uint32_t taddr =
                tmem + ((uint32_t)(warp * 32) << 16) + C::kDBase + dset * C::kDBuf;
#pragma unroll
            for (int t0 = 0; t0 < T; t0 += 16) {
                // issuer 0's chains in order, then issuer 1's, ... (a fixed
                // order); issuer i holds sums when the range has a group c with
                // c % 4 == i
                float sum[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) sum[i] = 0.f;
#pragma unroll
                for (int iss = 0; iss < kMmaWarps; ++iss) {
                    const bool valid = g1 - g0 >= kMmaWarps ||
                                       ((iss - c0) % kMmaWarps + kMmaWarps) % kMmaWarps < g1 - g0;
#pragma unroll
                    for (int ch = 0; ch < C::kChains; ++ch) {
                        float a0[16];
                        tmem_ld_x16(taddr + (iss * C::kChains + ch) * T + t0, a0);
                        tmem_wait_ld();
                        if (valid) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) sum[i] += a0[i];
                        }
                    }
                }
                if (!big) put16(t0, sum);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(d_empty + dset));
            // a row whose scales may overflow the fp16 restore: exact on the CUDA cores
            if (big) exact_row<kBf16>(L, p.M, n, g0, g1, direct, part);
            if (kRound && direct && p.done) {
                // a round with waits: this tile's outputs are all written
                __threadfence();
                asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
                if (threadIdx.x == 0) atomicAdd(p.done + l, 1u);
            }
            if (!direct) {
                __threadfence();
                asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
                // the CTAs whose slots hold the tile's sums: this one (a whole
                // tile), or every CTA whose range meets the tile
                const int b0 = whole ? (int)blockIdx.x : cta_of(p, tile0);
                const int b1 = whole ? (int)blockIdx.x : cta_of(p, tile0 + L.spt - 1);
                if (!whole) {
                    if (threadIdx.x == 0) {
                        const unsigned prev = atomicAdd(L.counters + t, 1u);
                        *s_last = prev == (unsigned)(b1 - b0) ? 1 : 0;
                    }
                    asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
                }
                if (whole || *s_last) {
                    __threadfence();
                    // the sums of tile row rr over the slots in K order (CTA
                    // order), 16 tokens per batch of independent loads (one
                    // round trip each, not one per token and piece)
                    auto gather = [&](int rr, int t0, float (&sum)[16]) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) sum[i] = 0.f;
                        for (int b = b0; b <= b1; ++b) {
                            const int sl =
                                2 * b + (whole || !starts_inside(p, b, tile0, L.spt) ? 1 : 0);
                            const float *src = p.partials + ((size_t)sl * p.M + t0) * kTileN + rr;
                            float v[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                v[i] = t0 + i < p.M ? __ldcg(src + (size_t)i * kTileN) : 0.f;
#pragma unroll
                            for (int i = 0; i < 16; ++i) sum[i] += v[i];
                        }
                    };
                    if (!L.silu) {
                        if (vrow) {
                            for (int t0 = 0; t0 < p.M; t0 += 16) {
                                float sum[16];
                                gather(r, t0, sum);
                                store_y16<kBf16>(L, p.M, n, t0, sum);
                            }
                        }
                    } else if (r < 64 && vrow) {
                        // SiLU-and-mul: the gate row's thread takes its up row
                        // (tile row r + 64): y = silu(g) * u, silu(g) = g / (1 + e^-g)
                        const int ycols = L.N / 2, jcol = 64 * t + r;
                        for (int t0 = 0; t0 < p.M; t0 += 16) {
                            float gs[16], us[16];
                            gather(r, t0, gs);
                            gather(r + 64, t0, us);
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                if (t0 + i >= p.M) continue;
                                const float g = gs[i];
                                L.y[(size_t)(t0 + i) * ycols + jcol] =
                                    float_to_f16<kBf16>(us[i] * (g / (1.f + expf(-g))));
                            }
                        }
                    }
                    if (!whole && threadIdx.x == 0) L.counters[t] = 0u;  // ready for the next launch
                }
                // the slot and s_last are written again only after the next such
                // segment's first barrier, which every epilogue thread reaches
                // after its reads
                if (kRound && p.done) __threadfence();
                asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
                // a round with waits: the tile's outputs are all written
                if (kRound && p.done && threadIdx.x == 0 && (whole || *s_last)) atomicAdd(p.done + l, 1u);
            }
            ++q;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (kRound && p.done && threadIdx.x == 0) {
        // a round with waits: the last CTA out zeroes the linears' counters
        // (every wait of every CTA is over by then) for the next launch
        __threadfence();
        if (atomicAdd(p.done + n_lin, 1u) == gridDim.x - 1) {
            for (int i = 0; i < n_lin; ++i) p.done[i] = 0u;
            p.done[n_lin] = 0u;
            __threadfence();
        }
    }
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int T>
int stages_for() {
    int ns = (kSmemBudget - TcConfig<T>::kXRing - kBarBytes) / TcConfig<T>::kStageBytes;
    return ns > kMaxStages ? kMaxStages : ns;
}

template <int T>
int smem_for(int ns) {
    return 1024 /*align slack*/ + TcConfig<T>::kXRing + ns * TcConfig<T>::kStageBytes + kBarBytes;
}

cudaLaunchConfig_t pdl_config(dim3 grid, int threads, int smem, cudaStream_t stream,
                              cudaLaunchAttribute *attr) {
    // programmatic dependent launch: the grid may start while the previous
    // kernel in the stream drains; it waits for it (griddepcontrol) before
    // touching what that kernel may read or write
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int T>
cudaError_t launch_t(const TcParams &p, bool bf16, int grid, bool cooperative,
                     cudaStream_t stream) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pdl_config(dim3(grid), kThreads, smem_for<T>(p.n_stages), stream, attr);
    if (cooperative) {
        // linears wait for earlier ones: every CTA must be resident at once
        attr[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
        attr[cfg.numAttrs].val.cooperative = 1;
        cfg.numAttrs += 1;
    }
    if (p.lins)
        return bf16 ? cudaLaunchKernelEx(&cfg, tc_kernel<T, true, true>, p)
                    : cudaLaunchKernelEx(&cfg, tc_kernel<T, false, true>, p);
    return bf16 ? cudaLaunchKernelEx(&cfg, tc_kernel<T, true, false>, p)
                : cudaLaunchKernelEx(&cfg, tc_kernel<T, false, false>, p);
}

}  // namespace

TcPlan plan_tc(int M, int N, int K, int split, const DeviceInfo &dev, int epi) {
    TcPlan pl{};
    pl.M = M;
    pl.T = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    const int G = K / kGroup;
    const bool silu = epi == kEpiSiluMul;
    // SiLU-and-mul: 64 outputs (their gate and up rows) per tile
    pl.n_tiles = silu ? (N / 2 + 63) / 64 : (N + kTileN - 1) / kTileN;
    pl.spt = (G + kSG - 1) / kSG;
    pl.stages = pl.T == 16 ? stages_for<16>() : (pl.T == 32 ? stages_for<32>() : stages_for<64>());
    const long long total = (long long)pl.n_tiles * pl.spt;
    const int slots = dev.sm_count;  // one CTA per SM
    // whole tiles unless they leave SMs idle for long: with n tiles on s SMs
    // the busiest SM streams ceil(n / s) tiles against n / s on average.  From
    // 17 tokens on, a single wave of tiles with few stages each stays whole:
    // there the pieces' partial sums (M x 128 fp32 per piece) cost more than
    // the idle SMs (one launch, L2 evicted, M = 24: N 8192, K 4096, 8 stages a
    // tile: 24.8 us whole against 30.7 split; N 4096, K 2048: 17.9 against
    // 20.7), while 16 stages a tile and more still gain from the split (N 1024,
    // K 8192: 31.0 split against 42.0)
    bool streamk = split == 1;
    if (split < 0) {
        const double rounds = (double)((pl.n_tiles + slots - 1) / slots);
        streamk = (double)pl.n_tiles / slots < 0.9 * rounds && pl.spt > 1;
        if (M > 16 && pl.n_tiles <= slots && pl.spt < 12) streamk = false;
    }
    pl.S = streamk ? 2 : 1;
    if (streamk) pl.grid = total < slots ? (int)total : slots;
    else pl.grid = pl.n_tiles < slots ? pl.n_tiles : slots;
    // partial-sum slots: split tiles, and whole SiLU-and-mul tiles (where the
    // gate and up rows meet)
    pl.ws_bytes = streamk || silu ? (size_t)2 * pl.grid * M * kTileN * sizeof(float) : 0;
    pl.threads = kThreads;
    pl.ok = G >= 1 && pl.stages >= 2;
    return pl;
}

cudaError_t tc_init(const DeviceInfo &dev) {
    (void)dev;
    if (!tensor_map_encoder()) return cudaErrorSymbolNotFound;
    const void *fns[12] = {
        (const void *)tc_kernel<16, false, false>, (const void *)tc_kernel<32, false, false>,
        (const void *)tc_kernel<64, false, false>, (const void *)tc_kernel<16, true, false>,
        (const void *)tc_kernel<32, true, false>,  (const void *)tc_kernel<64, true, false>,
        (const void *)tc_kernel<16, false, true>,  (const void *)tc_kernel<32, false, true>,
        (const void *)tc_kernel<64, false, true>,  (const void *)tc_kernel<16, true, true>,
        (const void *)tc_kernel<32, true, true>,   (const void *)tc_kernel<64, true, true>};
    const int smem[3] = {smem_for<16>(stages_for<16>()), smem_for<32>(stages_for<32>()),
                         smem_for<64>(stages_for<64>())};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 12 && e == cudaSuccess; ++i)
        e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, smem[i % 3]);
    return e;
}

cudaError_t tc_describe(const LinearArgs &a, int T, TcLinDesc *d) {
    const EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorInitializationError;
    memset(d, 0, sizeof(*d));
    const int G = a.K / kGroup;
    {
        // qweight as (word in group, row, group): a box of 64 rows x 4 groups
        // (a tile's stage is two of them)
        const cuuint64_t dims[3] = {16, (cuuint64_t)a.N, (cuuint64_t)G};
        const cuuint64_t strides[2] = {(cuuint64_t)a.K / 2, 64};
        const cuuint32_t box[3] = {16, (cuuint32_t)(kTileN / 2), (cuuint32_t)kSG};
        const cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = encode(&d->wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, (void *)a.qw, dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        // x as (K, token): a box of 64 k x T tokens lands as T rows of 128
        // bytes, 128-byte swizzled, the MMA's K-major swizzled layout (one
        // 128-byte request per token; 16-byte rows cost 8 requests each);
        // tokens past M read zeros
        const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
        const cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)T};
        const cuuint32_t estr[2] = {1, 1};
        CUresult r = encode(&d->xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void *)a.x, dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    d->x = a.x;
    d->qw = a.qw;
    d->scales = a.scales;
    d->zeros = a.zeros;
    d->y = a.y;
    d->residual = a.epi == kEpiResidual ? a.residual : nullptr;
    d->N = a.N;
    d->K = a.K;
    d->G = G;
    d->ZW = (G + 7) / 8;
    d->silu = a.epi == kEpiSiluMul;
    d->wait_for = -1;
    return cudaSuccess;
}

cudaError_t launch_tc(const LinearArgs &a, const TcPlan &plan, const Workspace &ws, int *status,
                      cudaStream_t stream) {
    const bool bf16 = a.dtype == kDtypeBf16;
    TcParams p;
    memset(&p, 0, sizeof(p));
    cudaError_t e = tc_describe(a, plan.T, &p.single);
    if (e != cudaSuccess) return e;
    p.single.counters = ws.counters;
    p.single.n_tiles = plan.n_tiles;
    p.single.spt = plan.spt;
    p.single.start = 0;
    p.lins = nullptr;
    p.n_lin = 1;
    p.done = nullptr;
    p.partials = ws.partials;
    p.status = status;
    p.M = a.M;
    p.streamk = plan.S > 1;
    p.n_stages = plan.stages;
    p.total = (long long)plan.n_tiles * plan.spt;
    switch (plan.T) {
        case 16: return launch_t<16>(p, bf16, plan.grid, false, stream);
        case 32: return launch_t<32>(p, bf16, plan.grid, false, stream);
        case 64: return launch_t<64>(p, bf16, plan.grid, false, stream);
    }
    return cudaErrorInvalidValue;
}

bool plan_tc_round(int M, const int *N, const int *K, const int *epi, int n, const DeviceInfo &dev,
                   TcRound *r, TcLinDesc *descs, size_t *ws_floats) {
    if (M < 1 || M > kTcMaxTokens || n < 1) return false;
    memset(r, 0, sizeof(*r));
    r->n = n;
    r->M = M;
    r->T = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    r->stages = r->T == 16 ? stages_for<16>() : (r->T == 32 ? stages_for<32>() : stages_for<64>());
    if (r->stages < 2) return false;
    // one stream-K sequence: linear after linear, tile after tile, stage after stage
    long long total = 0;
    for (int l = 0; l < n; ++l) {
        const int G = K[l] / kGroup;
        if (G < 1) return false;
        descs[l].n_tiles = epi[l] == kEpiSiluMul ? (N[l] / 2 + 63) / 64 : (N[l] + kTileN - 1) / kTileN;
        descs[l].spt = (G + kSG - 1) / kSG;
        descs[l].start = total;
        total += (long long)descs[l].n_tiles * descs[l].spt;
    }
    r->total = total;
    r->grid = total < dev.sm_count ? (int)total : dev.sm_count;
    // partial-sum slots: two per CTA (its first and last segments), shared by the linears
    *ws_floats = (size_t)2 * r->grid * M * kTileN;
    return true;
}

cudaError_t launch_tc_round(const TcRound &r, int *status, cudaStream_t stream) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    p.lins = r.descs;
    p.n_lin = r.n;
    p.done = r.done;
    p.partials = r.partials;
    p.status = status;
    p.M = r.M;
    p.streamk = 1;
    p.n_stages = r.stages;
    p.total = r.total;
    const bool coop = r.done != nullptr;
    switch (r.T) {
        case 16: return launch_t<16>(p, r.bf16, r.grid, coop, stream);
        case 32: return launch_t<32>(p, r.bf16, r.grid, coop, stream);
        case 64: return launch_t<64>(p, r.bf16, r.grid, coop, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace w4a16
