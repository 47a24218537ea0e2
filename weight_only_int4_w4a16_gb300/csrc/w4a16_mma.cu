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
//   * every warp runs its own two-slot ring: it waits for a slot, computes
//     the stage from it and then refills it two stages ahead, after a
//     generic-to-async proxy fence (the lanes' shared-memory reads must be
//     ordered before the TMA's writes into the same slot);
//   * the unpack is one lop3 per pair of nibbles and adds no bias: a nibble at
//     bits 0..3 of an fp16 half is the subnormal q * 2^-24, at bits 4..7 it is
//     q * 2^-20, both exact.  The pairs (q0,q4) (q2,q6) of a word feed one
//     MMA chain (D_lo, scale 2^-24) and (q1,q5) (q3,q7) another (D_hi, scale
//     2^-20); the MMA k slots stand for k0,k4,k2,k6 and k1,k5,k3,k7, and x is
//     staged once per CTA in the same order;
//   * the zero point leaves the per-weight work: sum_k (q - z) x = sum_k q x
//     - z * S with S the group's sum of x (per token, computed once per CTA
//     when x is staged).  Per group
//         acc += s * (16 * D_lo + D_hi - z * S * 2^-20)
//     and y = 2^20 * acc, which is sum_g s_g * sum_k (q - z) x;
//   * work comes in units: one K slice of R strips per warp.  CTAs are
//     persistent and take units round-robin (or from a shared counter in a
//     fused round); per unit a CTA stages that slice of x (with each group's
//     sums of x) and its warps stream their strips, while each warp's copy
//     stream already runs ahead into its next unit;
//   * a CTA is 8 warps, two per SM, or 16 warps, one per SM: the larger CTA
//     has twice the shared memory for staged x (the x of a K 5120 slice of 8
//     tokens fits beside its 16 rings, where an 8-warp CTA must cut K in
//     two), the smaller lets one CTA stream while the other crosses a unit
//     boundary;
//   * a fused decode round is one launch over the units of all its linears
//     in order: the weight stream does not stop between linears.  Where a
//     linear reads activations an earlier one writes (or the like), it waits
//     on per-linear completion counters before staging them;
//   * split K: fp32 partials and a last-arriving-warp reduction in slice
//     order (deterministic, no warp waits for another).
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "../../include/w4a16.h"
#include "w4a16_device.cuh"
#include "w4a16_internal.h"
#include "w4a16_mma_common.cuh"

namespace w4a16 {
namespace {

using namespace warp_mma;

constexpr int kStageGroups = 4;                 // groups per box
constexpr int kDepth = 2;                       // ring slots per warp
constexpr int kStageW = kStageGroups * 16 * 64;  // 4 KB of weights
constexpr int kStageMeta = 16 * 16;             // per row: 3 scale words, 1 zeros word
constexpr int kStageBytes = kStageW + kStageMeta;
// A unit of the CTA's queue, decoded once by thread 0 into shared memory:
// everything the warps need of the unit and of its linear, so that none of
// them reads a descriptor from global memory on its way.
struct UnitInfo {
    uint64_t tmap;  // address of the linear's tensor map
    const __half *x;
    const __half *scales;
    const uint32_t *zeros;
    __half *y;
    float *partials;
    unsigned *counters;
    uintptr_t scales_first, scales_end;
    const __half *residual;
    int l, slice, sb;  // linear, K slice, strip block (l < 0: the queue has ended)
    int N, K, G, ZW, M, S, slice_groups, n_strips, strips_per_warp, xstride, wait_for;
    int epi, ycols, half_strips;
    int seq;  // the queue position this entry holds (written last)
};
constexpr int kSlots = 8;  // one per queue position (mod 8)
// ring barriers, then 16 flag ints, then the barrier of the x copies, then
// the decoded units
// The CTA's shape: W = 8 warps (two CTAs per SM) or 16 warps (one CTA per SM,
// with the whole SM's shared memory: room for the x of a K 5120 slice of 8
// tokens beside the 16 warps' rings, where two 8-warp CTAs must cut it in
// two).  An SM runs 16 warps either way.
template <int W>
struct CtaShape {
    static constexpr int kWarps = W;
    static constexpr int kThreads = W * 32;
    static constexpr int kCtasPerSm = 16 / W;
    static constexpr int kRingBytes = W * kDepth * kStageBytes;  // 69632 for 8 warps
    static constexpr int kSlotOffset = W * kDepth * 8 + 64 + 16;
    static constexpr int kBarBytes = kSlotOffset + kSlots * (int)sizeof(UnitInfo);
    static constexpr int kSmemPerCta = 228 * 1024 / kCtasPerSm - 1024;  // the per-CTA reserve
};
// the shape's constants as locals of a function templated on W
#define W4A16_CTA_SHAPE(W)                                          \
    constexpr int kWarps = CtaShape<W>::kWarps;                     \
    constexpr int kThreads = CtaShape<W>::kThreads;                 \
    constexpr int kRingBytes = CtaShape<W>::kRingBytes;             \
    constexpr int kSlotOffset = CtaShape<W>::kSlotOffset;           \
    constexpr int kBarBytes = CtaShape<W>::kBarBytes;               \
    (void)kWarps, (void)kThreads, (void)kRingBytes, (void)kSlotOffset, (void)kBarBytes
constexpr int kMaxSliceGroups = 128;
constexpr int kRoundStripsPerWarp = 8;  // fused rounds: strips per warp and unit
constexpr int kErrMmaWait = 128;  // device status bit: a ring wait expired
constexpr int kErrMmaDep = 256;   // device status bit: a wait for an earlier linear expired

struct MmaKernelParams {
    MmaLinDesc single;         // the linear of a one-linear launch
    const MmaLinDesc *descs;   // fused round: device array of n_lin linears
    unsigned *done;            // fused round with waits: n_lin completion counters, else null
    unsigned *sched;           // 2 zeroed words: next dynamic unit, CTAs finished
    int *status;
    int n_lin;
    int total_units;
    int dynamic;  // units after the first two: 0 = every grid-th, 1 = from *sched
    // descriptors written by the preceding kernel (expert groups): n_lin and
    // total_units are upper bounds, counts[1] the units that exist (the
    // unused descriptors start past every unit); thread 0 waits for that
    // kernel before it reads them
    const int *counts;
};

// Ints of the CTA's flag area in shared memory
constexpr int kFlagAbort = 0;   // a wait expired: the CTA's warps stop at their next unit
constexpr int kFlagRed = 2;     // 2 x 3 ints: whether this CTA reduces a block, its linear and block
constexpr int kFlagQueue = 8;   // 8 ints: the CTA's units by sequence index (mod 8)
constexpr int kQueueAhead = 1;  // units fetched ahead of the one being consumed

// The epilogue of one output: y = h, h + residual, or silu(gate) * h (the
// up projection h and its gate both in fp32; silu(g) = g / (1 + e^-g)).
template <bool kBf16, class Lin>
__device__ __forceinline__ void epilogue_store(const Lin &R, size_t o, float h, float gate) {
    if (R.epi == kEpiResidual) h += to_float<kBf16>(R.residual[o]);
    else if (R.epi == kEpiSiluMul) h *= gate / (1.f + expf(-gate));
    R.y[o] = from_float<kBf16>(h);
}

// y = the epilogue of the sum of the S partial slices of block sb of a linear,
// by the whole CTA.  With SiLU-and-mul an output needs its gate row and its up
// row: half of the sums a thread keeps are gate rows, the other half the up
// rows of the same outputs (the register footprint stays that of 8 sums: the
// callers keep their registers across this call).
template <bool kBf16, int W>
__device__ __forceinline__ void reduce_block(const MmaLinDesc &R, int sb) {
    W4A16_CTA_SHAPE(W);
    const int rows_per_block = kWarps * R.strips_per_warp * 16;
    const int row0 = sb * rows_per_block;
    const int nrows = min(R.ycols - row0, rows_per_block);
    const int n_out = R.M * nrows;
    const bool silu = R.epi == kEpiSiluMul;
    const size_t up = (size_t)R.half_strips * 16;  // the up rows sit N/2 below the gate rows
    // each thread sums up to 8 rows at a time, the 8 loads of one slice in
    // flight together (slices in order: the sum is the same every launch)
    constexpr int kR = 8, kH = kR / 2;
    const int per = silu ? kH : kR;  // outputs per thread and pass
    for (int base = 0; base < n_out; base += kThreads * per) {
        float sum[kR];
        size_t off[kR];
#pragma unroll
        for (int j = 0; j < kR; ++j) {
            const int jo = silu ? (j & (kH - 1)) : j;  // the output of sum j
            const int i = base + jo * kThreads + threadIdx.x;
            const int t = i / nrows, row = row0 + i - t * nrows;
            off[j] = i < n_out ? (size_t)t * R.N + row + (silu && j >= kH ? up : 0) : 0;
            sum[j] = 0.f;
        }
        for (int s2 = 0; s2 < R.S; ++s2) {
            const float *ps = R.partials + (size_t)s2 * R.M * R.N;
            float v[kR];
#pragma unroll
            for (int j = 0; j < kR; ++j) v[j] = __ldcg(ps + off[j]);
#pragma unroll
            for (int j = 0; j < kR; ++j) sum[j] += v[j];
        }
#pragma unroll
        for (int j = 0; j < kR; ++j) {
            const int i = base + j * kThreads + threadIdx.x;
            if ((silu && j >= kH) || i >= n_out) continue;
            const int t = i / nrows, row = row0 + i - t * nrows;
            const size_t o = (size_t)t * R.ycols + row;
            if (silu) epilogue_store<kBf16>(R, o, sum[j + kH], sum[j]);
            else epilogue_store<kBf16>(R, o, sum[j], 0.f);
        }
    }
    if (threadIdx.x == 0) R.counters[sb] = 0u;  // ready for the next launch
}

// The same reduction with the partial sums staged in shared memory.  The sum
// is latency-bound when each thread loads a few floats per round trip to L2
// (one slice after another), so each thread first copies its share of the
// block's slices into shared memory with 16-byte cp.async copies (as many rows
// at a time as the buffer holds: the staged-x region, free at a unit boundary
// where x is restaged next), all in flight together and without registers,
// then each output's slices are summed from shared memory in slice order: the
// same sums, the same bits as reduce_block.  cp.async goes through the
// load/store path: bulk copies would queue behind the warps' weight boxes in
// the SM's copy engine.  Needs rows that start on 16-byte boundaries (N a
// multiple of 4, 16-byte aligned partial sums); returns false otherwise, or
// when the buffer holds fewer than 4 rows, without touching anything.
template <bool kBf16, int W>
__device__ __forceinline__ bool reduce_block_staged(const MmaLinDesc &R, int sb, uint8_t *buf,
                                                    uint32_t buf_bytes) {
    W4A16_CTA_SHAPE(W);
    if (R.N % 4 != 0 || ((uintptr_t)R.partials & 15) != 0) return false;
    const int rows_per_block = kWarps * R.strips_per_warp * 16;
    const int row0 = sb * rows_per_block;
    const int nrows = min(R.ycols - row0, rows_per_block);  // a multiple of 4 here
    const int nh = R.epi == kEpiSiluMul ? 2 : 1;            // gate rows, then up rows
    const size_t up = (size_t)R.half_strips * 16;
    const uint32_t per_row = (uint32_t)(R.S * R.M * nh) * 4u;
    int C = (int)(buf_bytes / per_row) & ~3;
    if (C < 4) return false;
    if (C > nrows) C = nrows;
    const int ncopies = R.S * R.M * nh;
    const uint32_t buf_s = dev::smem_u32(buf);
    for (int r0 = 0; r0 < nrows; r0 += C) {
        const int c = min(C, nrows - r0);
        const int q4 = c >> 2;  // 16-byte pieces per copied row segment
        // piece j: segment i = j / q4 (slice s, token t, gate or up rows h, i =
        // (s * M + t) * nh + h), 4 sums from row r0 + 4 (j % q4); it lands at
        // buf[i][4 (j % q4) ...]
        for (int j = threadIdx.x; j < ncopies * q4; j += kThreads) {
            const int i = j / q4, e = 4 * (j - i * q4);
            const int h = i % nh, st = i / nh;
            const float *src = R.partials + (size_t)st * R.N + row0 + r0 + e + (h ? up : 0);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                             buf_s + (uint32_t)((i * c + e) * 4)),
                         "l"(src)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        const float *f = reinterpret_cast<const float *>(buf);
        for (int i = threadIdx.x; i < R.M * c; i += kThreads) {
            const int t = i / c, rr = i - t * c;
            float sum = 0.f, gate = 0.f;
            for (int s2 = 0; s2 < R.S; ++s2) {
                const float *b = f + (size_t)((s2 * R.M + t) * nh) * c + rr;
                if (nh == 2) {
                    gate += b[0];
                    sum += b[c];
                } else {
                    sum += b[0];
                }
            }
            epilogue_store<kBf16>(R, (size_t)t * R.ycols + row0 + r0 + rr, sum, gate);
        }
        // every thread's reads of the chunk come before the next chunk's copies
        // (and before the next x copy, which writes through the async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
    }
    if (threadIdx.x == 0) R.counters[sb] = 0u;  // ready for the next launch
    return true;
}

// One call site for the kernel, with few arguments (the callers keep their
// registers across it).  A launch of one linear takes the staged reduction
// where the staged-x region is free (x_free: the next unit restages x, or
// none follows) and the rows allow it: there the reduction sits on the
// launch's critical path (config K 17408, N 5120 at M = 4: 32.8 -> 30.7 us).
// A fused round keeps the register path: in A/B runs of the 64-layer round
// the staged form was 1-2% slower at every M (its reductions overlap the
// other CTAs' streaming, and the copies wait with the weight traffic).  The
// buffer comes from the CTA's shared-memory layout.
template <bool kRound, bool kBf16, int W>
__device__ __noinline__ void reduce_any(const MmaLinDesc &R, int sb, int x_free) {
    W4A16_CTA_SHAPE(W);
    if constexpr (!kRound) {
        extern __shared__ __align__(128) uint8_t smem[];
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        if (x_free && reduce_block_staged<kBf16, W>(R, sb, smem + kRingBytes + kBarBytes,
                                                 dyn - (uint32_t)(kRingBytes + kBarBytes)))
            return;
    }
    reduce_block<kBf16, W>(R, sb);
}

template <bool kRound, bool kBf16, int W>
__global__ void __launch_bounds__(CtaShape<W>::kThreads, CtaShape<W>::kCtasPerSm)
    mma_kernel(const __grid_constant__ MmaKernelParams P) {
    W4A16_CTA_SHAPE(W);
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    uint8_t *wring = smem + (size_t)warp * kDepth * kStageBytes;  // this warp's two slots
    uint8_t *xs = smem + kRingBytes + kBarBytes;                   // staged x, then the sums
    int *flags = reinterpret_cast<int *>(smem + kRingBytes + kWarps * kDepth * 8);
    const uint32_t x_bar = dev::smem_u32(smem + kRingBytes + kWarps * kDepth * 8 + 64);
    volatile int *vflags = flags;
    volatile int *unit_q = flags + kFlagQueue;
    UnitInfo *slots = reinterpret_cast<UnitInfo *>(smem + kRingBytes + kSlotOffset);
    // the next kernel in the stream may be scheduled as SMs free up; it waits
    // for this grid to finish before it touches anything this grid writes
    grid_dependents_launch();
    const int total = P.total_units;
    const int grid = gridDim.x;
    auto desc = [&](int l) -> const MmaLinDesc & { return kRound ? P.descs[l] : P.single; };

    const uint32_t bar0 = dev::smem_u32(smem + kRingBytes) + 8 * kDepth * warp;
    const uint32_t ring0 = dev::smem_u32(wring);
    if (lane == 0) {
        // one arrival with the box's byte count, plus one per lane once its
        // metadata copies have landed
        for (int s = 0; s < kDepth; ++s) mbar_init(bar0 + 8 * s, 1 + 32);
        if (warp == 0) mbar_init(x_bar, 1);  // the x copies: bytes only
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // thread 0: decode queue position seq (its unit is in unit_q) into its
    // slot; the descriptors are read-only inputs
    int dl = 0;  // thread 0: the decoder's linear (units come in increasing order)
    auto fill_slot = [&](int seq) {
        UnitInfo &U = slots[seq & (kSlots - 1)];
        const int u = unit_q[seq & 7];
        if (u >= total || (kRound && P.counts && u >= P.counts[1])) {
            U.l = -1;
        } else {
            if (kRound) {
                // the last linear starting at or before u, four descriptors
                // per round trip (a CTA's first unit may lie many linears in)
                for (;;) {
                    int st[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st[i] = dl + 1 + i < P.n_lin ? P.descs[dl + 1 + i].unit_start : 0x7fffffff;
                    int adv = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) adv += u >= st[i];
                    dl += adv;
                    if (adv < 4) break;
                }
            }
            const MmaLinDesc &D = desc(dl);
            const int ul = u - D.unit_start;
            U.tmap = reinterpret_cast<uint64_t>(D.tmap_ref ? D.tmap_ref : &D.tmap);
            U.x = D.x;
            U.scales = D.scales;
            U.zeros = D.zeros;
            U.y = D.y;
            U.partials = D.partials;
            U.counters = D.counters;
            U.scales_first = D.scales_first;
            U.scales_end = D.scales_end;
            U.residual = D.residual;
            U.epi = D.epi;
            U.ycols = D.ycols;
            U.half_strips = D.half_strips;
            U.N = D.N;
            U.K = D.K;
            U.G = D.G;
            U.ZW = D.ZW;
            U.M = D.M;
            U.S = D.S;
            U.slice_groups = D.slice_groups;
            U.n_strips = D.n_strips;
            U.strips_per_warp = D.strips_per_warp;
            U.xstride = D.xstride;
            U.wait_for = D.wait_for;
            U.l = dl;
            U.slice = ul / D.n_blocks;
            U.sb = ul - U.slice * D.n_blocks;
        }
        st_release_cta(&U.seq, seq);
    };
    if (threadIdx.x == 0) {
        // descriptors written by the preceding kernel: wait for it before the
        // first read (the other threads read them after the barrier below)
        if (kRound && P.counts) grid_dependency_wait();
        // the CTA's first two units are fixed; the rest come every grid-th or
        // from a counter
        vflags[kFlagAbort] = 0;
        vflags[kFlagRed] = 0;
        for (int i = 0; i < kSlots; ++i) slots[i].seq = -1;
        unit_q[0] = blockIdx.x;
        unit_q[1] = blockIdx.x + grid < total ? blockIdx.x + grid : total;
        fill_slot(0);
        fill_slot(1);
    }
    __syncthreads();

    // ---- copy stream.  The issue cursor walks this warp's stages (unit by
    // unit, linear by linear) kDepth stages ahead of the consume cursor.
    // Weights, scales and zeros are never written by a preceding kernel, so
    // the stream starts before the grid-dependency wait.  Metadata: lane
    // (r = lane % 16, h = lane / 16) copies, for row r of the strip, scale
    // words 0 and 1 of the stage (h = 0) or scale word 2 and the zeros word
    // (h = 1): the three aligned words that hold the stage's four (2-byte
    // aligned) scales, and the zeros word of its groups.
    const int r = lane & 15, h = lane >> 4;
    int ik = 0;                   // queue position of the issue cursor's unit
    int ij = 0, inst = 0;         // stage within the strip, stages per strip
    bool i_wait = false;          // the next unit is not in the queue yet
    bool i_done = false;          // no units left
    unsigned t_iss = 0;           // stages issued by this warp
    uint64_t i_map = 0;           // tensor map of the unit's linear
    int i_g0 = 0, i_row16 = 0;    // first group of the slice, first row of the strip
    uintptr_t i_sfirst = 0;       // a valid source address for zero-byte copies
    uintptr_t is_s = 0;           // next scale word to copy (h = 0: it and the next)
    int is_avail = 0;             // bytes from is_s to the end of the scales (0 past row N)
    uintptr_t is_z = 0;           // zeros word of the next stage
    uint32_t is_zbytes = 0;
    // this warp's strips in a unit: strip0 + 8r for r < strips per warp; with
    // SiLU-and-mul the gate strip s, then the up strip s + half_strips
    int i_strip = 0, i_last = 0;  // current strip (of weight rows), the unit's last gate strip
    const UnitInfo *iD = nullptr;
    // copy sources of the issue cursor's strip
    auto i_strip_enter = [&]() {
        const UnitInfo &D = *iD;
        i_row16 = i_strip * 16;
        const int row = i_row16 + r;
        const bool vr = row < D.N;
        const size_t rr = (size_t)(vr ? row : 0);
        is_s = (((uintptr_t)(D.scales + rr * D.G + i_g0)) & ~(uintptr_t)3) + 8 * (uintptr_t)h;
        const uintptr_t rem = is_s < D.scales_end ? D.scales_end - is_s : 0;
        is_avail = vr ? (int)(rem > (1u << 30) ? (1u << 30) : rem) : 0;
        is_z = (uintptr_t)(D.zeros + rr * D.ZW + (i_g0 >> 3));
        is_zbytes = vr ? 4u : 0u;
        ij = 0;
    };
    // move the issue cursor to the first unit, at or after sequence index ik,
    // in which this warp has a strip (warp 0 always has one: it also asks L2
    // for the unit's slice of x); stop at a unit the queue does not hold yet
    auto i_enter = [&]() {
        for (;; ++ik) {
            const UnitInfo &D = slots[ik & (kSlots - 1)];
            if (ld_acquire_cta(&D.seq) != ik) {  // not decoded yet
                i_wait = true;
                return;
            }
            i_wait = false;
            if (D.l < 0) {
                i_done = true;
                return;
            }
            const int strip0 = D.sb * kWarps * D.strips_per_warp + warp;
            if (strip0 >= D.n_strips) continue;
            i_g0 = D.slice * D.slice_groups;
            const int ng = min(D.G, i_g0 + D.slice_groups) - i_g0;
            inst = (ng + kStageGroups - 1) / kStageGroups;
            if (warp == 0 && lane < D.M)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                 D.x + (size_t)lane * D.K + (size_t)i_g0 * kGroup),
                             "r"(ng * kGroup * 2)
                             : "memory");
            iD = &D;
            i_map = D.tmap;
            i_sfirst = D.scales_first;
            const int nr = min(D.strips_per_warp, (D.n_strips - 1 - strip0) / kWarps + 1);
            i_strip = strip0;
            i_last = strip0 + kWarps * (nr - 1);
            i_strip_enter();
            return;
        }
    };
    auto issue_next = [&]() {
        if (i_done) return;
        if (i_wait) {
            i_enter();
            if (i_wait || i_done) return;
        }
        const uint32_t slot = t_iss & 1u;  // kDepth == 2
        const uint32_t bar = bar0 + 8 * slot;
        const uint32_t dst = ring0 + slot * kStageBytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, kStageW);
            tma_box(dst, reinterpret_cast<const CUtensorMap *>(i_map), i_row16,
                    i_g0 + ij * kStageGroups, bar);
        }
        // a scale word copies the part of it inside the array; a word past
        // the end, or of a row past N, becomes zeros, reads nothing and takes
        // a valid source address
        const uint32_t md = dst + kStageW + r * 16 + 8 * h;
        const int n0 = min(max(is_avail, 0), 4);
        cp4(md, n0 ? is_s : i_sfirst, (uint32_t)n0);
        if (h == 0) {
            const int n1 = min(max(is_avail - 4, 0), 4);
            cp4(md + 4, n1 ? is_s + 4 : i_sfirst, (uint32_t)n1);
        } else {
            cp4(md + 4, is_z, is_zbytes);
        }
        cp_arrive_noinc(bar);
        ++t_iss;
        is_s += 8;
        is_avail -= 8;
        // stage j covers groups g0 + 4j .. g0 + 4j + 3: a new zeros word
        // starts with every second stage
        if (((i_g0 + (ij + 1) * kStageGroups) & 7) == 0) is_z += 4;
        if (++ij == inst) {
            // gate strip: its up strip next; then the next gate strip
            const int up = iD->epi == kEpiSiluMul ? iD->half_strips : 0;
            if (up && i_strip < up) {
                i_strip += up;
                i_strip_enter();
            } else if (i_strip - up < i_last) {  // the warp's next strip of the unit
                i_strip += kWarps - up;
                i_strip_enter();
            } else {
                ++ik;
                i_enter();
            }
        }
    };
    static_assert(kDepth == 2, "the slot and phase arithmetic assumes two slots");
    i_enter();
    issue_next();

    // ---- from here on: activations, outputs, the split-K workspace and the
    // counters may belong to the preceding kernel
    grid_dependency_wait();

    // x of the CTA's first unit goes out before the second weight stage, so
    // that it does not queue behind the weights
    int xpend_l = -1, xpend_slice = -1;  // the x copy in flight (-1: none)
    uint32_t x_par = 0;
    // thread 0: bulk-copy groups xg0 .. xg0 + xng - 1 of every token's x into
    // its staged row (raw order; rewritten in place once it lands)
    auto issue_x = [&](const UnitInfo &L, int xg0, int xng) {
        const uint32_t row_bytes = (uint32_t)xng * kGroup * 2;
        if (kBf16) {
            // the tokens' largest exponents, gathered once the copy lands:
            // cleared before the arrival, which releases the stores to every
            // thread that waits on the barrier
            int *xe = token_exps(xs, L.M, L.xstride, L.slice_groups);
            for (int t = 0; t < kMmaMaxTokens; ++t) xe[t] = 0;
        }
        mbar_arrive_expect_tx(x_bar, row_bytes * L.M);
        for (int t = 0; t < L.M; ++t)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                " [%0], [%1], %2, [%3];" ::"r"(dev::smem_u32(xs) + t * L.xstride),
                "l"(L.x + (size_t)t * L.K + (size_t)xg0 * kGroup), "r"(row_bytes), "r"(x_bar)
                : "memory");
    };
    {
        const UnitInfo &D0 = slots[0];  // a fixed unit, decoded before the barrier above
        if (D0.l >= 0 && !(kRound && P.done && D0.wait_for >= 0)) {
            const int xg0 = D0.slice * D0.slice_groups;
            if (threadIdx.x == 0) issue_x(D0, xg0, min(D0.G, xg0 + D0.slice_groups) - xg0);
            xpend_l = D0.l;
            xpend_slice = D0.slice;
        }
    }
    issue_next();

    // unit of word u of this lane's chunk in a group: x_unit(4c + u)
    const int xo0 = 16 * x_unit(4 * c + 0), xo1 = 16 * x_unit(4 * c + 1);
    const int xo2 = 16 * x_unit(4 * c + 2), xo3 = 16 * x_unit(4 * c + 3);
    unsigned t_cons = 0;  // stages consumed by this warp
    int cl = 0;           // linear of the consumer's unit
    int passed = 0;       // linears below this one are counted in P.done
    int staged_l = -1, staged_slice = -1;  // the (linear, slice) whose x is staged
    bool dead = false;
    // split K, one arrival per unit and CTA: the CTA that brings the last
    // slice of a block reduces it.  Thread 0 counts the arrival of the
    // previous unit at a unit boundary and reads the count's result at the
    // next boundary, so the atomic's latency hides behind a unit of work.
    int arr_l = -1, arr_sb = 0;  // split unit whose arrival is still to count
    unsigned *arr_cnt = nullptr;  // its linear's counters
    int arr_S = 0;                // its linear's slices
    int red_l = -1, red_sb = 0;  // arrival counted, its result in red_prev (thread 0)
    int red_S = 0;
    unsigned red_prev = 0;
    // The CTA's units after the first two: every grid-th unit (a launch of
    // one linear, whose few units per CTA are balanced best that way), or
    // from a shared counter (a fused round: CTAs that run faster take more).
    unsigned fetched = 0;  // thread 0, dynamic: counter value for sequence index k + kQueueAhead + 1
    auto seq_unit = [&](int seq, unsigned counter_value) -> int {
        const unsigned un = P.dynamic ? 2u * grid + counter_value
                                      : (unsigned)blockIdx.x + (unsigned)seq * grid;
        return un < (unsigned)total ? (int)un : total;
    };
    if (threadIdx.x == 0) {
        // sequence indices 2 .. kQueueAhead (none when the queue runs one ahead)
        if (kQueueAhead > 1) {
            const unsigned f = P.dynamic ? atomicAdd(P.sched, (unsigned)(kQueueAhead - 1)) : 0u;
            for (int i = 0; i < kQueueAhead - 1; ++i) unit_q[2 + i] = seq_unit(2 + i, f + i);
        }
        if (P.dynamic) fetched = atomicAdd(P.sched, 1u);
    }
    // thread 0: publish whether this CTA reduces the block whose arrival it
    // counted (the result is read here, a unit after the atomic), into the
    // flag slot of the boundary that reads it (two slots by parity: a slot is
    // rewritten only after every warp has passed the barrier after its read)
    auto publish_reduction = [&](int boundary) {
        if (threadIdx.x != 0) return;
        volatile int *f = vflags + kFlagRed + 3 * (boundary & 1);
        f[0] = red_l >= 0 && red_prev == (unsigned)(red_S - 1);
        f[1] = red_l;
        f[2] = red_sb;
        red_l = -1;
    };
    // count the arrival of the pending split unit (thread 0's atomic; all
    // warps have stored their partials: call after a CTA barrier).  arr_l and
    // red_pending are the same in every thread.
    bool red_pending = false;  // an arrival is counted, its result not yet published
    auto count_arrival = [&]() {
        if (arr_l < 0) return;
        if (threadIdx.x == 0) {
            unsigned prev;
            asm volatile("fence.acq_rel.gpu;\n\tatom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                         : "=r"(prev)
                         : "l"(arr_cnt + arr_sb)
                         : "memory");
            red_prev = prev;
            red_l = arr_l;
            red_sb = arr_sb;
            red_S = arr_S;
        }
        red_pending = true;
        arr_l = -1;
    };
    // all threads, after the barrier that follows publish_reduction(boundary).
    // x_free: the staged x is not needed again (the next unit restages it, or
    // no unit follows), so the reduction may stage partial sums over it: every
    // warp has passed the barrier after its last read, and no x copy is in
    // flight at a boundary
    auto maybe_reduce = [&](int boundary, bool x_free) {
        volatile int *f = vflags + kFlagRed + 3 * (boundary & 1);
        if (f[0]) reduce_any<kRound, kBf16, W>(desc(f[1]), f[2], x_free ? 1 : 0);
    };

    // boundary b: the barrier at the top of iteration b (b = k), or an extra
    // one inside it (b = k + 1 ... ); `bnd` counts them
    int bnd = 0;
    for (int k = 0;; ++k) {
        if (threadIdx.x == 0 && k >= 1) {
            // the unit fetched at the previous boundary joins the queue
            unit_q[(k + kQueueAhead) & 7] = seq_unit(k + kQueueAhead, fetched);
            if (P.dynamic) fetched = atomicAdd(P.sched, 1u);
        }
        // this unit, decoded by thread 0 a unit ago (warps that run ahead of
        // warp 0 wait for it here)
        const UnitInfo &D = slots[k & (kSlots - 1)];
        if (ld_acquire_cta(&D.seq) != k) {
            const unsigned long long tq = dev::globaltimer();
            while (ld_acquire_cta(&D.seq) != k) {
                if (vflags[kFlagAbort] || dev::globaltimer() - tq > kWaitNs) {
                    if (lane == 0) atomicOr(P.status, kErrMmaWait);
                    vflags[kFlagAbort] = 1;
                    break;
                }
            }
        }
        const bool have = !vflags[kFlagAbort] && D.l >= 0;
        if (have) cl = D.l;
        const int slice = D.slice, sb = D.sb;
        // A CTA barrier is needed to restage x, for the split-K arrival and
        // reduction protocol and for a new linear of a round with waits;
        // otherwise the warps go on without one, but at least every fourth
        // unit, so that no warp falls far enough behind warp 0 for the queue
        // (8 entries) to overwrite a unit it has still to read.
        const bool restage = have && (cl != staged_l || slice != staged_slice);
        if (restage || arr_l >= 0 || red_pending || (k & 3) == 0 ||
            (kRound && P.done && passed < cl && have)) {
            publish_reduction(bnd);
            red_pending = false;
            __syncthreads();  // the previous unit's staged x is no longer read
            if (vflags[kFlagAbort]) {
                dead = true;
                break;
            }
            maybe_reduce(bnd++, restage || !have);
        } else if (vflags[kFlagAbort]) {
            dead = true;
            break;
        }
        if (!have) break;
        const int M = D.M;
        const int g0 = slice * D.slice_groups;  // a multiple of kStageGroups
        const int ng = min(D.G, g0 + D.slice_groups) - g0;
        const int nst = (ng + kStageGroups - 1) / kStageGroups;
        float *sums = reinterpret_cast<float *>(xs + (size_t)M * D.xstride);  // [group][8]

        if (kRound && P.done && passed < cl) {
            // A new linear.  Settle this CTA's pending split arrival now (its
            // linear may be one that others wait for), count the linears this
            // CTA is done with, then wait for the linear this one depends on.
            count_arrival();
            publish_reduction(bnd);
            __syncthreads();
            maybe_reduce(bnd++, restage);  // a new linear: x is restaged
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                for (; passed < cl; ++passed) atomicAdd(P.done + passed, 1u);
                if (D.wait_for >= 0 && !wait_counter(P.done + D.wait_for, (unsigned)grid)) {
                    atomicOr(P.status, kErrMmaDep);
                    vflags[kFlagAbort] = 1;
                }
            }
            __syncthreads();
            if (vflags[kFlagAbort]) {
                dead = true;
                break;
            }
        }
        if (restage) {
            // ---- stage x[:, slice]: the slice lands by bulk copy in its rows
            // in raw order; then each lane rewrites its 16-byte unit J in MMA
            // pair order at unit x_unit(J) (a unit and its partner sit in the
            // same half warp: all of a warp's reads come before its writes),
            // and each (group, token)'s sum S of x is formed (kept as S *
            // 2^-20): the 16 lanes of a half warp hold the 16 units of one
            // group of one token and add theirs with shuffles
            if (xpend_l != cl || xpend_slice != slice) {  // not copied ahead
                if (threadIdx.x == 0) {
                    // the previous unit's reads of these rows are behind the
                    // barrier above; order them before the copy's writes
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue_x(D, g0, ng);
                }
            }
            // thread 0 decodes the next unit while the copy is in flight
            if (threadIdx.x == 0 && k >= 1) fill_slot(k + 1);
            xpend_l = cl;  // in flight until the wait below
            xpend_slice = slice;
            if (!__all_sync(0xffffffffu, mbar_wait(x_bar, x_par))) {
                if (lane == 0) {
                    atomicOr(P.status, kErrMmaWait);
                    vflags[kFlagAbort] = 1;
                }
                dead = true;
                break;
            }
            x_par ^= 1u;
            xpend_l = -1;
            const int nunits = ng * (kGroup / 8);
            const int xtotal = M * nunits;  // a multiple of 16
            int *xexp = token_exps(xs, M, D.xstride, D.slice_groups);
            // Unit i = t * nunits + J of this thread: 32 warp + lane, then
            // kThreads further per pass.  With bf16, t and J step without a
            // division (the fp16 kernel keeps the division: the stepped form
            // costs it registers elsewhere)
            const int i0 = warp * 32 + lane;
            const int dt = kThreads / nunits, dJ = kThreads - dt * nunits;
            if (kBf16) {
                // each token's largest exponent: a half warp holds 16 units of
                // one token (nunits is a multiple of 16)
                for (int i = i0, t = i0 / nunits, J = i0 - t * nunits; i - lane < xtotal;
                     i += kThreads) {
                    int e = 0;
                    if (i < xtotal)
                        e = max_bf16_exp(*reinterpret_cast<const uint4 *>(
                            xs + (size_t)t * D.xstride + 16 * J));
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) e = max(e, __shfl_xor_sync(0xffffffffu, e, off));
                    if (i < xtotal && (J & 15) == 0) atomicMax(xexp + t, e);
                    t += dt;
                    J += dJ;
                    if (J >= nunits) {
                        J -= nunits;
                        ++t;
                    }
                }
                __syncthreads();
            }
            for (int base = warp * 32, ts = i0 / nunits, Js = i0 - ts * nunits; base < xtotal;
                 base += kThreads) {
                const int i = base + lane;
                const bool valid = i < xtotal;
                int t, J;
                if constexpr (kBf16) {
                    t = ts;
                    J = Js;
                    ts += dt;
                    Js += dJ;
                    if (Js >= nunits) {
                        Js -= nunits;
                        ++ts;
                    }
                } else {
                    t = i / nunits;
                    J = i - t * nunits;
                }
                uint8_t *row = xs + (size_t)t * D.xstride;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (valid) v = *reinterpret_cast<const uint4 *>(row + 16 * J);
                if (kBf16 && valid) v = bf16_to_scaled_f16(v, pow2(bf16_stage_shift(xexp[t])));
                __syncwarp();
                if (valid) *reinterpret_cast<uint4 *>(row + 16 * x_unit(J)) = mma_pair_order(v);
                const float2 a = pair_to_float2<false>(v.x), bb = pair_to_float2<false>(v.y);
                const float2 e = pair_to_float2<false>(v.z), f = pair_to_float2<false>(v.w);
                float sum = ((a.x + a.y) + (bb.x + bb.y)) + ((e.x + e.y) + (f.x + f.y));
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                if (valid && (J & 15) == 0) sums[(J >> 4) * 8 + t] = sum * kTwoM20;
            }
            // tokens M..7 have no x: their sums are zero
            for (int i = threadIdx.x; i < ng * (8 - M); i += kThreads)
                sums[(i / (8 - M)) * 8 + M + i % (8 - M)] = 0.f;
            __syncthreads();
            staged_l = cl;
            staged_slice = slice;
        } else if (threadIdx.x == 0 && k >= 1) {
            fill_slot(k + 1);  // the next unit (slot 1 is decoded at the start)
        }
        // after the staging: thread 0's release fence and atomic would
        // otherwise hold up warp 0, and with it the staging
        count_arrival();
        // this warp's strips of the unit: strip0, strip0 + 8, ... (the tail
        // block of a slice may hold fewer); with SiLU-and-mul each is the
        // strip's gate rows, then its up rows
        const int nparts = D.epi == kEpiSiluMul ? 2 : 1;
        // The block's sums go to the workspace and the CTA that brings the
        // last slice reduces them (reduce_block, which applies the epilogue)
        // with split K, and always with SiLU-and-mul: its gate and up sums
        // meet there, so that no warp keeps the gate sums in registers
        // across the up rows (registers every linear would pay for).
        const bool to_ws = D.S > 1 || nparts == 2;
        for (int strip = sb * kWarps * D.strips_per_warp + warp, rs = 0;
             rs < D.strips_per_warp && strip < D.n_strips; ++rs, strip += kWarps) {
            // lanes of tokens >= M compute a column nobody stores: they read token 0
            const int tok = g < M ? g : 0;
            const uint8_t *xrow = xs + (size_t)tok * D.xstride;
            float acc[4];
            for (int part = 0; part < nparts; ++part) {
                const int ra = (strip + (part ? D.half_strips : 0)) * 16 + g, rb = ra + 8;
                const bool va = ra < D.N, vb = rb < D.N;
                // where the slice's first scale of each row sits in its aligned word
                // (the same in every stage: a stage advances 8 bytes)
                const uintptr_t s0A = (uintptr_t)(D.scales + (size_t)(va ? ra : 0) * D.G + g0);
                const uintptr_t s0B = (uintptr_t)(D.scales + (size_t)(vb ? rb : 0) * D.G + g0);
                const uint32_t offA = (uint32_t)(s0A >> 1) & 1u, offB = (uint32_t)(s0B >> 1) & 1u;
                const uint32_t shA = 16u * offA, shB = 16u * offB;
                const uint32_t selA = offA ? 0x54u : 0x32u, selB = offB ? 0x54u : 0x32u;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] = 0.f;
                for (int j = 0; j < nst; ++j) {
                    // the issue cursor may have stopped at a unit the queue did not
                    // hold yet: this stage belongs to a unit it holds
                    if (t_iss == t_cons) issue_next();
                    const uint32_t slot = t_cons & 1u, par = (t_cons >> 1) & 1u;
                    if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * slot, par))) {
                        if (lane == 0) {
                            atomicOr(P.status, kErrMmaWait);
                            vflags[kFlagAbort] = 1;  // the other warps stop at their next unit
                        }
                        dead = true;
                        break;
                    }
                    // this lane's part of the stage: 16 bytes of rows g and g + 8 of
                    // each group (read just before the group), the metadata of both rows
                    const uint8_t *st = wring + slot * kStageBytes;
                    const uint8_t *stA = st + g * 64 + 16 * c, *stB = st + (g + 8) * 64 + 16 * c;
                    const uint4 ma = *reinterpret_cast<const uint4 *>(st + kStageW + g * 16);
                    const uint4 mb = *reinterpret_cast<const uint4 *>(st + kStageW + (g + 8) * 16);
                    // zero nibbles of the stage's groups: the stage starts at group
                    // g0 + 4j, nibble (g0 + 4j) % 8 of its zeros word
                    const uint32_t zsh = ((g0 + j * kStageGroups) & 4) ? 16u : 0u;
                    const uint32_t zwA = ma.w >> zsh, zwB = mb.w >> zsh;
                    const uint32_t mA[3] = {ma.x, ma.y, ma.z}, mB[3] = {mb.x, mb.y, mb.z};
                    const int n_in = min(kStageGroups, ng - j * kStageGroups);
                    const uint8_t *xg = xrow + (size_t)j * (kStageGroups * 256);
                    const float *sg = sums + (j * kStageGroups) * 8 + 2 * c;  // tokens 2c, 2c+1
                    // one group of the stage
                    auto group = [&](const int i) {
                        // scales of rows ra and rb: half (off + i) of the words
                        uint32_t hA, hB;
                        if (i & 1) {
                            hA = dev::prmt(mA[i >> 1], mA[(i >> 1) + 1], selA);
                            hB = dev::prmt(mB[i >> 1], mB[(i >> 1) + 1], selB);
                        } else {
                            hA = mA[i >> 1] >> shA;
                            hB = mB[i >> 1] >> shB;
                        }
                        const float sA = bits_to_float<kBf16>(hA & 0xffffu);
                        const float sB = bits_to_float<kBf16>(hB & 0xffffu);
                        // zero points of rows ra and rb as floats (2^23 + z, minus 2^23)
                        const float zA =
                            __uint_as_float(0x4b000000u | ((zwA >> (4 * i)) & 0xfu)) - 8388608.f;
                        const float zB =
                            __uint_as_float(0x4b000000u | ((zwB >> (4 * i)) & 0xfu)) - 8388608.f;
                        // S * 2^-20 of tokens 2c, 2c + 1
                        const float2 sx = *reinterpret_cast<const float2 *>(sg + i * 8);
                        const uint8_t *xi = xg + i * 256;
                        uint4 xv[4];
                        xv[0] = *reinterpret_cast<const uint4 *>(xi + xo0);
                        xv[1] = *reinterpret_cast<const uint4 *>(xi + xo1);
                        xv[2] = *reinterpret_cast<const uint4 *>(xi + xo2);
                        xv[3] = *reinterpret_cast<const uint4 *>(xi + xo3);
                        const uint4 wa = *reinterpret_cast<const uint4 *>(stA + i * 1024);
                        const uint4 wb = *reinterpret_cast<const uint4 *>(stB + i * 1024);
                        const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
                        const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
                        float dl[4] = {0.f, 0.f, 0.f, 0.f}, dh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int uu = 0; uu < 4; ++uu) {
                            const uint32_t a = wA[uu], b = wB[uu], a8 = a >> 8, b8 = b >> 8;
                            mma16816(dl, a & 0x000f000fu, b & 0x000f000fu, a8 & 0x000f000fu,
                                     b8 & 0x000f000fu, xv[uu].x, xv[uu].y);
                            mma16816(dh, a & 0x00f000f0u, b & 0x00f000f0u, a8 & 0x00f000f0u,
                                     b8 & 0x00f000f0u, xv[uu].z, xv[uu].w);
                        }
                        // 2^-20 sum (q - z) x = 16 D_lo + D_hi - z S 2^-20
                        acc[0] = fmaf(sA, fmaf(-zA, sx.x, fmaf(16.f, dl[0], dh[0])), acc[0]);
                        acc[1] = fmaf(sA, fmaf(-zA, sx.y, fmaf(16.f, dl[1], dh[1])), acc[1]);
                        acc[2] = fmaf(sB, fmaf(-zB, sx.x, fmaf(16.f, dl[2], dh[2])), acc[2]);
                        acc[3] = fmaf(sB, fmaf(-zB, sx.y, fmaf(16.f, dl[3], dh[3])), acc[3]);
                    };
                    if (n_in == kStageGroups) {
#pragma unroll
                        for (int i = 0; i < kStageGroups; ++i) group(i);
                    } else {  // the last stage of a slice that ends at K
#pragma unroll
                        for (int i = 0; i < kStageGroups; ++i)
                            if (i < n_in) group(i);
                    }
                    // Refill the slot kDepth stages ahead once every lane is done with
                    // it.  The lanes read it through the generic proxy and the box
                    // lands through the async proxy: the proxy fence orders those
                    // reads before the new box's writes.
                    __syncwarp();
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    ++t_cons;
                    issue_next();
                }
                if (dead) break;

                // ---- end of the rows: acc[0..1] row ra, tokens 2c, 2c+1; acc[2..3] row rb
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] *= kTwo20;
                const int t0 = 2 * c, t1 = 2 * c + 1;
                if (kBf16) {  // undo the tokens' staging scales
                    const int *xexp = token_exps(xs, M, D.xstride, D.slice_groups);
                    const float u0 = pow2(-bf16_stage_shift(xexp[t0]));
                    const float u1 = pow2(-bf16_stage_shift(xexp[t1]));
                    acc[0] *= u0;
                    acc[1] *= u1;
                    acc[2] *= u0;
                    acc[3] *= u1;
                }
                if (to_ws) {  // this slice's partial sums, by weight row
                    float *ps = D.partials + (size_t)slice * M * D.N;
                    if (va && t0 < M) ps[(size_t)t0 * D.N + ra] = acc[0];
                    if (va && t1 < M) ps[(size_t)t1 * D.N + ra] = acc[1];
                    if (vb && t0 < M) ps[(size_t)t0 * D.N + rb] = acc[2];
                    if (vb && t1 < M) ps[(size_t)t1 * D.N + rb] = acc[3];
                    continue;
                }
                // y, or y + residual (read as fp32, one rounding)
                const size_t ya = (size_t)t0 * D.ycols + ra, yb = (size_t)t0 * D.ycols + rb;
                if (D.epi == kEpiResidual) {
                    if (va && t0 < M) acc[0] += to_float<kBf16>(D.residual[ya]);
                    if (va && t1 < M) acc[1] += to_float<kBf16>(D.residual[ya + D.ycols]);
                    if (vb && t0 < M) acc[2] += to_float<kBf16>(D.residual[yb]);
                    if (vb && t1 < M) acc[3] += to_float<kBf16>(D.residual[yb + D.ycols]);
                }
                if (va && t0 < M) D.y[ya] = from_float<kBf16>(acc[0]);
                if (va && t1 < M) D.y[ya + D.ycols] = from_float<kBf16>(acc[1]);
                if (vb && t0 < M) D.y[yb] = from_float<kBf16>(acc[2]);
                if (vb && t1 < M) D.y[yb + D.ycols] = from_float<kBf16>(acc[3]);
            }
            if (dead) break;
        }
        if (dead) break;
        if (to_ws) {  // count this unit's arrival at the next boundary
            arr_l = cl;
            arr_sb = sb;
            arr_cnt = D.counters;
            arr_S = D.S;
        }
    }


    if (dead) {
        // a wait expired: let this warp's copies in flight land (bounded)
        // before the CTA's shared memory goes away
        for (; t_cons < t_iss; ++t_cons) mbar_wait(bar0 + 8 * (t_cons & 1u), (t_cons >> 1) & 1u);
        if (xpend_l >= 0) mbar_wait(x_bar, x_par);  // an x copy in flight
        cp_wait_all();
        return;
    }
    cp_wait_all();
    // split K still pending: the decision on the arrival counted at the last
    // boundary, then the arrival of the last unit (arr_l and red_pending are
    // the same in every thread)
    if (red_pending || arr_l >= 0) {
        publish_reduction(bnd);
        red_pending = false;
        __syncthreads();
        maybe_reduce(bnd++, true);
        count_arrival();
        publish_reduction(bnd);
        __syncthreads();
        maybe_reduce(bnd++, true);
    }
    if (P.dynamic || (kRound && P.done)) {
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            if (kRound && P.done)
                for (; passed < P.n_lin; ++passed) atomicAdd(P.done + passed, 1u);
            // the last CTA out leaves the counters zeroed for the next launch
            const unsigned prev = atomicAdd(P.sched + 1, 1u);
            if (prev == (unsigned)grid - 1) {
                __threadfence();
                P.sched[0] = 0u;
                P.sched[1] = 0u;
                if (kRound && P.done)
                    for (int l = 0; l < P.n_lin; ++l) P.done[l] = 0u;
            }
        }
    }
}

int xstride_for(int slice_groups) { return slice_groups * kGroup * 2 + 16; }


cudaLaunchConfig_t launch_config(int grid, int threads, int smem, cudaStream_t stream,
                                 cudaLaunchAttribute *attr) {
    // programmatic dependent launch: the grid may start while the previous
    // kernel in the stream drains; the kernel waits for it (griddepcontrol)
    // before touching activations, outputs or the workspace
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// the shape's sizes on the host, by width (8 or 16 warps)
int ring_bytes(int w) { return w == 16 ? CtaShape<16>::kRingBytes : CtaShape<8>::kRingBytes; }
int bar_bytes(int w) { return w == 16 ? CtaShape<16>::kBarBytes : CtaShape<8>::kBarBytes; }
int smem_per_cta(int w) { return w == 16 ? CtaShape<16>::kSmemPerCta : CtaShape<8>::kSmemPerCta; }
int ctas_per_sm(int w) { return 16 / w; }

// the largest slice (a whole number of stages) whose staged x and sums fit
// beside the rings of a CTA of w warps
int max_slice_groups(int M, int w) {
    const int budget = smem_per_cta(w) - ring_bytes(w) - bar_bytes(w);
    int g = (budget - 16 * M - kMmaMaxTokens * 4) / (kGroup * 2 * M + 32);
    g = g / kStageGroups * kStageGroups;
    if (g > kMaxSliceGroups) g = kMaxSliceGroups;
    if (g < kStageGroups) g = kStageGroups;
    return g;
}

}  // namespace

int mma_smem_bytes(int M, int slice_groups, int warps) {
    return ring_bytes(warps) + bar_bytes(warps) + M * xstride_for(slice_groups) +
           slice_groups * 8 * 4 + kMmaMaxTokens * 4;
}

int mma_round_grid(const DeviceInfo &dev, int warps) { return ctas_per_sm(warps) * dev.sm_count; }

int mma_round_warps(int M, const int *K, const int *N, int n) {
    // The 16-warp CTA pays for its one-CTA-per-SM shape (a unit boundary
    // stalls all 16 warps of the SM, where two 8-warp CTAs cover each other's
    // barriers and x staging): in the 64-layer round at M = 1..4 it ran
    // 3-6% slower.  It wins where its room for x removes the K split from
    // most of the round's bytes: at M = 5..8 the K 5120 linears no longer fit
    // an 8-warp CTA unsplit (2.18-2.30 ms on 8 warps, 2.01-2.08 ms on 16).
    double all = 0, split8 = 0, split16 = 0;
    for (int l = 0; l < n; ++l) {
        const int G = K[l] / kGroup;
        const double b = (double)N[l] * K[l];
        all += b;
        if (G > max_slice_groups(M, 8)) split8 += b;
        if (G > max_slice_groups(M, 16)) split16 += b;
    }
    return all > 0 && split8 - split16 > 0.5 * all ? 16 : 8;
}

MmaPlan plan_mma(int M, int N, int K, int split, const DeviceInfo &dev, int epi, int copies,
                 int warps) {
    MmaPlan pl{};
    pl.M = M;
    const int G = K / kGroup;
    if (warps == 0) {
        // one linear alone: 16 warps when that CTA holds the whole K's x and
        // the 8-warp CTA would have to split K for room (K 5120, N 27648 at
        // M = 8: 36.9 -> 28.7 us); else 8 (where both split, as K 17408 at
        // M = 4 and 8, the 8-warp plans measured 2 us faster)
        warps = G > max_slice_groups(M, 8) && G <= max_slice_groups(M, 16) ? 16 : 8;
    }
    pl.warps = warps;
    const int kWarps = warps;
    // SiLU-and-mul: a logical strip is a gate strip and its up strip (N/2 a
    // multiple of 16), twice the work of a strip
    const int work = epi == kEpiSiluMul ? 2 : 1;
    pl.n_strips = (out_cols(N, epi) + 15) / 16;
    pl.strips_per_warp = split == 2 ? kRoundStripsPerWarp / work : 1;
    if (split == 3) split = 2;  // a round's last linears: fewest slices, small units
    pl.n_blocks = (pl.n_strips + kWarps * pl.strips_per_warp - 1) / (kWarps * pl.strips_per_warp);
    const int max_groups = max_slice_groups(M, warps);
    const int s_min = (G + max_groups - 1) / max_groups;
    if (split == 0 && s_min > 1) {
        pl.ok = false;
        return pl;
    }
    const int grid_max = ctas_per_sm(warps) * dev.sm_count;
    int best_sg = 0;
    if (split == 2) {
        // fewest slices: spread evenly over whole stages
        best_sg = (G + s_min - 1) / s_min;
        best_sg = (best_sg + kStageGroups - 1) / kStageGroups * kStageGroups;
    } else {
        // Pick the strips per warp and the K slices (whole stages) with the
        // least cost in a model tuned on single-launch times measured on
        // GB300 (one linear, L2 evicted, 14 shapes with K 5120..17408,
        // N 5120..139264, M 1..8, every feasible plan; the model's pick is
        // within 1.5% of the best plan on average): per unit a CTA pays
        // ~2.2 us (barrier, x staging) plus its stages, a stage per warp
        // 0.85 us plus 0.45 us at full load (16 warps share an SM's issue
        // slots); a split adds ~3 us plus 0.75 us per slice (partials, the
        // reducing CTA on the critical path; the reduction stages the slices'
        // partial sums through shared memory: with its earlier charge of 4.5 us
        // plus 2 us per slice, K 17408, N 5120 at M = 4 took 30.7 us, now 27.3).
        // Fewer, longer units win unless the staged x needs the slices or many
        // SMs would sit idle.
        int s_lo = s_min;
        if (split == 1 && s_lo < 2 && G > kStageGroups) s_lo = 2;
        int s_hi = split == 0 ? 1 : (G + kStageGroups - 1) / kStageGroups;
        if (s_hi < s_lo) s_hi = s_lo;
        double best_cost = 1e30;
        for (int spw = 1; spw <= kRoundStripsPerWarp; spw *= 2) {
            const int nb = (pl.n_strips + kWarps * spw - 1) / (kWarps * spw);
            for (int S = s_lo; S <= s_hi; ++S) {
                int sg = (G + S - 1) / S;
                sg = (sg + kStageGroups - 1) / kStageGroups * kStageGroups;
                if (sg > max_groups) continue;
                const int S_eff = (G + sg - 1) / sg;
                if (split == 1 && S_eff < 2 && G > kStageGroups) continue;
                const long long units = (long long)nb * S_eff * copies;
                const long long per_cta = (units + grid_max - 1) / grid_max;
                const double load = (double)(units < grid_max ? units : grid_max) / grid_max;
                const double stages = (double)spw * work * ((sg + kStageGroups - 1) / kStageGroups);
                // (SiLU-and-mul reduces through the workspace at any S)
                const bool reduces = S_eff > 1 || epi == kEpiSiluMul;
                const double cost = (double)per_cta * (2.2 + stages * (0.85 + 0.45 * load)) +
                                    (reduces ? 3.0 + 0.75 * S_eff : 0.0);
                if (cost < best_cost - 1e-9) {
                    best_cost = cost;
                    best_sg = sg;
                    pl.strips_per_warp = spw;
                    pl.n_blocks = nb;
                }
            }
        }
    }
    if (best_sg == 0) {  // split == 1 and too few groups to split along stage lines
        pl.ok = false;
        return pl;
    }
    pl.slice_groups = best_sg;
    pl.S = (G + best_sg - 1) / best_sg;
    pl.units = pl.S * pl.n_blocks;
    pl.grid = pl.units < grid_max ? pl.units : grid_max;
    pl.smem_bytes = mma_smem_bytes(M, pl.slice_groups, warps);
    // split K, and SiLU-and-mul with any number of slices: the partial sums
    pl.reduce = pl.S > 1 || epi == kEpiSiluMul;
    pl.ws_bytes = pl.reduce ? (size_t)pl.S * M * N * sizeof(float) : 0;
    pl.ok = true;
    return pl;
}

cudaError_t mma_describe(const LinearArgs &a, const MmaPlan &plan, float *partials,
                         unsigned *counters, int unit_start, int wait_for, MmaLinDesc *d) {
    const EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorInitializationError;
    memset(d, 0, sizeof(*d));
    const int G = a.K / kGroup;
    // qweight as a 3-D tensor of uint32: (word in group, row, group), so one
    // box brings a strip's 16 rows x 4 groups, group-major
    const cuuint64_t dims[3] = {16, (cuuint64_t)a.N, (cuuint64_t)G};
    const cuuint64_t strides[2] = {(cuuint64_t)a.K / 2, 64};
    const cuuint32_t box[3] = {16, 16, (cuuint32_t)kStageGroups};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(&d->tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, (void *)a.qw, dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    d->x = a.x;
    d->scales = a.scales;
    d->zeros = a.zeros;
    d->y = a.y;
    d->partials = partials;
    d->counters = counters;
    d->scales_first = (uintptr_t)a.scales & ~(uintptr_t)3;
    d->scales_end = (uintptr_t)(a.scales + (size_t)a.N * G);
    d->residual = a.epi == kEpiResidual ? a.residual : nullptr;
    d->epi = a.epi;
    d->ycols = out_cols(a.N, a.epi);
    d->half_strips = a.epi == kEpiSiluMul ? a.N / 32 : 0;
    d->N = a.N;
    d->K = a.K;
    d->G = G;
    d->ZW = (G + 7) / 8;
    d->M = a.M;
    d->S = plan.S;
    d->slice_groups = plan.slice_groups;
    d->n_strips = plan.n_strips;
    d->strips_per_warp = plan.strips_per_warp;
    d->n_blocks = plan.n_blocks;
    d->unit_start = unit_start;
    d->xstride = xstride_for(plan.slice_groups);
    d->wait_for = wait_for;
    return cudaSuccess;
}

cudaError_t launch_mma(const LinearArgs &a, const MmaPlan &plan, const Workspace &ws,
                       cudaStream_t stream) {
    const bool bf16 = a.dtype == kDtypeBf16;
    MmaKernelParams P;
    memset(&P, 0, sizeof(P));
    cudaError_t e = mma_describe(a, plan, ws.partials, ws.counters, 0, -1, &P.single);
    if (e != cudaSuccess) return e;
    P.status = ws.status;
    P.sched = ws.counters + ws.n_counters - kMmaSchedWords;
    P.n_lin = 1;
    P.total_units = plan.units;
    P.dynamic = 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_config(plan.grid, plan.warps * 32, plan.smem_bytes, stream, attr);
    if (plan.warps == 16)
        return bf16 ? cudaLaunchKernelEx(&cfg, mma_kernel<false, true, 16>, P)
                    : cudaLaunchKernelEx(&cfg, mma_kernel<false, false, 16>, P);
    return bf16 ? cudaLaunchKernelEx(&cfg, mma_kernel<false, true, 8>, P)
                : cudaLaunchKernelEx(&cfg, mma_kernel<false, false, 8>, P);
}

cudaError_t launch_mma_round(const MmaRound &r, const Workspace &ws, const DeviceInfo &dev,
                             cudaStream_t stream) {
    MmaKernelParams P;
    memset(&P, 0, sizeof(P));
    P.descs = r.descs;
    P.done = r.done;
    P.status = ws.status;
    P.sched = ws.counters + ws.n_counters - kMmaSchedWords;
    P.n_lin = r.n;
    P.total_units = r.total_units;
    P.counts = r.counts;
    P.dynamic = 1;
    int grid = mma_round_grid(dev, r.warps);
    if (grid > r.total_units) grid = r.total_units;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config(grid, r.warps * 32, r.smem_bytes, stream, attr);
    if (r.done) {
        // linears wait for earlier ones: every CTA must be resident at once
        attr[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
        attr[cfg.numAttrs].val.cooperative = 1;
        cfg.numAttrs += 1;
    }
    if (r.warps == 16)
        return r.bf16 ? cudaLaunchKernelEx(&cfg, mma_kernel<true, true, 16>, P)
                      : cudaLaunchKernelEx(&cfg, mma_kernel<true, false, 16>, P);
    return r.bf16 ? cudaLaunchKernelEx(&cfg, mma_kernel<true, true, 8>, P)
                  : cudaLaunchKernelEx(&cfg, mma_kernel<true, false, 8>, P);
}

EncodeTiledFn tensor_map_encoder() {
    // looked up once, on first use (a function-local static: thread-safe)
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                               cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

cudaError_t mma_init(const DeviceInfo &dev) {
    if (!tensor_map_encoder()) return cudaErrorSymbolNotFound;
    cudaError_t e = cudaSuccess;
    const void *fns[8] = {(const void *)mma_kernel<false, false, 8>,
                          (const void *)mma_kernel<true, false, 8>,
                          (const void *)mma_kernel<false, true, 8>,
                          (const void *)mma_kernel<true, true, 8>,
                          (const void *)mma_kernel<false, false, 16>,
                          (const void *)mma_kernel<true, false, 16>,
                          (const void *)mma_kernel<false, true, 16>,
                          (const void *)mma_kernel<true, true, 16>};
    for (int k = 0; k < 8 && e == cudaSuccess; ++k) {
        const void *fn = fns[k];
        int dyn = smem_per_cta(k < 4 ? 8 : 16);
        if (dyn > dev.max_smem_optin - 1024) dyn = dev.max_smem_optin - 1024;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
    }
    return e;
}

}  // namespace w4a16

// ---- allocation-free entry point ------------------------------------------
// Callers that cannot allocate device memory: a process whose device memory
// is wholly reserved by its own caching allocator, or a serving loop that must
// not call cudaMalloc (which synchronises the device and can fail when memory
// is reserved).  w4a16_linear_noalloc needs neither w4a16_init nor any
// allocation: its split-K scratch is this statically sized device array.
namespace {
// 4 MiB of fp32 partial sums: enough for the split every M <= 8 linear of a
// 27B-class decode layer takes (the largest, the fused gate+up projection
// K 5120, N 34816 at M = 8, splits K in two: 2.2 MB)
constexpr size_t kNoAllocPartialFloats = size_t(1) << 20;
constexpr int kNoAllocCounters = 4096;  // per-block arrival counters
// partials, then the counters, the kernel's scheduling words and a status word
constexpr size_t kNoAllocCounterBytes =
    (size_t)(kNoAllocCounters + w4a16::kMmaSchedWords) * sizeof(unsigned);
constexpr size_t kNoAllocBytes =
    kNoAllocPartialFloats * sizeof(float) + kNoAllocCounterBytes + 4 * sizeof(unsigned);
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {
struct NoAllocDevice {
    bool ready = false;
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch
    w4a16::DeviceInfo dev{};
};
constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

unsigned *noalloc_counters(unsigned char *scratch) {
    return reinterpret_cast<unsigned *>(scratch + kNoAllocPartialFloats * sizeof(float));
}
int *noalloc_status(unsigned char *scratch) {
    return reinterpret_cast<int *>(scratch + kNoAllocPartialFloats * sizeof(float) +
                                   kNoAllocCounterBytes);
}

// Once per device, with that device current: the scratch's device address
// (cudaGetSymbolAddress), zeroed counters and status, the kernel attributes.
int noalloc_setup(int device, NoAllocDevice **out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice &d = g_noalloc[device];
    if (!d.ready) {
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return (int)e;
        unsigned char *base = (unsigned char *)ptr;
        // the counters, scheduling words and status word must start at zero
        // (the kernels leave them zeroed after each launch)
        e = cudaMemset(base + kNoAllocPartialFloats * sizeof(float), 0,
                       kNoAllocBytes - kNoAllocPartialFloats * sizeof(float));
        w4a16::DeviceInfo info{};
        info.device = device;
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, device);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&info.max_smem_optin,
                                       cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
        if (e == cudaSuccess) e = w4a16::mma_init(info);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return (int)e;
        d.scratch = base;
        d.dev = info;
        d.ready = true;
    }
    *out = &d;
    return 0;
}
}  // namespace

namespace w4a16 {
bool noalloc_scratch(int device, NoAllocScratch *out) {
    if (device < 0 || device >= kNoAllocMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const NoAllocDevice &d = g_noalloc[device];
    if (!d.ready) return false;
    out->status = noalloc_status(d.scratch);
    out->counters = noalloc_counters(d.scratch);
    out->counter_bytes = kNoAllocCounterBytes;
    return true;
}
}  // namespace w4a16

extern "C" int w4a16_linear_noalloc(const uint16_t *x, const uint32_t *qweight,
                                    const uint16_t *scales, const uint32_t *zeros, int M, int N,
                                    int K, int group, uint16_t *y, void *stream) {
    using namespace w4a16;
    // the argument rules of w4a16_linear, then this entry point's own limit
    int st = check_linear_args(x, qweight, scales, zeros, M, N, K, group, y);
    if (st) return st;
    if (M > kMmaMaxTokens) return W4A16_ERR_UNSUPPORTED;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return W4A16_ERR_CUDA;
    if (device < 0 || device >= kNoAllocMaxDevices) return W4A16_ERR_UNSUPPORTED;
    NoAllocDevice *nd = nullptr;
    if (noalloc_setup(device, &nd)) return W4A16_ERR_CUDA;
    MmaPlan plan = plan_mma(M, N, K, -1, nd->dev);
    if (!plan.ok) return W4A16_ERR_UNSUPPORTED;
    // sizes over the scratch are rejected before anything is launched
    if (plan.ws_bytes > kNoAllocPartialFloats * sizeof(float) ||
        (plan.S > 1 && plan.n_blocks > kNoAllocCounters))
        return W4A16_ERR_WORKSPACE;
    Workspace ws{};
    ws.partials = reinterpret_cast<float *>(nd->scratch);
    ws.partial_bytes = kNoAllocPartialFloats * sizeof(float);
    ws.counters = noalloc_counters(nd->scratch);
    ws.n_counters = kNoAllocCounters + kMmaSchedWords;
    ws.status = noalloc_status(nd->scratch);
    LinearArgs a{reinterpret_cast<const __half *>(x), qweight,
                 reinterpret_cast<const __half *>(scales), zeros, reinterpret_cast<__half *>(y), M,
                 N, K};
    e = launch_mma(a, plan, ws, (cudaStream_t)stream);
    if (e != cudaSuccess) return W4A16_ERR_CUDA;
    // one kernel, one linear, under the rung that computed it
    count_launches(plan.S > 1 ? W4A16_RUNG_MMA_SPLITK : W4A16_RUNG_MMA, 1, 1);
    return W4A16_OK;
}
