// Expert MLP decode kernel: a whole mixture-of-experts MLP for a few tokens in
// ONE launch (forum.sourcefind.cn thread "vLLM on Hygon Z100", section 七:
// tokens regrouped by expert, the W4A16 expert small-M GEMV over packed INT4
// experts, each token's expert outputs summed with the router's weights).
//
//   out[t] = sum_j w[t, j] * down_e(silu(gate_e(x[t])) * up_e(x[t])),  e = ids[t, j]
//
// At decode a token meets k of E experts and each expert in use sees one or
// two tokens: the weights of the experts in use are the whole cost, and the
// chain of align / prepare / GEMV / sum launches spends far longer on its own
// latency than on them.  Here every CTA derives the routing itself (at most
// 128 slots: a stable rank per slot), and the two linears run as two phases
// of one persistent grid:
//
//   * phase 1, gate+up with SiLU-and-mul: a unit is one warp's 16-row MMA
//     strip of one tile (an expert's slots, up to 8 = the MMA's N): rows
//     0..7 of the MMA are 8 gate rows, rows 8..15 the matching up rows, so
//     each lane holds a gate sum and its up sum for the same output and token
//     and applies silu(gate) * up in registers.  Units go to warps
//     interleaved across CTAs (warp w of CTA c takes units w * grid + c, ...),
//     spreading the few strips of a decode step over every SM.  x of every
//     token is copied (cp.async) as soon as the kernel may read it, while the
//     routing is worked out, and staged once per CTA;
//   * phase 2, down: a unit is one tile and a block of 128 output rows, one
//     16-row strip per warp of a CTA, and a CTA takes a contiguous range of
//     units (tile-major, so mostly blocks of one tile); for each new tile it
//     waits (bounded) for the tile's phase-1 strips (a completion counter per
//     tile) and stages the tile's intermediate rows once; it writes its
//     slots' outputs.  The CTA that brings a block's last tile sums the
//     block's outputs over each token's experts (j in order, fp32, one
//     rounding) into out;
//   * every warp streams its weights through its own two-slot ring of TMA
//     boxes (two 8-row boxes per stage: 16 rows x 4 groups x 64 bytes, the
//     rows' scale and zero words copied by the lanes onto the same
//     mbarrier), and the stream runs straight from a warp's phase-1 strips
//     into its phase-2 strips: the down weights are in flight while the
//     warp waits for the intermediate rows, which are the only thing phase 2
//     waits for;
//   * the inner product is the 4-bit mma rung's: one lop3 per nibble pair as
//     an exact fp16 subnormal, mma.sync.m16n8k16 with fp32 accumulation, the
//     zero point folded in through each group's sum of the activations, the
//     scale applied per group in fp32.  bf16 activations are staged as fp16
//     scaled by a power of two per row (undone at the end of each strip).
//
// The intermediate and the experts' outputs are rounded to the 16-bit type,
// as the chain of separate calls rounds them.  Every wait is bounded; an
// expired wait sets a status bit and the CTA drains its copies and leaves.
#include <cuda.h>
#include <string.h>

#include "../../include/w4a16.h"
#include "w4a16_internal.h"
#include "w4a16_mma_common.cuh"

namespace w4a16 {
namespace {

using namespace warp_mma;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCtasPerSm = 2;
constexpr int kStageGroups = 4;                          // groups per stage
constexpr int kHalfBox = 8 * kStageGroups * 64;          // 8 rows x 4 groups x 64 B
constexpr int kStageW = 2 * kHalfBox;                    // 4 KB of weights
constexpr int kStageMeta = 16 * 16;                      // per row: 3 scale words, 1 zeros word
constexpr int kStageBytes = kStageW + kStageMeta;
constexpr int kDepth = 2;                                // ring slots per warp
constexpr int kRingBytes = kWarps * kDepth * kStageBytes;  // 69632
constexpr int kBarBytes = kWarps * kDepth * 8;
constexpr int kMaxSlots = kMoeDecodeMaxSlots;
// routing tables: 10 arrays of kMaxSlots ints, then 16 flag ints
constexpr int kRouteInts = 10 * kMaxSlots + 16;
constexpr int kRouteBytes = kRouteInts * 4;
constexpr int kStagedOffset = kRingBytes + kBarBytes + kRouteBytes;
constexpr int kSmemPerCta = 228 * 1024 / kCtasPerSm - 1024;  // leaves the per-CTA reserve
constexpr int kBlockRows = kWarps * 16;                  // down rows per phase-2 unit
constexpr int kErrDecodeWait = 2048;  // device status bit: a wait of the decode kernel expired

static_assert(kStagedOffset % 16 == 0, "staged rows need 16-byte alignment");

// Flag ints after the routing arrays
constexpr int kFlagTiles = 0;      // number of tiles
constexpr int kFlagAbortC = 1;     // a ring wait expired (written while computing)
constexpr int kFlagAbortW = 2;     // thread 0's wait for a tile expired
constexpr int kFlagLast = 3;       // this CTA sums the current block
constexpr int kFlagWarpSum = 4;    // 4 ints: tile starts per warp of positions

struct MoeDecodeParams {
    CUtensorMap map1;  // gate+up qweight as (word in group, stacked row, group), box {16, 8, 4}
    CUtensorMap map2;  // down qweight, the same
    const __half *x;   // [T, H] by token
    const int32_t *ids;
    const float *w;    // [T * k]
    const __half *s1, *s2;  // scales [E * 2I, G1], [E * H, G2]
    const uint32_t *z1, *z2;
    uintptr_t s1_end, s2_end;  // one past each scales array
    uintptr_t z1_end, z2_end;  // one past each zeros array
    __half *h;         // [T * k, I]: the intermediate rows by sorted position
    __half *o;         // [T * k, H]: each slot's down output by sorted position
    __half *out;       // [T, H]
    unsigned *tile_done;  // [kMaxSlots] phase-1 strips finished per tile
    unsigned *blk;        // [H / 128] tiles finished per block of down rows
    unsigned *fin;        // CTAs finished
    int *status;
    int E, k, T, I, H;
    int G1, ZW1, G2, ZW2;
    int xstride1, xstride2;  // bytes per staged row of x (phase 1) and of h (phase 2)
    int sums_off;            // bytes from the staged rows to their group sums, then 8 exponents
};

// Staging of activation rows for the MMA's B operand, in two steps so that
// the copy overlaps other work:
//   copy_rows_async: every thread issues 16-byte cp.async copies (L2 only:
//     the rows may have been written by other CTAs of this grid) of `rows`
//     rows (row r at src + r * src_stride) into the staged rows, raw order,
//     committed as one group;
//   permute_rows (after cp.async.wait_group 0 and a barrier): 16-byte unit J
//     of a row moves to unit x_unit(J) in MMA pair order (bf16 as fp16 scaled
//     by 2^shift(row), shift from the row's largest exponent, kept in
//     exps[r]), and each group's sum of the staged values times 2^-20 goes to
//     sums[group * 8 + r].  A unit and its destination sit in the same half
//     warp, so a warp reads all its units before it writes.  Ends with a
//     barrier.
__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_committed() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void copy_rows_async(uint8_t *xs, int xstride, const __half *src,
                                                size_t src_stride, int rows, int G) {
    const int nunits = G * 16, total = rows * nunits;
    for (int i = threadIdx.x; i < total; i += kThreads) {
        const int r = i / nunits, J = i - r * nunits;
        cp16(dev::smem_u32(xs + (size_t)r * xstride + 16 * J), src + r * src_stride + 8 * J);
    }
    cp_commit();
}

template <bool kBf16>
__device__ __forceinline__ void permute_rows(uint8_t *xs, int xstride, int rows, int G,
                                             float *sums, int *exps) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nunits = G * 16;
    const int total = rows * nunits;  // a multiple of 16: a half warp holds one group
    if (kBf16) {
        // exps[] were cleared before the barrier that follows the copies
        for (int base = warp * 32; base < total; base += kThreads) {
            const int i = base + lane;
            const int r = i / nunits, J = i - r * nunits;
            int e = 0;
            if (i < total)
                e = max_bf16_exp(*reinterpret_cast<const uint4 *>(xs + (size_t)r * xstride + 16 * J));
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) e = max(e, __shfl_xor_sync(0xffffffffu, e, off));
            if (i < total && (J & 15) == 0) atomicMax(exps + r, e);
        }
        __syncthreads();
    }
    for (int base = warp * 32; base < total; base += kThreads) {
        const int i = base + lane;
        const bool valid = i < total;
        const int r = i / nunits, J = i - r * nunits;
        uint8_t *row = xs + (size_t)r * xstride;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (valid) v = *reinterpret_cast<const uint4 *>(row + 16 * J);
        if (kBf16 && valid) v = bf16_to_scaled_f16(v, pow2(bf16_stage_shift(exps[r])));
        __syncwarp();
        if (valid) *reinterpret_cast<uint4 *>(row + 16 * x_unit(J)) = mma_pair_order(v);
        const float2 a = pair_to_float2<false>(v.x), b = pair_to_float2<false>(v.y);
        const float2 e = pair_to_float2<false>(v.z), f = pair_to_float2<false>(v.w);
        float sum = ((a.x + a.y) + (b.x + b.y)) + ((e.x + e.y) + (f.x + f.y));
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (valid && (J & 15) == 0) sums[(J >> 4) * 8 + r] = sum * kTwoM20;
    }
    __syncthreads();
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    moe_decode_kernel(const __grid_constant__ MoeDecodeParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int cta = blockIdx.x, grid = gridDim.x;
    uint8_t *wring = smem + (size_t)warp * kDepth * kStageBytes;  // this warp's slots
    const uint32_t ring0 = dev::smem_u32(wring);
    const uint32_t bar0 = dev::smem_u32(smem + kRingBytes) + 8 * kDepth * warp;
    int *route = reinterpret_cast<int *>(smem + kRingBytes + kBarBytes);
    int *key = route;                      // per slot: expert << 8 | slot (INT_MAX: no expert)
    int *spos = route + kMaxSlots;         // per slot: its sorted position, -1 without expert
    int *ptok = route + 2 * kMaxSlots;     // per sorted position: its token
    int *pexp = route + 3 * kMaxSlots;     // per sorted position: its expert
    int *pend = route + 4 * kMaxSlots;     // per sorted position: end of its expert's run
    int *pstart = route + 5 * kMaxSlots;   // per sorted position: a tile starts here
    int *t_p0 = route + 6 * kMaxSlots;     // per tile: first sorted position
    int *t_e = route + 7 * kMaxSlots;      // per tile: expert
    int *t_n = route + 8 * kMaxSlots;      // per tile: slots (1..8)
    float *wts = reinterpret_cast<float *>(route + 9 * kMaxSlots);  // per slot: router weight
    volatile int *flags = route + 10 * kMaxSlots;
    uint8_t *xs = smem + kStagedOffset;
    float *sums = reinterpret_cast<float *>(xs + P.sums_off);
    const int Gmax = P.G1 > P.G2 ? P.G1 : P.G2;
    int *exps = reinterpret_cast<int *>(xs + P.sums_off + Gmax * 8 * 4);

    if (lane == 0) {
        // one arrival with the boxes' byte count, plus one per lane once its
        // metadata copies have landed
        for (int s = 0; s < kDepth; ++s) mbar_init(bar0 + 8 * s, 1 + 32);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x < 16) flags[threadIdx.x] = 0;
    grid_dependents_launch();
    // the routing, x and the router weights may come from the preceding
    // kernel; the intermediate rows, outputs and counters from the previous
    // launch of this kernel
    grid_dependency_wait();
    // x of every token goes out first (raw order), to be staged once it lands
    copy_rows_async(xs, P.xstride1, P.x, (size_t)P.H, P.T, P.G1);
    if (kBf16 && threadIdx.x < 8) exps[threadIdx.x] = 0;

    // ---- routing: slots grouped by expert, stable in slot order.  A slot's
    // sorted position is the number of (expert, slot) keys below its own.
    const int n_slots = P.T * P.k;
    const int tid = threadIdx.x;
    int my_key = 0x7fffffff;
    if (tid < n_slots) {
        const int e = P.ids[tid];
        const bool ok = e >= 0 && e < P.E;
        if (ok) my_key = (e << 8) | tid;
        else if (cta == 0) atomicOr(P.status, kErrMoeIds);
        wts[tid] = P.w[tid];
    }
    const int n4 = (n_slots + 3) & ~3;
    if (tid < n4) key[tid] = my_key;
    const int n_valid = __syncthreads_count(my_key != 0x7fffffff);
    if (tid < n_slots) {
        if (my_key != 0x7fffffff) {
            const int e = my_key >> 8, lo = e << 8, hi = (e + 1) << 8;
            int rank = 0, run0 = 0, run1 = 0;
            for (int s = 0; s < n4; s += 4) {
                const int4 kv = *reinterpret_cast<const int4 *>(key + s);
                rank += (kv.x < my_key) + (kv.y < my_key) + (kv.z < my_key) + (kv.w < my_key);
                run0 += (kv.x < lo) + (kv.y < lo) + (kv.z < lo) + (kv.w < lo);
                run1 += (kv.x < hi) + (kv.y < hi) + (kv.z < hi) + (kv.w < hi);
            }
            spos[tid] = rank;
            ptok[rank] = tid / P.k;
            pexp[rank] = e;
            pend[rank] = run1;
            pstart[rank] = ((rank - run0) & 7) == 0;  // every 8th slot of a run opens a tile
        } else {
            spos[tid] = -1;
        }
    }
    __syncthreads();
    // number the tiles in position order: warps 0..3 hold positions 0..127
    const bool opens = tid < n_valid && pstart[tid];
    const unsigned opens_mask = __ballot_sync(0xffffffffu, opens);
    if (warp < kMaxSlots / 32 && lane == 0) flags[kFlagWarpSum + warp] = __popc(opens_mask);
    __syncthreads();
    if (warp < kMaxSlots / 32) {
        int before = 0;
        for (int w2 = 0; w2 < warp; ++w2) before += flags[kFlagWarpSum + w2];
        if (opens) {
            const int t = before + __popc(opens_mask & ((1u << lane) - 1u));
            t_p0[t] = tid;
            t_e[t] = pexp[tid];
            t_n[t] = min(8, pend[tid] - tid);
        }
        if (tid == 0) {
            int total = 0;
            for (int w2 = 0; w2 < kMaxSlots / 32; ++w2) total += flags[kFlagWarpSum + w2];
            flags[kFlagTiles] = total;
        }
    }
    __syncthreads();
    const int n_tiles = flags[kFlagTiles];

    const int S1 = P.I / 8;               // phase-1 strips per tile (8 outputs each)
    const int B2 = P.H / kBlockRows;      // phase-2 blocks per tile
    const int n_u1 = n_tiles * S1, n_u2 = n_tiles * B2;
    // phase-2 units of this CTA: a contiguous range (units are tile-major, so
    // a CTA waits for and stages few tiles)
    const int u2_lo = (int)((long long)cta * n_u2 / grid);
    const int u2_hi = (int)((long long)(cta + 1) * n_u2 / grid);
    const int nst1 = (P.G1 + kStageGroups - 1) / kStageGroups;
    const int nst2 = (P.G2 + kStageGroups - 1) / kStageGroups;

    // ---- copy stream: this warp's phase-1 strips, then its strips of the
    // CTA's phase-2 units, stage by stage, kDepth stages ahead of the
    // consumer.  Stage t of the stream: box A (rows rowA..rowA+7) and box B
    // (rows rowB..rowB+7) of groups 4j..4j+3 of one strip.  Metadata: lane (r = lane % 16, hh = lane / 16) copies, for row r of the
    // stage (rows 0..7 box A's, 8..15 box B's), scale words 0 and 1 of the
    // stage (hh = 0) or scale word 2 and the zeros word (hh = 1): the three
    // aligned words that hold the stage's four scales.
    const int r = lane & 15, hh = lane >> 4;
    const int w_base = warp * grid + cta;  // this warp's first phase-1 unit
    const int w_step = grid * kWarps;
    const int n1w = w_base < n_u1 ? (n_u1 - 1 - w_base) / w_step + 1 : 0;
    const unsigned n_st1 = (unsigned)(n1w * nst1);
    const unsigned n_stages = n_st1 + (unsigned)((u2_hi - u2_lo) * nst2);
    struct StageLoc {
        int rowA, rowB, j;
        bool p1;
    };
    auto stage_at = [&](unsigned t) -> StageLoc {
        StageLoc L;
        if (t < n_st1) {
            const int q = (int)t / nst1;
            L.j = (int)t - q * nst1;
            const int u = w_base + q * w_step;
            const int tile = u / S1, st = u - tile * S1;
            L.rowA = t_e[tile] * 2 * P.I + 8 * st;  // gate rows
            L.rowB = L.rowA + P.I;                  // their up rows
            L.p1 = true;
        } else {
            const int t2 = (int)(t - n_st1), q = t2 / nst2;
            L.j = t2 - q * nst2;
            const int u = u2_lo + q;
            const int tile = u / B2, b = u - tile * B2;
            L.rowA = t_e[tile] * P.H + (b * kWarps + warp) * 16;
            L.rowB = L.rowA + 8;
            L.p1 = false;
        }
        return L;
    };
    unsigned t_iss = 0;  // stages issued by this warp
    auto issue_stage = [&](unsigned t) {
        const StageLoc L = stage_at(t);
        const CUtensorMap *map = L.p1 ? &P.map1 : &P.map2;
        const int G = L.p1 ? P.G1 : P.G2, ZW = L.p1 ? P.ZW1 : P.ZW2;
        const uint32_t slot = t & 1u;  // kDepth == 2
        const uint32_t bar = bar0 + 8 * slot;
        const uint32_t dst = ring0 + slot * kStageBytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, kStageW);
            tma_box(dst, map, L.rowA, kStageGroups * L.j, bar);
            tma_box(dst + kHalfBox, map, L.rowB, kStageGroups * L.j, bar);
        }
        // a scale word copies the part of it inside the array; a word past the
        // end becomes zeros, reads nothing and takes a valid source address
        const size_t row = (size_t)(r < 8 ? L.rowA + r : L.rowB + (r - 8));
        const __half *sc = L.p1 ? P.s1 : P.s2;
        const uintptr_t s_w = (((uintptr_t)(sc + row * G)) & ~(uintptr_t)3) + 8 * (uintptr_t)hh +
                              8 * (uintptr_t)L.j;
        const uintptr_t end = L.p1 ? P.s1_end : P.s2_end;
        const int avail = s_w < end ? (int)min((uintptr_t)16, end - s_w) : 0;
        const uint32_t md = dst + kStageW + r * 16 + 8 * hh;
        const int n0 = min(avail, 4);
        cp4(md, n0 ? s_w : (uintptr_t)sc, (uint32_t)n0);
        if (hh == 0) {
            const int n1 = min(max(avail - 4, 0), 4);
            cp4(md + 4, n1 ? s_w + 4 : (uintptr_t)sc, (uint32_t)n1);
        } else {
            cp4(md + 4, (uintptr_t)((L.p1 ? P.z1 : P.z2) + row * ZW + ((kStageGroups * L.j) >> 3)), 4u);
        }
        cp_arrive_noinc(bar);
    };
    auto issue_next = [&]() {
        if (t_iss >= n_stages) return;
        issue_stage(t_iss);
        ++t_iss;
    };
    static_assert(kDepth == 2, "the slot and phase arithmetic assumes two slots");
    for (int s = 0; s < kDepth; ++s) issue_next();

    // ---- consumer.  One strip: MMA rows 0..7 from box A, rows 8..15 from box
    // B; lane (g, c) feeds staged row xrow (its MMA column g) and keeps the
    // sums of MMA rows g and g + 8 for columns 2c, 2c + 1 (staged rows r0, r1
    // for the group sums).  acc: (row g, 2c) (row g, 2c+1) (row g+8, 2c)
    // (row g+8, 2c+1), each sum_g s * sum_k (q - z) x times 2^-20.
    const int xo0 = 16 * x_unit(4 * c + 0), xo1 = 16 * x_unit(4 * c + 1);
    const int xo2 = 16 * x_unit(4 * c + 2), xo3 = 16 * x_unit(4 * c + 3);
    unsigned t_cons = 0;  // stages consumed by this warp
    auto run_strip = [&](const __half *sc, int G, int nst, size_t rowa, size_t rowb,
                         const uint8_t *xrow, int r0, int r1, float (&acc)[4]) -> bool {
        const uintptr_t s0A = (uintptr_t)(sc + rowa * G), s0B = (uintptr_t)(sc + rowb * G);
        const uint32_t offA = (uint32_t)(s0A >> 1) & 1u, offB = (uint32_t)(s0B >> 1) & 1u;
        const uint32_t shA = 16u * offA, shB = 16u * offB;
        const uint32_t selA = offA ? 0x54u : 0x32u, selB = offB ? 0x54u : 0x32u;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = 0.f;
        for (int j = 0; j < nst; ++j) {
            const uint32_t slot = t_cons & 1u, par = (t_cons >> 1) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * slot, par))) return false;
            const uint8_t *st = wring + slot * kStageBytes;
            const uint8_t *stA = st + g * 64 + 16 * c, *stB = stA + kHalfBox;
            const uint4 ma = *reinterpret_cast<const uint4 *>(st + kStageW + g * 16);
            const uint4 mb = *reinterpret_cast<const uint4 *>(st + kStageW + (g + 8) * 16);
            const uint32_t zsh = ((j * kStageGroups) & 4) ? 16u : 0u;
            const uint32_t zwA = ma.w >> zsh, zwB = mb.w >> zsh;
            const uint32_t mA[3] = {ma.x, ma.y, ma.z}, mB[3] = {mb.x, mb.y, mb.z};
            const int n_in = min(kStageGroups, G - j * kStageGroups);
            const uint8_t *xg = xrow + (size_t)j * (kStageGroups * 256);
            const float *sg = sums + (j * kStageGroups) * 8;
            auto group = [&](const int i) {
                uint32_t hA, hB;  // scales of rows A and B: half (off + i) of the words
                if (i & 1) {
                    hA = dev::prmt(mA[i >> 1], mA[(i >> 1) + 1], selA);
                    hB = dev::prmt(mB[i >> 1], mB[(i >> 1) + 1], selB);
                } else {
                    hA = mA[i >> 1] >> shA;
                    hB = mB[i >> 1] >> shB;
                }
                const float sA = bits_to_float<kBf16>(hA & 0xffffu);
                const float sB = bits_to_float<kBf16>(hB & 0xffffu);
                // zero points as floats (2^23 + z, minus 2^23)
                const float zA = __uint_as_float(0x4b000000u | ((zwA >> (4 * i)) & 0xfu)) - 8388608.f;
                const float zB = __uint_as_float(0x4b000000u | ((zwB >> (4 * i)) & 0xfu)) - 8388608.f;
                const float sx0 = sg[i * 8 + r0], sx1 = sg[i * 8 + r1];  // S * 2^-20
                const uint8_t *xi = xg + i * 256;
                uint4 xv[4];
                xv[0] = *reinterpret_cast<const uint4 *>(xi + xo0);
                xv[1] = *reinterpret_cast<const uint4 *>(xi + xo1);
                xv[2] = *reinterpret_cast<const uint4 *>(xi + xo2);
                xv[3] = *reinterpret_cast<const uint4 *>(xi + xo3);
                const uint4 wa = *reinterpret_cast<const uint4 *>(stA + i * 512);
                const uint4 wb = *reinterpret_cast<const uint4 *>(stB + i * 512);
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
                acc[0] = fmaf(sA, fmaf(-zA, sx0, fmaf(16.f, dl[0], dh[0])), acc[0]);
                acc[1] = fmaf(sA, fmaf(-zA, sx1, fmaf(16.f, dl[1], dh[1])), acc[1]);
                acc[2] = fmaf(sB, fmaf(-zB, sx0, fmaf(16.f, dl[2], dh[2])), acc[2]);
                acc[3] = fmaf(sB, fmaf(-zB, sx1, fmaf(16.f, dl[3], dh[3])), acc[3]);
            };
            if (n_in == kStageGroups) {
#pragma unroll
                for (int i = 0; i < kStageGroups; ++i) group(i);
            } else {  // the last stage of a row whose groups are not a multiple of 4
#pragma unroll
                for (int i = 0; i < kStageGroups; ++i)
                    if (i < n_in) group(i);
            }
            // refill the slot once every lane is done with it: the lanes'
            // generic-proxy reads before the next box's async-proxy writes
            __syncwarp();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            ++t_cons;
            issue_next();
        }
        return true;
    };
    // acc -> the sums themselves (times 2^20), bf16 staging scales undone
    // (two multiplications: 2^20 times the unscale factor may not be finite)
    auto finish = [&](float (&acc)[4], int r0, int r1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] *= kTwo20;
        if (kBf16) {
            const float u0 = pow2(-bf16_stage_shift(exps[r0]));
            const float u1 = pow2(-bf16_stage_shift(exps[r1]));
            acc[0] *= u0;
            acc[1] *= u1;
            acc[2] *= u0;
            acc[3] *= u1;
        }
    };

    // ---- phase 1: gate+up with SiLU-and-mul, on x staged once per CTA
    bool dead = false;
    cp_wait_committed();
    __syncthreads();
    permute_rows<kBf16>(xs, P.xstride1, P.T, P.G1, sums, exps);
    for (int u = w_base; u < n_u1; u += w_step) {
        const int tile = u / S1, s = u - tile * S1;
        const int p0 = t_p0[tile], n = t_n[tile];
        // lanes of columns >= n compute a column nobody stores: they read column 0
        const int cb = g < n ? g : 0, c0 = 2 * c < n ? 2 * c : 0, c1 = 2 * c + 1 < n ? 2 * c + 1 : 0;
        const int tb = ptok[p0 + cb], tk0 = ptok[p0 + c0], tk1 = ptok[p0 + c1];
        const size_t ra = (size_t)t_e[tile] * 2 * P.I + 8 * s + g, rb = ra + P.I;
        float acc[4];
        if (!run_strip(P.s1, P.G1, nst1, ra, rb, xs + (size_t)tb * P.xstride1, tk0, tk1, acc)) {
            if (lane == 0) {
                atomicOr(P.status, kErrDecodeWait);
                flags[kFlagAbortC] = 1;
            }
            dead = true;
            break;
        }
        finish(acc, tk0, tk1);
        // h = silu(gate) * up, rounded once (silu(g) = g / (1 + e^-g))
        const int nout = 8 * s + g;
        if (2 * c < n)
            P.h[(size_t)(p0 + 2 * c) * P.I + nout] =
                from_float<kBf16>(acc[2] * (acc[0] / (1.f + expf(-acc[0]))));
        if (2 * c + 1 < n)
            P.h[(size_t)(p0 + 2 * c + 1) * P.I + nout] =
                from_float<kBf16>(acc[3] * (acc[1] / (1.f + expf(-acc[1]))));
        __syncwarp();  // the lanes' rows, then the strip's arrival
        if (lane == 0) {
            __threadfence();
            atomicAdd(P.tile_done + tile, 1u);
        }
    }

    // ---- phase 2: down, a tile and a block of 128 rows per unit, then the
    // weighted sum of a block by the CTA that finishes its last tile.  Every
    // warp reaches every barrier; an expired wait stops the CTA at the next.
    int staged_tile = -1;
    for (int u = u2_lo; u < u2_hi; ++u) {
        __syncthreads();  // the staged rows and the flags are settled
        if (flags[kFlagAbortC]) break;
        const int tile = u / B2, b = u - tile * B2;
        const int p0 = t_p0[tile], n = t_n[tile];
        if (tile != staged_tile) {
            // wait for the tile's phase-1 strips, then stage its intermediate rows
            if (threadIdx.x == 0 && !wait_counter(P.tile_done + tile, (unsigned)S1)) {
                atomicOr(P.status, kErrDecodeWait);
                flags[kFlagAbortW] = 1;
            }
            if (kBf16 && threadIdx.x < 8) exps[threadIdx.x] = 0;
            __syncthreads();
            if (flags[kFlagAbortW]) break;
            copy_rows_async(xs, P.xstride2, P.h + (size_t)p0 * P.I, (size_t)P.I, n, P.G2);
            cp_wait_committed();
            __syncthreads();
            permute_rows<kBf16>(xs, P.xstride2, n, P.G2, sums, exps);
            staged_tile = tile;
        }
        const int cb = g < n ? g : 0, c0 = 2 * c < n ? 2 * c : 0, c1 = 2 * c + 1 < n ? 2 * c + 1 : 0;
        const int row = (b * kWarps + warp) * 16 + g;  // output row of MMA row g
        const size_t ra = (size_t)t_e[tile] * P.H + row, rb = ra + 8;
        float acc[4];
        if (!dead &&
            !run_strip(P.s2, P.G2, nst2, ra, rb, xs + (size_t)cb * P.xstride2, c0, c1, acc)) {
            if (lane == 0) {
                atomicOr(P.status, kErrDecodeWait);
                flags[kFlagAbortC] = 1;
            }
            dead = true;
        }
        if (!dead) {
            finish(acc, c0, c1);
            if (2 * c < n) {
                __half *o = P.o + (size_t)(p0 + 2 * c) * P.H;
                o[row] = from_float<kBf16>(acc[0]);
                o[row + 8] = from_float<kBf16>(acc[2]);
            }
            if (2 * c + 1 < n) {
                __half *o = P.o + (size_t)(p0 + 2 * c + 1) * P.H;
                o[row] = from_float<kBf16>(acc[1]);
                o[row + 8] = from_float<kBf16>(acc[3]);
            }
        }
        __syncthreads();  // the CTA's outputs of the unit, then its arrival
        if (flags[kFlagAbortC]) break;
        if (threadIdx.x == 0) {
            __threadfence();
            flags[kFlagLast] = atomicAdd(P.blk + b, 1u) == (unsigned)n_tiles - 1u;
        }
        __syncthreads();
        if (flags[kFlagLast]) {
            // every tile of block b is in: out[t, rows of b] = sum_j w[t, j] *
            // o[pos(t, j)], j in order, fp32, one rounding
            __threadfence();
            for (int i = threadIdx.x; i < P.T * kBlockRows; i += kThreads) {
                const int t = i / kBlockRows, nrow = b * kBlockRows + (i - t * kBlockRows);
                // eight loads in flight at a time; a slot with an invalid
                // expert id (no position) is left out
                float a = 0.f;
                for (int j0 = 0; j0 < P.k; j0 += 8) {
                    __half v[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = j0 + jj, p = j < P.k ? spos[t * P.k + j] : -1;
                        v[jj] = p >= 0 ? __ldcg(P.o + (size_t)p * P.H + nrow) : __ushort_as_half(0);
                    }
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = j0 + jj, sl = t * P.k + j;
                        if (j < P.k && spos[sl] >= 0) a = fmaf(wts[sl], to_float<kBf16>(v[jj]), a);
                    }
                }
                P.out[(size_t)t * P.H + nrow] = from_float<kBf16>(a);
            }
            if (threadIdx.x == 0) P.blk[b] = 0u;  // ready for the next launch
        }
    }
    if (n_tiles == 0) {  // no slot has an expert: every output is an empty sum
        for (int i = cta * kThreads + threadIdx.x; i < P.T * P.H; i += grid * kThreads)
            P.out[i] = from_float<kBf16>(0.f);
    }

    // copies still in flight (an expired wait) land before shared memory goes
    for (; t_cons < t_iss; ++t_cons) mbar_wait(bar0 + 8 * (t_cons & 1u), (t_cons >> 1) & 1u);
    cp_wait_all();
    __syncthreads();
    if (threadIdx.x == 0 && !flags[kFlagAbortC] && !flags[kFlagAbortW]) {
        // the last CTA out leaves the tiles' counters zeroed for the next launch
        __threadfence();
        if (atomicAdd(P.fin, 1u) == (unsigned)grid - 1u) {
            __threadfence();
            for (int t = 0; t < n_tiles; ++t) P.tile_done[t] = 0u;
            *P.fin = 0u;
        }
    }
}

}  // namespace

bool moe_decode_shape_ok(int E, int H, int I) {
    // whole groups and whole 128-row blocks; gate+up rows of a strip in one expert
    return E >= 1 && E <= kMaxMoeExperts && H % kBlockRows == 0 && I % kGroup == 0 && H > 0 &&
           I > 0 && (long long)E * 2 * I < (1ll << 31) && (long long)E * H < (1ll << 31);
}


// qweight [rows, K/8] as (word in group, row, group), boxes of 8 rows x 4 groups
static cudaError_t encode_experts(CUtensorMap *map, const uint32_t *qw, long long rows, int K) {
    const EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorInitializationError;
    const cuuint64_t dims[3] = {16, (cuuint64_t)rows, (cuuint64_t)(K / kGroup)};
    const cuuint64_t strides[2] = {(cuuint64_t)K / 2, 64};
    const cuuint32_t box[3] = {16, 8, (cuuint32_t)kStageGroups};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, (void *)qw, dims, strides,
                                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                 CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t moe_decode_describe(const uint32_t *qw1, const __half *s1, const uint32_t *z1,
                                const uint32_t *qw2, const __half *s2, const uint32_t *z2, int E,
                                int H, int I, bool bf16, MoeDecodeWeights *w) {
    if (!tensor_map_encoder() || !moe_decode_shape_ok(E, H, I)) return cudaErrorInvalidValue;
    memset(w, 0, sizeof(*w));
    w->E = E;
    w->H = H;
    w->I = I;
    w->G1 = H / kGroup;
    w->ZW1 = (w->G1 + 7) / 8;
    w->G2 = I / kGroup;
    w->ZW2 = (w->G2 + 7) / 8;
    w->s1 = s1;
    w->s2 = s2;
    w->z1 = z1;
    w->z2 = z2;
    w->s1_end = (uintptr_t)(s1 + (size_t)E * 2 * I * w->G1);
    w->s2_end = (uintptr_t)(s2 + (size_t)E * H * w->G2);
    w->z1_end = (uintptr_t)(z1 + (size_t)E * 2 * I * w->ZW1);
    w->z2_end = (uintptr_t)(z2 + (size_t)E * H * w->ZW2);
    w->bf16 = bf16;
    cudaError_t e = encode_experts(&w->map1, qw1, (long long)E * 2 * I, H);
    if (e == cudaSuccess) e = encode_experts(&w->map2, qw2, (long long)E * H, I);
    return e;
}

// staged rows: x (T rows of H) in phase 1, a tile's intermediate rows (up to
// min(8, T*k) rows of I) in phase 2, in one area; then the group sums and 8
// exponents
static int staged_rows_bytes(const MoeDecodeWeights &w, int T, int k) {
    const int x1 = T * (w.H * 2 + 16);
    const int r2 = T * k < kMmaMaxTokens ? T * k : kMmaMaxTokens;
    const int x2 = r2 * (w.I * 2 + 16);
    return ((x1 > x2 ? x1 : x2) + 15) & ~15;
}

int moe_decode_smem(const MoeDecodeWeights &w, int T, int k) {
    if (T < 1 || k < 1 || T > kMoeDecodeMaxTokens || T * k > kMaxSlots) return -1;
    const int Gmax = w.G1 > w.G2 ? w.G1 : w.G2;
    const int bytes = kStagedOffset + staged_rows_bytes(w, T, k) + Gmax * 8 * 4 + 8 * 4;
    return bytes <= kSmemPerCta ? bytes : -1;
}

size_t moe_decode_counter_words(const MoeDecodeWeights &w) {
    return (size_t)kMaxSlots + w.H / kBlockRows + 1;
}

cudaError_t launch_moe_decode(const MoeDecodeWeights &w, const __half *x, const int32_t *ids,
                              const float *wts, int T, int k, __half *out,
                              const MoeDecodeBuffers &b, int *status, const DeviceInfo &dev,
                              cudaStream_t stream) {
    const int smem = moe_decode_smem(w, T, k);
    if (smem < 0) return cudaErrorInvalidValue;
    MoeDecodeParams P;
    memset(&P, 0, sizeof(P));
    P.map1 = w.map1;
    P.map2 = w.map2;
    P.x = x;
    P.ids = ids;
    P.w = wts;
    P.s1 = w.s1;
    P.s2 = w.s2;
    P.z1 = w.z1;
    P.z2 = w.z2;
    P.s1_end = w.s1_end;
    P.s2_end = w.s2_end;
    P.z1_end = w.z1_end;
    P.z2_end = w.z2_end;
    P.h = b.h;
    P.o = b.o;
    P.out = out;
    P.tile_done = b.counters;
    P.blk = b.counters + kMaxSlots;
    P.fin = b.counters + kMaxSlots + w.H / kBlockRows;
    P.status = status;
    P.E = w.E;
    P.k = k;
    P.T = T;
    P.I = w.I;
    P.H = w.H;
    P.G1 = w.G1;
    P.ZW1 = w.ZW1;
    P.G2 = w.G2;
    P.ZW2 = w.ZW2;
    P.xstride1 = w.H * 2 + 16;
    P.xstride2 = w.I * 2 + 16;
    P.sums_off = staged_rows_bytes(w, T, k);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCtasPerSm * dev.sm_count);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // every CTA resident at once (phase 2 waits for other CTAs' phase 1), and
    // the launch may begin while the preceding kernel drains
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return w.bf16 ? cudaLaunchKernelEx(&cfg, moe_decode_kernel<true>, P)
                  : cudaLaunchKernelEx(&cfg, moe_decode_kernel<false>, P);
}

cudaError_t moe_decode_init(const DeviceInfo &dev) {
    if (!tensor_map_encoder()) return cudaErrorSymbolNotFound;
    int dyn = kSmemPerCta;
    if (dyn > dev.max_smem_optin - 1024) dyn = dev.max_smem_optin - 1024;
    const void *fns[2] = {(const void *)moe_decode_kernel<false>,
                          (const void *)moe_decode_kernel<true>};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fns[i], cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
    }
    return e;
}

}  // namespace w4a16
