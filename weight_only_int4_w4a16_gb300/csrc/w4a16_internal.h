// Internal interface between the C ABI (w4a16_api.cu) and the kernel files.
// Nothing here is exported from the shared library.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace w4a16 {

constexpr int kGroup = 128;  // inputs per quantisation group

// What follows the linear in the same kernel (the values of w4a16_epilogue):
// nothing; y = h + residual; y = silu(h[:, :N/2]) * h[:, N/2:], h = x W^T.
constexpr int kEpiNone = 0;
constexpr int kEpiResidual = 1;
constexpr int kEpiSiluMul = 2;
// The 16-bit type of x, scales, y and the residual (the values of w4a16_dtype).
constexpr int kDtypeF16 = 0;
constexpr int kDtypeBf16 = 1;

// One W4A16 linear, device pointers.  x [M, K] fp16; qw [N, K/8]; scales
// [N, G] fp16; zeros [N, ceil(G/8)]; y [M, N] fp16 ([M, N/2] for SiLU-and-mul);
// residual [M, N] fp16 (the residual epilogue only).
struct LinearArgs {
    const __half *x;
    const uint32_t *qw;
    const __half *scales;
    const uint32_t *zeros;
    __half *y;
    int M, N, K;
    int epi = kEpiNone;
    const __half *residual = nullptr;
    int dtype = kDtypeF16;  // bf16 data travels in __half storage, reinterpreted
};

// Output columns of a linear with epilogue epi.
inline int out_cols(int N, int epi) { return epi == kEpiSiluMul ? N / 2 : N; }

// Library-owned scratch for the split-K rungs: fp32 partial outputs and one
// arrival counter per output tile (zeroed at init, reset by the reducing CTA).
struct Workspace {
    float *partials;
    size_t partial_bytes;
    unsigned *counters;
    int n_counters;
    int *status;  // device word: kernels OR in an error code when a bounded wait expires
};

// cuTensorMapEncodeTiled from the driver, looked up once (null if the driver
// lacks it); every kernel that reads through TMA encodes its maps with it.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;
};

// ---- CUDA-core GEMV rungs (w4a16_gemv.cu) --------------------------------
constexpr int kGemvMaxTokens = 8;  // tokens per launch on the CUDA-core rungs

struct GemvPlan {
    bool ok;            // false: the shape cannot run with the requested split rule
    int M;              // tokens handled by this launch (1..8)
    int S;              // K slices (1 = no split)
    int slice_groups;   // groups per slice (last slice may hold fewer)
    int rows_per_cta;   // output rows per row block
    int n_row_blocks;   // ceil(N / rows_per_cta)
    int grid_x;         // CTAs per slice (grid-stride over row blocks)
    int smem_bytes;     // dynamic shared memory (staged activations)
    size_t ws_bytes;    // split-K partial bytes (0 when S == 1)
    int threads;        // per CTA
};

// split: 0 = never split K, 1 = split K (at least 2 slices when G >= 2),
// -1 = let the planner decide.
GemvPlan plan_gemv(int M, int N, int K, int split, const DeviceInfo &dev);
cudaError_t launch_gemv(const LinearArgs &a, const GemvPlan &plan, const Workspace &ws,
                        cudaStream_t stream);
cudaError_t gemv_init_attributes(const DeviceInfo &dev);

// ---- tcgen05 dequant-GEMM rungs (w4a16_tc.cu) -----------------------------
constexpr int kTcMaxTokens = 64;  // tokens per launch on the tensor-core rungs

struct TcPlan {
    bool ok;
    int M;             // real tokens in this launch (1..64)
    int T;             // MMA N: tokens padded to 16, 32 or 64
    int S;             // 1: every CTA takes whole 128-row tiles; 2: stream-K (CTAs take equal
                       // runs of (tile, stage) work and a tile split between CTAs is summed
                       // by the last of them)
    int n_tiles;       // 128-row weight tiles
    int spt;           // stages (4 groups each) per tile
    int grid;          // CTAs (one per SM)
    int stages;        // shared-memory stages in flight per CTA
    size_t ws_bytes;   // workspace: stream-K partial sums
    int threads;       // per CTA
};

// split: 0 = whole tiles only, 1 = stream-K, -1 = planner decides.  epi: the
// linear's epilogue (SiLU-and-mul tiles hold 64 outputs' gate and up rows).
TcPlan plan_tc(int M, int N, int K, int split, const DeviceInfo &dev, int epi = kEpiNone);
// status: device word the kernel ORs an error code into when a bounded wait expires.
cudaError_t launch_tc(const LinearArgs &a, const TcPlan &plan, const Workspace &ws, int *status,
                      cudaStream_t stream);
cudaError_t tc_init(const DeviceInfo &dev);

// One linear of a fused tcgen05 round, as the kernel reads it (device memory;
// the tensor maps are written by the host only).  A round is one stream-K
// sequence of (linear, tile, stage) work: linear l owns stages [start, start
// + n_tiles * spt).
struct TcLinDesc {
    CUtensorMap wmap;  // qweight 3-D: (16 words, N rows, G groups), box {16, 64, 4}
    CUtensorMap xmap;  // x 2-D: (K, M), box {64, T}, 128-byte swizzle
    const __half *x;
    const uint32_t *qw;
    const __half *scales;
    const uint32_t *zeros;
    __half *y;
    const __half *residual;  // y = h + residual, else null
    unsigned *counters;      // this linear's per-tile arrival counters (split tiles)
    long long start;         // its first stage in the round's sequence
    int N, K, G, ZW;
    int silu;                // SiLU-and-mul tiles (64 gate rows, their up rows N/2 below)
    int n_tiles, spt;
    int wait_for;            // -1, or an earlier linear that must finish first
};
// A fused tcgen05 round: n linears of M (9..64) tokens.
struct TcRound {
    const TcLinDesc *descs;  // device [n]
    int n;
    int M, T;
    long long total;         // stages of all linears
    int grid, stages;
    float *partials;         // [2 * grid][M][128] fp32
    unsigned *done;          // [n] tiles finished per linear, then 1 word: CTAs finished;
                             // null when no linear waits for another
    bool bf16;
};
// Fills r (except descs and done) and the descriptors' plan fields (n_tiles,
// spt, start) for linears of shapes (N[l], K[l], epi[l]); false when the
// round cannot take them.  ws_floats: the partial sums it needs.
bool plan_tc_round(int M, const int *N, const int *K, const int *epi, int n, const DeviceInfo &dev,
                   TcRound *r, TcLinDesc *descs, size_t *ws_floats);
// The tensor maps and pointers of one linear of a round.
cudaError_t tc_describe(const LinearArgs &a, int T, TcLinDesc *d);
cudaError_t launch_tc_round(const TcRound &r, int *status, cudaStream_t stream);

// ---- warp-level tensor-core MMA rungs (w4a16_mma.cu) ----------------------
constexpr int kMmaMaxTokens = 8;  // tokens per launch (the MMA's N = 8)

// The work of one linear is cut into units: one K slice of 8 * strips_per_warp
// strips of 16 rows (strips_per_warp per warp of a CTA, which stages the
// slice's activations once for all of them).  CTAs take units round-robin.
// With SiLU-and-mul a strip is logical: 16 gate rows and the 16 up rows N/2
// below them, computed one after the other by the same warp.
struct MmaPlan {
    bool ok;
    int M;             // tokens (1..8)
    int S;             // K slices
    int slice_groups;  // groups per slice (a multiple of 4; the last slice may hold fewer)
    int n_strips;      // 16-row strips
    int strips_per_warp;
    int n_blocks;      // units per slice: ceil(n_strips / (warps * strips_per_warp))
    int units;         // S * n_blocks
    bool reduce;       // sums go to the workspace, a block's last CTA reduces them
                       // (S > 1, or SiLU-and-mul); n_blocks arrival counters
    int grid;          // CTAs of a launch of this linear alone
    int smem_bytes;    // dynamic shared memory of such a launch
    size_t ws_bytes;   // split-K partial bytes (0 when S == 1)
    int warps;         // CTA shape: 8 warps (two CTAs per SM) or 16 (one per SM)
};

// One linear as the kernel reads it: in the kernel's parameters for a launch
// of one linear, in device memory for a fused round.
struct MmaLinDesc {
    CUtensorMap tmap;  // qweight as a 3-D tensor: (word in group, row, group)
    // when set, the tensor map to use instead of tmap: one written by the host
    // (expert tiles, whose descriptors a kernel writes, point at their
    // expert's map; a tensor map is never written by a kernel)
    const CUtensorMap *tmap_ref;
    const __half *x;
    const __half *scales;
    const uint32_t *zeros;
    __half *y;
    float *partials;      // this linear's partial sums (S > 1 or SiLU-and-mul)
    unsigned *counters;   // this linear's per-block arrival counters (the same)
    uintptr_t scales_first;  // the aligned word holding the first scale
    uintptr_t scales_end;    // one past the last byte of the scales array
    const __half *residual;  // kEpiResidual: [M, N], read before y is written
    int epi;                 // kEpiNone, kEpiResidual or kEpiSiluMul
    int ycols;               // columns of y (and of the residual)
    int half_strips;         // kEpiSiluMul: strips of the gate half (the up strip of
                             // logical strip s is strip s + half_strips)
    int N, K, G, ZW, M, S, slice_groups, n_strips, strips_per_warp, n_blocks;
    int unit_start;  // index of the linear's first unit in the fused list
    int xstride;     // bytes per staged token row
    int wait_for;    // fused round: linear that must be complete before this one reads x (-1: none)
};

// split: 0 = never split K, 1 = split K, -1 = planner balances the warps,
// 2 = fused rounds: fewest slices the staged activations allow, and units of
// kRoundStripsPerWarp strips per warp (the round's units balance each other),
// 3 = the same slices with one strip per warp (the round's last linears, so
// that the CTAs finish together).
// copies: the number of such linears that run side by side in one launch
// (the expert tiles of a mixture of experts); the one-linear cost model
// weighs their units together.
// warps: the CTA shape, 8 or 16; 0 = chosen for a linear launched alone (a
// fused round chooses one shape for all its linears: mma_round_warps)
MmaPlan plan_mma(int M, int N, int K, int split, const DeviceInfo &dev, int epi = kEpiNone,
                 int copies = 1, int warps = 0);
cudaError_t mma_describe(const LinearArgs &a, const MmaPlan &plan, float *partials,
                         unsigned *counters, int unit_start, int wait_for, MmaLinDesc *d);
cudaError_t launch_mma(const LinearArgs &a, const MmaPlan &plan, const Workspace &ws,
                       cudaStream_t stream);

// A fused round: n linears in one launch, their units in order.  done points
// at n zeroed counters when some linear waits for another (else null); the
// kernel leaves them zeroed again.
// The mma kernels take their scheduling counters from the last
// kMmaSchedWords words of the workspace counters.
constexpr int kMmaSchedWords = 2;

struct MmaRound {
    const MmaLinDesc *descs;  // device array of n descriptors
    int n;
    int total_units;
    int smem_bytes;
    unsigned *done;
    bool bf16;  // every linear of the round has bf16 data
    int warps = 8;  // the CTA shape of every linear's plan
    // expert groups: the descriptors come from the preceding kernel, which
    // writes the linear count and total units here (n and total_units are
    // then upper bounds, for the grid)
    const int *counts = nullptr;
};
int mma_round_grid(const DeviceInfo &dev, int warps);
int mma_smem_bytes(int M, int slice_groups, int warps);
// the CTA shape for a fused round of n linears (K[l] x N[l]) at M tokens:
// 16 warps where their room for x removes the K split from most bytes
int mma_round_warps(int M, const int *K, const int *N, int n);
cudaError_t launch_mma_round(const MmaRound &r, const Workspace &ws, const DeviceInfo &dev,
                             cudaStream_t stream);
cudaError_t mma_init(const DeviceInfo &dev);

// ---- dense 16-bit linear (w4a16_dense.cu) ---------------------------------
struct DensePlan {
    bool ok;
    int M;               // tokens (1..8)
    int S;               // K slices
    int slice_stages;    // 128-k stages per slice
    int n_strips;        // 16-row strips
    int strips_per_warp;
    int n_blocks;        // blocks of 8 * strips_per_warp strips
    int units;           // S * n_blocks
    int grid;
    int smem_bytes;
    size_t ws_bytes;     // split-K partial bytes (0 when S == 1)
};
DensePlan plan_dense(int M, int N, int K, const DeviceInfo &dev);
// y [M, N] = x [M, K] @ w [N, K]^T, 16-bit data (bf16: bfloat16 in __half storage)
cudaError_t launch_dense(const __half *x, const __half *w, __half *y, int M, int N, int K,
                         bool bf16, const DensePlan &plan, const Workspace &ws,
                         cudaStream_t stream);
cudaError_t dense_init(const DeviceInfo &dev);

// ---- mixture of experts (w4a16_moe.cu) -------------------------------------
constexpr int kMaxMoeExperts = 1024;
constexpr int kMaxMoeTiles = 2048;  // tiles of up to 8 slots per launch
constexpr int kErrMoeIds = 1024;  // device status bit: an expert id outside [0, E)
// Where the tiles of one expert-group launch put their results: y rows in
// sorted order, and per tile its own split-K partials and counters.
struct MoeTileSpace {
    __half *y;
    float *partials;        // null when the plan needs none
    size_t partial_stride;  // floats per tile
    unsigned *counters;
    size_t counter_stride;  // counters per tile
};
cudaError_t launch_moe_align(const int32_t *ids, int n_slots, int E, int32_t *sorted,
                             int32_t *pos, int32_t *offsets, int *status, cudaStream_t stream);
// tmpl2: null, or a second linear (the expert MLP's down projection) whose
// tiles follow the first's, read its outputs and wait for them
cudaError_t launch_moe_prepare(const MmaLinDesc *tmpl, const MmaLinDesc *tmpl2,
                               const int32_t *offsets, const int32_t *sorted, int E, int k,
                               int max_tiles, int units1, int units2, const MoeTileSpace &sp,
                               const MoeTileSpace &sp2, const __half *x, bool gather, __half *xs,
                               int n_slots, int K, MmaLinDesc *tiles, int *counts,
                               cudaStream_t stream);
cudaError_t launch_moe_sum(const __half *y, const int32_t *pos, const float *w, int T, int k,
                           int N, bool bf16, __half *out, cudaStream_t stream);

// ---- expert MLP decode kernel (w4a16_moe_decode.cu) ------------------------
constexpr int kMoeDecodeMaxSlots = 128;  // T * k per launch
constexpr int kMoeDecodeMaxTokens = 8;
// The two expert layers of an MLP as the decode kernel reads them: gate+up
// [E, 2I, H] (gate rows first, SiLU-and-mul) and down [E, H, I], stacked
// experts, with the tensor maps written once.
struct MoeDecodeWeights {
    CUtensorMap map1, map2;
    const __half *s1, *s2;
    const uint32_t *z1, *z2;
    uintptr_t s1_end, s2_end, z1_end, z2_end;
    int E, I, H, G1, ZW1, G2, ZW2;
    bool bf16;
};
// per call: intermediate rows [T*k, I] and expert outputs [T*k, H] (16-bit),
// and moe_decode_counter_words zeroed counters (the kernel leaves them zeroed)
struct MoeDecodeBuffers {
    __half *h, *o;
    unsigned *counters;
};
bool moe_decode_shape_ok(int E, int H, int I);
cudaError_t moe_decode_describe(const uint32_t *qw1, const __half *s1, const uint32_t *z1,
                                const uint32_t *qw2, const __half *s2, const uint32_t *z2, int E,
                                int H, int I, bool bf16, MoeDecodeWeights *w);
// dynamic shared memory of a launch for T tokens of k choices; -1: does not fit
int moe_decode_smem(const MoeDecodeWeights &w, int T, int k);
size_t moe_decode_counter_words(const MoeDecodeWeights &w);
cudaError_t launch_moe_decode(const MoeDecodeWeights &w, const __half *x, const int32_t *ids,
                              const float *wts, int T, int k, __half *out,
                              const MoeDecodeBuffers &b, int *status, const DeviceInfo &dev,
                              cudaStream_t stream);
cudaError_t moe_decode_init(const DeviceInfo &dev);

// ---- expired-wait probe (w4a16_waitprobe.cu) -------------------------------
constexpr int kErrProbeCounterWait = 4096;  // device status bit: the probe's counter wait expired
constexpr int kErrProbeBarrierWait = 8192;  // device status bit: the probe's mbarrier wait expired
// stale: null, or an arrival counter the probe increments first, leaving it as
// a split-K launch cut short by an expired wait can leave one (an arrival
// counted, the block never reduced)
cudaError_t launch_wait_probe(int *status, unsigned *stale, cudaStream_t stream);

// ---- shared by the entry points (w4a16_api.cu) -----------------------------
// The argument rules of w4a16_linear (and of the epilogue and dtype variants):
// a w4a16_status, W4A16_OK when the call may launch.
int check_linear_args(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                      const uint32_t *zeros, int M, int N, int K, int group, const uint16_t *y,
                      int epi = kEpiNone, const uint16_t *residual = nullptr,
                      int dtype = kDtypeF16);
// Record `linears` linears computed by `rung` and `kernels` kernel launches in
// the per-rung probe counters and the launch count (w4a16_probe_counts,
// w4a16_kernel_launches).
void count_launches(int rung, unsigned long long linears, unsigned long long kernels);

// ---- the allocation-free linear's scratch (w4a16_mma.cu) -------------------
// Where a device's static scratch keeps its status word and its counters
// (block arrival counters, then the kernel's scheduling words), once a
// w4a16_linear_noalloc call has set that device up.
struct NoAllocScratch {
    int *status;
    unsigned *counters;
    size_t counter_bytes;  // the counters and scheduling words, all zero between launches
};
// false when no w4a16_linear_noalloc call has set up `device` yet
bool noalloc_scratch(int device, NoAllocScratch *out);

// ---- pack / unpack / dequant (w4a16_pack.cu) ------------------------------
cudaError_t launch_pack(const uint8_t *q, const uint8_t *z, int N, int K, uint32_t *qw,
                        uint32_t *zeros, cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t *qw, const uint32_t *zeros, int N, int K, uint8_t *q,
                          uint8_t *z, cudaStream_t stream);
cudaError_t launch_dequant(const uint32_t *qw, const __half *scales, const uint32_t *zeros,
                           int N, int K, float *w_f32, __half *w_f16, cudaStream_t stream);
// src [rows, cols/8] words packed along cols (nibble order `order`) ->
// dst [cols, ceil(rows/8)] words packed along rows, sequential, pad nibbles 0.
cudaError_t launch_transpose_u4(const uint32_t *src, int rows, int cols, uint32_t order,
                                uint32_t *dst, cudaStream_t stream);
// src [rows, cols] -> dst [cols, rows], 16-bit elements.
cudaError_t launch_transpose_u16(const uint16_t *src, int rows, int cols, uint16_t *dst,
                                 cudaStream_t stream);

}  // namespace w4a16
