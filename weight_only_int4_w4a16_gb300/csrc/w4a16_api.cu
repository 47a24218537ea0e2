// C ABI of the W4A16 library: argument validation, the dispatch table with its
// per-rung probe counters, the split-K workspace, decode rounds and their
// CUDA-graph capture.  See include/w4a16.h for the contract of each call.
//
// Dispatch follows the ninfer-perf-tuning notes (section 二, "first ask which
// rung ran"): rungs are chosen from the shape (M, N, K), the table is frozen
// for the process, an environment variable read once at init can pin a rung,
// and every launch bumps its rung's counter so a run can prove which branch it
// took.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/w4a16.h"
#include "w4a16_internal.h"

using namespace w4a16;

namespace {

struct State {
    bool initialized = false;
    DeviceInfo dev{};
    Workspace ws{};
    void *ws_base = nullptr;
    void *round_descs = nullptr;  // device copy of the last fused round's descriptors
    std::vector<unsigned char> round_uploaded;  // what that copy holds
    int forced_rung = W4A16_RUNG_AUTO;
    bool log = false;
};

State g_state;
std::mutex g_mutex;
std::atomic<unsigned long long> g_probe[W4A16_NUM_RUNGS];
std::atomic<unsigned long long> g_launches{0};
thread_local int t_last_cuda_error = 0;

constexpr size_t kDefaultWorkspace = 64ull << 20;
constexpr int kCounters = 1 << 20;       // split-K arrival counters (and round completion counters)
constexpr int kMaxRoundLinears = 4096;   // linears of one fused decode round
constexpr int kRoundTailLinears = 24;    // a round's last linears, planned with small units
constexpr int kMaxM = 65535;

const char *const kRungNames[W4A16_NUM_RUNGS] = {"gemv", "gemv_splitk", "tc",
                                                  "tc_splitk", "mma", "mma_splitk"};

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return W4A16_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

constexpr int kMaxK = 1 << 22;
constexpr int kMaxRepackDim = 1 << 24;  // rows and columns of a repacked matrix
static_assert(kEpiNone == W4A16_EPILOGUE_NONE && kEpiResidual == W4A16_EPILOGUE_RESIDUAL &&
                  kEpiSiluMul == W4A16_EPILOGUE_SILU_MUL,
              "internal epilogue codes follow the ABI");
static_assert(kDtypeF16 == W4A16_DTYPE_F16 && kDtypeBf16 == W4A16_DTYPE_BF16,
              "internal 16-bit type codes follow the ABI");

int check_shape(int N, int K, int group) {
    if (N < 1 || K < 1 || K > kMaxK) return W4A16_ERR_INVALID_ARG;
    if (group != kGroup) return W4A16_ERR_UNSUPPORTED;
    if (K % kGroup != 0) return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

int check_linear(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                 const uint32_t *zeros, int M, int N, int K, int group, const uint16_t *y,
                 int epi = W4A16_EPILOGUE_NONE, const uint16_t *residual = nullptr,
                 int dtype = W4A16_DTYPE_F16) {
    if (!x || !qweight || !scales || !zeros || !y) return W4A16_ERR_INVALID_ARG;
    if (M < 1 || M > kMaxM) return W4A16_ERR_INVALID_ARG;
    if (dtype != W4A16_DTYPE_F16 && dtype != W4A16_DTYPE_BF16) return W4A16_ERR_INVALID_ARG;
    int st = check_shape(N, K, group);
    if (st) return st;
    if (epi != W4A16_EPILOGUE_NONE && epi != W4A16_EPILOGUE_RESIDUAL &&
        epi != W4A16_EPILOGUE_SILU_MUL)
        return W4A16_ERR_INVALID_ARG;
    // a residual exactly when the epilogue adds one
    if ((epi == W4A16_EPILOGUE_RESIDUAL) != (residual != nullptr)) return W4A16_ERR_INVALID_ARG;
    if (epi == W4A16_EPILOGUE_SILU_MUL && N % 32 != 0) return W4A16_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(qweight, 16) || !aligned(y, 16) || !aligned(scales, 2) ||
        !aligned(zeros, 4) || (residual && !aligned(residual, 2)))
        return W4A16_ERR_MISALIGNED;
    const size_t ybytes = (size_t)M * out_cols(N, epi) * 2;
    if (overlaps(x, (size_t)M * K * 2, y, ybytes)) return W4A16_ERR_INVALID_ARG;
    // the residual is y itself (y += x W^T) or lies apart from it
    if (residual && residual != y && overlaps(residual, ybytes, y, ybytes))
        return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

// The dispatch table.  Rungs that cannot run a shape are skipped in auto mode;
// a forced rung that cannot run it makes the call fail with UNSUPPORTED.
// Auto: up to 8 tokens on the CUDA-core GEMV (split K when the row blocks
// alone cannot fill the GPU), more tokens on the tcgen05 dequant-GEMM.
struct Decision {
    int rung;
    int status;
};

bool is_tc(int rung) { return rung == W4A16_RUNG_TC || rung == W4A16_RUNG_TC_SPLITK; }
bool is_mma(int rung) { return rung == W4A16_RUNG_MMA || rung == W4A16_RUNG_MMA_SPLITK; }

int tile_tokens(int rung) {
    return is_tc(rung) ? kTcMaxTokens : (is_mma(rung) ? kMmaMaxTokens : kGemvMaxTokens);
}

// A small fp16 linear without an epilogue, launched alone, runs faster on the
// CUDA-core gemv kernel: its launch is lighter than the warp-MMA kernel's
// (no tensor maps, no staged x, no mbarrier ring), and the weights are too few
// for the MMA kernel's per-weight advantage to pay that back.  The weight
// counts up to which it wins come from single launches with L2 evicted (one
// GB300): at 1..2 tokens up to 24 Mi weights (N 6144, K 4096: 14.3 against
// 16.4 us; a tie at 32 Mi), at 3..4 tokens up to 16 Mi (N 4096, K 4096: 16.4
// against 18.4 us; slower at 24 Mi), at 5..8 tokens up to 8 Mi (N 512, K 16384
// split: 18.4 against 24.5 us; slower at 16 Mi on most shapes).
bool gemv_small(int M, int N, int K) {
    const long long w = (long long)N * K;
    const long long lim = M <= 2 ? (24ll << 20) : M <= 4 ? (16ll << 20) : (8ll << 20);
    return M <= kMmaMaxTokens && w <= lim;
}

Decision decide(int M, int N, int K, const DeviceInfo &dev, int forced, int epi = kEpiNone,
                int dtype = kDtypeF16) {
    const int Mt = M < kGemvMaxTokens ? M : kGemvMaxTokens;
    const int G = K / kGroup;
    if (epi != kEpiNone || dtype != kDtypeF16) {
        // the epilogues and bf16 data run in the warp-MMA kernel (tiles of up
        // to 8 tokens, each reading the weights) and in the tcgen05 kernel (up
        // to 64 tokens per reading of the weights), not on the CUDA cores
        if (forced != W4A16_RUNG_AUTO && !is_mma(forced) && !is_tc(forced))
            return {forced, W4A16_ERR_UNSUPPORTED};
        if (forced == W4A16_RUNG_AUTO) {
            if (M > kMmaMaxTokens) {
                const int Mtc = M < kTcMaxTokens ? M : kTcMaxTokens;
                TcPlan t = plan_tc(Mtc, N, K, -1, dev, epi);
                return {t.S > 1 ? W4A16_RUNG_TC_SPLITK : W4A16_RUNG_TC, W4A16_OK};
            }
            MmaPlan p = plan_mma(Mt, N, K, -1, dev, epi);
            return {p.S > 1 ? W4A16_RUNG_MMA_SPLITK : W4A16_RUNG_MMA, W4A16_OK};
        }
    }
    switch (forced) {
        case W4A16_RUNG_GEMV: {
            GemvPlan p = plan_gemv(Mt, N, K, 0, dev);
            return {W4A16_RUNG_GEMV, p.ok ? W4A16_OK : W4A16_ERR_UNSUPPORTED};
        }
        case W4A16_RUNG_GEMV_SPLITK:
        case W4A16_RUNG_TC_SPLITK:
        case W4A16_RUNG_MMA_SPLITK:
            return {forced, G >= 2 ? W4A16_OK : W4A16_ERR_UNSUPPORTED};
        case W4A16_RUNG_TC:
            return {W4A16_RUNG_TC, W4A16_OK};
        case W4A16_RUNG_MMA: {
            MmaPlan p = plan_mma(Mt, N, K, 0, dev, epi);
            return {W4A16_RUNG_MMA, p.ok ? W4A16_OK : W4A16_ERR_UNSUPPORTED};
        }
        default:
            break;
    }
    if (M <= kMmaMaxTokens) {
        if (gemv_small(M, N, K)) {
            // the whole K per warp where the plan allows it (faster on every
            // small shape measured), else K split
            if (plan_gemv(Mt, N, K, 0, dev).ok) return {W4A16_RUNG_GEMV, W4A16_OK};
            if (G >= 2) return {W4A16_RUNG_GEMV_SPLITK, W4A16_OK};
        }
        MmaPlan p = plan_mma(Mt, N, K, -1, dev, epi);
        return {p.S > 1 ? W4A16_RUNG_MMA_SPLITK : W4A16_RUNG_MMA, W4A16_OK};
    }
    const int Mtc = M < kTcMaxTokens ? M : kTcMaxTokens;
    TcPlan t = plan_tc(Mtc, N, K, -1, dev);
    return {t.S > 1 ? W4A16_RUNG_TC_SPLITK : W4A16_RUNG_TC, W4A16_OK};
}

int split_rule(int rung) {
    switch (rung) {
        case W4A16_RUNG_GEMV:
        case W4A16_RUNG_TC:
        case W4A16_RUNG_MMA: return 0;
        case W4A16_RUNG_GEMV_SPLITK:
        case W4A16_RUNG_TC_SPLITK:
        case W4A16_RUNG_MMA_SPLITK: return 1;
    }
    return -1;
}

// Workspace bytes and counters one launch of `rung` needs for Mt tokens;
// false if the rung cannot run the shape.
bool launch_needs(int rung, int Mt, int N, int K, const DeviceInfo &dev, size_t *bytes,
                  int *counters, int epi) {
    if (is_tc(rung)) {
        TcPlan p = plan_tc(Mt, N, K, split_rule(rung), dev, epi);
        *bytes = p.ws_bytes;
        *counters = p.S > 1 ? p.n_tiles : 0;
        return p.ok;
    }
    if (is_mma(rung)) {
        MmaPlan p = plan_mma(Mt, N, K, split_rule(rung), dev, epi);
        *bytes = p.ws_bytes;
        *counters = p.reduce ? p.n_blocks : 0;
        return p.ok;
    }
    GemvPlan p = plan_gemv(Mt, N, K, split_rule(rung), dev);
    *bytes = p.ws_bytes;
    *counters = p.S > 1 ? p.n_row_blocks : 0;
    return p.ok;
}

size_t workspace_for(int rung, int M, int N, int K, const DeviceInfo &dev, int *status,
                     int epi = kEpiNone) {
    const int tt = tile_tokens(rung);
    size_t need = 0;
    *status = W4A16_OK;
    // every full token tile shares one plan; the last tile may be shorter
    int sizes[2] = {M < tt ? M : tt, M > tt && M % tt ? M % tt : 0};
    for (int Mt : sizes) {
        if (Mt == 0) continue;
        size_t b = 0;
        int c = 0;
        if (!launch_needs(rung, Mt, N, K, dev, &b, &c, epi)) {
            *status = W4A16_ERR_UNSUPPORTED;
            return 0;
        }
        if (b > need) need = b;
        if (c > kCounters - kMmaSchedWords) *status = W4A16_ERR_WORKSPACE;
    }
    return need;
}

int check_workspace(int rung, int M, int N, int K, const State &st, int epi = kEpiNone) {
    int status = W4A16_OK;
    size_t need = workspace_for(rung, M, N, K, st.dev, &status, epi);
    if (status) return status;
    if (need > st.ws.partial_bytes) return W4A16_ERR_WORKSPACE;
    return W4A16_OK;
}

int launch_linear(const LinearArgs &a, int rung, const State &st, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    const int tt = tile_tokens(rung);
    const int ycols = out_cols(a.N, a.epi);
    for (int m0 = 0; m0 < a.M && e == cudaSuccess; m0 += tt) {
        const int Mt = a.M - m0 < tt ? a.M - m0 : tt;
        LinearArgs t = a;
        t.x = a.x + (size_t)m0 * a.K;
        t.y = a.y + (size_t)m0 * ycols;
        if (a.residual) t.residual = a.residual + (size_t)m0 * ycols;
        t.M = Mt;
        if (is_tc(rung)) {
            TcPlan p = plan_tc(Mt, a.N, a.K, split_rule(rung), st.dev, a.epi);
            e = launch_tc(t, p, st.ws, st.ws.status, stream);
        } else if (is_mma(rung)) {
            MmaPlan p = plan_mma(Mt, a.N, a.K, split_rule(rung), st.dev, a.epi);
            e = launch_mma(t, p, st.ws, stream);
        } else {
            GemvPlan p = plan_gemv(Mt, a.N, a.K, split_rule(rung), st.dev);
            e = launch_gemv(t, p, st.ws, stream);
        }
        g_probe[rung].fetch_add(1, std::memory_order_relaxed);
        g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    if (st.log)
        fprintf(stderr, "[w4a16] linear M=%d N=%d K=%d -> %s\n", a.M, a.N, a.K, kRungNames[rung]);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int parse_rung(const char *s) {
    if (!s || !*s) return W4A16_RUNG_AUTO;
    for (int i = 0; i < W4A16_NUM_RUNGS; ++i)
        if (!strcmp(s, kRungNames[i])) return i;
    if (!strcmp(s, "auto")) return W4A16_RUNG_AUTO;
    char *end = nullptr;
    long v = strtol(s, &end, 10);
    if (end && *end == 0 && v >= 0 && v < W4A16_NUM_RUNGS) return (int)v;
    return W4A16_RUNG_AUTO;
}

int linear_impl(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                const uint32_t *zeros, int M, int N, int K, int group, uint16_t *y,
                void *stream, bool validated, int epi = kEpiNone,
                const uint16_t *residual = nullptr, int dtype = kDtypeF16) {
    if (!validated) {
        int st = check_linear(x, qweight, scales, zeros, M, N, K, group, y, epi, residual, dtype);
        if (st) return st;
    }
    const State &s = g_state;
    if (!s.initialized) return W4A16_ERR_NOT_INITIALIZED;
    Decision d = decide(M, N, K, s.dev, s.forced_rung, epi, dtype);
    if (d.status) return d.status;
    int st = check_workspace(d.rung, M, N, K, s, epi);
    if (st) return st;
    LinearArgs a{reinterpret_cast<const __half *>(x), qweight,
                 reinterpret_cast<const __half *>(scales), zeros,
                 reinterpret_cast<__half *>(y), M, N, K, epi,
                 reinterpret_cast<const __half *>(residual), dtype};
    return launch_linear(a, d.rung, s, (cudaStream_t)stream);
}

// ---- fused decode rounds ----------------------------------------------------
// A round whose linears all take the mma rungs (auto dispatch, M <= 8) runs as
// one launch of the mma kernel over the units of all its linears.  Each
// linear gets its own slices of the split-K workspace, so linears in flight
// at the same time never share partials or counters.  A linear that reads
// what an earlier one writes, writes what an earlier one reads, or writes
// what an earlier one writes waits (on per-linear completion counters) for
// the latest such linear to finish: the results are those of running the
// linears one after another.
struct FusedRound {
    bool tc = false;                  // a tcgen05 round (9..64 tokens), else warp-MMA
    std::vector<MmaLinDesc> descs;    // the warp-MMA round
    MmaRound round{};
    std::vector<TcLinDesc> tc_descs;  // the tcgen05 round
    TcRound tc_round{};
    int counters_used = 0;  // split-K counters, then the completion counters if waits exist
    const void *desc_data() const {
        return tc ? (const void *)tc_descs.data() : (const void *)descs.data();
    }
    size_t desc_bytes() const {
        return tc ? tc_descs.size() * sizeof(TcLinDesc) : descs.size() * sizeof(MmaLinDesc);
    }
    size_t done_words() const {  // completion counters a graph of this round owns
        if (tc) return tc_round.done ? tc_descs.size() + 1 : 0;
        return round.done ? descs.size() : 0;
    }
};

size_t bytes_of(int rows, int cols) { return (size_t)rows * cols * 2; }

// The latest earlier linear of a round that linear l must wait for: one whose
// output l reads (x, the residual), or whose input or output l writes over;
// -1 if none.
int round_wait_for(const w4a16_linear_desc *descs, int l, int M) {
    const w4a16_linear_desc &d = descs[l];
    const size_t dy = bytes_of(M, out_cols(d.N, d.epilogue));
    for (int j = l - 1; j >= 0; --j) {
        const w4a16_linear_desc &e = descs[j];
        const size_t ey = bytes_of(M, out_cols(e.N, e.epilogue));
        if (overlaps(e.y, ey, d.x, bytes_of(M, d.K)) ||
            (d.residual && overlaps(e.y, ey, d.residual, dy)) ||
            overlaps(e.x, bytes_of(M, e.K), d.y, dy) ||
            (e.residual && overlaps(e.residual, ey, d.y, dy)) || overlaps(e.y, ey, d.y, dy))
            return j;
    }
    return -1;
}

// A round of 9..64 tokens as one tcgen05 launch: one stream-K sequence over
// every linear's tiles and stages.
int plan_tc_fused_round(const w4a16_linear_desc *descs, int n, int M, const State &st,
                        FusedRound *fr) {
    if (M > kTcMaxTokens) return W4A16_ERR_UNSUPPORTED;
    fr->tc = true;
    fr->tc_descs.resize(n);
    std::vector<int> Ns(n), Ks(n), epis(n);
    bool waits = false;
    for (int l = 0; l < n; ++l) {
        const w4a16_linear_desc &d = descs[l];
        Ns[l] = d.N;
        Ks[l] = d.K;
        epis[l] = d.epilogue;
    }
    TcRound &r = fr->tc_round;
    size_t ws_floats = 0;
    std::vector<TcLinDesc> plan(n);
    if (!plan_tc_round(M, Ns.data(), Ks.data(), epis.data(), n, st.dev, &r, plan.data(),
                       &ws_floats))
        return W4A16_ERR_UNSUPPORTED;
    if (ws_floats * sizeof(float) > st.ws.partial_bytes) return W4A16_ERR_WORKSPACE;
    int counters = 0;
    for (int l = 0; l < n; ++l) {
        const w4a16_linear_desc &d = descs[l];
        LinearArgs a{reinterpret_cast<const __half *>(d.x), d.qweight,
                     reinterpret_cast<const __half *>(d.scales), d.zeros,
                     reinterpret_cast<__half *>(d.y), M, d.N, d.K, d.epilogue,
                     reinterpret_cast<const __half *>(d.residual), d.dtype};
        TcLinDesc &t = fr->tc_descs[l];
        cudaError_t e = tc_describe(a, r.T, &t);
        if (e != cudaSuccess) return cuda_fail(e);
        t.n_tiles = plan[l].n_tiles;
        t.spt = plan[l].spt;
        t.start = plan[l].start;
        t.counters = st.ws.counters + counters;  // one arrival counter per tile
        counters += t.n_tiles;
        t.wait_for = round_wait_for(descs, l, M);
        waits |= t.wait_for >= 0;
    }
    if (counters + (waits ? n + 1 : 0) > st.ws.n_counters - kMmaSchedWords)
        return W4A16_ERR_WORKSPACE;
    r.partials = st.ws.partials;
    r.done = waits ? st.ws.counters + counters : nullptr;
    r.bf16 = descs[0].dtype == W4A16_DTYPE_BF16;
    fr->counters_used = counters + (waits ? n + 1 : 0);
    return W4A16_OK;
}

// OK, UNSUPPORTED (the round is not eligible: launch linear by linear), or an error.
int plan_fused_round(const w4a16_linear_desc *descs, int n, int M, const State &st,
                     FusedRound *fr) {
    if (st.forced_rung != W4A16_RUNG_AUTO || n > kMaxRoundLinears) return W4A16_ERR_UNSUPPORTED;
    // one launch instantiates one 16-bit type
    for (int l = 1; l < n; ++l)
        if (descs[l].dtype != descs[0].dtype) return W4A16_ERR_UNSUPPORTED;
    if (M > kMmaMaxTokens) return plan_tc_fused_round(descs, n, M, st, fr);
    fr->descs.resize(n);
    size_t partial_floats = 0;
    int counters = 0, units = 0, smem = 0;
    bool waits = false;
    // one CTA shape for the whole launch
    std::vector<int> Ks(n), Ns(n);
    for (int l = 0; l < n; ++l) {
        Ks[l] = descs[l].K;
        Ns[l] = descs[l].N;
    }
    const int warps = mma_round_warps(M, Ks.data(), Ns.data(), n);
    for (int l = 0; l < n; ++l) {
        const w4a16_linear_desc &d = descs[l];
        // the last linears of a round come in small units: the CTAs then
        // run out of work within a small unit of each other
        MmaPlan p = plan_mma(M, d.N, d.K, l >= n - kRoundTailLinears ? 3 : 2, st.dev, d.epilogue,
                             1, warps);
        if (!p.ok) return W4A16_ERR_UNSUPPORTED;
        float *part = nullptr;
        unsigned *cnt = nullptr;
        if (p.reduce) {  // split K, or SiLU-and-mul
            part = st.ws.partials + partial_floats;
            partial_floats += (p.ws_bytes / sizeof(float) + 63) / 64 * 64;
            cnt = st.ws.counters + counters;
            counters += p.n_blocks;
        }
        // what a linear reads (x, the residual) and writes (y)
        const int wait_for = round_wait_for(descs, l, M);
        waits |= wait_for >= 0;
        LinearArgs a{reinterpret_cast<const __half *>(d.x), d.qweight,
                     reinterpret_cast<const __half *>(d.scales), d.zeros,
                     reinterpret_cast<__half *>(d.y), M, d.N, d.K, d.epilogue,
                     reinterpret_cast<const __half *>(d.residual), d.dtype};
        cudaError_t e = mma_describe(a, p, part, cnt, units, wait_for, &fr->descs[l]);
        if (e != cudaSuccess) return cuda_fail(e);
        units += p.units;
        if (p.smem_bytes > smem) smem = p.smem_bytes;
    }
    if (partial_floats * sizeof(float) > st.ws.partial_bytes) return W4A16_ERR_WORKSPACE;
    if (counters + (waits ? n : 0) > st.ws.n_counters - kMmaSchedWords) return W4A16_ERR_WORKSPACE;
    fr->round.n = n;
    fr->round.total_units = units;
    fr->round.smem_bytes = smem;
    fr->round.done = waits ? st.ws.counters + counters : nullptr;
    fr->round.bf16 = descs[0].dtype == W4A16_DTYPE_BF16;
    fr->round.warps = warps;
    fr->counters_used = counters + (waits ? n : 0);
    return W4A16_OK;
}

void count_fused_probes(const FusedRound &fr) {
    if (fr.tc) {
        // every linear of a tcgen05 round is a part of one stream-K sequence
        g_probe[W4A16_RUNG_TC_SPLITK].fetch_add(fr.tc_descs.size(), std::memory_order_relaxed);
        return;
    }
    for (const MmaLinDesc &d : fr.descs)
        g_probe[d.S > 1 ? W4A16_RUNG_MMA_SPLITK : W4A16_RUNG_MMA].fetch_add(
            1, std::memory_order_relaxed);
}

cudaError_t launch_fused(FusedRound &fr, const void *descs_dev, unsigned *done_dev,
                         const State &s, cudaStream_t stream) {
    if (fr.tc) {
        fr.tc_round.descs = (const TcLinDesc *)descs_dev;
        if (done_dev && fr.tc_round.done) fr.tc_round.done = done_dev;
        return launch_tc_round(fr.tc_round, s.ws.status, stream);
    }
    fr.round.descs = (const MmaLinDesc *)descs_dev;
    if (done_dev && fr.round.done) fr.round.done = done_dev;
    return launch_mma_round(fr.round, s.ws, s.dev, stream);
}

int validate_round(const w4a16_linear_desc *descs, int n_descs, int M) {
    if (!descs || n_descs < 1) return W4A16_ERR_INVALID_ARG;
    for (int i = 0; i < n_descs; ++i) {
        const w4a16_linear_desc &d = descs[i];
        int st = check_linear(d.x, d.qweight, d.scales, d.zeros, M, d.N, d.K, d.group, d.y,
                              d.epilogue, d.residual, d.dtype);
        if (st) return st;
    }
    if (!g_state.initialized) return W4A16_ERR_NOT_INITIALIZED;
    return W4A16_OK;
}

// Linear by linear (rounds the fused kernel does not take).
int round_per_linear(const w4a16_linear_desc *descs, int n_descs, int M, void *stream) {
    for (int i = 0; i < n_descs; ++i) {
        const w4a16_linear_desc &d = descs[i];
        Decision dec = decide(M, d.N, d.K, g_state.dev, g_state.forced_rung, d.epilogue, d.dtype);
        if (dec.status) return dec.status;
        int st = check_workspace(dec.rung, M, d.N, d.K, g_state, d.epilogue);
        if (st) return st;
    }
    for (int i = 0; i < n_descs; ++i) {
        const w4a16_linear_desc &d = descs[i];
        int st = linear_impl(d.x, d.qweight, d.scales, d.zeros, M, d.N, d.K, d.group, d.y, stream,
                             true, d.epilogue, d.residual, d.dtype);
        if (st) return st;
    }
    return W4A16_OK;
}

// A mixture-of-experts layer: the experts' descriptor templates (tensor maps
// written once here), room for the tile descriptors a call's prepare kernel
// writes, and the gathered activations.
struct MoeHandle {
    int E, N, K, epi, dtype, max_slots, max_tiles;
    MmaPlan plan;             // every tile's plan (M = 8 for the shared-memory budget)
    MmaLinDesc *tmpl = nullptr;   // device [E]
    MmaLinDesc *tiles = nullptr;  // device [max_tiles]
    int *counts = nullptr;        // device [2]: tiles, units
    __half *xs = nullptr;         // device [max_slots, K]
    const uint32_t *qweight = nullptr;  // the experts, as given
    const __half *scales = nullptr;
    const uint32_t *zeros = nullptr;
    void *buffer = nullptr;
};

// An expert MLP: gate+up and down expert layers and the per-call buffers of
// their chain (alignment, the intermediate and output rows in sorted order,
// both linears' tile descriptors, their completion counters).
struct MoeMlpHandle {
    MoeHandle *gu = nullptr, *dn = nullptr;
    int max_tokens = 0, k = 0, max_slots = 0, max_tiles = 0;
    int32_t *sorted = nullptr, *pos = nullptr, *offsets = nullptr;
    __half *h = nullptr, *o = nullptr;
    MmaLinDesc *tiles = nullptr;
    unsigned *done = nullptr;
    int *counts = nullptr;
    // the one-launch decode kernel (gate+up with SiLU-and-mul, whole groups)
    bool dec_ok = false;
    MoeDecodeWeights dec{};
    unsigned *dec_counters = nullptr;
    int path = W4A16_MOE_PATH_AUTO;
    void *buffer = nullptr;
};

// The path of an expert-MLP call with T tokens; -1 when the forced decode
// path cannot take it.
int mlp_path(const MoeMlpHandle *m, int T) {
    const bool dec = m->dec_ok && moe_decode_smem(m->dec, T, m->k) >= 0;
    if (m->path == W4A16_MOE_PATH_CHAIN) return W4A16_MOE_PATH_CHAIN;
    if (m->path == W4A16_MOE_PATH_DECODE) return dec ? W4A16_MOE_PATH_DECODE : -1;
    return dec ? W4A16_MOE_PATH_DECODE : W4A16_MOE_PATH_CHAIN;
}

struct RoundGraphHandle {
    cudaGraphExec_t exec = nullptr;
    void *buffer = nullptr;  // the fused round's descriptors and completion counters
};

}  // namespace

namespace w4a16 {
int check_linear_args(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                      const uint32_t *zeros, int M, int N, int K, int group, const uint16_t *y,
                      int epi, const uint16_t *residual, int dtype) {
    return check_linear(x, qweight, scales, zeros, M, N, K, group, y, epi, residual, dtype);
}

void count_launches(int rung, unsigned long long linears, unsigned long long kernels) {
    if (rung >= 0 && rung < W4A16_NUM_RUNGS)
        g_probe[rung].fetch_add(linears, std::memory_order_relaxed);
    g_launches.fetch_add(kernels, std::memory_order_relaxed);
}
}  // namespace w4a16

extern "C" {

int w4a16_init(int device, size_t workspace_bytes) {
    std::lock_guard<std::mutex> lock(g_mutex);
    State &s = g_state;
    if (s.initialized) {
        cudaDeviceSynchronize();
        cudaFree(s.ws_base);
        s = State{};
    }
    cudaError_t e = cudaSetDevice(device);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceInfo dev{};
    dev.device = device;
    e = cudaDeviceGetAttribute(&dev.sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&dev.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                   device);
    if (e != cudaSuccess) return cuda_fail(e);
    if (workspace_bytes == 0) workspace_bytes = kDefaultWorkspace;
    workspace_bytes = (workspace_bytes + 255) & ~(size_t)255;
    // counters, then one status word (kept 256-byte aligned), then the fused
    // round descriptors
    const size_t counter_bytes = (size_t)kCounters * sizeof(unsigned) + 256;
    const size_t desc_bytes =
        (size_t)kMaxRoundLinears *
        (sizeof(MmaLinDesc) > sizeof(TcLinDesc) ? sizeof(MmaLinDesc) : sizeof(TcLinDesc));
    void *base = nullptr;
    e = cudaMalloc(&base, workspace_bytes + counter_bytes + desc_bytes);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemset((char *)base + workspace_bytes, 0, counter_bytes);
    if (e == cudaSuccess) e = gemv_init_attributes(dev);
    if (e == cudaSuccess) e = tc_init(dev);
    if (e == cudaSuccess) e = mma_init(dev);
    if (e == cudaSuccess) e = dense_init(dev);
    if (e == cudaSuccess) e = moe_decode_init(dev);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(base);
        return cuda_fail(e);
    }
    s.dev = dev;
    s.ws_base = base;
    s.ws.partials = (float *)base;
    s.ws.partial_bytes = workspace_bytes;
    s.ws.counters = (unsigned *)((char *)base + workspace_bytes);
    s.ws.n_counters = kCounters;
    s.ws.status = (int *)((char *)base + workspace_bytes + (size_t)kCounters * sizeof(unsigned));
    s.round_descs = (char *)base + workspace_bytes + counter_bytes;
    s.round_uploaded.clear();
    s.forced_rung = parse_rung(getenv("W4A16_FORCE_RUNG"));
    const char *lg = getenv("W4A16_LOG");
    s.log = lg && *lg && strcmp(lg, "0") != 0;
    s.initialized = true;
    return W4A16_OK;
}

int w4a16_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mutex);
    State &s = g_state;
    if (!s.initialized) return W4A16_OK;
    cudaError_t e = cudaDeviceSynchronize();
    cudaError_t f = cudaFree(s.ws_base);
    s = State{};
    if (e != cudaSuccess) return cuda_fail(e);
    if (f != cudaSuccess) return cuda_fail(f);
    return W4A16_OK;
}

size_t w4a16_workspace_bytes(int M, int N, int K, int group) {
    if (M < 1 || M > kMaxM || check_shape(N, K, group)) return 0;
    DeviceInfo dev = g_state.dev;
    if (!g_state.initialized) dev.sm_count = 152;
    Decision d = decide(M, N, K, dev, g_state.forced_rung);
    if (d.status) return 0;
    int status = W4A16_OK;
    size_t need = workspace_for(d.rung, M, N, K, dev, &status);
    return status == W4A16_ERR_UNSUPPORTED ? 0 : need;
}

int w4a16_pack(const uint8_t *q, const uint8_t *z, int N, int K, int group, uint32_t *qweight,
               uint32_t *zeros, void *stream) {
    if (!q || !z || !qweight || !zeros) return W4A16_ERR_INVALID_ARG;
    int st = check_shape(N, K, group);
    if (st) return st;
    if (!aligned(q, 16) || !aligned(qweight, 16) || !aligned(z, 4) || !aligned(zeros, 4))
        return W4A16_ERR_MISALIGNED;
    cudaError_t e = launch_pack(q, z, N, K, qweight, zeros, (cudaStream_t)stream);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_unpack(const uint32_t *qweight, const uint32_t *zeros, int N, int K, int group,
                 uint8_t *q, uint8_t *z, void *stream) {
    if (!q || !z || !qweight || !zeros) return W4A16_ERR_INVALID_ARG;
    int st = check_shape(N, K, group);
    if (st) return st;
    if (!aligned(q, 16) || !aligned(qweight, 16) || !aligned(z, 4) || !aligned(zeros, 4))
        return W4A16_ERR_MISALIGNED;
    cudaError_t e = launch_unpack(qweight, zeros, N, K, q, z, (cudaStream_t)stream);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_dequant(const uint32_t *qweight, const uint16_t *scales, const uint32_t *zeros, int N,
                  int K, int group, float *w_f32, uint16_t *w_f16, void *stream) {
    if (!qweight || !scales || !zeros || (!w_f32 && !w_f16)) return W4A16_ERR_INVALID_ARG;
    int st = check_shape(N, K, group);
    if (st) return st;
    if (!aligned(qweight, 16) || !aligned(scales, 2) || !aligned(zeros, 4) ||
        (w_f32 && !aligned(w_f32, 16)) || (w_f16 && !aligned(w_f16, 16)))
        return W4A16_ERR_MISALIGNED;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = launch_dequant(qweight, reinterpret_cast<const __half *>(scales), zeros, N, K,
                                   w_f32, reinterpret_cast<__half *>(w_f16), (cudaStream_t)stream);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_repack_transpose(const uint32_t *src, int rows, int cols, uint32_t src_order,
                           uint32_t *dst, void *stream) {
    if (!src || !dst || rows < 1 || cols < 8 || cols % 8 != 0 || rows > kMaxRepackDim ||
        cols > kMaxRepackDim)
        return W4A16_ERR_INVALID_ARG;
    // the order must name each of the 8 nibble positions once
    unsigned seen = 0;
    for (int j = 0; j < 8; ++j) seen |= 1u << ((src_order >> (4 * j)) & 0xfu);
    if (seen != 0xffu) return W4A16_ERR_INVALID_ARG;
    if (!aligned(src, 4) || !aligned(dst, 4)) return W4A16_ERR_MISALIGNED;
    if (overlaps(src, (size_t)rows * (cols / 8) * 4, dst, (size_t)cols * ((rows + 7) / 8) * 4))
        return W4A16_ERR_INVALID_ARG;
    cudaError_t e = launch_transpose_u4(src, rows, cols, src_order, dst, (cudaStream_t)stream);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_transpose_f16(const uint16_t *src, int rows, int cols, uint16_t *dst, void *stream) {
    if (!src || !dst || rows < 1 || cols < 1 || rows > kMaxRepackDim || cols > kMaxRepackDim)
        return W4A16_ERR_INVALID_ARG;
    if (!aligned(src, 2) || !aligned(dst, 2)) return W4A16_ERR_MISALIGNED;
    if (overlaps(src, (size_t)rows * cols * 2, dst, (size_t)rows * cols * 2))
        return W4A16_ERR_INVALID_ARG;
    cudaError_t e = launch_transpose_u16(src, rows, cols, dst, (cudaStream_t)stream);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_dense_linear(const uint16_t *x, const uint16_t *w, int M, int N, int K, int dtype,
                       uint16_t *y, void *stream) {
    if (!x || !w || !y || M < 1 || M > kMaxM || N < 1 || K < kGroup || K > kMaxK ||
        K % kGroup != 0)
        return W4A16_ERR_INVALID_ARG;
    if (dtype != W4A16_DTYPE_F16 && dtype != W4A16_DTYPE_BF16) return W4A16_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16)) return W4A16_ERR_MISALIGNED;
    const size_t ybytes = (size_t)M * N * 2;
    if (overlaps(x, (size_t)M * K * 2, y, ybytes) || overlaps(w, (size_t)N * K * 2, y, ybytes))
        return W4A16_ERR_INVALID_ARG;
    const State &st = g_state;
    if (!st.initialized) return W4A16_ERR_NOT_INITIALIZED;
    // tiles of up to 8 tokens, each streaming the weights once
    for (int m0 = 0; m0 < M; m0 += kMmaMaxTokens) {
        const int Mt = M - m0 < kMmaMaxTokens ? M - m0 : kMmaMaxTokens;
        DensePlan p = plan_dense(Mt, N, K, st.dev);
        if (!p.ok) return W4A16_ERR_UNSUPPORTED;
        if (p.ws_bytes > st.ws.partial_bytes ||
            (p.S > 1 && p.n_blocks > st.ws.n_counters - kMmaSchedWords))
            return W4A16_ERR_WORKSPACE;
    }
    cudaError_t e = cudaSuccess;
    for (int m0 = 0; m0 < M && e == cudaSuccess; m0 += kMmaMaxTokens) {
        const int Mt = M - m0 < kMmaMaxTokens ? M - m0 : kMmaMaxTokens;
        DensePlan p = plan_dense(Mt, N, K, st.dev);
        e = launch_dense(reinterpret_cast<const __half *>(x) + (size_t)m0 * K,
                         reinterpret_cast<const __half *>(w),
                         reinterpret_cast<__half *>(y) + (size_t)m0 * N, Mt, N, K,
                         dtype == W4A16_DTYPE_BF16, p, st.ws, (cudaStream_t)stream);
        g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    if (st.log)
        fprintf(stderr, "[w4a16] dense linear M=%d N=%d K=%d dtype=%d\n", M, N, K, dtype);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_moe_create(int E, int N, int K, int group, const uint32_t *qweight,
                     const uint16_t *scales, const uint32_t *zeros, int epilogue, int dtype,
                     int max_slots, void **moe) {
    if (!moe) return W4A16_ERR_INVALID_ARG;
    *moe = nullptr;
    if (!qweight || !scales || !zeros || E < 1 || E > kMaxMoeExperts || max_slots < 1)
        return W4A16_ERR_INVALID_ARG;
    int st = check_shape(N, K, group);
    if (st) return st;
    if (dtype != W4A16_DTYPE_F16 && dtype != W4A16_DTYPE_BF16) return W4A16_ERR_INVALID_ARG;
    if (epilogue != W4A16_EPILOGUE_NONE && epilogue != W4A16_EPILOGUE_SILU_MUL)
        return epilogue == W4A16_EPILOGUE_RESIDUAL ? W4A16_ERR_UNSUPPORTED : W4A16_ERR_INVALID_ARG;
    if (epilogue == W4A16_EPILOGUE_SILU_MUL && N % 32 != 0) return W4A16_ERR_UNSUPPORTED;
    if (!aligned(qweight, 16) || !aligned(scales, 2) || !aligned(zeros, 4))
        return W4A16_ERR_MISALIGNED;
    State &s = g_state;
    if (!s.initialized) return W4A16_ERR_NOT_INITIALIZED;
    // tiles: one per expert that gets a slot, one more per further 8 slots
    long long max_tiles = (long long)max_slots < E ? max_slots : E;
    max_tiles += max_slots / kMmaMaxTokens;
    if (max_tiles > max_slots) max_tiles = max_slots;
    if (max_tiles > kMaxMoeTiles) return W4A16_ERR_UNSUPPORTED;
    MoeHandle *h = new MoeHandle();
    h->E = E;
    h->N = N;
    h->K = K;
    h->epi = epilogue;
    h->dtype = dtype;
    h->max_slots = max_slots;
    h->max_tiles = (int)max_tiles;
    h->qweight = qweight;
    h->scales = reinterpret_cast<const __half *>(scales);
    h->zeros = zeros;
    // one plan for every tile, weighing the tiles expected side by side (one
    // per expert in use, up to the slots)
    const int copies = max_slots < E ? max_slots : E;
    // (8-warp CTAs: an expert MLP's launch holds the plans of two linears)
    h->plan = plan_mma(kMmaMaxTokens, N, K, -1, s.dev, epilogue, copies, 8);
    if (!h->plan.ok) {
        delete h;
        return W4A16_ERR_UNSUPPORTED;
    }
    const size_t part_floats = h->plan.reduce ? (size_t)h->plan.S * kMmaMaxTokens * N : 0;
    if (part_floats * max_tiles * sizeof(float) > s.ws.partial_bytes ||
        (h->plan.reduce &&
         (long long)h->plan.n_blocks * max_tiles > s.ws.n_counters - kMmaSchedWords)) {
        delete h;
        return W4A16_ERR_WORKSPACE;
    }
    const int G = K / kGroup, ZW = (G + 7) / 8;
    std::vector<MmaLinDesc> tmpl(E);
    for (int e = 0; e < E; ++e) {
        LinearArgs a{nullptr, qweight + (size_t)e * N * (K / 8),
                     reinterpret_cast<const __half *>(scales) + (size_t)e * N * G,
                     zeros + (size_t)e * N * ZW, nullptr, kMmaMaxTokens, N, K, epilogue,
                     nullptr, dtype};
        cudaError_t e2 = mma_describe(a, h->plan, nullptr, nullptr, 0, -1, &tmpl[e]);
        if (e2 != cudaSuccess) {
            delete h;
            return cuda_fail(e2);
        }
    }
    const size_t tb = sizeof(MmaLinDesc) * E, lb = sizeof(MmaLinDesc) * max_tiles;
    const size_t xb = ((size_t)max_slots * K * 2 + 255) & ~(size_t)255;
    cudaError_t e = cudaMalloc(&h->buffer, tb + lb + 256 + xb);
    if (e == cudaSuccess) {
        char *b = (char *)h->buffer;
        h->tmpl = (MmaLinDesc *)b;
        h->tiles = (MmaLinDesc *)(b + tb);
        h->counts = (int *)(b + tb + lb);
        h->xs = (__half *)(b + tb + lb + 256);
        e = cudaMemcpy(h->tmpl, tmpl.data(), tb, cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
        if (h->buffer) cudaFree(h->buffer);
        delete h;
        return cuda_fail(e);
    }
    *moe = h;
    return W4A16_OK;
}

int w4a16_moe_destroy(void *moe) {
    if (!moe) return W4A16_ERR_INVALID_ARG;
    MoeHandle *h = (MoeHandle *)moe;
    cudaError_t e = h->buffer ? cudaFree(h->buffer) : cudaSuccess;
    delete h;
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_moe_align(const int32_t *topk_ids, int n_slots, int E, int32_t *sorted, int32_t *pos,
                    int32_t *offsets, void *stream) {
    if (!topk_ids || !sorted || !pos || !offsets || n_slots < 1 || E < 1 || E > kMaxMoeExperts)
        return W4A16_ERR_INVALID_ARG;
    if (!aligned(topk_ids, 4) || !aligned(sorted, 4) || !aligned(pos, 4) || !aligned(offsets, 4))
        return W4A16_ERR_MISALIGNED;
    if (!g_state.initialized) return W4A16_ERR_NOT_INITIALIZED;
    cudaError_t e = launch_moe_align(topk_ids, n_slots, E, sorted, pos, offsets, g_state.ws.status,
                                     (cudaStream_t)stream);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_moe_linear(void *moe, const uint16_t *x, int gather_k, const int32_t *sorted,
                     const int32_t *offsets, int n_slots, uint16_t *y, void *stream) {
    if (!moe || !x || !sorted || !offsets || !y || n_slots < 1 || gather_k < 0)
        return W4A16_ERR_INVALID_ARG;
    MoeHandle *h = (MoeHandle *)moe;
    if (n_slots > h->max_slots || (gather_k > 0 && n_slots % gather_k != 0))
        return W4A16_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16)) return W4A16_ERR_MISALIGNED;
    const State &st = g_state;
    if (!st.initialized) return W4A16_ERR_NOT_INITIALIZED;
    const int ycols = out_cols(h->N, h->epi);
    const size_t xrows = gather_k > 0 ? (size_t)(n_slots / gather_k) : (size_t)n_slots;
    if (overlaps(x, xrows * h->K * 2, y, (size_t)n_slots * ycols * 2)) return W4A16_ERR_INVALID_ARG;
    MoeTileSpace sp{};
    sp.y = reinterpret_cast<__half *>(y);
    if (h->plan.reduce) {
        sp.partials = st.ws.partials;
        sp.partial_stride = (size_t)h->plan.S * kMmaMaxTokens * h->N;
        sp.counters = st.ws.counters;
        sp.counter_stride = (size_t)h->plan.n_blocks;
    }
    cudaStream_t cs = (cudaStream_t)stream;
    cudaError_t e = launch_moe_prepare(h->tmpl, nullptr, offsets, sorted, h->E,
                                       gather_k > 0 ? gather_k : 1, h->max_tiles, h->plan.units, 0,
                                       sp, MoeTileSpace{}, reinterpret_cast<const __half *>(x),
                                       gather_k > 0, h->xs, n_slots, h->K, h->tiles, h->counts,
                                       cs);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (e != cudaSuccess) return cuda_fail(e);
    MmaRound r{};
    r.descs = h->tiles;
    r.n = h->max_tiles;
    r.total_units = h->max_tiles * h->plan.units;
    r.smem_bytes = h->plan.smem_bytes;
    r.done = nullptr;
    r.bf16 = h->dtype == W4A16_DTYPE_BF16;
    r.counts = h->counts;
    e = launch_mma_round(r, st.ws, st.dev, cs);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    g_probe[h->plan.S > 1 ? W4A16_RUNG_MMA_SPLITK : W4A16_RUNG_MMA].fetch_add(
        1, std::memory_order_relaxed);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_moe_mlp_create(void *gate_up, void *down, int max_tokens, int k, void **mlp) {
    if (!mlp) return W4A16_ERR_INVALID_ARG;
    *mlp = nullptr;
    if (!gate_up || !down || max_tokens < 1 || k < 1) return W4A16_ERR_INVALID_ARG;
    MoeHandle *gu = (MoeHandle *)gate_up, *dn = (MoeHandle *)down;
    // down reads what gate+up writes, and gives back rows of gate+up's input width
    if (gu->E != dn->E || gu->dtype != dn->dtype || dn->K != out_cols(gu->N, gu->epi) ||
        dn->epi != W4A16_EPILOGUE_NONE || dn->N != gu->K)
        return W4A16_ERR_INVALID_ARG;
    const long long slots = (long long)max_tokens * k;
    if (slots > gu->max_slots || slots > dn->max_slots) return W4A16_ERR_INVALID_ARG;
    const State &st = g_state;
    if (!st.initialized) return W4A16_ERR_NOT_INITIALIZED;
    // both linears' split-K spaces side by side in the workspace
    const size_t part_a = gu->plan.reduce ? (size_t)gu->plan.S * kMmaMaxTokens * gu->N : 0;
    const size_t part_b = dn->plan.reduce ? (size_t)dn->plan.S * kMmaMaxTokens * dn->N : 0;
    const int tiles = gu->max_tiles;
    const long long cnt_a = gu->plan.reduce ? (long long)gu->plan.n_blocks * tiles : 0;
    const long long cnt_b = dn->plan.reduce ? (long long)dn->plan.n_blocks * tiles : 0;
    if ((part_a + part_b) * tiles * sizeof(float) > st.ws.partial_bytes ||
        cnt_a + cnt_b > st.ws.n_counters - kMmaSchedWords)
        return W4A16_ERR_WORKSPACE;
    MoeMlpHandle *m = new MoeMlpHandle();
    m->gu = gu;
    m->dn = dn;
    m->max_tokens = max_tokens;
    m->k = k;
    m->max_slots = (int)slots;
    m->max_tiles = tiles;
    const size_t al = 256;
    auto up = [&](size_t b) { return (b + al - 1) / al * al; };
    const size_t b_sorted = up(slots * 4), b_pos = up(slots * 4), b_off = up((gu->E + 1) * 4);
    const size_t b_h = up(slots * dn->K * 2), b_o = up(slots * dn->N * 2);
    const size_t b_tiles = up(sizeof(MmaLinDesc) * 2 * tiles), b_done = up(2 * tiles * 4);
    // the decode kernel: gate+up rows [gate; up] with SiLU-and-mul over whole
    // groups and 128-row blocks of down
    if (gu->epi == W4A16_EPILOGUE_SILU_MUL && moe_decode_shape_ok(gu->E, gu->K, dn->K)) {
        cudaError_t e0 = moe_decode_describe(gu->qweight, gu->scales, gu->zeros, dn->qweight,
                                             dn->scales, dn->zeros, gu->E, gu->K, dn->K,
                                             gu->dtype == W4A16_DTYPE_BF16, &m->dec);
        m->dec_ok = e0 == cudaSuccess;
    }
    const size_t b_dec = m->dec_ok ? up(moe_decode_counter_words(m->dec) * 4) : 0;
    const size_t total = b_sorted + b_pos + b_off + b_h + b_o + b_tiles + b_done + b_dec + al;
    cudaError_t e = cudaMalloc(&m->buffer, total);
    if (e == cudaSuccess) {
        char *b = (char *)m->buffer;
        m->sorted = (int32_t *)b;
        b += b_sorted;
        m->pos = (int32_t *)b;
        b += b_pos;
        m->offsets = (int32_t *)b;
        b += b_off;
        m->h = (__half *)b;
        b += b_h;
        m->o = (__half *)b;
        b += b_o;
        m->tiles = (MmaLinDesc *)b;
        b += b_tiles;
        m->done = (unsigned *)b;
        b += b_done;
        m->counts = (int *)b;
        b += al;
        m->dec_counters = m->dec_ok ? (unsigned *)b : nullptr;
        e = cudaMemset(m->done, 0, b_done);  // the kernel leaves them zeroed again
        if (e == cudaSuccess && m->dec_ok) e = cudaMemset(m->dec_counters, 0, b_dec);
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        if (m->buffer) cudaFree(m->buffer);
        delete m;
        return cuda_fail(e);
    }
    *mlp = m;
    return W4A16_OK;
}

int w4a16_moe_mlp_destroy(void *mlp) {
    if (!mlp) return W4A16_ERR_INVALID_ARG;
    MoeMlpHandle *m = (MoeMlpHandle *)mlp;
    cudaError_t e = m->buffer ? cudaFree(m->buffer) : cudaSuccess;
    delete m;
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_moe_mlp_set_path(void *mlp, int path) {
    if (!mlp || path < W4A16_MOE_PATH_AUTO || path > W4A16_MOE_PATH_DECODE)
        return W4A16_ERR_INVALID_ARG;
    ((MoeMlpHandle *)mlp)->path = path;
    return W4A16_OK;
}

int w4a16_moe_mlp_path(void *mlp, int T, int *path) {
    if (!mlp || !path || T < 1) return W4A16_ERR_INVALID_ARG;
    const MoeMlpHandle *m = (const MoeMlpHandle *)mlp;
    if (T > m->max_tokens) return W4A16_ERR_INVALID_ARG;
    const int p = mlp_path(m, T);
    if (p < 0) return W4A16_ERR_UNSUPPORTED;
    *path = p;
    return W4A16_OK;
}

int w4a16_moe_mlp_buffers(void *mlp, uint16_t **h, uint16_t **o) {
    if (!mlp || !h || !o) return W4A16_ERR_INVALID_ARG;
    const MoeMlpHandle *m = (const MoeMlpHandle *)mlp;
    *h = reinterpret_cast<uint16_t *>(m->h);
    *o = reinterpret_cast<uint16_t *>(m->o);
    return W4A16_OK;
}

int w4a16_moe_mlp(void *mlp, const uint16_t *x, const int32_t *topk_ids, const float *weights,
                  int T, uint16_t *out, void *stream) {
    if (!mlp || !x || !topk_ids || !weights || !out || T < 1) return W4A16_ERR_INVALID_ARG;
    MoeMlpHandle *m = (MoeMlpHandle *)mlp;
    if (T > m->max_tokens) return W4A16_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(out, 2) || !aligned(topk_ids, 4) || !aligned(weights, 4))
        return W4A16_ERR_MISALIGNED;
    MoeHandle *gu = m->gu, *dn = m->dn;
    if (overlaps(x, (size_t)T * gu->K * 2, out, (size_t)T * dn->N * 2)) return W4A16_ERR_INVALID_ARG;
    const State &st = g_state;
    if (!st.initialized) return W4A16_ERR_NOT_INITIALIZED;
    const int path = mlp_path(m, T);
    if (path < 0) return W4A16_ERR_UNSUPPORTED;
    cudaStream_t cs = (cudaStream_t)stream;
    if (path == W4A16_MOE_PATH_DECODE) {
        const MoeDecodeBuffers b{m->h, m->o, m->dec_counters};
        cudaError_t e = launch_moe_decode(m->dec, reinterpret_cast<const __half *>(x), topk_ids,
                                          weights, T, m->k, reinterpret_cast<__half *>(out), b,
                                          st.ws.status, st.dev, cs);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
    }
    const int n_slots = T * m->k;
    cudaError_t e = launch_moe_align(topk_ids, n_slots, gu->E, m->sorted, m->pos, m->offsets,
                                     st.ws.status, cs);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (e != cudaSuccess) return cuda_fail(e);
    MoeTileSpace sa{}, sb{};
    sa.y = m->h;
    sb.y = m->o;
    size_t part_off = 0, cnt_off = 0;
    if (gu->plan.reduce) {
        sa.partials = st.ws.partials;
        sa.partial_stride = (size_t)gu->plan.S * kMmaMaxTokens * gu->N;
        sa.counters = st.ws.counters;
        sa.counter_stride = (size_t)gu->plan.n_blocks;
        part_off = sa.partial_stride * m->max_tiles;
        cnt_off = sa.counter_stride * m->max_tiles;
    }
    if (dn->plan.reduce) {
        sb.partials = st.ws.partials + part_off;
        sb.partial_stride = (size_t)dn->plan.S * kMmaMaxTokens * dn->N;
        sb.counters = st.ws.counters + cnt_off;
        sb.counter_stride = (size_t)dn->plan.n_blocks;
    }
    e = launch_moe_prepare(gu->tmpl, dn->tmpl, m->offsets, m->sorted, gu->E, m->k, m->max_tiles,
                           gu->plan.units, dn->plan.units, sa, sb,
                           reinterpret_cast<const __half *>(x), true, gu->xs, n_slots, gu->K,
                           m->tiles, m->counts, cs);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (e != cudaSuccess) return cuda_fail(e);
    // both linears in one launch: tile t of down waits for tile t of gate+up
    MmaRound r{};
    r.descs = m->tiles;
    r.n = 2 * m->max_tiles;
    r.total_units = m->max_tiles * (gu->plan.units + dn->plan.units);
    r.smem_bytes = gu->plan.smem_bytes > dn->plan.smem_bytes ? gu->plan.smem_bytes
                                                             : dn->plan.smem_bytes;
    r.done = m->done;
    r.bf16 = gu->dtype == W4A16_DTYPE_BF16;
    r.counts = m->counts;
    e = launch_mma_round(r, st.ws, st.dev, cs);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_moe_sum(m->o, m->pos, weights, T, m->k, dn->N, gu->dtype == W4A16_DTYPE_BF16,
                       reinterpret_cast<__half *>(out), cs);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_moe_sum(const uint16_t *y_sorted, const int32_t *pos, const float *weights, int T,
                  int k, int N, int dtype, uint16_t *out, void *stream) {
    if (!y_sorted || !pos || !weights || !out || T < 1 || k < 1 || N < 1)
        return W4A16_ERR_INVALID_ARG;
    if (dtype != W4A16_DTYPE_F16 && dtype != W4A16_DTYPE_BF16) return W4A16_ERR_INVALID_ARG;
    if (!aligned(y_sorted, 2) || !aligned(out, 2) || !aligned(pos, 4) || !aligned(weights, 4))
        return W4A16_ERR_MISALIGNED;
    if (overlaps(y_sorted, (size_t)T * k * N * 2, out, (size_t)T * N * 2))
        return W4A16_ERR_INVALID_ARG;
    cudaError_t e = launch_moe_sum(reinterpret_cast<const __half *>(y_sorted), pos, weights, T, k,
                                   N, dtype == W4A16_DTYPE_BF16, reinterpret_cast<__half *>(out),
                                   (cudaStream_t)stream);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_linear(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                 const uint32_t *zeros, int M, int N, int K, int group, uint16_t *y,
                 void *stream) {
    return linear_impl(x, qweight, scales, zeros, M, N, K, group, y, stream, false);
}

int w4a16_linear_epilogue(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                          const uint32_t *zeros, int M, int N, int K, int group, int epilogue,
                          const uint16_t *residual, uint16_t *y, void *stream) {
    return linear_impl(x, qweight, scales, zeros, M, N, K, group, y, stream, false, epilogue,
                       residual);
}

int w4a16_linear_ex(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                    const uint32_t *zeros, int M, int N, int K, int group, int dtype,
                    int epilogue, const uint16_t *residual, uint16_t *y, void *stream) {
    return linear_impl(x, qweight, scales, zeros, M, N, K, group, y, stream, false, epilogue,
                       residual, dtype);
}

int w4a16_decode_round(const w4a16_linear_desc *descs, int n_descs, int M, void *stream) {
    int st = validate_round(descs, n_descs, M);
    if (st) return st;
    State &s = g_state;
    // A graph captured from this call would keep pointing at the shared
    // descriptor copy that later rounds overwrite: under capture, launch linear
    // by linear (w4a16_round_graph_create captures a fused round with its own
    // descriptors).
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing((cudaStream_t)stream, &cap);
    if (ce != cudaSuccess) return cuda_fail(ce);
    if (cap != cudaStreamCaptureStatusNone) return round_per_linear(descs, n_descs, M, stream);
    FusedRound fr;
    st = plan_fused_round(descs, n_descs, M, s, &fr);
    if (st == W4A16_ERR_UNSUPPORTED) return round_per_linear(descs, n_descs, M, stream);
    if (st) return st;
    // upload the descriptors unless the device copy already holds these
    // (the copy is ordered on the stream after earlier rounds that read it)
    const size_t bytes = fr.desc_bytes();
    const unsigned char *src = (const unsigned char *)fr.desc_data();
    if (s.round_uploaded.size() != bytes || memcmp(s.round_uploaded.data(), src, bytes) != 0) {
        cudaError_t e = cudaMemcpyAsync(s.round_descs, src, bytes, cudaMemcpyHostToDevice,
                                        (cudaStream_t)stream);
        if (e != cudaSuccess) {
            s.round_uploaded.clear();
            return cuda_fail(e);
        }
        s.round_uploaded.assign(src, src + bytes);
    }
    cudaError_t e = launch_fused(fr, s.round_descs, nullptr, s, (cudaStream_t)stream);
    count_fused_probes(fr);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (s.log)
        fprintf(stderr, "[w4a16] decode round of %d linears M=%d -> fused %s%s\n", n_descs, M,
                fr.tc ? "tcgen05" : "mma",
                (fr.tc ? fr.tc_round.done != nullptr : fr.round.done != nullptr) ? ", with waits"
                                                                                  : "");
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_round_graph_create(const w4a16_linear_desc *descs, int n_descs, int M, void **graph) {
    if (!graph) return W4A16_ERR_INVALID_ARG;
    *graph = nullptr;
    int st = validate_round(descs, n_descs, M);
    if (st) return st;
    State &s = g_state;
    FusedRound fr;
    st = plan_fused_round(descs, n_descs, M, s, &fr);
    const bool fused = st == W4A16_OK;
    if (st && st != W4A16_ERR_UNSUPPORTED) return st;
    RoundGraphHandle *hd = new RoundGraphHandle();
    cudaError_t e = cudaSuccess;
    void *graph_descs = nullptr;
    unsigned *graph_done = nullptr;
    if (fused) {
        // the graph owns its descriptors and completion counters
        const size_t dbytes = (fr.desc_bytes() + 255) & ~(size_t)255;
        const size_t cbytes = fr.done_words() * sizeof(unsigned);
        e = cudaMalloc(&hd->buffer, dbytes + cbytes);
        if (e == cudaSuccess)
            e = cudaMemcpy(hd->buffer, fr.desc_data(), fr.desc_bytes(), cudaMemcpyHostToDevice);
        if (e == cudaSuccess && cbytes) e = cudaMemset((char *)hd->buffer + dbytes, 0, cbytes);
        graph_descs = hd->buffer;
        graph_done = cbytes ? (unsigned *)((char *)hd->buffer + dbytes) : nullptr;
    }
    cudaStream_t cs = nullptr;
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        if (cs) cudaStreamDestroy(cs);
        if (hd->buffer) cudaFree(hd->buffer);
        delete hd;
        return cuda_fail(e);
    }
    if (fused) {
        cudaError_t le = launch_fused(fr, graph_descs, graph_done, s, cs);
        st = le == cudaSuccess ? W4A16_OK : cuda_fail(le);
        if (!st) count_fused_probes(fr);
    } else {
        st = round_per_linear(descs, n_descs, M, cs);
    }
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (!st && e != cudaSuccess) st = cuda_fail(e);
    if (!st) {
        e = cudaGraphInstantiate(&hd->exec, g, 0);
        if (e != cudaSuccess) st = cuda_fail(e);
    }
    if (g) cudaGraphDestroy(g);
    if (st) {
        if (hd->buffer) cudaFree(hd->buffer);
        delete hd;
        return st;
    }
    *graph = (void *)hd;
    return W4A16_OK;
}

int w4a16_round_graph_launch(void *graph, void *stream) {
    if (!graph) return W4A16_ERR_INVALID_ARG;
    RoundGraphHandle *hd = (RoundGraphHandle *)graph;
    cudaError_t e = cudaGraphLaunch(hd->exec, (cudaStream_t)stream);
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_round_graph_destroy(void *graph) {
    if (!graph) return W4A16_ERR_INVALID_ARG;
    RoundGraphHandle *hd = (RoundGraphHandle *)graph;
    cudaError_t e = cudaGraphExecDestroy(hd->exec);
    cudaError_t f = hd->buffer ? cudaFree(hd->buffer) : cudaSuccess;
    delete hd;
    if (e != cudaSuccess) return cuda_fail(e);
    return f == cudaSuccess ? W4A16_OK : cuda_fail(f);
}

int w4a16_select_rung(int M, int N, int K, int group) {
    if (M < 1 || M > kMaxM || check_shape(N, K, group)) return -1;
    DeviceInfo dev = g_state.dev;
    if (!g_state.initialized) dev.sm_count = 152;
    Decision d = decide(M, N, K, dev, g_state.forced_rung);
    return d.status ? -1 : d.rung;
}

int w4a16_plan_info(int M, int N, int K, int group, int epilogue, int dtype, int32_t *info) {
    if (!info || M < 1 || M > kMaxM || check_shape(N, K, group)) return W4A16_ERR_INVALID_ARG;
    if (epilogue < kEpiNone || epilogue > kEpiSiluMul || (dtype != kDtypeF16 && dtype != kDtypeBf16))
        return W4A16_ERR_INVALID_ARG;
    if (epilogue == kEpiSiluMul && N % 32 != 0) return W4A16_ERR_INVALID_ARG;
    DeviceInfo dev = g_state.dev;
    if (!g_state.initialized) dev.sm_count = 152;
    const Decision d = decide(M, N, K, dev, g_state.forced_rung, epilogue, dtype);
    if (d.status) return d.status;
    const int Mt = M < tile_tokens(d.rung) ? M : tile_tokens(d.rung);
    info[0] = d.rung;
    if (is_mma(d.rung)) {
        const MmaPlan p = plan_mma(Mt, N, K, split_rule(d.rung), dev, epilogue);
        if (!p.ok) return W4A16_ERR_UNSUPPORTED;
        info[1] = p.warps * 32;
        info[2] = p.S;
        info[3] = p.grid;
    } else if (is_tc(d.rung)) {
        const TcPlan p = plan_tc(Mt, N, K, split_rule(d.rung), dev, epilogue);
        if (!p.ok) return W4A16_ERR_UNSUPPORTED;
        info[1] = p.threads;
        info[2] = p.S;
        info[3] = p.grid;
    } else {
        const GemvPlan p = plan_gemv(Mt, N, K, split_rule(d.rung), dev);
        if (!p.ok) return W4A16_ERR_UNSUPPORTED;
        info[1] = p.threads;
        info[2] = p.S;
        info[3] = p.grid_x * p.S;
    }
    return W4A16_OK;
}

int w4a16_set_forced_rung(int rung) {
    if (rung < W4A16_RUNG_AUTO || rung >= W4A16_NUM_RUNGS) return -2;
    std::lock_guard<std::mutex> lock(g_mutex);
    int prev = g_state.forced_rung;
    g_state.forced_rung = rung;
    return prev;
}

int w4a16_probe_counts(uint64_t *counts, int n) {
    if (!counts || n < 0) return 0;
    int k = n < W4A16_NUM_RUNGS ? n : W4A16_NUM_RUNGS;
    for (int i = 0; i < k; ++i) counts[i] = g_probe[i].load(std::memory_order_relaxed);
    return k;
}

uint64_t w4a16_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

void w4a16_probe_reset(void) {
    for (auto &c : g_probe) c.store(0, std::memory_order_relaxed);
    g_launches.store(0, std::memory_order_relaxed);
}

const char *w4a16_rung_name(int rung) {
    if (rung == W4A16_RUNG_AUTO) return "auto";
    if (rung < 0 || rung >= W4A16_NUM_RUNGS) return "?";
    return kRungNames[rung];
}

const char *w4a16_status_string(int status) {
    switch (status) {
        case W4A16_OK: return "ok";
        case W4A16_ERR_INVALID_ARG: return "invalid argument";
        case W4A16_ERR_UNSUPPORTED: return "unsupported shape or rung";
        case W4A16_ERR_MISALIGNED: return "misaligned pointer";
        case W4A16_ERR_WORKSPACE: return "split-K workspace too small";
        case W4A16_ERR_NOT_INITIALIZED: return "w4a16_init has not succeeded";
        case W4A16_ERR_CUDA: return "CUDA runtime error";
        case W4A16_ERR_DEVICE: return "a kernel reported a device-side error (bounded wait expired)";
    }
    return "?";
}

int w4a16_device_status(void *stream, int *code) {
    if (code) *code = 0;
    // the allocation-free linear's scratch on the current device, if a call
    // has set it up
    NoAllocScratch na{};
    int device = 0;
    const bool have_na = cudaGetDevice(&device) == cudaSuccess && noalloc_scratch(device, &na);
    if (!g_state.initialized && !have_na) return W4A16_ERR_NOT_INITIALIZED;
    cudaStream_t st = (cudaStream_t)stream;
    int h = 0, hn = 0;
    cudaError_t e = cudaSuccess;
    if (g_state.initialized)
        e = cudaMemcpyAsync(&h, g_state.ws.status, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && have_na)
        e = cudaMemcpyAsync(&hn, na.status, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && h != 0)
        e = cudaMemsetAsync(g_state.ws.status, 0, sizeof(int), st);
    // an expired wait in the allocation-free kernel may have left a block's
    // arrival counted and never reduced, or the scheduling words set: zero
    // them with the word, so that later calls start clean
    if (e == cudaSuccess && hn != 0) e = cudaMemsetAsync(na.counters, 0, na.counter_bytes, st);
    if (e == cudaSuccess && hn != 0) e = cudaMemsetAsync(na.status, 0, sizeof(int), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    h |= hn;
    if (code) *code = h;
    return h ? W4A16_ERR_DEVICE : W4A16_OK;
}

int w4a16_wait_probe(void *stream) {
    if (!g_state.initialized) return W4A16_ERR_NOT_INITIALIZED;
    cudaError_t e = launch_wait_probe(g_state.ws.status, nullptr, (cudaStream_t)stream);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    // the allocation-free linear's scratch, when set up on this device: the
    // same expired waits report into its word, and its first block counter is
    // left as a cut-short split-K launch can leave one
    NoAllocScratch na{};
    int device = 0;
    if (e == cudaSuccess && cudaGetDevice(&device) == cudaSuccess &&
        noalloc_scratch(device, &na)) {
        e = launch_wait_probe(na.status, na.counters, (cudaStream_t)stream);
        g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

int w4a16_last_cuda_error(void) { return t_last_cuda_error; }

int w4a16_device_sm_count(void) { return g_state.initialized ? g_state.dev.sm_count : 0; }

}  // extern "C"
