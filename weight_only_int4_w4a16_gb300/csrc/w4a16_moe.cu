// Mixture of experts on the W4A16 rungs (forum.sourcefind.cn thread "vLLM on
// Hygon Z100", section 七: a router picks a few experts per token; the tokens
// are rearranged by expert, aligned and padded; the W4A16 expert small-M GEMV
// runs over packed INT4 experts; each token's expert outputs are summed with
// the router's weights).
//
//   * align: a stable counting sort of the T*k slots (token t's j-th choice is
//     slot t*k + j) by expert: per-expert offsets, the slot at each sorted
//     position and the sorted position of each slot;
//   * prepare: one CTA cuts every expert's range of slots into tiles of up to
//     8 (the MMA's N) and writes one fused-round descriptor per tile (the
//     expert's tensor map and arrays from a per-expert template, the tile's
//     rows of the sorted activations and outputs, its own split-K partials
//     and counters); the other CTAs gather each sorted slot's activation row
//     from its token when the input is by token;
//   * the tiles then run as one launch of the fused-round mma kernel, which
//     reads the descriptors written just before it (after waiting for that
//     kernel) and skips descriptor slots past the last tile;
//   * sum: out[t] = sum_j w[t, j] * y[pos(t*k + j)] in fp32, j increasing,
//     rounded once.
#include <string.h>

#include "../../include/w4a16.h"
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kAlignThreads = 1024;

// Each kernel here may start while the previous one in the stream drains
// (programmatic dependent launch): it lets its own successor start early,
// then waits for its predecessor before reading anything.
__device__ __forceinline__ void chain_start() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... Params, typename... Args>
cudaError_t launch_chained(void (*kernel)(Params...), int grid, int threads, cudaStream_t stream,
                           Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
constexpr int kAlignChunk = 4096;  // slots staged in shared memory per pass

// One CTA.  Thread e owns expert e: counts, the exclusive prefix, then a scan
// over the slots in order that places expert e's slots (stable by slot).  A
// slot whose id is outside [0, E) gets no position (pos = -1, it is left out
// of every expert and of the sum) and sets a status bit.
__global__ void __launch_bounds__(kAlignThreads)
    moe_align_kernel(const int32_t *__restrict__ ids, int n_slots, int E,
                     int32_t *__restrict__ sorted, int32_t *__restrict__ pos,
                     int32_t *__restrict__ offsets, int *status) {
    __shared__ int count[kMaxMoeExperts];
    __shared__ int32_t chunk[kAlignChunk];
    chain_start();
    for (int e = threadIdx.x; e < E; e += blockDim.x) count[e] = 0;
    __syncthreads();
    for (int s = threadIdx.x; s < n_slots; s += blockDim.x) {
        const int e = ids[s];
        if (e >= 0 && e < E) {
            atomicAdd(&count[e], 1);
        } else {
            pos[s] = -1;
            atomicOr(status, kErrMoeIds);
        }
    }
    __syncthreads();
    {
        // exclusive scan of the counts, one expert per thread (E <= 1024)
        __shared__ int warp_sum[kAlignThreads / 32];
        const int e = threadIdx.x, lane = e & 31, wid = e >> 5;
        const int c = e < E ? count[e] : 0;
        int incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) warp_sum[wid] = incl;
        __syncthreads();
        int before = incl - c;
        for (int w = 0; w < wid; ++w) before += warp_sum[w];
        if (e < E) {
            offsets[e] = before;
            count[e] = before;  // becomes the expert's fill cursor
        }
        if (e == E - 1) offsets[E] = before + c;
    }
    __syncthreads();
    for (int base = 0; base < n_slots; base += kAlignChunk) {
        const int n = min(kAlignChunk, n_slots - base);
        for (int i = threadIdx.x; i < n; i += blockDim.x) chunk[i] = ids[base + i];
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            int p = count[e];
            for (int i = 0; i < n; ++i)
                if (chunk[i] == e) {
                    sorted[p] = base + i;
                    pos[base + i] = p;
                    ++p;
                }
            count[e] = p;
        }
        __syncthreads();
    }
}

// Block 0: the tile descriptors.  Blocks 1..: the gathered activation rows.
// With a second linear (tmpl2: an expert MLP's down projection) block 0 also
// writes its tiles right after the first linear's: tile t of the second reads
// the first's output rows of tile t and waits for that tile (wait_for).
__global__ void __launch_bounds__(256)
    moe_prepare_kernel(const MmaLinDesc *__restrict__ tmpl, const MmaLinDesc *__restrict__ tmpl2,
                       const int32_t *__restrict__ offsets, const int32_t *__restrict__ sorted,
                       int E, int k, int max_tiles, int units1, int units2, MoeTileSpace sp,
                       MoeTileSpace sp2, const __half *__restrict__ x, int gather,
                       __half *__restrict__ xs, int n_slots, int K,
                       MmaLinDesc *__restrict__ tiles, int *__restrict__ counts) {
    chain_start();
    if (blockIdx.x > 0) {
        // sorted position p reads its token's row: x[sorted[p] / k] (positions
        // up to offsets[E]: slots with an invalid id have none)
        const int kw = K / 8;  // 16-byte words per row
        const int n_valid = min(offsets[E], n_slots);
        for (long long i = (blockIdx.x - 1) * (long long)blockDim.x + threadIdx.x;
             i < (long long)n_valid * kw; i += (long long)(gridDim.x - 1) * blockDim.x) {
            const int p = (int)(i / kw), w = (int)(i - (long long)p * kw);
            const int t = sorted[p] / k;
            reinterpret_cast<uint4 *>(xs + (size_t)p * K)[w] =
                reinterpret_cast<const uint4 *>(x + (size_t)t * K)[w];
        }
        return;
    }
    __shared__ int tile_expert[kMaxMoeTiles];
    __shared__ int tile_row[kMaxMoeTiles];
    __shared__ int tile_m[kMaxMoeTiles];
    __shared__ int warp_sum[8];
    __shared__ int n_tiles;
    // the tiles of each expert (ceil(slots / 8)), numbered by an exclusive
    // scan over the experts: each thread takes up to 4 consecutive experts
    constexpr int kPer = kMaxMoeExperts / 256;
    const int e0 = threadIdx.x * kPer;
    int cnt[kPer], local = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = e0 + i;
        cnt[i] = e < E ? (offsets[e + 1] - offsets[e] + kMmaMaxTokens - 1) / kMmaMaxTokens : 0;
        local += cnt[i];
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sum[wid] = incl;
    __syncthreads();
    int before = incl - local;
    for (int w = 0; w < wid; ++w) before += warp_sum[w];
    if (threadIdx.x == blockDim.x - 1) {
        const int total = before + local;
        const int nt = total < max_tiles ? total : max_tiles;
        n_tiles = nt;
        counts[0] = tmpl2 ? 2 * nt : nt;
        counts[1] = nt * (units1 + (tmpl2 ? units2 : 0));
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = e0 + i;
        for (int t = 0; t < cnt[i]; ++t) {
            const int idx = before + t;
            if (idx >= max_tiles) break;
            const int r = offsets[e] + t * kMmaMaxTokens;
            tile_expert[idx] = e;
            tile_row[idx] = r;
            tile_m[idx] = min(kMmaMaxTokens, offsets[e + 1] - r);
        }
        before += cnt[i];
    }
    __syncthreads();
    const int nt = n_tiles;
    const int slots = (tmpl2 ? 2 : 1) * max_tiles;
    // which linear (0, 1) and tile a descriptor slot holds (-1: unused)
    auto role = [&](int i, int &lin, int &t) {
        lin = i < nt ? 0 : (tmpl2 && i < 2 * nt ? 1 : -1);
        t = lin == 0 ? i : i - nt;
    };
    // copy each tile's template, then its own fields; slots past the last
    // tile only start past every unit
    const int words = (int)(sizeof(MmaLinDesc) / 4);
    const int used = (tmpl2 ? 2 : 1) * nt;
    for (int i = threadIdx.x; i < used * words; i += blockDim.x) {
        const int d = i / words, w = i - d * words;
        int lin, t;
        role(d, lin, t);
        const MmaLinDesc *src = lin == 1 ? tmpl2 + tile_expert[t] : tmpl + tile_expert[t];
        reinterpret_cast<uint32_t *>(tiles + d)[w] = reinterpret_cast<const uint32_t *>(src)[w];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < slots; i += blockDim.x) {
        MmaLinDesc &d = tiles[i];
        int lin, t;
        role(i, lin, t);
        d.wait_for = -1;
        if (lin < 0) {
            d.M = 1;
            d.unit_start = 0x7fffffff;
            continue;
        }
        const int r = tile_row[t], e = tile_expert[t];
        const MoeTileSpace &q = lin == 0 ? sp : sp2;
        d.M = tile_m[t];
        d.y = q.y + (size_t)r * d.ycols;
        d.partials = q.partials ? q.partials + (size_t)t * q.partial_stride : nullptr;
        d.counters = q.counters ? q.counters + (size_t)t * q.counter_stride : nullptr;
        if (lin == 0) {
            d.x = (gather ? xs : x) + (size_t)r * K;
            d.unit_start = t * units1;
            d.tmap_ref = &tmpl[e].tmap;
        } else {
            d.x = sp.y + (size_t)r * tmpl[e].ycols;  // the first linear's rows of this tile
            d.unit_start = nt * units1 + t * units2;
            d.tmap_ref = &tmpl2[e].tmap;
            d.wait_for = t;
        }
    }
}

template <bool kBf16>
__global__ void __launch_bounds__(256)
    moe_sum_kernel(const __half *__restrict__ y, const int32_t *__restrict__ pos,
                   const float *__restrict__ w, int T, int k, int N, __half *__restrict__ out) {
    chain_start();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)T * N;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / N), n = (int)(i - (long long)t * N);
        float acc = 0.f;
        for (int j = 0; j < k; ++j) {
            const int s = t * k + j;
            if (pos[s] < 0) continue;  // a slot with an invalid expert id
            const __half v = y[(size_t)pos[s] * N + n];
            const float f = kBf16 ? __uint_as_float((uint32_t)__half_as_ushort(v) << 16)
                                  : __half2float(v);
            acc = fmaf(w[s], f, acc);
        }
        out[i] = kBf16 ? __ushort_as_half(__bfloat16_as_ushort(__float2bfloat16_rn(acc)))
                       : __float2half_rn(acc);
    }
}

}  // namespace

cudaError_t launch_moe_align(const int32_t *ids, int n_slots, int E, int32_t *sorted,
                             int32_t *pos, int32_t *offsets, int *status, cudaStream_t stream) {
    return launch_chained(moe_align_kernel, 1, kAlignThreads, stream, ids, n_slots, E, sorted, pos,
                          offsets, status);
}

cudaError_t launch_moe_prepare(const MmaLinDesc *tmpl, const MmaLinDesc *tmpl2,
                               const int32_t *offsets, const int32_t *sorted, int E, int k,
                               int max_tiles, int units1, int units2, const MoeTileSpace &sp,
                               const MoeTileSpace &sp2, const __half *x, bool gather, __half *xs,
                               int n_slots, int K, MmaLinDesc *tiles, int *counts,
                               cudaStream_t stream) {
    int blocks = 1;
    if (gather) {
        const long long words = (long long)n_slots * (K / 8);
        long long b = (words + 255) / 256;
        if (b > 1024) b = 1024;
        blocks += (int)(b < 1 ? 1 : b);
    }
    return launch_chained(moe_prepare_kernel, blocks, 256, stream, tmpl, tmpl2, offsets, sorted, E,
                          k, max_tiles, units1, units2, sp, sp2, x, gather ? 1 : 0, xs, n_slots,
                          K, tiles, counts);
}

cudaError_t launch_moe_sum(const __half *y, const int32_t *pos, const float *w, int T, int k,
                           int N, bool bf16, __half *out, cudaStream_t stream) {
    long long b = ((long long)T * N + 255) / 256;
    if (b > 4096) b = 4096;
    if (b < 1) b = 1;
    return bf16 ? launch_chained(moe_sum_kernel<true>, (int)b, 256, stream, y, pos, w, T, k, N, out)
                : launch_chained(moe_sum_kernel<false>, (int)b, 256, stream, y, pos, w, T, k, N,
                                 out);
}

}  // namespace w4a16
