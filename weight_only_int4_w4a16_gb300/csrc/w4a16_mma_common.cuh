// Device helpers of the warp-level tensor-core kernels (the 4-bit mma rung,
// the dense 16-bit rung and the expert decode kernel): the m16n8k16 MMA, the
// staged-activation layout and pair order, bf16 staging as scaled fp16, and
// the copy, mbarrier and counter primitives with bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "w4a16_device.cuh"

namespace w4a16 {
namespace warp_mma {

constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // 200 ms per wait
constexpr float kTwo20 = 1048576.f;
constexpr float kTwoM20 = 1.f / 1048576.f;

// Staged x: 16-byte unit J of a token row lives at unit J ^ (bit 3 of J moved
// to bit 1).  With a row stride of 16 (mod 128) bytes the 16-byte reads of a
// quarter warp (two tokens x four lanes) fall on distinct banks.
__device__ __forceinline__ int x_unit(int J) { return J ^ (((J >> 3) & 1) << 1); }

// bf16 activations are staged as fp16 for the fp16 MMA: token t's values are
// scaled by 2^k_t, k_t chosen from the largest exponent field E_t among them so
// that every scaled value is below 2^15 (fp16's range); the scale leaves at
// the end of each strip.  Values 2^29 below the token's largest lose bits to
// fp16's subnormals (an error under 2^-39 of the largest).  The exponents sit
// in 8 ints after the staged x and its sums.
__device__ __forceinline__ int *token_exps(uint8_t *xs, int M, int xstride, int slice_groups) {
    return reinterpret_cast<int *>(xs + (size_t)M * xstride + (size_t)slice_groups * 8 * 4);
}
// k_t for a largest biased exponent E (values below 2^(E - 126)), kept within
// the float exponent range so that 2^k and 2^-k are finite
__device__ __forceinline__ int bf16_stage_shift(int E) { return max(-126, min(126, 141 - E)); }
__device__ __forceinline__ float pow2(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }
// largest exponent field among the 8 bf16 values of a 16-byte unit
__device__ __forceinline__ int max_bf16_exp(uint4 v) {
    // the exponent fields in place (sign cleared), the largest by 16-bit
    // SIMD max: the unsigned order of the masked halves is that of the fields
    constexpr uint32_t kExp = 0x7f807f80u;
    const uint32_t m = __vmaxu2(__vmaxu2(v.x & kExp, v.y & kExp), __vmaxu2(v.z & kExp, v.w & kExp));
    return (int)(max(m & 0xffffu, m >> 16) >> 7);
}
// 8 bf16 values times 2^k, rounded to fp16 (exact but for the subnormal tail)
__device__ __forceinline__ uint4 bf16_to_scaled_f16(uint4 v, float scale) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16) * scale,
                                            __uint_as_float(w[i] & 0xffff0000u) * scale);
        o[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-bit activations, scales and outputs are IEEE binary16 or bfloat16 (the
// top half of a binary32); storage is 16-bit either way.
template <bool kBf16>
__device__ __forceinline__ float to_float(__half h) {
    if constexpr (kBf16) return __uint_as_float((uint32_t)__half_as_ushort(h) << 16);
    else return __half2float(h);
}
template <bool kBf16>
__device__ __forceinline__ float bits_to_float(uint32_t bits16) {  // low 16 bits
    if constexpr (kBf16) return __uint_as_float(bits16 << 16);
    else return __half2float(__ushort_as_half((unsigned short)bits16));
}
template <bool kBf16>
__device__ __forceinline__ __half from_float(float v) {  // round to nearest even
    if constexpr (kBf16) return __ushort_as_half(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
    else return __float2half_rn(v);
}
template <bool kBf16>
__device__ __forceinline__ float2 pair_to_float2(uint32_t v) {
    if constexpr (kBf16) return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    else return __half22float2(*reinterpret_cast<const __half2 *>(&v));
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

// box of a 3-D tensor map at (word 0, row, group): the qweight boxes of the
// warp-MMA kernels.  The weights are read once, so the copy carries an L2
// evict-first policy: they do not push out what is read again (activations,
// scale and zero words shared by neighbouring rows, split-K partials).
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap *map, int row, int grp,
                                        uint32_t bar) {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(grp), "r"(bar), "l"(pol)
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


// Bounded wait until *p >= target (acquire); false once kWaitNs has passed.
__device__ __forceinline__ bool wait_counter(const unsigned *p, unsigned target) {
    const unsigned long long t0 = dev::globaltimer();
    for (uint32_t i = 0;; ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        if ((i & 15) == 15) {
            if (dev::globaltimer() - t0 > kWaitNs) return false;
            __nanosleep(256);
        }
    }
}

__device__ __forceinline__ int ld_acquire_cta(const int *p) {
    int v;
    asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(v) : "r"(dev::smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_cta(int *p, int v) {
    asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(dev::smem_u32(p)), "r"(v) : "memory");
}

}  // namespace warp_mma
}  // namespace w4a16
