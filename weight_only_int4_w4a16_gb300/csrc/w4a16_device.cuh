// Device helpers shared by the W4A16 kernels: the nibble unpack, the
// activation pair order that matches it, and mbarrier / timer wrappers.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace w4a16 {
namespace dev {

// (a & b) | c in one instruction.
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

// The nibble unpack.  A nibble OR-ed into the mantissa of the fp16 constant
// 1024 (0x6400) is the fp16 value 1024 + q; a nibble at mantissa bits 4..7 of
// the constant 64 (0x5400, mantissa unit 1/16) is 64 + q.  One lop3 thus turns
// two nibbles of a word into an fp16 pair, and subtracting the matching
// (1024 + z) or (64 + z) pair is exact and leaves q - z.  For the word
// w = q0 | q1 << 4 | ... | q7 << 28 the four pairs are
//   d[0] = (q0 - z, q4 - z), d[1] = (q1 - z, q5 - z),
//   d[2] = (q2 - z, q6 - z), d[3] = (q3 - z, q7 - z)   (low half first).
struct ZeroPair {
    uint32_t hi;  // (1024 + z, 1024 + z)
    uint32_t lo;  // (64 + z, 64 + z)
};

__device__ __forceinline__ ZeroPair zero_pair(uint32_t z) {
    return {0x64006400u | z | (z << 16), 0x54005400u | (z << 4) | (z << 20)};
}

__device__ __forceinline__ void unpack_word(uint32_t w, ZeroPair zz, uint32_t (&d)[4]) {
    const uint32_t w8 = w >> 8;
    d[0] = hsub2(lop3_and_or(w, 0x000f000fu, 0x64006400u), zz.hi);
    d[1] = hsub2(lop3_and_or(w, 0x00f000f0u, 0x54005400u), zz.lo);
    d[2] = hsub2(lop3_and_or(w8, 0x000f000fu, 0x64006400u), zz.hi);
    d[3] = hsub2(lop3_and_or(w8, 0x00f000f0u, 0x54005400u), zz.lo);
}

// 8 consecutive fp16 activations (h0..h7) -> (h0,h4) (h1,h5) (h2,h6) (h3,h7):
// the order unpack_word yields the weights of one word.
__device__ __forceinline__ uint4 pair_order(uint4 v) {
    uint4 o;
    o.x = prmt(v.x, v.z, 0x5410);
    o.y = prmt(v.x, v.z, 0x7632);
    o.z = prmt(v.y, v.w, 0x5410);
    o.w = prmt(v.y, v.w, 0x7632);
    return o;
}

// Streaming 128-bit load: read-only, not kept in L1, L2 fetches 256 bytes.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace dev
}  // namespace w4a16
