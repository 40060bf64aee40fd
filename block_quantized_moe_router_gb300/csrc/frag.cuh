// frag.cuh -- m16n8k16 A-fragments built from packed E2M1 weight rows (internal).
//
// A warp owns 16 weight rows; lane (g = lane/4, q = lane%4) streams 16 contiguous bytes
// (32 codes) of rows g and g+8 per 128-element K step.  Within the step the MMA K order is
// permuted so that MMA sub-step I takes chunk elements 4I..4I+3 of every lane: k-slots
// (2q, 2q+1) <- elements 4I, 4I+1 and (2q+8, 2q+9) <- elements 4I+2, 4I+3.  The B operand
// uses the same permutation (a lane's column reads the same 32 elements), so the dot
// product is unchanged.
#pragma once
#include "common.cuh"

namespace moe {

// Block-scale of the 16-byte chunk (32 codes) a lane holds, as f16x2 pairs for the chunk's
// first and second 16 elements.
template <int FMT>
__device__ __forceinline__ void chunk_scales(const uint8_t* srow, int step, int q, int mxbias,
                                             uint32_t& lo, uint32_t& hi) {
    if constexpr (FMT == MOE_FMT_NVFP4) {
        const uint32_t s2 = ldg_u16(srow + step * 8 + 2 * q);
        const uint32_t h = e4m3x2_to_f16x2(s2);
        lo = __byte_perm(h, h, 0x1010);
        hi = __byte_perm(h, h, 0x3232);
    } else {
        const int b = (int)ldg_u8(srow + step * 4 + q);
        const int field = min(30, max(0, b - mxbias));
        const uint32_t bits = (uint32_t)field << 10;
        lo = hi = bits | (bits << 16);
    }
}

struct ChunkA {
    uint4 r0, r1;       // packed codes of rows g and g+8
    uint32_t s0lo, s0hi, s1lo, s1hi;
};

template <int FMT>
__device__ __forceinline__ void load_chunk(ChunkA& c, const uint8_t* p0, const uint8_t* p1,
                                           const uint8_t* s0, const uint8_t* s1, int step, int q,
                                           int mxbias) {
    c.r0 = ldg_stream128(p0 + step * 64);
    c.r1 = ldg_stream128(p1 + step * 64);
    chunk_scales<FMT>(s0, step, q, mxbias, c.s0lo, c.s0hi);
    chunk_scales<FMT>(s1, step, q, mxbias, c.s1lo, c.s1hi);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// A fragment of MMA step i (0..7) from a chunk: rows g / g+8, k-slots (2q,2q+1) = chunk
// elements 4i, 4i+1 and k-slots (2q+8, 2q+9) = chunk elements 4i+2, 4i+3.
template <int I>
__device__ __forceinline__ void frag_a(const ChunkA& c, uint32_t (&a)[4]) {
    const uint32_t w0 = word_of(c.r0, I >> 1), w1 = word_of(c.r1, I >> 1);
    const uint32_t sc0 = (I < 4) ? c.s0lo : c.s0hi;
    const uint32_t sc1 = (I < 4) ? c.s1lo : c.s1hi;
    constexpr int SEL = (I & 1) * 2;
    a[0] = hmul2(e2m1x2_to_f16x2<SEL>(w0), sc0);
    a[1] = hmul2(e2m1x2_to_f16x2<SEL>(w1), sc1);
    a[2] = hmul2(e2m1x2_to_f16x2<SEL + 1>(w0), sc0);
    a[3] = hmul2(e2m1x2_to_f16x2<SEL + 1>(w1), sc1);
}

// ---- asynchronous global -> shared copies (per-thread, no register staging) ----------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t saddr, const void* g) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t saddr, const void* g) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(saddr), "l"(g) : "memory");
}
// The same copies with an L2 cache policy (streamed weights: evict first, so that they do not
// push the kernel's code and the small per-step tensors out of L2).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void cp_async16_pol(uint32_t saddr, const void* g, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(saddr), "l"(g),
                 "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async8_pol(uint32_t saddr, const void* g, uint64_t pol) {
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 8, %2;" ::"r"(saddr), "l"(g),
                 "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async4_pol(uint32_t saddr, const void* g, uint64_t pol) {
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 4, %2;" ::"r"(saddr), "l"(g),
                 "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Block scales of a lane's 32-element chunk from the raw scale bits of its row and step:
// NVFP4 -- the 8 bytes of the row's 128-element step, this lane's pair at byte 2q;
// MXFP4 -- the 4 bytes of the row's step, this lane's byte at q.
template <int FMT>
__device__ __forceinline__ void scales_from_raw(uint2 raw, int q, int mxbias, uint32_t& lo,
                                                uint32_t& hi) {
    if constexpr (FMT == MOE_FMT_NVFP4) {
        const uint32_t word = (q < 2) ? raw.x : raw.y;
        const uint32_t s2 = (q & 1) ? (word >> 16) : (word & 0xFFFFu);
        const uint32_t h = e4m3x2_to_f16x2(s2);
        lo = __byte_perm(h, h, 0x1010);
        hi = __byte_perm(h, h, 0x3232);
    } else {
        const int b = (int)((raw.x >> (8 * q)) & 0xFFu);
        const int field = min(30, max(0, b - mxbias));
        const uint32_t bits = (uint32_t)field << 10;
        lo = hi = bits | (bits << 16);
    }
}

}  // namespace moe
