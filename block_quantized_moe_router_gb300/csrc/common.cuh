// common.cuh -- device helpers shared by the library's kernels (sm_103a only).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

#ifndef __CUDA_ARCH__
#define MOE_HOST_ONLY 1
#endif

namespace moe {

constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;

// ---- loads --------------------------------------------------------------------------------
// 16-byte read-only streaming load (weights are read once per launch: keep them out of L1).
__device__ __forceinline__ uint4 ldg_stream128(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// 16-byte read-only load that may be cached in L1 (activations shared by many warps).
__device__ __forceinline__ uint4 ldg_cached128(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u16(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u8(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// ---- FP4 / FP8 conversions (hardware cvt, exact) --------------------------------------------
// Two E2M1 codes of byte `sel` of w -> f16x2 (low nibble -> low half).
template <int SEL>
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t w) {
    uint32_t r;
    if constexpr (SEL == 0) {
        asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
            " cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n" : "=r"(r) : "r"(w));
    } else if constexpr (SEL == 1) {
        asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
            " cvt.rn.f16x2.e2m1x2 %0, b1;\n}\n" : "=r"(r) : "r"(w));
    } else if constexpr (SEL == 2) {
        asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
            " cvt.rn.f16x2.e2m1x2 %0, b2;\n}\n" : "=r"(r) : "r"(w));
    } else {
        asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
            " cvt.rn.f16x2.e2m1x2 %0, b3;\n}\n" : "=r"(r) : "r"(w));
    }
    return r;
}
// Two E4M3 bytes (low 16 bits of v) -> f16x2 (low byte -> low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
    uint32_t r;
    asm("{\n .reg .b16 h;\n cvt.u16.u32 h, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}\n"
        : "=r"(r) : "r"(v));
    return r;
}
// fp32 pair -> two E2M1 codes in one byte: `lo` -> low nibble (round to nearest even,
// saturating at +-6).
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n .reg .b8 b;\n cvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n cvt.u32.u8 %0, b;\n}\n"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r & 0xFFu;
}
// fp32 -> E4M3 byte (round to nearest even, saturating at 448).
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
    uint32_t h2 = e4m3x2_to_f16x2(byte & 0xFFu);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}
__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
    uint32_t h2 = e2m1x2_to_f16x2<0>(code & 0xFu);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// D = A (16x16 f16, row) * B (16x8 f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + __expf(-g)); }

__device__ __forceinline__ void status_or(int32_t* status, int32_t bits) {
    if (status && bits) atomicOr(status, bits);
}

// Programmatic dependent launch: wait until the preceding kernel on the stream has finished
// and its writes are visible; allow the next kernel on the stream to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

}  // namespace moe

// ---- host-side launch helpers ----------------------------------------------------------------
namespace moe {
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Launch with programmatic stream serialization: the kernel may be scheduled while its
// predecessor on the stream is still running and must call pdl_wait() before reading
// anything that predecessor writes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Which implementation of the expert FFN a call takes (shared by moe_workspace_size and
// moe_ffn_forward, so the workspace always matches the path).
enum FfnPath { PATH_DECODE = 0, PATH_GENERIC = 1, PATH_TC = 2 };

// The tcgen05 path needs K / N extents in whole 256-element tiles (NVFP4 or MXFP4 weights;
// MXFP4 block scales are re-expressed as E4M3 powers of two at preparation).
inline bool tc_shape_ok(int H, int I, int I_shared, int fmt_routed, int fmt_shared) {
    (void)fmt_routed;
    (void)fmt_shared;
    return H % 256 == 0 && I % 256 == 0 && I_shared % 256 == 0;
}

inline int select_path(int T, int H, int top_k, int act, bool tc_shape) {
    if (T <= 8 && T * top_k <= 64 && act == MOE_ACT_BF16 && H <= 8192) return PATH_DECODE;
    if (act == MOE_ACT_NVFP4 && tc_shape) return PATH_TC;
    return PATH_GENERIC;
}

// Workspace carve-up shared by moe_workspace_size and moe_ffn_forward.
struct Workspace {
    size_t counts, offsets, active, meta, sorted_pair, pos_of_pair, x16, xq, xs, h16, hq, hs, y;
    // tcgen05 path
    size_t mblock_expert, padrow_pair, tiles1, tiles2, tokq, toks, txq, txsf, thq, thsf, ybf, tscan;
    int max_blocks;
    size_t total;
    static Workspace plan(int E, int H, int I, int I_shared, int top_k, int T, int act, int path) {
        Workspace w{};
        const size_t P = (size_t)T * top_k;
        const size_t R = P + (I_shared > 0 ? (size_t)T : 0);
        const size_t Imax = (size_t)(I > I_shared ? I : I_shared);
        size_t off = 0;
        auto take = [&](size_t bytes) {
            size_t o = off;
            off = align_up(off + bytes, 256);
            return o;
        };
        w.counts = take(sizeof(int32_t) * (E + 1));
        w.offsets = take(sizeof(int32_t) * (E + 2));
        w.active = take(sizeof(int32_t) * (E + 1));
        w.meta = take(sizeof(int32_t) * 64);
        if (path == PATH_DECODE) {
            // h token-major per expert slot: [routed slots + shared][8][Imax]
            const size_t rows = ((size_t)(E < T * top_k ? E : T * top_k) + (I_shared > 0 ? 1 : 0)) * 8;
            w.h16 = take(sizeof(__half) * rows * Imax);
            w.x16 = take(sizeof(__half) * (size_t)T * H);
        } else if (path == PATH_GENERIC) {
            w.sorted_pair = take(sizeof(int32_t) * (P + 1));
            w.pos_of_pair = take(sizeof(int32_t) * (P + 1));
            w.x16 = take(sizeof(__half) * (size_t)T * H);
            w.xq = take(act == MOE_ACT_NVFP4 ? (size_t)T * H / 2 : 0);
            w.xs = take(act == MOE_ACT_NVFP4 ? (size_t)T * H / 16 : 0);
            w.h16 = take(sizeof(__half) * R * Imax);
            w.hq = take(act == MOE_ACT_NVFP4 ? R * Imax / 2 : 0);
            w.hs = take(act == MOE_ACT_NVFP4 ? R * Imax / 16 : 0);
            w.y = take(sizeof(float) * R * H);
        } else {
            // expert rows padded to 128: at most one partial block per active expert
            const size_t active = (size_t)E < P ? (size_t)E : P;
            w.max_blocks = (int)((P + 127) / 128 + active + (I_shared > 0 ? (T + 127) / 128 : 0));
            const size_t rows = (size_t)w.max_blocks * 128;
            w.tscan = take(sizeof(int32_t) * 5 * ((size_t)E + 2));  // counts, bases, cursors
            w.mblock_expert = take(sizeof(int32_t) * w.max_blocks);
            w.padrow_pair = take(sizeof(int32_t) * rows);
            w.tiles1 = take(16 * (size_t)w.max_blocks * (Imax / 128));
            w.tiles2 = take(16 * (size_t)w.max_blocks * (H / 256));
            w.tokq = take((size_t)T * H / 2);   // each token quantized once
            w.toks = take((size_t)T * H / 16);
            w.txq = take(rows * H / 2);
            w.txsf = take(rows * H / 16);
            w.thq = take(rows * Imax / 2);
            w.thsf = take(rows * Imax / 16);
            w.ybf = take(sizeof(__nv_bfloat16) * R * H);
        }
        w.total = off;
        return w;
    }
};
}  // namespace moe
