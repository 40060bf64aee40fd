// quant.cuh -- the NVFP4 activation quantizer on 16 values (internal).
//
// Per 16 consecutive elements: s = E4M3(amax / 6 / g) (round to nearest even, saturating at
// 448), code = E2M1(v / (e4m3(s) * g)) (round to nearest even, saturating at 6), all-zero codes
// when s decodes to 0 -- the `quantize_bf16_to_nvfp4` step of the FP4 x FP4 recipe
// (qwen3_attention/init.rs handle list; moe/mod.rs `moe_fused_gate_up_t_k64_fp4` doc).
#pragma once
#include "common.cuh"

namespace moe {

// Writes 8 packed bytes (element 2i in the low nibble), one E4M3 scale byte and, when `deq` is
// not null, the 16 exact dequantized values as f16.
__device__ __forceinline__ void quant16(const float (&v)[16], float g, uint8_t* packed,
                                        uint8_t* scale, __half* deq) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    float qs = amax / 6.0f;
    qs = qs / g;
    const uint32_t s = f32_to_e4m3(qs);
    const float denom = e4m3_to_f32(s) * g;
    uint32_t bytes[8];
    float dq[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t b = 0;
        if (denom != 0.f) b = f32x2_to_e2m1x2(v[2 * i] / denom, v[2 * i + 1] / denom);
        bytes[i] = b;
        dq[2 * i] = e2m1_to_f32(b & 0xF) * denom;
        dq[2 * i + 1] = e2m1_to_f32(b >> 4) * denom;
    }
    uint2 pk;
    pk.x = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
    pk.y = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
    *reinterpret_cast<uint2*>(packed) = pk;
    *scale = (uint8_t)s;
    if (deq) {
        uint4 a, b;
        a.x = pack_half2(dq[0], dq[1]);   a.y = pack_half2(dq[2], dq[3]);
        a.z = pack_half2(dq[4], dq[5]);   a.w = pack_half2(dq[6], dq[7]);
        b.x = pack_half2(dq[8], dq[9]);   b.y = pack_half2(dq[10], dq[11]);
        b.z = pack_half2(dq[12], dq[13]); b.w = pack_half2(dq[14], dq[15]);
        reinterpret_cast<uint4*>(deq)[0] = a;
        reinterpret_cast<uint4*>(deq)[1] = b;
    }
}

__device__ __forceinline__ void load_bf16x16(const __nv_bfloat16* src, float (&v)[16]) {
    const uint4 a = ldg_cached128(src), b = ldg_cached128(src + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// The same recipe with the 16 per-element divisions replaced by one reciprocal per block
// (v * (1 / denom)); the scale byte is computed exactly as above.  Used where the input is
// itself an fp32 intermediate (h inside the tensor-core GEMM epilogue), so a code can differ
// from the divided form only when v / denom lies within one ulp of an E2M1 midpoint.
__device__ __forceinline__ void quant16_rcp(const float (&v)[16], float g, uint8_t* packed,
                                            uint8_t* scale) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    float qs = amax / 6.0f;
    qs = qs / g;
    const uint32_t s = f32_to_e4m3(qs);
    const float denom = e4m3_to_f32(s) * g;
    const float inv = denom != 0.f ? 1.0f / denom : 0.f;
    uint2 pk;
    uint32_t bytes[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) bytes[i] = f32x2_to_e2m1x2(v[2 * i] * inv, v[2 * i + 1] * inv);
    pk.x = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
    pk.y = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
    *reinterpret_cast<uint2*>(packed) = pk;
    *scale = (uint8_t)s;
}

}  // namespace moe
