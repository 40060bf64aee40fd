// topk.cuh -- one warp's top-K routing of one token (internal; used by the routing kernel and
// by the fused few-token kernel).
//
// Routing kinds (spark_model MoE pages): softmax top-K (moe/init.rs, `moe_topk_softmax`
// handles); sigmoid scores with a correction bias that only affects the selection
// (moe/mod.rs, `correction_bias_dev` field doc); sqrt(softplus) scores in the same scheme
// (moe/mod.rs, `moe_topk_sqrtsoftplus` handles); softmax probabilities with a selection bias
// (moe/mod.rs, the LongCat `moe_topk_softmax_bias` handles).
#pragma once
#include "common.cuh"

namespace moe {

__device__ __forceinline__ float gate_score(int scoring, float l) {
    if (scoring == MOE_SCORE_SQRTSOFTPLUS) return sqrtf(l > 30.f ? l : log1pf(expf(l)));
    return 1.0f / (1.0f + expf(-l));
}

// fp32 -> uint32 with the same order as the floats (for packed 64-bit selection keys).
__device__ __forceinline__ uint32_t orderable(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Selects the top k of E <= 32 * EPL experts for one token.  `load(e)` returns logit e.
// Keys pack (selection score, ~expert) so one 64-bit max picks the higher score and, on a
// tie, the lower expert index; non-finite logits rank below every finite one.  Each round
// takes the lane's maximum with a tree and the warp's with two 32-bit reductions (high word,
// then the low word among the lanes holding that high word).  On return lanes < k hold
// their pick in my_e / my_w (descending selection score); the result says whether any logit
// was non-finite.
template <int EPL, typename Load>
__device__ __forceinline__ bool warp_topk(const Load& load, const float* bias, int E, int k,
                                          int scoring, int renorm, float scaling, int lane,
                                          int& my_e, float& my_w) {
    unsigned long long key[EPL];
    float lg[EPL], raw[EPL], bv[EPL];
    bool nonfinite = false;
    float lmax = -INFINITY;
    const bool use_bias = bias != nullptr && scoring != MOE_SCORE_SOFTMAX;
    const bool softmax = scoring == MOE_SCORE_SOFTMAX || scoring == MOE_SCORE_SOFTMAX_BIAS;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {  // every load issued before any is used
        const int e = lane + 32 * j;
        raw[j] = e < E ? load(e) : 0.f;
        bv[j] = (use_bias && e < E) ? bias[e] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        lg[j] = -INFINITY;
        if (e < E) {
            if (isfinite(raw[j])) {
                lg[j] = raw[j];
                lmax = fmaxf(lmax, raw[j]);
            } else {
                nonfinite = true;
            }
        }
    }
    const bool any_nonfinite = __any_sync(0xffffffffu, nonfinite);
#pragma unroll
    for (int o = 16; o; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    // softmax denominator over every finite logit (plain softmax needs it only unrenormalised)
    float zall = 1.f;
    if (scoring == MOE_SCORE_SOFTMAX_BIAS || (scoring == MOE_SCORE_SOFTMAX && !renorm)) {
        zall = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            if (isfinite(lg[j])) zall += expf(lg[j] - lmax);
#pragma unroll
        for (int o = 16; o; o >>= 1) zall += __shfl_xor_sync(0xffffffffu, zall, o);
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        key[j] = 0ull;
        if (e < E) {
            float v = -INFINITY;
            if (isfinite(lg[j])) {
                if (scoring == MOE_SCORE_SOFTMAX) v = lg[j];  // softmax is monotone in the logit
                else if (scoring == MOE_SCORE_SOFTMAX_BIAS) v = expf(lg[j] - lmax) / zall + bv[j];
                else v = gate_score(scoring, lg[j]) + bv[j];
            }
            key[j] = ((unsigned long long)orderable(v) << 32) | (0xFFFFFFFFu - (uint32_t)e);
        }
    }

    my_e = 0;
    float my_l = 0.f;  // the logit of this lane's pick, passed on by the lane that held it
    for (int r = 0; r < k; ++r) {
        unsigned long long t[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) t[j] = key[j];
#pragma unroll
        for (int w = EPL / 2; w >= 1; w >>= 1)
#pragma unroll
            for (int j = 0; j < w; ++j) t[j] = t[j + w] > t[j] ? t[j + w] : t[j];
        const uint32_t hi = (uint32_t)(t[0] >> 32);
        const uint32_t whi = __reduce_max_sync(0xffffffffu, hi);
        const uint32_t wlo = __reduce_max_sync(0xffffffffu, hi == whi ? (uint32_t)t[0] : 0u);
        const unsigned long long best = ((unsigned long long)whi << 32) | wlo;
        // keys are unique (they hold the expert index): clear the winner by value, so the key
        // array is never indexed at run time and stays in registers
        float hit = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const bool won = key[j] == best;
            hit = won ? raw[j] : hit;
            key[j] = won ? 0ull : key[j];
        }
        const int e = (int)(0xFFFFFFFFu - wlo);
        const float l = __shfl_sync(0xffffffffu, hit, e & 31);  // expert e sits in lane e % 32
        if (lane == r) {
            my_e = e;
            my_l = l;
        }
    }
    float num = 0.f;
    if (lane < k && isfinite(my_l)) num = softmax ? expf(my_l - lmax) : gate_score(scoring, my_l);
    float den = 1.f;
    if (renorm) {
        den = num;
#pragma unroll
        for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    } else if (softmax) {
        den = zall;
    }
    my_w = lane < k ? (den > 0.f ? num / den : 0.f) * scaling : 0.f;
    return any_nonfinite;
}

}  // namespace moe
