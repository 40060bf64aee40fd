// route.cu -- router GEMM (bf16 x bf16 -> fp32 logits) and the top-K routing kernels.
//
// Routing kinds (spark_model MoE pages):
//   softmax top-K           -- moe/init.rs, the `moe_topk_softmax` handles;
//   sigmoid + correction bias (selection on sigmoid+bias, weights from the unbiased sigmoid,
//     renormalised and scaled) -- moe/mod.rs, `correction_bias_dev` field doc;
//   sqrt(softplus) scores in the same scheme -- moe/mod.rs, `moe_topk_sqrtsoftplus` handles;
//   static hash routing through tid2eid [vocab, top_k] -- moe/init.rs, `new_with_hash` doc;
//     its weights either equal or, for the family that ships both the hash and the
//     sqrt(softplus) routing handles (moe/init.rs lookups), the sqrt(softplus) router scores
//     of the table's experts.
// The router keeps fp32 logits (moe/mod.rs, `dense_gemm_f32out` field doc: an fp32-output
// router GEMM feeding an fp32-input top-K).  Ids and weights stay on the device.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

// ------------------------------------------------------------------------------------------
// Router logits: logits[t][e] = sum_h x[t][h] * Wr[e][h].
// One CTA computes 16 experts x (8*NT) tokens; its KSPLIT warps split H and reduce through
// shared memory.  Each warp runs bf16 m16n8k16 MMAs with fp32 accumulation.  Within a warp
// the K order of the fragments is permuted so that every lane reads 16 contiguous bytes of
// its expert row and of its token row per 32-element step (both operands use the same
// permutation, so the dot product is unchanged).
// ------------------------------------------------------------------------------------------
template <int NT, int KSPLIT>
__global__ void __launch_bounds__(KSPLIT * 32)
router_logits_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wr,
                     float* __restrict__ logits, int T, int E, int H) {
    __shared__ float red[KSPLIT][NT * 4][32];
    pdl_wait();  // x may come from the preceding kernel
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int e0 = blockIdx.x * 16;
    const int t0 = blockIdx.y * 8 * NT;
    const int steps = H / 32;                       // 32 K-elements per warp step
    const int per = (steps + KSPLIT - 1) / KSPLIT;
    const int s_begin = warp * per;
    const int s_end = min(steps, s_begin + per);

    const int ea = e0 + g, eb = e0 + g + 8;
    const bool va = ea < E, vb = eb < E;
    const __nv_bfloat16* wa = wr + (size_t)(va ? ea : 0) * H + 8 * q;
    const __nv_bfloat16* wb = wr + (size_t)(vb ? eb : 0) * H + 8 * q;
    const __nv_bfloat16* xp[NT];
    bool vt[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int t = t0 + nt * 8 + g;
        vt[nt] = t < T;
        xp[nt] = x + (size_t)(vt[nt] ? t : 0) * H + 8 * q;
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;

    for (int s = s_begin; s < s_end; ++s) {
        const int kofs = s * 32;
        uint4 A0 = va ? ldg_stream128(wa + kofs) : make_uint4(0, 0, 0, 0);
        uint4 A1 = vb ? ldg_stream128(wb + kofs) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            uint4 B = vt[nt] ? ldg_cached128(xp[nt] + kofs) : make_uint4(0, 0, 0, 0);
            mma_bf16_16816(acc[nt], A0.x, A1.x, A0.y, A1.y, B.x, B.y);
            mma_bf16_16816(acc[nt], A0.z, A1.z, A0.w, A1.w, B.z, B.w);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[warp][nt * 4 + i][lane] = acc[nt][i];
    __syncthreads();
    for (int idx = threadIdx.x; idx < NT * 4 * 32; idx += blockDim.x) {
        const int slot = idx >> 5, ln = idx & 31;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < KSPLIT; ++w) sum += red[w][slot][ln];
        const int nt = slot >> 2, i = slot & 3;
        const int gg = ln >> 2, qq = ln & 3;
        const int e = e0 + gg + ((i & 2) ? 8 : 0);
        const int t = t0 + nt * 8 + 2 * qq + (i & 1);
        if (e < E && t < T) logits[(size_t)t * E + e] = sum;
    }
}

// ------------------------------------------------------------------------------------------
// Router logits for many tokens: CTA tile 128 tokens x 64 experts, K staged 64 at a time
// through a 3-stage cp.async ring in shared memory (rows padded to 144 bytes so ldmatrix is
// conflict-free), 8 warps of 32 tokens x 32 experts on bf16 m16n8k16 MMAs, fp32 accumulation.
// Rows beyond T or E are zero-filled by the copies and never stored.
// ------------------------------------------------------------------------------------------
constexpr int kRgBM = 128, kRgBN = 64, kRgBK = 64, kRgStages = 3;
constexpr int kRgRow = kRgBK * 2 + 16;  // bytes per staged row (64 bf16 + 16 bytes of padding)
constexpr int kRgSmem = kRgStages * (kRgBM + kRgBN) * kRgRow;

__device__ __forceinline__ void cp_async16_zfill(uint32_t saddr, const void* g, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(g), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t saddr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(saddr));
}

__global__ void __launch_bounds__(256)
router_gemm_tiled_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wr,
                         float* __restrict__ logits, int T, int E, int H) {
    extern __shared__ __align__(16) uint8_t rsm[];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kRgBM, e0 = blockIdx.y * kRgBN;
    const int wm = warp & 3, wn = warp >> 2;  // warp tile: tokens 32 wm.., experts 32 wn..
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(rsm));
    auto a_row = [&](int st, int r) { return sbase + (st * (kRgBM + kRgBN) + r) * kRgRow; };
    auto b_row = [&](int st, int r) { return sbase + (st * (kRgBM + kRgBN) + kRgBM + r) * kRgRow; };
    const int nk = H / kRgBK;

    auto issue = [&](int kt) {
        if (kt < nk) {
            const int st = kt % kRgStages;
            // 128 token rows + 64 expert rows, 8 x 16 bytes each: 1536 chunks over 256 threads
            for (int c = tid; c < (kRgBM + kRgBN) * 8; c += 256) {
                const int r = c >> 3, j = c & 7;
                if (r < kRgBM) {
                    const int t = t0 + r;
                    cp_async16_zfill(a_row(st, r) + j * 16,
                                     x + (size_t)(t < T ? t : 0) * H + kt * kRgBK + j * 8, t < T);
                } else {
                    const int e = e0 + r - kRgBM;
                    cp_async16_zfill(b_row(st, r - kRgBM) + j * 16,
                                     wr + (size_t)(e < E ? e : 0) * H + kt * kRgBK + j * 8, e < E);
                }
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    float acc[2][4][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[i][j][c] = 0.f;

#pragma unroll
    for (int kt = 0; kt < kRgStages - 1; ++kt) issue(kt);
    for (int kt = 0; kt < nk; ++kt) {
        issue(kt + kRgStages - 1);
        asm volatile("cp.async.wait_group %0;" ::"n"(kRgStages - 1) : "memory");
        __syncthreads();
        const int st = kt % kRgStages;
#pragma unroll
        for (int kk = 0; kk < kRgBK; kk += 16) {
            uint32_t a[2][4], b[4][2];
#pragma unroll
            for (int i = 0; i < 2; ++i)  // 16 tokens x 16 k per fragment
                ldmatrix_x4(a_row(st, wm * 32 + i * 16 + (lane & 15)) + (kk + (lane >> 4) * 8) * 2,
                            a[i][0], a[i][1], a[i][2], a[i][3]);
#pragma unroll
            for (int j = 0; j < 4; j += 2) {  // two 8-expert tiles per ldmatrix.x4
                const int r = wn * 32 + j * 8 + (lane & 7) + ((lane >> 4) << 3);
                ldmatrix_x4(b_row(st, r) + (kk + ((lane >> 3) & 1) * 8) * 2, b[j][0], b[j][1],
                            b[j + 1][0], b[j + 1][1]);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_bf16_16816(acc[i][j], a[i][0], a[i][1], a[i][2], a[i][3], b[j][0], b[j][1]);
        }
        __syncthreads();  // the stage is refilled by the next iteration's copies
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int t = t0 + wm * 32 + i * 16 + g + ((c & 2) ? 8 : 0);
                const int e = e0 + wn * 32 + j * 8 + 2 * q + (c & 1);
                if (t < T && e < E) logits[(size_t)t * E + e] = acc[i][j][c];
            }
}

// ------------------------------------------------------------------------------------------
// Top-K over fp32 logits: one warp per token; lane l holds experts l, l+32, ... (EPL of them).
// Each expert gets a 64-bit key (order-preserving bits of its selection score, then the
// complemented index), so one warp max per round picks the highest score with ties to the
// lower index.  Non-finite logits get score -inf and weight 0.
// ------------------------------------------------------------------------------------------
// score of the sigmoid-style routers
template <int EPL>
__global__ void __launch_bounds__(256)
topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
            int scoring, int renorm, float scaling, int32_t* __restrict__ ids,
            float* __restrict__ wout, int32_t* __restrict__ status) {
    pdl_wait();  // logits come from the router kernel
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    if (t >= T) return;
    const float* row = logits + (size_t)t * E;
    int my_e;
    float my_w;
    const bool nonfinite = warp_topk<EPL>([&](int e) { return row[e]; }, bias, E, k, scoring,
                                          renorm, scaling, lane, my_e, my_w);
    if (nonfinite && lane == 0) status_or(status, MOE_DEV_NONFINITE);
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_e;
        wout[(size_t)t * k + lane] = my_w;
    }
}

// ------------------------------------------------------------------------------------------
// Hash routing: ids = tid2eid[token_ids[t]] (table order).  One warp per token, lane j < k
// holds pair j.  Weights: scaling / k; or, with router logits (the hash layers of the family
// that also routes by sqrt(softplus) scores), s_j = sqrt(softplus(logit[t][id_j])),
// renormalised over the token's kept pairs when asked, times scaling.  A bad table entry or
// token id drops the pair (id -1, weight 0); a non-finite logit gives weight 0.
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
hash_route_kernel(const int64_t* __restrict__ tid2eid, const int32_t* __restrict__ token_ids,
                  int64_t vocab, int T, int E, int k, float scaling,
                  const float* __restrict__ logits, int renorm, int32_t* __restrict__ ids,
                  float* __restrict__ wout, int32_t* __restrict__ status) {
    pdl_wait();  // token ids (and the logits) may come from the preceding kernel
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int64_t tok = token_ids[t];
    const bool tok_ok = tok >= 0 && tok < vocab;
    if (!tok_ok && lane == 0) status_or(status, MOE_DEV_BAD_TOKEN_ID);
    int32_t e = -1;
    float w = 0.f;
    if (lane < k && tok_ok) {
        const int64_t te = tid2eid[tok * k + lane];
        if (te < 0 || te >= E) {
            status_or(status, MOE_DEV_BAD_EXPERT_ID);
        } else {
            e = (int32_t)te;
            w = 1.f;
            if (logits) {
                const float l = logits[(size_t)t * E + e];
                if (isfinite(l)) {
                    w = gate_score(MOE_SCORE_SQRTSOFTPLUS, l);
                } else {
                    w = 0.f;
                    status_or(status, MOE_DEV_NONFINITE);
                }
            }
        }
    }
    if (logits) {
        float den = 1.f;
        if (renorm) {
            den = w;
#pragma unroll
            for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        }
        w = den > 0.f ? w / den * scaling : 0.f;
    } else {
        w *= scaling / (float)k;
    }
    if (lane < k) {
        ids[(size_t)t * k + lane] = e;
        wout[(size_t)t * k + lane] = w;
    }
}

// ------------------------------------------------------------------------------------------
cudaError_t launch_router_logits(const void* x, const void* wr, float* logits, int T, int E,
                                 int H, cudaStream_t st) {
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* wb = static_cast<const __nv_bfloat16*>(wr);
    if (T <= 8) {
        return launch_pdl(router_logits_kernel<1, 16>, dim3((E + 15) / 16, (T + 7) / 8),
                          dim3(16 * 32), st, xb, wb, logits, T, E, H);
    }
    if (H % kRgBK == 0) {
        cudaError_t err = cudaFuncSetAttribute(router_gemm_tiled_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kRgSmem);
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((T + kRgBM - 1) / kRgBM, (E + kRgBN - 1) / kRgBN);
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = kRgSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, router_gemm_tiled_kernel, xb, wb, logits, T, E, H);
    }
    return launch_pdl(router_logits_kernel<4, 8>, dim3((E + 15) / 16, (T + 31) / 32),
                      dim3(8 * 32), st, xb, wb, logits, T, E, H);
}

template <int EPL>
static cudaError_t launch_topk_epl(const float* logits, const float* bias, int T, int E, int k,
                                   int scoring, int renorm, float scaling, int32_t* ids, float* w,
                                   int32_t* status, cudaStream_t st) {
    const int warps = T < 8 ? T : 8;
    return launch_pdl(topk_kernel<EPL>, dim3((T + warps - 1) / warps), dim3(32 * warps), st,
                      logits, bias, T, E, k, scoring, renorm, scaling, ids, w, status);
}

cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int scoring,
                        int renorm, float scaling, int32_t* ids, float* w, int32_t* status,
                        cudaStream_t st) {
    if (E <= 32) return launch_topk_epl<1>(logits, bias, T, E, k, scoring, renorm, scaling, ids, w, status, st);
    if (E <= 64) return launch_topk_epl<2>(logits, bias, T, E, k, scoring, renorm, scaling, ids, w, status, st);
    if (E <= 128) return launch_topk_epl<4>(logits, bias, T, E, k, scoring, renorm, scaling, ids, w, status, st);
    if (E <= 256) return launch_topk_epl<8>(logits, bias, T, E, k, scoring, renorm, scaling, ids, w, status, st);
    return launch_topk_epl<16>(logits, bias, T, E, k, scoring, renorm, scaling, ids, w, status, st);
}

cudaError_t launch_hash_route(const int64_t* tid2eid, const int32_t* token_ids, int64_t vocab,
                              int T, int E, int k, float scaling, const float* logits, int renorm,
                              int32_t* ids, float* w, int32_t* status, cudaStream_t st) {
    const int warps = T < 8 ? T : 8;
    return launch_pdl(hash_route_kernel, dim3((T + warps - 1) / warps), dim3(32 * warps), st,
                      tid2eid, token_ids, vocab, T, E, k, scaling, logits, renorm, ids, w, status);
}

}  // namespace moe
