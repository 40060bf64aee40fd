// decode.cu -- the expert FFN for a few tokens (T <= 8 and T * top_k <= 64, bf16
// activations): two launches.
//
//   dec_gateup_kernel   every CTA rebuilds the dispatch (which experts received tokens, in
//                       ascending id order, and which tokens each one received) from the
//                       routing ids in shared memory -- no separate sort launch -- then one
//                       CTA computes 32 (or 16) gate and up rows of one expert for all its
//                       tokens, with K split over warps and reduced through shared memory;
//                       writes h = SiLU(gate) * up token-major: hT[slot][token][I] (f16).
//   dec_down_kernel     the down projection fused with the top-K weighted sum and the shared
//                       expert: the MMA columns are the T tokens and the sum runs over
//                       (expert, I).  Each warp walks a subset of the active experts; per
//                       expert it accumulates W_down . h in fp32 and adds it scaled by that
//                       expert's per-tensor post-scale and each token's routing weight, so no
//                       per-pair outputs reach memory.  Warps are reduced through shared
//                       memory in a fixed order and bf16 rows are written directly.
//
// This is the "gate+up, silu+down in two fused launches" structure of the spark_model MoE
// module doc (moe/mod.rs), with the weighted sum (init.rs `moe_weighted_sum_blend`) folded
// into the second launch.  Both kernels are launched with programmatic dependent launch so
// their CTAs are resident when the producer finishes.
#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace moe {

constexpr int kDecMaxT = 8;
constexpr int kDecMaxSlots = 65;  // at most 64 routed pairs (T * top_k <= 64) + the shared expert

// Dispatch of T <= 8 tokens, rebuilt by every CTA from ids/w.
struct DecDispatch {
    uint32_t bitmap[kMaxExperts / 32];
    int n_active;                 // routed experts with >= 1 token
    int expert[kDecMaxSlots];     // slot -> expert id (ascending), shared slot -> 0
    uint32_t tokmask[kDecMaxSlots];
    float w[kDecMaxSlots][kDecMaxT];
};

__device__ __forceinline__ void dec_dispatch(const FfnLaunch& L, DecDispatch& D) {
    const int tid = threadIdx.x;
    const int P = L.T * L.k;
    for (int i = tid; i < kMaxExperts / 32; i += blockDim.x) D.bitmap[i] = 0;
    for (int i = tid; i < kDecMaxSlots; i += blockDim.x) {
        D.tokmask[i] = 0;
        for (int t = 0; t < kDecMaxT; ++t) D.w[i][t] = 0.f;
    }
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = L.ids[p];
        if (e >= 0 && e < L.E) atomicOr(&D.bitmap[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    // slot of expert e = number of set bits below e
    __shared__ int s_base[kMaxExperts / 32 + 1];
    if (tid == 0) {
        int b = 0;
        for (int i = 0; i < kMaxExperts / 32; ++i) { s_base[i] = b; b += __popc(D.bitmap[i]); }
        s_base[kMaxExperts / 32] = b;
        D.n_active = b;
    }
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = L.ids[p];
        if (e >= 0 && e < L.E) {
            const int slot = s_base[e >> 5] + __popc(D.bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
            const int t = p / L.k;
            D.expert[slot] = e;
            atomicOr(&D.tokmask[slot], 1u << t);
            atomicAdd(&D.w[slot][t], L.w[p]);  // a table may route a token to an expert twice
        }
    }
    if (L.I_shared > 0 && tid == 0) {
        const int s = s_base[kMaxExperts / 32];
        D.expert[s] = 0;
        D.tokmask[s] = (1u << L.T) - 1u;
        for (int t = 0; t < L.T; ++t) D.w[s][t] = 1.f;
    }
    __syncthreads();
}

// bf16x2 -> f16x2 (via fp32; exact for |x| >= 2^-14)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack_half2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// ------------------------------------------------------------------------------------------
// gate+up: CTA = ROWS16 row tiles of 16 (gate and up) x KSPLIT warps over K.
// ------------------------------------------------------------------------------------------
template <int FMT, int KSPLIT>
__device__ __forceinline__ void dec_gateup_rows(const FfnLaunch& L, const DecDispatch& D, int slot,
                                                bool shared, __half* hT) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int e = D.expert[slot];
    const uint32_t mask = D.tokmask[slot];
    const ProjView& PG = shared ? L.sh_gate : L.gate;
    const ProjView& PU = shared ? L.sh_up : L.up;
    const int N = shared ? L.I_shared : L.I;
    const int K = L.H;
    const int ks = warp % KSPLIT, rg = warp / KSPLIT;
    constexpr int RG = 8 / KSPLIT;  // row tiles per CTA
    const int n0 = (blockIdx.x * RG + rg) * 16;
    const int sv = FMT == MOE_FMT_NVFP4 ? 16 : 32;
    const int steps = K / 128;
    const int per = (steps + KSPLIT - 1) / KSPLIT;
    const int s0 = ks * per, s1 = min(steps, s0 + per);
    const bool rows_ok = n0 < N;

    // column g <-> the g-th token of this expert (ascending token index)
    int tok = -1;
    {
        uint32_t m = mask;
        for (int c = 0; c < g && m; ++c) m &= m - 1;
        if (m) tok = __ffs(m) - 1;
    }
    const __nv_bfloat16* xrow =
        static_cast<const __nv_bfloat16*>(L.x) + (size_t)(tok >= 0 ? tok : 0) * K + 32 * q;

    float accG[4] = {0.f, 0.f, 0.f, 0.f}, accU[4] = {0.f, 0.f, 0.f, 0.f};
    if (rows_ok) {
        const size_t rowA = (size_t)e * N + n0 + g;
        const uint8_t* pg0 = PG.packed + rowA * (K / 2) + 16 * q;
        const uint8_t* pg1 = pg0 + (size_t)8 * (K / 2);
        const uint8_t* sg0 = PG.scales + rowA * (K / sv);
        const uint8_t* sg1 = sg0 + (size_t)8 * (K / sv);
        const uint8_t* pu0 = PU.packed + rowA * (K / 2) + 16 * q;
        const uint8_t* pu1 = pu0 + (size_t)8 * (K / 2);
        const uint8_t* su0 = PU.scales + rowA * (K / sv);
        const uint8_t* su1 = su0 + (size_t)8 * (K / sv);
        const int mxg = FMT == MOE_FMT_MXFP4 ? 112 + PG.mx_off[e] : 0;
        const int mxu = FMT == MOE_FMT_MXFP4 ? 112 + PU.mx_off[e] : 0;
        ChunkA cg, cu;
        if (s0 < s1) {
            load_chunk<FMT>(cg, pg0, pg1, sg0, sg1, s0, q, mxg);
            load_chunk<FMT>(cu, pu0, pu1, su0, su1, s0, q, mxu);
        }
        for (int s = s0; s < s1; ++s) {
            ChunkA ng = cg, nu = cu;
            if (s + 1 < s1) {
                load_chunk<FMT>(ng, pg0, pg1, sg0, sg1, s + 1, q, mxg);
                load_chunk<FMT>(nu, pu0, pu1, su0, su1, s + 1, q, mxu);
            }
            // the lane's 32 token elements as f16x2 pairs (16 registers)
            uint32_t bx[16];
            {
                const uint4 r0 = tok >= 0 ? ldg_cached128(xrow + s * 128 + 0) : make_uint4(0, 0, 0, 0);
                const uint4 r1 = tok >= 0 ? ldg_cached128(xrow + s * 128 + 8) : make_uint4(0, 0, 0, 0);
                const uint4 r2 = tok >= 0 ? ldg_cached128(xrow + s * 128 + 16) : make_uint4(0, 0, 0, 0);
                const uint4 r3 = tok >= 0 ? ldg_cached128(xrow + s * 128 + 24) : make_uint4(0, 0, 0, 0);
                const uint32_t w[16] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w,
                                        r2.x, r2.y, r2.z, r2.w, r3.x, r3.y, r3.z, r3.w};
#pragma unroll
                for (int i = 0; i < 16; ++i) bx[i] = bf16x2_to_f16x2(w[i]);
            }
#define DEC_STEP(I)                                                         \
    {                                                                       \
        uint32_t fa[4], fb[4];                                              \
        frag_a<I>(cg, fa);                                                  \
        frag_a<I>(cu, fb);                                                  \
        mma_f16_16816(accG, fa[0], fa[1], fa[2], fa[3], bx[2 * I], bx[2 * I + 1]); \
        mma_f16_16816(accU, fb[0], fb[1], fb[2], fb[3], bx[2 * I], bx[2 * I + 1]); \
    }
            DEC_STEP(0) DEC_STEP(1) DEC_STEP(2) DEC_STEP(3)
            DEC_STEP(4) DEC_STEP(5) DEC_STEP(6) DEC_STEP(7)
#undef DEC_STEP
            cg = ng;
            cu = nu;
        }
    }
    // reduce the KSPLIT partial sums of each row tile through shared memory
    __shared__ float red[8][8][32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        red[warp][i][lane] = accG[i];
        red[warp][4 + i][lane] = accU[i];
    }
    __syncthreads();
    if (ks == 0 && rows_ok) {
        float G[4] = {0.f, 0.f, 0.f, 0.f}, U[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < KSPLIT; ++w) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                G[i] += red[rg * KSPLIT + w][i][lane];
                U[i] += red[rg * KSPLIT + w][4 + i][lane];
            }
        }
        const float pg = PG.post[e], pu = PU.post[e];
        const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = 2 * q + j;  // column -> c-th token of this expert
            uint32_t m = mask;
            for (int cc = 0; cc < c && m; ++cc) m &= m - 1;
            if (!m) continue;
            const int t = __ffs(m) - 1;
            __half* hrow = hT + ((size_t)slot * kDecMaxT + t) * Imax + n0;
            hrow[g] = __float2half_rn(silu_f32(G[j] * pg) * (U[j] * pu));
            hrow[g + 8] = __float2half_rn(silu_f32(G[2 + j] * pg) * (U[2 + j] * pu));
        }
    }
}

template <int FMT_R, int FMT_S, int KSPLIT>
__global__ void __launch_bounds__(256) dec_gateup_kernel(FfnLaunch L) {
    __shared__ DecDispatch D;
    pdl_wait();  // ids / w come from the routing kernels
    dec_dispatch(L, D);
    const int slot = blockIdx.y;
    const bool shared = L.I_shared > 0 && slot == D.n_active;
    if (slot > D.n_active || (slot == D.n_active && !shared)) return;
    if (shared) dec_gateup_rows<FMT_S, KSPLIT>(L, D, slot, true, L.h16);
    else dec_gateup_rows<FMT_R, KSPLIT>(L, D, slot, false, L.h16);
    pdl_trigger();
}

// ------------------------------------------------------------------------------------------
// down + weighted sum + shared expert: CTA = 16 output rows, 8 warps over the active slots.
// ------------------------------------------------------------------------------------------
template <int FMT>
__device__ __forceinline__ void dec_down_slot(const FfnLaunch& L, const DecDispatch& D, int slot,
                                              bool shared, int n0, float (&acc)[4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int e = D.expert[slot];
    const uint32_t mask = D.tokmask[slot];
    const ProjView& PD = shared ? L.sh_down : L.down;
    const int K = shared ? L.I_shared : L.I;
    const int N = L.H;
    const int sv = FMT == MOE_FMT_NVFP4 ? 16 : 32;
    const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
    const size_t rowA = (size_t)e * N + n0 + g;
    const uint8_t* p0 = PD.packed + rowA * (K / 2) + 16 * q;
    const uint8_t* p1 = p0 + (size_t)8 * (K / 2);
    const uint8_t* s0p = PD.scales + rowA * (K / sv);
    const uint8_t* s1p = s0p + (size_t)8 * (K / sv);
    const int mx = FMT == MOE_FMT_MXFP4 ? 112 + PD.mx_off[e] : 0;
    const bool tok_ok = (mask >> g) & 1u;  // column g = token g
    const __half* hrow = L.h16 + ((size_t)slot * kDecMaxT + g) * Imax + 32 * q;
    float part[4] = {0.f, 0.f, 0.f, 0.f};
    const int steps = K / 128;
    ChunkA c;
    load_chunk<FMT>(c, p0, p1, s0p, s1p, 0, q, mx);
    for (int s = 0; s < steps; ++s) {
        ChunkA n = c;
        if (s + 1 < steps) load_chunk<FMT>(n, p0, p1, s0p, s1p, s + 1, q, mx);
        uint4 b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            b[j] = tok_ok ? ldg_cached128(hrow + s * 128 + 8 * j) : make_uint4(0, 0, 0, 0);
#define DOWN_STEP(I)                                                            \
    {                                                                           \
        uint32_t fa[4];                                                         \
        frag_a<I>(c, fa);                                                       \
        mma_f16_16816(part, fa[0], fa[1], fa[2], fa[3], word_of(b[I >> 1], (I & 1) * 2), \
                      word_of(b[I >> 1], (I & 1) * 2 + 1));                     \
    }
        DOWN_STEP(0) DOWN_STEP(1) DOWN_STEP(2) DOWN_STEP(3)
        DOWN_STEP(4) DOWN_STEP(5) DOWN_STEP(6) DOWN_STEP(7)
#undef DOWN_STEP
        c = n;
    }
    const float post = PD.post[e];
    // accumulator columns 2q, 2q+1 are tokens 2q, 2q+1
    const float w0 = D.w[slot][2 * q] * post, w1 = D.w[slot][2 * q + 1] * post;
    acc[0] += part[0] * w0;
    acc[1] += part[1] * w1;
    acc[2] += part[2] * w0;
    acc[3] += part[3] * w1;
}

template <int FMT_R, int FMT_S>
__global__ void __launch_bounds__(256) dec_down_kernel(FfnLaunch L) {
    __shared__ DecDispatch D;
    __shared__ float red[8][4][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    pdl_wait();  // h comes from the gate+up kernel
    dec_dispatch(L, D);
    const int n0 = blockIdx.x * 16;
    const int nslots = D.n_active + (L.I_shared > 0 ? 1 : 0);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int slot = warp; slot < nslots; slot += 8) {
        const bool shared = slot == D.n_active;
        if (shared) dec_down_slot<FMT_S>(L, D, slot, true, n0, acc);
        else dec_down_slot<FMT_R>(L, D, slot, false, n0, acc);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) red[warp][i][lane] = acc[i];
    __syncthreads();
    pdl_trigger();
    if (warp == 0) {
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < 8; ++w)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] += red[w][i][lane];
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(L.out);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int t = 2 * q + j;
            if (t < L.T) {
                out[(size_t)t * L.H + n0 + g] = __float2bfloat16_rn(o[j]);
                out[(size_t)t * L.H + n0 + g + 8] = __float2bfloat16_rn(o[2 + j]);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
template <int FR, int FS>
static cudaError_t launch_decode_fmt(const FfnLaunch& L, int phase, cudaStream_t st) {
    const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
    const int slots = (L.E < L.T * L.k ? L.E : L.T * L.k) + (L.I_shared > 0 ? 1 : 0);
    if (phase == 1) {
        if (L.H <= 2048) {  // short K: 8-way split, one row tile per CTA
            return launch_pdl(dec_gateup_kernel<FR, FS, 8>, dim3(Imax / 16, slots), dim3(256), st, L);
        }
        return launch_pdl(dec_gateup_kernel<FR, FS, 4>, dim3(Imax / 32, slots), dim3(256), st, L);
    }
    return launch_pdl(dec_down_kernel<FR, FS>, dim3(L.H / 16), dim3(256), st, L);
}

cudaError_t launch_decode_phase(const FfnLaunch& L, int phase, cudaStream_t st) {
    const int fr = L.gate.fmt;
    const int fs = L.I_shared > 0 ? L.sh_gate.fmt : fr;
    if (fr == MOE_FMT_NVFP4 && fs == MOE_FMT_NVFP4) return launch_decode_fmt<0, 0>(L, phase, st);
    if (fr == MOE_FMT_NVFP4 && fs == MOE_FMT_MXFP4) return launch_decode_fmt<0, 1>(L, phase, st);
    if (fr == MOE_FMT_MXFP4 && fs == MOE_FMT_NVFP4) return launch_decode_fmt<1, 0>(L, phase, st);
    return launch_decode_fmt<1, 1>(L, phase, st);
}

}  // namespace moe
