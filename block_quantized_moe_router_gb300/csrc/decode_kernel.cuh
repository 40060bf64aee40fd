// decode_kernel.cuh -- the whole MoE block for a few tokens (T <= 8, T * top_k <= 64, bf16
// activations) in ONE persistent cooperative launch, one CTA per SM.
//
//   phase 0  every CTA converts a slice of x to f16 and, when the router runs here, computes
//            the router logits of the experts e = cta, cta + G, ... (fp32 dot products on
//            the CUDA cores, the 8 warps splitting H).                 -> grid barrier 1
//   phase 1  every CTA selects the top-K of all T tokens itself (one warp per token), or
//            looks the experts up in the hash table, or reads the given ids; CTA 0 writes
//            the routing outputs.  Each CTA then derives the dispatch: the active experts in
//            ascending id order, each with its tokens and routing weights.
//   phase 2  gate+up: tasks (expert slot, 32 rows of I) dealt round-robin to the CTAs; the 8
//            warps split K = H, partial sums meet in shared memory and h = SiLU(g) * u is
//            written token-major to hT[slot][token][I] (f16).          -> grid barrier 2
//   phase 3  down fused with the top-K weighted sum and the shared expert: each CTA owns
//            16-row tiles of the output; its (tile, slot) pairs are dealt to its warps, each
//            folds W_down . h of a slot into its tile with the expert's post-scale and each
//            token's weight; warps are reduced in a fixed order and bf16 rows are written.
//
// Every warp streams its operands through its own ring of asynchronous copies, S - 1 stages
// ahead of the MMAs, in ONE sequence that runs from its first gate+up stage to its last down
// stage.  A gate+up stage is one 128-element K-step of 32 rows of gate and up (two MMA
// tiles sharing the activation chunk of the step); a down stage is two K-steps of 16 rows.
// A stage also holds the block scales and the activations (x in f16 for gate+up, h for
// down).  The activations take 256 B per token column and K-step, so a one-token launch
// has stages of 3 KiB instead of 6.5 KiB.  The down weights depend only on the routing, so they are already in flight while
// the CTA waits at barrier 2; the h chunks of the down stages issued before that barrier are
// copied right after it.
//
// This is the "gate + top-K fused, expert FFN in two fused stages" structure of the
// spark_model MoE module doc (moe/mod.rs) taken to a single launch, with the weighted sum
// (init.rs `moe_weighted_sum_blend`) folded into the down stage.  Grid barriers are bounded
// spins on a 64-bit arrival counter owned by the weights handle, next to an epoch word (the
// launches completed on the handle) that fixes each launch's targets; a wait that runs out sets
// MOE_DEV_TIMEOUT and the kernel carries on (its results are then invalid) instead of hanging.
#pragma once
#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

constexpr int kDecMaxT = 8;
constexpr int kDecMaxSlots = 65;   // at most 64 routed pairs (T * top_k <= 64) + the shared expert
constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
// the gate+up partial sums (double-buffered) and, after barrier 2, the down partial sums
// (one 16-row output tile per 4 KB) share one region
constexpr int kDecRedG = 2 * kDecWarps * 512 * 4;
// dynamic shared memory left for the eight rings: the opt-in maximum per block less the
// partial-sum region and the static DecShared block (< 6 KiB)
constexpr int kDecRingBudget = 232448 - kDecRedG - 6144;

// Ring geometry for TPS gate+up tiles per stage and activation chunks laid out for NTOK token
// columns (MMA column g <-> 64 B per lane, 16 B per lane and 8-element group c at
// c * NTOK * 64 + lane * 16, so one token takes 256 B per 128-element K-step).  512 B =
// 32 lanes x 16 B; MMA row g = lane / 4.
//   gate+up: [0, kGuAct)  codes, 512 B each of (tile t, matrix m, rows +8 r) at (4t + 2m + r)
//            [kGuAct, kGuSc) activation chunk, [kGuSc, +256 TPS) scales, 256 B per tile
//   down:    [0, kDnCodes) activation chunks of the two K-steps, kAct each
//            [kDnCodes, kDnSc) codes, 512 B each of (step u, rows +8 r) at (2u + r)
//            [kDnSc, +512) scales, 256 B per step
// Three stages per warp.  A one-token stage is 3 KiB, so seven would fit, but priming six of
// them per warp on every SM asks for most of a layer's weights in one burst and delays each
// warp's first stage: one token took 24.3 us per layer step with 7-stage rings, 23.5 with 5,
// 22.6 with 4 and 22.0 with 3.
template <int TPS, int NTOK>
struct DecGeom {
    static constexpr int kAct = NTOK * 256;
    static constexpr int kGuAct = TPS * 2048, kGuSc = kGuAct + kAct, kGuBytes = kGuSc + TPS * 256;
    static constexpr int kDnCodes = 2 * kAct, kDnSc = kDnCodes + 2048, kDnBytes = kDnSc + 512;
    static constexpr int kStageBytes = ((kGuBytes > kDnBytes ? kGuBytes : kDnBytes) + 127) / 128 * 128;
    static constexpr int kStages = 3;
    static constexpr int kRingBytes = kDecWarps * kStages * kStageBytes;
    static_assert(kRingBytes <= kDecRingBudget, "ring does not fit");
};
constexpr int kDecRedDTile = kDecWarps * 128 * 4;
constexpr int kDecMaxTilesPerCta = 4;
// router phase: experts handled together per CTA, 8-element chunks per thread and expert
constexpr int kDecRouterBatch = 4, kDecRouterChunks = 4;  // H <= 8 * 256 * 4 = 8192
constexpr long long kBarrierCycles = 4000000000ll;  // default wait limit: ~2 s at 2 GHz

// Dispatch of T <= 8 tokens, derived by every CTA from the routing ids / weights.
struct DecDispatch {
    uint32_t bitmap[kMaxExperts / 32];
    int base[kMaxExperts / 32];
    int n_active;                 // routed experts with >= 1 token
    int expert[kDecMaxSlots];     // slot -> expert id (ascending), shared slot -> 0
    uint32_t tokmask[kDecMaxSlots];
    float w[kDecMaxSlots][kDecMaxT];
    // per slot and projection (gate, up, down): the fp32 post-scale and, for MXFP4, the
    // exponent bias of the f16 block-scale conversion -- read once here instead of once per task
    float post[kDecMaxSlots][3];
    int mxb[kDecMaxSlots][3];
};

struct DecShared {
    DecDispatch D;
    int32_t ids[64];
    float w[64];
    float zw[kDecMaxT];  // per token: summed weight of its zero-computation experts
    float red_router[4][kDecWarps][kDecMaxT];
    float sh_post[3];    // the shared expert's post-scales and MXFP4 biases (gate, up, down)
    int sh_mxb[3];
};

// ---- small helpers ---------------------------------------------------------------------------
// L2-only load: for data written earlier in this launch by other CTAs.
__device__ __forceinline__ float ld_cg_f32(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// bf16x2 -> f16x2 (via fp32; exact for |x| >= 2^-14)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack_half2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// the g-th set bit of mask (ascending), or -1
__device__ __forceinline__ int nth_bit(uint32_t mask, int g) {
    for (int c = 0; c < g && mask; ++c) mask &= mask - 1;
    return mask ? __ffs(mask) - 1 : -1;
}

// Grid-wide barrier of a cooperative launch.  bar[0] counts arrivals and is never reset;
// bar[1] counts the launches completed on it, so a launch starts with bar[0] = 2 G bar[1] and
// its two barriers complete at 2 G bar[1] + G and + 2 G (`target`, known to thread 0 of every
// block from the start).  Thread 0 arrives with a release add that needs no reply and polls
// with acquire loads.  The wait is bounded: after `limit` SM cycles it sets MOE_DEV_TIMEOUT and
// returns.
__device__ __forceinline__ void grid_barrier(unsigned long long* bar, unsigned long long target,
                                             int32_t* status, long long limit) {
    __syncthreads();
    if (threadIdx.x == 0) {
        red_release_add_u64(bar, 1ull);
        const long long t0 = clock64();
        bool done = ld_acquire_u64(bar) >= target;
        int spins = 0;
        while (!done) {
            if (++spins > 64) __nanosleep(64);
            done = ld_acquire_u64(bar) >= target;
            if (!done && clock64() - t0 > limit) break;
        }
        if (!done) status_or(status, MOE_DEV_TIMEOUT);
    }
    __syncthreads();
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// ---- phase 1: dispatch from the routing ids / weights in shared memory --------------------------
__device__ __forceinline__ void dec_dispatch(int T, int k, int E, int I_shared, const int32_t* ids,
                                             const float* wts, DecDispatch& D) {
    const int tid = threadIdx.x;
    for (int i = tid; i < kMaxExperts / 32; i += blockDim.x) D.bitmap[i] = 0;
    for (int i = tid; i < kDecMaxSlots * (kDecMaxT + 1); i += blockDim.x) {
        if (i < kDecMaxSlots) D.tokmask[i] = 0;
        else (&D.w[0][0])[i - kDecMaxSlots] = 0.f;
    }
    __syncthreads();
    if (tid < 32) {  // one warp: at most 64 pairs, two per lane
        const int lane = tid, P = T * k;
        const int e0 = lane < P ? ids[lane] : -1, e1 = lane + 32 < P ? ids[lane + 32] : -1;
        const float w0 = lane < P ? wts[lane] : 0.f, w1 = lane + 32 < P ? wts[lane + 32] : 0.f;
        if (e0 >= 0 && e0 < E) atomicOr(&D.bitmap[e0 >> 5], 1u << (e0 & 31));
        if (e1 >= 0 && e1 < E) atomicOr(&D.bitmap[e1 >> 5], 1u << (e1 & 31));
        __syncwarp();
        const int cnt = lane < kMaxExperts / 32 ? __popc(D.bitmap[lane]) : 0;
        int inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane < kMaxExperts / 32) D.base[lane] = inc - cnt;
        const int n_active = __shfl_sync(0xffffffffu, inc, 31);
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = h ? e1 : e0;
            const int p = lane + 32 * h;
            if (e >= 0 && e < E) {
                const int slot = D.base[e >> 5] + __popc(D.bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
                const int t = p / k;
                D.expert[slot] = e;
                atomicOr(&D.tokmask[slot], 1u << t);
                atomicAdd(&D.w[slot][t], h ? w1 : w0);  // a table may route a token to an expert twice
            }
        }
        if (lane == 0) {
            D.n_active = n_active;
            if (I_shared > 0) {
                D.expert[n_active] = 0;
                D.tokmask[n_active] = (1u << T) - 1u;
                for (int t = 0; t < T; ++t) D.w[n_active][t] = 1.f;
            }
        }
    }
    __syncthreads();
}

// ---- the MMAs of one ring stage ---------------------------------------------------------------
// gate+up: one K-step of 16 * TPS rows (tiles t < TPS) of gate and up; B = x in f16.
// acc[t][m][p]: tile t, matrix m (gate, up), MMA chain p (even / odd sub-steps).
template <int FMT, int TPS, int NTOK>
__device__ __forceinline__ void gu_stage(const uint8_t* st, bool has_tok, int lane, int g, int q,
                                         int mxg, int mxu, float (&acc)[2][2][2][4]) {
    using Geo = DecGeom<TPS, NTOK>;
    uint4 bx[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        bx[c] = has_tok ? *reinterpret_cast<const uint4*>(st + Geo::kGuAct + c * NTOK * 64 + lane * 16)
                        : make_uint4(0, 0, 0, 0);
    ChunkA cw[TPS][2];
#pragma unroll
    for (int t = 0; t < TPS; ++t) {
        const uint2* sc = reinterpret_cast<const uint2*>(st + Geo::kGuSc + t * 256);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            cw[t][m].r0 = *reinterpret_cast<const uint4*>(st + (4 * t + 2 * m) * 512 + lane * 16);
            cw[t][m].r1 = *reinterpret_cast<const uint4*>(st + (4 * t + 2 * m + 1) * 512 + lane * 16);
            scales_from_raw<FMT>(sc[g * 4 + 2 * m], q, m ? mxu : mxg, cw[t][m].s0lo, cw[t][m].s0hi);
            scales_from_raw<FMT>(sc[g * 4 + 2 * m + 1], q, m ? mxu : mxg, cw[t][m].s1lo, cw[t][m].s1hi);
        }
    }
    __syncwarp();  // every lane has read the stage before it is refilled
#define DEC_GU(I)                                                                        \
    {                                                                                    \
        const uint32_t b0 = word_of(bx[I >> 1], (I & 1) * 2);                            \
        const uint32_t b1 = word_of(bx[I >> 1], (I & 1) * 2 + 1);                        \
        _Pragma("unroll") for (int t = 0; t < TPS; ++t)                                  \
        _Pragma("unroll") for (int m = 0; m < 2; ++m) {                                  \
            uint32_t fa[4];                                                              \
            frag_a<I>(cw[t][m], fa);                                                     \
            mma_f16_16816(acc[t][m][I & 1], fa[0], fa[1], fa[2], fa[3], b0, b1);         \
        }                                                                                \
    }
    DEC_GU(0) DEC_GU(1) DEC_GU(2) DEC_GU(3) DEC_GU(4) DEC_GU(5) DEC_GU(6) DEC_GU(7)
#undef DEC_GU
}

// down: U (1 or 2) K-steps of 16 rows of W_down; B = h in f16.  part[u][p]: step u, chain p.
template <int FMT, int U, int TPS, int NTOK>
__device__ __forceinline__ void dn_stage(const uint8_t* st, bool has_tok, int lane, int g, int q,
                                         int mx, float (&part)[2][2][4]) {
    using Geo = DecGeom<TPS, NTOK>;
    uint4 hb[U][4];
    ChunkA c[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            hb[u][j] = has_tok ? *reinterpret_cast<const uint4*>(st + u * Geo::kAct + j * NTOK * 64 + lane * 16)
                               : make_uint4(0, 0, 0, 0);
        c[u].r0 = *reinterpret_cast<const uint4*>(st + Geo::kDnCodes + (2 * u) * 512 + lane * 16);
        c[u].r1 = *reinterpret_cast<const uint4*>(st + Geo::kDnCodes + (2 * u + 1) * 512 + lane * 16);
        const uint2* sc = reinterpret_cast<const uint2*>(st + Geo::kDnSc + u * 256);
        scales_from_raw<FMT>(sc[g * 4 + 0], q, mx, c[u].s0lo, c[u].s0hi);
        scales_from_raw<FMT>(sc[g * 4 + 1], q, mx, c[u].s1lo, c[u].s1hi);
    }
    __syncwarp();
#define DEC_DN(I)                                                                          \
    _Pragma("unroll") for (int u = 0; u < U; ++u) {                                        \
        uint32_t fa[4];                                                                    \
        frag_a<I>(c[u], fa);                                                               \
        mma_f16_16816(part[u][I & 1], fa[0], fa[1], fa[2], fa[3],                          \
                      word_of(hb[u][I >> 1], (I & 1) * 2), word_of(hb[u][I >> 1], (I & 1) * 2 + 1)); \
    }
    DEC_DN(0) DEC_DN(1) DEC_DN(2) DEC_DN(3) DEC_DN(4) DEC_DN(5) DEC_DN(6) DEC_DN(7)
#undef DEC_DN
}

__device__ __forceinline__ float sum4(const float (&a)[2][2][4], int i) {
    return (a[0][0][i] + a[0][1][i]) + (a[1][0][i] + a[1][1][i]);
}

// ------------------------------------------------------------------------------------------
// TPS: MMA tiles (16 rows each) per gate+up ring stage -- 2, or 1 when a layer has too few
// 32-row tasks to give every CTA at least two.  NTOK: token columns the activation chunks
// are laid out for (T <= NTOK).
template <int FR, int FS, int TPS, int NTOK>
__global__ void __launch_bounds__(kDecThreads, 1)
dec_fused_kernel(FfnLaunch L, DecRoute R, unsigned long long* bar) {
    using Geo = DecGeom<TPS, NTOK>;
    constexpr int kStages = Geo::kStages, kStageBytes = Geo::kStageBytes;
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ DecShared S;
    DecDispatch& D = S.D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
    const int G = gridDim.x, cta = blockIdx.x;
    const int T = L.T, H = L.H, E = L.E, k = L.k;
    const int Er = L.E + L.Z;  // router outputs: real experts, then zero-computation experts
    const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
    const int tiles_out = H / 16;
    const int cnt_d = cta < tiles_out ? (tiles_out - cta + G - 1) / G : 0;
    float* red_g = reinterpret_cast<float*>(dsm + Geo::kRingBytes);
    float* red_d = red_g;  // reused for the down partial sums after barrier 2
    unsigned long long epoch = 0, bar_base = 0;  // this launch's barrier targets (thread 0)

    // ---- phase 0 ----------------------------------------------------------------------------
    // The post-scales (and MXFP4 exponent offsets) of the routed projections for ALL experts
    // go into the idle partial-sum region now, so that once the routing is known the per-slot
    // values come from shared memory instead of a dependent global round trip.
    float* tab_post = red_g;                                                    // [3][kMaxExperts]
    int32_t* tab_mx = reinterpret_cast<int32_t*>(red_g + 3 * kMaxExperts);     // [3][kMaxExperts]
    for (int i = tid; i < 3 * E; i += kDecThreads) {
        const int pj = i / E, e = i - pj * E;
        const ProjView& PV = pj == 0 ? L.gate : pj == 1 ? L.up : L.down;
        cp_async4(smem_addr(tab_post + pj * kMaxExperts + e), PV.post + e);
        if (PV.fmt == MOE_FMT_MXFP4) cp_async4(smem_addr(tab_mx + pj * kMaxExperts + e), PV.mx_off + e);
    }
    cp_async_commit();
    if (tid < 3 && L.I_shared > 0) {
        const ProjView& PV = tid == 0 ? L.sh_gate : tid == 1 ? L.sh_up : L.sh_down;
        S.sh_post[tid] = PV.post[0];
        S.sh_mxb[tid] = PV.fmt == MOE_FMT_MXFP4 ? 112 + PV.mx_off[0] : 0;
    }
    // Everything above reads only tables of the prepared weights.  The inputs, the barrier words
    // and the workspace may belong to the preceding kernel on the stream (a programmatic
    // launch: this grid may be scheduled before that kernel has finished).
    pdl_wait();
    pdl_trigger();
    if (tid == 0) {  // thread 0 of each block runs the barriers
        epoch = ld_acquire_u64(bar + 1);
        bar_base = 2ull * (unsigned long long)G * epoch;
    }
    {   // x -> f16 (this CTA's slice of the flat array)
        const int n8 = T * H / 8;
        const uint4* xs = static_cast<const uint4*>(L.x);
        uint4* xd = reinterpret_cast<uint4*>(L.x16);
        for (int c = cta * kDecThreads + tid; c < n8; c += G * kDecThreads) {
            const uint4 v = ldg_cached128(xs + c);
            xd[c] = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                               bf16x2_to_f16x2(v.w));
        }
    }
    if (R.mode == DEC_ROUTE_ROUTER && cta < Er) {
        // router logits of experts e = cta, cta + G, ...: x (bf16) is staged in the idle ring,
        // each thread loads its router chunks of all these experts before any arithmetic
        const int chunks = H / 8;
        const uint4* xs_smem = reinterpret_cast<const uint4*>(dsm);
        const uint4* xg = static_cast<const uint4*>(L.x);
        for (int c = tid; c < T * chunks; c += kDecThreads) cp_async16(smem_addr(dsm + 16 * c), xg + c);
        cp_async_commit();
        const uint4* wr = static_cast<const uint4*>(R.w_router);
        for (int e0 = cta; e0 < Er; e0 += kDecRouterBatch * G) {
            uint4 wv[kDecRouterBatch][kDecRouterChunks];
#pragma unroll
            for (int b = 0; b < kDecRouterBatch; ++b)
#pragma unroll
                for (int m = 0; m < kDecRouterChunks; ++m) {
                    const int e = e0 + b * G, c = tid + m * kDecThreads;
                    wv[b][m] = (e < Er && c < chunks) ? ldg_stream128(wr + (size_t)e * chunks + c)
                                                     : make_uint4(0, 0, 0, 0);
                }
            cp_async_wait<0>();
            __syncthreads();  // x is staged
            float acc[kDecRouterBatch][NTOK];
#pragma unroll
            for (int b = 0; b < kDecRouterBatch; ++b)
#pragma unroll
                for (int t = 0; t < NTOK; ++t) acc[b][t] = 0.f;
            const int nb = min(kDecRouterBatch, (Er - e0 + G - 1) / G);  // experts of this batch
#pragma unroll
            for (int m = 0; m < kDecRouterChunks; ++m) {
                const int c = tid + m * kDecThreads;
                if (c < chunks) {
                    float wf[kDecRouterBatch][8];
#pragma unroll
                    for (int b = 0; b < kDecRouterBatch; ++b) unpack_bf16x8(wv[b][m], wf[b]);
#pragma unroll
                    for (int t = 0; t < NTOK; ++t) {
                        if (t < T) {
                            float xf[8];
                            unpack_bf16x8(xs_smem[t * chunks + c], xf);
#pragma unroll
                            for (int b = 0; b < kDecRouterBatch; ++b) {
                                if (b < nb) {
#pragma unroll
                                    for (int i = 0; i < 8; ++i) acc[b][t] = fmaf(wf[b][i], xf[i], acc[b][t]);
                                }
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < kDecRouterBatch; ++b) {
                if (b < nb) {
#pragma unroll
                    for (int t = 0; t < NTOK; ++t)
                        if (t < T)
#pragma unroll
                            for (int o = 16; o; o >>= 1) acc[b][t] += __shfl_xor_sync(0xffffffffu, acc[b][t], o);
                    if (lane == 0)
#pragma unroll
                        for (int t = 0; t < NTOK; ++t) S.red_router[b][warp][t] = acc[b][t];
                }
            }
            __syncthreads();
            if (tid < kDecRouterBatch * kDecMaxT) {
                const int b = tid / kDecMaxT, t = tid - b * kDecMaxT, e = e0 + b * G;
                if (t < T && e < Er) {
                    float s = 0.f;
#pragma unroll
                    for (int w = 0; w < kDecWarps; ++w) s += S.red_router[b][w][t];
                    R.logits_out[(size_t)t * Er + e] = s;
                }
            }
        }
    }
    cp_async_wait<0>();           // the post-scale tables are in
    const long long wait_limit = L.wait_cycles ? (long long)L.wait_cycles : kBarrierCycles;
    grid_barrier(bar, bar_base + G, L.status, wait_limit);  // x16 and the logits are written

    // ---- phase 1: routing and dispatch ---------------------------------------------------------
    const int P = T * k;
    // one routed token: its warp builds the dispatch itself (the picks of a top-K are distinct)
    const bool fast1 = NTOK == 1 && !R.hash_ids && (R.mode == DEC_ROUTE_ROUTER || R.mode == DEC_ROUTE_LOGITS);
    if (R.hash_ids) {
        // ids from the table; weights scaling / k, or from the sqrt(softplus) router scores of
        // the table's experts (logits from phase 0 or given), renormalised per token
        float wv = 0.f;
        if (tid < P) {
            const int t = tid / k, j = tid - t * k;
            const int64_t tok = R.token_ids[t];
            int32_t e = -1;
            if (tok < 0 || tok >= R.vocab) {
                if (cta == 0) status_or(L.status, MOE_DEV_BAD_TOKEN_ID);
            } else {
                const int64_t te = R.tid2eid[tok * k + j];
                if (te < 0 || te >= Er) {
                    if (cta == 0) status_or(L.status, MOE_DEV_BAD_EXPERT_ID);
                } else {
                    e = (int32_t)te;
                    wv = 1.f;
                    if (R.mode != DEC_ROUTE_HASH) {
                        const float l = R.mode == DEC_ROUTE_ROUTER
                                            ? ld_cg_f32(R.logits_out + (size_t)t * Er + e)
                                            : R.logits_in[(size_t)t * Er + e];
                        if (isfinite(l)) {
                            wv = gate_score(MOE_SCORE_SQRTSOFTPLUS, l);
                        } else {
                            wv = 0.f;
                            if (cta == 0) status_or(L.status, MOE_DEV_NONFINITE);
                        }
                    }
                }
            }
            S.ids[tid] = e;
            S.w[tid] = wv;
        }
        __syncthreads();
        if (tid < P) {
            if (R.mode == DEC_ROUTE_HASH) {
                wv *= R.scaling / (float)k;
            } else {
                float den = 1.f;
                if (R.renorm) {
                    const int t0 = (tid / k) * k;
                    den = 0.f;
                    for (int j = 0; j < k; ++j) den += S.w[t0 + j];
                }
                wv = den > 0.f ? wv / den * R.scaling : 0.f;
            }
        }
        __syncthreads();
        if (tid < P) S.w[tid] = wv;
    } else if (R.mode == DEC_ROUTE_ROUTER || R.mode == DEC_ROUTE_LOGITS) {
        if (warp < T) {
            const bool in_launch = R.mode == DEC_ROUTE_ROUTER;
            const float* row = (in_launch ? R.logits_out : R.logits_in) + (size_t)warp * Er;
            int my_e;
            float my_w;
            auto load = [&](int e) { return in_launch ? ld_cg_f32(row + e) : row[e]; };
            bool nonfinite;
            if (Er <= 64)
                nonfinite = warp_topk<2>(load, R.bias, Er, k, R.scoring, R.renorm, R.scaling, lane, my_e, my_w);
            else if (Er <= 128)
                nonfinite = warp_topk<4>(load, R.bias, Er, k, R.scoring, R.renorm, R.scaling, lane, my_e, my_w);
            else if (Er <= 256)
                nonfinite = warp_topk<8>(load, R.bias, Er, k, R.scoring, R.renorm, R.scaling, lane, my_e, my_w);
            else
                nonfinite = warp_topk<16>(load, R.bias, Er, k, R.scoring, R.renorm, R.scaling, lane, my_e, my_w);
            if (nonfinite && lane == 0 && cta == 0) status_or(L.status, MOE_DEV_NONFINITE);
            if (fast1) {
                // the real experts among the picks become the slots, in ascending id order; the
                // zero-computation ones fold into one weight
                const bool real = lane < k && my_e < E;
                int rank = 0;
                for (int j = 0; j < k; ++j) {
                    const int ej = __shfl_sync(0xffffffffu, my_e, j);
                    rank += (ej < E && ej < my_e) ? 1 : 0;
                }
                const int n_act = __popc(__ballot_sync(0xffffffffu, real));
                float z = (lane < k && !real) ? my_w : 0.f;
#pragma unroll
                for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
                for (int i = lane; i < (k + 1) * (kDecMaxT - 1); i += 32)
                    D.w[i / (kDecMaxT - 1)][1 + i % (kDecMaxT - 1)] = 0.f;
                if (real) {
                    D.expert[rank] = my_e;
                    D.tokmask[rank] = 1u;
                    D.w[rank][0] = my_w;
#pragma unroll
                    for (int pj = 0; pj < 3; ++pj) {
                        const bool mx = (pj == 0 ? L.gate.fmt : pj == 1 ? L.up.fmt : L.down.fmt) == MOE_FMT_MXFP4;
                        D.post[rank][pj] = tab_post[pj * kMaxExperts + my_e];
                        D.mxb[rank][pj] = mx ? 112 + tab_mx[pj * kMaxExperts + my_e] : 0;
                    }
                }
                if (lane == 0) {
                    D.n_active = n_act;
                    S.zw[0] = z;
                    if (L.I_shared > 0) {
                        D.expert[n_act] = 0;
                        D.tokmask[n_act] = 1u;
                        D.w[n_act][0] = 1.f;
#pragma unroll
                        for (int pj = 0; pj < 3; ++pj) {
                            D.post[n_act][pj] = S.sh_post[pj];
                            D.mxb[n_act][pj] = S.sh_mxb[pj];
                        }
                    }
                }
                if (cta == 0 && lane < k) {
                    R.ids_out[lane] = my_e;
                    R.w_out[lane] = my_w;
                }
            } else if (lane < k) {
                S.ids[warp * k + lane] = my_e;
                S.w[warp * k + lane] = my_w;
            }
        }
    } else if (tid < P) {
        // given ids: anything but -1, a real expert or a zero-computation expert is dropped
        // (the dispatch ignores it) and flagged, as on the many-token paths
        const int32_t e = L.ids[tid];
        if (e != -1 && (e < 0 || e >= Er) && cta == 0) status_or(L.status, MOE_DEV_BAD_EXPERT_ID);
        S.ids[tid] = e;
        S.w[tid] = L.w[tid];
    }
    __syncthreads();
    if (!fast1) {
    if (R.mode != DEC_ROUTE_GIVEN && cta == 0 && tid < P) {
        R.ids_out[tid] = S.ids[tid];
        R.w_out[tid] = S.w[tid];
    }
    dec_dispatch(T, k, E, L.I_shared, S.ids, S.w, D);
    if (tid < kDecMaxT) {  // zero-computation experts: their weights fold into one per token
        float z = 0.f;
        for (int j = 0; tid < T && j < k; ++j) {
            const int e = S.ids[tid * k + j];
            if (e >= E && e < Er) z += S.w[tid * k + j];
        }
        S.zw[tid] = z;
    }
    {
        const int nsl = D.n_active + (L.I_shared > 0 ? 1 : 0);
        for (int i = tid; i < nsl * 3; i += kDecThreads) {
            const int slot = i / 3, pj = i - slot * 3;
            if (slot == D.n_active) {
                D.post[slot][pj] = S.sh_post[pj];
                D.mxb[slot][pj] = S.sh_mxb[pj];
            } else {
                const int e = D.expert[slot];
                const bool mx = (pj == 0 ? L.gate.fmt : pj == 1 ? L.up.fmt : L.down.fmt) == MOE_FMT_MXFP4;
                D.post[slot][pj] = tab_post[pj * kMaxExperts + e];
                D.mxb[slot][pj] = mx ? 112 + tab_mx[pj * kMaxExperts + e] : 0;
            }
        }
        __syncthreads();
    }
    }

    // ---- the work of this CTA and of this warp ----------------------------------------------------
    // gate+up: tasks (slot, 32 rows) dealt round-robin to the CTAs; in each task warp w takes the
    // K-steps w, w + 8, ..., so at any time the 8 warps read 512 contiguous bytes of every row.
    const int n_active = D.n_active;
    const bool has_shared = L.I_shared > 0;
    const int rows_t = 16 * TPS;
    const int tilesR = L.I / rows_t;
    const int ntasks = n_active * tilesR + (has_shared ? L.I_shared / rows_t : 0);
    const int cnt_g = cta < ntasks ? (ntasks - cta + G - 1) / G : 0;
    const int ksteps_g = H / 128;
    const int n_g = ksteps_g > warp ? (ksteps_g - warp + kDecWarps - 1) / kDecWarps : 0;
    const int done_g = n_g > 0 ? cnt_g * n_g : 0;  // gate+up stages of this warp
    // down: 16-row output tiles dealt round-robin to the CTAs; the CTA's (tile, slot) pairs are
    // dealt to its warps (warp w takes pairs w, w + 8, ...), each streams the whole K of a pair,
    // two K-steps per stage.  Slots are visited in an order rotated by the CTA index so that
    // the CTAs read different experts at any one time.
    const int nslots = n_active + (has_shared ? 1 : 0);
    const int npairs = cnt_d * nslots;

    auto task_of = [&](int j, int& slot, int& n0) {  // task j of this CTA -> (slot, first row)
        const int tau = cta + j * G;
        if (tau < n_active * tilesR) {
            slot = tau / tilesR;
            n0 = (tau - slot * tilesR) * rows_t;
        } else {
            slot = n_active;
            n0 = (tau - n_active * tilesR) * rows_t;
        }
    };
    auto pair_of = [&](int p, int& tl, int& slot) {  // pair p of this CTA -> (tile, slot)
        tl = p / nslots;
        slot = (p - tl * nslots + cta) % nslots;
    };
    // activation chunk of a lane: x (task j) / h (slot), at K-step 0
    auto x_src = [&](int j) -> const __half* {
        int slot, n0;
        task_of(j, slot, n0);
        const int tok = nth_bit(D.tokmask[slot], g);  // MMA column g <-> the g-th token of the slot
        return tok < 0 ? nullptr : L.x16 + (size_t)tok * H + 32 * q;
    };
    auto h_src = [&](int slot) -> const __half* {
        const bool ok = (D.tokmask[slot] >> g) & 1u;  // MMA column g = token g
        return ok ? L.h16 + ((size_t)slot * kDecMaxT + g) * Imax + 32 * q : nullptr;
    };
    auto copy_act = [&](uint32_t dst, const __half* a) {  // 64 B of activations of this lane
        if (a) {
#pragma unroll
            for (int c = 0; c < 4; ++c) cp_async16(dst + c * NTOK * 64 + lane * 16, a + 8 * c);
        }
    };

    // ---- the ring: one flat issue sequence per warp ------------------------------------------------
    uint8_t* ring = dsm + warp * kStages * kStageBytes;
    const uint32_t rbase = smem_addr(ring);
    int ic_phase = done_g > 0 ? 0 : 1;
    // gate+up: task, K-step; down: pair, first K-step of the stage
    int ic_j = ic_phase == 0 ? 0 : warp, ic_s = ic_phase == 0 ? warp : 0, ic_ns = 0;
    int ic_sfb = 8;
    size_t ic_rs = 0;      // row stride of the scales (bytes)
    bool h_ready = false;  // h may be copied only after barrier 2
    const uint8_t *ic_c0 = nullptr, *ic_c1 = nullptr, *ic_sp = nullptr;
    size_t ic_rb = 0;      // row stride of the codes (bytes)
    const __half* ic_ap = nullptr;
    auto ic_enter = [&]() {  // base pointers of the issue cursor's task / pair
        if (ic_phase == 0) {
            int slot, n0;
            task_of(ic_j, slot, n0);
            const bool sh = slot == n_active;
            const ProjView& PG = sh ? L.sh_gate : L.gate;
            const ProjView& PU = sh ? L.sh_up : L.up;
            const int N = sh ? L.I_shared : L.I;
            const int fmt = sh ? FS : FR;
            const size_t rowA = (size_t)D.expert[slot] * N + n0 + g;
            ic_rb = (size_t)(H / 2);
            ic_c0 = PG.packed + rowA * ic_rb + 16 * q;
            ic_c1 = PU.packed + rowA * ic_rb + 16 * q;
            ic_sfb = fmt == MOE_FMT_NVFP4 ? 8 : 4;
            ic_rs = (size_t)(H / (fmt == MOE_FMT_NVFP4 ? 16 : 32));
            const ProjView& PS = (q >> 1) ? PU : PG;  // this lane stages (row g + 8 (q & 1), matrix q >> 1)
            ic_sp = PS.scales + (rowA + 8 * (q & 1)) * ic_rs;
            ic_ap = x_src(ic_j);
        } else if (ic_phase == 1) {
            if (ic_j >= npairs) {
                ic_phase = 2;
                return;
            }
            int tl, slot;
            pair_of(ic_j, tl, slot);
            const bool sh = slot == n_active;
            const ProjView& PD = sh ? L.sh_down : L.down;
            const int K = sh ? L.I_shared : L.I;
            const int fmt = sh ? FS : FR;
            const size_t rowA = (size_t)D.expert[slot] * H + (size_t)(cta + tl * G) * 16 + g;
            ic_rb = (size_t)(K / 2);
            ic_c0 = PD.packed + rowA * ic_rb + 16 * q;
            ic_sfb = fmt == MOE_FMT_NVFP4 ? 8 : 4;
            ic_rs = (size_t)(K / (fmt == MOE_FMT_NVFP4 ? 16 : 32));
            ic_sp = PD.scales + (rowA + 8 * (q & 1)) * ic_rs;
            ic_ap = h_src(slot);
            ic_ns = K / 128;
        }
    };
    const uint64_t wpol = l2_evict_first_policy();  // expert weights are read once per launch
    auto copy_scales = [&](uint32_t dst, const uint8_t* src) {
        if (ic_sfb == 8) cp_async8_pol(dst, src, wpol);
        else cp_async4_pol(dst, src, wpol);
    };
    ic_enter();
    int issued = 0;
    auto issue_next = [&]() {
        const uint32_t st = rbase + (issued % kStages) * kStageBytes;
        if (ic_phase == 0) {
            const int o = ic_s * 64;
#pragma unroll
            for (int t = 0; t < TPS; ++t) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const size_t ro = (size_t)(16 * t + 8 * r) * ic_rb + o;
                    cp_async16_pol(st + (4 * t + r) * 512 + lane * 16, ic_c0 + ro, wpol);
                    cp_async16_pol(st + (4 * t + 2 + r) * 512 + lane * 16, ic_c1 + ro, wpol);
                }
                copy_scales(st + Geo::kGuSc + t * 256 + lane * 8, ic_sp + 16 * t * ic_rs + ic_s * ic_sfb);
            }
            copy_act(st + Geo::kGuAct, ic_ap ? ic_ap + ic_s * 128 : nullptr);
            ic_s += kDecWarps;
            if (ic_s >= ksteps_g) {
                ic_s = warp;
                if (++ic_j == cnt_g) {
                    ic_phase = 1;
                    ic_j = warp;
                    ic_s = 0;
                }
                ic_enter();
            }
        } else if (ic_phase == 1) {
            const int nst = ic_ns - ic_s < 2 ? 1 : 2;
            for (int u = 0; u < nst; ++u) {
                const int o = (ic_s + u) * 64;
                cp_async16_pol(st + Geo::kDnCodes + (2 * u) * 512 + lane * 16, ic_c0 + o, wpol);
                cp_async16_pol(st + Geo::kDnCodes + (2 * u + 1) * 512 + lane * 16, ic_c0 + 8 * ic_rb + o, wpol);
                if (q < 2) copy_scales(st + Geo::kDnSc + u * 256 + lane * 8, ic_sp + (ic_s + u) * ic_sfb);
                if (h_ready) copy_act(st + u * Geo::kAct, ic_ap ? ic_ap + (ic_s + u) * 128 : nullptr);
            }
            ic_s += 2;
            if (ic_s >= ic_ns) {
                ic_s = 0;
                ic_j += kDecWarps;
                ic_enter();
            }
        }
        cp_async_commit();
        ++issued;
    };
#pragma unroll 1
    for (int i = 0; i < kStages - 1; ++i) issue_next();
    int consumed = 0;
    auto stage_ptr = [&](int c) { return ring + (c % kStages) * kStageBytes; };

    // ---- phase 2: gate+up ------------------------------------------------------------------------
    for (int j = 0; j < cnt_g; ++j) {
        int slot, n0;
        task_of(j, slot, n0);
        const bool sh = slot == n_active;
        const int fmt = sh ? FS : FR;
        const int mxg = D.mxb[slot][0], mxu = D.mxb[slot][1];
        const bool has_tok = nth_bit(D.tokmask[slot], g) >= 0;
        float acc[2][2][2][4] = {};
        for (int s = 0; s < n_g; ++s) {
            issue_next();
            cp_async_wait<kStages - 1>();
            __syncwarp();
            const uint8_t* st = stage_ptr(consumed);
            if (fmt == MOE_FMT_NVFP4) gu_stage<MOE_FMT_NVFP4, TPS, NTOK>(st, has_tok, lane, g, q, mxg, mxu, acc);
            else gu_stage<MOE_FMT_MXFP4, TPS, NTOK>(st, has_tok, lane, g, q, mxg, mxu, acc);
            ++consumed;
        }
        // K-split reduction, double-buffered: one CTA barrier per task
        float* rg = red_g + (j & 1) * kDecWarps * 512;
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    rg[(warp * 16 + t * 8 + m * 4 + i) * 32 + lane] = acc[t][m][0][i] + acc[t][m][1][i];
        __syncthreads();
        if (tid < 128 * TPS) {  // thread -> (tile, accumulator index, lane) of the MMA layout
            const int t = tid >> 7, i = (tid >> 5) & 3, ln = tid & 31;
            float Gs = 0.f, Us = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) {
                Gs += rg[(w * 16 + t * 8 + i) * 32 + ln];
                Us += rg[(w * 16 + t * 8 + 4 + i) * 32 + ln];
            }
            const int row = 16 * t + (ln >> 2) + 8 * (i >> 1), col = 2 * (ln & 3) + (i & 1);
            const int tok = nth_bit(D.tokmask[slot], col);  // column -> token
            if (tok >= 0) {
                const float hv = silu_f32(Gs * D.post[slot][0]) * (Us * D.post[slot][1]);
                L.h16[((size_t)slot * kDecMaxT + tok) * Imax + n0 + row] = __float2half_rn(hv);
            }
        }
    }
    grid_barrier(bar, bar_base + 2ull * G, L.status, wait_limit);  // every h is written (and red_g is no longer read)
    if (cta == 0 && tid == 0) bar[1] = epoch + 1ull;  // every block has passed barrier 1

    // ---- phase 3: down + weighted sum + shared expert ----------------------------------------------
    // the h chunks of the down stages already in the ring, then every later stage copies its own
    h_ready = true;
    for (int p = warp, idx = 0; p < npairs && done_g + idx < issued; p += kDecWarps) {
        int tl, slot;
        pair_of(p, tl, slot);
        const __half* a = h_src(slot);
        const int ns = (slot == n_active ? L.I_shared : L.I) / 128;
        for (int s = 0; s < ns && done_g + idx < issued; s += 2, ++idx) {
            const uint32_t st = rbase + ((done_g + idx) % kStages) * kStageBytes;
            for (int u = 0; u < 2 && s + u < ns; ++u) copy_act(st + u * Geo::kAct, a ? a + (s + u) * 128 : nullptr);
        }
    }
    cp_async_commit();
    cp_async_wait<0>();
    float acc[kDecMaxTilesPerCta][4] = {};
    for (int p = warp; p < npairs; p += kDecWarps) {
        int tl, slot;
        pair_of(p, tl, slot);
        const bool sh = slot == n_active;
        const int fmt = sh ? FS : FR;
        const int mx = D.mxb[slot][2];
        const int ns = (sh ? L.I_shared : L.I) / 128;
        const bool has_tok = (D.tokmask[slot] >> g) & 1u;
        float part[2][2][4] = {};
        for (int s = 0; s < ns; s += 2) {
            const bool two = s + 1 < ns;
            issue_next();
            cp_async_wait<kStages - 1>();
            __syncwarp();
            const uint8_t* st = stage_ptr(consumed);
            if (fmt == MOE_FMT_NVFP4) {
                if (two) dn_stage<MOE_FMT_NVFP4, 2, TPS, NTOK>(st, has_tok, lane, g, q, mx, part);
                else dn_stage<MOE_FMT_NVFP4, 1, TPS, NTOK>(st, has_tok, lane, g, q, mx, part);
            } else {
                if (two) dn_stage<MOE_FMT_MXFP4, 2, TPS, NTOK>(st, has_tok, lane, g, q, mx, part);
                else dn_stage<MOE_FMT_MXFP4, 1, TPS, NTOK>(st, has_tok, lane, g, q, mx, part);
            }
            ++consumed;
        }
        // expert done: fold in its post-scale and the token weights (MMA column = token)
        const float post = D.post[slot][2];
        const float w0 = D.w[slot][2 * q] * post, w1 = D.w[slot][2 * q + 1] * post;
#pragma unroll
        for (int t = 0; t < kDecMaxTilesPerCta; ++t) {
            if (t == tl) {
                acc[t][0] += sum4(part, 0) * w0;
                acc[t][1] += sum4(part, 1) * w1;
                acc[t][2] += sum4(part, 2) * w0;
                acc[t][3] += sum4(part, 3) * w1;
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp is done with the ring and red_g
#pragma unroll
    for (int t = 0; t < kDecMaxTilesPerCta; ++t)
        if (t < cnt_d)
#pragma unroll
            for (int i = 0; i < 4; ++i) red_d[(t * kDecWarps + warp) * 128 + i * 32 + lane] = acc[t][i];
    __syncthreads();
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(L.out);
    for (int o = tid; o < cnt_d * 128; o += kDecThreads) {
        const int tl = o >> 7, r = o & 127, i = r >> 5, ln = r & 31;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) sum += red_d[(tl * kDecWarps + w) * 128 + r];
        const int row = (ln >> 2) + 8 * (i >> 1), col = 2 * (ln & 3) + (i & 1);
        if (col < T) {
            const size_t o = (size_t)col * H + (size_t)(cta + tl * G) * 16 + row;
            if (S.zw[col] != 0.f)  // zero-computation experts return the token itself
                sum += S.zw[col] * __bfloat162float(static_cast<const __nv_bfloat16*>(L.x)[o]);
            out[o] = __float2bfloat16_rn(sum);
        }
    }
}

// ------------------------------------------------------------------------------------------
template <int TPS, int NTOK>
static int decode_smem_bytes(int H, int sms) {
    const int tpc = (H / 16 + sms - 1) / sms;
    if (tpc > kDecMaxTilesPerCta) return -1;
    return DecGeom<TPS, NTOK>::kRingBytes + (kDecRedG > tpc * kDecRedDTile ? kDecRedG : tpc * kDecRedDTile);
}

template <int FR, int FS, int TPS, int NTOK>
static cudaError_t launch_fused_tps(const FfnLaunch& L, const DecRoute& R, unsigned long long* bar,
                                    int sms, cudaStream_t st) {
    if (L.T > NTOK) return cudaErrorInvalidValue;
    // the router phase stages x in the (still idle) rings
    if ((size_t)L.T * L.H * 2 > (size_t)DecGeom<TPS, NTOK>::kRingBytes) return cudaErrorInvalidValue;
    const int smem = decode_smem_bytes<TPS, NTOK>(L.H, sms);
    if (smem < 0) return cudaErrorInvalidConfiguration;
    auto kern = dec_fused_kernel<FR, FS, TPS, NTOK>;
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
        return err;
    int per_sm = 0;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecThreads, smem)) != cudaSuccess)
        return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);  // one CTA per SM, all co-resident (cooperative launch)
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait in the kernel
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, L, R, bar);
}

template <int FR, int FS, int NTOK>
static cudaError_t launch_fused_fmt(const FfnLaunch& L, const DecRoute& R, unsigned long long* bar,
                                    int sms, cudaStream_t st) {
    // 32-row gate+up tasks unless even the most experts the routing can touch give fewer than
    // two per CTA (then 16-row tasks balance the CTAs better)
    const int slots = L.E < L.T * L.k ? L.E : L.T * L.k;
    const int tasks32 = slots * (L.I / 32) + (L.I_shared > 0 ? L.I_shared / 32 : 0);
    if (tasks32 >= 2 * sms) return launch_fused_tps<FR, FS, 2, NTOK>(L, R, bar, sms, st);
    return launch_fused_tps<FR, FS, 1, NTOK>(L, R, bar, sms, st);
}

// The fused launch with activation chunks laid out for NTOK token columns (T <= NTOK).
template <int NTOK>
static cudaError_t launch_decode_fused_ntok(const FfnLaunch& L, const DecRoute& R,
                                            unsigned long long* bar, int sms, cudaStream_t st) {
    const int fr = L.gate.fmt;
    const int fs = L.I_shared > 0 ? L.sh_gate.fmt : fr;
    if (fr == MOE_FMT_NVFP4 && fs == MOE_FMT_NVFP4) return launch_fused_fmt<0, 0, NTOK>(L, R, bar, sms, st);
    if (fr == MOE_FMT_NVFP4 && fs == MOE_FMT_MXFP4) return launch_fused_fmt<0, 1, NTOK>(L, R, bar, sms, st);
    if (fr == MOE_FMT_MXFP4 && fs == MOE_FMT_NVFP4) return launch_fused_fmt<1, 0, NTOK>(L, R, bar, sms, st);
    return launch_fused_fmt<1, 1, NTOK>(L, R, bar, sms, st);
}

// one token (compact activation chunks): compiled in its own translation unit
cudaError_t launch_decode_fused_t1(const FfnLaunch& L, const DecRoute& R, unsigned long long* bar,
                                   int sms, cudaStream_t st);

}  // namespace moe
