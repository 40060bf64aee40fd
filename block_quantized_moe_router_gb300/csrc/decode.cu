// decode.cu -- the expert FFN for a few tokens (T <= 8 and T * top_k <= 64, bf16
// activations): two launches.
//
//   dec_gateup_kernel   every CTA rebuilds the dispatch (which experts received tokens, in
//                       ascending id order, and which tokens each one received) from the
//                       routing ids -- no separate sort launch -- and then works through
//                       (expert, 16-row tile) tasks: 8 warps split K, each streams its gate and
//                       up rows, their block scales and the tokens through a per-warp ring of
//                       asynchronous copies; the partial sums meet in shared memory and
//                       h = SiLU(gate) * up is written token-major, hT[slot][token][I] (f16).
//   dec_down_kernel     the down projection fused with the top-K weighted sum and the shared
//                       expert: the MMA columns are the T tokens and the sum runs over
//                       (expert, I).  Each of the 8 warps walks a subset of the active experts
//                       through its copy ring; per expert it accumulates W_down . h in fp32 and
//                       adds it scaled by that expert's per-tensor post-scale and each token's
//                       routing weight, so no per-pair outputs reach memory.  Warps are
//                       reduced through shared memory in a fixed order and bf16 rows are
//                       written directly.
//
// This is the "gate+up, silu+down in two fused launches" structure of the spark_model MoE
// module doc (moe/mod.rs), with the weighted sum (init.rs `moe_weighted_sum_blend`) folded
// into the second launch.  Both kernels are launched with programmatic dependent launch.
//
// Copy ring: a warp's stage holds, per lane, its 16-byte code chunks (rows g and g+8 of each
// matrix), its 64 bytes of activations and one 8-byte word of block scales; the stage for step
// i + S - 1 is issued before step i is consumed, so S - 1 steps of every warp are in flight
// without holding registers.
#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace moe {

constexpr int kDecMaxT = 8;
constexpr int kDecMaxSlots = 65;  // at most 64 routed pairs (T * top_k <= 64) + the shared expert

// Dispatch of T <= 8 tokens, rebuilt by every CTA from ids/w.
struct DecDispatch {
    uint32_t bitmap[kMaxExperts / 32];
    int base[kMaxExperts / 32];
    int n_active;                 // routed experts with >= 1 token
    int expert[kDecMaxSlots];     // slot -> expert id (ascending), shared slot -> 0
    uint32_t tokmask[kDecMaxSlots];
    float w[kDecMaxSlots][kDecMaxT];
};

__device__ __forceinline__ void dec_dispatch(const FfnLaunch& L, DecDispatch& D) {
    const int tid = threadIdx.x;
    for (int i = tid; i < kMaxExperts / 32; i += blockDim.x) D.bitmap[i] = 0;
    for (int i = tid; i < kDecMaxSlots * (kDecMaxT + 1); i += blockDim.x) {
        if (i < kDecMaxSlots) D.tokmask[i] = 0;
        else (&D.w[0][0])[i - kDecMaxSlots] = 0.f;
    }
    __syncthreads();
    if (tid < 32) {  // one warp: at most 64 ids, two per lane
        const int lane = tid, P = L.T * L.k;
        int e0 = -1, e1 = -1;
        float w0 = 0.f, w1 = 0.f;  // loaded with the ids: one global round trip
        if (lane < P) { e0 = L.ids[lane]; w0 = L.w[lane]; }
        if (lane + 32 < P) { e1 = L.ids[lane + 32]; w1 = L.w[lane + 32]; }
        if (e0 >= 0 && e0 < L.E) atomicOr(&D.bitmap[e0 >> 5], 1u << (e0 & 31));
        if (e1 >= 0 && e1 < L.E) atomicOr(&D.bitmap[e1 >> 5], 1u << (e1 & 31));
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
            if (e >= 0 && e < L.E) {
                const int slot = D.base[e >> 5] + __popc(D.bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
                const int t = p / L.k;
                D.expert[slot] = e;
                atomicOr(&D.tokmask[slot], 1u << t);
                atomicAdd(&D.w[slot][t], h ? w1 : w0);  // a table may route a token to an expert twice
            }
        }
        if (lane == 0) {
            D.n_active = n_active;
            if (L.I_shared > 0) {
                D.expert[n_active] = 0;
                D.tokmask[n_active] = (1u << L.T) - 1u;
                for (int t = 0; t < L.T; ++t) D.w[n_active][t] = 1.f;
            }
        }
    }
    __syncthreads();
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

// ------------------------------------------------------------------------------------------
// gate+up
// ------------------------------------------------------------------------------------------
constexpr int kGuWarps = 8;  // K split over 8 warps
constexpr int kGuStages = 2;
constexpr int kGuStageBytes = 4 * 512 + 4 * 512 + 32 * 8;  // codes, tokens, scales
// the K-split reduction (8 warps x 8 x 32 floats) reuses the rings once they are drained
constexpr int kGuSmem = kGuWarps * kGuStages * kGuStageBytes;
static_assert(kGuWarps * 8 * 32 * 4 <= kGuSmem, "reduction buffer must fit in the rings");

template <int FMT>
__device__ __forceinline__ void dec_gateup_task(const FfnLaunch& L, const DecDispatch& D, int slot,
                                                int n0, uint8_t* ring, float* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const bool shared = slot == D.n_active;
    const int e = D.expert[slot];
    const uint32_t mask = D.tokmask[slot];
    const ProjView& PG = shared ? L.sh_gate : L.gate;
    const ProjView& PU = shared ? L.sh_up : L.up;
    const int N = shared ? L.I_shared : L.I;
    const int K = L.H;
    const int sv = FMT == MOE_FMT_NVFP4 ? 16 : 32;
    const int steps = K / 128;
    const int per = (steps + kGuWarps - 1) / kGuWarps;
    const int s0 = warp * per, s1 = min(steps, s0 + per);
    const int n = max(0, s1 - s0);

    const size_t rowA = (size_t)e * N + n0 + g;
    const uint8_t* pa[4] = {PG.packed + rowA * (K / 2) + 16 * q,
                            PG.packed + (rowA + 8) * (K / 2) + 16 * q,
                            PU.packed + rowA * (K / 2) + 16 * q,
                            PU.packed + (rowA + 8) * (K / 2) + 16 * q};
    // this lane stages the scales of (row g + 8 * (q & 1), matrix q >> 1)
    const ProjView& PS = (q >> 1) ? PU : PG;
    const uint8_t* sp = PS.scales + (rowA + 8 * (q & 1)) * (K / sv);
    const int mxg = FMT == MOE_FMT_MXFP4 ? 112 + PG.mx_off[e] : 0;
    const int mxu = FMT == MOE_FMT_MXFP4 ? 112 + PU.mx_off[e] : 0;
    const int tok = nth_bit(mask, g);  // column g <-> the g-th token of this expert
    const __nv_bfloat16* xrow =
        static_cast<const __nv_bfloat16*>(L.x) + (size_t)(tok >= 0 ? tok : 0) * K + 32 * q;
    const uint32_t rbase = smem_addr(ring);

    auto issue = [&](int i) {
        if (i < n) {
            const int s = s0 + i;
            const uint32_t st = rbase + (i % kGuStages) * kGuStageBytes;
#pragma unroll
            for (int c = 0; c < 4; ++c) cp_async16(st + c * 512 + lane * 16, pa[c] + s * 64);
            if (tok >= 0) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    cp_async16(st + 2048 + c * 512 + lane * 16, xrow + s * 128 + 8 * c);
            }
            if constexpr (FMT == MOE_FMT_NVFP4) cp_async8(st + 4096 + lane * 8, sp + s * 8);
            else cp_async4(st + 4096 + lane * 8, sp + s * 4);
        }
        cp_async_commit();
    };

    float accG[4] = {0.f, 0.f, 0.f, 0.f}, accU[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kGuStages - 1; ++i) issue(i);
    for (int i = 0; i < n; ++i) {
        issue(i + kGuStages - 1);
        cp_async_wait<kGuStages - 1>();
        __syncwarp();
        const uint8_t* st = ring + (i % kGuStages) * kGuStageBytes;
        ChunkA cg, cu;
        cg.r0 = *reinterpret_cast<const uint4*>(st + 0 * 512 + lane * 16);
        cg.r1 = *reinterpret_cast<const uint4*>(st + 1 * 512 + lane * 16);
        cu.r0 = *reinterpret_cast<const uint4*>(st + 2 * 512 + lane * 16);
        cu.r1 = *reinterpret_cast<const uint4*>(st + 3 * 512 + lane * 16);
        const uint2* sc = reinterpret_cast<const uint2*>(st + 4096);
        scales_from_raw<FMT>(sc[g * 4 + 0], q, mxg, cg.s0lo, cg.s0hi);
        scales_from_raw<FMT>(sc[g * 4 + 1], q, mxg, cg.s1lo, cg.s1hi);
        scales_from_raw<FMT>(sc[g * 4 + 2], q, mxu, cu.s0lo, cu.s0hi);
        scales_from_raw<FMT>(sc[g * 4 + 3], q, mxu, cu.s1lo, cu.s1hi);
        uint32_t bx[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 r = tok >= 0 ? *reinterpret_cast<const uint4*>(st + 2048 + c * 512 + lane * 16)
                                     : make_uint4(0, 0, 0, 0);
            bx[4 * c + 0] = bf16x2_to_f16x2(r.x);
            bx[4 * c + 1] = bf16x2_to_f16x2(r.y);
            bx[4 * c + 2] = bf16x2_to_f16x2(r.z);
            bx[4 * c + 3] = bf16x2_to_f16x2(r.w);
        }
        __syncwarp();  // every lane has read this stage before it is refilled
#define DEC_STEP(I)                                                                \
    {                                                                              \
        uint32_t fa[4], fb[4];                                                     \
        frag_a<I>(cg, fa);                                                         \
        frag_a<I>(cu, fb);                                                         \
        mma_f16_16816(accG, fa[0], fa[1], fa[2], fa[3], bx[2 * I], bx[2 * I + 1]); \
        mma_f16_16816(accU, fb[0], fb[1], fb[2], fb[3], bx[2 * I], bx[2 * I + 1]); \
    }
        DEC_STEP(0) DEC_STEP(1) DEC_STEP(2) DEC_STEP(3)
        DEC_STEP(4) DEC_STEP(5) DEC_STEP(6) DEC_STEP(7)
#undef DEC_STEP
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp's ring is drained: its space now holds the reduction
    // reduce the K-split partial sums through shared memory
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        red[(warp * 8 + i) * 32 + lane] = accG[i];
        red[(warp * 8 + 4 + i) * 32 + lane] = accU[i];
    }
    __syncthreads();
    if (warp == 0) {
        float G[4] = {0.f, 0.f, 0.f, 0.f}, U[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < kGuWarps; ++w) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                G[i] += red[(w * 8 + i) * 32 + lane];
                U[i] += red[(w * 8 + 4 + i) * 32 + lane];
            }
        }
        const float pg = PG.post[e], pu = PU.post[e];
        const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int t = nth_bit(mask, 2 * q + j);  // column -> token
            if (t < 0) continue;
            __half* hrow = L.h16 + ((size_t)slot * kDecMaxT + t) * Imax + n0;
            hrow[g] = __float2half_rn(silu_f32(G[j] * pg) * (U[j] * pu));
            hrow[g + 8] = __float2half_rn(silu_f32(G[2 + j] * pg) * (U[2 + j] * pu));
        }
    }
    __syncthreads();  // the rings are refilled by the next task
}

template <int FMT_R, int FMT_S>
__global__ void __launch_bounds__(kGuWarps * 32, 3) dec_gateup_kernel(FfnLaunch L, int tiles_per_slot) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ DecDispatch D;
    pdl_wait();  // ids / w come from the routing kernels
    dec_dispatch(L, D);
    // let the down kernel's CTAs start now: they stream their weights while this grid runs
    pdl_trigger();
    const int nslots = D.n_active + (L.I_shared > 0 ? 1 : 0);
    const int warp = threadIdx.x >> 5;
    uint8_t* ring = dsm + warp * kGuStages * kGuStageBytes;
    float* red = reinterpret_cast<float*>(dsm);
    const int ntasks = nslots * tiles_per_slot;
    for (int task = blockIdx.x; task < ntasks; task += gridDim.x) {
        const int slot = task / tiles_per_slot;
        const int n0 = (task - slot * tiles_per_slot) * 16;
        const bool shared = slot == D.n_active;
        if (n0 >= (shared ? L.I_shared : L.I)) continue;  // uniform over the CTA
        if (shared) dec_gateup_task<FMT_S>(L, D, slot, n0, ring, red);
        else dec_gateup_task<FMT_R>(L, D, slot, n0, ring, red);
    }
}

// ------------------------------------------------------------------------------------------
// down + weighted sum + shared expert
//
// The down weights depend only on the routing, not on h, so the CTAs (launched while the
// gate+up grid still runs) issue their first kDnStages - 1 weight steps before waiting for h.
// h itself is read from L2 one step ahead in registers.
// ------------------------------------------------------------------------------------------
constexpr int kDnWarps = 8;
constexpr int kDnStages = 6;
constexpr int kDnStageBytes = 2 * 512 + 32 * 8;  // codes of rows g and g+8, scales
constexpr int kDnSmem = kDnWarps * kDnStages * kDnStageBytes + kDnWarps * 4 * 32 * 4;

template <int FMT_R, int FMT_S>
__global__ void __launch_bounds__(kDnWarps * 32) dec_down_kernel(FfnLaunch L) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ DecDispatch D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    // the routing ids were complete before the gate+up grid let this grid start
    dec_dispatch(L, D);
    const int n0 = blockIdx.x * 16;
    const int nslots = D.n_active + (L.I_shared > 0 ? 1 : 0);
    const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
    uint8_t* ring = dsm + warp * kDnStages * kDnStageBytes;
    float* red = reinterpret_cast<float*>(dsm + kDnWarps * kDnStages * kDnStageBytes);
    const uint32_t rbase = smem_addr(ring);

    // this warp's work: slots warp, warp + 8, ...; their K steps in one flat sequence
    int total = 0;
    for (int slot = warp; slot < nslots; slot += kDnWarps)
        total += (slot == D.n_active ? L.I_shared : L.I) / 128;

    int is_slot = warp, is_s = 0;  // weight issue cursor
    auto issue = [&](int i) {
        if (i < total) {
            const bool sh = is_slot == D.n_active;
            const int e = D.expert[is_slot];
            const ProjView& PD = sh ? L.sh_down : L.down;
            const int K = sh ? L.I_shared : L.I;
            const int svb = (sh ? FMT_S : FMT_R) == MOE_FMT_NVFP4 ? 16 : 32;
            const size_t rowA = (size_t)e * L.H + n0 + g;
            const uint32_t st = rbase + (i % kDnStages) * kDnStageBytes;
            cp_async16(st + lane * 16, PD.packed + rowA * (K / 2) + 16 * q + is_s * 64);
            cp_async16(st + 512 + lane * 16, PD.packed + (rowA + 8) * (K / 2) + 16 * q + is_s * 64);
            if (q < 2) {  // scales of row g + 8q
                const uint8_t* sp = PD.scales + (rowA + 8 * q) * (K / svb);
                if (svb == 16) cp_async8(st + 1024 + lane * 8, sp + is_s * 8);
                else cp_async4(st + 1024 + lane * 8, sp + is_s * 4);
            }
            if (++is_s == K / 128) {
                is_s = 0;
                is_slot += kDnWarps;
            }
        }
        cp_async_commit();
    };
#pragma unroll 1
    for (int i = 0; i < kDnStages - 1; ++i) issue(i);

    pdl_wait();  // h comes from the gate+up kernel

    int hs_slot = warp, hs_s = 0;  // h cursor (one step ahead of the compute)
    auto load_h = [&](uint4 (&b)[4]) {
        const bool ok = hs_slot < nslots && ((D.tokmask[hs_slot] >> g) & 1u);  // column g = token g
        const __half* hrow = L.h16 + ((size_t)hs_slot * kDecMaxT + g) * Imax + 32 * q + hs_s * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = ok ? ldg_cached128(hrow + 8 * j) : make_uint4(0, 0, 0, 0);
        if (hs_slot < nslots && ++hs_s == (hs_slot == D.n_active ? L.I_shared : L.I) / 128) {
            hs_s = 0;
            hs_slot += kDnWarps;
        }
    };
    uint4 hb[4], hn[4];
    if (total > 0) load_h(hb);

    float acc[4] = {0.f, 0.f, 0.f, 0.f}, part[4] = {0.f, 0.f, 0.f, 0.f};
    int cs_slot = warp, cs_s = 0;  // consume cursor
    for (int i = 0; i < total; ++i) {
        issue(i + kDnStages - 1);
        if (i + 1 < total) load_h(hn);
        cp_async_wait<kDnStages - 1>();
        __syncwarp();
        const bool sh = cs_slot == D.n_active;
        const int e = D.expert[cs_slot];
        const uint8_t* st = ring + (i % kDnStages) * kDnStageBytes;
        ChunkA c;
        c.r0 = *reinterpret_cast<const uint4*>(st + lane * 16);
        c.r1 = *reinterpret_cast<const uint4*>(st + 512 + lane * 16);
        const uint2* sc = reinterpret_cast<const uint2*>(st + 1024);
        if ((sh ? FMT_S : FMT_R) == MOE_FMT_NVFP4) {
            scales_from_raw<MOE_FMT_NVFP4>(sc[g * 4 + 0], q, 0, c.s0lo, c.s0hi);
            scales_from_raw<MOE_FMT_NVFP4>(sc[g * 4 + 1], q, 0, c.s1lo, c.s1hi);
        } else {
            const int mx = 112 + (sh ? L.sh_down : L.down).mx_off[e];
            scales_from_raw<MOE_FMT_MXFP4>(sc[g * 4 + 0], q, mx, c.s0lo, c.s0hi);
            scales_from_raw<MOE_FMT_MXFP4>(sc[g * 4 + 1], q, mx, c.s1lo, c.s1hi);
        }
        __syncwarp();  // every lane has read this stage before it is refilled
#define DOWN_STEP(I)                                                                       \
    {                                                                                      \
        uint32_t fa[4];                                                                    \
        frag_a<I>(c, fa);                                                                  \
        mma_f16_16816(part, fa[0], fa[1], fa[2], fa[3], word_of(hb[I >> 1], (I & 1) * 2),  \
                      word_of(hb[I >> 1], (I & 1) * 2 + 1));                               \
    }
        DOWN_STEP(0) DOWN_STEP(1) DOWN_STEP(2) DOWN_STEP(3)
        DOWN_STEP(4) DOWN_STEP(5) DOWN_STEP(6) DOWN_STEP(7)
#undef DOWN_STEP
#pragma unroll
        for (int j = 0; j < 4; ++j) hb[j] = hn[j];
        const int K = sh ? L.I_shared : L.I;
        if (++cs_s == K / 128) {  // expert done: fold in with its post-scale and token weights
            const float post = (sh ? L.sh_down : L.down).post[e];
            const float w0 = D.w[cs_slot][2 * q] * post, w1 = D.w[cs_slot][2 * q + 1] * post;
            acc[0] += part[0] * w0;
            acc[1] += part[1] * w1;
            acc[2] += part[2] * w0;
            acc[3] += part[3] * w1;
            part[0] = part[1] = part[2] = part[3] = 0.f;
            cs_s = 0;
            cs_slot += kDnWarps;
        }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int i = 0; i < 4; ++i) red[(warp * 4 + i) * 32 + lane] = acc[i];
    __syncthreads();
    pdl_trigger();
    if (warp == 0) {
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < kDnWarps; ++w)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] += red[(w * 4 + i) * 32 + lane];
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
template <typename Kern>
static cudaError_t set_smem(Kern kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl_smem(void (*kernel)(KArgs...), dim3 grid, dim3 block, int smem,
                                   cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int FR, int FS>
static cudaError_t launch_decode_fmt(const FfnLaunch& L, int phase, cudaStream_t st) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t err;
    if (phase == 1) {
        const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
        const int tiles = Imax / 16;
        const int slots = (L.E < L.T * L.k ? L.E : L.T * L.k) + (L.I_shared > 0 ? 1 : 0);
        int grid = slots * tiles;
        if (grid > 2 * sms) grid = 2 * sms;  // two per SM, leaving room for the down kernel
        if ((err = set_smem(dec_gateup_kernel<FR, FS>, kGuSmem)) != cudaSuccess) return err;
        return launch_pdl_smem(dec_gateup_kernel<FR, FS>, dim3(grid), dim3(kGuWarps * 32), kGuSmem,
                               st, L, tiles);
    }
    if ((err = set_smem(dec_down_kernel<FR, FS>, kDnSmem)) != cudaSuccess) return err;
    return launch_pdl_smem(dec_down_kernel<FR, FS>, dim3(L.H / 16), dim3(kDnWarps * 32), kDnSmem,
                           st, L);
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
