// ffn.cu -- expert dispatch and the grouped expert FFN on the warp-level tensor-core path.
//
// Structure (spark_model MoE pages, moe/mod.rs module doc and `MoeLayer` field docs):
//   1. dispatch: histogram of the routed (token, slot) pairs per expert, offsets, the list of
//      experts that received tokens, and the permutation grouping pairs by expert
//      (`moe_sort_by_expert`, `moe_build_tile_worklist` handles);
//   2. gate+up projection of every routed pair and of the shared expert, SiLU(gate)*up fused
//      into its epilogue (`moe_expert_gate_up_shared`);
//   3. down projection, the routing weight applied in its epilogue
//      (`moe_expert_silu_down_shared`);
//   4. top-K weighted sum plus the shared expert (`moe_weighted_sum_blend`).
//
// Weight formats (moe/mod.rs, `MoeLayer::experts_scale_kind` field doc): NVFP4 = E2M1 codes,
// FP8-E4M3 scale per 16, f32 per-tensor global; MXFP4 = E2M1 codes, E8M0 scale per 32.
//
// The grouped GEMM: each warp owns 16 output rows of one expert and streams their packed
// weight rows with 16-byte loads (32 E2M1 codes per lane per step).  Codes are converted to
// f16 with the hardware E2M1->f16x2 conversion and multiplied by the f16 block scale (both
// exact: an E2M1 value times an E4M3 value has at most 6 significant bits and lies within
// [2^-10, 2688]); the per-tensor global is applied in fp32 at the end.  The columns are the
// expert's routed pairs (8 per m16n8k16 MMA tile), so each weight row is read once per
// launch whatever the number of tokens routed to the expert.  Activations enter as f16
// (bf16 tokens converted once; the NVFP4-quantized tokens and h are exact in f16).
#include <type_traits>

#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"
#include "quant.cuh"

namespace moe {

enum { MODE_GATEUP = 0, MODE_DOWN = 1 };

// ------------------------------------------------------------------------------------------
// Dispatch (block 0) + activation conversion/quantization (blocks 1..).
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(512) prep_kernel(FfnLaunch L) {
    const int tid = threadIdx.x;
    if (blockIdx.x == 0) {
        __shared__ int s_cnt[kMaxExperts];
        __shared__ int s_cur[kMaxExperts];
        const int E = L.E, P = L.T * L.k;
        for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
        __syncthreads();
        int bad = 0;
        for (int p = tid; p < P; p += blockDim.x) {
            const int e = L.ids[p];
            if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
            else if (e != -1 && !(e >= E && e < E + L.Z)) bad = 1;  // zero-computation experts are valid
        }
        if (bad) status_or(L.status, MOE_DEV_BAD_EXPERT_ID);
        __syncthreads();
        if (tid < 32) {
            const int lane = tid;
            const int per = (E + 31) / 32;
            const int lo = min(E, lane * per), hi = min(E, lo + per);
            int sum = 0, nz = 0;
            for (int e = lo; e < hi; ++e) { sum += s_cnt[e]; nz += s_cnt[e] > 0; }
            int isum = sum, inz = nz;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, isum, o);
                const int b = __shfl_up_sync(0xffffffffu, inz, o);
                if (lane >= o) { isum += a; inz += b; }
            }
            int off = isum - sum, act = inz - nz;
            for (int e = lo; e < hi; ++e) {
                const int c = s_cnt[e];
                L.offsets[e] = off;
                L.counts[e] = c;
                s_cur[e] = off;
                if (c > 0) L.active[act++] = e;
                off += c;
            }
            if (lane == 31) {
                L.offsets[E] = isum;
                L.meta[0] = inz;  // number of experts with at least one pair
                L.meta[1] = isum; // number of valid routed pairs
            }
        }
        __syncthreads();
        for (int p = tid; p < P; p += blockDim.x) {
            const int e = L.ids[p];
            if (e >= 0 && e < E) {
                const int pos = atomicAdd(&s_cur[e], 1);
                L.sorted_pair[pos] = p;
                L.pos_of_pair[p] = pos;
            } else {
                L.pos_of_pair[p] = -1;
            }
        }
        return;
    }
    // activation conversion: one thread per 16 elements of x
    const int64_t n16 = (int64_t)L.T * L.H / 16;
    const int64_t stride = (int64_t)(gridDim.x - 1) * blockDim.x;
    const auto* x = static_cast<const __nv_bfloat16*>(L.x);
    for (int64_t i = (int64_t)(blockIdx.x - 1) * blockDim.x + tid; i < n16; i += stride) {
        float v[16];
        load_bf16x16(x + i * 16, v);
        if (L.act == MOE_ACT_NVFP4) {
            quant16(v, L.g1, L.xq + i * 8, L.xs + i, L.x16 + i * 16);
        } else {
            uint4 a, b;
            a.x = pack_half2(v[0], v[1]);   a.y = pack_half2(v[2], v[3]);
            a.z = pack_half2(v[4], v[5]);   a.w = pack_half2(v[6], v[7]);
            b.x = pack_half2(v[8], v[9]);   b.y = pack_half2(v[10], v[11]);
            b.z = pack_half2(v[12], v[13]); b.w = pack_half2(v[14], v[15]);
            reinterpret_cast<uint4*>(L.x16 + i * 16)[0] = a;
            reinterpret_cast<uint4*>(L.x16 + i * 16)[1] = b;
        }
    }
}

// ------------------------------------------------------------------------------------------
// Grouped expert GEMM on m16n8k16 f16 MMAs.
//
// A CTA of kErWarps warps owns rows of one expert's projection over the whole K -- gate+up:
// 16 rows of gate and the same 16 of up per warp; down: two 16-row tiles per warp, as matrices
// A and B -- and the expert's tokens in passes of up to NT = 2 MMA column tiles of 8;
// each dequantized A fragment serves every column tile of the pass.  The
// operands stream through a CTA ring of kErStages shared-memory stages filled by cp.async,
// kErStages - 1 K-steps ahead of the MMAs (one flat sequence over all passes): every warp
// copies its own weight rows, and the token chunks, the same for all warps, are copied once
// by the whole CTA.  One CTA barrier per K-step both publishes a stage and frees the one the
// next copies refill.  Stage layout (512 B = 32 lanes x 16 B; MMA row g = lane / 4):
//   per warp w at w * kErWarpBytes: [0, 1024) codes of matrix A (rows g, g + 8),
//     [1024, 2048) codes of matrix B (up, or down's second tile), [2048, 2304) block scales (lane (g, q) stages
//     row g + 8 (q & 1) of matrix q >> 1);
//   token chunks at kErBOff: tile t at t * 2048, 16 B per (8-element group c, column j, q) at
//     c * 512 + (4 j + q) * 16.
// ------------------------------------------------------------------------------------------
constexpr int kErWarps = 4;
constexpr int kErStages = 3;
constexpr int kErNT = 2;
constexpr int kErWarpBytes = 2304;
constexpr int kErBOff = kErWarps * kErWarpBytes;
constexpr int kErStageBytes = kErBOff + kErNT * 2048;
constexpr int kErSmemBytes = kErStages * kErStageBytes;

// Work items: (routed slot, 64-row block) for the routed experts, slot-major; then, for the
// shared expert, which takes every token, (64-row block, 16-token tile: one pass of the NT = 2
// MMA column tiles) with the tiles of one row block adjacent.  The shared expert's items then
// cost about as much as a routed item with its few tokens, so the CTAs, which take items
// strided by the grid, finish together; its weight rows are read by the few CTAs running its
// adjacent items at the same time (L2 hits after the first).  A shared expert taken as
// whole-row-block items with all its tokens made those items several times heavier than the
// rest and left a tail.
struct ErItem {
    bool valid, shared;
    int e, row0, cnt, N, K;
    int xb, tb;  // 64-row block; first token of the item (shared expert)
};
template <int MODE>
__device__ __forceinline__ ErItem er_item(const FfnLaunch& L, int max_routed_slots, int xblocks,
                                          int it) {
    ErItem w{};
    const int routed_items = max_routed_slots * xblocks;
    if (it < routed_items) {
        const int slot = it / xblocks;
        w.xb = it - slot * xblocks;
        if (slot >= L.meta[0]) return w;
        w.e = L.active[slot];
        w.row0 = L.offsets[w.e];
        w.cnt = L.offsets[w.e + 1] - w.row0;
    } else {
        const int tiles = (L.T + 8 * kErNT - 1) / (8 * kErNT), j = it - routed_items;
        w.shared = true;
        w.xb = j / tiles;
        w.tb = (j - w.xb * tiles) * 8 * kErNT;
        w.e = 0;
        w.row0 = 0;
        w.cnt = min(8 * kErNT, L.T - w.tb);
    }
    const int Iexp = w.shared ? L.I_shared : L.I;
    w.N = MODE == MODE_GATEUP ? Iexp : L.H;
    w.K = MODE == MODE_GATEUP ? L.H : Iexp;
    w.valid = w.xb * kErWarps * 16 * (MODE == MODE_GATEUP ? 1 : 2) < w.N && w.cnt > 0;
    return w;
}

template <int MODE, int FR, int FS>
__global__ void __launch_bounds__(kErWarps * 32)
expert_mma_kernel(FfnLaunch L, int max_routed_slots, int xblocks, int items) {
    extern __shared__ __align__(16) uint8_t er_smem[];
    constexpr int NT = kErNT;
    // rows per warp: gate+up 16 of gate and 16 of up; down two 16-row tiles (matrices A and B)
    constexpr int kErRowsW = MODE == MODE_GATEUP ? 16 : 32;
    uint8_t* ring = er_smem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
    const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
    const int P = L.T * L.k;
    const uint32_t rbase = smem_addr(ring);
    // this thread's token chunk: group c = tid / 32, column j = (tid % 32) / 4, q = tid % 4
    const int bc = tid >> 5, bj = (tid & 31) >> 2, bq = tid & 3;
    auto b_src = [&](const ErItem& w, int col) -> const __half* {  // column col, K-step 0
        if (col >= w.cnt) return nullptr;
        if (MODE == MODE_GATEUP) {
            const int tok = w.shared ? w.tb + col : L.sorted_pair[w.row0 + col] / L.k;
            return L.x16 + (size_t)tok * L.H + 32 * bq + 8 * bc;
        }
        const int r = w.shared ? P + w.tb + col : w.row0 + col;
        return L.h16 + (size_t)r * Imax + 32 * bq + 8 * bc;
    };

    // ---- issue cursor: item, pass, K-step; one flat sequence over this CTA's items ----
    int ci = blockIdx.x, ip = 0, is = 0;
    ErItem cw{};
    int c_steps = 1, c_passes = 0, c_sfb = 8;
    // weight rows read once (one pass over the item's tokens) stream with an L2 evict-first
    // policy; rows read again in a later pass stay at the normal priority
    const uint64_t pol_once = l2_evict_first_policy(), pol_again = l2_evict_normal_policy();
    uint64_t c_pol = pol_once;
    size_t c_rstride = 0;
    const uint8_t *pa = nullptr, *pb = nullptr, *ps = nullptr;
    const __half* ib[NT];
    auto enter_pass = [&]() {
#pragma unroll
        for (int t = 0; t < NT; ++t) ib[t] = b_src(cw, ip * 8 * NT + 8 * t + bj);
    };
    auto enter_item = [&]() {  // the first valid item at or after ci
        for (; ci < items; ci += gridDim.x) {
            cw = er_item<MODE>(L, max_routed_slots, xblocks, ci);
            if (cw.valid) break;
        }
        if (ci >= items) return;
        const int fmt = cw.shared ? FS : FR;
        const int sv = fmt == MOE_FMT_NVFP4 ? 16 : 32;
        c_sfb = 128 / sv;
        c_steps = cw.K / 128;
        c_passes = (cw.cnt + 8 * NT - 1) / (8 * NT);
        // the shared expert's rows are read by the items of all its token tiles
        c_pol = (c_passes > 1 || cw.shared) ? pol_again : pol_once;
        c_rstride = (size_t)8 * (cw.K / 2);
        const int xb = cw.xb;
        const int n0 = (xb * kErWarps + warp) * kErRowsW;
        const bool rows_ok = n0 < cw.N;
        const ProjView& PA = MODE == MODE_GATEUP ? (cw.shared ? L.sh_gate : L.gate)
                                                 : (cw.shared ? L.sh_down : L.down);
        const ProjView& PB = cw.shared ? L.sh_up : L.up;
        const size_t rowA = (size_t)cw.e * cw.N + n0 + g;
        pa = rows_ok ? PA.packed + rowA * (cw.K / 2) + 16 * q : nullptr;
        // matrix B: up (gate+up), or the warp's second 16-row tile of down
        const bool rows2 = MODE == MODE_GATEUP ? rows_ok : n0 + 16 < cw.N;
        const size_t rowB = MODE == MODE_GATEUP ? rowA : rowA + 16;
        pb = rows2 ? (MODE == MODE_GATEUP ? PB : PA).packed + rowB * (cw.K / 2) + 16 * q : nullptr;
        // lane (g, q) stages the scales of row g + 8 (q & 1) of matrix q >> 1
        ps = ((q >> 1) ? rows2 : rows_ok)
                 ? ((q >> 1) && MODE == MODE_GATEUP ? PB : PA).scales +
                       ((q >> 1) ? rowB : rowA) * (size_t)(cw.K / sv) + 8 * (q & 1) * (size_t)(cw.K / sv)
                 : nullptr;
        ip = 0;
        is = 0;
        enter_pass();
    };
    enter_item();
    int issued = 0;
    auto issue = [&]() {
        if (ci < items) {
            const uint32_t st = rbase + (issued % kErStages) * kErStageBytes;
            const uint32_t sw = st + warp * kErWarpBytes;
            const int o = is * 64;
            if (pa) {
                cp_async16_pol(sw + lane * 16, pa + o, c_pol);
                cp_async16_pol(sw + 512 + lane * 16, pa + c_rstride + o, c_pol);
            }
            if (pb) {
                cp_async16_pol(sw + 1024 + lane * 16, pb + o, c_pol);
                cp_async16_pol(sw + 1536 + lane * 16, pb + c_rstride + o, c_pol);
            }
            if (ps) {
                if (c_sfb == 8) cp_async8_pol(sw + 2048 + lane * 8, ps + is * c_sfb, c_pol);
                else cp_async4_pol(sw + 2048 + lane * 8, ps + is * c_sfb, c_pol);
            }
#pragma unroll
            for (int t = 0; t < NT; ++t)
                if (ib[t]) cp_async16(st + kErBOff + t * 2048 + bc * 512 + (tid & 31) * 16, ib[t] + is * 128);
            if (++is == c_steps) {
                is = 0;
                if (++ip == c_passes) {
                    ci += gridDim.x;
                    enter_item();
                } else {
                    enter_pass();
                }
            }
        }
        cp_async_commit();
        ++issued;
    };
#pragma unroll 1
    for (int i = 0; i < kErStages - 1; ++i) issue();
    int consumed = 0;

    // ---- consumer: the same items, passes and K-steps in the same order ----
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const ErItem w = er_item<MODE>(L, max_routed_slots, xblocks, it);
        if (!w.valid) continue;  // CTA-uniform
        const bool shared = w.shared;
        const int e = w.e, row0 = w.row0, cnt = w.cnt, N = w.N, K = w.K, tb = w.tb;
        const int n0 = (w.xb * kErWarps + warp) * kErRowsW;
        const bool rows_ok = n0 < N;
        const int steps = K / 128;
        auto body = [&](auto fmt_c) {
            constexpr int FMT = decltype(fmt_c)::value;
            const ProjView& PA = MODE == MODE_GATEUP ? (shared ? L.sh_gate : L.gate)
                                                     : (shared ? L.sh_down : L.down);
            const ProjView& PB = shared ? L.sh_up : L.up;
            const int mxa = (FMT == MOE_FMT_MXFP4) ? 112 + PA.mx_off[e] : 0;
            const int mxb = FMT != MOE_FMT_MXFP4 ? 0 : MODE == MODE_GATEUP ? 112 + PB.mx_off[e] : mxa;
            const float postA = PA.post[e];
            const float postB = (MODE == MODE_GATEUP) ? PB.post[e] : 1.f;
            for (int c0 = 0; c0 < cnt; c0 += 8 * NT) {
                bool bval[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) bval[nt] = c0 + nt * 8 + g < cnt;
                float accA[NT][4], accB[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) { accA[nt][i] = 0.f; accB[nt][i] = 0.f; }
                for (int s = 0; s < steps; ++s) {
                    cp_async_wait<kErStages - 2>();
                    __syncthreads();  // stage `consumed` is in; every warp is done with the one refilled next
                    issue();
                    const uint8_t* st = ring + (consumed % kErStages) * kErStageBytes;
                    const uint8_t* sw = st + warp * kErWarpBytes;
                    const uint2* sc = reinterpret_cast<const uint2*>(sw + 2048);
                    ChunkA ca, cb;
                    ca.r0 = *reinterpret_cast<const uint4*>(sw + lane * 16);
                    ca.r1 = *reinterpret_cast<const uint4*>(sw + 512 + lane * 16);
                    scales_from_raw<FMT>(sc[g * 4 + 0], q, mxa, ca.s0lo, ca.s0hi);
                    scales_from_raw<FMT>(sc[g * 4 + 1], q, mxa, ca.s1lo, ca.s1hi);
                    {   // matrix B: up, or down's second 16-row tile
                        cb.r0 = *reinterpret_cast<const uint4*>(sw + 1024 + lane * 16);
                        cb.r1 = *reinterpret_cast<const uint4*>(sw + 1536 + lane * 16);
                        scales_from_raw<FMT>(sc[g * 4 + 2], q, mxb, cb.s0lo, cb.s0hi);
                        scales_from_raw<FMT>(sc[g * 4 + 3], q, mxb, cb.s1lo, cb.s1hi);
                    }
                    if (rows_ok) {
                        // the column tiles of this pass that hold tokens (warp-uniform); each A
                        // fragment is dequantized once and used for all of them
                        const int ntv = min(NT, (cnt - c0 + 7) / 8);
                        uint4 b[NT][4];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                b[nt][j] = (nt < ntv && bval[nt])
                                               ? *reinterpret_cast<const uint4*>(st + kErBOff + nt * 2048 + j * 512 + lane * 16)
                                               : make_uint4(0, 0, 0, 0);
#define MOE_STEP(I)                                                                   \
            {                                                                                 \
                uint32_t fa[4], fb[4];                                                        \
                frag_a<I>(ca, fa);                                                            \
                frag_a<I>(cb, fb);                                                            \
                _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                           \
                    if (nt < ntv) {                                                           \
                        const uint32_t b0 = word_of(b[nt][I >> 1], (I & 1) * 2);              \
                        const uint32_t b1 = word_of(b[nt][I >> 1], (I & 1) * 2 + 1);          \
                        mma_f16_16816(accA[nt], fa[0], fa[1], fa[2], fa[3], b0, b1);          \
                        mma_f16_16816(accB[nt], fb[0], fb[1], fb[2], fb[3], b0, b1);          \
                    }                                                                         \
                }                                                                             \
            }
                        MOE_STEP(0) MOE_STEP(1) MOE_STEP(2) MOE_STEP(3)
                        MOE_STEP(4) MOE_STEP(5) MOE_STEP(6) MOE_STEP(7)
#undef MOE_STEP
                    }
                    ++consumed;
                }
                if (!rows_ok) continue;

                // ---- epilogue ----
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (c0 + nt * 8 >= cnt) break;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int col = c0 + nt * 8 + 2 * q + j;
                        const bool valid = col < cnt;
                        const int r = shared ? P + tb + col : row0 + col;
                        if (MODE == MODE_GATEUP) {
                            const float h0 = silu_f32(accA[nt][j] * postA) * (accB[nt][j] * postB);
                            const float h1 = silu_f32(accA[nt][2 + j] * postA) * (accB[nt][2 + j] * postB);
                            if (L.act == MOE_ACT_NVFP4) {
                                // quantize h over the 16 consecutive rows n0..n0+15 of this column
                                float amax = fmaxf(fabsf(h0), fabsf(h1));
                                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
                                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 8));
                                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
                                float qs = amax / 6.0f;
                                qs = qs / L.g2;
                                const uint32_t sbyte = f32_to_e4m3(qs);
                                const float denom = e4m3_to_f32(sbyte) * L.g2;
                                uint32_t c0b = 0, c1b = 0;
                                if (denom != 0.f) {
                                    c0b = f32x2_to_e2m1x2(h0 / denom, 0.f) & 0xF;
                                    c1b = f32x2_to_e2m1x2(h1 / denom, 0.f) & 0xF;
                                }
                                const uint32_t n0c = __shfl_down_sync(0xffffffffu, c0b, 4);
                                const uint32_t n1c = __shfl_down_sync(0xffffffffu, c1b, 4);
                                if (valid) {
                                    __half* hrow = L.h16 + (size_t)r * Imax + n0;
                                    hrow[g] = __float2half_rn(e2m1_to_f32(c0b) * denom);
                                    hrow[g + 8] = __float2half_rn(e2m1_to_f32(c1b) * denom);
                                    uint8_t* qrow = L.hq + (size_t)r * (Imax / 2) + n0 / 2;
                                    if ((g & 1) == 0) {
                                        qrow[g / 2] = (uint8_t)(c0b | (n0c << 4));
                                        qrow[(g + 8) / 2] = (uint8_t)(c1b | (n1c << 4));
                                    }
                                    if (g == 0) L.hs[(size_t)r * (Imax / 16) + n0 / 16] = (uint8_t)sbyte;
                                }
                            } else if (valid) {
                                __half* hrow = L.h16 + (size_t)r * Imax + n0;
                                hrow[g] = __float2half_rn(h0);
                                hrow[g + 8] = __float2half_rn(h1);
                            }
                        } else if (valid) {
                            const float wcol = shared ? 1.f : L.w[L.sorted_pair[row0 + col]];
                            float* yrow = L.y + (size_t)r * L.H + n0;
                            yrow[g] = accA[nt][j] * postA * wcol;
                            yrow[g + 8] = accA[nt][2 + j] * postA * wcol;
                            if (n0 + 16 < N) {  // the second 16-row tile
                                yrow[16 + g] = accB[nt][j] * postA * wcol;
                                yrow[24 + g] = accB[nt][2 + j] * postA * wcol;
                            }
                        }
                    }
                }
            }
        };
        if (shared) body(std::integral_constant<int, FS>{});
        else body(std::integral_constant<int, FR>{});
    }
    cp_async_wait<0>();  // nothing may be in flight into shared memory when the CTA exits
}

// ------------------------------------------------------------------------------------------
// Combine: out[t] = sum_j y[pos(t,j)] + y[shared row t] + (folded weight of the
// zero-computation experts) * x[t], fixed j order, bf16 output.
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(FfnLaunch L) {
    const int H8 = L.H / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)L.T * H8) return;
    const int t = (int)(idx / H8), c = (int)(idx - (int64_t)t * H8);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    auto add_row = [&](int r) {
        const float4* src = reinterpret_cast<const float4*>(L.y + (size_t)r * L.H + c * 8);
        const float4 a = src[0], b = src[1];
        acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
        acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    };
    float zw = 0.f;
    for (int j = 0; j < L.k; ++j) {
        const int pos = L.pos_of_pair[t * L.k + j];
        if (pos >= 0) add_row(pos);
        const int e = L.ids[t * L.k + j];
        if (e >= L.E && e < L.E + L.Z) zw += L.w[t * L.k + j];
    }
    if (L.I_shared > 0) add_row(L.T * L.k + t);
    if (zw != 0.f) {
        const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(L.x) +
                                                         (size_t)t * L.H + c * 8);
        const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] += zw * __uint_as_float(xw[i] << 16);
            acc[2 * i + 1] += zw * __uint_as_float(xw[i] & 0xFFFF0000u);
        }
    }
    uint4 o;
    __nv_bfloat162 v;
    v = __floats2bfloat162_rn(acc[0], acc[1]); o.x = *reinterpret_cast<uint32_t*>(&v);
    v = __floats2bfloat162_rn(acc[2], acc[3]); o.y = *reinterpret_cast<uint32_t*>(&v);
    v = __floats2bfloat162_rn(acc[4], acc[5]); o.z = *reinterpret_cast<uint32_t*>(&v);
    v = __floats2bfloat162_rn(acc[6], acc[7]); o.w = *reinterpret_cast<uint32_t*>(&v);
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(L.out) + (size_t)t * L.H)[c] = o;
}

// ------------------------------------------------------------------------------------------
__global__ void quantize_act_kernel(const __nv_bfloat16* __restrict__ x, int64_t n16, float g,
                                    uint8_t* __restrict__ packed, uint8_t* __restrict__ scales,
                                    __half* deq16) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n16) return;
    float v[16];
    load_bf16x16(x + i * 16, v);
    quant16(v, g, packed + i * 8, scales + i, deq16 ? deq16 + i * 16 : nullptr);
}

__global__ void mx_offsets_kernel(const uint8_t* __restrict__ scales, int64_t per_expert,
                                  int32_t* __restrict__ off, float* __restrict__ post) {
    const int e = blockIdx.x;
    const uint8_t* s = scales + (size_t)e * per_expert;
    int m = 0;
    for (int64_t i = threadIdx.x; i < per_expert; i += blockDim.x) m = max(m, (int)s[i]);
    __shared__ int red[32];
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        int mm = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mm = max(mm, red[w]);
        if (mm == 255) mm = 254;  // 0xFF is NaN in E8M0; never produced by an encoder
        // f16 scale = 2^(byte - 127 - o) with o = max - 139: the largest block scale maps to
        // 2^12, so 6 * scale stays below the f16 maximum; post = 2^o restores the magnitude.
        const int o = mm - 139;
        off[e] = o;
        post[e] = ldexpf(1.0f, o);
    }
}

// ------------------------------------------------------------------------------------------
// Records a timing event on `st`; inside stream capture it becomes an event-record node.
cudaError_t record_phase_event(cudaEvent_t ev, cudaStream_t st) {
    if (!ev) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t err = cudaStreamIsCapturing(st, &cs);
    if (err != cudaSuccess) return err;
    return cs == cudaStreamCaptureStatusActive
               ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
               : cudaEventRecord(ev, st);
}

template <int MODE, int FR, int FS>
static cudaError_t launch_expert_gemm(const FfnLaunch& L, int slots_r, cudaStream_t st) {
    const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
    const int N = MODE == MODE_GATEUP ? Imax : L.H;
    auto kern = expert_mma_kernel<MODE, FR, FS>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kErSmemBytes);
    if (err != cudaSuccess) return err;
    int per_sm = 0, dev = 0, sms = 0;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kErWarps * 32, kErSmemBytes)) != cudaSuccess)
        return err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    // persistent CTAs: work items strided by the grid (er_item): routed (slot, 64-row block),
    // slot-major so that concurrently running CTAs read neighbouring rows of one expert, then
    // the shared expert's (64-row block, 16-token tile)
    const int rows_item = kErWarps * (MODE == MODE_GATEUP ? 16 : 32);  // down: two 16-row tiles a warp
    const int xblocks = (N + rows_item - 1) / rows_item;
    const int items = xblocks * slots_r + (L.I_shared > 0 ? xblocks * ((L.T + 8 * kErNT - 1) / (8 * kErNT)) : 0);
    int grid = (per_sm > 0 ? per_sm : 1) * sms;
    if (grid > items) grid = items;
    kern<<<grid, kErWarps * 32, kErSmemBytes, st>>>(L, slots_r, xblocks, items);
    return cudaGetLastError();
}

template <int MODE>
static cudaError_t launch_expert_phase(const FfnLaunch& L, int slots_r, cudaStream_t st) {
    const int fr = L.gate.fmt;
    const int fs = L.I_shared > 0 ? L.sh_gate.fmt : fr;
    if (fr == MOE_FMT_NVFP4 && fs == MOE_FMT_NVFP4)
        return launch_expert_gemm<MODE, MOE_FMT_NVFP4, MOE_FMT_NVFP4>(L, slots_r, st);
    if (fr == MOE_FMT_NVFP4 && fs == MOE_FMT_MXFP4)
        return launch_expert_gemm<MODE, MOE_FMT_NVFP4, MOE_FMT_MXFP4>(L, slots_r, st);
    if (fr == MOE_FMT_MXFP4 && fs == MOE_FMT_NVFP4)
        return launch_expert_gemm<MODE, MOE_FMT_MXFP4, MOE_FMT_NVFP4>(L, slots_r, st);
    return launch_expert_gemm<MODE, MOE_FMT_MXFP4, MOE_FMT_MXFP4>(L, slots_r, st);
}

cudaError_t launch_ffn(const FfnLaunch& L, cudaStream_t st, const PhaseEvents* ev) {
    cudaError_t err = cudaSuccess;
#define MOE_PHASE(i, body)                                                  \
    if (ev && (err = record_phase_event(ev->begin[i], st)) != cudaSuccess) return err; \
    body;                                                                  \
    if ((err = cudaGetLastError()) != cudaSuccess) return err;             \
    if (ev && (err = record_phase_event(ev->end[i], st)) != cudaSuccess) return err;
    const int64_t n16 = (int64_t)L.T * L.H / 16;
    int conv_blocks = (int)((n16 + 511) / 512);
    if (conv_blocks > 4 * 152) conv_blocks = 4 * 152;
    if (conv_blocks < 1) conv_blocks = 1;
    const int slots_r = L.E < L.T * L.k ? L.E : L.T * L.k;
    const int64_t nthreads = (int64_t)L.T * (L.H / 8);
    MOE_PHASE(0, (prep_kernel<<<1 + conv_blocks, 512, 0, st>>>(L)))
    MOE_PHASE(1, launch_expert_phase<MODE_GATEUP>(L, slots_r, st))
    MOE_PHASE(2, launch_expert_phase<MODE_DOWN>(L, slots_r, st))
    MOE_PHASE(3, (combine_kernel<<<(unsigned)((nthreads + 255) / 256), 256, 0, st>>>(L)))
#undef MOE_PHASE
    return cudaSuccess;
}

cudaError_t launch_quantize_act(const void* x, int64_t rows, int64_t K, float g, uint8_t* packed,
                                uint8_t* scales, __half* deq16, cudaStream_t st) {
    const int64_t n16 = rows * K / 16;
    quantize_act_kernel<<<(unsigned)((n16 + 255) / 256), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), n16, g, packed, scales, deq16);
    return cudaGetLastError();
}

cudaError_t launch_mx_offsets(const uint8_t* scales, int E, int64_t per_expert, int32_t* off,
                              float* post, cudaStream_t st) {
    mx_offsets_kernel<<<E, 256, 0, st>>>(scales, per_expert, off, post);
    return cudaGetLastError();
}

}  // namespace moe
