// prefill_tc.cu -- the many-token expert FFN with NVFP4 activations on the sm_103a tensor
// cores (tcgen05, block-scaled E2M1 x E2M1 with UE4M3 scales per 16, accumulators in TMEM).
//
// The block-scaled FP4 x FP4 product is the spark_model prefill recipe (moe/mod.rs,
// `moe_fused_gate_up_t_k64_fp4` field doc: one block-scaled MMA per 64-element K tile, NVFP4
// activations from the `quantize_bf16_to_nvfp4` step of qwen3_attention/init.rs); the pages
// run it as warp-level MMAs on GB10, here it is tcgen05 with operands staged by TMA.
//
// Data flow (every step on the device, no host synchronisation):
//   tc_hist_kernel / tc_scan_kernel / tc_scatter_kernel  histogram of the routed pairs,
//                    expert rows padded to 128 (one MMA M tile), padded-row -> pair map,
//                    per-128-row block -> expert map, and the two tile lists (expert-major;
//                    gate+up then M block, then N block, so that concurrently running CTAs
//                    share one block of token rows and the expert's weight tiles stay in L2 for
//                    its next block; down then N block, then M block);
//   tc_quant_tokens_kernel / tc_gather_rows_kernel  NVFP4 quantization of every token once,
//                    then a copy of each pair's token row into its padded row with the scales
//                    rearranged into the 128 x 4 scale-factor tile layout of the MMA;
//   tc_gemm_kernel   (gate+up) D[128 pairs][128 gate | 128 up] over K = H; the epilogue
//                    computes h = SiLU(g) * u and requantizes it to NVFP4 (codes + scale tiles)
//                    as the next GEMM's activation operand;
//   tc_gemm_kernel   (down) D[128 pairs][256 outputs] over K = I; the epilogue applies the
//                    per-tensor global and the routing weight and stores bf16 rows per pair;
//   tc_combine_kernel  out[t] = sum_j y[t, j] + y_shared[t].
//
// The GEMM kernel is persistent (one CTA per SM, tiles strided by the grid) and warp
// specialised: warp 0 issues TMA / bulk copies into a 4-stage shared-memory ring, warp 1
// allocates TMEM and one of its lanes issues tcgen05.mma, warps 2-9 drain the accumulator with
// tcgen05.ld, warps 10-13 (one per TMEM lane quarter) write the stage's scale factors into
// TMEM with tcgen05.st.  Every mbarrier wait is bounded; a wait
// that gives up sets MOE_DEV_TIMEOUT, the CTA stops issuing work, waits (bounded) for its
// copies and MMAs in flight, frees TMEM and returns.  The file also holds the many-token
// router GEMM on the tensor cores (tcgen05.mma.kind::f16, bf16 in, fp32 logits).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "quant.cuh"
#include "tc_ptx.cuh"

namespace moe {

using namespace tc;

constexpr int kTcABytes = 128 * 128;          // 128 rows x 128 B (256 E2M1 codes)
constexpr int kTcBBytes = 256 * 128;          // 256 rows x 128 B
constexpr int kTcSfaBytes = 4 * 512;          // 4 K blocks of 64 x one 128-row scale tile
constexpr int kTcSfaOff = kTcABytes + kTcBBytes;
constexpr uint32_t kTcTmemCols = 512;  // 256 accumulator + 4 stages x 48 scale columns, rounded
                                       // up to the power of two an allocation takes
// Scale factors: the MMA reads the same 32 lanes x 8 columns per K block of B's scales, and the
// same 32 lanes x 4 columns of A's, from each of the four TMEM lane quarters.  A stage's B
// scales (for a 256-row block of B and its 4 K blocks, the 16-byte lines of both 128-row scale
// tiles in the order the 32 lanes of one quarter read them) are prepared once as one 4 KB tile,
// A's as 4 tiles of 512 B; both are bulk-copied into the stage once, and four scale warps, one
// per lane quarter, load them from shared memory and write them into their quarter with
// tcgen05.st.  That keeps the scale copies off the tensor pipe (a 128-lane tcgen05.cp needs a
// tile four times in shared memory, a copy that replicates 32 lanes to the four quarters costs
// the pipe several times more) and leaves room for a fourth stage: 4 stages of 54 KiB.
constexpr int kTcStages = 4;
constexpr int kTcSfbBytes = 4096;
constexpr int kTcSfbOff = kTcSfaOff + kTcSfaBytes;
constexpr int kTcStageBytes = kTcSfbOff + kTcSfbBytes;  // 55296 (54 KiB, 1 KiB multiple)
constexpr int kTcSmemBytes = kTcStages * kTcStageBytes + 1024 + 256;
constexpr int kTcThreads = 448;    // producer warp, MMA warp, 8 epilogue warps, 4 scale warps
constexpr int kTcScaleWarp0 = 10;
// Registers: each of the SM's four sub-partitions holds 16384, and 14 warps put four warps on
// two of them, so a thread may use at most 128 (the epilogue's 128-column slice spills a little).
constexpr int kTcMaxRegs = 128;
constexpr int kTcEpiThreads = 256;
constexpr uint64_t kTcWaitLimit = 1ull << 26;  // polls before a wait is declared stuck

// Byte offset of the scale of (row r of a 128-row block, 16-element block j of a 64-element
// K block) inside that K block's 512-byte scale tile: rows r, r+32, r+64, r+96 share one
// 16-byte line, which the 32x128b tcgen05.cp spreads over TMEM lanes and columns.
__host__ __device__ __forceinline__ int sf_tile_offset(int r, int j) {
    return (r & 31) * 16 + (r >> 5) * 4 + j;
}

// ------------------------------------------------------------------------------------------
// dispatch + tile lists: a histogram over many CTAs, a one-warp scan, then the scatter of the
// pairs into their experts' padded rows, the padding marks, the block -> expert map and both
// tile lists over many CTAs.  a.scan holds 5 arrays of E + 2: per-expert counts (zeroed before
// the histogram; entry E = the shared expert), 128-row block bases, gate+up and down tile
// bases, and row cursors.
// ------------------------------------------------------------------------------------------
struct TcScan {
    int32_t *cnt, *mbase, *tb1, *tb2, *cursor;
    __device__ TcScan(int32_t* s, int E)
        : cnt(s), mbase(s + (E + 2)), tb1(s + 2 * (E + 2)), tb2(s + 3 * (E + 2)), cursor(s + 4 * (E + 2)) {}
};

__device__ __forceinline__ bool tc_routed(int e, int E) { return e >= 0 && e < E; }

__global__ void __launch_bounds__(1024) tc_hist_kernel(TcPrepArgs a) {
    __shared__ int cnt[kMaxExperts];
    const int E = a.E, P = a.T * a.k;
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    int bad = 0;
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
        const int e = a.ids[p];
        if (tc_routed(e, E)) atomicAdd(&cnt[e], 1);
        else if (e != -1 && !(e >= E && e < E + a.Z)) bad = 1;  // zero-computation experts are valid
    }
    if (bad) status_or(a.status, MOE_DEV_BAD_EXPERT_ID);
    __syncthreads();
    TcScan S(a.scan, E);
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (cnt[e]) atomicAdd(&S.cnt[e], cnt[e]);
}

// one warp: exclusive scans over E + 1 entries (routed experts, then the shared one)
__global__ void __launch_bounds__(32) tc_scan_kernel(TcPrepArgs a) {
    const int E = a.E, lane = threadIdx.x, n = E + 1, per = (n + 31) / 32;
    TcScan S(a.scan, E);
    if (lane == 0) S.cnt[E] = a.has_shared ? a.T : 0;  // the shared expert takes every token
    __syncwarp();
    const int lo = min(n, lane * per), hi = min(n, lo + per);
    int smb = 0, st1 = 0, st2 = 0;
    for (int e = lo; e < hi; ++e) {
        const int nmb = (S.cnt[e] + 127) / 128;
        smb += nmb;
        st1 += nmb * ((e < E ? a.I : a.I_shared) / 128);
        st2 += nmb * (a.H / 256);
    }
    int i_mb = smb, i_t1 = st1, i_t2 = st2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, i_mb, o);
        const int y = __shfl_up_sync(0xffffffffu, i_t1, o);
        const int z = __shfl_up_sync(0xffffffffu, i_t2, o);
        if (lane >= o) { i_mb += x; i_t1 += y; i_t2 += z; }
    }
    int b = i_mb - smb, t1 = i_t1 - st1, t2 = i_t2 - st2;
    for (int e = lo; e < hi; ++e) {
        const int nmb = (S.cnt[e] + 127) / 128;
        S.mbase[e] = b;
        S.tb1[e] = t1;
        S.tb2[e] = t2;
        S.cursor[e] = b * 128;
        b += nmb;
        t1 += nmb * ((e < E ? a.I : a.I_shared) / 128);
        t2 += nmb * (a.H / 256);
    }
    if (lane == 31) {
        S.mbase[n] = i_mb;
        S.tb1[n] = i_t1;
        S.tb2[n] = i_t2;
        a.meta[0] = i_t1;        // gate+up tiles
        a.meta[1] = i_t2;        // down tiles
        a.meta[2] = i_mb * 128;  // padded rows in use
        a.meta[3] = i_mb;        // 128-row blocks in use
    }
}

__global__ void __launch_bounds__(1024) tc_scatter_kernel(TcPrepArgs a) {
    __shared__ int cnt[kMaxExperts + 1];
    __shared__ int mbase[kMaxExperts + 2];
    __shared__ int tb1[kMaxExperts + 2];
    __shared__ int tb2[kMaxExperts + 2];
    __shared__ int lcur[kMaxExperts];
    const int tid = threadIdx.x, E = a.E, P = a.T * a.k;
    TcScan S(a.scan, E);
    for (int e = tid; e <= E + 1; e += blockDim.x) {
        if (e <= E) cnt[e] = S.cnt[e];
        mbase[e] = S.mbase[e];
        tb1[e] = S.tb1[e];
        tb2[e] = S.tb2[e];
        if (e < E) lcur[e] = 0;
    }
    __syncthreads();
    // this CTA's contiguous share of the pairs: count per expert, reserve a range of rows per
    // expert with one global atomic, then place each pair inside its range
    const int chunk = (P + gridDim.x - 1) / gridDim.x;
    const int p0 = min(P, blockIdx.x * chunk), p1 = min(P, p0 + chunk);
    for (int p = p0 + tid; p < p1; p += blockDim.x) {
        const int e = a.ids[p];
        if (tc_routed(e, E)) atomicAdd(&lcur[e], 1);
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x)
        if (lcur[e]) lcur[e] = atomicAdd(&S.cursor[e], lcur[e]);
    __syncthreads();
    for (int p = p0 + tid; p < p1; p += blockDim.x) {
        const int e = a.ids[p];
        if (tc_routed(e, E)) a.padrow_pair[atomicAdd(&lcur[e], 1)] = p;
    }
    const int g = blockIdx.x * blockDim.x + tid, G = gridDim.x * blockDim.x;
    if (a.has_shared)
        for (int t = g; t < a.T; t += G) a.padrow_pair[mbase[E] * 128 + t] = P + t;
    // the unused tail of each expert's last block (fewer than 128 rows)
    for (int i = g; i < (E + 1) * 128; i += G) {
        const int e = i >> 7, row = mbase[e] * 128 + cnt[e] + (i & 127);
        if (row < mbase[e + 1] * 128) a.padrow_pair[row] = -1;
    }
    const int nblocks = mbase[E + 1];
    for (int b = g; b < nblocks; b += G) {
        int lo = 0, hi = E + 1;  // largest e with mbase[e] <= b
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (mbase[mid] <= b) lo = mid; else hi = mid;
        }
        a.mblock_expert[b] = lo;
    }
    // tile lists: entry = (128-row block, N block, expert (E = shared), K stages)
    for (int pass = 0; pass < 2; ++pass) {
        const int* tb = pass == 0 ? tb1 : tb2;
        int4* out = pass == 0 ? a.tiles1 : a.tiles2;
        const int total = tb[E + 1];
        for (int t = g; t < total; t += G) {
            int lo = 0, hi = E + 1;  // largest e with tb[e] <= t and a nonzero range
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (tb[mid] <= t) lo = mid; else hi = mid;
            }
            while (lo < E && tb[lo + 1] <= t) ++lo;  // skip experts with no tiles
            // gate+up: M block outer, N block inner -- the 16 tiles of one block of token rows
            // run at the same time (its rows are read once from HBM) and the expert's weight
            // tiles are reused from L2 by its next row block (at 32768 tokens this halves the
            // launch's DRAM reads); down: N block outer, M block inner (measured faster there)
            const int nmb = mbase[lo + 1] - mbase[lo];
            const int nnb = (lo < E ? a.I : a.I_shared) / 128;
            const int r = t - tb[lo];
            const int mb = pass == 0 ? r / nnb : r % nmb;
            const int nb = pass == 0 ? r % nnb : r / nmb;
            const int K = pass == 0 ? a.H : (lo < E ? a.I : a.I_shared);
            out[t] = make_int4(mbase[lo] + mb, nb, lo, K / 256);
        }
    }
}

// ------------------------------------------------------------------------------------------
// NVFP4 quantization of the tokens (once per token), then a copy into the padded,
// expert-sorted rows with the scales rearranged into the MMA's scale tiles
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tc_quant_tokens_kernel(TcQuantArgs a) {
    const int nb16 = a.H / 16;
    const int64_t total = (int64_t)a.T * nb16;
    const auto* x = static_cast<const __nv_bfloat16*>(a.x);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        float v[16];
        load_bf16x16(x + i * 16, v);
        quant16(v, a.g1, a.tokq + i * 8, a.toks + i, nullptr);
    }
}

// Warp items, strided over the grid's warps: first one per padded row in use -- the warp
// copies the codes of the row's token (7 independent 16-byte loads per lane at H 7168) --,
// then one per (128-row block, 16 K blocks) -- lane l builds line l of each K block's scale
// tile (the scales of rows l, l + 32, l + 64, l + 96; 512 contiguous bytes per K block) from
// 16-byte runs of its four tokens' scales.  Rows without a pair keep whatever codes they had
// and get zero scales, so they contribute nothing.
constexpr int kGatherThreads = 256;
__global__ void __launch_bounds__(kGatherThreads) tc_gather_rows_kernel(TcQuantArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * kGatherThreads + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * kGatherThreads) >> 5;
    const int nblk = a.meta[3], rows = nblk * 128;
    const int KB = a.H / 64, wpr = a.H / 32;  // K blocks (a multiple of 4), 16-byte code words per row
    const int kch = (KB + 15) / 16;
    const uint4* src = reinterpret_cast<const uint4*>(a.tokq);
    uint4* dst = reinterpret_cast<uint4*>(a.xq);
    auto token_of = [&](int row) {
        const int p = a.padrow_pair[row];
        return p < 0 ? -1 : (p < a.P ? p / a.k : p - a.P);
    };
    const int64_t items = (int64_t)rows + (int64_t)nblk * kch;
    for (int64_t it = gw; it < items; it += nw) {
        if (it < rows) {
            const int row = (int)it;
            const int t = token_of(row);
            if (t < 0) continue;
            const uint4* s = src + (size_t)t * wpr;
            uint4* d = dst + (size_t)row * wpr;
            for (int w0 = 0; w0 < wpr; w0 += 8 * 32) {
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int w = w0 + 32 * u + lane;
                    if (w < wpr) v[u] = s[w];
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int w = w0 + 32 * u + lane;
                    if (w < wpr) d[w] = v[u];
                }
            }
        } else {
            const int64_t j = it - rows;
            const int mb = (int)(j / kch), kb0 = 16 * (int)(j - (int64_t)mb * kch);
            const int kb1 = min(KB, kb0 + 16);
            int tk[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) tk[q] = token_of(mb * 128 + 32 * q + lane);
            for (int kb = kb0; kb < kb1; kb += 4) {
                uint4 s4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    s4[q] = tk[q] < 0 ? make_uint4(0u, 0u, 0u, 0u)
                                      : *reinterpret_cast<const uint4*>(a.toks + ((size_t)tk[q] * KB + kb) * 4);
                uint8_t* line = a.xsf + ((size_t)mb * KB + kb) * 512 + 16 * lane;
                *reinterpret_cast<uint4*>(line) = make_uint4(s4[0].x, s4[1].x, s4[2].x, s4[3].x);
                *reinterpret_cast<uint4*>(line + 512) = make_uint4(s4[0].y, s4[1].y, s4[2].y, s4[3].y);
                *reinterpret_cast<uint4*>(line + 1024) = make_uint4(s4[0].z, s4[1].z, s4[2].z, s4[3].z);
                *reinterpret_cast<uint4*>(line + 1536) = make_uint4(s4[0].w, s4[1].w, s4[2].w, s4[3].w);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// the tcgen05 grouped GEMM
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tc_abort(TcGemmParams const& p, volatile int* flag) {
    *flag = 1;
    status_or(p.status, MOE_DEV_TIMEOUT);
}

// MODE 0: gate+up (epilogue h = SiLU(g) * u, requantized); MODE 1: down (epilogue bf16 pair
// rows).  p.mode must match.
template <int MODE>
__global__ void __maxnreg__(kTcMaxRegs)
tc_gemm_kernel(const __grid_constant__ TcTensorMaps maps, const TcGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTcStages * kTcStageBytes);
    uint64_t* empty = full + kTcStages;
    uint64_t* acc_full = empty + kTcStages;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain = acc_empty + 1;
    uint64_t* sfr = drain + 1;  // per stage: B's scales are in TMEM (one arrival per scale warp)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfr + kTcStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sfr[s], 4);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kTcEpiThreads);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&maps.a);
        prefetch_tmap(&maps.b0);
        prefetch_tmap(&maps.b1);
        prefetch_tmap(&maps.sb0);
        prefetch_tmap(&maps.sb1);
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTcTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int ntiles = p.num_tiles[0];

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            for (int tile = blockIdx.x; tile < ntiles && !*abort_flag; tile += gridDim.x) {
                const int4 tl = p.tiles[tile];
                const int b = tl.x, nb = tl.y, e = tl.z, kst = tl.w;
                const bool sh = e == p.E;
                const int es = sh ? 0 : e;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, kTcWaitLimit)) {
                        tc_abort(p, abort_flag);
                        break;
                    }
                    if (*abort_flag) break;
                    uint8_t* base = smem + stage * kTcStageBytes;
                    mbar_arrive_expect_tx(&full[stage], kTcStageBytes);
                    const int xb = ks * 128;
                    tma_load_2d(base, &maps.a, xb, b * 128, &full[stage]);
                    bulk_load(base + kTcSfaOff, p.sfa + ((size_t)b * p.sfa_kblocks + 4 * ks) * 512,
                              kTcSfaBytes, &full[stage]);
                    if (MODE == 0) {
                        const int N = sh ? p.I_shared : p.I;
                        const int row = es * N + nb * 128;
                        tma_load_2d(base + kTcABytes, sh ? &maps.sb0 : &maps.b0, xb, row, &full[stage]);
                        tma_load_2d(base + kTcABytes + 16384, sh ? &maps.sb1 : &maps.b1, xb, row,
                                    &full[stage]);
                        const size_t tix = ((size_t)es * (N / 128) + nb) * (p.H / 64) + 4 * ks;
                        const uint8_t* q4 = (sh ? p.ssfb0 : p.sfb0) + tix * 1024;  // quarter tile
                        bulk_load(base + kTcSfbOff, q4, kTcSfbBytes, &full[stage]);
                    } else {
                        const int K = sh ? p.I_shared : p.I;
                        const int row = es * p.H + nb * 256;
                        tma_load_2d(base + kTcABytes, sh ? &maps.sb0 : &maps.b0, xb, row, &full[stage]);
                        const uint8_t* q4 = (sh ? p.ssfb0 : p.sfb0) +
                                            (((size_t)es * (p.H / 256) + nb) * (K / 64) + 4 * ks) * 1024;
                        bulk_load(base + kTcSfbOff, q4, kTcSfbBytes, &full[stage]);
                    }
                    ++issued;
                    if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (*abort_flag) {
                // wait (bounded) for the copies this thread may still have in flight
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < kTcStages && i < issued; ++i) {
                    if (--s < 0) { s = kTcStages - 1; ph ^= 1u; }
                    mbar_wait_bounded(&full[s], ph, kTcWaitLimit);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            const uint32_t idesc = idesc_fp4(128, 256, 0);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool any = false;
            for (int tile = blockIdx.x; tile < ntiles && !*abort_flag; tile += gridDim.x) {
                const int kst = p.tiles[tile].w;
                if (!mbar_wait_bounded(acc_empty, acc_phase ^ 1u, kTcWaitLimit)) {
                    tc_abort(p, abort_flag);
                    break;
                }
                tc_fence_after();
                bool ok = true;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!mbar_wait_bounded(&full[stage], phase, kTcWaitLimit) ||
                        !mbar_wait_bounded(&sfr[stage], phase, kTcWaitLimit) || *abort_flag) {
                        tc_abort(p, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint8_t* base = smem + stage * kTcStageBytes;
                    const uint32_t sbase = smem_u32(base);
                    const uint32_t sfcol = 256 + stage * 48;
                    // scale columns of the stage (written by the scale warps), per K block j:
                    // B's 8 at +8 j, A's 4 at +32 + 4 j
                    uint32_t sfa_c[4], sfb_c[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        sfb_c[j] = tmem + sfcol + 8 * j;
                        sfa_c[j] = tmem + sfcol + 32 + 4 * j;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t ad = smem_desc(sbase + 32 * j, 16, 1024, kLayoutSw128);
                        const uint64_t bd = smem_desc(sbase + kTcABytes + 32 * j, 16, 1024, kLayoutSw128);
                        tc_mma_nvf4(tmem, ad, bd, idesc, sfa_c[j], sfb_c[j], (ks | j) != 0 ? 1u : 0u);
                    }
                    any = true;
                    tc_commit(&empty[stage]);
                    if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(acc_full);
                acc_phase ^= 1u;
            }
            if (any) {  // every MMA this thread issued has completed before TMEM is freed
                tc_commit(drain);
                mbar_wait_bounded(drain, 0, kTcWaitLimit);
            }
        }
    } else if (warp >= kTcScaleWarp0) {
        // ---------------- scales into TMEM (warps 10..13, lane quarter warp % 4) ----------
        // Lane l of every quarter takes, per K block j, the 32 bytes of line l of the stage's
        // B quarter tile (16 B at 1 KB (l / 8) + 256 j + 16 (l % 8) and 16 B at +128) into
        // columns 8 j .. 8 j + 7 of the stage's scale columns, and line l of A's K-block tile j
        // (16 B at 512 j + 16 l: rows l, l + 32, l + 64, l + 96) into columns 32 + 4 j .. +3.
        const uint32_t qlane = (uint32_t)((warp & 3) * 32) << 16;
        const int loff = 1024 * (lane >> 3) + 16 * (lane & 7);
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = blockIdx.x; tile < ntiles && !*abort_flag; tile += gridDim.x) {
            const int kst = p.tiles[tile].w;
            bool ok = true;
            for (int ks = 0; ks < kst; ++ks) {
                // the whole warp takes one decision (tcgen05.st below is warp-wide)
                const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&full[stage], phase, kTcWaitLimit) &&
                                                             !*abort_flag);
                if (!got) {
                    if (lane == 0) tc_abort(p, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* src = smem + stage * kTcStageBytes + kTcSfbOff + loff;
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 lo = *reinterpret_cast<const uint4*>(src + 256 * j);
                    const uint4 hi = *reinterpret_cast<const uint4*>(src + 256 * j + 128);
                    v[8 * j + 0] = lo.x; v[8 * j + 1] = lo.y; v[8 * j + 2] = lo.z; v[8 * j + 3] = lo.w;
                    v[8 * j + 4] = hi.x; v[8 * j + 5] = hi.y; v[8 * j + 6] = hi.z; v[8 * j + 7] = hi.w;
                }
                const uint8_t* sa = smem + stage * kTcStageBytes + kTcSfaOff + 16 * lane;
                uint32_t u[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 a = *reinterpret_cast<const uint4*>(sa + 512 * j);
                    u[4 * j + 0] = a.x; u[4 * j + 1] = a.y; u[4 * j + 2] = a.z; u[4 * j + 3] = a.w;
                }
                tmem_st_32(tmem + qlane + 256 + stage * 48, v);
                tmem_st_16(tmem + qlane + 256 + stage * 48 + 32, u);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sfr[stage]);
                if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
        }
    } else {
        // ---------------- epilogue (warps 2..9) ----------------
        // Two warps per TMEM lane quarter, each owning half of the tile's columns (128): a warp
        // reads its slice in two halves and releases the accumulator once the second half is
        // in registers, so the next tile's MMAs run while it finishes computing and storing.
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = quad * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t acc_phase = 0;
        // this row's pair, row block, N block and scales, read one tile ahead (dependent loads,
        // so they are not waited for between a tile's MMAs and the release of its accumulator):
        // gate+up the two post-scales, down the output scale (post-scale x routing weight)
        int pair_n = -1, b_n = 0, nb_n = 0;
        float s0_n = 0.f, s1_n = 0.f;
        auto row_scale = [&](int tile) {
            if (tile >= ntiles) return;
            const int4 tl = p.tiles[tile];
            const bool sh = tl.z == p.E;
            const int es = sh ? 0 : tl.z;
            pair_n = p.padrow_pair[tl.x * 128 + r];
            b_n = tl.x;
            nb_n = tl.y;
            s0_n = (sh ? p.spost0 : p.post0)[es];
            if (MODE == 0) s1_n = (sh ? p.spost1 : p.post1)[es];
            else s0_n = pair_n < 0 ? 0.f : s0_n * (pair_n < p.P ? p.topk_w[pair_n] : 1.f);
        };
        row_scale(blockIdx.x);
        const uint64_t ypol = MODE == 1 ? l2_policy_evict_first() : 0ull;  // down: the pair rows
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            if (!mbar_wait_bounded(acc_full, acc_phase, kTcWaitLimit)) {
                tc_abort(p, abort_flag);
                break;
            }
            if (*abort_flag) break;
            tc_fence_after();
            if constexpr (MODE == 1) {
                // output columns [128 half, +128) in two halves, packed to bf16 as they arrive,
                // so a thread holds 64 packed words instead of 128 accumulators
                const int pair = pair_n, nb = nb_n;
                const float sc = s0_n;
                uint32_t P[64];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t W[64];
#pragma unroll
                    for (int c = 0; c < 64; c += 16)
                        tmem_ld_16(trow + 128 * half + 64 * hh + c, *reinterpret_cast<uint32_t(*)[16]>(W + c));
                    tmem_ld_wait();
                    if (hh == 1) {
                        tc_fence_before();
                        mbar_arrive(acc_empty);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(W[2 * i]) * sc,
                                                                 __uint_as_float(W[2 * i + 1]) * sc);
                        P[32 * hh + i] = *reinterpret_cast<uint32_t*>(&v);
                    }
                }
                acc_phase ^= 1u;
                row_scale(tile + gridDim.x);
                if (pair < 0) continue;
                // 32-byte stores (the row segment is 256 B, 32-byte aligned): half as many
                // scattered store transactions as 16-byte ones.  The pair rows are read once, by
                // the combine after this launch, so they go to L2 evict-first and leave the
                // GEMM's operand tiles in place (32768 tokens: 4.2 GB of rows; the layer step
                // 7.75 -> 7.62 ms).
                __nv_bfloat16* dst = p.y + (size_t)pair * p.H + nb * 256 + 128 * half;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_global_v8_hint(dst + 16 * c, *reinterpret_cast<const uint32_t(*)[8]>(P + 8 * c), ypol);
            } else {
                // gate columns [64 half, +64) and up columns [128 + 64 half, +64), in two halves
                // of 32 + 32: the first half's h is computed and requantized before the second
                // half is read, so a thread holds 64 accumulators instead of 128
                const int pair = pair_n, b = b_n, nb = nb_n;
                const float pg = s0_n, pu = s1_n;
                const int prow = b * 128 + r;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t Gw[32], Uw[32];
#pragma unroll
                    for (int c = 0; c < 32; c += 16) {
                        tmem_ld_16(trow + 64 * half + 32 * hh + c, *reinterpret_cast<uint32_t(*)[16]>(Gw + c));
                        tmem_ld_16(trow + 128 + 64 * half + 32 * hh + c, *reinterpret_cast<uint32_t(*)[16]>(Uw + c));
                    }
                    tmem_ld_wait();
                    if (hh == 1) {
                        tc_fence_before();
                        mbar_arrive(acc_empty);
                    }
                    if (pair >= 0) {
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk) {
                            float h[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float gv = __uint_as_float(Gw[16 * blk + i]) * pg;
                                const float uv = __uint_as_float(Uw[16 * blk + i]) * pu;
                                h[i] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                            }
                            const int i = nb * 128 + 64 * half + 32 * hh + 16 * blk;
                            uint8_t* sf = p.hsf + ((size_t)b * p.hsf_kblocks + (i >> 6)) * 512 +
                                          sf_tile_offset(r, (i >> 4) & 3);
                            quant16_rcp(h, p.g2, p.hq + (size_t)prow * p.hq_row_bytes + i / 2, sf);
                        }
                    }
                }
                acc_phase ^= 1u;
                row_scale(tile + gridDim.x);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTcTmemCols);
    }
}

// ------------------------------------------------------------------------------------------
// combine: out[t] = sum_j y[t*k + j] (valid pairs) + y[P + t]
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tc_combine_kernel(TcCombineArgs a) {
    const int H8 = a.H / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)a.T * H8) return;
    const int t = (int)(idx / H8), c = (int)(idx - (int64_t)t * H8);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    auto add = [&](int row) {
        const uint4 v = *reinterpret_cast<const uint4*>(a.y + (size_t)row * a.H + c * 8);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] += __uint_as_float(w[i] << 16);
            acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
        }
    };
    float zw = 0.f;  // folded weight of the zero-computation experts
    for (int j = 0; j < a.k; ++j) {
        const int e = a.ids[t * a.k + j];
        if (e >= 0 && e < a.E) add(t * a.k + j);
        else if (e >= a.E && e < a.E + a.Z) zw += a.w[t * a.k + j];
    }
    if (a.has_shared) add(a.T * a.k + t);
    if (zw != 0.f) {
        const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) +
                                                         (size_t)t * a.H + c * 8);
        const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] += zw * __uint_as_float(xw[i] << 16);
            acc[2 * i + 1] += zw * __uint_as_float(xw[i] & 0xFFFF0000u);
        }
    }
    uint4 o;
    uint32_t* ow = &o.x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        ow[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + (size_t)t * a.H)[c] = o;
}

// ------------------------------------------------------------------------------------------
// weight preparation: scale-factor tiles and tensor maps
// ------------------------------------------------------------------------------------------
// out[((e * N/128 + rb) * K/64 + kb) * 512 + sf_tile_offset(r, j)] = in[e][rb*128 + r][kb*4 + j]
__global__ void sf_tiles_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out,
                                int E, int N, int K) {
    const int64_t total = (int64_t)E * N * (K / 16);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int kk = (int)(i % (K / 16));
        const int64_t row = i / (K / 16);
        const int e = (int)(row / N), n = (int)(row % N);
        const int rb = n >> 7, r = n & 127, kb = kk >> 2, j = kk & 3;
        out[(((size_t)e * (N / 128) + rb) * (K / 64) + kb) * 512 + sf_tile_offset(r, j)] = in[i];
    }
}

// MXFP4: block scale 2^(b - 127) = 2^d * 2^(bmax - 135) with d = b - bmax + 8 <= 8, written as
// the E4M3 byte of 2^d (exact for d >= -9; smaller blocks flush to zero); 32-element blocks
// become two 16-element ones.  post[e] = 2^(bmax - 135), bmax = off[e] + 139.
__device__ __forceinline__ uint8_t e8m0_as_e4m3(int b, int bmax) {
    const int d = b - bmax + 8;
    if (d >= -6) return (uint8_t)((d + 7) << 3);
    if (d >= -9) return (uint8_t)(1 << (d + 9));
    return 0;
}

__global__ void sf_tiles_mx_kernel(const uint8_t* __restrict__ in, const int32_t* __restrict__ off,
                                   uint8_t* __restrict__ out, float* __restrict__ post, int E,
                                   int N, int K) {
    const int64_t total = (int64_t)E * N * (K / 16);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int kk = (int)(i % (K / 16));
        const int64_t row = i / (K / 16);
        const int e = (int)(row / N), n = (int)(row % N);
        const int bmax = off[e] + 139;
        const int b = in[row * (K / 32) + kk / 2];
        const int rb = n >> 7, r = n & 127, kb = kk >> 2, j = kk & 3;
        out[(((size_t)e * (N / 128) + rb) * (K / 64) + kb) * 512 + sf_tile_offset(r, j)] =
            e8m0_as_e4m3(b, bmax);
        if (i < E) post[i] = ldexpf(1.0f, off[i] + 4);  // 2^(bmax - 135)
    }
}

// Quarter tiles of B's scales: the lines of the two 128-row scale tiles t = 0, 1 (tile index
// pidx * mul + add_t of src_t) of a pair's four K blocks of a K-stage, laid out as the 32 TMEM
// lanes of one lane quarter read them (4 KB): a stage's scales are this 4 KB copied to each of
// the four quarters' shared-memory slices.
__global__ void sf_pair_kernel(const uint8_t* __restrict__ src0, const uint8_t* __restrict__ src1,
                               uint8_t* __restrict__ out, int64_t npairs, int kblocks, int mul,
                               int add0, int add1) {
    const int64_t total = npairs * kblocks * 64;  // 16-byte pieces
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int piece = (int)(i & 63);  // line l of tile t
        const int64_t pk = i >> 6;          // pair * kblocks + kb
        const int64_t pidx = pk / kblocks;
        const int kb = (int)(pk - pidx * kblocks);
        const int t = piece >> 5, l = piece & 31;
        const uint8_t* src = t ? src1 : src0;
        const int64_t tile = pidx * mul + (t ? add1 : add0);
        const uint4 v = *reinterpret_cast<const uint4*>(src + (tile * kblocks + kb) * 512 + l * 16);
        // per pair and K-stage (4 K blocks) 4 KB: 8-line group g = l / 8 at 1 KB steps, K block
        // at 256 B, tile at 128 B, line in group at 16 B
        *reinterpret_cast<uint4*>(out + (pidx * kblocks + (kb & ~3)) * 1024 + (l >> 3) * 1024 +
                                  (kb & 3) * 256 + t * 128 + (l & 7) * 16) = v;
    }
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2D map over a [rows][row_bytes] uint8 matrix, 128-byte x box_rows boxes, 128B swizzle.
static bool encode_rows(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
                        uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn || rows < box_rows || row_bytes % 128) return false;
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale tiles of one projection; for MXFP4 also its MMA-path post-scales (owned).
static cudaError_t make_sf_tiles(const ProjView& pv, int E, int N, int K, uint8_t** out,
                                 const float** post, float** owned, cudaStream_t st) {
    const size_t bytes = (size_t)E * N * (K / 16);
    cudaError_t err = cudaMalloc(out, bytes);
    if (err != cudaSuccess) return err;
    if (pv.fmt == MOE_FMT_NVFP4) {
        sf_tiles_kernel<<<1024, 256, 0, st>>>(pv.scales, *out, E, N, K);
        *post = pv.post;
    } else {
        if ((err = cudaMalloc(owned, sizeof(float) * E)) != cudaSuccess) return err;
        sf_tiles_mx_kernel<<<1024, 256, 0, st>>>(pv.scales, pv.mx_off, *out, *owned, E, N, K);
        *post = *owned;
    }
    return cudaGetLastError();
}

// Quarter tiles from compact tiles: npairs pairs of K / 64 blocks.
static cudaError_t make_pairs(uint8_t** out, uint8_t* src0, uint8_t* src1, int64_t npairs, int K,
                              int mul, int add0, int add1, cudaStream_t st) {
    cudaError_t err = cudaMalloc(out, (size_t)npairs * (K / 64) * 1024);
    if (err != cudaSuccess) return err;
    sf_pair_kernel<<<1024, 256, 0, st>>>(src0, src1, *out, npairs, K / 64, mul, add0, add1);
    return cudaGetLastError();
}

bool tc_supported(int E, int H, int I, int I_shared, int fmt_routed, int fmt_shared) {
    (void)E;
    return tc_shape_ok(H, I, I_shared, fmt_routed, fmt_shared) && encode_fn() != nullptr;
}

cudaError_t tc_prepare(const FfnLaunch& L, TcWeights* tw, cudaStream_t st) {
    *tw = TcWeights{};
    const int E = L.E, H = L.H, I = L.I, Is = L.I_shared;
    cudaError_t err;
    if ((err = make_sf_tiles(L.gate, E, I, H, &tw->sf_gate, &tw->post_gate, &tw->owned_post[0], st)) != cudaSuccess) return err;
    if ((err = make_sf_tiles(L.up, E, I, H, &tw->sf_up, &tw->post_up, &tw->owned_post[1], st)) != cudaSuccess) return err;
    if ((err = make_sf_tiles(L.down, E, H, I, &tw->sf_down, &tw->post_down, &tw->owned_post[2], st)) != cudaSuccess) return err;
    bool ok = encode_rows(&tw->gate, L.gate.packed, H / 2, (uint64_t)E * I, 128) &&
              encode_rows(&tw->up, L.up.packed, H / 2, (uint64_t)E * I, 128) &&
              encode_rows(&tw->down, L.down.packed, I / 2, (uint64_t)E * H, 256);
    if (Is > 0) {
        if ((err = make_sf_tiles(L.sh_gate, 1, Is, H, &tw->sf_sh_gate, &tw->post_sh_gate, &tw->owned_post[3], st)) != cudaSuccess) return err;
        if ((err = make_sf_tiles(L.sh_up, 1, Is, H, &tw->sf_sh_up, &tw->post_sh_up, &tw->owned_post[4], st)) != cudaSuccess) return err;
        if ((err = make_sf_tiles(L.sh_down, 1, H, Is, &tw->sf_sh_down, &tw->post_sh_down, &tw->owned_post[5], st)) != cudaSuccess) return err;
        ok = ok && encode_rows(&tw->sh_gate, L.sh_gate.packed, H / 2, Is, 128) &&
             encode_rows(&tw->sh_up, L.sh_up.packed, H / 2, Is, 128) &&
             encode_rows(&tw->sh_down, L.sh_down.packed, Is / 2, H, 256);
    }
    if (!ok) return cudaErrorInvalidValue;
    // B's scales as quarter tiles: gate | up per 128-row block, 256-row blocks of down; the
    // compact tiles they are built from are freed
    if ((err = make_pairs(&tw->sfp_gu, tw->sf_gate, tw->sf_up, (int64_t)E * (I / 128), H, 1, 0, 0, st)) != cudaSuccess) return err;
    if ((err = make_pairs(&tw->sfp_dn, tw->sf_down, tw->sf_down, (int64_t)E * (H / 256), I, 2, 0, 1, st)) != cudaSuccess) return err;
    if (Is > 0) {
        if ((err = make_pairs(&tw->sfp_sh_gu, tw->sf_sh_gate, tw->sf_sh_up, Is / 128, H, 1, 0, 0, st)) != cudaSuccess) return err;
        if ((err = make_pairs(&tw->sfp_sh_dn, tw->sf_sh_down, tw->sf_sh_down, H / 256, Is, 2, 0, 1, st)) != cudaSuccess) return err;
    }
    if ((err = cudaStreamSynchronize(st)) != cudaSuccess) return err;
    for (uint8_t** b : {&tw->sf_gate, &tw->sf_up, &tw->sf_down, &tw->sf_sh_gate, &tw->sf_sh_up, &tw->sf_sh_down}) {
        if (*b) cudaFree(*b);
        *b = nullptr;
    }
    for (auto kern : {tc_gemm_kernel<0>, tc_gemm_kernel<1>}) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
        if (err != cudaSuccess) return err;
    }
    tw->ready = true;
    return cudaSuccess;
}

void tc_release(TcWeights* tw) {
    uint8_t* bufs[10] = {tw->sf_gate, tw->sf_up, tw->sf_down, tw->sf_sh_gate, tw->sf_sh_up,
                         tw->sf_sh_down, tw->sfp_gu, tw->sfp_dn, tw->sfp_sh_gu, tw->sfp_sh_dn};
    for (uint8_t* b : bufs)
        if (b) cudaFree(b);
    for (float* f : tw->owned_post)
        if (f) cudaFree(f);
    *tw = TcWeights{};
}

// ------------------------------------------------------------------------------------------
// Router logits of many tokens on the tensor cores: logits[t][e] = x[t] . W_r[e] (bf16 in,
// fp32 out), one 128-token x 128-expert tile and one half of K = H per CTA: the two halves are
// added into the zeroed logits with fp32 atomics (exactly two addends onto zero, so the result
// does not depend on their order), which doubles the CTAs a few tiles give.  Warp 0 issues the
// TMA loads into a 4-stage ring (64 elements of K per stage, 128-byte swizzled rows), one lane
// of warp 1 issues tcgen05.mma.kind::f16 (M 128, N 128, K 16; four per stage) into a 128-column
// TMEM accumulator, warps 2-5 (one per lane quarter) read it back and write fp32 rows.  Every
// wait is bounded: a wait that gives up sets MOE_DEV_TIMEOUT and the CTA winds down.
// ------------------------------------------------------------------------------------------
constexpr int kRtStages = 4;
constexpr int kRtStageBytes = 2 * 128 * 128;  // A and B: 128 rows x 128 B each
constexpr int kRtSmemBytes = kRtStages * kRtStageBytes + 1024 + 256;
constexpr int kRtThreads = 192;

struct RtMaps {
    CUtensorMap x, w;
};

__global__ void __launch_bounds__(kRtThreads, 1)
router_tc_kernel(const __grid_constant__ RtMaps maps, float* __restrict__ logits, int T, int E,
                 int H, int32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRtStages * kRtStageBytes);
    uint64_t* empty = full + kRtStages;
    uint64_t* acc_full = empty + kRtStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * 128, e0 = blockIdx.y * 128;
    const int nk = H / 128, k0 = blockIdx.z * nk;  // this CTA's half of the 64-element K steps
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRtStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.w);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto give_up = [&]() {
        *abort_flag = 1;
        if (status) status_or(status, MOE_DEV_TIMEOUT);
    };
    if (warp == 0 && lane == 0) {  // TMA producer
        int issued = 0;
        for (int ks = 0; ks < nk && !*abort_flag; ++ks) {
            const int s = ks % kRtStages;
            const uint32_t ph = (ks / kRtStages) & 1u;
            const int kx = (k0 + ks) * 128;  // bytes along the bf16 row
            if (!mbar_wait_bounded(&empty[s], ph ^ 1u, kTcWaitLimit)) {
                give_up();
                break;
            }
            uint8_t* base = smem + s * kRtStageBytes;
            mbar_arrive_expect_tx(&full[s], kRtStageBytes);
            tma_load_2d(base, &maps.x, kx, t0, &full[s]);
            tma_load_2d(base + 128 * 128, &maps.w, kx, e0, &full[s]);
            ++issued;
        }
        if (*abort_flag)  // wait (bounded) for the copies still in flight
            for (int i = issued - 1; i >= 0 && i >= issued - kRtStages; --i)
                mbar_wait_bounded(&full[i % kRtStages], (i / kRtStages) & 1u, kTcWaitLimit);
    } else if (warp == 1 && lane == 0) {  // MMA issuer
        const uint32_t idesc = idesc_bf16(128, 128);
        bool any = false;
        for (int ks = 0; ks < nk; ++ks) {
            const int s = ks % kRtStages;
            if (!mbar_wait_bounded(&full[s], (ks / kRtStages) & 1u, kTcWaitLimit) || *abort_flag) {
                give_up();
                break;
            }
            tc_fence_after();
            const uint32_t sbase = smem_u32(smem + s * kRtStageBytes);
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // K 16 per MMA: 32 bytes along the swizzled row
                const uint64_t ad = smem_desc(sbase + 32 * j, 16, 1024, kLayoutSw128);
                const uint64_t bd = smem_desc(sbase + 128 * 128 + 32 * j, 16, 1024, kLayoutSw128);
                tc_mma_bf16(tmem, ad, bd, idesc, (ks | j) != 0 ? 1u : 0u);
            }
            any = true;
            tc_commit(&empty[s]);
        }
        if (any) {
            tc_commit(acc_full);  // every MMA has completed when this arrives
            mbar_wait_bounded(acc_full, 0, kTcWaitLimit);  // before TMEM can be freed
        } else if (!*abort_flag) {
            give_up();
        }
    } else if (warp >= 2) {  // epilogue: lane quarter q reads rows 32 q .. 32 q + 31
        const int q = warp & 3;
        const int t = t0 + 32 * q + lane;
        bool ok = mbar_wait_bounded(acc_full, 0, kTcWaitLimit);
        if (ok && !*abort_flag) {
            tc_fence_after();
            const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
#pragma unroll
            for (int c = 0; c < 128; c += 32) {
                uint32_t v[32];
                tmem_ld_16(trow + c, *reinterpret_cast<uint32_t(*)[16]>(v));
                tmem_ld_16(trow + c + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
                tmem_ld_wait();
                if (t < T) {
                    float* dst = logits + (size_t)t * E + e0 + c;
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        red_add_v4(dst + i, __uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                   __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                }
            }
        } else if (!ok) {
            give_up();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

cudaError_t launch_router_tc(const void* x, const void* wr, float* logits, int T, int E, int H,
                             int32_t* status, cudaStream_t st) {
    if (T < 128 || E % 128 != 0 || H % 128 != 0 || encode_fn() == nullptr) return cudaErrorNotSupported;
    // TMA sources 16-byte aligned, 16-byte vector reductions
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(wr)) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(logits) % 32 != 0)
        return cudaErrorNotSupported;
    RtMaps m{};
    if (!encode_rows(&m.x, x, (uint64_t)H * 2, (uint64_t)T, 128) ||
        !encode_rows(&m.w, wr, (uint64_t)H * 2, (uint64_t)E, 128))
        return cudaErrorNotSupported;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kRtSmemBytes);
        if (err != cudaSuccess) return err;
        attr_set = true;
    }
    cudaError_t err = cudaMemsetAsync(logits, 0, sizeof(float) * (size_t)T * E, st);
    if (err != cudaSuccess) return err;
    router_tc_kernel<<<dim3((T + 127) / 128, E / 128, 2), kRtThreads, kRtSmemBytes, st>>>(m, logits, T, E, H, status);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
cudaError_t launch_ffn_tc(const FfnLaunch& L, const TcWeights& tw, const TcBuffers& B,
                          cudaStream_t st, const PhaseEvents* ev) {
    const int Imax = L.I > L.I_shared ? L.I : L.I_shared;
    const int P = L.T * L.k;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t err = cudaSuccess;
#define TC_PHASE(i, body)                                                            \
    if (ev && (err = record_phase_event(ev->begin[i], st)) != cudaSuccess) return err; \
    body;                                                                           \
    if ((err = cudaGetLastError()) != cudaSuccess) return err;                      \
    if (ev && (err = record_phase_event(ev->end[i], st)) != cudaSuccess) return err;

    TcPrepArgs pa{};
    pa.ids = L.ids; pa.T = L.T; pa.k = L.k; pa.E = L.E; pa.Z = L.Z; pa.H = L.H; pa.I = L.I;
    pa.I_shared = L.I_shared; pa.has_shared = L.I_shared > 0; pa.status = L.status;
    pa.meta = B.meta; pa.mblock_expert = B.mblock_expert; pa.padrow_pair = B.padrow_pair;
    pa.tiles1 = B.tiles1; pa.tiles2 = B.tiles2; pa.scan = B.scan;
    TcQuantArgs qa{};
    qa.x = L.x; qa.T = L.T; qa.H = L.H; qa.k = L.k; qa.P = P; qa.g1 = L.g1; qa.meta = B.meta;
    qa.padrow_pair = B.padrow_pair; qa.tokq = B.tokq; qa.toks = B.toks; qa.xq = B.xq; qa.xsf = B.xsf;
    const int hist_ctas = (int)std::min<int64_t>(2 * sms, std::max<int64_t>(1, ((int64_t)P + 4095) / 4096));
    if ((err = cudaMemsetAsync(B.scan, 0, sizeof(int32_t) * (L.E + 2), st)) != cudaSuccess) return err;
    TC_PHASE(0, (tc_hist_kernel<<<hist_ctas, 1024, 0, st>>>(pa),
                 tc_scan_kernel<<<1, 32, 0, st>>>(pa),
                 tc_scatter_kernel<<<sms, 1024, 0, st>>>(pa),
                 tc_quant_tokens_kernel<<<sms * 8, 256, 0, st>>>(qa),
                 tc_gather_rows_kernel<<<sms * 8, kGatherThreads, 0, st>>>(qa)))

    TcTensorMaps m1{}, m2{};
    const uint64_t rows = (uint64_t)B.max_blocks * 128;
    if (!encode_rows(&m1.a, B.xq, L.H / 2, rows, 128) ||
        !encode_rows(&m2.a, B.hq, Imax / 2, rows, 128))
        return cudaErrorInvalidValue;
    m1.b0 = tw.gate; m1.b1 = tw.up; m1.sb0 = tw.sh_gate; m1.sb1 = tw.sh_up;
    m2.b0 = tw.down; m2.b1 = tw.down; m2.sb0 = tw.sh_down; m2.sb1 = tw.sh_down;
    if (L.I_shared == 0) { m1.sb0 = tw.gate; m1.sb1 = tw.up; m2.sb0 = tw.down; m2.sb1 = tw.down; }

    TcGemmParams g{};
    g.E = L.E; g.H = L.H; g.I = L.I; g.I_shared = L.I_shared; g.k = L.k; g.T = L.T; g.P = P;
    g.mblock_expert = B.mblock_expert; g.padrow_pair = B.padrow_pair; g.topk_w = L.w;
    g.status = L.status; g.g2 = L.g2;
    g.hq = B.hq; g.hsf = B.hsf; g.hq_row_bytes = Imax / 2; g.hsf_kblocks = Imax / 64;
    g.y = B.y;

    TcGemmParams g1 = g;
    g1.mode = 0;
    g1.tiles = B.tiles1; g1.num_tiles = B.meta + 0;
    g1.sfa = B.xsf; g1.sfa_kblocks = L.H / 64;
    g1.sfb0 = tw.sfp_gu; g1.ssfb0 = tw.sfp_sh_gu;  // quarter tiles of gate | up
    g1.post0 = tw.post_gate; g1.post1 = tw.post_up; g1.spost0 = tw.post_sh_gate; g1.spost1 = tw.post_sh_up;
    TC_PHASE(1, (tc_gemm_kernel<0><<<sms, kTcThreads, kTcSmemBytes, st>>>(m1, g1)))

    TcGemmParams g2 = g;
    g2.mode = 1;
    g2.tiles = B.tiles2; g2.num_tiles = B.meta + 1;
    g2.sfa = B.hsf; g2.sfa_kblocks = Imax / 64;
    g2.sfb0 = tw.sfp_dn; g2.ssfb0 = tw.sfp_sh_dn;  // quarter tiles of down
    g2.post0 = tw.post_down; g2.post1 = tw.post_down; g2.spost0 = tw.post_sh_down; g2.spost1 = tw.post_sh_down;
    TC_PHASE(2, (tc_gemm_kernel<1><<<sms, kTcThreads, kTcSmemBytes, st>>>(m2, g2)))

    TcCombineArgs ca{};
    ca.y = B.y; ca.ids = L.ids; ca.out = L.out; ca.T = L.T; ca.H = L.H; ca.k = L.k; ca.E = L.E;
    ca.w = L.w; ca.x = L.x; ca.Z = L.Z;
    ca.has_shared = L.I_shared > 0;
    const int64_t n = (int64_t)L.T * (L.H / 8);
    TC_PHASE(3, (tc_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(ca)))
#undef TC_PHASE
    return cudaSuccess;
}

}  // namespace moe
