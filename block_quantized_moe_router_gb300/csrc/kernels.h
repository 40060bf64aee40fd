// kernels.h -- host-side launchers of the library's kernels (internal).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ---- routing (route.cu) -------------------------------------------------------------------
cudaError_t launch_router_logits(const void* x, const void* wr, float* logits, int T, int E,
                                 int H, cudaStream_t st);
// The same on the tensor cores (prefill_tc.cu): T >= 128 tokens, E a multiple of 128;
// cudaErrorNotSupported (nothing launched) otherwise.
cudaError_t launch_router_tc(const void* x, const void* wr, float* logits, int T, int E, int H,
                             int32_t* status, cudaStream_t st);
cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int scoring,
                        int renorm, float scaling, int32_t* ids, float* w, int32_t* status,
                        cudaStream_t st);
// ids = tid2eid[token] (table order).  Weights: scaling / k, or -- with router logits given --
// sqrt(softplus(logit at the id)), renormalised over the token's kept pairs when `renorm`,
// times scaling.
cudaError_t launch_hash_route(const int64_t* tid2eid, const int32_t* token_ids, int64_t vocab,
                              int T, int E, int k, float scaling, const float* logits, int renorm,
                              int32_t* ids, float* w, int32_t* status, cudaStream_t st);

// ---- expert FFN (ffn.cu) --------------------------------------------------------------------
// One projection as the kernels see it: packed codes, block scales, and a per-expert fp32
// post-scale (the NVFP4 global, or 2^offset for MXFP4) plus, for MXFP4, the per-expert
// exponent offset folded into the f16 scale conversion.
struct ProjView {
    const uint8_t* packed;
    const uint8_t* scales;
    const float* post;      // [E]
    const int32_t* mx_off;  // [E] (MXFP4) or nullptr
    int fmt;
};

struct FfnLaunch {
    int T, E, H, I, k, I_shared, act, path;
    int Z;                  // zero-computation experts: ids E .. E + Z - 1 add w * x
    float g1, g2;
    unsigned long long wait_cycles;  // device-wide barrier wait limit in SM cycles (0: default)
    const void* x;          // bf16 [T][H]
    const int32_t* ids;     // [T][k]
    const float* w;         // [T][k]
    void* out;              // bf16 [T][H]
    int32_t* status;
    ProjView gate, up, down, sh_gate, sh_up, sh_down;
    // workspace views
    int32_t *counts, *offsets, *active, *meta, *sorted_pair, *pos_of_pair;
    __half* x16;
    uint8_t *xq, *xs;
    __half* h16;
    uint8_t *hq, *hs;
    float* y;
};

// Optional timing events around the kernel phases of launch_ffn (null entries: untimed).
struct PhaseEvents {
    cudaEvent_t begin[4];
    cudaEvent_t end[4];
};

cudaError_t launch_ffn(const FfnLaunch& L, cudaStream_t st, const PhaseEvents* ev = nullptr);
cudaError_t record_phase_event(cudaEvent_t ev, cudaStream_t st);

// ---- many-token FFN on the tcgen05 tensor cores (prefill_tc.cu) -----------------------------
// Weights prepared once: TMA maps over the packed codes and the block scales rearranged into
// the MMA's 128-row x 4 scale-factor tiles (owned buffers).
struct TcWeights {
    bool ready = false;
    CUtensorMap gate, up, down, sh_gate, sh_up, sh_down;
    uint8_t *sf_gate = nullptr, *sf_up = nullptr, *sf_down = nullptr;
    uint8_t *sf_sh_gate = nullptr, *sf_sh_up = nullptr, *sf_sh_down = nullptr;
    // B-operand scales as quarter tiles (the compact tiles above are freed once these exist)
    uint8_t *sfp_gu = nullptr, *sfp_dn = nullptr, *sfp_sh_gu = nullptr, *sfp_sh_dn = nullptr;
    // per-expert post-scales seen by the MMA path: the NVFP4 globals, or for MXFP4 the power of
    // two left over after the E8M0 scales were re-expressed as E4M3 (owned when MXFP4)
    const float *post_gate = nullptr, *post_up = nullptr, *post_down = nullptr;
    const float *post_sh_gate = nullptr, *post_sh_up = nullptr, *post_sh_down = nullptr;
    float* owned_post[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
};
struct TcBuffers {  // workspace views
    int32_t *meta, *mblock_expert, *padrow_pair;
    int32_t* scan;  // 5 x (E + 2): counts, 128-row block bases, tile bases (gate+up, down), cursors
    int4 *tiles1, *tiles2;
    uint8_t *tokq, *toks;  // tokens quantized once: codes [T][H/2], scales [T][H/16]
    uint8_t *xq, *xsf, *hq, *hsf;
    __nv_bfloat16* y;
    int max_blocks;
};
struct TcPrepArgs {
    const int32_t* ids;
    int T, k, E, Z, H, I, I_shared, has_shared;
    int32_t* status;
    int32_t *meta, *mblock_expert, *padrow_pair;
    int4 *tiles1, *tiles2;
    int32_t* scan;
};
struct TcQuantArgs {
    const void* x;
    int T, H, k, P;
    float g1;
    const int32_t *meta, *padrow_pair;
    uint8_t *tokq, *toks;
    uint8_t *xq, *xsf;
};
struct TcTensorMaps {
    CUtensorMap a, b0, b1, sb0, sb1;
};
struct TcGemmParams {
    int mode;  // 0: gate+up -> NVFP4 h; 1: down -> bf16 rows per pair
    int E, H, I, I_shared, k, T, P;
    const int4* tiles;
    const int32_t* num_tiles;
    const int32_t *mblock_expert, *padrow_pair;
    const uint8_t* sfa;
    int sfa_kblocks;
    const uint8_t *sfb0, *ssfb0;  // B's scales as quarter tiles (routed, shared)
    const float *post0, *post1, *spost0, *spost1;
    const float* topk_w;
    uint8_t *hq, *hsf;
    int hq_row_bytes, hsf_kblocks;
    float g2;
    __nv_bfloat16* y;
    int32_t* status;
};
struct TcCombineArgs {
    const __nv_bfloat16* y;
    const int32_t* ids;
    const float* w;         // routing weights (zero-computation experts add w * x)
    const void* x;          // bf16 [T][H]
    void* out;
    int T, H, k, E, Z, has_shared;
};

bool tc_supported(int E, int H, int I, int I_shared, int fmt_routed, int fmt_shared);
cudaError_t tc_prepare(const FfnLaunch& L, TcWeights* tw, cudaStream_t st);
void tc_release(TcWeights* tw);
cudaError_t launch_ffn_tc(const FfnLaunch& L, const TcWeights& tw, const TcBuffers& B,
                          cudaStream_t st, const PhaseEvents* ev);

// Few-token path (T <= 8, T * top_k <= 64, bf16 activations): the whole block in one
// persistent cooperative launch of `sms` CTAs (decode.cu).  Where the routing comes from:
enum DecRouteMode {
    DEC_ROUTE_GIVEN = 0,   // ids / weights in L.ids / L.w
    DEC_ROUTE_ROUTER = 1,  // router GEMM (w_router, x) -> logits_out, then top-K
    DEC_ROUTE_LOGITS = 2,  // top-K of logits_in
    DEC_ROUTE_HASH = 3     // tid2eid[token_ids]
};
struct DecRoute {
    int mode;
    int hash_ids;             // ids from tid2eid[token_ids] (with mode ROUTER / LOGITS the
                              // weights come from the sqrt(softplus) scores of the logits)
    const void* w_router;     // bf16 [E][H]
    const float* logits_in;   // [T][E]
    float* logits_out;        // [T][E]
    const float* bias;        // [E] or null (selection only)
    int scoring, renorm;
    float scaling;
    const int64_t* tid2eid;   // [vocab][k]
    const int32_t* token_ids; // [T]
    int64_t vocab;
    int32_t* ids_out;         // [T][k] (modes 1-3)
    float* w_out;             // [T][k]
};
// `bar`: a device 64-bit counter, zero when first used, owned by the weights handle and used
// only by launches of `sms` CTAs.
cudaError_t launch_decode_fused(const FfnLaunch& L, const DecRoute& R, unsigned long long* bar,
                                int sms, cudaStream_t st);
// Moves the barrier epoch one launch ahead of the arrival counter (test aid: every barrier
// wait of the next fused launch then runs out its limit).
cudaError_t launch_barrier_skew(unsigned long long* bar, cudaStream_t st);

cudaError_t launch_quantize_act(const void* x, int64_t rows, int64_t K, float g, uint8_t* packed,
                                uint8_t* scales, __half* deq16, cudaStream_t st);

// Per-expert max of the E8M0 scale bytes of an MXFP4 tensor -> exponent offset and post-scale.
cudaError_t launch_mx_offsets(const uint8_t* scales, int E, int64_t per_expert, int32_t* off,
                              float* post, cudaStream_t st);

}  // namespace moe
