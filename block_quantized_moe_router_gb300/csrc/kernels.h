// kernels.h -- host-side launchers of the library's kernels (internal).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ---- routing (route.cu) -------------------------------------------------------------------
cudaError_t launch_router_logits(const void* x, const void* wr, float* logits, int T, int E,
                                 int H, cudaStream_t st);
cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int scoring,
                        int renorm, float scaling, int32_t* ids, float* w, int32_t* status,
                        cudaStream_t st);
cudaError_t launch_hash_route(const int64_t* tid2eid, const int32_t* token_ids, int64_t vocab,
                              int T, int E, int k, float scaling, int32_t* ids, float* w,
                              int32_t* status, cudaStream_t st);

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
    int T, E, H, I, k, I_shared, act;
    float g1, g2;
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

// Few-token path (T <= 8, bf16 activations): phase 1 = gate+up, phase 2 = down + combine.
cudaError_t launch_decode_phase(const FfnLaunch& L, int phase, cudaStream_t st);

cudaError_t launch_quantize_act(const void* x, int64_t rows, int64_t K, float g, uint8_t* packed,
                                uint8_t* scales, __half* deq16, cudaStream_t st);

// Per-expert max of the E8M0 scale bytes of an MXFP4 tensor -> exponent offset and post-scale.
cudaError_t launch_mx_offsets(const uint8_t* scales, int E, int64_t per_expert, int32_t* off,
                              float* post, cudaStream_t st);

}  // namespace moe
