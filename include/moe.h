/* moe.h -- C ABI of the GB300 (sm_103a) MoE FFN block library (libmoe_gb300.so).
 *
 * The library computes the Mixture-of-Experts FFN block of an LLM serving engine:
 *   router GEMM -> top-K routing (softmax, sigmoid + correction bias, or a static hash
 *   table) -> per-expert token dispatch -> block-quantized expert FFN
 *   (gate+up projection, SiLU(gate)*up, down projection) -> top-K weighted sum plus an
 *   optional shared expert.
 * Sources: the spark_model MoE pages -- moe/mod.rs (module doc: two fused expert launches,
 * routing ids and weights stay on the device with no device-to-host synchronisation; the
 * `MoeLayer` field docs for the weight formats, the correction bias and the tid2eid table)
 * and moe/init.rs (`MoeLayer::new_with_hash`: argument checks at construction).
 *
 * Conventions shared by every entry point:
 *   - Pointers marked [device] must point to device memory of the current CUDA device;
 *     pointers marked [host] to host memory.  The caller owns every buffer it passes.
 *     The library owns only the prepared-weights handle and the buffers behind it.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Every call is asynchronous on that stream: no host synchronisation, no device-to-host
 *     copy and no memory allocation happen inside moe_route / moe_ffn_forward / moe_forward /
 *     moe_quantize_act_nvfp4.  moe_forward_host alone copies, from and to the caller's host
 *     buffers, and those copies are enqueued on the stream too.
 *   - Errors detectable on the host return a nonzero moe_status_t BEFORE anything is
 *     launched.  A failed launch returns MOE_ERR_CUDA.  Problems found in the data on the
 *     device are OR-ed into the caller's int32 device status word (MOE_DEV_* bits); the
 *     kernels then skip or zero the affected work instead of trapping.
 *   - Layouts are row-major.  Block-quantized tensors are stacked over experts:
 *       packed  [E][N][K/2] uint8 -- E2M1 codes, element 2i in the LOW nibble of byte i,
 *                                   bit 3 of a code is its sign;
 *       scales  [E][N][K/16] uint8 FP8-E4M3 (NVFP4) or [E][N][K/32] uint8 E8M0 (MXFP4);
 *       globals [E] float32 per-tensor global (NVFP4, multiplies) or NULL (MXFP4).
 *     Value of element (e, n, k) = e2m1(code) * scale(e, n, k / block) * global(e).
 *     gate and up have N = I, K = H; down has N = H, K = I.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* a size, pointer or enum is out of its documented range  */
    MOE_ERR_UNSUPPORTED = 2,   /* a valid combination this library does not implement     */
    MOE_ERR_CUDA = 3,          /* a CUDA runtime call or a kernel launch failed            */
    MOE_ERR_WORKSPACE = 4      /* the workspace passed is smaller than moe_workspace_size */
} moe_status_t;

/* Bits of the caller-owned int32 device status word (atomically OR-ed by the kernels). */
#define MOE_DEV_BAD_EXPERT_ID 0x1 /* a tid2eid entry outside [0,E): that pair is dropped     */
#define MOE_DEV_BAD_TOKEN_ID 0x2  /* a token id outside [0,vocab): the token's pairs dropped */
#define MOE_DEV_NONFINITE 0x4     /* a NaN/Inf router logit: ranked below every finite one   */
#define MOE_DEV_TIMEOUT 0x8       /* a bounded device-side wait gave up                      */

typedef enum {
    MOE_SCORE_SOFTMAX = 0,
    MOE_SCORE_SIGMOID = 1,
    MOE_SCORE_HASH = 2,
    MOE_SCORE_SQRTSOFTPLUS = 3,
    MOE_SCORE_SOFTMAX_BIAS = 4,
    MOE_SCORE_HASH_SQRTSOFTPLUS = 5  /* hash ids, weights from sqrt(softplus) router scores */
} moe_scoring_t;
typedef enum { MOE_FMT_NVFP4 = 0, MOE_FMT_MXFP4 = 1 } moe_fmt_t;
/* Activation precision of the expert GEMMs.  BF16: W4A16 (bf16 tokens, dequantized
 * weights; tokens and h enter the MMAs as f16, so their magnitudes must stay within f16's
 * finite range, 65504).  NVFP4: W4A4 -- tokens and the intermediate h are quantized to NVFP4
 * (per 16 elements, E4M3 scale, static power-of-two f32 global) before the block-scaled FP4
 * MMA. */
typedef enum { MOE_ACT_BF16 = 0, MOE_ACT_NVFP4 = 1 } moe_act_t;

/* One block-quantized projection, stacked over experts (layout in the header comment). */
typedef struct {
    const void* packed;    /* [device] uint8 [E][N][K/2]                                  */
    const void* scales;    /* [device] uint8 [E][N][K/16] (NVFP4) or [E][N][K/32] (MXFP4) */
    const float* globals;  /* [device] float [E] (NVFP4) or NULL (MXFP4)                   */
    int32_t fmt;           /* moe_fmt_t                                                     */
} moe_qtensor;

/* The expert weights of one MoE layer.  Constraints (checked): 1 <= E, E + zero_experts <= 512,
 * 1 <= top_k <= min(E + zero_experts, 32); H, I, I_shared multiples of 128; I_shared == 0
 * means no shared expert.  A shared expert is one expert (E = 1 in its tensors) added with
 * weight 1.  zero_experts (Z >= 0) zero-computation experts have ids E .. E + Z - 1 and no
 * weights: such an expert returns its input, so a pair routed to it adds w * x[t] (the bf16
 * token, whatever act is) -- the LongCat zero-computation experts of the spark_model MoE
 * pages (moe/mod.rs, `moe_zero_expert_add` handle and `zero_accum_dev` field doc). */
typedef struct {
    int32_t E, H, I, top_k, I_shared;
    moe_qtensor gate, up, down;
    moe_qtensor sh_gate, sh_up, sh_down;
    int32_t zero_experts;
} moe_ffn_desc;

/* Routing of T tokens over E real experts and zero_experts zero-computation experts (ids
 * E .. E + zero_experts - 1; see moe_ffn_desc).  The router has E + zero_experts outputs:
 * w_router [E + Z][H], correction_bias [E + Z], logits [T][E + Z].  Constraints (checked):
 * 1 <= E, E + Z <= 512, 1 <= top_k <= min(E + Z, 32); learned routers: H a multiple of 32 when
 * the router GEMM runs; both hash kinds: tid2eid and token_ids non-NULL, vocab >= 1. */
typedef struct {
    int32_t T, E, H, top_k;
    int32_t scoring;           /* moe_scoring_t                                            */
    int32_t renormalize;       /* 1: weights renormalised over the selected experts        */
    float routed_scaling;      /* multiplies every routing weight (1.0 for plain top-K)    */
    const void* w_router;      /* [device] bf16 [E][H], or NULL when logits are supplied   */
    const float* correction_bias; /* [device] float [E] (sigmoid/sqrt-softplus selection) or NULL */
    const int64_t* tid2eid;    /* [device] int64 [vocab][top_k] (hash kinds only)         */
    int64_t vocab;
    const int32_t* token_ids;  /* [device] int32 [T] (hash kinds only)                    */
    int32_t zero_experts;      /* Z >= 0 zero-computation experts after the E real ones    */
} moe_route_desc;

/* Router GEMM + top-K (every rule below runs over the E + zero_experts router outputs).
 *   Softmax: p = softmax(logits) over all E; the top_k largest are selected; weight =
 *     p / sum(selected p) when renormalize, else p; times routed_scaling.
 *   Softmax + bias: p = softmax(logits); selection ranks p + correction_bias; weight = p /
 *     sum(selected p) when renormalize, else p; times routed_scaling (moe/mod.rs, the LongCat
 *     `moe_topk_softmax_bias` handles, whose router width is num_experts + zero_expert_num).
 *   Sigmoid: s = sigmoid(logits); selection ranks s + correction_bias; weight = s /
 *     sum(selected s) when renormalize, else s; times routed_scaling.  (moe/mod.rs,
 *     `correction_bias_dev` field doc.)
 *   Sqrt(softplus): the sigmoid scheme with s = sqrt(log(1 + exp(logits))) (moe/mod.rs, the
 *     `moe_topk_sqrtsoftplus` routing handles).
 *   Hash: ids = tid2eid[token_ids[t]] in table order; weight = routed_scaling / top_k.
 *     (moe/init.rs, `new_with_hash` doc.)
 *   Hash + sqrt(softplus) weights: ids as for Hash; the router GEMM still runs (or logits_in
 *     is read) and pair j gets s_j = sqrt(log(1 + exp(logits[t][id_j]))); weight = s_j /
 *     sum over the token's kept pairs of s when renormalize, else s_j; times routed_scaling.
 *     No correction bias (nothing is selected).  This is how this library reads the hash
 *     layers of the model family that ships both the `moe_hash_route` and the
 *     `moe_topk_sqrtsoftplus` routing handles (moe/init.rs handle lookups; moe/mod.rs,
 *     `tid2eid_dev` field doc): the table fixes the experts, the learned router their weights.
 *     A pair with a bad table entry is dropped (weight 0) and left out of the sum; a
 *     non-finite logit at a chosen id gives that pair weight 0 and sets MOE_DEV_NONFINITE.
 * Ids are written in descending selection-score order, ties to the lower expert index.
 * x_bf16      [device] bf16 [T][H]; used when w_router != NULL.
 * logits_in   [device] float [T][E] or NULL: precomputed router logits (then w_router and
 *             x_bf16 are ignored).
 * logits_out  [device] float [T][E]; required when the router GEMM runs, else may be NULL.
 * topk_ids    [device] int32 [T][top_k]; -1 marks a dropped pair.
 * topk_w      [device] float [T][top_k].
 * dev_status  [device] int32 [1]; bits are OR-ed in, never cleared by the library.
 * T == 0 is a valid no-op. */
moe_status_t moe_route(const moe_route_desc* desc, const void* x_bf16, const float* logits_in,
                       float* logits_out, int32_t* topk_ids, float* topk_w, int32_t* dev_status,
                       void* stream);

/* Bytes of device workspace moe_ffn_forward needs for T tokens in activation mode act.
 * Source: the spark_model MoE pages, moe/mod.rs, `zero_accum_dev` field doc (the layer's
 * scratch is a fixed-size allocation made once, so that the forward pass stays graph-safe):
 * here the caller makes that one allocation, sized by this call, and passes it to every
 * moe_ffn_forward / moe_forward with at most T tokens.  The size depends only on the
 * descriptor, T and act.  Host-only: launches nothing.  Errors: MOE_ERR_INVALID_ARG for a
 * NULL `bytes`, an invalid descriptor (the checks of moe_ffn_desc), T < 0 or an unknown act. */
moe_status_t moe_workspace_size(const moe_ffn_desc* desc, int32_t T, int32_t act, size_t* bytes);

/* One-time weight preparation.  Source: the spark_model MoE pages, moe/mod.rs, the
 * `cutlass_grouped_host` (`MoeCutlassHostTables`) and `_cutlass_sfb_owned` field docs: the
 * per-expert scale-factor (SFB) layout the grouped FP4 GEMM consumes is built ONCE at load
 * from the weights' scales and owned by the layer, dying with it.  Here: validates the
 * descriptor (the construction-time checks of moe/init.rs, `MoeLayer::new_with_hash`),
 * derives per-tensor post-scales (the NVFP4 globals; for MXFP4 a power-of-two exponent
 * offset) and the scale-factor tiles of the FP4 tensor-core path (3 * (E * I + I_shared) *
 * H / 16 bytes: the weights' scales in the order the tensor-core kernel copies them to TMEM).
 * desc        [host] read during the call only; the device buffers it points to must stay
 *             alive and unchanged until moe_release_weights.
 * handle_out  [host] receives the handle (NULL on error).
 * Allocates device memory and synchronises `stream` before returning.  Errors:
 * MOE_ERR_INVALID_ARG (descriptor checks), MOE_ERR_UNSUPPORTED (gate/up/down of mixed formats),
 * MOE_ERR_CUDA (allocation or launch failure; nothing is leaked). */
moe_status_t moe_prepare_weights(const moe_ffn_desc* desc, void** handle_out, void* stream);
/* Frees everything moe_prepare_weights allocated (moe/mod.rs, `_cutlass_sfb_owned` field doc:
 * the owned scale buffers live exactly as long as the layer).  The caller must make sure no
 * launch using the handle is still running.
 * Errors: MOE_ERR_INVALID_ARG for NULL or a pointer that is not a live handle. */
moe_status_t moe_release_weights(void* handle);

/* Expert FFN + weighted combine.  Source: the spark_model MoE pages, moe/mod.rs module doc
 * (the top-K experts of a batch run in two fused expert launches -- gate+up, then SiLU+down --
 * with ids and weights kept on the device) and moe/init.rs (`moe_weighted_sum_blend`: the
 * weighted sum plus the shared expert):
 *   out[t] = sum_j topk_w[t][j] * FFN_{topk_ids[t][j]}(x[t]) + FFN_shared(x[t]),
 *   FFN_e(a) = W_down,e (SiLU(W_gate,e a) * (W_up,e a)) for a real expert e < E,
 *   FFN_e(a) = x[t] for a zero-computation expert E <= e < E + zero_experts;
 *   pairs with any other id (e.g. -1) are dropped.
 * act = MOE_ACT_NVFP4 quantizes x with global g_act1 and h with global g_act2 (each a
 * power of two) before the FP4 products; MOE_ACT_BF16 ignores both.
 * x_bf16 [device] bf16 [T][H]; topk_ids/topk_w as written by moe_route;
 * out_bf16 [device] bf16 [T][H]; workspace [device], ws_bytes >= moe_workspace_size.
 * T == 0 is a valid no-op.  Few tokens (T <= 8, T * top_k <= 64, MOE_ACT_BF16) run as one
 * persistent cooperative launch with the constraints stated at moe_forward. */
moe_status_t moe_ffn_forward(const void* handle, int32_t T, int32_t act, float g_act1,
                             float g_act2, const void* x_bf16, const int32_t* topk_ids,
                             const float* topk_w, void* out_bf16, void* workspace,
                             size_t ws_bytes, int32_t* dev_status, void* stream);

/* Route + expert FFN in one call: the result of moe_route(route, x_bf16, logits_in,
 * logits_out, topk_ids, topk_w, dev_status) followed by moe_ffn_forward(handle, route->T, act,
 * g_act1, g_act2, x_bf16, topk_ids, topk_w, out_bf16, workspace, ws_bytes, dev_status), with the
 * same argument rules, outputs and workspace size (moe_workspace_size of the handle's
 * descriptor).  route->E, route->top_k, route->H and route->zero_experts must equal the
 * handle's E, top_k, H and zero_experts.
 * For a few tokens (T <= 8, T * top_k <= 64, act == MOE_ACT_BF16) the router GEMV, the top-K
 * selection (or the hash lookup), the expert FFN and the weighted sum run in ONE persistent
 * kernel launch with one thread block per SM and two device-wide barriers -- the single-launch
 * decode structure that the spark_model MoE module doc (moe/mod.rs) works towards by fusing
 * the gate with the top-K; there the router logits come from fp32 dot products on the CUDA
 * cores, so they can differ from moe_route's in the last bits.  That launch is cooperative:
 * it needs every SM of the device free to co-schedule (MOE_ERR_CUDA if the device cannot run
 * it), and calls on one handle must not overlap on the GPU (the handle owns the barrier
 * counter).  If a device-side barrier wait gives up (MOE_DEV_TIMEOUT) the outputs of that
 * call are invalid and the handle must be released and prepared again. */
moe_status_t moe_forward(const void* handle, const moe_route_desc* route, int32_t act,
                         float g_act1, float g_act2, const void* x_bf16, const float* logits_in,
                         float* logits_out, int32_t* topk_ids, float* topk_w, void* out_bf16,
                         void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* moe_forward for a caller whose tokens and results live in HOST memory.  It computes what
 * moe_forward computes (the spark_model MoE pages, moe/mod.rs module doc: router, top-K and
 * the expert FFN with the weighted sum); the pages' layer only ever sees device tensors, so
 * the copies around it are this library's.  Enqueued on `stream`, in order: the copy of
 * x_bf16_host (and, for both hash kinds, token_ids_host) into a staging area at the end of the
 * workspace; moe_forward on the staged copies, with the router logits, ids and weights in that
 * staging area; the copy of the output into out_bf16_host and, when those pointers are not
 * NULL, of the ids and weights into topk_ids_host / topk_w_host.  The call returns once all
 * of it is enqueued: the host buffers must stay valid, and the inputs unchanged, until the
 * stream has passed the copies -- synchronise the stream (or an event recorded after the call)
 * before reading the outputs.  Page-locked host memory (cudaHostAlloc / cudaHostRegister)
 * makes the copies asynchronous and lets the call be captured into a CUDA graph; with pageable
 * memory the runtime may block the host inside the copies.
 * x_bf16_host    [host] bf16 [T][H].
 * token_ids_host [host] int32 [T]; required for both hash kinds, ignored otherwise (the
 *                route descriptor's token_ids field is ignored).
 * out_bf16_host  [host] bf16 [T][H].
 * topk_ids_host  [host] int32 [T][top_k] or NULL;  topk_w_host [host] float [T][top_k] or NULL.
 * workspace      [device], ws_bytes >= moe_workspace_size_host for (desc, T, act).
 * dev_status     [device] int32 [1] or NULL, as for moe_forward.
 * The router must run in the call: route->w_router is required unless route->scoring is
 * MOE_SCORE_HASH (precomputed logits are not taken from the host).  Errors: those of
 * moe_forward; MOE_ERR_INVALID_ARG for a NULL x_bf16_host / out_bf16_host, a hash kind without
 * token_ids_host, or a learned router without w_router; MOE_ERR_WORKSPACE when ws_bytes is
 * below moe_workspace_size_host; MOE_ERR_CUDA when a copy cannot be enqueued.  T == 0 is a
 * valid no-op.
 * moe_workspace_size_host: moe_workspace_size plus the staging area (x and the output, T * H
 * bf16 each; ids, weights, token ids and the E + zero_experts router logits per token), each
 * part 256-byte aligned.  Host-only; errors as for moe_workspace_size. */
moe_status_t moe_workspace_size_host(const moe_ffn_desc* desc, int32_t T, int32_t act,
                                     size_t* bytes);
moe_status_t moe_forward_host(const void* handle, const moe_route_desc* route, int32_t act,
                              float g_act1, float g_act2, const void* x_bf16_host,
                              const int32_t* token_ids_host, void* out_bf16_host,
                              int32_t* topk_ids_host, float* topk_w_host, void* workspace,
                              size_t ws_bytes, int32_t* dev_status, void* stream);

/* The NVFP4 activation quantizer on its own (the `quantize_bf16_to_nvfp4` step of the
 * FP4 x FP4 recipe, qwen3_attention/init.rs handle list): per 16 consecutive elements of
 * each row, s = E4M3(amax / 6 / g) (round to nearest even, saturating), code =
 * E2M1(v / (e4m3(s) * g)) (round to nearest even, saturating at 6), all-zero codes when s
 * decodes to 0.  x_bf16 [device] bf16 [rows][K]; packed [device] uint8 [rows][K/2];
 * scales [device] uint8 [rows][K/16]; K a multiple of 16. */
moe_status_t moe_quantize_act_nvfp4(const void* x_bf16, int64_t rows, int64_t K, float g,
                                    uint8_t* packed, uint8_t* scales, void* stream);

/* moe_ffn_forward without a caller-provided workspace.  The pages have no counterpart: this is
 * for callers that cannot give the library device memory -- a host that freezes its device
 * memory plan at start-up and must see no cudaMalloc afterwards (cudaMalloc can synchronise
 * the device), or a plugin interface that passes tensors but no workspace or allocator.
 * Same arguments and result as moe_ffn_forward, minus workspace/ws_bytes.  The scratch is a
 * static 8 MiB device array inside the library (held on every GPU that loads it until the
 * process exits); a call whose workspace plan (moe_workspace_size) exceeds 8 MiB returns
 * MOE_ERR_WORKSPACE without launching (8 MiB holds up to 27 tokens at H 7168, I 2048, top-8
 * with a shared expert).  Allocates nothing.  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  All calls on a device share the one array, so calls whose
 * kernels overlap on the GPU race and must be serialised by the caller; no part of the array
 * needs clearing between calls. */
moe_status_t moe_ffn_forward_noalloc(const void* handle, int32_t T, int32_t act, float g_act1,
                                     float g_act2, const void* x_bf16, const int32_t* topk_ids,
                                     const float* topk_w, void* out_bf16, int32_t* dev_status,
                                     void* stream);

/* Diagnostics for the bounded device waits (no counterpart on the pages, which give no
 * device-side wait at all; the few-token kernel's device-wide barriers are this library's).
 * moe_set_wait_limit(handle, cycles): every device-wide barrier wait of the few-token kernel
 * launched on `handle` afterwards gives up after `cycles` SM clock cycles (0 = the default,
 * 4e9 cycles, about 2 s) and then sets MOE_DEV_TIMEOUT and carries on.  Host-only.
 * moe_skew_barrier(handle, stream): moves the handle's barrier epoch (the count of few-token
 * launches completed on it) one ahead of its arrival counter, on `stream`.  In the next
 * few-token launch no device-wide barrier can complete: every wait runs out after the limit,
 * MOE_DEV_TIMEOUT is set, the launch returns normally (after about twice the limit) and its
 * outputs are invalid.  Used by the tests of the timeout path; after it (or after any
 * MOE_DEV_TIMEOUT) release the handle and prepare the weights again.
 * Errors: MOE_ERR_INVALID_ARG for a bad handle, MOE_ERR_CUDA if the launch fails. */
moe_status_t moe_set_wait_limit(void* handle, uint64_t cycles);
moe_status_t moe_skew_barrier(void* handle, void* stream);

/* Kernel timing for benchmarks (no counterpart on the pages; a measurement aid).
 * moe_profile_enable(handle, mask) makes the handle record
 * a pair of CUDA timing events around each kernel phase selected by `mask` in every later
 * moe_ffn_forward on that handle (as external event nodes when the stream is being captured
 * into a CUDA graph); mask 0 stops it.  Phases: bit 0 dispatch + activation conversion,
 * bit 1 gate+up GEMM, bit 2 down GEMM, bit 3 combine.  moe_profile_read waits for the last
 * recorded end event and writes the duration in milliseconds of each phase's most recent
 * execution to ms_out[0..3] (-1 for phases not timed).  Not thread-safe per handle. */
moe_status_t moe_profile_enable(void* handle, uint32_t mask);
moe_status_t moe_profile_read(void* handle, float* ms_out);

/* A static, NUL-terminated description of a status code ("unknown moe_status_t" for values
 * outside the enum); never NULL, nothing to free.  Source: the loud construction-time errors
 * of the spark_model MoE layer (moe/init.rs, `MoeLayer::new_with_hash`: a top_k above the
 * expert count is refused at load with a message instead of routing out of bounds). */
const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
