// api.cu -- the C ABI declared in include/moe.h: argument validation, the prepared-weights
// handle and the launch sequence.  Argument checks follow the construction-time checks of
// the spark_model MoE layer (moe/init.rs, `MoeLayer::new_with_hash`: 1 <= top_k <= E, and
// top_k / E bounded by the routing kernels' fixed per-warp storage).
#include <cmath>
#include <cstring>
#include <new>

#include "common.cuh"
#include "kernels.h"

namespace {

using namespace moe;

bool pow2_positive(float g) {
    if (!(g > 0.f) || !std::isfinite(g)) return false;
    int ex = 0;
    return std::frexp(g, &ex) == 0.5f;
}

bool is_hash(int scoring) { return scoring == MOE_SCORE_HASH || scoring == MOE_SCORE_HASH_SQRTSOFTPLUS; }

bool valid_fmt(int f) { return f == MOE_FMT_NVFP4 || f == MOE_FMT_MXFP4; }

bool valid_qtensor(const moe_qtensor& t) {
    if (!t.packed || !t.scales || !valid_fmt(t.fmt)) return false;
    if (t.fmt == MOE_FMT_NVFP4 && !t.globals) return false;
    return true;
}

struct PreparedProj {
    ProjView view{};
    int32_t* mx_off = nullptr;  // owned
    float* mx_post = nullptr;   // owned
};

struct Handle {
    uint32_t magic = 0x4D4F4531u;  // "MOE1"
    moe_ffn_desc desc{};
    PreparedProj gate, up, down, sh_gate, sh_up, sh_down;
    uint32_t profile_mask = 0;
    PhaseEvents events{};  // owned; created by moe_profile_enable
    bool tc_shape = false;
    TcWeights tc{};        // owned; the tcgen05 path's scale tiles and tensor maps
    int sms = 0;           // SM count of the device the weights live on
    unsigned long long* bar = nullptr;  // owned; grid-barrier arrival counter and epoch (few-token kernel)
    unsigned long long wait_cycles = 0;  // device-wide barrier wait limit (0 = the default)
};

bool desc_tc_shape(const moe_ffn_desc& d) {
    return tc_shape_ok(d.H, d.I, d.I_shared, d.gate.fmt, d.I_shared > 0 ? d.sh_gate.fmt : d.gate.fmt);
}

void destroy_events(Handle* h) {
    for (int i = 0; i < 4; ++i) {
        if (h->events.begin[i]) cudaEventDestroy(h->events.begin[i]);
        if (h->events.end[i]) cudaEventDestroy(h->events.end[i]);
        h->events.begin[i] = h->events.end[i] = nullptr;
    }
    h->profile_mask = 0;
}

moe_status_t prepare_proj(const moe_qtensor& t, int E, int64_t N, int64_t K, PreparedProj& out,
                          cudaStream_t st) {
    out.view.packed = static_cast<const uint8_t*>(t.packed);
    out.view.scales = static_cast<const uint8_t*>(t.scales);
    out.view.fmt = t.fmt;
    if (t.fmt == MOE_FMT_NVFP4) {
        out.view.post = t.globals;
        out.view.mx_off = nullptr;
        return MOE_OK;
    }
    if (cudaMalloc(&out.mx_off, sizeof(int32_t) * E) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMalloc(&out.mx_post, sizeof(float) * E) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_mx_offsets(out.view.scales, E, N * (K / 32), out.mx_off, out.mx_post, st) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    out.view.post = out.mx_post;
    out.view.mx_off = out.mx_off;
    return MOE_OK;
}

void free_proj(PreparedProj& p) {
    if (p.mx_off) cudaFree(p.mx_off);
    if (p.mx_post) cudaFree(p.mx_post);
    p.mx_off = nullptr;
    p.mx_post = nullptr;
}

moe_status_t validate_ffn_desc(const moe_ffn_desc* d) {
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->E < 1 || d->zero_experts < 0 || d->E + d->zero_experts > kMaxExperts)
        return MOE_ERR_INVALID_ARG;
    if (d->top_k < 1 || d->top_k > d->E + d->zero_experts || d->top_k > kMaxTopK)
        return MOE_ERR_INVALID_ARG;
    if (d->H < 128 || d->H % 128 || d->I < 128 || d->I % 128) return MOE_ERR_INVALID_ARG;
    if (d->I_shared < 0 || d->I_shared % 128) return MOE_ERR_INVALID_ARG;
    if (!valid_qtensor(d->gate) || !valid_qtensor(d->up) || !valid_qtensor(d->down))
        return MOE_ERR_INVALID_ARG;
    if (d->gate.fmt != d->up.fmt || d->gate.fmt != d->down.fmt) return MOE_ERR_UNSUPPORTED;
    if (d->I_shared > 0) {
        if (!valid_qtensor(d->sh_gate) || !valid_qtensor(d->sh_up) || !valid_qtensor(d->sh_down))
            return MOE_ERR_INVALID_ARG;
        if (d->sh_gate.fmt != d->sh_up.fmt || d->sh_gate.fmt != d->sh_down.fmt)
            return MOE_ERR_UNSUPPORTED;
    }
    return MOE_OK;
}

moe_status_t validate_route(const moe_route_desc* d, const float* logits_in) {
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->T < 0 || d->E < 1 || d->zero_experts < 0 || d->E + d->zero_experts > kMaxExperts)
        return MOE_ERR_INVALID_ARG;
    if (d->top_k < 1 || d->top_k > d->E + d->zero_experts || d->top_k > kMaxTopK)
        return MOE_ERR_INVALID_ARG;
    if (!std::isfinite(d->routed_scaling)) return MOE_ERR_INVALID_ARG;
    if (d->scoring != MOE_SCORE_SOFTMAX && d->scoring != MOE_SCORE_SIGMOID &&
        d->scoring != MOE_SCORE_HASH && d->scoring != MOE_SCORE_SQRTSOFTPLUS &&
        d->scoring != MOE_SCORE_SOFTMAX_BIAS && d->scoring != MOE_SCORE_HASH_SQRTSOFTPLUS)
        return MOE_ERR_INVALID_ARG;
    if (is_hash(d->scoring) && d->vocab < 1) return MOE_ERR_INVALID_ARG;
    if (d->scoring != MOE_SCORE_HASH && !logits_in && (d->H < 32 || d->H % 32))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// The FFN launch description of one call; the workspace carve-up follows the path's plan.
FfnLaunch make_launch(const Handle* h, int T, int act, float g1, float g2, int path,
                      const Workspace& ws, char* base, const void* x, const int32_t* ids,
                      const float* w, void* out, int32_t* status) {
    const moe_ffn_desc& d = h->desc;
    FfnLaunch L{};
    L.T = T; L.E = d.E; L.H = d.H; L.I = d.I; L.k = d.top_k; L.I_shared = d.I_shared;
    L.Z = d.zero_experts;
    L.act = act; L.path = path; L.g1 = g1; L.g2 = g2;
    L.wait_cycles = h->wait_cycles;
    L.x = x; L.ids = ids; L.w = w; L.out = out; L.status = status;
    L.gate = h->gate.view; L.up = h->up.view; L.down = h->down.view;
    L.sh_gate = h->sh_gate.view; L.sh_up = h->sh_up.view; L.sh_down = h->sh_down.view;
    L.counts = reinterpret_cast<int32_t*>(base + ws.counts);
    L.offsets = reinterpret_cast<int32_t*>(base + ws.offsets);
    L.active = reinterpret_cast<int32_t*>(base + ws.active);
    L.meta = reinterpret_cast<int32_t*>(base + ws.meta);
    L.sorted_pair = reinterpret_cast<int32_t*>(base + ws.sorted_pair);
    L.pos_of_pair = reinterpret_cast<int32_t*>(base + ws.pos_of_pair);
    L.x16 = reinterpret_cast<__half*>(base + ws.x16);
    L.xq = reinterpret_cast<uint8_t*>(base + ws.xq);
    L.xs = reinterpret_cast<uint8_t*>(base + ws.xs);
    L.h16 = reinterpret_cast<__half*>(base + ws.h16);
    L.hq = reinterpret_cast<uint8_t*>(base + ws.hq);
    L.hs = reinterpret_cast<uint8_t*>(base + ws.hs);
    L.y = reinterpret_cast<float*>(base + ws.y);
    return L;
}

// The few-token path: one persistent launch (phase 1 timing events around it when profiled).
moe_status_t run_decode(const Handle* h, const FfnLaunch& L, const DecRoute& R, cudaStream_t st) {
    const PhaseEvents* ev = h->profile_mask ? &h->events : nullptr;
    if (ev && record_phase_event(ev->begin[1], st) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_decode_fused(L, R, h->bar, h->sms, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (ev && record_phase_event(ev->end[1], st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

// Staging area of moe_forward_host, after the FFN workspace: the step's inputs and outputs.
struct HostStage {
    size_t x, out, ids, w, logits, tok, total;
    static HostStage plan(const moe_ffn_desc& d, int T, int act) {
        const int path = select_path(T, d.H, d.top_k, act, desc_tc_shape(d));
        HostStage s{};
        size_t off = align_up(Workspace::plan(d.E, d.H, d.I, d.I_shared, d.top_k, T, act, path).total, 256);
        auto take = [&](size_t bytes) {
            const size_t o = off;
            off = align_up(off + bytes, 256);
            return o;
        };
        s.x = take(sizeof(uint16_t) * (size_t)T * d.H);
        s.out = take(sizeof(uint16_t) * (size_t)T * d.H);
        s.ids = take(sizeof(int32_t) * (size_t)T * d.top_k);
        s.w = take(sizeof(float) * (size_t)T * d.top_k);
        s.logits = take(sizeof(float) * (size_t)T * (d.E + d.zero_experts));
        s.tok = take(sizeof(int32_t) * (size_t)T);
        s.total = off;
        return s;
    }
};

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: argument out of range";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: combination not implemented";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA call or kernel launch failed";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
    }
    return "unknown moe_status_t";
}

moe_status_t moe_route(const moe_route_desc* d, const void* x_bf16, const float* logits_in,
                       float* logits_out, int32_t* topk_ids, float* topk_w, int32_t* dev_status,
                       void* stream) {
    const moe_status_t v = validate_route(d, logits_in);
    if (v != MOE_OK) return v;
    if (d->T == 0) return MOE_OK;
    if (!topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int Er = d->E + d->zero_experts;  // router outputs: real then zero-computation experts
    if (d->scoring == MOE_SCORE_HASH) {
        if (!d->tid2eid || !d->token_ids) return MOE_ERR_INVALID_ARG;
        return launch_hash_route(d->tid2eid, d->token_ids, d->vocab, d->T, Er, d->top_k,
                                 d->routed_scaling, nullptr, 0, topk_ids, topk_w, dev_status,
                                 st) == cudaSuccess
                   ? MOE_OK : MOE_ERR_CUDA;
    }
    if (d->scoring == MOE_SCORE_HASH_SQRTSOFTPLUS && (!d->tid2eid || !d->token_ids))
        return MOE_ERR_INVALID_ARG;
    const float* logits = logits_in;
    if (!logits) {
        if (!d->w_router || !x_bf16 || !logits_out) return MOE_ERR_INVALID_ARG;
        cudaError_t err = launch_router_tc(x_bf16, d->w_router, logits_out, d->T, Er, d->H,
                                           dev_status, st);
        if (err == cudaErrorNotSupported)
            err = launch_router_logits(x_bf16, d->w_router, logits_out, d->T, Er, d->H, st);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        logits = logits_out;
    }
    if (d->scoring == MOE_SCORE_HASH_SQRTSOFTPLUS)  // table ids, router-score weights
        return launch_hash_route(d->tid2eid, d->token_ids, d->vocab, d->T, Er, d->top_k,
                                 d->routed_scaling, logits, d->renormalize ? 1 : 0, topk_ids,
                                 topk_w, dev_status, st) == cudaSuccess
                   ? MOE_OK : MOE_ERR_CUDA;
    const float* bias = d->scoring != MOE_SCORE_SOFTMAX ? d->correction_bias : nullptr;
    return launch_topk(logits, bias, d->T, Er, d->top_k, d->scoring, d->renormalize ? 1 : 0,
                       d->routed_scaling, topk_ids, topk_w, dev_status, st) == cudaSuccess
               ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_workspace_size(const moe_ffn_desc* d, int32_t T, int32_t act, size_t* bytes) {
    if (!bytes) return MOE_ERR_INVALID_ARG;
    moe_status_t v = validate_ffn_desc(d);
    if (v != MOE_OK) return v;
    if (T < 0 || (act != MOE_ACT_BF16 && act != MOE_ACT_NVFP4)) return MOE_ERR_INVALID_ARG;
    const int path = select_path(T, d->H, d->top_k, act, desc_tc_shape(*d));
    *bytes = Workspace::plan(d->E, d->H, d->I, d->I_shared, d->top_k, T, act, path).total;
    return MOE_OK;
}

moe_status_t moe_prepare_weights(const moe_ffn_desc* d, void** handle_out, void* stream) {
    if (!handle_out) return MOE_ERR_INVALID_ARG;
    *handle_out = nullptr;
    moe_status_t v = validate_ffn_desc(d);
    if (v != MOE_OK) return v;
    Handle* h = new (std::nothrow) Handle();
    if (!h) return MOE_ERR_CUDA;
    h->desc = *d;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    moe_status_t s = MOE_OK;
    const int E = d->E, H = d->H, I = d->I, Is = d->I_shared;
    if (s == MOE_OK) s = prepare_proj(d->gate, E, I, H, h->gate, st);
    if (s == MOE_OK) s = prepare_proj(d->up, E, I, H, h->up, st);
    if (s == MOE_OK) s = prepare_proj(d->down, E, H, I, h->down, st);
    if (Is > 0) {
        if (s == MOE_OK) s = prepare_proj(d->sh_gate, 1, Is, H, h->sh_gate, st);
        if (s == MOE_OK) s = prepare_proj(d->sh_up, 1, Is, H, h->sh_up, st);
        if (s == MOE_OK) s = prepare_proj(d->sh_down, 1, H, Is, h->sh_down, st);
    }
    int dev = 0;
    if (s == MOE_OK && (cudaGetDevice(&dev) != cudaSuccess ||
                        cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess))
        s = MOE_ERR_CUDA;
    if (s == MOE_OK && (cudaMalloc(&h->bar, 256) != cudaSuccess ||
                        cudaMemsetAsync(h->bar, 0, 256, st) != cudaSuccess))
        s = MOE_ERR_CUDA;
    h->tc_shape = desc_tc_shape(*d);
    if (s == MOE_OK && h->tc_shape) {
        FfnLaunch L{};
        L.E = E; L.H = H; L.I = I; L.I_shared = Is;
        L.gate = h->gate.view; L.up = h->up.view; L.down = h->down.view;
        L.sh_gate = h->sh_gate.view; L.sh_up = h->sh_up.view; L.sh_down = h->sh_down.view;
        if (tc_prepare(L, &h->tc, st) != cudaSuccess) s = MOE_ERR_CUDA;
    }
    if (s == MOE_OK && cudaStreamSynchronize(st) != cudaSuccess) s = MOE_ERR_CUDA;
    if (s != MOE_OK) {
        moe_release_weights(h);
        return s;
    }
    *handle_out = h;
    return MOE_OK;
}

moe_status_t moe_release_weights(void* handle) {
    Handle* h = static_cast<Handle*>(handle);
    if (!h || h->magic != 0x4D4F4531u) return MOE_ERR_INVALID_ARG;
    free_proj(h->gate); free_proj(h->up); free_proj(h->down);
    free_proj(h->sh_gate); free_proj(h->sh_up); free_proj(h->sh_down);
    destroy_events(h);
    tc_release(&h->tc);
    if (h->bar) cudaFree(h->bar);
    h->magic = 0;
    delete h;
    return MOE_OK;
}

moe_status_t moe_ffn_forward(const void* handle, int32_t T, int32_t act, float g_act1,
                             float g_act2, const void* x_bf16, const int32_t* topk_ids,
                             const float* topk_w, void* out_bf16, void* workspace,
                             size_t ws_bytes, int32_t* dev_status, void* stream) {
    const Handle* h = static_cast<const Handle*>(handle);
    if (!h || h->magic != 0x4D4F4531u) return MOE_ERR_INVALID_ARG;
    if (T < 0 || (act != MOE_ACT_BF16 && act != MOE_ACT_NVFP4)) return MOE_ERR_INVALID_ARG;
    if (act == MOE_ACT_NVFP4 && (!pow2_positive(g_act1) || !pow2_positive(g_act2)))
        return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !topk_ids || !topk_w || !out_bf16 || !workspace) return MOE_ERR_INVALID_ARG;
    const moe_ffn_desc& d = h->desc;
    const int path = select_path(T, d.H, d.top_k, act, h->tc_shape);
    if (path == PATH_TC && !h->tc.ready) return MOE_ERR_UNSUPPORTED;
    const Workspace ws = Workspace::plan(d.E, d.H, d.I, d.I_shared, d.top_k, T, act, path);
    if (ws_bytes < ws.total) return MOE_ERR_WORKSPACE;
    char* base = static_cast<char*>(workspace);
    const FfnLaunch L = make_launch(h, T, act, g_act1, g_act2, path, ws, base, x_bf16, topk_ids,
                                    topk_w, out_bf16, dev_status);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (path == PATH_DECODE) {
        DecRoute R{};
        R.mode = DEC_ROUTE_GIVEN;
        return run_decode(h, L, R, st);
    }
    const PhaseEvents* ev = h->profile_mask ? &h->events : nullptr;
    cudaError_t err;
    if (path == PATH_TC) {
        TcBuffers B{};
        B.meta = L.meta;
        B.mblock_expert = reinterpret_cast<int32_t*>(base + ws.mblock_expert);
        B.scan = reinterpret_cast<int32_t*>(base + ws.tscan);
        B.padrow_pair = reinterpret_cast<int32_t*>(base + ws.padrow_pair);
        B.tiles1 = reinterpret_cast<int4*>(base + ws.tiles1);
        B.tiles2 = reinterpret_cast<int4*>(base + ws.tiles2);
        B.tokq = reinterpret_cast<uint8_t*>(base + ws.tokq);
        B.toks = reinterpret_cast<uint8_t*>(base + ws.toks);
        B.xq = reinterpret_cast<uint8_t*>(base + ws.txq);
        B.xsf = reinterpret_cast<uint8_t*>(base + ws.txsf);
        B.hq = reinterpret_cast<uint8_t*>(base + ws.thq);
        B.hsf = reinterpret_cast<uint8_t*>(base + ws.thsf);
        B.y = reinterpret_cast<__nv_bfloat16*>(base + ws.ybf);
        B.max_blocks = ws.max_blocks;
        err = launch_ffn_tc(L, h->tc, B, st, ev);
    } else {
        err = launch_ffn(L, st, ev);
    }
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_forward(const void* handle, const moe_route_desc* rd, int32_t act, float g_act1,
                         float g_act2, const void* x_bf16, const float* logits_in,
                         float* logits_out, int32_t* topk_ids, float* topk_w, void* out_bf16,
                         void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
    const Handle* h = static_cast<const Handle*>(handle);
    if (!h || h->magic != 0x4D4F4531u) return MOE_ERR_INVALID_ARG;
    const moe_status_t v = validate_route(rd, logits_in);
    if (v != MOE_OK) return v;
    const moe_ffn_desc& d = h->desc;
    if (rd->E != d.E || rd->top_k != d.top_k || rd->H != d.H || rd->zero_experts != d.zero_experts)
        return MOE_ERR_INVALID_ARG;
    if (act != MOE_ACT_BF16 && act != MOE_ACT_NVFP4) return MOE_ERR_INVALID_ARG;
    if (act == MOE_ACT_NVFP4 && (!pow2_positive(g_act1) || !pow2_positive(g_act2)))
        return MOE_ERR_INVALID_ARG;
    const int T = rd->T;
    if (T == 0) return MOE_OK;
    if (!x_bf16 || !topk_ids || !topk_w || !out_bf16 || !workspace) return MOE_ERR_INVALID_ARG;
    const bool hash = rd->scoring == MOE_SCORE_HASH;  // no router at all
    if (is_hash(rd->scoring) && (!rd->tid2eid || !rd->token_ids)) return MOE_ERR_INVALID_ARG;
    if (!hash && !logits_in && (!rd->w_router || !logits_out)) return MOE_ERR_INVALID_ARG;
    const int path = select_path(T, d.H, d.top_k, act, h->tc_shape);
    if (path != PATH_DECODE) {
        moe_status_t s = moe_route(rd, x_bf16, logits_in, logits_out, topk_ids, topk_w, dev_status,
                                   stream);
        if (s != MOE_OK) return s;
        return moe_ffn_forward(handle, T, act, g_act1, g_act2, x_bf16, topk_ids, topk_w, out_bf16,
                               workspace, ws_bytes, dev_status, stream);
    }
    const Workspace ws = Workspace::plan(d.E, d.H, d.I, d.I_shared, d.top_k, T, act, path);
    if (ws_bytes < ws.total) return MOE_ERR_WORKSPACE;
    const FfnLaunch L = make_launch(h, T, act, g_act1, g_act2, path, ws,
                                    static_cast<char*>(workspace), x_bf16, topk_ids, topk_w,
                                    out_bf16, dev_status);
    DecRoute R{};
    R.mode = hash ? DEC_ROUTE_HASH : (logits_in ? DEC_ROUTE_LOGITS : DEC_ROUTE_ROUTER);
    R.hash_ids = is_hash(rd->scoring) ? 1 : 0;  // ids from the table (weights as R.scoring says)
    R.w_router = rd->w_router;
    R.logits_in = logits_in;
    R.logits_out = logits_out;
    R.bias = (rd->scoring != MOE_SCORE_SOFTMAX && !is_hash(rd->scoring)) ? rd->correction_bias : nullptr;
    R.scoring = rd->scoring;
    R.renorm = rd->renormalize ? 1 : 0;
    R.scaling = rd->routed_scaling;
    R.tid2eid = rd->tid2eid;
    R.token_ids = rd->token_ids;
    R.vocab = rd->vocab;
    R.ids_out = topk_ids;
    R.w_out = topk_w;
    return run_decode(h, L, R, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_workspace_size_host(const moe_ffn_desc* d, int32_t T, int32_t act, size_t* bytes) {
    const moe_status_t v = moe_workspace_size(d, T, act, bytes);
    if (v != MOE_OK) return v;
    *bytes = HostStage::plan(*d, T, act).total;
    return MOE_OK;
}

moe_status_t moe_forward_host(const void* handle, const moe_route_desc* rd, int32_t act,
                              float g_act1, float g_act2, const void* x_host,
                              const int32_t* token_ids_host, void* out_host,
                              int32_t* topk_ids_host, float* topk_w_host, void* workspace,
                              size_t ws_bytes, int32_t* dev_status, void* stream) {
    const Handle* h = static_cast<const Handle*>(handle);
    if (!h || h->magic != 0x4D4F4531u) return MOE_ERR_INVALID_ARG;
    const moe_status_t v = validate_route(rd, nullptr);
    if (v != MOE_OK) return v;
    const moe_ffn_desc& d = h->desc;
    if (rd->E != d.E || rd->top_k != d.top_k || rd->H != d.H || rd->zero_experts != d.zero_experts)
        return MOE_ERR_INVALID_ARG;
    if (act != MOE_ACT_BF16 && act != MOE_ACT_NVFP4) return MOE_ERR_INVALID_ARG;
    if (act == MOE_ACT_NVFP4 && (!pow2_positive(g_act1) || !pow2_positive(g_act2)))
        return MOE_ERR_INVALID_ARG;
    const int T = rd->T;
    if (T == 0) return MOE_OK;
    if (!x_host || !out_host || !workspace) return MOE_ERR_INVALID_ARG;
    const bool hash_ids = is_hash(rd->scoring);
    if (hash_ids && (!token_ids_host || !rd->tid2eid)) return MOE_ERR_INVALID_ARG;
    if (rd->scoring != MOE_SCORE_HASH && !rd->w_router) return MOE_ERR_INVALID_ARG;
    // every check moe_forward makes on the host, before the first copy is enqueued
    if (select_path(T, d.H, d.top_k, act, h->tc_shape) == PATH_TC && !h->tc.ready)
        return MOE_ERR_UNSUPPORTED;
    const HostStage hs = HostStage::plan(d, T, act);
    if (ws_bytes < hs.total) return MOE_ERR_WORKSPACE;
    char* base = static_cast<char*>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t xbytes = sizeof(uint16_t) * (size_t)T * d.H;
    const size_t pbytes = (size_t)T * d.top_k * 4;
    moe_route_desc r = *rd;
    r.token_ids = hash_ids ? reinterpret_cast<const int32_t*>(base + hs.tok) : nullptr;
    if (cudaMemcpyAsync(base + hs.x, x_host, xbytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (hash_ids && cudaMemcpyAsync(base + hs.tok, token_ids_host, sizeof(int32_t) * (size_t)T,
                                    cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    const moe_status_t f = moe_forward(
        handle, &r, act, g_act1, g_act2, base + hs.x, nullptr,
        rd->scoring == MOE_SCORE_HASH ? nullptr : reinterpret_cast<float*>(base + hs.logits),
        reinterpret_cast<int32_t*>(base + hs.ids), reinterpret_cast<float*>(base + hs.w),
        base + hs.out, workspace, ws_bytes, dev_status, stream);
    if (f != MOE_OK) return f;
    if (cudaMemcpyAsync(out_host, base + hs.out, xbytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (topk_ids_host &&
        cudaMemcpyAsync(topk_ids_host, base + hs.ids, pbytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (topk_w_host &&
        cudaMemcpyAsync(topk_w_host, base + hs.w, pbytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status_t moe_set_wait_limit(void* handle, uint64_t cycles) {
    Handle* h = static_cast<Handle*>(handle);
    if (!h || h->magic != 0x4D4F4531u) return MOE_ERR_INVALID_ARG;
    h->wait_cycles = cycles;
    return MOE_OK;
}

moe_status_t moe_skew_barrier(void* handle, void* stream) {
    Handle* h = static_cast<Handle*>(handle);
    if (!h || h->magic != 0x4D4F4531u) return MOE_ERR_INVALID_ARG;
    return launch_barrier_skew(h->bar, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_profile_enable(void* handle, uint32_t mask) {
    Handle* h = static_cast<Handle*>(handle);
    if (!h || h->magic != 0x4D4F4531u || (mask & ~0xFu)) return MOE_ERR_INVALID_ARG;
    destroy_events(h);
    for (int i = 0; i < 4; ++i) {
        if (!(mask & (1u << i))) continue;
        if (cudaEventCreate(&h->events.begin[i]) != cudaSuccess ||
            cudaEventCreate(&h->events.end[i]) != cudaSuccess) {
            destroy_events(h);
            return MOE_ERR_CUDA;
        }
    }
    h->profile_mask = mask;
    return MOE_OK;
}

moe_status_t moe_profile_read(void* handle, float* ms_out) {
    Handle* h = static_cast<Handle*>(handle);
    if (!h || h->magic != 0x4D4F4531u || !ms_out) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i) {
        ms_out[i] = -1.f;
        if (!(h->profile_mask & (1u << i))) continue;
        if (cudaEventSynchronize(h->events.end[i]) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaEventElapsedTime(&ms_out[i], h->events.begin[i], h->events.end[i]) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status_t moe_quantize_act_nvfp4(const void* x_bf16, int64_t rows, int64_t K, float g,
                                    uint8_t* packed, uint8_t* scales, void* stream) {
    if (rows < 0 || K < 16 || K % 16 || !(g > 0.f) || !std::isfinite(g))
        return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!x_bf16 || !packed || !scales) return MOE_ERR_INVALID_ARG;
    return launch_quantize_act(x_bf16, rows, K, g, packed, scales, nullptr,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
