// moe_oracle.cpp -- plain, slow, obviously-correct CPU reference for the MoE FFN block.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the library's compute path may link, load or call
// this file; only the test-suite, the package smoke check and the benchmark's CPU-baseline
// leg use it.  It shares no code, header, table or helper with the CUDA library.
//
// What it computes (sources are the spark_model MoE pages):
//   * block-quantized weight formats -- moe/mod.rs, `MoeLayer::experts_scale_kind` field doc:
//       NVFP4 = packed E2M1 + FP8-E4M3 scale per 16 elements + f32 per-tensor global;
//       MXFP4 = packed E2M1 + E8M0 scale per 32 elements, no global.
//   * routing -- softmax top-K (moe/init.rs, `moe_topk_softmax` handles), sigmoid scoring
//     with a per-expert correction bias used for selection (moe/mod.rs, `correction_bias_dev`
//     field doc), sqrt(softplus) scoring (moe/mod.rs, the `moe_topk_sqrtsoftplus` handles of
//     the DeepSeek-V4 routing), static hash routing through a tid2eid [vocab, top_k] i64
//     table (moe/init.rs, `new_with_hash` doc; moe/mod.rs, `tid2eid_dev` field doc), and
//     softmax + bias routing over num_experts + zero_expert_num logits with zero-computation
//     experts (moe/mod.rs, the LongCat `moe_topk_softmax_bias` / `moe_zero_expert_add` handles
//     and the `router_logits_n` and `zero_accum_dev` field docs).
//   * per expert: gate+up projection, SiLU(gate)*up, down projection, then the top-K weighted
//     sum plus an optional shared expert (moe/mod.rs module doc: "gate+up, silu+down" and
//     `moe_weighted_sum_blend`).
//   * the FP4 x FP4 prefill recipe, whose activations are quantized to NVFP4 before the
//     block-scaled MMA (moe/mod.rs, `moe_fused_gate_up_t_k64_fp4` field doc;
//     qwen3_attention/init.rs, the `quantize_bf16_to_nvfp4` kernel handle).
//
// Floating point: every dot product and every nonlinearity is evaluated in fp64.  The only
// fp32 arithmetic is the activation quantizer Q (A4 mode), which is specified in fp32 so
// that it is reproducible from identical fp32 input.
//
// Readings of points the pages leave open (each is listed in the design notes):
//   - E2M1 element 2i sits in the LOW nibble of byte i, element 2i+1 in the high nibble.
//   - the NVFP4 per-tensor global MULTIPLIES: w = e2m1(code) * e4m3(scale) * global.
//   - top-K ties break toward the lower expert index; ids are emitted in descending
//     selection-score order; hash routing keeps the table's order.
//   - sigmoid routing selects on sigmoid(logit)+bias, weights with the unbiased sigmoid,
//     renormalised over the selected set and multiplied by the routed scaling factor.
//   - sqrt(softplus) routing is the sigmoid scheme with the score sqrt(log(1 + e^logit)).
//   - hash routing weights are 1/top_k.
//   - score-weighted hash routing (the hash layers of the family that ships both the hash and
//     the sqrt(softplus) routing handles): ids from the table in table order, weight of pair
//     j = sqrt(softplus(logit at id j)), renormalised over the token's kept pairs when asked,
//     times the routed scaling; no correction bias, since nothing is selected.
//   - softmax + bias routing: p = softmax over all router logits; selection ranks p + bias;
//     weights are p (renormalised over the selected set when asked) times the routed scaling.
//   - a zero-computation expert (id in [E, E + Z)) returns its input: it adds w * x, the
//     bf16 token itself, whatever the activation precision of the real experts.
//   - the shared expert is added with weight 1.
//   - Q: per 16 consecutive elements, s = E4M3_rne_satfinite(amax / 6 / g);
//     code = E2M1_rne_satfinite(v / (e4m3(s) * g)); all-zero codes when s decodes to 0.
//
// Build: g++ -O2 -fno-fast-math -std=c++17 -shared -fPIC -pthread moe_oracle.cpp
#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <thread>
#include <vector>
#include <functional>

namespace {

// ---------------------------------------------------------------------------------------
// Decode tables (written out by value; the tests pin them against closed forms and against
// an independent library conversion).
// ---------------------------------------------------------------------------------------

// E2M1: 1 sign bit (bit 3), 2 exponent bits, 1 mantissa bit.  Magnitudes by 3-bit code.
const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double g_e4m3[256];
double g_e8m0[256];
double g_e2m1[16];
bool g_tables_ready = false;

void build_tables() {
    if (g_tables_ready) return;
    for (int c = 0; c < 16; ++c) g_e2m1[c] = (c & 8) ? -kE2M1Mag[c & 7] : kE2M1Mag[c & 7];
    // E4M3 (OCP FP8, "fn" flavour): bias 7, no infinities, S.1111.111 is NaN.
    for (int b = 0; b < 256; ++b) {
        int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
        double v;
        if (e == 15 && m == 7) v = NAN;
        else if (e == 0) v = (m / 8.0) * std::ldexp(1.0, -6);
        else v = (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);
        g_e4m3[b] = s ? -v : v;
    }
    // E8M0: unsigned power of two 2^(b-127); 0xFF is NaN.
    for (int b = 0; b < 256; ++b) g_e8m0[b] = (b == 255) ? NAN : std::ldexp(1.0, b - 127);
    g_tables_ready = true;
}

inline double e2m1_val(int code) { return g_e2m1[code & 15]; }

// Nibble k of a packed row: element 2i in the low nibble of byte i.
inline int nibble(const uint8_t* row, int64_t k) {
    uint8_t b = row[k >> 1];
    return (k & 1) ? (b >> 4) : (b & 15);
}

// Round-to-nearest-even onto the E2M1 grid with saturation at +-6, evaluated in fp32
// semantics: the argument is an fp32 value; the nearest magnitude is chosen, ties go to the
// even code (mantissa bit 0).
uint8_t e2m1_encode_rne(float v) {
    if (std::isnan(v)) return 0;  // not produced by finite inputs; kept total
    uint8_t sign = std::signbit(v) ? 8 : 0;
    float a = std::fabs(v);
    int best = 0;
    float best_d = INFINITY;
    for (int c = 0; c < 8; ++c) {
        float d = std::fabs(a - (float)kE2M1Mag[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0)) { best = c; best_d = d; }
    }
    return (uint8_t)(sign | best);
}

// Round-to-nearest-even onto the non-negative finite E4M3 grid, saturating at 448.
uint8_t e4m3_encode_rne_sat(float v) {
    if (!(v > 0.0f)) return 0;  // zero, negative zero (amax is never negative) and NaN
    double a = (double)v;
    if (a >= 448.0) return 0x7E;
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = std::fabs(a - g_e4m3[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0)) { best = c; best_d = d; }
    }
    return (uint8_t)best;
}

// ---------------------------------------------------------------------------------------
// Threading helper: split [0, n) into contiguous chunks over nthreads std::threads.
// ---------------------------------------------------------------------------------------
int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    unsigned hc = std::thread::hardware_concurrency();
    return hc ? (int)hc : 1;
}

void parallel_for(int64_t n, int nthreads, const std::function<void(int64_t)>& body) {
    nthreads = resolve_threads(nthreads);
    if (n <= 0) return;
    if (nthreads == 1 || n == 1) {
        for (int64_t i = 0; i < n; ++i) body(i);
        return;
    }
    std::vector<std::thread> pool;
    int64_t chunk = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        int64_t lo = t * chunk, hi = std::min<int64_t>(n, lo + chunk);
        if (lo >= hi) break;
        pool.emplace_back([lo, hi, &body] { for (int64_t i = lo; i < hi; ++i) body(i); });
    }
    for (auto& th : pool) th.join();
}

inline double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

inline double sigmoid(double z) { return 1.0 / (1.0 + std::exp(-z)); }
inline double sqrt_softplus(double z) {
    const double sp = z > 30.0 ? z : std::log1p(std::exp(z));
    return std::sqrt(sp);
}
// score of the sigmoid-style routers: 1 = sigmoid, 3 = sqrt(softplus)
inline double gate_score(int scoring, double z) { return scoring == 3 ? sqrt_softplus(z) : sigmoid(z); }
inline double silu(double z) { return z * sigmoid(z); }

// One quantized matrix [rows, K] with its format.
struct QMat {
    const uint8_t* packed;   // [rows][K/2]
    const uint8_t* scales;   // [rows][K/16] (NVFP4, E4M3) or [rows][K/32] (MXFP4, E8M0)
    double global;           // NVFP4 per-tensor global; 1 for MXFP4
    int fmt;                 // 0 = NVFP4, 1 = MXFP4
    int64_t rows, K;
};

// Dequantize one row of a quantized matrix into fp64.
void dequant_row(const QMat& m, int64_t r, double* out) {
    const uint8_t* prow = m.packed + r * (m.K / 2);
    if (m.fmt == 0) {
        const uint8_t* srow = m.scales + r * (m.K / 16);
        for (int64_t k = 0; k < m.K; ++k)
            out[k] = e2m1_val(nibble(prow, k)) * g_e4m3[srow[k / 16]] * m.global;
    } else {
        const uint8_t* srow = m.scales + r * (m.K / 32);
        for (int64_t k = 0; k < m.K; ++k)
            out[k] = e2m1_val(nibble(prow, k)) * g_e8m0[srow[k / 32]];
    }
}

// y[r] = sum_k W[r,k] * a[k]  (fp64), for all rows of W.
void qmatvec(const QMat& m, const double* a, double* y, std::vector<double>& rowbuf) {
    rowbuf.resize(m.K);
    for (int64_t r = 0; r < m.rows; ++r) {
        dequant_row(m, r, rowbuf.data());
        double acc = 0.0;
        for (int64_t k = 0; k < m.K; ++k) acc += rowbuf[k] * a[k];
        y[r] = acc;
    }
}

// The activation quantizer Q, in fp32: see the file header.  Writes the dequantized fp32
// values (exactly representable) into out[0..n).
void quant_dequant_nvfp4_f32(const float* v, int64_t n, float g, double* out,
                             uint8_t* packed, uint8_t* scales) {
    for (int64_t b0 = 0; b0 < n; b0 += 16) {
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(v[b0 + i]));
        float q = amax / 6.0f;
        q = q / g;
        uint8_t s = e4m3_encode_rne_sat(q);
        float sdec = (float)g_e4m3[s];
        float denom = sdec * g;
        if (scales) scales[b0 / 16] = s;
        for (int i = 0; i < 16; ++i) {
            uint8_t code = 0;
            if (denom != 0.0f) code = e2m1_encode_rne(v[b0 + i] / denom);
            if (packed) {
                int64_t k = b0 + i;
                if ((k & 1) == 0) packed[k >> 1] = code;
                else packed[k >> 1] = (uint8_t)(packed[k >> 1] | (code << 4));
            }
            out[b0 + i] = e2m1_val(code) * (double)sdec * (double)g;
        }
    }
}

}  // namespace

extern "C" {

// ----- tables -----------------------------------------------------------------------------
void orc_tables(double* e2m1_16, double* e4m3_256, double* e8m0_256) {
    build_tables();
    if (e2m1_16) std::memcpy(e2m1_16, g_e2m1, sizeof(g_e2m1));
    if (e4m3_256) std::memcpy(e4m3_256, g_e4m3, sizeof(g_e4m3));
    if (e8m0_256) std::memcpy(e8m0_256, g_e8m0, sizeof(g_e8m0));
}

uint8_t orc_e2m1_encode(float v) { build_tables(); return e2m1_encode_rne(v); }
uint8_t orc_e4m3_encode(float v) { build_tables(); return e4m3_encode_rne_sat(v); }

// Activation quantizer Q over rows of length K (K % 16 == 0), fp32 input.
// packed [rows][K/2], scales [rows][K/16], deq [rows][K] (fp64 of the exact dequantized value).
void orc_quant_nvfp4(const float* v, int64_t rows, int64_t K, float g,
                     uint8_t* packed, uint8_t* scales, double* deq) {
    build_tables();
    std::vector<double> tmp(K);
    for (int64_t r = 0; r < rows; ++r) {
        if (packed) std::memset(packed + r * (K / 2), 0, K / 2);
        quant_dequant_nvfp4_f32(v + r * K, K, g, deq ? deq + r * K : tmp.data(),
                                packed ? packed + r * (K / 2) : nullptr,
                                scales ? scales + r * (K / 16) : nullptr);
    }
}

// Dequantize a whole [rows, K] matrix to fp64.
void orc_dequant(const uint8_t* packed, const uint8_t* scales, double global, int fmt,
                 int64_t rows, int64_t K, double* out) {
    build_tables();
    QMat m{packed, scales, fmt == 0 ? global : 1.0, fmt, rows, K};
    for (int64_t r = 0; r < rows; ++r) dequant_row(m, r, out + r * K);
}

// ----- routing ------------------------------------------------------------------------------
// scoring: 0 softmax, 1 sigmoid (+ correction bias for selection), 2 hash,
// 3 sqrt(softplus) (+ correction bias for selection), 4 softmax (+ correction bias for
// selection), 5 hash ids with sqrt(softplus) router-score weights.  E here is the router
// width (real + zero-computation experts).
// Inputs: either x_bf16 [T,H] + w_router_bf16 [E,H] (router GEMM) or logits_in f32 [T,E].
// Outputs: logits_out [T,E] fp64 (may be null), ids [T,k], w [T,k] fp64, score_out [T,E]
// fp64 selection score (may be null).  Returns 0, or -1 on an invalid argument.
// status_out (may be null) receives the same bits the device status word uses:
//   1 = a hash table entry outside [0,E) (pair dropped: id -1, weight 0),
//   2 = a token id outside [0,vocab) (all of the token's pairs dropped),
//   4 = a non-finite logit (ranked below every finite score).
int orc_route(int T, int E, int H, int k, int scoring, int renorm, double scaling,
              const uint16_t* x_bf16, const uint16_t* w_router_bf16, const float* logits_in,
              const float* bias, const int64_t* tid2eid, int64_t vocab, const int32_t* token_ids,
              double* logits_out, int32_t* ids, double* w, double* score_out, int32_t* status_out,
              int nthreads) {
    build_tables();
    if (T < 0 || E <= 0 || k <= 0 || k > E || scoring < 0 || scoring > 5) return -1;
    std::vector<int32_t> tok_status(T, 0);
    if (scoring == 2) {
        for (int t = 0; t < T; ++t) {
            int64_t tok = token_ids[t];
            if (tok < 0 || tok >= vocab) {
                tok_status[t] |= 2;
                for (int j = 0; j < k; ++j) { ids[t * k + j] = -1; w[t * k + j] = 0.0; }
                continue;
            }
            for (int j = 0; j < k; ++j) {
                int64_t e = tid2eid[tok * k + j];
                if (e < 0 || e >= E) {
                    tok_status[t] |= 1;
                    ids[t * k + j] = -1;
                    w[t * k + j] = 0.0;
                } else {
                    ids[t * k + j] = (int32_t)e;
                    w[t * k + j] = scaling / k;
                }
            }
        }
    } else {
        parallel_for(T, nthreads, [&](int64_t t) {
            std::vector<double> logit(E), v(E);
            for (int e = 0; e < E; ++e) {
                double l;
                if (logits_in) {
                    l = (double)logits_in[t * E + e];
                } else {
                    double acc = 0.0;
                    for (int h = 0; h < H; ++h)
                        acc += bf16_to_double(x_bf16[t * (int64_t)H + h]) *
                               bf16_to_double(w_router_bf16[(int64_t)e * H + h]);
                    l = acc;
                }
                logit[e] = l;
                if (logits_out) logits_out[t * E + e] = l;
            }
            if (scoring == 5) {
                // the table chooses the experts (in its order); the router's sqrt(softplus)
                // scores of those experts give the weights
                const int64_t tok = token_ids[t];
                if (score_out)
                    for (int e = 0; e < E; ++e)
                        score_out[t * E + e] = std::isfinite(logit[e]) ? sqrt_softplus(logit[e]) : 0.0;
                if (tok < 0 || tok >= vocab) {
                    tok_status[t] |= 2;
                    for (int j = 0; j < k; ++j) { ids[t * k + j] = -1; w[t * k + j] = 0.0; }
                    return;
                }
                std::vector<double> sj(k, 0.0);
                double ssum = 0.0;
                for (int j = 0; j < k; ++j) {
                    const int64_t e = tid2eid[tok * k + j];
                    if (e < 0 || e >= E) {
                        tok_status[t] |= 1;
                        ids[t * k + j] = -1;
                        continue;
                    }
                    ids[t * k + j] = (int32_t)e;
                    if (std::isfinite(logit[e])) sj[j] = sqrt_softplus(logit[e]);
                    else tok_status[t] |= 4;
                    ssum += sj[j];
                }
                for (int j = 0; j < k; ++j) {
                    const double v = renorm ? (ssum > 0.0 ? sj[j] / ssum : 0.0) : sj[j];
                    w[t * k + j] = v * scaling;
                }
                return;
            }
            bool nonfinite = false;
            double lmax = -INFINITY;
            for (int e = 0; e < E; ++e)
                if (std::isfinite(logit[e])) lmax = std::max(lmax, logit[e]);
            double zall = 0.0;  // softmax denominator over every finite logit
            for (int e = 0; e < E; ++e)
                if (std::isfinite(logit[e])) zall += std::exp(logit[e] - lmax);
            for (int e = 0; e < E; ++e) {
                double l = logit[e];
                if (!std::isfinite(l)) { nonfinite = true; v[e] = -INFINITY; continue; }
                if (scoring == 0) v[e] = l;  // softmax is monotone in the logit
                else if (scoring == 4) v[e] = std::exp(l - lmax) / zall + (bias ? (double)bias[e] : 0.0);
                else v[e] = gate_score(scoring, l) + (bias ? (double)bias[e] : 0.0);
            }
            if (nonfinite) tok_status[t] |= 4;
            if (score_out)
                for (int e = 0; e < E; ++e) score_out[t * E + e] = v[e];
            // full sort: descending score, ascending index on ties
            std::vector<int> order(E);
            for (int e = 0; e < E; ++e) order[e] = e;
            std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
                if (v[a] != v[b]) return v[a] > v[b];
                return a < b;
            });
            if (scoring == 0 || scoring == 4) {
                // softmax over all E, then the selected subset (optionally renormalised)
                double zsel = 0.0;
                for (int j = 0; j < k; ++j) {
                    double l = logit[order[j]];
                    if (std::isfinite(l)) zsel += std::exp(l - lmax);
                }
                for (int j = 0; j < k; ++j) {
                    int e = order[j];
                    double p = std::isfinite(logit[e]) ? std::exp(logit[e] - lmax) : 0.0;
                    ids[t * k + j] = e;
                    w[t * k + j] = (renorm ? p / zsel : p / zall) * scaling;
                }
            } else {
                double ssel = 0.0;
                for (int j = 0; j < k; ++j) {
                    double l = logit[order[j]];
                    if (std::isfinite(l)) ssel += gate_score(scoring, l);
                }
                for (int j = 0; j < k; ++j) {
                    int e = order[j];
                    double s = std::isfinite(logit[e]) ? gate_score(scoring, logit[e]) : 0.0;
                    ids[t * k + j] = e;
                    w[t * k + j] = (renorm ? s / ssel : s) * scaling;
                }
            }
        });
    }
    if (status_out) {
        int32_t st = 0;
        for (int t = 0; t < T; ++t) st |= tok_status[t];
        *status_out = st;
    }
    return 0;
}

// ----- expert FFN + combine ----------------------------------------------------------------
// Weight tensors are stacked over experts: packed [E][N][K/2], scales [E][N][K/sv],
// globals [E] (NVFP4) or null (MXFP4).  gate/up: N = I, K = H.  down: N = H, K = I.
// The shared expert (if sh_I > 0) has the same layout with one expert and intermediate sh_I.
// act_mode: 0 = bf16 activations (A16), 1 = NVFP4 activations (A4) with globals g1 (for x)
// and g2 (for h).  ids [T,k] (id -1 = dropped pair; E <= id < E + Z a zero-computation expert
// that adds w * x), w [T,k] fp64.  out [T,H] fp64.
struct OrcProj {
    const uint8_t* packed;
    const uint8_t* scales;
    const float* globals;
    int fmt;
};

int orc_moe_ffn(int T, int E, int H, int I, int k, int Z,
                OrcProj gate, OrcProj up, OrcProj down,
                int sh_I, OrcProj sh_gate, OrcProj sh_up, OrcProj sh_down,
                int act_mode, float g1, float g2,
                const uint16_t* x_bf16, const int32_t* ids, const double* w,
                double* out, int nthreads) {
    build_tables();
    if (T < 0 || E <= 0 || Z < 0 || H % 32 || I % 32 || (sh_I % 32)) return -1;
    auto sv = [](int fmt) { return fmt == 0 ? 16 : 32; };
    auto expert_mat = [&](const OrcProj& p, int e, int64_t N, int64_t K) {
        QMat m;
        m.packed = p.packed + (int64_t)e * N * (K / 2);
        m.scales = p.scales + (int64_t)e * N * (K / sv(p.fmt));
        m.global = (p.fmt == 0 && p.globals) ? (double)p.globals[e] : 1.0;
        m.fmt = p.fmt;
        m.rows = N;
        m.K = K;
        return m;
    };
    // one FFN evaluation: y = W_d * act(h), h = silu(W_g a) * (W_u a)
    auto ffn = [&](const QMat& mg, const QMat& mu, const QMat& md, const double* a,
                   int64_t Iexp, double* y, std::vector<double>& rowbuf) {
        std::vector<double> gv(Iexp), uv(Iexp), h(Iexp);
        qmatvec(mg, a, gv.data(), rowbuf);
        qmatvec(mu, a, uv.data(), rowbuf);
        for (int64_t i = 0; i < Iexp; ++i) h[i] = silu(gv[i]) * uv[i];
        if (act_mode == 1) {
            std::vector<float> hf(Iexp);
            for (int64_t i = 0; i < Iexp; ++i) hf[i] = (float)h[i];
            quant_dequant_nvfp4_f32(hf.data(), Iexp, g2, h.data(), nullptr, nullptr);
        }
        qmatvec(md, h.data(), y, rowbuf);
    };
    parallel_for(T, nthreads, [&](int64_t t) {
        std::vector<double> a(H), y(H), rowbuf;
        if (act_mode == 1) {
            std::vector<float> xf(H);
            for (int h = 0; h < H; ++h) xf[h] = (float)bf16_to_double(x_bf16[t * (int64_t)H + h]);
            quant_dequant_nvfp4_f32(xf.data(), H, g1, a.data(), nullptr, nullptr);
        } else {
            for (int h = 0; h < H; ++h) a[h] = bf16_to_double(x_bf16[t * (int64_t)H + h]);
        }
        double* o = out + t * (int64_t)H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = ids[t * k + j];
            double wj = w[t * k + j];
            if (e >= E && e < E + Z) {  // zero-computation expert: the input itself
                for (int h = 0; h < H; ++h) o[h] += wj * bf16_to_double(x_bf16[t * (int64_t)H + h]);
                continue;
            }
            if (e < 0 || e >= E) continue;
            ffn(expert_mat(gate, e, I, H), expert_mat(up, e, I, H), expert_mat(down, e, H, I),
                a.data(), I, y.data(), rowbuf);
            for (int h = 0; h < H; ++h) o[h] += wj * y[h];
        }
        if (sh_I > 0) {
            ffn(expert_mat(sh_gate, 0, sh_I, H), expert_mat(sh_up, 0, sh_I, H),
                expert_mat(sh_down, 0, H, sh_I), a.data(), sh_I, y.data(), rowbuf);
            for (int h = 0; h < H; ++h) o[h] += y[h];
        }
    });
    return 0;
}

int orc_hardware_threads() { return resolve_threads(0); }

}  // extern "C"
