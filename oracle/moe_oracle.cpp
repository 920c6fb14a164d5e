// Host-only reference ("oracle") for the routed mixture-of-experts FFN.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link or call this file:
// only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg use it.
// It includes no CUDA header and shares no code, table or constant generator with the GPU
// library; both sides read the same seeded input bytes and nothing else.
//
// What it computes, and where that is written down:
//   * Per (token, slot) expert chain: gate = Wg.x, up = Wu.x, clamped SwiGLU, down = Wd.a —
//     "memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs", `reference_expert` and
//     `reference_grouped_projections`; the projection order (gate, up, then down on the
//     activation) is the same in "memra-engine 0.131.0 src/dsv4_ep.rs", `chain`.
//   * Clamped SwiGLU  silu(min(g, L)) * clamp(u, -L, L) — "spark_model
//     layers/glm5next_mlp/forward.rs", doc comment of `swiglu_rows`; no clamp when L = +inf,
//     as the gate binary's `activation_limit = None` arm (`silu_mul`) does.
//   * Weighted combine  out[t] = sum_k w[t,k] * down[t,k], slots in order 0..top_k-1 —
//     ep_step_fp8_gate.rs, `combine_down_rows_host`.
//   * FP8 weight = e4m3(code) * S[n/128][k/128] with one fp32 scale per 128x128 block, banks
//     stacked [E][N][K] — ep_step_fp8_gate.rs, `expert_matrix` (expert stride N*K codes and
//     scale_rows*scale_cols scales).
//   * NVFP4 weight = e2m1(nibble) * e4m3(sf[n][k/16]) * scale_2, two codes per byte and one
//     scale byte per 16 elements — dsv4_ep.rs, `chain` (wstride = inter*hidden/2,
//     sstride = inter*hidden/16); scale_2 is a by-value f32 — forward.rs, `w4a16_gemv`. Or one
//     scale_2 per expert and projection (oracle_moe_nvfp4_expert_scale2) — forward.rs,
//     `w4a16_gemv_moe` (the expert table's scale2_vals) and dsv4_ep.rs's EP matrix test (one
//     macro scale per expert and projection).
//   * Route permutation: per-expert counts, exclusive offsets, expert-sorted pair list and its
//     inverse — forward.rs, `Glm5NextMlpWorkspace` (sorted ids, expert_offsets[E+1],
//     token_to_perm). Ties inside one expert are broken by ascending pair index t*top_k+k
//     (the pages leave this open; this is the stable reading).
//
// Arithmetic: every product and sum is carried in IEEE double. E4M3, E2M1 and bf16 are decoded
// from their bit definitions. Results do not depend on the thread count: each output element is
// produced by one thread, summing in index order.
//
//   * Router (in front of the FFN): fp32 logits = bf16 x . bf16 router rows [E][H]; sigmoid, plus a
//     per-expert bias for the selection only; top-k by that score; weights = the selected
//     sigmoids, optionally renormalised to sum 1, times routed_scale; one expert group — "spark_model
//     layers/glm5next_mlp/forward.rs", `forward_moe` router step (logits GEMM with f32 output, then
//     one top-k launch taking logits, router_bias, top_k, n_group = 1, routed_scale, renormalize)
//     and the Step gate's `upload_sigmoid_topk_router(router, bias, top_k, router_scale,
//     route_norm)`. The pages print no body for the top-k step; the reading here: selection by
//     sigmoid(l) + bias, descending, ties to the lower expert index; weights from sigmoid(l)
//     without the bias.
//
// Parity pins (tests/test_oracle_pins.py): all 256 E4M3 codes against torch's float8_e4m3fn,
// the E2M1 magnitude table, hand-built code/scale bytes, clamp boundary values, the pages' combine
// worked example, brute-force dense float64 matmul on tiny banks, and a brute-force stable sort
// for the permutation. No function here is "parity unpinned".

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---- number formats, from their bit definitions ----------------------------------------------

// E4M3 ("FN" variant): sign | 4 exponent bits, bias 7 | 3 mantissa bits. Exponent field 0 is
// subnormal (m/8 * 2^-6). S.1111.111 is NaN; there is no infinity; the largest finite is 448.
double e4m3_value(uint8_t code) {
    const int sign = code >> 7;
    const int exp_field = (code >> 3) & 0xF;
    const int mant = code & 0x7;
    if (exp_field == 0xF && mant == 0x7) return std::nan("");
    double mag;
    if (exp_field == 0)
        mag = std::ldexp(mant / 8.0, -6);
    else
        mag = std::ldexp(1.0 + mant / 8.0, exp_field - 7);
    return sign ? -mag : mag;
}

// E2M1: sign | 2 exponent bits, bias 1 | 1 mantissa bit. Exponent field 0 is subnormal
// (m/2 * 2^0). Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no NaN or infinity.
double e2m1_value(uint8_t nibble) {
    const int sign = (nibble >> 3) & 1;
    const int exp_field = (nibble >> 1) & 0x3;
    const int mant = nibble & 0x1;
    double mag;
    if (exp_field == 0)
        mag = mant * 0.5;
    else
        mag = std::ldexp(1.0 + mant / 2.0, exp_field - 1);
    return sign ? -mag : mag;
}

// bf16 is the top half of an IEEE binary32, so widening is exact.
double bf16_value(uint16_t bits) {
    uint32_t u = static_cast<uint32_t>(bits) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return static_cast<double>(f);
}

// Round a double to bf16 (8 significant bits, binary32 exponent range), nearest-even, in ONE
// step from the double (no intermediate binary32 rounding).
uint16_t bf16_round(double v) {
    if (std::isnan(v)) return 0x7FC0;
    const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
    double a = std::fabs(v);
    if (a == 0.0) return sign;
    if (std::isinf(a)) return sign | 0x7F80;
    int e;
    std::frexp(a, &e);                       // a = f * 2^e, f in [0.5, 1)
    int q = e - 8;                           // unit of the last kept bit for a normal bf16
    if (q < -133) q = -133;                  // subnormal step is 2^-133
    double scaled = std::ldexp(a, -q);       // exact: power-of-two scaling
    double r = std::nearbyint(scaled);       // default rounding mode: nearest, ties to even
    double out = std::ldexp(r, q);
    if (out >= std::ldexp(1.0, 128)) return sign | 0x7F80;   // overflow to infinity
    float f = static_cast<float>(out);       // exact: out has <= 8 significant bits
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return sign | static_cast<uint16_t>((u >> 16) & 0x7FFF);
}

// silu(z) = z / (1 + exp(-z)); the clamp is asymmetric: gate only from above, up both ways.
double clamped_swiglu(double g, double u, double limit) {
    if (g > limit) g = limit;
    if (u > limit) u = limit;
    if (u < -limit) u = -limit;
    return g / (1.0 + std::exp(-g)) * u;
}

// ---- dequantised weight access -------------------------------------------------------------

struct Bank {
    int fmt;            // 1 = FP8 E4M3 with [N/128][K/128] fp32 block scales; 2 = NVFP4
    const uint8_t* codes;
    const float* block_scale;   // FP8
    const uint8_t* sf;          // NVFP4, [E][N][K/16] E4M3 bytes
    double scale_2;             // NVFP4
    int N, K;
    // NVFP4 with one scale_2 per expert: expert e's is s2e[e * s2_stride] (null: scale_2 for all)
    const float* s2e = nullptr;
    int s2_stride = 1;
    // Dequantised W[e][n][k].
    double w(int e, int n, int k) const {
        if (fmt == 1) {
            const size_t idx = (static_cast<size_t>(e) * N + n) * K + k;
            const int sr = N / 128, sc = K / 128;
            const size_t sidx = (static_cast<size_t>(e) * sr + n / 128) * sc + k / 128;
            return e4m3_value(codes[idx]) * static_cast<double>(block_scale[sidx]);
        }
        const size_t byte = (static_cast<size_t>(e) * N + n) * (K / 2) + k / 2;
        const uint8_t nib = (k % 2 == 0) ? (codes[byte] & 0xF) : (codes[byte] >> 4);
        const size_t sfi = (static_cast<size_t>(e) * N + n) * (K / 16) + k / 16;
        const double s2 = s2e != nullptr ? static_cast<double>(s2e[static_cast<size_t>(e) * s2_stride]) : scale_2;
        return e2m1_value(nib) * e4m3_value(sf[sfi]) * s2;
    }
};

template <class F>
void parallel_for(int64_t n, int nthreads, F fn) {
    if (nthreads <= 1 || n < 2) {
        for (int64_t i = 0; i < n; ++i) fn(i);
        return;
    }
    if (nthreads > n) nthreads = static_cast<int>(n);
    std::vector<std::thread> pool;
    pool.reserve(nthreads);
    for (int t = 0; t < nthreads; ++t) {
        const int64_t lo = n * t / nthreads, hi = n * (t + 1) / nthreads;   // static partition
        pool.emplace_back([=] {
            for (int64_t i = lo; i < hi; ++i) fn(i);
        });
    }
    for (auto& th : pool) th.join();
}

int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    unsigned hc = std::thread::hardware_concurrency();
    return hc ? static_cast<int>(hc) : 1;
}

// One routed MoE FFN over the selected tokens. All intermediates optional.
//   g, u, a : [T*topk][I]   y : [T*topk][H]   out : [T][H] (double and bf16)
int moe_forward(const uint16_t* x, int T, int H, int I, int E, int topk, const int32_t* ids,
                const float* wts, const Bank& gate, const Bank& up, const Bank& down, double limit,
                const int32_t* token_list, int n_tokens, double* out_f64, uint16_t* out_bf16,
                double* g_out, double* u_out, double* a_out, double* y_out, int nthreads,
                int32_t* err) {
    nthreads = resolve_threads(nthreads);
    int32_t flags = 0;
    if (token_list == nullptr) n_tokens = T;
    std::vector<int> tokens(n_tokens);
    for (int i = 0; i < n_tokens; ++i) tokens[i] = token_list ? token_list[i] : i;
    for (int i = 0; i < n_tokens; ++i)
        if (tokens[i] < 0 || tokens[i] >= T) return -2;

    // Which (token, slot) pairs contribute: id -1 is an unfilled slot; any other id outside
    // [0, E) is an error that contributes nothing and raises bit 0 of the error word.
    const int64_t npairs = static_cast<int64_t>(n_tokens) * topk;
    std::vector<int> pair_expert(npairs);
    for (int64_t q = 0; q < npairs; ++q) {
        const int t = tokens[q / topk], k = static_cast<int>(q % topk);
        const int32_t e = ids[static_cast<size_t>(t) * topk + k];
        if (e >= 0 && e < E)
            pair_expert[q] = e;
        else {
            pair_expert[q] = -1;
            if (e != -1) flags |= 1;
        }
    }

    std::vector<double> xd(static_cast<size_t>(n_tokens) * H);
    for (int i = 0; i < n_tokens; ++i)
        for (int h = 0; h < H; ++h)
            xd[static_cast<size_t>(i) * H + h] = bf16_value(x[static_cast<size_t>(tokens[i]) * H + h]);

    // gate / up / activation for every (pair, n)
    std::vector<double> act(static_cast<size_t>(npairs) * I, 0.0);
    parallel_for(npairs * I, nthreads, [&](int64_t idx) {
        const int64_t q = idx / I;
        const int n = static_cast<int>(idx % I);
        const int e = pair_expert[q];
        if (e < 0) return;
        const double* xr = &xd[static_cast<size_t>(q / topk) * H];
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            g += xr[h] * gate.w(e, n, h);
            u += xr[h] * up.w(e, n, h);
        }
        const double a = clamped_swiglu(g, u, limit);
        act[idx] = a;
        if (g_out) g_out[idx] = g;
        if (u_out) u_out[idx] = u;
        if (a_out) a_out[idx] = a;
    });

    // down projection for every (pair, j)
    std::vector<double> y(static_cast<size_t>(npairs) * H, 0.0);
    parallel_for(npairs * H, nthreads, [&](int64_t idx) {
        const int64_t q = idx / H;
        const int j = static_cast<int>(idx % H);
        const int e = pair_expert[q];
        if (e < 0) return;
        const double* ar = &act[static_cast<size_t>(q) * I];
        double s = 0.0;
        for (int n = 0; n < I; ++n) s += ar[n] * down.w(e, j, n);
        y[idx] = s;
        if (y_out) y_out[idx] = s;
    });

    // weighted combine, slot order
    for (int i = 0; i < n_tokens; ++i) {
        const int t = tokens[i];
        for (int j = 0; j < H; ++j) {
            double s = 0.0;
            for (int k = 0; k < topk; ++k) {
                const int64_t q = static_cast<int64_t>(i) * topk + k;
                if (pair_expert[q] < 0) continue;
                s += static_cast<double>(wts[static_cast<size_t>(t) * topk + k]) *
                     y[static_cast<size_t>(q) * H + j];
            }
            if (out_f64) out_f64[static_cast<size_t>(i) * H + j] = s;
            if (out_bf16) out_bf16[static_cast<size_t>(i) * H + j] = bf16_round(s);
        }
    }
    if (err) *err |= flags;
    return 0;
}

bool shapes_ok(int T, int H, int I, int E, int topk) {
    return T >= 1 && H >= 128 && I >= 128 && H % 128 == 0 && I % 128 == 0 && E >= 1 && topk >= 1;
}

}  // namespace

extern "C" {

double oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }
double oracle_e2m1_value(uint8_t nibble) { return e2m1_value(nibble & 0xF); }
double oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }
uint16_t oracle_bf16_round(double v) { return bf16_round(v); }
double oracle_clamped_swiglu(double g, double u, double limit) { return clamped_swiglu(g, u, limit); }

// Combine only: down [T*topk][width] rows, weights [T*topk] -> out [T][width], slot order.
// Mirrors ep_step_fp8_gate.rs `combine_down_rows_host` (which also rejects mismatched sizes).
int oracle_combine(const double* down, const double* weights, int T, int topk, int width,
                   double* out) {
    if (T < 1 || topk < 1 || width < 1) return -2;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < width; ++j) {
            double s = 0.0;
            for (int k = 0; k < topk; ++k) {
                const size_t q = static_cast<size_t>(t) * topk + k;
                s += weights[q] * down[q * width + j];
            }
            out[static_cast<size_t>(t) * width + j] = s;
        }
    return 0;
}

// Dequantise one expert's full [N][K] matrix to doubles (test helper).
int oracle_dequant_fp8(const uint8_t* codes, const float* scales, int E, int N, int K, int e,
                       double* out) {
    if (N % 128 || K % 128 || e < 0 || e >= E) return -2;
    Bank b{1, codes, scales, nullptr, 0.0, N, K};
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) out[static_cast<size_t>(n) * K + k] = b.w(e, n, k);
    return 0;
}

int oracle_dequant_nvfp4(const uint8_t* packed, const uint8_t* sf, double scale_2, int E, int N,
                         int K, int e, double* out) {
    if (K % 16 || e < 0 || e >= E) return -2;
    Bank b{2, packed, nullptr, sf, scale_2, N, K};
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) out[static_cast<size_t>(n) * K + k] = b.w(e, n, k);
    return 0;
}

// Route histogram / counting-sort permutation.
//   counts[E], offsets[E+1] (offsets[E] = number of valid pairs), sorted_pair[T*topk]
//   (first offsets[E] entries valid, value = t*topk+k), pair_to_sorted[T*topk] (-1 = not routed).
int oracle_route_permute(const int32_t* ids, int T, int topk, int E, int32_t* counts,
                         int32_t* offsets, int32_t* sorted_pair, int32_t* pair_to_sorted,
                         int32_t* err) {
    if (T < 1 || topk < 1 || E < 1) return -2;
    const int64_t P = static_cast<int64_t>(T) * topk;
    int32_t flags = 0;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) {
        const int32_t e = ids[p];
        if (e >= 0 && e < E)
            ++counts[e];
        else if (e != -1)
            flags |= 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    std::vector<int32_t> cursor(offsets, offsets + E);
    for (int64_t p = 0; p < P; ++p) {
        const int32_t e = ids[p];
        if (e >= 0 && e < E) {
            const int32_t pos = cursor[e]++;
            sorted_pair[pos] = static_cast<int32_t>(p);
            pair_to_sorted[p] = pos;
        } else {
            pair_to_sorted[p] = -1;
        }
    }
    for (int64_t s = offsets[E]; s < P; ++s) sorted_pair[s] = -1;
    if (err) *err |= flags;
    return 0;
}

// Full FP8 routed FFN. token_list (nullable) restricts the computation to those tokens; the
// outputs are then laid out in token_list order.
int oracle_moe_fp8(const uint16_t* x, int T, int H, int I, int E, int topk, const int32_t* ids,
                   const float* wts, const uint8_t* w_gate, const float* s_gate,
                   const uint8_t* w_up, const float* s_up, const uint8_t* w_down,
                   const float* s_down, double limit, const int32_t* token_list, int n_tokens,
                   double* out_f64, uint16_t* out_bf16, double* g_out, double* u_out,
                   double* a_out, double* y_out, int nthreads, int32_t* err) {
    if (!shapes_ok(T, H, I, E, topk)) return -2;
    if (!(limit > 0.0)) return -4;
    Bank g{1, w_gate, s_gate, nullptr, 0.0, I, H};
    Bank u{1, w_up, s_up, nullptr, 0.0, I, H};
    Bank d{1, w_down, s_down, nullptr, 0.0, H, I};
    return moe_forward(x, T, H, I, E, topk, ids, wts, g, u, d, limit, token_list, n_tokens,
                       out_f64, out_bf16, g_out, u_out, a_out, y_out, nthreads, err);
}

// Full NVFP4 (W4A16) routed FFN; scale_2 is one by-value scalar per projection.
int oracle_moe_nvfp4(const uint16_t* x, int T, int H, int I, int E, int topk, const int32_t* ids,
                     const float* wts, const uint8_t* w_gate, const uint8_t* sf_gate,
                     float scale2_gate, const uint8_t* w_up, const uint8_t* sf_up,
                     float scale2_up, const uint8_t* w_down, const uint8_t* sf_down,
                     float scale2_down, double limit, const int32_t* token_list, int n_tokens,
                     double* out_f64, uint16_t* out_bf16, double* g_out, double* u_out,
                     double* a_out, double* y_out, int nthreads, int32_t* err) {
    if (!shapes_ok(T, H, I, E, topk)) return -2;
    if (!(limit > 0.0)) return -4;
    Bank g{2, w_gate, nullptr, sf_gate, scale2_gate, I, H};
    Bank u{2, w_up, nullptr, sf_up, scale2_up, I, H};
    Bank d{2, w_down, nullptr, sf_down, scale2_down, H, I};
    return moe_forward(x, T, H, I, E, topk, ids, wts, g, u, d, limit, token_list, n_tokens,
                       out_f64, out_bf16, g_out, u_out, a_out, y_out, nthreads, err);
}

// The same with one scale_2 per expert and projection: expert e's is scale2_x[e * stride]
// ("memra-engine 0.131.0 src/dsv4_ep.rs", the EP matrix test's macro scales, one per expert and
// projection; "spark_model layers/glm5next_mlp/forward.rs", `w4a16_gemv_moe`: the expert table's
// scale2_vals, one per expert).
int oracle_moe_nvfp4_expert_scale2(const uint16_t* x, int T, int H, int I, int E, int topk,
                                   const int32_t* ids, const float* wts, const uint8_t* w_gate,
                                   const uint8_t* sf_gate, const float* scale2_gate, const uint8_t* w_up,
                                   const uint8_t* sf_up, const float* scale2_up, const uint8_t* w_down,
                                   const uint8_t* sf_down, const float* scale2_down, int stride,
                                   double limit, const int32_t* token_list, int n_tokens, double* out_f64,
                                   uint16_t* out_bf16, double* g_out, double* u_out, double* a_out,
                                   double* y_out, int nthreads, int32_t* err) {
    if (!shapes_ok(T, H, I, E, topk)) return -2;
    if (!(limit > 0.0)) return -4;
    if (scale2_gate == nullptr || scale2_up == nullptr || scale2_down == nullptr || stride < 1) return -3;
    Bank g{2, w_gate, nullptr, sf_gate, 0.0, I, H, scale2_gate, stride};
    Bank u{2, w_up, nullptr, sf_up, 0.0, I, H, scale2_up, stride};
    Bank d{2, w_down, nullptr, sf_down, 0.0, H, I, scale2_down, stride};
    return moe_forward(x, T, H, I, E, topk, ids, wts, g, u, d, limit, token_list, n_tokens,
                       out_f64, out_bf16, g_out, u_out, a_out, y_out, nthreads, err);
}

// Router logits in double: logits[t][e] = sum_h x[t][h] * W[e][h] (bf16 inputs, exact products).
int oracle_router_logits(const uint16_t* x, int T, int H, const uint16_t* w, int E, double* logits) {
    if (T < 1 || H < 1 || E < 1) return -2;
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += bf16_value(x[static_cast<size_t>(t) * H + h]) * bf16_value(w[static_cast<size_t>(e) * H + h]);
            logits[static_cast<size_t>(t) * E + e] = acc;
        }
    return 0;
}

// Router top-k from given logits, in double: score = sigmoid(l) + bias (bias nullable), the topk
// largest scores in descending order (ties: lower expert index first); weight = sigmoid(l) of the
// pick, divided by the sum over the picks when renormalize != 0, times routed_scale.
int oracle_router_topk(const double* logits, int T, int E, const double* bias, int topk,
                       double routed_scale, int renormalize, int32_t* ids, double* weights) {
    if (T < 1 || E < 1 || topk < 1 || topk > E) return -2;
    std::vector<double> sig(E), score(E);
    std::vector<char> taken(E);
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            sig[e] = 1.0 / (1.0 + std::exp(-logits[static_cast<size_t>(t) * E + e]));
            score[e] = sig[e] + (bias ? bias[e] : 0.0);
            taken[e] = 0;
        }
        double sum = 0.0;
        for (int k = 0; k < topk; ++k) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || score[e] > score[best])) best = e;   // first max wins
            taken[best] = 1;
            ids[static_cast<size_t>(t) * topk + k] = best;
            weights[static_cast<size_t>(t) * topk + k] = sig[best];
            sum += sig[best];
        }
        for (int k = 0; k < topk; ++k) {
            double& w = weights[static_cast<size_t>(t) * topk + k];
            if (renormalize) w /= sum;
            w *= routed_scale;
        }
    }
    return 0;
}

// Shared expert in double: out[t] = Wd . (silu(min(Wg.x, L)) * clamp(Wu.x, -L, L)), bf16 weights
// and x decoded exactly, no intermediate rounding ("spark_model layers/glm5next_mlp/forward.rs",
// `forward_moe`: `forward_dense` on the shared weights).
int oracle_shared_expert(const uint16_t* x, int T, int H, int S, const uint16_t* wg, const uint16_t* wu,
                         const uint16_t* wd, double limit, double* out, int nthreads) {
    if (T < 1 || H < 1 || S < 1 || !(limit > 0.0)) return -2;
    std::vector<double> act(static_cast<size_t>(T) * S);
    parallel_for(static_cast<int64_t>(T) * S, resolve_threads(nthreads), [&](int64_t idx) {
        const int64_t t = idx / S, n = idx % S;
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            const double xv = bf16_value(x[t * H + h]);
            g += xv * bf16_value(wg[n * H + h]);
            u += xv * bf16_value(wu[n * H + h]);
        }
        act[idx] = clamped_swiglu(g, u, limit);
    });
    parallel_for(static_cast<int64_t>(T) * H, resolve_threads(nthreads), [&](int64_t idx) {
        const int64_t t = idx / H, j = idx % H;
        double s = 0.0;
        for (int n = 0; n < S; ++n) s += act[t * S + n] * bf16_value(wd[j * S + n]);
        out[idx] = s;
    });
    return 0;
}

// The layer epilogue: out = bf16(routed + shared + residual), exact sum then one rounding
// (forward.rs `forward_moe`: shared output added in the routed combine; the Step gate's
// final add order routed-plus-shared-then-residual). shared / residual: bf16 bits, nullable.
int oracle_layer_epilogue(const double* routed, const uint16_t* shared, const uint16_t* residual, int64_t n,
                          double* out_f64, uint16_t* out_bf16) {
    for (int64_t i = 0; i < n; ++i) {
        double s = routed[i];
        if (shared) s += bf16_value(shared[i]);
        if (residual) s += bf16_value(residual[i]);
        if (out_f64) out_f64[i] = s;
        if (out_bf16) out_bf16[i] = bf16_round(s);
    }
    return 0;
}

int oracle_hardware_threads(void) { return resolve_threads(0); }

}  // extern "C"
