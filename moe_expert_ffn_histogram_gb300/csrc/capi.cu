// C ABI of libmoe_ffn_gb300 (declared in include/moe_ffn.h): synchronous argument checks,
// workspace carving, tier selection and the kernel launches. No allocation, no host sync.
//
// Tiers ("spark_model layers/glm5next_mlp/forward.rs", `gemm` / `forward_moe` tier policy:
// M = 1 decode -> GEMV, M = 2..8 verify -> one weight sweep per union expert), chosen by
// measurement on GB300:
//   T == 1      : gate_up kernel (group = slot) -> down_combine kernel, the latter launched as a
//                 programmatic dependent that starts its weight stream while gate_up drains.
//   2 <= T <= 8 : one fused cooperative launch (fused.cu): in-kernel expert grouping, gate/up +
//                 SwiGLU, grid barrier, down + slot-order combine (after a 4-byte barrier memset).
//   T >= 9 (the measured crossover, kGroupedMinRows*): grouped GEMMs over expert-sorted rows on
//                 the tcgen05 tensor cores (prefill.cu). Shapes the grouped tier does not cover
//                 (NVFP4 with H or I not a multiple of 256; H or I above 8192; E above 4096) run as
//                 even row groups of <= 8 tokens ("forward.rs", `moe_row_groups`), each through
//                 the cooperative kernel.
// The stage entry points (moe_plan, moe_*_gate_up, moe_*_down_combine) run the same work items
// as separate kernels and give the same bits.
#include <cmath>
#include <cstdint>

#include "../../include/moe_ffn.h"
#include "kernels.cuh"
#include "stage_timing.cuh"


using namespace moe;

#ifndef MOE_FORWARD_FUSED
#define MOE_FORWARD_FUSED 1
#endif
#ifndef MOE_FP4_TOKEN
#define MOE_FP4_TOKEN 1
#endif
#ifndef MOE_FORCE_FUSED
#define MOE_FORCE_FUSED 0
#endif

namespace {

constexpr int kMaxRowsPerSweep = 8;
constexpr size_t kMaxSmem = 227 * 1024;

bool shape_ok(int T, int H, int I, int E, int topk) {
    return T >= 1 && topk >= 1 && topk <= kMaxTopk && H >= 128 && I >= 128 && H % 128 == 0 &&
           I % 128 == 0 && E >= 1;
}

int rows_per_sweep(int T) { return T < kMaxRowsPerSweep ? T : kMaxRowsPerSweep; }

// The grouped-GEMM (prefill) tier: more than one 8-token sweep, and shapes its tiles cover
// (per-K-block scale tables of <= 64 entries). Smallest T the grouped-GEMM tier takes; below it,
// sweeps of <= 8 tokens through the cooperative kernel. Measured on GB300 with the decode banks
// (uniform routes over 256 / 160 experts, L2 flushed): the grouped tier wins from the first width
// past one sweep - FP8 T = 9: 0.549 vs 0.561 ms, T = 24: 1.16 vs 1.38 ms; NVFP4 T = 9: 0.32 vs
// 0.38 ms, T = 16: 0.46 vs 0.58 ms - so every T > 8 that it covers goes to it.
#ifndef MOE_PREFILL_MIN_T
#define MOE_PREFILL_MIN_T 0
#endif
constexpr int kGroupedMinRowsFp8 = 9, kGroupedMinRowsFp4 = 9;

bool uses_prefill(int T, int H, int I, int E, int fmt) {
    const int min_t = MOE_PREFILL_MIN_T > 0 ? MOE_PREFILL_MIN_T : (fmt == 0 ? kGroupedMinRowsFp8 : kGroupedMinRowsFp4);
    // NVFP4 also needs K % 256 == 0 (16-byte loads of 4 slices' scale bytes per row)
    return T > kMaxRowsPerSweep && T >= min_t && H <= 8192 && I <= 8192 && E <= kMaxPlanExperts &&
           static_cast<long long>(T) * kMaxTopk < (1LL << 30) &&
           (fmt == 0 || (H % 256 == 0 && I % 256 == 0));
}


// Largest number of columns a group can have for a sub-batch of `rows` tokens.
int group_cap(int rows, int topk) {
    const int p = rows * topk;
    int cap = rows < kMaxCols ? rows : kMaxCols;
    return cap < p ? cap : p;
}

// Columns per group in the fused kernel: its x staging is cap x H f16 of shared memory, and a cap
// of 4 (57 KB at H = 7168) leaves room for two CTAs per SM. An expert picked by more tokens of
// one sweep becomes several groups (its rows are then read once per group) - rare for sweeps of
// <= 8 tokens over many experts.
#ifndef MOE_FUSED_CAP
#define MOE_FUSED_CAP 4
#endif
constexpr int kFusedCap = MOE_FUSED_CAP;
int fused_cap(int rows, int topk) {
    const int c = group_cap(rows, topk);
    return c < kFusedCap ? c : kFusedCap;
}

int check_sizes(int T, int H, int I, int E, int topk) {
    if (!shape_ok(T, H, I, E, topk)) return MOE_ERR_SHAPE;
    const int rows = rows_per_sweep(T);
    if (rows > 1 && E > kMaxPlanExperts) return MOE_ERR_UNSUPPORTED;
    if (rows > 1 && route_plan_smem_bytes(E) > kMaxSmem) return MOE_ERR_UNSUPPORTED;
    const int cap = rows == 1 ? 1 : group_cap(rows, topk);
    if (gate_up_smem_bytes(H, cap) > kMaxSmem) return MOE_ERR_UNSUPPORTED;
    if (down_smem_bytes(rows, topk) > kMaxSmem) return MOE_ERR_UNSUPPORTED;
    if (fused_smem_bytes(H, rows, topk, rows == 1 ? 1 : fused_cap(rows, topk)) > kMaxSmem)
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

struct Ws {
    WsLayout L;
    uint8_t* base;
    template <class P> P* at(size_t off) const { return reinterpret_cast<P*>(base + off); }
};

// fmt: 0 FP8, 1 NVFP4 (whose layout has room for the single-token kernels' activation scales)
int check_ws(void* ws, size_t bytes, int rows, int I, int E, int topk, int fmt, Ws& out) {
    if (ws == nullptr) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return MOE_ERR_WORKSPACE;
    out.L = ws_layout(rows, I, E, topk, fmt == 1 ? kFp4TokFeat : kFeatBlock);
    out.base = static_cast<uint8_t*>(ws);
    if (bytes < out.L.total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

Groups groups_for(const Ws& w, const int32_t* ids, int rows, int topk, int E) {
    Groups g{};
    g.ids = ids;
    g.topk = topk;
    g.E = E;
    if (rows > 1) {
        g.count = w.at<int32_t>(w.L.group_count);
        g.expert = w.at<int32_t>(w.L.group_expert);
        g.start = w.at<int32_t>(w.L.group_start);
        g.ncols = w.at<int32_t>(w.L.group_ncols);
        g.sorted_pair = w.at<int32_t>(w.L.sorted_pair);
    }
    return g;
}

int cuda_status(cudaError_t st) { return st == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ---- the three stages for one sub-batch of rows <= 8 tokens --------------------------------

int stage_plan(int rows, int E, int topk, const int32_t* ids, const Ws& w, int32_t* err,
               cudaStream_t s) {
    if (rows <= 1) return MOE_OK;
    return cuda_status(launch_route_plan(
        ids, rows * topk, E, group_cap(rows, topk), w.at<int32_t>(w.L.counts),
        w.at<int32_t>(w.L.offsets), w.at<int32_t>(w.L.sorted_pair),
        w.at<int32_t>(w.L.pair_to_sorted), w.at<int32_t>(w.L.group_count),
        w.at<int32_t>(w.L.group_expert), w.at<int32_t>(w.L.group_start),
        w.at<int32_t>(w.L.group_ncols), err, s));
}

// NVFP4 with one scale_2 per expert and projection: expert e's gate value is g[e * stride]
// (all null: the projections' scalars)
struct ExpertScale2 {
    const float* g = nullptr;
    const float* u = nullptr;
    const float* d = nullptr;
    int stride = 1;
};

template <int FMT>
int stage_gate_up(const uint16_t* x, int rows, int H, int I, int E, int topk, const int32_t* ids,
                  const uint8_t* wg, const float* sg, const uint8_t* sfg, float s2g,
                  const uint8_t* wu, const float* su, const uint8_t* sfu, float s2u, float limit,
                  const Ws& w, int32_t* err, cudaStream_t s, const uint8_t* wd = nullptr,
                  const uint8_t* sfd = nullptr, const ExpertScale2& xs2 = {}) {
    GateUpArgs a{};
    a.x = reinterpret_cast<const __nv_bfloat16*>(x);
    a.H = H;
    a.I = I;
    a.wg = wg;
    a.wu = wu;
    a.sg = sg;
    a.su = su;
    a.sfg = sfg;
    a.sfu = sfu;
    a.s2g = s2g;
    a.s2u = s2u;
    a.s2g_e = xs2.g;
    a.s2u_e = xs2.u;
    a.s2_stride = xs2.stride;
    a.limit = limit;
    a.grp = groups_for(w, ids, rows, topk, E);
    a.act = w.at<__half>(w.L.act);
    a.act_scale = w.at<float>(w.L.act_scale);
    a.err = err;
    if (MOE_FP4_TOKEN && FMT == 1 && rows == 1)   // one NVFP4 token: the lean single-token kernel
        return cuda_status(launch_fp4_token_gate_up(a, topk, s));
    const int ngroups = rows * topk;     // implicit: topk slots; table: at most one per pair
    const int cap = rows == 1 ? 1 : group_cap(rows, topk);
    // NVFP4, one token: prefetch the call's whole weight set into L2 when it fits (<= 96 MB,
    // under the 129 MB L2 with room for the rest)
    if (MOE_FP4_L2_PREFETCH && FMT == 1 && rows == 1 && wd != nullptr && sfd != nullptr) {
        const double per_expert = 3.0 * I * (H / 2.0 + H / 16.0);
        if (per_expert * topk <= 96.0 * (1 << 20)) {
            a.l2_prefetch = 1;
            a.pf_wd = wd;
            a.pf_sfd = sfd;
        }
    }
    return cuda_status(launch_gate_up<FMT>(a, ngroups, cap, s));
}

template <int FMT>
int stage_down(int rows, int H, int I, int E, int topk, const int32_t* ids, const float* wts,
               const uint8_t* wd, const float* sd, const uint8_t* sfd, float s2d, uint16_t* out,
               const Ws& w, cudaStream_t s, const uint16_t* shared = nullptr,
               const uint16_t* residual = nullptr, const ExpertScale2& xs2 = {}) {
    DownArgs a{};
    a.T = rows;
    a.H = H;
    a.I = I;
    a.topk = topk;
    a.E = E;
    a.ids = ids;
    a.wts = wts;
    a.wd = wd;
    a.sd = sd;
    a.sfd = sfd;
    a.s2d = s2d;
    a.s2d_e = xs2.d;
    a.s2_stride = xs2.stride;
    a.grp = groups_for(w, ids, rows, topk, E);
    a.act = w.at<__half>(w.L.act);
    a.act_scale = w.at<float>(w.L.act_scale);
    a.out = reinterpret_cast<__nv_bfloat16*>(out);
    a.shared = reinterpret_cast<const __nv_bfloat16*>(shared);
    a.residual = reinterpret_cast<const __nv_bfloat16*>(residual);
    if (MOE_FP4_TOKEN && FMT == 1 && rows == 1)
        return cuda_status(launch_fp4_token_down(a, MOE_PDL != 0, s));
    return cuda_status(launch_down_combine<FMT>(a, s));
}

// The whole forward of one sub-batch as one fused cooperative launch (grouping done in-kernel).
template <int FMT>
int stage_fused(const uint16_t* x, int rows, int H, int I, int E, int topk, const int32_t* ids,
                const float* wts, const uint8_t* wg, const float* sg, const uint8_t* sfg, float s2g,
                const uint8_t* wu, const float* su, const uint8_t* sfu, float s2u,
                const uint8_t* wd, const float* sd, const uint8_t* sfd, float s2d, float limit,
                uint16_t* out, const Ws& w, int32_t* err, cudaStream_t s,
                const uint16_t* shared = nullptr, const uint16_t* residual = nullptr,
                const ExpertScale2& xs2 = {}) {
    Groups grp{};
    grp.ids = ids;
    grp.topk = topk;
    grp.E = E;
    GateUpArgs ga{};
    ga.x = reinterpret_cast<const __nv_bfloat16*>(x);
    ga.H = H;
    ga.I = I;
    ga.wg = wg;
    ga.wu = wu;
    ga.sg = sg;
    ga.su = su;
    ga.sfg = sfg;
    ga.sfu = sfu;
    ga.s2g = s2g;
    ga.s2u = s2u;
    ga.s2g_e = xs2.g;
    ga.s2u_e = xs2.u;
    ga.s2_stride = xs2.stride;
    ga.limit = limit;
    ga.grp = grp;
    ga.act = w.at<__half>(w.L.act);
    ga.act_scale = w.at<float>(w.L.act_scale);
    ga.err = err;
    DownArgs da{};
    da.T = rows;
    da.H = H;
    da.I = I;
    da.topk = topk;
    da.E = E;
    da.ids = ids;
    da.wts = wts;
    da.wd = wd;
    da.sd = sd;
    da.sfd = sfd;
    da.s2d = s2d;
    da.s2d_e = xs2.d;
    da.s2_stride = xs2.stride;
    da.grp = grp;
    da.act = ga.act;
    da.act_scale = ga.act_scale;
    da.out = reinterpret_cast<__nv_bfloat16*>(out);
    da.shared = reinterpret_cast<const __nv_bfloat16*>(shared);
    da.residual = reinterpret_cast<const __nv_bfloat16*>(residual);
    const int cap = rows == 1 ? 1 : fused_cap(rows, topk);
    return cuda_status(launch_fused_forward<FMT>(ga, da, w.at<unsigned>(w.L.barrier), rows, cap, s));
}

struct Proj {
    const uint8_t* w;
    const float* s;       // FP8
    const uint8_t* sf;    // NVFP4
    float s2;
};

template <int FMT>
int forward(const uint16_t* x, int T, int H, int I, int E, int topk, const int32_t* ids,
            const float* wts, Proj pg, Proj pu, Proj pd, float limit, uint16_t* out, void* ws,
            size_t ws_bytes, int32_t* err, cudaStream_t s, const uint16_t* shared = nullptr,
            const uint16_t* residual = nullptr, const ExpertScale2& xs2 = {}) {
    int rc = check_sizes(T, H, I, E, topk);
    if (rc) return rc;
    StageScope timing(s, FMT == 0 ? "moe_fp8_forward" : "moe_nvfp4_forward");
    if (uses_prefill(T, H, I, E, FMT)) {
        if (ws == nullptr || reinterpret_cast<uintptr_t>(ws) % 256 != 0) return MOE_ERR_WORKSPACE;
        const PrefillLayout L = prefill_layout(T, H, I, E, topk);
        if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
        PrefillWeights wt{pg.w,  pu.w,  pd.w,  pg.s, pu.s, pd.s, pg.sf, pu.sf, pd.sf, pg.s2, pu.s2, pd.s2,
                          xs2.g, xs2.u, xs2.d, xs2.stride};
        return cuda_status(launch_prefill(FMT, reinterpret_cast<const __nv_bfloat16*>(x), T, H, I, E, topk,
                                          ids, wts, wt, limit, reinterpret_cast<__nv_bfloat16*>(out),
                                          static_cast<uint8_t*>(ws), L, err, s,
                                          reinterpret_cast<const __nv_bfloat16*>(shared),
                                          reinterpret_cast<const __nv_bfloat16*>(residual)));
    }
    const int rows_max = rows_per_sweep(T);
    Ws w;
    if ((rc = check_ws(ws, ws_bytes, rows_max, I, E, topk, FMT, w))) return rc;
    // even split into ceil(T/8) groups, never a trailing group of one ("forward.rs",
    // `moe_row_groups`); the workspace is rebuilt per group, in stream order.
    const int ngroups = (T + kMaxRowsPerSweep - 1) / kMaxRowsPerSweep;
    int start = 0;
    for (int i = 0; i < ngroups; ++i) {
        const int rows = (T - start + (ngroups - i) - 1) / (ngroups - i);
        const int32_t* ids_g = ids + static_cast<size_t>(start) * topk;
        const float* wts_g = wts + static_cast<size_t>(start) * topk;
        const uint16_t* x_g = x + static_cast<size_t>(start) * H;
        uint16_t* out_g = out + static_cast<size_t>(start) * H;
        const uint16_t* sh_g = shared ? shared + static_cast<size_t>(start) * H : nullptr;
        const uint16_t* rs_g = residual ? residual + static_cast<size_t>(start) * H : nullptr;
        if (MOE_FORWARD_FUSED && (rows > 1 || MOE_FORCE_FUSED)) {
            stage_mark(s, "fused");
            if ((rc = stage_fused<FMT>(x_g, rows, H, I, E, topk, ids_g, wts_g, pg.w, pg.s, pg.sf,
                                       pg.s2, pu.w, pu.s, pu.sf, pu.s2, pd.w, pd.s, pd.sf, pd.s2,
                                       limit, out_g, w, err, s, sh_g, rs_g, xs2)))
                return rc;
        } else {
            stage_mark(s, "plan");
            if ((rc = stage_plan(rows, E, topk, ids_g, w, err, s))) return rc;
            stage_mark(s, "gate_up");
            if ((rc = stage_gate_up<FMT>(x_g, rows, H, I, E, topk, ids_g, pg.w, pg.s, pg.sf, pg.s2,
                                         pu.w, pu.s, pu.sf, pu.s2, limit, w, err, s, pd.w, pd.sf, xs2)))
                return rc;
            stage_mark(s, "down_combine");
            if ((rc = stage_down<FMT>(rows, H, I, E, topk, ids_g, wts_g, pd.w, pd.s, pd.sf, pd.s2,
                                      out_g, w, s, sh_g, rs_g, xs2)))
                return rc;
        }
        start += rows;
    }
    return MOE_OK;
}

bool limit_ok(float limit) { return !std::isnan(limit) && limit > 0.0f; }

// The kernels read weights and activations with 16-byte (FP8) / 8-byte (NVFP4) vector loads.
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
template <class... P>
bool all_aligned(const P*... p) { return (aligned16(p) && ...); }

// The per-expert scale_2 tables: present, 4-byte aligned, a stride of at least one element.
int check_expert_scale2(const ExpertScale2& t) {
    if (!t.g || !t.u || !t.d) return MOE_ERR_NULL;
    if (t.stride < 1) return MOE_ERR_VALUE;
    if ((reinterpret_cast<uintptr_t>(t.g) | reinterpret_cast<uintptr_t>(t.u) | reinterpret_cast<uintptr_t>(t.d)) & 3u)
        return MOE_ERR_ALIGN;
    return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(int T, int H, int I, int E, int topk, int fmt) {
    if (fmt != MOE_FMT_FP8_E4M3_B128 && fmt != MOE_FMT_NVFP4) return 0;
    if (check_sizes(T, H, I, E, topk) != MOE_OK) return 0;
    if (uses_prefill(T, H, I, E, fmt == MOE_FMT_FP8_E4M3_B128 ? 0 : 1))
        return prefill_layout(T, H, I, E, topk).total;
    return ws_layout(rows_per_sweep(T), I, E, topk, fmt == MOE_FMT_NVFP4 ? kFp4TokFeat : kFeatBlock).total;
}

int moe_route_permute(const int32_t* topk_ids, int T, int topk, int E, int32_t* counts,
                      int32_t* offsets, int32_t* sorted_pair, int32_t* pair_to_sorted,
                      int32_t* err, void* stream) {
    if (!topk_ids || !counts || !offsets || !sorted_pair || !pair_to_sorted) return MOE_ERR_NULL;
    if (T < 1 || topk < 1 || E < 1) return MOE_ERR_SHAPE;
    if (E > kMaxPlanExperts || route_plan_smem_bytes(E) > kMaxSmem) return MOE_ERR_UNSUPPORTED;
    const long long P = static_cast<long long>(T) * topk;
    if (P > (1LL << 30)) return MOE_ERR_SHAPE;
    return cuda_status(launch_route_plan(topk_ids, static_cast<int>(P), E, 1, counts, offsets,
                                         sorted_pair, pair_to_sorted, nullptr, nullptr, nullptr,
                                         nullptr, err, static_cast<cudaStream_t>(stream)));
}

int moe_fp8_forward(const uint16_t* x, int T, int H, int I, int E, int topk,
                    const int32_t* topk_ids, const float* topk_weights, const uint8_t* w_gate,
                    const float* s_gate, const uint8_t* w_up, const float* s_up,
                    const uint8_t* w_down, const float* s_down, float limit, uint16_t* out,
                    void* workspace, size_t workspace_bytes, int32_t* err, void* stream) {
    if (!x || !topk_ids || !topk_weights || !w_gate || !s_gate || !w_up || !s_up || !w_down ||
        !s_down || !out)
        return MOE_ERR_NULL;
    if (!limit_ok(limit)) return MOE_ERR_VALUE;
    if (!all_aligned(x, w_gate, w_up, w_down, out)) return MOE_ERR_ALIGN;
    return forward<0>(x, T, H, I, E, topk, topk_ids, topk_weights, Proj{w_gate, s_gate, nullptr, 1.f},
                      Proj{w_up, s_up, nullptr, 1.f}, Proj{w_down, s_down, nullptr, 1.f}, limit,
                      out, workspace, workspace_bytes, err, static_cast<cudaStream_t>(stream));
}

int moe_nvfp4_forward(const uint16_t* x, int T, int H, int I, int E, int topk,
                      const int32_t* topk_ids, const float* topk_weights, const uint8_t* w_gate,
                      const uint8_t* sf_gate, float scale2_gate, const uint8_t* w_up,
                      const uint8_t* sf_up, float scale2_up, const uint8_t* w_down,
                      const uint8_t* sf_down, float scale2_down, float limit, uint16_t* out,
                      void* workspace, size_t workspace_bytes, int32_t* err, void* stream) {
    if (!x || !topk_ids || !topk_weights || !w_gate || !sf_gate || !w_up || !sf_up || !w_down ||
        !sf_down || !out)
        return MOE_ERR_NULL;
    if (!limit_ok(limit)) return MOE_ERR_VALUE;
    if (!std::isfinite(scale2_gate) || !std::isfinite(scale2_up) || !std::isfinite(scale2_down))
        return MOE_ERR_VALUE;
    if (!all_aligned(x, w_gate, w_up, w_down, sf_gate, sf_up, sf_down, out)) return MOE_ERR_ALIGN;
    return forward<1>(x, T, H, I, E, topk, topk_ids, topk_weights,
                      Proj{w_gate, nullptr, sf_gate, scale2_gate},
                      Proj{w_up, nullptr, sf_up, scale2_up},
                      Proj{w_down, nullptr, sf_down, scale2_down}, limit, out, workspace,
                      workspace_bytes, err, static_cast<cudaStream_t>(stream));
}

int moe_nvfp4_forward_expert_scale2(const uint16_t* x, int T, int H, int I, int E, int topk,
                                    const int32_t* topk_ids, const float* topk_weights,
                                    const uint8_t* w_gate, const uint8_t* sf_gate, const float* scale2_gate,
                                    const uint8_t* w_up, const uint8_t* sf_up, const float* scale2_up,
                                    const uint8_t* w_down, const uint8_t* sf_down, const float* scale2_down,
                                    int scale2_stride, float limit, uint16_t* out, void* workspace,
                                    size_t workspace_bytes, int32_t* err, void* stream) {
    if (!x || !topk_ids || !topk_weights || !w_gate || !sf_gate || !w_up || !sf_up || !w_down ||
        !sf_down || !out)
        return MOE_ERR_NULL;
    if (!limit_ok(limit)) return MOE_ERR_VALUE;
    if (!all_aligned(x, w_gate, w_up, w_down, sf_gate, sf_up, sf_down, out)) return MOE_ERR_ALIGN;
    const ExpertScale2 xs2{scale2_gate, scale2_up, scale2_down, scale2_stride};
    if (const int rc = check_expert_scale2(xs2)) return rc;
    return forward<1>(x, T, H, I, E, topk, topk_ids, topk_weights, Proj{w_gate, nullptr, sf_gate, 1.f},
                      Proj{w_up, nullptr, sf_up, 1.f}, Proj{w_down, nullptr, sf_down, 1.f}, limit, out,
                      workspace, workspace_bytes, err, static_cast<cudaStream_t>(stream), nullptr, nullptr, xs2);
}

// ---- the forwards with the layer epilogue ---------------------------------------------------

int moe_fp8_forward_layer(const uint16_t* x, int T, int H, int I, int E, int topk,
                          const int32_t* topk_ids, const float* topk_weights, const uint8_t* w_gate,
                          const float* s_gate, const uint8_t* w_up, const float* s_up,
                          const uint8_t* w_down, const float* s_down, float limit,
                          const uint16_t* shared, const uint16_t* residual, uint16_t* out,
                          void* workspace, size_t workspace_bytes, int32_t* err, void* stream) {
    if (!x || !topk_ids || !topk_weights || !w_gate || !s_gate || !w_up || !s_up || !w_down ||
        !s_down || !out)
        return MOE_ERR_NULL;
    if (!limit_ok(limit)) return MOE_ERR_VALUE;
    if (!all_aligned(x, w_gate, w_up, w_down, out)) return MOE_ERR_ALIGN;
    if ((shared && !aligned16(shared)) || (residual && !aligned16(residual))) return MOE_ERR_ALIGN;
    return forward<0>(x, T, H, I, E, topk, topk_ids, topk_weights, Proj{w_gate, s_gate, nullptr, 1.f},
                      Proj{w_up, s_up, nullptr, 1.f}, Proj{w_down, s_down, nullptr, 1.f}, limit,
                      out, workspace, workspace_bytes, err, static_cast<cudaStream_t>(stream), shared,
                      residual);
}

int moe_nvfp4_forward_layer(const uint16_t* x, int T, int H, int I, int E, int topk,
                            const int32_t* topk_ids, const float* topk_weights, const uint8_t* w_gate,
                            const uint8_t* sf_gate, float scale2_gate, const uint8_t* w_up,
                            const uint8_t* sf_up, float scale2_up, const uint8_t* w_down,
                            const uint8_t* sf_down, float scale2_down, float limit,
                            const uint16_t* shared, const uint16_t* residual, uint16_t* out,
                            void* workspace, size_t workspace_bytes, int32_t* err, void* stream) {
    if (!x || !topk_ids || !topk_weights || !w_gate || !sf_gate || !w_up || !sf_up || !w_down ||
        !sf_down || !out)
        return MOE_ERR_NULL;
    if (!limit_ok(limit)) return MOE_ERR_VALUE;
    if (!std::isfinite(scale2_gate) || !std::isfinite(scale2_up) || !std::isfinite(scale2_down))
        return MOE_ERR_VALUE;
    if (!all_aligned(x, w_gate, w_up, w_down, sf_gate, sf_up, sf_down, out)) return MOE_ERR_ALIGN;
    if ((shared && !aligned16(shared)) || (residual && !aligned16(residual))) return MOE_ERR_ALIGN;
    return forward<1>(x, T, H, I, E, topk, topk_ids, topk_weights,
                      Proj{w_gate, nullptr, sf_gate, scale2_gate},
                      Proj{w_up, nullptr, sf_up, scale2_up},
                      Proj{w_down, nullptr, sf_down, scale2_down}, limit, out, workspace,
                      workspace_bytes, err, static_cast<cudaStream_t>(stream), shared, residual);
}

int moe_nvfp4_forward_layer_expert_scale2(const uint16_t* x, int T, int H, int I, int E, int topk,
                                          const int32_t* topk_ids, const float* topk_weights,
                                          const uint8_t* w_gate, const uint8_t* sf_gate, const float* scale2_gate,
                                          const uint8_t* w_up, const uint8_t* sf_up, const float* scale2_up,
                                          const uint8_t* w_down, const uint8_t* sf_down, const float* scale2_down,
                                          int scale2_stride, float limit, const uint16_t* shared,
                                          const uint16_t* residual, uint16_t* out, void* workspace,
                                          size_t workspace_bytes, int32_t* err, void* stream) {
    if (!x || !topk_ids || !topk_weights || !w_gate || !sf_gate || !w_up || !sf_up || !w_down ||
        !sf_down || !out)
        return MOE_ERR_NULL;
    if (!limit_ok(limit)) return MOE_ERR_VALUE;
    if (!all_aligned(x, w_gate, w_up, w_down, sf_gate, sf_up, sf_down, out)) return MOE_ERR_ALIGN;
    if ((shared && !aligned16(shared)) || (residual && !aligned16(residual))) return MOE_ERR_ALIGN;
    const ExpertScale2 xs2{scale2_gate, scale2_up, scale2_down, scale2_stride};
    if (const int rc = check_expert_scale2(xs2)) return rc;
    return forward<1>(x, T, H, I, E, topk, topk_ids, topk_weights, Proj{w_gate, nullptr, sf_gate, 1.f},
                      Proj{w_up, nullptr, sf_up, 1.f}, Proj{w_down, nullptr, sf_down, 1.f}, limit, out,
                      workspace, workspace_bytes, err, static_cast<cudaStream_t>(stream), shared, residual, xs2);
}

// ---- stage entry points (T <= 8: one sweep) -------------------------------------------------

int moe_plan(int T, int H, int I, int E, int topk, int fmt, const int32_t* topk_ids,
             void* workspace, size_t workspace_bytes, int32_t* err, void* stream) {
    if (!topk_ids) return MOE_ERR_NULL;
    if (fmt != MOE_FMT_FP8_E4M3_B128 && fmt != MOE_FMT_NVFP4) return MOE_ERR_VALUE;
    int rc = check_sizes(T, H, I, E, topk);
    if (rc) return rc;
    if (T > kMaxRowsPerSweep) return MOE_ERR_UNSUPPORTED;
    Ws w;
    if ((rc = check_ws(workspace, workspace_bytes, T, I, E, topk, fmt == MOE_FMT_NVFP4 ? 1 : 0, w))) return rc;
    return stage_plan(T, E, topk, topk_ids, w, err, static_cast<cudaStream_t>(stream));
}

int moe_fp8_gate_up(const uint16_t* x, int T, int H, int I, int E, int topk,
                    const int32_t* topk_ids, const uint8_t* w_gate, const float* s_gate,
                    const uint8_t* w_up, const float* s_up, float limit, void* workspace,
                    size_t workspace_bytes, int32_t* err, void* stream) {
    if (!x || !topk_ids || !w_gate || !s_gate || !w_up || !s_up) return MOE_ERR_NULL;
    if (!limit_ok(limit)) return MOE_ERR_VALUE;
    if (!all_aligned(x, w_gate, w_up)) return MOE_ERR_ALIGN;
    int rc = check_sizes(T, H, I, E, topk);
    if (rc) return rc;
    if (T > kMaxRowsPerSweep) return MOE_ERR_UNSUPPORTED;
    Ws w;
    if ((rc = check_ws(workspace, workspace_bytes, T, I, E, topk, 0, w))) return rc;
    return stage_gate_up<0>(x, T, H, I, E, topk, topk_ids, w_gate, s_gate, nullptr, 1.f, w_up,
                            s_up, nullptr, 1.f, limit, w, err, static_cast<cudaStream_t>(stream));
}

int moe_fp8_down_combine(int T, int H, int I, int E, int topk, const int32_t* topk_ids,
                         const float* topk_weights, const uint8_t* w_down, const float* s_down,
                         uint16_t* out, void* workspace, size_t workspace_bytes, void* stream) {
    if (!topk_ids || !topk_weights || !w_down || !s_down || !out) return MOE_ERR_NULL;
    if (!all_aligned(w_down, out)) return MOE_ERR_ALIGN;
    int rc = check_sizes(T, H, I, E, topk);
    if (rc) return rc;
    if (T > kMaxRowsPerSweep) return MOE_ERR_UNSUPPORTED;
    Ws w;
    if ((rc = check_ws(workspace, workspace_bytes, T, I, E, topk, 0, w))) return rc;
    return stage_down<0>(T, H, I, E, topk, topk_ids, topk_weights, w_down, s_down, nullptr, 1.f,
                         out, w, static_cast<cudaStream_t>(stream));
}

int moe_nvfp4_gate_up(const uint16_t* x, int T, int H, int I, int E, int topk,
                      const int32_t* topk_ids, const uint8_t* w_gate, const uint8_t* sf_gate,
                      float scale2_gate, const uint8_t* w_up, const uint8_t* sf_up,
                      float scale2_up, float limit, void* workspace, size_t workspace_bytes,
                      int32_t* err, void* stream) {
    if (!x || !topk_ids || !w_gate || !sf_gate || !w_up || !sf_up) return MOE_ERR_NULL;
    if (!limit_ok(limit)) return MOE_ERR_VALUE;
    if (!std::isfinite(scale2_gate) || !std::isfinite(scale2_up)) return MOE_ERR_VALUE;
    if (!all_aligned(x, w_gate, w_up, sf_gate, sf_up)) return MOE_ERR_ALIGN;
    int rc = check_sizes(T, H, I, E, topk);
    if (rc) return rc;
    if (T > kMaxRowsPerSweep) return MOE_ERR_UNSUPPORTED;
    Ws w;
    if ((rc = check_ws(workspace, workspace_bytes, T, I, E, topk, 1, w))) return rc;
    return stage_gate_up<1>(x, T, H, I, E, topk, topk_ids, w_gate, nullptr, sf_gate, scale2_gate,
                            w_up, nullptr, sf_up, scale2_up, limit, w, err,
                            static_cast<cudaStream_t>(stream));
}

int moe_nvfp4_down_combine(int T, int H, int I, int E, int topk, const int32_t* topk_ids,
                           const float* topk_weights, const uint8_t* w_down,
                           const uint8_t* sf_down, float scale2_down, uint16_t* out,
                           void* workspace, size_t workspace_bytes, void* stream) {
    if (!topk_ids || !topk_weights || !w_down || !sf_down || !out) return MOE_ERR_NULL;
    if (!std::isfinite(scale2_down)) return MOE_ERR_VALUE;
    if (!all_aligned(w_down, sf_down, out)) return MOE_ERR_ALIGN;
    int rc = check_sizes(T, H, I, E, topk);
    if (rc) return rc;
    if (T > kMaxRowsPerSweep) return MOE_ERR_UNSUPPORTED;
    Ws w;
    if ((rc = check_ws(workspace, workspace_bytes, T, I, E, topk, 1, w))) return rc;
    return stage_down<1>(T, H, I, E, topk, topk_ids, topk_weights, w_down, nullptr, sf_down,
                         scale2_down, out, w, static_cast<cudaStream_t>(stream));
}

// ---- router ---------------------------------------------------------------------------------

namespace {
bool router_shape_ok(int T, int H, int E) {
    return T >= 1 && H >= 32 && H % 32 == 0 && E >= 16 && E <= 1024 && E % 16 == 0;
}
int device_sms(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}
}  // namespace

size_t moe_router_workspace_bytes(int T, int H, int E) {
    if (!router_shape_ok(T, H, E)) return 0;
    int sms = 0;
    if (device_sms(&sms) != MOE_OK) sms = 152;
    const int ks = router_ksplit(T, H, E, sms);
    return align_up(static_cast<size_t>(ks) * T * E * sizeof(float), 256);
}

int moe_router(const uint16_t* x, int T, int H, const uint16_t* router_w, const float* bias, int E, int topk,
               float routed_scale, int renormalize, float* logits, int32_t* topk_ids, float* topk_weights,
               void* workspace, size_t workspace_bytes, void* stream) {
    if (!x || !router_w || !topk_ids || !topk_weights) return MOE_ERR_NULL;
    if (!router_shape_ok(T, H, E) || topk < 1 || topk > kMaxTopk || topk > E) return MOE_ERR_SHAPE;
    if (!std::isfinite(routed_scale) || !(routed_scale > 0.0f)) return MOE_ERR_VALUE;
    if (!all_aligned(x, router_w)) return MOE_ERR_ALIGN;
    if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MOE_ERR_WORKSPACE;
    int sms = 0;
    int rc = device_sms(&sms);
    if (rc) return rc;
    const int ks = router_ksplit(T, H, E, sms);
    if (workspace_bytes < static_cast<size_t>(ks) * T * E * sizeof(float)) return MOE_ERR_WORKSPACE;
    if (router_topk_smem_bytes(E) > kMaxSmem) return MOE_ERR_UNSUPPORTED;
    return cuda_status(launch_router(reinterpret_cast<const __nv_bfloat16*>(x), T, H,
                                     reinterpret_cast<const __nv_bfloat16*>(router_w), bias, E, topk, routed_scale,
                                     renormalize != 0, logits, topk_ids, topk_weights, static_cast<float*>(workspace),
                                     ks, static_cast<cudaStream_t>(stream)));
}

// ---- shared expert ----------------------------------------------------------------------------

namespace {
bool shared_shape_ok(int T, int H, int S) {
    return T >= 1 && H >= 32 && S >= 32 && H % 32 == 0 && S % 32 == 0;
}
}  // namespace

size_t moe_shared_expert_workspace_bytes(int T, int H, int S) {
    if (!shared_shape_ok(T, H, S)) return 0;
    int sms = 0;
    if (device_sms(&sms) != MOE_OK) sms = 152;
    return shared_expert_ws_bytes(T, H, S, sms);
}

int moe_shared_expert_bf16(const uint16_t* x, int T, int H, int S, const uint16_t* w_gate,
                           const uint16_t* w_up, const uint16_t* w_down, float limit, uint16_t* out,
                           void* workspace, size_t workspace_bytes, void* stream) {
    if (!x || !w_gate || !w_up || !w_down || !out) return MOE_ERR_NULL;
    if (!shared_shape_ok(T, H, S)) return MOE_ERR_SHAPE;
    if (!limit_ok(limit)) return MOE_ERR_VALUE;
    if (!all_aligned(x, w_gate, w_up, w_down, out)) return MOE_ERR_ALIGN;
    if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MOE_ERR_WORKSPACE;
    int sms = 0;
    int rc = device_sms(&sms);
    if (rc) return rc;
    if (workspace_bytes < shared_expert_ws_bytes(T, H, S, sms)) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_shared_expert(
        reinterpret_cast<const __nv_bfloat16*>(x), T, H, S, reinterpret_cast<const __nv_bfloat16*>(w_gate),
        reinterpret_cast<const __nv_bfloat16*>(w_up), reinterpret_cast<const __nv_bfloat16*>(w_down), limit,
        reinterpret_cast<__nv_bfloat16*>(out), static_cast<uint8_t*>(workspace), sms,
        static_cast<cudaStream_t>(stream)));
}

int moe_stream_read(const void* buf, size_t bytes, uint32_t* sink, void* stream) {
    if (buf == nullptr || sink == nullptr) return MOE_ERR_NULL;
    if (bytes == 0 || bytes % 16 != 0) return MOE_ERR_SHAPE;
    if (!aligned16(buf) || (reinterpret_cast<uintptr_t>(sink) & 3u) != 0) return MOE_ERR_ALIGN;
    int sms = 0;
    if (const int st = device_sms(&sms); st != MOE_OK) return st;
    return cuda_status(launch_stream_read(buf, bytes, sink, sms, static_cast<cudaStream_t>(stream)));
}

int moe_test_barrier_timeout(int enable) {
    set_test_barrier_timeout(enable != 0);
    return MOE_OK;
}

const char* moe_build_arch(void) { return "sm_103a"; }

}  // extern "C"
