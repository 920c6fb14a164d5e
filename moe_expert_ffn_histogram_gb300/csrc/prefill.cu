// Wide (prefill) tier: the routed pairs of a whole batch, sorted by expert, go through two
// grouped GEMMs instead of per-token GEMV sweeps, so each expert's weights are read once per
// 128-row tile of its routed rows rather than once per 8 tokens.
//
// "spark_model layers/glm5next_mlp/forward.rs": `forward_moe` sends rows > 8 (and above a
// measured width floor) to the grouped tensor-core GEMM over expert-sorted rows, one launch per
// projection, with `moe_sort_by_expert` before it and the `_indexed` combine after it (same slot
// order and rounding as the narrow tiers). Here:
//
//   route plan               counts / offsets / sorted_pair / pair_to_sorted (route_plan.cu)
//   prefill_tiles            the m-tile list: (expert, first sorted row) per 128-row tile
//   prefill_x_prep           x (bf16) -> x16 (f16, one power-of-two range scale per token), each
//                            token's row written to its routed pairs' sorted rows
//   gate/up grouped GEMM     per tile of 128 sorted rows x 128 features: gate and up, clamped
//                            SwiGLU in the epilogue -> a (prefill_tw.cu, the TMEM core)
//   prefill_act_prep         a (fp32) -> a16 (f16, one power-of-two range scale per sorted row),
//                            only when no clamp limit bounds a (with one the GEMM writes a16)
//   down grouped GEMM        per tile of 128 sorted rows x 128 output rows: y, stored in f16 times
//                            a power of two per (sorted row, 128-row block) from a bound on |y|
//   prefill_combine          out[t] = sum over slots k in order of w[t,k] * y[pair_to_sorted], bf16
//
// Weights are dequantised by the GEMM's converter warps: E4M3 -> f16 exactly, times the block
// scale pre-multiplied by a power of two chosen per (expert, 128-row weight block) so the product
// stays in f16's normal range (one f16 rounding per weight); the power of two is undone in the
// fp32 epilogue. Products accumulate in fp32.
#include <cmath>

#include "prefill.cuh"
#include "stage_timing.cuh"

namespace moe {


// ---- tile list -----------------------------------------------------------------------------------

// One block: the m-tile list from the per-expert counts (after the single-block route plan; the
// multi-block plan builds it in its middle launch).
__global__ void __launch_bounds__(1024) prefill_tiles_kernel(const int32_t* __restrict__ counts,
                                                             const int32_t* __restrict__ offsets, int E,
                                                             TileList tl) {
    build_tile_list(counts, offsets, E, tl);
}

// ---- x prep ---------------------------------------------------------------------------------------

// One block per token: x16[t] = f16(x[t] * s_t), xinv[t] = 1 / s_t, s_t a power of two. With
// pair_to_sorted given, the row is instead written to each of the token's topk sorted rows of
// x16 (then [P][H]; pairs marked -1 are skipped), so that the gate/up GEMM reads its A tiles as
// plain boxes.
__global__ void __launch_bounds__(256) prefill_x_prep_kernel(const __nv_bfloat16* __restrict__ x,
                                                             int H, __half* __restrict__ x16,
                                                             float* __restrict__ xinv,
                                                             const int32_t* __restrict__ pair_to_sorted,
                                                             int topk) {
    __shared__ float red[8];
    pdl_launch_dependents();                           // the gate/up GEMM may start its setup
    const int t = blockIdx.x, tid = threadIdx.x;
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    const int nv = H / 8;
    float m = 0.0f;
    for (int v = tid; v < nv; v += 256) {
        const uint4 q = __ldg(xr + v);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
            m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
        }
    }
    m = warp_max(m);
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    float mm = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) mm = fmaxf(mm, red[w]);
    float inv;
    const float s = pow2_range_scale(mm, inv);
    pdl_wait();                        // the route plan's pair_to_sorted (programmatic dependent launch)
    if (tid == 0) xinv[t] = inv;
    const int ncopy = pair_to_sorted != nullptr ? topk : 1;
    for (int v = tid; v < nv; v += 256) {
        const uint4 q = __ldg(xr + v);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h2 = __floats2half2_rn(__uint_as_float(w[i] << 16) * s,
                                                 __uint_as_float(w[i] & 0xFFFF0000u) * s);
            o[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        for (int c = 0; c < ncopy; ++c) {
            const int row = pair_to_sorted != nullptr ? pair_to_sorted[static_cast<size_t>(t) * topk + c] : t;
            if (row < 0) continue;                            // pair with an out-of-range expert id
            reinterpret_cast<uint4*>(x16 + static_cast<size_t>(row) * H)[v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// ---- activation prep -------------------------------------------------------------------------------

// One block per sorted row: a16[r] = f16(a[r] * s_r), ainv[r] = 1 / s_r, from the row's max |a|
// (kept as the float's bit pattern by the gate/up GEMM's integer atomicMax).
__global__ void __launch_bounds__(256) prefill_act_prep_kernel(const float* __restrict__ a32,
                                                               const uint32_t* __restrict__ amax,
                                                               const int32_t* __restrict__ nrows,
                                                               int I, __half* __restrict__ a16,
                                                               float* __restrict__ ainv) {
    const int r = blockIdx.x;
    if (r >= *nrows) return;
    float inv;
    const float s = pow2_range_scale(__uint_as_float(amax[r]), inv);
    if (threadIdx.x == 0) ainv[r] = inv;
    const float4* src = reinterpret_cast<const float4*>(a32 + static_cast<size_t>(r) * I);
    uint2* dst = reinterpret_cast<uint2*>(a16 + static_cast<size_t>(r) * I);
    for (int v = threadIdx.x; v < I / 4; v += 256) {
        const float4 q = src[v];
        const __half2 lo = __floats2half2_rn(q.x * s, q.y * s), hi = __floats2half2_rn(q.z * s, q.w * s);
        dst[v] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
}

// ---- combine ----------------------------------------------------------------------------------------

// out[t][j] = bf16( sum_{k in slot order} w[t,k] * y[pair_to_sorted[t*topk+k]][j] ), a separate
// rounded multiply and add per term (ep_step_fp8_gate.rs, `combine_down_rows_host`; the indexed
// twin of forward.rs's `glm5next_moe_combine_indexed`). y arrives as f16 y * 2^g with g per sorted
// row and 128-row output block (yexp); y16 * 2^-g is exact in fp32. One block per token, 8
// consecutive outputs per thread and step (16-byte loads).
__global__ void __launch_bounds__(256) prefill_combine_kernel(const __half* __restrict__ y16,
                                                              const int8_t* __restrict__ yexp,
                                                              const int32_t* __restrict__ pair_to_sorted,
                                                              const float* __restrict__ wts,
                                                              int topk, int H,
                                                              __nv_bfloat16* __restrict__ out,
                                                              const __nv_bfloat16* __restrict__ shared,
                                                              const __nv_bfloat16* __restrict__ residual) {
    const int t = blockIdx.x, nb = H / 128;
    pdl_wait();                                        // y of the down GEMM (programmatic dependent)
    int rows[kMaxTopk];
    float w[kMaxTopk];
#pragma unroll
    for (int k = 0; k < kMaxTopk; ++k) {
        rows[k] = k < topk ? pair_to_sorted[t * topk + k] : -1;
        w[k] = k < topk ? wts[t * topk + k] : 0.0f;
    }
    for (int j = threadIdx.x * 8; j < H; j += 256 * 8) {
        float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kMaxTopk; ++k) {
            if (rows[k] < 0) continue;
            const size_t r = static_cast<size_t>(rows[k]);
            const uint4 v = __ldcs(reinterpret_cast<const uint4*>(y16 + r * H + j));
            const float unscale = __int_as_float((127 - yexp[r * nb + (j >> 7)]) << 23);   // 2^-g
            const uint32_t hv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hv[q]));
                s[2 * q] = __fadd_rn(s[2 * q], __fmul_rn(w[k], f.x * unscale));
                s[2 * q + 1] = __fadd_rn(s[2 * q + 1], __fmul_rn(w[k], f.y * unscale));
            }
        }
        const size_t oj = static_cast<size_t>(t) * H + j;
        if (shared != nullptr || residual != nullptr) {   // layer epilogue: (routed + shared) + residual
            uint4 sh = make_uint4(0, 0, 0, 0), rs = make_uint4(0, 0, 0, 0);
            if (shared != nullptr) sh = *reinterpret_cast<const uint4*>(shared + oj);
            if (residual != nullptr) rs = *reinterpret_cast<const uint4*>(residual + oj);
            const uint32_t shv[4] = {sh.x, sh.y, sh.z, sh.w}, rsv[4] = {rs.x, rs.y, rs.z, rs.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (shared != nullptr) {
                    s[2 * q] = __fadd_rn(s[2 * q], __uint_as_float(shv[q] << 16));
                    s[2 * q + 1] = __fadd_rn(s[2 * q + 1], __uint_as_float(shv[q] & 0xFFFF0000u));
                }
                if (residual != nullptr) {
                    s[2 * q] = __fadd_rn(s[2 * q], __uint_as_float(rsv[q] << 16));
                    s[2 * q + 1] = __fadd_rn(s[2 * q + 1], __uint_as_float(rsv[q] & 0xFFFF0000u));
                }
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(s[2 * q], s[2 * q + 1]);
            o[q] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(out + oj) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ---- workspace and launch sequence ------------------------------------------------------------------

// pairs from which the prefill tier plans its permutation over several blocks
constexpr int kWidePlanPairs = 4096;
// largest clamp limit L for which a (|a| <= L^2) is stored in f16 without a range scale
constexpr float kA16DirectLimit = 255.0f;

PrefillLayout prefill_layout(int T, int H, int I, int E, int topk) {
    const size_t P = static_cast<size_t>(T) * topk;
    const size_t mtiles = P / prefill::kBM + static_cast<size_t>(E) + 1;
    PrefillLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    L.counts = take(static_cast<size_t>(E) * 4);
    L.offsets = take((static_cast<size_t>(E) + 1) * 4);
    L.sorted_pair = take(P * 4);
    L.pair_to_sorted = take(P * 4);
    L.tiles = take(16);
    L.tile_e = take(mtiles * 4);
    L.tile_r0 = take(mtiles * 4);
    L.tile_first = take(mtiles * 4);
    L.tile_cnt = take(mtiles * 4);
    L.x16 = take(P * H * 2);                       // [P][H], in sorted-row order for the TMA boxes
    L.xinv = take(static_cast<size_t>(T) * 4);
    L.amax = take(P * 4);
    L.a16 = take(P * static_cast<size_t>(I) * 2);
    L.ainv = take(P * 4);
    L.f32 = take(P * static_cast<size_t>(H > I ? H : I) * 4);   // a (fp32), later y (f16)
    L.tmax = take(mtiles * 4);                                 // max |a| per m-tile
    L.yexp = take(P * static_cast<size_t>(H / prefill::kBN));   // y's power of two per row and block
    L.plan_blk = take(route_plan_wide_ws_bytes(static_cast<int>(P), E));
    L.total = o;
    return L;
}


cudaError_t launch_prefill(int fmt, const __nv_bfloat16* x, int T, int H, int I, int E, int topk,
                           const int32_t* ids, const float* wts, const PrefillWeights& wt, float limit,
                           __nv_bfloat16* out, uint8_t* ws, const PrefillLayout& L, int32_t* err,
                           cudaStream_t stream, const __nv_bfloat16* shared, const __nv_bfloat16* residual) {
    const uint8_t *wg = wt.wg, *wu = wt.wu, *wd = wt.wd;
    const float *sg = wt.sg, *su = wt.su, *sd = wt.sd;
    const int P = T * topk;
    auto I32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
    cudaError_t st;
    const TileList tl{I32(L.tiles), I32(L.tile_e), I32(L.tile_r0), I32(L.tile_first), I32(L.tile_cnt),
                      prefill::kBM};
    uint32_t* amax = reinterpret_cast<uint32_t*>(ws + L.amax);
    // a finite clamp limit L <= 255 bounds |a| = |silu(min(g, L)) * clamp(u, -L, L)| by L^2, which
    // f16 holds without a range scale: the TMEM core then writes a in f16 itself
    const bool a16_direct = std::isfinite(limit) && limit <= kA16DirectLimit;
    // the direct f16 activations carry one power of two 2^s with L^2 * 2^s < 2^15, so that small
    // activations stay clear of f16's subnormal range
    int l2e = 0;
    if (a16_direct) std::frexp(static_cast<double>(limit) * limit, &l2e);
    const int a16_s = a16_direct && limit > 0.0f ? 15 - l2e : 0;
    // max |a| per sorted row (range-scaled activations: their scale, and y's f16 factor) or per
    // m-tile (f16 activations under the clamp: y's f16 factor); zeroed before the route plan, so
    // that the plan kernels, x prep and the gate/up GEMM follow one another as programmatic
    // dependent launches
    uint32_t* tmax = reinterpret_cast<uint32_t*>(ws + L.tmax);
    if (!a16_direct && (st = cudaMemsetAsync(amax, 0, static_cast<size_t>(P) * 4, stream)) != cudaSuccess)
        return st;
    if (a16_direct && (st = cudaMemsetAsync(tmax, 0, L.yexp - L.tmax, stream)) != cudaSuccess) return st;
    stage_mark(stream, "route_plan");
    // many pairs: the multi-block plan (one block serialises ~32 rounds of 1024 pairs), which also
    // builds the m-tile list
    if (P >= kWidePlanPairs) {
        st = launch_route_plan_wide(ids, P, E, I32(L.counts), I32(L.offsets), I32(L.sorted_pair),
                                    I32(L.pair_to_sorted), I32(L.plan_blk), err, stream, tl);
        if (st != cudaSuccess) return st;
    } else {
        st = launch_route_plan(ids, P, E, 1, I32(L.counts), I32(L.offsets), I32(L.sorted_pair),
                               I32(L.pair_to_sorted), nullptr, nullptr, nullptr, nullptr, err, stream);
        if (st != cudaSuccess) return st;
        stage_mark(stream, "tile_list");
        prefill_tiles_kernel<<<1, 1024, 0, stream>>>(I32(L.counts), I32(L.offsets), E, tl);
        if ((st = cudaGetLastError()) != cudaSuccess) return st;
    }
    __half* x16 = reinterpret_cast<__half*>(ws + L.x16);
    float* xinv = reinterpret_cast<float*>(ws + L.xinv);
    stage_mark(stream, "x_prep");
    {
        // a programmatic dependent of the last plan kernel: x's range scales overlap its tail
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(T);
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((st = cudaLaunchKernelEx(&cfg, prefill_x_prep_kernel, x, H, x16, xinv,
                                     static_cast<const int32_t*>(I32(L.pair_to_sorted)), topk)) != cudaSuccess)
            return st;
    }

    float* f32 = reinterpret_cast<float*>(ws + L.f32);
    PrefillGemmArgs gu{};
    gu.tiles = I32(L.tiles);
    gu.tile_e = I32(L.tile_e);
    gu.tile_r0 = I32(L.tile_r0);
    gu.tile_first = I32(L.tile_first);
    gu.tile_cnt = I32(L.tile_cnt);
    gu.offsets = I32(L.offsets);
    gu.sorted_pair = I32(L.sorted_pair);
    gu.topk = topk;
    gu.K = H;
    gu.n_tiles = I / prefill::kBN;
    gu.a = x16;
    gu.a_inv = xinv;
    gu.w0 = wg;
    gu.s0 = sg;
    gu.w1 = wu;
    gu.s1 = su;
    gu.wrows = I;
    gu.limit = limit;
    gu.out = f32;
    gu.amax = amax;
    gu.tmax = tmax;
    gu.out16 = a16_direct ? reinterpret_cast<__half*>(ws + L.a16) : nullptr;
    gu.a16_scale = std::ldexp(1.0f, a16_s);
    gu.out_ld = I;
    gu.err = err;
    gu.a_rows = P;
    gu.experts = E;
    gu.fmt = fmt;
    gu.sf0 = wt.sfg;
    gu.sf1 = wt.sfu;
    gu.s2_0 = wt.s2g;
    gu.s2_1 = wt.s2u;
    gu.s2e_0 = wt.s2g_e;
    gu.s2e_1 = wt.s2u_e;
    gu.s2_stride = wt.s2_stride;
    stage_mark(stream, "gate_up_gemm");
    if ((st = launch_prefill_gemm_tw(0, gu, I, stream)) != cudaSuccess) return st;

    __half* a16 = reinterpret_cast<__half*>(ws + L.a16);
    float* ainv = reinterpret_cast<float*>(ws + L.ainv);
    if (!a16_direct) {
        stage_mark(stream, "act_prep");
        prefill_act_prep_kernel<<<P, 256, 0, stream>>>(f32, amax, I32(L.offsets) + E, I, a16, ainv);
        if ((st = cudaGetLastError()) != cudaSuccess) return st;
    }

    PrefillGemmArgs dn = gu;
    dn.K = I;
    dn.n_tiles = H / prefill::kBN;
    dn.a = a16;
    dn.a_inv = a16_direct ? nullptr : ainv;
    dn.a16_scale = std::ldexp(1.0f, -a16_s);
    dn.out16 = nullptr;
    dn.w0 = wd;
    dn.s0 = sd;
    dn.w1 = wd;
    dn.s1 = sd;
    dn.wrows = H;
    dn.sf0 = wt.sfd;
    dn.sf1 = wt.sfd;
    dn.s2_0 = wt.s2d;
    dn.s2_1 = wt.s2d;
    dn.s2e_0 = wt.s2d_e;
    dn.s2e_1 = wt.s2d_e;
    dn.out = nullptr;
    dn.y16 = reinterpret_cast<__half*>(f32);
    dn.yexp = reinterpret_cast<int8_t*>(ws + L.yexp);
    dn.amax = amax;
    dn.out_ld = H;
    dn.a_rows = P;
    stage_mark(stream, "down_gemm");
    if ((st = launch_prefill_gemm_tw(1, dn, H, stream)) != cudaSuccess) return st;

    stage_mark(stream, "combine");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((st = cudaLaunchKernelEx(&cfg, prefill_combine_kernel, static_cast<const __half*>(dn.y16),
                                 static_cast<const int8_t*>(dn.yexp), static_cast<const int32_t*>(I32(L.pair_to_sorted)),
                                 wts, topk, H, out, shared, residual)) != cudaSuccess)
        return st;
    return cudaGetLastError();
}

}  // namespace moe
