// Router in front of the routed FFN: fp32 logits = bf16 x . bf16 router rows, then sigmoid, a
// per-expert selection bias, top-k, optional renormalisation and routed_scale
// ("spark_model layers/glm5next_mlp/forward.rs", `forward_moe` router step: one logits GEMM with
// f32 output for all rows, then one top-k launch over all rows taking logits, router_bias, top_k,
// n_group = 1, routed_scale and renormalize; the Step gate builds the same sigmoid top-k router from
// its router matrix, bias, top_k, router_scale and route_norm).
//
//   router_logits_kernel: tensor-core GEMV/GEMM. A = 16 router rows per warp (bf16 straight from
//     HBM, no conversion), B = 8 tokens per MMA column tile, mma.sync m16n8k16 bf16 -> f32, with
//     the lane layout of the FFN kernels (lane c streams 16 bytes of each of its two rows per
//     32-wide K chunk; elements 4i+{0,1} / 4i+{2,3} are logical K (2c,2c+1) / (2c+8,2c+9) of step
//     i, and B is read at the same physical positions). Few-token calls (T <= 32) take one CTA per
//     16 rows x 8 tokens x K part (up to 8 parts, summed in order by the consumer); its 16 warps
//     split the part again and meet in shared memory (dense_small_kernel). Wide calls take 32
//     tokens per CTA so that the matrix is re-read from L2 once per 32 tokens.
//   router_topk_kernel: one CTA per token sums the K parts in order and computes sigmoid and score
//     for every expert; its first warp selects top-k by repeated warp arg-max (score descending,
//     ties to the lower expert index, NaN scores after every number) over the experts not yet
//     taken (a flag per expert, so a -inf or NaN score never makes an index invalid); weights are
//     the picks' sigmoids (renormalised in pick order, times routed_scale).
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kRtWarps = 4;                       // expert tiles of 16 per logits CTA
constexpr int kRtTopkWarps = 4;                   // warps of a top-k CTA (one token)

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// part[ks][t][e] for K chunks (32 wide) [ks*NC/KS, (ks+1)*NC/KS), tokens blockIdx.y*8*TS ..
template <int TS>
__global__ void __launch_bounds__(kRtWarps * 32) router_logits_kernel(const __nv_bfloat16* __restrict__ x, int T,
                                                                     int H, const __nv_bfloat16* __restrict__ w,
                                                                     int E, float* __restrict__ part) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int e0 = (blockIdx.x * kRtWarps + warp) * 16;
    if (e0 >= E) return;
    const int KS = gridDim.z, ks = blockIdx.z, NC = H / 32;
    const int k0 = ks * NC / KS, k1 = (ks + 1) * NC / KS;
    const int tbase = blockIdx.y * 8 * TS;
    const uint4* ra = reinterpret_cast<const uint4*>(w + static_cast<size_t>(e0 + g) * H + c * 8);
    const uint4* rb = reinterpret_cast<const uint4*>(w + static_cast<size_t>(e0 + g + 8) * H + c * 8);
    const uint4* xb[TS];
    bool tv[TS];
#pragma unroll
    for (int j = 0; j < TS; ++j) {
        const int t = tbase + 8 * j + g;
        tv[j] = t < T;
        xb[j] = reinterpret_cast<const uint4*>(x + static_cast<size_t>(tv[j] ? t : 0) * H + c * 8);
    }
    float acc[TS][4];
#pragma unroll
    for (int j = 0; j < TS; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
    for (int kc = k0; kc < k1; ++kc) {
        const uint4 qa = ld_stream_v4(ra + kc * 4), qb = ld_stream_v4(rb + kc * 4);   // 32 bf16 = 4 uint4
#pragma unroll
        for (int j = 0; j < TS; ++j) {
            const uint4 bx = tv[j] ? __ldg(xb[j] + kc * 4) : make_uint4(0, 0, 0, 0);
            mma_bf16(acc[j], qa.x, qb.x, qa.y, qb.y, bx.x, bx.y);
            mma_bf16(acc[j], qa.z, qb.z, qa.w, qb.w, bx.z, bx.w);
        }
    }
    float* dst = part + static_cast<size_t>(ks) * T * E;
#pragma unroll
    for (int j = 0; j < TS; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int t = tbase + 8 * j + 2 * c + (q & 1), e = e0 + g + 8 * (q >> 1);
            if (t < T) dst[static_cast<size_t>(t) * E + e] = acc[j][q];
        }
    }
}

// Few tokens (T <= 32): one CTA per (16 rows, 8 tokens); its 16 warps split K, keep four 32-wide
// chunks of loads in flight each, and meet in shared memory (fixed order) - no partial buffer.
constexpr int kRtSmallWarps = 16;
__global__ void __launch_bounds__(kRtSmallWarps * 32) dense_small_kernel(const __nv_bfloat16* __restrict__ x, int T,
                                                                         int H, const __nv_bfloat16* __restrict__ w,
                                                                         int E, float* __restrict__ out) {
    __shared__ float red[kRtSmallWarps][32][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int e0 = blockIdx.x * 16, tbase = blockIdx.y * 8;
    // this CTA's K part (grid z), split again over its 16 warps
    const int KS = gridDim.z, ks = blockIdx.z, NC = H / 32;
    const int c0 = ks * NC / KS, nc = (ks + 1) * NC / KS - c0;
    const int k0 = c0 + warp * nc / kRtSmallWarps, k1 = c0 + (warp + 1) * nc / kRtSmallWarps;
    const uint4* ra = reinterpret_cast<const uint4*>(w + static_cast<size_t>(e0 + g) * H + c * 8);
    const uint4* rb = reinterpret_cast<const uint4*>(w + static_cast<size_t>(e0 + g + 8) * H + c * 8);
    const int t = tbase + g;
    const bool tv = t < T;
    const uint4* xb = reinterpret_cast<const uint4*>(x + static_cast<size_t>(tv ? t : 0) * H + c * 8);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    constexpr int kU = 4;
    for (int kc = k0; kc < k1; kc += kU) {
        uint4 qa[kU], qb[kU], bx[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const bool in = kc + u < k1;
            qa[u] = in ? ld_stream_v4(ra + (kc + u) * 4) : make_uint4(0, 0, 0, 0);
            qb[u] = in ? ld_stream_v4(rb + (kc + u) * 4) : make_uint4(0, 0, 0, 0);
            bx[u] = in && tv ? __ldg(xb + (kc + u) * 4) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            mma_bf16(acc, qa[u].x, qb[u].x, qa[u].y, qb[u].y, bx[u].x, bx[u].y);
            mma_bf16(acc, qa[u].z, qb[u].z, qa[u].w, qb[u].w, bx[u].z, bx[u].w);
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) red[warp][lane][q] = acc[q];
    __syncthreads();
    if (warp == 0) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int v = 0; v < kRtSmallWarps; ++v)
#pragma unroll
            for (int q = 0; q < 4; ++q) s[q] += red[v][lane][q];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int tt = tbase + 2 * c + (q & 1), e = e0 + g + 8 * (q >> 1);
            if (tt < T) out[(static_cast<size_t>(ks) * T + tt) * E + e] = s[q];
        }
    }
}

// Selection order of the top-k scan: a higher score first, equal scores to the lower expert index,
// and a NaN score after every number (a NaN logit or bias cannot pick an expert ahead of a finite
// or infinite score; NaN scores among themselves go by index). `be` < 0 means no candidate yet.
__device__ __forceinline__ bool topk_better(float v, int e, float bs, int be) {
    if (be < 0) return true;
    const bool vn = isnan(v), bn = isnan(bs);
    if (vn != bn) return bn;
    if (vn) return e < be;
    return v > bs || (v == bs && e < be);
}

__global__ void __launch_bounds__(kRtTopkWarps * 32) router_topk_kernel(const float* __restrict__ part, int KS,
                                                                        int T, int E, const float* __restrict__ bias,
                                                                        int topk, float routed_scale, int renorm,
                                                                        float* __restrict__ logits,
                                                                        int32_t* __restrict__ ids,
                                                                        float* __restrict__ wts) {
    // one CTA per token: all its threads sum the K parts and score the experts, warp 0 selects
    extern __shared__ float rt_smem[];                // [2][E] fp32: sigmoid, score; then [E] taken flags
    const int lane = threadIdx.x & 31, t = blockIdx.x;
    float* sig = rt_smem;
    float* score = sig + E;
    unsigned char* taken = reinterpret_cast<unsigned char*>(score + E);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float l = 0.0f;
#pragma unroll 8
        for (int q = 0; q < KS; ++q) l += part[(static_cast<size_t>(q) * T + t) * E + e];
        if (logits != nullptr) logits[static_cast<size_t>(t) * E + e] = l;
        const float s = 1.0f / (1.0f + expf(-l));
        sig[e] = s;
        score[e] = s + (bias != nullptr ? bias[e] : 0.0f);
        taken[e] = 0;
    }
    __syncthreads();
    if (threadIdx.x >= 32) return;
    float picked[kMaxTopk];                          // unrolled to kMaxTopk: stays in registers
    int pid[kMaxTopk];
#pragma unroll
    for (int k = 0; k < kMaxTopk; ++k) {
        if (k >= topk) break;
        // a lane's candidate is always an untaken expert (or none): taken experts are skipped by
        // their flag, not by a marker score, so -inf and NaN scores stay selectable
        float bs = 0.0f;
        int be = -1;
        for (int e = lane; e < E; e += 32) {
            if (taken[e]) continue;
            const float v = score[e];
            if (topk_better(v, e, bs, be)) {
                bs = v;
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (oe >= 0 && topk_better(os, oe, bs, be)) {
                bs = os;
                be = oe;
            }
        }
        // k < topk <= E experts are taken, so some lane had an untaken candidate; the clamp only
        // keeps every index in [0, E) by construction
        be = be < 0 ? 0 : (be >= E ? E - 1 : be);
        __syncwarp();
        if (lane == 0) taken[be] = 1;
        __syncwarp();
        pid[k] = be;
        picked[k] = sig[be];
    }
    if (lane == 0) {
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < kMaxTopk; ++k)
            if (k < topk) sum += picked[k];
#pragma unroll
        for (int k = 0; k < kMaxTopk; ++k) {
            if (k >= topk) break;
            const float wv = renorm ? picked[k] / sum : picked[k];
            ids[static_cast<size_t>(t) * topk + k] = pid[k];
            wts[static_cast<size_t>(t) * topk + k] = wv * routed_scale;
        }
    }
}

}  // namespace

int router_ksplit(int T, int H, int E, int sms) {
    if (T > 32) return 1;
    // few tokens: enough CTAs (one per 16 rows x 8 tokens x K part) to cover the SMs; each CTA
    // splits its part again over 16 warps
    const int ctas = (E / 16) * ((T + 7) / 8);
    int ks = (sms + ctas - 1) / ctas;
    if (ks > 8) ks = 8;
    if (ks > H / 32 / 16) ks = H / 32 / 16;
    return ks < 1 ? 1 : ks;
}

cudaError_t launch_dense_bf16(const __nv_bfloat16* x, int T, int K, const __nv_bfloat16* w, int N, float* part,
                              int KS, cudaStream_t stream) {
    const int ex = (N / 16 + kRtWarps - 1) / kRtWarps;
    if (T > 32)
        router_logits_kernel<4><<<dim3(ex, (T + 31) / 32, KS), kRtWarps * 32, 0, stream>>>(x, T, K, w, N, part);
    else
        dense_small_kernel<<<dim3(N / 16, (T + 7) / 8, KS), kRtSmallWarps * 32, 0, stream>>>(x, T, K, w, N, part);
    return cudaGetLastError();
}

size_t router_topk_smem_bytes(int E) { return static_cast<size_t>(2) * E * sizeof(float) + static_cast<size_t>(E); }

cudaError_t launch_router(const __nv_bfloat16* x, int T, int H, const __nv_bfloat16* w, const float* bias, int E,
                          int topk, float routed_scale, int renorm, float* logits, int32_t* ids, float* wts,
                          float* part, int KS, cudaStream_t stream) {
    cudaError_t st = launch_dense_bf16(x, T, H, w, E, part, KS, stream);
    if (st != cudaSuccess) return st;
    const size_t smem = router_topk_smem_bytes(E);
    if (smem > 48 * 1024 &&
        (st = cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem))) != cudaSuccess)
        return st;
    router_topk_kernel<<<T, kRtTopkWarps * 32, smem, stream>>>(
        part, KS, T, E, bias, topk, routed_scale, renorm, logits, ids, wts);
    return cudaGetLastError();
}

}  // namespace moe
