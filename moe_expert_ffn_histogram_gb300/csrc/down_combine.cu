// Dequant-fused down projection fused with the fixed-order top-k weighted combine.
//
//     y(t,k)[j] = sum_n a(t,k)[n] * Wd[e][j][n]
//     out[t][j] = bf16( sum_{k = 0 .. topk-1, in slot order} w[t][k] * y(t,k)[j] )
//
// Sources: "memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs", `combine_down_rows_host` (slot
// order, a separate round-to-nearest multiply and add per term) and `reference_expert` (down on
// the activation); "spark_model layers/glm5next_mlp/forward.rs", `glm5next_moe_combine` call site
// in `forward_moe` (one combine for every row instead of per-row launches). Here the combine is
// the epilogue of the down GEMV: a CTA owns 16 output rows j for every token, sweeps the down
// rows of every routed group through its 8 warps, keeps y in shared memory and combines in slot
// order, so there is no expert_out buffer and no atomics; the result is deterministic.
#include "kernels.cuh"

namespace moe {


namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;          // 64-wide K segments per load batch

}  // namespace

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) down_combine_kernel(const DownArgs a) {
    extern __shared__ __align__(16) float ys[];     // [P][16]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int H = a.H, I = a.I;
    const int j0 = blockIdx.x * kDownRows;
    const Groups& G = a.grp;
    const int ngroups = G.count == nullptr ? a.topk : *G.count;
    const int nseg = I / 64;

    for (int gi = warp; gi < ngroups; gi += kWarps) {
        int e, ncols, st = 0;
        if (G.count == nullptr) {
            e = G.ids[gi];
            ncols = 1;
            if (e < 0 || e >= G.E) continue;
        } else {
            e = G.expert[gi];
            ncols = G.ncols[gi];
            st = G.start[gi];
        }
        auto pair_of = [&](int col) { return G.count == nullptr ? gi : G.sorted_pair[st + col]; };
        const bool has_b = g < ncols;
        const int pb = has_b ? pair_of(g) : 0;
        const int col0 = 2 * c, col1 = 2 * c + 1;
        const int p0 = col0 < ncols ? pair_of(col0) : -1;
        const int p1 = col1 < ncols ? pair_of(col1) : -1;
        const __half* hb = a.act + static_cast<size_t>(pb) * I + c * 16;
        const float* hs0 = a.act_scale + static_cast<size_t>(p0 < 0 ? 0 : p0) * (I / kFeatBlock);
        const float* hs1 = a.act_scale + static_cast<size_t>(p1 < 0 ? 0 : p1) * (I / kFeatBlock);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};   // (row g: col0, col1), (row g+8: col0, col1)

        if constexpr (FMT == 0) {
            const size_t r0 = static_cast<size_t>(e) * H + j0 + g;
            const uint8_t* pa0 = a.wd + r0 * I + c * 16;
            const uint8_t* pa1 = pa0 + static_cast<size_t>(8) * I;
            const float* wsr = a.sd + (static_cast<size_t>(e) * (H / 128) + j0 / 128) * (I / 128);
            for (int s0 = 0; s0 < nseg; s0 += kStages) {
                uint4 qa[kStages], qb[kStages];
#pragma unroll
                for (int s = 0; s < kStages; ++s) {
                    if (s0 + s < nseg) {
                        qa[s] = ld_stream_v4(pa0 + (s0 + s) * 64);
                        qb[s] = ld_stream_v4(pa1 + (s0 + s) * 64);
                    }
                }
#pragma unroll
                for (int s = 0; s < kStages; ++s) {
                    const int seg = s0 + s;
                    if (seg < nseg) {
                        uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
                        if (has_b) {
                            const uint4* bp = reinterpret_cast<const uint4*>(hb + seg * 64);
                            b0 = __ldg(bp);
                            b1 = __ldg(bp + 1);
                        }
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        const uint32_t wa[4] = {qa[s].x, qa[s].y, qa[s].z, qa[s].w};
                        const uint32_t wb[4] = {qb[s].x, qb[s].y, qb[s].z, qb[s].w};
                        const uint32_t bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t a_lo, a_hi, b_lo, b_hi;
                            e4m3x4_to_f16x2x2(wa[i], a_lo, a_hi);
                            e4m3x4_to_f16x2x2(wb[i], b_lo, b_hi);
                            mma_f16(d, a_lo, b_lo, a_hi, b_hi, bb[2 * i], bb[2 * i + 1]);
                        }
                        const float wsc = __ldg(wsr + seg / 2);
                        const float f0 = p0 >= 0 ? wsc * __ldg(hs0 + seg) : 0.0f;
                        const float f1 = p1 >= 0 ? wsc * __ldg(hs1 + seg) : 0.0f;
                        acc[0] = fmaf(d[0], f0, acc[0]);
                        acc[1] = fmaf(d[1], f1, acc[1]);
                        acc[2] = fmaf(d[2], f0, acc[2]);
                        acc[3] = fmaf(d[3], f1, acc[3]);
                    }
                }
            }
        } else {
            const size_t r0 = static_cast<size_t>(e) * H + j0 + g;
            const uint8_t* pa0 = a.wd + r0 * (I / 2) + c * 8;
            const uint8_t* pa1 = pa0 + static_cast<size_t>(8) * (I / 2);
            const uint8_t* fa0 = a.sfd + r0 * (I / 16) + c;
            const uint8_t* fa1 = fa0 + static_cast<size_t>(8) * (I / 16);
            constexpr int kS = 2 * kStages;
            for (int s0 = 0; s0 < nseg; s0 += kS) {
                uint2 qa[kS], qb[kS];
                uint32_t fa[kS], fb[kS];
#pragma unroll
                for (int s = 0; s < kS; ++s) {
                    if (s0 + s < nseg) {
                        qa[s] = ld_stream_v2(pa0 + (s0 + s) * 32);
                        qb[s] = ld_stream_v2(pa1 + (s0 + s) * 32);
                        fa[s] = ld_stream_u8(fa0 + (s0 + s) * 4);
                        fb[s] = ld_stream_u8(fa1 + (s0 + s) * 4);
                    }
                }
#pragma unroll
                for (int s = 0; s < kS; ++s) {
                    const int seg = s0 + s;
                    if (seg < nseg) {
                        uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
                        if (has_b) {
                            const uint4* bp = reinterpret_cast<const uint4*>(hb + seg * 64);
                            b0 = __ldg(bp);
                            b1 = __ldg(bp + 1);
                        }
                        const uint32_t sa = e4m3_splat_f16x2(fa[s]), sb = e4m3_splat_f16x2(fb[s]);
                        uint32_t xa[8], xb[8];
                        e2m1x8_to_f16x2x4(qa[s].x, xa[0], xa[1], xa[2], xa[3]);
                        e2m1x8_to_f16x2x4(qa[s].y, xa[4], xa[5], xa[6], xa[7]);
                        e2m1x8_to_f16x2x4(qb[s].x, xb[0], xb[1], xb[2], xb[3]);
                        e2m1x8_to_f16x2x4(qb[s].y, xb[4], xb[5], xb[6], xb[7]);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            xa[j] = hmul2(xa[j], sa);
                            xb[j] = hmul2(xb[j], sb);
                        }
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_f16(d, xa[0], xb[0], xa[1], xb[1], b0.x, b0.y);
                        mma_f16(d, xa[2], xb[2], xa[3], xb[3], b0.z, b0.w);
                        mma_f16(d, xa[4], xb[4], xa[5], xb[5], b1.x, b1.y);
                        mma_f16(d, xa[6], xb[6], xa[7], xb[7], b1.z, b1.w);
                        const float f0 = p0 >= 0 ? __ldg(hs0 + seg) : 0.0f;
                        const float f1 = p1 >= 0 ? __ldg(hs1 + seg) : 0.0f;
                        acc[0] = fmaf(d[0], f0, acc[0]);
                        acc[1] = fmaf(d[1], f1, acc[1]);
                        acc[2] = fmaf(d[2], f0, acc[2]);
                        acc[3] = fmaf(d[3], f1, acc[3]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] *= a.s2d;
        }
        if (p0 >= 0) {
            ys[p0 * kDownRows + g] = acc[0];
            ys[p0 * kDownRows + g + 8] = acc[2];
        }
        if (p1 >= 0) {
            ys[p1 * kDownRows + g] = acc[1];
            ys[p1 * kDownRows + g + 8] = acc[3];
        }
    }
    __syncthreads();

    // slot-order combine: one thread per (token, row); a separate rounded multiply and add per
    // term, so the order and the roundings are fixed
    for (int i = tid; i < a.T * kDownRows; i += kThreads) {
        const int t = i / kDownRows, r = i % kDownRows;
        float s = 0.0f;
        for (int k = 0; k < a.topk; ++k) {
            const int p = t * a.topk + k;
            const int e = a.ids[p];
            if (e < 0 || e >= a.E) continue;
            s = __fadd_rn(s, __fmul_rn(a.wts[p], ys[p * kDownRows + r]));
        }
        a.out[static_cast<size_t>(t) * H + j0 + r] = __float2bfloat16_rn(s);
    }
}

size_t down_smem_bytes(int T, int topk) {
    return static_cast<size_t>(T) * topk * kDownRows * sizeof(float);
}

template <int FMT>
cudaError_t launch_down_combine(const DownArgs& a, cudaStream_t stream) {
    const size_t smem = down_smem_bytes(a.T, a.topk);
    if (smem > 48 * 1024) {
        cudaError_t st = cudaFuncSetAttribute(down_combine_kernel<FMT>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem));
        if (st != cudaSuccess) return st;
    }
    down_combine_kernel<FMT><<<a.H / kDownRows, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template cudaError_t launch_down_combine<0>(const DownArgs&, cudaStream_t);
template cudaError_t launch_down_combine<1>(const DownArgs&, cudaStream_t);

}  // namespace moe
