// Dequant-fused gate + up projections with the clamped SwiGLU fused into the epilogue.
//
// For every routed group (one expert, up to 8 columns = routed pairs) and every block of 64
// intermediate features n, computes
//     g[n] = sum_k x[k] * Wg[e][n][k]      u[n] = sum_k x[k] * Wu[e][n][k]
//     a[n] = silu(min(g, limit)) * clamp(u, -limit, limit)
// and stores a as f16 with one power-of-two range scale per (pair, 64-feature block).
//
// Sources: "memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs", `reference_expert` (gate, up,
// activation); "spark_model layers/glm5next_mlp/forward.rs", `swiglu_rows` (the asymmetric clamp)
// and `w4a16_gemv_moe` / `w4a16_gemv_moe_batchm` (every routed slot in one launch; each union
// expert swept once for all the rows that selected it). Here gate and up share one pass: the 16
// MMA rows of a warp are 8 gate rows and the same 8 up rows, so g and u of a feature meet in one
// lane and the SwiGLU needs no extra launch or buffer.
//
// Layout: CTA = 8 warps x 8 features; warp w owns features n0 + 8w .. n0 + 8w + 7. A lane streams
// 16 bytes (FP8) or 8 bytes (NVFP4) of each of its two weight rows per 64-wide K segment with
// L1-bypassing 128/64-bit loads; the columns' activations sit in shared memory as f16.
#include "kernels.cuh"

namespace moe {


namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStagesFp8 = 4;    // 128-wide K blocks per load batch (64 B per row per lane)
constexpr int kStagesFp4 = 8;    // 64-wide K segments per load batch (64 B per row per lane)

__device__ __forceinline__ float clamped_swiglu(float g, float u, float limit) {
    g = fminf(g, limit);
    u = fminf(fmaxf(u, -limit), limit);
    return g / (1.0f + expf(-g)) * u;
}

// One MMA step for FP8 rows: 4 code bytes of the gate row (qg) and of the up row (qu).
__device__ __forceinline__ void mma_step_fp8(float (&d)[4], uint32_t qg, uint32_t qu,
                                             uint32_t b0, uint32_t b1) {
    uint32_t g_lo, g_hi, u_lo, u_hi;
    e4m3x4_to_f16x2x2(qg, g_lo, g_hi);
    e4m3x4_to_f16x2x2(qu, u_lo, u_hi);
    mma_f16(d, g_lo, u_lo, g_hi, u_hi, b0, b1);
}

}  // namespace

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) gate_up_kernel(const GateUpArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __half* xs = reinterpret_cast<__half*>(smem_raw);       // [ncols][H] f16, range-scaled
    __shared__ float x_inv[kMaxCols];
    __shared__ int col_pair[kMaxCols];
    __shared__ int s_expert, s_ncols;
    __shared__ float red[kWarps][kMaxCols];
    __shared__ float a_scale[kMaxCols], a_inv[kMaxCols];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int H = a.H, I = a.I;
    const Groups& G = a.grp;

    if (tid == 0) {
        int e = -1, nc = 0;
        const int gi = blockIdx.y;
        if (G.count == nullptr) {           // implicit: group = slot of the single token
            e = G.ids[gi];
            nc = 1;
            col_pair[0] = gi;
            if (e < 0 || e >= G.E) {
                if (e != -1 && blockIdx.x == 0 && a.err) atomicOr(a.err, 1);
                e = -1;
            }
        } else if (gi < *G.count) {
            e = G.expert[gi];
            nc = G.ncols[gi];
            const int st = G.start[gi];
            for (int j = 0; j < nc; ++j) col_pair[j] = G.sorted_pair[st + j];
        }
        s_expert = e;
        s_ncols = nc;
    }
    __syncthreads();
    const int e = s_expert;
    if (e < 0) return;
    const int ncols = s_ncols;

    // ---- stage the columns' activations as f16 with a per-column power-of-two scale ----
    {
        const int nv = H / 8;                       // 16-byte vectors of 8 bf16
        float m[kMaxCols];
#pragma unroll
        for (int j = 0; j < kMaxCols; ++j) m[j] = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxCols; ++j) {
            if (j < ncols) {
                const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(col_pair[j] / G.topk) * H);
                float mj = 0.0f;
                for (int v = tid; v < nv; v += kThreads) {
                    const uint4 q = __ldg(xr + v);
                    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        mj = fmaxf(mj, fabsf(__uint_as_float(w[i] << 16)));
                        mj = fmaxf(mj, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
                    }
                }
                m[j] = mj;
            }
        }
#pragma unroll
        for (int j = 0; j < kMaxCols; ++j) {
            const float r = warp_max(m[j]);
            if (lane == 0) red[warp][j] = r;
        }
        __syncthreads();
        if (tid < ncols) {
            float mm = 0.0f;
            for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, red[w][tid]);
            float inv;
            a_scale[tid] = pow2_range_scale(mm, inv);
            x_inv[tid] = inv;
        }
        __syncthreads();
        for (int j = 0; j < ncols; ++j) {
            const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(col_pair[j] / G.topk) * H);
            const float s = a_scale[j];
            uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<size_t>(j) * H);
            for (int v = tid; v < nv; v += kThreads) {
                const uint4 q = __ldg(xr + v);
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const __half2 h2 = __floats2half2_rn(__uint_as_float(w[i] << 16) * s,
                                                         __uint_as_float(w[i] & 0xFFFF0000u) * s);
                    o[i] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        __syncthreads();
    }

    // ---- main loop: 16 MMA rows = 8 gate rows + the same 8 up rows ----
    const int n = blockIdx.x * kFeatBlock + warp * 8 + g;
    const bool has_b = g < ncols;
    const __half* xb = xs + static_cast<size_t>(has_b ? g : 0) * H + c * 16;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};   // gate(col 2c), gate(col 2c+1), up(2c), up(2c+1)

    if constexpr (FMT == 0) {
        const size_t row = static_cast<size_t>(e) * I + n;
        const uint8_t* pg = a.wg + row * H + c * 16;
        const uint8_t* pu = a.wu + row * H + c * 16;
        const int nkb = H / 128;
        const size_t srow = (static_cast<size_t>(e) * (I / 128) + (blockIdx.x * kFeatBlock) / 128) * (H / 128);
        const float* sgr = a.sg + srow;
        const float* sur = a.su + srow;
        for (int kb0 = 0; kb0 < nkb; kb0 += kStagesFp8) {
            uint4 q[kStagesFp8][4];
#pragma unroll
            for (int s = 0; s < kStagesFp8; ++s) {
                if (kb0 + s < nkb) {
                    const size_t off = static_cast<size_t>(kb0 + s) * 128;
                    q[s][0] = ld_stream_v4(pg + off);
                    q[s][1] = ld_stream_v4(pu + off);
                    q[s][2] = ld_stream_v4(pg + off + 64);
                    q[s][3] = ld_stream_v4(pu + off + 64);
                }
            }
#pragma unroll
            for (int s = 0; s < kStagesFp8; ++s) {
                const int kb = kb0 + s;
                if (kb < nkb) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
                        if (has_b) {
                            const uint4* bp = reinterpret_cast<const uint4*>(xb + kb * 128 + h * 64);
                            b0 = bp[0];
                            b1 = bp[1];
                        }
                        const uint4 qg = q[s][2 * h], qu = q[s][2 * h + 1];
                        mma_step_fp8(d, qg.x, qu.x, b0.x, b0.y);
                        mma_step_fp8(d, qg.y, qu.y, b0.z, b0.w);
                        mma_step_fp8(d, qg.z, qu.z, b1.x, b1.y);
                        mma_step_fp8(d, qg.w, qu.w, b1.z, b1.w);
                    }
                    const float fg = __ldg(sgr + kb), fu = __ldg(sur + kb);
                    acc[0] = fmaf(d[0], fg, acc[0]);
                    acc[1] = fmaf(d[1], fg, acc[1]);
                    acc[2] = fmaf(d[2], fu, acc[2]);
                    acc[3] = fmaf(d[3], fu, acc[3]);
                }
            }
        }
    } else {
        const size_t row = static_cast<size_t>(e) * I + n;
        const uint8_t* pg = a.wg + row * (H / 2) + c * 8;
        const uint8_t* pu = a.wu + row * (H / 2) + c * 8;
        const uint8_t* fgp = a.sfg + row * (H / 16) + c;
        const uint8_t* fup = a.sfu + row * (H / 16) + c;
        const int nseg = H / 64;
        for (int s0 = 0; s0 < nseg; s0 += kStagesFp4) {
            uint2 qg[kStagesFp4], qu[kStagesFp4];
            uint32_t fg[kStagesFp4], fu[kStagesFp4];
#pragma unroll
            for (int s = 0; s < kStagesFp4; ++s) {
                if (s0 + s < nseg) {
                    qg[s] = ld_stream_v2(pg + (s0 + s) * 32);
                    qu[s] = ld_stream_v2(pu + (s0 + s) * 32);
                    fg[s] = ld_stream_u8(fgp + (s0 + s) * 4);
                    fu[s] = ld_stream_u8(fup + (s0 + s) * 4);
                }
            }
#pragma unroll
            for (int s = 0; s < kStagesFp4; ++s) {
                const int seg = s0 + s;
                if (seg < nseg) {
                    uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
                    if (has_b) {
                        const uint4* bp = reinterpret_cast<const uint4*>(xb + seg * 64);
                        b0 = bp[0];
                        b1 = bp[1];
                    }
                    const uint32_t sg2 = e4m3_splat_f16x2(fg[s]), su2 = e4m3_splat_f16x2(fu[s]);
                    uint32_t ga[8], ua[8];
                    e2m1x8_to_f16x2x4(qg[s].x, ga[0], ga[1], ga[2], ga[3]);
                    e2m1x8_to_f16x2x4(qg[s].y, ga[4], ga[5], ga[6], ga[7]);
                    e2m1x8_to_f16x2x4(qu[s].x, ua[0], ua[1], ua[2], ua[3]);
                    e2m1x8_to_f16x2x4(qu[s].y, ua[4], ua[5], ua[6], ua[7]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        ga[j] = hmul2(ga[j], sg2);
                        ua[j] = hmul2(ua[j], su2);
                    }
                    mma_f16(acc, ga[0], ua[0], ga[1], ua[1], b0.x, b0.y);
                    mma_f16(acc, ga[2], ua[2], ga[3], ua[3], b0.z, b0.w);
                    mma_f16(acc, ga[4], ua[4], ga[5], ua[5], b1.x, b1.y);
                    mma_f16(acc, ga[6], ua[6], ga[7], ua[7], b1.z, b1.w);
                }
            }
        }
    }

    // ---- epilogue: unscale, clamped SwiGLU, per-(pair, 64-block) range scale, f16 store ----
    float hv[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int col = 2 * c + j;
        hv[j] = 0.0f;
        if (col < ncols) {
            float gv = acc[j] * x_inv[col], uv = acc[2 + j] * x_inv[col];
            if constexpr (FMT == 1) {
                gv *= a.s2g;
                uv *= a.s2u;
            }
            hv[j] = clamped_swiglu(gv, uv, a.limit);
        }
    }
    float m0 = fabsf(hv[0]), m1 = fabsf(hv[1]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    if (g == 0) {
        red[warp][2 * c] = m0;
        red[warp][2 * c + 1] = m1;
    }
    __syncthreads();
    if (tid < ncols) {
        float mm = 0.0f;
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, red[w][tid]);
        float inv;
        a_scale[tid] = pow2_range_scale(mm, inv);
        a_inv[tid] = inv;
        a.act_scale[static_cast<size_t>(col_pair[tid]) * (I / kFeatBlock) + blockIdx.x] = inv;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int col = 2 * c + j;
        if (col < ncols)
            a.act[static_cast<size_t>(col_pair[col]) * I + n] = __float2half_rn(hv[j] * a_scale[col]);
    }
}

size_t gate_up_smem_bytes(int H, int max_cols) {
    return static_cast<size_t>(max_cols) * H * sizeof(__half);
}

template <int FMT>
cudaError_t launch_gate_up(const GateUpArgs& a, int num_groups, int max_cols, cudaStream_t stream) {
    const size_t smem = gate_up_smem_bytes(a.H, max_cols);
    if (smem > 48 * 1024) {
        cudaError_t st = cudaFuncSetAttribute(gate_up_kernel<FMT>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem));
        if (st != cudaSuccess) return st;
    }
    dim3 grid(a.I / kFeatBlock, num_groups);
    gate_up_kernel<FMT><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template cudaError_t launch_gate_up<0>(const GateUpArgs&, int, int, cudaStream_t);
template cudaError_t launch_gate_up<1>(const GateUpArgs&, int, int, cudaStream_t);

}  // namespace moe
