// The two GEMV work items of the routed MoE FFN, as CTA-level device functions shared by the
// stage kernels (gate_up.cu, down_combine.cu) and the fused persistent kernel (fused.cu).
//
//   gate_up_item: one routed group (one expert, up to 8 columns = routed pairs) x one block of 64
//     intermediate features: g and u for the block, the clamped SwiGLU, and the activation a as
//     f16 with one power-of-two range scale per (pair, 64-feature block).
//     Sources: "memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs", `reference_expert`;
//     "spark_model layers/glm5next_mlp/forward.rs", `swiglu_rows` (asymmetric clamp) and
//     `w4a16_gemv_moe_batchm` (each union expert swept once for all rows that selected it).
//   down_item: 16 output rows j for every group, then the slot-order weighted combine of those
//     rows for every token ("memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs",
//     `combine_down_rows_host`: slot order, separate rounded multiply and add).
//
// Both run on 8 warps (256 threads). Every warp owns one 16-row MMA tile (see moe_common.cuh for
// the lane layout) and streams its two weight rows with L1-bypassing vector loads in batches of
// 512 B per row, the batch size at which this row-interleaved stream matches a plain sequential
// read on GB300 HBM.
#pragma once
#include "kernels.cuh"

namespace moe {

constexpr int kItemWarps = 8;
constexpr int kItemThreads = kItemWarps * 32;
constexpr int kMaxPairs = kMaxTopk * kMaxCols;   // pairs of one sub-batch (<= 8 tokens x top-8)
#ifndef MOE_GU_BATCH
#define MOE_GU_BATCH 4
#endif
#ifndef MOE_GU_BATCH_FP4
#define MOE_GU_BATCH_FP4 4
#endif
#ifndef MOE_DN_BATCH
#define MOE_DN_BATCH 4
#endif
#ifndef MOE_DN_BATCH_FP4
#define MOE_DN_BATCH_FP4 2
#endif
#ifndef MOE_FUSED_DN_BATCH
#define MOE_FUSED_DN_BATCH 1
#endif
#ifndef MOE_FUSED_GU_BATCH
#define MOE_FUSED_GU_BATCH MOE_GU_BATCH
#endif
#ifndef MOE_FUSED_GU_BATCH_FP4
#define MOE_FUSED_GU_BATCH_FP4 MOE_GU_BATCH_FP4
#endif
#ifndef MOE_FUSED_DN_BATCH_FP4
#define MOE_FUSED_DN_BATCH_FP4 4
#endif
#ifndef MOE_MIN_BLOCKS
#define MOE_MIN_BLOCKS 2
#endif
#ifndef MOE_DN_MIN_BLOCKS
#define MOE_DN_MIN_BLOCKS 3
#endif
constexpr int kStagesFp8 = MOE_GU_BATCH;      // 128-wide K blocks per load batch (128 B per row each)
constexpr int kStagesFp4 = MOE_GU_BATCH_FP4;  // 128-wide K super-segments per batch (64 B per row each)
constexpr int kFusedStagesFp8 = MOE_FUSED_GU_BATCH;       // the same in the fused kernel
constexpr int kFusedStagesFp4 = MOE_FUSED_GU_BATCH_FP4;
// 64-wide K segments per down load batch: the stage kernel's (FP8, NVFP4) and the fused kernel's
// (measured: single-token NVFP4 down 26.0 -> 19.3 us with 2 instead of 4; the fused FP8 batch-M
// step 400 -> 346 us with 1; the fused NVFP4 step at T=8 best with 4)
constexpr int kDownBatch = MOE_DN_BATCH;
constexpr int kDownBatchFp4 = MOE_DN_BATCH_FP4;
constexpr int kFusedDownBatch = MOE_FUSED_DN_BATCH;
constexpr int kFusedDownBatchFp4 = MOE_FUSED_DN_BATCH_FP4;
constexpr int kMinBlocks = MOE_MIN_BLOCKS;    // CTAs per SM the register budget is sized for
constexpr int kDownMinBlocks = MOE_DN_MIN_BLOCKS;   // the same, for the down stage kernel

// One routed group as a CTA sees it: its expert and the routed pairs (t*topk + k) it serves.
struct GroupView {
    int e;
    int ncols;
    int pair[kMaxCols];
};

// Every group of one sub-batch, in shared memory.
struct GroupList {
    int count;
    GroupView g[kMaxPairs];
};

// Small shared scratch of gate_up_item.
struct GateUpShared {
    uint4 zeros[2];                        // a zero B fragment pair (single-token NVFP4 path)
    float x_inv[kMaxCols];
    float red[kItemWarps][kMaxCols];
    float a_scale[kMaxCols];
};

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

// One 128-wide super-segment of the single-token NVFP4 gate/up product for lane (g, c) of a warp:
// the MMA's 8 B columns carry the super-segment's 8 scale groups instead of tokens. In half h
// lane c's codes belong to group 2c + h; only the lane that holds B column 2c + h at lane c's
// positions, (g = 2c + h, c), has the token's x there (xh[2h], xh[2h+1]) and every other B value
// is zero (d[h] collects half h, so the two halves are two independent MMA chains), so D[row][n] is the row's partial dot product over group n, scaled once per
// (row, group) in fp32 with no per-element multiply. The lane keeps groups 2c and 2c+1 of its
// gate row and of its up row in accg / accu.
__device__ __forceinline__ void fp4_token_superseg(const uint4& qg, const uint4& qu, const uint2& fg,
                                                   const uint2& fu, const uint4 (&xh)[4], int c,
                                                   int sf_shift, float& accg, float& accu) {
    const uint32_t wgq[4] = {qg.x, qg.y, qg.z, qg.w};
    const uint32_t wuq[4] = {qu.x, qu.y, qu.z, qu.w};
    float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // one chain per half
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t ga[8], ua[8];
        e2m1x8_to_f16x2x4(wgq[2 * h], ga[0], ga[1], ga[2], ga[3]);
        e2m1x8_to_f16x2x4(wgq[2 * h + 1], ga[4], ga[5], ga[6], ga[7]);
        e2m1x8_to_f16x2x4(wuq[2 * h], ua[0], ua[1], ua[2], ua[3]);
        e2m1x8_to_f16x2x4(wuq[2 * h + 1], ua[4], ua[5], ua[6], ua[7]);
        const uint4 b0 = xh[2 * h], b1 = xh[2 * h + 1];
        float (&dh)[4] = d[h];                 // half h only feeds the columns 2c' + h
        mma_f16(dh, ga[0], ua[0], ga[1], ua[1], b0.x, b0.y);
        mma_f16(dh, ga[2], ua[2], ga[3], ua[3], b0.z, b0.w);
        mma_f16(dh, ga[4], ua[4], ga[5], ua[5], b1.x, b1.y);
        mma_f16(dh, ga[6], ua[6], ga[7], ua[7], b1.z, b1.w);
    }
    // the scales of groups 2c and 2c+1 of the gate row and of the up row
    const uint32_t sg = e4m3x2_to_f16x2(((c >> 1) ? fg.y : fg.x) >> sf_shift);
    const uint32_t su = e4m3x2_to_f16x2(((c >> 1) ? fu.y : fu.x) >> sf_shift);
    const float2 sgf = __half22float2(*reinterpret_cast<const __half2*>(&sg));
    const float2 suf = __half22float2(*reinterpret_cast<const __half2*>(&su));
    accg = fmaf(d[0][0], sgf.x, accg);
    accg = fmaf(d[1][1], sgf.y, accg);
    accu = fmaf(d[0][2], suf.x, accu);
    accu = fmaf(d[1][3], suf.y, accu);
}

// Dynamic shared memory of the items: x staging [max_cols][H] f16, y rows [P][16] fp32.
__host__ __device__ inline size_t gate_up_item_smem(int H, int max_cols) {
    return static_cast<size_t>(max_cols) * H * sizeof(__half);
}
__host__ __device__ inline size_t down_item_smem(int rows, int topk) {
    return static_cast<size_t>(rows) * topk * kDownRows * sizeof(float);
}

// ---- gate + up + SwiGLU for (group gv, feature block fb) --------------------------------------
// kToken1: compile the single-token NVFP4 loop (the stage kernel; the fused batch kernel leaves it
// out to stay within its register budget and runs one-column groups on the general loop).
template <int FMT, int kSF8 = kStagesFp8, int kSF4 = kStagesFp4, bool kToken1 = true>
__device__ void gate_up_item(const GateUpArgs& a, const GroupView& gv, int fb, __half* xs,
                             GateUpShared& sh) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int H = a.H, I = a.I;
    const int e = gv.e, ncols = gv.ncols;
    const int topk = a.grp.topk;
    const int n = fb * kFeatBlock + warp * 8 + g;       // this lane's gate / up row in the block

    if (tid < 2) sh.zeros[tid] = make_uint4(0, 0, 0, 0);   // visible after the staging barriers

    // ---- stage the columns' activations as f16 with a per-column power-of-two scale ----
    {
        const int nv = H / 8;                       // 16-byte vectors of 8 bf16
        float m[kMaxCols];
#pragma unroll
        for (int j = 0; j < kMaxCols; ++j) m[j] = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxCols; ++j) {
            if (j < ncols) {
                const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(gv.pair[j] / topk) * H);
                float mj = 0.0f;
                for (int v = tid; v < nv; v += kItemThreads) {
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
            if (lane == 0) sh.red[warp][j] = r;
        }
        __syncthreads();
        if (tid < ncols) {
            float mm = 0.0f;
            for (int w = 0; w < kItemWarps; ++w) mm = fmaxf(mm, sh.red[w][tid]);
            float inv;
            sh.a_scale[tid] = pow2_range_scale(mm, inv);
            sh.x_inv[tid] = inv;
        }
        __syncthreads();
        for (int j = 0; j < ncols; ++j) {
            const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(gv.pair[j] / topk) * H);
            const float s = sh.a_scale[j];
            uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<size_t>(j) * H);
            for (int v = tid; v < nv; v += kItemThreads) {
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
    const bool has_b = g < ncols;
    const __half* xb = xs + static_cast<size_t>(has_b ? g : 0) * H + c * 16;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};   // gate(col 2c), gate(col 2c+1), up(2c), up(2c+1)

    if constexpr (FMT == 0) {
        const size_t row = static_cast<size_t>(e) * I + n;
        const uint8_t* pg = a.wg + row * H + c * 16;
        const uint8_t* pu = a.wu + row * H + c * 16;
        const int nkb = H / 128;
        const size_t srow = (static_cast<size_t>(e) * (I / 128) + (fb * kFeatBlock) / 128) * (H / 128);
        const float* sgr = a.sg + srow;
        const float* sur = a.su + srow;
        for (int kb0 = 0; kb0 < nkb; kb0 += kSF8) {
            uint4 q[kSF8][4];
#pragma unroll
            for (int s = 0; s < kSF8; ++s) {
                if (kb0 + s < nkb) {
                    const size_t off = static_cast<size_t>(kb0 + s) * 128;
                    q[s][0] = ld_stream_v4(pg + off);
                    q[s][1] = ld_stream_v4(pu + off);
                    q[s][2] = ld_stream_v4(pg + off + 64);
                    q[s][3] = ld_stream_v4(pu + off + 64);
                }
            }
#pragma unroll
            for (int s = 0; s < kSF8; ++s) {
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
        // NVFP4: the per-16 scale bytes fold into A, so nothing needs the 64-wide K interleave of
        // the FP8 path. A lane streams 16 bytes (32 codes) of each row per 128-wide super-segment
        // t: elements 128t + 32c .. +31, i.e. MMA step i (0..7) takes elements 4i..4i+3 of those;
        // B is read at the same physical positions. The row's 8 scale bytes of a super-segment
        // come in one 8-byte load shared by the row's 4 lanes; lane c uses bytes 2c and 2c+1.
        const size_t row = static_cast<size_t>(e) * I + n;
        const uint8_t* pg = a.wg + row * (H / 2) + c * 16;
        const uint8_t* pu = a.wu + row * (H / 2) + c * 16;
        const uint8_t* fgp = a.sfg + row * (H / 16);
        const uint8_t* fup = a.sfu + row * (H / 16);
        const __half* xb4 = xs + static_cast<size_t>(has_b ? g : 0) * H + c * 32;
        const int nsup = H / 128;
        const int sf_shift = 16 * (c & 1);
        if (kToken1 && ncols == 1) {
            // one token: fp4_token_superseg per super-segment, the 4 lanes of a row summed at the end
            const int act = (g >> 1) == c ? (g & 1) : -1;   // the half whose x this lane carries
            const __half* xr = xs + c * 32;                   // the token row, lane c's positions
            // every lane loads its B pair of each half, branch-free: x where it carries that
            // half, else the zero pair (stride 0)
            const uint4* xp0 = act == 0 ? reinterpret_cast<const uint4*>(xr) : sh.zeros;
            const uint4* xp1 = act == 1 ? reinterpret_cast<const uint4*>(xr) + 2 : sh.zeros;
            const int xst0 = act == 0 ? 16 : 0, xst1 = act == 1 ? 16 : 0;
            float accg = 0.0f, accu = 0.0f;
            for (int t0 = 0; t0 < nsup; t0 += kSF4) {
                uint4 qg[kSF4], qu[kSF4];
                uint2 fg[kSF4], fu[kSF4];
#pragma unroll
                for (int s = 0; s < kSF4; ++s) {
                    if (t0 + s < nsup) {
                        qg[s] = ld_stream_v4(pg + (t0 + s) * 64);
                        qu[s] = ld_stream_v4(pu + (t0 + s) * 64);
                        fg[s] = ld_stream_v2(fgp + (t0 + s) * 8);
                        fu[s] = ld_stream_v2(fup + (t0 + s) * 8);
                    }
                }
#pragma unroll
                for (int s = 0; s < kSF4; ++s) {
                    const int t = t0 + s;
                    if (t < nsup) {
                        const uint4 xh[4] = {xp0[t * xst0], xp0[t * xst0 + 1], xp1[t * xst1],
                                             xp1[t * xst1 + 1]};
                        fp4_token_superseg(qg[s], qu[s], fg[s], fu[s], xh, c, sf_shift, accg, accu);
                    }
                }
            }
            accg += __shfl_xor_sync(0xffffffffu, accg, 1);
            accg += __shfl_xor_sync(0xffffffffu, accg, 2);
            accu += __shfl_xor_sync(0xffffffffu, accu, 1);
            accu += __shfl_xor_sync(0xffffffffu, accu, 2);
            acc[0] = c == 0 ? accg : 0.0f;                    // column 0 = the token
            acc[2] = c == 0 ? accu : 0.0f;
        } else
        for (int t0 = 0; t0 < nsup; t0 += kSF4) {
            uint4 qg[kSF4], qu[kSF4];
            uint2 fg[kSF4], fu[kSF4];
#pragma unroll
            for (int s = 0; s < kSF4; ++s) {
                if (t0 + s < nsup) {
                    qg[s] = ld_stream_v4(pg + (t0 + s) * 64);
                    qu[s] = ld_stream_v4(pu + (t0 + s) * 64);
                    fg[s] = ld_stream_v2(fgp + (t0 + s) * 8);
                    fu[s] = ld_stream_v2(fup + (t0 + s) * 8);
                }
            }
#pragma unroll
            for (int s = 0; s < kSF4; ++s) {
                const int t = t0 + s;
                if (t < nsup) {
                    uint4 bq[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                                   make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
                    if (has_b) {
                        const uint4* bp = reinterpret_cast<const uint4*>(xb4 + t * 128);
#pragma unroll
                        for (int j = 0; j < 4; ++j) bq[j] = bp[j];
                    }
                    const uint32_t sgw = ((c >> 1) ? fg[s].y : fg[s].x) >> sf_shift;
                    const uint32_t suw = ((c >> 1) ? fu[s].y : fu[s].x) >> sf_shift;
                    const uint32_t wgq[4] = {qg[s].x, qg[s].y, qg[s].z, qg[s].w};
                    const uint32_t wuq[4] = {qu[s].x, qu[s].y, qu[s].z, qu[s].w};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {          // elements 16h .. 16h+15 of the lane's 32
                        const uint32_t sg2 = e4m3_splat_f16x2((sgw >> (8 * h)) & 0xFFu);
                        const uint32_t su2 = e4m3_splat_f16x2((suw >> (8 * h)) & 0xFFu);
                        uint32_t ga[8], ua[8];
                        e2m1x8_to_f16x2x4(wgq[2 * h], ga[0], ga[1], ga[2], ga[3]);
                        e2m1x8_to_f16x2x4(wgq[2 * h + 1], ga[4], ga[5], ga[6], ga[7]);
                        e2m1x8_to_f16x2x4(wuq[2 * h], ua[0], ua[1], ua[2], ua[3]);
                        e2m1x8_to_f16x2x4(wuq[2 * h + 1], ua[4], ua[5], ua[6], ua[7]);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            ga[j] = hmul2(ga[j], sg2);
                            ua[j] = hmul2(ua[j], su2);
                        }
                        const uint4 b0 = bq[2 * h], b1 = bq[2 * h + 1];
                        mma_f16(acc, ga[0], ua[0], ga[1], ua[1], b0.x, b0.y);
                        mma_f16(acc, ga[2], ua[2], ga[3], ua[3], b0.z, b0.w);
                        mma_f16(acc, ga[4], ua[4], ga[5], ua[5], b1.x, b1.y);
                        mma_f16(acc, ga[6], ua[6], ga[7], ua[7], b1.z, b1.w);
                    }
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
            float gv_ = acc[j] * sh.x_inv[col], uv = acc[2 + j] * sh.x_inv[col];
            if constexpr (FMT == 1) {
                gv_ *= scale2_of(a.s2g, a.s2g_e, a.s2_stride, e);
                uv *= scale2_of(a.s2u, a.s2u_e, a.s2_stride, e);
            }
            hv[j] = clamped_swiglu(gv_, uv, a.limit);
        }
    }
    float m0 = fabsf(hv[0]), m1 = fabsf(hv[1]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    __syncthreads();                       // the staging reads of sh.red are long done
    if (g == 0) {
        sh.red[warp][2 * c] = m0;
        sh.red[warp][2 * c + 1] = m1;
    }
    __syncthreads();
    if (tid < ncols) {
        float mm = 0.0f;
        for (int w = 0; w < kItemWarps; ++w) mm = fmaxf(mm, sh.red[w][tid]);
        float inv;
        sh.a_scale[tid] = pow2_range_scale(mm, inv);
        a.act_scale[static_cast<size_t>(gv.pair[tid]) * (I / kFeatBlock) + fb] = inv;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int col = 2 * c + j;
        if (col < ncols)
            a.act[static_cast<size_t>(gv.pair[col]) * I + n] = __float2half_rn(hv[j] * sh.a_scale[col]);
    }
}

// ---- down + combine for output rows jt*16 .. jt*16+15 ------------------------------------------
// The activation a and its scales are read with plain (coherent) loads, never the read-only path:
// in the fused kernel they were written by other CTAs of the same grid before a grid barrier
// whose acquire fence makes those writes visible.
// With kWaitDeps (the stage kernel launched as a programmatic dependent of the gate/up kernel),
// each thread issues its first weight batch BEFORE waiting for the gate/up grid, so the down
// weight stream starts while the gate/up kernel drains.
template <int FMT, bool kWaitDeps = false, int kStages = kDownBatch>
__device__ void down_item(const DownArgs& a, const GroupList& gl, int jt, float* ys) {
    bool waited = false;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int H = a.H, I = a.I;
    const int j0 = jt * kDownRows;
    const int nseg = I / 64;

    for (int gi = warp; gi < gl.count; gi += kItemWarps) {
        const GroupView& gv = gl.g[gi];
        const int e = gv.e, ncols = gv.ncols;
        const bool has_b = g < ncols;
        const int pb = has_b ? gv.pair[g] : 0;
        const int col0 = 2 * c, col1 = 2 * c + 1;
        const int p0 = col0 < ncols ? gv.pair[col0] : -1;
        const int p1 = col1 < ncols ? gv.pair[col1] : -1;
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
                if (kWaitDeps && !waited) {
                    pdl_wait();
                    waited = true;
                }
#pragma unroll
                for (int s = 0; s < kStages; ++s) {
                    const int seg = s0 + s;
                    if (seg < nseg) {
                        uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
                        if (has_b) {
                            const uint4* bp = reinterpret_cast<const uint4*>(hb + seg * 64);
                            b0 = bp[0];
                            b1 = bp[1];
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
                        const float f0 = p0 >= 0 ? wsc * hs0[seg] : 0.0f;
                        const float f1 = p1 >= 0 ? wsc * hs1[seg] : 0.0f;
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
            // the row's scale bytes of two segments come in one 8-byte load shared by its 4 lanes
            const uint8_t* fa0 = a.sfd + r0 * (I / 16);
            const uint8_t* fa1 = fa0 + static_cast<size_t>(8) * (I / 16);
            constexpr int kS = 2 * kStages;
            for (int s0 = 0; s0 < nseg; s0 += kS) {
                uint2 qa[kS], qb[kS];
                uint2 fa2[kS / 2], fb2[kS / 2];
#pragma unroll
                for (int s = 0; s < kS; ++s) {
                    if (s0 + s < nseg) {
                        qa[s] = ld_stream_v2(pa0 + (s0 + s) * 32);
                        qb[s] = ld_stream_v2(pa1 + (s0 + s) * 32);
                    }
                }
#pragma unroll
                for (int s = 0; s < kS; s += 2) {
                    if (s0 + s < nseg) {
                        fa2[s / 2] = ld_stream_v2(fa0 + (s0 + s) * 4);
                        fb2[s / 2] = ld_stream_v2(fa1 + (s0 + s) * 4);
                    }
                }
                if (kWaitDeps && !waited) {
                    pdl_wait();
                    waited = true;
                }
#pragma unroll
                for (int s = 0; s < kS; ++s) {
                    const int seg = s0 + s;
                    if (seg < nseg) {
                        uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
                        if (has_b) {
                            const uint4* bp = reinterpret_cast<const uint4*>(hb + seg * 64);
                            b0 = bp[0];
                            b1 = bp[1];
                        }
                        const uint32_t wa_ = (s & 1) ? fa2[s / 2].y : fa2[s / 2].x;
                        const uint32_t wb_ = (s & 1) ? fb2[s / 2].y : fb2[s / 2].x;
                        const uint32_t sa = e4m3_splat_f16x2((wa_ >> (8 * c)) & 0xFFu);
                        const uint32_t sb = e4m3_splat_f16x2((wb_ >> (8 * c)) & 0xFFu);
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
                        const float f0 = p0 >= 0 ? hs0[seg] : 0.0f;
                        const float f1 = p1 >= 0 ? hs1[seg] : 0.0f;
                        acc[0] = fmaf(d[0], f0, acc[0]);
                        acc[1] = fmaf(d[1], f1, acc[1]);
                        acc[2] = fmaf(d[2], f0, acc[2]);
                        acc[3] = fmaf(d[3], f1, acc[3]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] *= scale2_of(a.s2d, a.s2d_e, a.s2_stride, e);
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
    if (kWaitDeps && !waited) pdl_wait();
    __syncthreads();

    // slot-order combine: one thread per (token, row); a separate rounded multiply and add per
    // term, so the order and the roundings are fixed
    for (int i = tid; i < a.T * kDownRows; i += kItemThreads) {
        const int t = i / kDownRows, r = i % kDownRows;
        float s = 0.0f;
        for (int k = 0; k < a.topk; ++k) {
            const int p = t * a.topk + k;
            const int e = a.ids[p];
            if (e < 0 || e >= a.E) continue;
            s = __fadd_rn(s, __fmul_rn(a.wts[p], ys[p * kDownRows + r]));
        }
        const size_t o = static_cast<size_t>(t) * H + j0 + r;
        if (a.shared != nullptr) s = __fadd_rn(s, __bfloat162float(a.shared[o]));
        if (a.residual != nullptr) s = __fadd_rn(s, __bfloat162float(a.residual[o]));
        a.out[o] = __float2bfloat16_rn(s);
    }
}

// ---- group lists --------------------------------------------------------------------------------

// From the stage-kernel group description (implicit T == 1 slots, or the plan kernel's table).
// Called by all threads; ends with a barrier.
__device__ inline void load_group_list(const Groups& G, GroupList& gl) {
    if (threadIdx.x == 0) {
        int n = 0;
        if (G.count == nullptr) {
            for (int k = 0; k < G.topk; ++k) {
                const int e = G.ids[k];
                if (e < 0 || e >= G.E) continue;
                gl.g[n].e = e;
                gl.g[n].ncols = 1;
                gl.g[n].pair[0] = k;
                ++n;
            }
        } else {
            n = *G.count;
            for (int i = 0; i < n; ++i) {
                gl.g[i].e = G.expert[i];
                gl.g[i].ncols = G.ncols[i];
                for (int j = 0; j < G.ncols[i]; ++j) gl.g[i].pair[j] = G.sorted_pair[G.start[i] + j];
            }
        }
        gl.count = n;
    }
    __syncthreads();
}

// Group the P <= 64 routed pairs of a sub-batch by expert inside one CTA (ascending expert, then
// ascending pair; at most `cap` columns per group) - the same grouping the plan kernel builds,
// computed redundantly by every CTA of the fused kernel instead of by a separate launch.
// Returns true if an id outside [-1, E) was seen. Called by all threads; ends with a barrier.
__device__ inline bool plan_groups_in_cta(const int32_t* ids, int P, int E, int cap, GroupList& gl) {
    constexpr int kNone = 0x7fffffff;
    __shared__ int key[kMaxPairs];     // e * 64 + pair, kNone if the pair is not routed
    __shared__ int rnk[kMaxPairs];     // rank of the pair among its expert's pairs
    __shared__ int cnt[kMaxPairs];     // number of pairs of its expert
    __shared__ int bad;
    const int tid = threadIdx.x;
    if (tid == 0) bad = 0;
    __syncthreads();
    if (tid < P) {
        const int e = ids[tid];
        const bool valid = e >= 0 && e < E;
        key[tid] = valid ? e * kMaxPairs + tid : kNone;
        if (!valid && e != -1) bad = 1;
    }
    __syncthreads();
    if (tid < P) {
        const int mine = key[tid];
        int r = 0, n = 0;
        if (mine != kNone) {
            const int e = mine / kMaxPairs;
            for (int q = 0; q < P; ++q) {
                const int k = key[q];
                if (k != kNone && k / kMaxPairs == e) {
                    ++n;
                    if (k < mine) ++r;
                }
            }
        }
        rnk[tid] = r;
        cnt[tid] = n;
    }
    __syncthreads();
    if (tid < P && key[tid] != kNone) {
        const int e = key[tid] / kMaxPairs;
        int groups_before = 0;             // groups of the experts below e
        for (int q = 0; q < P; ++q)
            if (key[q] != kNone && rnk[q] == 0 && key[q] / kMaxPairs < e)
                groups_before += (cnt[q] + cap - 1) / cap;
        const int gi = groups_before + rnk[tid] / cap;
        const int col = rnk[tid] % cap;
        gl.g[gi].pair[col] = tid;
        if (col == 0) {
            gl.g[gi].e = e;
            const int left = cnt[tid] - (rnk[tid] / cap) * cap;
            gl.g[gi].ncols = left < cap ? left : cap;
        }
    }
    if (tid == 0) {
        int n = 0;
        for (int q = 0; q < P; ++q)
            if (key[q] != kNone && rnk[q] == 0) n += (cnt[q] + cap - 1) / cap;
        gl.count = n;
    }
    __syncthreads();
    return bad != 0;
}

}  // namespace moe
