// Single-token (T = 1) NVFP4 decode: gate/up + clamped SwiGLU, then down + slot-order combine,
// both written for the fewest instructions per weight byte, since at one token these GEMVs are
// paced by instruction issue, not by bytes in flight.
//
// Both kernels use the single-token super-segment product: a lane streams 16 bytes (32 E2M1
// codes, scale groups 2c and 2c + 1 of a 128-wide super-segment) of each of its two weight rows
// and the MMA's 8 B columns carry the super-segment's 8 scale groups instead of tokens (column n
// holds the token's values on group n and zeros elsewhere), so D[row][n] is the row's partial dot
// product over group n, scaled once per (row, group) in fp32 - no per-element scale multiply.
// Per lane and super-segment: two 16-byte code loads, two 16-bit scale loads (the lane's own two
// groups), 32 code conversions, 8 MMAs (two independent chains), the scales; addresses advance by
// constant strides and full load batches run without bounds checks.
//
//   gate/up: rows g / g + 8 of the MMA tile are gate row n / up row n; B is x (f16 in shared
//            memory with a power-of-two scale); writes a as f16 with one power-of-two scale per
//            kFp4TokFeat-feature block (one block per CTA; the down kernel below reads them).
//   down:    rows g / g + 8 are output rows j0 + g / j0 + g + 8 of the slot's expert; B is the
//            slot's activation a; the group scale also carries a's inverse block scale (a lane's
//            two groups, 32 consecutive features, lie in one block).
//
// Sources: "memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs", `reference_expert` (gate, up,
// SwiGLU, down) and `combine_down_rows_host` (slot order, separate rounded multiply and add);
// "memra-engine 0.131.0 src/dsv4_ep.rs", `chain` (NVFP4 strides: codes K/2, scale bytes K/16
// per row); "spark_model layers/glm5next_mlp/forward.rs", `w4a16_gemv` (scale_2 by value) and
// `swiglu_rows` (the asymmetric clamp).
#include "gemv_items.cuh"

#ifndef MOE_FP4T_GU_BATCH
#define MOE_FP4T_GU_BATCH 4
#endif
#ifndef MOE_FP4T_DN_BATCH
#define MOE_FP4T_DN_BATCH 2
#endif

namespace moe {

namespace {

constexpr int kGuB = MOE_FP4T_GU_BATCH;     // super-segments per load batch, gate/up
constexpr int kGuWarps = kFp4TokFeat / 8;   // gate/up warps per CTA: 8 features (gate + up rows) each
constexpr int kGuThreads = 32 * kGuWarps;
constexpr int kGuMinBlocks = 2 * kItemThreads / kGuThreads;   // 128 registers per thread
constexpr int kDnB = MOE_FP4T_DN_BATCH;     // the same, down

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p) {
    uint16_t v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// One super-segment for lane (g, c): row-A codes qa, row-B codes qb (16 bytes each), the B
// fragments of the two halves (x0: the lane's half-0 values or zeros, x1: half 1), and the four
// f16->f32 scales of groups 2c, 2c + 1 of rows A and B; adds the scaled group sums to accA / accB.
__device__ __forceinline__ void fp4_superseg(const uint4& qa, const uint4& qb, const uint4 (&x0)[2],
                                             const uint4 (&x1)[2], float2 sa, float2 sb, float& accA,
                                             float& accB) {
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
    float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // one MMA chain per half
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t ra[8], rb[8];
        e2m1x8_to_f16x2x4(wa[2 * h], ra[0], ra[1], ra[2], ra[3]);
        e2m1x8_to_f16x2x4(wa[2 * h + 1], ra[4], ra[5], ra[6], ra[7]);
        e2m1x8_to_f16x2x4(wb[2 * h], rb[0], rb[1], rb[2], rb[3]);
        e2m1x8_to_f16x2x4(wb[2 * h + 1], rb[4], rb[5], rb[6], rb[7]);
        const uint4 b0 = h == 0 ? x0[0] : x1[0], b1 = h == 0 ? x0[1] : x1[1];
        mma_f16(d[h], ra[0], rb[0], ra[1], rb[1], b0.x, b0.y);
        mma_f16(d[h], ra[2], rb[2], ra[3], rb[3], b0.z, b0.w);
        mma_f16(d[h], ra[4], rb[4], ra[5], rb[5], b1.x, b1.y);
        mma_f16(d[h], ra[6], rb[6], ra[7], rb[7], b1.z, b1.w);
    }
    // column 2c (group 2c) lives in chain 0, column 2c + 1 in chain 1
    accA = fmaf(d[0][0], sa.x, accA);
    accA = fmaf(d[1][1], sa.y, accA);
    accB = fmaf(d[0][2], sb.x, accB);
    accB = fmaf(d[1][3], sb.y, accB);
}

__device__ __forceinline__ float2 e4m3x2_f32(uint32_t two_bytes) {
    const uint32_t h = e4m3x2_to_f16x2(two_bytes);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// ---- gate/up ------------------------------------------------------------------------------------

// grid (I / kFp4TokFeat, topk), kGuWarps warps: warp w computes features fb*kFp4TokFeat + 8w .. +7
// of slot blockIdx.y.
__global__ void __launch_bounds__(kGuThreads, kGuMinBlocks) fp4_token_gate_up_kernel(const GateUpArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];    // x as f16 [H]
    __shared__ GateUpShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int H = a.H, I = a.I, slot = blockIdx.y, fb = blockIdx.x;
    const int e = a.grp.ids[slot];                          // the same word for every thread
    pdl_launch_dependents();                                // the down kernel may start its stream
    if (e < 0 || e >= a.grp.E) {
        if (e != -1 && fb == 0 && tid == 0 && a.err != nullptr) atomicOr(a.err, 1);
        return;
    }
    const int n = fb * kFp4TokFeat + warp * 8 + g;
    const size_t row = static_cast<size_t>(e) * I + n;
    const uint8_t* pg = a.wg + row * (H / 2) + c * 16;     // codes: 64 bytes per super-segment
    const uint8_t* pu = a.wu + row * (H / 2) + c * 16;
    const uint8_t* fg = a.sfg + row * (H / 16) + 2 * c;    // the lane's two scale bytes, 8 per super-segment
    const uint8_t* fu = a.sfu + row * (H / 16) + 2 * c;
    const int nsup = H / 128;

    // the first batch of weights is in flight while x is staged
    uint4 qg[kGuB], qu[kGuB];
    uint32_t sg[kGuB], su[kGuB];
    const int first = nsup < kGuB ? nsup : kGuB;
#pragma unroll
    for (int s = 0; s < kGuB; ++s)
        if (s < first) {
            qg[s] = ld_stream_v4(pg + s * 64);
            qu[s] = ld_stream_v4(pu + s * 64);
            sg[s] = ld_stream_u16(fg + s * 8);
            su[s] = ld_stream_u16(fu + s * 8);
        }

    // ---- x as f16 with a power-of-two range scale ----
    __half* xs = reinterpret_cast<__half*>(smem_raw);
    {
        const int nv = H / 8;
        const uint4* xr = reinterpret_cast<const uint4*>(a.x);
        float m = 0.0f;
        for (int v = tid; v < nv; v += kGuThreads) {
            const uint4 q = __ldg(xr + v);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
                m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
            }
        }
        m = warp_max(m);
        if (lane == 0) sh.red[warp][0] = m;
        if (tid < 2) sh.zeros[tid] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        if (tid == 0) {
            float mm = 0.0f;
            for (int w = 0; w < kGuWarps; ++w) mm = fmaxf(mm, sh.red[w][0]);
            float inv;
            sh.a_scale[0] = pow2_range_scale(mm, inv);
            sh.x_inv[0] = inv;
        }
        __syncthreads();
        const float s = sh.a_scale[0];
        for (int v = tid; v < nv; v += kGuThreads) {
            const uint4 q = __ldg(xr + v);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half2 h2 = __floats2half2_rn(__uint_as_float(w[i] << 16) * s,
                                                     __uint_as_float(w[i] & 0xFFFF0000u) * s);
                o[i] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            reinterpret_cast<uint4*>(xs)[v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        __syncthreads();
    }

    // B fragments: lane (g, c) carries x only in column 2c + h of half h, i.e. when g == 2c + h;
    // every other lane reads the zero pair (stride 0)
    const int hx = g - 2 * c;                                // the half this lane carries, if 0 or 1
    const uint4* xp0 = hx == 0 ? reinterpret_cast<const uint4*>(xs + c * 32) : sh.zeros;
    const uint4* xp1 = hx == 1 ? reinterpret_cast<const uint4*>(xs + c * 32 + 16) : sh.zeros;
    const int xs0 = hx == 0 ? 16 : 0, xs1 = hx == 1 ? 16 : 0; // uint4 per super-segment
    float accg = 0.0f, accu = 0.0f;
    auto compute = [&](int s) {
        const uint4 x0[2] = {xp0[0], xp0[1]}, x1[2] = {xp1[0], xp1[1]};
        xp0 += xs0;
        xp1 += xs1;
        fp4_superseg(qg[s], qu[s], x0, x1, e4m3x2_f32(sg[s]), e4m3x2_f32(su[s]), accg, accu);
    };
    int t = first;
    if (first == kGuB) {
        for (; t + kGuB <= nsup; t += kGuB) {                // full batches: no bounds checks
#pragma unroll
            for (int s = 0; s < kGuB; ++s) compute(s);
            pg += kGuB * 64;
            pu += kGuB * 64;
            fg += kGuB * 8;
            fu += kGuB * 8;
#pragma unroll
            for (int s = 0; s < kGuB; ++s) {
                qg[s] = ld_stream_v4(pg + s * 64);
                qu[s] = ld_stream_v4(pu + s * 64);
                sg[s] = ld_stream_u16(fg + s * 8);
                su[s] = ld_stream_u16(fu + s * 8);
            }
        }
#pragma unroll
        for (int s = 0; s < kGuB; ++s) compute(s);
        pg += kGuB * 64;
        pu += kGuB * 64;
        fg += kGuB * 8;
        fu += kGuB * 8;
        for (; t < nsup; ++t) {                              // the ragged tail, one at a time
            qg[0] = ld_stream_v4(pg);
            qu[0] = ld_stream_v4(pu);
            sg[0] = ld_stream_u16(fg);
            su[0] = ld_stream_u16(fu);
            compute(0);
            pg += 64;
            pu += 64;
            fg += 8;
            fu += 8;
        }
    } else {
#pragma unroll
        for (int s = 0; s < kGuB; ++s)
            if (s < first) compute(s);
    }
    // the four lanes of a row hold disjoint groups: sum them
    accg += __shfl_xor_sync(0xffffffffu, accg, 1);
    accg += __shfl_xor_sync(0xffffffffu, accg, 2);
    accu += __shfl_xor_sync(0xffffffffu, accu, 1);
    accu += __shfl_xor_sync(0xffffffffu, accu, 2);

    // ---- epilogue: scales, clamped SwiGLU, per-64-block range scale, f16 store ----
    float hv = 0.0f;
    if (c == 0) {
        const float gv = accg * sh.x_inv[0] * scale2_of(a.s2g, a.s2g_e, a.s2_stride, e),
                    uv = accu * sh.x_inv[0] * scale2_of(a.s2u, a.s2u_e, a.s2_stride, e);
        hv = clamped_swiglu(gv, uv, a.limit);
    }
    const float m = warp_max(fabsf(hv));
    if (lane == 0) sh.red[warp][1] = m;
    __syncthreads();
    float mm = 0.0f;
#pragma unroll
    for (int w = 0; w < kGuWarps; ++w) mm = fmaxf(mm, sh.red[w][1]);
    float inv;
    const float s_a = pow2_range_scale(mm, inv);
    if (tid == 0) a.act_scale[static_cast<size_t>(slot) * (I / kFp4TokFeat) + fb] = inv;
    if (c == 0) a.act[static_cast<size_t>(slot) * I + n] = __float2half_rn(hv * s_a);
}

// ---- down + combine -------------------------------------------------------------------------------

// grid H / 16, 8 warps: warp k = slot k, rows j0 + g and j0 + g + 8 of its expert's down matrix;
// then the slot-order combine of the 8 results per row. Launched as a programmatic dependent of
// the gate/up kernel: the first weight batch is issued before the wait for its activations.
__global__ void __launch_bounds__(kItemThreads, 3) fp4_token_down_kernel(const DownArgs a) {
    __shared__ float ys[kMaxTopk][kDownRows];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int H = a.H, I = a.I, j0 = blockIdx.x * kDownRows;
    const int k = warp;
    const int e = k < a.topk ? a.ids[k] : -1;
    const bool live = e >= 0 && e < a.E;
    const int nsup = I / 128;
    float accA = 0.0f, accB = 0.0f;                         // rows j0 + g, j0 + g + 8 (lane's groups)
    if (live) {
        const size_t r0 = static_cast<size_t>(e) * H + j0 + g;
        const uint8_t* pa = a.wd + r0 * (I / 2) + c * 16;
        const uint8_t* pb = pa + static_cast<size_t>(8) * (I / 2);
        const uint8_t* fa = a.sfd + r0 * (I / 16) + 2 * c;
        const uint8_t* fb_ = fa + static_cast<size_t>(8) * (I / 16);
        // the slot's activation: lane (g, c) carries half h = g - 2c of its 32 positions, if any
        const int hx = g - 2 * c;
        const bool carrier = hx == 0 || hx == 1;
        const __half* hb = a.act + static_cast<size_t>(k) * I + c * 32 + (hx == 1 ? 16 : 0);
        // the scale block of the lane's 32 features c*32 .. c*32+31 of each 128-wide super-segment
        const float* hs = a.act_scale + static_cast<size_t>(k) * (I / kFp4TokFeat) + (32 * c) / kFp4TokFeat;

        uint4 qa[kDnB], qb[kDnB], xa[kDnB][2];
        uint32_t sa[kDnB], sb[kDnB];
        float ai[kDnB];
        // the batch's activations and their scales: plain loads (written by the preceding grid,
        // visible after the dependency wait)
        auto load_x = [&](int cnt, int t0) {
#pragma unroll
            for (int s = 0; s < kDnB; ++s)
                if (s < cnt) {
                    xa[s][0] = xa[s][1] = make_uint4(0, 0, 0, 0);
                    if (carrier) {
                        xa[s][0] = *reinterpret_cast<const uint4*>(hb + (t0 + s) * 128);
                        xa[s][1] = *reinterpret_cast<const uint4*>(hb + (t0 + s) * 128 + 8);
                    }
                    ai[s] = hs[(128 / kFp4TokFeat) * (t0 + s)];   // a's scale of the lane's block
                }
        };
        auto load_w = [&](int cnt) {
#pragma unroll
            for (int s = 0; s < kDnB; ++s)
                if (s < cnt) {
                    qa[s] = ld_stream_v4(pa + s * 64);
                    qb[s] = ld_stream_v4(pb + s * 64);
                    sa[s] = ld_stream_u16(fa + s * 8);
                    sb[s] = ld_stream_u16(fb_ + s * 8);
                }
        };
        auto advance = [&](int cnt) {
            pa += cnt * 64;
            pb += cnt * 64;
            fa += cnt * 8;
            fb_ += cnt * 8;
        };
        // The lane's fragments go to half hx by bit masks, not by a branch: the MMAs are
        // warp-synchronous and every lane must execute the same instruction sequence.
        const uint32_t m0 = hx == 0 ? 0xffffffffu : 0u, m1 = hx == 1 ? 0xffffffffu : 0u;
        auto mask4 = [](const uint4& v, uint32_t m) { return make_uint4(v.x & m, v.y & m, v.z & m, v.w & m); };
        auto compute = [&](int s) {
            const uint4 x0[2] = {mask4(xa[s][0], m0), mask4(xa[s][1], m0)};
            const uint4 x1[2] = {mask4(xa[s][0], m1), mask4(xa[s][1], m1)};
            const float ainv = ai[s];
            float2 fa2 = e4m3x2_f32(sa[s]), fb2 = e4m3x2_f32(sb[s]);
            fa2.x *= ainv;
            fa2.y *= ainv;
            fb2.x *= ainv;
            fb2.y *= ainv;
            __syncwarp();                                      // converged after the carriers' loads
            fp4_superseg(qa[s], qb[s], x0, x1, fa2, fb2, accA, accB);
        };
        const int first = nsup < kDnB ? nsup : kDnB;
        load_w(first);
        pdl_wait();
        load_x(first, 0);
        int t = 0;
        if (first == kDnB) {
            for (; t + 2 * kDnB <= nsup; t += kDnB) {        // full batches: no bounds checks
#pragma unroll
                for (int s = 0; s < kDnB; ++s) compute(s);
                advance(kDnB);
                load_w(kDnB);
                load_x(kDnB, t + kDnB);
            }
#pragma unroll
            for (int s = 0; s < kDnB; ++s) compute(s);
            advance(kDnB);
            t += kDnB;
            for (; t < nsup; ++t) {
                load_w(1);
                load_x(1, t);
                compute(0);
                advance(1);
            }
        } else {
#pragma unroll
            for (int s = 0; s < kDnB; ++s)
                if (s < first) compute(s);
        }
    } else {
        pdl_wait();
    }
    accA += __shfl_xor_sync(0xffffffffu, accA, 1);
    accA += __shfl_xor_sync(0xffffffffu, accA, 2);
    accB += __shfl_xor_sync(0xffffffffu, accB, 1);
    accB += __shfl_xor_sync(0xffffffffu, accB, 2);
    if (c == 0 && k < a.topk) {
        const int ek = a.ids[k];                            // reloaded: not kept live through the loop
        const float s2 = ek >= 0 && ek < a.E ? scale2_of(a.s2d, a.s2d_e, a.s2_stride, ek) : 0.0f;
        ys[k][g] = accA * s2;
        ys[k][g + 8] = accB * s2;
    }
    __syncthreads();
    // slot-order combine: one thread per output row; a separate rounded multiply and add per term
    if (tid < kDownRows) {
        float s = 0.0f;
        for (int kk = 0; kk < a.topk; ++kk) {
            const int ek = a.ids[kk];
            if (ek < 0 || ek >= a.E) continue;
            s = __fadd_rn(s, __fmul_rn(a.wts[kk], ys[kk][tid]));
        }
        const size_t o = static_cast<size_t>(j0) + tid;
        if (a.shared != nullptr) s = __fadd_rn(s, __bfloat162float(a.shared[o]));
        if (a.residual != nullptr) s = __fadd_rn(s, __bfloat162float(a.residual[o]));
        a.out[o] = __float2bfloat16_rn(s);
    }
}

}  // namespace

cudaError_t launch_fp4_token_gate_up(const GateUpArgs& a, int topk, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(a.H) * sizeof(__half);
    if (smem > 48 * 1024) {
        const cudaError_t st = cudaFuncSetAttribute(fp4_token_gate_up_kernel,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    static_cast<int>(smem));
        if (st != cudaSuccess) return st;
    }
    fp4_token_gate_up_kernel<<<dim3(a.I / kFp4TokFeat, topk), kGuThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fp4_token_down(const DownArgs& a, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.H / kDownRows);
    cfg.blockDim = dim3(kItemThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t st = cudaLaunchKernelEx(&cfg, fp4_token_down_kernel, a);
    if (st != cudaSuccess) return st;
    return cudaGetLastError();
}

}  // namespace moe
