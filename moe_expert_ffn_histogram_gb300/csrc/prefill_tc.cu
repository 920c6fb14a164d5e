// tcgen05 core of the prefill grouped GEMMs: the same 128-row x 128-column tiles and the same
// device-built tile list as the mma.sync core in prefill.cu, with the accumulator in tensor memory.
//
// Per CTA (8 warps, persistent over tiles): every thread streams A (f16 activation rows) and the
// raw E4M3 weight rows of the next K slices into shared memory with cp.async, three slices ahead;
// for the current slice the threads dequantise the weight bytes to f16 (times the prescaled block
// scale) into the canonical no-swizzle K-major layout the tensor core reads, fence the async
// proxy, and one thread issues four tcgen05.mma (M=128, N=128, K=16, f16 x f16 -> f32 in TMEM)
// and commits them to the slice's mbarrier. The epilogue reads the accumulator with tcgen05.ld
// (warp w owns TMEM lanes 32*(w%4) .. +31) and applies the SwiGLU (gate/up) or the row scale
// (down) as the mma.sync core does.
//
// Canonical K-major layout without swizzle: an operand tile of R rows x 64 K halves is stored as
// 8-row x 16-byte core matrices, (r, k) at (r/8)*1024 + (k/8)*128 + (r%8)*16 + (k%8)*2 bytes; so
// the descriptor's leading-dimension offset (next core matrix along K) is 128 B and its
// stride-dimension offset (next 8-row group) is 1024 B.
//
// Every wait is bounded (about one second of SM clock); on a timeout the CTA sets bit 1 of the
// error word, stops issuing work, waits (bounded) for its MMAs, frees its TMEM and exits.
#include "prefill.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kTcStages = 4;
constexpr int kTcA = 128 * 64 * 2;            // A slice, canonical layout (16 KB)
constexpr int kTcB = 128 * 64 * 2;            // B slice as f16, canonical layout (16 KB)
constexpr int kTcRawRow = 64 + 16;            // raw E4M3 row pitch (padded: conflict-free reads)
constexpr int kTcRaw = 128 * kTcRawRow;       // raw B slice (10 KB)
constexpr int kTcStage = kTcA + kTcB + kTcRaw;
constexpr int kTcSmem = kTcStages * kTcStage + 1024;   // + alignment slack
constexpr uint32_t kTmemCols = 128;
constexpr int kErrBitTimeout = 2;

}  // namespace

template <int KIND>
__global__ void __launch_bounds__(prefill::kThreads, 1) prefill_tc_gemm_kernel(const PrefillGemmArgs p) {
    using namespace prefill;
    extern __shared__ uint8_t smem_dyn[];
    // 1024-byte aligned base for the operand slices
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ const __half* a_row[kBM];
    __shared__ float a_scale[kBM];
    __shared__ uint32_t w_scale[2][64];
    __shared__ float w_inv[2];
    __shared__ __align__(8) uint64_t mbar[kTcStages];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = p.K, KT = K / kBK, KB = K / 128;
    const int total = p.tiles[0] * p.n_tiles;

    if (tid == 0) {
        for (int s = 0; s < kTcStages; ++s) mbar_init(&mbar[s], 1);
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    auto stA = [&](int s) { return smem + s * kTcStage; };
    auto stB = [&](int s) { return smem + s * kTcStage + kTcA; };
    auto stRaw = [&](int s) { return smem + s * kTcStage + kTcA + kTcB; };

    uint32_t git = 0;                                  // slices processed by this CTA so far
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const int mt = tile / p.n_tiles, nt = tile % p.n_tiles;
        const int e = p.tile_e[mt], r0 = p.tile_r0[mt];
        const int rows = min(kBM, p.offsets[e + 1] - r0);

        tc_fence_before();
        __syncthreads();                               // previous epilogue's TMEM reads are done
        if (abort_s) break;
        if (tid < kBM) {
            const int r = r0 + min(tid, rows - 1);     // padded rows repeat the last valid row
            if (KIND == 0) {
                const int t = p.sorted_pair[r] / p.topk;
                a_row[tid] = p.a + static_cast<size_t>(t) * K;
                a_scale[tid] = p.a_inv[t];
            } else {
                a_row[tid] = p.a + static_cast<size_t>(r) * K;
                a_scale[tid] = p.a_inv[r];
            }
        }
        if (warp < 2) {                                // warp 0: gate / down scales, warp 1: up
            const int nb = KIND == 0 ? (nt * 64) / 128 : nt;
            const float* srow = ((KIND == 0 && warp == 1) ? p.s1 : p.s0) +
                                (static_cast<size_t>(e) * (p.wrows / 128) + nb) * KB;
            float m = 0.0f;
            for (int kb = lane; kb < KB; kb += 32) m = fmaxf(m, fabsf(srow[kb]));
            m = warp_max(m) * 448.0f;
            float inv;
            const float pre = pow2_range_scale(m, inv);
            for (int kb = lane; kb < KB; kb += 32) {
                const __half h = __float2half_rn(srow[kb] * pre);
                const uint16_t hb = *reinterpret_cast<const uint16_t*>(&h);
                w_scale[warp][kb] = static_cast<uint32_t>(hb) * 0x10001u;
            }
            if (lane == 0) w_inv[warp] = inv;
        }
        __syncthreads();

        // ---- loader: slice kt -> stage s (A rows in canonical layout, raw weight rows) ----
        auto load = [&](int kt, int s) {
            uint8_t* dA = stA(s);
            uint8_t* dR = stRaw(s);
#pragma unroll
            for (int i = 0; i < 4; ++i) {              // A: 128 rows x 8 chunks of 8 halves
                const int ch = tid + i * kThreads, r = ch & 127, q = ch >> 7;
                cp_async16(dA + (r >> 3) * 1024 + q * 128 + (r & 7) * 16, a_row[r] + kt * kBK + q * 8);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {              // raw B: 128 weight rows x 4 chunks of 16 B
                const int ch = tid + i * kThreads, n = ch & 127, q = ch >> 7;
                const uint8_t* src;
                if (KIND == 0)                         // rows 0..63 gate, 64..127 the same up rows
                    src = (n < 64 ? p.w0 : p.w1) +
                          (static_cast<size_t>(e) * p.wrows + nt * 64 + (n & 63)) * K;
                else
                    src = p.w0 + (static_cast<size_t>(e) * p.wrows + nt * kBN + n) * K;
                cp_async16(dR + n * kTcRawRow + q * 16, src + kt * kBK + q * 16);
            }
        };

#pragma unroll
        for (int s = 0; s < kTcStages - 1; ++s) {
            if (s < KT) load(s, (git + s) % kTcStages);
            cp_async_commit();
        }
        for (int kt = 0; kt < KT; ++kt) {
            const uint32_t g = git + kt, s = g % kTcStages;
            cp_async_wait<kTcStages - 2>();
            __syncthreads();
            if (abort_s) break;                        // uniform: written only after barrier B
            // dequantise this slice's weight bytes into the canonical f16 layout
            {
                const uint8_t* raw = stRaw(s);
                uint8_t* dB = stB(s);
                const int kb = (kt * kBK) / 128;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int it = tid + i * kThreads, n = it & 127, q = it >> 7;
                    const uint4 w = lds128(raw + n * kTcRawRow + q * 16);
                    const uint32_t sc = w_scale[(KIND == 0 && n >= 64) ? 1 : 0][kb];
                    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                    uint32_t h[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        e4m3x4_to_f16x2x2(wv[j], h[2 * j], h[2 * j + 1]);
                        h[2 * j] = hmul2(h[2 * j], sc);
                        h[2 * j + 1] = hmul2(h[2 * j + 1], sc);
                    }
                    uint8_t* d = dB + (n >> 3) * 1024 + (2 * q) * 128 + (n & 7) * 16;
                    *reinterpret_cast<uint4*>(d) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4*>(d + 128) = make_uint4(h[4], h[5], h[6], h[7]);
                }
            }
            fence_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t a0 = smem_u32(stA(s)), b0 = smem_u32(stB(s));
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    mma_issue(tmem, smem_desc(a0 + kk * 256, 128, 1024),
                              smem_desc(b0 + kk * 256, 128, 1024), (kt > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&mbar[s]);
            }
            if (kt > 0) {                              // the previous slice's MMAs are done
                const uint32_t gp = g - 1;
                if (!mbar_wait(&mbar[gp % kTcStages], (gp / kTcStages) & 1u)) abort_s = 1;
            }
            if (kt + kTcStages - 1 < KT) load(kt + kTcStages - 1, (g + kTcStages - 1) % kTcStages);
            cp_async_commit();
        }
        cp_async_wait<0>();
        {
            const uint32_t gl = git + KT - 1;
            if (!mbar_wait(&mbar[gl % kTcStages], (gl / kTcStages) & 1u)) abort_s = 1;
        }
        git += KT;
        __syncthreads();
        if (abort_s) break;
        tc_fence_after();

        // ---- epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (tile rows) ----
        const int row = 32 * (warp & 3) + lane;
        const int half = warp >> 2;
        const uint32_t trow = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        if (KIND == 0) {
            const float xs = a_scale[row];
            float m = 0.0f;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                float gv[16], uv[16];
                tmem_ld16(trow + 32 * half + 16 * b, gv);
                tmem_ld16(trow + 64 + 32 * half + 16 * b, uv);
                float hv[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    hv[j] = clamped_swiglu(gv[j] * xs * w_inv[0], uv[j] * xs * w_inv[1], p.limit);
                    m = fmaxf(m, fabsf(hv[j]));
                }
                if (row < rows) {
                    float4* dst = reinterpret_cast<float4*>(p.out + static_cast<size_t>(r0 + row) * p.out_ld +
                                                            nt * 64 + 32 * half + 16 * b);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        dst[j] = make_float4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]);
                }
            }
            if (row < rows) atomicMax(p.amax + r0 + row, __float_as_uint(m));
        } else {
            const float sc = a_scale[row] * w_inv[0];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                float v[16];
                tmem_ld16(trow + 64 * half + 16 * b, v);
                if (row < rows) {
                    float4* dst = reinterpret_cast<float4*>(p.out + static_cast<size_t>(r0 + row) * p.out_ld +
                                                            nt * kBN + 64 * half + 16 * b);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        dst[j] = make_float4(v[4 * j] * sc, v[4 * j + 1] * sc, v[4 * j + 2] * sc, v[4 * j + 3] * sc);
                }
            }
        }
    }

    // ---- teardown: report a timeout, then free TMEM (all MMAs were waited for above) ----
    tc_fence_before();
    __syncthreads();
    if (abort_s) {                                     // let any MMA still in flight finish
        if (tid == 0 && p.err != nullptr) atomicOr(p.err, kErrBitTimeout);
        const long long t0 = clock64();
        while (clock64() - t0 < (1ll << 22)) {
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

cudaError_t launch_prefill_gemm_tc(int kind, const PrefillGemmArgs& p, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t st;
    if ((st = cudaGetDevice(&dev)) != cudaSuccess) return st;
    if ((st = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return st;
    if (kind == 0) {
        if ((st = cudaFuncSetAttribute(prefill_tc_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kTcSmem)) != cudaSuccess)
            return st;
        prefill_tc_gemm_kernel<0><<<sms, prefill::kThreads, kTcSmem, stream>>>(p);
    } else {
        if ((st = cudaFuncSetAttribute(prefill_tc_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kTcSmem)) != cudaSuccess)
            return st;
        prefill_tc_gemm_kernel<1><<<sms, prefill::kThreads, kTcSmem, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace moe
