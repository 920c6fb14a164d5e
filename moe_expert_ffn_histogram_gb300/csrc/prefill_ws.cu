// Warp-specialised tcgen05 core of the prefill grouped GEMMs (the default core of the wide tier).
//
// Same tiles and tile list as prefill.cu, but every role runs decoupled, linked by mbarriers:
//   warps 0-3  producers  cp.async the next K slices of A (128 f16 activation rows, canonical
//                         K-major core-matrix layout) and of the raw E4M3 weight rows, three
//                         slices ahead; arrive on full[s] when their copies land;
//   warps 4-7  converters dequantise slice s's weight bytes to f16 (times the prescaled block
//                         scale, from tables each warp builds per tile) into the canonical layout,
//                         fence the async proxy, arrive conv[s];
//   warp 12    one thread issues the four M=128 x N=BN x K=16 tcgen05.mma of slice s into one of
//                         two TMEM accumulators, and commits them to empty[s] (stage reusable)
//                         and, after a tile's last slice, to acc_full[b];
//   warps 8-11 epilogue   read the finished accumulator with tcgen05.ld (warp w owns TMEM lanes
//                         32*(w%4) .. +31), apply the SwiGLU (gate/up) or the row scale (down),
//                         store, and arrive acc_empty[b] - while the MMAs of the next tile already
//                         run into the other accumulator.
// gate/up: BN = 256 (128 gate rows and the same 128 up rows of one 128-feature block).
// down:    BN = 256 output columns (128 when H is not a multiple of 256).
// Every wait is bounded (~1 s of SM clock); on a timeout the CTA records bit 1 in the error word,
// all roles leave their loops, and the CTA frees its TMEM and exits.
#include "prefill.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kWsStages = 3;
constexpr int kWsA = 128 * 64 * 2;           // A slice, canonical layout (16 KB)
constexpr int kWsRawRow = 64 + 16;           // raw E4M3 row pitch (padded: conflict-free reads)
constexpr int kProdThreads = 128, kConvThreads = 128, kEpiThreads = 128;
constexpr int kWsThreads = kProdThreads + kConvThreads + kEpiThreads + 32;   // + MMA warp
constexpr int kMmaWarp = 12;

template <int BN>
struct WsCfg {
    static constexpr int kRaw = BN * kWsRawRow;
    static constexpr int kB = BN * 64 * 2;
    static constexpr int kStage = kWsA + kRaw + kB;
    static constexpr int kSmem = kWsStages * kStage + 1024;   // + 1024 B alignment slack
    static constexpr uint32_t kTmemCols = 2 * BN;               // two fp32 accumulators
    static_assert(kStage % 1024 == 0 && (kWsA + kRaw) % 1024 == 0, "stage alignment");
};

}  // namespace

template <int KIND, int BN>
__global__ void __launch_bounds__(kWsThreads, 1) prefill_ws_gemm_kernel(const PrefillGemmArgs p) {
    using Cfg = WsCfg<BN>;
    constexpr int NS = kWsStages;
    constexpr uint32_t kIdescN = idesc_f16_f32<128, BN>();
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[NS], conv[NS], empty[NS], acc_full[2], acc_empty[2];
    __shared__ uint32_t w_scale[4][2][64];          // per converter warp: two scale tables
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = p.K, KT = K / 64, KB = K / 128;
    const int total = p.tiles[0] * p.n_tiles;
    auto stA = [&](uint32_t s) { return smem + s * Cfg::kStage; };
    auto stRaw = [&](uint32_t s) { return smem + s * Cfg::kStage + kWsA; };
    auto stB = [&](uint32_t s) { return smem + s * Cfg::kStage + kWsA + Cfg::kRaw; };

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], kProdThreads);
            mbar_init(&conv[s], kConvThreads);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiThreads);
        }
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (tid < kProdThreads) {
        // ---------------- producers ----------------
        // Lane l of warp w copies 16-byte chunk (l >> 3) (+4) of rows 8g + (l & 7): each warp
        // instruction reads whole 64-byte row segments (coalesced) and its eight-lane phases write
        // eight distinct shared-memory bank groups (conflict-free in both layouts).
        const int rr = tid & 7, cc = (tid >> 3) & 3, w = tid >> 5;
        uint32_t sc = 0;
        for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x) {
            int mt, nt;
            decode_tile(p, tile, mt, nt);
            const int e = p.tile_e[mt], r0 = p.tile_r0[mt];
            const int rows = min(128, p.offsets[e + 1] - r0);
            const __half* asrc[4];                            // A rows 8 * (4w + j) + rr
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = r0 + min(8 * (4 * w + j) + rr, rows - 1);   // padded rows repeat the last
                asrc[j] = (KIND == 0 ? p.a + static_cast<size_t>(p.sorted_pair[r] / p.topk) * K
                                     : p.a + static_cast<size_t>(r) * K) + cc * 8;
            }
            const uint8_t* bsrc[BN / 32];                     // weight rows 8 * (w + 4i) + rr
#pragma unroll
            for (int i = 0; i < BN / 32; ++i) {
                const int n = 8 * (w + 4 * i) + rr;
                if (KIND == 0)                                // rows 0..127 gate, 128..255 up
                    bsrc[i] = (n < 128 ? p.w0 : p.w1) + (static_cast<size_t>(e) * p.wrows + nt * 128 + (n & 127)) * K;
                else
                    bsrc[i] = p.w0 + (static_cast<size_t>(e) * p.wrows + nt * BN + n) * K;
                bsrc[i] += cc * 16;
            }
            for (int kt = 0; kt < KT; ++kt, ++sc) {
                const uint32_t s = sc % NS, u = sc / NS;
                if (u > 0 && !mbar_wait(&empty[s], (u - 1) & 1u)) {
                    abort_s = 1;
                    break;
                }
                uint8_t* dA = stA(s) + (4 * w) * 1024 + cc * 128 + rr * 16;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    cp_async16(dA + j * 1024, asrc[j] + kt * 64);
                    cp_async16(dA + j * 1024 + 512, asrc[j] + kt * 64 + 32);
                }
                uint8_t* dR = stRaw(s) + (8 * w + rr) * kWsRawRow + cc * 16;
#pragma unroll
                for (int i = 0; i < BN / 32; ++i) cp_async16(dR + i * 32 * kWsRawRow, bsrc[i] + kt * 64);
                cp_async_mbar_arrive(&full[s]);
            }
        }
        cp_async_wait<0>();
    } else if (tid < kProdThreads + kConvThreads) {
        // ---------------- converters ----------------
        // Each converter warp builds its own copy of the tile's scale tables, so the four warps
        // never wait on one another; a wait that times out is made warp-uniform before leaving.
        const int ct = tid - kProdThreads, cw = ct >> 5;
        uint32_t sc = 0;
        for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x) {
            int mt, nt;
            decode_tile(p, tile, mt, nt);
            const int e = p.tile_e[mt];
            __syncwarp();                                     // the old tables are no longer read
            const size_t sblk = static_cast<size_t>(e) * (p.wrows / 128);
            if (KIND == 0) {
                weight_prescale(p.s0 + (sblk + nt) * KB, KB, w_scale[cw][0]);
                weight_prescale(p.s1 + (sblk + nt) * KB, KB, w_scale[cw][1]);
            } else {
                // down tiles of 256 columns span two 128-row scale blocks: rows 128.. use the next
                const int nb = (nt * BN) / 128;
                weight_prescale(p.s0 + (sblk + nb) * KB, KB, w_scale[cw][0]);
                if (BN == 256) weight_prescale(p.s0 + (sblk + nb + 1) * KB, KB, w_scale[cw][1]);
            }
            __syncwarp();
            for (int kt = 0; kt < KT; ++kt, ++sc) {
                const uint32_t s = sc % NS, u = sc / NS;
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], u & 1u))) {
                    abort_s = 1;
                    break;
                }
                const int kb = kt >> 1;
#pragma unroll
                for (int j = 0; j < BN / 128; ++j) {
                    const int n = ct + 128 * j;
                    const uint32_t sc2 = w_scale[cw][(BN == 256 && j == 1) ? 1 : 0][kb];
                    const uint8_t* raw = stRaw(s) + n * kWsRawRow;
                    uint8_t* dB = stB(s) + (n >> 3) * 1024 + (n & 7) * 16;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 w = lds128(raw + q * 16);
                        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                        uint32_t h[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            e4m3x4_to_f16x2x2(wv[i], h[2 * i], h[2 * i + 1]);
                            h[2 * i] = hmul2(h[2 * i], sc2);
                            h[2 * i + 1] = hmul2(h[2 * i + 1], sc2);
                        }
                        *reinterpret_cast<uint4*>(dB + (2 * q) * 128) = make_uint4(h[0], h[1], h[2], h[3]);
                        *reinterpret_cast<uint4*>(dB + (2 * q + 1) * 128) = make_uint4(h[4], h[5], h[6], h[7]);
                    }
                }
                fence_async_smem();                           // A (cp.async) and B visible to the MMA
                mbar_arrive(&conv[s]);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            uint32_t sc = 0, tcount = 0;
            for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x, ++tcount) {
                const uint32_t b = tcount & 1u, v = tcount >> 1;
                if (v > 0 && !mbar_wait(&acc_empty[b], (v - 1) & 1u)) {
                    abort_s = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + b * BN;
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt, ++sc) {
                    const uint32_t s = sc % NS, u = sc / NS;
                    if (!mbar_wait(&conv[s], u & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    fence_async_smem();
                    const uint32_t a0 = smem_u32(stA(s)), b0 = smem_u32(stB(s));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_issue_id(d, smem_desc(a0 + kk * 256, 128, 1024), smem_desc(b0 + kk * 256, 128, 1024),
                                     kIdescN, (kt > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                    if (kt == KT - 1) mma_commit(&acc_full[b]);
                }
                if (!ok) {
                    abort_s = 1;
                    break;
                }
            }
        }
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;
        const int row = 32 * q + lane;
        uint32_t tcount = 0;
        for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x, ++tcount) {
            int mt, nt;
            decode_tile(p, tile, mt, nt);
            const int e = p.tile_e[mt], r0 = p.tile_r0[mt];
            const int rows = min(128, p.offsets[e + 1] - r0);
            const int rr = r0 + min(row, rows - 1);
            const float xs = KIND == 0 ? p.a_inv[p.sorted_pair[rr] / p.topk] : p.a_inv[rr];
            float winv[2];
            if (KIND == 0) {
                winv[0] = weight_prescale(p.s0 + (static_cast<size_t>(e) * (p.wrows / 128) + nt) * KB, KB, nullptr);
                winv[1] = weight_prescale(p.s1 + (static_cast<size_t>(e) * (p.wrows / 128) + nt) * KB, KB, nullptr);
            } else {
                const int nb = (nt * BN) / 128;
                winv[0] = weight_prescale(p.s0 + (static_cast<size_t>(e) * (p.wrows / 128) + nb) * KB, KB, nullptr);
                winv[1] = BN == 256 ? weight_prescale(p.s0 + (static_cast<size_t>(e) * (p.wrows / 128) + nb + 1) * KB,
                                                      KB, nullptr)
                                    : winv[0];
            }
            const uint32_t b = tcount & 1u, v = tcount >> 1;
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(&acc_full[b], v & 1u))) {
                abort_s = 1;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + b * BN;
            const bool valid = row < rows;
            if (KIND == 0) {
                float m = 0.0f;
                float* dst = p.out + static_cast<size_t>(r0 + row) * p.out_ld + nt * 128;
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    float gv[16], uv[16];
                    tmem_ld16(taddr + c0, gv);
                    tmem_ld16(taddr + 128 + c0, uv);
                    float hv[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        hv[j] = clamped_swiglu(gv[j] * xs * winv[0], uv[j] * xs * winv[1], p.limit);
                        m = fmaxf(m, fabsf(hv[j]));
                    }
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            reinterpret_cast<float4*>(dst + c0)[j] =
                                make_float4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]);
                    }
                }
                if (valid) atomicMax(p.amax + r0 + row, __float_as_uint(m));
            } else {
                float* dst = p.out + static_cast<size_t>(r0 + row) * p.out_ld + nt * BN;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    float yv[16];
                    tmem_ld16(taddr + c0, yv);
                    const float sc = xs * winv[c0 < 128 ? 0 : 1];
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            reinterpret_cast<float4*>(dst + c0)[j] = make_float4(
                                yv[4 * j] * sc, yv[4 * j + 1] * sc, yv[4 * j + 2] * sc, yv[4 * j + 3] * sc);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
        }
    }

    // ---------------- teardown ----------------
    __syncthreads();
    if (abort_s) {                                        // let any MMA still in flight finish
        if (tid == 0 && p.err != nullptr) atomicOr(p.err, 2);
        const long long t0 = clock64();
        while (clock64() - t0 < (1ll << 22)) {
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

cudaError_t launch_prefill_gemm_ws(int kind, const PrefillGemmArgs& p, int N_total, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t st;
    if ((st = cudaGetDevice(&dev)) != cudaSuccess) return st;
    if ((st = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return st;
    PrefillGemmArgs q = p;
    if (kind == 0) {
        q.n_tiles = N_total / 128;
        if ((st = cudaFuncSetAttribute(prefill_ws_gemm_kernel<0, 256>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, WsCfg<256>::kSmem)) != cudaSuccess)
            return st;
        prefill_ws_gemm_kernel<0, 256><<<sms, kWsThreads, WsCfg<256>::kSmem, stream>>>(q);
    } else if (N_total % 256 == 0) {
        q.n_tiles = N_total / 256;
        if ((st = cudaFuncSetAttribute(prefill_ws_gemm_kernel<1, 256>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, WsCfg<256>::kSmem)) != cudaSuccess)
            return st;
        prefill_ws_gemm_kernel<1, 256><<<sms, kWsThreads, WsCfg<256>::kSmem, stream>>>(q);
    } else {
        q.n_tiles = N_total / 128;
        if ((st = cudaFuncSetAttribute(prefill_ws_gemm_kernel<1, 128>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, WsCfg<128>::kSmem)) != cudaSuccess)
            return st;
        prefill_ws_gemm_kernel<1, 128><<<sms, kWsThreads, WsCfg<128>::kSmem, stream>>>(q);
    }
    return cudaGetLastError();
}

}  // namespace moe
