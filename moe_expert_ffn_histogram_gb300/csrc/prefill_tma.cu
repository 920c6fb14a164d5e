// TMA-fed warp-specialised tcgen05 core of the prefill grouped GEMMs (the default prefill core).
//
// Tiles and epilogues are those of prefill_ws.cu; what changes is how operands reach shared
// memory (there one cp.async per 16 bytes per thread, which bounded the kernel) and how the
// weight conversion overlaps:
//   warps 0-2   producers  warp w owns load stage w: one thread arms full[w] with the slice's
//                          byte count and issues three TMA boxes - 128 sorted rows x 64 f16 of A
//                          (128-byte swizzle: the K-major layout the MMA reads directly) and the
//                          slice's E4M3 weight rows (64-byte swizzle);
//   warps 3-10  converters two groups of four warps take alternate slices: dequantise the weight
//                          slice to f16 x prescaled block scale into B buffer sc % 3 (canonical
//                          no-swizzle K-major), fence the async proxy, arrive bfull;
//   warps 11-14 epilogue   as in prefill_ws.cu (warp w reads TMEM lanes 32*(w%4) .. +31);
//   warp 15     MMA        one thread: four M=128 x N=BN x K=16 tcgen05.mma per slice into one of
//                          two TMEM accumulators; commits free the load stage, the B buffer and,
//                          after a tile's last slice, hand the accumulator to the epilogue.
// Gate/up reads A from the sorted copy of x16 that the x prep kernel writes ([P][H]); down reads
// a16 ([P][I]). Every wait is bounded (~1 s of SM clock); on a timeout the CTA sets bit 1 of the
// error word, every role leaves its loop, and the CTA frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "prefill.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kTmStages = 3;                     // load stages = converted-weight buffers: slice sc
                                                 // uses load stage and B buffer sc % 3
constexpr int kTmA = 128 * 128;                  // A slice: 128 rows x 64 f16, 128B-swizzled (16 KB)
constexpr int kTmProdWarps = kTmStages;          // producer warp w owns load stage w
constexpr int kTmConvGroups = 2;                 // converter group g takes slices sc % 2 == g
constexpr int kTmGroupWarps = 4;
constexpr int kTmGroupThreads = 32 * kTmGroupWarps;
constexpr int kTmConvWarps = kTmConvGroups * kTmGroupWarps;
constexpr int kTmEpiThreads = 128;
constexpr int kTmConvWarp0 = kTmProdWarps;                 // 3
constexpr int kTmEpiWarp0 = kTmConvWarp0 + kTmConvWarps;   // 11
constexpr int kTmMmaWarp = kTmEpiWarp0 + 4;                // 15
constexpr int kTmThreads = 32 * (kTmMmaWarp + 1);          // 512

template <int BN>
struct TmCfg {
    static constexpr int kRaw = BN * 64;                   // raw E4M3 slice, 64B-swizzled rows
    static constexpr int kLoad = kTmA + kRaw;              // one load stage
    static constexpr int kB = BN * 128;                    // converted f16 slice
    static constexpr int kSmem = kTmStages * (kLoad + kB) + 1024;
    static constexpr uint32_t kTmemCols = 2 * BN;          // two fp32 accumulators
    static_assert(kLoad % 1024 == 0 && kB % 1024 == 0, "stage alignment");
};

}  // namespace

template <int KIND, int BN>
__global__ void __launch_bounds__(kTmThreads, 1)
    prefill_tma_gemm_kernel(const PrefillGemmArgs p, const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1) {
    using Cfg = TmCfg<BN>;
    constexpr int NL = kTmStages, NB = kTmStages;
    constexpr uint32_t kIdescN = idesc_f16_f32<128, BN>();
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[NL], empty[NL], bfull[NB], bempty[NB], acc_full[2], acc_empty[2];
    __shared__ uint32_t w_scale[kTmConvWarps][2][64];    // per converter warp: the tile's two tables
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = p.K, KT = K / 64, KB = K / 128;
    const int total = p.tiles[0] * p.n_tiles;
    auto stA = [&](uint32_t s) { return smem + s * Cfg::kLoad; };
    auto stRaw = [&](uint32_t s) { return smem + s * Cfg::kLoad + kTmA; };
    auto stB = [&](uint32_t b) { return smem + NL * Cfg::kLoad + b * Cfg::kB; };

    if (tid == 0) {
        for (int s = 0; s < NL; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(&bfull[b], kTmGroupWarps);
            mbar_init(&bempty[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kTmEpiThreads);
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

    if (warp < kTmProdWarps) {
        // ---------------- producers ----------------
        // A TMA issue costs the issuing thread tens to hundreds of cycles; three warps, each
        // owning one load stage (slices sc with sc % 3 == warp), keep the copies flowing.
        if (lane == 0) {
            uint32_t sc = 0;
            for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x) {
                int mt, nt;
                decode_tile(p, tile, mt, nt);
                const int e = p.tile_e[mt], r0 = p.tile_r0[mt];
                const int wy0 = e * p.wrows + (KIND == 0 ? nt * 128 : nt * BN);
                const int wy1 = KIND == 0 ? wy0 : wy0 + 128;
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt, ++sc) {
                    const uint32_t s = sc % NL, u = sc / NL;
                    if (static_cast<int>(s) != warp) continue;
                    if (u > 0 && !mbar_wait(&empty[s], (u - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], kTmA + Cfg::kRaw);
                    const uint32_t a_dst = smem_u32(stA(s)), r_dst = smem_u32(stRaw(s));
                    tma_load_2d(a_dst, &tmA, kt * 64, r0, &full[s]);   // rows past the expert: unused
                    tma_load_2d(r_dst, &tmW0, kt * 64, wy0, &full[s]);
                    if (BN == 256) tma_load_2d(r_dst + 128 * 64, KIND == 0 ? &tmW1 : &tmW0, kt * 64, wy1, &full[s]);
                }
                if (!ok) {
                    abort_s = 1;
                    break;
                }
            }
        }
    } else if (warp < kTmEpiWarp0) {
        // ---------------- converters ----------------
        // Two groups of four warps take alternate slices, so one slice's conversion overlaps the
        // next. Work item i = gt + 128 j of a slice is the 16-byte raw chunk q = i / BN of weight
        // row n = i % BN: eight consecutive lanes take eight consecutive rows of one chunk, which
        // the 64-byte swizzle spreads over eight bank groups for the reads, as (n & 7) does for
        // the writes. A slice waits first for its B buffer (whose previous slice, three back,
        // the MMA has then consumed) and only then for its load stage, so that parity waits
        // never run two phases ahead.
        const int ct = tid - 32 * kTmConvWarp0, cw = ct >> 5;
        const int grp = cw / kTmGroupWarps, gt = ct % kTmGroupThreads;
        uint32_t(*tbl)[64] = w_scale[cw];
        uint32_t sc = 0;
        for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x) {
            int mt, nt;
            decode_tile(p, tile, mt, nt);
            const int e = p.tile_e[mt];
            __syncwarp();                                  // the old tables are no longer read
            const size_t sblk = static_cast<size_t>(e) * (p.wrows / 128);
            if (KIND == 0) {                               // rows 0..127 gate, 128..255 up
                weight_prescale(p.s0 + (sblk + nt) * KB, KB, tbl[0]);
                weight_prescale(p.s1 + (sblk + nt) * KB, KB, tbl[1]);
            } else {                                       // rows 128.. in the next 128-row block
                weight_prescale(p.s0 + (sblk + (nt * BN) / 128) * KB, KB, tbl[0]);
                if (BN == 256) weight_prescale(p.s0 + (sblk + (nt * BN) / 128 + 1) * KB, KB, tbl[1]);
            }
            __syncwarp();
            bool ok = true;
            for (int kt = 0; kt < KT; ++kt, ++sc) {
                if (static_cast<int>(sc % kTmConvGroups) != grp) continue;
                const uint32_t s = sc % NL, u = sc / NL;
                bool w_ok = u == 0 || mbar_wait(&bempty[s], (u - 1) & 1u);
                if (w_ok) w_ok = mbar_wait(&full[s], u & 1u);
                if (!__all_sync(0xffffffffu, w_ok)) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = stRaw(s);
                uint8_t* dst = stB(s);
                constexpr int kItems = BN * 4 / kTmGroupThreads;
                // All of this slice's raw chunks are read before the first store, so the reads
                // are not held behind stores the compiler cannot prove disjoint from them.
                uint4 wr[kItems];
#pragma unroll
                for (int j = 0; j < kItems; ++j) {
                    const int item = gt + kTmGroupThreads * j;
                    const int n = item % BN, q = item / BN;
                    wr[j] = lds128(raw + n * 64 + ((q ^ ((n >> 1) & 3)) << 4));
                }
#pragma unroll
                for (int j = 0; j < kItems; ++j) {
                    const int item = gt + kTmGroupThreads * j;
                    const int n = item % BN, q = item / BN;
                    const uint32_t sc2 = tbl[n >> 7][kt >> 1];
                    const uint32_t wv[4] = {wr[j].x, wr[j].y, wr[j].z, wr[j].w};
                    uint32_t h[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        e4m3x4_to_f16x2x2(wv[i], h[2 * i], h[2 * i + 1]);
                        h[2 * i] = hmul2(h[2 * i], sc2);
                        h[2 * i + 1] = hmul2(h[2 * i + 1], sc2);
                    }
                    uint8_t* dB = dst + (n >> 3) * 1024 + (2 * q) * 128 + (n & 7) * 16;
                    *reinterpret_cast<uint4*>(dB) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4*>(dB + 128) = make_uint4(h[4], h[5], h[6], h[7]);
                }
                fence_async_smem();                        // B visible to the MMA (async proxy)
                __syncwarp();
                if (lane == 0) mbar_arrive(&bfull[s]);
            }
            if (!ok) {
                abort_s = 1;
                break;
            }
        }
    } else if (warp == kTmMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            uint32_t sc = 0, tcount = 0;
            for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x, ++tcount) {
                const uint32_t ab = tcount & 1u, v = tcount >> 1;
                if (v > 0 && !mbar_wait(&acc_empty[ab], (v - 1) & 1u)) {
                    abort_s = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + ab * BN;
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt, ++sc) {
                    const uint32_t s = sc % NL, u = sc / NL, b = s, ub = u;
                    if (!mbar_wait(&full[s], u & 1u) || !mbar_wait(&bfull[b], ub & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(stA(s)), b0 = smem_u32(stB(b));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_issue_id(d, smem_desc_sw128(a0 + kk * 32), smem_desc(b0 + kk * 256, 128, 1024), kIdescN,
                                     (kt > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                    mma_commit(&bempty[b]);
                    if (kt == KT - 1) mma_commit(&acc_full[ab]);
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


namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// 2-D map over a row-major [rows][inner] matrix of elem-byte elements, box box_inner x box_rows.
bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem, const void* base, uint64_t inner, uint64_t rows,
                 uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem)};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND, int BN>
cudaError_t launch_tma(const PrefillGemmArgs& q, const CUtensorMap& a, const CUtensorMap& w0, const CUtensorMap& w1,
                       int grid, cudaStream_t stream) {
    cudaError_t st = cudaFuncSetAttribute(prefill_tma_gemm_kernel<KIND, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          TmCfg<BN>::kSmem);
    if (st != cudaSuccess) return st;
    prefill_tma_gemm_kernel<KIND, BN><<<grid, kTmThreads, TmCfg<BN>::kSmem, stream>>>(q, a, w0, w1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_gemm_tma(int kind, const PrefillGemmArgs& p, int N_total, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t st;
    if ((st = cudaGetDevice(&dev)) != cudaSuccess) return st;
    if ((st = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return st;
    // TMA wants 16-byte aligned bases and row strides (K is a multiple of 128 here).
    if ((reinterpret_cast<uintptr_t>(p.a) | reinterpret_cast<uintptr_t>(p.w0) | reinterpret_cast<uintptr_t>(p.w1)) &
        15u)
        return cudaErrorMisalignedAddress;
    PrefillGemmArgs q = p;
    const int BN = (kind == 0 || N_total % 256 == 0) ? 256 : 128;
    q.n_tiles = kind == 0 ? N_total / 128 : N_total / BN;
    CUtensorMap ma, mw0, mw1;
    const uint64_t wrows_all = static_cast<uint64_t>(p.experts) * p.wrows;
    bool ok = make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.a, p.K, p.a_rows, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map_2d(&mw0, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w0, p.K, wrows_all, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_64B) &&
              make_map_2d(&mw1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w1, p.K, wrows_all, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return cudaErrorInvalidValue;
    if (kind == 0) return launch_tma<0, 256>(q, ma, mw0, mw1, sms, stream);
    if (BN == 256) return launch_tma<1, 256>(q, ma, mw0, mw1, sms, stream);
    return launch_tma<1, 128>(q, ma, mw0, mw1, sms, stream);
}

}  // namespace moe
