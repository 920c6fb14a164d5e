// Prefill grouped-GEMM core with the dequantised weights in tensor memory (the default core).
//
// Each GEMM is computed transposed: D[weight row][token] = W x A^T, with the weight slice (f16,
// produced by the converter warps) as the MMA's A operand in TMEM and 128 sorted activation rows
// (TMA, 128-byte swizzled) as its B operand in shared memory. Dequantised weights thus never
// pass through shared memory: per 64-wide K slice shared memory carries the token box, the raw
// E4M3 box and its one read by the converters - the f16 round trip through shared memory is what
// bounded the core that staged the dequantised weights there (prefill_tma.cu).
//   warps 0-1    token producers  slice sc -> slot sc % 4 (TMA box 128 rows x 64 f16), once the
//                                 slot's previous MMAs are done;
//   warps 2-3    raw producers    slice sc -> raw stage sc % 6 (NM boxes of 128 rows x 64 E4M3
//                                 bytes, 64-byte swizzled), once the converters have read it;
//   warps 4-11   converters       warp w writes TMEM lanes 32*(w%4)..+31 (the hardware's lane
//                                 quarter), lane = weight row; warps 4-7 take matrix (or K half) 0,
//                                 warps 8-11 matrix (or K half) 1. Read the raw row slice into
//                                 registers, release the raw stage, dequantise to f16 pairs x
//                                 prescaled block scale, tcgen05.st into TMEM slot sc % 4;
//   warps 12-19  epilogue         read D (lane = weight row, column = token) with tcgen05.ld,
//                                 SwiGLU (gate/up) or the row scales (down), token-major stores;
//   warp 20      MMA              one thread: per slice and K=16 step one M=128 x N MMA per weight
//                                 matrix (N = the tile's valid rows rounded up to 16); one commit
//                                 per slice frees the slot (token box and TMEM slice), one per
//                                 tile hands the accumulator over.
// gate/up: NM = 2 (gate rows nt*128.., up rows nt*128..), one accumulator (the two D matrices
// fill 256 TMEM columns, the four slots the other 256). down: NM = 1 (output rows nt*128..), the
// K halves of the slice split over the two converter groups, two accumulators so that the
// epilogue overlaps the next tile.
// Every wait is bounded (~1 s of SM clock); on a timeout the CTA sets bit 1 of the error word,
// every role leaves its loop, and the CTA frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "prefill.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kTwSlotsMax = 8;                   // token boxes in smem = weight slices in TMEM
constexpr int kTwRawStages = 6;                  // raw E4M3 weight boxes in smem
constexpr int kTwTok = 128 * 128;                // token slice: 128 rows x 64 f16 (16 KB)
constexpr int kTwTokWarps = 2;                   // producer warps for token boxes (slots w, w+2)
constexpr int kTwRawWarps = 2;                   // producer warps for raw boxes (stages w, w+2, w+4)
constexpr int kTwConvWarp0 = kTwTokWarps + kTwRawWarps;    // 4
constexpr int kTwConvWarps = 8;
constexpr int kTwEpiWarp0 = kTwConvWarp0 + kTwConvWarps;   // 12
constexpr int kTwEpiWarps = 8;
constexpr int kTwMmaWarp = kTwEpiWarp0 + kTwEpiWarps;      // 20
constexpr int kTwThreads = 32 * (kTwMmaWarp + 1);          // 672

template <int NM, int DB, int FMT>
struct TwCfg {
    static constexpr int kRowBytes = FMT == 0 ? 64 : 32;   // raw bytes of one row's 64-wide slice
    static constexpr int kRaw = NM * 128 * kRowBytes;      // raw weight boxes of one slice
    // (at least 120 KB, so that one CTA - and one 512-column TMEM allocation - fits per SM)
    // slots: 4 with two weight matrices (their TMEM slices and the accumulator fill 512 columns),
    // 8 with one
    static constexpr int kSlots = NM == 2 ? 4 : 8;
    static constexpr int kSmemUsed = kSlots * kTwTok + kTwRawStages * kRaw + 1024;
    static constexpr int kSmem = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
    static constexpr int kAcc = DB ? 2 : 1;                // accumulator buffers
    static constexpr uint32_t kAccCols = NM * 128;         // one buffer: NM matrices x 128 tokens
    static constexpr uint32_t kACols = NM * 32;            // one slot: 64 K (32 f16 pairs) per matrix
    static constexpr uint32_t kA0 = kAcc * kAccCols;       // first A column
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kA0 + kSlots * kACols <= kTmemCols && kSlots <= kTwSlotsMax && kSlots % 2 == 0, "TMEM budget");
    static_assert(kRaw % 1024 == 0, "stage alignment");
};

}  // namespace

template <int KIND, int NM, int DB, int FMT>
__global__ void __launch_bounds__(kTwThreads, 1)
    prefill_tw_gemm_kernel(const PrefillGemmArgs p, const __grid_constant__ CUtensorMap tmTok,
                           const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1) {
    using Cfg = TwCfg<NM, DB, FMT>;
    constexpr int NS = Cfg::kSlots, NR = kTwRawStages;
    constexpr uint32_t kIdesc128 = idesc_f16_f32<128, 128>();
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    // tfull[s]: token box s landed; rfull/rempty[r]: raw box r landed / read by all converters;
    // afull[s]: weight slice s in TMEM; sempty[s]: the MMAs of slot s (token box and TMEM slice)
    // are done; acc_full/acc_empty[b]: accumulator b complete / drained.
    __shared__ __align__(8) uint64_t tfull[NS], afull[NS], sempty[NS], rfull[NR], rempty[NR], acc_full[2], acc_empty[2];
    __shared__ uint32_t w_scale[kTwConvWarps][64];       // per converter warp: its rows' scale table
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = p.K, KT = K / 64, KB = K / 128;
    const int total = p.tiles[0] * p.n_tiles;
    auto stTok = [&](uint32_t s) { return smem + s * kTwTok; };
    auto stRaw = [&](uint32_t r) { return smem + NS * kTwTok + r * Cfg::kRaw; };

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&tfull[s], 1);
            mbar_init(&afull[s], kTwConvWarps);
            mbar_init(&sempty[s], 1);
        }
        for (int r = 0; r < NR; ++r) {
            mbar_init(&rfull[r], 1);
            mbar_init(&rempty[r], kTwConvWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kTwEpiWarps);
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

    if (warp < kTwConvWarp0) {
        // ---------------- producers ----------------
        // Warps 0-1 issue token boxes (slice sc by warp sc % 2 into slot sc % 4, once the slot's
        // previous MMAs are done); warps 2-3 issue raw weight boxes (slice sc by warp 2 + sc % 2
        // into raw stage sc % 6, once all converters have read its previous box). Each warp
        // always serves the same slots / stages, in order.
        if (lane == 0) {
            const bool tok = warp < kTwTokWarps;
            const int pw = tok ? warp : warp - kTwTokWarps;
            uint32_t sc = 0;
            for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x) {
                int mt, nt;
                decode_tile(p, tile, mt, nt);
                const int e = p.tile_e[mt], r0 = p.tile_r0[mt];
                const int wy = e * p.wrows + nt * 128;        // first weight row of the slab
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt, ++sc) {
                    if (static_cast<int>(sc % 2) != pw) continue;
                    if (tok) {
                        const uint32_t s = sc % NS, u = sc / NS;
                        if (u > 0 && !mbar_wait(&sempty[s], (u - 1) & 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&tfull[s], kTwTok);
                        tma_load_2d(smem_u32(stTok(s)), &tmTok, kt * 64, r0, &tfull[s]);   // rows past the expert: unused
                    } else {
                        const uint32_t r = sc % NR, u = sc / NR;
                        if (u > 0 && !mbar_wait(&rempty[r], (u - 1) & 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&rfull[r], Cfg::kRaw);
                        tma_load_2d(smem_u32(stRaw(r)), &tmW0, kt * Cfg::kRowBytes, wy, &rfull[r]);
                        if (NM == 2)
                            tma_load_2d(smem_u32(stRaw(r)) + 128 * Cfg::kRowBytes, &tmW1, kt * Cfg::kRowBytes, wy,
                                        &rfull[r]);
                    }
                }
                if (!ok) {
                    abort_s = 1;
                    break;
                }
            }
        }
    } else if (warp < kTwEpiWarp0) {
        // ---------------- converters ----------------
        // Lane quarter qd = warp % 4 (TMEM access rule); part 0/1 = matrix (NM = 2) or K half
        // (NM = 1). Eight consecutive lanes read eight consecutive raw rows of one 16-byte chunk,
        // which the 64-byte swizzle places in eight distinct bank groups. The raw box is
        // released as soon as it is in registers; the TMEM slot is waited for only then.
        const int cw = warp - kTwConvWarp0, qd = warp & 3, part = cw / 4;
        const int rrow = (NM == 2 ? part * 128 : 0) + 32 * qd + lane;       // raw row of this thread
        const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
        // FP8: 16-byte chunks of 16 codes, 64-byte rows, 64-byte swizzle. NVFP4: 16-byte chunks of
        // 32 codes, 32-byte rows, 32-byte swizzle (chunk ^ bit 2 of the row).
        constexpr int kChunks = FMT == 0 ? (NM == 2 ? 4 : 2) : (NM == 2 ? 2 : 1);
        const int c0 = NM == 2 ? 0 : kChunks * part;
        const int sw = FMT == 0 ? (rrow >> 1) & 3 : (rrow >> 2) & 1;
        uint32_t* tbl = w_scale[cw];
        const uint8_t* sfrow = nullptr;                    // NVFP4: this row's scale bytes
        uint4 sfv = make_uint4(0, 0, 0, 0);                // NVFP4: scale bytes of 4 slices (K 256)
        uint32_t sc = 0;
        for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x) {
            int mt, nt;
            decode_tile(p, tile, mt, nt);
            const int e = p.tile_e[mt];
            if constexpr (FMT == 0) {
                __syncwarp();                              // the old table is no longer read
                const size_t sblk = static_cast<size_t>(e) * (p.wrows / 128) + nt;
                weight_prescale((NM == 2 && part == 1 ? p.s1 : p.s0) + sblk * KB, KB, tbl);
                __syncwarp();
            } else {
                const size_t wr_ = static_cast<size_t>(e) * p.wrows + nt * 128 + (rrow & 127);
                sfrow = (NM == 2 && part == 1 ? p.sf1 : p.sf0) + wr_ * (K / 16);
            }
            bool ok = true;
            for (int kt = 0; kt < KT; ++kt, ++sc) {
                const uint32_t r = sc % NR, ur = sc / NR, s = sc % NS, us = sc / NS;
                if (FMT == 1 && (kt & 3) == 0) sfv = __ldg(reinterpret_cast<const uint4*>(sfrow + kt * 4));
                if (!__all_sync(0xffffffffu, mbar_wait(&rfull[r], ur & 1u))) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = stRaw(r) + rrow * Cfg::kRowBytes;
                uint4 wr[kChunks];
#pragma unroll
                for (int c = 0; c < kChunks; ++c) wr[c] = lds128(raw + (((c0 + c) ^ sw) << 4));
                __syncwarp();
                if (lane == 0) mbar_arrive(&rempty[r]);
                if (!__all_sync(0xffffffffu, us == 0 || mbar_wait(&sempty[s], (us - 1) & 1u))) {
                    ok = false;
                    break;
                }
                uint32_t h[NM == 2 ? 32 : 16];
                if constexpr (FMT == 0) {
                    const uint32_t sc2 = tbl[kt >> 1];
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        const uint32_t wv[4] = {wr[c].x, wr[c].y, wr[c].z, wr[c].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t lo, hi;
                            e4m3x4_to_f16x2x2(wv[i], lo, hi);
                            h[8 * c + 2 * i] = hmul2(lo, sc2);
                            h[8 * c + 2 * i + 1] = hmul2(hi, sc2);
                        }
                    }
                } else {
                    // the slice's 4 scale bytes (one per 16 codes); E2M1 x E4M3 products are exact
                    const uint32_t sfw = (kt & 2) ? ((kt & 1) ? sfv.w : sfv.z) : ((kt & 1) ? sfv.y : sfv.x);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        const uint32_t wv[4] = {wr[c].x, wr[c].y, wr[c].z, wr[c].w};
                        const int grp0 = 2 * (c0 + c);     // scale group of the chunk's first 16 codes
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t sf2 = e4m3_splat_f16x2((sfw >> (8 * (grp0 + (i >> 1)))) & 0xFFu);
                            uint32_t q[4];
                            e2m1x8_to_f16x2x4(wv[i], q[0], q[1], q[2], q[3]);
#pragma unroll
                            for (int b = 0; b < 4; ++b) h[16 * c + 4 * i + b] = hmul2(q[b], sf2);
                        }
                    }
                }
                const uint32_t ta = tmem + lane_off + Cfg::kA0 + s * Cfg::kACols + (NM == 2 ? part * 32 : part * 16);
                if constexpr (NM == 2)
                    tmem_st32(ta, h);
                else
                    tmem_st16(ta, h);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[s]);
            }
            if (!ok) {
                abort_s = 1;
                break;
            }
        }
    } else if (warp == kTwMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            uint32_t sc = 0, tcount = 0;
            for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x, ++tcount) {
                const uint32_t b = tcount % Cfg::kAcc, v = tcount / Cfg::kAcc;
                if (v > 0 && !mbar_wait(&acc_empty[b], (v - 1) & 1u)) {
                    abort_s = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem + b * Cfg::kAccCols;
                // MMA width = the tile's valid rows rounded up to 16: the last m-tile of an expert
                // is often far from full, and the MMA time scales with N
                int mt, nt;
                decode_tile(p, tile, mt, nt);
                const int rows = min(128, p.offsets[p.tile_e[mt] + 1] - p.tile_r0[mt]);
                const uint32_t n_eff = static_cast<uint32_t>((rows + 15) & ~15);
                const uint32_t idesc = (kIdesc128 & ~(0x3Fu << 17)) | ((n_eff >> 3) << 17);
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt, ++sc) {
                    const uint32_t s = sc % NS, us = sc / NS;
                    if (!mbar_wait(&tfull[s], us & 1u) || !mbar_wait(&afull[s], us & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tok = smem_u32(stTok(s));
                    const uint32_t a0 = tmem + Cfg::kA0 + s * Cfg::kACols;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bdesc = smem_desc_sw128(tok + kk * 32);
#pragma unroll
                        for (int m = 0; m < NM; ++m)
                            mma_issue_tmem_a(d0 + m * 128, a0 + m * 32 + kk * 8, bdesc, idesc,
                                             (kt > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&sempty[s]);
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
        // Warp w reads TMEM lanes 32*(w%4)..+31 (lane = weight row f of the tile's slab) and token
        // columns 64*h..+63, h = (w - 12) / 4. Each store instruction writes one token row's 32
        // consecutive features (128 contiguous bytes).
        __shared__ float xs_s[kTwEpiWarps][64];            // per epilogue warp: its tokens' scales
        const int ew = warp - kTwEpiWarp0, qd = warp & 3, cbase = 64 * (ew / 4);
        const int f = 32 * qd + lane;
        const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
        uint32_t tcount = 0;
        for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x, ++tcount) {
            int mt, nt;
            decode_tile(p, tile, mt, nt);
            const int e = p.tile_e[mt], r0 = p.tile_r0[mt];
            const int rows = min(128, p.offsets[e + 1] - r0);
            __syncwarp();                                  // the previous tile's scales are read
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int rr = r0 + min(cbase + 32 * i + lane, rows - 1);
                xs_s[ew][32 * i + lane] = KIND == 0 ? p.a_inv[p.sorted_pair[rr] / p.topk] : p.a_inv[rr];
            }
            const size_t sblk = static_cast<size_t>(e) * (p.wrows / 128) + nt;
            float winv0, winv1;                            // undo the converters' weight scaling
            if constexpr (FMT == 0) {
                winv0 = weight_prescale(p.s0 + sblk * KB, KB, nullptr);
                winv1 = KIND == 0 ? weight_prescale(p.s1 + sblk * KB, KB, nullptr) : winv0;
            } else {
                winv0 = p.s2_0;                            // NVFP4: scale_2 of the projection
                winv1 = KIND == 0 ? p.s2_1 : winv0;
            }
            __syncwarp();
            const uint32_t b = tcount % Cfg::kAcc, v = tcount / Cfg::kAcc;
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(&acc_full[b], v & 1u))) {
                abort_s = 1;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem + lane_off + b * Cfg::kAccCols + cbase;
            float* dst = p.out + static_cast<size_t>(r0 + cbase) * p.out_ld + nt * 128 + f;
            const int vrows = rows - cbase;                // valid columns of this warp
#pragma unroll 1
            for (int c0 = 0; c0 < 64 && c0 < vrows; c0 += 16) {
                if (KIND == 0) {
                    float gv[16], uv[16];
                    tmem_ld16(taddr + c0, gv);
                    tmem_ld16(taddr + 128 + c0, uv);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = c0 + j;
                        const float xs = xs_s[ew][t];
                        // the same clamped SwiGLU with the SFU exponential and divide (a few ulp; the
                        // epilogue holds the single accumulator, so its length stalls the MMA)
                        const float gg = fminf(gv[j] * xs * winv0, p.limit);
                        const float uu = fminf(fmaxf(uv[j] * xs * winv1, -p.limit), p.limit);
                        const float h = __fdividef(gg, 1.0f + __expf(-gg)) * uu;
                        const uint32_t mb = warp_max_bits(fabsf(h));
                        if (t < vrows) {
                            dst[static_cast<size_t>(t) * p.out_ld] = h;
                            if (lane == 0) atomicMax(p.amax + r0 + cbase + t, mb);
                        }
                    }
                } else {
                    float yv[16];
                    tmem_ld16(taddr + c0, yv);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = c0 + j;
                        if (t < vrows) dst[static_cast<size_t>(t) * p.out_ld] = yv[j] * xs_s[ew][t] * winv0;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
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

PFN_cuTensorMapEncodeTiled_v12000 tw_encoder() {
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

// 2-D map over a row-major [rows][inner] matrix of elem-byte elements, box box_inner x 128.
bool tw_map(CUtensorMap* m, CUtensorMapDataType dt, int elem, const void* base, uint64_t inner, uint64_t rows,
            uint32_t box_inner, CUtensorMapSwizzle sw) {
    auto enc = tw_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem)};
    const cuuint32_t box[2] = {box_inner, 128};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND, int NM, int DB, int FMT>
cudaError_t launch_tw(const PrefillGemmArgs& q, const CUtensorMap& a, const CUtensorMap& w0, const CUtensorMap& w1,
                      int grid, cudaStream_t stream) {
    using Cfg = TwCfg<NM, DB, FMT>;
    cudaError_t st = cudaFuncSetAttribute(prefill_tw_gemm_kernel<KIND, NM, DB, FMT>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (st != cudaSuccess) return st;
    prefill_tw_gemm_kernel<KIND, NM, DB, FMT><<<grid, kTwThreads, Cfg::kSmem, stream>>>(q, a, w0, w1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_gemm_tw(int kind, const PrefillGemmArgs& p, int N_total, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t st;
    if ((st = cudaGetDevice(&dev)) != cudaSuccess) return st;
    if ((st = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return st;
    // TMA wants 16-byte aligned bases and row strides (K is a multiple of 128 here).
    if ((reinterpret_cast<uintptr_t>(p.a) | reinterpret_cast<uintptr_t>(p.w0) | reinterpret_cast<uintptr_t>(p.w1)) &
        15u)
        return cudaErrorMisalignedAddress;
    PrefillGemmArgs q = p;
    q.n_tiles = N_total / 128;
    CUtensorMap ma, mw0, mw1;
    const uint64_t wrows_all = static_cast<uint64_t>(p.experts) * p.wrows;
    const bool fp4 = p.fmt == 1;
    if (fp4 && ((reinterpret_cast<uintptr_t>(p.sf0) | reinterpret_cast<uintptr_t>(p.sf1)) & 15u))
        return cudaErrorMisalignedAddress;
    // FP8: rows of K code bytes, boxes of 64 bytes (64-byte swizzle); NVFP4: rows of K/2 bytes of
    // packed codes, boxes of 32 bytes (32-byte swizzle)
    const uint64_t wbytes = fp4 ? p.K / 2 : p.K;
    const uint32_t wbox = fp4 ? 32 : 64;
    const CUtensorMapSwizzle wsw = fp4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
    const bool ok = tw_map(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.a, p.K, p.a_rows, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
                    tw_map(&mw0, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w0, wbytes, wrows_all, wbox, wsw) &&
                    tw_map(&mw1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w1, wbytes, wrows_all, wbox, wsw);
    if (!ok) return cudaErrorInvalidValue;
    if (kind == 0) return fp4 ? launch_tw<0, 2, 0, 1>(q, ma, mw0, mw1, sms, stream)
                              : launch_tw<0, 2, 0, 0>(q, ma, mw0, mw1, sms, stream);
    return fp4 ? launch_tw<1, 1, 1, 1>(q, ma, mw0, mw1, sms, stream) : launch_tw<1, 1, 1, 0>(q, ma, mw0, mw1, sms, stream);
}

}  // namespace moe
