// Prefill grouped-GEMM core with the dequantised weights in tensor memory (the default core).
//
// Each GEMM is computed transposed: D[weight row][token] = W x A^T, with the weight slice (f16,
// produced by the converter warps) as the MMA's A operand in TMEM and 128 sorted activation rows
// (TMA, 128-byte swizzled) as its B operand in shared memory. Dequantised weights thus never
// pass through shared memory: per 128-wide K slice shared memory carries the token boxes, the
// raw weight boxes and their one read by the converters - the f16 round trip through shared
// memory is what bounded an earlier core that staged the dequantised weights there.
//   warps 0-1    token producers  slice sc -> token slot sc % NT (two TMA boxes of 128 rows x 64
//                                 f16), once the slot's previous MMAs are done;
//   warps 2-3    raw producers    slice sc -> raw stage sc % NR (per weight matrix one box of 128
//                                 rows x 128 E4M3 bytes, 128-byte swizzle, or x 64 bytes of packed
//                                 E2M1 codes, 64-byte swizzle), once the converters have read it;
//   warps 4-11   converters       warp w writes TMEM lanes 32*(w%4)..+31 (the hardware's lane
//                                 quarter), lane = weight row; warps 4-7 take matrix (or K half) 0,
//                                 warps 8-11 matrix (or K half) 1. Read the raw row slice into
//                                 registers, release the raw stage, dequantise to f16 pairs x
//                                 prescaled block scale, tcgen05.st into TMEM slot sc % NS;
//   warps 12-19  epilogue         read D (lane = weight row, column = token) with tcgen05.ld,
//                                 SwiGLU (gate/up) or the row scales (down), token-major stores;
//   warp 20      MMA              one thread: per slice and K=16 step one M=128 x N MMA per weight
//                                 matrix (N = the tile's valid rows rounded up to 16); a commit
//                                 per slice frees its TMEM slice (and with its own token slots a
//                                 second one its token boxes), one per tile hands the accumulator
//                                 over. No memory access in its loop;
//   warp 21      watcher          waits on the slice's mbarriers for the MMA warp and releases it
//                                 through a named barrier (per tile a reduction that carries N).
// gate/up: NM = 2 (gate rows nt*128.., up rows nt*128..), one accumulator (the two D matrices
// fill 256 TMEM columns, two slots of 2 x 64 columns the other 256). down: NM = 1 (output rows
// nt*128..), the K halves of the slice split over the two converter groups, two accumulators so
// that the epilogue overlaps the next tile, four slots of 64 columns.
// The slice is 128 wide because every slice costs the converters, the watcher and the MMA warp
// a fixed round of barrier traffic (~500 cycles measured for an empty pipeline of this shape);
// 128-wide slices double the MMA work that pays for it.
// Every wait is bounded (~1 s of SM clock); on a timeout the CTA sets bit 1 of the error word and
// every role leaves its loop; the producers issue no further box once any role has given up. The
// CTA then waits (bounded again) until every TMA box it issued has landed and every MMA it queued
// has completed, and only then frees its TMEM and exits, so that no asynchronous write reaches
// its shared memory or TMEM after it has gone (if that drain also times out: bit 2 as well).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "prefill.cuh"
#include "tc_ptx.cuh"
#include "tma_map.cuh"


namespace moe {

namespace {

// tanh(x) by the SFU's approximation (tanh.approx.f32).
__device__ __forceinline__ float tanh_approx(float x) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Bounded mbarrier wait of this core's pipeline roles.
__device__ __forceinline__ bool tw_wait(uint64_t* m, uint32_t parity) {
    if (mbar_test(m, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_test(m, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

constexpr int kTwSliceK = 128;                   // K per slice
constexpr int kTwSlotsMax = 4;                   // token slots in smem / weight slices in TMEM
constexpr int kTwBox = 128 * 128;                // one token box: 128 rows x 64 f16 (16 KB)
constexpr int kTwTok = 2 * kTwBox;               // token slice: 128 rows x 128 f16 (32 KB)
constexpr int kTwTokWarps = 2;                   // producer warps for token boxes (odd / even slices)
constexpr int kTwRawWarps = 2;                   // producer warps for raw boxes (odd / even slices)
constexpr int kTwConvWarp0 = kTwTokWarps + kTwRawWarps;    // 4
constexpr int kTwConvWarps = 8;
constexpr int kTwEpiWarp0 = kTwConvWarp0 + kTwConvWarps;   // 12
constexpr int kTwEpiWarps = 8;
constexpr int kTwMmaWarp = kTwEpiWarp0 + kTwEpiWarps;      // 20
constexpr int kTwWatchWarp = kTwMmaWarp + 1;               // 21
constexpr int kTwThreads = 32 * (kTwWatchWarp + 1);        // 704
constexpr uint32_t kTwIssueBar = 1;                        // named barrier: watcher <-> MMA warp

template <int NM, int DB, int FMT>
struct TwCfg {
    static constexpr int kRowBytes = FMT == 0 ? 128 : 64;  // raw bytes of one row's 128-wide slice
    static constexpr int kRaw = NM * 128 * kRowBytes;      // raw weight boxes of one slice
    // slots: 2 with two weight matrices (their TMEM slices and the accumulator fill 512 columns),
    // 4 with one
    static constexpr int kSlots = NM == 2 ? 2 : 4;
    // token slots: with two weight matrices more than TMEM slots (their own release barrier,
    // a second commit per slice), so that the token boxes are loaded ahead of the slot
    // recycling; with one matrix one per TMEM slot (released with it)
    static constexpr int kTokSlots = NM == 2 ? (FMT == 0 ? 3 : 4) : kSlots;
    static constexpr bool kTokOwn = kTokSlots != kSlots;
    // raw stages: as many as fit beside the token slots (at least 120 KB in all, so that one CTA
    // - and one 512-column TMEM allocation - fits per SM)
    static constexpr int kRawStages = (NM == 2 && FMT == 0) ? 3 : (NM == 1 && FMT == 0) ? 5 : (NM == 2) ? 5 : 6;
    static constexpr int kSmemUsed = kTokSlots * kTwTok + kRawStages * kRaw + 1024;
    static constexpr int kSmem = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
    static constexpr int kAcc = DB ? 2 : 1;                // accumulator buffers
    static constexpr uint32_t kAccCols = NM * 128;         // one buffer: NM matrices x 128 tokens
    static constexpr uint32_t kMCols = kTwSliceK / 2;      // one matrix's slice: 128 K = 64 f16 pairs
    static constexpr uint32_t kACols = NM * kMCols;        // one slot
    static constexpr uint32_t kA0 = kAcc * kAccCols;       // first A column
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kA0 + kSlots * kACols <= kTmemCols && kSlots <= kTwSlotsMax && kTokSlots <= kTwSlotsMax, "TMEM budget");
    static_assert(kSmemUsed + 8 * 1024 <= 227 * 1024, "shared memory");
    static_assert(kRaw % 1024 == 0 && kTwTok % 1024 == 0, "stage alignment");
};

}  // namespace

// 1: a tile's token boxes hold its valid rows rounded up to 16; 0: always 128 rows.
#ifndef MOE_TOK_FIT
#define MOE_TOK_FIT 1
#endif

// Token-row maps of one matrix with boxes of 16, 32, ..., 128 rows (x 64 f16): a tile loads only
// its valid rows rounded up to 16 (the width its MMAs run at), so narrow tiles of rarely routed
// experts do not fill shared memory with rows they never read.
struct TokMaps {
    CUtensorMap m[8];
};

template <int KIND, int NM, int DB, int FMT>
__global__ void __launch_bounds__(kTwThreads, 1)
    prefill_tw_gemm_kernel(const PrefillGemmArgs p, const __grid_constant__ TokMaps tmTok,
                           const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1) {
    using Cfg = TwCfg<NM, DB, FMT>;
    constexpr int NS = Cfg::kSlots, NT = Cfg::kTokSlots, NR = Cfg::kRawStages;
    constexpr uint32_t kIdesc128 = idesc_f16_f32<128, 128>();
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    // tfull[t]: token boxes of token slot t landed; tempty[t]: its MMAs are done (own token
    // slots only); rfull/rempty[r]: raw boxes r landed / read by all converters; afull[s]: weight
    // slice s in TMEM; sempty[s]: the MMAs of slot s are done (its TMEM slice - and its token
    // boxes when those are not on their own - may be refilled); acc_full/acc_empty[b]:
    // accumulator b complete / drained.
    __shared__ __align__(8) uint64_t tfull[NT], tempty[NT], afull[NS], sempty[NS], rfull[NR], rempty[NR], acc_full[2],
        acc_empty[2], mma_done;
    // boxes issued into each token slot / raw stage so far: the phase of the last one is what
    // the teardown waits for after an abort
    __shared__ volatile uint32_t tok_issued[NT], raw_issued[NR];
    __shared__ uint32_t w_scale[kTwConvWarps][64];       // per converter warp: its rows' scale table
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = p.K, KT = K / kTwSliceK, KB = K / 128;
    const int total = p.tiles[0] * p.n_tiles;
    auto stTok = [&](uint32_t s) { return smem + s * kTwTok; };
    auto stRaw = [&](uint32_t r) { return smem + NT * kTwTok + r * Cfg::kRaw; };

    if (tid == 0) {
        for (int t = 0; t < NT; ++t) {
            mbar_init(&tfull[t], 1);
            mbar_init(&tempty[t], 1);
        }
        for (int s = 0; s < NS; ++s) {
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
        mbar_init(&mma_done, 1);
        for (int t = 0; t < NT; ++t) tok_issued[t] = 0;
        for (int r = 0; r < NR; ++r) raw_issued[r] = 0;
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    // launched as a programmatic dependent: the setup above overlaps the previous kernel's tail;
    // nothing it wrote is read before this wait
    pdl_wait();
    pdl_launch_dependents();

    if (warp < kTwConvWarp0) {
        // ---------------- producers ----------------
        // Warps 0-1 issue token boxes (slice sc by warp sc % 2 into slot sc % NS, once the slot's
        // previous MMAs are done); warps 2-3 issue raw weight boxes (slice sc by warp 2 + sc % 2
        // into raw stage sc % NR, once all converters have read its previous boxes).
        if (lane == 0) {
            const bool tok = warp < kTwTokWarps;
            const int pw = tok ? warp : warp - kTwTokWarps;
            uint32_t sc = 0;
            for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x) {
                int mt, nt;
                decode_tile(p, tile, mt, nt);
                const int e = p.tile_e[mt], r0 = p.tile_r0[mt];
                const int wy = e * p.wrows + nt * 128;        // first weight row of the slab
                // token boxes of the tile's valid rows rounded up to 16 (1..8 sixteen-row groups)
                const int n16 = !tok ? 0 : MOE_TOK_FIT ? (min(128, p.offsets[e + 1] - r0) + 15) / 16 : 8;
                const CUtensorMap* tmap = tok ? &tmTok.m[n16 - 1] : nullptr;
                bool ok = true;
                for (int kt = 0; kt < KT; ++kt, ++sc) {
                    if (static_cast<int>(sc % 2) != pw) continue;
                    if (abort_s) {                             // another role gave up: issue no more
                        ok = false;
                        break;
                    }
                    if (tok) {
                        const uint32_t s = sc % NT, u = sc / NT;
                        if (u > 0 && !tw_wait(Cfg::kTokOwn ? &tempty[s] : &sempty[s], (u - 1) & 1u)) {
                            ok = false;
                            break;
                        }
                        // rows past the expert's last row, up to the next 16, are loaded and never used
                        mbar_arrive_expect_tx(&tfull[s], static_cast<uint32_t>(n16) * 16 * 256);
                        tma_load_2d(smem_u32(stTok(s)), tmap, kt * kTwSliceK, r0, &tfull[s]);
                        tma_load_2d(smem_u32(stTok(s)) + kTwBox, tmap, kt * kTwSliceK + 64, r0, &tfull[s]);
                        tok_issued[s] = u + 1;
                    } else {
                        const uint32_t r = sc % NR, u = sc / NR;
                        if (u > 0 && !tw_wait(&rempty[r], (u - 1) & 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&rfull[r], Cfg::kRaw);
                        tma_load_2d(smem_u32(stRaw(r)), &tmW0, kt * Cfg::kRowBytes, wy, &rfull[r]);
                        if (NM == 2)
                            tma_load_2d(smem_u32(stRaw(r)) + 128 * Cfg::kRowBytes, &tmW1, kt * Cfg::kRowBytes, wy,
                                        &rfull[r]);
                        raw_issued[r] = u + 1;
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
        // (NM = 1). A thread converts its row's slice in pieces of 64 K (32 f16 pairs, one
        // 32-column TMEM store each): two pieces per matrix slice with NM = 2, its K half with
        // NM = 1. Raw rows: FP8 128 bytes in 16-byte chunks, 128-byte swizzle (chunk ^ row % 8);
        // NVFP4 64 bytes of packed codes, 64-byte swizzle (chunk ^ (row / 2) % 4). Eight
        // consecutive lanes read eight consecutive rows of one chunk, which the swizzle places in
        // eight distinct bank groups. The raw boxes are released once the last piece has been
        // converted; the TMEM slot is waited for only before the first store.
        const int cw = warp - kTwConvWarp0, qd = warp & 3, part = cw / 4;
        const int rrow = (NM == 2 ? part * 128 : 0) + 32 * qd + lane;       // raw row of this thread
        const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
        constexpr int kPieces = NM == 2 ? 2 : 1;                  // 64-K pieces per thread
        constexpr int kPieceChunks = FMT == 0 ? 4 : 2;            // 16-byte chunks per piece
        const int c0 = NM == 2 ? 0 : kPieceChunks * part;         // first chunk of this thread
        const int sw = FMT == 0 ? (rrow & 7) : ((rrow >> 1) & 3);
        uint32_t* tbl = w_scale[cw];
        const uint8_t* sfrow = nullptr;                    // NVFP4: this row's scale bytes
        uint4 sfv = make_uint4(0, 0, 0, 0);                // NVFP4: scale bytes of 2 slices (K 256)
        // FP8 block scales of (expert e, 128-row block nt), one per 128-wide K block
        const float* const sbase = NM == 2 && part == 1 ? p.s1 : p.s0;
        auto scale_row = [&](int e, int nt) { return sbase + (static_cast<size_t>(e) * (p.wrows / 128) + nt) * KB; };
        // FP8 gate/up: the next tile's expert, block and scales are fetched over the current
        // tile's last three slices (dependent loads one per slice, off the new tile's ramp) and
        // the scale table is rebuilt from registers between the tiles (measured: 2,178 -> 2,075
        // us). The others fetch them at the tile's start: the same prefetch made the down GEMMs
        // slower (FP8 1,294 -> 1,452 us) and left NVFP4 gate/up no faster.
        constexpr bool kAhead = NM == 2 && FMT == 0;
        int e_cur = 0, nt_cur = 0;
        if (kAhead && blockIdx.x < total) {
            int mt;
            decode_tile(p, blockIdx.x, mt, nt_cur);
            e_cur = p.tile_e[mt];
            if constexpr (FMT == 0) weight_prescale(scale_row(e_cur, nt_cur), KB, tbl);
            __syncwarp();
        }
        const int kt1 = KT >= 3 ? KT - 3 : 0, kt2 = KT >= 2 ? KT - 2 : 0, kt3 = KT - 1;
        uint32_t sc = 0;
        for (int tile = blockIdx.x; tile < total && !abort_s; tile += gridDim.x) {
            if constexpr (!kAhead) {
                int mt;
                decode_tile(p, tile, mt, nt_cur);
                e_cur = p.tile_e[mt];
                if constexpr (FMT == 0) {
                    __syncwarp();                          // the old table is no longer read
                    weight_prescale(scale_row(e_cur, nt_cur), KB, tbl);
                    __syncwarp();
                }
            }
            const int e = e_cur, nt = nt_cur;
            if constexpr (FMT == 1) {
                const size_t wr_ = static_cast<size_t>(e) * p.wrows + nt * 128 + (rrow & 127);
                sfrow = (NM == 2 && part == 1 ? p.sf1 : p.sf0) + wr_ * (K / 16);
            }
            const int ntile = tile + gridDim.x;
            int nf = 0, nc = 1, ne = 0, nnt = 0;
            float nsv0 = 0.0f, nsv1 = 0.0f;                // FP8: the next tile's scales kb = lane, lane + 32
            bool ok = true;
            for (int kt = 0; kt < KT; ++kt, ++sc) {
                if (kAhead && ntile < total) {
                    if (kt == kt1) {
                        const int m = ntile / p.n_tiles;
                        nf = p.tile_first[m];
                        nc = p.tile_cnt[m];
                    }
                    if (kt == kt2) {
                        const int local = ntile - p.n_tiles * nf;
                        nnt = local / nc;
                        ne = p.tile_e[nf + (local - nnt * nc)];
                    }
                    if (FMT == 0 && kt == kt3) {
                        const float* srow = scale_row(ne, nnt);
                        if (lane < KB) nsv0 = srow[lane];
                        if (lane + 32 < KB) nsv1 = srow[lane + 32];
                    }
                }
                const uint32_t r = sc % NR, ur = sc / NR, s = sc % NS, us = sc / NS;
                if (FMT == 1 && (kt & 1) == 0) sfv = __ldg(reinterpret_cast<const uint4*>(sfrow + kt * 8));
                if (!__all_sync(0xffffffffu, tw_wait(&rfull[r], ur & 1u))) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = stRaw(r) + rrow * Cfg::kRowBytes;
                const uint32_t ta = tmem + lane_off + Cfg::kA0 + s * Cfg::kACols + (NM == 2 ? part * Cfg::kMCols : part * 32);
#pragma unroll
                for (int pc = 0; pc < kPieces; ++pc) {
                    // the piece's chunks
                    uint4 wr[kPieceChunks];
#pragma unroll
                    for (int c = 0; c < kPieceChunks; ++c)
                        wr[c] = lds128(raw + (((c0 + pc * kPieceChunks + c) ^ sw) << 4));
                    uint32_t h[32];
                    if constexpr (FMT == 0) {
                        const uint32_t sc2 = tbl[kt];
#pragma unroll
                        for (int c = 0; c < kPieceChunks; ++c) {
                            const uint4 q = wr[c];
                            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                uint32_t lo, hi;
                                e4m3x4_to_f16x2x2(wv[i], lo, hi);
                                h[8 * c + 2 * i] = hmul2(lo, sc2);
                                h[8 * c + 2 * i + 1] = hmul2(hi, sc2);
                            }
                        }
                    } else {
                        // the piece's 4 scale bytes (one per 16 codes); E2M1 x E4M3 products are exact
                        const int wsel = (kt & 1) * 2 + (NM == 2 ? pc : part);
                        const uint32_t sfw = wsel == 0 ? sfv.x : wsel == 1 ? sfv.y : wsel == 2 ? sfv.z : sfv.w;
#pragma unroll
                        for (int c = 0; c < kPieceChunks; ++c) {
                            const uint4 q = wr[c];
                            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const uint32_t sf2 = e4m3_splat_f16x2((sfw >> (8 * (2 * c + (i >> 1)))) & 0xFFu);
                                uint32_t qq[4];
                                e2m1x8_to_f16x2x4(wv[i], qq[0], qq[1], qq[2], qq[3]);
#pragma unroll
                                for (int b = 0; b < 4; ++b) h[16 * c + 4 * i + b] = hmul2(qq[b], sf2);
                            }
                        }
                    }
                    // the raw boxes are released once the last piece has been converted (the
                    // conversion consumes the loaded registers): a release right after the
                    // shared-memory loads can let the next box land before they have returned
                    if (pc == kPieces - 1) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&rempty[r]);
                    }
                    if (pc == 0 && !__all_sync(0xffffffffu, us == 0 || tw_wait(&sempty[s], (us - 1) & 1u))) {
                        ok = false;
                        break;
                    }
                    tmem_st32(ta + pc * 32, h);
                }
                if (!ok) break;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[s]);
            }
            if (!ok) {
                abort_s = 1;
                break;
            }
            if (kAhead && ntile < total) {
                e_cur = ne;
                nt_cur = nnt;
                if constexpr (FMT == 0) {
                    __syncwarp();                          // the old table is no longer read
                    prescale_from_regs(nsv0, nsv1, KB, tbl);
                    __syncwarp();
                }
            }
        }
    } else if (warp == kTwMmaWarp) {
        // ---------------- MMA issuer ----------------
        // Lane 0 issues. This warp touches no memory in its loop: a shared-memory access (an
        // mbarrier wait included) by the issuing thread waits for the MMAs queued before it,
        // i.e. drains the tensor pipe (measured: ~290 instead of ~70 cycles per M=128 MMA).
        // The watcher warp waits for each slice's operands instead and releases this warp
        // through named barrier kTwIssueBar: per tile one reduction whose result is the tile's
        // MMA width / 16 (0: stop), then a plain barrier per further slice (a reduction per
        // slice costs ~250 cycles more than a plain barrier and starves the pipe).
        uint32_t sc = 0, tcount = 0;
        while (true) {
            const uint32_t n16 = bar_red_popc(kTwIssueBar, 64, false);
            if (n16 == 0) break;
            const uint32_t b = tcount % Cfg::kAcc;
            const uint32_t d0 = tmem + b * Cfg::kAccCols;
            // MMA width = the tile's valid rows rounded up to 16
            const uint32_t idesc = (kIdesc128 & ~(0x3Fu << 17)) | ((2u * n16) << 17);
            for (int kt = 0; kt < KT; ++kt, ++sc) {
                if (kt > 0) named_bar_sync(kTwIssueBar, 64);
                if (lane == 0) {
                    const uint32_t s = sc % NS, t = sc % NT;
                    tc_fence_after();
                    const uint32_t tok = smem_u32(stTok(t));
                    const uint32_t a0 = tmem + Cfg::kA0 + s * Cfg::kACols;
#pragma unroll
                    for (int kk = 0; kk < kTwSliceK / 16; ++kk) {
                        // K16 step kk: token box kk / 4, 32-byte column group kk % 4 of its rows
                        const uint64_t bdesc = smem_desc_sw128(tok + (kk >> 2) * kTwBox + (kk & 3) * 32);
#pragma unroll
                        for (int m = 0; m < NM; ++m)
                            mma_issue_tmem_a(d0 + m * 128, a0 + m * Cfg::kMCols + kk * 8, bdesc, idesc,
                                             (kt > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&sempty[s]);
                    if (Cfg::kTokOwn) mma_commit(&tempty[t]);
                    if (kt == KT - 1) mma_commit(&acc_full[b]);
                }
            }
            ++tcount;
        }
        // one more commit: it arrives once every MMA this thread queued has completed (the
        // teardown waits for it before TMEM and shared memory are released)
        if (lane == 0) mma_commit(&mma_done);
    } else if (warp == kTwWatchWarp) {
        // ---------------- watcher ----------------
        // Per slice: the accumulator drained (first slice of a tile), the token boxes landed and
        // the weight slice in TMEM; then the release of the MMA warp - the tile's first slice
        // by a reduction carrying the MMA width (lanes < n16 vote true; 0 on a timeout or an
        // abort), every further slice by a plain barrier. After a failed wait the rest of the
        // tile is released without waiting (the MMA warp cannot be stopped inside a tile; its
        // results are discarded with the error bit) and the next reduction stops it. A final 0
        // ends the MMA warp's loop.
        uint32_t sc = 0, tcount = 0;
        bool ok = true;
        bool live = true;                                  // the MMA warp is still in its loop
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++tcount) {
            int mt, nt;
            decode_tile(p, tile, mt, nt);
            const int rows = min(128, p.offsets[p.tile_e[mt] + 1] - p.tile_r0[mt]);
            const int n16 = (rows + 15) >> 4;              // >= 1: a tile has at least one row
            const uint32_t b = tcount % Cfg::kAcc, v = tcount / Cfg::kAcc;
            for (int kt = 0; kt < KT; ++kt, ++sc) {
                const uint32_t s = sc % NS, us = sc / NS, t = sc % NT, ut = sc / NT;
                if (lane == 0 && ok) {
                    ok = !abort_s;
                    if (ok && kt == 0 && v > 0) ok = tw_wait(&acc_empty[b], (v - 1) & 1u);
                    if (ok) ok = tw_wait(&tfull[t], ut & 1u) && tw_wait(&afull[s], us & 1u);
                    if (!ok) {                                 // stop the producers before the MMA
                        abort_s = 1;                           // warp is released without operands
                        __threadfence_block();
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (kt == 0) {
                    if (bar_red_popc(kTwIssueBar, 64, ok && lane < n16) == 0) {
                        live = false;                      // the MMA warp has left its loop
                        break;
                    }
                } else {
                    named_bar_sync(kTwIssueBar, 64);
                }
            }
        }
        // every release the MMA warp waits for is sent: a final 0 unless a reduction already
        // returned 0 (then both warps left their loops at the same barrier)
        if (live) bar_red_popc(kTwIssueBar, 64, false);
        if (!ok && lane == 0) abort_s = 1;
    } else {
        // ---------------- epilogue ----------------
        // Warp w reads TMEM lanes 32*(w%4)..+31 (lane = weight row f of the tile's slab) and token
        // columns 64*h..+63, h = (w - 12) / 4. Each store instruction writes one token row's 32
        // consecutive features (128 contiguous bytes).
        // per epilogue warp and column: the factor of the accumulator - the token's or row's
        // activation scale times the weight block's inverse prescale (gate/up: gate in xs_s, up
        // in ys_s; down: in ys_s, with y's power of two for f16)
        __shared__ float xs_s[kTwEpiWarps][64];
        __shared__ float ys_s[kTwEpiWarps][64];
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
                xs_s[ew][32 * i + lane] = KIND == 0       ? p.a_inv[p.sorted_pair[rr] / p.topk]
                                          : p.a_inv != nullptr ? p.a_inv[rr]
                                                               : p.a16_scale;
            }
            const size_t sblk = static_cast<size_t>(e) * (p.wrows / 128) + nt;
            float winv0, winv1;                            // undo the converters' weight scaling
            if constexpr (FMT == 0) {
                winv0 = weight_prescale(p.s0 + sblk * KB, KB, nullptr);
                winv1 = KIND == 0 ? weight_prescale(p.s1 + sblk * KB, KB, nullptr) : winv0;
            } else {
                winv0 = scale2_of(p.s2_0, p.s2e_0, p.s2_stride, e);   // NVFP4: the expert's scale_2
                winv1 = KIND == 0 ? scale2_of(p.s2_1, p.s2e_1, p.s2_stride, e) : winv0;
            }
            if constexpr (KIND == 1) {
                // y goes out in f16 times 2^g, g from |y[r][j]| <= A_r * sum_i |W[j][i]|: A_r the
                // row's max |a| (range-scaled activations) or the m-tile's (f16 activations under
                // the clamp), both from the gate/up epilogue - the f16 rounding of a and the fp32
                // sums stay inside the factor 2 between 2^15 and f16's largest value - and the
                // weight sum 128 * 448 * (sum of the block's scales) for FP8, K * 6 * 448 *
                // |the expert's scale_2| for NVFP4 (E2M1 <= 6, E4M3 scale bytes <= 448)
                const float wsum = FMT == 0 ? 57344.0f * block_scale_abs_sum(p.s0 + sblk * KB, KB)
                                            : static_cast<float>(p.K) * 2688.0f * fabsf(winv0);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int t = 32 * i + lane;
                    const float arow = p.a_inv != nullptr ? __uint_as_float(p.amax[r0 + min(cbase + t, rows - 1)])
                                                          : __uint_as_float(p.tmax[mt]);
                    const int g = pow2_bound_exponent(arow, wsum);
                    ys_s[ew][t] = (xs_s[ew][t] * winv0) * __int_as_float((127 + g) << 23);
                    if (qd == 0 && cbase + t < rows)
                        p.yexp[static_cast<size_t>(r0 + cbase + t) * p.n_tiles + nt] = static_cast<int8_t>(g);
                }
            }
            if constexpr (KIND == 0) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int t = 32 * i + lane;
                    ys_s[ew][t] = xs_s[ew][t] * winv1;
                    xs_s[ew][t] = xs_s[ew][t] * winv0;
                }
            }
            __syncwarp();
            const uint32_t b = tcount % Cfg::kAcc, v = tcount / Cfg::kAcc;
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(&acc_full[b], v & 1u))) {
                abort_s = 1;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem + lane_off + b * Cfg::kAccCols + cbase;
            float* dst = KIND == 0 ? p.out + static_cast<size_t>(r0 + cbase) * p.out_ld + nt * 128 + f : nullptr;
            __half* dsty = KIND == 1 ? p.y16 + static_cast<size_t>(r0 + cbase) * p.out_ld + nt * 128 + f : nullptr;
            __half* dst16 = KIND == 0 && p.out16 != nullptr
                                ? p.out16 + static_cast<size_t>(r0 + cbase) * p.out_ld + nt * 128 + f
                                : nullptr;
            const int vrows = rows - cbase;                // valid columns of this warp
            float amax_t = 0.0f;                           // gate/up, f16 path: max |a| seen in the tile
#pragma unroll 1
            for (int c0 = 0; c0 < 64 && c0 < vrows; c0 += 16) {
                if (KIND == 0) {
                    float gv[16], uv[16];
                    tmem_ld16x2(taddr + c0, taddr + 128 + c0, gv, uv);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = c0 + j;
                        // the clamped SwiGLU with silu(g) = g/2 * (1 + tanh(g/2)): one SFU operation
                        // (tanh.approx, about 2^-11 absolute error) instead of an exponential and a
                        // divide - the epilogue holds the single accumulator, so its length stalls
                        // the MMA (measured: gate/up GEMM 2,164 -> 2,134 us)
                        const float gg = fminf(gv[j] * xs_s[ew][t], p.limit);
                        const float uu = fminf(fmaxf(uv[j] * ys_s[ew][t], -p.limit), p.limit);
                        const float hg = 0.5f * gg;
                        const float h = hg * (1.0f + tanh_approx(hg)) * uu;
                        if (dst16 != nullptr) {                // bounded by the clamp: f16 as is
                            if (t < vrows) {
                                dst16[static_cast<size_t>(t) * p.out_ld] = __float2half_rn(h * p.a16_scale);
                                amax_t = fmaxf(amax_t, fabsf(h));
                            }
                        } else {
                            const uint32_t mb = warp_max_bits(fabsf(h));
                            if (t < vrows) {
                                dst[static_cast<size_t>(t) * p.out_ld] = h;
                                if (lane == 0) atomicMax(p.amax + r0 + cbase + t, mb);
                            }
                        }
                    }
                } else {
                    float yv[16];
                    tmem_ld16(taddr + c0, yv);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = c0 + j;
                        if (t < vrows) dsty[static_cast<size_t>(t) * p.out_ld] = __float2half_rn(yv[j] * ys_s[ew][t]);
                    }
                }
            }
            if (KIND == 0 && dst16 != nullptr) {           // the m-tile's max |a| (all its n-tiles)
                const uint32_t mb = warp_max_bits(amax_t);
                if (lane == 0) atomicMax(p.tmax + mt, mb);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
    }

    // ---------------- teardown ----------------
    // Every role has left its loop. Without an abort every box issued was waited for by its
    // consumer and every MMA by the epilogue; after one, boxes may still be landing and MMAs still
    // running, so the CTA waits for the last phase of each token slot and raw stage that received
    // a box, and for the MMA warp's final commit, before TMEM and shared memory are released.
    __syncthreads();
    {
        bool drained = true;
        if (tid == 0) {
            drained = tw_wait(&mma_done, 0);
        } else if (abort_s && tid <= NT) {
            const uint32_t n = tok_issued[tid - 1];
            if (n > 0) drained = tw_wait(&tfull[tid - 1], (n - 1) & 1u);
        } else if (abort_s && tid <= NT + NR) {
            const uint32_t n = raw_issued[tid - 1 - NT];
            if (n > 0) drained = tw_wait(&rfull[tid - 1 - NT], (n - 1) & 1u);
        }
        if (abort_s && tid == 0 && p.err != nullptr) atomicOr(p.err, 2);
        if (!drained && p.err != nullptr) atomicOr(p.err, 4);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

namespace {

// 2-D map over a row-major [rows][inner] matrix of elem-byte elements, box box_inner x 128.
bool tw_map(CUtensorMap* m, CUtensorMapDataType dt, int elem, const void* base, uint64_t inner, uint64_t rows,
            uint32_t box_inner, CUtensorMapSwizzle sw) {
    return encode_map_2d(m, dt, elem, base, inner, rows, box_inner, 128, sw);
}

template <int KIND, int NM, int DB, int FMT>
cudaError_t launch_tw(const PrefillGemmArgs& q, const TokMaps& a, const CUtensorMap& w0, const CUtensorMap& w1,
                      int grid, cudaStream_t stream) {
    using Cfg = TwCfg<NM, DB, FMT>;
    cudaError_t st = cudaFuncSetAttribute(prefill_tw_gemm_kernel<KIND, NM, DB, FMT>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (st != cudaSuccess) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTwThreads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((st = cudaLaunchKernelEx(&cfg, prefill_tw_gemm_kernel<KIND, NM, DB, FMT>, q, a, w0, w1)) != cudaSuccess)
        return st;
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
    TokMaps ma;
    CUtensorMap mw0, mw1;
    const uint64_t wrows_all = static_cast<uint64_t>(p.experts) * p.wrows;
    const bool fp4 = p.fmt == 1;
    if (fp4 && ((reinterpret_cast<uintptr_t>(p.sf0) | reinterpret_cast<uintptr_t>(p.sf1)) & 15u))
        return cudaErrorMisalignedAddress;
    // FP8: rows of K code bytes, boxes of 128 bytes (128-byte swizzle); NVFP4: rows of K/2 bytes
    // of packed codes, boxes of 64 bytes (64-byte swizzle): one 128-wide K slice of 128 rows
    const uint64_t wbytes = fp4 ? p.K / 2 : p.K;
    const uint32_t wbox = fp4 ? 64 : 128;
    const CUtensorMapSwizzle wsw = fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    bool ok = tw_map(&mw0, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w0, wbytes, wrows_all, wbox, wsw) &&
              tw_map(&mw1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.w1, wbytes, wrows_all, wbox, wsw);
    // token rows (f16, 64-element boxes, 128-byte swizzle), one map per box height 16 .. 128
    for (int i = 0; i < 8 && ok; ++i)
        ok = encode_map_2d(&ma.m[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.a, p.K, p.a_rows, 64, 16 * (i + 1),
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;
    if (kind == 0) return fp4 ? launch_tw<0, 2, 0, 1>(q, ma, mw0, mw1, sms, stream)
                              : launch_tw<0, 2, 0, 0>(q, ma, mw0, mw1, sms, stream);
    return fp4 ? launch_tw<1, 1, 1, 1>(q, ma, mw0, mw1, sms, stream) : launch_tw<1, 1, 1, 0>(q, ma, mw0, mw1, sms, stream);
}

}  // namespace moe
