// Shared pieces of the grouped-GEMM (prefill) tier: tile shape, the GEMM argument block and the
// per-tile helpers of the tensor-memory GEMM core (prefill_tw.cu).
#pragma once
#include "gemv_items.cuh"

namespace moe {

namespace prefill {

constexpr int kBM = 128;               // sorted rows per tile
constexpr int kBN = 128;               // weight rows per tile (gate/up: 128 gate + the same 128 up)

}  // namespace prefill

struct PrefillGemmArgs {
    // tile schedule
    const int32_t* tiles;        // [1] number of m-tiles
    const int32_t* tile_e;       // [m-tiles]
    const int32_t* tile_r0;      // [m-tiles]
    const int32_t* tile_first;   // [m-tiles] first m-tile of the tile's expert
    const int32_t* tile_cnt;     // [m-tiles] number of m-tiles of the tile's expert
    const int32_t* offsets;      // [E+1]
    const int32_t* sorted_pair;  // [P]
    int topk, K, n_tiles;
    // A operand: sorted rows of x16 (KIND 0) or of a16 (KIND 1), f16
    const __half* a;
    const float* a_inv;          // per token (KIND 0) or per sorted row (KIND 1)
    // B operand: E4M3 weight rows and fp32 block scales; KIND 0 uses both gate (w0) and up (w1)
    const uint8_t* w0;
    const float* s0;
    const uint8_t* w1;
    const float* s1;
    int wrows;                   // rows of one expert's weight matrix (I for gate/up, H for down)
    float limit;
    // outputs
    float* out;                  // KIND 0: a32 [P][I]
    // KIND 1: y [P][H] in f16 as y * 2^g, g = yexp[row][n-tile] chosen per sorted row and 128-row
    // output block from a bound on |y| (so that |y| * 2^g < 2^15); the combine multiplies by 2^-g
    __half* y16;
    int8_t* yexp;                // [P][H / 128]
    uint32_t* amax;              // per sorted row max |a| (float bits) of the range-scaled path:
                                 // KIND 0 writes it (zeroed before), KIND 1 reads it for y's factor
    uint32_t* tmax;              // per m-tile max |a| (float bits) of the f16 path (out16): the same
    // KIND 0, TMEM core: when set, a goes straight to f16 here ([P][I]) as a * a16_scale, one power
    // of two for all rows (a finite clamp limit L <= 255 bounds |a| by L^2, and L^2 * a16_scale <
    // 2^15), out and amax are not used (tmax is); KIND 1 then runs with a_inv == nullptr and
    // a16_scale holding the inverse
    __half* out16;
    float a16_scale;
    int out_ld;                  // I (KIND 0) or H (KIND 1)
    int32_t* err;                // optional error word (bit 1: a bounded wait gave up)
    int a_rows;                  // rows of the A matrix: T (KIND 0) or P (KIND 1)
    int experts;                 // E
    // NVFP4 weights (prefill_tw.cu only): w0/w1 hold packed E2M1 codes [E][wrows][K/2], sf0/sf1
    // the E4M3 scale bytes [E][wrows][K/16], s2_0/s2_1 the per-projection scale_2
    int fmt;                     // 0 FP8 E4M3 block-128, 1 NVFP4
    const uint8_t* sf0;
    const uint8_t* sf1;
    float s2_0, s2_1;
    // NVFP4 with one scale_2 per expert (null: s2_0 / s2_1): expert e's is s2e_0[e * s2_stride]
    const float* s2e_0;
    const float* s2e_1;
    int s2_stride;
};

// (m-tile, n-tile) of work item `tile` in expert-major, n-tile-middle, m-tile-minor order: the
// CTAs running at one time share few weight slabs (each slab is read from HBM about once and
// served to the expert's m-tiles from L2) while the expert's activation rows stay in L2.
__device__ __forceinline__ void decode_tile(const PrefillGemmArgs& p, int tile, int& mt, int& nt) {
    const int m = tile / p.n_tiles;
    const int first = p.tile_first[m], cnt = p.tile_cnt[m];
    const int local = tile - p.n_tiles * first;
    nt = local / cnt;
    mt = first + (local - nt * cnt);
}

// Prescale of one (expert, 128-row weight block) scale row: f16x2 splats of scale * 2^p per
// 128-wide K block into tbl (if non-null) and 2^-p returned, with 2^p chosen so that 448 * scale
// * 2^p stays below 2^15. One warp.
__device__ __forceinline__ float weight_prescale(const float* srow, int KB, uint32_t* tbl) {
    const int lane = threadIdx.x & 31;
    float m = 0.0f;
    for (int kb = lane; kb < KB; kb += 32) m = fmaxf(m, fabsf(srow[kb]));
    m = warp_max(m) * 448.0f;
    float inv;
    const float pre = pow2_range_scale(m, inv);
    if (tbl != nullptr)
        for (int kb = lane; kb < KB; kb += 32) {
            const __half h = __float2half_rn(srow[kb] * pre);
            tbl[kb] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&h)) * 0x10001u;
        }
    return inv;
}

// sum over the KB 128-wide K blocks of |scale| of one (expert, 128-row weight block) scale row, the
// same value in every lane (a fixed shuffle tree). One warp.
__device__ __forceinline__ float block_scale_abs_sum(const float* srow, int KB) {
    const int lane = threadIdx.x & 31;
    float v = 0.0f;
    for (int kb = lane; kb < KB; kb += 32) v += fabsf(srow[kb]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exponent g with a * w * 2^g < 2^15 for positive finite a and w (0 when either is zero or not
// finite), clamped to [-100, 100]: with m = a * w < 2^(ea + ew), g = 15 - ea - ew.
__device__ __forceinline__ int pow2_bound_exponent(float a, float w) {
    if (!(a > 0.0f) || !(w > 0.0f) || !isfinite(a) || !isfinite(w)) return 0;
    int ea, ew;
    frexpf(a, &ea);
    frexpf(w, &ew);
    const int g = 15 - ea - ew;
    return g < -100 ? -100 : (g > 100 ? 100 : g);
}

// The same table from scales already in registers: lane holds kb = lane (v0) and lane + 32 (v1),
// zero past KB (KB <= 64). One warp.
__device__ __forceinline__ void prescale_from_regs(float v0, float v1, int KB, uint32_t* tbl) {
    const int lane = threadIdx.x & 31;
    const float m = warp_max(fmaxf(fabsf(v0), fabsf(v1))) * 448.0f;
    float inv;
    const float pre = pow2_range_scale(m, inv);
    auto splat = [&](float v) {
        const __half h = __float2half_rn(v * pre);
        return static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&h)) * 0x10001u;
    };
    if (lane < KB) tbl[lane] = splat(v0);
    if (lane + 32 < KB) tbl[lane + 32] = splat(v1);
}


// Transposed variant with the dequantised weights as the MMA's TMEM operand (prefill_tw.cu);
// FP8 or NVFP4 weights (p.fmt).
cudaError_t launch_prefill_gemm_tw(int kind, const PrefillGemmArgs& p, int N_total, cudaStream_t stream);

}  // namespace moe
