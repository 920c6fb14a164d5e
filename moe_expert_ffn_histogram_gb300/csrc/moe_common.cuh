// Device helpers and the workspace layout shared by the sm_103a kernels of libmoe_ffn_gb300.
//
// Tile convention used by every GEMV kernel (one warp = one 16-row tile of A):
//   mma.sync m16n8k16 (f16 x f16 -> f32). Lane L = 4*g + c (g = L>>2 in 0..7, c = L&3).
//   A rows g and g+8 are two weight rows; lane (g, c) loads the bytes of physical K positions
//   k0 + 16c .. k0 + 16c + 15 of each of its two rows, and feeds element 4i+{0,1} as logical
//   K (2c, 2c+1) and 4i+{2,3} as logical K (2c+8, 2c+9) of MMA step i (i = 0..3). B column n is
//   the activation vector of column n (a token or a routed pair), read at the SAME physical
//   positions, so each MMA step sums a permutation of 16 consecutive-in-memory K products.
//   One 64-wide K segment = 4 MMA steps.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

constexpr int kMaxTopk = 8;
constexpr int kMaxCols = 8;          // B columns per MMA tile (n = 8)
constexpr int kFeatBlock = 64;       // features per gate/up CTA, = K width of one a-scale block
// features per single-token NVFP4 gate/up CTA (decode_fp4.cu), = the K width of its a-scale
// blocks: 32 spreads the 2 x 8 x I/16 warps of one token over 4-warp CTAs (several per SM, so
// that no SM carries twice the loads of another); 64 is the 8-warp layout of the other kernels
#ifndef MOE_FP4T_FEAT
#define MOE_FP4T_FEAT 32
#endif
constexpr int kFp4TokFeat = MOE_FP4T_FEAT;
static_assert(kFp4TokFeat == 32 || kFp4TokFeat == 64, "single-token NVFP4 feature block");
constexpr int kDownRows = 16;        // output rows per down/combine CTA
constexpr int kPlanThreads = 1024;
constexpr int kMaxPlanExperts = 4096;

// ---- workspace -------------------------------------------------------------------------------

struct WsLayout {
    size_t barrier;
    size_t group_count, group_expert, group_start, group_ncols;
    size_t counts, offsets, sorted_pair, pair_to_sorted;
    size_t act, act_scale;
    size_t total;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// rows: tokens handled per sub-batch (<= 8); pairs = rows * topk. act_blk: the K width of one
// activation-scale block (kFeatBlock; NVFP4 banks reserve room for kFp4TokFeat-wide blocks, which
// the single-token kernels write).
__host__ __device__ inline WsLayout ws_layout(int rows, int I, int E, int topk, int act_blk = kFeatBlock) {
    const size_t P = static_cast<size_t>(rows) * topk;
    WsLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    L.barrier = take(16);
    L.group_count = take(16);
    L.group_expert = take(P * 4);
    L.group_start = take(P * 4);
    L.group_ncols = take(P * 4);
    L.counts = take(static_cast<size_t>(E) * 4);
    L.offsets = take((static_cast<size_t>(E) + 1) * 4);
    L.sorted_pair = take(P * 4);
    L.pair_to_sorted = take(P * 4);
    L.act = take(P * static_cast<size_t>(I) * 2);
    L.act_scale = take(P * static_cast<size_t>(I / (act_blk < kFeatBlock ? act_blk : kFeatBlock)) * 4);
    L.total = o;
    return L;
}

// How routed pairs are grouped for the GEMV kernels. Implicit mode (T == 1): group k is slot k
// with one column, its expert read straight from topk_ids. Table mode (T > 1): groups come from
// the plan kernel (one expert, up to `cap` columns each, columns = pairs in ascending order).
struct Groups {
    const int32_t* ids;           // [T*topk]
    const int32_t* count;         // nullptr = implicit
    const int32_t* expert;
    const int32_t* start;
    const int32_t* ncols;
    const int32_t* sorted_pair;
    int topk;
    int E;
};

// ---- conversions -----------------------------------------------------------------------------

// Two E4M3 bytes (low 16 bits of w, then high 16 bits) -> two f16x2 (exact: every E4M3 value,
// subnormals included, is an f16 normal).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 p, q;\n\tmov.b32 {p, q}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, p;\n\tcvt.rn.f16x2.e4m3x2 %1, q;\n\t}"
        : "=r"(lo), "=r"(hi) : "r"(w));
}

// Four bytes of packed E2M1 (two codes each) -> four f16x2, byte b -> r[b] (exact).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(w));
}

// Two E4M3 bytes (low 16 bits of w: byte 0, byte 1) -> f16x2 {byte 0, byte 1} (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
    uint32_t r;
    asm("{\n\t.reg .b16 p, q;\n\tmov.b32 {p, q}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, p;\n\t}" : "=r"(r) : "r"(w));
    return r;
}

// One E4M3 scale byte -> {sf, sf} as f16x2.
__device__ __forceinline__ uint32_t e4m3_splat_f16x2(uint32_t byte) {
    uint32_t r;
    const uint32_t two = (byte & 0xFFu) * 0x0101u;
    asm("{\n\t.reg .b16 p, q;\n\tmov.b32 {p, q}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, p;\n\t}"
        : "=r"(r) : "r"(two));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// D += A * B, m16n8k16, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- memory ----------------------------------------------------------------------------------

// Weight stream: read once, keep it out of L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream_u8(const void* p) {
    uint32_t v;
    asm("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Fire-and-forget bulk prefetch of [p, p + bytes) into L2 (bytes a multiple of 16, p 16-aligned):
// no registers, no shared memory, no completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Bulk L2 prefetch of [p, p + bytes) in chunks of at most 64 KB; p 16-byte aligned, the tail
// below 16 bytes is left out.
__device__ __forceinline__ void prefetch_l2_range(const uint8_t* p, size_t bytes) {
    bytes &= ~static_cast<size_t>(15);
    for (size_t o = 0; o < bytes; o += 65536) {
        const size_t n = bytes - o < 65536 ? bytes - o : 65536;
        prefetch_l2(p + o, static_cast<uint32_t>(n));
    }
}

// Programmatic dependent launch (1: on): a dependent kernel is launched while the one before it
// on the stream still runs, does its setup, and waits in griddepcontrol.wait for that grid's
// completion before it reads what the grid wrote.
#ifndef MOE_PDL
#define MOE_PDL 1
#endif

// Programmatic dependent launch: let the next kernel on the stream start launching, and (in that
// kernel) wait until every grid it depends on has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Asynchronous global -> shared copies (per-thread, completion tracked with commit/wait groups).
// 16-byte copies bypass L1 (.cg); 8- and 4-byte copies only exist in the .ca form.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint2 lds64(const void* p) { return *reinterpret_cast<const uint2*>(p); }

// ---- power-of-two range scales -----------------------------------------------------------------

// For a block whose largest magnitude is m, return s = 2^(15 - e) with m < 2^e, so |v * s| < 2^15
// (inside f16's finite range) for every v of the block, and set inv = 1/s. Both are exact powers
// of two, so scaling and unscaling add no rounding. m == 0 or non-finite -> s = 1.
__device__ __forceinline__ float pow2_range_scale(float m, float& inv) {
    if (!(m > 0.0f) || !isfinite(m)) {
        inv = 1.0f;
        return 1.0f;
    }
    int e;
    frexpf(m, &e);
    int s = 15 - e;
    s = s < -100 ? -100 : (s > 100 ? 100 : s);
    inv = __int_as_float((127 - s) << 23);
    return __int_as_float((127 + s) << 23);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace moe
