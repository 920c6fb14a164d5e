// Kernel argument blocks and launchers of libmoe_ffn_gb300 (internal to the library).
#pragma once
#include "moe_common.cuh"

namespace moe {

// Gate + up projections with the clamped SwiGLU fused (gate_up.cu).
struct GateUpArgs {
    const __nv_bfloat16* x;
    int H, I;
    const uint8_t* wg;
    const uint8_t* wu;
    const float* sg;      // FP8 block scales [E][I/128][H/128]
    const float* su;
    const uint8_t* sfg;   // NVFP4 scale bytes [E][I][H/16]
    const uint8_t* sfu;
    float s2g, s2u;       // NVFP4 scale_2
    // NVFP4 with one scale_2 per expert: expert e's is s2g_e[e * s2_stride] (null: s2g for all)
    const float* s2g_e;
    const float* s2u_e;
    int s2_stride;
    float limit;
    Groups grp;
    __half* act;          // [P][I] f16, range-scaled
    float* act_scale;     // [P][I/64] inverse range scale ([P][I/32] in the single-token NVFP4 kernels)
    int32_t* err;
    // Single-token NVFP4 calls whose weights fit in L2: each CTA first asks L2 for its own gate/up
    // rows and for its share of its expert's down matrix (bulk prefetch), so that HBM streams the
    // whole working set at once while the warps consume it from L2.
    int l2_prefetch;
    const uint8_t* pf_wd;  // down codes [E][H][I/2]
    const uint8_t* pf_sfd; // down scale bytes [E][H][I/16]
};

// NVFP4 scale_2 of expert e: its entry of the per-expert table when there is one, else the
// projection's scalar.
__device__ __forceinline__ float scale2_of(float s2, const float* s2e, int stride, int e) {
    return s2e != nullptr ? __ldg(s2e + static_cast<size_t>(e) * stride) : s2;
}

// Single-token NVFP4 calls ask L2 for their whole weight set up front (0: they do not).
#ifndef MOE_FP4_L2_PREFETCH
#define MOE_FP4_L2_PREFETCH 1
#endif

// Down projection fused with the slot-order combine (down_combine.cu).
struct DownArgs {
    int T, H, I, topk, E;
    const int32_t* ids;     // [T][topk]
    const float* wts;       // [T][topk]
    const uint8_t* wd;
    const float* sd;        // FP8 block scales [E][H/128][I/128]
    const uint8_t* sfd;     // NVFP4 scale bytes [E][H][I/16]
    float s2d;
    const float* s2d_e;     // NVFP4, one scale_2 per expert: s2d_e[e * s2_stride] (null: s2d)
    int s2_stride;
    Groups grp;
    const __half* act;      // [P][I]
    const float* act_scale; // [P][I/64] ([P][I/32] in the single-token NVFP4 kernels)
    __nv_bfloat16* out;     // [T][H]
    // layer epilogue (nullable): out = bf16((sum_k w*y + shared) + residual), fp32 adds in that order
    const __nv_bfloat16* shared;     // [T][H] shared-expert output
    const __nv_bfloat16* residual;   // [T][H]
};

// FMT: 0 = FP8 E4M3 with 128x128 block scales, 1 = NVFP4.
template <int FMT> cudaError_t launch_gate_up(const GateUpArgs& a, int num_groups, int max_cols,
                                              cudaStream_t stream);
template <int FMT> cudaError_t launch_down_combine(const DownArgs& a, cudaStream_t stream);
size_t gate_up_smem_bytes(int H, int max_cols);
size_t down_smem_bytes(int T, int topk);

// Single-token NVFP4 decode (decode_fp4.cu): the same workspace format as launch_gate_up /
// launch_down_combine for one token, fewer instructions per weight byte.
cudaError_t launch_fp4_token_gate_up(const GateUpArgs& a, int topk, cudaStream_t stream);
cudaError_t launch_fp4_token_down(const DownArgs& a, bool pdl, cudaStream_t stream);

// The whole forward of one sub-batch in one cooperative launch (fused.cu); `barrier` is a
// workspace word, zeroed by the launcher with a memset on `stream`.
template <int FMT> cudaError_t launch_fused_forward(const GateUpArgs& ga, const DownArgs& da,
                                                    unsigned* barrier, int rows, int cap,
                                                    cudaStream_t stream);
size_t fused_smem_bytes(int H, int rows, int topk, int cap);
// Test hook of the fused kernel's grid barrier (moe_test_barrier_timeout).
void set_test_barrier_timeout(bool on);

// Wide tier (prefill.cu): workspace layout and the launch sequence of the grouped-GEMM path.
struct PrefillLayout {
    size_t counts, offsets, sorted_pair, pair_to_sorted, tiles, tile_e, tile_r0, tile_first, tile_cnt;
    size_t x16, xinv, amax, a16, ainv, f32, tmax, yexp, plan_blk, total;
};
PrefillLayout prefill_layout(int T, int H, int I, int E, int topk);
// Weights of the three projections for the prefill tier: FP8 codes + fp32 block scales, or
// NVFP4 packed codes + E4M3 scale bytes + scale_2.
struct PrefillWeights {
    const uint8_t *wg, *wu, *wd;
    const float *sg, *su, *sd;        // FP8
    const uint8_t *sfg, *sfu, *sfd;   // NVFP4
    float s2g, s2u, s2d;              // NVFP4
    // NVFP4 with one scale_2 per expert and projection (null: the scalars above)
    const float *s2g_e, *s2u_e, *s2d_e;
    int s2_stride;
};
cudaError_t launch_prefill(int fmt, const __nv_bfloat16* x, int T, int H, int I, int E, int topk,
                           const int32_t* ids, const float* wts, const PrefillWeights& wt, float limit,
                           __nv_bfloat16* out, uint8_t* ws, const PrefillLayout& L, int32_t* err,
                           cudaStream_t stream, const __nv_bfloat16* shared = nullptr,
                           const __nv_bfloat16* residual = nullptr);

// Router (router.cu): K-split factor for (T, H, E), top-k shared memory, and the two launches.
int router_ksplit(int T, int H, int E, int sms);
size_t router_topk_smem_bytes(int E);
cudaError_t launch_router(const __nv_bfloat16* x, int T, int H, const __nv_bfloat16* w, const float* bias, int E,
                          int topk, float routed_scale, int renorm, float* logits, int32_t* ids, float* wts,
                          float* part, int KS, cudaStream_t stream);

// Dense bf16 product partials: part[ks][t][n] = sum over K chunk range ks of x[t][:] . w[n][:]
// (x [T][K], w [N][K], N % 16 == 0, K % 32 == 0; the router's logits kernel).
cudaError_t launch_dense_bf16(const __nv_bfloat16* x, int T, int K, const __nv_bfloat16* w, int N, float* part,
                              int KS, cudaStream_t stream);
// Plain streaming read of [p, p + bytes) (bytes a positive multiple of 16, p 16-byte aligned)
// XOR-folded into *sink (stream_read.cu): the benchmark's size-matched read ceiling.
cudaError_t launch_stream_read(const void* p, size_t bytes, uint32_t* sink, int sms, cudaStream_t stream);
// Shared expert (shared_expert.cu): workspace bytes and the launches.
size_t shared_expert_ws_bytes(int T, int H, int S, int sms);
cudaError_t launch_shared_expert(const __nv_bfloat16* x, int T, int H, int S, const __nv_bfloat16* wg,
                                 const __nv_bfloat16* wu, const __nv_bfloat16* wd, float limit,
                                 __nv_bfloat16* out, uint8_t* ws, int sms, cudaStream_t stream);

// The grouped tier's m-tile list (the tiles of rows_per_tile sorted rows of each expert, in
// ascending expert order): tiles[0] = number of m-tiles; tile_e[i], tile_r0[i] = expert and first
// sorted row of tile i; tile_first[i], tile_cnt[i] = first m-tile and number of m-tiles of that
// expert. Null tiles: no list.
struct TileList {
    int32_t* tiles;
    int32_t* tile_e;
    int32_t* tile_r0;
    int32_t* tile_first;
    int32_t* tile_cnt;
    int rows_per_tile;
};

// Builds the list from per-expert counts and offsets (global or shared memory) with the whole
// block (any size up to 1024 threads, a multiple of 32; every thread calls it).
__device__ __forceinline__ void build_tile_list(const int* counts, const int* offsets, int E, const TileList& tl) {
    __shared__ int warp_sum[32];
    __shared__ int base_s;
    if (threadIdx.x == 0) base_s = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, rpt = tl.rows_per_tile;
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const int n = e < E ? (counts[e] + rpt - 1) / rpt : 0;
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int v = lane < static_cast<int>(blockDim.x >> 5) ? warp_sum[lane] : 0;
            int wi = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += u;
            }
            warp_sum[lane] = wi - v;
        }
        __syncthreads();
        const int start = base_s + warp_sum[warp] + incl - n;
        for (int i = 0; i < n; ++i) {
            tl.tile_e[start + i] = e;
            tl.tile_r0[start + i] = offsets[e] + i * rpt;
            tl.tile_first[start + i] = start;
            tl.tile_cnt[start + i] = n;
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) base_s = start + n;
        __syncthreads();
    }
    if (threadIdx.x == 0) tl.tiles[0] = base_s;
}

// Route histogram / stable counting sort, optionally emitting expert groups (route_plan.cu).
cudaError_t launch_route_plan(const int32_t* ids, int P, int E, int cap, int32_t* counts,
                              int32_t* offsets, int32_t* sorted_pair, int32_t* pair_to_sorted,
                              int32_t* group_count, int32_t* group_expert, int32_t* group_start,
                              int32_t* group_ncols, int32_t* err, cudaStream_t stream);
// The same permutation (no groups) over several blocks for many pairs; blk is scratch of
// route_plan_wide_ws_bytes(P, E) bytes (route_plan.cu). Three launches; with tl.tiles set the
// middle one also builds the grouped tier's m-tile list.
size_t route_plan_wide_ws_bytes(int P, int E);
cudaError_t launch_route_plan_wide(const int32_t* ids, int P, int E, int32_t* counts, int32_t* offsets,
                                   int32_t* sorted_pair, int32_t* pair_to_sorted, int32_t* blk,
                                   int32_t* err, cudaStream_t stream, const TileList& tl);
size_t route_plan_smem_bytes(int E);

}  // namespace moe
