// Route histogram + stable counting sort of (token, slot) pairs by expert, and the expert groups
// that the batched GEMV kernels sweep (each selected expert's weights read once per call).
//
// "spark_model layers/glm5next_mlp/forward.rs": the expert-sorted row order, expert_offsets[E+1]
// and token_to_perm of `Glm5NextMlpWorkspace`, built by the `moe_sort_by_expert` step of
// `forward_moe`; the "union" of a few rows' experts swept once each (doc comment of
// `forward_moe`, `w4a16_gemv_moe_batchm`). Here both come from ONE single-block launch that
// never returns to the host.
#include "kernels.cuh"

namespace moe {

namespace {

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan of in[0..n) into out[0..n) by the whole block (blockDim.x == kPlanThreads).
// Returns the total. in and out may alias. Uses scratch[33].
__device__ int block_exclusive_scan(const int* in, int* out, int n, int* scratch) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + kPlanThreads - 1) / kPlanThreads;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += in[i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = scratch[lane];
        int wi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += u;
        }
        scratch[lane] = wi - v;
        if (lane == 31) scratch[32] = wi;
    }
    __syncthreads();
    int run = scratch[warp] + incl - local;
    for (int i = lo; i < hi; ++i) {
        const int v = in[i];
        out[i] = run;
        run += v;
    }
    const int total = scratch[32];
    __syncthreads();
    return total;
}

}  // namespace

// One block of kPlanThreads threads. Dynamic shared memory: 3*E ints + 32*E bytes.
// group_* may be null (plain permutation). cap = max columns per group (1..8).
__global__ void __launch_bounds__(kPlanThreads, 1)
route_plan_kernel(const int32_t* __restrict__ ids, int P, int E, int cap,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ sorted_pair, int32_t* __restrict__ pair_to_sorted,
                  int32_t* __restrict__ group_count, int32_t* __restrict__ group_expert,
                  int32_t* __restrict__ group_start, int32_t* __restrict__ group_ncols,
                  int32_t* __restrict__ err) {
    extern __shared__ __align__(16) int smem_i[];
    int* cnt = smem_i;                 // [E]
    int* run = cnt + E;                // [E] offsets, then running cursor
    int* tmp = run + E;                // [E] group counts / group bases
    uint8_t* pre = reinterpret_cast<uint8_t*>(tmp + E);   // [32][E] per-warp counts of a round
    __shared__ int scratch[33];
    __shared__ int bad;

    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) bad = 0;
    for (int e = tid; e < E; e += kPlanThreads) cnt[e] = 0;
    for (int i = tid; i < 32 * E; i += kPlanThreads) pre[i] = 0;
    __syncthreads();

    // 1. histogram (integer atomics: the result does not depend on their order)
    for (int p = tid; p < P; p += kPlanThreads) {
        const int e = ids[p];
        if (e >= 0 && e < E)
            atomicAdd(&cnt[e], 1);
        else if (e != -1)
            bad = 1;
    }
    __syncthreads();

    // 2. offsets
    const int total = block_exclusive_scan(cnt, run, E, scratch);
    for (int e = tid; e < E; e += kPlanThreads) {
        counts[e] = cnt[e];
        offsets[e] = run[e];
    }
    if (tid == 0) offsets[E] = total;

    // 3. groups: ceil(count/cap) per expert, ascending expert, contiguous sorted pairs
    if (group_count != nullptr) {
        for (int e = tid; e < E; e += kPlanThreads) tmp[e] = (cnt[e] + cap - 1) / cap;
        __syncthreads();
        const int G = block_exclusive_scan(tmp, tmp, E, scratch);
        for (int e = tid; e < E; e += kPlanThreads) {
            const int c = cnt[e];
            for (int j = 0, gi = tmp[e]; j * cap < c; ++j, ++gi) {
                group_expert[gi] = e;
                group_start[gi] = run[e] + j * cap;
                group_ncols[gi] = min(cap, c - j * cap);
            }
        }
        if (tid == 0) *group_count = G;
    }
    __syncthreads();

    // 4. stable scatter, in rounds of kPlanThreads pairs (ascending pair index)
    for (int base = 0; base < P; base += kPlanThreads) {
        const int p = base + tid;
        const int e = p < P ? ids[p] : -1;
        const bool valid = p < P && e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
        const int rank = __popc(peers & lanemask_lt());
        const bool leader = valid && rank == 0;
        const int wc = __popc(peers);
        if (leader) pre[warp * E + e] = static_cast<uint8_t>(wc);
        __syncthreads();
        if (valid) {
            int s = 0;
            for (int w = 0; w < warp; ++w) s += pre[w * E + e];
            const int pos = run[e] + s + rank;
            sorted_pair[pos] = p;
            pair_to_sorted[p] = pos;
        } else if (p < P) {
            pair_to_sorted[p] = -1;
        }
        __syncthreads();
        if (leader) {
            atomicAdd(&run[e], wc);
            pre[warp * E + e] = 0;
        }
        __syncthreads();
    }
    for (int s = total + tid; s < P; s += kPlanThreads) sorted_pair[s] = -1;
    if (tid == 0 && bad && err != nullptr) atomicOr(err, 1);
}

// ---- the same permutation for many pairs, over several blocks --------------------------------------

// shared memory up to which plan_base_kernel stages the per-block counts
constexpr size_t kPlanStageBytes = 160 * 1024;
// Block b owns pairs [b*kPlanThreads, (b+1)*kPlanThreads). plan_hist_kernel counts each block's
// pairs per expert; plan_base_kernel turns the counts into each (block, expert) first position -
// the expert's offset plus the counts of the earlier blocks - and the offsets; plan_scatter_kernel
// places each block's pairs in one round of the single-block kernel's stable scatter. Same result,
// bit for bit: within an expert, pairs keep ascending pair order.

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_hist_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ blk,
                 int32_t* __restrict__ err) {
    extern __shared__ __align__(16) int smem_i[];
    int* cnt = smem_i;                 // [E]
    const int tid = threadIdx.x;
    pdl_launch_dependents();           // the base kernel may start; it waits for this grid
    for (int e = tid; e < E; e += kPlanThreads) cnt[e] = 0;
    __syncthreads();
    const int p = blockIdx.x * kPlanThreads + tid;
    bool bad = false;
    if (p < P) {
        const int e = ids[p];
        if (e >= 0 && e < E)
            atomicAdd(&cnt[e], 1);
        else if (e != -1)
            bad = true;
    }
    if (__syncthreads_or(bad) && tid == 0 && err != nullptr) atomicOr(err, 1);
    for (int e = tid; e < E; e += kPlanThreads) blk[static_cast<size_t>(blockIdx.x) * E + e] = cnt[e];
}

// staged: the [nblk][E] counts go through shared memory (one coalesced read and write of blk
// instead of nblk dependent accesses per expert in each of two passes)
__global__ void __launch_bounds__(kPlanThreads, 1)
plan_base_kernel(int P, int E, int nblk, int32_t* __restrict__ blk, int32_t* __restrict__ counts,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pair, int staged, TileList tl) {
    extern __shared__ __align__(16) int smem_i[];
    int* cnt = smem_i;                 // [E]
    int* run = cnt + E;                // [E]
    int* bc = run + E;                 // [nblk][E] when staged
    __shared__ int scratch[33];
    const int tid = threadIdx.x;
    const size_t nall = static_cast<size_t>(nblk) * E;
    pdl_wait();                        // the histogram grid's counts (programmatic dependent launch)
    pdl_launch_dependents();
    if (staged) {
        for (size_t i = tid; i < nall; i += kPlanThreads) bc[i] = blk[i];
        __syncthreads();
    }
    int* src = staged ? bc : blk;
    // per expert: block bases relative to the expert, and its total
    for (int e = tid; e < E; e += kPlanThreads) {
        int acc = 0;
        for (int b = 0; b < nblk; ++b) {
            int* q = src + static_cast<size_t>(b) * E + e;
            const int c = *q;
            *q = acc;
            acc += c;
        }
        cnt[e] = acc;
    }
    __syncthreads();
    const int total = block_exclusive_scan(cnt, run, E, scratch);
    if (staged) {
        for (size_t i = tid; i < nall; i += kPlanThreads) blk[i] = bc[i] + run[i % E];
    } else {
        for (int e = tid; e < E; e += kPlanThreads)
            for (int b = 0; b < nblk; ++b) blk[static_cast<size_t>(b) * E + e] += run[e];
    }
    for (int e = tid; e < E; e += kPlanThreads) {
        counts[e] = cnt[e];
        offsets[e] = run[e];
    }
    if (tid == 0) offsets[E] = total;
    for (int s = total + tid; s < P; s += kPlanThreads) sorted_pair[s] = -1;
    if (tl.tiles != nullptr) build_tile_list(cnt, run, E, tl);   // cnt / run are final here
}

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_scatter_kernel(const int32_t* __restrict__ ids, int P, int E, const int32_t* __restrict__ blk,
                    int32_t* __restrict__ sorted_pair, int32_t* __restrict__ pair_to_sorted) {
    extern __shared__ __align__(16) int smem_i[];
    uint8_t* pre = reinterpret_cast<uint8_t*>(smem_i);   // [32][E] per-warp counts
    const int tid = threadIdx.x, warp = tid >> 5;
    pdl_wait();                        // the base kernel's block bases (programmatic dependent launch)
    pdl_launch_dependents();
    for (int i = tid; i < 32 * E; i += kPlanThreads) pre[i] = 0;
    __syncthreads();
    const int p = blockIdx.x * kPlanThreads + tid;
    const int e = p < P ? ids[p] : -1;
    const bool valid = p < P && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    const int rank = __popc(peers & lanemask_lt());
    if (valid && rank == 0) pre[warp * E + e] = static_cast<uint8_t>(__popc(peers));
    __syncthreads();
    if (valid) {
        int s = 0;
        for (int w = 0; w < warp; ++w) s += pre[w * E + e];
        const int pos = blk[static_cast<size_t>(blockIdx.x) * E + e] + s + rank;
        sorted_pair[pos] = p;
        pair_to_sorted[p] = pos;
    } else if (p < P) {
        pair_to_sorted[p] = -1;
    }
}

size_t route_plan_wide_ws_bytes(int P, int E) {
    const size_t nblk = (static_cast<size_t>(P) + kPlanThreads - 1) / kPlanThreads;
    return nblk * E * 4;
}

cudaError_t launch_route_plan_wide(const int32_t* ids, int P, int E, int32_t* counts, int32_t* offsets,
                                   int32_t* sorted_pair, int32_t* pair_to_sorted, int32_t* blk,
                                   int32_t* err, cudaStream_t stream, const TileList& tl) {
    const int nblk = (P + kPlanThreads - 1) / kPlanThreads;
    // the per-block counts fit shared memory beside the two [E] arrays: stage them
    const size_t staged_bytes = (static_cast<size_t>(nblk) + 2) * E * 4;
    const bool staged = staged_bytes <= kPlanStageBytes;
    const size_t s1 = static_cast<size_t>(E) * 4, s2 = staged ? staged_bytes : static_cast<size_t>(E) * 8,
                 s3 = static_cast<size_t>(E) * 32;
    const void* fns[3] = {reinterpret_cast<const void*>(plan_hist_kernel),
                          reinterpret_cast<const void*>(plan_base_kernel),
                          reinterpret_cast<const void*>(plan_scatter_kernel)};
    const size_t sm[3] = {s1, s2, s3};
    for (int i = 0; i < 3; ++i)
        if (sm[i] > 48 * 1024) {
            cudaError_t st = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(sm[i]));
            if (st != cudaSuccess) return st;
        }
    plan_hist_kernel<<<nblk, kPlanThreads, s1, stream>>>(ids, P, E, blk, err);
    cudaError_t st = cudaGetLastError();
    if (st != cudaSuccess) return st;
    // the base and scatter kernels are programmatic dependents of the kernel before them: each
    // is resident and waiting (griddepcontrol.wait) when its predecessor completes
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(1);
    cfg.dynamicSmemBytes = s2;
    if ((st = cudaLaunchKernelEx(&cfg, plan_base_kernel, P, E, nblk, blk, counts, offsets, sorted_pair,
                                 staged ? 1 : 0, tl)) != cudaSuccess)
        return st;
    cfg.gridDim = dim3(nblk);
    cfg.dynamicSmemBytes = s3;
    if ((st = cudaLaunchKernelEx(&cfg, plan_scatter_kernel, ids, P, E, static_cast<const int32_t*>(blk),
                                 sorted_pair, pair_to_sorted)) != cudaSuccess)
        return st;
    return cudaGetLastError();
}

size_t route_plan_smem_bytes(int E) { return static_cast<size_t>(E) * (3 * 4 + 32); }

cudaError_t launch_route_plan(const int32_t* ids, int P, int E, int cap, int32_t* counts,
                              int32_t* offsets, int32_t* sorted_pair, int32_t* pair_to_sorted,
                              int32_t* group_count, int32_t* group_expert, int32_t* group_start,
                              int32_t* group_ncols, int32_t* err, cudaStream_t stream) {
    const size_t smem = route_plan_smem_bytes(E);
    if (smem > 48 * 1024) {
        cudaError_t st = cudaFuncSetAttribute(route_plan_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem));
        if (st != cudaSuccess) return st;
    }
    route_plan_kernel<<<1, kPlanThreads, smem, stream>>>(ids, P, E, cap, counts, offsets,
                                                         sorted_pair, pair_to_sorted, group_count,
                                                         group_expert, group_start, group_ncols,
                                                         err);
    return cudaGetLastError();
}

}  // namespace moe
