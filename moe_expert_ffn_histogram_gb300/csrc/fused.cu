// The whole routed-MoE forward of one sub-batch (T <= 8 tokens) in ONE persistent cooperative
// launch: every CTA groups the routed pairs by expert itself, sweeps its share of the gate/up work
// items, meets the other CTAs at a grid-wide barrier, and sweeps its share of the down+combine
// work items. One launch instead of three removes the per-kernel ramp-up and drain of the weight
// stream (on GB300 each extra kernel boundary costs about 5 us of HBM time at these sizes), and
// while waiting at the barrier a CTA already pulls its first down tiles into L2.
//
// The barrier counter lives in the workspace and is zeroed by a memset on the same stream right
// before the launch. The wait is bounded: if it ever exceeds ~2 s of SM clock (possible only if the
// GPU could not keep every CTA resident, which the cooperative launch rules out), the CTA sets
// MOE_ERRBIT_BARRIER in the error word, writes NaN to the output rows it owns (so an incomplete
// result is visible even to a caller that passed no error word) and returns instead of hanging.
// moe_test_barrier_timeout() makes the barrier wait for one CTA more than the grid holds, with a
// ~10 ms bound, so that a test can drive that path.
#include <atomic>
#include <mutex>

#include "../../include/moe_ffn.h"

#include "gemv_items.cuh"

#ifndef MOE_FUSED_PREFETCH
#define MOE_FUSED_PREFETCH 0
#endif

namespace moe {

namespace {

constexpr long long kBarrierTimeoutCycles = 1ll << 32;
constexpr long long kTestBarrierTimeoutCycles = 1ll << 24;   // ~10 ms: the test hook's bound
constexpr int kErrBitBarrier = MOE_ERRBIT_BARRIER;

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier over gridDim.x CTAs (plus `extra`, which only the test hook sets) on a zeroed
// counter; false after `limit` cycles of SM clock.
__device__ bool grid_barrier(unsigned* counter, int32_t* err, unsigned extra, long long limit) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();                          // publish this CTA's phase-1 writes
        atomicAdd(counter, 1u);
        const long long t0 = clock64();
        int good = 1;
        while (ld_acquire_gpu(counter) < gridDim.x + extra) {
            if (clock64() - t0 > limit) {
                good = 0;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        ok = good;
        if (!good && err != nullptr) atomicOr(err, kErrBitBarrier);
    }
    __syncthreads();
    return ok != 0;
}

}  // namespace

struct FusedCtl {
    unsigned* barrier;   // zeroed before the launch
    int rows;            // tokens of this sub-batch (1..8)
    int cap;             // columns per group
    unsigned barrier_extra;        // 0; 1 under the test hook (the barrier can never complete)
    long long barrier_limit;       // wait bound in SM clock cycles
};

template <int FMT>
#ifndef MOE_FUSED_MIN_BLOCKS
#define MOE_FUSED_MIN_BLOCKS kMinBlocks
#endif
__global__ void __launch_bounds__(kItemThreads, MOE_FUSED_MIN_BLOCKS)
fused_forward_kernel(const GateUpArgs ga, const DownArgs da, const FusedCtl ctl) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ GroupList gl;
    __shared__ GateUpShared sh;
    const int topk = ga.grp.topk, E = ga.grp.E;

    // ---- expert groups of this sub-batch, computed by every CTA ----
    bool bad;
    if (ctl.rows == 1) {
        __shared__ int s_bad;
        if (threadIdx.x == 0) {
            int b = 0;
            for (int k = 0; k < topk; ++k) {
                const int e = ga.grp.ids[k];
                if ((e < 0 || e >= E) && e != -1) b = 1;
            }
            s_bad = b;
        }
        Groups implicit = ga.grp;
        implicit.count = nullptr;
        load_group_list(implicit, gl);
        bad = s_bad != 0;
    } else {
        bad = plan_groups_in_cta(ga.grp.ids, ctl.rows * topk, E, ctl.cap, gl);
    }
    if (bad && blockIdx.x == 0 && threadIdx.x == 0 && ga.err != nullptr) atomicOr(ga.err, 1);

    // ---- phase 1: gate/up + SwiGLU items (group, 64-feature block) ----
    const int nfb = ga.I / kFeatBlock;
    const int n1 = gl.count * nfb;
    for (int it = blockIdx.x; it < n1; it += gridDim.x) {
        gate_up_item<FMT, kFusedStagesFp8, kFusedStagesFp4, false>(
            ga, gl.g[it / nfb], it % nfb, reinterpret_cast<__half*>(smem_raw), sh);
        __syncthreads();
    }

    // ---- warm L2 with this CTA's first down tiles (they do not depend on phase 1) ----
    const int n2 = da.H / kDownRows;
    if (MOE_FUSED_PREFETCH && blockIdx.x < n2 && threadIdx.x < gl.count) {
        const int e = gl.g[threadIdx.x].e;
        const size_t r0 = static_cast<size_t>(e) * da.H + static_cast<size_t>(blockIdx.x) * kDownRows;
        const size_t row_bytes = FMT == 0 ? static_cast<size_t>(da.I) : static_cast<size_t>(da.I / 2);
        prefetch_l2(da.wd + r0 * row_bytes, static_cast<uint32_t>(kDownRows * row_bytes));
        if (FMT == 1)
            prefetch_l2(da.sfd + r0 * (da.I / 16), static_cast<uint32_t>(kDownRows * (da.I / 16)));
    }

    if (!grid_barrier(ctl.barrier, ga.err, ctl.barrier_extra, ctl.barrier_limit)) {
        // the rows this CTA would have written (down items jt = blockIdx.x + i * gridDim.x, no
        // other CTA writes them) become NaN: the call's output is invalid, and visibly so
        const __nv_bfloat16 qnan = __ushort_as_bfloat16(0x7FC0);
        for (int jt = blockIdx.x; jt < n2; jt += gridDim.x)
            for (int i = threadIdx.x; i < da.T * kDownRows; i += blockDim.x)
                da.out[static_cast<size_t>(i / kDownRows) * da.H + jt * kDownRows + i % kDownRows] = qnan;
        return;
    }

    // ---- phase 2: down + slot-order combine items (16 output rows each) ----
    for (int jt = blockIdx.x; jt < n2; jt += gridDim.x) {
        down_item<FMT, false, FMT == 0 ? kFusedDownBatch : kFusedDownBatchFp4>(da, gl, jt, reinterpret_cast<float*>(smem_raw));
        __syncthreads();
    }
}

namespace {

std::atomic<int> g_test_barrier_timeout{0};

// Co-resident CTAs per SM for a (kernel, dynamic smem) pair, times the SM count; cached per
// device because the occupancy query costs host time on every call.
template <int FMT>
cudaError_t fused_grid(size_t smem, int* grid) {
    struct Entry { int dev; size_t smem; int grid; };
    static std::mutex mu;
    static Entry cache[16];
    static int n = 0;
    int dev = 0;
    cudaError_t st = cudaGetDevice(&dev);
    if (st != cudaSuccess) return st;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n; ++i)
            if (cache[i].dev == dev && cache[i].smem == smem) {
                *grid = cache[i].grid;
                return cudaSuccess;
            }
    }
    int sms = 0, per_sm = 0;
    if ((st = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return st;
    if ((st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_forward_kernel<FMT>,
                                                            kItemThreads, smem)) != cudaSuccess)
        return st;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    *grid = per_sm * sms;
    std::lock_guard<std::mutex> lock(mu);
    if (n < 16) cache[n++] = Entry{dev, smem, *grid};
    return cudaSuccess;
}

}  // namespace

size_t fused_smem_bytes(int H, int rows, int topk, int cap) {
    const size_t a = gate_up_item_smem(H, cap), b = down_item_smem(rows, topk);
    return a > b ? a : b;
}

template <int FMT>
cudaError_t launch_fused_forward(const GateUpArgs& ga, const DownArgs& da, unsigned* barrier,
                                 int rows, int cap, cudaStream_t stream) {
    const size_t smem = fused_smem_bytes(ga.H, rows, ga.grp.topk, cap);
    cudaError_t st;
    if (smem > 48 * 1024 &&
        (st = cudaFuncSetAttribute(fused_forward_kernel<FMT>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem))) != cudaSuccess)
        return st;
    int grid = 0;
    if ((st = fused_grid<FMT>(smem, &grid)) != cudaSuccess) return st;
    if ((st = cudaMemsetAsync(barrier, 0, sizeof(unsigned), stream)) != cudaSuccess) return st;
    const bool test_timeout = g_test_barrier_timeout.load(std::memory_order_relaxed) != 0;
    FusedCtl ctl{barrier, rows, cap, test_timeout ? 1u : 0u,
                 test_timeout ? kTestBarrierTimeoutCycles : kBarrierTimeoutCycles};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kItemThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((st = cudaLaunchKernelEx(&cfg, fused_forward_kernel<FMT>, ga, da, ctl)) != cudaSuccess) return st;
    return cudaGetLastError();
}

void set_test_barrier_timeout(bool on) { g_test_barrier_timeout.store(on ? 1 : 0); }

template cudaError_t launch_fused_forward<0>(const GateUpArgs&, const DownArgs&, unsigned*, int, int,
                                             cudaStream_t);
template cudaError_t launch_fused_forward<1>(const GateUpArgs&, const DownArgs&, unsigned*, int, int,
                                             cudaStream_t);

}  // namespace moe
