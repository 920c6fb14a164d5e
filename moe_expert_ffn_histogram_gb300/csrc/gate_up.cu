// Stage kernel: dequant-fused gate + up projections with the clamped SwiGLU epilogue, one CTA per
// (feature block of 64, routed group). The work item itself is gate_up_item (gemv_items.cuh).
#include "gemv_items.cuh"

namespace moe {

size_t gate_up_smem_bytes(int H, int max_cols) { return gate_up_item_smem(H, max_cols); }

template <int FMT>
__global__ void __launch_bounds__(kItemThreads, kMinBlocks) gate_up_kernel(const GateUpArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ GroupView gv;
    __shared__ GateUpShared sh;
    const Groups& G = a.grp;
    if (threadIdx.x == 0) {
        const int gi = blockIdx.y;
        gv.e = -1;
        if (G.count == nullptr) {           // implicit: group = slot of the single token
            const int e = G.ids[gi];
            if (e >= 0 && e < G.E) {
                gv.e = e;
                gv.ncols = 1;
                gv.pair[0] = gi;
            } else if (e != -1 && blockIdx.x == 0 && a.err) {
                atomicOr(a.err, 1);
            }
        } else if (gi < *G.count) {
            gv.e = G.expert[gi];
            gv.ncols = G.ncols[gi];
            for (int j = 0; j < gv.ncols; ++j) gv.pair[j] = G.sorted_pair[G.start[gi] + j];
        }
    }
    __syncthreads();
    pdl_launch_dependents();      // the down kernel may launch; it waits for this grid's results
    if (gv.e < 0) return;
    if (FMT == 1 && a.l2_prefetch && threadIdx.x == 0) {
        const int e = gv.e, nfb = gridDim.x, fb = blockIdx.x;
        const size_t rows = static_cast<size_t>(e) * a.I + static_cast<size_t>(fb) * kFeatBlock;
        prefetch_l2_range(a.wg + rows * (a.H / 2), static_cast<size_t>(kFeatBlock) * (a.H / 2));
        prefetch_l2_range(a.wu + rows * (a.H / 2), static_cast<size_t>(kFeatBlock) * (a.H / 2));
        prefetch_l2_range(a.sfg + rows * (a.H / 16), static_cast<size_t>(kFeatBlock) * (a.H / 16));
        prefetch_l2_range(a.sfu + rows * (a.H / 16), static_cast<size_t>(kFeatBlock) * (a.H / 16));
        // this block's 1/nfb share of expert e's down matrix (codes, then scale bytes)
        const size_t dcodes = static_cast<size_t>(a.H) * (a.I / 2), dsf = static_cast<size_t>(a.H) * (a.I / 16);
        const size_t c0 = (dcodes * fb / nfb) & ~static_cast<size_t>(15), c1 = (dcodes * (fb + 1) / nfb) & ~static_cast<size_t>(15);
        const size_t s0 = (dsf * fb / nfb) & ~static_cast<size_t>(15), s1 = (dsf * (fb + 1) / nfb) & ~static_cast<size_t>(15);
        prefetch_l2_range(a.pf_wd + static_cast<size_t>(e) * dcodes + c0, c1 - c0);
        prefetch_l2_range(a.pf_sfd + static_cast<size_t>(e) * dsf + s0, s1 - s0);
    }
    gate_up_item<FMT>(a, gv, blockIdx.x, reinterpret_cast<__half*>(smem_raw), sh);
}

template <int FMT>
cudaError_t launch_gate_up(const GateUpArgs& a, int num_groups, int max_cols, cudaStream_t stream) {
    const size_t smem = gate_up_item_smem(a.H, max_cols);
    if (smem > 48 * 1024) {
        cudaError_t st = cudaFuncSetAttribute(gate_up_kernel<FMT>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem));
        if (st != cudaSuccess) return st;
    }
    dim3 grid(a.I / kFeatBlock, num_groups);
    gate_up_kernel<FMT><<<grid, kItemThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template cudaError_t launch_gate_up<0>(const GateUpArgs&, int, int, cudaStream_t);
template cudaError_t launch_gate_up<1>(const GateUpArgs&, int, int, cudaStream_t);

}  // namespace moe
