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
