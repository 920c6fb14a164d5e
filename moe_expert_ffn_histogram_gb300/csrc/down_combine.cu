// Stage kernel: dequant-fused down projection with the slot-order combine, one CTA per 16 output
// rows. The work item itself is down_item (gemv_items.cuh).
#include "gemv_items.cuh"

// Launched as a programmatic dependent of the preceding gate/up kernel (see down_item).

namespace moe {

size_t down_smem_bytes(int T, int topk) { return down_item_smem(T, topk); }

template <int FMT>
__global__ void __launch_bounds__(kItemThreads, kDownMinBlocks) down_combine_kernel(const DownArgs a) {
    extern __shared__ __align__(16) float ys[];     // [P][16]
    __shared__ GroupList gl;
    load_group_list(a.grp, gl);
    down_item<FMT, MOE_PDL != 0, FMT == 0 ? kDownBatch : kDownBatchFp4>(a, gl, blockIdx.x, ys);
}

template <int FMT>
cudaError_t launch_down_combine(const DownArgs& a, cudaStream_t stream) {
    const size_t smem = down_item_smem(a.T, a.topk);
    if (smem > 48 * 1024) {
        cudaError_t st = cudaFuncSetAttribute(down_combine_kernel<FMT>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(smem));
        if (st != cudaSuccess) return st;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.H / kDownRows);
    cfg.blockDim = dim3(kItemThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t st = cudaLaunchKernelEx(&cfg, down_combine_kernel<FMT>, a);
    if (st != cudaSuccess) return st;
    return cudaGetLastError();
}

template cudaError_t launch_down_combine<0>(const DownArgs&, cudaStream_t);
template cudaError_t launch_down_combine<1>(const DownArgs&, cudaStream_t);

}  // namespace moe
