// The shared expert of the MoE layer: a dense BF16 SwiGLU MLP over every token, not routed and not
// route-weighted ("spark_model layers/glm5next_mlp/forward.rs", `forward_moe`: `forward_dense` on the
// shared weights into `shared_out`, which the combine then adds; the Step gate uploads the shared
// gate/up/down as a replicated BF16 SwiGLU with its own activation limit).
//
//   shared = Wd . bf16(silu(min(Wg.x, L)) * clamp(Wu.x, -L, L))
//
// Three tensor-core passes of the router's dense bf16 kernel (K split over the grid for small T, so
// that enough warps stream the weights), a SwiGLU pass that sums the gate/up parts in order and
// rounds the activation to bf16 (the input precision of the down product), and a final pass that
// sums the down parts in order and rounds to bf16. Deterministic.
#include <algorithm>

#include "kernels.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) shared_swiglu_kernel(const float* __restrict__ pg, const float* __restrict__ pu,
                                                            int KS, int T, int S, float limit,
                                                            __nv_bfloat16* __restrict__ a) {
    const size_t n = static_cast<size_t>(T) * S;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float g = 0.0f, u = 0.0f;
        for (int q = 0; q < KS; ++q) {
            g += pg[q * n + i];
            u += pu[q * n + i];
        }
        g = fminf(g, limit);
        u = fminf(fmaxf(u, -limit), limit);
        a[i] = __float2bfloat16_rn(g / (1.0f + expf(-g)) * u);
    }
}

__global__ void __launch_bounds__(256) dense_reduce_bf16_kernel(const float* __restrict__ part, int KS, size_t n,
                                                                __nv_bfloat16* __restrict__ out) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float s = 0.0f;
        for (int q = 0; q < KS; ++q) s += part[q * n + i];
        out[i] = __float2bfloat16_rn(s);
    }
}

struct SharedLayout {
    int ks1, ks2;
    size_t pg, pu, a, pd, total;
};

SharedLayout shared_layout(int T, int H, int S, int sms) {
    SharedLayout L{};
    L.ks1 = router_ksplit(T, H, S, sms);
    L.ks2 = router_ksplit(T, S, H, sms);
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    L.pg = take(static_cast<size_t>(L.ks1) * T * S * 4);
    L.pu = take(static_cast<size_t>(L.ks1) * T * S * 4);
    L.a = take(static_cast<size_t>(T) * S * 2);
    L.pd = take(static_cast<size_t>(L.ks2) * T * H * 4);
    L.total = o;
    return L;
}

}  // namespace

size_t shared_expert_ws_bytes(int T, int H, int S, int sms) { return shared_layout(T, H, S, sms).total; }

cudaError_t launch_shared_expert(const __nv_bfloat16* x, int T, int H, int S, const __nv_bfloat16* wg,
                                 const __nv_bfloat16* wu, const __nv_bfloat16* wd, float limit,
                                 __nv_bfloat16* out, uint8_t* ws, int sms, cudaStream_t stream) {
    const SharedLayout L = shared_layout(T, H, S, sms);
    float* pg = reinterpret_cast<float*>(ws + L.pg);
    float* pu = reinterpret_cast<float*>(ws + L.pu);
    __nv_bfloat16* a = reinterpret_cast<__nv_bfloat16*>(ws + L.a);
    float* pd = reinterpret_cast<float*>(ws + L.pd);
    cudaError_t st;
    if ((st = launch_dense_bf16(x, T, H, wg, S, pg, L.ks1, stream)) != cudaSuccess) return st;
    if ((st = launch_dense_bf16(x, T, H, wu, S, pu, L.ks1, stream)) != cudaSuccess) return st;
    const size_t ns = static_cast<size_t>(T) * S, nh = static_cast<size_t>(T) * H;
    const int g1 = static_cast<int>(std::min<size_t>((ns + 255) / 256, static_cast<size_t>(sms) * 8));
    shared_swiglu_kernel<<<g1, 256, 0, stream>>>(pg, pu, L.ks1, T, S, limit, a);
    if ((st = cudaGetLastError()) != cudaSuccess) return st;
    if ((st = launch_dense_bf16(a, T, S, wd, H, pd, L.ks2, stream)) != cudaSuccess) return st;
    const int g2 = static_cast<int>(std::min<size_t>((nh + 255) / 256, static_cast<size_t>(sms) * 8));
    dense_reduce_bf16_kernel<<<g2, 256, 0, stream>>>(pd, L.ks2, nh, out);
    return cudaGetLastError();
}

}  // namespace moe
