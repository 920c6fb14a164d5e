// moe_fp8_forward_noalloc: the FP8 routed-MoE forward for callers that cannot allocate device
// memory.
//
// Some callers of this library cannot call cudaMalloc or hand it a workspace: a plugin that only
// receives input and output pointers through a fixed interface (no workspace argument, no access
// to the host framework's allocator), or a latency-critical serving loop that forbids device
// allocation because cudaMalloc/cudaFree can implicitly synchronise the device and stall every
// stream. This entry point gives them the forward without a workspace argument: its scratch is a
// file-scope device array of fixed size, so nothing is allocated at call time.
//
// Contract:
//   * The scratch is MOE_NOALLOC_SCRATCH_BYTES (1 MiB) in every GPU's memory that loads the library,
//     held until the process exits. Calls whose moe_workspace_bytes() exceeds it are rejected
//     with MOE_ERR_WORKSPACE before anything is enqueued.
//   * All calls on one device share that array, and it keeps the last call's contents. Nothing in
//     it needs to start at zero: every call writes each region before reading it. Calls that
//     overlap on the GPU (e.g. on two streams at once) race on the array; serialise them (one
//     stream, or events).
//   * The first call on each device, with that device current, looks up the array's device
//     address with cudaGetSymbolAddress (which may load the library's kernels on that device).
//     Make that first call before any stream capture. The address is cached per device and per
//     CUDA context: after cudaDeviceReset() the device gets a new context, the next call looks the
//     address up again (so, again, make it outside a capture).
//   * No cudaMalloc, cudaFree or allocating library routine is called.
// The pages have no counterpart to this entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe_ffn.h"

namespace {

constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // id of the context the address belongs to

// Unique id of the calling thread's current CUDA context (0 if the driver cannot tell): a reset
// device gets a new context and so a new id.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device (host code must not use the
// array's name as a pointer: on the host it is only a stand-in for the symbol).
int scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    // a thread that has not used the runtime yet has no current context (id 0): the lookup then
    // runs once more, which makes the device's primary context current, and the id read after it
    // is the one kept
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_ptr[dev] == nullptr || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        const cudaError_t st = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (st != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = current_context_id();
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" {

int moe_fp8_forward_noalloc(const uint16_t* x, int T, int H, int I, int E, int topk,
                            const int32_t* topk_ids, const float* topk_weights,
                            const uint8_t* w_gate, const float* s_gate, const uint8_t* w_up,
                            const float* s_up, const uint8_t* w_down, const float* s_down,
                            float limit, uint16_t* out, int32_t* err, void* stream) {
    const size_t need = moe_workspace_bytes(T, H, I, E, topk, MOE_FMT_FP8_E4M3_B128);
    if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
    if (need == 0)   // invalid sizes: report exactly what moe_fp8_forward reports, enqueue nothing
        return moe_fp8_forward(x, T, H, I, E, topk, topk_ids, topk_weights, w_gate, s_gate, w_up,
                               s_up, w_down, s_down, limit, out, nullptr, 0, err, stream);
    void* scratch = nullptr;
    const int rc = scratch_on_current_device(&scratch);
    if (rc != MOE_OK) return rc;
    return moe_fp8_forward(x, T, H, I, E, topk, topk_ids, topk_weights, w_gate, s_gate, w_up, s_up,
                           w_down, s_down, limit, out, scratch, kNoAllocScratchBytes, err, stream);
}

}  // extern "C"
