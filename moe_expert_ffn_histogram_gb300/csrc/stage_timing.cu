// Stage hooks. NVTX: every forward opens a range named after its entry point and, inside it, one
// range per stage (route plan, gate/up, down and combine, ...), on the calling host thread, so
// that a profiler can select a stage's kernels (ncu --nvtx --nvtx-include). Always on unless
// built with MOE_NVTX=0; without an attached tool an NVTX call is a null-pointer check.
//
// Stage timing: CUDA events recorded on the forward's own stream between its kernel launches.
// Off by default. When on, each forward records one event at the start of every stage and one
// after the last; moe_stage_times turns the most recent forward's events into per-stage
// durations. The events sit between launches, so a stage that normally starts early as a
// programmatic dependent launch waits for its predecessor instead: the intervals are the
// stages' serialised device times. One process-wide recorder, for profiling from one host
// thread at a time.
#include "stage_timing.cuh"
#include "../../include/moe_ffn.h"

#ifndef MOE_NVTX
#define MOE_NVTX 1
#endif
#if MOE_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace moe {

namespace {

// NVTX: the calling host thread's open stage range (closed by the next stage or the call's end)
thread_local bool t_stage_open = false;

void nvtx_push(const char* name) {
#if MOE_NVTX
    nvtxRangePushA(name);
#else
    (void)name;
#endif
}
void nvtx_pop() {
#if MOE_NVTX
    nvtxRangePop();
#endif
}

constexpr int kMaxMarks = 64;

struct StageRecorder {
    bool on = false;
    bool created = false;
    int n = 0;          // marks of the forward in progress
    int done = -1;      // stages of the last completed forward (-1: none)
    cudaEvent_t ev[kMaxMarks];
    const char* name[kMaxMarks];
};

StageRecorder g_rec;

bool create_events() {
    if (g_rec.created) return true;
    for (int i = 0; i < kMaxMarks; ++i)
        if (cudaEventCreate(&g_rec.ev[i]) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(g_rec.ev[j]);
            return false;
        }
    g_rec.created = true;
    return true;
}

}  // namespace

void stage_begin(cudaStream_t, const char* call) {
    nvtx_push(call);
    t_stage_open = false;
    if (g_rec.on) g_rec.n = 0;
}

void stage_mark(cudaStream_t s, const char* name) {
    if (t_stage_open) nvtx_pop();
    nvtx_push(name);
    t_stage_open = true;
    if (!g_rec.on || g_rec.n >= kMaxMarks - 1) return;
    if (cudaEventRecord(g_rec.ev[g_rec.n], s) != cudaSuccess) return;
    g_rec.name[g_rec.n++] = name;
}

void stage_end(cudaStream_t s) {
    if (t_stage_open) nvtx_pop();
    t_stage_open = false;
    nvtx_pop();
    if (!g_rec.on || g_rec.n == 0) return;
    if (cudaEventRecord(g_rec.ev[g_rec.n], s) != cudaSuccess) return;
    g_rec.done = g_rec.n;
}

}  // namespace moe

extern "C" {

int moe_stage_timing(int enable) {
    using moe::g_rec;
    if (enable && !moe::create_events()) return MOE_ERR_CUDA;
    g_rec.on = enable != 0;
    g_rec.n = 0;
    g_rec.done = -1;
    return MOE_OK;
}

int moe_stage_times(float* ms, const char** names, int max_stages) {
    using moe::g_rec;
    if (ms == nullptr || max_stages < 0) return MOE_ERR_NULL;
    if (!g_rec.on || g_rec.done < 0) return 0;
    if (cudaEventSynchronize(g_rec.ev[g_rec.done]) != cudaSuccess) return MOE_ERR_CUDA;
    const int n = g_rec.done < max_stages ? g_rec.done : max_stages;
    for (int i = 0; i < n; ++i) {
        if (cudaEventElapsedTime(&ms[i], g_rec.ev[i], g_rec.ev[i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
        if (names) names[i] = g_rec.name[i];
    }
    return n;
}

}  // extern "C"
