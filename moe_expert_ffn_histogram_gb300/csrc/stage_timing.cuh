// Stage hooks of the forward paths (stage_timing.cu): NVTX ranges for profilers (one per call,
// one per stage inside it; MOE_NVTX=0 builds them out), and CUDA events per stage once
// moe_stage_timing(1) switched the recorder on.
#pragma once
#include <cuda_runtime.h>

namespace moe {

void stage_begin(cudaStream_t s, const char* call);   // a forward called `call` starts
void stage_mark(cudaStream_t s, const char* name);    // a stage called `name` starts here
void stage_end(cudaStream_t s);

// begin on construction, end (one event after the last stage) on every return path
struct StageScope {
    cudaStream_t s;
    StageScope(cudaStream_t st, const char* call) : s(st) { stage_begin(s, call); }
    ~StageScope() { stage_end(s); }
};

}  // namespace moe
