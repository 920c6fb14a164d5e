// Stage timing hooks of the forward paths (stage_timing.cu); no-ops unless moe_stage_timing(1)
// switched the recorder on.
#pragma once
#include <cuda_runtime.h>

namespace moe {

void stage_begin(cudaStream_t s);
void stage_mark(cudaStream_t s, const char* name);   // a stage called `name` starts here
void stage_end(cudaStream_t s);

// begin on construction, end (one event after the last stage) on every return path
struct StageScope {
    cudaStream_t s;
    explicit StageScope(cudaStream_t st) : s(st) { stage_begin(s); }
    ~StageScope() { stage_end(s); }
};

}  // namespace moe
