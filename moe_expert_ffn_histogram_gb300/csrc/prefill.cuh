// Shared pieces of the grouped-GEMM (prefill) tier: tile shape, the GEMM argument block, and
// the two GEMM cores (mma.sync in prefill.cu, tcgen05/TMEM in prefill_tc.cu).
#pragma once
#include "gemv_items.cuh"

namespace moe {

namespace prefill {

constexpr int kBM = 128;               // sorted rows per tile
constexpr int kBN = 128;               // weight rows per tile (gate/up: 64 gate + the same 64 up)
constexpr int kBK = 64;                // K per pipeline stage
constexpr int kThreads = 256;          // 8 warps: 2 (rows) x 4 (columns), warp tile 64 x 32
constexpr int kStages = 3;
constexpr int kARow = kBK * 2 + 32;    // A smem row pitch in bytes (f16 + 32 B pad: no conflicts)
constexpr int kBRow = kBK + 16;        // B smem row pitch in bytes (fp8 + 16 B pad: no conflicts)
constexpr int kAStage = kBM * kARow;
constexpr int kBStage = kBN * kBRow;
constexpr int kSmem = kStages * (kAStage + kBStage);

}  // namespace prefill

struct PrefillGemmArgs {
    // tile schedule
    const int32_t* tiles;        // [1] number of m-tiles
    const int32_t* tile_e;       // [m-tiles]
    const int32_t* tile_r0;      // [m-tiles]
    const int32_t* offsets;      // [E+1]
    const int32_t* sorted_pair;  // [P]
    int topk, K, n_tiles;
    // A operand: rows of a16 (KIND 1) or rows of x16 gathered through sorted_pair (KIND 0)
    const __half* a;
    const float* a_inv;          // per token (KIND 0) or per sorted row (KIND 1)
    // B operand: E4M3 weight rows and fp32 block scales; KIND 0 uses both gate (w0) and up (w1)
    const uint8_t* w0;
    const float* s0;
    const uint8_t* w1;
    const float* s1;
    int wrows;                   // rows of one expert's weight matrix (I for gate/up, H for down)
    float limit;
    // outputs
    float* out;                  // KIND 0: a32 [P][I]; KIND 1: y [P][H]
    uint32_t* amax;              // KIND 0: per sorted row max |a| (float bits), zeroed before
    int out_ld;                  // I (KIND 0) or H (KIND 1)
    int32_t* err;                // optional error word (bit 1: a bounded wait gave up)
};

// Launch one grouped GEMM (KIND 0: gate/up + SwiGLU, KIND 1: down) on the simple tcgen05 core
// (prefill_tc.cu) or the warp-specialised one (prefill_ws.cu; N_total = I or H, it picks its own
// column tiling and sets n_tiles).
cudaError_t launch_prefill_gemm_tc(int kind, const PrefillGemmArgs& p, cudaStream_t stream);
cudaError_t launch_prefill_gemm_ws(int kind, const PrefillGemmArgs& p, int N_total, cudaStream_t stream);

}  // namespace moe
