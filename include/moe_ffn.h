/*
 * moe_ffn.h - C ABI of the GB300 (sm_103a) routed mixture-of-experts FFN library
 * (libmoe_ffn_gb300.so).
 *
 * The operation (one MoE FFN site, top-k routing):
 *
 *   for each token t and slot k with expert e = topk_ids[t][k]:
 *       g = Wg[e] . x[t]        u = Wu[e] . x[t]                      (gate, up: [I] each)
 *       a = silu(min(g, limit)) * clamp(u, -limit, limit)             (clamped SwiGLU)
 *       y = Wd[e] . a                                                  (down: [H])
 *   out[t] = sum_{k = 0 .. topk-1, in slot order} topk_weights[t][k] * y(t, k)   -> bf16
 *
 * Sources: the per-expert chain is "memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs",
 * `reference_expert`; the asymmetric clamp is "spark_model layers/glm5next_mlp/forward.rs",
 * `swiglu_rows`; the slot-order combine is ep_step_fp8_gate.rs, `combine_down_rows_host`.
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except where a comment
 *     says otherwise. No call allocates memory. The only state the library keeps between calls
 *     is the scratch array of moe_fp8_forward_noalloc (and its cached device address), a few
 *     per-device launch parameters it caches, and the switches of moe_stage_timing and
 *     moe_test_barrier_timeout. Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *     stream) and the function returns after enqueueing; nothing is synchronised.
 *   - Argument checks are synchronous: on any MOE_ERR_* return nothing has been enqueued, except
 *     MOE_ERR_CUDA, which reports a launch failure (work before the failing launch may be queued).
 *   - Route ids: -1 marks an unfilled slot and contributes exactly 0. Any other id outside
 *     [0, E) also contributes 0 and ORs bit 0 (MOE_ERRBIT_BAD_ID) into *err when err != NULL.
 *     err is never cleared by the library. Duplicate ids within one token are legal and summed.
 *   - Outputs are a deterministic function of the inputs: no floating-point atomics, fixed
 *     reduction order. `out` must not alias x, the weights or the workspace.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Shapes: 1 <= topk <= 8; H and I are multiples of 128; E >= 1.
 */
#ifndef MOE_FFN_GB300_H
#define MOE_FFN_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_NULL = -1,        /* a required pointer is NULL                                   */
    MOE_ERR_SHAPE = -2,       /* T < 1, topk outside 1..8, H or I not a positive multiple of 128,
                                 E < 1, or a size too large for the tier                       */
    MOE_ERR_WORKSPACE = -3,   /* workspace NULL or smaller than moe_workspace_bytes()         */
    MOE_ERR_VALUE = -4,       /* limit is NaN or <= 0 (use +INFINITY for "no clamp"), or a
                                 scale_2 that is not finite                                    */
    MOE_ERR_CUDA = -5,        /* a kernel launch or attribute call failed                      */
    MOE_ERR_UNSUPPORTED = -6, /* shape outside what this build's kernels cover                 */
    MOE_ERR_ALIGN = -7        /* x, out or a weight/scale array is not 16-byte aligned          */
} moe_status;

typedef enum {
    MOE_FMT_FP8_E4M3_B128 = 1, /* E4M3 codes + one fp32 scale per 128x128 block              */
    MOE_FMT_NVFP4 = 2          /* packed E2M1 + E4M3 scale per 16 elements + fp32 scale_2     */
} moe_format;

#define MOE_ERRBIT_BAD_ID 1
/* A bounded wait gave up (about 1-2 s of SM clock): the grid-wide barrier of the cooperative
 * forward (possible only if the GPU could not keep all of its CTAs resident) or a pipeline wait of
 * the grouped-GEMM tier. The output of that call is invalid. The cooperative forward writes NaN to
 * the output rows of every CTA that gave up, so the failure shows in `out` even when err is NULL;
 * the grouped-GEMM tier leaves the rows of the tiles it abandoned unwritten and reports the
 * failure only through *err. */
#define MOE_ERRBIT_BARRIER 2
/* After such an abort, a grouped-GEMM CTA's wait for its own TMA loads and MMAs in flight also
 * timed out before it released its shared and tensor memory. */
#define MOE_ERRBIT_DRAIN 4

/*
 * moe_workspace_bytes - device scratch needed by moe_fp8_forward / moe_nvfp4_forward for a call
 * with these sizes (and any smaller T). A pure function of its arguments; 0 on invalid sizes.
 * The workspace is fully rewritten by every call before it is read, so it needs no clearing.
 * Sizing idea: "spark_model layers/glm5next_mlp/forward.rs", `mlp_ws_bytes` (scratch sized once
 * for the widest call a site can make).
 */
MOE_API size_t moe_workspace_bytes(int T, int H, int I, int E, int topk, int fmt);

/*
 * moe_route_permute - route histogram and stable counting-sort of (token, slot) pairs by expert.
 *
 *   topk_ids        [T][topk] int32, row-major.
 *   counts          [E]       out: number of pairs routed to each expert.
 *   offsets         [E+1]     out: exclusive prefix sum of counts; offsets[E] = routed pairs.
 *   sorted_pair     [T*topk]  out: sorted_pair[offsets[e] + r] = the r-th pair p = t*topk + k
 *                             (ascending p) with topk_ids[p] == e; entries from offsets[E] on
 *                             are -1.
 *   pair_to_sorted  [T*topk]  out: inverse of sorted_pair; -1 for pairs that are not routed.
 *   err             nullable; bit 0 set on an id outside [-1, E).
 *
 * Equal keys keep ascending pair order, so every output is unique and bit-exact.
 * Source: "spark_model layers/glm5next_mlp/forward.rs", `Glm5NextMlpWorkspace` (sorted token ids,
 * expert_offsets[E+1], token_to_perm) and the `moe_sort_by_expert` step of `forward_moe`.
 * Limits: E <= 4096 (MOE_ERR_UNSUPPORTED beyond). One launch, no host synchronisation.
 */
MOE_API int moe_route_permute(const int32_t* topk_ids, int T, int topk, int E, int32_t* counts,
                      int32_t* offsets, int32_t* sorted_pair, int32_t* pair_to_sorted,
                      int32_t* err, void* stream);

/*
 * moe_fp8_forward - routed MoE FFN with E4M3 weights and one fp32 scale per 128x128 block.
 *
 *   x             [T][H]      bf16 activations.
 *   topk_ids      [T][topk]   int32 expert ids.
 *   topk_weights  [T][topk]   fp32 router weights.
 *   w_gate, w_up  [E][I][H]   uint8 E4M3 codes (K = H contiguous);
 *   s_gate, s_up  [E][I/128][H/128] fp32 block scales.
 *   w_down        [E][H][I]   uint8 E4M3 codes;  s_down [E][H/128][I/128] fp32.
 *                 Dequantised weight W[e][n][k] = e4m3(code) * s[e][n/128][k/128]
 *                 ("memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs", `expert_matrix`).
 *   limit         SwiGLU clamp (> 0; +INFINITY = no clamp).
 *   out           [T][H]      bf16, fully written (zero for a token with no routed slot).
 *   workspace     >= moe_workspace_bytes(T, H, I, E, topk, MOE_FMT_FP8_E4M3_B128) bytes,
 *                 256-byte aligned.
 *
 * Arithmetic: weight codes decode exactly to f16 (the grouped-GEMM tier then multiplies each by
 * its block scale times a power of two in f16, one rounding per weight; the GEMV tiers apply the
 * scale in fp32), activations are carried as f16 with a power-of-two scale per token (and per
 * 64-wide block of the activation a in the GEMV tiers; per sorted row in the grouped-GEMM tier,
 * or one fixed power of two there when a clamp limit <= 255 bounds |a| by limit^2), products
 * accumulate in fp32, the grouped-GEMM tier keeps each pair's down output in f16 times a power of
 * two chosen from a bound on it, the combine runs in slot order in fp32, and the result is
 * rounded once to bf16.
 *
 * Tiers (chosen from the sizes alone): T == 1 two kernels; 2 <= T <= 8 one cooperative kernel;
 * larger T the grouped GEMM over expert-sorted rows on the tcgen05 tensor cores (measured faster
 * than sweeps of <= 8 rows from T = 9 on) when it covers the shape - H, I <= 8192, E <= 4096 -
 * the workspace then holding the sorted rows, about P*(2H + 2I + 4*max(H,I)) bytes for
 * P = T*topk; otherwise the cooperative kernel in even sweeps of <= 8 rows.
 */
MOE_API int moe_fp8_forward(const uint16_t* x, int T, int H, int I, int E, int topk,
                    const int32_t* topk_ids, const float* topk_weights,
                    const uint8_t* w_gate, const float* s_gate,
                    const uint8_t* w_up, const float* s_up,
                    const uint8_t* w_down, const float* s_down,
                    float limit, uint16_t* out, void* workspace, size_t workspace_bytes,
                    int32_t* err, void* stream);

/*
 * moe_nvfp4_forward - routed MoE FFN with NVFP4 (W4A16) weights.
 *
 *   w_gate, w_up  [E][I][H/2]   packed E2M1 codes: element 2j in the low nibble of byte j.
 *   sf_gate, sf_up [E][I][H/16] E4M3 scale bytes, one per 16 consecutive K elements.
 *   w_down        [E][H][I/2];  sf_down [E][H][I/16].
 *   scale2_*      one fp32 per projection, passed BY VALUE.
 *                 W[e][n][k] = e2m1(nibble) * e4m3(sf[e][n][k/16]) * scale_2
 *                 ("memra-engine 0.131.0 src/dsv4_ep.rs", `chain`: wstride = inter*hidden/2,
 *                 sstride = inter*hidden/16; "spark_model layers/glm5next_mlp/forward.rs",
 *                 `w4a16_gemv`: scale_2 is a by-value scalar).
 * Everything else as moe_fp8_forward; the grouped-GEMM tier (T > 8) also needs H and I to be
 * multiples of 256, otherwise T > 8 runs as sweeps of <= 8 tokens through the cooperative kernel.
 * Arithmetic: an E2M1 code times its E4M3 scale is exact in f16, so every stage scales each code
 * in f16 with no rounding, except a single token's gate/up, which scales each 16-wide group's
 * fp32 partial sum once (and gives its activation a one power-of-two scale per 32-wide block
 * instead of 64). scale_2 and the activation scales apply in fp32.
 */
MOE_API int moe_nvfp4_forward(const uint16_t* x, int T, int H, int I, int E, int topk,
                      const int32_t* topk_ids, const float* topk_weights,
                      const uint8_t* w_gate, const uint8_t* sf_gate, float scale2_gate,
                      const uint8_t* w_up, const uint8_t* sf_up, float scale2_up,
                      const uint8_t* w_down, const uint8_t* sf_down, float scale2_down,
                      float limit, uint16_t* out, void* workspace, size_t workspace_bytes,
                      int32_t* err, void* stream);

/*
 * moe_nvfp4_forward_expert_scale2 - moe_nvfp4_forward with one scale_2 per expert and projection,
 * as a checkpoint quantised expert by expert stores it:
 *   W[e][n][k] = e2m1(nibble) * e4m3(sf[e][n][k/16]) * scale2_x[e * scale2_stride]
 * ("spark_model layers/glm5next_mlp/forward.rs", `w4a16_gemv_moe`: the expert table passes its
 * scale2_vals, one per expert; "memra-engine 0.131.0 src/dsv4_ep.rs", the EP matrix test: one
 * macro scale per expert and projection).
 *   scale2_gate, scale2_up, scale2_down  device fp32 arrays, 4-byte aligned; expert e's value at
 *                 element e * scale2_stride, so separate [E] arrays (stride 1) and one [E][3]
 *                 table (the three pointers offset by the projection's column, stride 3) both work.
 *   scale2_stride >= 1.
 * Everything else (sizes, tiers, workspace, err, stream, arithmetic) as moe_nvfp4_forward, the
 * per-expert value taking the scalar's place in each tier. The values are read on the device:
 * they are not checked, and a non-finite one makes that expert's outputs non-finite.
 * Errors: MOE_ERR_NULL for a null table, MOE_ERR_VALUE for scale2_stride < 1 (and as
 * moe_nvfp4_forward), MOE_ERR_ALIGN for a table that is not 4-byte aligned.
 */
MOE_API int moe_nvfp4_forward_expert_scale2(const uint16_t* x, int T, int H, int I, int E, int topk,
                                            const int32_t* topk_ids, const float* topk_weights,
                                            const uint8_t* w_gate, const uint8_t* sf_gate,
                                            const float* scale2_gate, const uint8_t* w_up,
                                            const uint8_t* sf_up, const float* scale2_up,
                                            const uint8_t* w_down, const uint8_t* sf_down,
                                            const float* scale2_down, int scale2_stride, float limit,
                                            uint16_t* out, void* workspace, size_t workspace_bytes,
                                            int32_t* err, void* stream);

/*
 * moe_fp8_forward_layer / moe_nvfp4_forward_layer - the forwards above with the MoE layer's
 * epilogue fused into the combine: out = bf16(((sum_k w[t,k] * y[t,k]) + shared[t]) + residual[t]),
 * the two adds in fp32 in that order after the slot-order sum, one rounding
 * ("spark_model layers/glm5next_mlp/forward.rs", `forward_moe`: the shared expert's output enters
 * the routed combine, not routed-scaled; the Step gate's full-layer check: final add order
 * routed-plus-shared-then-residual).
 *   shared    [T][H] bf16 shared-expert output (e.g. from moe_shared_expert_bf16), or NULL.
 *   residual  [T][H] bf16 residual stream, or NULL.  Both device pointers, 16-byte aligned, and
 *             neither may alias out.
 * Everything else as the forwards above (same workspace size).
 */
MOE_API int moe_fp8_forward_layer(const uint16_t* x, int T, int H, int I, int E, int topk,
                                  const int32_t* topk_ids, const float* topk_weights,
                                  const uint8_t* w_gate, const float* s_gate,
                                  const uint8_t* w_up, const float* s_up,
                                  const uint8_t* w_down, const float* s_down, float limit,
                                  const uint16_t* shared, const uint16_t* residual, uint16_t* out,
                                  void* workspace, size_t workspace_bytes, int32_t* err, void* stream);
MOE_API int moe_nvfp4_forward_layer(const uint16_t* x, int T, int H, int I, int E, int topk,
                                    const int32_t* topk_ids, const float* topk_weights,
                                    const uint8_t* w_gate, const uint8_t* sf_gate, float scale2_gate,
                                    const uint8_t* w_up, const uint8_t* sf_up, float scale2_up,
                                    const uint8_t* w_down, const uint8_t* sf_down, float scale2_down,
                                    float limit, const uint16_t* shared, const uint16_t* residual,
                                    uint16_t* out, void* workspace, size_t workspace_bytes,
                                    int32_t* err, void* stream);

/*
 * moe_nvfp4_forward_layer_expert_scale2 - moe_nvfp4_forward_layer with one scale_2 per expert and
 * projection: the tables, stride and errors of moe_nvfp4_forward_expert_scale2, the shared and
 * residual inputs and the single-rounding epilogue of moe_nvfp4_forward_layer.
 */
MOE_API int moe_nvfp4_forward_layer_expert_scale2(const uint16_t* x, int T, int H, int I, int E, int topk,
                                                  const int32_t* topk_ids, const float* topk_weights,
                                                  const uint8_t* w_gate, const uint8_t* sf_gate,
                                                  const float* scale2_gate, const uint8_t* w_up,
                                                  const uint8_t* sf_up, const float* scale2_up,
                                                  const uint8_t* w_down, const uint8_t* sf_down,
                                                  const float* scale2_down, int scale2_stride, float limit,
                                                  const uint16_t* shared, const uint16_t* residual,
                                                  uint16_t* out, void* workspace, size_t workspace_bytes,
                                                  int32_t* err, void* stream);

/*
 * Stage entry points. moe_plan, then moe_*_gate_up, then moe_*_down_combine (on one stream, same
 * workspace, same arguments as the forward they stand for) compute exactly the bits of
 * moe_*_forward for T <= 8, as three separate kernels; moe_*_forward runs the same work items in
 * one fused cooperative launch. They are exported so that a caller (or a profiler) can time or
 * interleave the stages.
 *
 * moe_plan            - groups the routed (token, slot) pairs by expert into the workspace
 *                       (one launch; a no-op for T == 1, where slot k is group k).
 * moe_*_gate_up       - dequant-fused gate and up projections for every group, clamped SwiGLU
 *                       fused in; writes the activation a (f16, per-64 power-of-two scales) to
 *                       the workspace.
 * moe_*_down_combine  - dequant-fused down projection fused with the slot-order weighted
 *                       combine; writes out.
 */
MOE_API int moe_plan(int T, int H, int I, int E, int topk, int fmt, const int32_t* topk_ids,
             void* workspace, size_t workspace_bytes, int32_t* err, void* stream);

MOE_API int moe_fp8_gate_up(const uint16_t* x, int T, int H, int I, int E, int topk,
                    const int32_t* topk_ids, const uint8_t* w_gate, const float* s_gate,
                    const uint8_t* w_up, const float* s_up, float limit, void* workspace,
                    size_t workspace_bytes, int32_t* err, void* stream);

MOE_API int moe_fp8_down_combine(int T, int H, int I, int E, int topk, const int32_t* topk_ids,
                         const float* topk_weights, const uint8_t* w_down, const float* s_down,
                         uint16_t* out, void* workspace, size_t workspace_bytes, void* stream);

MOE_API int moe_nvfp4_gate_up(const uint16_t* x, int T, int H, int I, int E, int topk,
                      const int32_t* topk_ids, const uint8_t* w_gate, const uint8_t* sf_gate,
                      float scale2_gate, const uint8_t* w_up, const uint8_t* sf_up,
                      float scale2_up, float limit, void* workspace, size_t workspace_bytes,
                      int32_t* err, void* stream);

MOE_API int moe_nvfp4_down_combine(int T, int H, int I, int E, int topk, const int32_t* topk_ids,
                           const float* topk_weights, const uint8_t* w_down,
                           const uint8_t* sf_down, float scale2_down, uint16_t* out,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_fp8_forward_noalloc - moe_fp8_forward for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point. It exists for callers that cannot call
 * cudaMalloc or pass a workspace: for example a plugin that only receives input and output
 * pointers through a fixed interface, or a latency-critical loop that forbids device allocation
 * because cudaMalloc/cudaFree can implicitly synchronise the device. Arguments are those of
 * moe_fp8_forward without the workspace; the caller still passes every input and the output.
 *
 * Scratch: a file-scope device array of MOE_NOALLOC_SCRATCH_BYTES inside the library, present on
 * every GPU that loads the library until the process exits. Calls whose
 * moe_workspace_bytes(T, H, I, E, topk, MOE_FMT_FP8_E4M3_B128) exceeds it return
 * MOE_ERR_WORKSPACE with nothing enqueued (e.g. T <= 8, I = 2048, E = 256 needs about 270 KB).
 * All calls on a device share the array and it keeps the last call's contents; nothing in it
 * needs to start at zero. Calls that overlap on the GPU race on it: serialise them.
 * The first call on each device (with that device current) looks up the array's device address
 * with cudaGetSymbolAddress, which may load the library's kernels; make it before any stream
 * capture. The address is kept per device and per CUDA context: after cudaDeviceReset() the next
 * call on that device looks it up again (make that call outside a capture too). No cudaMalloc,
 * cudaFree or allocating library routine is ever called.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)
MOE_API int moe_fp8_forward_noalloc(const uint16_t* x, int T, int H, int I, int E, int topk,
                                    const int32_t* topk_ids, const float* topk_weights,
                                    const uint8_t* w_gate, const float* s_gate,
                                    const uint8_t* w_up, const float* s_up,
                                    const uint8_t* w_down, const float* s_down, float limit,
                                    uint16_t* out, int32_t* err, void* stream);

/*
 * moe_router - the router in front of the FFN: logits, sigmoid, selection bias, top-k, weights.
 * ("spark_model layers/glm5next_mlp/forward.rs", `forward_moe` router step: one f32-output logits
 * GEMM over all rows, then one top-k launch taking logits, router_bias, top_k, n_group = 1,
 * routed_scale, renormalize; the Step gate's sigmoid top-k router takes the same router matrix,
 * bias, top_k, router_scale and route_norm.)
 *
 *   x            [T][H]  bf16 (device).         router_w [E][H] bf16 (device, K = H contiguous).
 *   bias         [E] fp32 selection bias (device) or NULL for none.
 *   logits       [T][E] fp32 out (device) or NULL: l = sum_h x[t][h] * router_w[e][h], fp32 MMA
 *                accumulation.
 *   topk_ids     [T][topk] int32 out: experts by descending sigmoid(l) + bias; equal scores go to
 *                the lower expert index (the pages print no tie rule; this is the stable one). The
 *                ids of a token are always distinct and in [0, E): a -inf score is picked only
 *                after every finite one, a NaN score (NaN logit or bias) only after every number.
 *   topk_weights [T][topk] fp32 out: sigmoid(l) of each pick (the bias only selects), divided by
 *                the sum over the picks if renormalize != 0, times routed_scale.
 *   workspace    >= moe_router_workspace_bytes(T, H, E) bytes (device, 256-byte aligned): partial
 *                logits of a K split for small T.
 * Limits: 16 <= E <= 1024 with E % 16 == 0, H % 32 == 0, 1 <= topk <= min(8, E), routed_scale
 * finite and > 0, x and router_w 16-byte aligned. Errors return synchronously (MOE_ERR_*) with
 * nothing enqueued; otherwise two launches on `stream`, no host synchronisation. Deterministic.
 */
MOE_API size_t moe_router_workspace_bytes(int T, int H, int E);
MOE_API int moe_router(const uint16_t* x, int T, int H, const uint16_t* router_w, const float* bias,
                       int E, int topk, float routed_scale, int renormalize, float* logits,
                       int32_t* topk_ids, float* topk_weights, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * moe_shared_expert_bf16 - the MoE layer's shared expert, a dense BF16 SwiGLU MLP over all tokens
 * ("spark_model layers/glm5next_mlp/forward.rs", `forward_moe`: `forward_dense` on the shared
 * weights into `shared_out`; the Step gate's replicated BF16 SwiGLU with its own limit):
 *   out[t] = bf16( Wd . bf16( silu(min(Wg.x[t], L)) * clamp(Wu.x[t], -L, L) ) ), fp32 accumulation.
 *   x [T][H] bf16; w_gate, w_up [S][H] bf16; w_down [H][S] bf16; out [T][H] bf16 (device).
 *   workspace >= moe_shared_expert_workspace_bytes(T, H, S) bytes, 256-byte aligned.
 * Limits: H, S multiples of 32; limit > 0 (+INFINITY: no clamp); 16-byte aligned arrays. Errors
 * return synchronously with nothing enqueued; otherwise five launches, no host synchronisation.
 */
MOE_API size_t moe_shared_expert_workspace_bytes(int T, int H, int S);
MOE_API int moe_shared_expert_bf16(const uint16_t* x, int T, int H, int S, const uint16_t* w_gate,
                                   const uint16_t* w_up, const uint16_t* w_down, float limit,
                                   uint16_t* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Stage timing (tracing, off by default). moe_stage_timing(1) makes every moe_*_forward and
 * moe_*_forward_layer call record a CUDA event on its stream before each of its stages (kernel
 * launches) and one after the last; moe_stage_timing(0) stops it. moe_stage_times blocks until
 * the most recent such call's last event has completed and writes, for its first
 * min(stages, max_stages) stages, the device time in ms (ms[i]) and a static stage name owned by
 * the library (names[i], when names != NULL). It returns the number written, 0 when timing is
 * off or no forward ran since it was switched on, MOE_ERR_NULL for ms == NULL, or MOE_ERR_CUDA.
 * The events serialise stages that otherwise overlap (programmatic dependent launches), so the
 * intervals are per-stage device times, and a timed forward can be slightly slower than an
 * untimed one. At most 63 stages per forward are kept. One process-wide recorder: call from one
 * host thread at a time.
 */
MOE_API int moe_stage_timing(int enable);
MOE_API int moe_stage_times(float* ms, const char** names, int max_stages);

/*
 * moe_test_barrier_timeout - test hook, off by default. While enabled (enable != 0), every
 * cooperative forward (2 <= T <= 8 rows per sweep) makes its grid-wide barrier wait for one CTA
 * more than the grid holds and gives up after about 10 ms instead of about 2 s, so that a test can
 * check the timeout path without a GPU fault: MOE_ERRBIT_BARRIER is set in *err, `out` holds NaN,
 * and the CUDA context stays usable. Returns MOE_OK. Process-wide; not for production calls.
 */
MOE_API int moe_test_barrier_timeout(int enable);

/*
 * moe_stream_read - measurement aid, not part of the forward. Reads the device buffer
 * [buf, buf + bytes) once with one plain streaming kernel (16-byte loads, consecutive threads on
 * consecutive words, two 512-thread blocks per SM) and XORs every 32-bit word of it into *sink
 * (device memory; not cleared by the library, so the caller zeroes it first; the fold does not
 * depend on the order of the blocks). What this kernel reaches on a given byte count, timed the
 * way a forward is timed, is the read throughput one kernel of that size gets from HBM on the
 * device: launch latency and the ramp at either end weigh more the fewer bytes a call moves, so
 * the fraction of the peak copy bandwidth a forward can reach depends on its size. The benchmark
 * reports it beside each bandwidth-bound workload's fraction.
 *   buf    device pointer, 16-byte aligned (MOE_ERR_ALIGN), read only.
 *   bytes  a positive multiple of 16 (MOE_ERR_SHAPE otherwise).
 *   sink   device pointer to one uint32_t, 4-byte aligned.
 * Returns MOE_OK, MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_ALIGN or MOE_ERR_CUDA. One launch.
 */
MOE_API int moe_stream_read(const void* buf, size_t bytes, uint32_t* sink, void* stream);

/* Library build identification: the compiled CUDA architecture string (e.g. "sm_103a"). */
MOE_API const char* moe_build_arch(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_FFN_GB300_H */
