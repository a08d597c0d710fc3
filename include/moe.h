/*
 * moe.h: C ABI of the GB300 (sm_103a) MoE layer forward hot path and its backward.
 *
 *   router -> dispatch -> grouped SwiGLU expert FFN -> combine
 *
 * The steps follow the MoE data flow of "Megatron-LM 分布式训练（六）：MoE 专家并行 EP 与上下文并行 CP"
 * (section "MoE 层的数据流") and the shape table of "v6 长序列和 MoE: Context Parallel 与 Expert Parallel"
 * (section "NVIDIA 原题: Implement MoE and show the dimensions"):
 *   x [T,h] -> router logits [T,E] -> top-k [T,k] -> dispatch [E,C,h] (or dropless blocks) -> expert FFN
 *   -> combine y [T,h].
 *
 * Conventions (every entry point):
 *   - Tensor arguments are DEVICE pointers owned by the caller, row-major with the last dimension
 *     contiguous. The library never allocates memory: calls that need scratch take a caller-provided
 *     device workspace whose size the matching *_workspace_size() function returns. One exception:
 *     moe_dispatch_static keeps its scratch in a fixed 1 MiB device array of the library's own (held for the
 *     life of the process and shared by all its calls, so overlapping calls must be serialised by the caller).
 *   - Per-device state the library caches (the device error word's and that array's addresses, kernel
 *     attributes) is keyed by the CUDA context it was set up in and set up again in a new context, e.g. after
 *     cudaDeviceReset; the first call in a new context should come before any stream capture in it.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Every call only
 *     enqueues work on that stream; none synchronizes the host.
 *   - Return value: MOE_OK, or an error code with a message retrievable by moe_last_error_string()
 *     (per host thread). Argument checks happen before anything is enqueued, so a call that returns
 *     MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE has not touched device memory.
 *     MOE_ERR_CUDA reports a failed launch. Errors detected on the device (a bounded wait that ran out,
 *     an expert id outside [0, E)) are latched in a device word and reported by moe_check_device_error().
 *   - dtype: MOE_F32 (fp32 in/out, fp32 arithmetic) or MOE_BF16 (bf16 tensors, fp32 accumulation).
 *     Gates, logits, f, P and aux are always fp32.
 *   - Sizes: T >= 0; 1 <= k <= min(E, 16); 1 <= E <= 1024; h % 8 == 0; F % 8 == 0. All tensor pointers
 *     must be 16-byte aligned.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, size out of range */
    MOE_ERR_UNSUPPORTED = 2,  /* dtype, gating mode or shape this build does not handle */
    MOE_ERR_WORKSPACE = 3,    /* workspace smaller than *_workspace_size() */
    MOE_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed */
    MOE_ERR_TIMEOUT = 5       /* a bounded device-side wait ran out (see moe_check_device_error) */
};

enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 };

/* Gating modes ("Megatron-LM ... （六）", section "Router": top-k on the logits with softmax or sigmoid
 * weights; "v6 长序列和 MoE ...", "Load balancing loss" bullet: DeepSeek-V3 selection-only bias). */
enum moe_gating {
    MOE_GATING_SOFTMAX = 0,            /* gate = full-softmax probability of the chosen expert */
    MOE_GATING_SOFTMAX_RENORM = 1,     /* gate = softmax probability / sum over the k chosen */
    MOE_GATING_SIGMOID_BIAS_RENORM = 2, /* select on sigmoid(L)+bias; gate = s / sum_chosen s */
    MOE_GATING_SOFTMAX_SELBIAS = 3      /* select on L+bias (bias: selection only, e.g. the Sinkhorn log column
                                           scalings of moe_sinkhorn_bias); gate = full-softmax probability */
};

/* Rows per tile of the device tile schedule written by moe_dispatch and read by the expert FFN. */
#define MOE_TILE_M 128

/* ---------------------------------------------------------------------------------------------------
 * moe_router: gating GEMM, top-k, gates, per-expert counts and Switch aux-loss terms.
 *   "Megatron-LM ... （六）", section "Router" (logits = hidden_states @ W_router, then top-k with
 *   softmax/sigmoid weights); "v6 长序列和 MoE ...", table rows "router" and "top-k", and the
 *   "Load balancing loss" bullet (aux = alpha * E * sum_i f_i P_i).
 *
 *   x        [T,h]  dtype        tokens
 *   w_r      [h,E]  dtype        router weight
 *   bias     [E]    fp32 or NULL softmax modes: added to the logits; sigmoid mode: selection only
 *   logits   [T,E]  fp32 or NULL x @ w_r (+ bias in softmax modes)
 *   topk_ids [T,k]  int32        chosen experts, by descending selection score, ties -> lower index
 *   gates    [T,k]  fp32         gate of each chosen expert (see enum moe_gating)
 *   counts   [E]    int32        assignments per expert before any capacity limit (sum = k*T)
 *   f        [E]    fp32         counts / (k*T)
 *   P        [E]    fp32         mean over tokens of the router probability (softmax modes: the full
 *                                softmax; sigmoid mode: s_e / sum_e' s_e')
 *   aux      [1]    fp32         alpha * E * sum_e f_e * P_e
 *   Deterministic: the same inputs give bitwise-identical outputs on every call.
 *   Errors: MOE_ERR_UNSUPPORTED for a dtype or gating value outside the enums; MOE_ERR_INVALID_ARG for
 *   h % 8 != 0, E or k out of range, a null output, or x / w_r / logits not 16-byte aligned;
 *   MOE_ERR_WORKSPACE if ws_bytes < moe_router_workspace_size().
 * ------------------------------------------------------------------------------------------------- */
size_t moe_router_workspace_size(int T, int h, int E, int k, int dtype);
int moe_router(const void* x, const void* w_r, const float* bias, int T, int h, int E, int k, int dtype,
               int gating, float alpha, float* logits, int32_t* topk_ids, float* gates, int32_t* counts,
               float* f, float* P, float* aux, void* ws, size_t ws_bytes, void* stream);

/* moe_pack_router_weight / moe_router_packed: moe_router on a router weight repacked once ("Megatron-LM ...
 *   （六）", section "Router": the same logits GEMM; the packing is this library's operand layout, not the pages').
 *   moe_pack_router_weight writes `packed` (moe_router_packed_bytes(h, E, dtype) bytes): for bf16 the transpose
 *   W_r^T [E,h] (the K-major operand of the logits GEMM, which moe_router otherwise builds in its workspace on
 *   every call), for fp32 a copy of w_r [h,E]. moe_router_packed takes that buffer in place of w_r; every other
 *   argument, the workspace size and the outputs (bitwise) are those of moe_router. Errors as moe_router;
 *   moe_pack_router_weight: MOE_ERR_INVALID_ARG for h % 8 != 0, E outside [1, 1024] or a null / misaligned
 *   pointer. With bf16 and E <= 32 the kernel's blocks wait (bounded, moe_set_wait_limit) for the packed rows'
 *   bulk copy into shared memory: if the wait runs out, moe_check_device_error() then reports MOE_ERR_TIMEOUT
 *   (site 0x130) and that call's outputs are not to be used; the context stays usable. */
size_t moe_router_packed_bytes(int h, int E, int dtype);
int moe_pack_router_weight(const void* w_r, int h, int E, int dtype, void* packed, void* stream);
int moe_router_packed(const void* x, const void* w_packed, const float* bias, int T, int h, int E, int k, int dtype,
                      int gating, float alpha, float* logits, int32_t* topk_ids, float* gates, int32_t* counts,
                      float* f, float* P, float* aux, void* ws, size_t ws_bytes, void* stream);

/* moe_router_from_logits: the gating part of moe_router (top-k, gates, counts, f, P, aux) on given fp32
 * logits [T,E] (as moe_router writes them: bias already added in the two plain softmax modes; in the sigmoid
 * and selection-bias modes `bias` is the selection-only term). Workspace: moe_router_from_logits_workspace_size. */
size_t moe_router_from_logits_workspace_size(int T, int E);
int moe_router_from_logits(const float* logits, const float* bias, int T, int E, int k, int gating, float alpha,
                           int32_t* topk_ids, float* gates, int32_t* counts, float* f, float* P, float* aux,
                           void* ws, size_t ws_bytes, void* stream);

/* moe_sinkhorn_bias: Sinkhorn routing ("Megatron-LM ... （六）", section "Router": Sinkhorn iterations make the
 * routing matrix doubly stochastic, balancing the experts without an aux loss). On K = exp(L - rowmax) [T,E]
 * and starting from row scalings r = 1, n_iter times: c_e = (T/E) / sum_t K[t,e] r_t, then
 * r_t = 1 / sum_e K[t,e] c_e. Writes sel_bias[e] = log c_e; the top-k of the balanced matrix
 * diag(r) K diag(c) is the top-k of L + sel_bias (moe_router_from_logits with MOE_GATING_SOFTMAX_SELBIAS).
 * fp32 with fixed-order sums (deterministic). Workspace: moe_sinkhorn_workspace_size(T, E). */
size_t moe_sinkhorn_workspace_size(int T, int E);
int moe_sinkhorn_bias(const float* logits, int T, int E, int n_iter, float* sel_bias, void* ws, size_t ws_bytes,
                      void* stream);

/* ---------------------------------------------------------------------------------------------------
 * moe_dispatch: histogram, exclusive scan, stable scatter, capacity mask, permutation indices, EP send
 * layout and the expert FFN's tile schedule.
 *   "v6 长序列和 MoE ...", table row "dispatch" (group by expert, at most C per expert, pad) and the
 *   "Capacity" bullet (C = cf*k*T/E; tokens over capacity are dropped); the follow-up note there (sort
 *   tokens by expert, one grouped GEMM); "专家并行" (formulaic), section "All2All" (the (E,C,M) buffer
 *   pre-sorted by destination expert; the all-to-all as a block transpose).
 *
 *   capacity  0 = dropless (rows = k*T, offsets = exclusive scan of counts), else C (rows = E*C,
 *             offsets[e] = e*C, pad rows zero). moe_dispatch_rows() returns rows.
 *   slot(t,j) = number of earlier assignments to the same expert in token order; kept iff dropless or
 *             slot < C.
 *   x           [T,h] dtype      tokens
 *   topk_ids    [T,k] int32      from moe_router (values in [0,E); a token never repeats an expert)
 *   buf         [rows,h] dtype   buf[dest_row[t,j]] = x[t]; pad rows zero
 *   offsets     [E+1] int32      first row of each expert block (offsets[E] = rows)
 *   kept_counts [E]   int32      rows used by each expert
 *   dest_row    [T,k] int32      row of (t,j) in buf, -1 if dropped
 *   drop_mask   [T,k] uint8      1 if (t,j) was dropped
 *   src_token   [rows] int32     token of each row, -1 on pad rows
 *   src_slot    [rows] int32     j of each row, -1 on pad rows
 *   rank_counts [R]   int32      kept rows of each virtual EP rank (rank r owns experts
 *                                [r*E/R, (r+1)*E/R); the expert-major buffer is already rank-major)
 *   rank_offsets[R+1] int32      first row of each rank block (= offsets[r*E/R])
 *   tile_sched  moe_tile_sched_bytes() bytes, opaque: per-expert MOE_TILE_M-row tiles for the FFN
 *   Deterministic and stable (token order inside every expert block).
 *   Errors: MOE_ERR_INVALID_ARG if num_ranks does not divide E, rows >= 2^31, capacity < 0, or a pointer
 *   is null or not 16-byte aligned (x, buf, tile_sched); MOE_ERR_WORKSPACE if ws_bytes <
 *   moe_dispatch_workspace_size(). An id outside [0, E) is treated as dropped and latched:
 *   moe_check_device_error() then returns MOE_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------------------------------- */
size_t moe_dispatch_rows(int T, int E, int k, int capacity);
size_t moe_tile_sched_bytes(int T, int E, int k, int capacity);
size_t moe_dispatch_workspace_size(int T, int E, int k, int capacity);
int moe_dispatch(const void* x, const int32_t* topk_ids, int T, int h, int E, int k, int capacity,
                 int num_ranks, int dtype, void* buf, int32_t* offsets, int32_t* kept_counts,
                 int32_t* dest_row, uint8_t* drop_mask, int32_t* src_token, int32_t* src_slot,
                 int32_t* rank_counts, int32_t* rank_offsets, int32_t* tile_sched, void* ws,
                 size_t ws_bytes, void* stream);

/* moe_dispatch_static: moe_dispatch for callers that cannot allocate device memory, such as a plugin whose
 * host framework owns all device memory, a latency-critical thread that may not allocate, or a program that
 * reserves all its memory at start-up. The paper has no counterpart: this is a library-usage variant.
 * Arguments and outputs are those of moe_dispatch minus the workspace: the scratch lives in a fixed 1 MiB
 * (1048576-byte) array of the library's own device memory, held by every GPU that loads the library until
 * the process exits. A size whose scratch (moe_dispatch_workspace_size) exceeds 1 MiB is rejected with
 * MOE_ERR_INVALID_ARG before anything is enqueued. The first call on a device (with that device current)
 * looks up the array's device address, and so does the first call in a new context of that device (after
 * cudaDeviceReset); make those calls before any stream capture on the device. All calls
 * share the array and each overwrites it: calls that may overlap on the GPU race and must be serialised by
 * the caller. No call allocates memory. */
int moe_dispatch_static(const void* x, const int32_t* topk_ids, int T, int h, int E, int k, int capacity,
                        int num_ranks, int dtype, void* buf, int32_t* offsets, int32_t* kept_counts,
                        int32_t* dest_row, uint8_t* drop_mask, int32_t* src_token, int32_t* src_slot,
                        int32_t* rank_counts, int32_t* rank_offsets, int32_t* tile_sched, void* stream);

/* Writes a tile schedule for one dense group of `rows` rows (offsets {0, rows}): the shared expert of a
 * DeepSeek-V3-shaped layer runs through the expert FFN with E = 1 and this schedule. */
int moe_dense_tile_sched(int rows, int32_t* tile_sched, void* stream);

/* ---------------------------------------------------------------------------------------------------
 * Expert-choice routing ("10.5 序列并行与专家并行", section 10.5.6, expert-choice bullet: the routing
 * direction is reversed and every expert takes a fixed number C of the highest-scoring tokens among all
 * tokens, which balances the expert load by construction).
 *   score[t,e] = softmax over experts of logits[t,:] (the logits of moe_router); expert e takes the C tokens
 *   with the highest score[:,e] (equal scores -> lower token index) and lays them out in rows e*C .. e*C+C-1
 *   in ascending token order; gate = score. A token chosen by no expert gets y = 0 (plus shared_out).
 *   moe_expert_choice_route:   logits [T,E] fp32 -> tokens [E,C] int32, gates [E,C] fp32, slot [T,E] int32
 *                              (row of (t,e) inside expert e's block, -1 if e did not choose t).
 *                              Workspace: moe_expert_choice_workspace_size(T, E) bytes. 1 <= C <= T, E <= 256.
 *   moe_expert_choice_dispatch: buf [E*C,h] dtype, buf[e*C+j] = x[tokens[e][j]]; tile_sched for the expert
 *                              FFN (moe_tile_sched_bytes(T, E, 1, C) bytes).
 *   moe_expert_choice_combine: y[t] = shared_out[t] + sum over experts e with slot[t][e] >= 0, ascending e, of
 *                              gates[e][slot] * eout[e*C + slot[t][e]]; fp32 accumulation, deterministic.
 * ------------------------------------------------------------------------------------------------- */
size_t moe_expert_choice_workspace_size(int T, int E);
int moe_expert_choice_route(const float* logits, int T, int E, int C, int32_t* tokens, float* gates, int32_t* slot,
                            void* ws, size_t ws_bytes, void* stream);
int moe_expert_choice_dispatch(const void* x, const int32_t* tokens, int T, int h, int E, int C, int dtype,
                               void* buf, int32_t* tile_sched, void* stream);
int moe_expert_choice_combine(const void* eout, const int32_t* slot, const float* gates, const void* shared_out,
                              int T, int h, int E, int C, int dtype, void* y, void* stream);

/* ---------------------------------------------------------------------------------------------------
 * moe_pack_expert_weights: one-time repack of the SwiGLU expert weights for the grouped GEMM.
 *   "v6 长序列和 MoE ...", section "MoE" (a SwiGLU FFN has three h x F matrices).
 *   w_gate [E,F,h], w_up [E,F,h], w_down [E,h,F] (nn.Linear layout, dtype) -> packed
 *   (moe_packed_weights_bytes() bytes, opaque): gate and up rows interleaved in blocks of 128 so that one
 *   GEMM tile computes both halves of the SwiGLU for the same 128 columns of F, and w_down.
 * ------------------------------------------------------------------------------------------------- */
size_t moe_packed_weights_bytes(int E, int h, int F, int dtype);
int moe_pack_expert_weights(const void* w_gate, const void* w_up, const void* w_down, int E, int h, int F,
                            int dtype, void* packed, void* stream);

/* ---------------------------------------------------------------------------------------------------
 * Grouped SwiGLU expert FFN ("Megatron-LM ... （六）", data flow: experts run as one GroupedGEMM;
 * "v6 长序列和 MoE ...", table row "expert": each expert runs its own FFN h -> F -> h).
 *   For every expert e and every kept row r in [offsets[e], offsets[e] + kept_counts[e]):
 *     act[r]  = silu(buf[r] @ W_gate[e]^T) * (buf[r] @ W_up[e]^T)     [rows,F] dtype
 *     eout[r] = act[r] @ W_down[e]^T                                    [rows,h] dtype
 *   Rows outside the kept ranges are not written. bf16 runs on the tcgen05 tensor cores (bf16 operands,
 *   fp32 accumulation in tensor memory; act is stored in bf16); fp32 runs on the CUDA cores.
 *   moe_expert_up_gate and moe_expert_down are the two steps; moe_expert_ffn runs both with act in the
 *   workspace.
 *   Errors: MOE_ERR_UNSUPPORTED for a dtype outside the enum; MOE_ERR_INVALID_ARG for E, h, F or rows out
 *   of range (h % 8, F % 8), a null pointer with rows > 0, or a pointer not 16-byte aligned.
 * ------------------------------------------------------------------------------------------------- */
int moe_expert_up_gate(const void* buf, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                       int rows, int dtype, void* act, void* stream);
int moe_expert_down(const void* act, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                    int rows, int dtype, void* eout, void* stream);
/* Routed experts and one shared expert in the same launch per GEMM ("Megatron-LM ... （六）", data flow:
 * the shared experts see every token and their output is added in the combine; the page's overlap
 * guidance is realised by appending the shared expert's tiles to the routed experts' work list of one
 * persistent tensor-core kernel, so they fill the routed GEMM's last partial wave instead of starting a
 * launch of their own).
 *   Routed part exactly as moe_expert_up_gate / moe_expert_down. Shared part, one dense group of T rows:
 *     act_shared[t] = silu(x[t] @ Ws_gate^T) * (x[t] @ Ws_up^T)          [T,F]
 *     out_shared[t] = act_shared[t] @ Ws_down^T                          [T,h]
 *   packed_shared: the shared expert packed by moe_pack_expert_weights with E = 1 (same h, F).
 *   bf16 only (MOE_ERR_UNSUPPORTED otherwise: fp32 callers make one call per group). tile_sched must be
 *   valid even when rows == 0. All pointers 16-byte aligned; rows == 0 and T == 0 is a no-op. */
int moe_expert_up_gate_shared(const void* buf, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                              int rows, const void* x, int T, const void* packed_shared, void* act_shared,
                              int dtype, void* act, void* stream);
int moe_expert_down_shared(const void* act, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                           int rows, const void* act_shared, int T, const void* packed_shared, void* out_shared,
                           int dtype, void* eout, void* stream);
/* moe_expert_up_gate_save: moe_expert_up_gate_shared (packed_shared may be NULL: routed experts only, x, T,
 *   act_shared and gu_shared unused) that also stores the pre-activations for the backward:
 *     gu [rows, 2*Fp] (Fp = F rounded up to 128; columns in blocks of 256: 128 of g = buf W_gate^T, then the
 *     u = buf W_up^T of the same f; f >= F zero), gu_shared [T, 2*Fp] likewise for the shared expert,
 *   both bf16 (rows outside the tiles' kept ranges not written). bf16 only; pointers 16-byte aligned. */
int moe_expert_up_gate_save(const void* buf, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                            int rows, const void* x, int T, const void* packed_shared, void* act_shared,
                            void* gu_shared, int dtype, void* act, void* gu, void* stream);
size_t moe_expert_ffn_workspace_size(int rows, int F, int dtype);
int moe_expert_ffn(const void* buf, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                   int rows, int dtype, void* eout, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------------
 * moe_combine: un-permute and gate-weighted sum of the k expert outputs.
 *   "v6 长序列和 MoE ...", table row "combine" (back to the original position, k outputs summed weighted
 *   by gate); "专家并行" (formulaic), forward pass (top-2 weighted merge); "Megatron-LM ... （六）" data flow
 *   (+ shared experts).
 *   y[t] = shared_out[t] (if not NULL) + sum over j with dest_row[t,j] >= 0 of gates[t,j] * eout[dest_row[t,j]]
 *   accumulated in fp32 in ascending j, rounded once to dtype. Dropped pairs add nothing; no residual.
 *   eout [rows,h] dtype; dest_row [T,k] int32; gates [T,k] fp32; shared_out [T,h] dtype or NULL;
 *   y [T,h] dtype. Deterministic (no atomics).
 *   Errors: MOE_ERR_UNSUPPORTED for a dtype outside the enum; MOE_ERR_INVALID_ARG for h % 8 != 0, k outside
 *   [1, 16], a null pointer, or eout / shared_out / y not 16-byte aligned.
 * ------------------------------------------------------------------------------------------------- */
int moe_combine(const void* eout, const int32_t* dest_row, const float* gates, const void* shared_out, int T,
                int h, int k, int dtype, void* y, void* stream);

/* ---------------------------------------------------------------------------------------------------
 * moe_expert_down_combine: the down GEMM with the combine in its epilogue (one launch instead of
 *   moe_expert_down[_shared] followed by moe_combine).
 *   "v6 长序列和 MoE ...", table row "combine"; "专家并行" (formulaic), section "通信与计算的重叠" (work on
 *   the outputs that are ready while the rest is still being computed); "Megatron-LM ... （六）" data flow
 *   (+ shared experts).
 *   Writes eout [rows,h] (and, when act_shared is not NULL, out_shared [T,h] of the shared expert, whose tiles run in
 *   the same launch) exactly as moe_expert_down / moe_expert_down_shared, and y [T,h] bit-identical to
 *   moe_combine(eout, dest_row, gates, out_shared or NULL): the tile that completes a token's 256-column block
 *   sums that block from the token's rows in ascending j with fp32 fused multiply-adds, rounded once to bf16.
 *   src_token [rows] int32 (moe_dispatch's; -1 for pads), dest_row / gates [T,k] as for moe_combine.
 *   arrivals [T * ceil(h/256)] int32, size from moe_combine_arrivals_bytes: per-(token, column block) arrival
 *   counters; they must be zero before the first call (e.g. one cudaMemsetAsync at allocation) and every call that
 *   completes leaves them zero again. Two calls that may run at the same time must not share them. After a call
 *   whose launch was cut short (moe_check_device_error reports MOE_ERR_TIMEOUT) zero them again.
 *   bf16 only (MOE_ERR_UNSUPPORTED otherwise); tile_sched, packed_w, rows as moe_expert_down; act_shared /
 *   packed_shared / out_shared all NULL or all set. All pointers 16-byte aligned.
 * ------------------------------------------------------------------------------------------------- */
size_t moe_combine_arrivals_bytes(int T, int h);
int moe_expert_down_combine(const void* act, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                            int rows, const int32_t* src_token, const int32_t* dest_row, const float* gates, int T,
                            int k, const void* act_shared, const void* packed_shared, int dtype, void* eout,
                            void* out_shared, void* y, int32_t* arrivals, void* stream);

/* ---------------------------------------------------------------------------------------------------
 * The whole layer forward in one call ("Megatron-LM ... （六）", section "MoE 层的数据流": router ->
 * dispatch -> experts as one GroupedGEMM -> combine, plus the shared expert; "v6 长序列和 MoE ...", the worked shape
 * table of section "NVIDIA 原题").
 *   moe_layer_forward enqueues on `stream` the calls of one layer forward, the same launches (so the same output
 *   bits) as those calls made one after the other with the intermediates in the workspace:
 *     x [T,h] dtype (device)  ->  y [T,h] dtype (device)
 *   routing MOE_ROUTING_TOKEN: moe_router_packed (gating), moe_dispatch (or moe_dispatch_fp8 + moe_dequant_fp8 with
 *     payload MOE_PAYLOAD_FP8), moe_expert_up_gate[_shared], moe_expert_down[_shared], moe_combine;
 *   MOE_ROUTING_SINKHORN: moe_router_packed (softmax mode, for the logits), moe_sinkhorn_bias (sinkhorn_iters, 0 =
 *     16), moe_router_from_logits (MOE_GATING_SOFTMAX_SELBIAS), then as token routing (`gating` unused);
 *   MOE_ROUTING_EXPERT_CHOICE: moe_router_packed (gating, for the logits), moe_expert_choice_route /
 *     _dispatch with C = capacity tokens per expert (1 <= C <= T, E <= 256), the expert FFN,
 *     moe_expert_choice_combine.
 *   The shared expert runs inside the routed GEMM launches with bf16 and the dtype payload, otherwise as a dense
 *   group of T rows after them.
 *   moe_layer_forward_host runs it on n_batches batches that live in page-locked host memory (cudaHostAlloc or
 *   cudaHostRegister), x_host[i] [T,h] -> y_host[i] [T,h]: one host->device copy of each x and one device->host
 *   copy of each y (cudaMemcpyAsync), on two streams that the call creates and releases (the first copy waits for
 *   the work already enqueued on `stream`), so that batch i's copies overlap the layer working on its neighbours on
 *   `stream` (two device buffers for x and two for y inside the workspace; a buffer is refilled only after the
 *   layer or the copy that last read it has finished). `stream`
 *   then waits for the last copy: once `stream` has been synchronised, every y_host[i] is written. Neither call
 *   waits for the host. moe_layer_forward only launches kernels on `stream` and may be captured into a CUDA graph
 *   (after one call outside the capture on the device); moe_layer_forward_host creates streams and may not.
 *   desc: the layer's sizes, dtype, gating (MOE_GATING_SOFTMAX, _SOFTMAX_RENORM or _SIGMOID_BIAS_RENORM), alpha,
 *     capacity (0: dropless) and num_ranks as for moe_router / moe_dispatch, routing, payload (FP8: bf16, token
 *     routing, h % 128 == 0), sinkhorn_iters, and its device-resident parameters:
 *     w_r_packed (moe_pack_router_weight's output), bias ([E] fp32 or NULL, as for moe_router), packed_w
 *     (moe_pack_expert_weights for the E routed experts), packed_shared (one shared expert packed with E = 1,
 *     or NULL for none). The caller owns all of it.
 *   ws: moe_layer_workspace_size(desc) bytes of device memory (moe_layer_host_workspace_size(desc) for the host
 *     variant), 16-byte aligned. moe_layer_views_of(desc, ws, &v) gives the device addresses of the intermediates
 *     inside it (the router's and the dispatch's outputs, act, eout, the shared expert's act and output), as the
 *     last forward left them.
 *   Errors: MOE_ERR_INVALID_ARG for a null desc or pointer, n_batches < 0, a host buffer that is not
 *     page-locked, or what the chained calls reject; MOE_ERR_UNSUPPORTED for MOE_GATING_SOFTMAX_SELBIAS, a dtype,
 *     routing or payload outside the enums, or the FP8 payload with fp32 or without token routing;
 *     MOE_ERR_WORKSPACE if ws_bytes is short; MOE_ERR_CUDA. The arguments are checked before anything is
 *     enqueued; a call that fails later returns the failing step's status with the steps before it already
 *     enqueued (the host variant then still makes `stream` wait for every copy it issued).
 * ------------------------------------------------------------------------------------------------- */
enum moe_routing { MOE_ROUTING_TOKEN = 0, MOE_ROUTING_EXPERT_CHOICE = 1, MOE_ROUTING_SINKHORN = 2 };
enum moe_payload { MOE_PAYLOAD_DTYPE = 0, MOE_PAYLOAD_FP8 = 1 };

typedef struct moe_layer_desc {
    int T, h, E, k, F;
    int dtype;                  /* enum moe_dtype */
    int gating;                 /* enum moe_gating */
    float alpha;                /* aux-loss coefficient */
    int capacity;               /* expert capacity C (0: dropless) */
    int num_ranks;              /* virtual EP ranks of the send layout (divides E) */
    const void* w_r_packed;     /* moe_pack_router_weight(w_r) */
    const float* bias;          /* [E] fp32 or NULL */
    const void* packed_w;       /* moe_pack_expert_weights of the routed experts */
    const void* packed_shared;  /* the shared expert (E = 1) or NULL */
    int routing;                /* enum moe_routing */
    int payload;                /* enum moe_payload: the send buffer in dtype, or e4m3 with per-128-column scales */
    int sinkhorn_iters;         /* MOE_ROUTING_SINKHORN: iterations (0: 16) */
} moe_layer_desc;

typedef struct moe_layer_views {
    float* logits;              /* [T,E] */
    int32_t* topk_ids;          /* [T,k] */
    float* gates;               /* [T,k] */
    int32_t* counts;            /* [E] */
    float* f;                   /* [E] */
    float* P;                   /* [E] */
    float* aux;                 /* [1] */
    void* buf;                  /* [rows,h] dtype */
    /* offsets .. rank_offsets: token and Sinkhorn routing (NULL for expert choice) */
    int32_t* offsets;           /* [E+1] */
    int32_t* kept_counts;       /* [E] */
    int32_t* dest_row;          /* [T,k] */
    uint8_t* drop_mask;         /* [T,k] */
    int32_t* src_token;         /* [rows] */
    int32_t* src_slot;          /* [rows] */
    int32_t* rank_counts;       /* [num_ranks] */
    int32_t* rank_offsets;      /* [num_ranks+1] */
    int32_t* tile_sched;        /* moe_tile_sched_bytes() */
    void* act;                  /* [rows,F] dtype */
    void* eout;                 /* [rows,h] dtype */
    void* act_shared;           /* [T,F] dtype, NULL without a shared expert */
    void* out_shared;           /* [T,h] dtype, NULL without a shared expert */
    long long rows;             /* rows of buf: moe_dispatch_rows(T, E, k, capacity), E * capacity for expert choice */
    int32_t* ec_tokens;         /* expert choice: [E,C] (else NULL) */
    float* ec_gates;            /* expert choice: [E,C] */
    int32_t* ec_slot;           /* expert choice: [T,E] */
    float* sel_bias;            /* Sinkhorn: [E] log column scalings (else NULL) */
    uint8_t* buf8;              /* FP8 payload: [rows,h] e4m3 codes (else NULL; buf then holds the dequantised rows) */
    float* scales;              /* FP8 payload: [rows,h/128] */
} moe_layer_views;

size_t moe_layer_workspace_size(const moe_layer_desc* desc);
size_t moe_layer_host_workspace_size(const moe_layer_desc* desc);
int moe_layer_views_of(const moe_layer_desc* desc, void* ws, moe_layer_views* views);
int moe_layer_forward(const moe_layer_desc* desc, const void* x, void* y, void* ws, size_t ws_bytes, void* stream);
int moe_layer_forward_host(const moe_layer_desc* desc, int n_batches, const void* const* x_host,
                           void* const* y_host, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------------
 * FP8 dispatch payload ("10.5 序列并行与专家并行", section 10.5.7: activations that cross nodes can travel in
 * a low-precision format such as FP8, halving the bytes with negligible effect on model quality).
 * moe_dispatch_fp8: moe_dispatch with the send buffer in e4m3 (finite-only variant: bias 7, 3 mantissa bits,
 *   largest magnitude 448). bf16 x, h % 128 == 0. For every kept row r of token t and every block b of 128
 *   columns: scales[r, b] = max |x[t, block b]| / 448 in fp32 (1 for an all-zero block) and
 *   buf8[r, col] = e4m3(x[t, col] / scales[r, b]) rounded to nearest, ties to even, saturating at +-448;
 *   pad rows: codes 0, scale 0. buf8 [rows,h] uint8, scales [rows,h/128] fp32; every other output and the
 *   workspace as moe_dispatch.
 * moe_expert_up_gate_fp8: moe_expert_up_gate reading that buffer: each code is dequantised to
 *   bf16(fp32(value) * scale) inside the GEMM (converter warps turn each staged e4m3 tile into the bf16
 *   operand tile in shared memory), so the bf16 buffer never exists in memory. act [rows,F] bf16.
 * moe_dequant_fp8: the same dequantisation as a pass of its own (the receive side of the FP8 exchange):
 *   out [rows,h] bf16 = bf16(fp32(value) * scale), bit-identical to the operand moe_expert_up_gate_fp8 builds;
 *   moe_expert_up_gate on out then gives the same act. h % 128 == 0; buf8 and out 16-byte aligned. On GB300
 *   this pass plus the bf16 GEMM is the faster of the two routes (the converter warps limit the fused one).
 * ------------------------------------------------------------------------------------------------- */
int moe_dispatch_fp8(const void* x, const int32_t* topk_ids, int T, int h, int E, int k, int capacity, int num_ranks,
                     uint8_t* buf8, float* scales, int32_t* offsets, int32_t* kept_counts, int32_t* dest_row,
                     uint8_t* drop_mask, int32_t* src_token, int32_t* src_slot, int32_t* rank_counts,
                     int32_t* rank_offsets, int32_t* tile_sched, void* ws, size_t ws_bytes, void* stream);
int moe_expert_up_gate_fp8(const uint8_t* buf8, const float* scales, const int32_t* tile_sched, const void* packed_w,
                           int E, int h, int F, int rows, void* act, void* stream);
int moe_dequant_fp8(const uint8_t* buf8, const float* scales, int rows, int h, void* out, void* stream);

/* ---------------------------------------------------------------------------------------------------
 * Backward of the layer ("专家并行" (formulaic), section "BWD（反向传播）" and the overlap notes: the
 * gradients return to the experts along the routing path; each expert computes its own weight gradients).
 * The pages give no formulas: these are the chain rule through the forward calls above with the top-k
 * selection, the counts and the capacity drops held constant. Upstream gradients: dy for y and d_aux for the
 * aux loss. Every reduction runs in a fixed order; all outputs are deterministic.
 *
 * moe_combine_backward: through moe_combine.
 *   d_eout[r] = gates[t,j] * dy[t] for every kept row r (t = src_token[r], j = src_slot[r]), 0 on pad rows;
 *   d_gates[t,j] = sum_d dy[t,d] * eout[dest_row[t,j], d] (fp32) for kept pairs, 0 for dropped ones.
 *   dy [T,h], eout [rows,h], d_eout [rows,h] dtype; src_token/src_slot [rows], dest_row [T,k] from
 *   moe_dispatch; gates [T,k] and d_gates [T,k] fp32. The shared expert's output gradient is dy itself.
 * ------------------------------------------------------------------------------------------------- */
int moe_combine_backward(const void* dy, const void* eout, const int32_t* src_token, const int32_t* src_slot,
                         const int32_t* dest_row, const float* gates, int T, int h, int k, int rows, int dtype,
                         void* d_eout, float* d_gates, void* stream);

/* moe_router_backward: d_logits [T,E] fp32 from d_gates [T,k] and the aux loss, for the forward's logits,
 *   topk_ids, gates and f (all as moe_router wrote them) and its gating mode and alpha.
 *   With c_e = d_aux * alpha * E * f_e / T:
 *     softmax / softmax_selbias: dp_e = sum_j [ids_j = e] d_g_j + c_e, d_logits = p * (dp - <dp, p>)
 *     softmax_renorm: dp_e = sum_j [ids_j = e] (d_g_j - sum_i d_g_i g_i) / S + c_e (S = sum_j p[ids_j]), same
 *     sigmoid_bias_renorm: ds_e = sum_j [ids_j = e] (d_g_j - sum_i d_g_i g_i) / S + (c_e - <c, q>) / sum(s),
 *       q = s / sum(s), S = sum_j s[ids_j]; d_logits = ds * s * (1 - s)   (the selection bias gets none).
 *   d_bias [E] fp32 (may be NULL) = sum over t of d_logits: the gradient of the bias the softmax modes add to
 *   the logits. Workspace: moe_router_backward_workspace_size(T, E) bytes when d_bias is given. */
size_t moe_router_backward_workspace_size(int T, int E);
int moe_router_backward(const float* logits, const int32_t* topk_ids, const float* gates, const float* d_gates,
                        const float* f, int T, int E, int k, int gating, float alpha, float d_aux, float* d_logits,
                        float* d_bias, void* ws, size_t ws_bytes, void* stream);

/* moe_router_weight_grad: dW_r [h,E] fp32 = x^T d_logits (x [T,h] dtype, d_logits [T,E] fp32), fp32
 *   accumulation in a fixed order. bf16 with E >= 64 (E % 8 == 0, h % 8 == 0): on the tensor cores, each fp32
 *   d_logits value split into three bf16 pieces whose sum is the value to 2^-24 relative, so the products are
 *   fp32-exact; the K range is split over token blocks and the parts added in order. Otherwise per token
 *   slice on the CUDA cores, then the slices in order. Workspace: moe_router_weight_grad_workspace_size(T, h, E)
 *   bytes (enough for either path). */
size_t moe_router_weight_grad_workspace_size(int T, int h, int E);
int moe_router_weight_grad(const void* x, const float* d_logits, int T, int h, int E, int dtype, float* dW_r,
                           void* ws, size_t ws_bytes, void* stream);

/* moe_dispatch_backward: through moe_dispatch and the router's x W_r.
 *   dx[t] = dx_extra[t] + sum over kept j of d_buf[dest_row[t,j]] + sum_e d_logits[t,e] * W_r[:, e]
 *   accumulated in fp32 in that order (j ascending), rounded once to dtype. The router term: bf16 with
 *   E >= 64 (E % 8 == 0): one tensor-core GEMM of the three bf16 pieces of d_logits (as in
 *   moe_router_weight_grad) with W_r, fp32 [T,h] in the workspace; otherwise e ascending on the CUDA cores.
 *   dx_extra [T,h] dtype (e.g. the shared expert's input gradient) and d_logits may be NULL (their terms are
 *   then absent; w_r is only read with d_logits). d_buf [rows,h], dx [T,h], w_r [h,E] dtype (16-byte aligned
 *   on the tensor-core path). Workspace (with d_logits): moe_dispatch_backward_workspace_size(T, h, E, dtype)
 *   bytes, 16-byte aligned. */
size_t moe_dispatch_backward_workspace_size(int T, int h, int E, int dtype);
int moe_dispatch_backward(const void* d_buf, const int32_t* dest_row, const float* d_logits, const void* w_r,
                          const void* dx_extra, int T, int h, int k, int E, int dtype, void* dx, void* ws,
                          size_t ws_bytes, void* stream);

/* Expert FFN backward (bf16, tcgen05 tensor cores; MOE_ERR_UNSUPPORTED for fp32). With g = buf W_gate^T,
 * u = buf W_up^T, s the logistic of g and act = silu(g) u as in moe_expert_up_gate:
 *   moe_pack_expert_weights_backward: one-time repack of the same three matrices as the dgrad GEMMs'
 *     operands (moe_packed_weights_backward_bytes() bytes, opaque).
 *   moe_expert_down_backward:    d_act [rows,F] = d_eout [rows,h] @ W_down[e]          for the kept rows
 *   moe_expert_up_gate_backward: recomputes g and u, then
 *     d_gu [rows, 2*Fp] (Fp = F rounded up to 128; columns in blocks of 256: 128 of d_g then the d_u of the same
 *       f, f >= F zero): d_g = d_act * u * s * (1 + g (1 - s)), d_u = d_act * silu(g)
 *     d_buf [rows,h] = d_g @ W_gate[e] + d_u @ W_up[e]
 *   moe_expert_weight_grads: fp32 [E,F,h] dW_gate = d_g^T buf, dW_up = d_u^T buf, [E,h,F] dW_down = d_eout^T act
 *     over each expert's kept rows [offsets[e], offsets[e] + kept_counts[e]) (zero for an expert without rows),
 *     from buf, act (the forward's), d_gu and d_eout (all pointers 16-byte aligned). Workspace:
 *     moe_expert_weight_grads_workspace_size() bytes (each expert's rows transposed into a 64-aligned column
 *     segment).
 *   Rows outside the kept ranges are not read (weight gradients) or not written (d_act, d_gu, d_buf). */
size_t moe_packed_weights_backward_bytes(int E, int h, int F, int dtype);
int moe_pack_expert_weights_backward(const void* w_gate, const void* w_up, const void* w_down, int E, int h, int F,
                                     int dtype, void* packed_bwd, void* stream);
int moe_expert_down_backward(const void* d_eout, const int32_t* tile_sched, const void* packed_bwd, int E, int h,
                             int F, int rows, int dtype, void* d_act, void* stream);
int moe_expert_up_gate_backward(const void* buf, const void* d_act, const int32_t* tile_sched, const void* packed_w,
                                const void* packed_bwd, int E, int h, int F, int rows, int dtype, void* d_gu,
                                void* d_buf, void* stream);
/* moe_expert_up_gate_backward_saved: moe_expert_up_gate_backward from the pre-activations gu that
 *   moe_expert_up_gate_save stored instead of recomputing them: d_gu by the same formulas from the bf16 g and u
 *   (an elementwise pass over the tiles' kept rows), then d_buf as there. */
int moe_expert_up_gate_backward_saved(const void* gu, const void* d_act, const int32_t* tile_sched,
                                      const void* packed_bwd, int E, int h, int F, int rows, int dtype, void* d_gu,
                                      void* d_buf, void* stream);
size_t moe_expert_weight_grads_workspace_size(int E, int h, int F, int rows, int dtype);
int moe_expert_weight_grads(const void* buf, const void* act, const void* d_gu, const void* d_eout,
                            const int32_t* offsets, const int32_t* kept_counts, int E, int h, int F, int rows,
                            int dtype, float* dW_gate, float* dW_up, float* dW_down, void* ws, size_t ws_bytes,
                            void* stream);

/* ---------------------------------------------------------------------------------------------------
 * Errors and diagnostics.
 * ------------------------------------------------------------------------------------------------- */
/* Message of the last failing call on this host thread ("" if none). */
const char* moe_last_error_string(void);
/* Synchronizes `stream`, then reads and clears the device error word of the current device. Returns
 * MOE_OK, MOE_ERR_TIMEOUT if a bounded device-side wait ran out since the last check, MOE_ERR_INVALID_ARG
 * if a kernel met an expert id outside [0, E), or MOE_ERR_CUDA. */
int moe_check_device_error(void* stream);
/* Sets the iteration limit of the bounded device-side waits (mbarrier polls) of later launches: those of the
 * tensor-core GEMMs and of moe_dispatch's row copy; spins <= 0 restores the default. A small limit makes
 * those waits give up early, which exercises the error path: the kernel latches MOE_ERR_TIMEOUT, waits
 * (bounded) for its copies and MMAs in flight, frees its tensor memory and returns. */
void moe_set_wait_limit(long long spins);
/* Number of kernels this process has launched through the library (all devices, all threads). */
unsigned long long moe_launch_count(void);
/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
