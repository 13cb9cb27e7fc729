/*
 * moe.h — C ABI of the B300 (sm_103a) forward pass of a DeepSeekMoE layer with
 * auxiliary-loss-free load balancing.
 *
 * Sources (web pages about the DeepSeek-V3 technical report, cited by site, title
 * and section):
 *   [P1] szhzxw.cn, DeepSeek-V3 解读: "无辅助损失负载平衡的DeepSeekMoE",
 *        "互补序列级辅助损失", "节点限制路由", "无Token丢弃".
 *   [P3] pwwt.cn, "DeepSeek-V3 Technical Report" 笔记: §一, §1.1.2, §1.1.3, §1.2,
 *        §1.3, §1.4, §三 (FP8), §四 (dispatch / combine).
 *   [P4] xyznot.com, "DeepSeek-V3 Technical Report" reading guide: Method §2
 *        (equations for h'_t, s_{i,t}, g'_{i,t}; gamma = 0.001, alpha = 0.0001) and
 *        Key ideas (1 shared + 256 routed experts, 8 active; E4M3 with 1x128 /
 *        128x128 scaling).
 *
 * Conventions shared by every call
 *   - All tensor arguments are DEVICE pointers owned by the caller, row-major, and
 *     16-byte aligned.  The library allocates no device memory and keeps no state
 *     between calls, except device arrays built into it: one error word (see
 *     moe_device_error), the bf16 expert GEMMs' tile counters (see
 *     moe_expert_gate_up) and the scratch of moe_dispatch_noalloc.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call only
 *     enqueues work on it and returns; no call synchronises with the device.
 *   - Arguments are validated before anything is launched: on an invalid argument a
 *     call returns MOE_ERR_INVALID_ARG (or MOE_ERR_UNSUPPORTED for a dtype/shape
 *     combination with no kernel, MOE_ERR_WORKSPACE for a missing or short
 *     workspace) and enqueues nothing.  MOE_ERR_CUDA reports a failed launch.
 *   - Values of device-resident inputs are checked by the kernels that read them:
 *     an expert index outside [0, N_r), an inv_row outside [0, T*K_r), an
 *     expert_offset segment outside [0, T*K_r), or seq_offsets that are not
 *     0 = off[0] <= ... <= off[n_seq] = T are skipped (the entry adds nothing; an
 *     out-of-order sequence counts as empty), no memory outside the buffers is
 *     touched, and MOE_ERR_INVALID_ARG is recorded in the device error word (see
 *     moe_device_error).  The results of such a call are meaningless.  NaN/Inf
 *     inputs are undefined behaviour.
 *   - The library caches, per device, the addresses of its built-in device arrays
 *     (tile counters, dispatch scratch).  A device reset (cudaDeviceReset) frees
 *     them: do not call the library on a device that has been reset in the same
 *     process.
 *   - Token-level notation follows [P4] Method §2: u_t the layer input of token t,
 *     e_i the centroid of routed expert i, b_i its routing bias, N_r routed and
 *     N_s shared experts, K_r experts active per token, I the SwiGLU width.
 */
#ifndef MOE_ALF_H
#define MOE_ALF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_UNSUPPORTED = 2,
    MOE_ERR_WORKSPACE = 3,
    MOE_ERR_CUDA = 4,
    MOE_ERR_TIMEOUT = 5
} moe_status;

typedef enum {
    MOE_F32 = 0,   /* IEEE fp32 */
    MOE_BF16 = 1,  /* bfloat16, fp32 accumulation */
    MOE_E4M3 = 2   /* FP8 E4M3 codes (uint8) with fp32 block scales */
} moe_dtype;

/* Layer shape.  G = M = 1 disables the group limit.  Requirements checked by every
 * call that takes a shape: 1 <= K_r <= N_r <= 256, K_r <= 32, N_r % G == 0,
 * 1 <= M <= G <= 32, K_r % M == 0, M*(N_r/G) >= K_r, T >= 0, d and I multiples of
 * 8 (of 128 for E4M3), N_s >= 0. */
typedef struct {
    int32_t T, d, N_r, K_r, N_s, I, G, M;
} moe_shape;

/* Expert weights, all K-major.  Routed: gate and up [N_r, I, d], down [N_r, d, I];
 * shared (s_*): the same with N_s.  For E4M3 the *_scale arrays hold one fp32 scale
 * per 128x128 block: gate/up [E, I/128, d/128], down [E, d/128, I/128]; they are
 * ignored otherwise. */
typedef struct {
    moe_dtype dtype;
    const void* gate;
    const void* up;
    const void* down;
    const float* gate_scale;
    const float* up_scale;
    const float* down_scale;
    const void* s_gate;
    const void* s_up;
    const void* s_down;
    const float* s_gate_scale;
    const float* s_up_scale;
    const float* s_down_scale;
} moe_expert_weights;

MOE_API const char* moe_status_string(moe_status s);
MOE_API int moe_abi_version(void);

/* --------------------------------------------------------------------------------
 * Routing: affinities, biased Top-K_r with optional group limit, gates.
 * [P4] Method §2 (s_{i,t} = Sigmoid(u_t^T e_i); g'_{i,t} = s_{i,t} if s_{i,t}+b_i is
 * in TopK({s_{j,t}+b_j}, K_r), else 0; g normalises g'); [P3] §1.1.2 (bias only
 * decides selection), §1.3 (at most M groups, ranked by the sum of their K_r/M
 * largest scores); [P1] (bias used for routing only).
 *
 *   u [T, d], e [N_r, d]: both dtype `dt` (MOE_F32 or MOE_BF16).
 *   b [N_r] fp32: routing bias, read only.
 *   seq_offsets [n_seq+1] int32 (device), 0 = off[0] <= off[1] <= ... <= off[n_seq]
 *     = T (checked on the device, see above); may be NULL with n_seq == 0 when no
 *     sequence statistic is wanted.
 *   topk_idx [T, K_r] int32 out: selected experts in descending s+b order, ties to
 *     the lower index.  topk_gate [T, K_r] fp32 out: s_{i,t} / sum over the
 *     selected s (raw s, never s+b).
 *   s_out [T, N_r] fp32 out or NULL: the affinities in fp32.
 *   seq_p_sum [n_seq, N_r] fp32 out or NULL: sum over tokens t of sequence j of
 *     s_{i,t} / sum_k s_{k,t} (input of moe_seq_balance_stat).
 *   workspace: moe_route_workspace(sh, n_seq) bytes, queried with the device that
 *     will run the call current (the affinity GEMM splits the d dimension according
 *     to the device's SM count; the partial products live there).  Pass n_seq = 0 to
 *     the query when seq_p_sum will be NULL.
 * The keys s+b are formed as one fp32 addition; a group's score is the fp32 sum of
 * its K_r/M largest keys in descending order. */
MOE_API size_t moe_route_workspace(moe_shape sh, int32_t n_seq);
MOE_API moe_status moe_route(const void* u, const void* e, moe_dtype dt, const float* b,
                     moe_shape sh, const int32_t* seq_offsets, int32_t n_seq,
                     int32_t* topk_idx, float* topk_gate, float* s_out,
                     float* seq_p_sum, void* workspace, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------------
 * Dispatch: whole-batch expert load, per-expert token lists, gathered rows.
 * [P3] §1.4 and [P1] "无Token丢弃" (no token is dropped: segments hold 0..T tokens);
 * [P1] and [P3] §1.1.3 (the load of the whole batch is monitored every step);
 * [P3] §四 (dispatch sends tokens to their experts; here the local analogue).
 *
 *   topk_idx [T, K_r] int32 from moe_route.
 *   load [N_r] int32 out: tokens routed to each expert.
 *   expert_offset [N_r+1] int32 out: exclusive prefix sum of load.
 *   perm_token [T*K_r] int32 out: expert by expert, the tokens routed there in
 *     ascending token order.  inv_row [T, K_r] int32 out: the row of (t, k) in it.
 *   u, x_perm: when both are non-NULL the rows u[perm_token[r]] are gathered into
 *     x_perm [T*K_r, d] (dtype `u_dt`; for MOE_E4M3 u holds codes and u_scale /
 *     x_perm_scale [*, d/128] fp32 scales are gathered alongside).
 *   workspace: moe_dispatch_workspace(sh) bytes.
 * Deterministic: identical inputs give bit-identical outputs. */
MOE_API size_t moe_dispatch_workspace(moe_shape sh);
MOE_API moe_status moe_dispatch(const int32_t* topk_idx, moe_shape sh, const void* u,
                        moe_dtype u_dt, const float* u_scale, int32_t* load,
                        int32_t* expert_offset, int32_t* perm_token, int32_t* inv_row,
                        void* x_perm, float* x_perm_scale, void* workspace,
                        size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------------
 * Dispatch without any allocation.  The pages have no counterpart: this exists for
 * callers that cannot call cudaMalloc or hand out device scratch, such as code running
 * under an allocator that owns all device memory, or a host runtime whose buffers are
 * fixed up front.  It computes exactly what moe_dispatch computes, with the same
 * arguments minus the workspace.
 *
 *   Scratch: the per-chunk expert counts live in one device array built into the
 *   library, 2 MiB per GPU (524288 int32), held by every GPU that loads the library
 *   until the process exits.  ceil(T/32) * N_r must fit in it (T <= 65536 tokens with
 *   N_r = 256); a larger batch returns MOE_ERR_INVALID_ARG and launches nothing.
 *   Allocation: none; no cudaMalloc, cudaFree or allocating library routine.
 *   First call per device: looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current and caches it; make that first call before any stream
 *     capture.
 *   Sharing: every call on a device uses the same array, which keeps the last call's
 *     contents.  Each entry a call reads is written earlier in the same call, so
 *     nothing has to be cleared, but calls that overlap on the GPU (different streams
 *     without ordering between them) race on it: serialise them.
 * Returns what moe_dispatch returns; MOE_ERR_CUDA if the address lookup fails. */
MOE_API moe_status moe_dispatch_noalloc(const int32_t* topk_idx, moe_shape sh, const void* u,
                                moe_dtype u_dt, const float* u_scale, int32_t* load,
                                int32_t* expert_offset, int32_t* perm_token,
                                int32_t* inv_row, void* x_perm, float* x_perm_scale,
                                void* stream);

/* --------------------------------------------------------------------------------
 * FP8 E4M3 quantisation with fp32 block scales ([P4] Key ideas: E4M3 on all
 * tensors, activations per 1x128 tile, weights per 128x128 block; [P3] §三).
 * x [rows, cols] (dtype x_dt: MOE_F32 or MOE_BF16) -> q [rows, cols] E4M3 codes and
 * scale [rows/block_rows, cols/128] fp32, block_rows 1 (activations) or 128
 * (weights; stack experts along rows).  scale = amax/448 (fp32), 1 for an all-zero
 * block; code = E4M3(x / scale) rounded to nearest-even, saturating at 448. */
MOE_API moe_status moe_quantize_e4m3(const void* x, moe_dtype x_dt, int64_t rows, int64_t cols,
                             int32_t block_rows, uint8_t* q, float* scale, void* stream);

/* --------------------------------------------------------------------------------
 * Expert FFNs, routed and shared: FFN(x) = W_down (silu(W_gate x) * (W_up x)).
 * [P4] Method §2, equation for h'_t (the experts' FFN terms); SwiGLU without biases
 * is the reading taken for the pages' unnamed FFN.
 *
 * Row space R = T*K_r + N_s*T: rows [0, T*K_r) are the routed rows in dispatch
 * order (expert i owns [expert_offset[i], expert_offset[i+1])), rows
 * T*K_r + s*T + t hold shared expert s applied to token t.
 *
 * moe_expert_gate_up: h [R, I] = silu(x W_gate^T) * (x W_up^T), x = x_perm rows for
 *   routed experts and u for shared ones.  bf16: h is bf16.  f32: h is fp32.
 *   E4M3: x_perm/u are codes with 1x128 scales, h is written as E4M3 codes with
 *   1x128 scales h_scale [R, I/128].
 * moe_expert_down: y [R, d] = h W_down^T (y bf16 for bf16/E4M3, fp32 for f32).
 * moe_expert_ffn: both, with h in the workspace (moe_expert_ffn_workspace bytes).
 * expert_offset [N_r+1] comes from moe_dispatch.
 * The bf16 GEMMs hand out their tiles from one of 64 device counters built into the
 * library, taken round-robin per call; the last CTA of a call puts its counter back to
 * zero, so at most 64 bf16 gate/up or down calls may be in flight on a device at once. */
MOE_API size_t moe_expert_ffn_workspace(moe_shape sh, moe_dtype w_dt);
MOE_API moe_status moe_expert_gate_up(const void* x_perm, const float* x_perm_scale,
                              const void* u, const float* u_scale,
                              const int32_t* expert_offset, moe_shape sh,
                              const moe_expert_weights* w, void* h, float* h_scale,
                              void* stream);
/* moe_expert_gate_up_gather: the bf16 moe_expert_gate_up, with the routed rows' tokens
 * read straight from u: row r < T*K_r of the row space is u[perm_token[r]] (perm_token
 * [T*K_r] from moe_dispatch), so the dispatch need not write x_perm (call it with u and
 * x_perm null).  h is bit-identical to moe_expert_gate_up's on x_perm = u[perm_token].
 * A perm_token entry outside [0, T) is read as a zero row and reported through
 * moe_device_error() (MOE_ERR_INVALID_ARG).  bf16 weights only; u 16-byte aligned.
 * It saves the x_perm buffer and the dispatch's row copy but not time: the GEMM ran
 * about 2.5 times longer than moe_expert_gate_up on x_perm (DeepSeek-V3 and 64-expert
 * shapes). */
MOE_API moe_status moe_expert_gate_up_gather(const void* u, const int32_t* perm_token,
                              const int32_t* expert_offset, moe_shape sh,
                              const moe_expert_weights* w, void* h, void* stream);
MOE_API moe_status moe_expert_down(const void* h, const float* h_scale,
                           const int32_t* expert_offset, moe_shape sh,
                           const moe_expert_weights* w, void* y, void* stream);
MOE_API moe_status moe_expert_ffn(const void* x_perm, const float* x_perm_scale, const void* u,
                          const float* u_scale, const int32_t* expert_offset,
                          moe_shape sh, const moe_expert_weights* w, void* y,
                          void* workspace, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------------
 * Combine: h'_t = u_t + sum_s y[T*K_r + s*T + t] + sum_k g_{t,k} y[inv_row[t,k]].
 * [P4] Method §2, equation for h'_t; [P3] §四 (combine: gate-weighted sum of the
 * experts' outputs back at the token).  fp32 accumulation in the fixed order u,
 * shared experts ascending, routed slots k ascending.
 *   u [T, d] and y [R, d] in dtype `dt` (MOE_F32 or MOE_BF16); topk_gate and
 *   inv_row [T, K_r] from moe_route / moe_dispatch; h_out [T, d] in out_dt. */
MOE_API moe_status moe_combine(const void* u, const void* y, moe_dtype dt, const float* topk_gate,
                       const int32_t* inv_row, moe_shape sh, void* h_out,
                       moe_dtype out_dt, void* stream);

/* --------------------------------------------------------------------------------
 * End-of-step bias update ([P3] §1.1.3; [P1] "在每个步骤的末尾"; gamma in [P4]
 * Method §2): b_i += gamma * sign(T*K_r - N_r*load_i), i.e. -gamma above the mean
 * load T*K_r/N_r, +gamma below it, unchanged at it (exact integer comparison, then
 * one fp32 addition).  b [N_r] is updated in place; load [N_r] from moe_dispatch
 * (the whole batch's load; with token-parallel replicas, sum it across them first). */
MOE_API moe_status moe_bias_update(float* b, const int32_t* load, moe_shape sh, float gamma,
                           void* stream);

/* --------------------------------------------------------------------------------
 * Complementary sequence-wise balance statistic ([P3] §1.2; alpha in [P4] Method §2):
 * stat_j = alpha * sum_i f_i P_i for each sequence j of length T_j, with
 * f_i = N_r/(K_r*T_j) * #{t in j : i in topk_idx[t]} and P_i = seq_p_sum[j,i] / T_j.
 * stat_per_seq [n_seq] fp32 out; stat_mean [1] fp32 out (mean over sequences).
 * Deterministic fixed-order reduction (fp64 inside). */
MOE_API moe_status moe_seq_balance_stat(const float* seq_p_sum, const int32_t* topk_idx,
                                const int32_t* seq_offsets, int32_t n_seq, moe_shape sh,
                                float alpha, float* stat_per_seq, float* stat_mean,
                                void* stream);

/* --------------------------------------------------------------------------------
 * Backward pass of the layer at the forward pass's selection (bf16 layers).  The pages
 * define the forward pass ([P4] Method §2: h'_t = u_t + sum_s FFN_s(u_t) +
 * sum_k g_{k,t} FFN_{idx_k}(u_t), s_{i,t} = Sigmoid(u_t^T e_i), gates from the raw s of
 * the selected experts); this call returns the gradients of
 *     J = sum(dh * h') + mean over sequences of alpha * sum_i f_i P_i
 * with respect to u, the centroids e and every expert weight, holding the selection
 * fixed: Top-K_r and the group limit are piecewise constant, the bias b enters only the
 * selection and gets no gradient ([P3] §1.1.3: it is moved by the sign rule), f_i counts
 * selections and passes none; the gates pass theirs through the raw s ([P3] §1.1.2).
 *
 *   Forward state (from one moe_route / moe_dispatch / moe_expert_ffn step on the same
 *   u): u [T, d] and e [N_r, d] bf16, s [T, N_r] fp32 (moe_route's s_out), topk_idx,
 *   topk_gate, expert_offset, inv_row, x_perm [T*K_r, d] bf16, y [R, d] bf16 (the expert
 *   outputs, R = T*K_r + N_s*T).  w: bf16 weights.  seq_offsets / n_seq / alpha: the
 *   balance-loss term (n_seq = 0 or alpha = 0 leaves it out).
 *   dh [T, d] fp32: dJ/dh'.
 *   Outputs, fp32: du [T, d], de [N_r, d], dw_gate / dw_up [N_r, I, d], dw_down
 *   [N_r, d, I], and the shared experts' dws_* [N_s, ...] (may be NULL when N_s = 0).
 *   workspace: moe_backward_workspace(sh, n_seq) bytes.  The SwiGLU pre-activations are
 *   recomputed (one gate/up GEMM) rather than kept from the forward pass.
 * Requirements beyond the shape checks: N_r % 64 == 0, weights MOE_BF16. */
MOE_API size_t moe_backward_workspace(moe_shape sh, int32_t n_seq);
MOE_API moe_status moe_backward(const void* u, const void* e, const float* s,
                                const int32_t* topk_idx, const float* topk_gate,
                                const int32_t* expert_offset, const int32_t* inv_row,
                                const void* x_perm, const void* y, const moe_expert_weights* w,
                                moe_shape sh, const int32_t* seq_offsets, int32_t n_seq,
                                float alpha, const float* dh, float* du, float* de,
                                float* dw_gate, float* dw_up, float* dw_down, float* dws_gate,
                                float* dws_up, float* dws_down, void* workspace,
                                size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------------
 * FP8 backward pass: the same gradients for a layer whose expert GEMMs run in E4M3.
 * pwwt.cn notes §三: the three GEMMs of a linear layer - Fprop, Dgrad (activation
 * gradient) and Wgrad (weight gradient) - take E4M3 inputs with fp32 outputs, and
 * Wgrad reads activations kept in E4M3 from the forward pass; the reading guide's FP8
 * bullet (Key ideas): activations scaled per 1x128 tile, weights per 128x128 block,
 * promotion to fp32 every 128 elements of the contraction.  Here an activation tile
 * lies along the contraction of the GEMM that reads it: 1x128 in Fprop and Dgrad,
 * 128x1 (one feature over 128 tokens of an expert's segment, the last tile short) in
 * Wgrad; dY = g*dh, dA and dC are quantised from their own values for each; Wgrad's
 * activations are the forward's E4M3 tokens and E4M3 h (the latter recomputed by the
 * forward's FP8 gate/up kernel), re-tiled 128x1.  Routing, gates, the balance loss and
 * the affinity gradients du = dz e, de = dz^T u stay bf16 / fp32, as in the FP8 forward.
 *
 * moe_fp8_dgrad_weights_make: the transposed E4M3 weights Dgrad multiplies by (once per
 * weight update): for the routed experts (E = N_r) and the shared ones (E = N_s, s_*),
 *   wdt  [E, I, d]  = W_down^T                    scales [E, I/128, d/128]
 *   wgut [E, d, 2I] = [W_gate^T | W_up^T]         scales [E, d/128, 2I/128]
 * taken from w (MOE_E4M3, d and I multiples of 128); the codes and scales are those of
 * w, moved (a 128x128 block of W is one of W^T).
 *
 * moe_backward_fp8: inputs as moe_backward, plus the forward's E4M3 state: u_q / u_scale
 * (moe_quantize_e4m3 of u, 1x128), x_perm_q / x_perm_scale (the dispatched codes and
 * scales); y: the FP8 forward's expert outputs (bf16); w: the E4M3 weights; wt: from
 * moe_fp8_dgrad_weights_make.  u (bf16) feeds the router gradients.  Outputs as
 * moe_backward.  workspace: moe_backward_fp8_workspace(sh, n_seq) bytes.
 * Requirements beyond the shape checks: N_r % 64 == 0, d % 128 == 0, I % 128 == 0. */
typedef struct {
    void* wdt;
    float* wdt_scale;
    void* wgut;
    float* wgut_scale;
    void* s_wdt;
    float* s_wdt_scale;
    void* s_wgut;
    float* s_wgut_scale;
} moe_fp8_dgrad_weights;
MOE_API moe_status moe_fp8_dgrad_weights_make(const moe_expert_weights* w, moe_shape sh,
                                              const moe_fp8_dgrad_weights* wt, void* stream);
MOE_API size_t moe_backward_fp8_workspace(moe_shape sh, int32_t n_seq);
MOE_API moe_status moe_backward_fp8(const void* u, const void* u_q, const float* u_scale,
                                    const void* e, const float* s, const int32_t* topk_idx,
                                    const float* topk_gate, const int32_t* expert_offset,
                                    const int32_t* inv_row, const void* x_perm_q,
                                    const float* x_perm_scale, const void* y,
                                    const moe_expert_weights* w, const moe_fp8_dgrad_weights* wt,
                                    moe_shape sh, const int32_t* seq_offsets, int32_t n_seq,
                                    float alpha, const float* dh, float* du, float* de,
                                    float* dw_gate, float* dw_up, float* dw_down, float* dws_gate,
                                    float* dws_up, float* dws_down, void* workspace,
                                    size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------------
 * Device error word.  Kernels that wait on asynchronous copies bound every wait;
 * a wait that runs out records MOE_ERR_TIMEOUT here and the kernel returns early.
 * Kernels that find an invalid device-resident value record MOE_ERR_INVALID_ARG.
 * The word keeps the largest code recorded.  This call synchronises the current
 * device, copies the word to *code (MOE_OK if nothing was recorded) and, if `clear`
 * is non-zero, resets it. */
MOE_API moe_status moe_device_error(int32_t* code, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ALF_H */
