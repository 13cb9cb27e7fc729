// Internal launchers (host side).  The C ABI in api.cu validates arguments and then
// calls these; each enqueues its kernels on `st` and returns the launch status.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

struct RouteOut;

constexpr int kDispatchChunk = 32;  // tokens per warp chunk in count / scatter
// Capacity (int32 entries) of the dispatch's built-in chunk-count array.
constexpr size_t kDispatchStaticCounts = (size_t)1 << 19;

// Segments of the expert FFN row space: routed expert i owns rows
// [expert_offset[i], expert_offset[i+1]); shared expert s owns T rows starting at
// T*K_r + s*T and reads its inputs from u.
struct FfnShape {
  int T, d, I, N_r, K_r, N_s;
};

int device_sm_count();
int32_t* dev_error_ptr();                        // device address of the error word
cudaError_t read_dev_error(int32_t* code, bool clear);   // synchronises the device

int router_tc_splits(int T, int d);   // split-K factor of the tensor-core affinity GEMM
cudaError_t launch_router_gemm_tc(const void* u, const void* e, int T, int d, int N_r,
                                  float* z_part, cudaStream_t st);
cudaError_t launch_router_gemm_simt(const void* u, const void* e, moe_dtype dt, int T, int d,
                                    int N_r, float* z, cudaStream_t st);
cudaError_t launch_router_select(const float* z_part, int S, const float* b, const RouteOut& p,
                                 cudaStream_t st);
// Fused routing (affinity GEMM, sigmoid, keys, group limit, Top-K_r, gates, P sums in
// one launch) for bf16 layers: 64, 128 or 256 experts, K_r <= 8, groups of whole
// 32-expert blocks with K_r/M <= 2, d >= 128.  done_ctr: scratch of 256 bytes (the
// counter) and then the [n_seq, N_r] fixed-point P accumulators, zeroed on the stream
// before the kernel when P sums are wanted and the batch is more than one cluster.
bool router_fused_ok(int N_r, int K_r, int G, int M, int d);
cudaError_t launch_router_fused(const void* u, const void* e, int d, const float* b,
                                const RouteOut& p, float* seq_p_sum, int* done_ctr,
                                cudaStream_t st);
cudaError_t launch_seq_psum(const float* pwin, const int32_t* seq_offsets, int n_seq, int T,
                            int N_r, float* out, cudaStream_t st);

cudaError_t launch_dispatch(const int32_t* topk_idx, int T, int N_r, int K_r,
                            const void* u, size_t row_bytes, const float* u_scale,
                            int scale_cols, int32_t* load, int32_t* expert_offset,
                            int32_t* perm_token, int32_t* inv_row, void* x_perm,
                            float* x_perm_scale, int32_t* ws_counts, cudaStream_t st);

// Device address of the built-in chunk-count array (kDispatchStaticCounts entries) on
// the current device; looked up on the first call per device.
cudaError_t dispatch_static_counts(int32_t** out);

cudaError_t launch_quantize_e4m3(const void* x, moe_dtype x_dt, int64_t rows, int64_t cols,
                                 int block_rows, uint8_t* q, float* scale, cudaStream_t st);

cudaError_t launch_ffn_up_simt(const FfnShape& s, const float* x_perm, const float* u,
                               const int32_t* expert_offset, const moe_expert_weights* w,
                               float* h, cudaStream_t st);
cudaError_t launch_ffn_down_simt(const FfnShape& s, const float* h,
                                 const int32_t* expert_offset, const moe_expert_weights* w,
                                 float* y, cudaStream_t st);

// save_a / save_c (optional, bf16 [R, I]): also write the pre-activations x W_gate^T
// and x W_up^T (the backward pass reads them).
cudaError_t launch_ffn_up_tc(const FfnShape& s, const void* x_perm, const void* u,
                             const int32_t* expert_offset, const moe_expert_weights* w,
                             void* h, cudaStream_t st, void* save_a = nullptr,
                             void* save_c = nullptr);
// The same with the routed token rows read straight from u at the rows perm_token gives
// (no x_perm); bf16 only.
cudaError_t launch_ffn_up_tc_gather(const FfnShape& s, const void* u, const int32_t* perm_token,
                                    const int32_t* expert_offset, const moe_expert_weights* w, void* h,
                                    cudaStream_t st);
cudaError_t launch_ffn_down_tc(const FfnShape& s, const void* h,
                               const int32_t* expert_offset, const moe_expert_weights* w,
                               void* y, cudaStream_t st);

cudaError_t launch_ffn_up_fp8(const FfnShape& s, const void* x_perm, const float* x_perm_scale,
                              const void* u, const float* u_scale, const int32_t* expert_offset,
                              const moe_expert_weights* w, void* h, float* h_scale,
                              cudaStream_t st, void* save_a = nullptr, void* save_c = nullptr);
cudaError_t launch_ffn_down_fp8(const FfnShape& s, const void* h, const float* h_scale,
                                const int32_t* expert_offset, const moe_expert_weights* w,
                                void* y, cudaStream_t st);

// Backward pass (bwd_gemm.cu, bwd_misc.cu).  All activation arrays are in the FFN row
// space R = T*K_r + N_s*T and bf16 unless noted.
struct BwdGemmIo {
  FfnShape s;
  const int32_t* expert_offset;
  const void *w_gate, *w_up, *w_down, *ws_gate, *ws_up, *ws_down;   // bf16 weights
  const void* x_perm;   // [T*K_r, d]
  const void* u;        // [T, d]
  const void* e;        // [N_r, d]
  const __nv_bfloat16 *a, *c, *h;   // [R, I]: pre-activations and SwiGLU output
  const void* dY;       // [R, d]
  const void* dz;       // [T, N_r]
  __nv_bfloat16 *dA, *dC;           // [R, I]
  __nv_bfloat16* dX;                // [R, d]
  float *dw_gate, *dw_up, *dw_down, *dws_gate, *dws_up, *dws_down;
  float* du_router;     // [T, d]
  float* de;            // [N_r, d]
  bool experts = true;  // the expert GEMMs (dH, dX, dW_*) ...
  bool router = true;   // ... and the router's (du = dz e, de = dz^T u)
};
cudaError_t launch_bwd_gemms(const BwdGemmIo& io, cudaStream_t st);

// FP8 backward (bwd_fp8.cu).
// dst [E][C, ldd] at column col0 <- src [E][R, C]^T (E4M3 codes), and the 128x128 block
// scales dst_s [E][C/128, ldd/128] at column col0/128 <- src_s [E][R/128, C/128]^T.
cudaError_t launch_fp8_transpose(const uint8_t* src, const float* src_s, int E, int R, int C,
                                 uint8_t* dst, float* dst_s, int ldd, int col0, cudaStream_t st);
// SwiGLU backward from dH, a, c (bf16 [rows, I]): dA = dH c silu'(a), dC = dH silu(a) in
// fp32; ac_q [rows, 2I] = E4M3 1x128 tiles of (dA | dC) with scales ac_s [rows, 2I/128],
// and dA, dC rounded to bf16.
cudaError_t launch_fp8_swiglu_bwd(const void* dH, const void* a, const void* c, long long rows, int I,
                                  uint8_t* ac_q, float* ac_s, void* dA, void* dC, cudaStream_t st);
// Wgrad operand: the columns of an activation [rows, C] over each expert segment's tokens,
// E4M3 per 128x1 tile, transposed: q [C, Rp] (segment s at column pstart(s), padded to a
// multiple of 128 with zero codes) and scales [Rp/128, C].  Segment i < N_r is rows
// [off[i], off[i+1]) of `routed`; shared segment j reads rows j*shared_stride .. + T of
// `shared`.  Source values: bf16 (src_scale null) or E4M3 codes with 1x128 scales
// (src_scale [rows, C/128], shared_scale likewise).
struct ColQuantSrc {
  const void* routed;
  const void* shared;
  const float* routed_scale;
  const float* shared_scale;
  long long shared_stride;   // rows between shared segments in `shared`
};
cudaError_t launch_fp8_colquant(const ColQuantSrc& src, const int32_t* expert_offset, int T, int K_r,
                                int N_r, int N_s, int C, uint8_t* q, float* scale, long long Rp,
                                cudaStream_t st);
// Wgrad GEMM per expert segment: out_e [M, N] (fp32, row-major) = sum over the segment's
// 128-token blocks kb of diag(sa[kb, :]) (A_kb B_kb^T) diag(sb[kb, :]), with A = qa [M, Rp],
// B = qb [N, Rp] E4M3 (K = tokens), sa [Rp/128, M], sb [Rp/128, N]; routed experts to out
// [N_r][M, N], shared ones to out_s [N_s][M, N].  An expert without tokens gets zeros.
cudaError_t launch_fp8_wgrad(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                             int M, int N, long long Rp, const int32_t* expert_offset, int T, int K_r,
                             int N_r, int N_s, float* out, float* out_s, cudaStream_t st);
// Per (sequence, expert) selection counts (int32 [n_seq, N_r], zeroed here first).
cudaError_t launch_seq_counts(const int32_t* topk_idx, const int32_t* seq_offsets, int n_seq,
                              int T, int N_r, int K_r, int32_t* counts, cudaStream_t st);
// Per token: dgate = dh . y rows, the gate and balance-loss backward to dz (bf16
// [T, N_r]), and the expert-output gradients dY rows (bf16 [R, d]).
cudaError_t launch_bwd_prep(const float* dh, const void* y, const float* s, const int32_t* topk_idx,
                            const float* topk_gate, const int32_t* inv_row, const int32_t* counts,
                            const int32_t* seq_offsets, int n_seq, float alpha, int T, int d,
                            int N_r, int K_r, int N_s, void* dz, void* dY, cudaStream_t st);
// du = dh + du_router + sum of the token's dX rows (routed slots and shared experts).
cudaError_t launch_bwd_combine(const float* dh, const float* du_router, const void* dX,
                               const int32_t* inv_row, int T, int d, int K_r, int N_s, float* du,
                               cudaStream_t st);

cudaError_t launch_combine(const void* u, const void* y, moe_dtype dt, const float* gate,
                           const int32_t* inv_row, int T, int d, int K_r, int N_s,
                           void* out, moe_dtype out_dt, cudaStream_t st);

cudaError_t launch_bias_update(float* b, const int32_t* load, int T, int N_r, int K_r,
                               float gamma, cudaStream_t st);
cudaError_t launch_seq_stat(const float* seq_p_sum, const int32_t* topk_idx,
                            const int32_t* seq_offsets, int n_seq, int T, int N_r, int K_r,
                            float alpha, float* stat_per_seq, float* stat_mean,
                            cudaStream_t st);

}  // namespace moe
