// Internal launchers (host side).  The C ABI in api.cu validates arguments and then
// calls these; each enqueues its kernels on `st` and returns the launch status.
#pragma once

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
// 32-expert blocks with K_r/M <= 2, d >= 128.  done_ctr: one int of scratch (zeroed on
// the stream before the kernel when P sums are wanted).
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

cudaError_t launch_ffn_up_tc(const FfnShape& s, const void* x_perm, const void* u,
                             const int32_t* expert_offset, const moe_expert_weights* w,
                             void* h, cudaStream_t st);
cudaError_t launch_ffn_down_tc(const FfnShape& s, const void* h,
                               const int32_t* expert_offset, const moe_expert_weights* w,
                               void* y, cudaStream_t st);

cudaError_t launch_ffn_up_fp8(const FfnShape& s, const void* x_perm, const float* x_perm_scale,
                              const void* u, const float* u_scale, const int32_t* expert_offset,
                              const moe_expert_weights* w, void* h, float* h_scale,
                              cudaStream_t st);
cudaError_t launch_ffn_down_fp8(const FfnShape& s, const void* h, const float* h_scale,
                                const int32_t* expert_offset, const moe_expert_weights* w,
                                void* y, cudaStream_t st);

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
