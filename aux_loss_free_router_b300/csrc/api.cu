// The C ABI: argument validation, workspace layout and kernel selection.  Nothing is
// launched unless every check passes; no call synchronises or allocates.
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "launch.h"
#include "ffn_sched.cuh"
#include "route_select.cuh"

using namespace moe;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
inline bool ok_opt(const void* p) { return p == nullptr || aligned16(p); }
inline cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status check_shape(const moe_shape& s) {
  if (s.T < 0 || s.d <= 0 || s.I <= 0 || s.N_s < 0 || s.N_s > kMaxShared) return MOE_ERR_INVALID_ARG;
  if (s.N_r < 1 || s.N_r > kMaxExperts || s.K_r < 1 || s.K_r > s.N_r || s.K_r > 32)
    return MOE_ERR_INVALID_ARG;
  if (s.G < 1 || s.G > 32 || s.M < 1 || s.M > s.G || s.N_r % s.G != 0 || s.K_r % s.M != 0)
    return MOE_ERR_INVALID_ARG;
  if ((long long)s.M * (s.N_r / s.G) < s.K_r) return MOE_ERR_INVALID_ARG;
  if (s.d % 8 != 0 || s.I % 8 != 0) return MOE_ERR_INVALID_ARG;
  if ((long long)s.T * s.K_r + (long long)s.N_s * s.T >= (1LL << 31)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

bool is_float_dtype(moe_dtype dt) { return dt == MOE_F32 || dt == MOE_BF16; }
size_t elem_bytes(moe_dtype dt) { return dt == MOE_F32 ? 4 : dt == MOE_BF16 ? 2 : 1; }

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported dtype or shape";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA launch error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int moe_abi_version(void) { return MOE_ABI_VERSION; }

// ------------------------------------------------------------------------ route ----

namespace {

bool router_uses_tc(const moe_shape& sh, moe_dtype dt) { return dt == MOE_BF16 && sh.N_r % 32 == 0; }

struct RouteWs {
  size_t z_bytes, pwin_bytes;
  size_t total() const { return z_bytes + pwin_bytes; }
};

RouteWs route_ws(const moe_shape& sh, int n_seq, int S) {
  RouteWs w{0, 0};
  if (sh.T <= 0) return w;
  w.z_bytes = align256((size_t)S * sh.T * sh.N_r * sizeof(float));
  if (n_seq > 0) w.pwin_bytes = align256((size_t)sh.T * sh.N_r * sizeof(float));
  return w;
}

}  // namespace

size_t moe_route_workspace(moe_shape sh, int32_t n_seq) {
  if (sh.T <= 0 || sh.N_r <= 0 || sh.d <= 0) return 0;
  // sized for the split path's partial products (the CUDA-core path uses one split);
  // the fused path needs a counter and the P-sum rows, which is less
  const size_t split = route_ws(sh, n_seq, router_tc_splits(sh.T, sh.d)).total();
  const size_t fused = 256 + (n_seq > 0 ? align256((size_t)n_seq * sh.N_r * 8) : 0);
  return split > fused ? split : fused;
}

moe_status moe_route(const void* u, const void* e, moe_dtype dt, const float* b, moe_shape sh,
                     const int32_t* seq_offsets, int32_t n_seq, int32_t* topk_idx,
                     float* topk_gate, float* s_out, float* seq_p_sum, void* workspace,
                     size_t ws_bytes, void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if (!is_float_dtype(dt)) return MOE_ERR_UNSUPPORTED;
  if (sh.T > 0 && (!ok_ptr(u) || !ok_ptr(e) || !ok_ptr(b) || !ok_ptr(topk_idx) || !ok_ptr(topk_gate)))
    return MOE_ERR_INVALID_ARG;
  if (!ok_opt(s_out) || !ok_opt(seq_p_sum) || n_seq < 0) return MOE_ERR_INVALID_ARG;
  const bool want_stat = seq_p_sum != nullptr;
  if (want_stat && (n_seq < 1 || seq_offsets == nullptr)) return MOE_ERR_INVALID_ARG;
  if (sh.T == 0) {
    if (!want_stat) return MOE_OK;
    return cuda_status(cudaMemsetAsync(seq_p_sum, 0, sizeof(float) * n_seq * sh.N_r, S(stream)));
  }
  if (dt == MOE_BF16 && router_fused_ok(sh.N_r, sh.K_r, sh.G, sh.M, sh.d)) {
    // one launch: a counter (256 bytes), then the fixed-point P sums [n_seq, N_r] (8 bytes each)
    const size_t need = 256 + (want_stat ? align256((size_t)n_seq * sh.N_r * 8) : 0);
    if (workspace == nullptr || !aligned16(workspace) || ws_bytes < need) return MOE_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    RouteOut p{sh.T, sh.N_r, sh.K_r, sh.G, sh.M, topk_idx, topk_gate, s_out,
               want_stat ? reinterpret_cast<float*>(ws + 256) : nullptr, seq_offsets,
               want_stat ? n_seq : 0};
    return cuda_status(launch_router_fused(u, e, sh.d, b, p, seq_p_sum,
                                           reinterpret_cast<int*>(ws), S(stream)));
  }
  const bool tc = router_uses_tc(sh, dt);
  const int splits = tc ? router_tc_splits(sh.T, sh.d) : 1;
  const RouteWs w = route_ws(sh, want_stat ? n_seq : 0, splits);
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < w.total()) return MOE_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  float* z_part = reinterpret_cast<float*>(ws);
  float* pwin = want_stat ? reinterpret_cast<float*>(ws + w.z_bytes) : nullptr;
  RouteOut p{sh.T, sh.N_r, sh.K_r, sh.G, sh.M, topk_idx, topk_gate, s_out, pwin,
             seq_offsets, want_stat ? n_seq : 0};
  cudaError_t err = tc ? launch_router_gemm_tc(u, e, sh.T, sh.d, sh.N_r, z_part, S(stream))
                       : launch_router_gemm_simt(u, e, dt, sh.T, sh.d, sh.N_r, z_part, S(stream));
  if (err == cudaSuccess) err = launch_router_select(z_part, splits, b, p, S(stream));
  if (err == cudaSuccess && want_stat)
    err = launch_seq_psum(pwin, seq_offsets, n_seq, sh.T, sh.N_r, seq_p_sum, S(stream));
  return cuda_status(err);
}

// --------------------------------------------------------------------- dispatch ----

size_t moe_dispatch_workspace(moe_shape sh) {
  if (sh.T <= 0 || sh.N_r <= 0) return 0;
  const size_t chunks = ((size_t)sh.T + kDispatchChunk - 1) / kDispatchChunk;
  return align256(chunks * sh.N_r * sizeof(int32_t));
}

moe_status moe_dispatch(const int32_t* topk_idx, moe_shape sh, const void* u, moe_dtype u_dt,
                        const float* u_scale, int32_t* load, int32_t* expert_offset,
                        int32_t* perm_token, int32_t* inv_row, void* x_perm,
                        float* x_perm_scale, void* workspace, size_t ws_bytes, void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if (!ok_ptr(load) || !ok_ptr(expert_offset)) return MOE_ERR_INVALID_ARG;
  if (sh.T > 0 && (!ok_ptr(topk_idx) || !ok_ptr(perm_token) || !ok_ptr(inv_row)))
    return MOE_ERR_INVALID_ARG;
  const bool gather = u != nullptr && x_perm != nullptr;
  if ((u == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (gather && (!aligned16(u) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  size_t row_bytes = 0;
  int scale_cols = 0;
  if (gather) {
    if (u_dt != MOE_F32 && u_dt != MOE_BF16 && u_dt != MOE_E4M3) return MOE_ERR_UNSUPPORTED;
    row_bytes = (size_t)sh.d * elem_bytes(u_dt);
    if (row_bytes % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (u_dt == MOE_E4M3) {
      if (sh.d % 128 != 0 || !ok_ptr(u_scale) || !ok_ptr(x_perm_scale)) return MOE_ERR_INVALID_ARG;
      scale_cols = sh.d / 128;
    }
  }
  const size_t need = moe_dispatch_workspace(sh);
  if (need > 0 && (workspace == nullptr || !aligned16(workspace) || ws_bytes < need))
    return MOE_ERR_WORKSPACE;
  const cudaError_t err = launch_dispatch(
      topk_idx, sh.T, sh.N_r, sh.K_r, gather ? u : nullptr, row_bytes,
      u_dt == MOE_E4M3 ? u_scale : nullptr, scale_cols, load, expert_offset, perm_token, inv_row,
      gather ? x_perm : nullptr, u_dt == MOE_E4M3 ? x_perm_scale : nullptr,
      static_cast<int32_t*>(workspace), S(stream));
  return cuda_status(err);
}

// For callers that cannot allocate device memory: the same dispatch, with the chunk
// counts kept in the library's built-in device array instead of a workspace.
moe_status moe_dispatch_noalloc(const int32_t* topk_idx, moe_shape sh, const void* u,
                                moe_dtype u_dt, const float* u_scale, int32_t* load,
                                int32_t* expert_offset, int32_t* perm_token, int32_t* inv_row,
                                void* x_perm, float* x_perm_scale, void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  const size_t cap = kDispatchStaticCounts * sizeof(int32_t);
  if (moe_dispatch_workspace(sh) > cap) return MOE_ERR_INVALID_ARG;   // beyond the built-in size
  int32_t* counts = nullptr;
  if (dispatch_static_counts(&counts) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_dispatch(topk_idx, sh, u, u_dt, u_scale, load, expert_offset, perm_token, inv_row,
                      x_perm, x_perm_scale, counts, cap, stream);
}

// ------------------------------------------------------------------------- quant ----

moe_status moe_quantize_e4m3(const void* x, moe_dtype x_dt, int64_t rows, int64_t cols,
                             int32_t block_rows, uint8_t* q, float* scale, void* stream) {
  if (!is_float_dtype(x_dt)) return MOE_ERR_UNSUPPORTED;
  if (rows < 0 || cols <= 0 || cols % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (block_rows != 1 && block_rows != 128) return MOE_ERR_INVALID_ARG;
  if (block_rows == 128 && rows % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!ok_ptr(x) || !ok_ptr(q) || !ok_ptr(scale))) return MOE_ERR_INVALID_ARG;
  if (block_rows == 128 && rows / 128 > 65535) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_e4m3(x, x_dt, rows, cols, block_rows, q, scale, S(stream)));
}

// ------------------------------------------------------------------- expert FFN ----

namespace {

moe_status check_weights(const moe_shape& sh, const moe_expert_weights* w) {
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(w->gate) || !ok_ptr(w->up) || !ok_ptr(w->down)) return MOE_ERR_INVALID_ARG;
  if (sh.N_s > 0 && (!ok_ptr(w->s_gate) || !ok_ptr(w->s_up) || !ok_ptr(w->s_down)))
    return MOE_ERR_INVALID_ARG;
  if (w->dtype == MOE_E4M3) {
    if (sh.d % 128 != 0 || sh.I % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (!ok_ptr(w->gate_scale) || !ok_ptr(w->up_scale) || !ok_ptr(w->down_scale))
      return MOE_ERR_INVALID_ARG;
    if (sh.N_s > 0 && (!ok_ptr(w->s_gate_scale) || !ok_ptr(w->s_up_scale) || !ok_ptr(w->s_down_scale)))
      return MOE_ERR_INVALID_ARG;
    return MOE_OK;
  }
  if (!is_float_dtype(w->dtype)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

FfnShape ffn_shape(const moe_shape& sh) { return FfnShape{sh.T, sh.d, sh.I, sh.N_r, sh.K_r, sh.N_s}; }

size_t h_bytes(const moe_shape& sh, moe_dtype dt) {
  const size_t rows = (size_t)sh.T * sh.K_r + (size_t)sh.N_s * sh.T;
  return rows * sh.I * elem_bytes(dt);
}

size_t h_scale_bytes(const moe_shape& sh) {
  const size_t rows = (size_t)sh.T * sh.K_r + (size_t)sh.N_s * sh.T;
  return rows * (size_t)(sh.I / 128) * sizeof(float);
}

}  // namespace

size_t moe_expert_ffn_workspace(moe_shape sh, moe_dtype w_dt) {
  if (sh.T <= 0) return 0;
  if (w_dt == MOE_E4M3) return align256(h_bytes(sh, w_dt)) + align256(h_scale_bytes(sh));
  return align256(h_bytes(sh, w_dt));
}

moe_status moe_expert_gate_up(const void* x_perm, const float* x_perm_scale, const void* u,
                              const float* u_scale, const int32_t* expert_offset, moe_shape sh,
                              const moe_expert_weights* w, void* h, float* h_scale,
                              void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if ((st = check_weights(sh, w)) != MOE_OK) return st;
  if (sh.T == 0) return MOE_OK;
  if (!ok_ptr(x_perm) || !ok_ptr(u) || !ok_ptr(expert_offset) || !ok_ptr(h))
    return MOE_ERR_INVALID_ARG;
  const FfnShape fs = ffn_shape(sh);
  cudaError_t err;
  if (w->dtype == MOE_E4M3) {
    if (!ok_ptr(x_perm_scale) || !ok_ptr(h_scale) || (sh.N_s > 0 && !ok_ptr(u_scale)))
      return MOE_ERR_INVALID_ARG;
    err = launch_ffn_up_fp8(fs, x_perm, x_perm_scale, u, u_scale, expert_offset, w, h, h_scale,
                            S(stream));
  } else if (w->dtype == MOE_F32)
    err = launch_ffn_up_simt(fs, (const float*)x_perm, (const float*)u, expert_offset, w,
                             (float*)h, S(stream));
  else
    err = launch_ffn_up_tc(fs, x_perm, u, expert_offset, w, h, S(stream));
  return cuda_status(err);
}

moe_status moe_expert_gate_up_gather(const void* u, const int32_t* perm_token,
                                     const int32_t* expert_offset, moe_shape sh,
                                     const moe_expert_weights* w, void* h, void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if ((st = check_weights(sh, w)) != MOE_OK) return st;
  if (w->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (sh.T == 0) return MOE_OK;
  if (!ok_ptr(u) || !aligned16(u) || !ok_ptr(perm_token) || !ok_ptr(expert_offset) || !ok_ptr(h))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_ffn_up_tc_gather(ffn_shape(sh), u, perm_token, expert_offset, w, h, S(stream)));
}

moe_status moe_expert_down(const void* h, const float* h_scale, const int32_t* expert_offset,
                           moe_shape sh, const moe_expert_weights* w, void* y, void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if ((st = check_weights(sh, w)) != MOE_OK) return st;
  if (sh.T == 0) return MOE_OK;
  if (!ok_ptr(h) || !ok_ptr(expert_offset) || !ok_ptr(y)) return MOE_ERR_INVALID_ARG;
  const FfnShape fs = ffn_shape(sh);
  cudaError_t err;
  if (w->dtype == MOE_E4M3) {
    if (!ok_ptr(h_scale)) return MOE_ERR_INVALID_ARG;
    err = launch_ffn_down_fp8(fs, h, h_scale, expert_offset, w, y, S(stream));
  } else if (w->dtype == MOE_F32)
    err = launch_ffn_down_simt(fs, (const float*)h, expert_offset, w, (float*)y, S(stream));
  else
    err = launch_ffn_down_tc(fs, h, expert_offset, w, y, S(stream));
  return cuda_status(err);
}

moe_status moe_expert_ffn(const void* x_perm, const float* x_perm_scale, const void* u,
                          const float* u_scale, const int32_t* expert_offset, moe_shape sh,
                          const moe_expert_weights* w, void* y, void* workspace,
                          size_t ws_bytes, void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if ((st = check_weights(sh, w)) != MOE_OK) return st;
  if (sh.T == 0) return MOE_OK;
  const size_t need = moe_expert_ffn_workspace(sh, w->dtype);
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < need) return MOE_ERR_WORKSPACE;
  float* h_scale = nullptr;
  if (w->dtype == MOE_E4M3)
    h_scale = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(h_bytes(sh, w->dtype)));
  st = moe_expert_gate_up(x_perm, x_perm_scale, u, u_scale, expert_offset, sh, w, workspace,
                          h_scale, stream);
  if (st != MOE_OK) return st;
  return moe_expert_down(workspace, h_scale, expert_offset, sh, w, y, stream);
}

// ---------------------------------------------------------------------- combine ----

moe_status moe_combine(const void* u, const void* y, moe_dtype dt, const float* topk_gate,
                       const int32_t* inv_row, moe_shape sh, void* h_out, moe_dtype out_dt,
                       void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if (!is_float_dtype(dt) || !is_float_dtype(out_dt)) return MOE_ERR_UNSUPPORTED;
  if (sh.T == 0) return MOE_OK;
  if (!ok_ptr(u) || !ok_ptr(y) || !ok_ptr(topk_gate) || !ok_ptr(inv_row) || !ok_ptr(h_out))
    return MOE_ERR_INVALID_ARG;
  if (((size_t)sh.d * elem_bytes(dt)) % 16 != 0) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(u, y, dt, topk_gate, inv_row, sh.T, sh.d, sh.K_r, sh.N_s,
                                    h_out, out_dt, S(stream)));
}

// ------------------------------------------------------------------ end of step ----

moe_status moe_bias_update(float* b, const int32_t* load, moe_shape sh, float gamma,
                           void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if (!ok_ptr(b) || !ok_ptr(load)) return MOE_ERR_INVALID_ARG;
  if (!(gamma >= 0.f) || gamma > 1e30f) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_bias_update(b, load, sh.T, sh.N_r, sh.K_r, gamma, S(stream)));
}

moe_status moe_seq_balance_stat(const float* seq_p_sum, const int32_t* topk_idx,
                                const int32_t* seq_offsets, int32_t n_seq, moe_shape sh,
                                float alpha, float* stat_per_seq, float* stat_mean,
                                void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if (n_seq < 1 || !ok_ptr(seq_p_sum) || !ok_ptr(seq_offsets) || !ok_ptr(stat_per_seq) ||
      !ok_opt(stat_mean))
    return MOE_ERR_INVALID_ARG;
  if (sh.T > 0 && !ok_ptr(topk_idx)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_seq_stat(seq_p_sum, topk_idx, seq_offsets, n_seq, sh.T, sh.N_r, sh.K_r,
                                     alpha, stat_per_seq, stat_mean, S(stream)));
}

// ---------------------------------------------------------------------- backward ----

namespace {

struct BwdWs {
  size_t h, a, c, dY, dA, dC, dX, dz, dur, counts, total;
};

BwdWs bwd_ws(const moe_shape& sh, int n_seq) {
  const size_t R = (size_t)sh.T * sh.K_r + (size_t)sh.N_s * sh.T;
  const size_t ri = align256(R * sh.I * 2), rd = align256(R * sh.d * 2);
  BwdWs w;
  size_t o = 0;
  w.h = o; o += ri;
  w.a = o; o += ri;
  w.c = o; o += ri;
  w.dA = o; o += ri;
  w.dC = o; o += ri;
  w.dY = o; o += rd;
  w.dX = o; o += rd;
  w.dz = o; o += align256((size_t)sh.T * sh.N_r * 2);
  w.dur = o; o += align256((size_t)sh.T * sh.d * 4);
  w.counts = o; o += align256((size_t)(n_seq > 0 ? n_seq : 1) * sh.N_r * 4);
  w.total = o;
  return w;
}

}  // namespace

namespace {

moe_status zero_grads(const moe_shape& sh, float* de, float* dw_gate, float* dw_up, float* dw_down,
                      float* dws_gate, float* dws_up, float* dws_down, cudaStream_t cs) {
  const size_t gi = (size_t)sh.I * sh.d * 4;
  cudaError_t err = cudaMemsetAsync(de, 0, (size_t)sh.N_r * sh.d * 4, cs);
  if (err == cudaSuccess) err = cudaMemsetAsync(dw_gate, 0, sh.N_r * gi, cs);
  if (err == cudaSuccess) err = cudaMemsetAsync(dw_up, 0, sh.N_r * gi, cs);
  if (err == cudaSuccess) err = cudaMemsetAsync(dw_down, 0, sh.N_r * gi, cs);
  if (sh.N_s > 0) {
    if (err == cudaSuccess) err = cudaMemsetAsync(dws_gate, 0, sh.N_s * gi, cs);
    if (err == cudaSuccess) err = cudaMemsetAsync(dws_up, 0, sh.N_s * gi, cs);
    if (err == cudaSuccess) err = cudaMemsetAsync(dws_down, 0, sh.N_s * gi, cs);
  }
  return cuda_status(err);
}

}  // namespace

size_t moe_backward_workspace(moe_shape sh, int32_t n_seq) {
  if (sh.T <= 0 || sh.N_r <= 0 || sh.d <= 0 || sh.I <= 0 || n_seq < 0) return 0;
  return bwd_ws(sh, n_seq).total;
}

moe_status moe_backward(const void* u, const void* e, const float* s, const int32_t* topk_idx,
                        const float* topk_gate, const int32_t* expert_offset,
                        const int32_t* inv_row, const void* x_perm, const void* y,
                        const moe_expert_weights* w, moe_shape sh, const int32_t* seq_offsets,
                        int32_t n_seq, float alpha, const float* dh, float* du, float* de,
                        float* dw_gate, float* dw_up, float* dw_down, float* dws_gate,
                        float* dws_up, float* dws_down, void* workspace, size_t ws_bytes,
                        void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if ((st = check_weights(sh, w)) != MOE_OK) return st;
  if (w->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (sh.N_r % 64 != 0 || n_seq < 0 || !(alpha >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(e) || !ok_ptr(de) || !ok_ptr(dw_gate) || !ok_ptr(dw_up) || !ok_ptr(dw_down))
    return MOE_ERR_INVALID_ARG;
  if (sh.N_s > 0 && (!ok_ptr(dws_gate) || !ok_ptr(dws_up) || !ok_ptr(dws_down)))
    return MOE_ERR_INVALID_ARG;
  const bool balance = n_seq > 0 && alpha != 0.f;
  if (balance && !ok_ptr(seq_offsets)) return MOE_ERR_INVALID_ARG;
  const cudaStream_t cs = S(stream);
  if (sh.T == 0)   // no token: every gradient is zero
    return zero_grads(sh, de, dw_gate, dw_up, dw_down, dws_gate, dws_up, dws_down, cs);
  if (!ok_ptr(u) || !ok_ptr(s) || !ok_ptr(topk_idx) || !ok_ptr(topk_gate) || !ok_ptr(expert_offset) ||
      !ok_ptr(inv_row) || !ok_ptr(x_perm) || !ok_ptr(y) || !ok_ptr(dh) || !ok_ptr(du))
    return MOE_ERR_INVALID_ARG;
  const BwdWs L = bwd_ws(sh, n_seq);
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(ws + off); };
  const FfnShape fs = ffn_shape(sh);
  // the SwiGLU output and pre-activations, recomputed
  cudaError_t err = launch_ffn_up_tc(fs, x_perm, u, expert_offset, w, bf(L.h), cs, bf(L.a), bf(L.c));
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  if (err == cudaSuccess && balance)
    err = launch_seq_counts(topk_idx, seq_offsets, n_seq, sh.T, sh.N_r, sh.K_r, counts, cs);
  if (err == cudaSuccess)
    err = launch_bwd_prep(dh, y, s, topk_idx, topk_gate, inv_row, counts, seq_offsets,
                          balance ? n_seq : 0, balance ? alpha : 0.f, sh.T, sh.d, sh.N_r, sh.K_r,
                          sh.N_s, ws + L.dz, ws + L.dY, cs);
  if (err == cudaSuccess) {
    BwdGemmIo io{fs, expert_offset, w->gate, w->up, w->down, w->s_gate, w->s_up, w->s_down,
                 x_perm, u, e, bf(L.a), bf(L.c), bf(L.h), ws + L.dY, ws + L.dz, bf(L.dA), bf(L.dC),
                 bf(L.dX), dw_gate, dw_up, dw_down, dws_gate, dws_up, dws_down,
                 reinterpret_cast<float*>(ws + L.dur), de};
    err = launch_bwd_gemms(io, cs);
  }
  if (err == cudaSuccess)
    err = launch_bwd_combine(dh, reinterpret_cast<const float*>(ws + L.dur), ws + L.dX, inv_row,
                             sh.T, sh.d, sh.K_r, sh.N_s, du, cs);
  return cuda_status(err);
}

moe_status moe_fp8_dgrad_weights_make(const moe_expert_weights* w, moe_shape sh,
                                      const moe_fp8_dgrad_weights* wt, void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if ((st = check_weights(sh, w)) != MOE_OK) return st;
  if (w->dtype != MOE_E4M3 || wt == nullptr) return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(wt->wdt) || !ok_ptr(wt->wdt_scale) || !ok_ptr(wt->wgut) || !ok_ptr(wt->wgut_scale))
    return MOE_ERR_INVALID_ARG;
  if (sh.N_s > 0 && (!ok_ptr(wt->s_wdt) || !ok_ptr(wt->s_wdt_scale) || !ok_ptr(wt->s_wgut) ||
                     !ok_ptr(wt->s_wgut_scale)))
    return MOE_ERR_INVALID_ARG;
  const cudaStream_t cs = S(stream);
  auto u8 = [](const void* p) { return static_cast<const uint8_t*>(p); };
  auto m8 = [](void* p) { return static_cast<uint8_t*>(p); };
  cudaError_t err = cudaSuccess;
  for (int sh_part = 0; sh_part < 2 && err == cudaSuccess; ++sh_part) {
    const int E = sh_part ? sh.N_s : sh.N_r;
    if (E == 0) continue;
    const void* gate = sh_part ? w->s_gate : w->gate;
    const void* up = sh_part ? w->s_up : w->up;
    const void* down = sh_part ? w->s_down : w->down;
    const float* gs = sh_part ? w->s_gate_scale : w->gate_scale;
    const float* us = sh_part ? w->s_up_scale : w->up_scale;
    const float* ds = sh_part ? w->s_down_scale : w->down_scale;
    void* wdt = sh_part ? wt->s_wdt : wt->wdt;
    float* wdts = sh_part ? wt->s_wdt_scale : wt->wdt_scale;
    void* wgut = sh_part ? wt->s_wgut : wt->wgut;
    float* wguts = sh_part ? wt->s_wgut_scale : wt->wgut_scale;
    err = launch_fp8_transpose(u8(down), ds, E, sh.d, sh.I, m8(wdt), wdts, sh.d, 0, cs);
    if (err == cudaSuccess) err = launch_fp8_transpose(u8(gate), gs, E, sh.I, sh.d, m8(wgut), wguts, 2 * sh.I, 0, cs);
    if (err == cudaSuccess)
      err = launch_fp8_transpose(u8(up), us, E, sh.I, sh.d, m8(wgut), wguts, 2 * sh.I, sh.I, cs);
  }
  return cuda_status(err);
}

namespace {

struct Fp8BwdWs {
  size_t hq, hs, a, c, dY, dYq, dYs, dH, acq, acs, dA, dC, dX;
  size_t t_dY, s_dY, t_h, s_h, t_dA, s_dA, t_dC, s_dC, t_x, s_x, dz, dur, counts, total;
  long long Rp;
};

Fp8BwdWs fp8_bwd_ws(const moe_shape& sh, int n_seq) {
  const size_t R = (size_t)sh.T * sh.K_r + (size_t)sh.N_s * sh.T;
  const size_t d = sh.d, I = sh.I;
  Fp8BwdWs w;
  // padded Wgrad row space: every segment rounded up to whole 128-token blocks
  w.Rp = (long long)(((R + 127) / 128) * 128 + 128 * (size_t)(sh.N_r + sh.N_s));
  const size_t Rp = (size_t)w.Rp, nb = Rp / 128;
  size_t o = 0;
  auto take = [&](size_t& f, size_t bytes) { f = o; o += align256(bytes); };
  take(w.hq, R * I);
  take(w.hs, R * (I / 128) * 4);
  take(w.a, R * I * 2);
  take(w.c, R * I * 2);
  take(w.dY, R * d * 2);
  take(w.dYq, R * d);
  take(w.dYs, R * (d / 128) * 4);
  take(w.dH, R * I * 2);
  take(w.acq, R * 2 * I);
  take(w.acs, R * (2 * I / 128) * 4);
  take(w.dA, R * I * 2);
  take(w.dC, R * I * 2);
  take(w.dX, R * d * 2);
  take(w.t_dY, d * Rp);
  take(w.s_dY, nb * d * 4);
  take(w.t_h, I * Rp);
  take(w.s_h, nb * I * 4);
  take(w.t_dA, I * Rp);
  take(w.s_dA, nb * I * 4);
  take(w.t_dC, I * Rp);
  take(w.s_dC, nb * I * 4);
  take(w.t_x, d * Rp);
  take(w.s_x, nb * d * 4);
  take(w.dz, (size_t)sh.T * sh.N_r * 2);
  take(w.dur, (size_t)sh.T * d * 4);
  take(w.counts, (size_t)(n_seq > 0 ? n_seq : 1) * sh.N_r * 4);
  w.total = o;
  return w;
}

}  // namespace

size_t moe_backward_fp8_workspace(moe_shape sh, int32_t n_seq) {
  if (sh.T <= 0 || sh.N_r <= 0 || sh.d <= 0 || sh.I <= 0 || n_seq < 0) return 0;
  return fp8_bwd_ws(sh, n_seq).total;
}

moe_status moe_backward_fp8(const void* u, const void* u_q, const float* u_scale, const void* e,
                            const float* s, const int32_t* topk_idx, const float* topk_gate,
                            const int32_t* expert_offset, const int32_t* inv_row, const void* x_perm_q,
                            const float* x_perm_scale, const void* y, const moe_expert_weights* w,
                            const moe_fp8_dgrad_weights* wt, moe_shape sh, const int32_t* seq_offsets,
                            int32_t n_seq, float alpha, const float* dh, float* du, float* de,
                            float* dw_gate, float* dw_up, float* dw_down, float* dws_gate,
                            float* dws_up, float* dws_down, void* workspace, size_t ws_bytes,
                            void* stream) {
  moe_status st = check_shape(sh);
  if (st != MOE_OK) return st;
  if ((st = check_weights(sh, w)) != MOE_OK) return st;
  if (w->dtype != MOE_E4M3 || wt == nullptr) return MOE_ERR_INVALID_ARG;
  if (sh.N_r % 64 != 0 || n_seq < 0 || !(alpha >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(e) || !ok_ptr(de) || !ok_ptr(dw_gate) || !ok_ptr(dw_up) || !ok_ptr(dw_down))
    return MOE_ERR_INVALID_ARG;
  if (sh.N_s > 0 && (!ok_ptr(dws_gate) || !ok_ptr(dws_up) || !ok_ptr(dws_down)))
    return MOE_ERR_INVALID_ARG;
  const bool balance = n_seq > 0 && alpha != 0.f;
  if (balance && !ok_ptr(seq_offsets)) return MOE_ERR_INVALID_ARG;
  if (sh.T == 0)   // no token: every gradient is zero
    return zero_grads(sh, de, dw_gate, dw_up, dw_down, dws_gate, dws_up, dws_down, S(stream));
  if (!ok_ptr(u) || !ok_ptr(u_q) || !ok_ptr(u_scale) || !ok_ptr(s) || !ok_ptr(topk_idx) ||
      !ok_ptr(topk_gate) || !ok_ptr(expert_offset) || !ok_ptr(inv_row) || !ok_ptr(x_perm_q) ||
      !ok_ptr(x_perm_scale) || !ok_ptr(y) || !ok_ptr(dh) || !ok_ptr(du) || !ok_ptr(wt->wdt) ||
      !ok_ptr(wt->wdt_scale) || !ok_ptr(wt->wgut) || !ok_ptr(wt->wgut_scale))
    return MOE_ERR_INVALID_ARG;
  if (sh.N_s > 0 && (!ok_ptr(wt->s_wdt) || !ok_ptr(wt->s_wdt_scale) || !ok_ptr(wt->s_wgut) ||
                     !ok_ptr(wt->s_wgut_scale)))
    return MOE_ERR_INVALID_ARG;
  const Fp8BwdWs L = fp8_bwd_ws(sh, n_seq);
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  auto at = [&](size_t off) { return static_cast<void*>(ws + off); };
  auto u8 = [&](size_t off) { return reinterpret_cast<uint8_t*>(ws + off); };
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  const cudaStream_t cs = S(stream);
  const FfnShape fs = ffn_shape(sh);
  const long long R = (long long)sh.T * sh.K_r + (long long)sh.N_s * sh.T;
  const long long routed = (long long)sh.T * sh.K_r;
  // Fprop again: the E4M3 h Wgrad reads, and the pre-activations a, c (bf16)
  cudaError_t err = launch_ffn_up_fp8(fs, x_perm_q, x_perm_scale, u_q, u_scale, expert_offset, w, at(L.hq),
                                      f32(L.hs), cs, at(L.a), at(L.c));
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  if (err == cudaSuccess && balance)
    err = launch_seq_counts(topk_idx, seq_offsets, n_seq, sh.T, sh.N_r, sh.K_r, counts, cs);
  if (err == cudaSuccess)
    err = launch_bwd_prep(dh, y, s, topk_idx, topk_gate, inv_row, counts, seq_offsets, balance ? n_seq : 0,
                          balance ? alpha : 0.f, sh.T, sh.d, sh.N_r, sh.K_r, sh.N_s, at(L.dz), at(L.dY), cs);
  // Dgrad: dH = dY W_down (dY in 1x128 tiles), the SwiGLU backward, dX = [dA|dC] [W_gate; W_up]
  if (err == cudaSuccess) err = launch_quantize_e4m3(at(L.dY), MOE_BF16, R, sh.d, 1, u8(L.dYq), f32(L.dYs), cs);
  if (err == cudaSuccess) {
    FfnShape fd = fs;
    fd.d = sh.I;
    fd.I = sh.d;
    moe_expert_weights wd{};
    wd.dtype = MOE_E4M3;
    wd.down = wt->wdt;
    wd.down_scale = wt->wdt_scale;
    wd.s_down = wt->s_wdt;
    wd.s_down_scale = wt->s_wdt_scale;
    err = launch_ffn_down_fp8(fd, at(L.dYq), f32(L.dYs), expert_offset, &wd, at(L.dH), cs);
  }
  if (err == cudaSuccess)
    err = launch_fp8_swiglu_bwd(at(L.dH), at(L.a), at(L.c), R, sh.I, u8(L.acq), f32(L.acs), at(L.dA), at(L.dC), cs);
  if (err == cudaSuccess) {
    FfnShape fx = fs;
    fx.I = 2 * sh.I;
    moe_expert_weights wx{};
    wx.dtype = MOE_E4M3;
    wx.down = wt->wgut;
    wx.down_scale = wt->wgut_scale;
    wx.s_down = wt->s_wgut;
    wx.s_down_scale = wt->s_wgut_scale;
    err = launch_ffn_down_fp8(fx, at(L.acq), f32(L.acs), expert_offset, &wx, at(L.dX), cs);
  }
  // Wgrad operands: 128x1 tiles over each segment's tokens, transposed
  const auto bf = [&](size_t off, long long row, int C) {
    return static_cast<const void*>(ws + off + (size_t)row * C * 2);
  };
  const struct { ColQuantSrc src; int C; size_t q, sc; } ops[5] = {
      {{bf(L.dY, 0, sh.d), bf(L.dY, routed, sh.d), nullptr, nullptr, sh.T}, sh.d, L.t_dY, L.s_dY},
      {{ws + L.hq, ws + L.hq + (size_t)routed * sh.I, f32(L.hs), f32(L.hs) + (size_t)routed * (sh.I / 128), sh.T},
       sh.I, L.t_h, L.s_h},
      {{bf(L.dA, 0, sh.I), bf(L.dA, routed, sh.I), nullptr, nullptr, sh.T}, sh.I, L.t_dA, L.s_dA},
      {{bf(L.dC, 0, sh.I), bf(L.dC, routed, sh.I), nullptr, nullptr, sh.T}, sh.I, L.t_dC, L.s_dC},
      {{x_perm_q, u_q, x_perm_scale, u_scale, 0}, sh.d, L.t_x, L.s_x}};
  for (int i = 0; i < 5 && err == cudaSuccess; ++i)
    err = launch_fp8_colquant(ops[i].src, expert_offset, sh.T, sh.K_r, sh.N_r, sh.N_s, ops[i].C, u8(ops[i].q),
                              f32(ops[i].sc), L.Rp, cs);
  // Wgrad: dW_down = dY^T h, dW_gate = dA^T x, dW_up = dC^T x per expert
  if (err == cudaSuccess)
    err = launch_fp8_wgrad(u8(L.t_dY), f32(L.s_dY), u8(L.t_h), f32(L.s_h), sh.d, sh.I, L.Rp, expert_offset,
                           sh.T, sh.K_r, sh.N_r, sh.N_s, dw_down, dws_down, cs);
  if (err == cudaSuccess)
    err = launch_fp8_wgrad(u8(L.t_dA), f32(L.s_dA), u8(L.t_x), f32(L.s_x), sh.I, sh.d, L.Rp, expert_offset,
                           sh.T, sh.K_r, sh.N_r, sh.N_s, dw_gate, dws_gate, cs);
  if (err == cudaSuccess)
    err = launch_fp8_wgrad(u8(L.t_dC), f32(L.s_dC), u8(L.t_x), f32(L.s_x), sh.I, sh.d, L.Rp, expert_offset,
                           sh.T, sh.K_r, sh.N_r, sh.N_s, dw_up, dws_up, cs);
  // router: du = dz e, de = dz^T u (bf16, as in the FP8 forward)
  if (err == cudaSuccess) {
    BwdGemmIo io{fs, expert_offset, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, u, e,
                 nullptr, nullptr, nullptr, nullptr, at(L.dz), nullptr, nullptr, nullptr, nullptr, nullptr,
                 nullptr, nullptr, nullptr, nullptr, f32(L.dur), de};
    io.experts = false;
    err = launch_bwd_gemms(io, cs);
  }
  if (err == cudaSuccess)
    err = launch_bwd_combine(dh, f32(L.dur), at(L.dX), inv_row, sh.T, sh.d, sh.K_r, sh.N_s, du, cs);
  return cuda_status(err);
}

moe_status moe_device_error(int32_t* code, int32_t clear) {
  if (code == nullptr) return MOE_ERR_INVALID_ARG;
  return cuda_status(read_dev_error(code, clear != 0));
}

}  // extern "C"
