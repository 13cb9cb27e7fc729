// Backward pass, the parts around the GEMMs: per-sequence selection counts, the per-token
// gradients of the gates, affinities and expert outputs, and the sum into du.
//
// At the forward pass's selection the layer is h'_t = u_t + sum_s FFN_s(u_t) +
// sum_k g_{k,t} FFN_{idx_k}(u_t) with g_k = s_{idx_k} / sum_j s_{idx_j} and s = sigmoid(z),
// z = u e^T (DeepSeek-V3 Technical Report reading guide, Method §2), plus the
// sequence-wise balance loss alpha * sum_i f_i P_i averaged over the sequences (pwwt.cn
// notes §1.2; f_i counts selections and passes no gradient, P_i is the mean over the
// sequence of s_{i,t} / sum_j s_{j,t}).  For an upstream gradient dh = dJ/dh':
//   dgate_k   = dh_t . y_{t,k}                    (y_{t,k} = FFN_{idx_k}(u_t))
//   ds_{idx_j} = (dgate_j - sum_k g_k dgate_k) / sum_j s_{idx_j}   (raw s: the bias gets none)
//   ds_{i,t} += alpha/n_seq * (f_i - sum_j f_j s_{j,t}/R_t) / (T_S R_t),  R_t = sum_j s_{j,t}
//   dz = ds * s (1 - s)
//   dY rows: g_k dh_t for the routed slots, dh_t for the shared experts
#include "common.cuh"
#include "launch.h"
#include "route_select.cuh"

namespace moe {

namespace {

__global__ void seq_counts_kernel(const int32_t* __restrict__ topk_idx,
                                  const int32_t* __restrict__ seq_offsets, int n_seq, int T, int N_r,
                                  int K_r, int32_t* __restrict__ counts, int32_t* err) {
  const long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= (long long)T * K_r) return;
  const int t = (int)(x / K_r);
  const int ex = topk_idx[x];
  if ((unsigned)ex >= (unsigned)N_r) {
    record_error(err, MOE_ERR_INVALID_ARG);
    return;
  }
  const int j = seq_of(t, seq_offsets, n_seq);
  atomicAdd(counts + (size_t)j * N_r + ex, 1);   // integer adds: exact in any order
}

// One warp per token.  s and the counts give ds; dz is written for every expert.
__global__ void __launch_bounds__(256) bwd_prep_kernel(
    const float* __restrict__ dh, const __nv_bfloat16* __restrict__ y, const float* __restrict__ s,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_gate,
    const int32_t* __restrict__ inv_row, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ seq_offsets, int n_seq, float alpha, int T, int d, int N_r, int K_r,
    int N_s, __nv_bfloat16* __restrict__ dz, __nv_bfloat16* __restrict__ dY, int32_t* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  const size_t R0 = (size_t)T * K_r;
  const float* dht = dh + (size_t)t * d;
  // the token's slots: expert, gate, row (one per lane, K_r <= 32)
  int my_i = 0, my_r = 0;
  float my_g = 0.f;
  if (lane < K_r) {
    my_i = topk_idx[(size_t)t * K_r + lane];
    my_g = topk_gate[(size_t)t * K_r + lane];
    my_r = inv_row[(size_t)t * K_r + lane];
    if ((unsigned)my_i >= (unsigned)N_r || (size_t)(unsigned)my_r >= R0) {
      record_error(err, MOE_ERR_INVALID_ARG);
      my_i = 0;
      my_r = 0;
      my_g = 0.f;
    }
  }
  // dgate_k = dh_t . y_{t,k}; dY rows = g_k dh_t (routed) and dh_t (shared)
  float my_dg = 0.f;
  for (int k = 0; k < K_r; ++k) {
    const int r = __shfl_sync(0xffffffffu, my_r, k);
    const float gk = __shfl_sync(0xffffffffu, my_g, k);
    const __nv_bfloat16* yr = y + (size_t)r * d;
    __nv_bfloat16* dyr = dY + (size_t)r * d;
    float acc = 0.f;
    for (int j = lane * 8; j < d; j += 256) {
      const float4 h0 = *reinterpret_cast<const float4*>(dht + j);
      const float4 h1 = *reinterpret_cast<const float4*>(dht + j + 4);
      const uint4 yv = *reinterpret_cast<const uint4*>(yr + j);
      const __nv_bfloat16* yb = reinterpret_cast<const __nv_bfloat16*>(&yv);
      const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      uint4 ov;
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(&ov);
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        acc = fmaf(hv[x], __bfloat162float(yb[x]), acc);
        ob[x] = __float2bfloat16_rn(gk * hv[x]);
      }
      *reinterpret_cast<uint4*>(dyr + j) = ov;
    }
    acc = warp_sum(acc);
    if (lane == k) my_dg = acc;
  }
  for (int sh = 0; sh < N_s; ++sh) {
    __nv_bfloat16* dyr = dY + (R0 + (size_t)sh * T + t) * d;
    for (int j = lane * 8; j < d; j += 256) {
      const float4 h0 = *reinterpret_cast<const float4*>(dht + j);
      const float4 h1 = *reinterpret_cast<const float4*>(dht + j + 4);
      uint4 ov;
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(&ov);
      ob[0] = __float2bfloat16_rn(h0.x); ob[1] = __float2bfloat16_rn(h0.y);
      ob[2] = __float2bfloat16_rn(h0.z); ob[3] = __float2bfloat16_rn(h0.w);
      ob[4] = __float2bfloat16_rn(h1.x); ob[5] = __float2bfloat16_rn(h1.y);
      ob[6] = __float2bfloat16_rn(h1.z); ob[7] = __float2bfloat16_rn(h1.w);
      *reinterpret_cast<uint4*>(dyr + j) = ov;
    }
  }
  // gate backward: ds_{idx_j} = (dgate_j - sum_k g_k dgate_k) / S, S = sum of the raw s
  const float* st = s + (size_t)t * N_r;
  const float my_s = lane < K_r ? st[my_i] : 0.f;
  const float S = warp_sum(my_s);
  const float inner = warp_sum(lane < K_r ? my_g * my_dg : 0.f);
  const float my_ds_sel = lane < K_r ? (my_dg - inner) / S : 0.f;
  // balance-loss backward for the token's sequence
  float coef = 0.f, inner2 = 0.f, Rt = 1.f;
  int seq = 0;
  if (alpha != 0.f && n_seq > 0) {
    seq = seq_of(t, seq_offsets, n_seq);
    const int T_S = seq_offsets[seq + 1] - seq_offsets[seq];
    float rs = 0.f, fs = 0.f;
    for (int i = lane; i < N_r; i += 32) {
      const float f = (float)N_r / ((float)K_r * T_S) * (float)counts[(size_t)seq * N_r + i];
      rs += st[i];
      fs += f * st[i];
    }
    Rt = warp_sum(rs);
    inner2 = warp_sum(fs) / Rt;
    coef = T_S > 0 ? alpha / (float)n_seq / ((float)T_S * Rt) : 0.f;
  }
  for (int i0 = 0; i0 < N_r; i0 += 32) {   // warp-uniform: the shuffles need every lane
    const int i = i0 + lane;
    float ds = 0.f;
    for (int k = 0; k < K_r; ++k) {         // the selected slot of expert i, if any
      const int ik = __shfl_sync(0xffffffffu, my_i, k);
      const float dk = __shfl_sync(0xffffffffu, my_ds_sel, k);
      if (ik == i) ds += dk;
    }
    if (i < N_r) {
      const float si = st[i];
      if (coef != 0.f) {
        const float f = (float)N_r / ((float)K_r * (seq_offsets[seq + 1] - seq_offsets[seq])) *
                        (float)counts[(size_t)seq * N_r + i];
        ds += coef * (f - inner2);
      }
      dz[(size_t)t * N_r + i] = __float2bfloat16_rn(ds * si * (1.f - si));
    }
  }
}

// du_t = dh_t + du_router_t + sum_s dX[T*K_r + s*T + t] + sum_k dX[inv_row[t, k]], fp32,
// in that order; one warp per token, 8 columns per lane per pass.
__global__ void __launch_bounds__(256) bwd_combine_kernel(
    const float* __restrict__ dh, const float* __restrict__ du_router,
    const __nv_bfloat16* __restrict__ dX, const int32_t* __restrict__ inv_row, int T, int d, int K_r,
    int N_s, float* __restrict__ du, int32_t* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  const size_t R0 = (size_t)T * K_r;
  int my_r = lane < K_r ? inv_row[(size_t)t * K_r + lane] : 0;
  bool my_ok = lane < K_r;
  if (my_ok && (size_t)(unsigned)my_r >= R0) {
    record_error(err, MOE_ERR_INVALID_ARG);
    my_ok = false;
    my_r = 0;
  }
  for (int j = lane * 8; j < d; j += 256) {
    float acc[8];
    const float4 a0 = *reinterpret_cast<const float4*>(dh + (size_t)t * d + j);
    const float4 a1 = *reinterpret_cast<const float4*>(dh + (size_t)t * d + j + 4);
    acc[0] = a0.x; acc[1] = a0.y; acc[2] = a0.z; acc[3] = a0.w;
    acc[4] = a1.x; acc[5] = a1.y; acc[6] = a1.z; acc[7] = a1.w;
    if (du_router) {
      const float4 b0 = *reinterpret_cast<const float4*>(du_router + (size_t)t * d + j);
      const float4 b1 = *reinterpret_cast<const float4*>(du_router + (size_t)t * d + j + 4);
      acc[0] += b0.x; acc[1] += b0.y; acc[2] += b0.z; acc[3] += b0.w;
      acc[4] += b1.x; acc[5] += b1.y; acc[6] += b1.z; acc[7] += b1.w;
    }
    auto add_row = [&](size_t r) {
      const uint4 v = *reinterpret_cast<const uint4*>(dX + r * d + j);
      const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[x] += __bfloat162float(vb[x]);
    };
    for (int sh = 0; sh < N_s; ++sh) add_row(R0 + (size_t)sh * T + t);
    for (int k = 0; k < K_r; ++k) {
      const int r = __shfl_sync(0xffffffffu, my_r, k);
      const bool ok = __shfl_sync(0xffffffffu, my_ok, k);
      if (ok) add_row((size_t)r);
    }
    float4* o = reinterpret_cast<float4*>(du + (size_t)t * d + j);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

}  // namespace

cudaError_t launch_seq_counts(const int32_t* topk_idx, const int32_t* seq_offsets, int n_seq, int T,
                              int N_r, int K_r, int32_t* counts, cudaStream_t st) {
  cudaError_t err = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)n_seq * N_r, st);
  if (err != cudaSuccess || T == 0) return err;
  const long long n = (long long)T * K_r;
  seq_counts_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(topk_idx, seq_offsets, n_seq, T, N_r,
                                                                 K_r, counts, dev_error_ptr());
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const float* dh, const void* y, const float* s, const int32_t* topk_idx,
                            const float* topk_gate, const int32_t* inv_row, const int32_t* counts,
                            const int32_t* seq_offsets, int n_seq, float alpha, int T, int d,
                            int N_r, int K_r, int N_s, void* dz, void* dY, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  bwd_prep_kernel<<<(T + 7) / 8, 256, 0, st>>>(
      dh, (const __nv_bfloat16*)y, s, topk_idx, topk_gate, inv_row, counts, seq_offsets, n_seq,
      alpha, T, d, N_r, K_r, N_s, (__nv_bfloat16*)dz, (__nv_bfloat16*)dY, dev_error_ptr());
  return cudaGetLastError();
}

cudaError_t launch_bwd_combine(const float* dh, const float* du_router, const void* dX,
                               const int32_t* inv_row, int T, int d, int K_r, int N_s, float* du,
                               cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  bwd_combine_kernel<<<(T + 7) / 8, 256, 0, st>>>(dh, du_router, (const __nv_bfloat16*)dX, inv_row, T,
                                                  d, K_r, N_s, du, dev_error_ptr());
  return cudaGetLastError();
}

}  // namespace moe
