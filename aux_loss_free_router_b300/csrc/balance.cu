// End-of-step state: the bias update and the sequence-wise balance statistic.
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

// The library's device error word (one per device that loads the library).
__device__ int32_t g_dev_error = 0;


// b_i += gamma * sign(T*K_r - N_r*load_i): overloaded experts (load above the batch
// mean T*K_r/N_r) move down by gamma, underloaded ones up, experts exactly at the
// mean stay (pwwt.cn notes §1.1.3; gamma = 0.001 in the reading guide, Method §2).
__global__ void bias_update_kernel(float* __restrict__ b, const int32_t* __restrict__ load,
                                   long long total, int N_r, float gamma) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N_r) return;
  const long long diff = total - (long long)N_r * load[i];
  const float step = diff > 0 ? gamma : (diff < 0 ? -gamma : 0.f);
  b[i] = __fadd_rn(b[i], step);
}

// alpha * sum_i f_i P_i per sequence (pwwt.cn notes §1.2), one block for the batch:
// per sequence an integer histogram of the selected experts, then a fixed-order fp64
// sum.  f_i = N_r/(K_r*T_j) * count_i, P_i = seq_p_sum[j, i] / T_j.
__global__ void __launch_bounds__(1024) seq_stat_kernel(const float* __restrict__ seq_p_sum,
                                                        const int32_t* __restrict__ topk_idx,
                                                        const int32_t* __restrict__ seq_offsets,
                                                        int n_seq, int N_r, int K_r, float alpha,
                                                        float* __restrict__ stat_per_seq,
                                                        float* __restrict__ stat_mean) {
  __shared__ int32_t cnt[256];
  __shared__ double term[256];
  double mean_acc = 0.0;
  for (int j = 0; j < n_seq; ++j) {
    for (int i = threadIdx.x; i < N_r; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int a = seq_offsets[j], z = seq_offsets[j + 1];
    const long long n_ent = (long long)(z - a) * K_r;
    const int32_t* src = topk_idx + (size_t)a * K_r;
    for (long long x = threadIdx.x; x < n_ent; x += blockDim.x) atomicAdd(&cnt[src[x]], 1);
    __syncthreads();
    const int T_j = z - a;
    for (int i = threadIdx.x; i < N_r; i += blockDim.x) {
      double v = 0.0;
      if (T_j > 0) {
        const double f = (double)N_r / ((double)K_r * T_j) * (double)cnt[i];
        const double P = (double)seq_p_sum[(size_t)j * N_r + i] / (double)T_j;
        v = f * P;
      }
      term[i] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      double s = 0.0;
      for (int i = 0; i < N_r; ++i) s += term[i];
      const double st = (double)alpha * s;
      stat_per_seq[j] = (float)st;
      mean_acc += st;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0 && stat_mean) *stat_mean = n_seq > 0 ? (float)(mean_acc / n_seq) : 0.f;
}

}  // namespace

int32_t* dev_error_ptr() {
  // The symbol's device address differs per device: look it up for the current one.
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_dev_error) != cudaSuccess) return nullptr;
  return static_cast<int32_t*>(p);
}

cudaError_t read_dev_error(int32_t* code, bool clear) {
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  err = cudaMemcpyFromSymbol(code, g_dev_error, sizeof(int32_t));
  if (err != cudaSuccess || !clear) return err;
  const int32_t zero = 0;
  return cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(int32_t));
}

cudaError_t launch_bias_update(float* b, const int32_t* load, int T, int N_r, int K_r,
                               float gamma, cudaStream_t st) {
  bias_update_kernel<<<(N_r + 255) / 256, 256, 0, st>>>(b, load, (long long)T * K_r, N_r, gamma);
  return cudaGetLastError();
}

cudaError_t launch_seq_stat(const float* seq_p_sum, const int32_t* topk_idx,
                            const int32_t* seq_offsets, int n_seq, int N_r, int K_r,
                            float alpha, float* stat_per_seq, float* stat_mean,
                            cudaStream_t st) {
  seq_stat_kernel<<<1, 1024, 0, st>>>(seq_p_sum, topk_idx, seq_offsets, n_seq, N_r, K_r, alpha,
                                      stat_per_seq, stat_mean);
  return cudaGetLastError();
}

}  // namespace moe
