// End-of-step state: the bias update and the sequence-wise balance statistic.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace moe {

namespace {

// The library's device error word (one per device that loads the library).
__device__ int32_t g_dev_error = 0;


// b_i += gamma * sign(T*K_r - N_r*load_i): overloaded experts (load above the batch
// mean T*K_r/N_r) move down by gamma, underloaded ones up, experts exactly at the
// mean stay (pwwt.cn notes §1.1.3; gamma = 0.001 in the reading guide, Method §2).
__global__ void bias_update_kernel(float* __restrict__ b, const int32_t* __restrict__ load,
                                   long long total, int N_r, float gamma) {
  pdl_release();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N_r) return;
  const long long diff = total - (long long)N_r * load[i];
  const float step = diff > 0 ? gamma : (diff < 0 ? -gamma : 0.f);
  b[i] = __fadd_rn(b[i], step);
}

// alpha * sum_i f_i P_i per sequence (pwwt.cn notes §1.2).  A cluster of kStatSplit CTAs
// per sequence: each builds the integer histogram of the experts selected in its slab
// of the sequence's (token, slot) entries; CTA 0 of the cluster adds the histograms
// (integers: exact in any order) through distributed shared memory, then forms
// f_i = N_r/(K_r*T_j) * count_i and P_i = seq_p_sum[j, i] / T_j and sums f_i P_i by a
// fixed-order fp64 tree.  Offsets that are not 0 = off[0] <= ... <= off[n_seq] = T, and
// selected experts outside [0, N_r), record MOE_ERR_INVALID_ARG and are left out (a
// sequence whose own bounds are out of order or outside [0, T] counts as empty).
constexpr int kStatSplit = 8;

__global__ void __cluster_dims__(kStatSplit, 1, 1) __launch_bounds__(256)
    seq_stat_kernel(const float* __restrict__ seq_p_sum, const int32_t* __restrict__ topk_idx,
                    const int32_t* __restrict__ seq_offsets, int n_seq, int T, int N_r, int K_r,
                    float alpha, float* __restrict__ stat_per_seq, float* __restrict__ stat_mean,
                    int32_t* err) {
  __shared__ int32_t cnt[256];
  __shared__ double term[256];
  pdl_release();
  pdl_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int j = blockIdx.x / kStatSplit;
  cnt[threadIdx.x] = 0;
  __syncthreads();
  int a = seq_offsets[j], z = seq_offsets[j + 1];
  const bool bad = a < 0 || z < a || z > T || (j == 0 && a != 0) || (j == n_seq - 1 && z != T);
  if (bad) {
    if (threadIdx.x == 0 && rank == 0) record_error(err, MOE_ERR_INVALID_ARG);
    if (a < 0 || z < a || z > T) a = z = 0;
  }
  const long long n_ent = (long long)(z - a) * K_r;
  const long long slab = (n_ent + kStatSplit - 1) / kStatSplit;
  const long long x0 = rank * slab, x1 = min(n_ent, x0 + slab);
  const int32_t* src = topk_idx + (size_t)a * K_r;
  for (long long x = x0 + threadIdx.x; x < x1; x += blockDim.x) {
    const int ex = __ldg(src + x);
    if ((unsigned)ex < (unsigned)N_r) atomicAdd(&cnt[ex], 1);
    else record_error(err, MOE_ERR_INVALID_ARG);
  }
  cluster.sync();   // every CTA's histogram is complete and visible to the cluster
  if (rank == 0) {
    const int i = threadIdx.x;
    int c = 0;
    for (int r = 0; r < kStatSplit; ++r) c += cluster.map_shared_rank(cnt, r)[i];
    const int T_j = z - a;
    double v = 0.0;
    if (i < N_r && T_j > 0) {
      const double f = (double)N_r / ((double)K_r * T_j) * (double)c;
      v = f * ((double)seq_p_sum[(size_t)j * N_r + i] / (double)T_j);
    }
    term[i] = v;
    __syncthreads();
    for (int h = 128; h > 0; h >>= 1) {   // fixed pairing: deterministic
      if (threadIdx.x < h) term[threadIdx.x] += term[threadIdx.x + h];
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      stat_per_seq[j] = (float)((double)alpha * term[0]);
      if (stat_mean && n_seq == 1) *stat_mean = (float)((double)alpha * term[0]);   // its own mean
    }
  }
  cluster.sync();   // the peers' histograms stay in place until CTA 0 has read them
}

// Mean over sequences, summed in order in fp64 (one thread: n_seq is small).
__global__ void seq_mean_kernel(const float* __restrict__ stat_per_seq, int n_seq,
                                float* __restrict__ stat_mean) {
  pdl_release();
  pdl_wait();
  double s = 0.0;
  for (int j = 0; j < n_seq; ++j) s += (double)stat_per_seq[j];
  *stat_mean = n_seq > 0 ? (float)(s / n_seq) : 0.f;
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
  const cudaError_t err = launch_pdl(bias_update_kernel, dim3((N_r + 255) / 256), dim3(256), 0, st, 0, b,
                                     load, (long long)T * K_r, N_r, gamma);
  return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_seq_stat(const float* seq_p_sum, const int32_t* topk_idx,
                            const int32_t* seq_offsets, int n_seq, int T, int N_r, int K_r,
                            float alpha, float* stat_per_seq, float* stat_mean,
                            cudaStream_t st) {
  cudaError_t err = launch_pdl(seq_stat_kernel, dim3(n_seq * kStatSplit), dim3(256), 0, st, 0, seq_p_sum,
                               topk_idx, seq_offsets, n_seq, T, N_r, K_r, alpha, stat_per_seq,
                               stat_mean, dev_error_ptr());
  // one sequence: the statistic kernel wrote the mean itself
  if (err == cudaSuccess && stat_mean && n_seq > 1)
    err = launch_pdl(seq_mean_kernel, dim3(1), dim3(1), 0, st, 0, (const float*)stat_per_seq, n_seq, stat_mean);
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace moe
