// Dispatch: whole-batch expert load, stable per-expert token lists and the gather of
// token rows into expert order.  No token is dropped: an expert's segment holds
// anywhere from 0 to T rows (pwwt.cn notes §1.4; szhzxw.cn "无Token丢弃").
//
// The token range is cut into chunks of kDispatchChunk tokens, one warp each.  Batches
// with at most 512 (token, slot) entries per 32nd of the tokens (T <= 2048 at K_r = 8) run
// count, scan and scatter in one CTA (dispatch_small_kernel).
//   count:   per-chunk expert histogram (shared-memory integer atomics: exact),
//            stored expert-major.
//   scan:    one warp per expert: exclusive scan over its chunks; load = the total.
//   scatter: each warp scans load into expert offsets (the first warp publishes
//            them); chunk base = expert offset + the expert's chunk prefix.
//   scatter: each warp walks its chunk's (t, k) entries in order, 32 at a time;
//            __match_any_sync groups equal experts, the rank inside a group is the
//            number of lower lanes with the same expert.  Positions therefore grow
//            with t inside every expert: the order is deterministic and stable.
//   gather:  one warp per token (per column chunk in small batches) reads its row once
//            and writes it to its K_r rows.
// An entry of topk_idx outside [0, N_r) is skipped everywhere (no count, no row, inv_row
// = -1) and MOE_ERR_INVALID_ARG is recorded in the device error word: the caller's
// routing is wrong, and no memory outside the buffers is touched.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "route_select.cuh"

namespace moe {

namespace {

constexpr int kWarps = 4;
// Below this many token warps the gather splits each row into column chunks.
constexpr int kGatherTargetWarps = 2048;

__global__ void __launch_bounds__(kWarps * 32) dispatch_count_kernel(
    const int32_t* __restrict__ topk_idx, int T, int N_r, int K_r, int32_t* __restrict__ counts,
    int32_t* err) {
  extern __shared__ int32_t cnt_sm[];
  pdl_release();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kWarps + warp;
  const int n_chunks = (T + kDispatchChunk - 1) / kDispatchChunk;
  int32_t* cnt = cnt_sm + warp * N_r;
  for (int i = lane; i < N_r; i += 32) cnt[i] = 0;
  __syncwarp();
  if (chunk < n_chunks) {
    const int t0 = chunk * kDispatchChunk;
    const int n_ent = (min(T, t0 + kDispatchChunk) - t0) * K_r;
    const int32_t* src = topk_idx + (size_t)t0 * K_r;
    for (int x = lane; x < n_ent; x += 32) {
      const int ex = src[x];
      if ((unsigned)ex < (unsigned)N_r) atomicAdd(&cnt[ex], 1);
      else record_error(err, MOE_ERR_INVALID_ARG);
    }
    __syncwarp();
    for (int i = lane; i < N_r; i += 32) counts[(size_t)i * n_chunks + chunk] = cnt[i];
  }
}

// One warp per expert: exclusive scan of its chunk counts (expert-major rows, so the
// loads are coalesced) in place; the row total is the expert's load.
__global__ void __launch_bounds__(256) dispatch_scan_kernel(int32_t* __restrict__ counts,
                                                            int n_chunks, int N_r,
                                                            int32_t* __restrict__ load) {
  pdl_release();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= N_r) return;
  int32_t* row = counts + (size_t)i * n_chunks;
  int carry = 0;
  for (int c0 = 0; c0 < n_chunks; c0 += 32) {
    const int c = c0 + lane;
    const int v = c < n_chunks ? row[c] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (c < n_chunks) row[c] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) load[i] = carry;
}

// Exclusive scan of load over the N_r experts by one warp (each lane a contiguous span);
// result in shared memory, and in expert_offset when `out` is set.
__device__ __forceinline__ void expert_offsets(const int32_t* __restrict__ load, int N_r,
                                               int32_t* off_sm, int32_t* out) {
  const int lane = threadIdx.x & 31;
  const int span = (N_r + 31) / 32;
  int local = 0;
  for (int q = 0; q < span; ++q) {
    const int i = lane * span + q;
    if (i < N_r) local += load[i];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  int run = incl - local;
  for (int q = 0; q < span; ++q) {
    const int i = lane * span + q;
    if (i < N_r) {
      off_sm[i] = run;
      if (out) out[i] = run;
      run += load[i];
    }
  }
  if (out && lane == 31) out[N_r] = incl;
}

__global__ void __launch_bounds__(kWarps * 32) dispatch_scatter_kernel(
    const int32_t* __restrict__ topk_idx, int T, int N_r, int K_r,
    const int32_t* __restrict__ chunk_prefix, const int32_t* __restrict__ load,
    int32_t* __restrict__ expert_offset, int32_t* __restrict__ perm_token,
    int32_t* __restrict__ inv_row) {
  extern __shared__ int32_t run_sm[];
  pdl_release();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kWarps + warp;
  const int n_chunks = (T + kDispatchChunk - 1) / kDispatchChunk;
  if (chunk >= n_chunks) return;
  int32_t* run = run_sm + warp * N_r;
  // every warp derives the expert offsets itself; the first one also publishes them
  expert_offsets(load, N_r, run, chunk == 0 ? expert_offset : nullptr);
  __syncwarp();
  for (int i = lane; i < N_r; i += 32) run[i] += chunk_prefix[(size_t)i * n_chunks + chunk];
  __syncwarp();
  const int t0 = chunk * kDispatchChunk;
  const int n_ent = (min(T, t0 + kDispatchChunk) - t0) * K_r;
  const size_t e0 = (size_t)t0 * K_r;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < n_ent; base += 32) {
    const int x = base + lane;
    const bool in_range = x < n_ent;
    const int ex = in_range ? topk_idx[e0 + x] : -1;
    const bool valid = in_range && (unsigned)ex < (unsigned)N_r;
    if (in_range && !valid) inv_row[e0 + x] = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, ex);
    const int rank = __popc(peers & lt_mask);
    int pos = 0;
    if (valid) pos = run[ex] + rank;
    __syncwarp();
    if (valid && rank == 0) run[ex] += __popc(peers);
    __syncwarp();
    if (valid) {
      perm_token[pos] = (int32_t)((e0 + x) / K_r);
      inv_row[e0 + x] = pos;
    }
  }
}

// Small batches: count, scan and scatter in one CTA of 32 warps.  Warp w takes the w-th
// of 32 contiguous token chunks of ceil(T/32) tokens and loads its (token, slot) entries
// once, kSmallPerLane per lane, into registers; the chunk counts live in shared memory.
// The positions do not depend on the chunking (experts in order, tokens ascending within
// each expert): they are those of the three-kernel path.
constexpr int kSmallWarps = 32;
constexpr int kSmallPerLane = 16;   // entries per warp <= 32 * 16 = 512 (e.g. T = 2048, K_r = 8)

__host__ __device__ inline bool dispatch_small_ok(int T, int K_r) {
  return (long long)((T + kSmallWarps - 1) / kSmallWarps) * K_r <= 32 * kSmallPerLane;
}

__global__ void __launch_bounds__(kSmallWarps * 32) dispatch_small_kernel(
    const int32_t* __restrict__ topk_idx, int T, int N_r, int K_r, int32_t* __restrict__ load,
    int32_t* __restrict__ expert_offset, int32_t* __restrict__ perm_token,
    int32_t* __restrict__ inv_row, int32_t* err) {
  extern __shared__ int32_t cnt[];            // [kSmallWarps][N_r], then off [N_r]
  pdl_release();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* off = cnt + kSmallWarps * N_r;
  for (int i = threadIdx.x; i < kSmallWarps * N_r; i += blockDim.x) cnt[i] = 0;
  const int ct = (T + kSmallWarps - 1) / kSmallWarps;
  const int t0 = min(T, warp * ct), t1 = min(T, t0 + ct);
  const int n_ent = (t1 - t0) * K_r;                 // the same for every lane of the warp
  const size_t e0 = (size_t)t0 * K_r;
  pdl_wait();
  int ex[kSmallPerLane];
#pragma unroll
  for (int j = 0; j < kSmallPerLane; ++j) {
    const int x = j * 32 + lane;
    ex[j] = x < n_ent ? topk_idx[e0 + x] : -1;
  }
  __syncthreads();                                   // counts zeroed
#pragma unroll
  for (int j = 0; j < kSmallPerLane; ++j) {
    if (j * 32 + lane < n_ent) {
      if ((unsigned)ex[j] < (unsigned)N_r) atomicAdd(&cnt[warp * N_r + ex[j]], 1);
      else record_error(err, MOE_ERR_INVALID_ARG);
    }
  }
  __syncthreads();
  // per expert: exclusive scan over the chunks, the total is the load
  for (int i = threadIdx.x; i < N_r; i += blockDim.x) {
    int run = 0;
    for (int c = 0; c < kSmallWarps; ++c) {
      const int v = cnt[c * N_r + i];
      cnt[c * N_r + i] = run;
      run += v;
    }
    load[i] = run;
    off[i] = run;
  }
  __syncthreads();
  if (warp == 0) {    // exclusive scan of the loads over the experts
    const int span = (N_r + 31) / 32;
    int local = 0;
    for (int q = 0; q < span; ++q) {
      const int i = lane * span + q;
      if (i < N_r) local += off[i];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - local;
    for (int q = 0; q < span; ++q) {
      const int i = lane * span + q;
      if (i < N_r) {
        const int v = off[i];
        off[i] = run;
        expert_offset[i] = run;
        run += v;
      }
    }
    if (lane == 31) expert_offset[N_r] = incl;
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  int32_t* run = cnt + warp * N_r;                   // this chunk's next position per expert
  for (int i = lane; i < N_r; i += 32) run[i] += off[i];
  __syncwarp();
#pragma unroll
  for (int j = 0; j < kSmallPerLane; ++j) {
    if (j * 32 >= n_ent) break;                      // warp-uniform
    const int x = j * 32 + lane;
    const bool in_range = x < n_ent;
    const int e = in_range ? ex[j] : -1;
    const bool valid = in_range && (unsigned)e < (unsigned)N_r;
    if (in_range && !valid) inv_row[e0 + x] = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    int pos = 0;
    if (valid) pos = run[e] + rank;
    __syncwarp();
    if (valid && rank == 0) run[e] += __popc(peers);
    __syncwarp();
    if (valid) {
      perm_token[pos] = (int32_t)((e0 + x) / K_r);
      inv_row[e0 + x] = pos;
    }
  }
}

// 16-byte vector copy of each token's row to its K_r destination rows: one warp per
// token and column chunk (small batches split each row over gridDim.y so that enough
// warps have loads in flight); the chunk of blockIdx.y == 0 also copies the scales.
__global__ void __launch_bounds__(256) dispatch_gather_kernel(
    const uint8_t* __restrict__ u, size_t row_bytes, const float* __restrict__ u_scale,
    int scale_cols, const int32_t* __restrict__ inv_row, int T, int K_r, int pass_per_chunk,
    uint8_t* __restrict__ x_perm, float* __restrict__ x_perm_scale) {
  pdl_release();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  const int my_row = lane < K_r ? inv_row[(size_t)t * K_r + lane] : 0;
  const uint4* src = reinterpret_cast<const uint4*>(u + (size_t)t * row_bytes);
  const size_t nvec = row_bytes / 16;
  const size_t v_begin = (size_t)blockIdx.y * pass_per_chunk * 32;
  const size_t v_stop = v_begin + (size_t)pass_per_chunk * 32;
  const size_t v_end = v_stop < nvec ? v_stop : nvec;
  // Every lane runs every iteration so that the shuffles below see the full warp.
  for (size_t v0 = v_begin; v0 < v_end; v0 += 32) {
    const size_t v = v0 + lane;
    const bool ok = v < v_end;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (ok) val = __ldg(src + v);
    for (int k = 0; k < K_r; ++k) {
      const int r = __shfl_sync(0xffffffffu, my_row, k);
      if (ok && r >= 0) reinterpret_cast<uint4*>(x_perm + (size_t)r * row_bytes)[v] = val;
    }
  }
  if (u_scale && blockIdx.y == 0) {
    for (int c0 = 0; c0 < scale_cols; c0 += 32) {
      const int c = c0 + lane;
      const bool ok = c < scale_cols;
      const float sc = ok ? u_scale[(size_t)t * scale_cols + c] : 0.f;
      for (int k = 0; k < K_r; ++k) {
        const int r = __shfl_sync(0xffffffffu, my_row, k);
        if (ok && r >= 0) x_perm_scale[(size_t)r * scale_cols + c] = sc;
      }
    }
  }
}

}  // namespace

cudaError_t launch_dispatch(const int32_t* topk_idx, int T, int N_r, int K_r,
                            const void* u, size_t row_bytes, const float* u_scale,
                            int scale_cols, int32_t* load, int32_t* expert_offset,
                            int32_t* perm_token, int32_t* inv_row, void* x_perm,
                            float* x_perm_scale, int32_t* ws_counts, cudaStream_t st) {
  const int n_chunks = (T + kDispatchChunk - 1) / kDispatchChunk;
  if (n_chunks == 0) {
    cudaError_t err = cudaMemsetAsync(load, 0, sizeof(int32_t) * N_r, st);
    if (err == cudaSuccess) err = cudaMemsetAsync(expert_offset, 0, sizeof(int32_t) * (N_r + 1), st);
    return err;
  }
  if (dispatch_small_ok(T, K_r)) {
    // one launch for count, scan and scatter; at most 33 x 256 counts of shared memory
    const cudaError_t err = launch_pdl(dispatch_small_kernel, dim3(1), dim3(kSmallWarps * 32),
                                       sizeof(int32_t) * (size_t)(kSmallWarps + 1) * N_r, st, 0, topk_idx,
                                       T, N_r, K_r, load, expert_offset, perm_token, inv_row, dev_error_ptr());
    if (err != cudaSuccess) return err;
  } else {
    const int blocks = (n_chunks + kWarps - 1) / kWarps;
    const size_t smem = sizeof(int32_t) * kWarps * N_r;
    cudaError_t err = launch_pdl(dispatch_count_kernel, dim3(blocks), dim3(kWarps * 32), smem, st, 0,
                                 topk_idx, T, N_r, K_r, ws_counts, dev_error_ptr());
    if (err == cudaSuccess)
      err = launch_pdl(dispatch_scan_kernel, dim3((N_r + 7) / 8), dim3(256), 0, st, 0, ws_counts,
                       n_chunks, N_r, load);
    if (err == cudaSuccess)
      err = launch_pdl(dispatch_scatter_kernel, dim3(blocks), dim3(kWarps * 32), smem, st, 0, topk_idx,
                       T, N_r, K_r, (const int32_t*)ws_counts, (const int32_t*)load, expert_offset,
                       perm_token, inv_row);
    if (err != cudaSuccess) return err;
  }
  if (u && x_perm) {
    const int passes = (int)((row_bytes / 16 + 31) / 32);   // 512-byte passes of a warp
    const int chunks = std::min(passes, std::max(1, kGatherTargetWarps / T));
    const int ppc = (passes + chunks - 1) / chunks;
    const dim3 grid((T + 7) / 8, (passes + ppc - 1) / ppc);
    const cudaError_t err = launch_pdl(dispatch_gather_kernel, grid, dim3(256), 0, st, 0, (const uint8_t*)u,
                                       row_bytes, u_scale, scale_cols, (const int32_t*)inv_row, T, K_r,
                                       ppc, (uint8_t*)x_perm, x_perm_scale);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------ built-in chunk-count scratch ---
//
// moe_dispatch_noalloc runs the same kernels with their per-chunk expert counts in this
// file-scope device array instead of a caller workspace.  It is sized for
// kDispatchStaticCounts int32 entries (2 MiB): ceil(T/32) * N_r must not exceed it,
// e.g. T <= 65536 tokens with 256 experts.  Every GPU that loads the library keeps it
// until the process exits.
static __device__ __align__(256) int32_t g_dispatch_counts[kDispatchStaticCounts];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_counts_mu;
int32_t* g_counts_addr[kMaxDevices] = {};
}  // namespace

// Device address of g_dispatch_counts on the current device.  In host code the array's
// name only stands in for the symbol, so it is looked up with cudaGetSymbolAddress once
// per device, with that device current, and cached.
cudaError_t dispatch_static_counts(int32_t** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_counts_mu);
  if (g_counts_addr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_dispatch_counts);
    if (err != cudaSuccess) return err;
    g_counts_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_counts_addr[dev];
  return cudaSuccess;
}

}  // namespace moe
