// Router pieces on CUDA cores: the affinity GEMM for fp32 layers, the routing
// decision kernel shared by every layer dtype (sigmoid, bias, group limit, Top-K_r,
// gates; DeepSeek-V3 Technical Report reading guide, Method §2), and the
// deterministic per-sequence reduction of the normalised affinities.
#include "launch.h"
#include "route_oct.cuh"
#include "route_select.cuh"

namespace moe {

namespace {

constexpr int kTok = 32;   // tokens per block
// Reduction chunk of the SIMT affinity GEMM for JN accumulators per thread: wide
// chunks (fewer load round trips) while the centroid tile stays small.
template <int JN> constexpr int simt_kc() { return JN <= 4 ? 128 : (JN <= 8 ? 64 : 32); }

// z = u e^T on CUDA cores (fp32 layers, or shapes the tensor-core GEMM does not
// take): 32 tokens x N_r centroids per block, fp32 FMA over chunks of d.  Thread
// (ty, tx) owns token ty and centroids tx + 8j, j < JN (JN >= N_r / 8).
template <typename TIn, int JN, int kKc = simt_kc<JN>()>
__global__ void __launch_bounds__(256) router_gemm_simt_kernel(const TIn* __restrict__ u,
                                                               const TIn* __restrict__ e,
                                                               int T, int d, int N_r,
                                                               float* __restrict__ z) {
  extern __shared__ float sm[];
  float* u_tile = sm;                          // [kTok][kKc+1]
  float* e_tile = u_tile + kTok * (kKc + 1);   // [N_r][kKc+1]
  pdl_release();
  pdl_wait();
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kTok;
  const int ty = tid >> 3, tx = tid & 7;
  float acc[JN];
#pragma unroll
  for (int j = 0; j < JN; ++j) acc[j] = 0.f;
  // per chunk a thread loads UL token and up to EL centroid elements, all of them into
  // registers before any shared-memory store, so the loads are in flight together
  constexpr int UL = kTok * kKc / 256, EL = 8 * JN * kKc / 256;
  for (int k0 = 0; k0 < d; k0 += kKc) {
    float ru[UL], re[EL];
#pragma unroll
    for (int q = 0; q < UL; ++q) {
      const int x = tid + 256 * q, r = x / kKc, c = x % kKc, t = t0 + r, k = k0 + c;
      ru[q] = (t < T && k < d) ? to_f32(u[(size_t)t * d + k]) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < EL; ++q) {
      const int x = tid + 256 * q, r = x / kKc, c = x % kKc, k = k0 + c;
      re[q] = (r < N_r && k < d) ? to_f32(e[(size_t)r * d + k]) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < UL; ++q) {
      const int x = tid + 256 * q;
      u_tile[(x / kKc) * (kKc + 1) + x % kKc] = ru[q];
    }
#pragma unroll
    for (int q = 0; q < EL; ++q) {
      const int x = tid + 256 * q;
      if (x / kKc < N_r) e_tile[(x / kKc) * (kKc + 1) + x % kKc] = re[q];
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kKc; ++c) {
      const float uv = u_tile[ty * (kKc + 1) + c];
#pragma unroll
      for (int j = 0; j < JN; ++j) {
        const int i = tx + 8 * j;
        if (i < N_r) acc[j] = fmaf(uv, e_tile[i * (kKc + 1) + c], acc[j]);
      }
    }
    __syncthreads();
  }
  const int t = t0 + ty;
  if (t < T) {
#pragma unroll
    for (int j = 0; j < JN; ++j) {
      const int i = tx + 8 * j;
      if (i < N_r) z[(size_t)t * N_r + i] = acc[j];
    }
  }
}

// The routing decision for 32 tokens per block (eight warps), for the shapes the
// warp-per-token kernel below does not take: z = the fixed-order fp32 sum of the S
// split-K partials, s = sigmoid(z) into shared memory (the block's 256 threads over
// the tile's token x expert entries), then either one thread per token (select_row,
// warp 0) or one warp per token (route_token, warp w takes tokens w, w+8, ...); s is
// written out when asked for, and the block's P-sum window runs.
constexpr int kSelWarps = 8;
__global__ void __launch_bounds__(kSelWarps * 32) router_select_kernel(
    const float* __restrict__ z_part, int S, const float* __restrict__ b, RouteOut p, int fast) {
  static_assert(kTok == kPWindow, "one block covers one P-sum window");
  __shared__ float s_tile[kTok * (kMaxExperts + 1)];
  __shared__ float b_sm[kMaxExperts];
  __shared__ float rs_sm[kTok];
  __shared__ int seqid[kTok];
  pdl_release();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int N_r = p.N_r, T = p.T, stride = N_r + 1;
  const int t0 = blockIdx.x * kTok;
  const int ntok = min(kTok, T - t0);
  for (int i = threadIdx.x; i < N_r; i += blockDim.x) b_sm[i] = b[i];
  if (p.pwin && (int)threadIdx.x < ntok)
    seqid[threadIdx.x] = seq_of(t0 + threadIdx.x, p.seq_offsets, p.n_seq);
  for (int x = threadIdx.x; x < ntok * N_r; x += blockDim.x) {
    const int r = x / N_r, i = x - r * N_r, t = t0 + r;
    float z = z_part[(size_t)t * N_r + i];
    for (int sp = 1; sp < S; ++sp) z = __fadd_rn(z, z_part[((size_t)sp * T + t) * N_r + i]);
    s_tile[r * stride + i] = sigmoid_f32(z);
  }
  __syncthreads();
  if (!fast) {
    for (int r = warp; r < ntok; r += kSelWarps) {
      route_token(s_tile + r * stride, b_sm, t0 + r, p);
      if (p.pwin) {
        float part = 0.f;
        for (int i = lane; i < N_r; i += 32) part = __fadd_rn(part, s_tile[r * stride + i]);
        const float rs = warp_sum(part);
        if (lane == 0) rs_sm[r] = rs;
      }
    }
  } else if (warp == 0) {
    const int t = t0 + lane;
    float rowsum = 0.f;
    if (t < T) {
      const float* row = s_tile + lane * stride;
      float c1[kMaxSlots], c2[kMaxSlots];
#pragma unroll
      for (int c = 0; c < kMaxSlots; ++c) {
        c1[c] = c2[c] = -CUDART_INF_F;
        if (c < N_r / 32) {
#pragma unroll 8
          for (int j = 0; j < 32; ++j) {
            const int i = c * 32 + j;
            const float sv = row[i];
            rowsum = __fadd_rn(rowsum, sv);
            const float k = __fadd_rn(sv, b_sm[i]);
            c2[c] = fmaxf(c2[c], fminf(c1[c], k));
            c1[c] = fmaxf(c1[c], k);
          }
        }
      }
      select_row(row, b_sm, c1, c2, t, p);
    }
    rs_sm[lane] = rowsum;
  }
  __syncthreads();
  if (p.s_out) {
    for (int x = threadIdx.x; x < ntok * N_r; x += blockDim.x) {
      const int r = x / N_r, i = x - r * N_r;
      p.s_out[(size_t)(t0 + r) * N_r + i] = s_tile[r * stride + i];
    }
  }
  if (p.pwin) {
    for (int i = threadIdx.x; i < N_r; i += blockDim.x)
      window_runs([&](int r) { return __fdiv_rn(s_tile[r * stride + i], rs_sm[r]); }, seqid, ntok,
                  t0, N_r, i, p.pwin);
  }
}

// The routing decision with one warp per token, for N_r = 32*E experts: lane l holds
// experts [l*E, l*E + E).  With the group limit a group is 32/G whole lanes, so a
// group's two best keys merge in log2(32/G) shuffle steps; Top-K_r takes K_r rounds
// of a warp-wide (key, index) argmax.  A block covers one P-sum window of 32 tokens
// (8 warps x 4 tokens); the normalised affinities go through shared memory to the
// window's per-sequence run sums.
// E consecutive floats (16-byte vectors when E is a multiple of 4; the rows are
// 16-byte aligned then).
template <int E>
__device__ __forceinline__ void load_row(const float* __restrict__ src, float (&v)[E]) {
  if constexpr (E % 4 == 0) {
#pragma unroll
    for (int q = 0; q < E / 4; ++q) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(src) + q);
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) v[j] = __ldg(src + j);
  }
}

template <int E>
__device__ __forceinline__ void store_row(float* dst, const float (&v)[E]) {
  if constexpr (E % 4 == 0) {
#pragma unroll
    for (int q = 0; q < E / 4; ++q)
      reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) dst[j] = v[j];
  }
}

template <int E>
__global__ void __launch_bounds__(256, 2) router_select_warp_kernel(const float* __restrict__ z_part,
                                                                 int S, const float* __restrict__ b,
                                                                 RouteOut p) {
  constexpr int WARPS = 8, TPW = kPWindow / WARPS, N = 32 * E;
  __shared__ __align__(16) float sp_tile[kPWindow][N];
  __shared__ int seqid[kPWindow];
  pdl_release();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T, t0 = blockIdx.x * kPWindow;
  const int ntok = min(kPWindow, T - t0);
  const bool want_p = p.pwin != nullptr;
  if (want_p && (int)threadIdx.x < ntok) seqid[threadIdx.x] = seq_of(t0 + threadIdx.x, p.seq_offsets, p.n_seq);
  float bl[E];
#pragma unroll
  for (int j = 0; j < E; ++j) bl[j] = __ldg(b + lane * E + j);
  const int G = p.G, lpg = 32 / G, my_group = lane / lpg;
  const int kg = p.K_r / p.M;

  for (int r = 0; r < TPW; ++r) {
    const int tl = warp * TPW + r, t = t0 + tl;
    if (tl >= ntok) break;                       // warp-uniform
    float z[E];
    const float* zp = z_part + (size_t)t * N + lane * E;
    load_row<E>(zp, z);
    for (int sp = 1; sp < S; ++sp) {
      float zs[E];
      load_row<E>(zp + (size_t)sp * T * N, zs);
#pragma unroll
      for (int j = 0; j < E; ++j) z[j] = __fadd_rn(z[j], zs[j]);
    }
    float sv[E], key[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
      sv[j] = sigmoid_f32(z[j]);
      key[j] = __fadd_rn(sv[j], bl[j]);           // one fp32 rounding
    }
    if (p.s_out) store_row<E>(p.s_out + (size_t)t * N + lane * E, sv);
    if (want_p) {
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < E; ++j) part = __fadd_rn(part, sv[j]);
      const float rs = warp_sum(part);
      float spv[E];
#pragma unroll
      for (int j = 0; j < E; ++j) spv[j] = __fdiv_rn(sv[j], rs);
      store_row<E>(&sp_tile[tl][lane * E], spv);
    }

    if (G > 1) {
      // the group's kg <= 2 best keys (values only: ties do not change the sum)
      float t1 = -CUDART_INF_F, t2 = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const float lo = fminf(t1, key[j]);
        t1 = fmaxf(t1, key[j]);
        t2 = fmaxf(t2, lo);
      }
      for (int o = 1; o < lpg; o <<= 1) {
        const float a1 = __shfl_xor_sync(0xffffffffu, t1, o);
        const float a2 = __shfl_xor_sync(0xffffffffu, t2, o);
        const float lo = fminf(t1, a1);
        t1 = fmaxf(t1, a1);
        t2 = fmaxf(fmaxf(t2, a2), lo);
      }
      const float gs = kg == 1 ? t1 : __fadd_rn(t1, t2);   // descending order
      int rank = 0;                                          // groups ranked above mine
      for (int g = 0; g < G; ++g) {
        const float o = __shfl_sync(0xffffffffu, gs, g * lpg);
        rank += (o > gs || (o == gs && g < my_group)) ? 1 : 0;
      }
      if (rank >= p.M) {
#pragma unroll
        for (int j = 0; j < E; ++j) key[j] = -CUDART_INF_F;
      }
    }

    // Top-K_r: the lane's best entry (lowest index among equal keys), then K_r rounds
    // of the warp argmax; only the winning lane recomputes its best.
    float bk = -CUDART_INF_F;
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < E; ++j)
      if (key[j] > bk) { bk = key[j]; bi = lane * E + j; }
    int my_idx = 0;
    for (int k = 0; k < p.K_r; ++k) {
      float wk = bk;
      int wi = bi;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float k2 = __shfl_xor_sync(0xffffffffu, wk, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, wi, o);
        if (better(k2, i2, wk, wi)) { wk = k2; wi = i2; }
      }
      if (lane == k) my_idx = wi;
      if (wi == bi) {                 // this lane's entry was taken
        bk = -CUDART_INF_F;
        bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < E; ++j) {
          if (lane * E + j == wi) key[j] = -CUDART_INF_F;
          else if (key[j] > bk) { bk = key[j]; bi = lane * E + j; }
        }
      }
    }
    // raw s of the selected experts, gates normalised over them in selection order
    const int owner = my_idx / E, slot = my_idx - owner * E;
    float my_s = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const float v = __shfl_sync(0xffffffffu, sv[j], owner);
      if (slot == j) my_s = v;
    }
    float total = 0.f;
    for (int k = 0; k < p.K_r; ++k) total = __fadd_rn(total, __shfl_sync(0xffffffffu, my_s, k));
    if (lane < p.K_r) {
      p.topk_idx[(size_t)t * p.K_r + lane] = my_idx;
      p.topk_gate[(size_t)t * p.K_r + lane] = __fdiv_rn(my_s, total);
    }
  }
  if (want_p) {
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x)
      window_runs([&](int r) { return sp_tile[r][i]; }, seqid, ntok, t0, N, i, p.pwin);
  }
}

// The routing decision with eight threads per token, for N_r = 32*Q experts: thread p
// of a token holds experts 32q + 4p .. 32q + 4p + 3 of every 32-expert block q (16-byte
// loads; a warp load covers 64 contiguous bytes of each of its 4 tokens).  With the
// group limit a group is bq = Q/G whole blocks: each block's two best keys come from the
// thread's four and three shuffle steps over the token's eight threads.  Each thread
// then keeps the top 8 of its eligible experts and three merge steps give all eight
// threads the token's top 8.  A block covers one P-sum window of 32 tokens (8 warps x
// 4 tokens).
template <int Q>
__global__ void __launch_bounds__(256, 2) router_select_oct_kernel(const float* __restrict__ z_part,
                                                                int S, const float* __restrict__ b,
                                                                RouteOut p) {
  constexpr int N = 32 * Q;
  __shared__ __align__(16) float sp_tile[kPWindow][N];
  __shared__ int seqid[kPWindow];
  pdl_release();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T, t0 = blockIdx.x * kPWindow;
  const int ntok = min(kPWindow, T - t0);
  const int tl = warp * 4 + (lane >> 3), part = lane & 7;
  const int t = t0 + tl;
  const bool valid = tl < ntok;
  const bool want_p = p.pwin != nullptr;
  if (want_p && (int)threadIdx.x < ntok)
    seqid[threadIdx.x] = seq_of(t0 + threadIdx.x, p.seq_offsets, p.n_seq);

  float sv[Q][4], bv[Q][4];
  // z = the split-K partials added in split order; the loads of PB splits (8 float4 per
  // thread) are issued before their adds, so a small batch with many splits waits for
  // a few load round trips, not one per split
  constexpr int PB = Q >= 8 ? 1 : 8 / Q;
  float4 z[Q];
  const float* zp = z_part + (size_t)t * N + 4 * part;
  const size_t split_stride = (size_t)T * N;
#pragma unroll
  for (int q = 0; q < Q; ++q)
    z[q] = valid ? __ldg(reinterpret_cast<const float4*>(zp + 32 * q)) : make_float4(0.f, 0.f, 0.f, 0.f);
  if (valid) {
    for (int sp0 = 1; sp0 < S; sp0 += PB) {
      float4 w[PB][Q];
#pragma unroll
      for (int j = 0; j < PB; ++j)
#pragma unroll
        for (int q = 0; q < Q; ++q)
          if (sp0 + j < S)
            w[j][q] = __ldg(reinterpret_cast<const float4*>(zp + (size_t)(sp0 + j) * split_stride + 32 * q));
#pragma unroll
      for (int j = 0; j < PB; ++j)
#pragma unroll
        for (int q = 0; q < Q; ++q)
          if (sp0 + j < S) {
            z[q].x = __fadd_rn(z[q].x, w[j][q].x); z[q].y = __fadd_rn(z[q].y, w[j][q].y);
            z[q].z = __fadd_rn(z[q].z, w[j][q].z); z[q].w = __fadd_rn(z[q].w, w[j][q].w);
          }
    }
  }
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const float4 bb = __ldg(reinterpret_cast<const float4*>(b + 32 * q + 4 * part));
    bv[q][0] = bb.x; bv[q][1] = bb.y; bv[q][2] = bb.z; bv[q][3] = bb.w;
    sv[q][0] = sigmoid_f32(z[q].x); sv[q][1] = sigmoid_f32(z[q].y);
    sv[q][2] = sigmoid_f32(z[q].z); sv[q][3] = sigmoid_f32(z[q].w);
  }
  if (valid && p.s_out) {
#pragma unroll
    for (int q = 0; q < Q; ++q)
      *reinterpret_cast<float4*>(p.s_out + (size_t)t * N + 32 * q + 4 * part) =
          make_float4(sv[q][0], sv[q][1], sv[q][2], sv[q][3]);
  }
  if (want_p) {
    float rs = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) rs = __fadd_rn(rs, sv[q][j]);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) rs = __fadd_rn(rs, __shfl_xor_sync(0xffffffffu, rs, o));
    if (valid) {
      const float inv = __frcp_rn(rs);
#pragma unroll
      for (int q = 0; q < Q; ++q)
        *reinterpret_cast<float4*>(&sp_tile[tl][32 * q + 4 * part]) =
            make_float4(sv[q][0] * inv, sv[q][1] * inv, sv[q][2] * inv, sv[q][3] * inv);
    }
  }

  oct_decide<Q>(sv, bv, part, t, valid, p);
  if (want_p) {
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x)
      window_runs([&](int r) { return sp_tile[r][i]; }, seqid, ntok, t0, N, i, p.pwin);
  }
}

// Whether router_select_warp_kernel takes the shape: 32, 64, 128 or 256 experts and,
// with the group limit, groups of whole lanes (G divides 32) keeping K_r/M <= 2 keys.
inline bool warp_select_ok(int N_r, int K_r, int G, int M) {
  if (N_r != 32 && N_r != 64 && N_r != 128 && N_r != 256) return false;
  if (G == 1) return true;
  return 32 % G == 0 && K_r / M <= 2;
}

// out[j, i] = sum over the P-sum windows' run sums of sequence j: the run starting at
// the sequence's first token and one at every window start inside the sequence.  A
// block takes one sequence and 32 experts (lane = expert); its 8 warps take every 8th
// run, accumulate in fp64, and the 8 partial sums are added in warp order.  Offsets
// that are not 0 = off[0] <= ... <= off[n_seq] = T record MOE_ERR_INVALID_ARG; a
// sequence whose own bounds are out of order or outside [0, T] is summed as empty.
__global__ void __launch_bounds__(256) seq_psum_kernel(const float* __restrict__ pwin,
                                                       const int32_t* __restrict__ seq_offsets,
                                                       int n_seq, int T, int N_r,
                                                       float* __restrict__ out, int32_t* err) {
  __shared__ double part[8][32];
  pdl_release();
  pdl_wait();
  const int j = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.y * 32 + lane;
  int a = seq_offsets[j], z = seq_offsets[j + 1];
  const bool bad = a < 0 || z < a || z > T || (j == 0 && a != 0) || (j == n_seq - 1 && z != T);
  if (bad) {
    if (threadIdx.x == 0 && blockIdx.y == 0) record_error(err, MOE_ERR_INVALID_ARG);
    if (a < 0 || z < a || z > T) a = z = 0;
  }
  double acc = 0.0;
  if (i < N_r && a < z) {
    // run r = 0 starts at a; run r >= 1 at the r-th window start after a
    const int w1 = (a / kPWindow + 1) * kPWindow;
    const int n_runs = 1 + (z > w1 ? (z - w1 + kPWindow - 1) / kPWindow : 0);
    for (int r = warp; r < n_runs; r += 8) {
      const int t = r == 0 ? a : w1 + (r - 1) * kPWindow;
      acc += (double)__ldg(pwin + (size_t)t * N_r + i);
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && i < N_r) {
    double s = 0.0;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += part[w][lane];
    out[(size_t)j * N_r + i] = (float)s;
  }
}

}  // namespace

cudaError_t launch_router_gemm_simt(const void* u, const void* e, moe_dtype dt, int T, int d,
                                    int N_r, float* z, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((T + kTok - 1) / kTok);
  // accumulators per thread: N_r / 8 rounded up to a power of two
  int jn = 1;
  while (jn * 8 < N_r) jn <<= 1;
  auto smem = [&](int kc) { return sizeof(float) * (size_t)(kTok + N_r) * (kc + 1); };
  cudaError_t err;
#define MOE_SIMT_GEMM(TIN, JN)                                                                   \
  err = launch_pdl(router_gemm_simt_kernel<TIN, JN>, grid, dim3(256), smem(simt_kc<JN>()), st, 0, \
                   (const TIN*)u, (const TIN*)e, T, d, N_r, z)
  if (dt == MOE_F32) {
    switch (jn) {
      case 1: MOE_SIMT_GEMM(float, 1); break;
      case 2: MOE_SIMT_GEMM(float, 2); break;
      case 4: MOE_SIMT_GEMM(float, 4); break;
      case 8: MOE_SIMT_GEMM(float, 8); break;
      case 16: MOE_SIMT_GEMM(float, 16); break;
      default: MOE_SIMT_GEMM(float, 32); break;
    }
  } else {
    switch (jn) {
      case 1: MOE_SIMT_GEMM(__nv_bfloat16, 1); break;
      case 2: MOE_SIMT_GEMM(__nv_bfloat16, 2); break;
      case 4: MOE_SIMT_GEMM(__nv_bfloat16, 4); break;
      case 8: MOE_SIMT_GEMM(__nv_bfloat16, 8); break;
      case 16: MOE_SIMT_GEMM(__nv_bfloat16, 16); break;
      default: MOE_SIMT_GEMM(__nv_bfloat16, 32); break;
    }
  }
#undef MOE_SIMT_GEMM
  return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_router_select(const float* z_part, int S, const float* b, const RouteOut& p,
                                 cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  const dim3 blocks((p.T + kPWindow - 1) / kPWindow);
  auto go = [&](auto kernel) { return launch_pdl(kernel, blocks, dim3(256), 0, st, 0, z_part, S, b, p); };
  cudaError_t err;
  if (oct_select_ok(p.N_r, p.K_r, p.G, p.M)) {
    switch (p.N_r) {
      case 64: err = go(router_select_oct_kernel<2>); break;
      case 128: err = go(router_select_oct_kernel<4>); break;
      default: err = go(router_select_oct_kernel<8>); break;
    }
  } else if (warp_select_ok(p.N_r, p.K_r, p.G, p.M)) {
    switch (p.N_r) {
      case 32: err = go(router_select_warp_kernel<1>); break;
      case 64: err = go(router_select_warp_kernel<2>); break;
      case 128: err = go(router_select_warp_kernel<4>); break;
      default: err = go(router_select_warp_kernel<8>); break;
    }
  } else {
    const int fast = fast_select_ok(p.N_r, p.K_r, p.G, p.M) ? 1 : 0;
    err = launch_pdl(router_select_kernel, blocks, dim3(kSelWarps * 32), 0, st, 0, z_part, S, b, p, fast);
  }
  return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_seq_psum(const float* pwin, const int32_t* seq_offsets, int n_seq, int T,
                            int N_r, float* out, cudaStream_t st) {
  if (n_seq == 0) return cudaSuccess;
  const dim3 grid(n_seq, (N_r + 31) / 32);
  const cudaError_t err = launch_pdl(seq_psum_kernel, grid, dim3(256), 0, st, 0, pwin, seq_offsets, n_seq,
                                     T, N_r, out, dev_error_ptr());
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace moe
