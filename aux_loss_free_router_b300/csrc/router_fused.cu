// Fused routing for bf16 layers with 64, 128 or 256 experts and K_r <= 8: the affinity
// GEMM z = u e^T on the tensor cores, s = sigmoid(z), the keys s + b, the group limit,
// Top-K_r, the gates and the per-sequence P sums, in one launch (DeepSeek-V3 Technical
// Report reading guide, Method §2: s_{i,t} = Sigmoid(u_t^T e_i), g'_{i,t} from
// TopK({s_{j,t} + b_j}, K_r), gates from the raw s; pwwt.cn notes §1.2: P_i of the
// sequence-wise statistic; §1.3: the group limit).
//
// A cluster of C CTAs (C = 2, 4 or 8) takes 128 tokens.  CTA c forms the fp32 product
// of the 128 tokens with all N_r centroids over the c-th slice of d (single-CTA M=128
// MMAs, TMEM lane = token, column = expert; u and e stream through a 4-stage TMA ring)
// and writes its partial tile to its own shared memory.  After a cluster barrier CTA c
// takes tokens [c*R, (c+1)*R), R = 128/C: one warp per token (lane l: experts l + 32j)
// reads the C partials over distributed shared memory and adds them in slice order (z is
// the same for every C-way split of a given launch shape, and bit-identical run to run),
// then forms s, the keys and the decision with warp reductions (route_warp.cuh).  Each CTA sums s_{i,t}/sum_j s_{j,t} over each
// run of its tokens that lies in one sequence (fp32, token order) and adds the run sum
// to that sequence's accumulator as a 64-bit fixed-point integer (units of 2^-32):
// integer addition is exact and associative, so the totals do not depend on the order
// the CTAs finish in.  The last CTA to finish (a per-launch atomic counter) converts the
// totals to fp32 seq_p_sum.  A batch of at most 128 tokens is one cluster: there CTA 0
// adds the CTAs' run sums over distributed shared memory instead (fp32, token order).
// C is chosen so that the clusters fill the SMs: 2 at 8192 tokens, 8 for decode batches.
#include <algorithm>

#include "launch.h"
#include "route_oct.cuh"
#include "route_warp.cuh"
#include "route_select.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {

namespace {

constexpr int BM = 128, BK = 64, STAGES = 4, THREADS = 256;
constexpr int A_BYTES = BM * BK * 2;

struct FCtrl {
  uint64_t full[STAGES], empty[STAGES], tfull, fin;
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
  int nruns;            // one-cluster launches: runs of one sequence among this CTA's tokens
  int seqid[BM];
  int runseq[BM];       // ... and the sequence of each run
};

// Row stride (floats) of a partial tile in shared memory: N_r + 4 keeps the float4
// stores of the 32 token rows of a warp off each other's banks.
__host__ __device__ constexpr int part_stride(int n_r) { return n_r + 4; }

// Shared memory: the TMA ring during the K loop; afterwards the same space holds the
// partial tile [128][N_r + 4] and the normalised affinities of the CTA's 128/C tokens
// [128/C][N_r].  The control block follows the larger of the two.
__host__ __device__ constexpr size_t fused_ctrl_offset(int n_r, int C) {
  return (size_t)STAGES * (A_BYTES + (size_t)n_r * BK * 2) >
                 (size_t)BM * part_stride(n_r) * 4 + (size_t)(BM / C) * n_r * 4
             ? (size_t)STAGES * (A_BYTES + (size_t)n_r * BK * 2)
             : (size_t)BM * part_stride(n_r) * 4 + (size_t)(BM / C) * n_r * 4;
}

struct FusedArgs {
  RouteOut p;
  const float* b;
  int d, C;
  int one_cluster;               // the launch is one cluster (T <= 128): P sums over DSMEM
  int* done_ctr;                 // zeroed before a launch of more than one cluster
  unsigned long long* p_acc;     // [n_seq, N_r] fixed-point P sums, zeroed with done_ctr
  float* seq_p_sum;              // [n_seq, N_r] or null
  int32_t* err;
};

constexpr double kFix = 4294967296.0;   // 2^32: fixed-point units of the P accumulators

// z[j] = sum over the CC slices, in slice order, of the value at row + 32*j in the
// partial tile of each CTA of the cluster.  The loads of a batch of slices (at most 16
// values) are all issued before the first add.
template <int Q, int CC>
__device__ __forceinline__ void sum_cols(float (&z)[Q], const float* row) {
  constexpr int PER = (16 / Q) < CC ? (16 / Q) : CC;
#pragma unroll
  for (int s0 = 0; s0 < CC; s0 += PER) {
    float w[PER][Q];
#pragma unroll
    for (int bb = 0; bb < PER; ++bb)
#pragma unroll
      for (int j = 0; j < Q; ++j) w[bb][j] = tc::ld_cluster_f32(tc::cluster_addr(row + 32 * j, (uint32_t)(s0 + bb)));
#pragma unroll
    for (int bb = 0; bb < PER; ++bb)
#pragma unroll
      for (int j = 0; j < Q; ++j) z[j] = (s0 + bb == 0) ? w[bb][j] : __fadd_rn(z[j], w[bb][j]);
  }
}

template <int Q, int G>
__global__ void __launch_bounds__(THREADS, 1)
    router_fused_kernel(const __grid_constant__ CUtensorMap mU, const __grid_constant__ CUtensorMap mE,
                        FusedArgs a) {
  constexpr int N = 32 * Q;
  constexpr int LD = part_stride(N);
  extern __shared__ uint8_t smem_raw[];
  pdl_release();
  pdl_wait();
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  constexpr int SBYTES = A_BYTES + N * BK * 2;
  // after the K loop the ring's space holds the partial tile [128][LD] and the
  // normalised affinities of this CTA's tokens [R][N] (P sums)
  float* part = reinterpret_cast<float*>(base);
  float* sp_tile = part + BM * LD;
  FCtrl& F = *reinterpret_cast<FCtrl*>(base + fused_ctrl_offset(N, a.C));

  const RouteOut& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.C;
  const int c = (int)tc::cluster_rank();
  const int tile0 = (blockIdx.x / C) * BM;                 // first token of the cluster
  const int nk = (a.d + BK - 1) / BK;
  const int kb0 = c * nk / C, kb1 = (c + 1) * nk / C;     // this CTA's slice of d (>= 1 block)
  const int R = BM / C;
  const int my0 = tile0 + c * R;                           // this CTA's tokens
  const int ntok = max(0, min(R, p.T - my0));
  const bool want_p = p.pwin != nullptr;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(&F.full[i], 1);
      tc::mbar_init(&F.empty[i], 1);
    }
    tc::mbar_init(&F.tfull, 1);
    tc::mbar_init(&F.fin, 1);
    F.abort_flag = 0;
    F.is_last = 0;
    tc::fence_mbar_init();
  }
  if (want_p && (int)threadIdx.x < ntok) F.seqid[threadIdx.x] = seq_of(my0 + threadIdx.x, p.seq_offsets, p.n_seq);
  if (warp == 1) {
    tc::tmem_alloc(&F.tmem_base, N < 32 ? 32 : N);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = F.tmem_base;
  volatile int* abort_flag = &F.abort_flag;

  // ------------------------------------------------ partial GEMM over this slice --
  if (warp == 0) {
    if (lane == 0) {
      for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
        const int st = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!tc::mbar_wait(&F.empty[st], ph ^ 1, abort_flag, a.err)) break;
        tc::mbar_arrive_expect_tx(&F.full[st], (uint32_t)SBYTES);
        uint8_t* sa = base + st * SBYTES;
        tc::tma_load_2d(sa, &mU, &F.full[st], kb * BK, tile0);
        tc::tma_load_2d(sa + A_BYTES, &mE, &F.full[st], kb * BK, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(BM, N);
      bool ok = true;
      for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
        const int st = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!tc::mbar_wait(&F.full[st], ph, abort_flag, a.err)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t s0 = tc::smem_u32(base + st * SBYTES);
        const uint64_t ad = tc::sdesc_sw128(s0), bd = tc::sdesc_sw128(s0 + A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc::mma_bf16(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (it | kk) != 0);
        tc::mma_commit(&F.empty[st]);
      }
      if (ok) tc::mma_commit(&F.tfull);
      tc::mma_commit(&F.fin);
    }
  } else if (warp >= 4 && warp < 8) {
    // TMEM -> shared memory: lane quarter q = warp - 4 holds tokens 32q .. 32q + 31
    const int q = warp - 4;
    const bool got = tc::mbar_wait(&F.tfull, 0, abort_flag, a.err);
    if (__all_sync(0xffffffffu, got)) {
      tc::fence_after_sync();
      float* row = part + (size_t)(q * 32 + lane) * LD;
#pragma unroll 1
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t z[32];
        tc::tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + c0, z);
        tc::tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 8; ++v)
          *reinterpret_cast<float4*>(row + c0 + 4 * v) =
              make_float4(__uint_as_float(z[4 * v]), __uint_as_float(z[4 * v + 1]),
                          __uint_as_float(z[4 * v + 2]), __uint_as_float(z[4 * v + 3]));
      }
    }
  }
  if (warp == 1 && lane == 0) tc::mbar_drain(&F.fin, 0);   // every MMA has finished
  tc::fence_before_sync();
  __syncthreads();
  // every CTA's partial tile is written and visible to the cluster (every CTA reaches
  // this barrier, also after a timed-out wait)
  tc::cluster_sync();

  // ------------- reduce over the slices, decide, P contributions: a warp per token pair --
  // A warp takes tokens tl and tl + 8 together (two independent reduction chains) and
  // loads the next pair's partials over distributed shared memory while it decides.
  const bool aborted = *abort_flag != 0;
  {
    constexpr int NW = THREADS / 32;
    float bv[Q];
#pragma unroll
    for (int j = 0; j < Q; ++j) bv[j] = __ldg(a.b + lane + 32 * j);
    auto load_pair = [&](int tl0, float (&z)[2][Q]) {
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int tl = min(tl0 + n * NW, max(ntok - 1, 0));          // a spare token re-reads a valid row
        const float* row = part + (size_t)(c * R + tl) * LD + lane;  // row of the partial tiles
        if (C == 2) sum_cols<Q, 2>(z[n], row);
        else if (C == 4) sum_cols<Q, 4>(z[n], row);
        else sum_cols<Q, 8>(z[n], row);
      }
    };
    float z[2][Q];
    if (warp < ntok && !aborted) load_pair(warp, z);
    for (int tl0 = warp; tl0 < ntok && !aborted; tl0 += 2 * NW) {
      float sv[2][Q];
      int tt[2];
      bool ok[2];
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        tt[n] = my0 + tl0 + n * NW;
        ok[n] = tl0 + n * NW < ntok;
#pragma unroll
        for (int j = 0; j < Q; ++j) sv[n][j] = sigmoid_f32(z[n][j]);
      }
      if (tl0 + 2 * NW < ntok) load_pair(tl0 + 2 * NW, z);            // in flight while deciding
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        if (!ok[n]) continue;
        if (p.s_out) {
#pragma unroll
          for (int j = 0; j < Q; ++j) p.s_out[(size_t)tt[n] * N + lane + 32 * j] = sv[n][j];
        }
        if (want_p) {
          float rs = 0.f;
#pragma unroll
          for (int j = 0; j < Q; ++j) rs = __fadd_rn(rs, sv[n][j]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) rs = __fadd_rn(rs, __shfl_xor_sync(0xffffffffu, rs, o));
          const float inv = __frcp_rn(rs);
          const int tl = tl0 + n * NW;
#pragma unroll
          for (int j = 0; j < Q; ++j) sp_tile[(size_t)tl * N + lane + 32 * j] = sv[n][j] * inv;
        }
      }
      warp_decide<Q, G, 2>(sv, bv, tt, ok, p);
    }
  }
  __syncthreads();

  if (a.one_cluster) {
    // One cluster covers the batch: each CTA leaves its run sums in shared memory and
    // CTA 0 adds them per sequence over distributed shared memory, in token order (fp32;
    // no atomics and no scratch to zero).
    if (want_p) {
      if (threadIdx.x == 0) {
        int n = 0;
        for (int r = 0; r < ntok && !aborted; ++r)
          if (r == 0 || F.seqid[r] != F.seqid[r - 1]) F.runseq[n++] = F.seqid[r];
        F.nruns = n;
      }
      if (!aborted) {
        for (int i = threadIdx.x; i < N; i += blockDim.x) {   // run k's sum goes to row k
          float acc = 0.f;
          for (int r = 0, k = 0; r < ntok; ++r) {
            acc = __fadd_rn(acc, sp_tile[(size_t)r * N + i]);
            if (r == ntok - 1 || F.seqid[r + 1] != F.seqid[r]) {
              sp_tile[(size_t)(k++) * N + i] = acc;
              acc = 0.f;
            }
          }
        }
      }
    }
    tc::cluster_sync();   // every CTA's run sums and run list are in place
    if (want_p && c == 0) {
      for (int j = threadIdx.x; j < p.n_seq; j += blockDim.x) {   // offsets 0 <= ... <= T
        const int s0 = p.seq_offsets[j], s1 = p.seq_offsets[j + 1];
        if (s0 < 0 || s1 < s0 || s1 > p.T || (j == 0 && s0 != 0) || (j == p.n_seq - 1 && s1 != p.T))
          record_error(a.err, MOE_ERR_INVALID_ARG);
      }
      for (int i = threadIdx.x; i < N; i += blockDim.x) {
        int j = 0;
        float acc = 0.f;
        for (int src = 0; src < C; ++src) {
          const int nr = tc::ld_cluster_s32(tc::cluster_addr(&F.nruns, (uint32_t)src));
          for (int k = 0; k < nr; ++k) {
            const int sid = tc::ld_cluster_s32(tc::cluster_addr(&F.runseq[k], (uint32_t)src));
            const float v = tc::ld_cluster_f32(tc::cluster_addr(sp_tile + (size_t)k * N + i, (uint32_t)src));
            for (; j < sid && j < p.n_seq; ++j) {
              a.seq_p_sum[(size_t)j * N + i] = acc;
              acc = 0.f;
            }
            acc = __fadd_rn(acc, v);
          }
        }
        for (; j < p.n_seq; ++j) {
          a.seq_p_sum[(size_t)j * N + i] = acc;
          acc = 0.f;
        }
      }
    }
  } else {
    if (want_p && !aborted && ntok > 0) {
      for (int i = threadIdx.x; i < N; i += blockDim.x) {
        float acc = 0.f;
        for (int r = 0; r < ntok; ++r) {
          acc = __fadd_rn(acc, sp_tile[(size_t)r * N + i]);
          if (r == ntok - 1 || F.seqid[r + 1] != F.seqid[r]) {   // end of a run
            const unsigned long long v = (unsigned long long)__double2ll_rn((double)acc * kFix);
            atomicAdd(a.p_acc + (size_t)F.seqid[r] * N + i, v);
            acc = 0.f;
          }
        }
      }
      __threadfence();
    }
    __syncthreads();
    if (want_p) {
      // the last CTA to get here adds the run sums of every sequence
      if (threadIdx.x == 0) {
        __threadfence();
        F.is_last = atomicAdd(a.done_ctr, 1) == (int)gridDim.x - 1;
      }
      __syncthreads();
      if (F.is_last) {
        __threadfence();
        if (threadIdx.x < p.n_seq) {   // offsets that are not 0 <= ... <= T are reported
          const int j = threadIdx.x, s0 = p.seq_offsets[j], s1 = p.seq_offsets[j + 1];
          if (s0 < 0 || s1 < s0 || s1 > p.T || (j == 0 && s0 != 0) || (j == p.n_seq - 1 && s1 != p.T))
            record_error(a.err, MOE_ERR_INVALID_ARG);
        }
        for (int x = threadIdx.x; x < p.n_seq * N; x += blockDim.x)
          a.seq_p_sum[x] = (float)((double)(long long)__ldcg(a.p_acc + x) / kFix);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // a wait that ran out may have left TMA copies in flight: give them time to land
    const uint64_t w0 = global_ns();
    while (global_ns() - w0 < 10000000ull) {
    }
  }
  tc::cluster_sync();   // the peers have read this CTA's partial tile
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, N < 32 ? 32 : N);
  }
}

// CTAs per 128-token tile: the largest power of two from 2 to 8 with the clusters still
// fitting the SMs in one wave (2 when they do not), and no more than d's 64-wide blocks
// (d >= 128, so every CTA gets at least one).
int fused_cluster(int T, int d) {
  const int tiles = (T + BM - 1) / BM;
  const int nk = (d + BK - 1) / BK;
  int C = 2;
  while (C < 8 && (long long)tiles * C * 2 <= device_sm_count() && C * 2 <= nk) C *= 2;
  return C;
}

size_t fused_smem(int n_r, int C) { return fused_ctrl_offset(n_r, C) + sizeof(FCtrl) + 1024; }

}  // namespace

bool router_fused_ok(int N_r, int K_r, int G, int M, int d) {
  return oct_select_ok(N_r, K_r, G, M) && d >= 2 * BK;
}

cudaError_t launch_router_fused(const void* u, const void* e, int d, const float* b,
                                const RouteOut& p, float* seq_p_sum, int* done_ctr,
                                cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  CUtensorMap mU, mE;
  const uint64_t rb = (uint64_t)d * 2;
  if (!make_tmap_2d(&mU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u, d, p.T, rb, BK, BM) ||
      !make_tmap_2d(&mE, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, e, d, p.N_r, rb, BK, p.N_r))
    return cudaErrorInvalidValue;
  const int C = fused_cluster(p.T, d);
  // scratch: the counter, then the fixed-point accumulators, zeroed together
  unsigned long long* p_acc = reinterpret_cast<unsigned long long*>(done_ctr + 64);
  const int one = (p.T + BM - 1) / BM == 1 ? 1 : 0;
  FusedArgs a{p, b, d, C, one, done_ctr, p_acc, seq_p_sum, dev_error_ptr()};
  cudaError_t err = cudaSuccess;
  if (p.pwin && !one)
    err = cudaMemsetAsync(done_ctr, 0, 256 + (size_t)p.n_seq * p.N_r * sizeof(unsigned long long), st);
  if (err != cudaSuccess) return err;
  const size_t smem = fused_smem(p.N_r, C);
  auto go = [&](auto kernel) {
    cudaError_t e2 = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e2 != cudaSuccess) return e2;
    return launch_pdl(kernel, dim3(((p.T + BM - 1) / BM) * C), dim3(THREADS), smem, st, (unsigned)C, mU, mE, a);
  };
  // N_r = 32 Q experts in G groups (G divides Q: router_fused_ok)
  switch (p.N_r * 16 + p.G) {
    case 64 * 16 + 1: err = go(router_fused_kernel<2, 1>); break;
    case 64 * 16 + 2: err = go(router_fused_kernel<2, 2>); break;
    case 128 * 16 + 1: err = go(router_fused_kernel<4, 1>); break;
    case 128 * 16 + 2: err = go(router_fused_kernel<4, 2>); break;
    case 128 * 16 + 4: err = go(router_fused_kernel<4, 4>); break;
    case 256 * 16 + 1: err = go(router_fused_kernel<8, 1>); break;
    case 256 * 16 + 2: err = go(router_fused_kernel<8, 2>); break;
    case 256 * 16 + 4: err = go(router_fused_kernel<8, 4>); break;
    case 256 * 16 + 8: err = go(router_fused_kernel<8, 8>); break;
    default: return cudaErrorInvalidValue;
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace moe
