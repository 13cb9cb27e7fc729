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
//
// With 256 experts and at least 2048 tokens the product is formed by CTA pairs instead
// (cta_group::2 MMAs of M = 256 tokens): a cluster of C CTAs takes 256 tokens, its C/2
// pairs split d, and in each pair the even CTA holds tokens 0..127 of the product and the
// odd one tokens 128..255, each loading its own 128 token rows and half of the centroid
// rows per K step.  An SM then takes in a third less per K step (the centroid slice is
// the larger part of a single CTA's intake).  The decisions are as above, over the C/2
// partial tiles that hold a token; 16 warps decide.
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
// pair launches: CTA pairs multiply 256 tokens at a time, each CTA taking in half of the
// centroids per K step, through a deeper ring; 16 warps decide
constexpr int PSTAGES = 6, PTHREADS = 512;
constexpr int A_BYTES = BM * BK * 2;

struct FCtrl {
  uint64_t full[PSTAGES], empty[PSTAGES], tfull, fin;
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
  int nruns;            // one-cluster launches: runs of one sequence among this CTA's tokens
  int seqid[BM];
  int runseq[BM];       // ... and the sequence of each run
  float psh[2][256];    // P sums of one run: the two halves of the tokens, per expert
};

// Row stride (floats) of a partial tile in shared memory: N_r + 4 keeps the float4
// stores of the 32 token rows of a warp off each other's banks.
__host__ __device__ constexpr int part_stride(int n_r) { return n_r + 4; }

// Shared memory: the TMA ring during the K loop; afterwards the same space holds the
// partial tile [128][N_r + 4] and the normalised affinities of the CTA's 128/KS tokens
// [128/KS][N_r] (KS: the K slices of a cluster, C for single-CTA launches and C/2 for
// pair launches).  The control block follows the larger of the two.
__host__ __device__ constexpr size_t fused_ring_bytes(int n_r, bool pair) {
  return (size_t)(pair ? PSTAGES : STAGES) * (A_BYTES + (size_t)(pair ? n_r / 2 : n_r) * BK * 2);
}
__host__ __device__ constexpr size_t fused_ctrl_offset(int n_r, int C, bool pair) {
  return fused_ring_bytes(n_r, pair) >
                 (size_t)BM * part_stride(n_r) * 4 + (size_t)(BM / (pair ? C / 2 : C)) * n_r * 4
             ? fused_ring_bytes(n_r, pair)
             : (size_t)BM * part_stride(n_r) * 4 + (size_t)(BM / (pair ? C / 2 : C)) * n_r * 4;
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
// partial tile of slice s's CTA, cluster rank s*RS + hf.  The loads of a batch of slices
// (at most 16 values) are all issued before the first add.
template <int Q, int CC, int RS>
__device__ __forceinline__ void sum_cols(float (&z)[Q], const float* row, int hf) {
  constexpr int PER = (16 / Q) < CC ? (16 / Q) : CC;
#pragma unroll
  for (int s0 = 0; s0 < CC; s0 += PER) {
    float w[PER][Q];
#pragma unroll
    for (int bb = 0; bb < PER; ++bb)
#pragma unroll
      for (int j = 0; j < Q; ++j)
        w[bb][j] = tc::ld_cluster_f32(tc::cluster_addr(row + 32 * j, (uint32_t)((s0 + bb) * RS + hf)));
#pragma unroll
    for (int bb = 0; bb < PER; ++bb)
#pragma unroll
      for (int j = 0; j < Q; ++j) z[j] = (s0 + bb == 0) ? w[bb][j] : __fadd_rn(z[j], w[bb][j]);
  }
}

template <int Q, int G, bool PAIR>
__global__ void __launch_bounds__(PAIR ? PTHREADS : THREADS, 1)
    router_fused_kernel(const __grid_constant__ CUtensorMap mU, const __grid_constant__ CUtensorMap mE,
                        FusedArgs a) {
  constexpr int N = 32 * Q;
  constexpr int LD = part_stride(N);
  constexpr int STG = PAIR ? PSTAGES : STAGES;
  constexpr int NTHR = PAIR ? PTHREADS : THREADS;
  constexpr int NB = PAIR ? N / 2 : N;                 // centroid rows this CTA loads
  extern __shared__ uint8_t smem_raw[];
  pdl_release();
  pdl_wait();
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  constexpr int SBYTES = A_BYTES + NB * BK * 2;
  // after the K loop the ring's space holds the partial tile [128][LD] and the
  // normalised affinities of this CTA's tokens [R][N] (P sums)
  float* part = reinterpret_cast<float*>(base);
  float* sp_tile = part + BM * LD;
  FCtrl& F = *reinterpret_cast<FCtrl*>(base + fused_ctrl_offset(N, a.C, PAIR));

  const RouteOut& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.C;
  const int c = (int)tc::cluster_rank();
  // A single-CTA launch: the cluster's C CTAs each multiply the cluster's 128 tokens
  // over one slice of d.  A pair launch: the cluster's C/2 CTA pairs each multiply its
  // 256 tokens over one slice of d; the even CTA of a pair holds the first 128 tokens of
  // the product, the odd one the next 128.
  const int KS = PAIR ? C / 2 : C;                          // slices of d
  const int ks = PAIR ? c >> 1 : c;                         // this CTA's slice
  const int hf = PAIR ? c & 1 : 0;                          // this CTA's half of a pair tile
  const int tile0 = (blockIdx.x / C) * (PAIR ? 2 * BM : BM);  // first token of the cluster
  const int row0 = tile0 + hf * BM;                         // this CTA's 128 product rows
  const int nk = (a.d + BK - 1) / BK;
  const int kb0 = ks * nk / KS, kb1 = (ks + 1) * nk / KS;   // this CTA's slice of d (>= 1 block)
  const int R = BM / KS;
  const int my0 = row0 + ks * R;                            // the tokens this CTA decides
  const int ntok = max(0, min(R, p.T - my0));
  const bool want_p = p.pwin != nullptr;
  const bool leader = !PAIR || hf == 0;                     // issues the MMAs
  const uint16_t pmask = (uint16_t)(3u << (2 * ks));        // PAIR: the pair's two ranks

  if (threadIdx.x == 0) {
    for (int i = 0; i < STG; ++i) {
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
    if constexpr (PAIR) {
      tc::tmem_alloc_pair(&F.tmem_base, N < 32 ? 32 : N);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(&F.tmem_base, N < 32 ? 32 : N);
      tc::tmem_relinquish();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // pairs: both CTAs' barriers exist before a copy or a commit reaches the peer's
  if constexpr (PAIR) tc::cluster_sync();
  const uint32_t tmem_base = F.tmem_base;
  volatile int* abort_flag = &F.abort_flag;

  // ------------------------------------------------ partial GEMM over this slice --
  if (warp == 0) {
    if (lane == 0) {
      for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
        const int st = it % STG;
        const uint32_t ph = (it / STG) & 1;
        if (!tc::mbar_wait(&F.empty[st], ph ^ 1, abort_flag, a.err)) break;
        uint8_t* sa = base + st * SBYTES;
        if constexpr (PAIR) {
          // both CTAs' copies complete on the even CTA's barrier
          const uint32_t bar = tc::cluster_addr(&F.full[st], (uint32_t)(c & ~1));
          if (leader) tc::mbar_arrive_expect_tx(&F.full[st], (uint32_t)(2 * SBYTES));
          tc::tma_load_2d_pair(sa, &mU, bar, kb * BK, row0);
          tc::tma_load_2d_pair(sa + A_BYTES, &mE, bar, kb * BK, hf * NB);
        } else {
          tc::mbar_arrive_expect_tx(&F.full[st], (uint32_t)SBYTES);
          tc::tma_load_2d(sa, &mU, &F.full[st], kb * BK, tile0);
          tc::tma_load_2d(sa + A_BYTES, &mE, &F.full[st], kb * BK, 0);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      const uint32_t idesc = tc::idesc_bf16(PAIR ? 2 * BM : BM, N);
      bool ok = true;
      for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
        const int st = it % STG;
        const uint32_t ph = (it / STG) & 1;
        if (!tc::mbar_wait(&F.full[st], ph, abort_flag, a.err)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t s0 = tc::smem_u32(base + st * SBYTES);
        const uint64_t ad = tc::sdesc_sw128(s0), bd = tc::sdesc_sw128(s0 + A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          if constexpr (PAIR) tc::mma_bf16_pair(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (it | kk) != 0);
          else tc::mma_bf16(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (it | kk) != 0);
        }
        if constexpr (PAIR) tc::mma_commit_pair_mask(&F.empty[st], pmask);
        else tc::mma_commit(&F.empty[st]);
      }
      if constexpr (PAIR) {
        if (ok) tc::mma_commit_pair_mask(&F.tfull, pmask);
        tc::mma_commit_pair_mask(&F.fin, pmask);
      } else {
        if (ok) tc::mma_commit(&F.tfull);
        tc::mma_commit(&F.fin);
      }
    }
  } else if (warp >= 4 && warp < (PAIR ? 12 : 8)) {
    // TMEM -> shared memory: lane quarter q = warp & 3 holds tokens 32q .. 32q + 31;
    // pair launches split the columns over two warps per quarter
    const int q = warp & 3;
    constexpr int CW = PAIR ? N / 2 : N;                  // columns per drain warp
    const int cbeg = PAIR ? ((warp - 4) >> 2) * CW : 0;
    const bool got = tc::mbar_wait(&F.tfull, 0, abort_flag, a.err);
    if (__all_sync(0xffffffffu, got)) {
      tc::fence_after_sync();
      float* row = part + (size_t)(q * 32 + lane) * LD;
#pragma unroll 1
      for (int c0 = cbeg; c0 < cbeg + CW; c0 += 32) {
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
    constexpr int NW = NTHR / 32;
    float bv[Q];
#pragma unroll
    for (int j = 0; j < Q; ++j) bv[j] = __ldg(a.b + lane + 32 * j);
    auto load_pair = [&](int tl0, float (&z)[2][Q]) {
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int tl = min(tl0 + n * NW, max(ntok - 1, 0));          // a spare token re-reads a valid row
        const float* row = part + (size_t)(ks * R + tl) * LD + lane;  // row of the partial tiles
        if constexpr (PAIR) {
          if (KS == 1) sum_cols<Q, 1, 2>(z[n], row, hf);
          else if (KS == 2) sum_cols<Q, 2, 2>(z[n], row, hf);
          else sum_cols<Q, 4, 2>(z[n], row, hf);
        } else {
          if (C == 2) sum_cols<Q, 2, 1>(z[n], row, 0);
          else if (C == 4) sum_cols<Q, 4, 1>(z[n], row, 0);
          else sum_cols<Q, 8, 1>(z[n], row, 0);
        }
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

  if (!PAIR && a.one_cluster) {
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
      if (F.seqid[0] == F.seqid[ntok - 1]) {
        // the CTA's tokens lie in one sequence (the usual case): with two threads per
        // expert, each adds a fixed half of the tokens in order, and the halves are added
        // in order before the one fixed-point update
        const int SH = (int)blockDim.x >= 2 * N ? 2 : 1;
        const int half = (ntok + SH - 1) / SH;
        if ((int)threadIdx.x < SH * N) {
          const int i = (int)threadIdx.x % N, h = (int)threadIdx.x / N;
          const int r1 = min(ntok, (h + 1) * half);
          int r = h * half;
          float acc = 0.f;
          for (; r + 8 <= r1; r += 8) {
            float v[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) v[x] = sp_tile[(size_t)(r + x) * N + i];
#pragma unroll
            for (int x = 0; x < 8; ++x) acc = __fadd_rn(acc, v[x]);
          }
          for (; r < r1; ++r) acc = __fadd_rn(acc, sp_tile[(size_t)r * N + i]);
          F.psh[h][i] = acc;
        }
        __syncthreads();
        if ((int)threadIdx.x < N) {
          const int i = (int)threadIdx.x;
          const float acc = SH == 2 ? __fadd_rn(F.psh[0][i], F.psh[1][i]) : F.psh[0][i];
          const unsigned long long v = (unsigned long long)__double2ll_rn((double)acc * kFix);
          atomicAdd(a.p_acc + (size_t)F.seqid[0] * N + i, v);
        }
      } else {
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
    if constexpr (PAIR) tc::tmem_dealloc_pair(tmem_base, N < 32 ? 32 : N);
    else tc::tmem_dealloc(tmem_base, N < 32 ? 32 : N);
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

// Pair launches, for 256 experts, d >= 256 and batches of at least kPairMinTokens (the
// centroid slice is then two thirds of what a single CTA takes in per K step; with 64
// experts the pairs measured slower): C/2 pairs per 256-token tile, C/2 a power of two
// from 2 to 4, the largest with the clusters still fitting the SMs in one wave and no more
// slices than d's 64-wide blocks.  At least two slices: a CTA then decides at most 64
// tokens, whose normalised affinities fit beside the partial tile in shared memory.
constexpr int kPairMinTokens = 2048;
bool fused_pair_ok(int T, int d, int N_r) { return T >= kPairMinTokens && N_r == 256 && d >= 4 * BK; }
int fused_cluster_pair(int T, int d) {
  const int tiles = (T + 2 * BM - 1) / (2 * BM);
  const int nk = (d + BK - 1) / BK;
  int KS = 2;
  while (KS < 4 && (long long)tiles * 2 * KS * 2 <= device_sm_count() && KS * 2 <= nk) KS *= 2;
  return 2 * KS;
}

size_t fused_smem(int n_r, int C, bool pair) {
  return fused_ctrl_offset(n_r, C, pair) + sizeof(FCtrl) + 1024;
}

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
  // large batches: CTA pairs (each CTA loads half of the centroid rows per K step)
  const bool pair = fused_pair_ok(p.T, d, p.N_r);
  if (!make_tmap_2d(&mU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u, d, p.T, rb, BK, BM) ||
      !make_tmap_2d(&mE, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, e, d, p.N_r, rb, BK, pair ? p.N_r / 2 : p.N_r))
    return cudaErrorInvalidValue;
  const int C = pair ? fused_cluster_pair(p.T, d) : fused_cluster(p.T, d);
  // scratch: the counter, then the fixed-point accumulators, zeroed together
  unsigned long long* p_acc = reinterpret_cast<unsigned long long*>(done_ctr + 64);
  const int tile = pair ? 2 * BM : BM;
  const int one = (p.T + tile - 1) / tile == 1 ? 1 : 0;   // never for pair launches
  FusedArgs a{p, b, d, C, one, done_ctr, p_acc, seq_p_sum, dev_error_ptr()};
  cudaError_t err = cudaSuccess;
  if (p.pwin && !one)
    err = cudaMemsetAsync(done_ctr, 0, 256 + (size_t)p.n_seq * p.N_r * sizeof(unsigned long long), st);
  if (err != cudaSuccess) return err;
  const size_t smem = fused_smem(p.N_r, C, pair);
  const dim3 grid(((p.T + tile - 1) / tile) * C);
  auto go = [&](auto single, auto paired) {
    auto run = [&](auto kernel, int threads) {
      cudaError_t e2 = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e2 != cudaSuccess) return e2;
      return launch_pdl(kernel, grid, dim3(threads), smem, st, (unsigned)C, mU, mE, a);
    };
    return pair ? run(paired, PTHREADS) : run(single, THREADS);
  };
  // N_r = 32 Q experts in G groups (G divides Q: router_fused_ok)
#define MOE_RF(Q, G) go(router_fused_kernel<Q, G, false>, router_fused_kernel<Q, G, true>)
  switch (p.N_r * 16 + p.G) {
    case 64 * 16 + 1: err = MOE_RF(2, 1); break;
    case 64 * 16 + 2: err = MOE_RF(2, 2); break;
    case 128 * 16 + 1: err = MOE_RF(4, 1); break;
    case 128 * 16 + 2: err = MOE_RF(4, 2); break;
    case 128 * 16 + 4: err = MOE_RF(4, 4); break;
    case 256 * 16 + 1: err = MOE_RF(8, 1); break;
    case 256 * 16 + 2: err = MOE_RF(8, 2); break;
    case 256 * 16 + 4: err = MOE_RF(8, 4); break;
    case 256 * 16 + 8: err = MOE_RF(8, 8); break;
    default: return cudaErrorInvalidValue;
  }
#undef MOE_RF
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace moe
