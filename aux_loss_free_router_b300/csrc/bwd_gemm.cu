// Backward-pass GEMMs of the layer on the sm_103a tensor cores (tcgen05 MMAs over TMEM,
// fed by TMA), at the forward pass's selection.  The pages define the forward pass only
// (DeepSeek-V3 Technical Report reading guide, Method §2: h'_t = u_t + shared FFNs +
// sum_k g_{k,t} FFN_k(u_t), s = Sigmoid(u e^T)); the gradients are those of that
// function, with the selection held fixed (pwwt.cn notes §1.1.3: the bias is moved by
// the sign rule, not learned).  With dY the gradient of an expert's output rows:
//
//   kDH    dH  = dY W_down, and in the epilogue dA = dH * c * silu'(a), dC = dH * silu(a)
//          (a = x W_gate^T, c = x W_up^T: the SwiGLU pre-activations)
//   kDX    dX  = dA W_gate + dC W_up
//   kDWD   dW_down[e] = sum over the expert's rows of dY^T h
//   kDWGU  dW_gate[e] = dA^T x, dW_up[e] = dC^T x
//   kDUR   du (router part) = dz e           (dz: gradient of the affinity logits)
//   kDE    de = dz^T u
//
// One persistent kernel template serves all six: single-CTA M=128 x N=256 tiles (a tile
// of token rows sizes N to its tokens in steps of 16), K steps of 64 through a 4-stage
// TMA ring of 48 KB, two 256-column TMEM accumulators (the epilogue of a tile overlaps
// the next tile's MMAs), tiles handed out round-robin.  An SM takes in 48 KB per
// 128 x 256 x 64 MACs.  Each
// operand is read in place, K-major or MN-major (shared-memory descriptor: 128-byte
// swizzle; for MN-major the leading byte offset is the stride between 64-element chunks
// of M or N and the stride byte offset the stride between 8-row groups of K), so no
// weight or activation is transposed in memory.  Where K runs over an expert's token
// rows (kDWD, kDWGU), the rows of the last K step that belong to the next segment are
// zeroed in shared memory before the MMAs read them.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "ffn_sched.cuh"
#include "launch.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moe {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4, THREADS = 192;
constexpr int OPA = BM * BK * 2;           // A of a K step: 16 KB
constexpr int OPB = BN * BK * 2;           // B of a K step: 32 KB
constexpr int STAGE = OPA + OPB;
constexpr int TMEM_COLS = 512, ACC = 256;
constexpr int SCR = 32 * 32 * 4;           // per epilogue warp: 32 x 32 fp32 (the store box)

enum : int { kDH = 0, kDX = 1, kDWD = 2, kDWGU = 3, kDUR = 4, kDE = 5 };

template <int KIND> struct Traits {
  static constexpr bool A_MN = KIND != kDUR;                         // A is MN-major
  static constexpr bool B_MN = KIND == kDWD || KIND == kDWGU || KIND == kDUR || KIND == kDE;
  static constexpr bool ROW_K = KIND == kDWD || KIND == kDWGU;        // K = a segment's rows
  static constexpr bool TRANSPOSED = KIND == kDH || KIND == kDX;      // out rows = tokens = N
};

struct BCtrl {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], fin;
  uint32_t tmem_base;
  int abort_flag;
  SegTable tab;
};

constexpr size_t kSmemBytes = (size_t)STAGES * STAGE + 4 * SCR + sizeof(BCtrl) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

struct BwdArgs {
  int T, d, I, N_r, K_r, N_s;
  const int32_t* expert_offset;
  const __nv_bfloat16* a;     // kDH: pre-activations [R, I]
  const __nv_bfloat16* c;
  __nv_bfloat16* o_bf0;       // kDH: dA [R, I]; kDX: dX [R, d]
  __nv_bfloat16* o_bf1;       // kDH: dC [R, I]
  float* o_f0;                // kDWD: dW_down; kDWGU: dW_gate; kDUR: du [T, d]; kDE: de [N_r, d]
  float* o_f1;                // kDWGU: dW_up
  float* o_fs0;               // kDWD / kDWGU: the shared experts' dW_down / dW_gate
  float* o_fs1;               // kDWGU: the shared experts' dW_up
  int32_t* err;
  int mn3d = 0;               // MN-major maps are 3-D: one copy per operand per K step
};

// One output tile: M index = TMEM lane, N index = accumulator column.
struct BTile {
  int seg;          // expert segment (routed < N_r, shared >= N_r), or -1
  int part;         // kDWGU: 0 gate, 1 up
  int m0, n0;       // origin of the tile in the output's M and N
  int nk;           // K steps (0: the output tile is zero)
  int kv_last;      // kinds with ROW_K: rows of the last K step inside the segment
  int a_row0;       // first K row of A (ROW_K) / first token row of the tile (TRANSPOSED)
  int b_row0;       // first K row of B (ROW_K)
  int n_tok;        // TRANSPOSED: tokens of the tile
};

template <int KIND>
__device__ __forceinline__ int tile_count(const SegTable& tab, const BwdArgs& g) {
  const int segs = g.N_r + g.N_s;
  if (KIND == kDH || KIND == kDX) return tab.total;
  if (KIND == kDWD) return segs * ((g.d + BM - 1) / BM) * ((g.I + BN - 1) / BN);
  if (KIND == kDWGU) return 2 * segs * ((g.I + BM - 1) / BM) * ((g.d + BN - 1) / BN);
  if (KIND == kDUR) return ((g.T + BM - 1) / BM) * ((g.d + BN - 1) / BN);
  return ((g.N_r + BM - 1) / BM) * ((g.d + BN - 1) / BN);   // kDE
}

template <int KIND>
__device__ __forceinline__ BTile decode(const SegTable& tab, const BwdArgs& g, int tile) {
  BTile b;
  b.seg = -1;
  b.part = 0;
  b.kv_last = BK;
  b.a_row0 = b.b_row0 = 0;
  b.n_tok = 0;
  if (KIND == kDH || KIND == kDX) {
    const int mt = KIND == kDH ? (g.I + BM - 1) / BM : (g.d + BM - 1) / BM;
    const TileCoord t = decode_tile(tab, tile, mt);
    b.seg = t.seg;
    b.m0 = t.n * BM;                        // features of the output row
    b.n0 = 0;
    b.a_row0 = t.out_row0 + t.tok0;         // token rows in the FFN row space
    b.n_tok = t.n_tok;
    b.nk = KIND == kDH ? (g.d + BK - 1) / BK : 2 * ((g.I + BK - 1) / BK);
    return b;
  }
  if (KIND == kDWD || KIND == kDWGU) {
    const int segs = g.N_r + g.N_s;
    const int Mx = KIND == kDWD ? g.d : g.I, Nx = KIND == kDWD ? g.I : g.d;
    const int mt = (Mx + BM - 1) / BM, nt = (Nx + BN - 1) / BN;
    int t = tile;
    if (KIND == kDWGU) {
      b.part = t / (segs * mt * nt);
      t -= b.part * segs * mt * nt;
    }
    b.seg = t / (mt * nt);
    t -= b.seg * mt * nt;
    b.m0 = (t / nt) * BM;
    b.n0 = (t % nt) * BN;
    const bool shared = b.seg >= g.N_r;
    const int rows = tab.rows[b.seg];
    b.a_row0 = shared ? g.T * g.K_r + (b.seg - g.N_r) * g.T : tab.row0[b.seg];
    b.b_row0 = (KIND == kDWGU && shared) ? 0 : b.a_row0;   // x rows: x_perm or u
    b.nk = (rows + BK - 1) / BK;
    b.kv_last = rows - (b.nk - 1) * BK;
    return b;
  }
  const int nt = (g.d + BN - 1) / BN;
  b.m0 = (tile / nt) * BM;
  b.n0 = (tile % nt) * BN;
  b.nk = KIND == kDUR ? (g.N_r + BK - 1) / BK : (g.T + BK - 1) / BK;
  return b;
}

// Shared-memory descriptors of one operand: K-major (128-byte rows of K) or MN-major
// (64-element chunks of M or N, 8 KB apart, each with 64 rows of K).
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) { return tc::sdesc_sw128(saddr); }
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(8192 >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Advance a descriptor by 16 rows of K: 32 bytes (K-major) or 2048 bytes (MN-major).
template <bool MN> __device__ __forceinline__ uint64_t desc_k16(uint64_t d, int kk) {
  return d + (uint64_t)(MN ? 128 * kk : 2 * kk);
}

__host__ __device__ constexpr uint32_t idesc(bool a_mn, bool b_mn, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// Loads of one operand of ROWS rows (M or N): MN-major -> ROWS/64 boxes of (64, 64) at
// x, x + 64, ...; K-major -> one (64, ROWS) box.
template <bool MN, int ROWS>
__device__ __forceinline__ void load_op(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int x_mn,
                                        int k_or_row, bool mn3d) {
  if (MN && mn3d) {
    tc::tma_load_3d(dst, m, bar, 0, k_or_row, x_mn / 64);   // ROWS/64 chunks in one copy
  } else if (MN) {
#pragma unroll
    for (int c = 0; c < ROWS / 64; ++c) tc::tma_load_2d(dst + c * 8192, m, bar, x_mn + 64 * c, k_or_row);
  } else {
    tc::tma_load_2d(dst, m, bar, k_or_row, x_mn);
  }
}

__device__ __forceinline__ float sigm(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

// m0..m5 per kind:
//   kDH:   m0 W_down routed  [N_r*d, I] MN   m1 W_down shared  m4 dY [R, d] K
//   kDX:   m0 W_gate routed  [N_r*I, d] MN   m1 W_up routed    m2 W_gate shared
//          m3 W_up shared    m4 dA [R, I] K  m5 dC [R, I] K
//   kDWD:  m0 dY [R, d] MN   m4 h [R, I] MN
//   kDWGU: m0 dA [R, I] MN   m1 dC [R, I] MN m4 x_perm [T*K_r, d] MN   m5 u [T, d] MN
//   kDUR:  m0 dz [T, N_r] K  m4 e [N_r, d] MN
//   kDE:   m0 dz [T, N_r] MN m4 u [T, d] MN
template <int KIND>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_gemm_kernel(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
                    const __grid_constant__ CUtensorMap m2, const __grid_constant__ CUtensorMap m3,
                    const __grid_constant__ CUtensorMap m4, const __grid_constant__ CUtensorMap m5,
                    const __grid_constant__ CUtensorMap o0, const __grid_constant__ CUtensorMap o1,
                    const __grid_constant__ CUtensorMap o2, const __grid_constant__ CUtensorMap o3,
                    BwdArgs g) {
  using Tr = Traits<KIND>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_off = tc::smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_off & 1023u)) & 1023u);
  float* scr_all = reinterpret_cast<float*>(base + STAGES * STAGE);
  BCtrl& C = *reinterpret_cast<BCtrl*>(base + STAGES * STAGE + 4 * SCR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(&C.full[i], 1);
      tc::mbar_init(&C.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&C.tfull[i], 1);
      tc::mbar_init(&C.tempty[i], 4);
    }
    tc::mbar_init(&C.fin, 1);
    C.abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&C.tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (KIND == kDH || KIND == kDX) {
    const int mt = KIND == kDH ? (g.I + BM - 1) / BM : (g.d + BM - 1) / BM;
    build_seg_table(C.tab, g.expert_offset, g.T, g.K_r, g.N_r, g.N_s, BN, mt, true, g.err);
  } else if (KIND == kDWD || KIND == kDWGU) {
    build_seg_table(C.tab, g.expert_offset, g.T, g.K_r, g.N_r, g.N_s, 1 << 30, 1, false, g.err);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = C.tmem_base;
  volatile int* abort_flag = &C.abort_flag;
  const int total = tile_count<KIND>(C.tab, g);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer --
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const BTile b = decode<KIND>(C.tab, g, tile);
        const bool sh = b.seg >= g.N_r;
        const int e = sh ? b.seg - g.N_r : b.seg;
        for (int ks = 0; ks < b.nk; ++ks, ++it) {
          const int st = it % STAGES;
          if (!tc::mbar_wait(&C.empty[st], ((it / STAGES) & 1) ^ 1, abort_flag, g.err)) { ok = false; break; }
          uint64_t* bar = &C.full[st];
          tc::mbar_arrive_expect_tx(bar, STAGE);
          uint8_t* sa = base + st * STAGE;
          uint8_t* sb = sa + OPA;
          if (KIND == kDH) {
            load_op<true, BM>(sa, sh ? &m1 : &m0, bar, b.m0, e * g.d + ks * BK, g.mn3d != 0);
            load_op<false, BN>(sb, &m4, bar, b.a_row0, ks * BK, g.mn3d != 0);
          } else if (KIND == kDX) {
            const int nkI = b.nk / 2, ph = ks >= nkI, kk = ks - ph * nkI;
            const CUtensorMap* ma = ph ? (sh ? &m3 : &m1) : (sh ? &m2 : &m0);
            load_op<true, BM>(sa, ma, bar, b.m0, e * g.I + kk * BK, g.mn3d != 0);
            load_op<false, BN>(sb, ph ? &m5 : &m4, bar, b.a_row0, kk * BK, g.mn3d != 0);
          } else if (KIND == kDWD) {
            load_op<true, BM>(sa, &m0, bar, b.m0, b.a_row0 + ks * BK, g.mn3d != 0);
            load_op<true, BN>(sb, &m4, bar, b.n0, b.b_row0 + ks * BK, g.mn3d != 0);
          } else if (KIND == kDWGU) {
            load_op<true, BM>(sa, b.part ? &m1 : &m0, bar, b.m0, b.a_row0 + ks * BK, g.mn3d != 0);
            load_op<true, BN>(sb, sh ? &m5 : &m4, bar, b.n0, b.b_row0 + ks * BK, g.mn3d != 0);
          } else if (KIND == kDUR) {
            load_op<false, BM>(sa, &m0, bar, b.m0, ks * BK, g.mn3d != 0);
            load_op<true, BN>(sb, &m4, bar, b.n0, ks * BK, g.mn3d != 0);
          } else {
            load_op<true, BM>(sa, &m0, bar, b.m0, ks * BK, g.mn3d != 0);
            load_op<true, BN>(sb, &m4, bar, b.n0, ks * BK, g.mn3d != 0);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer --
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++tcount) {
        const BTile b = decode<KIND>(C.tab, g, tile);
        // token tiles: N sized to the tile's tokens in steps of 16
        const uint32_t id = idesc(Tr::A_MN, Tr::B_MN, Tr::TRANSPOSED ? (b.n_tok + 15) & ~15 : BN);
        const int acc = tcount & 1;
        if (!tc::mbar_wait(&C.tempty[acc], ((tcount >> 1) & 1) ^ 1, abort_flag, g.err)) break;
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC);
        for (int ks = 0; ks < b.nk; ++ks, ++it) {
          const int st = it % STAGES;
          if (!tc::mbar_wait(&C.full[st], (it / STAGES) & 1, abort_flag, g.err)) { ok = false; break; }
          tc::fence_after_sync();
          uint8_t* sa = base + st * STAGE;
          int k16 = BK / 16;
          if (Tr::ROW_K && ks == b.nk - 1 && b.kv_last < BK) {
            // rows kv_last .. (next multiple of 16) - 1 hold the next segment's rows: zero
            // them (whole 128-byte rows, so the swizzle does not matter) in all six 8 KB
            // chunks of the stage (two of A, four of B)
            const int kv = b.kv_last, kend = (kv + 15) & ~15;
            for (int ch = 0; ch < STAGE / 8192; ++ch)
              for (int r = kv; r < kend; ++r) {
                uint4* row = reinterpret_cast<uint4*>(sa + ch * 8192 + r * 128);
#pragma unroll
                for (int v = 0; v < 8; ++v) row[v] = make_uint4(0, 0, 0, 0);
              }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            k16 = kend / 16;
          }
          const uint32_t s0 = tc::smem_u32(sa);
          const uint64_t ad = Tr::A_MN ? desc_mn(s0) : desc_k(s0);
          const uint64_t bd = Tr::B_MN ? desc_mn(s0 + OPA) : desc_k(s0 + OPA);
          for (int kk = 0; kk < k16; ++kk)
            tc::mma_bf16(d_tmem, desc_k16<Tr::A_MN>(ad, kk), desc_k16<Tr::B_MN>(bd, kk), id,
                         (ks | kk) != 0);
          tc::mma_commit(&C.empty[st]);
        }
        if (!ok) break;
        tc::mma_commit(&C.tfull[acc]);   // with no K steps it arrives at once
      }
      tc::mma_commit(&C.fin);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;
    float* scr = scr_all + q * (SCR / 4);
    int tcount = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++tcount) {
      const BTile b = decode<KIND>(C.tab, g, tile);
      const int acc = tcount & 1;
      const bool got = tc::mbar_wait(&C.tfull[acc], (tcount >> 1) & 1, abort_flag, g.err);
      if (!__all_sync(0xffffffffu, got)) break;
      tc::fence_after_sync();
      const uint32_t t_base = tmem_base + (uint32_t)(acc * ACC) + ((uint32_t)(q * 32) << 16);
      if (Tr::TRANSPOSED) {
        // lane = feature m0 + 32q + lane, column = token; out rows are tokens
        const int Fx = KIND == kDH ? g.I : g.d;
        if (KIND == kDH) {
          // bring the next tile's pre-activations into L2 while this tile is written
          const int nt = tile + gridDim.x;
          if (nt < total) {
            const BTile nb = decode<KIND>(C.tab, g, nt);
            const int f0 = nb.m0 + q * 32;
            if (f0 < Fx)
              for (int r = lane; r < nb.n_tok; r += 32) {
                const size_t o = (size_t)(nb.a_row0 + r) * Fx + f0;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(g.a + o));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(g.c + o));
              }
          }
        }
        // a and c of a 16-token group are loaded one group ahead of their use
        uint4 pa[2], pc[2];
        auto fetch = [&](int j0) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int item = i * 32 + lane, tok = item >> 2, piece = item & 3;
            const int f = b.m0 + q * 32 + piece * 8;
            pa[i] = pc[i] = make_uint4(0, 0, 0, 0);
            if (KIND == kDH && j0 + tok < b.n_tok && f < Fx) {
              const size_t o = (size_t)(b.a_row0 + j0 + tok) * Fx + f;
              pa[i] = *reinterpret_cast<const uint4*>(g.a + o);
              pc[i] = *reinterpret_cast<const uint4*>(g.c + o);
            }
          }
        };
        if (KIND == kDH) fetch(0);
#pragma unroll 1
        for (int j0 = 0; j0 < b.n_tok; j0 += 16) {
          uint4 ca[2], cc2[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) { ca[i] = pa[i]; cc2[i] = pc[i]; }
          if (KIND == kDH && j0 + 16 < b.n_tok) fetch(j0 + 16);
          uint32_t r[16];
          tc::tmem_ld16(t_base + j0, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) scr[j * 32 + lane] = __uint_as_float(r[j]);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int item = i * 32 + lane;             // 16 tokens x 4 pieces of 8 features
            const int tok = item >> 2, piece = item & 3;
            const int f = b.m0 + q * 32 + piece * 8;
            if (j0 + tok < b.n_tok && f < Fx) {
              const size_t o = (size_t)(b.a_row0 + j0 + tok) * Fx + f;
              float v[8];
#pragma unroll
              for (int x = 0; x < 8; ++x) v[x] = scr[tok * 32 + piece * 8 + x];
              if (KIND == kDH) {
                const uint4 av = ca[i];
                const uint4 cv = cc2[i];
                const __nv_bfloat16* ah = reinterpret_cast<const __nv_bfloat16*>(&av);
                const __nv_bfloat16* ch = reinterpret_cast<const __nv_bfloat16*>(&cv);
                uint4 da, dc;
                __nv_bfloat16* dah = reinterpret_cast<__nv_bfloat16*>(&da);
                __nv_bfloat16* dch = reinterpret_cast<__nv_bfloat16*>(&dc);
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                  const float aa = __bfloat162float(ah[x]), cc = __bfloat162float(ch[x]);
                  const float sg = sigm(aa);
                  // silu(a) = a s(a); silu'(a) = s(a) (1 + a (1 - s(a)))
                  dah[x] = __float2bfloat16_rn(v[x] * cc * (sg * (1.f + aa * (1.f - sg))));
                  dch[x] = __float2bfloat16_rn(v[x] * aa * sg);
                }
                *reinterpret_cast<uint4*>(g.o_bf0 + o) = da;
                *reinterpret_cast<uint4*>(g.o_bf1 + o) = dc;
              } else {
                uint4 ov;
                __nv_bfloat16* oh = reinterpret_cast<__nv_bfloat16*>(&ov);
#pragma unroll
                for (int x = 0; x < 8; ++x) oh[x] = __float2bfloat16_rn(v[x]);
                *reinterpret_cast<uint4*>(g.o_bf0 + o) = ov;
              }
            }
          }
          __syncwarp();
        }
      } else {
        // lane = output row m0 + 32q + lane, column = n0 + c: fp32 rows, 32 x 32 blocks
        // written to the warp's scratch as one 128-byte-swizzled box and stored by TMA
        // (o0/o1: routed / shared outputs; kDWGU o2/o3 for dW_up; kDUR, kDE: o0)
        const CUtensorMap* om = &o0;
        int z = 0;
        if (KIND == kDWD || KIND == kDWGU) {
          const bool sh = b.seg >= g.N_r;
          z = sh ? b.seg - g.N_r : b.seg;
          om = KIND == kDWGU && b.part ? (sh ? &o3 : &o2) : (sh ? &o1 : &o0);
        }
        const int Nx = (KIND == kDWD) ? g.I : g.d;
        const int Mx = KIND == kDWD ? g.d : KIND == kDWGU ? g.I : KIND == kDUR ? g.T : g.N_r;
        const int y0 = b.m0 + q * 32;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          if (b.n0 + c0 >= Nx) break;
          uint32_t r[32];
          tc::tmem_ld32(t_base + c0, r);
          tc::tmem_ld_wait();
          if (lane == 0) tc::bulk_wait_read();   // the previous box has left the scratch
          __syncwarp();
          uint8_t* rowp = reinterpret_cast<uint8_t*>(scr) + lane * 128;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 val = b.nk > 0 ? make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                      __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(rowp + ((v ^ (lane & 7)) << 4)) = val;   // 128-byte swizzle
          }
          tc::fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0 && y0 < Mx) {   // rows past Mx (and columns past Nx) are clipped
            tc::tma_store_3d(om, scr, b.n0 + c0, y0, z);
            tc::bulk_commit();
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&C.tempty[acc]);
    }
  }

  if (warp >= 2 && lane == 0) tc::bulk_wait_all();   // this warp's output stores are done
  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // a wait that ran out may have left TMA copies in flight: give them time to land
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 10000000ull) {
    }
  }
  if (warp == 1 && lane == 0) tc::mbar_drain(&C.fin, 0);
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

constexpr CUtensorMapDataType kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

// fp32 output [E][rows][cols] seen by TMA stores of 32 x 32 boxes (rows past `rows` and
// columns past `cols` are clipped).
bool out_map(CUtensorMap* m, const float* p, uint64_t cols, uint64_t rows, uint64_t E) {
  return make_tmap_3d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p, cols, rows, E, cols * 4, rows * cols * 4, 32, 32);
}

// MN-major map: inner = the M/N extent (contiguous), outer = K rows; box 64 x 64.
bool map_mn(CUtensorMap* m, const void* p, uint64_t inner, uint64_t rows) {
  return make_tmap_2d(m, kBF16, p, inner, rows, inner * 2, 64, 64);
}
// K-major map: inner = K (contiguous), outer = M/N rows; box 64 x `box_rows`.
bool map_k(CUtensorMap* m, const void* p, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  return make_tmap_2d(m, kBF16, p, inner, rows, inner * 2, 64, box_rows);
}

template <int KIND>
cudaError_t launch_kind(const CUtensorMap* m, const CUtensorMap* o, const BwdArgs& g, long long tiles_ub,
                        cudaStream_t st) {
  static std::mutex mu;
  static bool attr_set[64] = {};
  auto k = bwd_gemm_kernel<KIND>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
      if (err != cudaSuccess) return err;
      attr_set[dev] = true;
    }
  }
  const int grid = (int)std::max<long long>(1, std::min<long long>(device_sm_count(), tiles_ub));
  k<<<grid, THREADS, kSmemBytes, st>>>(m[0], m[1], m[2], m[3], m[4], m[5], o[0], o[1], o[2], o[3], g);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_gemms(const BwdGemmIo& io, cudaStream_t st) {
  const FfnShape& s = io.s;
  const uint64_t R = (uint64_t)s.T * s.K_r + (uint64_t)s.N_s * s.T;
  const int segs = s.N_r + s.N_s;
  // with no shared expert the shared maps repeat the routed ones (never read)
  const uint64_t Es = s.N_s ? s.N_s : s.N_r;
  const void* wsg = s.N_s ? io.ws_gate : io.w_gate;
  const void* wsu = s.N_s ? io.ws_up : io.w_up;
  const void* wsd = s.N_s ? io.ws_down : io.w_down;
  BwdArgs g{s.T, s.d, s.I, s.N_r, s.K_r, s.N_s, io.expert_offset, io.a, io.c, nullptr, nullptr,
            nullptr, nullptr, nullptr, nullptr, dev_error_ptr()};
  const long long tok_tiles =
      (long long)s.T * s.K_r / BN + s.N_r + (long long)s.N_s * ((s.T + BN - 1) / BN);
  CUtensorMap m[6];
  // MN-major operands: one 3-D box of 2 (A, slots 0-3) or 4 (B, slots 4-5) 64-element
  // chunks per K step when every MN extent (d, I, N_r) is a multiple of 64, else 2-D
  // boxes of one chunk each
  if (s.d % 64 == 0 && s.I % 64 == 0 && s.N_r % 64 == 0) {
    CUtensorMap probe;
    g.mn3d = make_tmap_mn3d(&probe, kBF16, io.u, s.d, s.T, (uint64_t)s.d * 2, 64, BN / 64) ? 1 : 0;
  }
  auto mn = [&](int slot, const void* p, uint64_t inner, uint64_t rows) {
    return g.mn3d ? make_tmap_mn3d(&m[slot], kBF16, p, inner, rows, inner * 2, 64, slot < 4 ? BM / 64 : BN / 64)
                  : map_mn(&m[slot], p, inner, rows);
  };
  auto same = [&](int from) {       // unused map slots: copies of a valid map
    for (int i = from; i < 6; ++i)
      if (i != 4) m[i] = m[0];
  };
  cudaError_t err;

  if (io.experts) {
    // dH = dY W_down, then the SwiGLU backward -> dA, dC
    if (!mn(0, io.w_down, s.I, (uint64_t)s.N_r * s.d) || !mn(1, wsd, s.I, Es * s.d) ||
        !map_k(&m[4], io.dY, s.d, R, BN))
      return cudaErrorInvalidValue;
    same(2);
    g.o_bf0 = io.dA;
    g.o_bf1 = io.dC;
    const CUtensorMap od[4] = {m[0], m[0], m[0], m[0]};
    if ((err = launch_kind<kDH>(m, od, g, tok_tiles * ((s.I + BM - 1) / BM), st)) != cudaSuccess) return err;

    // dX = dA W_gate + dC W_up
    if (!mn(0, io.w_gate, s.d, (uint64_t)s.N_r * s.I) ||
        !mn(1, io.w_up, s.d, (uint64_t)s.N_r * s.I) || !mn(2, wsg, s.d, Es * s.I) ||
        !mn(3, wsu, s.d, Es * s.I) || !map_k(&m[4], io.dA, s.I, R, BN) || !map_k(&m[5], io.dC, s.I, R, BN))
      return cudaErrorInvalidValue;
    g.o_bf0 = io.dX;
    g.o_bf1 = nullptr;
    const CUtensorMap ox[4] = {m[0], m[0], m[0], m[0]};
    if ((err = launch_kind<kDX>(m, ox, g, tok_tiles * ((s.d + BM - 1) / BM), st)) != cudaSuccess) return err;

    // dW_down[e] = dY^T h over the expert's rows
    if (!mn(0, io.dY, s.d, R) || !mn(4, io.h, s.I, R)) return cudaErrorInvalidValue;
    same(1);
    g.o_f0 = io.dw_down;
    g.o_fs0 = io.dws_down;
    CUtensorMap ow[4];
    if (!out_map(&ow[0], io.dw_down, s.I, s.d, s.N_r) || !out_map(&ow[1], s.N_s ? io.dws_down : io.dw_down, s.I, s.d,
                                                                   s.N_s ? s.N_s : s.N_r))
      return cudaErrorInvalidValue;
    ow[2] = ow[3] = ow[0];
    if ((err = launch_kind<kDWD>(m, ow, g, (long long)segs * ((s.d + BM - 1) / BM) * ((s.I + BN - 1) / BN),
                                 st)) != cudaSuccess)
      return err;

    // dW_gate[e] = dA^T x, dW_up[e] = dC^T x (x: x_perm rows, or u for the shared experts)
    if (!mn(0, io.dA, s.I, R) || !mn(1, io.dC, s.I, R) ||
        !mn(4, io.x_perm, s.d, (uint64_t)s.T * s.K_r) || !mn(5, io.u, s.d, s.T))
      return cudaErrorInvalidValue;
    m[2] = m[3] = m[0];
    g.o_f0 = io.dw_gate;
    g.o_f1 = io.dw_up;
    g.o_fs0 = io.dws_gate;
    g.o_fs1 = io.dws_up;
    CUtensorMap og[4];
    const int Es2 = s.N_s ? s.N_s : s.N_r;
    if (!out_map(&og[0], io.dw_gate, s.d, s.I, s.N_r) || !out_map(&og[1], s.N_s ? io.dws_gate : io.dw_gate, s.d, s.I, Es2) ||
        !out_map(&og[2], io.dw_up, s.d, s.I, s.N_r) || !out_map(&og[3], s.N_s ? io.dws_up : io.dw_up, s.d, s.I, Es2))
      return cudaErrorInvalidValue;
    if ((err = launch_kind<kDWGU>(m, og, g, 2LL * segs * ((s.I + BM - 1) / BM) * ((s.d + BN - 1) / BN),
                                  st)) != cudaSuccess)
      return err;
  }
  if (!io.router) return cudaSuccess;

  // router: du = dz e, de = dz^T u
  if (!map_k(&m[0], io.dz, s.N_r, s.T, BM) || !mn(4, io.e, s.d, s.N_r)) return cudaErrorInvalidValue;
  same(1);
  g.o_f0 = io.du_router;
  g.o_f1 = g.o_fs0 = g.o_fs1 = nullptr;
  CUtensorMap ou[4];
  if (!out_map(&ou[0], io.du_router, s.d, s.T, 1)) return cudaErrorInvalidValue;
  ou[1] = ou[2] = ou[3] = ou[0];
  if ((err = launch_kind<kDUR>(m, ou, g, (long long)((s.T + BM - 1) / BM) * ((s.d + BN - 1) / BN), st)) !=
      cudaSuccess)
    return err;
  if (!mn(0, io.dz, s.N_r, s.T) || !mn(4, io.u, s.d, s.T)) return cudaErrorInvalidValue;
  same(1);
  g.o_f0 = io.de;
  CUtensorMap oe[4];
  if (!out_map(&oe[0], io.de, s.d, s.N_r, 1)) return cudaErrorInvalidValue;
  oe[1] = oe[2] = oe[3] = oe[0];
  return launch_kind<kDE>(m, oe, g, (long long)((s.N_r + BM - 1) / BM) * ((s.d + BN - 1) / BN), st);
}

}  // namespace moe
