// Tile schedule over the variable-size expert segments, built on the device from
// expert_offset (no host round trip).  Segment i < N_r is routed expert i with
// rows [expert_offset[i], expert_offset[i+1]); segment N_r + s is shared expert s
// over all T tokens.  Tiles are numbered segment-major, then m-tile (token rows),
// then n-tile (weight rows), so CTAs running at the same time share a token tile
// through L2, and a segment's few m-tiles reuse its weight tiles soon after.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kMaxShared = 32;
constexpr int kMaxSegs = 256 + kMaxShared;

struct SegTable {
  int total, nseg, T, K_r, N_r;
  int prefix[kMaxSegs + 1];  // tiles before segment i
  int row0[kMaxSegs];        // first input row of the segment
  int rows[kMaxSegs];        // rows in the segment (0..T)
  int mt[kMaxSegs];          // m-tiles in the segment
  int q[kMaxSegs];           // rows per m-tile (the last one may have fewer)
};

struct TileCoord {
  int seg, m, n;
  int row0;      // first input row (x_perm row for routed, u row 0 for shared)
  int rows;      // rows in the segment
  int out_row0;  // first row in the FFN row space [T*K_r + N_s*T]
  int tok0;      // first row of this tile within the segment (m * q)
  int n_tok;     // rows of this tile
};

// All threads of the block call this; the caller synchronises afterwards.  With
// `balanced` a segment's rows are cut into ceil(rows/BM) tiles of equal size rounded up
// to 16 (at most BM), so that the tiles of one segment take the same time; otherwise
// into tiles of exactly BM rows.  A routed segment that does not lie inside
// [0, T*K_r) (expert_offset not produced by the dispatch) is treated as empty and
// MOE_ERR_INVALID_ARG is recorded in `err`.
__device__ __forceinline__ void build_seg_table(SegTable& tab, const int32_t* __restrict__ off,
                                                int T, int K_r, int N_r, int N_s, int BM,
                                                int n_tiles_n, bool balanced, int32_t* err) {
  const int nseg = N_r + N_s;
  for (int i = threadIdx.x; i < nseg; i += blockDim.x) {
    int r0 = 0, rows = T;
    if (i < N_r) {
      r0 = off[i];
      rows = off[i + 1] - r0;
      if (r0 < 0 || rows < 0 || (long long)r0 + rows > (long long)T * K_r) {
        if (blockIdx.x == 0) record_error(err, MOE_ERR_INVALID_ARG);
        r0 = 0;
        rows = 0;
      }
    }
    tab.row0[i] = r0;
    tab.rows[i] = rows;
    const int mt = (rows + BM - 1) / BM;
    tab.mt[i] = mt;
    tab.q[i] = (balanced && mt > 0) ? min(BM, (((rows + mt - 1) / mt) + 15) & ~15) : BM;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int span = (nseg + 31) / 32;
    int local = 0;
    for (int q = 0; q < span; ++q) {
      const int i = lane * span + q;
      if (i < nseg) local += tab.mt[i] * n_tiles_n;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int q = 0; q < span; ++q) {
      const int i = lane * span + q;
      if (i < nseg) {
        tab.prefix[i] = run;
        run += tab.mt[i] * n_tiles_n;
      }
    }
    if (lane == 31) {
      tab.prefix[nseg] = incl;
      tab.total = incl;
      tab.nseg = nseg;
      tab.T = T;
      tab.K_r = K_r;
      tab.N_r = N_r;
    }
  }
}

__device__ __forceinline__ TileCoord decode_tile(const SegTable& tab, int tile, int n_tiles_n) {
  // largest segment i with prefix[i] <= tile; then prefix[i+1] > tile, so i is non-empty
  int lo = 0, hi = tab.nseg;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tab.prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  TileCoord c;
  c.seg = lo;
  const int within = tile - tab.prefix[lo];
  c.m = within / n_tiles_n;
  c.n = within - c.m * n_tiles_n;
  c.row0 = tab.row0[lo];
  c.rows = tab.rows[lo];
  c.out_row0 = lo < tab.N_r ? c.row0 : tab.T * tab.K_r + (lo - tab.N_r) * tab.T;
  c.tok0 = c.m * tab.q[lo];
  c.n_tok = min(tab.q[lo], c.rows - c.tok0);
  return c;
}

}  // namespace moe
