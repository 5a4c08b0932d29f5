// Shared by the index scorers: arguments, query-row tiles, and the helper that
// hands out block-table entries to a warp.
#pragma once

#include <cuda.h>

#include "m3s_device.cuh"

namespace m3s {

constexpr int kMaxTiles = 8192;

struct ScoreArgs {
  const uint16_t* q_idx;
  const float* w;
  int Hi;
  const uint8_t* codes;
  const uint8_t* scales;
  int num_pages;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* row_req;  // index path (QT == 1)
  const int32_t* cu_q;     // verify path (QT == 8)
  const int32_t* row_len;
  int R, B, ntiles, cpr;   // cpr: row chunks per request (verify path)
  float* bscores;
  int bs_stride;
  int32_t* err;
  int mx;                  // 1: the index plane is MXFP4 (E8M0 per 32), else NVFP4
};

template <int QT>
struct TileInfo {
  int row0, nrows, req, len;
};

// Rows, request and key count of tile t. Invalid tiles (pad rows, bad request,
// a length beyond the block table) come back with nrows == 0.
template <int QT>
__device__ TileInfo<QT> tile_info(const ScoreArgs& a, int t, bool report) {
  TileInfo<QT> ti{0, 0, -1, 0};
  if (QT == 1) {
    ti.row0 = t;
    ti.req = a.row_req[t];
    ti.len = a.row_len[t];
    if (ti.req < 0 || ti.len <= 0) { ti.len = 0; return ti; }
    ti.nrows = 1;
  } else {
    const int b = t / a.cpr, j = t % a.cpr;
    const int c0 = a.cu_q[b], qb = a.cu_q[b + 1] - c0;
    const int n = min(QT, qb - j * QT);
    if (n <= 0) return ti;
    ti.row0 = c0 + j * QT;
    ti.req = b;
    ti.nrows = n;
    for (int i = 0; i < n; ++i) ti.len = max(ti.len, a.row_len[ti.row0 + i]);
    if (ti.len <= 0) { ti.nrows = 0; ti.len = 0; return ti; }
  }
  if (ti.req >= a.B || ti.len > a.bt_stride * kPage) {
    if (report) raise(a.err, M3S_DEVERR_ROW);
    ti.nrows = 0;
    ti.len = 0;
  }
  return ti;
}

// Exclusive prefix over tiles of their block counts, into pre[0 .. ntiles]
// (shared memory), by the whole CTA. red: one int per warp of scratch.
template <int QT>
__device__ __forceinline__ void tile_prefix(const ScoreArgs& a, int* pre, int* red, int nthreads) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ntiles = a.ntiles;
  const int per = (ntiles + nthreads - 1) / nthreads;
  const int i0 = min(ntiles, tid * per), i1 = min(ntiles, i0 + per);
  int local = 0;
  for (int i = i0; i < i1; ++i) {
    const TileInfo<QT> ti = tile_info<QT>(a, i, blockIdx.x == 0);
    local += ti.nrows ? (ti.len + kPage - 1) / kPage : 0;
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int wv = 0; wv < warp; ++wv) base += red[wv];
  int run = base + incl - local;
  if (tid == 0) pre[0] = 0;
  for (int i = i0; i < i1; ++i) {
    const TileInfo<QT> ti = tile_info<QT>(a, i, false);
    run += ti.nrows ? (ti.len + kPage - 1) / kPage : 0;
    pre[i + 1] = run;
  }
  __syncthreads();
}

// First tile whose block range holds position lo (pre[t] <= lo < pre[t+1]).
__device__ __forceinline__ int tile_at(const int* pre, int ntiles, int lo) {
  int l = 0, h = ntiles;
  while (h - l > 1) {
    const int m = (l + h) >> 1;
    if (pre[m] <= lo) l = m; else h = m;
  }
  return l;
}

// Page id of block j of the segment for a warp that walks j = j0, j0 + step, ...:
// the warp loads 32 upcoming entries of the block table at once (one coalesced
// load) and hands them out with a shuffle, so no role waits on a dependent
// global load per block. Must be called by all 32 lanes with the same j.
struct PageWindow {
  int base = -1, val = -1;
  __device__ __forceinline__ int get(const int32_t* bt_row, int j, int step, int jend, int lane) {
    const int slot = (j - base) / step;
    if (base < 0 || slot >= 32) {
      base = j;
      const int jl = j + lane * step;
      val = jl < jend ? bt_row[jl] : -1;
    }
    return __shfl_sync(0xffffffffu, val, (j - base) / step);
  }
};

int sm_count();
// Tensor map over a one-head index code plane viewed as [num_pages * 128 rows]
// x [64 bytes], boxes of one page (128 rows), 64-byte swizzle.
bool make_codes_map(CUtensorMap* map, const uint8_t* codes, int num_pages);
int launch_score_decode(const ScoreArgs& a, cudaStream_t st);

}  // namespace m3s
