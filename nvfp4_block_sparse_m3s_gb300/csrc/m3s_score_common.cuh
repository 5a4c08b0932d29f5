// Shared by the index scorers: arguments, query-row tiles, and the helper that
// hands out block-table entries to a warp.
#pragma once

#include <cuda.h>

#include "m3s_device.cuh"

namespace m3s {

constexpr int kMaxTiles = 8192;

// Persistent grids run at most this many CTAs (candidate slots are sized by it).
constexpr int kMaxGrid = 256;

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
  // streaming top-k (cand == nullptr: block scores only, into bscores)
  unsigned long long* cand;   // candidate lists [ntiles + grid - 1][QT][topk], packed keys
  unsigned* ticket;           // per tile: blocks scored so far in this call (0 between calls)
  int topk, init_blocks, local_blocks;
  int32_t* ids;               // [R][topk] output ids, or nullptr when keys_out is given
  unsigned long long* keys_out;  // [R][topk] merged keys (candidate output), or nullptr
  const int32_t* blk_base;    // per request: the request's id of the call's block 0 (or nullptr)
  const int32_t* blk_count;   // per request: blocks of the call's slice (with blk_base)
  float* seg_scores;          // verify path: per CTA, [QT][bt_stride] block maxima of its segment
  int2* meta;                 // partials mode (no merge here): per tile (first slot, lists), or nullptr
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
    if (a.blk_base && ti.req < a.B) {   // a slice of the request's blocks: its causal part
      const int base = a.blk_base[ti.req], cnt = max(a.blk_count[ti.req], 0);
      ti.len = min(max(ti.len - base * kPage, 0), cnt * kPage);
      if (base < 0 || ti.len <= 0) {   // nothing of this row in the slice
        ti.nrows = 0;
        ti.len = 0;
        return ti;
      }
    }
  } else {
    const int b = t / a.cpr, j = t % a.cpr;
    const int c0 = a.cu_q[b], qb = a.cu_q[b + 1] - c0;
    const int n = min(min(QT, qb - j * QT), a.R - (c0 + j * QT));   // rows past R do not exist
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

// The tiles' layout in the work split, in shared memory:
//   pre[t]   exclusive prefix of the tiles' block counts (pre[ntiles] = all blocks);
//   nz[w]    bit t % 32 of word t / 32 set when tile t has blocks;
//   nzc[w]   set bits in the words before w.
// A tile with blocks costs c set-up units plus one per block in the work split;
// an empty tile costs nothing.
struct TileLayout {
  long long* bnd;   // bnd[k] = floor(C k / g): CTA k's first cost position (k <= g; C beyond)
  int* pre;
  unsigned* nz;
  int* nzc;
  int ntiles;
  int c;
  int g;   // the CTAs the cost is cut over: min(grid, C), so each has at least one unit
  static constexpr size_t bytes(int ntiles) {
    return static_cast<size_t>(kMaxGrid + 1) * 8 + static_cast<size_t>(ntiles + 1) * 4 +
           2 * static_cast<size_t>((ntiles + 32) / 32) * 4;
  }
  __device__ __forceinline__ void bind(void* base, int n, int setup) {
    bnd = static_cast<long long*>(base);   // (8-byte aligned base)
    pre = reinterpret_cast<int*>(bnd + kMaxGrid + 1);
    nz = reinterpret_cast<unsigned*>(pre + n + 1);
    nzc = reinterpret_cast<int*>(nz + (n + 32) / 32);
    ntiles = n;
    c = setup;
  }
  __device__ __forceinline__ int blocks(int t) const { return pre[t + 1] - pre[t]; }
  // cost position of tile t's start
  __device__ __forceinline__ long long cost_at(int t) const {
    const int w = t >> 5;
    const int ne = nzc[w] + __popc(nz[w] & ((1u << (t & 31)) - 1u));
    return pre[t] + static_cast<long long>(c) * ne;
  }
  __device__ __forceinline__ long long total_cost() const { return cost_at(ntiles); }
  // Block position of cost position x: monotone, so consecutive cost ranges
  // give contiguous, disjoint block ranges covering every block.
  __device__ __forceinline__ int cost_to_block(long long x) const {
    if (x >= total_cost()) return pre[ntiles];
    int l = 0, h = ntiles;   // cost_at(l) <= x < cost_at(h)
    while (h - l > 1) {
      const int m = (l + h) >> 1;
      if (cost_at(m) <= x) l = m; else h = m;
    }
    const long long o = x - cost_at(l);
    return pre[l] + static_cast<int>(o > c ? o - c : 0);
  }
  // the block range [lo, hi) of CTA k (of the grid the boundaries were made for)
  __device__ __forceinline__ int2 cta_range(int k) const {
    return make_int2(cost_to_block(bnd[k]), cost_to_block(bnd[k + 1]));
  }
  // The CTAs (of g) whose ranges hold the first and the last block of tile t
  // (which has blocks). Block b0 + j of the tile sits at cost position base + j
  // (base = the tile's start + its set-up: the set-up units map to b0 too), and
  // CTA k starts at cost position floor(C k / g), so the CTA holding cost
  // position X is the largest k with floor(C k / g) <= X.
  __device__ __forceinline__ int2 covering_ctas(int t, int g) const {
    const long long C = total_cost(), base = cost_at(t) + c;
    const long long X0 = base, X1 = base + blocks(t) - 1;
    return make_int2(static_cast<int>(min(static_cast<long long>(g - 1), ((X0 + 1) * g - 1) / C)),
                     static_cast<int>(min(static_cast<long long>(g - 1), ((X1 + 1) * g - 1) / C)));
  }
  // CTA k's blocks of tile t, relative to the tile's first block: [x, y), empty
  // when y <= x (a CTA between the covering ones whose cost range holds no block
  // of the tile).
  __device__ __forceinline__ int2 cta_blocks(int t, int k) const {
    const long long base = cost_at(t) + c, nb = blocks(t);
    const long long lo = min(max(bnd[k] - base, 0ll), nb);
    const long long hi = min(max(bnd[k + 1] - base, 0ll), nb);
    return make_int2(static_cast<int>(lo), static_cast<int>(hi));
  }
};

// Fill a TileLayout (bound to shared memory) by the whole CTA. red: one int
// per warp of scratch.
template <int QT>
__device__ __forceinline__ void tile_prefix(const ScoreArgs& a, TileLayout& L, int* red, int nthreads) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ntiles = a.ntiles;
  const int nw = (ntiles + 32) / 32;
  for (int i = tid; i < nw; i += nthreads) L.nz[i] = 0u;
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
  if (tid == 0) L.pre[0] = 0;
  for (int i = i0; i < i1; ++i) {
    const TileInfo<QT> ti = tile_info<QT>(a, i, false);
    const int nb = ti.nrows ? (ti.len + kPage - 1) / kPage : 0;
    run += nb;
    L.pre[i + 1] = run;
    if (nb) atomicOr(&L.nz[i >> 5], 1u << (i & 31));
  }
  __syncthreads();
  if (warp == 0) {   // exclusive prefix of the words' bit counts
    int carry = 0;
    for (int w0 = 0; w0 < nw; w0 += 32) {
      const int w = w0 + lane;
      const int cnt = w < nw ? __popc(L.nz[w]) : 0;
      int inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      if (w < nw) L.nzc[w] = carry + inc - cnt;
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  __syncthreads();
  const long long C = L.total_cost();
  L.g = static_cast<int>(min(static_cast<long long>(gridDim.x), max(C, 1ll)));
  for (int k = tid; k <= static_cast<int>(gridDim.x); k += nthreads) L.bnd[k] = k <= L.g ? C * k / L.g : C;
  __syncthreads();
}

// This CTA's share (of the grid's) of an input's bytes, brought into L2 ahead
// of its use; a hint only, skipped for an unaligned base.
__device__ __forceinline__ void prefetch_share_l2(const void* base, size_t bytes) {
  if (!base || bytes == 0 || (reinterpret_cast<uintptr_t>(base) & 15u) != 0) return;
  const size_t chunk = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~static_cast<size_t>(15);
  const size_t off = static_cast<size_t>(blockIdx.x) * chunk;
  if (off >= bytes) return;
  const size_t n = min(chunk, bytes - off) & ~static_cast<size_t>(15);
  if (n > 0) bulk_prefetch_l2(static_cast<const uint8_t*>(base) + off, static_cast<uint32_t>(n));
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

// ---- streaming block top-k ------------------------------------------------
//
// Selection keys (64-bit): a scored block's key is topk_key(score, id) (the
// higher score, then the lower id); forced blocks rank above every score: init
// blocks (the row's first init blocks) 0xFFFFFFFF:~id (lower id first), local
// blocks (its last local blocks) 0xFFFFFFFE:id (most recent first). Keys of
// distinct blocks are distinct; 0 is below every key (an empty slot).
__device__ __forceinline__ unsigned long long select_key(float score, int id, int nb, int init, int local) {
  if (id < init) return (0xFFFFFFFFull << 32) | static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(id));
  if (id >= nb - local) return (0xFFFFFFFEull << 32) | static_cast<unsigned long long>(static_cast<uint32_t>(id));
  return topk_key(score, id);
}

// The block id of a selection key (local keys hold the id itself, the others
// its complement).
__device__ __forceinline__ int select_key_id(unsigned long long key) {
  const uint32_t lo = static_cast<uint32_t>(key);
  return static_cast<int>((key >> 32) == 0xFFFFFFFEull ? lo : 0xFFFFFFFFu - lo);
}

// A warp's running top-k (k <= 64) of distinct keys, sorted descending: slot s
// lives in lane s % 32, register s / 32; empty slots hold 0.
struct WarpTopk {
  unsigned long long a, b;   // slots lane and 32 + lane
  unsigned long long kth;    // the k-th largest so far (0 while fewer than k)
  __device__ __forceinline__ void clear() { a = b = kth = 0ull; }
  // Insert x (the same value in every lane; distinct from every key held).
  __device__ __forceinline__ void insert(unsigned long long x, int k, int lane) {
    if (x <= kth) return;
    const int pos = __popc(__ballot_sync(0xffffffffu, a > x)) + __popc(__ballot_sync(0xffffffffu, b > x));
    const unsigned long long a_up = __shfl_up_sync(0xffffffffu, a, 1);
    const unsigned long long b_up = __shfl_up_sync(0xffffffffu, b, 1);
    const unsigned long long a31 = __shfl_sync(0xffffffffu, a, 31);
    const int sa = lane, sb = 32 + lane;
    unsigned long long na = sa < pos ? a : (sa == pos ? x : a_up);
    unsigned long long nb = sb < pos ? b : (sb == pos ? x : (lane == 0 ? a31 : b_up));
    if (sa >= k) na = 0ull;
    if (sb >= k) nb = 0ull;
    a = na;
    b = nb;
    kth = __shfl_sync(0xffffffffu, k > 32 ? b : a, (k - 1) & 31);
  }
  // Append slot s = the next largest key (used by merges that produce keys in
  // descending order).
  __device__ __forceinline__ void put(int s, unsigned long long x, int lane) {
    if (s < 32) { if (lane == s) a = x; }
    else if (lane == s - 32) b = x;
  }
};

// Merge nl descending candidate lists (kc keys each, 0-padded) into the top k
// keys, by one warp. List j starts at base + (slot ? slot[j] : j) * stride;
// GLOBAL = the lists are in global memory, written by other CTAs of this
// launch (read through L2), else in shared memory. Lane l owns lists l, l + 32,
// ... (at most OWN each) and keeps the best of their heads; each round takes
// the warp's best key (one 32-bit reduction on the high words, a second only
// when several lanes share the highest) and its owner advances that list.
template <int OWN, bool GLOBAL>
__device__ __forceinline__ void warp_merge_own(const unsigned long long* base, const int* slot, int stride,
                                               int nl, int kc, int k, int lane, WarpTopk& out) {
  const unsigned long long* lp[OWN];
  int p[OWN];
  unsigned long long h[OWN];
  unsigned long long best = 0ull;
#pragma unroll
  for (int j = 0; j < OWN; ++j) {
    const int li = lane + 32 * j;
    lp[j] = li < nl ? base + static_cast<size_t>(slot ? slot[li] : li) * stride : nullptr;
    p[j] = 0;
    h[j] = lp[j] ? (GLOBAL ? __ldcg(lp[j]) : *lp[j]) : 0ull;
    best = h[j] > best ? h[j] : best;
  }
  out.clear();
  for (int s = 0; s < k; ++s) {
    const uint32_t bh = static_cast<uint32_t>(best >> 32);
    const uint32_t mh = __reduce_max_sync(0xffffffffu, bh);
    const unsigned tied = __ballot_sync(0xffffffffu, bh == mh);
    const uint32_t lo = static_cast<uint32_t>(best);
    const uint32_t ml = __popc(tied) > 1 ? __reduce_max_sync(0xffffffffu, bh == mh ? lo : 0u)
                                         : __shfl_sync(0xffffffffu, lo, __ffs(tied) - 1);
    const unsigned long long m = (static_cast<unsigned long long>(mh) << 32) | ml;
    if (m == 0ull) break;   // every list is exhausted
    out.put(s, m, lane);
    if (best == m) {   // the one owner (keys are distinct): advance that list, refresh its best
      best = 0ull;
#pragma unroll
      for (int j = 0; j < OWN; ++j) {
        if (h[j] == m) {
          ++p[j];
          h[j] = p[j] < kc ? (GLOBAL ? __ldcg(lp[j] + p[j]) : lp[j][p[j]]) : 0ull;
        }
        best = h[j] > best ? h[j] : best;
      }
    }
  }
}

template <bool GLOBAL>
__device__ __forceinline__ void warp_merge(const unsigned long long* base, const int* slot, int stride,
                                           int nl, int kc, int k, int lane, WarpTopk& out) {
  static_assert(kMaxGrid <= 256, "at most 8 lists a lane");
  if (nl <= 32) warp_merge_own<1, GLOBAL>(base, slot, stride, nl, kc, k, lane, out);
  else if (nl <= 64) warp_merge_own<2, GLOBAL>(base, slot, stride, nl, kc, k, lane, out);
  else if (nl <= 128) warp_merge_own<4, GLOBAL>(base, slot, stride, nl, kc, k, lane, out);
  else warp_merge_own<8, GLOBAL>(base, slot, stride, nl, kc, k, lane, out);
}

// x = the top k (k <= 64) of the union of two descending warp lists x and y
// (distinct keys, 0-padded), descending: y reversed against x elementwise gives
// the 64 largest as a bitonic sequence (the classic bitonic split), which a
// bitonic merge network then sorts, larger keys to lower slots.
__device__ __forceinline__ void warp_merge2(WarpTopk& x, const WarpTopk& y, int k, int lane) {
  if (k <= 32) {
    const unsigned long long r = __shfl_sync(0xffffffffu, y.a, 31 - lane);
    unsigned long long z = x.a > r ? x.a : r;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, z, d);
      z = (lane & d) ? (o < z ? o : z) : (o > z ? o : z);
    }
    x.a = lane < k ? z : 0ull;
    x.b = 0ull;
    return;
  }
  const unsigned long long ra = __shfl_sync(0xffffffffu, y.b, 31 - lane);   // reversed y, slots 0 .. 31
  const unsigned long long rb = __shfl_sync(0xffffffffu, y.a, 31 - lane);   // slots 32 .. 63
  unsigned long long za = x.a > ra ? x.a : ra;
  unsigned long long zb = x.b > rb ? x.b : rb;
  if (zb > za) {   // distance 32: slot s against slot s + 32, in the lane
    const unsigned long long t = za;
    za = zb;
    zb = t;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const unsigned long long oa = __shfl_xor_sync(0xffffffffu, za, d);
    const unsigned long long ob = __shfl_xor_sync(0xffffffffu, zb, d);
    za = (lane & d) ? (oa < za ? oa : za) : (oa > za ? oa : za);
    zb = (lane & d) ? (ob < zb ? ob : zb) : (ob > zb ? ob : zb);
  }
  x.a = lane < k ? za : 0ull;
  x.b = 32 + lane < k ? zb : 0ull;
}

// Sort a warp list descending (slots past k hold 0): a bitonic sorting network
// over the 32 (k <= 32) or 64 slots; in the stage of block size `size`, slot i
// is ordered against slot i ^ d descending when i & size is 0, else ascending.
__device__ __forceinline__ void warp_sort_desc(WarpTopk& t, int k, int lane) {
  auto cx = [&](unsigned long long x, int i, int size, int d) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, x, d);
    const bool desc = (i & size) == 0, lower = (i & d) == 0;
    return (desc == lower) ? (o > x ? o : x) : (o < x ? o : x);
  };
  if (k <= 32) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int d = size >> 1; d > 0; d >>= 1) t.a = cx(t.a, lane, size, d);
    return;
  }
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int d = size >> 1; d > 0; d >>= 1) {
      t.a = cx(t.a, lane, size, d);
      t.b = cx(t.b, 32 + lane, size, d);   // (slot 32 + lane: ascending blocks at size 32)
    }
  if (t.b > t.a) {   // size 64, distance 32: in the lane
    const unsigned long long x = t.a;
    t.a = t.b;
    t.b = x;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    t.a = cx(t.a, lane, 64, d);
    t.b = cx(t.b, 32 + lane, 64, d);
  }
}

// A warp list from / to n <= 64 keys at p (slot s at p[s]).
__device__ __forceinline__ WarpTopk warp_load(const unsigned long long* p, int n, int lane) {
  WarpTopk t;
  t.a = lane < n ? p[lane] : 0ull;
  t.b = 32 + lane < n ? p[32 + lane] : 0ull;
  t.kth = 0ull;
  return t;
}
__device__ __forceinline__ void warp_store(const WarpTopk& t, unsigned long long* p, int n, int lane) {
  if (lane < n) p[lane] = t.a;
  if (32 + lane < n) p[32 + lane] = t.b;
}

// For each of `groups` groups of nl descending lists of k keys in shared memory
// (list j of group g at lists + (g * nl + j) * k), merge the group's lists into
// its list 0: a tree of pairwise warp merges, level by level (the lists i and
// i + st merged into list i, st = 1, 2, 4, ...), the pairs of a level spread
// over the warps, a barrier after each level. Called by the whole CTA.
__device__ __forceinline__ void tree_merge_lists(unsigned long long* lists, int groups, int nl, int k, int nthreads) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = nthreads >> 5;
  for (int st = 1; st < nl; st <<= 1) {
    const int pairs = (nl + 2 * st - 1) / (2 * st);   // list i = 2 st q, partner i + st
    for (int item = warp; item < groups * pairs; item += nwarps) {
      const int g = item / pairs, i = (item % pairs) * 2 * st;
      if (i + st >= nl) continue;   // (warp-uniform) no partner this level
      unsigned long long* li = lists + (static_cast<size_t>(g) * nl + i) * k;
      WarpTopk x = warp_load(li, k, lane);
      const WarpTopk y = warp_load(li + static_cast<size_t>(st) * k, k, lane);
      warp_merge2(x, y, k, lane);
      warp_store(x, li, k, lane);
    }
    __syncthreads();
  }
}

// Write a row's merged keys as ids: the selected ids ascending, then -1.
__device__ __forceinline__ void write_ids(const WarpTopk& sel, int k, int32_t* out, int lane) {
  const int ia = sel.a ? select_key_id(sel.a) : 0x7FFFFFFF;
  const int ib = sel.b ? select_key_id(sel.b) : 0x7FFFFFFF;
  const int cnt = __popc(__ballot_sync(0xffffffffu, sel.a != 0ull)) + __popc(__ballot_sync(0xffffffffu, sel.b != 0ull));
  int ra = 0, rb = 0;
  for (int j = 0; j < 32; ++j) {
    const int xa = __shfl_sync(0xffffffffu, ia, j);
    ra += xa < ia;
    rb += xa < ib;
    if (k > 32) {
      const int xb = __shfl_sync(0xffffffffu, ib, j);
      ra += xb < ia;
      rb += xb < ib;
    }
  }
  if (sel.a) out[ra] = ia;
  if (sel.b) out[rb] = ib;
  for (int i = cnt + lane; i < k; i += 32) out[i] = -1;
}

__device__ __forceinline__ void write_keys(const WarpTopk& sel, int k, unsigned long long* out, int lane) {
  if (lane < k) out[lane] = sel.a;
  if (32 + lane < k) out[32 + lane] = sel.b;
}

// The rows a tile stands for, valid or not: (first row, count).
template <int QT>
__device__ __forceinline__ int2 tile_rows(const ScoreArgs& a, int t) {
  if (QT == 1) return make_int2(t, 1);
  const int b = t / a.cpr, j = t % a.cpr;
  const int c0 = a.cu_q[b], qb = a.cu_q[b + 1] - c0;
  return make_int2(c0 + j * QT, max(0, min(min(QT, qb - j * QT), a.R - (c0 + j * QT))));
}

// Rows that no CTA scores get no candidates: the rows of tiles without blocks
// (pad rows, empty or invalid requests) and, on the verify path, the rows past
// cu_q[B]. CTA k writes theirs (ids -1, or zero keys) for tiles t = k mod grid.
template <int QT>
__device__ void write_unscored_rows(const ScoreArgs& a, const TileLayout& L, int nthreads) {
  const int tid = threadIdx.x, G = gridDim.x;
  auto blank = [&](int r) {
    for (int i = tid; i < a.topk; i += nthreads) {
      if (a.ids) a.ids[static_cast<size_t>(r) * a.topk + i] = -1;
      else if (a.keys_out) a.keys_out[static_cast<size_t>(r) * a.topk + i] = 0ull;
    }
    if (a.meta && tid == 0) a.meta[r] = make_int2(0, 0);   // no candidate lists
  };
  for (int t = blockIdx.x; t < L.ntiles; t += G) {
    if (L.blocks(t) != 0) continue;
    const int2 rows = tile_rows<QT>(a, t);
    for (int r = rows.x; r < rows.x + rows.y; ++r) blank(r);
  }
  if (QT > 1)
    for (int r = max(0, a.cu_q[a.B]) + blockIdx.x; r < a.R; r += G) blank(r);
}

// atomicAdd at GPU scope with acquire-release semantics: it publishes the
// writes that happen before it (the CTA barrier before it makes the other
// threads' writes among them) and, when it observes another CTA's addition,
// makes that CTA's published writes visible to what follows it (the barrier
// after it extends that to the CTA's other threads).
__device__ __forceinline__ unsigned atomic_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// End of a CTA's segment of tile t, called by every thread of the CTA after a
// __syncthreads that follows this segment's candidate writes. The segment's
// block count is added to the tile's ticket (one acquire-release atomic); the
// CTA whose addition completes the tile (every block scored) merges
// the tile's rows: their lists in slots t + c for the CTAs c whose ranges meet
// the tile, staged through buf (buf_keys keys of shared memory) and merged by a
// tree of pairwise warp merges (one warp per row reading L2 when they do not
// fit), and resets the ticket for the next call. Shared scratch: vslot
// (kMaxGrid + 32 ints), cnt (one int).
template <int QT>
__device__ void tile_finish(const ScoreArgs& a, const TileLayout& L, int t, int seg_blocks,
                            unsigned long long* buf, int buf_keys, int* vslot, int* cnt, int nthreads) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  const int G = L.g, kc = a.topk;
  // thread 0's ticket addition is in flight while the CTA works out which CTAs
  // hold blocks of the tile (all the merge needs; unused unless this CTA merges)
  unsigned old = 0u;
  if (tid == 0) old = atomic_add_acq_rel_gpu(&a.ticket[t], static_cast<unsigned>(seg_blocks));
  const int2 cc = L.covering_ctas(t, G);
  bool has = false;
  if (tid <= cc.y - cc.x) {   // (at most kMaxGrid covering CTAs: one thread each)
    const int2 r = L.cta_blocks(t, cc.x + tid);
    has = r.y > r.x;
  }
  int* vcount = vslot + kMaxGrid;
  const unsigned bal = __ballot_sync(0xffffffffu, has);   // compact the holders' slots, in CTA order
  if (lane == 0) vcount[warp] = __popc(bal);
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += vcount[w];
  if (has) vslot[base + __popc(bal & ((1u << lane) - 1u))] = t + cc.x + tid;
  if (tid == 0) {
    int n = 0;
    for (int w = 0; w < nwarps; ++w) n += vcount[w];
    *cnt = old + static_cast<unsigned>(seg_blocks) == static_cast<unsigned>(L.blocks(t)) ? n : -1;
  }
  __syncthreads();
  if (*cnt < 0) return;            // (uniform) another CTA completes this tile; else every
                                    // CTA's list of the tile is visible from here on
  const int nl = *cnt;
  const int2 rows = tile_rows<QT>(a, t);
  const int per_row = nl * kc;
  const int rp = per_row > 0 ? buf_keys / per_row : 0;   // rows staged per pass
  for (int r0 = 0; r0 < rows.y; r0 += (rp > 0 ? rp : rows.y)) {
    const int nr = rp > 0 ? min(rp, rows.y - r0) : rows.y - r0;
    if (rp > 0) {
      for (int e = tid; e < nr * per_row; e += nthreads) {
        const int rr = e / per_row, j = (e / kc) % nl, i = e % kc;
        buf[e] = __ldcg(a.cand + (static_cast<size_t>(vslot[j]) * QT + r0 + rr) * kc + i);
      }
      __syncthreads();
      tree_merge_lists(buf, nr, nl, kc, nthreads);
      for (int rr = warp; rr < nr; rr += nwarps) {
        const WarpTopk sel = warp_load(buf + static_cast<size_t>(rr) * per_row, kc, lane);
        const size_t row = static_cast<size_t>(rows.x + r0 + rr);
        if (a.ids) write_ids(sel, a.topk, a.ids + row * a.topk, lane);
        else write_keys(sel, a.topk, a.keys_out + row * a.topk, lane);
      }
    } else {   // too many lists to stage: one warp per row merges them from L2
      for (int rr = warp; rr < nr; rr += nwarps) {
        WarpTopk sel;
        warp_merge<true>(a.cand + static_cast<size_t>(r0 + rr) * kc, vslot, QT * kc, nl, kc, a.topk, lane, sel);
        const size_t row = static_cast<size_t>(rows.x + r0 + rr);
        if (a.ids) write_ids(sel, a.topk, a.ids + row * a.topk, lane);
        else write_keys(sel, a.topk, a.keys_out + row * a.topk, lane);
      }
    }
    fence_proxy_async();   // buf may be shared memory that bulk copies refill next
    __syncthreads();
  }
  if (tid == 0) {
    a.ticket[t] = 0u;
    *cnt = 0;
  }
}

// Streaming top-k workspace: a ticket per tile (rounded up to 256 bytes), then
// candidate lists for ntiles + kMaxGrid - 1 slots of qt rows x topk keys, then
// (multi-row tiles) each CTA's segment score scratch, qt rows x bt_stride fp32.
__host__ __device__ constexpr size_t topk_ticket_bytes(int ntiles) {
  return (static_cast<size_t>(ntiles) * 4 + 255) & ~static_cast<size_t>(255);
}
__host__ __device__ constexpr size_t topk_cand_bytes(int ntiles, int qt, int topk) {
  return static_cast<size_t>(ntiles + kMaxGrid - 1) * qt * topk * 8;
}
__host__ __device__ constexpr size_t topk_ws_bytes(int ntiles, int qt, int topk, int bt_stride = 0) {
  return topk_ticket_bytes(ntiles) + topk_cand_bytes(ntiles, qt, topk) +
         (qt > 1 ? static_cast<size_t>(kMaxGrid) * qt * (bt_stride > 0 ? bt_stride : 1) * 4 : 0);
}

// Which form a score + top-k call takes. With more tiles than CTAs can run,
// tiles finish throughout the launch and each tile's candidate merge overlaps
// other tiles' scoring: the top-k streams inside the scorer (one launch, no
// block-score matrix). With at most kMaxGrid tiles every tile ends with the
// launch and the merges form its tail; there the block scores go to the
// workspace and a second launch selects (it starts while the scorer ends).
// Measured on the decode batches (1-8 rows) and the 16 x 8 verify batch, the
// two-launch form was the faster one; on the 8192-row prefill chunk (1024
// tiles), streaming.
// m3s_index_attention's workspace: candidate lists for R + kMaxGrid - 1 slots
// of topk keys, then each row's (first slot, lists).
__host__ __device__ constexpr size_t index_attention_meta_offset(int R, int topk) {
  return (static_cast<size_t>(R + kMaxGrid - 1) * topk * 8 + 255) & ~static_cast<size_t>(255);
}
__host__ __device__ constexpr size_t index_attention_ws_bytes(int R, int topk) {
  return index_attention_meta_offset(R, topk) + static_cast<size_t>(R) * 8;
}

// m3s_verify_index_attention's workspace: the candidate lists (slots of 8 rows
// x topk keys, as in the streaming form), the CTAs' block-maximum scratch
// ([grid][8][bt_stride] fp32), then each row's list range (int2 per row).
__host__ __device__ constexpr size_t verify_attention_seg_offset(int ntiles, int topk) {
  return (topk_cand_bytes(ntiles, 8, topk) + 255) & ~static_cast<size_t>(255);
}
__host__ __device__ constexpr size_t verify_attention_meta_offset(int ntiles, int topk, int bt_stride) {
  return (verify_attention_seg_offset(ntiles, topk) +
          static_cast<size_t>(kMaxGrid) * 8 * (bt_stride > 0 ? bt_stride : 1) * 4 + 255) &
         ~static_cast<size_t>(255);
}
__host__ __device__ constexpr size_t verify_attention_ws_bytes(int ntiles, int R, int topk, int bt_stride) {
  return verify_attention_meta_offset(ntiles, topk, bt_stride) + static_cast<size_t>(R) * 8;
}

__host__ __device__ constexpr bool topk_streams(long long ntiles) { return ntiles > kMaxGrid; }

// Workspace bytes of a score + top-k call: the streaming state, or the block
// scores (rows x bt_stride fp32) of the two-launch form.
__host__ __device__ constexpr size_t score_topk_ws_bytes(long long ntiles, int qt, int R, int bt_stride, int topk) {
  return topk_streams(ntiles) ? topk_ws_bytes(static_cast<int>(ntiles), qt, topk, bt_stride)
                              : static_cast<size_t>(R) * (bt_stride > 0 ? bt_stride : 1) * 4;
}

int sm_count();
int grid_size();   // the persistent scorers' CTA count: min(SMs, kMaxGrid)
// Tensor map over a one-head index code plane viewed as [num_pages * 128 rows]
// x [64 bytes], boxes of one page (128 rows), 64-byte swizzle.
bool make_codes_map(CUtensorMap* map, const uint8_t* codes, int num_pages);
int launch_score_decode(const ScoreArgs& a, cudaStream_t st);

}  // namespace m3s
