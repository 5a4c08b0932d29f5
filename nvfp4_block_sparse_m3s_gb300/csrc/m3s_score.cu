// Lightning-indexer scoring over paged NVFP4 index keys with block top-k.
//
// "[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (ROCm/ATOM
// #2744): Design / Index (FP4 index keys decoded to 16-bit in registers),
// Design / Decode score grid (a long request must not serialise the kernel)
// and Design / Fused verify top-k (rows of one request scored together, ids
// only). Token score = sum_h w_h * ReLU(q_h . k_t); block score = max over the
// block's causal tokens; top-k blocks with ties to the lower block id.
//
// Work decomposition. A "tile" is a set of query rows that read the same keys:
// one row (index path) or up to 8 consecutive rows of one request (verify /
// prefill path). Every tile owns ceil(len/128) blocks of 128 keys; the blocks
// of all tiles are laid end to end and the persistent grid cuts that sequence
// into equal contiguous ranges, one per CTA, so a 450K-token request is spread
// over every SM exactly like the short ones.
//
// Inner loop (tcgen05). A warpgroup owns a block of 128 keys at a time: its
// 128 threads each dequantise one key (e2m1 x E4M3 -> f16, exact) straight from
// the bulk-copied (TMA) page in shared memory into tensor memory, which is the
// A operand (M = 128 keys) of tcgen05.mma kind::f16; B is the tile's queries
// (N = 16 heads x rows) in shared memory; the f32 scores accumulate in tensor
// memory and come back with tcgen05.ld, one key per thread, for the
// ReLU-weighted head sum and the block maximum.
#include <cuda_runtime.h>

#include "m3s_device.cuh"

namespace m3s {
namespace {

constexpr int kStages = 3;                                      // per warpgroup
constexpr int kStageBytes = kPageCodeBytes + kPageScaleBytes;   // one block: 9216
constexpr int kMaxTiles = 8192;

// Warpgroups per CTA and the tensor-memory plan: per warpgroup 64 columns of
// A (128 keys x 128 dims of f16) and N = 16 * QT columns of f32 scores.
template <int QT>
struct Cfg {
  static constexpr int kWG = QT == 1 ? 4 : 2;
  static constexpr int kThreads = kWG * 128;
  static constexpr int kN = 16 * QT;
  static constexpr int kACols = kHeadDim / 2;
  static constexpr int kWGCols = kACols + kN;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kQBytes = kN * kHeadDim * 2;
};

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

template <int QT>
struct __align__(128) ScoreSmem {
  uint8_t stage[Cfg<QT>::kWG][kStages][kStageBytes];
  uint8_t bq[Cfg<QT>::kQBytes];  // B operand: queries, f16, K-major, no swizzle
  uint64_t sbar[Cfg<QT>::kWG][kStages];
  uint64_t mbar[Cfg<QT>::kWG];
  float blkmax[Cfg<QT>::kWG][4][QT];
  float wsm[QT * 16];
  int lensm[QT];
  int svalid[Cfg<QT>::kWG][kStages];
  int abort_wg[Cfg<QT>::kWG];
  uint32_t tmem_base;
  int qbad;
};

template <int QT>
size_t score_smem_bytes(int ntiles) {
  return sizeof(ScoreSmem<QT>) + (ntiles + 1) * 4 + 128;
}

// B layout: core matrix (8 rows x 8 f16 = 128 B) for K-chunk kc (dims 8kc ..
// 8kc+7) and row group rg sits at (kc * N/8 + rg) * 128 B: the K-direction
// stride (LBO) is 16 N bytes, the row-group stride (SBO) 128 bytes.
template <int QT>
__device__ __forceinline__ uint32_t bq_offset(int n, int kc) {
  return (kc * (Cfg<QT>::kN / 8) + (n >> 3)) * 128 + (n & 7) * 16;
}

template <int QT>
__global__ void __launch_bounds__(Cfg<QT>::kThreads, 1) score_kernel(const ScoreArgs a) {
  using C = Cfg<QT>;
  constexpr uint32_t kIdesc = idesc_f16(128, C::kN);
  extern __shared__ __align__(128) uint8_t smem_raw[];
  ScoreSmem<QT>& sm = *reinterpret_cast<ScoreSmem<QT>*>(smem_raw);
  int* pre = reinterpret_cast<int*>(smem_raw + sizeof(ScoreSmem<QT>));
  __shared__ int red[C::kThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wg = warp >> 2, wq = warp & 3;  // warpgroup; quarter = TMEM lanes 32wq .. 32wq+31
  const int wtid = tid & 127;               // = key index within the block
  const bool issuer = wtid == 0;
  const int bar_id = 1 + wg;

  // ---- prologue: barriers and tensor memory (touches no input) ----
  if (tid < C::kWG * kStages) mbar_init(&sm.sbar[tid / kStages][tid % kStages], 1);
  if (tid < C::kWG) {
    mbar_init(&sm.mbar[tid], 1);
    sm.abort_wg[tid] = 0;
  }
  if (tid == 0) sm.qbad = 0;
  if (warp == 0) tmem_alloc(&sm.tmem_base, C::kTmemCols);
  mbar_fence_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t a_tm = tmem + wg * C::kWGCols;  // lane 0, first A column of this warpgroup
  const uint32_t d_tm = a_tm + C::kACols;        // lane 0, first score column
  const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
  pdl_trigger();
  pdl_wait();

  // ---- exclusive prefix of block counts over tiles (block-wide scan) ----
  const int ntiles = a.ntiles;
  const int per = (ntiles + C::kThreads - 1) / C::kThreads;
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

  const long long N = pre[ntiles];
  const int lo = static_cast<int>(N * blockIdx.x / gridDim.x);
  const int hi = static_cast<int>(N * (blockIdx.x + 1) / gridDim.x);
  int tile = 0;
  {
    int l = 0, h = ntiles;  // pre[l] <= lo < pre[h]
    while (h - l > 1) {
      const int m = (l + h) >> 1;
      if (pre[m] <= lo) l = m; else h = m;
    }
    tile = l;
  }

  uint32_t sphase = 0;    // expected parity per stage of this warpgroup
  uint32_t mphase = 0;    // expected parity of the MMA barrier
  uint32_t pending = 0;   // issuer: stages with a copy not yet waited for
  bool mma_pending = false;
  float wreg[16];

  int pos = lo;
  while (pos < hi) {
    while (pre[tile + 1] <= pos) ++tile;
    const int seg_lo = pos - pre[tile];
    const int seg_hi = min(hi, pre[tile + 1]) - pre[tile];
    const TileInfo<QT> ti = tile_info<QT>(a, tile, false);

    // ---- stage the tile's queries (the B operand), weights and lengths ----
    __syncthreads();
    for (int e = tid; e < C::kN * 16; e += C::kThreads) {
      const int n = e >> 4, kc = e & 15;
      const int rho = n >> 4, h = n & 15;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (rho < ti.nrows && h < a.Hi) {
        const uint4 raw = *reinterpret_cast<const uint4*>(
            a.q_idx + (static_cast<size_t>(ti.row0 + rho) * a.Hi + h) * kHeadDim + 8 * kc);
        bool bad = false;
        v.x = bf16x2_to_f16x2(raw.x, bad);
        v.y = bf16x2_to_f16x2(raw.y, bad);
        v.z = bf16x2_to_f16x2(raw.z, bad);
        v.w = bf16x2_to_f16x2(raw.w, bad);
        if (bad) sm.qbad = 1;
      }
      *reinterpret_cast<uint4*>(sm.bq + bq_offset<QT>(n, kc)) = v;
    }
    for (int e = tid; e < QT * 16; e += C::kThreads) {
      const int rho = e >> 4, h = e & 15;
      sm.wsm[e] = (rho < ti.nrows && h < a.Hi) ? a.w[static_cast<size_t>(ti.row0 + rho) * a.Hi + h] : 0.f;
    }
    if (tid < QT) sm.lensm[tid] = tid < ti.nrows ? a.row_len[ti.row0 + tid] : 0;
    fence_proxy_async();  // the queries are read by the tensor core (async proxy)
    __syncthreads();
    int rlen[QT];
#pragma unroll
    for (int rho = 0; rho < QT; ++rho) rlen[rho] = sm.lensm[rho];
    if constexpr (QT == 1) {
#pragma unroll
      for (int h = 0; h < 16; ++h) wreg[h] = sm.wsm[h];
    }

    // ---- this warpgroup's blocks: seg_lo + wg + k * kWG ----
    const int first = seg_lo + wg;
    const int count = first < seg_hi ? (seg_hi - first + C::kWG - 1) / C::kWG : 0;
    const int32_t* bt_row = a.block_table + static_cast<size_t>(ti.req) * a.bt_stride;

    auto issue = [&](int k) {  // issuer thread only
      const int s = k % kStages;
      const int page = bt_row[first + k * C::kWG];
      int ok = 0;
      if (page < 0 || page >= a.num_pages) {
        raise(a.err, M3S_DEVERR_PAGE);
      } else if (!sm.abort_wg[wg]) {
        fence_proxy_async();
        mbar_expect_tx(&sm.sbar[wg][s], kStageBytes);
        bulk_g2s(sm.stage[wg][s], a.codes + static_cast<size_t>(page) * kPageCodeBytes,
                 kPageCodeBytes, &sm.sbar[wg][s]);
        bulk_g2s(sm.stage[wg][s] + kPageCodeBytes,
                 a.scales + static_cast<size_t>(page) * kPageScaleBytes, kPageScaleBytes,
                 &sm.sbar[wg][s]);
        pending |= 1u << s;
        ok = 1;
      }
      sm.svalid[wg][s] = ok;
    };
    if (issuer)
      for (int k = 0; k < count && k < kStages; ++k) issue(k);
    named_bar_sync(bar_id, 128);

    for (int k = 0; k < count; ++k) {
      const int s = k % kStages;
      const int blk = first + k * C::kWG;
      const bool issued = sm.svalid[wg][s] != 0;
      const bool valid = issued && !sm.abort_wg[wg];
      if (valid) {
        if (!mbar_wait(&sm.sbar[wg][s], (sphase >> s) & 1u)) {
          sm.abort_wg[wg] = 1;
          raise(a.err, M3S_DEVERR_TIMEOUT);
        } else if (issuer) {
          pending &= ~(1u << s);
        }
        // dequantise key wtid into A (TMEM lane = key, column i = dims 2i, 2i+1)
        const uint8_t* cs = sm.stage[wg][s];
        const uint8_t* ss = cs + kPageCodeBytes;
        const uint4* kp = reinterpret_cast<const uint4*>(cs + wtid * kCodeBytes);
        const uint2 sc = *reinterpret_cast<const uint2*>(ss + wtid * kScaleBytes);
        const uint32_t s01 = e4m3x2_to_f16x2(sc.x & 0xFFFFu), s23 = e4m3x2_to_f16x2(sc.x >> 16);
        const uint32_t s45 = e4m3x2_to_f16x2(sc.y & 0xFFFFu), s67 = e4m3x2_to_f16x2(sc.y >> 16);
        const uint32_t spair[4] = {s01, s23, s45, s67};
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // chunk c = dims 32c .. 32c+31 = scale groups 2c, 2c+1
          const uint4 wv = kp[c];
          const uint32_t g0 = bcast_lo(spair[c]), g1 = bcast_hi(spair[c]);
          uint32_t v[16];
          e2m1x8_to_f16x2(wv.x, v[0], v[1], v[2], v[3]);
          e2m1x8_to_f16x2(wv.y, v[4], v[5], v[6], v[7]);
          e2m1x8_to_f16x2(wv.z, v[8], v[9], v[10], v[11]);
          e2m1x8_to_f16x2(wv.w, v[12], v[13], v[14], v[15]);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = hmul2(v[i], g0);
#pragma unroll
          for (int i = 8; i < 16; ++i) v[i] = hmul2(v[i], g1);
          tmem_st16(lane_base + a_tm + 16 * c, v);
        }
        tmem_wait_st();
      }
      if (issued) sphase ^= 1u << s;
      tc_fence_before();
      named_bar_sync(bar_id, 128);
      const bool go = valid && !sm.abort_wg[wg];
      if (issuer) {
        if (k + kStages < count) issue(k + kStages);  // stage s has been read by all
        if (go) {
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t bdesc = smem_desc_noswizzle(sm.bq + ks * 32 * C::kN, 16 * C::kN, 128);
            tc_mma_ts(d_tm, a_tm + 8 * ks, bdesc, kIdesc, ks > 0 ? 1u : 0u);
          }
          tc_commit(&sm.mbar[wg]);
          mma_pending = true;
        }
      }
      if (go) {
        if (!mbar_wait(&sm.mbar[wg], mphase & 1u)) {
          sm.abort_wg[wg] = 1;
          raise(a.err, M3S_DEVERR_TIMEOUT);
        } else if (issuer) {
          mma_pending = false;
        }
        mphase ^= 1u;
        tc_fence_after();
        const int tok = blk * kPage + wtid;
#pragma unroll
        for (int rho = 0; rho < QT; ++rho) {
          float d[16];
          tmem_ld16(lane_base + d_tm + 16 * rho, d);
          tmem_wait_ld();
          float sc = 0.f;
          if constexpr (QT == 1) {
#pragma unroll
            for (int h = 0; h < 16; ++h) sc = fmaf(wreg[h], fmaxf(d[h], 0.f), sc);
          } else {
            const float4* w4 = reinterpret_cast<const float4*>(sm.wsm + 16 * rho);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float4 wv = w4[q4];
              sc = fmaf(wv.x, fmaxf(d[4 * q4 + 0], 0.f), sc);
              sc = fmaf(wv.y, fmaxf(d[4 * q4 + 1], 0.f), sc);
              sc = fmaf(wv.z, fmaxf(d[4 * q4 + 2], 0.f), sc);
              sc = fmaf(wv.w, fmaxf(d[4 * q4 + 3], 0.f), sc);
            }
          }
          float m = tok < rlen[rho] ? sc : -INFINITY;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) sm.blkmax[wg][wq][rho] = m;
        }
      }
      tc_fence_before();
      named_bar_sync(bar_id, 128);
      if (wtid < QT) {
        const int rho = wtid;
        if (rho < ti.nrows && blk * kPage < rlen[rho]) {
          float m = -INFINITY;
          if (go) {
#pragma unroll
            for (int q = 0; q < 4; ++q) m = fmaxf(m, sm.blkmax[wg][q][rho]);
          }
          a.bscores[static_cast<size_t>(ti.row0 + rho) * a.bs_stride + blk] = m;
        }
      }
    }
    pos = pre[tile] + seg_hi;
    ++tile;
  }

  // ---- leave: drain anything still in flight after a timeout, free TMEM ----
  if (issuer) {
    for (int s = 0; s < kStages; ++s)
      if (pending & (1u << s)) mbar_wait(&sm.sbar[wg][s], (sphase >> s) & 1u);
    if (mma_pending) mbar_wait(&sm.mbar[wg], mphase & 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && sm.qbad) raise(a.err, M3S_DEVERR_QRANGE);
}

// ---- top-k over block scores: one CTA per row, exact radix select ----
// Keys are 64-bit (ordered score bits, then the complemented block id), all
// distinct. The leading bytes every key shares are skipped; then one byte per
// pass from the top: a histogram of the byte over the keys that still match
// the chosen prefix locates the bin holding the k-th largest key; keys in
// higher bins are in, lower bins out. The loop stops as soon as the bin's keys
// are exactly the ones still needed (at the latest on the last byte).
constexpr int kTopkThreads = 1024;

__device__ __forceinline__ unsigned long long topk_key_at(const float* row, const unsigned long long* keys,
                                                        bool in_smem, int i) {
  return in_smem ? keys[i] : topk_key(row[i], i);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(
    const float* __restrict__ bscores, int bs_stride, const int32_t* __restrict__ row_req,
    const int32_t* __restrict__ row_len, int B, int bt_stride, int topk, int smem_keys,
    int32_t* __restrict__ ids) {
  extern __shared__ unsigned long long keys[];
  __shared__ unsigned int hist[256];
  __shared__ unsigned long long wmax[kTopkThreads / 32], wmin[kTopkThreads / 32];
  __shared__ unsigned long long sh_prefix, sh_mask;
  __shared__ int sh_krem, sh_done, sh_shift, nsel;
  __shared__ int sel[M3S_MAX_TOPK];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int len = row_len[r];
  const int req = row_req ? row_req[r] : 0;
  const bool ok = len > 0 && req >= 0 && req < B && len <= bt_stride * kPage;
  const int nb = ok ? (len + kPage - 1) / kPage : 0;
  const int cnt = min(topk, nb);
  int32_t* out = ids + static_cast<size_t>(r) * topk;
  for (int i = cnt + tid; i < topk; i += kTopkThreads) out[i] = -1;
  if (cnt == 0) return;
  if (cnt == nb) {  // every block is selected: ids 0 .. nb-1
    for (int i = tid; i < nb; i += kTopkThreads) out[i] = i;
    return;
  }
  const float* row = bscores + static_cast<size_t>(r) * bs_stride;
  const bool in_smem = nb <= smem_keys;
  unsigned long long kmax = 0, kmin = ~0ull;
  for (int i = tid; i < nb; i += kTopkThreads) {
    const unsigned long long key = topk_key(row[i], i);
    if (in_smem) keys[i] = key;
    kmax = key > kmax ? key : kmax;
    kmin = key < kmin ? key : kmin;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long x = __shfl_xor_sync(0xffffffffu, kmax, o);
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, kmin, o);
    kmax = x > kmax ? x : kmax;
    kmin = y < kmin ? y : kmin;
  }
  if (lane == 0) {
    wmax[warp] = kmax;
    wmin[warp] = kmin;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 0; w < kTopkThreads / 32; ++w) {
      kmax = wmax[w] > kmax ? wmax[w] : kmax;
      kmin = wmin[w] < kmin ? wmin[w] : kmin;
    }
    const int common = (__clzll(static_cast<long long>(kmax ^ kmin)) / 8) * 8;  // shared leading bits
    const unsigned long long mask = common ? ~0ull << (64 - common) : 0ull;
    sh_prefix = kmax & mask;
    sh_mask = mask;
    sh_shift = 56 - common;
    sh_krem = cnt;
    sh_done = 0;
    nsel = 0;
  }
  __syncthreads();

  for (int shift = sh_shift; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += kTopkThreads) hist[b] = 0;
    const unsigned long long prefix = sh_prefix, mask = sh_mask;
    const int krem = sh_krem;
    __syncthreads();
    for (int i = tid; i < nb; i += kTopkThreads) {
      const unsigned long long key = topk_key_at(row, keys, in_smem, i);
      if ((key & mask) == prefix) atomicAdd(&hist[static_cast<unsigned>(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      int loc = 0;
#pragma unroll
      for (int d = 0; d < 8; ++d) loc += hist[8 * tid + d];
      int suf = loc;  // sum over lanes >= this one
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_down_sync(0xffffffffu, suf, o);
        if (tid + o < 32) suf += u;
      }
      int above = suf - loc;
#pragma unroll
      for (int d = 7; d >= 0; --d) {
        const int bin = 8 * tid + d;
        const int h = hist[bin];
        if (above < krem && above + h >= krem) {
          sh_prefix = prefix | (static_cast<unsigned long long>(bin) << shift);
          sh_mask = mask | (255ull << shift);
          sh_krem = krem - above;
          sh_done = (h == krem - above);
        }
        above += h;
      }
    }
    __syncthreads();
    if (sh_done) break;
  }
  const unsigned long long prefix = sh_prefix, mask = sh_mask;
  for (int i = tid; i < nb; i += kTopkThreads) {
    const unsigned long long key = topk_key_at(row, keys, in_smem, i);
    if ((key & mask) >= prefix) {
      const int slot = atomicAdd(&nsel, 1);
      if (slot < M3S_MAX_TOPK) sel[slot] = i;
    }
  }
  __syncthreads();
  if (tid < cnt) {
    const int mine = sel[tid];
    int rank = 0;
    for (int j = 0; j < cnt; ++j) rank += sel[j] < mine;
    out[rank] = mine;
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t topk_smem(int bt_stride, int* keys_out) {
  const int k = bt_stride < 12288 ? bt_stride : 12288;
  *keys_out = k;
  return static_cast<size_t>(k) * 8;
}

template <int QT>
int launch_score(const ScoreArgs& a, cudaStream_t st) {
  const size_t smem = score_smem_bytes<QT>(a.ntiles);
  if (smem > 227 * 1024) return M3S_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(score_kernel<QT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return M3S_ERR_LAUNCH;
  return launch_kernel(score_kernel<QT>, dim3(sm_count()), dim3(Cfg<QT>::kThreads), smem, st, 0, a) ==
                 cudaSuccess
             ? M3S_OK
             : M3S_ERR_LAUNCH;
}

int launch_topk(const float* bscores, int bs_stride, const int32_t* row_req, const int32_t* row_len,
                int R, int B, int bt_stride, int topk, int32_t* ids, cudaStream_t st) {
  int keys = 0;
  const size_t smem = topk_smem(bt_stride, &keys);
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return M3S_ERR_LAUNCH;
  return launch_kernel(topk_kernel, dim3(R), dim3(kTopkThreads), smem, st, 0, bscores, bs_stride,
                       row_req, row_len, B, bt_stride, topk, keys, ids) == cudaSuccess
             ? M3S_OK
             : M3S_ERR_LAUNCH;
}

int check_common(const uint16_t* q_idx, const float* w, int Hi, const m3s_nvfp4_plane& idx_k,
                 const int32_t* block_table, int bt_stride, int R, int B, int topk,
                 const int32_t* topk_ids) {
  if (R < 0 || B < 0 || topk < 0 || bt_stride < 0) return M3S_ERR_INVALID;
  if (Hi < 1 || Hi > M3S_MAX_INDEX_HEADS || topk > M3S_MAX_TOPK) return M3S_ERR_UNSUPPORTED;
  if (idx_k.num_heads != 1 || idx_k.num_pages < 0) return M3S_ERR_INVALID;
  if (R == 0) return M3S_OK;
  if (!q_idx || !w || !topk_ids || (B > 0 && (!block_table || bt_stride < 1))) return M3S_ERR_INVALID;
  if (!aligned16(q_idx) || (idx_k.num_pages > 0 && (!idx_k.codes || !idx_k.scales ||
                                                    !aligned16(idx_k.codes) || !aligned16(idx_k.scales))))
    return M3S_ERR_INVALID;
  return M3S_OK;
}

}  // namespace
}  // namespace m3s

extern "C" int m3s_index_block_scores(const uint16_t* q_idx, const float* w, int32_t Hi,
                                      m3s_nvfp4_plane idx_k, const int32_t* block_table,
                                      int32_t bt_stride, const int32_t* row_req,
                                      const int32_t* row_len, int32_t R, int32_t B,
                                      float* block_scores, int32_t bs_stride, int32_t* err,
                                      void* stream) {
  using namespace m3s;
  int32_t dummy_ids = 0;
  const int rc = check_common(q_idx, w, Hi, idx_k, block_table, bt_stride, R, B, 0, &dummy_ids);
  if (rc != M3S_OK || R == 0) return rc;
  if (!row_req || !row_len || !block_scores || bs_stride < bt_stride || bs_stride < 1)
    return M3S_ERR_INVALID;
  if (R > kMaxTiles) return M3S_ERR_UNSUPPORTED;
  if (B == 0) return M3S_OK;
  ScoreArgs a{q_idx, w, Hi, idx_k.codes, idx_k.scales, idx_k.num_pages, block_table, bt_stride,
              row_req, nullptr, row_len, R, B, R, 1, block_scores, bs_stride, err};
  return launch_score<1>(a, static_cast<cudaStream_t>(stream));
}

extern "C" int m3s_block_topk(const float* block_scores, int32_t bs_stride, const int32_t* row_req,
                              const int32_t* row_len, int32_t R, int32_t B, int32_t bt_stride,
                              int32_t topk, int32_t* topk_ids, void* stream) {
  using namespace m3s;
  if (R < 0 || B < 0 || topk < 0 || bt_stride < 0 || bs_stride < bt_stride) return M3S_ERR_INVALID;
  if (topk > M3S_MAX_TOPK) return M3S_ERR_UNSUPPORTED;
  if (R == 0 || topk == 0) return M3S_OK;
  if (!row_len || !topk_ids || (B > 0 && !block_scores)) return M3S_ERR_INVALID;
  return launch_topk(block_scores, bs_stride > 0 ? bs_stride : 1, row_req, row_len, R, B,
                     bt_stride, topk, topk_ids, static_cast<cudaStream_t>(stream));
}

extern "C" int m3s_index_score_topk(const uint16_t* q_idx, const float* w, int32_t Hi,
                                    m3s_nvfp4_plane idx_k, const int32_t* block_table,
                                    int32_t bt_stride, const int32_t* row_req,
                                    const int32_t* row_len, int32_t R, int32_t B, int32_t topk,
                                    int32_t* topk_ids, float* block_scores, void* ws,
                                    size_t ws_bytes, int32_t* err, void* stream) {
  using namespace m3s;
  int rc = check_common(q_idx, w, Hi, idx_k, block_table, bt_stride, R, B, topk, topk_ids);
  if (rc != M3S_OK || R == 0) return rc;
  if (!row_req || !row_len) return M3S_ERR_INVALID;
  if (R > kMaxTiles) return M3S_ERR_UNSUPPORTED;
  if (topk == 0) return M3S_OK;
  const int stride = bt_stride > 0 ? bt_stride : 1;
  float* bs = block_scores;
  if (!bs) {
    if (ws_bytes < m3s_workspace_bytes(M3S_OP_INDEX_SCORE_TOPK, R, B, bt_stride, 0, 0, Hi, topk, 1))
      return M3S_ERR_WORKSPACE;
    if (!ws || !aligned16(ws)) return M3S_ERR_INVALID;
    bs = static_cast<float*>(ws);
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B > 0) {
    ScoreArgs a{q_idx, w, Hi, idx_k.codes, idx_k.scales, idx_k.num_pages, block_table, bt_stride,
                row_req, nullptr, row_len, R, B, R, 1, bs, stride, err};
    rc = launch_score<1>(a, st);
    if (rc != M3S_OK) return rc;
  }
  return launch_topk(bs, stride, row_req, row_len, R, B, bt_stride, topk, topk_ids, st);
}

extern "C" int m3s_verify_score_topk(const uint16_t* q_idx, const float* w, int32_t Hi,
                                     m3s_nvfp4_plane idx_k, const int32_t* block_table,
                                     int32_t bt_stride, const int32_t* cu_q,
                                     const int32_t* row_len, int32_t B, int32_t R, int32_t max_q,
                                     int32_t topk, int32_t* topk_ids, void* ws, size_t ws_bytes,
                                     int32_t* err, void* stream) {
  using namespace m3s;
  int rc = check_common(q_idx, w, Hi, idx_k, block_table, bt_stride, R, B, topk, topk_ids);
  if (rc != M3S_OK || R == 0) return rc;
  if (!cu_q || !row_len || max_q < 0) return M3S_ERR_INVALID;
  if (topk == 0 || B == 0) {
    if (topk > 0) {
      // no requests: every row is padding
      return launch_topk(nullptr, 1, nullptr, row_len, R, 0, bt_stride, topk, topk_ids,
                         static_cast<cudaStream_t>(stream));
    }
    return M3S_OK;
  }
  const int cpr = max_q > 0 ? (max_q + 7) / 8 : 1;
  const long long ntiles = static_cast<long long>(B) * cpr;
  if (ntiles > kMaxTiles) return M3S_ERR_UNSUPPORTED;
  if (ws_bytes < m3s_workspace_bytes(M3S_OP_VERIFY_SCORE_TOPK, R, B, bt_stride, 0, 0, Hi, topk, max_q))
    return M3S_ERR_WORKSPACE;
  if (!ws || !aligned16(ws)) return M3S_ERR_INVALID;
  float* bs = static_cast<float*>(ws);
  ScoreArgs a{q_idx, w, Hi, idx_k.codes, idx_k.scales, idx_k.num_pages, block_table, bt_stride,
              nullptr, cu_q, row_len, R, B, static_cast<int>(ntiles), cpr, bs, bt_stride, err};
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = launch_score<8>(a, st);
  if (rc != M3S_OK) return rc;
  return launch_topk(bs, bt_stride, nullptr, row_len, R, B, bt_stride, topk, topk_ids, st);
}
