// Lightning-indexer scoring over paged NVFP4 index keys with block top-k.
//
// "[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (ROCm/ATOM
// #2744): Design / Index (FP4 index keys decoded to fp16 in registers),
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
// Inner loop. Each warp streams whole blocks (9216 B: 8192 B of codes + 1024 B
// of scales) into its own double-buffered shared-memory stages with 1-D bulk
// copies (TMA) and an mbarrier, dequantises e2m1 x E4M3 to fp16 in registers
// (exact) and feeds mma.sync m16n8k16 with the 16 keys of an m-tile as M and
// (row, head) pairs as N. The head dimension is walked in a permuted order so
// that every thread's key bytes are one contiguous 16-byte chunk; the query
// fragments use the same permutation, which leaves every dot product unchanged.
#include <cuda_runtime.h>

#include "m3s_device.cuh"

namespace m3s {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;
constexpr int kStageBytes = kPageCodeBytes + kPageScaleBytes;  // 9216
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

struct __align__(16) ScoreSmem {
  uint8_t stage[kWarps][kStages][kStageBytes];
  uint64_t bar[kWarps][kStages];
};

// Shared-memory layout: ScoreSmem | q fragments (8 k-steps x NT n-tiles x 32 lanes
// x 8 B) | w (QT x 16 floats) | row lengths (QT ints) | tile prefix (ntiles+1 ints).
template <int QT>
__host__ __device__ constexpr int qfrag_bytes() { return 8 * (2 * QT) * 32 * 8; }

template <int QT>
size_t score_smem_bytes(int ntiles) {
  return sizeof(ScoreSmem) + qfrag_bytes<QT>() + QT * 16 * 4 + QT * 4 + (ntiles + 1) * 4 + 16;
}

template <int QT>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const ScoreArgs a) {
  constexpr int NT = 2 * QT;  // n8 tiles of (row, head) columns
  extern __shared__ __align__(128) uint8_t smem_raw[];
  ScoreSmem& sm = *reinterpret_cast<ScoreSmem*>(smem_raw);
  uint2* qfrag = reinterpret_cast<uint2*>(smem_raw + sizeof(ScoreSmem));
  float* wsm = reinterpret_cast<float*>(smem_raw + sizeof(ScoreSmem) + qfrag_bytes<QT>());
  int* lensm = reinterpret_cast<int*>(wsm + QT * 16);
  int* pre = lensm + QT;
  __shared__ int red[kWarps];
  __shared__ int qbad;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  if (tid < kWarps * kStages) mbar_init(&sm.bar[tid / kStages][tid % kStages], 1);
  if (tid == 0) qbad = 0;
  mbar_fence_init();

  // ---- exclusive prefix of block counts over tiles (block-wide scan) ----
  const int ntiles = a.ntiles;
  const int per = (ntiles + kThreads - 1) / kThreads;
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
  if (lo >= hi) return;

  // first tile with pre[t+1] > lo
  int tile = 0;
  {
    int l = 0, h = ntiles;  // pre[l] <= lo < pre[h]
    while (h - l > 1) {
      const int m = (l + h) >> 1;
      if (pre[m] <= lo) l = m; else h = m;
    }
    tile = l;
  }

  uint32_t phase_bits = 0;  // per-stage mbarrier parity of this warp
  bool aborted = false;
  uint32_t qa[8][NT == 2 ? 2 : 1][2];  // decode path: q fragments kept in registers
  (void)qa;

  int pos = lo;
  while (pos < hi) {
    while (pre[tile + 1] <= pos) ++tile;
    const int seg_lo = pos - pre[tile];
    const int seg_hi = min(hi, pre[tile + 1]) - pre[tile];
    const TileInfo<QT> ti = tile_info<QT>(a, tile, false);

    // ---- stage the tile's queries (fp16, fragment order) and weights ----
    __syncthreads();
    for (int e = tid; e < 8 * NT * 32; e += kThreads) {
      const int ln = e & 31, c = (e >> 5) % NT, j = (e >> 5) / NT;
      const int col = 8 * c + (ln >> 2), tt = ln & 3;
      const int rho = col >> 4, h = col & 15;
      uint2 v = make_uint2(0u, 0u);
      if (rho < ti.nrows && h < a.Hi) {
        const uint2 raw = *reinterpret_cast<const uint2*>(
            a.q_idx + (static_cast<size_t>(ti.row0 + rho) * a.Hi + h) * kHeadDim + 32 * tt + 4 * j);
        bool bad = false;
        v.x = bf16x2_to_f16x2(raw.x, bad);
        v.y = bf16x2_to_f16x2(raw.y, bad);
        if (bad) qbad = 1;
      }
      qfrag[e] = v;
    }
    for (int e = tid; e < QT * 16; e += kThreads) {
      const int rho = e >> 4, h = e & 15;
      wsm[e] = (rho < ti.nrows && h < a.Hi) ? a.w[static_cast<size_t>(ti.row0 + rho) * a.Hi + h] : 0.f;
    }
    if (tid < QT) lensm[tid] = tid < ti.nrows ? a.row_len[ti.row0 + tid] : 0;
    __syncthreads();

    float wreg[QT][4];
    int rlen[QT];
#pragma unroll
    for (int rho = 0; rho < QT; ++rho) {
      wreg[rho][0] = wsm[rho * 16 + 2 * t];
      wreg[rho][1] = wsm[rho * 16 + 2 * t + 1];
      wreg[rho][2] = wsm[rho * 16 + 8 + 2 * t];
      wreg[rho][3] = wsm[rho * 16 + 9 + 2 * t];
      rlen[rho] = lensm[rho];
    }
    if constexpr (NT == 2) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint2 v = qfrag[(j * NT + c) * 32 + lane];
          qa[j][c][0] = v.x;
          qa[j][c][1] = v.y;
        }
    }

    // ---- this warp's blocks of the segment: seg_lo + warp + k * kWarps ----
    const int first = seg_lo + warp;
    const int count = first < seg_hi ? (seg_hi - first + kWarps - 1) / kWarps : 0;
    const int32_t* bt_row = a.block_table + static_cast<size_t>(ti.req) * a.bt_stride;
    uint32_t valid_bits = 0;

    auto issue = [&](int k) {
      const int s = k & 1;
      const int blk = first + k * kWarps;
      int ok = 0;
      if (lane == 0 && !aborted) {
        const int page = bt_row[blk];
        if (page < 0 || page >= a.num_pages) {
          raise(a.err, M3S_DEVERR_PAGE);
        } else {
          fence_proxy_async();
          mbar_expect_tx(&sm.bar[warp][s], kStageBytes);
          bulk_g2s(sm.stage[warp][s], a.codes + static_cast<size_t>(page) * kPageCodeBytes,
                   kPageCodeBytes, &sm.bar[warp][s]);
          bulk_g2s(sm.stage[warp][s] + kPageCodeBytes,
                   a.scales + static_cast<size_t>(page) * kPageScaleBytes, kPageScaleBytes,
                   &sm.bar[warp][s]);
          ok = 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      valid_bits = (valid_bits & ~(1u << s)) | (static_cast<uint32_t>(ok) << s);
    };

    if (count > 0) issue(0);
    if (count > 1) issue(1);
    for (int k = 0; k < count; ++k) {
      const int s = k & 1;
      const int blk = first + k * kWarps;
      bool have = (valid_bits >> s) & 1u;
      if (have) {
        const bool done = mbar_wait(&sm.bar[warp][s], (phase_bits >> s) & 1u);
        phase_bits ^= 1u << s;
        if (!done) {
          if (lane == 0) raise(a.err, M3S_DEVERR_TIMEOUT);
          aborted = true;
          have = false;
          // give the copies still in flight one more bounded wait before leaving
          mbar_wait(&sm.bar[warp][s], (phase_bits >> s) & 1u ^ 1u);
          if (k + 1 < count && ((valid_bits >> (s ^ 1)) & 1u))
            mbar_wait(&sm.bar[warp][s ^ 1], (phase_bits >> (s ^ 1)) & 1u);
          valid_bits = 0;
        }
      }
      float best[QT];
#pragma unroll
      for (int rho = 0; rho < QT; ++rho) best[rho] = -INFINITY;

      if (have) {
        const uint8_t* cs = sm.stage[warp][s];
        const uint8_t* ss = cs + kPageCodeBytes;
#pragma unroll 1
        for (int mt = 0; mt < 8; ++mt) {
          const int key0 = mt * 16 + g;
          const uint4 ca = *reinterpret_cast<const uint4*>(cs + key0 * kCodeBytes + 16 * t);
          const uint4 cb = *reinterpret_cast<const uint4*>(cs + (key0 + 8) * kCodeBytes + 16 * t);
          const uint32_t sa = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(ss + key0 * kScaleBytes + 2 * t));
          const uint32_t sb = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(ss + (key0 + 8) * kScaleBytes + 2 * t));
          const uint32_t sa0 = bcast_lo(sa), sa1 = bcast_hi(sa);
          const uint32_t sb0 = bcast_lo(sb), sb1 = bcast_hi(sb);
          const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w};
          const uint32_t wb[4] = {cb.x, cb.y, cb.z, cb.w};
          float acc[NT][4];
#pragma unroll
          for (int c = 0; c < NT; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            // bytes 2j, 2j+1 of the thread's chunk = dims 32t+4j .. 32t+4j+3,
            // scale group 2t + (j >= 4)
            const uint32_t xa = wa[j >> 1] >> (16 * (j & 1));
            const uint32_t xb = wb[j >> 1] >> (16 * (j & 1));
            const uint32_t scA = j < 4 ? sa0 : sa1, scB = j < 4 ? sb0 : sb1;
            const uint32_t a0 = hmul2(e2m1x2_to_f16x2(xa & 0xFFu), scA);
            const uint32_t a2 = hmul2(e2m1x2_to_f16x2((xa >> 8) & 0xFFu), scA);
            const uint32_t a1 = hmul2(e2m1x2_to_f16x2(xb & 0xFFu), scB);
            const uint32_t a3 = hmul2(e2m1x2_to_f16x2((xb >> 8) & 0xFFu), scB);
#pragma unroll
            for (int c = 0; c < NT; ++c) {
              uint32_t b0, b1;
              if constexpr (NT == 2) {
                b0 = qa[j][c][0];
                b1 = qa[j][c][1];
              } else {
                const uint2 v = qfrag[(j * NT + c) * 32 + lane];
                b0 = v.x;
                b1 = v.y;
              }
              mma16816(acc[c], a0, a1, a2, a3, b0, b1);
            }
          }
          // token scores of keys key0 and key0 + 8 for each row of the tile
          const int tok0 = blk * kPage + key0;
#pragma unroll
          for (int rho = 0; rho < QT; ++rho) {
            const float* w4 = wreg[rho];
            float p0 = w4[0] * fmaxf(acc[2 * rho][0], 0.f) + w4[1] * fmaxf(acc[2 * rho][1], 0.f) +
                       w4[2] * fmaxf(acc[2 * rho + 1][0], 0.f) + w4[3] * fmaxf(acc[2 * rho + 1][1], 0.f);
            float p1 = w4[0] * fmaxf(acc[2 * rho][2], 0.f) + w4[1] * fmaxf(acc[2 * rho][3], 0.f) +
                       w4[2] * fmaxf(acc[2 * rho + 1][2], 0.f) + w4[3] * fmaxf(acc[2 * rho + 1][3], 0.f);
            p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
            p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
            if (tok0 < rlen[rho]) best[rho] = fmaxf(best[rho], p0);
            if (tok0 + 8 < rlen[rho]) best[rho] = fmaxf(best[rho], p1);
          }
        }
      }
#pragma unroll
      for (int rho = 0; rho < QT; ++rho) {
        float m = best[rho];
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (lane == 0 && rho < ti.nrows && blk * kPage < rlen[rho])
          a.bscores[static_cast<size_t>(ti.row0 + rho) * a.bs_stride + blk] = m;
      }
      __syncwarp();
      if (k + 2 < count) issue(k + 2);
    }
    pos = pre[tile] + seg_hi;
    ++tile;
  }
  __syncthreads();
  if (tid == 0 && qbad) raise(a.err, M3S_DEVERR_QRANGE);
}

// ---- top-k over block scores: one CTA per row ----
// Round i picks the largest key below the previous pick (keys are distinct:
// the block id sits in the low half), so nothing has to be removed.
constexpr int kTopkThreads = 256;

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(
    const float* __restrict__ bscores, int bs_stride, const int32_t* __restrict__ row_req,
    const int32_t* __restrict__ row_len, int B, int bt_stride, int topk, int smem_keys,
    int32_t* __restrict__ ids) {
  extern __shared__ unsigned long long keys[];
  __shared__ unsigned long long wbest[kTopkThreads / 32];
  __shared__ int sel[M3S_MAX_TOPK];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int len = row_len[r];
  const int req = row_req ? row_req[r] : 0;
  const bool ok = len > 0 && req >= 0 && req < B && len <= bt_stride * kPage;
  const int nb = ok ? (len + kPage - 1) / kPage : 0;
  const float* row = bscores + static_cast<size_t>(r) * bs_stride;
  const bool in_smem = nb <= smem_keys;
  if (in_smem)
    for (int i = tid; i < nb; i += kTopkThreads) keys[i] = topk_key(row[i], i);
  __syncthreads();
  const int cnt = min(topk, nb);
  unsigned long long prev = ~0ull;
  for (int k = 0; k < cnt; ++k) {
    unsigned long long best = 0;
    for (int i = tid; i < nb; i += kTopkThreads) {
      const unsigned long long key = in_smem ? keys[i] : topk_key(row[i], i);
      if (key < prev && key > best) best = key;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long v = __shfl_xor_sync(0xffffffffu, best, o);
      best = v > best ? v : best;
    }
    if (lane == 0) wbest[warp] = best;
    __syncthreads();
    best = wbest[0];
#pragma unroll
    for (int wv = 1; wv < kTopkThreads / 32; ++wv) best = wbest[wv] > best ? wbest[wv] : best;
    if (tid == 0) sel[k] = key_id(best);
    prev = best;
    __syncthreads();
  }
  // write ascending ids, then -1 padding
  if (tid < topk) {
    int out = -1;
    if (tid < cnt) {
      const int mine = sel[tid];
      int rank = 0;
      for (int j = 0; j < cnt; ++j) rank += sel[j] < mine;
      ids[static_cast<size_t>(r) * topk + rank] = mine;
    } else {
      ids[static_cast<size_t>(r) * topk + tid] = out;
    }
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
  score_kernel<QT><<<sm_count(), kThreads, smem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? M3S_OK : M3S_ERR_LAUNCH;
}

int launch_topk(const float* bscores, int bs_stride, const int32_t* row_req, const int32_t* row_len,
                int R, int B, int bt_stride, int topk, int32_t* ids, cudaStream_t st) {
  int keys = 0;
  const size_t smem = topk_smem(bt_stride, &keys);
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return M3S_ERR_LAUNCH;
  topk_kernel<<<R, kTopkThreads, smem, st>>>(bscores, bs_stride, row_req, row_len, B, bt_stride,
                                             topk, keys, ids);
  return cudaGetLastError() == cudaSuccess ? M3S_OK : M3S_ERR_LAUNCH;
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
