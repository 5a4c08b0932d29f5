// Index scorer for single-row tiles (decode rows), on mma.sync tensor cores.
//
// "[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (ROCm/ATOM
// #2744), Design / Index and Decode score grid: score[t] = sum_h w_h *
// ReLU(q_h . k_t) over NVFP4 index keys decoded to 16-bit, block score = max
// over the block's causal tokens, work spread so a long request cannot
// serialise the kernel.
//
// With one query row per tile the product has only 16 columns (the index
// heads), which is far too narrow for tcgen05.mma (every M128 x K16
// instruction costs about the same time up to N = 128). The warp-level
// m16n8k16 instruction fits this shape: the 16 keys of an m-tile are M, the
// 16 heads two n8 tiles, and K walks the head dimension in a permuted order so
// every thread's key bytes are one contiguous 16-byte chunk (the query
// fragments use the same order, which leaves every dot product unchanged).
//
// MXFP4 keys (one E8M0 scale per 32 elements) take the same loop: a thread's
// 16-byte chunk of a key is exactly one of its four 32-element groups, so the
// chunk is scaled by 2^(E_t - E_max) (E_max = the key's largest exponent; exact
// in fp16 while the key's exponents span at most 23) and the key's score by
// 2^(E_max - 127) in fp32 after the head sum. When a half lands, its warp turns
// each key's four E8M0 bytes into those factors once (two keys per lane, into a
// per-warp scratch), so the tile loop only loads them.
//
// Each of the 16 warps streams whole blocks of its share (every 16th block of
// the CTA's contiguous range) as two halves of 64 keys through its own
// double-buffered shared-memory stages, filled by 1-D bulk copies (TMA) that
// complete on an mbarrier. Block-table entries are fetched 32 at a time.
//
// The CTA ranges are cut in a cost space where every row costs its blocks plus
// kSegCost: each row segment a CTA takes on pays a fixed set-up (its query row
// and first block-table entries come from HBM), so a CTA whose range spans two
// rows is given that many fewer blocks.
#include <cuda_runtime.h>

#include "m3s_score_common.cuh"

namespace m3s {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;                                    // per warp
constexpr int kHalfKeys = 64;                                 // keys per stage
constexpr int kHalfCodeBytes = kHalfKeys * kCodeBytes;        // 4096
constexpr int kHalfScaleBytes = kHalfKeys * kScaleBytes;      // 512
constexpr int kStageBytes = kHalfCodeBytes + kHalfScaleBytes; // 4608
constexpr int kQFragWords = 8 * 2 * 32;                       // k-steps x n-tiles x lanes (uint2)
constexpr int kSegCost = 6;                                   // set-up of a row segment, in blocks
constexpr int kSegCostStreaming = 14;   // ... plus its candidates' merge and ticket (streaming top-k)
static_assert(kQFragWords == kThreads, "one query fragment word per thread");

// MXFP4 factors of one warp's current half: per key the fp16x2 factor of each
// of its four groups and its fp32 2^(E_max - 127).
struct MxScratch {
  uint32_t fac[kWarps][kHalfKeys][4];
  float key[kWarps][kHalfKeys];
};

struct __align__(16) DecodeSmem {
  uint8_t stage[kWarps][kStages][kStageBytes];
  uint64_t bar[kWarps][kStages];
  uint2 qfrag[kQFragWords];
  float w[16];           // the row's weights times 2^(e_h - e_ref)
  unsigned qmax[2][16];  // per head: the largest query magnitude's BF16 bits (by segment parity)
  float escale;          // 2^e_ref: the row's block maxima are scaled back by it
  unsigned long long wlist[kWarps][64];   // the warps' top-k lists at a segment's end
  int vslot[kMaxGrid + 32];   // candidate slots of a tile being merged
  int fin;
  int len;
  int qbad;
};

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <bool MX>
__global__ void __launch_bounds__(kThreads, 1) score_decode_kernel(const ScoreArgs a) {
  constexpr int kKeyScaleBytes = MX ? kMxScaleBytes : kScaleBytes;
  constexpr int kHalfScaleB = kHalfKeys * kKeyScaleBytes;  // 256 or 512
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);
  MxScratch& mxs = *reinterpret_cast<MxScratch*>(smem_raw + sizeof(DecodeSmem));   // MX only
  TileLayout L;
  L.bind(smem_raw + sizeof(DecodeSmem) + (MX ? sizeof(MxScratch) : 0), a.ntiles,
         a.cand ? kSegCostStreaming : kSegCost);
  const int* pre = L.pre;
  __shared__ int red[kWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  if (tid < kWarps * kStages) mbar_init(&sm.bar[tid / kStages][tid % kStages], 1);
  if (tid == 0) {
    sm.qbad = 0;
    sm.fin = 0;
  }
  if (tid < 32) (&sm.qmax[0][0])[tid] = 0u;
  mbar_fence_init();
  __syncthreads();
  // The next kernel may launch once every CTA has signalled. Its CTAs then wait
  // for this grid on SMs this grid has freed; with the streaming top-k the grid
  // ends with a few CTAs merging candidates, so those signal only when their
  // blocks are scored (early waiting CTAs of the next kernel were measured to
  // slow the step down).
  const bool late = a.cand && !a.meta;   // the grid ends merging candidates
  if (!late) pdl_trigger();
  // Before the wait, each CTA brings its share of the queries, weights and
  // block table into L2: the set-up after the wait is a chain of dependent
  // loads, each a DRAM miss after an L2 flush otherwise. (A hint only: a line
  // an earlier kernel writes later is updated in L2, which every read goes
  // through.)
  if (tid == 0) {
    prefetch_share_l2(a.q_idx, static_cast<size_t>(a.R) * a.Hi * kHeadDim * 2);
    prefetch_share_l2(a.w, static_cast<size_t>(a.R) * a.Hi * 4);
    prefetch_share_l2(a.block_table, static_cast<size_t>(a.B) * a.bt_stride * 4);
  }
  pdl_wait();

  tile_prefix<1>(a, L, red, kThreads);
  const int ntiles = a.ntiles;
  if (a.cand) write_unscored_rows<1>(a, L, kThreads);
  const int2 range = L.cta_range(blockIdx.x);
  const int lo = range.x, hi = range.y;
  int tile = tile_at(pre, ntiles, lo);
  if (late && lo >= hi) pdl_trigger();   // no blocks

  uint32_t phase_bits = 0;  // per-stage mbarrier parity of this warp
  bool aborted = false;

  int pos = lo;
  int par = 0;   // parity of this CTA's segment count (selects the qmax buffer)
  while (pos < hi) {
    while (pre[tile + 1] <= pos) ++tile;
    const int seg_lo = pos - pre[tile];
    const int seg_hi = min(hi, pre[tile + 1]) - pre[tile];
    const TileInfo<1> ti = tile_info<1>(a, tile, false);
    if (a.meta && seg_lo == 0 && tid == 0) {   // this CTA holds the tile's first block
      const int2 cc = L.covering_ctas(tile, L.g);
      if (cc.x != static_cast<int>(blockIdx.x)) raise(a.err, M3S_DEVERR_ROW);   // (invariant)
      a.meta[tile] = make_int2(tile + cc.x, cc.y - cc.x + 1);   // its lists: consecutive slots
    }

    // ---- the row's queries (one fragment word per thread), weights and length:
    // the loads go out first, so their round trip overlaps the block-table
    // fetch of the first copies below ----
    uint2 qraw = make_uint2(0u, 0u);
    int hq = -1;   // the head of this thread's query word (-1: none)
    {
      const int ln = tid & 31, c = (tid >> 5) & 1, j = tid >> 6;
      const int h = 8 * c + (ln >> 2), tt = ln & 3;
      if (ti.nrows && h < a.Hi) {
        qraw = *reinterpret_cast<const uint2*>(
            a.q_idx + (static_cast<size_t>(ti.row0) * a.Hi + h) * kHeadDim + 32 * tt + 4 * j);
        hq = h;
      }
    }
    const float wrow = (tid < 16 && ti.nrows && tid < a.Hi) ? a.w[static_cast<size_t>(ti.row0) * a.Hi + tid] : 0.f;
    const int lrow = (tid == 0 && ti.nrows) ? a.row_len[ti.row0] : 0;

    // ---- a range that goes on into the next row warms L2 with that row's
    // queries and first block-table entries while this segment runs ----
    const int next_pos = pre[tile] + seg_hi;
    if (warp == kWarps - 1 && next_pos < hi) {
      int nt = tile + 1;
      while (pre[nt + 1] <= next_pos) ++nt;
      const TileInfo<1> tn = tile_info<1>(a, nt, false);
      if (tn.nrows) {
        if (lane * 64 < a.Hi * kHeadDim)
          prefetch_l2(a.q_idx + static_cast<size_t>(tn.row0) * a.Hi * kHeadDim + lane * 64);
        const int j0 = next_pos - pre[nt] + 32 * lane;
        if (lane < 16 && j0 < min(hi, pre[nt + 1]) - pre[nt])
          prefetch_l2(a.block_table + static_cast<size_t>(tn.req) * a.bt_stride + j0);
      }
    }

    // ---- this warp's blocks: every kWarps-th block of the segment, two halves
    // each, the warp order carried on from the CTA's previous segment (so a
    // range over two rows does not give the low warps an extra block in each);
    // its first two copies go out before the queries are staged ----
    const int rot = (pos - lo) % kWarps;
    const int first = seg_lo + (warp - rot + kWarps) % kWarps;
    const int count = first < seg_hi ? (seg_hi - first + kWarps - 1) / kWarps : 0;
    const int nhalf = 2 * count;
    const int32_t* bt_row = a.block_table + static_cast<size_t>(ti.req) * a.bt_stride;
    PageWindow pw;
    uint32_t valid_bits = 0;

    auto issue = [&](int hh) {  // all lanes (the page window is warp-wide)
      const int s = hh & 1;
      const int blk = first + (hh >> 1) * kWarps;
      const int half = hh & 1;
      const int page = pw.get(bt_row, blk, kWarps, seg_hi, lane);   // (warp-uniform)
      const bool ok = !aborted && page >= 0 && page < a.num_pages;
      if (lane == 0 && !aborted) {
        if (!ok) {
          if (half == 0) raise(a.err, M3S_DEVERR_PAGE);
        } else {
          // (no proxy fence: every generic read of this stage has returned, its
          // values having gone through the mma and the shuffles above)
          mbar_expect_tx(&sm.bar[warp][s], kHalfCodeBytes + kHalfScaleB);
          bulk_g2s(sm.stage[warp][s],
                   a.codes + static_cast<size_t>(page) * kPageCodeBytes + half * kHalfCodeBytes,
                   kHalfCodeBytes, &sm.bar[warp][s]);
          bulk_g2s(sm.stage[warp][s] + kHalfCodeBytes,
                   a.scales + static_cast<size_t>(page) * (kPage * kKeyScaleBytes) + half * kHalfScaleB,
                   kHalfScaleB, &sm.bar[warp][s]);
        }
      }
      valid_bits = (valid_bits & ~(1u << s)) | (static_cast<uint32_t>(ok) << s);
    };

    if (nhalf > 0) issue(0);
    if (nhalf > 1) issue(1);

    // ---- the queries to fp16 in fragment order, each head scaled by 2^-e_h
    // (its largest magnitude taken over the CTA with shared-memory atomics);
    // the previous segment's readers are past the first barrier ----
    if (hq >= 0) {
      const unsigned m = max(bf16x2_absmax_bits(qraw.x), bf16x2_absmax_bits(qraw.y));
      if (m) atomicMax(&sm.qmax[par][hq], m);
    }
    __syncthreads();
    if (tid < 16) sm.qmax[par ^ 1][tid] = 0u;   // the next segment's (its last readers are done)
    {
      uint2 v = make_uint2(0u, 0u);
      if (hq >= 0) {
        const unsigned m = sm.qmax[par][hq];
        if (m >= kBf16InfBits) sm.qbad = 1;
        if (m) {
          const QScale sc = q_scale(q_scale_exp(min(m, kBf16InfBits - 1)));
          v.x = bf16x2_to_f16x2_scaled(qraw.x, sc);
          v.y = bf16x2_to_f16x2_scaled(qraw.y, sc);
        }
      }
      sm.qfrag[tid] = v;
    }
    if (warp == 0) {
      // score = 2^e_ref * sum_h (w_h 2^(e_h - e_ref)) ReLU(scaled dot product),
      // e_ref the largest e_h over the heads that contribute
      int eh = kQNoExp;
      if (lane < 16 && ti.nrows && lane < a.Hi) {
        const unsigned m = sm.qmax[par][lane];
        if (m && wrow != 0.f) eh = q_scale_exp(min(m, kBf16InfBits - 1));
      }
      const int eref = __reduce_max_sync(0xffffffffu, eh);
      if (lane < 16) sm.w[lane] = eh == kQNoExp ? 0.f : wrow * exp2i_f32(max(eh - eref, -150));
      if (lane == 0) sm.escale = eref == kQNoExp ? 1.f : exp2i_f32(eref);
    }
    if (tid == 0) sm.len = lrow;
    __syncthreads();

    const float w0 = sm.w[2 * t], w1 = sm.w[2 * t + 1], w2 = sm.w[8 + 2 * t], w3 = sm.w[9 + 2 * t];
    const float escale = sm.escale;
    const int rlen = sm.len;
    const int nbr = (rlen + kPage - 1) / kPage;   // the row's blocks (forced-block rule)
    // a slice of the request's blocks (context parallelism): local block j is the
    // request's block j + boff, and token positions and ids are the request's
    const int boff = (a.blk_base && ti.nrows) ? a.blk_base[ti.req] : 0;
    WarpTopk list;   // this warp's running top-k of the segment's blocks
    list.clear();
    uint32_t qa[8][2][2];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint2 v = sm.qfrag[(j * 2 + c) * 32 + lane];
        qa[j][c][0] = v.x;
        qa[j][c][1] = v.y;
      }

    float best = -INFINITY;
    for (int hh = 0; hh < nhalf; ++hh) {
      const int s = hh & 1;
      const int blk = first + (hh >> 1) * kWarps;
      const int half = hh & 1;
      if (half == 0) best = -INFINITY;
      bool have = (valid_bits >> s) & 1u;
      if (have) {
        // every lane waits; the warp takes one decision (the loop below is warp-collective)
        const bool done = __all_sync(0xffffffffu, mbar_wait(&sm.bar[warp][s], (phase_bits >> s) & 1u));
        phase_bits ^= 1u << s;
        if (!done) {
          if (lane == 0) raise(a.err, M3S_DEVERR_TIMEOUT);
          aborted = true;
          have = false;
          // give the copies still in flight one more bounded wait before leaving
          mbar_wait(&sm.bar[warp][s], ((phase_bits >> s) & 1u) ^ 1u);
          if (hh + 1 < nhalf && ((valid_bits >> (s ^ 1)) & 1u))
            mbar_wait(&sm.bar[warp][s ^ 1], (phase_bits >> (s ^ 1)) & 1u);
          valid_bits = 0;
        }
      }
      if (have) {
        const uint8_t* cs = sm.stage[warp][s];
        const uint8_t* ss = cs + kHalfCodeBytes;
        if constexpr (MX) {
          // the half's per-key factors, two keys per lane (the previous half's
          // readers are this warp's lanes, all past the loop below)
#pragma unroll
          for (int kk = lane; kk < kHalfKeys; kk += 32) {
            const uint32_t w4 = *reinterpret_cast<const uint32_t*>(ss + kk * kMxScaleBytes);
            const int em = e8m0_max4(w4);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              mxs.fac[warp][kk][j] = pow2_neg_f16x2(em - static_cast<int>((w4 >> (8 * j)) & 0xFFu));
            mxs.key[warp][kk] = pow2_f32(em - 127);
          }
          __syncwarp();
        }
        // (fully unrolled: the shared loads and the head-sum shuffles of one
        // m-tile overlap the others' conversions and products; 5% faster than
        // one m-tile at a time although ptxas then spills 12 bytes)
#pragma unroll
        for (int mt = 0; mt < kHalfKeys / 16; ++mt) {
          const int key0 = mt * 16 + g;
          const uint4 ca = *reinterpret_cast<const uint4*>(cs + key0 * kCodeBytes + 16 * t);
          const uint4 cb = *reinterpret_cast<const uint4*>(cs + (key0 + 8) * kCodeBytes + 16 * t);
          uint32_t sa0, sa1, sb0, sb1;
          float fa = 1.f, fb = 1.f;   // MXFP4: the keys' 2^(E_max - 127)
          if constexpr (MX) {   // this thread's chunk is group t of keys key0, key0 + 8
            sa0 = sa1 = mxs.fac[warp][key0][t];
            sb0 = sb1 = mxs.fac[warp][key0 + 8][t];
            fa = mxs.key[warp][key0];
            fb = mxs.key[warp][key0 + 8];
          } else {
            const uint32_t sa = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(ss + key0 * kScaleBytes + 2 * t));
            const uint32_t sb = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(ss + (key0 + 8) * kScaleBytes + 2 * t));
            sa0 = bcast_lo(sa);
            sa1 = bcast_hi(sa);
            sb0 = bcast_lo(sb);
            sb1 = bcast_hi(sb);
          }
          const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w};
          const uint32_t wb[4] = {cb.x, cb.y, cb.z, cb.w};
          float acc[2][4];
#pragma unroll
          for (int c = 0; c < 2; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) {
            // word jw of the thread's chunk = bytes 4jw .. 4jw+3 = k-steps 2jw
            // (bytes 4jw, 4jw+1) and 2jw+1 (bytes 4jw+2, 4jw+3); the chunk holds
            // dims 32t .. 32t+31, scale group 2t for words 0-1, 2t+1 for 2-3
            uint32_t xa[4], xb[4];
            e2m1x8_to_f16x2(wa[jw], xa[0], xa[1], xa[2], xa[3]);
            e2m1x8_to_f16x2(wb[jw], xb[0], xb[1], xb[2], xb[3]);
            const uint32_t scA = jw < 2 ? sa0 : sa1, scB = jw < 2 ? sb0 : sb1;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              xa[e] = hmul2(xa[e], scA);
              xb[e] = hmul2(xb[e], scB);
            }
#pragma unroll
            for (int js = 0; js < 2; ++js) {
              const int j = 2 * jw + js;
#pragma unroll
              for (int c = 0; c < 2; ++c)
                mma16816(acc[c], xa[2 * js], xb[2 * js], xa[2 * js + 1], xb[2 * js + 1], qa[j][c][0],
                         qa[j][c][1]);
            }
          }
          // token scores of keys key0 and key0 + 8
          float p0 = w0 * fmaxf(acc[0][0], 0.f) + w1 * fmaxf(acc[0][1], 0.f) +
                     w2 * fmaxf(acc[1][0], 0.f) + w3 * fmaxf(acc[1][1], 0.f);
          float p1 = w0 * fmaxf(acc[0][2], 0.f) + w1 * fmaxf(acc[0][3], 0.f) +
                     w2 * fmaxf(acc[1][2], 0.f) + w3 * fmaxf(acc[1][3], 0.f);
          p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
          p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
          p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
          p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
          if constexpr (MX) {
            p0 *= fa;
            p1 *= fb;
          }
          const int tok0 = (blk + boff) * kPage + half * kHalfKeys + key0;
          if (tok0 < rlen) best = fmaxf(best, p0);
          if (tok0 + 8 < rlen) best = fmaxf(best, p1);
        }
      }
      if (half == 1) {
        float m = best;
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (ti.nrows && (blk + boff) * kPage < rlen) {   // warp-uniform
          const float sc = m * escale;
          if (a.bscores && lane == 0) a.bscores[static_cast<size_t>(ti.row0) * a.bs_stride + blk] = sc;
          if (a.cand) list.insert(select_key(sc, blk + boff, nbr, a.init_blocks, a.local_blocks), a.topk, lane);
        }
      }
      __syncwarp();
      if (hh + 2 < nhalf) issue(hh + 2);
    }
    if (late && pre[tile] + seg_hi >= hi) pdl_trigger();   // this CTA's blocks are scored
    if (a.cand) {
      // the segment's candidates: the top k of the 16 warps' lists into slot
      // tile + CTA; then (unless the attention merges) the tile's ticket, and
      // the last CTA of the tile merges it
      unsigned long long* slot = a.cand + static_cast<size_t>(tile + blockIdx.x) * a.topk;
      // (a tree of pairwise bitonic merges: measured faster here than ranking
      // the 16 lists' keys by counting, 1.2 against 2.1 us a segment end)
      for (int half = kWarps / 2; half >= 1; half >>= 1) {
        if (warp >= half && warp < 2 * half) warp_store(list, &sm.wlist[warp][0], 64, lane);
        __syncthreads();
        if (warp < half) warp_merge2(list, warp_load(&sm.wlist[warp + half][0], 64, lane), a.topk, lane);
      }
      if (warp == 0) write_keys(list, a.topk, slot, lane);
      __syncthreads();
      if (!a.meta)
        tile_finish<1>(a, L, tile, seg_hi - seg_lo, reinterpret_cast<unsigned long long*>(&sm.stage[0][0][0]),
                       static_cast<int>(sizeof(sm.stage) / 8), sm.vslot, &sm.fin, kThreads);
    }
    pos = pre[tile] + seg_hi;
    ++tile;
    par ^= 1;
  }
  __syncthreads();
  if (tid == 0 && sm.qbad) raise(a.err, M3S_DEVERR_QRANGE);
}

}  // namespace

int launch_score_decode(const ScoreArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(DecodeSmem) + (a.mx ? sizeof(MxScratch) : 0) + TileLayout::bytes(a.ntiles) + 16;
  if (smem > 227 * 1024) return M3S_ERR_UNSUPPORTED;
  const auto kernel = a.mx ? score_decode_kernel<true> : score_decode_kernel<false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return M3S_ERR_LAUNCH;
  return launch_kernel(kernel, dim3(grid_size()), dim3(kThreads), smem, st, 0, a) ==
                 cudaSuccess
             ? M3S_OK
             : M3S_ERR_LAUNCH;
}

}  // namespace m3s
