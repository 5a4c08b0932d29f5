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
// Inner loop (tcgen05, warp-specialised). A producer warp streams whole
// blocks (8 KB of codes through a 2-D tensor map with 64-byte swizzle, so the
// per-key reads below are free of bank conflicts, plus 1 KB of scales) into a
// ring of shared-memory stages. Dequantising warpgroups turn a block into the
// A operand: each of their 128 threads decodes one key (e2m1 x E4M3 -> f16,
// exact) straight into its lane of a tensor-memory slot (M = 128 keys). One
// thread issues tcgen05.mma kind::f16 against the tile's queries in shared
// memory (B: N = 16 heads x rows) into a ring of tensor-memory accumulators,
// and an epilogue warpgroup reads the f32 scores back one key per thread for
// the ReLU-weighted head sum and the block maximum. mbarriers hand stages,
// A slots and accumulators from one role to the next, so no role waits on a
// round trip of another.
#include <cstddef>
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "m3s_score_common.cuh"

namespace m3s {
namespace {

// (a.x * b.x + c.x, a.y * b.y + c.y): two IEEE fma (round to nearest) in one
// packed f32x2 instruction.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 pa, pb, pc;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n"
      " mov.b64 pc, {%6, %7};\n fma.rn.f32x2 pc, pa, pb, pc;\n mov.b64 {%0, %1}, pc;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

constexpr int kStageBytes = kPageCodeBytes + kPageScaleBytes;  // one block: 9216 = 9 x 1024

// The CTA ranges are cut in a cost space where every tile costs its blocks plus
// kTileSetUp: a tile segment that a CTA takes on stages that tile's queries and
// refills the role pipeline after the CTA-wide barrier that ends its previous
// segment (about 5 us, some 7 blocks, on the verify batch), so a CTA whose
// range spans two tiles is given that many fewer blocks.
constexpr int kTileSetUp = 7;
// With the streaming top-k a segment's end also merges its candidates and
// arrives on the tile's ticket (and the last CTA of a tile merges it): charged
// as 3 more blocks.
constexpr int kTileSetUpStreaming = 10;

// Roles and resources. Warp 0: producer (bulk copies); warps 1 .. kND: MMA
// issuers, one per accumulator slot (block g -> issuer g % kND, so one issuer's
// commits overlap the other's MMAs); warps 1 + kND .. kND + 4 kNEpi: epilogue
// warpgroups (block g -> g % kNEpi, which owns accumulator slot g % kND); then
// kNDQ dequantising warpgroups. With the streaming top-k the epilogue (the
// busiest role) only stores each row's block maximum into the CTA's score
// scratch (L2-resident, reused every segment); at the segment's end one warp
// per row selects the row's top-k from it.
// Tensor memory: kNA A slots of 64 columns (128 keys x 128 f16) and kND
// accumulator slots of N = 16 * QT f32 columns.
template <int QT>
struct Cfg {
  static_assert(QT % 2 == 0 && QT <= 8, "rows per tile: an even count up to 8");
  static constexpr int kN = 16 * QT;
  // 15 warps: the register file is split over the four SM sub-partitions, so
  // at most four warps a partition keep 128 registers a thread (the kernel is
  // compiled for 512 threads to hold it there)
  static constexpr int kNDQ = 1;
  static constexpr int kNEpi = 2;
  static constexpr int kIssuers = kNEpi;  // == kND
  static constexpr int kWarps = 1 + kIssuers + 4 * kNEpi + 4 * kNDQ;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kBoundThreads = 512;
  static_assert(kThreads <= kBoundThreads, "register budget");
  // Stages and A slots are multiples of kNDQ: block g goes to warpgroup g % kNDQ,
  // stage g % kNS and slot g % kNA, so each stage and each slot is only ever used
  // by one warpgroup, in order, and a parity wait can never see a phase two back.
  static constexpr int kNS = 8;
  static constexpr int kNA = 4;
  static constexpr int kND = kNEpi;
  static constexpr int kACols = kHeadDim / 2;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kQBytes = kN * kHeadDim * 2;
  static_assert(kNA * kACols + kND * kN <= 512, "tensor memory plan exceeds 512 columns");
  static_assert(kNS % kNDQ == 0 && kNA % kNDQ == 0, "stages and slots must partition by warpgroup");
};

template <int QT>
struct __align__(1024) ScoreSmem {
  uint8_t stage[Cfg<QT>::kNS][kStageBytes];  // codes (swizzled, 1024-aligned) then scales
  uint8_t bq[Cfg<QT>::kQBytes];              // B operand: queries, f16, K-major, no swizzle
  uint64_t full[Cfg<QT>::kNS], empty[Cfg<QT>::kNS];
  uint64_t afull[Cfg<QT>::kNA], aempty[Cfg<QT>::kNA];
  uint64_t dfull[Cfg<QT>::kND], dempty[Cfg<QT>::kND];
  // order-preserving bits of per-warp block maxima, by accumulator slot and by the
  // parity of the warpgroup's block count: a buffer is written again only after
  // the warpgroup's next barrier, which its reader passes first
  uint32_t blkmax[Cfg<QT>::kND][2][4][QT];
  int vslot[kMaxGrid + 32];                   // candidate slots of a tile being merged
  int fin;
  alignas(16) float wsm[QT * 16];        // weights times 2^(e_h - e_ref) of their row (read as float4)
  int qexp[Cfg<QT>::kN];                 // per (row, head): the query scale exponent e_h
  float rowscale[QT];                    // per row: 2^e_ref, applied to its block maxima
  int lensm[QT];
  uint32_t tmem_base;
  int qbad;
  int abort;
};

static_assert(offsetof(ScoreSmem<8>, wsm) % 16 == 0, "the epilogue reads the weights as float4");
static_assert(offsetof(ScoreSmem<8>, full) % 8 == 0, "8-byte members");

template <int QT>
size_t score_smem_bytes(int ntiles) {
  return sizeof(ScoreSmem<QT>) + TileLayout::bytes(ntiles) + 1024;  // + alignment slack
}

// B layout: core matrix (8 rows x 8 f16 = 128 B) for K-chunk kc (dims 8kc ..
// 8kc+7) and row group rg sits at (kc * N/8 + rg) * 128 B: the K-direction
// stride (LBO) is 16 N bytes, the row-group stride (SBO) 128 bytes.
template <int QT>
__device__ __forceinline__ uint32_t bq_offset(int n, int kc) {
  return (kc * (Cfg<QT>::kN / 8) + (n >> 3)) * 128 + (n & 7) * 16;
}

// Bounded wait that gives up at once when the CTA has aborted; raises on timeout.
template <int QT>
__device__ __forceinline__ bool role_wait(ScoreSmem<QT>& sm, uint64_t* bar, uint32_t parity, int32_t* err) {
  if (*reinterpret_cast<volatile int*>(&sm.abort)) return false;
  if (mbar_wait(bar, parity)) return true;
  raise(err, M3S_DEVERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
  return false;
}

// MX: MXFP4 index keys (one E8M0 scale per 32 elements). The dequantising
// thread of a key scales each 32-dim chunk by 2^(E_chunk - E_max) in fp16 (exact
// while the key's exponents span at most 23), and the key's epilogue thread
// multiplies its head sums by 2^(E_max - 127), reading the key's four scale
// bytes from the plane itself (L2-resident: the stage holding them is recycled
// long before the epilogue runs).
template <int QT, bool MX>
__global__ void __launch_bounds__(Cfg<QT>::kBoundThreads, 1)
    score_kernel(const ScoreArgs a, const __grid_constant__ CUtensorMap codes_map) {
  using C = Cfg<QT>;
  constexpr int kPageScaleB = MX ? kMxPageScaleBytes : kPageScaleBytes;
  constexpr uint32_t kIdesc = idesc_f16(128, C::kN);
  extern __shared__ uint8_t smem_raw[];
  ScoreSmem<QT>& sm = *reinterpret_cast<ScoreSmem<QT>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TileLayout L;
  // (partials mode, meta set: candidate lists without the tiles' merges)
  const bool late = a.cand && !a.meta;   // the grid ends merging candidates
  L.bind(reinterpret_cast<uint8_t*>(&sm) + sizeof(ScoreSmem<QT>), a.ntiles,
         late ? kTileSetUpStreaming : kTileSetUp);
  const int* pre = L.pre;
  __shared__ int red[C::kWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;  // TMEM lane quarter

  // ---- prologue: barriers and tensor memory (touches no input) ----
  if (tid < C::kNS) {
    mbar_init(&sm.full[tid], 1);
    mbar_init(&sm.empty[tid], 128);
  }
  if (tid < C::kNA) {
    mbar_init(&sm.afull[tid], 128);
    mbar_init(&sm.aempty[tid], 1);
  }
  if (tid < C::kND) {
    mbar_init(&sm.dfull[tid], 1);
    mbar_init(&sm.dempty[tid], 128);
  }
  if (tid == 0) {
    sm.qbad = 0;
    sm.abort = 0;
    sm.fin = 0;
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, C::kTmemCols);
  mbar_fence_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // with the streaming top-k the next kernel is let launch only when this CTA's
  // blocks are scored (its waiting CTAs slowed the step when launched early)
  if (!late) pdl_trigger();
  pdl_wait();

  // ---- exclusive prefix of block counts over tiles, then this CTA's range ----
  tile_prefix<QT>(a, L, red, C::kThreads);
  const int ntiles = a.ntiles;
  if (a.cand) write_unscored_rows<QT>(a, L, C::kThreads);
  const int2 range = L.cta_range(blockIdx.x);
  const int lo = range.x, hi = range.y;
  int tile = tile_at(pre, ntiles, lo);
  if (late && lo >= hi) pdl_trigger();   // no blocks

  int g0 = 0;               // sequence number of the segment's first block in this CTA
  bool mma_issued = false;  // MMA thread: a commit may still be outstanding
  uint32_t last_d = 0, last_ud = 0;
  int pos = lo;
  while (pos < hi) {
    while (pre[tile + 1] <= pos) ++tile;
    const int seg_lo = pos - pre[tile];
    const int seg_hi = min(hi, pre[tile + 1]) - pre[tile];
    const int nseg = seg_hi - seg_lo;
    const TileInfo<QT> ti = tile_info<QT>(a, tile, false);
    const int32_t* bt_row = a.block_table + static_cast<size_t>(ti.req) * a.bt_stride;
    if (a.meta && seg_lo == 0 && tid < ti.nrows) {   // this CTA holds the tile's first block
      // row rho's lists: slots tile + c of the covering CTAs c, QT lists apart
      const int2 cc = L.covering_ctas(tile, L.g);
      if (cc.x != static_cast<int>(blockIdx.x)) raise(a.err, M3S_DEVERR_ROW);   // (invariant)
      a.meta[ti.row0 + tid] = make_int2((tile + cc.x) * QT + tid, cc.y - cc.x + 1);
    }

    // ---- stage the tile's queries (the B operand), weights and lengths. Each
    // (row, head) is scaled by 2^-e_h before its f16 conversion (its largest
    // magnitude from the 16 lanes of a half-warp, which hold its 16 chunks: both
    // loop bounds are multiples of 32, so whole warps iterate together) ----
    for (int e = tid; e < C::kN * 16; e += C::kThreads) {
      const int n = e >> 4, kc = e & 15;
      const int rho = n >> 4, h = n & 15;
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (rho < ti.nrows && h < a.Hi)
        raw = *reinterpret_cast<const uint4*>(
            a.q_idx + (static_cast<size_t>(ti.row0 + rho) * a.Hi + h) * kHeadDim + 8 * kc);
      unsigned m = max(max(bf16x2_absmax_bits(raw.x), bf16x2_absmax_bits(raw.y)),
                       max(bf16x2_absmax_bits(raw.z), bf16x2_absmax_bits(raw.w)));
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m >= kBf16InfBits) sm.qbad = 1;
      const int eh = m ? q_scale_exp(min(m, kBf16InfBits - 1)) : kQNoExp;
      if (m) {
        const QScale sc = q_scale(eh);
        v.x = bf16x2_to_f16x2_scaled(raw.x, sc);
        v.y = bf16x2_to_f16x2_scaled(raw.y, sc);
        v.z = bf16x2_to_f16x2_scaled(raw.z, sc);
        v.w = bf16x2_to_f16x2_scaled(raw.w, sc);
      }
      *reinterpret_cast<uint4*>(sm.bq + bq_offset<QT>(n, kc)) = v;
      if (kc == 0) sm.qexp[n] = eh;
    }
    if (tid < QT) sm.lensm[tid] = tid < ti.nrows ? a.row_len[ti.row0 + tid] : 0;
    fence_proxy_async();  // the queries are read by the tensor core (async proxy)
    __syncthreads();
    // score = 2^e_ref * sum_h (w_h 2^(e_h - e_ref)) ReLU(scaled dot product), per
    // row e_ref = the largest e_h over its contributing heads (the row's 16 heads
    // are a half-warp; QT * 16 is a multiple of 32)
    for (int e = tid; e < QT * 16; e += C::kThreads) {
      const int rho = e >> 4, h = e & 15;
      const float wv = (rho < ti.nrows && h < a.Hi) ? a.w[static_cast<size_t>(ti.row0 + rho) * a.Hi + h] : 0.f;
      const int eh = wv != 0.f ? sm.qexp[e] : kQNoExp;
      int eref = eh;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) eref = max(eref, __shfl_xor_sync(0xffffffffu, eref, o));
      sm.wsm[e] = eh == kQNoExp ? 0.f : wv * exp2i_f32(max(eh - eref, -150));
      if (h == 0) sm.rowscale[rho] = eref == kQNoExp ? 1.f : exp2i_f32(eref);
    }
    __syncthreads();

    if (warp == 0) {
      // ================= producer =================
      PageWindow pw;
      for (int j = 0; j < nseg; ++j) {
        const int g = g0 + j, s = g % C::kNS, u = g / C::kNS;
        const int page = pw.get(bt_row + seg_lo, j, 1, nseg, lane);
        int ok = 1;
        if (lane == 0) {
          if (!role_wait(sm, &sm.empty[s], (u & 1) ^ 1, a.err)) {
            ok = 0;
          } else if (page < 0 || page >= a.num_pages) {
            raise(a.err, M3S_DEVERR_PAGE);
            mbar_arrive(&sm.full[s]);  // nothing to copy: complete the phase empty
          } else {
            mbar_expect_tx(&sm.full[s], kPageCodeBytes + kPageScaleB);
            tma_load_2d(sm.stage[s], &codes_map, 0, page * kPage, &sm.full[s]);
            bulk_g2s(sm.stage[s] + kPageCodeBytes,
                     a.scales + static_cast<size_t>(page) * kPageScaleB, kPageScaleB,
                     &sm.full[s]);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
    } else if (warp <= C::kIssuers) {
      // ================= MMA issuers (issuer i: blocks g with g % kND == i) =================
      const int iss = warp - 1;
      if (lane == 0) {
        for (int j = ((iss - g0) % C::kND + C::kND) % C::kND; j < nseg; j += C::kND) {
          const int g = g0 + j;
          const int as = g % C::kNA, ua = g / C::kNA, ds = g % C::kND, ud = g / C::kND;
          if (!role_wait(sm, &sm.afull[as], ua & 1, a.err)) break;
          if (!role_wait(sm, &sm.dempty[ds], (ud & 1) ^ 1, a.err)) break;
          tc_fence_after();
          const uint32_t a_tm = tmem + as * C::kACols;
          const uint32_t d_tm = tmem + C::kNA * C::kACols + ds * C::kN;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t bdesc = smem_desc_noswizzle(sm.bq + ks * 32 * C::kN, 16 * C::kN, 128);
            tc_mma_ts(d_tm, a_tm + 8 * ks, bdesc, kIdesc, ks > 0 ? 1u : 0u);
          }
          tc_commit(&sm.dfull[ds]);
          tc_commit(&sm.aempty[as]);
          mma_issued = true;
          last_d = ds;
          last_ud = ud;
        }
      }
    } else if (warp < 1 + C::kIssuers + 4 * C::kNEpi) {
      // ================= epilogue warpgroups =================
      // Per block: the accumulator (rows x 16 heads, one key per thread) in two
      // loads of half the rows each; the slot is released to the MMA as soon as
      // the second load has landed, before the second half is reduced. Each
      // row's weighted ReLU head sum runs as packed f32x2 fma (even heads in one
      // lane of the pair, odd heads in the other), and the block maximum over
      // the warp's 32 keys is one redux on order-preserving integer keys.
      const int ep = (warp - 1 - C::kIssuers) >> 2;          // warpgroup: blocks g with g % kNEpi == ep
      const int etid = tid - 32 * (1 + C::kIssuers) - 128 * ep;  // 0 .. 127 within the warpgroup
      const int wq = warp & 3;                   // lane quarter: keys 32 wq .. 32 wq + 31
      constexpr int kHalfRows = QT / 2;
      int rlen[QT];
      int rlen_min = INT_MAX;   // over the tile's rows: a block below it is causal for every row
#pragma unroll
      for (int rho = 0; rho < QT; ++rho) {
        rlen[rho] = sm.lensm[rho];
        if (rho < ti.nrows) rlen_min = min(rlen_min, rlen[rho]);
      }
      const float rscale = sm.rowscale[etid < QT ? etid : 0];   // this thread's row's 2^e_ref
      PageWindow pw;
      for (int j = ((ep - g0) % C::kNEpi + C::kNEpi) % C::kNEpi; j < nseg; j += C::kNEpi) {
        const int g = g0 + j, ds = g % C::kND, ud = g / C::kND;
        const int blk = seg_lo + j;
        const int page = pw.get(bt_row + seg_lo, j, C::kNEpi, nseg, lane);
        uint32_t kexp = 0;   // MX: the key's four E8M0 bytes, loaded while the MMA runs
        if constexpr (MX) {
          if (page >= 0 && page < a.num_pages)
            kexp = *reinterpret_cast<const uint32_t*>(
                a.scales + static_cast<size_t>(page) * kMxPageScaleBytes + (32 * wq + lane) * kMxScaleBytes);
        }
        const bool ok = __all_sync(0xffffffffu, role_wait(sm, &sm.dfull[ds], ud & 1, a.err));
        tc_fence_after();
        const int tok = blk * kPage + (32 * wq + lane);
        const uint32_t d_tm = tmem + C::kNA * C::kACols + ds * C::kN;
        float sc[QT];
#pragma unroll
        for (int rho = 0; rho < QT; ++rho) sc[rho] = 0.f;
        if (ok) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float d[16 * kHalfRows];
#pragma unroll
            for (int c = 0; c < kHalfRows / 2; ++c)
              tmem_ld32(lane_base + d_tm + 16 * kHalfRows * half + 32 * c,
                        *reinterpret_cast<float(*)[32]>(&d[32 * c]));
            tmem_wait_ld();
            reg_fence(d);
            if (half == 1) {
              tc_fence_before();
              mbar_arrive(&sm.dempty[ds]);
            }
#pragma unroll
            for (int r = 0; r < kHalfRows; ++r) {
              const int rho = kHalfRows * half + r;
              const float4* w4 = reinterpret_cast<const float4*>(sm.wsm + 16 * rho);
              // even heads in .x, odd heads in .y, one packed fma per head pair
              float2 s = make_float2(0.f, 0.f);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                const float4 wv = w4[q4];
                s = ffma2(make_float2(wv.x, wv.y),
                          make_float2(fmaxf(d[16 * r + 4 * q4 + 0], 0.f), fmaxf(d[16 * r + 4 * q4 + 1], 0.f)), s);
                s = ffma2(make_float2(wv.z, wv.w),
                          make_float2(fmaxf(d[16 * r + 4 * q4 + 2], 0.f), fmaxf(d[16 * r + 4 * q4 + 3], 0.f)), s);
              }
              sc[rho] = s.x + s.y;
            }
          }
          if constexpr (MX) {   // the key's 2^(E_max - 127): positive, so it commutes with ReLU
            const float kf = pow2_f32(e8m0_max4(kexp) - 127);
#pragma unroll
            for (int rho = 0; rho < QT; ++rho) sc[rho] *= kf;
          }
        } else {
          tc_fence_before();
          mbar_arrive(&sm.dempty[ds]);
        }
        if ((blk + 1) * kPage <= rlen_min) {   // (warp-uniform) every key is causal for every row
#pragma unroll
          for (int rho = 0; rho < QT; ++rho) {
            const uint32_t mx = __reduce_max_sync(0xffffffffu, ordered_bits(sc[rho]));
            if (lane == 0) sm.blkmax[ds][ud & 1][wq][rho] = mx;
          }
        } else {
#pragma unroll
          for (int rho = 0; rho < QT; ++rho) {
            const uint32_t key = ordered_bits(tok < rlen[rho] ? sc[rho] : -INFINITY);
            const uint32_t mx = __reduce_max_sync(0xffffffffu, key);
            if (lane == 0) sm.blkmax[ds][ud & 1][wq][rho] = mx;
          }
        }
        named_bar_sync(1 + ep, 128);
        if (*reinterpret_cast<volatile int*>(&sm.abort)) break;  // uniform: read after the barrier
        {
          // rows: threads 0 .. QT-1 of the warpgroup (its first warp's lanes)
          // take their block maxima right after the barrier
          if (etid < QT) {
            const int rho = etid;
            float m = -INFINITY;
            if (rho < ti.nrows && blk * kPage < rlen[rho]) {
              if (page >= 0 && page < a.num_pages) {
                uint32_t mk = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) mk = max(mk, sm.blkmax[ds][ud & 1][q][rho]);
                m = from_ordered_bits(mk) * rscale;
              }
              if (a.bscores) a.bscores[static_cast<size_t>(ti.row0 + rho) * a.bs_stride + blk] = m;
            }
            if (a.cand) a.seg_scores[(static_cast<size_t>(blockIdx.x) * QT + rho) * a.bt_stride + j] = m;
          }
        }
      }
    } else {
      // ================= dequantising warpgroups =================
      const int dq = (warp - 1 - C::kIssuers - 4 * C::kNEpi) >> 2;    // which warpgroup
      const int key = tid & 127;         // TMEM lane = key within the block
      const int sw = (key >> 1) & 3;     // 64-byte swizzle of this key's row
      PageWindow pw;
      // block g = g0 + j belongs to warpgroup g % kNDQ, whatever g0 the segment
      // starts at: each stage and A slot is then used by one warpgroup only
      for (int j = ((dq - g0) % C::kNDQ + C::kNDQ) % C::kNDQ; j < nseg; j += C::kNDQ) {
        const int g = g0 + j, s = g % C::kNS, us = g / C::kNS;
        const int as = g % C::kNA, ua = g / C::kNA;
        const int page = pw.get(bt_row + seg_lo, j, C::kNDQ, nseg, lane);
        // failed (timed-out) waits are made warp-uniform before any warp-collective op
        if (!__all_sync(0xffffffffu, role_wait(sm, &sm.full[s], us & 1, a.err))) break;
        if (!__all_sync(0xffffffffu, role_wait(sm, &sm.aempty[as], (ua & 1) ^ 1, a.err))) break;
        if (page >= 0 && page < a.num_pages) {
          const uint8_t* cs = sm.stage[s];
          const uint8_t* ss = cs + kPageCodeBytes;
          uint32_t spair[4];
          if constexpr (MX) {   // chunk c is E8M0 group c: one factor for both halves
            const uint32_t w4 = *reinterpret_cast<const uint32_t*>(ss + key * kMxScaleBytes);
            const int em = e8m0_max4(w4);
#pragma unroll
            for (int c = 0; c < 4; ++c) spair[c] = pow2_neg_f16x2(em - static_cast<int>((w4 >> (8 * c)) & 0xFFu));
          } else {
            const uint2 sc = *reinterpret_cast<const uint2*>(ss + key * kScaleBytes);
            spair[0] = e4m3x2_to_f16x2(sc.x & 0xFFFFu);
            spair[1] = e4m3x2_to_f16x2(sc.x >> 16);
            spair[2] = e4m3x2_to_f16x2(sc.y & 0xFFFFu);
            spair[3] = e4m3x2_to_f16x2(sc.y >> 16);
          }
          const uint32_t a_tm = tmem + as * C::kACols;
#pragma unroll
          for (int c = 0; c < 4; ++c) {  // chunk c = dims 32c .. 32c+31 = scale groups 2c, 2c+1
            const uint4 wv = *reinterpret_cast<const uint4*>(cs + key * kCodeBytes + 16 * (c ^ sw));
            const uint32_t g0s = MX ? spair[c] : bcast_lo(spair[c]);
            const uint32_t g1s = MX ? spair[c] : bcast_hi(spair[c]);
            uint32_t v[16];
            e2m1x8_to_f16x2(wv.x, v[0], v[1], v[2], v[3]);
            e2m1x8_to_f16x2(wv.y, v[4], v[5], v[6], v[7]);
            e2m1x8_to_f16x2(wv.z, v[8], v[9], v[10], v[11]);
            e2m1x8_to_f16x2(wv.w, v[12], v[13], v[14], v[15]);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = hmul2(v[i], g0s);
#pragma unroll
            for (int i = 8; i < 16; ++i) v[i] = hmul2(v[i], g1s);
            tmem_st16(lane_base + a_tm + 16 * c, v);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&sm.afull[as]);
        mbar_arrive(&sm.empty[s]);
      }
    }
    __syncthreads();  // every role is done with this segment (and its queries)
    if (late && pre[tile] + seg_hi >= hi) pdl_trigger();   // this CTA's blocks are scored
    if (a.cand) {
      // the segment's candidates: warp rho takes row rho's block maxima from the
      // CTA's score scratch 32 at a time and keeps their top-k (a key enters
      // only above the list's k-th), into slot tile + CTA; then the tile's
      // ticket (the last CTA of the tile merges it)
      if (warp < ti.nrows) {
        const int rho = warp;
        const int rl_r = sm.lensm[rho];
        const int nbr = (rl_r + kPage - 1) / kPage;
        const float* row_sc = a.seg_scores + (static_cast<size_t>(blockIdx.x) * QT + rho) * a.bt_stride;
        WarpTopk list;
        list.clear();
        // the maxima 32 x kListBatch at a time (their loads issued together);
        // a chunk with more than kInsertMax keys above the list's k-th is sorted
        // across the lanes and merged in (a bitonic split), fewer are inserted
        // one by one (the first chunks of a segment insert almost every key:
        // one at a time that took 11 us a segment on the verify batch)
        constexpr int kListBatch = 4, kInsertMax = 4;
        for (int j0 = 0; j0 < nseg; j0 += 32 * kListBatch) {
          unsigned long long key[kListBatch];
#pragma unroll
          for (int u = 0; u < kListBatch; ++u) {
            const int j = j0 + 32 * u + lane;
            const int blk = seg_lo + j;
            key[u] = (j < nseg && blk * kPage < rl_r)
                         ? select_key(__ldcg(row_sc + j), blk, nbr, a.init_blocks, a.local_blocks)
                         : 0ull;
          }
#pragma unroll
          for (int u = 0; u < kListBatch; ++u) {
            unsigned over = __ballot_sync(0xffffffffu, key[u] > list.kth);
            if (__popc(over) > kInsertMax) {
              WarpTopk c;
              c.a = key[u];
              c.b = 0ull;
              c.kth = 0ull;
              warp_sort_desc(c, 32, lane);   // the chunk, descending in slots 0 .. 31
              warp_merge2(list, c, a.topk, lane);
              list.kth = __shfl_sync(0xffffffffu, a.topk > 32 ? list.b : list.a, (a.topk - 1) & 31);
            } else {
              while (over) {   // ascending lanes: each key is inserted in turn
                const int l = __ffs(over) - 1;
                over &= over - 1;
                list.insert(__shfl_sync(0xffffffffu, key[u], l), a.topk, lane);
              }
            }
          }
        }
        write_keys(list, a.topk, a.cand + (static_cast<size_t>(tile + blockIdx.x) * QT + rho) * a.topk, lane);
      }
      __syncthreads();
      if (!a.meta)
        tile_finish<QT>(a, L, tile, nseg, reinterpret_cast<unsigned long long*>(&sm.stage[0][0]),
                        static_cast<int>(sizeof(sm.stage) / 8), sm.vslot, &sm.fin, C::kThreads);
    }
    g0 += nseg;
    pos = pre[tile] + seg_hi;
    ++tile;
  }

  // ---- leave: after a timeout, give the last MMA one more bounded wait; free TMEM ----
  if (warp >= 1 && warp <= C::kIssuers && lane == 0 && mma_issued && sm.abort)
    mbar_wait(&sm.dfull[last_d], last_ud & 1);
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

// Forced blocks (the first init blocks and the last local blocks of the row)
// rank above every score: their keys' high words, 0xFFFFFFFF (init) and
// 0xFFFFFFFE (local), sit above ordered_bits(+inf). Init keys keep the
// complemented id (lower id first), local keys the id itself (most recent
// first), so init + local beyond k keeps the row's newest blocks.
__device__ __forceinline__ unsigned long long block_key(const float* row, int i, int nb, int init, int local) {
  if (i < init) return (0xFFFFFFFFull << 32) | static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(i));
  if (i >= nb - local) return (0xFFFFFFFEull << 32) | static_cast<unsigned long long>(static_cast<uint32_t>(i));
  return topk_key(row[i], i);
}

__device__ __forceinline__ unsigned long long topk_key_at(const float* row, const unsigned long long* keys,
                                                        bool in_smem, int i, int nb, int init, int local) {
  return in_smem ? keys[i] : block_key(row, i, nb, init, local);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(
    const float* __restrict__ bscores, int bs_stride, const int32_t* __restrict__ row_req,
    const int32_t* __restrict__ row_len, int B, int bt_stride, int topk, int init_blocks,
    int local_blocks, int smem_keys, int32_t* __restrict__ ids) {
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
    const unsigned long long key = block_key(row, i, nb, init_blocks, local_blocks);
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
      const unsigned long long key = topk_key_at(row, keys, in_smem, i, nb, init_blocks, local_blocks);
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
    const unsigned long long key = topk_key_at(row, keys, in_smem, i, nb, init_blocks, local_blocks);
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

}  // namespace

// Tensor map over a one-head index code plane viewed as [num_pages * 128 rows]
// x [64 bytes], boxes of one page (128 rows), 64-byte swizzle.
bool make_codes_map(CUtensorMap* map, const uint8_t* codes, int num_pages) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kCodeBytes),
                              static_cast<cuuint64_t>(num_pages > 0 ? num_pages : 1) * kPage};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kCodeBytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kCodeBytes), static_cast<cuuint32_t>(kPage)};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

int grid_size() { return min(sm_count(), kMaxGrid); }

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The streaming top-k's workspace (sized by m3s_workspace_bytes): the tiles'
// tickets, then the candidate lists.
void bind_topk_workspace(ScoreArgs& a, void* ws, int ntiles, int topk, int init_blocks, int local_blocks,
                         int32_t* ids) {
  a.ticket = static_cast<unsigned*>(ws);
  a.cand = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + topk_ticket_bytes(ntiles));
  a.topk = topk;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  a.ids = ids;
}

size_t topk_smem(int bt_stride, int* keys_out) {
  const int k = bt_stride < 12288 ? bt_stride : 12288;
  *keys_out = k;
  return static_cast<size_t>(k) * 8;
}

template <int QT>
int launch_score(const ScoreArgs& a, cudaStream_t st) {
  const size_t smem = score_smem_bytes<QT>(a.ntiles);
  if (smem > 227 * 1024) return M3S_ERR_UNSUPPORTED;
  CUtensorMap map;
  if (a.num_pages > 0 && !make_codes_map(&map, a.codes, a.num_pages)) return M3S_ERR_LAUNCH;
  if (a.num_pages <= 0) memset(&map, 0, sizeof(map));
  const auto kernel = a.mx ? score_kernel<QT, true> : score_kernel<QT, false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return M3S_ERR_LAUNCH;
  return launch_kernel(kernel, dim3(grid_size()), dim3(Cfg<QT>::kThreads), smem, st, 0, a,
                       map) == cudaSuccess
             ? M3S_OK
             : M3S_ERR_LAUNCH;
}

int launch_topk(const float* bscores, int bs_stride, const int32_t* row_req, const int32_t* row_len,
                int R, int B, int bt_stride, int topk, int init_blocks, int local_blocks, int32_t* ids,
                cudaStream_t st) {
  int keys = 0;
  const size_t smem = topk_smem(bt_stride, &keys);
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return M3S_ERR_LAUNCH;
  return launch_kernel(topk_kernel, dim3(R), dim3(kTopkThreads), smem, st, 0, bscores, bs_stride,
                       row_req, row_len, B, bt_stride, topk, init_blocks, local_blocks, keys, ids) ==
                 cudaSuccess
             ? M3S_OK
             : M3S_ERR_LAUNCH;
}

int check_common(const uint16_t* q_idx, const float* w, int Hi, const m3s_fp4_plane& idx_k,
                 const int32_t* block_table, int bt_stride, int R, int B, int topk,
                 const int32_t* topk_ids) {
  if (R < 0 || B < 0 || topk < 0 || bt_stride < 0) return M3S_ERR_INVALID;
  if (idx_k.format != M3S_FMT_NVFP4 && idx_k.format != M3S_FMT_MXFP4) return M3S_ERR_INVALID;
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
                                      m3s_fp4_plane idx_k, const int32_t* block_table,
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
              row_req, nullptr, row_len, R, B, R, 1, block_scores, bs_stride, err,
              idx_k.format == M3S_FMT_MXFP4 ? 1 : 0};
  return launch_score_decode(a, static_cast<cudaStream_t>(stream));
}

extern "C" int m3s_block_topk(const float* block_scores, int32_t bs_stride, const int32_t* row_req,
                              const int32_t* row_len, int32_t R, int32_t B, int32_t bt_stride,
                              int32_t topk, int32_t init_blocks, int32_t local_blocks,
                              int32_t* topk_ids, void* stream) {
  using namespace m3s;
  if (R < 0 || B < 0 || topk < 0 || bt_stride < 0 || bs_stride < bt_stride) return M3S_ERR_INVALID;
  if (init_blocks < 0 || local_blocks < 0) return M3S_ERR_INVALID;
  if (topk > M3S_MAX_TOPK) return M3S_ERR_UNSUPPORTED;
  if (R == 0 || topk == 0) return M3S_OK;
  if (!row_len || !topk_ids || (B > 0 && !block_scores)) return M3S_ERR_INVALID;
  return launch_topk(block_scores, bs_stride > 0 ? bs_stride : 1, row_req, row_len, R, B,
                     bt_stride, topk, init_blocks, local_blocks, topk_ids,
                     static_cast<cudaStream_t>(stream));
}

extern "C" int m3s_index_score_topk(const uint16_t* q_idx, const float* w, int32_t Hi,
                                    m3s_fp4_plane idx_k, const int32_t* block_table,
                                    int32_t bt_stride, const int32_t* row_req,
                                    const int32_t* row_len, int32_t R, int32_t B, int32_t topk,
                                    int32_t init_blocks, int32_t local_blocks, int32_t* topk_ids,
                                    float* block_scores, void* ws, size_t ws_bytes, int32_t* err,
                                    void* stream) {
  using namespace m3s;
  int rc = check_common(q_idx, w, Hi, idx_k, block_table, bt_stride, R, B, topk, topk_ids);
  if (rc != M3S_OK || R == 0) return rc;
  if (!row_req || !row_len || init_blocks < 0 || local_blocks < 0) return M3S_ERR_INVALID;
  if (R > kMaxTiles) return M3S_ERR_UNSUPPORTED;
  if (topk == 0) return M3S_OK;
  const int stride = bt_stride > 0 ? bt_stride : 1;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool streams = topk_streams(R);
  if (streams || !block_scores) {
    if (ws_bytes < m3s_workspace_bytes(M3S_OP_INDEX_SCORE_TOPK, R, B, bt_stride, 0, 0, Hi, topk, 1))
      return M3S_ERR_WORKSPACE;
    if (!ws || !aligned16(ws)) return M3S_ERR_INVALID;
  }
  float* bs = block_scores ? block_scores : static_cast<float*>(ws);
  ScoreArgs a{q_idx, w, Hi, idx_k.codes, idx_k.scales, idx_k.num_pages, block_table, bt_stride,
              row_req, nullptr, row_len, R, B, R, 1, streams ? block_scores : bs, stride, err,
              idx_k.format == M3S_FMT_MXFP4 ? 1 : 0};
  if (streams) {
    bind_topk_workspace(a, ws, R, topk, init_blocks, local_blocks, topk_ids);
    return launch_score_decode(a, st);
  }
  if (B > 0) {   // two launches: block scores, then the top-k
    rc = launch_score_decode(a, st);
    if (rc != M3S_OK) return rc;
  }
  return launch_topk(bs, stride, row_req, row_len, R, B, bt_stride, topk, init_blocks, local_blocks,
                     topk_ids, st);
}

extern "C" int m3s_verify_score_topk(const uint16_t* q_idx, const float* w, int32_t Hi,
                                     m3s_fp4_plane idx_k, const int32_t* block_table,
                                     int32_t bt_stride, const int32_t* cu_q,
                                     const int32_t* row_len, int32_t B, int32_t R, int32_t max_q,
                                     int32_t topk, int32_t init_blocks, int32_t local_blocks,
                                     int32_t* topk_ids, void* ws, size_t ws_bytes, int32_t* err,
                                     void* stream) {
  using namespace m3s;
  int rc = check_common(q_idx, w, Hi, idx_k, block_table, bt_stride, R, B, topk, topk_ids);
  if (rc != M3S_OK || R == 0) return rc;
  if (!cu_q || !row_len || max_q < 0 || init_blocks < 0 || local_blocks < 0) return M3S_ERR_INVALID;
  if (topk == 0) return M3S_OK;
  const int cpr = max_q > 0 ? (max_q + 7) / 8 : 1;
  const long long ntiles = static_cast<long long>(B) * cpr;   // B == 0: every row is padding
  if (ntiles > kMaxTiles) return M3S_ERR_UNSUPPORTED;
  if (ws_bytes < m3s_workspace_bytes(M3S_OP_VERIFY_SCORE_TOPK, R, B, bt_stride, 0, 0, Hi, topk, max_q))
    return M3S_ERR_WORKSPACE;
  if (!ws || !aligned16(ws)) return M3S_ERR_INVALID;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool streams = topk_streams(ntiles);
  const int stride = bt_stride > 0 ? bt_stride : 1;
  ScoreArgs a{q_idx, w, Hi, idx_k.codes, idx_k.scales, idx_k.num_pages, block_table, bt_stride,
              nullptr, cu_q, row_len, R, B, static_cast<int>(ntiles), cpr,
              streams ? nullptr : static_cast<float*>(ws), stride, err,
              idx_k.format == M3S_FMT_MXFP4 ? 1 : 0};
  if (streams) {
    bind_topk_workspace(a, ws, static_cast<int>(ntiles), topk, init_blocks, local_blocks, topk_ids);
    a.seg_scores = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(a.cand) +
                                            topk_cand_bytes(static_cast<int>(ntiles), 8, topk));
    return launch_score<8>(a, st);
  }
  if (ntiles > 0) {   // two launches: block scores, then the top-k (rows past cu_q[B]: -1)
    rc = launch_score<8>(a, st);
    if (rc != M3S_OK) return rc;
  }
  return launch_topk(static_cast<float*>(ws), stride, nullptr, row_len, R, B, bt_stride, topk, init_blocks,
                     local_blocks, topk_ids, st);
}

// ---------------------------------------------------------------------------
// Indexer context parallelism: a slice's candidates, and their merge.
// ---------------------------------------------------------------------------
namespace m3s {
namespace {

// One warp per row: the k best keys of the n_lists ranks' lists (list i of row r
// at cand + (i * R + r) * topk), as ids ascending (-1 padded).
__global__ void __launch_bounds__(256) merge_candidates_kernel(const unsigned long long* __restrict__ cand,
                                                               int n_lists, int R, int topk,
                                                               int32_t* __restrict__ ids) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= R) return;   // (warp-uniform)
  WarpTopk sel;
  warp_merge<true>(cand + static_cast<size_t>(r) * topk, nullptr, R * topk, n_lists, topk, topk, lane, sel);
  write_ids(sel, topk, ids + static_cast<size_t>(r) * topk, lane);
}

}  // namespace
}  // namespace m3s

extern "C" int m3s_index_score_candidates(const uint16_t* q_idx, const float* w, int32_t Hi,
                                          m3s_fp4_plane idx_k, const int32_t* block_table,
                                          int32_t bt_stride, const int32_t* blk_begin,
                                          const int32_t* blk_count, const int32_t* row_req,
                                          const int32_t* row_len, int32_t R, int32_t B, int32_t topk,
                                          int32_t init_blocks, int32_t local_blocks,
                                          uint64_t* cand_keys, void* ws, size_t ws_bytes, int32_t* err,
                                          void* stream) {
  using namespace m3s;
  int32_t dummy = 0;
  int rc = check_common(q_idx, w, Hi, idx_k, block_table, bt_stride, R, B, topk, &dummy);
  if (rc != M3S_OK || R == 0) return rc;
  if (!row_req || !row_len || !cand_keys || init_blocks < 0 || local_blocks < 0) return M3S_ERR_INVALID;
  if (B > 0 && (!blk_begin || !blk_count)) return M3S_ERR_INVALID;
  if (R > kMaxTiles) return M3S_ERR_UNSUPPORTED;
  if (topk == 0) return M3S_OK;
  if (ws_bytes < m3s_workspace_bytes(M3S_OP_INDEX_CANDIDATES, R, B, bt_stride, 0, 0, Hi, topk, 1))
    return M3S_ERR_WORKSPACE;
  if (!ws || !aligned16(ws) || (reinterpret_cast<uintptr_t>(cand_keys) & 7u)) return M3S_ERR_INVALID;
  ScoreArgs a{q_idx, w, Hi, idx_k.codes, idx_k.scales, idx_k.num_pages, block_table, bt_stride,
              row_req, nullptr, row_len, R, B, R, 1, nullptr, bt_stride > 0 ? bt_stride : 1, err,
              idx_k.format == M3S_FMT_MXFP4 ? 1 : 0};
  bind_topk_workspace(a, ws, R, topk, init_blocks, local_blocks, nullptr);
  a.keys_out = reinterpret_cast<unsigned long long*>(cand_keys);
  a.blk_base = blk_begin;
  a.blk_count = blk_count;
  return launch_score_decode(a, static_cast<cudaStream_t>(stream));
}

extern "C" int m3s_merge_candidates(const uint64_t* cand_keys, int32_t n_lists, int32_t R, int32_t topk,
                                    int32_t* topk_ids, void* stream) {
  using namespace m3s;
  if (n_lists < 0 || R < 0 || topk < 0) return M3S_ERR_INVALID;
  if (topk > M3S_MAX_TOPK || n_lists > kMaxGrid) return M3S_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(R) * topk > INT32_MAX) return M3S_ERR_UNSUPPORTED;   // list stride is int
  if (R == 0 || topk == 0) return M3S_OK;
  if (!topk_ids || (n_lists > 0 && !cand_keys) || (reinterpret_cast<uintptr_t>(cand_keys) & 7u))
    return M3S_ERR_INVALID;
  const int rows_per_cta = 8;
  return launch_kernel(merge_candidates_kernel, dim3((R + rows_per_cta - 1) / rows_per_cta),
                       dim3(32 * rows_per_cta), 0, static_cast<cudaStream_t>(stream), 0,
                       reinterpret_cast<const unsigned long long*>(cand_keys), n_lists, R, topk, topk_ids) ==
                 cudaSuccess
             ? M3S_OK
             : M3S_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// Decode rows end to end in two launches: the scorer leaves each CTA's top-k
// candidates of every row it scores (and each row's slot range); the
// attention merges a row's candidates before it reads its pages.
// ---------------------------------------------------------------------------
namespace m3s {
int check_attention(const uint16_t* q, int32_t Hq, int32_t Hkv, m3s_fp4_plane k, m3s_fp4_plane v,
                    const int32_t* block_table, int32_t bt_stride, int32_t B, const int32_t* row_req,
                    const int32_t* row_len, bool have_ids, int32_t topk, int32_t R, const uint16_t* out);
int launch_attention(const uint16_t* q, int32_t Hq, int32_t Hkv, m3s_fp4_plane k, m3s_fp4_plane v,
                     const int32_t* block_table, int32_t bt_stride, int32_t B, const int32_t* row_req,
                     const int32_t* row_len, const int32_t* topk_ids, int32_t topk, int32_t R,
                     float sm_scale, uint16_t* out, float* lse, int32_t* err, cudaStream_t stream,
                     const unsigned long long* cand, const int2* meta, int32_t* ids_out, int cand_lists,
                     int cand_stride);
}  // namespace m3s

extern "C" int m3s_index_attention(const uint16_t* q_idx, const float* w, int32_t Hi, m3s_fp4_plane idx_k,
                                   const uint16_t* q, int32_t Hq, int32_t Hkv, m3s_fp4_plane k,
                                   m3s_fp4_plane v, const int32_t* block_table, int32_t bt_stride,
                                   int32_t B, const int32_t* row_req, const int32_t* row_len, int32_t R,
                                   int32_t topk, int32_t init_blocks, int32_t local_blocks, float sm_scale,
                                   int32_t* topk_ids, uint16_t* out, float* lse, void* ws, size_t ws_bytes,
                                   int32_t* err, void* stream) {
  using namespace m3s;
  int32_t no_ids = 0;   // (top-k 0 writes no id)
  int rc = check_common(q_idx, w, Hi, idx_k, block_table, bt_stride, R, B, topk, topk > 0 ? topk_ids : &no_ids);
  if (rc != M3S_OK) return rc;
  rc = check_attention(q, Hq, Hkv, k, v, block_table, bt_stride, B, row_req, row_len, true, topk, R, out);
  if (rc != M3S_OK || R == 0) return rc;
  if (!row_req || !row_len || init_blocks < 0 || local_blocks < 0) return M3S_ERR_INVALID;
  if (R > kMaxTiles) return M3S_ERR_UNSUPPORTED;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (topk == 0)   // nothing selected: every row attends over no token
    return launch_attention(q, Hq, Hkv, k, v, block_table, bt_stride, B, row_req, row_len, topk_ids, 0, R,
                            sm_scale, out, lse, err, st, nullptr, nullptr, nullptr, 0, 1);
  if (ws_bytes < m3s_workspace_bytes(M3S_OP_INDEX_ATTENTION, R, B, bt_stride, Hq, Hkv, Hi, topk, 1))
    return M3S_ERR_WORKSPACE;
  if (!ws || !aligned16(ws)) return M3S_ERR_INVALID;
  ScoreArgs a{q_idx, w, Hi, idx_k.codes, idx_k.scales, idx_k.num_pages, block_table, bt_stride,
              row_req, nullptr, row_len, R, B, R, 1, nullptr, bt_stride > 0 ? bt_stride : 1, err,
              idx_k.format == M3S_FMT_MXFP4 ? 1 : 0};
  uint8_t* base = static_cast<uint8_t*>(ws);
  a.cand = reinterpret_cast<unsigned long long*>(base);
  a.meta = reinterpret_cast<int2*>(base + index_attention_meta_offset(R, topk));
  a.topk = topk;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  rc = launch_score_decode(a, st);
  if (rc != M3S_OK) return rc;
  return launch_attention(q, Hq, Hkv, k, v, block_table, bt_stride, B, row_req, row_len, nullptr, topk, R,
                          sm_scale, out, lse, err, st, a.cand, a.meta, topk_ids, R + kMaxGrid - 1, 1);
}

// Verify rows (tiles of up to 8 rows of one request) the same way: the verify
// scorer in partials mode leaves each CTA's top-k of every row it scores (the
// streaming form's lists, without the tiles' merges) and each row's list range,
// and the attention merges a row's lists before it reads the row's pages.
extern "C" int m3s_verify_index_attention(const uint16_t* q_idx, const float* w, int32_t Hi,
                                          m3s_fp4_plane idx_k, const uint16_t* q, int32_t Hq, int32_t Hkv,
                                          m3s_fp4_plane k, m3s_fp4_plane v, const int32_t* block_table,
                                          int32_t bt_stride, int32_t B, const int32_t* cu_q,
                                          const int32_t* row_req, const int32_t* row_len, int32_t R,
                                          int32_t max_q, int32_t topk, int32_t init_blocks,
                                          int32_t local_blocks, float sm_scale, int32_t* topk_ids,
                                          uint16_t* out, float* lse, void* ws, size_t ws_bytes, int32_t* err,
                                          void* stream) {
  using namespace m3s;
  int32_t no_ids = 0;   // (top-k 0 writes no id)
  int rc = check_common(q_idx, w, Hi, idx_k, block_table, bt_stride, R, B, topk, topk > 0 ? topk_ids : &no_ids);
  if (rc != M3S_OK) return rc;
  rc = check_attention(q, Hq, Hkv, k, v, block_table, bt_stride, B, row_req, row_len, true, topk, R, out);
  if (rc != M3S_OK || R == 0) return rc;
  if (!cu_q || !row_req || !row_len || max_q < 0 || init_blocks < 0 || local_blocks < 0) return M3S_ERR_INVALID;
  const int cpr = max_q > 0 ? (max_q + 7) / 8 : 1;
  const long long ntiles = static_cast<long long>(B) * cpr;   // B == 0: every row is padding
  if (ntiles > kMaxTiles) return M3S_ERR_UNSUPPORTED;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (topk == 0)   // nothing selected: every row attends over no token
    return launch_attention(q, Hq, Hkv, k, v, block_table, bt_stride, B, row_req, row_len, topk_ids, 0, R,
                            sm_scale, out, lse, err, st, nullptr, nullptr, nullptr, 0, 1);
  if (ws_bytes < m3s_workspace_bytes(M3S_OP_VERIFY_INDEX_ATTENTION, R, B, bt_stride, Hq, Hkv, Hi, topk, max_q))
    return M3S_ERR_WORKSPACE;
  if (!ws || !aligned16(ws)) return M3S_ERR_INVALID;
  const int nt = static_cast<int>(ntiles);
  ScoreArgs a{q_idx, w, Hi, idx_k.codes, idx_k.scales, idx_k.num_pages, block_table, bt_stride,
              nullptr, cu_q, row_len, R, B, nt, cpr, nullptr, bt_stride > 0 ? bt_stride : 1, err,
              idx_k.format == M3S_FMT_MXFP4 ? 1 : 0};
  uint8_t* base = static_cast<uint8_t*>(ws);
  a.cand = reinterpret_cast<unsigned long long*>(base);
  a.seg_scores = reinterpret_cast<float*>(base + verify_attention_seg_offset(nt, topk));
  a.meta = reinterpret_cast<int2*>(base + verify_attention_meta_offset(nt, topk, bt_stride));
  a.topk = topk;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  if (nt > 0) {
    rc = launch_score<8>(a, st);
    if (rc != M3S_OK) return rc;
  } else {   // no tile: every row is padding, with an empty list range
    if (cudaMemsetAsync(a.meta, 0, static_cast<size_t>(R) * 8, st) != cudaSuccess) return M3S_ERR_LAUNCH;
  }
  return launch_attention(q, Hq, Hkv, k, v, block_table, bt_stride, B, row_req, row_len, nullptr, topk, R,
                          sm_scale, out, lse, err, st, a.cand, a.meta, topk_ids, (nt + kMaxGrid - 1) * 8, 8);
}

// ---------------------------------------------------------------------------
// m3s_index_score_topk_static: m3s_index_score_topk with its block-score
// scratch in a file-scope device array instead of a caller workspace.
//
// It serves callers that cannot allocate device memory when they call: a
// plain C host that links only this library and owns no device allocator,
// and an engine plugin whose device memory budget is fixed at start-up, so
// it cannot size a workspace per call. Those callers get a scratch whose
// size is fixed when the library is built.
//
// The host side looks the array's address up on every call
// (cudaGetSymbolAddress, with the caller's device current), so the address is
// always the one of the current context, also after a cudaDeviceReset. The
// first call on a device also loads the module that holds the array, so it
// should come before any stream capture. Nothing in the scratch has to start at
// zero: the scorer writes every block score that the top-k reads (each block
// below the row's block count, -inf for a skipped page). All calls share one
// scratch per device, so two calls that overlap on the GPU (different
// streams, no ordering between them) race on it.
// ---------------------------------------------------------------------------
namespace m3s {
namespace {

constexpr size_t kStaticScratchFloats = M3S_STATIC_SCRATCH_BYTES / sizeof(float);
static_assert(M3S_STATIC_SCRATCH_BYTES % 256 == 0, "static scratch size");

static __device__ __align__(256) float g_static_block_scores[kStaticScratchFloats];

// The array's address in the current context (nullptr when the lookup fails).
// Not cached: a cached address would dangle after cudaDeviceReset or under
// another context of the same device.
float* static_scratch() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_block_scores) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<float*>(p);
}

}  // namespace
}  // namespace m3s

extern "C" int m3s_index_score_topk_static(const uint16_t* q_idx, const float* w, int32_t Hi,
                                           m3s_fp4_plane idx_k, const int32_t* block_table,
                                           int32_t bt_stride, const int32_t* row_req,
                                           const int32_t* row_len, int32_t R, int32_t B,
                                           int32_t topk, int32_t* topk_ids, int32_t* err,
                                           void* stream) {
  using namespace m3s;
  int rc = check_common(q_idx, w, Hi, idx_k, block_table, bt_stride, R, B, topk, topk_ids);
  if (rc != M3S_OK || R == 0) return rc;
  if (!row_req || !row_len) return M3S_ERR_INVALID;
  if (R > kMaxTiles) return M3S_ERR_UNSUPPORTED;
  if (topk == 0) return M3S_OK;
  const int stride = bt_stride > 0 ? bt_stride : 1;
  // the block-score matrix [R][stride] must fit the fixed scratch
  if (static_cast<size_t>(R) * static_cast<size_t>(stride) > kStaticScratchFloats)
    return M3S_ERR_WORKSPACE;
  float* bs = static_scratch();
  if (!bs) return M3S_ERR_LAUNCH;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B > 0) {
    ScoreArgs a{q_idx, w, Hi, idx_k.codes, idx_k.scales, idx_k.num_pages, block_table, bt_stride,
                row_req, nullptr, row_len, R, B, R, 1, bs, stride, err,
                idx_k.format == M3S_FMT_MXFP4 ? 1 : 0};
    rc = launch_score_decode(a, st);
    if (rc != M3S_OK) return rc;
  }
  return launch_topk(bs, stride, row_req, row_len, R, B, bt_stride, topk, 0, 0, topk_ids, st);
}
