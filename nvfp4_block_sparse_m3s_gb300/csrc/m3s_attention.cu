// Block-sparse softmax attention over the selected NVFP4 pages.
//
// "NVFP4 sparse KV" (ROCm/ATOM #2746), Summary / Attention and "[MiniMax-M3.1]
// FP4 index cache and NVFP4 sparse KV cache" (#2744), Design / Attention: a
// row attends over its top-k blocks, addressed through the request's block
// table, against the dequantised K/V. Bad ids are reported, never wrapped
// (review of #2744: a modulo silently mapped an invalid id onto a valid page).
//
// Split-K inside a thread-block cluster: the CTAs (split, kv head, row) of one
// (kv head, row) form a cluster; each runs an online softmax over its share of
// the row's blocks, leaves (m, l, o) in its shared memory, and the cluster's
// CTAs combine the partials through distributed shared memory and write the
// output, so there is no second launch and no workspace round trip. Inside a
// CTA a group of four warps takes 32 tokens each of a 128-token block; a CTA
// has one group, or two taking alternate blocks (each with its own two-stage
// page ring) when the grid has at most one CTA per SM. S = Q K^T
// with the q heads of the KV head as M (m16), then P V with P re-used from the
// S accumulators as the A operand. K and V are dequantised from the
// shared-memory copy of the page straight into mma fragments: K in a permuted
// head-dim order (each thread reads one 16-byte chunk of a token, the q
// fragments follow the same order), V two tokens at a time with the nibbles of
// the same byte interleaved (each n8 tile covers every other dimension).
//
// MXFP4 K/V (one E8M0 scale per 32 elements) run the same fp16 products after
// exponent normalisation, since e2m1 x 2^(E-127) does not fit fp16 over E8M0's
// range. K: a thread's 16-byte chunk of a token is one 32-element group, scaled
// by 2^(E - E_max) (E_max = the token's largest exponent), and the token's scores
// by 2^(E_max - 127) in fp32. V: every output accumulator of a thread lies in one
// 32-dim group, so each warp keeps a running reference exponent R per group (the
// largest of its live tokens so far), scales V by 2^(E - R), rescales its
// accumulators exactly when R grows, and multiplies them by 2^(R - 127) at the
// end. Both are exact while the exponents involved span at most 23.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "m3s_score_common.cuh"

namespace m3s {
namespace {

// 2^x by the PTX ex2.approx.ftz instruction (inputs here are at most 2^8;
// results below 2^-126 flush to 0, far below the resolution of the fp32 sum
// they join).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// How far (log2 units) a head's running maximum may rise above the reference
// its sums are kept relative to before they are rescaled.
constexpr float kMaxSlack = 8.f;

struct AttnArgs {
  const uint16_t* q;
  int Hq, Hkv, G;
  const uint8_t *kc, *ks, *vc, *vs;
  int num_pages;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* row_req;
  const int32_t* row_len;
  const int32_t* ids;
  int topk, R, B;
  float scale_log2;  // sm_scale * log2(e)
  int nsplit, ips;
  uint16_t* out;
  float* lse;
  int32_t* err;
  // candidates mode (ids == nullptr): the scorer's per-CTA candidate lists and
  // each row's (first list, lists), its lists cand_stride lists apart; the
  // row's ids are written to ids_out
  const unsigned long long* cand;
  const int2* meta;
  int32_t* ids_out;
  int nlists;        // lists of topk keys in cand
  int cand_stride;   // 1 (decode rows: a row's lists are consecutive) or 8 (verify tiles)
};

// Per-warp partial outputs are stored at [head][dim + dim / 32] in rows of
// kMergeRow floats: the 32 lanes of one store (8 heads x 4 dim groups of 32)
// then fall in 32 different banks (bank = 4 head + dim / 32 + const).
constexpr int kMergeRow = kHeadDim + 4;
__device__ __forceinline__ int merge_at(int head, int dim) { return head * kMergeRow + dim + (dim >> 5); }

// The warps' partial outputs, merged after the block loop (over the page stages).
template <int NW>
struct AttnMerge {
  float o[NW][16 * kMergeRow];
  float m[NW][16];
  float l[NW][16];
  float f[NW][16];   // exp2(m_warp - M) per warp and head
};

// Dynamic shared memory: this part, then the page stages (K codes, K scales,
// V codes, V scales of one page each), which the merge buffers reuse.
struct __align__(16) AttnFixed {
  uint4 qa[8][32];            // the q fragments (A operand) per k-step and lane
  float lsc[16];              // per-head logit scales (log2 units)
  float cta_o[16][kHeadDim];  // this CTA's partial: sum p v, relative to cta_m (log2 units)
  float cta_m[16];
  float cta_l[16];
  uint64_t bar[4];            // two stages per warp group
  uint64_t cand_bar;          // candidates mode: the staging copy of the row's lists
  int sel_id[M3S_MAX_TOPK];   // candidates mode: the row's selected ids, ascending
  unsigned long long sel_tau; // candidates mode: the selection's lower bound
  int sel_n;                  // ... and its candidate count
  int page[M3S_MAX_TOPK];
  int ntok[M3S_MAX_TOPK];
  int nblocks;
};
constexpr size_t kAttFixedBytes = (sizeof(AttnFixed) + 127) / 128 * 128;

// Named barrier over the n threads of barrier `id`, and the same with an OR
// vote across them.
__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool bar_or(bool p, int id, int n) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.or.pred b, %2, %3, a;\n"
      " selp.u32 %0, 1, 0, b;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 2^d as fp32 for d <= 0, zero below fp32's subnormal range.
__device__ __forceinline__ float pow2_f32_nonpos(int d) {
  if (d >= -126) return __uint_as_float(static_cast<uint32_t>(d + 127) << 23);
  return d >= -149 ? __uint_as_float(1u << (d + 149)) : 0.f;
}

// Candidates mode, the whole CTA: the row's top-k from its candidate lists
// (mt.y lists of topk keys, each descending, list j at list index
// mt.x + j * cand_stride), its ids ranked ascending into sel_id (-1 padded);
// split 0 of the first KV head also writes them to ids_out. Consecutive lists
// (decode rows) are one contiguous run, staged into buf by one bulk copy
// (thread 0); strided lists, or a run that is not 16-byte aligned, by loads
// from every thread. Selection by counting, in three CTA-wide passes: the k-th largest
// list head is a lower bound for the row's k-th key (the k largest heads are
// k keys at least that large; with fewer lists than k every key is a
// candidate: bounding by the smallest of the lists' ceil(k / nl)-th keys
// instead timed 0.25 us slower on the skewed decode step), so only keys at or
// above it are candidates; each candidate's rank is the number of larger ones,
// and the k best land at their ranks. (More than kSelCap candidates: a
// pairwise merge of all lists instead.) Kept out of line: inlined, merge code
// of this kind slowed the block loop of the whole kernel (measured: decode-row
// attention 20 us against 12). Returns false when the copy's bounded wait runs
// out (the row then gets no block).
constexpr int kSelCap = 512;
__device__ __noinline__ bool select_row_candidates(const AttnArgs& a, int2 mt, int r, int split, int kvh,
                                                   unsigned long long* buf, size_t buf_bytes, uint64_t* bar,
                                                   int nthreads, int* sel_id, unsigned long long* tau_s,
                                                   int* n_s) {
  const int tid = threadIdx.x, k = a.topk;
  // a range outside the lists is reported and skipped (the scorer writes every
  // row's range each call; this guards against a stale or foreign workspace)
  const int cs = a.cand_stride;
  if (mt.x < 0 || mt.y < 0 || mt.y > a.nlists ||
      (mt.y > 0 && static_cast<long long>(mt.x) + static_cast<long long>(mt.y - 1) * cs >= a.nlists)) {
    if (tid == 0) raise(a.err, M3S_DEVERR_ROW);
    mt = make_int2(0, 0);
  }
  const int nl = mt.y;
  const int nkeys = nl * k;
  const unsigned long long* src = a.cand + static_cast<size_t>(mt.x) * k;
  // (the copy may read up to 8 bytes past the run: the workspace's slot area is
  // followed by its 256-byte padding and the row ranges)
  const uint32_t bytes = (static_cast<uint32_t>(nkeys) * 8 + 15) & ~15u;
  unsigned long long* cand = buf + ((nkeys + 1) & ~1);   // kSelCap candidates
  unsigned long long* top = cand + kSelCap;              // the k best, descending
  bool ok = static_cast<size_t>(bytes) + (kSelCap + M3S_MAX_TOPK) * 8 + M3S_MAX_TOPK * 4 <= buf_bytes;
  if (ok && nkeys > 0) {
    if (cs == 1 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
      if (tid == 0) {
        mbar_expect_tx(bar, bytes);
        bulk_g2s(buf, src, bytes, bar);
      }
      // one decision for the whole CTA (a late copy seen by some threads only)
      if (__syncthreads_or(!mbar_wait(bar, 0))) {
        if (tid == 0) raise(a.err, M3S_DEVERR_TIMEOUT);
        mbar_wait(bar, 0);
        ok = false;
      }
    } else {   // (list e / k at src + (e / k) * cs * k)
      for (int e = tid; e < nkeys; e += nthreads)
        buf[e] = __ldcg(src + static_cast<size_t>(e / k) * cs * k + e % k);
      __syncthreads();
    }
  }
  int nsel = 0;   // keys selected (<= k)
  if (ok && nkeys > 0) {
    // the lower bound: the k-th largest head (every nonzero key when fewer lists)
    if (tid == 0) {
      *tau_s = 1ull;
      *n_s = 0;
    }
    __syncthreads();
    if (nl >= k) {
      for (int j = tid; j < nl; j += nthreads) {
        const unsigned long long h = buf[j * k];
        int rank = 0;
#pragma unroll 8
        for (int i = 0; i < nl; ++i) rank += buf[i * k] > h;
        if (rank == k - 1) *tau_s = h > 1ull ? h : 1ull;   // (zero heads: empty lists)
      }
      __syncthreads();
    }
    const unsigned long long tau = *tau_s;
    for (int e = tid; e < nkeys; e += nthreads) {
      const unsigned long long x = buf[e];
      if (x >= tau) {
        const int s = atomicAdd(n_s, 1);
        if (s < kSelCap) cand[s] = x;
      }
    }
    __syncthreads();
    const int m = *n_s;
    for (int i = tid; i < k; i += nthreads) top[i] = 0ull;   // (an unfilled place: no id)
    __syncthreads();
    if (m <= kSelCap) {
      for (int c = tid; c < m; c += nthreads) {
        const unsigned long long x = cand[c];
        int rank = 0;
#pragma unroll 8
        for (int i = 0; i < m; ++i) rank += cand[i] > x;
        if (rank < k) top[rank] = x;
      }
      nsel = min(m, k);
    } else {   // (many equal-looking lists: merge them all)
      tree_merge_lists(buf, 1, nl, k, nthreads);
      for (int i = tid; i < k; i += nthreads) top[i] = buf[i];
      nsel = k;
    }
    __syncthreads();
  }
  // the ids, ascending (rank of each selected id among them)
  int* top_id = reinterpret_cast<int*>(top + M3S_MAX_TOPK);
  if (tid < nsel) top_id[tid] = top[tid] ? select_key_id(top[tid]) : -1;
  __syncthreads();
  if (tid < k) {
    int id = -1, rank = tid;
    if (tid < nsel && top_id[tid] >= 0) {
      id = top_id[tid];
      rank = 0;
#pragma unroll 8
      for (int i = 0; i < nsel; ++i) rank += top_id[i] >= 0 && top_id[i] < id;
    } else if (tid < nsel) {   // (unfilled: after the filled ones)
      rank = 0;
      for (int i = 0; i < nsel; ++i) rank += top_id[i] >= 0 || i < tid;
    }
    sel_id[rank] = id;
    if (split == 0 && kvh == 0 && a.ids_out) a.ids_out[static_cast<size_t>(r) * k + rank] = id;
  }
  fence_proxy_async();   // bulk copies refill the stage memory read and written here
  __syncthreads();
  return ok;
}

template <bool MX, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 4 ? 4 : 1) attention_kernel(const AttnArgs a) {
  // a page's K (or V) scale bytes, and where they sit in a stage
  constexpr int kPageScaleB = MX ? kMxPageScaleBytes : kPageScaleBytes;
  constexpr int kStageB = 2 * (kPageCodeBytes + kPageScaleB);
  constexpr int kThreads = NW * 32;
  constexpr int kGroups = NW / 4;   // groups of four warps, each a two-stage ring
  extern __shared__ __align__(128) uint8_t att_smem[];
  AttnFixed& sm = *reinterpret_cast<AttnFixed*>(att_smem);
  uint8_t* const stage0 = att_smem + kAttFixedBytes;
  AttnMerge<NW>& mg = *reinterpret_cast<AttnMerge<NW>*>(stage0);
  const int split = blockIdx.x, kvh = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int gi = warp >> 2;   // this warp's group

  if (tid == 0) {
    for (int i = 0; i < 2 * kGroups; ++i) mbar_init(&sm.bar[i], 1);
    mbar_init(&sm.cand_bar, 1);
    mbar_fence_init();
    // Before the wait, bring this row's q and a share of the block table into
    // L2: no earlier kernel of the step writes the block table, and a q line a
    // producer writes later is updated in L2, which every read below goes through.
    if (split == 0)
      bulk_prefetch_l2(a.q + (static_cast<size_t>(r) * a.Hq + kvh * a.G) * kHeadDim,
                       static_cast<uint32_t>(a.G * kHeadDim * 2));
    const size_t tb = static_cast<size_t>(a.B) * a.bt_stride * sizeof(int32_t);
    const size_t nctas = static_cast<size_t>(gridDim.x) * gridDim.y * gridDim.z;
    const size_t me = blockIdx.x + static_cast<size_t>(gridDim.x) * (blockIdx.y + static_cast<size_t>(gridDim.y) * blockIdx.z);
    const size_t chunk = ((tb + nctas - 1) / nctas + 15) & ~static_cast<size_t>(15);
    const size_t off = me * chunk;
    if ((reinterpret_cast<uintptr_t>(a.block_table) & 15u) == 0 && off < tb) {
      const size_t n = min(chunk, tb - off) & ~static_cast<size_t>(15);
      if (n > 0) bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(a.block_table) + off, static_cast<uint32_t>(n));
    }
  }
  pdl_trigger();
  pdl_wait();
  // q fragments (A operand, heads as rows) in the permuted head-dim order:
  // k-step j covers dims 32t+4j .. 32t+4j+3 for thread t. Warp 1 loads and
  // converts them into shared memory while warp 0 works out the block list.
  uint2 qr[8][2];
  if (warp == 1) {
    const int h0 = g, h1 = g + 8;
    const uint16_t* q0 = a.q + (static_cast<size_t>(r) * a.Hq + kvh * a.G + h0) * kHeadDim + 32 * t;
    const uint16_t* q1 = a.q + (static_cast<size_t>(r) * a.Hq + kvh * a.G + h1) * kHeadDim + 32 * t;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qr[j][0] = h0 < a.G ? *reinterpret_cast<const uint2*>(q0 + 4 * j) : make_uint2(0u, 0u);
      qr[j][1] = h1 < a.G ? *reinterpret_cast<const uint2*>(q1 + 4 * j) : make_uint2(0u, 0u);
    }
  }

  // The block list of this split: warp 0 reads the ids (together with the row's
  // request and length), checks them, looks the pages up in parallel and
  // compacts the valid ones; the lane that finds block 0 or 1 starts its copy.
  // Candidates mode: the whole CTA selects the row's top-k first.
  const bool cands = a.cand != nullptr;
  if (cands)
    select_row_candidates(a, a.meta[r], r, split, kvh, reinterpret_cast<unsigned long long*>(stage0),
                          static_cast<size_t>(2 * kGroups) * kStageB, &sm.cand_bar, kThreads, sm.sel_id,
                          &sm.sel_tau, &sm.sel_n);
  // block i of the list goes to group i mod kGroups, as that group's
  // (i / kGroups)-th block, into the group's stage 2 group + (that & 1)
  auto issue = [&](int i, int page) {
    const int s = 2 * (i % kGroups) + ((i / kGroups) & 1);
    const size_t rec = static_cast<size_t>(page) * a.Hkv + kvh;
    uint8_t* dst = stage0 + s * kStageB;
    fence_proxy_async();
    mbar_expect_tx(&sm.bar[s], kStageB);
    bulk_g2s(dst, a.kc + rec * kPageCodeBytes, kPageCodeBytes, &sm.bar[s]);
    bulk_g2s(dst + kPageCodeBytes, a.ks + rec * kPageScaleB, kPageScaleB, &sm.bar[s]);
    bulk_g2s(dst + kPageCodeBytes + kPageScaleB, a.vc + rec * kPageCodeBytes, kPageCodeBytes,
             &sm.bar[s]);
    bulk_g2s(dst + 2 * kPageCodeBytes + kPageScaleB, a.vs + rec * kPageScaleB, kPageScaleB,
             &sm.bar[s]);
  };
  if (warp == 0) {
    __syncwarp();   // the barriers lane 0 initialised
    const int i0 = split * a.ips, i1 = min(a.topk, i0 + a.ips);
    const int id_first = !cands && i0 + lane < i1 ? a.ids[static_cast<size_t>(r) * a.topk + i0 + lane] : -1;
    const int len = a.row_len[r];
    const int req = a.row_req[r];
    const bool row_ok = req >= 0 && len > 0;
    const bool row_bad = row_ok && (req >= a.B || len > a.bt_stride * kPage);
    if (row_bad && lane == 0 && split == 0 && kvh == 0) raise(a.err, M3S_DEVERR_ROW);
    const int nb = (len + kPage - 1) / kPage;
    int n = 0;
    for (int base = i0; base < i1; base += 32) {
      const int i = base + lane;
      int page = -1, ntok = 0;
      if (row_ok && !row_bad && i < i1) {
        const int id = cands ? sm.sel_id[i] : (base == i0 ? id_first : a.ids[static_cast<size_t>(r) * a.topk + i]);
        if (id >= 0) {
          if (id >= nb || id >= a.bt_stride) {
            if (kvh == 0) raise(a.err, M3S_DEVERR_BLOCK_ID);
          } else {
            page = a.block_table[static_cast<size_t>(req) * a.bt_stride + id];
            if (page < 0 || page >= a.num_pages) {
              if (kvh == 0) raise(a.err, M3S_DEVERR_PAGE);
              page = -1;
            } else {
              ntok = min(kPage, len - id * kPage);
            }
          }
        }
      }
      const unsigned keep = __ballot_sync(0xffffffffu, page >= 0);
      if (page >= 0) {
        const int at = n + __popc(keep & ((1u << lane) - 1u));
        sm.page[at] = page;
        sm.ntok[at] = ntok;
        if (at < 2 * kGroups) issue(at, page);
      }
      n += __popc(keep);
    }
    if (lane == 0) sm.nblocks = n;
  }
  // Heads g and g + 8 are scaled by 2^-e before their f16 conversion (e from
  // the head's largest magnitude, over the four lanes t that hold its 128 dims)
  // and their logits by sm_scale log2(e) 2^e, which undoes it.
  if (warp == 1) {
    unsigned m0 = 0u, m1 = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      m0 = max(m0, max(bf16x2_absmax_bits(qr[j][0].x), bf16x2_absmax_bits(qr[j][0].y)));
      m1 = max(m1, max(bf16x2_absmax_bits(qr[j][1].x), bf16x2_absmax_bits(qr[j][1].y)));
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      m0 = max(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = max(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    if ((m0 >= kBf16InfBits || m1 >= kBf16InfBits) && t == 0) raise(a.err, M3S_DEVERR_QRANGE);
    const int e0 = m0 ? q_scale_exp(min(m0, kBf16InfBits - 1)) : 0;
    const int e1 = m1 ? q_scale_exp(min(m1, kBf16InfBits - 1)) : 0;
    const QScale sc0 = q_scale(e0), sc1 = q_scale(e1);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      sm.qa[j][lane] = make_uint4(bf16x2_to_f16x2_scaled(qr[j][0].x, sc0), bf16x2_to_f16x2_scaled(qr[j][1].x, sc1),
                                  bf16x2_to_f16x2_scaled(qr[j][0].y, sc0), bf16x2_to_f16x2_scaled(qr[j][1].y, sc1));
    if (t == 0) {
      sm.lsc[g] = a.scale_log2 * exp2i_f32(e0);
      sm.lsc[g + 8] = a.scale_log2 * exp2i_f32(e1);
    }
  }
  __syncthreads();
  const int nblocks = sm.nblocks;
  const float lsc0 = sm.lsc[g], lsc1 = sm.lsc[g + 8];


  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running max (log2 units) of heads g, g+8
  float l0 = 0.f, l1 = 0.f;              // this thread's share of the sums
  uint32_t vref = 0;                     // MX: this warp's V reference exponent per group (bytes)
  bool aborted = false;

  // this group's blocks i = gi, gi + kGroups, ... (its k-th in stage 2 gi + (k & 1))
  for (int i = gi, k = 0; i < nblocks; i += kGroups, ++k) {
    const int s = 2 * gi + (k & 1);
    const uint32_t par = static_cast<uint32_t>(k >> 1) & 1u;
    const bool fail = !aborted && !mbar_wait(&sm.bar[s], par);
    // one decision for the whole group before any warp-collective work
    if (bar_or(fail, 1 + gi, 128) && !aborted) {
      aborted = true;
      if ((warp & 3) == 0 && lane == 0) raise(a.err, M3S_DEVERR_TIMEOUT);
      // give the group's copies still in flight one more bounded wait before leaving
      mbar_wait(&sm.bar[s], par);
      if (i + kGroups < nblocks) mbar_wait(&sm.bar[s ^ 1], static_cast<uint32_t>((k + 1) >> 1) & 1u);
    }
    if (!aborted) {
      const uint8_t* kcs = stage0 + s * kStageB;
      const uint8_t* kss = kcs + kPageCodeBytes;
      const uint8_t* vcs = kss + kPageScaleB;
      const uint8_t* vss = vcs + kPageCodeBytes;
      const int ntok = sm.ntok[i];
      const int tb = (warp & 3) * 32;  // this warp's first token in the block

      // ---- S = Q K^T for 32 tokens (4 n8 tiles) ----
      float sacc[4][4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        sacc[c][0] = sacc[c][1] = sacc[c][2] = sacc[c][3] = 0.f;
        const int tok = tb + 8 * c + g;
        const uint4 kw = *reinterpret_cast<const uint4*>(kcs + tok * kCodeBytes + 16 * t);
        const uint32_t wv[4] = {kw.x, kw.y, kw.z, kw.w};
        if constexpr (MX) {
          // the thread's 16-byte chunk (dims 32t .. 32t+31) is E8M0 group t
          const uint32_t kw4 = *reinterpret_cast<const uint32_t*>(kss + tok * kMxScaleBytes);
          const int em = e8m0_max4(kw4);
          const uint32_t sj = pow2_neg_f16x2(em - static_cast<int>((kw4 >> (8 * t)) & 0xFFu));
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) {   // word jw: bytes 0, 1 = k-step 2jw, bytes 2, 3 = 2jw + 1
            uint32_t x[4];
            e2m1x8_to_f16x2(wv[jw], x[0], x[1], x[2], x[3]);
#pragma unroll
            for (int js = 0; js < 2; ++js) {
              const uint4 qv = sm.qa[2 * jw + js][lane];
              mma16816(sacc[c], qv.x, qv.y, qv.z, qv.w, hmul2(x[2 * js], sj), hmul2(x[2 * js + 1], sj));
            }
          }
          // columns 2t, 2t + 1 of this tile are the tokens decoded by lanes 8t, 8t + 4
          const float fk = pow2_f32(em - 127);
          const float f0 = __shfl_sync(0xffffffffu, fk, 8 * t);
          const float f1 = __shfl_sync(0xffffffffu, fk, 8 * t + 4);
          sacc[c][0] *= f0;
          sacc[c][1] *= f1;
          sacc[c][2] *= f0;
          sacc[c][3] *= f1;
        } else {
          const uint32_t sc = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(kss + tok * kScaleBytes + 2 * t));
          const uint32_t s0 = bcast_lo(sc), s1 = bcast_hi(sc);
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) {   // word jw: bytes 0, 1 = k-step 2jw, bytes 2, 3 = 2jw + 1
            uint32_t x[4];
            e2m1x8_to_f16x2(wv[jw], x[0], x[1], x[2], x[3]);
            const uint32_t sj = jw < 2 ? s0 : s1;
#pragma unroll
            for (int js = 0; js < 2; ++js) {
              const uint4 qv = sm.qa[2 * jw + js][lane];
              mma16816(sacc[c], qv.x, qv.y, qv.z, qv.w, hmul2(x[2 * js], sj), hmul2(x[2 * js + 1], sj));
            }
          }
        }
      }
      // ---- online softmax (log2 domain), causal mask inside the block. (The
      // logits are scaled one by one before the maximum: the reference is a
      // rounded logit and each term's exponent is a rounded logit minus it, so
      // the largest term is exactly 2^0 at any magnitude; folding the scale
      // into an fma with the reference took the product's rounding error, up
      // to 2^88 for logits near 2^112, into the exponent.) ----
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (ntok >= kPage) {   // (block-uniform) every token of the block is live
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            sacc[c][e] *= lsc0;
            sacc[c][2 + e] *= lsc1;
            mx0 = fmaxf(mx0, sacc[c][e]);
            mx1 = fmaxf(mx1, sacc[c][2 + e]);
          }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int tk = tb + 8 * c + 2 * t;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool live = tk + e < ntok;
            sacc[c][e] = live ? sacc[c][e] * lsc0 : -INFINITY;
            sacc[c][2 + e] = live ? sacc[c][2 + e] * lsc1 : -INFINITY;
            mx0 = fmaxf(mx0, sacc[c][e]);
            mx1 = fmaxf(mx1, sacc[c][2 + e]);
          }
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      // The reference m of a head moves only when the block's maximum exceeds
      // it by more than kMaxSlack (and on the head's first live token): the
      // sums stay relative to a reference up to 2^kMaxSlack below the true
      // maximum, so p <= 2^kMaxSlack, and the accumulators are rescaled rarely
      // (a warp-uniform skip) instead of on every block.
      const float n0 = mx0 > m0 + kMaxSlack ? mx0 : m0;
      const float n1 = mx1 > m1 + kMaxSlack ? mx1 : m1;
      if (__any_sync(0xffffffffu, n0 != m0 || n1 != m1)) {
        const float c0 = n0 == m0 ? 1.f : exp2f(m0 - n0);   // (0 from an empty reference)
        const float c1 = n1 == m1 ? 1.f : exp2f(m1 - n1);
        l0 *= c0;
        l1 *= c1;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[n][0] *= c0;
          o[n][1] *= c0;
          o[n][2] *= c1;
          o[n][3] *= c1;
        }
      }
      m0 = n0;
      m1 = n1;
      // (a head whose reference is still -inf has only masked logits: -inf - 0
      // gives p = 0 with no test per element)
      const float b0 = n0 == -INFINITY ? 0.f : n0, b1 = n1 == -INFINITY ? 0.f : n1;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float p0 = ex2_ftz(sacc[c][e] - b0);
          const float p1 = ex2_ftz(sacc[c][2 + e] - b1);
          sacc[c][e] = p0;
          sacc[c][2 + e] = p1;
          l0 += p0;
          l1 += p1;
        }
      }
      if constexpr (MX) {
        // the reference exponents take in this block's live tokens; the
        // accumulators (all of group t for this thread) follow exactly
        uint32_t e4 = tb + lane < ntok
                          ? *reinterpret_cast<const uint32_t*>(vss + (tb + lane) * kMxScaleBytes)
                          : 0u;
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) e4 = __vmaxu4(e4, __shfl_xor_sync(0xffffffffu, e4, sh));
        const uint32_t rnew = __vmaxu4(vref, e4);
        if (rnew != vref) {   // warp-uniform
          const float f = pow2_f32_nonpos(static_cast<int>((vref >> (8 * t)) & 0xFFu) -
                                          static_cast<int>((rnew >> (8 * t)) & 0xFFu));
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            o[n][0] *= f;
            o[n][1] *= f;
            o[n][2] *= f;
            o[n][3] *= f;
          }
          vref = rnew;
        }
      }
      // ---- O += P V over the warp's 32 tokens (2 k-steps of 16) ----
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t pa0 = pack_f16x2(sacc[2 * kk][0], sacc[2 * kk][1]);
        const uint32_t pa1 = pack_f16x2(sacc[2 * kk][2], sacc[2 * kk][3]);
        const uint32_t pa2 = pack_f16x2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        const uint32_t pa3 = pack_f16x2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
        const int t0 = tb + 16 * kk + 2 * t;  // tokens t0, t0+1 (b0) and t0+8, t0+9 (b1)
        // bytes 8g .. 8g+7 of each token: dims 16g .. 16g+15 (scale group g)
        const uint2 v0 = *reinterpret_cast<const uint2*>(vcs + t0 * kCodeBytes + 8 * g);
        const uint2 v1 = *reinterpret_cast<const uint2*>(vcs + (t0 + 1) * kCodeBytes + 8 * g);
        const uint2 v2 = *reinterpret_cast<const uint2*>(vcs + (t0 + 8) * kCodeBytes + 8 * g);
        const uint2 v3 = *reinterpret_cast<const uint2*>(vcs + (t0 + 9) * kCodeBytes + 8 * g);
        uint32_t s01, s23;   // the (token, token + 1) scale pairs of these dims
        if constexpr (MX) {   // dims 16g .. 16g+15 lie in E8M0 group g / 2: 2^(E - R)
          const int gm = g >> 1;
          const int rg = static_cast<int>((vref >> (8 * gm)) & 0xFFu);
          // (a masked token's exponent may exceed R: its weight is 0, keep its factor finite)
          const auto fac = [&](int tk) {
            return pow2_neg_f16x2(max(rg - static_cast<int>(vss[tk * kMxScaleBytes + gm]), 0)) & 0xFFFFu;
          };
          s01 = fac(t0) | (fac(t0 + 1) << 16);
          s23 = fac(t0 + 8) | (fac(t0 + 9) << 16);
        } else {
          s01 = e4m3x2_to_f16x2(vss[t0 * kScaleBytes + g] | (vss[(t0 + 1) * kScaleBytes + g] << 8));
          s23 = e4m3x2_to_f16x2(vss[(t0 + 8) * kScaleBytes + g] | (vss[(t0 + 9) * kScaleBytes + g] << 8));
        }
        const uint32_t wa[2] = {v0.x, v0.y}, wb[2] = {v1.x, v1.y};
        const uint32_t wc[2] = {v2.x, v2.y}, wd[2] = {v3.x, v3.y};
#pragma unroll
        for (int hw = 0; hw < 2; ++hw) {
          // interleave the nibbles of the two tokens: byte jj of lo01 holds
          // (token t0, token t0+1) low nibbles = dim 16g + 2jj of both tokens
          const uint32_t lo01 = (wa[hw] & 0x0F0F0F0Fu) | ((wb[hw] & 0x0F0F0F0Fu) << 4);
          const uint32_t hi01 = ((wa[hw] >> 4) & 0x0F0F0F0Fu) | (wb[hw] & 0xF0F0F0F0u);
          const uint32_t lo23 = (wc[hw] & 0x0F0F0F0Fu) | ((wd[hw] & 0x0F0F0F0Fu) << 4);
          const uint32_t hi23 = ((wc[hw] >> 4) & 0x0F0F0F0Fu) | (wd[hw] & 0xF0F0F0F0u);
          uint32_t xe0[4], xe1[4], xo0[4], xo1[4];   // byte bb of each word, decoded
          e2m1x8_to_f16x2(lo01, xe0[0], xe0[1], xe0[2], xe0[3]);
          e2m1x8_to_f16x2(lo23, xe1[0], xe1[1], xe1[2], xe1[3]);
          e2m1x8_to_f16x2(hi01, xo0[0], xo0[1], xo0[2], xo0[3]);
          e2m1x8_to_f16x2(hi23, xo1[0], xo1[1], xo1[2], xo1[3]);
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const int jj = 4 * hw + bb;
            mma16816(o[2 * jj], pa0, pa1, pa2, pa3, hmul2(xe0[bb], s01), hmul2(xe1[bb], s23));
            mma16816(o[2 * jj + 1], pa0, pa1, pa2, pa3, hmul2(xo0[bb], s01), hmul2(xo1[bb], s23));
          }
        }
      }
    }
    bar_sync(1 + gi, 128);  // every warp of the group is done with stage s
    if ((warp & 3) == 0 && lane == 0 && !aborted && i + 2 * kGroups < nblocks)
      issue(i + 2 * kGroups, sm.page[i + 2 * kGroups]);
  }

  if constexpr (MX) {   // undo the V reference: this thread's accumulators are group t
    const float f = pow2_f32(static_cast<int>((vref >> (8 * t)) & 0xFFu) - 127);
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= f;
      o[n][1] *= f;
      o[n][2] *= f;
      o[n][3] *= f;
    }
  }
  // ---- merge the four warps ----
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __syncthreads();   // every group is done with its stages (all copies landed)
  if (t == 0) {
    mg.m[warp][g] = m0;
    mg.m[warp][g + 8] = m1;
    mg.l[warp][g] = l0;
    mg.l[warp][g + 8] = l1;
  }
  // o[2jj + odd][e]: head g (e < 2) or g+8, dim 16*(2t + (e&1)) + 2jj + odd
#pragma unroll
  for (int jj = 0; jj < 8; ++jj)
#pragma unroll
    for (int odd = 0; odd < 2; ++odd)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int head = e < 2 ? g : g + 8;
        const int dim = 16 * (2 * t + (e & 1)) + 2 * jj + odd;
        mg.o[warp][merge_at(head, dim)] = o[2 * jj + odd][e];
      }
  __syncthreads();

  // this CTA's partial over its blocks: (M, L, O) per head, O relative to 2^M;
  // each warp's factor 2^(m_warp - M) once per head
  const int G = a.G;
  if (tid < 16) {
    const int head = tid;
    float M = -INFINITY;
#pragma unroll
    for (int wv = 0; wv < NW; ++wv) M = fmaxf(M, mg.m[wv][head]);
    float L = 0.f;
#pragma unroll
    for (int wv = 0; wv < NW; ++wv) {
      const float f = M == -INFINITY ? 0.f : exp2f(mg.m[wv][head] - M);
      mg.f[wv][head] = f;
      L += f * mg.l[wv][head];
    }
    sm.cta_m[head] = M;
    sm.cta_l[head] = L;
  }
  __syncthreads();
  const int dim = tid & (kHeadDim - 1);   // thread = (head half, output dim)
  for (int head = tid >> 7; head < 16; head += kThreads / kHeadDim) {
    float O = 0.f;
#pragma unroll
    for (int wv = 0; wv < NW; ++wv) O += mg.f[wv][head] * mg.o[wv][merge_at(head, dim)];
    sm.cta_o[head][dim] = O;
  }
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int nrank = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  if (nrank > 1) cluster.sync(); else __syncthreads();
  // rank k merges heads k, k + nrank, ...: thread = dim, every partial read
  // once through distributed shared memory, all loads independent
  const AttnFixed* peer[8];
#pragma unroll
  for (int rk = 0; rk < 8; ++rk) peer[rk] = rk < nrank ? cluster.map_shared_rank(&sm, rk) : &sm;
  for (int head = rank + nrank * (tid >> 7); head < G; head += nrank * (kThreads / kHeadDim)) {
    float mr[8], lr[8], orr[8];
#pragma unroll
    for (int rk = 0; rk < 8; ++rk) {
      if (rk < nrank) {
        mr[rk] = peer[rk]->cta_m[head];
        lr[rk] = peer[rk]->cta_l[head];
        orr[rk] = peer[rk]->cta_o[head][dim];
      } else {
        mr[rk] = -INFINITY;
        lr[rk] = 0.f;
        orr[rk] = 0.f;
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int rk = 0; rk < 8; ++rk) M = fmaxf(M, mr[rk]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int rk = 0; rk < 8; ++rk) {
        const float f = mr[rk] == -INFINITY ? 0.f : exp2f(mr[rk] - M);
        L += f * lr[rk];
        O += f * orr[rk];
      }
    }
    const int qh = kvh * G + head;
    a.out[(static_cast<size_t>(r) * a.Hq + qh) * kHeadDim + dim] = f32_to_bf16_bits(L > 0.f ? O / L : 0.f);
    if (a.lse && dim == 0)
      a.lse[static_cast<size_t>(r) * a.Hq + qh] =
          L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
  if (nrank > 1) cluster.sync();  // keep every rank's shared memory alive until rank 0 is done
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int sm_count_cached() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      return 148;
  }
  return n;
}

// Split count: enough CTAs for four per SM (the one-group CTA's residency), at
// most one block per split and at most 8 splits (one portable thread-block
// cluster per (kv head, row)).
int attention_splits(int R, int Hkv, int topk, int* ips) {
  if (topk <= 0) { *ips = 0; return 1; }
  const long long ctas = static_cast<long long>(R) * Hkv;
  const long long slots = 4ll * sm_count_cached();
  long long want = ctas > 0 ? (slots + ctas - 1) / ctas : 1;
  if (want < 1) want = 1;
  if (want > 8) want = 8;
  if (want > topk) want = topk;
  const int per = static_cast<int>((topk + want - 1) / want);
  *ips = per;
  return (topk + per - 1) / per;
}

// Dynamic shared memory of a CTA of nw warps: the fixed part, then the page
// stages (two per group of four warps) or the merge buffers, whichever is larger.
size_t attention_smem(int nw, bool mx) {
  const size_t stage = 2 * (kPageCodeBytes + static_cast<size_t>(mx ? kMxPageScaleBytes : kPageScaleBytes));
  const size_t st = static_cast<size_t>(nw / 2) * stage;
  const size_t mrg = nw == 8 ? sizeof(AttnMerge<8>) : sizeof(AttnMerge<4>);
  return kAttFixedBytes + (st > mrg ? st : mrg);
}

}  // namespace m3s

namespace m3s {

// m3s_sparse_attention, or (topk_ids == nullptr) its candidates mode: the row's
// top-k merged from the scorer's lists cand / meta, its ids written to ids_out.
// The argument checks of m3s_sparse_attention (before anything is launched).
int check_attention(const uint16_t* q, int32_t Hq, int32_t Hkv, m3s_fp4_plane k, m3s_fp4_plane v,
                    const int32_t* block_table, int32_t bt_stride, int32_t B, const int32_t* row_req,
                    const int32_t* row_len, bool have_ids, int32_t topk, int32_t R, const uint16_t* out) {
  if (R < 0 || B < 0 || Hq < 1 || Hkv < 1 || topk < 0 || bt_stride < 0) return M3S_ERR_INVALID;
  if (Hq % Hkv != 0) return M3S_ERR_INVALID;
  if (Hq / Hkv > M3S_MAX_GQA || topk > M3S_MAX_TOPK) return M3S_ERR_UNSUPPORTED;
  if (k.num_heads != Hkv || v.num_heads != Hkv || k.num_pages != v.num_pages || k.num_pages < 0)
    return M3S_ERR_INVALID;
  if ((k.format != M3S_FMT_NVFP4 && k.format != M3S_FMT_MXFP4) ||
      (v.format != M3S_FMT_NVFP4 && v.format != M3S_FMT_MXFP4))
    return M3S_ERR_INVALID;
  if (k.format != v.format) return M3S_ERR_UNSUPPORTED;   // one format per cache
  if (R == 0) return M3S_OK;
  if (R > 65535) return M3S_ERR_UNSUPPORTED;
  if (!q || !out || !row_req || !row_len || (topk > 0 && !have_ids)) return M3S_ERR_INVALID;
  if (!aligned16(q) || !aligned16(out)) return M3S_ERR_INVALID;
  if (k.num_pages > 0 && (!k.codes || !k.scales || !v.codes || !v.scales || !aligned16(k.codes) ||
                          !aligned16(k.scales) || !aligned16(v.codes) || !aligned16(v.scales)))
    return M3S_ERR_INVALID;
  if (B > 0 && (bt_stride < 1 || !block_table)) return M3S_ERR_INVALID;
  return M3S_OK;
}

int launch_attention(const uint16_t* q, int32_t Hq, int32_t Hkv, m3s_fp4_plane k, m3s_fp4_plane v,
                     const int32_t* block_table, int32_t bt_stride, int32_t B, const int32_t* row_req,
                     const int32_t* row_len, const int32_t* topk_ids, int32_t topk, int32_t R,
                     float sm_scale, uint16_t* out, float* lse, int32_t* err, cudaStream_t stream,
                     const unsigned long long* cand, const int2* meta, int32_t* ids_out, int cand_lists,
                     int cand_stride) {
  const int rc = check_attention(q, Hq, Hkv, k, v, block_table, bt_stride, B, row_req, row_len,
                                 topk_ids != nullptr || (cand && meta), topk, R, out);
  if (rc != M3S_OK || R == 0) return rc;
  int ips = 0;
  const int nsplit = attention_splits(R, Hkv, topk, &ips);
  AttnArgs a{q, Hq, Hkv, Hq / Hkv, k.codes, k.scales, v.codes, v.scales, k.num_pages, block_table,
             bt_stride, row_req, row_len, topk_ids, topk, R, B,
             sm_scale * 1.4426950408889634f, nsplit, ips, out, lse, err, cand, meta, ids_out,
             cand_lists, cand_stride};
  // two warp groups when the grid has at most one CTA per SM (each SM then
  // computes two of its blocks at once), else one (more CTAs resident per SM)
  const bool mx = k.format == M3S_FMT_MXFP4;
  const bool wide = static_cast<long long>(nsplit) * Hkv * R <= sm_count_cached();
  const int nw = wide ? 8 : 4;
  const auto kernel = mx ? (wide ? attention_kernel<true, 8> : attention_kernel<true, 4>)
                         : (wide ? attention_kernel<false, 8> : attention_kernel<false, 4>);
  const size_t smem = attention_smem(nw, mx);
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return M3S_ERR_LAUNCH;
  if (launch_kernel(kernel, dim3(nsplit, Hkv, R), dim3(nw * 32), smem, stream, nsplit, a) != cudaSuccess)
    return M3S_ERR_LAUNCH;
  return M3S_OK;
}

}  // namespace m3s

extern "C" int m3s_sparse_attention(const uint16_t* q, int32_t Hq, int32_t Hkv, m3s_fp4_plane k,
                                    m3s_fp4_plane v, const int32_t* block_table,
                                    int32_t bt_stride, int32_t B, const int32_t* row_req,
                                    const int32_t* row_len, const int32_t* topk_ids, int32_t topk,
                                    int32_t R, float sm_scale, uint16_t* out, float* lse, void* ws,
                                    size_t ws_bytes, int32_t* err, void* stream) {
  (void)ws;
  (void)ws_bytes;
  return m3s::launch_attention(q, Hq, Hkv, k, v, block_table, bt_stride, B, row_req, row_len, topk_ids,
                               topk, R, sm_scale, out, lse, err, static_cast<cudaStream_t>(stream),
                               nullptr, nullptr, nullptr, 0, 1);
}
