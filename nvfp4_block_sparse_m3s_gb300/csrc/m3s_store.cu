// Quantise-store of BF16 rows into paged NVFP4 or MXFP4 planes, and the row map.
//
// Quantisation: "[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache"
// (ROCm/ATOM #2744), Design / Write path -- per 16 elements
// scale = e4m3(amax / 6), codes rounded half-to-even on the e2m1 grid and
// saturating at 6. MXFP4 (same page, Follow-up: MXFP4 caches) -- one E8M0
// scale per 32 elements, 2^E with E = floor(log2(amax)) - 2 clamped to
// [-127, 127] (the OCP MX shared exponent), codes |x| / 2^E rounded the same
// way. Row map: same page, Design / Attention (one launch maps each row to
// its request and causal length).
#include <cuda_runtime.h>

#include "m3s_device.cuh"

namespace m3s {
namespace {

// e2m1 magnitude code of |x| for scale s, decided without division: the seven
// decision points are the grid midpoints times s, which are exact in fp32 (s
// has 4 significant bits, the midpoints at most 3). A tie (|x| equal to a
// midpoint) goes to the even code, hence '>' below an even code and '>=' below
// an odd one. Values beyond 5*s saturate to code 7 (6*s).
__device__ __forceinline__ uint32_t e2m1_code(uint32_t bf16, const float (&thr)[7]) {
  const float ax = __uint_as_float((bf16 & 0x7FFFu) << 16);
  const uint32_t mag = (ax > thr[0]) + (ax >= thr[1]) + (ax > thr[2]) + (ax >= thr[3]) +
                       (ax > thr[4]) + (ax >= thr[5]) + (ax > thr[6]);
  return mag | ((bf16 >> 12) & 8u);  // sign = the sign bit of the BF16 input
}

// One 16-element group held as 8 words of BF16 pairs -> 2 words of packed codes
// (element e in nibble e) and the scale byte.
__device__ __forceinline__ void quantise_group(const uint32_t (&x)[8], uint32_t& lo, uint32_t& hi,
                                               float scale) {
  float thr[7];
  const float mids[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
#pragma unroll
  for (int i = 0; i < 7; ++i) thr[i] = mids[i] * scale;
  lo = hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lo |= e2m1_code(x[i] & 0xFFFFu, thr) << (8 * i);
    lo |= e2m1_code(x[i] >> 16, thr) << (8 * i + 4);
    hi |= e2m1_code(x[i + 4] & 0xFFFFu, thr) << (8 * i);
    hi |= e2m1_code(x[i + 4] >> 16, thr) << (8 * i + 4);
  }
  if (scale == 0.0f) lo = hi = 0;  // a zero (or underflowed) scale stores zero codes
}

// The MXFP4 shared exponent of a group whose largest magnitude has BF16 bits
// am: floor(log2(amax)) - 2, clamped to E8M0's [-127, 127]. A normal BF16's
// floor(log2) is its exponent field minus 127; a subnormal one is m * 2^-133
// (m = its mantissa bits); amax 0 gives -127.
__device__ __forceinline__ int mx_shared_exponent(uint32_t am) {
  int fl;
  if (am >= 0x80u) fl = static_cast<int>(am >> 7) - 127;
  else if (am != 0) fl = (31 - __clz(static_cast<int>(am))) - 133;
  else fl = -200;
  return min(127, max(-127, fl - 2));
}

// Largest |x| of a group, as BF16 magnitude bits (non-negative floats order as
// their bit patterns).
__device__ __forceinline__ uint32_t group_amax_bits(const uint32_t (&x)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = __vmaxu2(m, x[i] & 0x7FFF7FFFu);
  return max(m & 0xFFFFu, m >> 16);
}

// One thread quantises 32 elements (two NVFP4 scale groups, one MXFP4 group)
// of one (row, head): it reads 64 B, writes 16 B of codes with one 128-bit
// store, and the four threads of a (row, head) gather their scale bytes so one
// of them writes the record's 8 (NVFP4) or 4 (MXFP4) scale bytes in one store.
struct StoreJob {
  const uint16_t* src;
  int64_t stride;
  int64_t total_threads;  // T * H * 4
  int32_t H;
  int32_t mx;             // 1: MXFP4 plane
  uint8_t* codes;
  uint8_t* scales;
  int64_t capacity;       // num_pages * 128
};

struct StoreBatch {
  StoreJob job[M3S_MAX_STORE_JOBS];
  // the row map in the same launch (grid row njobs), or rows_job = -1
  int rows_job;
  const int32_t* cu_q;
  const int32_t* seq_len;
  int32_t B, R;
  int32_t* row_req;
  int32_t* row_len;
};

// Row r's request and causal length (m3s_decode_rows): a binary search over cu_q.
__device__ __forceinline__ void row_of(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ seq_len,
                                      int32_t B, int r, int32_t* req_out, int32_t* len_out) {
  int32_t req = -1, len = 0;
  if (B > 0 && r < cu_q[B]) {
    int lo = 0, hi = B;  // cu_q[lo] <= r < cu_q[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu_q[mid] <= r) lo = mid; else hi = mid;
    }
    const int qb = cu_q[lo + 1] - cu_q[lo];
    req = lo;
    len = seq_len[lo] - qb + (r - cu_q[lo]) + 1;
  }
  *req_out = req;
  *len_out = len;
}

__global__ void __launch_bounds__(256) nvfp4_store_kernel(const StoreBatch batch,
                                                         const int64_t* __restrict__ slots,
                                                         int32_t* err) {
  pdl_trigger();
  pdl_wait();
  if (static_cast<int>(blockIdx.y) == batch.rows_job) {   // the row map's grid row
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < batch.R) row_of(batch.cu_q, batch.seq_len, batch.B, r, &batch.row_req[r], &batch.row_len[r]);
    return;
  }
  const StoreJob& jb = batch.job[blockIdx.y];
  const uint16_t* __restrict__ src = jb.src;
  const int64_t stride = jb.stride;
  const int32_t H = jb.H;
  uint8_t* __restrict__ codes = jb.codes;
  uint8_t* __restrict__ scales = jb.scales;
  const int64_t capacity = jb.capacity;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= jb.total_threads) return;
  const int part = static_cast<int>(idx & 3);
  const int64_t rh = idx >> 2;
  const int h = static_cast<int>(rh % H);
  const int64_t r = rh / H;
  const int64_t slot = slots[r];
  if (slot < 0) return;  // pad row: untouched
  if (slot >= capacity) {
    if (part == 0 && h == 0) raise(err, M3S_DEVERR_SLOT);
    return;
  }
  const uint4* p = reinterpret_cast<const uint4*>(src + r * stride + h * kHeadDim + part * 32);
  const uint4 v0 = __ldg(p), v1 = __ldg(p + 1), v2 = __ldg(p + 2), v3 = __ldg(p + 3);
  const uint32_t g0[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  const uint32_t g1[8] = {v2.x, v2.y, v2.z, v2.w, v3.x, v3.y, v3.z, v3.w};
  const int64_t page = slot / kPage, pos = slot % kPage;
  const int64_t rec = (page * H + h) * kPage + pos;
  const int lane = threadIdx.x & 31;
  const unsigned mask = 0xFu << (lane & 28);

  if (jb.mx) {
    // one E8M0 group: the codes are |x| / 2^E on the grid, decided against the
    // midpoints times 2^E (exact in fp32 down to 2^-129)
    const int E = mx_shared_exponent(max(group_amax_bits(g0), group_amax_bits(g1)));
    const float s = pow2_f32(E);
    uint4 out;
    quantise_group(g0, out.x, out.y, s);
    quantise_group(g1, out.z, out.w, s);
    *reinterpret_cast<uint4*>(codes + rec * kCodeBytes + part * 16) = out;
    const uint32_t mine = static_cast<uint32_t>(E + 127);
    const uint32_t p1 = __shfl_sync(mask, mine, (lane & 28) + 1);
    const uint32_t p2 = __shfl_sync(mask, mine, (lane & 28) + 2);
    const uint32_t p3 = __shfl_sync(mask, mine, (lane & 28) + 3);
    if (part == 0)
      *reinterpret_cast<uint32_t*>(scales + rec * kMxScaleBytes) = mine | (p1 << 8) | (p2 << 16) | (p3 << 24);
    return;
  }

  // scale = E4M3(amax / 6): the correctly rounded fp32 quotient cannot sit on or
  // across an E4M3 rounding boundary unless the exact quotient does (amax has 8
  // significant bits), so fp32 division followed by a round-to-nearest-even,
  // saturate-finite conversion gives the exact result.
  const float q0 = __fdiv_rn(bf16_bits_to_f32(group_amax_bits(g0)), 6.0f);
  const float q1 = __fdiv_rn(bf16_bits_to_f32(group_amax_bits(g1)), 6.0f);
  uint16_t pair;  // byte 0 = group 2*part, byte 1 = group 2*part+1
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(q1), "f"(q0));
  uint32_t sw = e4m3x2_to_f16x2(pair);
  const __half2 s2 = *reinterpret_cast<const __half2*>(&sw);
  const float s0 = __low2float(s2), s1 = __high2float(s2);

  uint4 out;
  quantise_group(g0, out.x, out.y, s0);
  quantise_group(g1, out.z, out.w, s1);
  *reinterpret_cast<uint4*>(codes + rec * kCodeBytes + part * 16) = out;

  const uint32_t mine = pair;
  const uint32_t p1 = __shfl_sync(mask, mine, (lane & 28) + 1);
  const uint32_t p2 = __shfl_sync(mask, mine, (lane & 28) + 2);
  const uint32_t p3 = __shfl_sync(mask, mine, (lane & 28) + 3);
  if (part == 0) {
    *reinterpret_cast<uint2*>(scales + rec * kScaleBytes) = make_uint2(mine | (p1 << 16), p2 | (p3 << 16));
  }
}

// ---- quantise-at-write: RMSNorm / rotate-half RoPE / BF16 round / store ----
// #2744, Follow-up: MXFP4 caches: the quantisation inside the kernel that
// normalises, rotates and writes the step's rows. One warp per (job, row,
// head); lane l owns elements 4l .. 4l+3. Every float operation is rounded on
// its own and the sum of squares runs in one fixed order, so the BF16 values
// (and hence the stored bytes) are those of the unfused path.
struct WriteJob {
  const uint16_t* src;
  int64_t stride;
  int32_t H;
  int32_t rope;
  int32_t mx;            // destination plane format (1: MXFP4)
  const float* weight;   // RMSNorm weight [128] or null
  uint8_t* codes;        // destination plane, or null when out is given
  uint8_t* scales;
  int64_t capacity;
  uint16_t* out;         // BF16 rows, or null
  int64_t out_stride;
  int64_t warp0;         // first warp (over the whole launch) of this job
};

struct WriteBatch {
  WriteJob job[M3S_MAX_WRITE_JOBS];
  int32_t njobs;
  int64_t total_warps;
};

// Heads of one row handled by one warp: their loads are all issued before any
// arithmetic, so a warp keeps this many 256-byte rows in flight.
constexpr int kWriteHeadsPerWarp = 4;

// One head of one row (its 4 elements per lane in raw): normalise, rotate,
// round to BF16 and write, as described above.
__device__ __forceinline__ void write_head(const WriteJob& jb, int64_t t, int h, int64_t slot, uint2 raw,
                                           const float4& w, const float4& c4, const float4& s4,
                                           int32_t rd, float eps, int lane) {
  float y[4] = {bf16_bits_to_f32(raw.x & 0xFFFFu), bf16_bits_to_f32(raw.x >> 16),
                bf16_bits_to_f32(raw.y & 0xFFFFu), bf16_bits_to_f32(raw.y >> 16)};
  if (jb.weight) {
    float p = __fmul_rn(y[0], y[0]);
#pragma unroll
    for (int i = 1; i < 4; ++i) p = __fadd_rn(p, __fmul_rn(y[i], y[i]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, off));
    const float ss = __shfl_sync(0xffffffffu, p, 0);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, 0.0078125f), eps)));
    const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = __fmul_rn(__fmul_rn(y[i], r), wv[i]);
  }
  if (jb.rope) {
    const int half = rd >> 1;  // a multiple of 4: a pair's partner is half / 4 lanes away
    const int d0 = 4 * lane;
    const int partner = d0 < half ? lane + (half >> 2) : (d0 < rd ? lane - (half >> 2) : lane);
    float py[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) py[i] = __shfl_sync(0xffffffffu, y[i], partner);
    if (d0 < rd) {
      const float c[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        y[i] = d0 < half ? __fsub_rn(__fmul_rn(y[i], c[i]), __fmul_rn(py[i], sn[i]))
                         : __fadd_rn(__fmul_rn(y[i], c[i]), __fmul_rn(py[i], sn[i]));
    }
  }
  uint32_t bv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) bv[i] = f32_to_bf16_bits(y[i]);
  if (jb.out) {
    *reinterpret_cast<uint2*>(jb.out + t * jb.out_stride + h * kHeadDim + 4 * lane) =
        make_uint2(bv[0] | (bv[1] << 16), bv[2] | (bv[3] << 16));
    return;
  }
  // quantise the BF16 values as the store does: NVFP4 groups of 16 span 4
  // lanes, MXFP4 groups of 32 span 8
  uint32_t am = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) am = max(am, bv[i] & 0x7FFFu);
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
  float s;
  uint32_t sbyte;
  if (jb.mx) {
    am = max(am, __shfl_xor_sync(0xffffffffu, am, 4));
    const int E = mx_shared_exponent(am);
    s = pow2_f32(E);
    sbyte = static_cast<uint32_t>(E + 127);
  } else {
    const float q = __fdiv_rn(bf16_bits_to_f32(am), 6.0f);
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(q));
    sbyte = pair & 0xFFu;
    const uint32_t sh = e4m3x2_to_f16x2(sbyte);
    s = __half2float(__ushort_as_half(static_cast<unsigned short>(sh & 0xFFFFu)));
  }
  const float mids[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
  float thr[7];
#pragma unroll
  for (int i = 0; i < 7; ++i) thr[i] = mids[i] * s;
  uint32_t code = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) code |= e2m1_code(bv[i], thr) << (4 * i);
  if (s == 0.0f) code = 0;  // NVFP4: a zero scale stores zero codes
  const int64_t page = slot / kPage, pos = slot % kPage;
  const int64_t rec = (page * jb.H + h) * kPage + pos;
  *reinterpret_cast<uint16_t*>(jb.codes + rec * kCodeBytes + 2 * lane) = static_cast<uint16_t>(code);
  if (jb.mx) {
    if ((lane & 7) == 0) jb.scales[rec * kMxScaleBytes + (lane >> 3)] = static_cast<uint8_t>(sbyte);
  } else {
    if ((lane & 3) == 0) jb.scales[rec * kScaleBytes + (lane >> 2)] = static_cast<uint8_t>(sbyte);
  }
}

__global__ void __launch_bounds__(256) write_kernel(const WriteBatch b, const int64_t* __restrict__ slots,
                                                   const float* __restrict__ cos_t,
                                                   const float* __restrict__ sin_t, int32_t rd,
                                                   float eps, int32_t* err) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (gw >= b.total_warps) return;  // warp-uniform
  int j = 0;
  while (j + 1 < b.njobs && gw >= b.job[j + 1].warp0) ++j;
  const WriteJob& jb = b.job[j];
  const int groups = (jb.H + kWriteHeadsPerWarp - 1) / kWriteHeadsPerWarp;
  const int64_t rg = gw - jb.warp0;
  const int h0 = static_cast<int>(rg % groups) * kWriteHeadsPerWarp;
  const int nh = min(kWriteHeadsPerWarp, jb.H - h0);
  const int64_t t = rg / groups;
  int64_t slot = 0;
  if (!jb.out) {
    slot = slots[t];
    if (slot < 0) return;  // pad row: untouched (warp-uniform)
    if (slot >= jb.capacity) {
      if (lane == 0 && h0 == 0) raise(err, M3S_DEVERR_SLOT);
      return;
    }
  }
  uint2 raw[kWriteHeadsPerWarp];
#pragma unroll
  for (int k = 0; k < kWriteHeadsPerWarp; ++k)
    if (k < nh) raw[k] = *reinterpret_cast<const uint2*>(jb.src + t * jb.stride + (h0 + k) * kHeadDim + 4 * lane);
  float4 w = make_float4(0.f, 0.f, 0.f, 0.f), c4 = w, s4 = w;
  if (jb.weight) w = *reinterpret_cast<const float4*>(jb.weight + 4 * lane);
  if (jb.rope && 4 * lane < rd) {
    const int half = rd >> 1, d0 = 4 * lane;
    const int ci = d0 < half ? d0 : d0 - half;
    c4 = *reinterpret_cast<const float4*>(cos_t + t * half + ci);
    s4 = *reinterpret_cast<const float4*>(sin_t + t * half + ci);
  }
#pragma unroll
  for (int k = 0; k < kWriteHeadsPerWarp; ++k)
    if (k < nh) write_head(jb, t, h0 + k, slot, raw[k], w, c4, s4, rd, eps, lane);   // nh is warp-uniform
}

__global__ void decode_rows_kernel(const int32_t* __restrict__ cu_q,
                                   const int32_t* __restrict__ seq_len, int32_t B, int32_t R,
                                   int32_t* __restrict__ row_req, int32_t* __restrict__ row_len) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  row_of(cu_q, seq_len, B, r, &row_req[r], &row_len[r]);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace m3s

namespace m3s {
namespace {
int check_job(const uint16_t* src, int64_t stride, int32_t H, const m3s_fp4_plane& dst) {
  if (H <= 0 || dst.num_pages < 0 || dst.num_heads != H) return M3S_ERR_INVALID;
  if (dst.format != M3S_FMT_NVFP4 && dst.format != M3S_FMT_MXFP4) return M3S_ERR_INVALID;
  if (!src || !dst.codes || !dst.scales) return M3S_ERR_INVALID;
  if (!aligned16(src) || !aligned16(dst.codes) || !aligned16(dst.scales)) return M3S_ERR_INVALID;
  if (stride < static_cast<int64_t>(H) * kHeadDim || (stride & 7)) return M3S_ERR_INVALID;
  return M3S_OK;
}

int launch_store(const m3s_store_job* jobs, int32_t njobs, int32_t T, const int64_t* slots,
                 int32_t* err, cudaStream_t st, const int32_t* cu_q = nullptr,
                 const int32_t* seq_len = nullptr, int32_t B = 0, int32_t R = 0,
                 int32_t* row_req = nullptr, int32_t* row_len = nullptr) {
  StoreBatch b{};
  b.rows_job = -1;
  int64_t most = 0;
  for (int i = 0; i < njobs; ++i) {
    const m3s_store_job& j = jobs[i];
    b.job[i] = StoreJob{j.src, j.src_row_stride, static_cast<int64_t>(T) * j.H * 4, j.H,
                        j.dst.format == M3S_FMT_MXFP4 ? 1 : 0, j.dst.codes, j.dst.scales,
                        static_cast<int64_t>(j.dst.num_pages) * kPage};
    most = b.job[i].total_threads > most ? b.job[i].total_threads : most;
  }
  int64_t blocks = (most + 255) / 256;
  int rows = njobs;
  if (R > 0) {   // the row map as one more grid row
    b.rows_job = njobs;
    b.cu_q = cu_q;
    b.seq_len = seq_len;
    b.B = B;
    b.R = R;
    b.row_req = row_req;
    b.row_len = row_len;
    blocks = blocks > (R + 255) / 256 ? blocks : (R + 255) / 256;
    ++rows;
  }
  if (blocks > 0x7FFFFFFF) return M3S_ERR_UNSUPPORTED;
  return launch_kernel(nvfp4_store_kernel, dim3(static_cast<unsigned>(blocks), rows), dim3(256), 0,
                       st, 0, b, slots, err) == cudaSuccess
             ? M3S_OK
             : M3S_ERR_LAUNCH;
}
}  // namespace
}  // namespace m3s

extern "C" int m3s_nvfp4_store(const uint16_t* src, int64_t src_row_stride, int32_t T, int32_t H,
                               const int64_t* slot_mapping, m3s_fp4_plane dst, int32_t* err,
                               void* stream) {
  using namespace m3s;
  if (T < 0 || H <= 0 || dst.num_pages < 0 || dst.num_heads != H) return M3S_ERR_INVALID;
  if (T == 0) return M3S_OK;
  if (!slot_mapping) return M3S_ERR_INVALID;
  const int rc = check_job(src, src_row_stride, H, dst);
  if (rc != M3S_OK) return rc;
  const m3s_store_job job{src, src_row_stride, H, dst};
  return launch_store(&job, 1, T, slot_mapping, err, static_cast<cudaStream_t>(stream));
}

extern "C" int m3s_nvfp4_store_batch(const m3s_store_job* jobs, int32_t njobs, int32_t T,
                                     const int64_t* slot_mapping, int32_t* err, void* stream) {
  using namespace m3s;
  if (T < 0 || njobs < 0 || njobs > M3S_MAX_STORE_JOBS || (njobs > 0 && !jobs)) return M3S_ERR_INVALID;
  if (T == 0 || njobs == 0) return M3S_OK;
  if (!slot_mapping) return M3S_ERR_INVALID;
  for (int i = 0; i < njobs; ++i) {
    const int rc = check_job(jobs[i].src, jobs[i].src_row_stride, jobs[i].H, jobs[i].dst);
    if (rc != M3S_OK) return rc;
  }
  return launch_store(jobs, njobs, T, slot_mapping, err, static_cast<cudaStream_t>(stream));
}

extern "C" int m3s_nvfp4_store_batch_rows(const m3s_store_job* jobs, int32_t njobs, int32_t T,
                                          const int64_t* slot_mapping, const int32_t* cu_q,
                                          const int32_t* seq_len, int32_t B, int32_t R, int32_t* row_req,
                                          int32_t* row_len, int32_t* err, void* stream) {
  using namespace m3s;
  if (T < 0 || njobs < 0 || njobs > M3S_MAX_STORE_JOBS || (njobs > 0 && !jobs)) return M3S_ERR_INVALID;
  if (B < 0 || R < 0) return M3S_ERR_INVALID;
  if (R > 0 && (!cu_q || !row_req || !row_len || (B > 0 && !seq_len))) return M3S_ERR_INVALID;
  const bool store = T > 0 && njobs > 0;
  if (store) {
    if (!slot_mapping) return M3S_ERR_INVALID;
    for (int i = 0; i < njobs; ++i) {
      const int rc = check_job(jobs[i].src, jobs[i].src_row_stride, jobs[i].H, jobs[i].dst);
      if (rc != M3S_OK) return rc;
    }
  }
  if (!store && R == 0) return M3S_OK;
  return launch_store(jobs, store ? njobs : 0, store ? T : 0, slot_mapping, err, static_cast<cudaStream_t>(stream),
                      cu_q, seq_len, B, R, row_req, row_len);
}

extern "C" int m3s_qk_norm_rope_store(const m3s_write_job* jobs, int32_t njobs, int32_t T,
                                      const int64_t* slot_mapping, const float* rope_cos,
                                      const float* rope_sin, int32_t rotary_dim, float eps,
                                      int32_t* err, void* stream) {
  using namespace m3s;
  if (T < 0 || njobs < 0 || njobs > M3S_MAX_WRITE_JOBS || (njobs > 0 && !jobs)) return M3S_ERR_INVALID;
  bool any_rope = false, any_plane = false;
  WriteBatch b{};
  b.njobs = njobs;
  int64_t warps = 0;
  for (int i = 0; i < njobs; ++i) {
    const m3s_write_job& j = jobs[i];
    if (j.H <= 0 || !j.src || !aligned16(j.src) || j.src_row_stride < static_cast<int64_t>(j.H) * kHeadDim ||
        (j.src_row_stride & 7))
      return M3S_ERR_INVALID;
    if (j.norm_weight && !aligned16(j.norm_weight)) return M3S_ERR_INVALID;
    if (j.out) {
      if (!aligned16(j.out) || j.out_row_stride < static_cast<int64_t>(j.H) * kHeadDim || (j.out_row_stride & 7))
        return M3S_ERR_INVALID;
    } else {
      const int rc = check_job(j.src, j.src_row_stride, j.H, j.dst);
      if (rc != M3S_OK) return rc;
      any_plane = true;
    }
    any_rope |= j.rope != 0;
    b.job[i] = WriteJob{j.src, j.src_row_stride, j.H, j.rope != 0 ? 1 : 0,
                        (!j.out && j.dst.format == M3S_FMT_MXFP4) ? 1 : 0, j.norm_weight,
                        j.out ? nullptr : j.dst.codes, j.out ? nullptr : j.dst.scales,
                        j.out ? 0 : static_cast<int64_t>(j.dst.num_pages) * kPage, j.out,
                        j.out_row_stride, warps};
    warps += static_cast<int64_t>(T) * ((j.H + kWriteHeadsPerWarp - 1) / kWriteHeadsPerWarp);
  }
  if (any_rope && (rotary_dim < 8 || rotary_dim > kHeadDim || (rotary_dim & 7) || !rope_cos || !rope_sin ||
                   !aligned16(rope_cos) || !aligned16(rope_sin)))
    return M3S_ERR_INVALID;
  if (T == 0 || njobs == 0) return M3S_OK;
  if (any_plane && !slot_mapping) return M3S_ERR_INVALID;
  b.total_warps = warps;
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > 0x7FFFFFFF) return M3S_ERR_UNSUPPORTED;
  return launch_kernel(write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                       static_cast<cudaStream_t>(stream), 0, b, slot_mapping, rope_cos, rope_sin,
                       any_rope ? rotary_dim : 0, eps, err) == cudaSuccess
             ? M3S_OK
             : M3S_ERR_LAUNCH;
}

extern "C" int m3s_decode_rows(const int32_t* cu_q, const int32_t* seq_len, int32_t B, int32_t R,
                               int32_t* row_req, int32_t* row_len, void* stream) {
  if (B < 0 || R < 0) return M3S_ERR_INVALID;
  if (R == 0) return M3S_OK;
  if (!cu_q || !row_req || !row_len || (B > 0 && !seq_len)) return M3S_ERR_INVALID;
  return m3s::launch_kernel(m3s::decode_rows_kernel, dim3((R + 255) / 256), dim3(256), 0,
                            static_cast<cudaStream_t>(stream), 0, cu_q, seq_len, B, R, row_req,
                            row_len) == cudaSuccess
             ? M3S_OK
             : M3S_ERR_LAUNCH;
}
