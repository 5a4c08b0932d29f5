// Device helpers shared by the m3s kernels (sm_103a): bounded mbarrier waits,
// bulk global->shared copies, f16 tensor-core mma, and the in-register NVFP4
// dequantisation.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/m3s.h"

namespace m3s {

constexpr int kHeadDim = 128;
constexpr int kPage = 128;
constexpr int kCodeBytes = 64;     // e2m1 payload per token and head
constexpr int kScaleBytes = 8;     // E4M3 scales per token and head
constexpr int kPageCodeBytes = kPage * kCodeBytes;    // 8192
constexpr int kPageScaleBytes = kPage * kScaleBytes;  // 1024
constexpr int kMxScaleBytes = 4;   // MXFP4: E8M0 scales per token and head (one per 32)
constexpr int kMxPageScaleBytes = kPage * kMxScaleBytes;  // 512

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void raise(int32_t* err, int32_t bits) {
  if (err != nullptr) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false after the limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---- bulk copies (TMA, 1-D) -------------------------------------------------

// Bring `bytes` (a multiple of 16, from a 16-byte aligned address) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Copy `bytes` (multiple of 16; both addresses 16-byte aligned) from global to
// this CTA's shared memory; completion is signalled as transaction bytes on bar.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Order this thread's earlier shared-memory accesses before later async-proxy
// (bulk copy) writes to the same buffer.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 2-D tiled bulk tensor copy (TMA): the box at (x, y) of the tensor map (a
// CUtensorMap kernel parameter) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- numeric conversions ----------------------------------------------------

// The four bytes of a word (byte b = elements 2b, 2b+1) -> four f16x2. Exact.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& o0, uint32_t& o1,
                                                uint32_t& o2, uint32_t& o3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) -> f16x2. Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
      : "=r"(r)
      : "r"(two));
  return r;
}

// fp16x2 broadcast of 2^-d (d >= 0): normal down to 2^-14, subnormal to 2^-24,
// zero beyond.
__device__ __forceinline__ uint32_t pow2_neg_f16x2(int d) {
  const uint32_t h = d <= 14 ? static_cast<uint32_t>(15 - d) << 10 : (d <= 24 ? 1u << (24 - d) : 0u);
  return h | (h << 16);
}

// 2^e as fp32 for e in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float pow2_f32(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// The largest of the four E8M0 bytes of a word (an MXFP4 record's exponents).
__device__ __forceinline__ int e8m0_max4(uint32_t w4) {
  const uint32_t m2 = __vmaxu4(w4, w4 >> 16);
  return static_cast<int>(max(m2 & 0xFFu, (m2 >> 8) & 0xFFu));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Broadcast the low (sel = 0) or high (sel = 1) half of an f16x2 into both halves.
__device__ __forceinline__ uint32_t bcast_lo(uint32_t x) { return __byte_perm(x, 0, 0x1010); }
__device__ __forceinline__ uint32_t bcast_hi(uint32_t x) { return __byte_perm(x, 0, 0x3232); }

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// ---- queries: BF16 -> f16 under a per-(row, head) power-of-two scale -------
//
// BF16 spans 2^-133 .. 2^128, f16 only 2^-24 .. 65504. A query head (128
// elements) is therefore multiplied by 2^-e before its conversion, with e
// chosen from the head's largest magnitude so that it lands in [2^15, 2^16):
// every element within 2^-29 of the largest converts exactly (an f16 normal
// holds BF16's 8 significant bits), smaller ones round as f16 subnormals or
// vanish (below 2^-40 of the largest). The readers undo the scale exactly in
// fp32: d_true = 2^e * d_scaled (ReLU and softmax logits commute with it).

// The largest magnitude of a BF16 pair, as 15-bit magnitude bits (which order
// like the values).
__device__ __forceinline__ uint32_t bf16x2_absmax_bits(uint32_t two) {
  return max(two & 0x7FFFu, (two >> 16) & 0x7FFFu);
}

// A head with no nonzero element has no scale exponent.
constexpr int kQNoExp = -100000;

// Scale exponent e of a head whose largest magnitude has bits m (0 < m <
// 0x7F80): the exponent of m's leading bit, minus 15.
__device__ __forceinline__ int q_scale_exp(uint32_t m) {
  const int E = static_cast<int>(m >> 7);
  const int lead = E > 0 ? E - 127 : (31 - __clz(static_cast<int>(m))) - 133;  // subnormal: mantissa's leading bit
  return lead - 15;
}

// 2^k as fp32 for any k (a subnormal below -126, 0 below -149, +inf above 127).
__device__ __forceinline__ float exp2i_f32(int k) {
  if (k > 127) return __uint_as_float(0x7F800000u);
  if (k >= -126) return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
  return k >= -149 ? __uint_as_float(1u << (k + 149)) : 0.f;
}

// The two factors whose product is 2^-e (each an exact fp32 power of two; the
// second is 1 unless -e > 127).
struct QScale {
  float s1, s2;
};
__device__ __forceinline__ QScale q_scale(int e) {
  const int k = -e, k1 = min(k, 127);
  return QScale{exp2i_f32(k1), exp2i_f32(k - k1)};
}

// BF16 pair (low element in the low half) * 2^-e -> f16x2. The two products are
// exact (powers of two, no overflow: the head's largest element lands below
// 2^16); the conversion is exact for f16 normals.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t two, QScale s) {
  const float a = (__uint_as_float(two << 16) * s.s1) * s.s2;
  const float b = (__uint_as_float(two & 0xFFFF0000u) * s.s1) * s.s2;
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Magnitude bits at or above this are inf or NaN (reported, never scaled).
constexpr uint32_t kBf16InfBits = 0x7F80u;

// f32 -> BF16 bits, round to nearest even (finite inputs; NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u) return static_cast<uint16_t>((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// ---- tensor core ------------------------------------------------------------

// D = A(16x16, row) * B(16x8, col) + C, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- programmatic dependent launch -----------------------------------------

// Let the next kernel in the stream start its prologue now.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the previous kernel in the stream has completed and its writes
// are visible (a no-op when this kernel was launched without the attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- tcgen05: tensor memory and the 5th-generation tensor core -------------

// Allocate `ncols` (power of two >= 32) TMEM columns; the base address is
// written to *dst (shared memory). Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: kind::f16, A and B both f16, f32 accumulate.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// 32 lanes x 16 columns of 32 bits: thread t <-> lane (base lane + t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]),
        "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]),
        "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]),
        "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
      : "r"(taddr)
      : "memory");
}
// After tcgen05.wait::ld: make the loaded registers count as written here, so
// no use of them can be scheduled above the wait (the load's asm already
// "defines" them for the compiler, before the data has landed).
template <int N>
__device__ __forceinline__ void reg_fence(float (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+f"(v[i]));
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, no swizzle: core matrices of 8 rows x 16 B;
// lbo = byte distance between core matrices along K, sbo = along M/N.
__device__ __forceinline__ uint64_t smem_desc_noswizzle(const void* base, uint32_t lbo, uint32_t sbo) {
  const uint64_t addr = smem_addr(base);
  return ((addr >> 4) & 0x3FFFull) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}

// Instruction descriptor for kind::f16: f16 A and B (K-major), f32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Order-preserving map of an fp32 score to uint32 (-0 folded onto +0).
__device__ __forceinline__ uint32_t ordered_bits(float s) {
  uint32_t u = __float_as_uint(s);
  if ((u << 1) == 0) u = 0;  // +-0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k key: the higher score wins, then the LOWER block id.
__device__ __forceinline__ unsigned long long topk_key(float s, int32_t id) {
  return (static_cast<unsigned long long>(ordered_bits(s)) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}

// Inverse of ordered_bits.
__device__ __forceinline__ float from_ordered_bits(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// ---- host: launches -----------------------------------------------------------

// Launch with programmatic stream serialisation (the kernel may start while the
// previous kernel in the stream finishes; it calls pdl_wait() before touching
// any input) and, when cluster_x > 0, thread-block clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

}  // namespace m3s
