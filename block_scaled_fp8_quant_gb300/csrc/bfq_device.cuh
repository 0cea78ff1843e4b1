// bfq_device.cuh — device-side building blocks for the sm_103a kernels:
// fp8 conversion, the FMA-corrected quotient, the fp32 exp used by silu,
// mbarrier waits with a watchdog, TMA loads and tcgen05 (UMMA / TMEM) helpers,
// all as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bfq_internal.h"

namespace bfq {

// ---------------------------------------------------------------------------
// host: TMA tensor maps (defined in gemm_kernels.cu)
// ---------------------------------------------------------------------------
// 2D map over a row-major byte matrix [rows][inner] with a 128 x box_rows box
// and 128-byte swizzling; out-of-range rows read as zero.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
              uint32_t box_rows);
// 2D map over the bf16 output [rows][cols] with a 64 x 128 box and 128-byte
// swizzling, for TMA stores of a staged tile.
bool make_out_map(CUtensorMap* map, void* base, uint64_t cols, uint64_t rows);

// Kernels whose bounded waits give up latch BFQ_ERR_TIMEOUT into the
// library's device status word (its address is a kernel argument, see
// device_status_ptr()); bfq_poll_device_status() reads and clears it.
__device__ __forceinline__ void record_timeout(int* status) {
  atomicExch(status, BFQ_ERR_TIMEOUT);
}

// Debug builds (compiled with BFQ_DEVICE_CHECKS): every global access whose
// offset the kernel computes checks it against the extent of its array, as
// the host derived it from the call's arguments; a failing check latches
// BFQ_ERR_DEVICE_BOUNDS in the status word (never overwriting an earlier
// error) and the access is skipped.  Release builds compile the checks away.
#ifdef BFQ_DEVICE_CHECKS
__device__ __forceinline__ bool in_bounds(int* status, int64_t off, int64_t len,
                                          int64_t extent) {
  if (off >= 0 && off + len <= extent) return true;
  atomicCAS(status, 0, BFQ_ERR_DEVICE_BOUNDS);
  return false;
}
#else
__device__ __forceinline__ bool in_bounds(int*, int64_t, int64_t, int64_t) { return true; }
#endif

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// numeric helpers
// ---------------------------------------------------------------------------
constexpr float kFp8Max = 448.0f;
constexpr float kEps = 1e-10f;

// Smallest power of two >= s for a positive normal float: bump the exponent
// when any mantissa bit is set (UE8M0 "ceil to a power of two").
__device__ __forceinline__ float ceil_pow2(float s) {
  uint32_t b = __float_as_uint(s);
  if (b & 0x007FFFFFu) b = (b & 0x7F800000u) + 0x00800000u;
  return __uint_as_float(b);
}

// Biased exponent byte of a positive power of two.
__device__ __forceinline__ uint32_t ue8m0_byte(float p) { return __float_as_uint(p) >> 23; }

// Two fp32 values -> two e4m3 codes, round-to-nearest-even, saturating to
// +-448.  Returns lo in byte 0 and hi in byte 1.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// Quotient a / s for a whole group sharing the divisor s, with y = RN(1/s):
// one correction step by fused multiply-add (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990).  The result equals the IEEE quotient whenever neither
// the residual nor the quotient underflows; otherwise both are below 2^-11
// and round to the same signed zero in e4m3.  The sign is taken from a so
// that a zero numerator keeps its sign as in the IEEE quotient.
__device__ __forceinline__ float group_div(float a, float s, float y) {
  float q0 = __fmul_rn(a, y);
  float r = __fmaf_rn(-q0, s, a);
  return copysignf(__fmaf_rn(r, y, q0), a);
}

// fp32 exp by Cody-Waite range reduction and a degree-7 Taylor polynomial:
//   n = rint(x * log2 e),  r = (x - n * ln2_hi) - n * ln2_lo,
//   exp(r) ~ sum_{k<=7} r^k / k!  (Horner with fused multiply-adds),
//   exp(x) = exp(r) * 2^n, the power applied as two exact factors.
// ln2_hi = 0x1.62e4p-1 has 15 significant bits; ln2_lo = fl32(ln2 - ln2_hi).
// x < -88 -> 0, x > 89 -> +inf.  Every step is an explicitly rounded fp32
// operation so the result does not depend on compiler contraction.
__device__ __forceinline__ float pow2_int(int k) {  // -126 <= k <= 127
  return __uint_as_float((uint32_t)(k + 127) << 23);
}

__device__ __forceinline__ float bfq_expf(float x) {
  if (isnan(x)) return x;
  if (x < -88.0f) return 0.0f;
  if (x > 89.0f) return __int_as_float(0x7F800000);
  const float log2e = 0x1.715476p+0f;
  const float ln2_hi = 0x1.62e4p-1f;
  const float ln2_lo = 0x1.7f7d1cp-20f;
  float n = rintf(__fmul_rn(x, log2e));
  float r = __fmaf_rn(-n, ln2_hi, x);
  r = __fmaf_rn(-n, ln2_lo, r);
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, r, 0x1.111112p-7f);
  p = __fmaf_rn(p, r, 0x1.555556p-5f);
  p = __fmaf_rn(p, r, 0x1.555556p-3f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  int k = (int)n;
  int k1 = k / 2;
  int k2 = k - k1;
  return __fmul_rn(__fmul_rn(p, pow2_int(k1)), pow2_int(k2));
}

__device__ __forceinline__ float bfq_silu(float g) {
  return __fdiv_rn(g, __fadd_rn(1.0f, bfq_expf(-g)));
}

// Bring the 128-byte line holding p into L2 (no register result, no wait).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// 16-byte streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// Wait until the grids this one depends on (the previous kernel in the
// stream, when launched with programmatic serialization) have completed and
// their memory is visible; a no-op otherwise.  Every kernel calls it before
// its first global-memory access.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next kernel in the stream to start launching (it still waits in
// griddep_wait() for this grid to finish before touching memory).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// shared memory / mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// timeout_ns (globaltimer) or as soon as *abort is set by another role of the
// CTA; on giving up it latches BFQ_ERR_TIMEOUT in *status, sets *abort and
// returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort, int* status,
                                          uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      record_timeout(status);
      *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) — 2D tiled load into shared memory, completing
// on an mbarrier with a transaction count.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 1D bulk copy of `bytes` (a multiple of 16) from global to shared memory,
// both addresses 16-byte aligned, completing on an mbarrier with a
// transaction count.
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2D tiled store from shared memory (bulk-group completion).  Elements of the
// box outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x,
                                             int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          map),
      "r"(smem_u32(src)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_and_wait_all() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group 0;" ::: "memory");
}

// Close the current bulk async-group (TMA stores issued so far).
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store has finished reading its shared
// memory source (the global writes may still be in flight).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA) before a barrier.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, UMMA issue/commit, TMEM loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row (1024-byte) swizzle atoms
// stacked along M/N (stride byte offset 1024), descriptor version 1, layout
// type SWIZZLE_128B.  The tile base must be 1024-byte aligned.
__host__ __device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address      [0,14)
  d |= (uint64_t)1 << 16;                     // leading byte offset (unused) [16,30)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset [32,46)
  d |= (uint64_t)1 << 46;                     // version            [46,48)
  d |= (uint64_t)2 << 61;                     // SWIZZLE_128B       [61,64)
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4: A and B e4m3, fp32
// accumulator, both operands K-major, M x N tile.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (0u << 7)                    // A format: e4m3
         | (0u << 10)                   // B format: e4m3
         | ((uint32_t)(N >> 3) << 17)   // N >> 3
         | ((uint32_t)(M >> 4) << 24);  // M >> 4
}

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4.block_scale: A and B
// e4m3, both K-major, M x N tile, fp32 accumulator, UE8M0 scale factors;
// sf_byte (0..3) selects which byte of A's and of B's 32-bit scale words in
// TMEM this MMA applies (scale_vec::1X: one scale per row for its K = 32).
__host__ __device__ constexpr uint32_t idesc_e4m3_bs(int M, int N, uint32_t sf_byte) {
  return (sf_byte << 4)                 // B scale-factor byte    [4,6)
         | (0u << 7)                    // A format: e4m3         [7,10)
         | (0u << 10)                   // B format: e4m3         [10,13)
         | ((uint32_t)(N >> 3) << 17)   // N >> 3                 [17,23)
         | (1u << 23)                   // scale factors UE8M0    [23]
         | ((uint32_t)(M >> 4) << 24)   // M >> 4                 [24,29)
         | (sf_byte << 29);             // A scale-factor byte    [29,31)
}

// D[tmem] (+)= (A[smem] * 2^(sA - 127)) * (B[smem] * 2^(sB - 127))^T for one
// K = 32 step, sA / sB the UE8M0 scale of each row of A / B: the selected
// byte of the 32-bit words at TMEM columns sfa.. / sfb.. (M = 128 rows of A:
// row 32 c + r at lane r of column sfa + c; N rows of B likewise from sfb),
// issued by a single thread.
__device__ __forceinline__ void umma_e4m3_bs(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor of a tcgen05.cp source of 16-byte rows: row r at
// byte 16 r, i.e. 8-row (128-byte) core matrices stacked contiguously
// (stride byte offset 128), one core matrix along K (leading byte offset
// unused), no swizzle, descriptor version 1.  16-byte aligned base.
__host__ __device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address      [0,14)
  d |= (uint64_t)(128 >> 4) << 32;            // stride byte offset [32,46)
  d |= (uint64_t)1 << 46;                     // version            [46,48)
  return d;                                   // layout type 0: no swizzle
}

// Copy 32 rows x 128 bits from shared memory (descriptor above) into 4
// consecutive TMEM columns of lanes 0-31, replicated into each of the four
// 32-lane quarters (lane 32 q + r, column c = bytes 16 r + 4 c .. + 3 of the
// source).  Asynchronous; ordered before later tcgen05.mma of this thread.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by a single thread.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on *bar when all tcgen05 operations issued so far by this
// thread have completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 64 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per
// thread) as 32 register pairs (column 2i in the low half of p[i]).  Load and
// wait are one asm statement, so no use of the registers can be scheduled
// before the data is valid.
__device__ __forceinline__ void tmem_ld64_pairs_wait(uint32_t taddr, uint64_t (&p)[32]) {
  asm volatile(
      "{\n\t.reg .b32 t<64>;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15,t16,t17,t18,t19,t20,t21,t22,t23,t24,t25,t26,t27,t28,t29,t30,t31,t32,t33,t34,t35,t36,t37,t38,t39,t40,t41,t42,t43,t44,t45,t46,t47,t48,t49,t50,t51,t52,t53,t54,t55,t56,t57,t58,t59,t60,t61,t62,t63}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "mov.b64 %0, {t0,t1};\n\t"
      "mov.b64 %1, {t2,t3};\n\t"
      "mov.b64 %2, {t4,t5};\n\t"
      "mov.b64 %3, {t6,t7};\n\t"
      "mov.b64 %4, {t8,t9};\n\t"
      "mov.b64 %5, {t10,t11};\n\t"
      "mov.b64 %6, {t12,t13};\n\t"
      "mov.b64 %7, {t14,t15};\n\t"
      "mov.b64 %8, {t16,t17};\n\t"
      "mov.b64 %9, {t18,t19};\n\t"
      "mov.b64 %10, {t20,t21};\n\t"
      "mov.b64 %11, {t22,t23};\n\t"
      "mov.b64 %12, {t24,t25};\n\t"
      "mov.b64 %13, {t26,t27};\n\t"
      "mov.b64 %14, {t28,t29};\n\t"
      "mov.b64 %15, {t30,t31};\n\t"
      "mov.b64 %16, {t32,t33};\n\t"
      "mov.b64 %17, {t34,t35};\n\t"
      "mov.b64 %18, {t36,t37};\n\t"
      "mov.b64 %19, {t38,t39};\n\t"
      "mov.b64 %20, {t40,t41};\n\t"
      "mov.b64 %21, {t42,t43};\n\t"
      "mov.b64 %22, {t44,t45};\n\t"
      "mov.b64 %23, {t46,t47};\n\t"
      "mov.b64 %24, {t48,t49};\n\t"
      "mov.b64 %25, {t50,t51};\n\t"
      "mov.b64 %26, {t52,t53};\n\t"
      "mov.b64 %27, {t54,t55};\n\t"
      "mov.b64 %28, {t56,t57};\n\t"
      "mov.b64 %29, {t58,t59};\n\t"
      "mov.b64 %30, {t60,t61};\n\t"
      "mov.b64 %31, {t62,t63};\n\t"
      "}\n"
      : "=l"(p[0]), "=l"(p[1]), "=l"(p[2]), "=l"(p[3]), "=l"(p[4]), "=l"(p[5]), "=l"(p[6]), "=l"(p[7]), "=l"(p[8]), "=l"(p[9]), "=l"(p[10]), "=l"(p[11]), "=l"(p[12]), "=l"(p[13]), "=l"(p[14]), "=l"(p[15]), "=l"(p[16]), "=l"(p[17]), "=l"(p[18]), "=l"(p[19]), "=l"(p[20]), "=l"(p[21]), "=l"(p[22]), "=l"(p[23]), "=l"(p[24]), "=l"(p[25]), "=l"(p[26]), "=l"(p[27]), "=l"(p[28]), "=l"(p[29]), "=l"(p[30]), "=l"(p[31])
      : "r"(taddr)
      : "memory");
}

// Cluster-wide barrier (all threads of all CTAs of the cluster), with
// release/acquire ordering of the memory operations around it.
// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

// 16-byte load from a cluster shared-memory address (distributed shared memory).
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// 16-byte shared-memory load.
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// acc = v * s + acc on a pair of fp32 lanes (packed f32x2 fused multiply-add).
__device__ __forceinline__ void ffma2(uint64_t& acc, uint64_t v, uint64_t s2) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(v), "l"(s2));
}

__device__ __forceinline__ uint64_t splat2(float s) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(s));
  return r;
}

__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
  return f;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// Packed f32x2 arithmetic: each lane of the pair is rounded exactly as the
// scalar fp32 operation (round to nearest even, subnormals kept).
__device__ __forceinline__ uint64_t fma2_rn(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2_rn(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2_rn(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// bfq_silu on two values at once: the same fp32 operations as bfq_expf and
// bfq_silu in the same order (so bit-identical results), with the
// multiplies and FMAs of the range reduction, the polynomial and the
// scaling issued as f32x2 pairs, and the range cases of bfq_expf applied by
// selection afterwards.
__device__ __forceinline__ float exp_range_fix(float x, float v) {
  return isnan(x) ? x : (x < -88.0f ? 0.0f : (x > 89.0f ? __int_as_float(0x7F800000) : v));
}

__device__ __forceinline__ float2 bfq_silu2(float g0, float g1) {
  const float x0 = -g0, x1 = -g1;
  const uint64_t x = pack2(x0, x1);
  const float2 t = unpack2(mul2_rn(x, splat2(0x1.715476p+0f)));
  const float n0 = rintf(t.x), n1 = rintf(t.y);
  const uint64_t n = pack2(n0, n1);
  // fma(-n, c, x) == fma(n, -c, x) exactly
  uint64_t r = fma2_rn(n, splat2(-0x1.62e4p-1f), x);
  r = fma2_rn(n, splat2(-0x1.7f7d1cp-20f), r);
  uint64_t p = splat2(0x1.a01a02p-13f);
  p = fma2_rn(p, r, splat2(0x1.6c16c2p-10f));
  p = fma2_rn(p, r, splat2(0x1.111112p-7f));
  p = fma2_rn(p, r, splat2(0x1.555556p-5f));
  p = fma2_rn(p, r, splat2(0x1.555556p-3f));
  p = fma2_rn(p, r, splat2(0.5f));
  p = fma2_rn(p, r, splat2(1.0f));
  p = fma2_rn(p, r, splat2(1.0f));
  const int k0 = (int)n0, k1 = (int)n1;
  const int h0 = k0 / 2, h1 = k1 / 2;
  const float2 e = unpack2(mul2_rn(mul2_rn(p, pack2(pow2_int(h0), pow2_int(h1))),
                                   pack2(pow2_int(k0 - h0), pow2_int(k1 - h1))));
  const float2 d =
      unpack2(add2_rn(pack2(exp_range_fix(x0, e.x), exp_range_fix(x1, e.y)), splat2(1.0f)));
  return make_float2(__fdiv_rn(g0, d.x), __fdiv_rn(g1, d.y));
}

// 4-byte asynchronous global -> shared copy (no register round trip).
__device__ __forceinline__ void cp_async_4(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)), "l"(src)
               : "memory");
}

// Arrive on *bar once every cp.async this thread issued so far has landed;
// the arrival counts against the barrier's expected count (.noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Register reconfiguration of a whole warpgroup (all 128 threads execute it).
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N) : "memory");
}

// Named barrier over `count` threads (a multiple of 32), id 1..15, that
// returns in every participating thread whether any of them passed true.
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Named barrier over `count` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace bfq
