// gemm_kernels.cu — block-scaled FP8 GEMM on sm_103a tensor cores.
//
//   out[m, n] = sum_b sA[m, b] * sW[n / 128, b] * sum_{k in block b} a[m, k] w[n, k]
//
// ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.2: fp8_gemm_nt and the Triton
// loop that multiplies each K-block product by a_s * b_s; "[Kernel]
// Integrate batched/masked deepgemm kernel": the masked per-expert form.)
//
// Design (one CTA per output tile and K split, one CTA per SM):
//   warp 0      TMA producer: per 128-deep K block, one 128 x 128 A tile and
//               one BN x 128 W tile (128-byte swizzle) into a smem ring.
//   warp 1      allocates TMEM; lane 0 issues 4 tcgen05.mma (K = 32 each,
//               kind::f8f6f4, e4m3 x e4m3 -> fp32) per K block into one of two
//               TMEM partial-sum buffers, then commits to the ring's "empty"
//               barrier and to the buffer's "full" barrier.
//   warps 2..   epilogue ("promotion"): per K block, read the fp32 partial of
//               its 32 rows x 128 columns from TMEM, multiply by the scale
//               product sA[m, b] * sW[nblk, b] and accumulate in registers.
//               At the end convert to bf16 and store the tile through shared
//               memory, or (K split over a thread-block cluster) keep the
//               fp32 partial in the CTA's shared memory; every CTA of the
//               cluster then sums its slice of the tile over the splits, read
//               through distributed shared memory in split order
//               (deterministic), and stores bf16.
// The persistent form (one CTA per SM walking many tiles) and the masked
// per-expert forms are described at their kernel.
// Every wait is bounded: a wait that gives up latches BFQ_ERR_TIMEOUT in the
// library's status word, every role drains and the CTA frees its TMEM and
// exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "bfq_device.cuh"
#include "gemm_common.cuh"

namespace bfq {


// BN = 256: three warpgroups.  Warpgroup 0 (warps 0-3) holds the TMA
// producer (warp 0) and the MMA issuer (warp 1) and gives registers away
// (setmaxnreg 24); warpgroups 1-2 (warps 4-11) are the eight epilogue warps
// (setmaxnreg 240).  128*24 + 256*240 = 64512 = 384 threads * 168 registers,
// the allocation the kernel is launched with (checked on the host).
// Warp 2 streams the scales into shared memory.  BN = 128: seven warps, two
// per sub-partition at most, no reconfiguration.
template <int BN>
struct GemmCfg {
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr int kEpiWarps = BN / 32;  // 128 columns per warp
  static constexpr int kEpiWarp0 = (BN == 256) ? 4 : 3;
  static constexpr int kScaleWarp = 2;       // streams the scales into smem
  static constexpr int kScaleSlots = 8;      // K blocks of scales in flight
  static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
  static constexpr bool kRegSplit = (BN == 256);
  static constexpr int kLaunchRegs = 168;
  static constexpr int kProducerRegs = 24;
  static constexpr int kEpilogueRegs = 240;
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;
  // scale ring: [slot][128] activation scales (raw bits) + [slot][2] weight scales
  static constexpr int kScaleBytes = kScaleSlots * (kBM + 2) * 4;
  static constexpr int kBarrierBytes = 512;
  static constexpr size_t kSmemBytes =
      (size_t)kStages * kStageBytes + kScaleBytes + kBarrierBytes + 1024;
};



// Fused output quant of one row's 128 accumulated columns, which form exactly
// one 1 x 128 group (the tile's column halves start at multiples of 128): the
// values are rounded to bf16 as the output is stored, then quantized as the
// per-token-group quant kernel quantizes a bf16 input — group amax, scale
// fl32(max(amax, eps) / 448) (power of two for the pow2 and UE8M0 formats),
// correctly rounded quotient, saturating e4m3 — so the codes and scales are
// those of quantizing the stored bf16 output ("[Perf] Deepgemm fused layout
// kernel for activations": no separate quant or layout pass).
//   row m, columns col0 .. col0 + 127 of q_out; group = col0 / 128; the
//   row's last group zeroes the bytes a partial packed word leaves unused.
__device__ __forceinline__ void quant_store_row_group(const uint64_t (&acc)[64],
                                                      const GemmParams& p, int m, int col0) {
  const int fmt = p.q_fmt, group = col0 >> 7;
  const bool last = col0 + 128 >= p.N;
  const int64_t ld = p.q_scale_ld;
  const int64_t qoff = (int64_t)m * p.N + col0;
  uint8_t* q_row = p.q_out + qoff;
  const bool q_ok = in_bounds(p.status, qoff, 128, p.n_q);
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const float2 f = unpack2(acc[j]);
    const uint32_t b = pack_bf16x2(f.x, f.y);
    amax = fmaxf(amax, fmaxf(fabsf(bf16lo(b)), fabsf(bf16hi(b))));
  }
  float s = __fdiv_rn(fmaxf(amax, kEps), kFp8Max);
  if (fmt != BFQ_SCALE_F32) s = ceil_pow2(s);
  const float y = __frcp_rn(s);  // exact for a power of two
#pragma unroll
  for (int c = 0; c < 8; ++c) {  // 16 codes per 16-byte store
    uint32_t w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 f0 = unpack2(acc[c * 8 + 2 * t]), f1 = unpack2(acc[c * 8 + 2 * t + 1]);
      const uint32_t b0 = pack_bf16x2(f0.x, f0.y), b1 = pack_bf16x2(f1.x, f1.y);
      const float v0 = bf16lo(b0), v1 = bf16hi(b0), v2 = bf16lo(b1), v3 = bf16hi(b1);
      uint32_t lo, hi;
      if (fmt == BFQ_SCALE_F32) {
        lo = cvt_e4m3x2(group_div(v0, s, y), group_div(v1, s, y));
        hi = cvt_e4m3x2(group_div(v2, s, y), group_div(v3, s, y));
      } else {
        lo = cvt_e4m3x2(__fmul_rn(v0, y), __fmul_rn(v1, y));
        hi = cvt_e4m3x2(__fmul_rn(v2, y), __fmul_rn(v3, y));
      }
      w[t] = lo | (hi << 16);
    }
    if (q_ok) st_v4(q_row + c * 16, make_uint4(w[0], w[1], w[2], w[3]));
  }
  if (fmt == BFQ_SCALE_UE8M0_PACKED) {
    const int64_t woff = (int64_t)(group >> 2) * ld + m;
    if (!in_bounds(p.status, woff, 1, p.n_qs)) return;
    uint8_t* word = (uint8_t*)p.q_scales + woff * 4;
    word[group & 3] = (uint8_t)ue8m0_byte(s);
    if (last)
      for (int b = (group & 3) + 1; b < 4; ++b) word[b] = 0;
  } else {
    const int64_t soff = (int64_t)group * ld + m;
    if (in_bounds(p.status, soff, 1, p.n_qs)) ((float*)p.q_scales)[soff] = s;
  }
}

template <int BN, bool MASKED, bool QOUT = false>
__global__ void __launch_bounds__(GemmCfg<BN>::kThreads, 1)
    gemm_block_fp8_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmW,
                          const __grid_constant__ CUtensorMap tmO, const GemmParams p) {
  using C = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::kStages * C::kABytes;
  uint32_t* sc_a = (uint32_t*)(smem + (size_t)C::kStages * C::kStageBytes);  // [slot][128]
  uint32_t* sc_w = sc_a + C::kScaleSlots * kBM;                                 // [slot][2]
  uint64_t* full = (uint64_t*)(smem + (size_t)C::kStages * C::kStageBytes + C::kScaleBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* sfull = tempty + 2;
  uint64_t* sempty = sfull + C::kScaleSlots;
  uint64_t* drain = sempty + C::kScaleSlots;
  uint32_t* tmem_slot = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  // ---- tile decode: split fastest, then m tile, then n tile, then expert ----
  const int split = blockIdx.x % p.splits;
  const int tile = blockIdx.x / p.splits;
  const int mt = tile % p.m_tiles;
  const int rest = tile / p.m_tiles;
  const int nt = rest % p.n_tiles;
  const int e = MASKED ? rest / p.n_tiles : 0;
  const int m0 = mt * kBM, n0 = nt * BN;
  int m_limit = p.M;
  if (MASKED) {
    griddep_wait();  // the counts may come from the previous kernel
    int c = __ldg(p.counts + e);
    m_limit = c < 0 ? 0 : (c > p.M ? p.M : c);
    if (m0 >= m_limit) return;  // whole tile is padding: no loads, no MMA
  }
  const int KB = p.K / kBK;
  const int kb_begin = (int)((int64_t)split * KB / p.splits);
  const int kb_end = (int)((int64_t)(split + 1) * KB / p.splits);
  const int nk = kb_end - kb_begin;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], C::kEpiWarps);
    }
    for (int b = 0; b < C::kScaleSlots; ++b) {
      mbar_init(&sfull[b], 32);
      mbar_init(&sempty[b], C::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // The set-up above overlaps the previous kernel's tail; nothing below may
  // touch global memory before that kernel has finished.
  if (!MASKED) griddep_wait();
  griddep_launch_dependents();
  static_assert(!C::kRegSplit || 128 * C::kProducerRegs +
                                         (C::kThreads - 128) * C::kEpilogueRegs <=
                                     C::kThreads * C::kLaunchRegs,
                "register split exceeds the launch allocation");

  if (warp < C::kEpiWarp0) {
    if (C::kRegSplit) setmaxnreg_dec<C::kProducerRegs>();
    if (warp == 0) {
      // ------------------------------ TMA producer ------------------------------
      if (lane == 0) {
        const int a_row = (MASKED ? e * p.M : 0) + m0;
        const int w_row = (MASKED ? e * p.N : 0) + n0;
        int issued = 0;
        for (int i = 0; i < nk; ++i) {
          const int s = i % C::kStages;
          const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status, kWaitTimeoutNs)) break;
          mbar_arrive_expect_tx(&full[s], (uint32_t)C::kStageBytes);
          const int kx = (kb_begin + i) * kBK;
          tma_load_2d(sA + (size_t)s * C::kABytes, &tmA, &full[s], kx, a_row);
          tma_load_2d(sB + (size_t)s * C::kBBytes, &tmW, &full[s], kx, w_row);
          ++issued;
        }
        if (*abort_flag) {
          // let the copies already issued land before the CTA can exit
          for (int j = issued - C::kStages < 0 ? 0 : issued - C::kStages; j < issued; ++j) {
            volatile int no_abort = 0;
            (void)mbar_wait(&full[j % C::kStages], (uint32_t)(j / C::kStages) & 1u, &no_abort,
                            p.status, kWaitTimeoutNs / 8);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------- MMA issuer -------------------------------
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
        bool issued_any = false;
        for (int i = 0; i < nk; ++i) {
          const int s = i % C::kStages;
          const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
          const int buf = i & 1;
          const uint32_t tph = (uint32_t)(i >> 1) & 1u;
          if (!mbar_wait(&tempty[buf], tph ^ 1u, abort_flag, p.status, kWaitTimeoutNs)) break;
          tc_fence_after_sync();
          if (!mbar_wait(&full[s], ph, abort_flag, p.status, kWaitTimeoutNs)) break;
          tc_fence_after_sync();
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + (size_t)s * C::kABytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + (size_t)s * C::kBBytes));
          const uint32_t d = tmem_base + (uint32_t)(buf * BN);
  #pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            umma_e4m3(d, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                      kk > 0 ? 1u : 0u);
          umma_commit(&empty[s]);
          umma_commit(&tfull[buf]);
          issued_any = true;
        }
        if (*abort_flag && issued_any) {
          // wait for the MMAs already issued before TMEM is released
          umma_commit(drain);
          volatile int no_abort = 0;
          (void)mbar_wait(drain, 0, &no_abort, p.status, kWaitTimeoutNs / 8);
        }
      }
    } else if (warp == C::kScaleWarp) {
      // ------------------------------ scale loader ------------------------------
      // Per K block: raw bits of sA for the tile's 128 rows (fp32 bits, or the
      // packed word that holds this block's exponent) and sW for its 1-2 weight
      // row-blocks, copied asynchronously into a ring slot.  Rows past the valid
      // range are not copied (their outputs are never stored).
      const int KBs = KB;
      const int nb0 = n0 / 128;
      const int nblks = (int)((p.N + 127) / 128);
      const void* sa = MASKED ? (const void*)((const char*)p.sa + (int64_t)e * p.sa_estride * 4)
                              : p.sa;
      const float* sw = p.sw + (MASKED ? (int64_t)e * p.sw_estride : 0);
      const bool packed = p.a_fmt == BFQ_SCALE_UE8M0_PACKED;
      for (int i = 0; i < nk; ++i) {
        const int slot = i % C::kScaleSlots;
        const uint32_t ph = (uint32_t)(i / C::kScaleSlots) & 1u;
        if (!mbar_wait(&sempty[slot], ph ^ 1u, abort_flag, p.status, kWaitTimeoutNs)) break;
        const int kb = kb_begin + i;
        const int64_t col_off = (MASKED ? (int64_t)e * p.sa_estride : 0) +
                                (int64_t)(packed ? (kb >> 2) : kb) * p.sa_ld + m0;
        const int64_t w_off = (MASKED ? (int64_t)e * p.sw_estride : 0) +
                              (int64_t)(nb0 + lane) * KBs + kb;
        const uint32_t* col = (const uint32_t*)sa + (int64_t)(packed ? (kb >> 2) : kb) * p.sa_ld;
  #pragma unroll
        for (int r = lane; r < kBM; r += 32)
          if (m0 + r < m_limit && in_bounds(p.status, col_off + r, 1, p.n_sa))
            cp_async_4(&sc_a[slot * kBM + r], col + m0 + r);
        if (lane < BN / 128 && nb0 + lane < nblks && in_bounds(p.status, w_off, 1, p.n_sw))
          cp_async_4(&sc_w[slot * 2 + lane], sw + (int64_t)(nb0 + lane) * KBs + kb);
        cp_async_arrive_noinc(&sfull[slot]);
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
    __syncwarp();
    if (p.splits > 1) {  // pair with the epilogue's two cluster barriers
      cluster_sync();
      cluster_sync();
    }
  } else {
    if (C::kRegSplit) setmaxnreg_inc<C::kEpilogueRegs>();
    // ------------------------- epilogue / promotion ---------------------------
    const int ew = warp - C::kEpiWarp0;
    const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
    const int half = (BN == 256) ? (ew >> 2) : 0;
    const int row_local = quarter * 32 + lane;
    const int m = m0 + row_local;
    const bool row_ok = m < m_limit;
    const int col0 = n0 + half * 128;
    const bool warp_active = (m0 + quarter * 32 < m_limit) && (col0 < p.N);
    const int ncols = min(128, p.N - col0);  // multiple of 64 when positive

    uint64_t acc[64];  // 128 fp32 accumulators as pairs (column 2i low)
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0ull;

    for (int i = 0; i < nk; ++i) {
      const int buf = i & 1;
      const uint32_t tph = (uint32_t)(i >> 1) & 1u;
      const int slot = i % C::kScaleSlots;
      const uint32_t sph = (uint32_t)(i / C::kScaleSlots) & 1u;
      if (!mbar_wait(&sfull[slot], sph, abort_flag, p.status, kWaitTimeoutNs)) break;
      const uint32_t a_bits = sc_a[slot * kBM + row_local];
      const float w_s = __uint_as_float(sc_w[slot * 2 + half]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[slot]);
      float sa_v;
      if (p.a_fmt == BFQ_SCALE_UE8M0_PACKED) {
        const uint32_t b = (a_bits >> (8 * ((kb_begin + i) & 3))) & 0xFFu;
        sa_v = b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);  // 2^(b-127)
      } else {
        sa_v = __uint_as_float(a_bits);
      }
      const uint64_t s2 = splat2(__fmul_rn(row_ok ? sa_v : 0.0f, w_s));
      if (!mbar_wait(&tfull[buf], tph, abort_flag, p.status, kWaitTimeoutNs)) break;
      tc_fence_after_sync();
      if (warp_active) {
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                               (uint32_t)(buf * BN + half * 128);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint64_t v[32];
          tmem_ld64_pairs_wait(taddr + (uint32_t)(h * 64), v);
#pragma unroll
          for (int t = 0; t < 32; ++t) ffma2(acc[h * 32 + t], v[t], s2);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }

    const bool ok = !*abort_flag;
    const int64_t out_row = (MASKED ? (int64_t)e * p.out_estride : 0) + (int64_t)m * p.N;
    if (p.splits == 1 && !MASKED) {
      // (fused output quant: the bf16 output is optional)
      if (!QOUT || p.out != nullptr) {
        // Dense tile: stage the bf16 tile in the (now idle) A stages as
        // [BN/64] boxes of 128 rows x 64 columns in the 128-byte swizzled layout
        // (16-byte chunk c of row r at chunk c ^ (r mod 8): conflict-free), then
        // one thread writes them with TMA stores, which clip rows >= M.
        if (ok && warp_active) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int blk = half * 2 + j;
            if (j * 64 >= ncols) break;  // this 64-column block lies beyond N
            const uint32_t row_addr =
                smem_u32(smem) + (uint32_t)(blk * (kBM * 128) + row_local * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int a = j * 32 + c * 4;  // pair index of column j*64 + c*8
              const float2 f0 = unpack2(acc[a + 0]), f1 = unpack2(acc[a + 1]);
              const float2 f2 = unpack2(acc[a + 2]), f3 = unpack2(acc[a + 3]);
              st_shared_v4(row_addr + (uint32_t)((c ^ (row_local & 7)) << 4),
                           make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f1.x, f1.y),
                                      pack_bf16x2(f2.x, f2.y), pack_bf16x2(f3.x, f3.y)));
            }
          }
        }
        fence_proxy_async_smem();
        named_barrier(1, C::kEpiWarps * 32);
        if (threadIdx.x == C::kEpiWarp0 * 32 && !*abort_flag) {
          for (int blk = 0; blk < BN / 64; ++blk)
            if (n0 + blk * 64 < p.N)
              tma_store_2d(&tmO, smem + blk * (kBM * 128), n0 + blk * 64, m0);
          bulk_commit_and_wait_all();
        }
      }
      if constexpr (QOUT) {
        if (ok && warp_active && row_ok)
          quant_store_row_group(acc, p, m, col0);
      }
    } else if (p.splits == 1) {
      if (ok && warp_active && row_ok) {
        __nv_bfloat16* dst = p.out + out_row + col0;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (c * 8 < ncols) {
            const float2 f0 = unpack2(acc[c * 4 + 0]), f1 = unpack2(acc[c * 4 + 1]);
            const float2 f2 = unpack2(acc[c * 4 + 2]), f3 = unpack2(acc[c * 4 + 3]);
            if (in_bounds(p.status, out_row + col0 + c * 8, 8, p.n_out))
              st_v4(dst + c * 8, make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f1.x, f1.y),
                                            pack_bf16x2(f2.x, f2.y), pack_bf16x2(f3.x, f3.y)));
          }
        }
      }
    } else {
      // split-K: publish this split's fp32 partial; the cluster reduces below.
      // split-K: this split's fp32 partial stays in the CTA's own shared
      // memory, in the (now idle) stage ring: every load has landed and every
      // MMA that read a stage has completed.  Row r of the tile holds BN
      // floats; 16-byte chunk j sits at chunk j ^ (r mod 8) (conflict-free
      // both for the row-per-thread writes here and the chunk-per-thread
      // reads below).  The K splits of one tile are one thread-block cluster:
      // after one cluster barrier, CTA `split` sums the split-th slice of the
      // tile over the splits' partials, read from the peers' shared memory in
      // split order (deterministic); a second barrier keeps every partial in
      // place until all peers have read it.
      static_assert(kBM * BN * 4 <= C::kStages * C::kStageBytes, "partial exceeds the stages");
      const uint32_t part_base = smem_u32(smem);
      auto part_addr = [&](int r, int j) {
        return part_base + (uint32_t)(r * BN * 4) + (uint32_t)((j ^ (r & 7)) << 4);
      };
      if (ok && warp_active && row_ok) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c * 4 < ncols)
            st_shared_v4(part_addr(row_local, half * 32 + c),
                         make_uint4((uint32_t)acc[c * 2], (uint32_t)(acc[c * 2] >> 32),
                                    (uint32_t)acc[c * 2 + 1], (uint32_t)(acc[c * 2 + 1] >> 32)));
      }
      cluster_sync();
      // Fused quant: the partials of a warp's next unit are loaded before the
      // current unit is summed and stored (its byte stores may alias the loads
      // for the compiler), so each warp keeps a unit's loads in flight.
      auto load_parts = [&](int r, int j, float4 (&v)[kMaxSplits]) {
        const uint32_t a = part_addr(r, j);
#pragma unroll
        for (int t = 0; t < kMaxSplits; ++t)
          if (t < p.splits) v[t] = ld_dsmem_v4(dsmem_addr(a, (uint32_t)t));
      };
      auto sum_parts = [&](const float4 (&v)[kMaxSplits]) {  // in split order
        float4 a4 = v[0];
#pragma unroll
        for (int t = 1; t < kMaxSplits; ++t)
          if (t < p.splits) {
            a4.x += v[t].x; a4.y += v[t].y; a4.z += v[t].z; a4.w += v[t].w;
          }
        return a4;
      };
      if (QOUT && !*abort_flag) {
        // Fused output quant: the reduction is shared out in whole 128-column
        // groups, one warp per (row, group) — 32 lanes x 4 columns — so each
        // group's amax is one warp reduction.  The sums are formed in split
        // order exactly as below, so the bf16 output is the same.
        const int rows = min(kBM, m_limit - m0);
        const int gpr = min(BN, p.N - n0) / 128;  // output groups per row
        const int total = rows * gpr;
        const int u_begin = (int)((int64_t)split * total / p.splits);
        const int u_end = (int)((int64_t)(split + 1) * total / p.splits);
        auto load_unit = [&](int u, float4 (&v)[kMaxSplits]) {
          const int r = u / gpr;
          load_parts(r, (u - r * gpr) * 32 + lane, v);
        };
        float4 vn[kMaxSplits];
        int u = u_begin + (warp - C::kEpiWarp0);
        if (u < u_end) load_unit(u, vn);
        for (; u < u_end; u += C::kEpiWarps) {
          float4 v[kMaxSplits];
#pragma unroll
          for (int t = 0; t < kMaxSplits; ++t) v[t] = vn[t];
          if (u + C::kEpiWarps < u_end) load_unit(u + C::kEpiWarps, vn);
          const int r = u / gpr;
          const int col = n0 + (u - r * gpr) * 128;
          const int64_t off = (int64_t)(m0 + r) * p.N + col + lane * 4;
          const float4 a4 = sum_parts(v);
          const uint32_t b01 = pack_bf16x2(a4.x, a4.y), b23 = pack_bf16x2(a4.z, a4.w);
          if (p.out && in_bounds(p.status, off, 4, p.n_out))
            *reinterpret_cast<uint2*>(p.out + off) = make_uint2(b01, b23);
          const float x0 = bf16lo(b01), x1 = bf16hi(b01), x2 = bf16lo(b23), x3 = bf16hi(b23);
          float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
          float sc = __fdiv_rn(fmaxf(amax, kEps), kFp8Max);
          if (p.q_fmt != BFQ_SCALE_F32) sc = ceil_pow2(sc);
          const float y = __frcp_rn(sc);
          uint32_t lo, hi;
          if (p.q_fmt == BFQ_SCALE_F32) {
            lo = cvt_e4m3x2(group_div(x0, sc, y), group_div(x1, sc, y));
            hi = cvt_e4m3x2(group_div(x2, sc, y), group_div(x3, sc, y));
          } else {
            lo = cvt_e4m3x2(__fmul_rn(x0, y), __fmul_rn(x1, y));
            hi = cvt_e4m3x2(__fmul_rn(x2, y), __fmul_rn(x3, y));
          }
          if (in_bounds(p.status, off, 4, p.n_q))
            *reinterpret_cast<uint32_t*>(p.q_out + off) = lo | (hi << 16);
          if (lane == 0) {
            const int m = m0 + r, group = col >> 7;
            if (p.q_fmt == BFQ_SCALE_UE8M0_PACKED) {
              const int64_t woff = (int64_t)(group >> 2) * p.q_scale_ld + m;
              if (in_bounds(p.status, woff, 1, p.n_qs)) {
                uint8_t* word = (uint8_t*)p.q_scales + woff * 4;
                word[group & 3] = (uint8_t)ue8m0_byte(sc);
                if (col + 128 >= p.N)
                  for (int bb = (group & 3) + 1; bb < 4; ++bb) word[bb] = 0;
              }
            } else {
              const int64_t soff = (int64_t)group * p.q_scale_ld + m;
              if (in_bounds(p.status, soff, 1, p.n_qs)) ((float*)p.q_scales)[soff] = sc;
            }
          }
        }
      } else if (!*abort_flag) {
        const int rows = min(kBM, m_limit - m0);
        const int upr = min(BN, p.N - n0) / 4;  // float4 units per row
        const int total = rows * upr;
        const int u_begin = (int)((int64_t)split * total / p.splits);
        const int u_end = (int)((int64_t)(split + 1) * total / p.splits);
        for (int u = u_begin + (int)threadIdx.x - C::kEpiWarp0 * 32; u < u_end;
             u += C::kEpiWarps * 32) {
          const int r = u / upr, c4 = u - (u / upr) * upr;
          const int64_t off = (int64_t)(m0 + r) * p.N + n0 + c4 * 4;
          float4 v[kMaxSplits];
          load_parts(r, c4, v);
          const float4 a4 = sum_parts(v);
          if (in_bounds(p.status, off, 4, p.n_out))
            *reinterpret_cast<uint2*>(p.out + off) =
                make_uint2(pack_bf16x2(a4.x, a4.y), pack_bf16x2(a4.z, a4.w));
        }
      }
      cluster_sync();  // the peers have read this CTA's partial
    }
  }

  // ---- teardown: everyone is done with TMEM before it is released ----
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}


// ----------------------------------------------------------------------------
// Persistent form (BN = 256, no K split): one CTA per SM walks its share of
// the tiles, tile t going to CTA t mod gridDim.x.  The TMA producer, the MMA
// issuer and the scale loader run ahead across tile boundaries, so a tile's
// promotion drain and store overlap the next tile's loads and first MMAs, and
// barrier and TMEM set-up are paid once per SM rather than once per tile.
// Tiles leave through a dedicated staging buffer (the stage ring stays busy
// with the next tile): dense tiles stage the whole 128 x 256 tile and issue
// its four TMA-store boxes together; masked tiles stage one 128 x 64 box at
// a time and copy its valid rows out with coalesced stores.
// Masked: the tile list holds only row tiles that start below their expert's
// count — per-expert tile counts are prefix-summed in shared memory at start
// — so padding costs no CTA time and the valid tiles spread evenly over the
// SMs; rows past the count are never written.
// ----------------------------------------------------------------------------

// STAGES: depth of the operand ring.  The shared memory a fourth stage would
// take holds three more output boxes instead, so the staging buffer holds one
// 128-row x 64-column bf16 box (4 stages: the masked forms) or the whole
// 128 x 256 tile (3 stages: dense tiles, whose four TMA stores then run on
// while the next tile is promoted, instead of each box waiting for the last
// to leave the buffer); the total is the same.
template <int STAGES>
struct PersistCfgT {
  using C = GemmCfg<256>;
  static_assert(STAGES == 3 || STAGES == 4, "3 or 4 operand stages");
  static constexpr int kStages = STAGES;
  static constexpr int kBoxBytes = kBM * 64 * 2;  // one 128-row x 64-column bf16 box
  static constexpr int kStagingBoxes = STAGES == 4 ? 1 : 4;
  static constexpr int kStagingBytes = kStagingBoxes * kBoxBytes;
  static constexpr int kPrefixBytes = (2 * kPersistMaxExperts + 2) * 4;
  static constexpr size_t kSmemBytes = (size_t)kStages * C::kStageBytes + kStagingBytes +
                                       C::kScaleBytes + kPrefixBytes + C::kBarrierBytes + 1024;
  // Register split of the 384-thread launch (168 each): warpgroup 0 keeps 40
  // (its tile walk spills at 24, which slowed every K block by ~30 %), the
  // epilogue 232 (no spills).
  static constexpr int kWg0Regs = 40;
  static constexpr int kEpiRegs = 232;
  static_assert(128 * kWg0Regs + 256 * kEpiRegs <= 384 * 168, "register split");
};
using PersistCfg = PersistCfgT<4>;
static_assert(PersistCfgT<3>::kSmemBytes == PersistCfgT<4>::kSmemBytes, "same footprint");


template <bool MASKED, bool QOUT = false, bool SILU = false, int STAGES = 4>
__global__ void __launch_bounds__(GemmCfg<256>::kThreads, 1)
    gemm_block_fp8_persistent(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmW,
                              const __grid_constant__ CUtensorMap tmO, const GemmParams p) {
  constexpr int BN = 256;
  using C = GemmCfg<BN>;
  using PC = PersistCfgT<STAGES>;
  static_assert(!SILU || (MASKED && !QOUT), "the fused silu-mul-quant output is a masked form");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + PC::kStages * C::kABytes;
  uint8_t* stg = smem + (size_t)PC::kStages * C::kStageBytes;  // 1024-byte aligned
  uint32_t* sc_a = (uint32_t*)(stg + PC::kStagingBytes);       // [slot][128]
  uint32_t* sc_w = sc_a + C::kScaleSlots * kBM;                // [slot][2]
  int* tpre = (int*)(sc_w + 2 * C::kScaleSlots);               // [E + 1]
  int* cnt = tpre + kPersistMaxExperts + 1;                    // [E]
  uint64_t* full = (uint64_t*)(cnt + kPersistMaxExperts + 1);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* sfull = tempty + 2;
  uint64_t* sempty = sfull + C::kScaleSlots;
  uint64_t* drain = sempty + C::kScaleSlots;
  uint32_t* tmem_slot = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = p.K / kBK;

  if (MASKED) masked_tile_prefix(p, tpre, cnt);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], C::kEpiWarps);
    }
    for (int b = 0; b < C::kScaleSlots; ++b) {
      mbar_init(&sfull[b], 32);
      mbar_init(&sempty[b], C::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmW);
    if (!MASKED) prefetch_tensormap(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  if (!MASKED) griddep_wait();
  griddep_launch_dependents();
  const int total = MASKED ? tpre[p.E] : p.m_tiles * p.n_tiles;

  // Tiles of this CTA and the K blocks they stream, as one flat sequence
  // g = 0 .. steps-1 (tile g / KB, K block g mod KB): the warps that run at
  // 24 registers keep only a counter and the current tile's coordinates.
  const int my_tiles =
      (int)blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int steps = my_tiles * KB;
  static_assert(PC::kStages <= C::kStages, "barrier slots for the operand ring");
  static_assert((C::kScaleSlots & (C::kScaleSlots - 1)) == 0, "scale ring of 2^n slots");

  if (warp < C::kEpiWarp0) {
    setmaxnreg_dec<PC::kWg0Regs>();
    if (warp == 0) {
      // ------------------------------ TMA producer ------------------------------
      if (lane == 0) {
        int g = 0, i = 0, t = blockIdx.x, a_row = 0, w_row = 0;
        for (; g < steps; ++g) {
          if (i == 0) {
            int e, m0, n0, ml;
            persist_tile<MASKED>(t, p, tpre, cnt, e, m0, n0, ml);
            a_row = (MASKED ? e * p.M : 0) + m0;
            w_row = (MASKED ? e * p.N : 0) + n0;
          }
          const int s = g % PC::kStages;
          const uint32_t ph = (uint32_t)(g / PC::kStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status, kWaitTimeoutNs)) break;
          mbar_arrive_expect_tx(&full[s], (uint32_t)C::kStageBytes);
          tma_load_2d(sA + (size_t)s * C::kABytes, &tmA, &full[s], i * kBK, a_row);
          tma_load_2d(sB + (size_t)s * C::kBBytes, &tmW, &full[s], i * kBK, w_row);
          if (++i == KB) {
            i = 0;
            t += gridDim.x;
          }
        }
        if (*abort_flag) {
          // let the copies already issued land before the CTA can exit
          for (int j = g - PC::kStages < 0 ? 0 : g - PC::kStages; j < g; ++j) {
            volatile int no_abort = 0;
            (void)mbar_wait(&full[j % PC::kStages], (uint32_t)(j / PC::kStages) & 1u, &no_abort,
                            p.status, kWaitTimeoutNs / 8);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------- MMA issuer -------------------------------
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
        int g = 0;
        for (; g < steps; ++g) {
          const int s = g % PC::kStages;
          const int buf = g & 1;
          if (!mbar_wait(&tempty[buf], ((uint32_t)(g >> 1) & 1u) ^ 1u, abort_flag, p.status,
                         kWaitTimeoutNs))
            break;
          tc_fence_after_sync();
          if (!mbar_wait(&full[s], (uint32_t)(g / PC::kStages) & 1u, abort_flag, p.status,
                         kWaitTimeoutNs))
            break;
          tc_fence_after_sync();
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + (size_t)s * C::kABytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + (size_t)s * C::kBBytes));
          const uint32_t d = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            umma_e4m3(d, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                      kk > 0 ? 1u : 0u);
          umma_commit(&empty[s]);
          umma_commit(&tfull[buf]);
        }
        if (*abort_flag && g > 0) {
          // wait for the MMAs already issued before TMEM is released
          umma_commit(drain);
          volatile int no_abort = 0;
          (void)mbar_wait(drain, 0, &no_abort, p.status, kWaitTimeoutNs / 8);
        }
      }
    } else if (warp == C::kScaleWarp) {
      // ------------------------------ scale loader ------------------------------
      const int nblks = (int)((p.N + 127) / 128);
      const bool packed = p.a_fmt == BFQ_SCALE_UE8M0_PACKED;
      const uint32_t* sa = (const uint32_t*)p.sa;
      const float* sw = p.sw;
      int i = 0, t = blockIdx.x, m0 = 0, ml = 0, nb0 = 0;
      for (int g = 0; g < steps; ++g) {
        if (i == 0) {
          int e, n0;
          persist_tile<MASKED>(t, p, tpre, cnt, e, m0, n0, ml);
          sa = (const uint32_t*)p.sa + (MASKED ? (int64_t)e * p.sa_estride : 0);
          sw = p.sw + (MASKED ? (int64_t)e * p.sw_estride : 0);
          nb0 = n0 / 128;
        }
        const int slot = g % C::kScaleSlots;
        if (!mbar_wait(&sempty[slot], ((uint32_t)(g / C::kScaleSlots) & 1u) ^ 1u, abort_flag,
                       p.status, kWaitTimeoutNs))
          break;
        const uint32_t* col = sa + (int64_t)(packed ? (i >> 2) : i) * p.sa_ld;
#pragma unroll
        for (int r = lane; r < kBM; r += 32)
          if (m0 + r < ml && in_bounds(p.status, (col - (const uint32_t*)p.sa) + m0 + r, 1, p.n_sa))
            cp_async_4(&sc_a[slot * kBM + r], col + m0 + r);
        if (lane < 2 && nb0 + lane < nblks &&
            in_bounds(p.status, (sw - p.sw) + (int64_t)(nb0 + lane) * KB + i, 1, p.n_sw))
          cp_async_4(&sc_w[slot * 2 + lane], sw + (int64_t)(nb0 + lane) * KB + i);
        cp_async_arrive_noinc(&sfull[slot]);
        if (++i == KB) {
          i = 0;
          t += gridDim.x;
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
    __syncwarp();
  } else {
    setmaxnreg_inc<PC::kEpiRegs>();
    // ------------------------- epilogue / promotion ---------------------------
    const int ew = warp - C::kEpiWarp0;
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int half = ew >> 2;
    const int row_local = quarter * 32 + lane;
    const bool store_thread = threadIdx.x == C::kEpiWarp0 * 32;
    int g = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int e, m0, n0, m_limit;
      persist_tile<MASKED>(t, p, tpre, cnt, e, m0, n0, m_limit);
      const int m = m0 + row_local;
      const bool row_ok = m < m_limit;
      const int col0 = n0 + half * 128;
      // SILU: the tile's columns are gate block n0/256 (0..127) and the
      // matching up block (128..255); warp half h accumulates gate and up
      // columns h*64 .. h*64+63 of each, i.e. the same 64 features.
      const bool warp_active = (m0 + quarter * 32 < m_limit) && (SILU || col0 < p.N);
      const int ncols = min(128, p.N - col0);

      uint64_t acc[64];
      // Stages output boxes r0 .. r0 + kStagingBoxes - 1 of the tile (box b =
      // columns b*64 .. b*64+63, held by warp half b/2) as bf16 in the 128-byte
      // swizzled layout: 16-byte chunk c of row r at chunk c ^ (r mod 8).
      auto stage_boxes = [&](int r0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int b = half * 2 + j;
          if (b < r0 || b >= r0 + PC::kStagingBoxes || !warp_active || j * 64 >= ncols) continue;
          const uint32_t row_addr =
              smem_u32(stg) + (uint32_t)((b - r0) * PC::kBoxBytes + row_local * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int a = j * 32 + c * 4;  // pair index of column j*64 + c*8 of this half
            const float2 f0 = unpack2(acc[a + 0]), f1 = unpack2(acc[a + 1]);
            const float2 f2 = unpack2(acc[a + 2]), f3 = unpack2(acc[a + 3]);
            st_shared_v4(row_addr + (uint32_t)((c ^ (row_local & 7)) << 4),
                         make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f1.x, f1.y),
                                    pack_bf16x2(f2.x, f2.y), pack_bf16x2(f3.x, f3.y)));
          }
        }
      };
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0ull;
      bool stop = false;
      for (int i = 0; i < KB; ++i, ++g) {
        const int buf = g & 1;
        const uint32_t tph = (uint32_t)(g >> 1) & 1u;
        const int slot = g % C::kScaleSlots;
        const uint32_t sph = (uint32_t)(g / C::kScaleSlots) & 1u;
        if (!mbar_wait(&sfull[slot], sph, abort_flag, p.status, kWaitTimeoutNs)) {
          stop = true;
          break;
        }
        const uint32_t a_bits = sc_a[slot * kBM + row_local];
        const float w_s = __uint_as_float(sc_w[slot * 2 + (SILU ? 0 : half)]);
        const float w_s_up = SILU ? __uint_as_float(sc_w[slot * 2 + 1]) : 0.0f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[slot]);
        float sa_v;
        if (p.a_fmt == BFQ_SCALE_UE8M0_PACKED) {
          const uint32_t b = (a_bits >> (8 * (i & 3))) & 0xFFu;
          sa_v = b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);  // 2^(b-127)
        } else {
          sa_v = __uint_as_float(a_bits);
        }
        const uint64_t s2 = splat2(__fmul_rn(row_ok ? sa_v : 0.0f, w_s));
        const uint64_t s2_up = SILU ? splat2(__fmul_rn(row_ok ? sa_v : 0.0f, w_s_up)) : 0ull;
        if (!mbar_wait(&tfull[buf], tph, abort_flag, p.status, kWaitTimeoutNs)) {
          stop = true;
          break;
        }
        tc_fence_after_sync();
        if (warp_active) {
          if constexpr (SILU) {
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                   (uint32_t)(buf * BN + half * 64);
            uint64_t v[32];
            tmem_ld64_pairs_wait(taddr, v);  // gate columns
#pragma unroll
            for (int q = 0; q < 32; ++q) ffma2(acc[q], v[q], s2);
            tmem_ld64_pairs_wait(taddr + 128u, v);  // the matching up columns
#pragma unroll
            for (int q = 0; q < 32; ++q) ffma2(acc[32 + q], v[q], s2_up);
          } else {
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                   (uint32_t)(buf * BN + half * 128);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint64_t v[32];
              tmem_ld64_pairs_wait(taddr + (uint32_t)(h * 64), v);
#pragma unroll
              for (int q = 0; q < 32; ++q) ffma2(acc[h * 32 + q], v[q], s2);
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
      // Every epilogue warp takes the same decision (the stores and the fused
      // silu-mul-quant below synchronise them on named barriers).
      if (named_barrier_or(2, C::kEpiWarps * 32, stop || *abort_flag)) break;

      if constexpr (SILU) {
        silu_quant_tile_rows<C::kEpiWarps * 32>(p, acc, acc + 32, (float*)stg, e, m, n0, half,
                                                row_local, warp_active && row_ok);
      } else if (MASKED) {
        // Rows past the count must not be written, so no TMA store: each
        // 128 x 64 box is staged in shared memory (128-byte swizzle, as for
        // dense tiles) and its valid rows are copied out with 16-byte stores,
        // eight lanes per 128-byte row segment, so one store instruction
        // writes four whole segments instead of 16 bytes of 32 rows.
        const int rows_valid = min(kBM, m_limit - m0);
        const int tid = (int)threadIdx.x - C::kEpiWarp0 * 32;
        for (int r0 = 0; r0 < BN / 64; r0 += PC::kStagingBoxes) {
          named_barrier(1, C::kEpiWarps * 32);
          stage_boxes(r0);
          named_barrier(1, C::kEpiWarps * 32);
          for (int b = r0; b < r0 + PC::kStagingBoxes; ++b) {
            if (n0 + b * 64 >= p.N) break;
            const uint32_t box = smem_u32(stg) + (uint32_t)((b - r0) * PC::kBoxBytes);
            __nv_bfloat16* base =
                p.out + (int64_t)e * p.out_estride + (int64_t)m0 * p.N + n0 + b * 64;
            for (int q = tid; q < rows_valid * 8; q += C::kEpiWarps * 32) {
              const int r = q >> 3, c = q & 7;
              if (in_bounds(p.status, (base - p.out) + (int64_t)r * p.N + c * 8, 8, p.n_out))
                st_v4(base + (int64_t)r * p.N + c * 8,
                      ld_shared_v4(box + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4))));
            }
          }
        }
      } else {
        // The tile's four 128 x 64 boxes through the staging buffer, one at
        // a time or all at once (3-stage ring); rows >= M are clipped by the
        // tensor map.  The stores run on while the next tile is promoted;
        // the buffer is only rewritten once they have read it.  (Fused output
        // quant: the bf16 output is optional; the condition is the same for
        // every thread.)
        if (!QOUT || p.out != nullptr) {
          for (int r0 = 0; r0 < BN / 64; r0 += PC::kStagingBoxes) {
            if (store_thread) bulk_wait_read_all();  // earlier boxes have left the buffer
            named_barrier(1, C::kEpiWarps * 32);
            stage_boxes(r0);
            fence_proxy_async_smem();
            named_barrier(1, C::kEpiWarps * 32);
            if (store_thread) {
              for (int b = r0; b < r0 + PC::kStagingBoxes; ++b)
                if (n0 + b * 64 < p.N)
                  tma_store_2d(&tmO, stg + (b - r0) * PC::kBoxBytes, n0 + b * 64, m0);
              bulk_commit();
            }
          }
        }
        if constexpr (QOUT) {
          if (warp_active && row_ok)
            quant_store_row_group(acc, p, m, col0);
        }
      }
    }
    if (!MASKED && store_thread) bulk_wait_read_all();
  }

  // ---- teardown: everyone is done with TMEM before it is released ----
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    else
      cudaGetLastError();
  });
  return g_encode;
}

// 2D map over a row-major byte matrix [rows][inner] with a 128 x box_rows box
// and 128-byte swizzling; out-of-range rows read as zero.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
              uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2D map over the bf16 output [rows][cols] with a 64 x 128 box and 128-byte
// swizzling, for TMA stores of the staged tile.
bool make_out_map(CUtensorMap* map, void* base, uint64_t cols, uint64_t rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

struct Plan {
  int bn = 256;
  bool persist = false;  // persistent 256-wide kernel (no K split)
  int m_tiles = 0, n_tiles = 0, splits = 1;
};

template <int BN>
int max_active_clusters(const DeviceInfo& dev, int cluster);

// Plan for one tile width: K is split over a cluster of CTAs when there are
// fewer tiles than SMs.
Plan plan_for_width(const DeviceInfo& dev, int bn, int64_t M, int64_t N, int64_t K) {
  Plan pl;
  pl.bn = bn;
  pl.m_tiles = (int)cdiv(M, kBM);
  pl.n_tiles = (int)cdiv(N, pl.bn);
  const int tiles = pl.m_tiles * pl.n_tiles;
  const int KB = (int)(K / kBK);
  int splits = 1;
  if (tiles < dev.sm_count) splits = dev.sm_count / tiles;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits > KB) splits = KB;
  if (splits < 1) splits = 1;
  // all clusters of the grid should be resident at once
  while (splits > 1 && (pl.bn == 256 ? max_active_clusters<256>(dev, splits)
                                     : max_active_clusters<128>(dev, splits)) < tiles)
    --splits;
  pl.splits = splits;
  return pl;
}

// 256-wide tiles, except where the 256-wide plan splits K and 128-wide tiles
// keep more CTAs busy, or as many with no K split at all (no partial sums to
// reduce, and the tile leaves through the TMA-store epilogue).  This pays
// once the tile holds more than 32 rows; with fewer rows the 256-wide tile's
// larger weight stages (more bytes in flight per SM) win.
Plan dense_plan(const DeviceInfo& dev, int64_t M, int64_t N, int64_t K) {
  Plan pl = plan_for_width(dev, N > 128 ? 256 : 128, M, N, K);
  if (pl.bn == 256 && pl.splits > 1 && M > 32) {
    const Plan alt = plan_for_width(dev, 128, M, N, K);
    const int ctas = pl.m_tiles * pl.n_tiles * pl.splits;
    const int alt_ctas = alt.m_tiles * alt.n_tiles * alt.splits;
    if (alt_ctas > ctas || (alt.splits == 1 && alt_ctas >= ctas)) pl = alt;
  }
  // More 256-wide tiles than SMs: one persistent CTA per SM walks them.
  if (pl.bn == 256 && pl.splits == 1 && pl.m_tiles * pl.n_tiles > dev.sm_count &&
      dev.smem_optin >= PersistCfg::kSmemBytes)
    pl.persist = true;
  // Between one and 1.5 waves of long-K tiles (the persistent schedule would
  // leave most SMs idle in its second round): K split two ways over 2-CTA
  // clusters instead, 2 x tiles half-length CTAs in about three half-waves.
  const int tiles = pl.m_tiles * pl.n_tiles;
  if (pl.persist && tiles < 2 * dev.sm_count && tiles % dev.sm_count <= dev.sm_count / 2 &&
      K / kBK >= 64 && max_active_clusters<256>(dev, 2) > 0) {
    pl.persist = false;
    pl.splits = 2;
  }
  return pl;
}

template <int BN, bool MASKED, bool QOUT = false>
bfq_status configure(const DeviceInfo& dev) {
  using C = GemmCfg<BN>;
  static bool configured[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (configured[dev.ordinal]) return BFQ_OK;
  if (C::kRegSplit) {
    // setmaxnreg.inc only completes if the launch allocation covers the
    // split; refuse to launch a build whose register count differs.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, gemm_block_fp8_kernel<BN, MASKED, QOUT>) != cudaSuccess) {
      cudaGetLastError();
      return BFQ_ERR_CUDA;
    }
    if (fa.numRegs != C::kLaunchRegs) return BFQ_ERR_DEVICE;
  }
  if (cudaFuncSetAttribute(gemm_block_fp8_kernel<BN, MASKED, QOUT>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)C::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return BFQ_ERR_CUDA;
  }
  configured[dev.ordinal] = true;
  return BFQ_OK;
}

// Clusters of `cluster` CTAs of the dense kernel that fit on the device at
// once (cached per device and size; 0 when unknown).
template <int BN>
int max_active_clusters(const DeviceInfo& dev, int cluster) {
  using C = GemmCfg<BN>;
  static int cache[64][kMaxSplits + 1];
  static std::mutex mu;
  if (cluster < 1 || cluster > kMaxSplits) return 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev.ordinal][cluster]) return cache[dev.ordinal][cluster];
  }
  if (configure<BN, false>(dev) != BFQ_OK) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(cluster * dev.sm_count));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_block_fp8_kernel<BN, false>, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[dev.ordinal][cluster] = n > 0 ? n : -1;
  return n;
}

template <int BN, bool MASKED, bool QOUT = false>
bfq_status launch(const DeviceInfo& dev, const CUtensorMap& ma, const CUtensorMap& mw,
                  const CUtensorMap& mo, const GemmParams& p, unsigned grid, cudaStream_t s) {
  using C = GemmCfg<BN>;
  bfq_status st = configure<BN, MASKED, QOUT>(dev);
  if (st != BFQ_OK) return st;
  return launch_status(launch_pdl(gemm_block_fp8_kernel<BN, MASKED, QOUT>, dim3(grid),
                                  dim3(C::kThreads), C::kSmemBytes, s,
                                  p.splits > 1 ? (unsigned)p.splits : 1u, ma, mw, mo, p));
}

// Tile configuration of the masked grouped GEMM (no K split).
Plan masked_plan(const DeviceInfo& dev, int64_t E, int64_t T, int64_t N, int64_t K) {
  (void)T;
  (void)K;
  Plan pl;
  pl.bn = N > 128 ? 256 : 128;
  pl.persist = pl.bn == 256 && E <= kPersistMaxExperts &&
               dev.smem_optin >= PersistCfg::kSmemBytes;
  return pl;
}

template <bool MASKED, bool QOUT = false, bool SILU = false, int STAGES = 4>
bfq_status configure_persistent(const DeviceInfo& dev) {
  static bool configured[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (configured[dev.ordinal]) return BFQ_OK;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, gemm_block_fp8_persistent<MASKED, QOUT, SILU, STAGES>) !=
      cudaSuccess) {
    cudaGetLastError();
    return BFQ_ERR_CUDA;
  }
  // setmaxnreg.inc only completes if the launch allocation covers the split
  if (fa.numRegs != GemmCfg<256>::kLaunchRegs) return BFQ_ERR_DEVICE;
  if (cudaFuncSetAttribute(gemm_block_fp8_persistent<MASKED, QOUT, SILU, STAGES>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)PersistCfgT<STAGES>::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return BFQ_ERR_CUDA;
  }
  configured[dev.ordinal] = true;
  return BFQ_OK;
}

template <bool MASKED, bool QOUT = false, bool SILU = false, int STAGES = 4>
bfq_status launch_persistent(const DeviceInfo& dev, const CUtensorMap& ma, const CUtensorMap& mw,
                             const CUtensorMap& mo, const GemmParams& p, unsigned grid,
                             cudaStream_t s) {
  bfq_status st = configure_persistent<MASKED, QOUT, SILU, STAGES>(dev);
  if (st != BFQ_OK) return st;
  return launch_status(launch_pdl(gemm_block_fp8_persistent<MASKED, QOUT, SILU, STAGES>,
                                  dim3(grid), dim3(GemmCfg<256>::kThreads),
                                  PersistCfgT<STAGES>::kSmemBytes, s, 1u, ma, mw, mo, p));
}

// Dense persistent launch: the 3-stage ring, so that the whole output tile is
// staged at once and its four TMA stores overlap the next tile's promotion.
template <bool QOUT>
bfq_status launch_dense_persistent(const DeviceInfo& dev, const CUtensorMap& ma,
                                   const CUtensorMap& mw, const CUtensorMap& mo,
                                   const GemmParams& p, unsigned grid, cudaStream_t s) {
  return launch_persistent<false, QOUT, false, 3>(dev, ma, mw, mo, p, grid, s);
}

bfq_status check_device(DeviceInfo* dev) {
  bfq_status st = current_device(dev);
  if (st != BFQ_OK) return st;
  if (dev->cc_major != 10) return BFQ_ERR_DEVICE;
  if (dev->smem_optin < GemmCfg<256>::kSmemBytes) return BFQ_ERR_DEVICE;
  return BFQ_OK;
}

}  // namespace
}  // namespace bfq

using namespace bfq;

// Every split reduces through distributed shared memory, so no plan needs a
// workspace.
extern "C" size_t bfq_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t E) {
  (void)M;
  (void)N;
  (void)K;
  (void)E;
  return 0;
}

namespace bfq {
namespace {

// Optional fused output quant of a dense GEMM (null: plain bf16 output).
struct QuantOut {
  int32_t fmt;
  void* q;
  void* scales;
  int64_t scale_ld;
};

bfq_status gemm_dense(const void* a_q, const void* a_scales, int32_t a_fmt, int64_t a_scale_ld,
                      const void* w_q, const float* w_scales, int64_t M, int64_t N, int64_t K,
                      void* out, void* workspace, size_t workspace_bytes, const QuantOut* qo,
                      void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || !valid_fmt(a_fmt) || a_scale_ld < M)
    return BFQ_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 64 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (qo) {
    if (!valid_fmt(qo->fmt) || qo->scale_ld < M) return BFQ_ERR_INVALID_ARG;
    if (N % 128 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  }
  if (M == 0) return BFQ_OK;
  if (!a_q || !a_scales || !w_q || !w_scales || (!out && !qo)) return BFQ_ERR_INVALID_ARG;
  if (qo && (!qo->q || !qo->scales)) return BFQ_ERR_INVALID_ARG;
  if (!aligned16(a_q) || !aligned16(w_q) || (out && !aligned16(out)) || a_scale_ld % 4 != 0 ||
      ((uintptr_t)a_scales & 3u) || ((uintptr_t)w_scales & 3u))
    return BFQ_ERR_MISALIGNED;
  if (qo && (!aligned16(qo->q) || ((uintptr_t)qo->scales & 3u) || qo->scale_ld % 4 != 0))
    return BFQ_ERR_MISALIGNED;
  if (workspace_bytes > 0 && !workspace) return BFQ_ERR_INVALID_ARG;
  if (workspace && !aligned16(workspace)) return BFQ_ERR_MISALIGNED;
  DeviceInfo dev;
  bfq_status st = check_device(&dev);
  if (st != BFQ_OK) return st;
  Plan pl = dense_plan(dev, M, N, K);
  CUtensorMap ma, mw, mo;
  if (!make_map(&ma, a_q, (uint64_t)K, (uint64_t)M, kBM) ||
      !make_map(&mw, w_q, (uint64_t)K, (uint64_t)N, (uint32_t)pl.bn))
    return BFQ_ERR_CUDA;
  if (out ? !make_out_map(&mo, out, (uint64_t)N, (uint64_t)M) : false) return BFQ_ERR_CUDA;
  if (!out) mo = ma;  // never used: the kernels skip the bf16 store
  GemmParams p{};
  p.sa = a_scales;
  p.sa_ld = a_scale_ld;
  p.sw = w_scales;
  p.out = (__nv_bfloat16*)out;
  p.status = device_status_ptr();
  if (!p.status) return BFQ_ERR_CUDA;
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.m_tiles = pl.m_tiles;
  p.n_tiles = pl.n_tiles;
  p.splits = pl.splits;
  p.a_fmt = a_fmt;
  if (qo) {
    p.q_out = (uint8_t*)qo->q;
    p.q_scales = qo->scales;
    p.q_scale_ld = qo->scale_ld;
    p.q_fmt = qo->fmt;
  }
  p.n_sa = scale_cols(K, a_fmt) * a_scale_ld;
  p.n_sw = cdiv(N, 128) * (K / 128);
  p.n_out = M * N;
  p.n_q = qo ? M * N : 0;
  p.n_qs = qo ? scale_cols(N, qo->fmt) * qo->scale_ld : 0;
  const unsigned grid = (unsigned)(pl.m_tiles * pl.n_tiles * pl.splits);
  const unsigned pgrid = grid < (unsigned)dev.sm_count ? grid : (unsigned)dev.sm_count;
  cudaStream_t s = (cudaStream_t)stream;
  if (qo) {
    if (pl.persist) return launch_dense_persistent<true>(dev, ma, mw, mo, p, pgrid, s);
    return pl.bn == 256 ? launch<256, false, true>(dev, ma, mw, mo, p, grid, s)
                        : launch<128, false, true>(dev, ma, mw, mo, p, grid, s);
  }
  if (pl.persist) return launch_dense_persistent<false>(dev, ma, mw, mo, p, pgrid, s);
  return pl.bn == 256 ? launch<256, false>(dev, ma, mw, mo, p, grid, s)
                      : launch<128, false>(dev, ma, mw, mo, p, grid, s);
}

}  // namespace
}  // namespace bfq

extern "C" bfq_status bfq_gemm_block_fp8(const void* a_q, const void* a_scales, int32_t a_fmt,
                                         int64_t a_scale_ld, const void* w_q,
                                         const float* w_scales, int64_t M, int64_t N,
                                         int64_t K, void* out, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  return gemm_dense(a_q, a_scales, a_fmt, a_scale_ld, w_q, w_scales, M, N, K, out, workspace,
                    workspace_bytes, nullptr, stream);
}

extern "C" bfq_status bfq_gemm_block_fp8_quant(const void* a_q, const void* a_scales,
                                               int32_t a_fmt, int64_t a_scale_ld,
                                               const void* w_q, const float* w_scales, int64_t M,
                                               int64_t N, int64_t K, void* out, int32_t q_fmt,
                                               void* q_out, void* q_scales, int64_t q_scale_ld,
                                               void* workspace, size_t workspace_bytes,
                                               void* stream) {
  const QuantOut qo{q_fmt, q_out, q_scales, q_scale_ld};
  return gemm_dense(a_q, a_scales, a_fmt, a_scale_ld, w_q, w_scales, M, N, K, out, workspace,
                    workspace_bytes, &qo, stream);
}

extern "C" bfq_status bfq_gemm_block_fp8_masked(
    const void* a_q, const void* a_scales, int32_t a_fmt, int64_t a_scale_ld, const void* w_q,
    const float* w_scales, const int32_t* valid_counts, int32_t E, int32_t T, int64_t N,
    int64_t K, int32_t expected_m, void* out, void* workspace, size_t workspace_bytes,
    void* stream) {
  (void)expected_m;
  (void)workspace;
  (void)workspace_bytes;
  if (E < 0 || T < 0 || N <= 0 || K <= 0 || !valid_fmt(a_fmt) || a_scale_ld < T)
    return BFQ_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 64 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)E * T > 0x7FFFFFFF || (int64_t)E * N > 0x7FFFFFFF || K > 0x7FFFFFFF)
    return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (E == 0 || T == 0) return BFQ_OK;
  if (!a_q || !a_scales || !w_q || !w_scales || !valid_counts || !out)
    return BFQ_ERR_INVALID_ARG;
  if (!aligned16(a_q) || !aligned16(w_q) || !aligned16(out) || a_scale_ld % 4 != 0 ||
      ((uintptr_t)a_scales & 3u) || ((uintptr_t)w_scales & 3u))
    return BFQ_ERR_MISALIGNED;
  DeviceInfo dev;
  bfq_status st = check_device(&dev);
  if (st != BFQ_OK) return st;
  const Plan mp = masked_plan(dev, E, T, N, K);
  const int bn = mp.bn;
  CUtensorMap ma, mw;
  if (!make_map(&ma, a_q, (uint64_t)K, (uint64_t)E * T, kBM) ||
      !make_map(&mw, w_q, (uint64_t)K, (uint64_t)E * N, (uint32_t)bn))
    return BFQ_ERR_CUDA;
  GemmParams p{};
  p.sa = a_scales;
  p.sa_ld = a_scale_ld;
  p.sa_estride = scale_cols(K, a_fmt) * a_scale_ld;
  p.sw = w_scales;
  p.sw_estride = cdiv(N, 128) * (K / 128);
  p.out = (__nv_bfloat16*)out;
  p.out_estride = (int64_t)T * N;
  p.counts = valid_counts;
  p.status = device_status_ptr();
  if (!p.status) return BFQ_ERR_CUDA;
  p.M = T;
  p.N = (int)N;
  p.K = (int)K;
  p.m_tiles = (int)cdiv(T, kBM);
  p.n_tiles = (int)cdiv(N, bn);
  p.splits = 1;
  p.a_fmt = a_fmt;
  p.E = E;
  p.n_sa = E * p.sa_estride;
  p.n_sw = E * p.sw_estride;
  p.n_out = (int64_t)E * T * N;
  const int64_t grid = (int64_t)p.m_tiles * p.n_tiles * E;
  if (grid > 0x7FFFFFFF) return BFQ_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  if (mp.persist)
    return launch_persistent<true>(dev, ma, mw, mw, p,
                                   (unsigned)(grid < dev.sm_count ? grid : dev.sm_count), s);
  return bn == 256 ? launch<256, true>(dev, ma, mw, mw, p, (unsigned)grid, s)
                   : launch<128, true>(dev, ma, mw, mw, p, (unsigned)grid, s);
}

// ----------------------------------------------------------------------------
// Entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc: plugins inside a host framework that
// owns every byte of device memory through its own allocator, and serving
// loops that forbid allocation after start-up because cudaMalloc can
// synchronize the device.  The K splits reduce through distributed shared memory, so no
// plan needs scratch: this is the regular call without a workspace.
// ----------------------------------------------------------------------------
extern "C" size_t bfq_gemm_noalloc_scratch_bytes(void) { return 0; }

extern "C" bfq_status bfq_gemm_block_fp8_noalloc(const void* a_q, const void* a_scales,
                                                 int32_t a_fmt, int64_t a_scale_ld,
                                                 const void* w_q, const float* w_scales,
                                                 int64_t M, int64_t N, int64_t K, void* out,
                                                 void* stream) {
  return bfq_gemm_block_fp8(a_q, a_scales, a_fmt, a_scale_ld, w_q, w_scales, M, N, K, out,
                            nullptr, 0, stream);
}

// ----------------------------------------------------------------------------
// masked up projection with silu-mul-quant fused into its epilogue
// ----------------------------------------------------------------------------
namespace bfq {
namespace {

// Copies 128-row blocks of each expert's [2I][K] weight (and the matching
// scale rows) so that output block 2j is gate block j and block 2j+1 is up
// block j.  One CTA per (output block, expert); 16-byte copies.
__global__ void __launch_bounds__(256)
    interleave_gate_up_kernel(const uint8_t* __restrict__ w, const float* __restrict__ sw,
                              int64_t I, int64_t K, uint8_t* __restrict__ w_out,
                              float* __restrict__ sw_out) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t nb = blockIdx.x, e = blockIdx.y;
  const int64_t G = I / 128, KB = K / 128;
  const int64_t src_blk = (nb & 1) ? G + (nb >> 1) : (nb >> 1);
  const uint4* src = (const uint4*)(w + (e * 2 * I + src_blk * 128) * K);
  uint4* dst = (uint4*)(w_out + (e * 2 * I + nb * 128) * K);
  const int64_t n16 = 128 * K / 16;
  for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
  const float* ssrc = sw + (e * 2 * G + src_blk) * KB;
  float* sdst = sw_out + (e * 2 * G + nb) * KB;
  for (int64_t i = threadIdx.x; i < KB; i += blockDim.x) sdst[i] = ssrc[i];
}

}  // namespace
}  // namespace bfq

extern "C" bfq_status bfq_interleave_gate_up(const void* w_q, const float* w_scales, int32_t E,
                                             int64_t I, int64_t K, void* w_q_out,
                                             float* w_scales_out, void* stream) {
  if (E <= 0 || I <= 0 || K <= 0) return BFQ_ERR_INVALID_ARG;
  if (I % 128 != 0 || K % 128 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (E > 65535 || 2 * I / 128 > 0x7FFFFFFF) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (!w_q || !w_scales || !w_q_out || !w_scales_out) return BFQ_ERR_INVALID_ARG;
  if (w_q == w_q_out || w_scales == w_scales_out) return BFQ_ERR_INVALID_ARG;
  if (!aligned16(w_q) || !aligned16(w_q_out) || ((uintptr_t)w_scales & 3u) ||
      ((uintptr_t)w_scales_out & 3u))
    return BFQ_ERR_MISALIGNED;
  DeviceInfo dev;
  bfq_status st = current_device(&dev);
  if (st != BFQ_OK) return st;
  return launch_status(launch_pdl(interleave_gate_up_kernel, dim3((unsigned)(2 * I / 128),
                                                                   (unsigned)E),
                                  dim3(256), 0, (cudaStream_t)stream, 1u,
                                  (const uint8_t*)w_q, w_scales, I, K, (uint8_t*)w_q_out,
                                  w_scales_out));
}

extern "C" bfq_status bfq_gemm_block_fp8_masked_silu_quant(
    const void* a_q, const void* a_scales, int32_t a_fmt, int64_t a_scale_ld, const void* w_q,
    const float* w_scales, const int32_t* valid_counts, int32_t E, int32_t T, int64_t I,
    int64_t K, int32_t q_fmt, void* q_out, void* q_scales, int64_t q_scale_ld, void* stream) {
  if (E < 0 || T < 0 || I <= 0 || K <= 0 || !valid_fmt(a_fmt) || !valid_fmt(q_fmt) ||
      a_scale_ld < T || q_scale_ld < T)
    return BFQ_ERR_INVALID_ARG;
  if (K % 128 != 0 || I % 128 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  const int64_t N = 2 * I;
  if ((int64_t)E * T > 0x7FFFFFFF || (int64_t)E * N > 0x7FFFFFFF || K > 0x7FFFFFFF ||
      (int64_t)T * I > 0x7FFFFFFF)
    return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (E > kPersistMaxExperts) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (E == 0 || T == 0) return BFQ_OK;
  if (!a_q || !a_scales || !w_q || !w_scales || !valid_counts || !q_out || !q_scales)
    return BFQ_ERR_INVALID_ARG;
  if (!aligned16(a_q) || !aligned16(w_q) || !aligned16(q_out) || a_scale_ld % 4 != 0 ||
      q_scale_ld % 4 != 0 || ((uintptr_t)a_scales & 3u) || ((uintptr_t)w_scales & 3u) ||
      ((uintptr_t)q_scales & 3u))
    return BFQ_ERR_MISALIGNED;
  DeviceInfo dev;
  bfq_status st = check_device(&dev);
  if (st != BFQ_OK) return st;
  if (dev.smem_optin < PersistCfg::kSmemBytes) return BFQ_ERR_DEVICE;
  CUtensorMap ma, mw;
  if (!make_map(&ma, a_q, (uint64_t)K, (uint64_t)E * T, kBM) ||
      !make_map(&mw, w_q, (uint64_t)K, (uint64_t)E * N, 256u))
    return BFQ_ERR_CUDA;
  GemmParams p{};
  p.sa = a_scales;
  p.sa_ld = a_scale_ld;
  p.sa_estride = scale_cols(K, a_fmt) * a_scale_ld;
  p.sw = w_scales;
  p.sw_estride = (N / 128) * (K / 128);
  p.counts = valid_counts;
  p.status = device_status_ptr();
  if (!p.status) return BFQ_ERR_CUDA;
  p.M = T;
  p.N = (int)N;
  p.K = (int)K;
  p.m_tiles = (int)cdiv(T, kBM);
  p.n_tiles = (int)(N / 256);
  p.splits = 1;
  p.a_fmt = a_fmt;
  p.E = E;
  p.q_out = (uint8_t*)q_out;
  p.q_scales = q_scales;
  p.q_scale_ld = q_scale_ld;
  p.q_fmt = q_fmt;
  p.silu_tab = silu_table(dev, (cudaStream_t)stream);
  p.n_sa = E * p.sa_estride;
  p.n_sw = E * p.sw_estride;
  p.n_q = (int64_t)E * T * I;
  p.n_qs = E * scale_cols(I, q_fmt) * q_scale_ld;
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles * E;
  const unsigned grid = (unsigned)(tiles < dev.sm_count ? tiles : dev.sm_count);
  return launch_persistent<true, false, true>(dev, ma, mw, mw, p, grid, (cudaStream_t)stream);
}
