// gemm_blockscaled.cu — block-scaled FP8 GEMM for power-of-two (UE8M0) scales,
// with the scales applied by the tensor cores' own block scaling.
//
//   out[m, n] = sum_b sA[m, b] * sW[n / 128, b] * sum_{k in block b} a[m, k] w[n, k]
//
// with every sA and sW a power of two ("vLLM DeepGEMM FP8 Block GEMM 基准测试"
// §4.1–4.2: UE8M0 scales are the hardware-friendly form; "[Perf] Deepgemm
// fused layout kernel for activations": four exponents packed per int32).
// Multiplying by a power of two is exact, so the MMA itself can scale each
// K = 32 step's products by 2^(eA + eB) (tcgen05.mma kind::mxf8f6f4
// .block_scale, scale_vec::1X) and accumulate the whole K range in TMEM: no
// per-K-block TMEM read and promotion FMAs as in the general kernel.
//
// One CTA per SM walks 128 x 256 output tiles (tile t to CTA t mod gridDim.x),
// dense or masked per expert as the persistent promotion kernel does:
//   warp 0      TMA producer: per 128-deep K block one 128 x 128 A tile and
//               one 256 x 128 W tile (128-byte swizzle) into a 4-stage ring.
//   warp 1      allocates 512 TMEM columns (accumulator 0-255, scale ring
//               256-319); lane 0 copies each group of four K blocks' scale
//               words from shared memory into a TMEM slot (tcgen05.cp) and
//               issues 4 block-scaled MMAs per K block, the scale byte being
//               the K block's position in its group of four.
//   warp 2      scale loader: per group of four K blocks, one 32-bit word per
//               activation row (the packed UE8M0 word as stored, brought in
//               by a bulk copy, or the exponent bytes of four fp32 powers of
//               two) and one per weight row (the exponent bytes of its
//               128-row block's four fp32 scales), in the row order the copy
//               into TMEM expects.
//   warps 4-11  epilogue: once per tile, read the fp32 accumulator (each warp
//               32 rows x 128 columns), release TMEM to the next tile's MMAs,
//               round to bf16 and store (TMA store of 128 x 64 boxes; masked
//               tiles copy only their valid rows).
// A scale that is not a positive power of two cannot be applied by the
// hardware: the loader latches BFQ_ERR_FORMAT in the library's status word
// (the output of that call is undefined).  Every wait is bounded as in the
// other GEMM kernels.
#include <cudaTypedefs.h>

#include <mutex>

#include "bfq_device.cuh"
#include "gemm_common.cuh"

namespace bfq {
namespace {

struct BsCfg {
  static constexpr int kBN = 256;
  static constexpr int kStages = 4;
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = kBN * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kGroup = 4;     // K blocks per scale word (one byte each)
  static constexpr int kSfSlots = 6;   // groups of scale words in flight
  static constexpr int kSfaWords = kBM;
  static constexpr int kSfbWords = kBN;
  static constexpr int kSfSlotWords = kSfaWords + kSfbWords;
  static constexpr int kBoxBytes = kBM * 64 * 2;  // one 128-row x 64-column bf16 box
  static constexpr int kEpiWarp0 = 4;
  static constexpr int kEpiWarps = 8;
  static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSfCol0 = kBN;     // scale ring after the accumulator
  static constexpr uint32_t kSfSlotCols = 16;  // 4 columns of A words, 8 of W words
  static constexpr int kPrefixBytes = (2 * kPersistMaxExperts + 2) * 4;
  static constexpr int kBarrierBytes = 256;
  static constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + kBoxBytes +
                                       (size_t)kSfSlots * kSfSlotWords * 4 + kPrefixBytes +
                                       kBarrierBytes + 1024;
};
static_assert(BsCfg::kSfCol0 + BsCfg::kSfSlots * BsCfg::kSfSlotCols <= BsCfg::kTmemCols,
              "scale ring inside the TMEM allocation");
static_assert(BsCfg::kSmemBytes <= 232448, "fits the opt-in shared memory of one CTA");
static_assert((2 * BsCfg::kStages + 3 * BsCfg::kSfSlots + 3) * 8 + 8 <= BsCfg::kBarrierBytes,
              "barriers, TMEM address and abort flag fit their area");

// A positive normal power of two (exponent byte 1..255, no mantissa, no sign).
__device__ __forceinline__ bool pow2_bits(uint32_t b) {
  return (b & 0x807FFFFFu) == 0 && (b >> 23) != 0;
}

// SILU (masked only): the up projection with silu-and-mul and its quant in
// the epilogue (interleaved gate/up weights; the output is q_out/q_scales).
template <bool MASKED, bool SILU = false>
__global__ void __launch_bounds__(BsCfg::kThreads, 1)
    gemm_block_fp8_bs(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmO, const GemmParams p) {
  using C = BsCfg;
  constexpr int BN = C::kBN;
  static_assert(!SILU || MASKED, "the fused silu-mul-quant output is a masked form");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::kStages * C::kABytes;
  uint8_t* stg = smem + (size_t)C::kStages * C::kStageBytes;  // 1024-byte aligned
  uint32_t* sf = (uint32_t*)(stg + C::kBoxBytes);              // [slot][A 128 | W 256]
  int* tpre = (int*)(sf + C::kSfSlots * C::kSfSlotWords);      // [E + 1]
  int* cnt = tpre + kPersistMaxExperts + 1;                    // [E]
  uint64_t* full = (uint64_t*)(cnt + kPersistMaxExperts + 1);
  uint64_t* empty = full + C::kStages;
  uint64_t* sfull = empty + C::kStages;
  uint64_t* sempty = sfull + C::kSfSlots;
  uint64_t* sload = sempty + C::kSfSlots;  // packed activation words landed in the slot
  uint64_t* tfull = sload + C::kSfSlots;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
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
    for (int s = 0; s < C::kSfSlots; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 1);
      mbar_init(&sload[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, C::kEpiWarps);
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
  const int my_tiles =
      (int)blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      const int steps = my_tiles * KB;
      int g = 0, i = 0, t = blockIdx.x, a_row = 0, w_row = 0;
      for (; g < steps; ++g) {
        if (i == 0) {
          int e, m0, n0, ml;
          persist_tile<MASKED>(t, p, tpre, cnt, e, m0, n0, ml);
          a_row = (MASKED ? e * p.M : 0) + m0;
          w_row = (MASKED ? e * p.N : 0) + n0;
        }
        const int s = g % C::kStages;
        const uint32_t ph = (uint32_t)(g / C::kStages) & 1u;
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
        for (int j = g - C::kStages < 0 ? 0 : g - C::kStages; j < g; ++j) {
          volatile int no_abort = 0;
          (void)mbar_wait(&full[j % C::kStages], (uint32_t)(j / C::kStages) & 1u, &no_abort,
                          p.status, kWaitTimeoutNs / 8);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0) {
      int g = 0, q = 0;
      bool ok = true;
      for (int tt = 0; tt < my_tiles && ok; ++tt) {
        if (!mbar_wait(tempty, ((uint32_t)tt & 1u) ^ 1u, abort_flag, p.status, kWaitTimeoutNs))
          break;
        tc_fence_after_sync();
        uint32_t sfa = 0;
        for (int i = 0; i < KB; ++i, ++g) {
          if ((i & 3) == 0) {
            const int slot = q % C::kSfSlots;
            if (!mbar_wait(&sfull[slot], (uint32_t)(q / C::kSfSlots) & 1u, abort_flag, p.status,
                           kWaitTimeoutNs)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            sfa = tmem_base + C::kSfCol0 + (uint32_t)slot * C::kSfSlotCols;
            const uint32_t src = smem_u32(sf + slot * C::kSfSlotWords);
            tmem_cp_32x128b_x4(sfa, sdesc_rows16(src));                 // A rows 0-127
            tmem_cp_32x128b_x4(sfa + 4, sdesc_rows16(src + 512));       // W rows 0-127
            tmem_cp_32x128b_x4(sfa + 8, sdesc_rows16(src + 1024));      // W rows 128-255
          }
          const int s = g % C::kStages;
          if (!mbar_wait(&full[s], (uint32_t)(g / C::kStages) & 1u, abort_flag, p.status,
                         kWaitTimeoutNs)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + (size_t)s * C::kABytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + (size_t)s * C::kBBytes));
          const uint32_t idesc = idesc_e4m3_bs(kBM, BN, (uint32_t)(i & 3));
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            umma_e4m3_bs(tmem_base, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk),
                         idesc, sfa, sfa + 4, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
          if ((i & 3) == 3 || i == KB - 1) {
            umma_commit(&sempty[q % C::kSfSlots]);  // this group's scale slot is free
            ++q;
          }
        }
        if (!ok) break;
        umma_commit(tfull);
      }
      if (*abort_flag && g > 0) {
        // wait for the MMAs already issued before TMEM is released
        umma_commit(drain);
        volatile int no_abort = 0;
        (void)mbar_wait(drain, 0, &no_abort, p.status, kWaitTimeoutNs / 8);
      }
    }
  } else if (warp == 2) {
    // ------------------------------ scale loader ------------------------------
    // Group q = tile q / gpt, K blocks 4 (q mod gpt) .. + 3.  Its global
    // reads are started kAhead groups before it is written out.  Packed
    // activation words come by one bulk copy into the group's slot (row r at
    // word r) and are permuted in place when the group is written out; the
    // weight scales (2 blocks x 4 K blocks: 16 contiguous bytes per block
    // when K / 128 is a multiple of 4 and the array 16-byte aligned) by bulk
    // copies into the slot's last 8 words, read before the slot's weight
    // words are written.  Both wait for the slot to be free.  Otherwise
    // (fp32 power-of-two activation scales; weight scales not so aligned)
    // the values are loaded into registers.  Scale lines are pulled into L2
    // kPrefetchGroups ahead.
    constexpr int kAhead = 3;
    constexpr int kPrefetchGroups = 8;
    static_assert(kAhead < C::kSfSlots, "a copy lands in a slot the MMA has released");
    const int gpt = (KB + C::kGroup - 1) / C::kGroup;
    const int ngroups = my_tiles * gpt;
    const bool packed = p.a_fmt == BFQ_SCALE_UE8M0_PACKED;
    const bool wbulk = (KB & 3) == 0 && ((uintptr_t)p.sw & 15u) == 0;
    const bool bulk = packed || wbulk;  // the group's slot receives bulk copies
    const int nblks = (p.N + 127) / 128;
    bool bad = false;
    struct Coord {
      int tt = -1, e = 0, m0 = 0, n0 = 0, ml = 0;
    };
    // first K block of group q; c holds its tile's coordinates (cached)
    auto coord = [&](int q, Coord& c) -> int {
      const int tt = q / gpt;
      if (tt != c.tt) {
        c.tt = tt;
        persist_tile<MASKED>(blockIdx.x + tt * gridDim.x, p, tpre, cnt, c.e, c.m0, c.n0, c.ml);
      }
      return (q - tt * gpt) * C::kGroup;
    };
    auto sa_of = [&](const Coord& c) {
      return (const uint32_t*)p.sa + (MASKED ? (int64_t)c.e * p.sa_estride : 0);
    };
    auto sw_of = [&](const Coord& c) {
      return p.sw + (MASKED ? (int64_t)c.e * p.sw_estride : 0);
    };
    Coord c_pf, c_ld, c_em;
    auto prefetch_group = [&](int q) {
      const int i0 = coord(q, c_pf);
      const int nk = min(C::kGroup, KB - i0);
      const uint32_t* sa = sa_of(c_pf);
      if (packed) {
        // four 128-byte lines: rows 32 lane .. of the group's word column
        if (lane < 4 && c_pf.m0 + 32 * lane < c_pf.ml)
          prefetch_l2(sa + (int64_t)(i0 >> 2) * p.sa_ld + c_pf.m0 + 32 * lane);
      } else if (lane < 16 && (lane >> 2) < nk && c_pf.m0 + 32 * (lane & 3) < c_pf.ml) {
        prefetch_l2(sa + (int64_t)(i0 + (lane >> 2)) * p.sa_ld + c_pf.m0 + 32 * (lane & 3));
      }
      const int nb = c_pf.n0 / 128 + ((lane - 16) >> 2);
      if (lane >= 16 && lane < 24 && nb < nblks && (lane & 3) < nk)
        prefetch_l2(sw_of(c_pf) + (int64_t)nb * KB + i0 + (lane & 3));
    };
    struct Fetched {
      uint32_t a[16];  // fp32 power-of-two scales: a[4 c + k] = bits of row 32 c + lane, K block k
      uint32_t w;      // lane j < 8: fp32 bits of weight block n0 / 128 + j / 4, K block j % 4
    };
    int q_copied = 0;  // groups whose bulk copies were issued
    auto fetch = [&](int q, Fetched& f) -> bool {
      const int i0 = coord(q, c_ld);
      const int nk = min(C::kGroup, KB - i0);
      const uint32_t* sa = sa_of(c_ld);
      const float* sw = sw_of(c_ld);
      const int nb0 = c_ld.n0 / 128;
      if (!wbulk) {
        const int nb = nb0 + (lane >> 2), kb = i0 + (lane & 3);
        f.w = (lane < 8 && nb < nblks && kb < KB &&
               in_bounds(p.status, (sw - p.sw) + (int64_t)nb * KB + kb, 1, p.n_sw))
                  ? __float_as_uint(__ldg(sw + (int64_t)nb * KB + kb))
                  : 0x3F800000u;
      }
      if (!packed) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int m = c_ld.m0 + c * 32 + lane;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            f.a[4 * c + k] =
                (m < c_ld.ml && k < nk &&
                 in_bounds(p.status, (sa - (const uint32_t*)p.sa) + (int64_t)(i0 + k) * p.sa_ld + m,
                           1, p.n_sa))
                    ? __ldg(sa + (int64_t)(i0 + k) * p.sa_ld + m)
                    : 0x3F800000u;
        }
      }
      if (!bulk) return true;
      const int slot = q % C::kSfSlots;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&sempty[slot], ((uint32_t)(q / C::kSfSlots) & 1u) ^ 1u, abort_flag,
                       p.status, kWaitTimeoutNs);
        if (ok) {
          uint32_t* wa = sf + slot * C::kSfSlotWords;
          // rows m0 .. of the group's word column, not past the column's end
          uint32_t abytes = packed ? (uint32_t)min(kBM, (int)(p.sa_ld - c_ld.m0)) * 4u : 0u;
          int nbw = wbulk ? min(2, nblks - nb0) : 0;
          if (packed && !in_bounds(p.status,
                                   (sa - (const uint32_t*)p.sa) + (int64_t)(i0 >> 2) * p.sa_ld +
                                       c_ld.m0,
                                   abytes / 4, p.n_sa))
            abytes = 0;
          if (nbw > 0 && !in_bounds(p.status, (sw - p.sw) + (int64_t)nb0 * KB + i0,
                                    (int64_t)(nbw - 1) * KB + 4, p.n_sw))
            nbw = 0;
          mbar_arrive_expect_tx(&sload[slot], abytes + 16u * (uint32_t)nbw);
          if (abytes)
            bulk_load_1d(wa, sa + (int64_t)(i0 >> 2) * p.sa_ld + c_ld.m0, abytes, &sload[slot]);
          for (int h = 0; h < nbw; ++h)
            bulk_load_1d(wa + C::kSfSlotWords - 8 + 4 * h, sw + (int64_t)(nb0 + h) * KB + i0, 16u,
                         &sload[slot]);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      if (ok) q_copied = q + 1;
      return ok;
    };
    auto emit = [&](int q, const Fetched& f) -> bool {
      const int i0 = coord(q, c_em);
      const int nk = min(C::kGroup, KB - i0);
      const int slot = q % C::kSfSlots;
      const uint32_t ph = (uint32_t)(q / C::kSfSlots) & 1u;
      // lane 0 waits and the warp takes its decision together (the shuffles
      // below need every lane)
      bool ok = true;
      if (lane == 0)
        ok = bulk ? mbar_wait(&sload[slot], ph, abort_flag, p.status, kWaitTimeoutNs)
                  : mbar_wait(&sempty[slot], ph ^ 1u, abort_flag, p.status, kWaitTimeoutNs);
      if (!__shfl_sync(0xFFFFFFFFu, (int)ok, 0)) return false;
      __syncwarp();
      uint32_t* wa = sf + slot * C::kSfSlotWords;
      uint32_t* wb = wa + C::kSfaWords;
      // activation row 32 c + lane -> word 4 lane + c (the copy into TMEM
      // puts bytes 16 r + 4 c of the source at lane r, column c)
      uint32_t v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int m = c_em.m0 + c * 32 + lane;
        if (packed) {
          v[c] = m < c_em.ml ? wa[c * 32 + lane] : 0u;
        } else {
          v[c] = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t b = f.a[4 * c + k];
            bad |= !pow2_bits(b);
            v[c] |= k < nk ? ((b >> 23) & 0xFFu) << (8 * k) : 0u;
          }
        }
      }
      // lane j < 8: fp32 bits of weight block n0 / 128 + j / 4, K block j % 4
      // (a block past N keeps the value 1.0, unused)
      uint32_t w = f.w;
      if (wbulk)
        w = (lane < 8 && c_em.n0 / 128 + (lane >> 2) < nblks) ? wb[C::kSfbWords - 8 + lane]
                                                             : 0x3F800000u;
      __syncwarp();  // every copied word is read before any is overwritten
#pragma unroll
      for (int c = 0; c < 4; ++c) wa[lane * 4 + c] = v[c];
      // weight rows: one word per 128-row block, the same for all its rows
      if (lane < 8) bad |= !pow2_bits(w);
      uint32_t wv0 = 0, wv1 = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, w, k);
        const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, w, 4 + k);
        if (k < nk) {
          wv0 |= ((b0 >> 23) & 0xFFu) << (8 * k);
          wv1 |= ((b1 >> 23) & 0xFFu) << (8 * k);
        }
      }
#pragma unroll
      for (int j = 0; j < C::kSfbWords / 32; ++j) wb[lane + 32 * j] = j < 4 ? wv0 : wv1;
      fence_proxy_async_smem();  // visible to the tensor cores' copy
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfull[slot]);
      return true;
    };
    Fetched f[kAhead + 1];
    bool stop = false;
    int q_emitted = 0;
    for (int q = 0; q < kPrefetchGroups && q < ngroups; ++q) prefetch_group(q);
#pragma unroll
    for (int d = 0; d < kAhead; ++d)
      if (!stop && d < ngroups) stop = !fetch(d, f[d]);
    for (int q0 = 0; q0 < ngroups && !stop; q0 += kAhead + 1) {
#pragma unroll
      for (int d = 0; d <= kAhead; ++d) {
        const int q = q0 + d;
        if (stop || q >= ngroups) continue;
        if (q + kPrefetchGroups < ngroups) prefetch_group(q + kPrefetchGroups);
        if (q + kAhead < ngroups)
          stop = !fetch(q + kAhead, f[(d + kAhead) % (kAhead + 1)]);
        if (!stop) {
          stop = !emit(q, f[d]);
          if (!stop) q_emitted = q + 1;
        }
      }
    }
    if (stop && lane == 0) {
      // let the bulk copies already issued land before the CTA can exit
      for (int q = q_emitted; q < q_copied; ++q) {
        volatile int no_abort = 0;
        (void)mbar_wait(&sload[q % C::kSfSlots], (uint32_t)(q / C::kSfSlots) & 1u, &no_abort,
                        p.status, kWaitTimeoutNs / 8);
      }
    }
    if (bad) atomicCAS(p.status, 0, BFQ_ERR_FORMAT);
  } else if (warp >= C::kEpiWarp0) {
    // -------------------------------- epilogue --------------------------------
    const int ew = warp - C::kEpiWarp0;
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int half = ew >> 2;      // accumulator columns 128*half .. +127
    const int row_local = quarter * 32 + lane;
    const bool store_thread = threadIdx.x == C::kEpiWarp0 * 32;
    const int tid = (int)threadIdx.x - C::kEpiWarp0 * 32;
    for (int tt = 0; tt < my_tiles; ++tt) {
      int e, m0, n0, m_limit;
      persist_tile<MASKED>(blockIdx.x + tt * gridDim.x, p, tpre, cnt, e, m0, n0, m_limit);
      const int col0 = n0 + half * 128;
      const bool warp_active = (m0 + quarter * 32 < m_limit) && (SILU || col0 < p.N);
      const int ncols = min(128, p.N - col0);
      uint64_t lo[32], hi[32];  // SILU: lo = 64 gate columns, hi = the matching up columns
      const bool stop = !mbar_wait(tfull, (uint32_t)tt & 1u, abort_flag, p.status,
                                   kWaitTimeoutNs);
      if (!stop) {
        tc_fence_after_sync();
        if (warp_active) {
          const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                 (uint32_t)(half * (SILU ? 64 : 128));
          tmem_ld64_pairs_wait(taddr, lo);
          tmem_ld64_pairs_wait(taddr + (SILU ? 128u : 64u), hi);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty);  // the next tile's MMAs may start
      }
      if (named_barrier_or(2, C::kEpiWarps * 32, stop || *abort_flag)) break;
      if constexpr (SILU) {
        silu_quant_tile_rows<C::kEpiWarps * 32>(p, lo, hi, (float*)stg, e, m0 + row_local, n0,
                                                half, row_local,
                                                warp_active && m0 + row_local < m_limit);
        continue;
      }

      // Box b (columns 64 b .. 64 b + 63 of the tile) is held by warp half
      // b / 2 (lo or hi); staged as bf16 in the 128-byte swizzled layout:
      // 16-byte chunk c of row r at chunk c ^ (r mod 8).
      for (int b = 0; b < BN / 64; ++b) {
        if (n0 + b * 64 >= p.N) break;
        if (!MASKED && store_thread) bulk_wait_read_all();  // the last box has left
        named_barrier(1, C::kEpiWarps * 32);
        if (half == (b >> 1) && warp_active && (b & 1) * 64 < ncols) {
          const uint64_t* v = (b & 1) ? hi : lo;
          const uint32_t row_addr = smem_u32(stg) + (uint32_t)(row_local * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float2 f0 = unpack2(v[c * 4 + 0]), f1 = unpack2(v[c * 4 + 1]);
            const float2 f2 = unpack2(v[c * 4 + 2]), f3 = unpack2(v[c * 4 + 3]);
            st_shared_v4(row_addr + (uint32_t)((c ^ (row_local & 7)) << 4),
                         make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f1.x, f1.y),
                                    pack_bf16x2(f2.x, f2.y), pack_bf16x2(f3.x, f3.y)));
          }
        }
        if (!MASKED) fence_proxy_async_smem();
        named_barrier(1, C::kEpiWarps * 32);
        if (!MASKED) {
          // rows >= M are clipped by the tensor map
          if (store_thread) {
            tma_store_2d(&tmO, stg, n0 + b * 64, m0);
            bulk_commit();
          }
        } else {
          // rows past the count must not be written: copy the valid rows of
          // the box with 16-byte stores, eight lanes per 128-byte row segment
          const int rows_valid = min(kBM, m_limit - m0);
          __nv_bfloat16* base =
              p.out + (int64_t)e * p.out_estride + (int64_t)m0 * p.N + n0 + b * 64;
          const uint32_t box = smem_u32(stg);
          for (int x = tid; x < rows_valid * 8; x += C::kEpiWarps * 32) {
            const int r = x >> 3, c = x & 7;
            if (in_bounds(p.status, (base - p.out) + (int64_t)r * p.N + c * 8, 8, p.n_out))
              st_v4(base + (int64_t)r * p.N + c * 8,
                    ld_shared_v4(box + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4))));
          }
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
template <bool MASKED, bool SILU = false>
bfq_status configure_bs(const DeviceInfo& dev) {
  static bool configured[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (configured[dev.ordinal]) return BFQ_OK;
  if (cudaFuncSetAttribute(gemm_block_fp8_bs<MASKED, SILU>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)BsCfg::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return BFQ_ERR_CUDA;
  }
  configured[dev.ordinal] = true;
  return BFQ_OK;
}

bfq_status check_device_bs(DeviceInfo* dev) {
  bfq_status st = current_device(dev);
  if (st != BFQ_OK) return st;
  if (dev->cc_major != 10 || dev->smem_optin < BsCfg::kSmemBytes) return BFQ_ERR_DEVICE;
  return BFQ_OK;
}

bool pow2_fmt(int32_t fmt) {
  return fmt == BFQ_SCALE_UE8M0_PACKED || fmt == BFQ_SCALE_F32_POW2;
}

template <bool MASKED, bool SILU = false>
bfq_status launch_bs(const DeviceInfo& dev, const CUtensorMap& ma, const CUtensorMap& mw,
                     const CUtensorMap& mo, const GemmParams& p, int64_t tiles,
                     cudaStream_t s) {
  bfq_status st = configure_bs<MASKED, SILU>(dev);
  if (st != BFQ_OK) return st;
  const unsigned grid = (unsigned)(tiles < dev.sm_count ? tiles : dev.sm_count);
  return launch_status(launch_pdl(gemm_block_fp8_bs<MASKED, SILU>, dim3(grid),
                                  dim3(BsCfg::kThreads), BsCfg::kSmemBytes, s, 1u, ma, mw, mo,
                                  p));
}

}  // namespace
}  // namespace bfq

using namespace bfq;

extern "C" bfq_status bfq_gemm_block_fp8_ue8m0(const void* a_q, const void* a_scales,
                                               int32_t a_fmt, int64_t a_scale_ld,
                                               const void* w_q, const float* w_scales,
                                               int64_t M, int64_t N, int64_t K, void* out,
                                               void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || !valid_fmt(a_fmt) || a_scale_ld < M)
    return BFQ_ERR_INVALID_ARG;
  if (!pow2_fmt(a_fmt)) return BFQ_ERR_FORMAT;
  if (K % 128 != 0 || N % 64 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BFQ_OK;
  if (!a_q || !a_scales || !w_q || !w_scales || !out) return BFQ_ERR_INVALID_ARG;
  if (!aligned16(a_q) || !aligned16(w_q) || !aligned16(out) || a_scale_ld % 4 != 0 ||
      ((uintptr_t)a_scales & 3u) || ((uintptr_t)w_scales & 3u) ||
      (a_fmt == BFQ_SCALE_UE8M0_PACKED && !aligned16(a_scales)))
    return BFQ_ERR_MISALIGNED;
  DeviceInfo dev;
  bfq_status st = check_device_bs(&dev);
  if (st != BFQ_OK) return st;
  // Launch plan: with one row tile, K < 1024 or fewer than half as many
  // tiles as SMs the promotion kernel's plan (K split over a cluster,
  // double-buffered accumulators) is faster (measured); it computes the same
  // result.
  const int64_t tiles = cdiv(M, kBM) * cdiv(N, BsCfg::kBN);
  if (M <= kBM || K < 1024 || 2 * tiles < dev.sm_count)
    return bfq_gemm_block_fp8(a_q, a_scales, a_fmt, a_scale_ld, w_q, w_scales, M, N, K, out,
                              nullptr, 0, stream);
  CUtensorMap ma, mw, mo;
  if (!make_map(&ma, a_q, (uint64_t)K, (uint64_t)M, kBM) ||
      !make_map(&mw, w_q, (uint64_t)K, (uint64_t)N, (uint32_t)BsCfg::kBN) ||
      !make_out_map(&mo, out, (uint64_t)N, (uint64_t)M))
    return BFQ_ERR_CUDA;
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
  p.m_tiles = (int)cdiv(M, kBM);
  p.n_tiles = (int)cdiv(N, BsCfg::kBN);
  p.splits = 1;
  p.a_fmt = a_fmt;
  p.n_sa = scale_cols(K, a_fmt) * a_scale_ld;
  p.n_sw = cdiv(N, 128) * (K / 128);
  p.n_out = M * N;
  return launch_bs<false>(dev, ma, mw, mo, p, (int64_t)p.m_tiles * p.n_tiles,
                          (cudaStream_t)stream);
}

extern "C" bfq_status bfq_gemm_block_fp8_masked_ue8m0(
    const void* a_q, const void* a_scales, int32_t a_fmt, int64_t a_scale_ld, const void* w_q,
    const float* w_scales, const int32_t* valid_counts, int32_t E, int32_t T, int64_t N,
    int64_t K, void* out, void* stream) {
  if (E < 0 || T < 0 || N <= 0 || K <= 0 || !valid_fmt(a_fmt) || a_scale_ld < T)
    return BFQ_ERR_INVALID_ARG;
  if (!pow2_fmt(a_fmt)) return BFQ_ERR_FORMAT;
  if (K % 128 != 0 || N % 64 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)E * T > 0x7FFFFFFF || (int64_t)E * N > 0x7FFFFFFF || K > 0x7FFFFFFF)
    return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (E > kPersistMaxExperts) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (E == 0 || T == 0) return BFQ_OK;
  if (!a_q || !a_scales || !w_q || !w_scales || !valid_counts || !out)
    return BFQ_ERR_INVALID_ARG;
  if (!aligned16(a_q) || !aligned16(w_q) || !aligned16(out) || a_scale_ld % 4 != 0 ||
      ((uintptr_t)a_scales & 3u) || ((uintptr_t)w_scales & 3u) ||
      (a_fmt == BFQ_SCALE_UE8M0_PACKED && !aligned16(a_scales)))
    return BFQ_ERR_MISALIGNED;
  DeviceInfo dev;
  bfq_status st = check_device_bs(&dev);
  if (st != BFQ_OK) return st;
  CUtensorMap ma, mw;
  if (!make_map(&ma, a_q, (uint64_t)K, (uint64_t)E * T, kBM) ||
      !make_map(&mw, w_q, (uint64_t)K, (uint64_t)E * N, (uint32_t)BsCfg::kBN))
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
  p.n_tiles = (int)cdiv(N, BsCfg::kBN);
  p.splits = 1;
  p.a_fmt = a_fmt;
  p.E = E;
  p.n_sa = E * p.sa_estride;
  p.n_sw = E * p.sw_estride;
  p.n_out = (int64_t)E * T * N;
  return launch_bs<true>(dev, ma, mw, mw, p, (int64_t)p.m_tiles * p.n_tiles * E,
                         (cudaStream_t)stream);
}

extern "C" bfq_status bfq_gemm_block_fp8_masked_silu_quant_ue8m0(
    const void* a_q, const void* a_scales, int32_t a_fmt, int64_t a_scale_ld, const void* w_q,
    const float* w_scales, const int32_t* valid_counts, int32_t E, int32_t T, int64_t I,
    int64_t K, int32_t q_fmt, void* q_out, void* q_scales, int64_t q_scale_ld, void* stream) {
  if (E < 0 || T < 0 || I <= 0 || K <= 0 || !valid_fmt(a_fmt) || !valid_fmt(q_fmt) ||
      a_scale_ld < T || q_scale_ld < T)
    return BFQ_ERR_INVALID_ARG;
  if (!pow2_fmt(a_fmt)) return BFQ_ERR_FORMAT;
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
      ((uintptr_t)q_scales & 3u) || (a_fmt == BFQ_SCALE_UE8M0_PACKED && !aligned16(a_scales)))
    return BFQ_ERR_MISALIGNED;
  DeviceInfo dev;
  bfq_status st = check_device_bs(&dev);
  if (st != BFQ_OK) return st;
  CUtensorMap ma, mw;
  if (!make_map(&ma, a_q, (uint64_t)K, (uint64_t)E * T, kBM) ||
      !make_map(&mw, w_q, (uint64_t)K, (uint64_t)E * N, (uint32_t)BsCfg::kBN))
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
  p.n_tiles = (int)(N / BsCfg::kBN);
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
  return launch_bs<true, true>(dev, ma, mw, mw, p, (int64_t)p.m_tiles * p.n_tiles * E,
                               (cudaStream_t)stream);
}
