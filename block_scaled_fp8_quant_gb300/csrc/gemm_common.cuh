// gemm_common.cuh — tile constants, kernel parameters and the persistent
// tile walk shared by the GEMM translation units.
#pragma once

#include "bfq_device.cuh"

namespace bfq {

constexpr int kBM = 128;  // rows of A per tile (UMMA M)
constexpr int kBK = 128;  // K per stage = one scale block
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s
constexpr int kMaxSplits = 8;  // K splits of a tile form one (portable-size) cluster

// Most experts the persistent masked kernels take (their per-expert tile
// prefix sums live in shared memory).
constexpr int kPersistMaxExperts = 1024;

struct GemmParams {
  const void* sa;          // activation scales (format a_fmt), column-major
  int64_t sa_ld;           // leading dimension of sa
  int64_t sa_estride;      // elements of sa per expert (masked)
  const float* sw;         // weight scales [nblk][KB]
  int64_t sw_estride;      // floats of sw per expert (masked)
  __nv_bfloat16* out;      // [rows][N]
  int64_t out_estride;     // elements of out per expert (masked)
  const int32_t* counts;   // masked: per-expert valid rows
  int* status;             // device error latch
  int M;                   // dense: rows of A; masked: rows per expert (T)
  int N, K;
  int m_tiles, n_tiles, splits;
  int a_fmt;
  int E;                   // masked: experts
  // fused output quant (QOUT kernels): the bf16-rounded output quantized per
  // 1 x 128 group into q_out (e4m3 [M][N]) and q_scales (format q_fmt,
  // column-major, leading dimension q_scale_ld); out may then be null.
  uint8_t* q_out;
  void* q_scales;
  int64_t q_scale_ld;
  int q_fmt;
  // fused silu-mul-quant (SILU kernel): silu of every bf16 gate, indexed by
  // its 16 bits (the library's table), or null to compute it
  const float* silu_tab;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Tile t of the persistent schedule -> (expert, first row, first column,
// valid rows of the expert).  Masked: tpre[e] = tiles of experts < e,
// cnt[e] = clamped valid rows of expert e.
template <bool MASKED>
__device__ __forceinline__ void persist_tile(int t, const GemmParams& p, const int* tpre,
                                             const int* cnt, int& e, int& m0, int& n0,
                                             int& m_limit) {
  if (MASKED) {
    int lo = 0, hi = p.E;  // tpre[lo] <= t < tpre[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tpre[mid] <= t) lo = mid;
      else hi = mid;
    }
    e = lo;
    m_limit = cnt[e];
    const int a = (m_limit + kBM - 1) / kBM;  // active row tiles of expert e
    const int r = t - tpre[e];
    const int nt = r / a;
    m0 = (r - nt * a) * kBM;
    n0 = nt * 256;
  } else {
    e = 0;
    m_limit = p.M;
    const int nt = t / p.m_tiles;
    m0 = (t - nt * p.m_tiles) * kBM;
    n0 = nt * 256;
  }
}

// Masked persistent kernels, all threads of the CTA: cnt[e] = expert e's
// valid rows clamped to [0, T] and tpre[e] = tiles of experts < e (exclusive
// prefix sum of ceil(cnt / 128) * n_tiles, tpre[E] = all tiles), in shared
// memory.  Waits for the previous grid first (the counts may come from it).
// The caller synchronizes the CTA before reading tpre.
__device__ __forceinline__ void masked_tile_prefix(const GemmParams& p, int* tpre, int* cnt) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  for (int x = threadIdx.x; x < p.E; x += blockDim.x) {
    int c = __ldg(p.counts + x);
    c = c < 0 ? 0 : (c > p.M ? p.M : c);
    cnt[x] = c;
    tpre[x + 1] = (c + kBM - 1) / kBM * p.n_tiles;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (p.E + 31) / 32;
    const int b = lane * per;
    const int b_end = min(p.E, b + per);
    int sum = 0;
    for (int x = b; x < b_end; ++x) sum += tpre[x + 1];
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= o) inc += y;
    }
    int run = inc - sum;
    for (int x = b; x < b_end; ++x) {
      run += tpre[x + 1];
      tpre[x + 1] = run;
    }
    if (lane == 0) tpre[0] = 0;
  }
}

}  // namespace bfq
