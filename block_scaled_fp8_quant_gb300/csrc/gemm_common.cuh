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
  // extents of the arrays, in their elements (32-bit scale words / floats,
  // bf16 outputs, e4m3 codes), for the debug build's bounds checks
  int64_t n_sa, n_sw, n_out, n_q, n_qs;
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

// Fused silu(gate) * up + 1 x 128 group quant of one output tile's features,
// exactly as the silu-mul-quant kernel computes them from the bf16
// up-projection output ("[EP+DP] Optimize the little operations in the
// DeepGEMM + DeepEP low latency case", Summary item 2): a 256-wide tile of
// the interleaved up projection holds gate block n0 / 256 (columns 0-127)
// and the matching up block (128-255).  Each thread holds, for its row, the
// fp32 accumulators of 64 gate features g[] and the same 64 up features u[]
// (features 64 half .. + 63, as 32 pairs each).  Gate and up are rounded to
// bf16, y = silu(g) * u in fp32 (silu looked up in the library's table of
// all bf16 gates, or computed while a graph is captured before the table
// exists — the same values), group amax over the 128 features (the two
// halves exchanged through xam, shared float[2][128]), scale, codes.  y
// overwrites g.  Called by all kNT epilogue threads (named barrier 1);
// active = the row is valid and the thread's warp holds data.
template <int kNT>
__device__ __forceinline__ void silu_quant_tile_rows(const GemmParams& p, uint64_t* g,
                                                     const uint64_t* u, float* xam, int e, int m,
                                                     int n0, int half, int row_local,
                                                     bool active) {
  float amax = 0.0f;
  if (active) {  // rows past the count: nothing to form
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float2 gf = unpack2(g[j]), uf = unpack2(u[j]);
      const uint32_t gb = pack_bf16x2(gf.x, gf.y), ub = pack_bf16x2(uf.x, uf.y);
      const float2 sg = p.silu_tab ? make_float2(__ldg(p.silu_tab + (gb & 0xFFFFu)),
                                                 __ldg(p.silu_tab + (gb >> 16)))
                                   : bfq_silu2(bf16lo(gb), bf16hi(gb));
      const float2 y = unpack2(mul2_rn(pack2(sg.x, sg.y), pack2(bf16lo(ub), bf16hi(ub))));
      g[j] = pack2(y.x, y.y);
      amax = fmaxf(amax, fmaxf(fabsf(y.x), fabsf(y.y)));
    }
  }
  xam[half * kBM + row_local] = amax;  // partial amax per half and row
  named_barrier(1, kNT);
  amax = fmaxf(xam[row_local], xam[kBM + row_local]);
  named_barrier(1, kNT);  // both read before the next tile writes
  if (!active) return;
  const int I = p.N >> 1;
  const int fg = n0 >> 8;  // 128-feature group of this tile
  float sc = __fdiv_rn(fmaxf(amax, kEps), kFp8Max);
  if (p.q_fmt != BFQ_SCALE_F32) sc = ceil_pow2(sc);
  const float y_inv = __frcp_rn(sc);
  const int64_t qoff = ((int64_t)e * p.M + m) * I + fg * 128 + half * 64;
  uint8_t* qrow = p.q_out + qoff;
  const bool q_ok = in_bounds(p.status, qoff, 64, p.n_q);
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // 16 codes per 16-byte store
    uint32_t w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 y0 = unpack2(g[c * 8 + 2 * t]), y1 = unpack2(g[c * 8 + 2 * t + 1]);
      uint32_t lo, hi;
      if (p.q_fmt == BFQ_SCALE_F32) {
        lo = cvt_e4m3x2(group_div(y0.x, sc, y_inv), group_div(y0.y, sc, y_inv));
        hi = cvt_e4m3x2(group_div(y1.x, sc, y_inv), group_div(y1.y, sc, y_inv));
      } else {
        lo = cvt_e4m3x2(__fmul_rn(y0.x, y_inv), __fmul_rn(y0.y, y_inv));
        hi = cvt_e4m3x2(__fmul_rn(y1.x, y_inv), __fmul_rn(y1.y, y_inv));
      }
      w[t] = lo | (hi << 16);
    }
    if (q_ok) st_v4(qrow + c * 16, make_uint4(w[0], w[1], w[2], w[3]));
  }
  if (half == 0) {
    const int G = I >> 7;
    if (p.q_fmt == BFQ_SCALE_UE8M0_PACKED) {
      const int64_t cols = (G + 3) >> 2;
      const int64_t woff = ((int64_t)e * cols + (fg >> 2)) * p.q_scale_ld + m;
      if (in_bounds(p.status, woff, 1, p.n_qs)) {
        uint8_t* word = (uint8_t*)p.q_scales + woff * 4;
        word[fg & 3] = (uint8_t)ue8m0_byte(sc);
        if (fg == G - 1)
          for (int b = (fg & 3) + 1; b < 4; ++b) word[b] = 0;
      }
    } else {
      const int64_t soff = ((int64_t)e * G + fg) * p.q_scale_ld + m;
      if (in_bounds(p.status, soff, 1, p.n_qs)) ((float*)p.q_scales)[soff] = sc;
    }
  }
}

}  // namespace bfq
