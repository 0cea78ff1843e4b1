// quant_kernels.cu — bandwidth-bound kernels of the block-FP8 path:
//   * per-token-group (1 x 128) activation quant, three scale formats, packed
//     UE8M0 words assembled in registers ("[Perf] Deepgemm fused layout kernel
//     for activations", Purpose: pack scales into a uint32 early and remove
//     the extra layout kernel);
//   * fused silu(gate) * up + quant over a masked per-expert batch
//     ("[EP+DP] Optimize the little operations in the DeepGEMM + DeepEP low
//     latency case", Summary item 2: padded tokens neither loaded nor
//     computed);
//   * 128 x 128 block weight quant ("vLLM DeepGEMM FP8 Block GEMM 基准测试"
//     §4.1, per_block_cast_to_fp8).
//
// Work unit of the activation kernels: one warp quantizes a 512-element chunk
// of one row (four 128-element groups, i.e. one packed scale word).  Lane l
// owns elements [16 l, 16 l + 16) and group l / 8; the 8 lanes of a group
// reduce their amax with three xor-shuffles.  Loads are 16-byte, coalesced
// (a warp reads 1 KiB of bf16 contiguous memory per unit) and bypass L1.
#include <map>
#include <mutex>

#include "bfq_device.cuh"

namespace bfq {

constexpr int kQuantWarps = 8;  // warps per block
constexpr int kUnroll = 1;      // units per warp and loop iteration

// Quantize the lane's 16 values of one group.  `gactive` says whether this
// lane's group exists (partial last chunk).  Returns the group's scale (all 8
// lanes of the group hold it) and writes 16 codes as one uint4.
template <int FMT>
__device__ __forceinline__ float quant16(const float (&v)[16], uint4& codes) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
  float s = __fdiv_rn(fmaxf(amax, kEps), kFp8Max);
  uint32_t c[8];
  // The quotients are formed two at a time with packed f32x2 operations; each
  // lane of a pair is rounded exactly as the scalar operation, so the codes
  // are those of group_div (fp32 scales) and of one multiply (powers of two).
  if (FMT == BFQ_SCALE_F32) {
    const float y = __frcp_rn(s);
    const uint64_t y2 = splat2(y), neg_s2 = splat2(-s);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t a = pack2(v[2 * i], v[2 * i + 1]);
      const uint64_t q0 = mul2_rn(a, y2);
      const uint64_t r = fma2_rn(q0, neg_s2, a);  // fma(-q0, s, a), exactly
      const float2 q = unpack2(fma2_rn(r, y2, q0));
      c[i] = cvt_e4m3x2(copysignf(q.x, v[2 * i]), copysignf(q.y, v[2 * i + 1]));
    }
  } else {
    s = ceil_pow2(s);
    const uint64_t y2 = splat2(__frcp_rn(s));  // exact: s is a power of two
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 q = unpack2(mul2_rn(pack2(v[2 * i], v[2 * i + 1]), y2));
      c[i] = cvt_e4m3x2(q.x, q.y);
    }
  }
  codes.x = c[0] | (c[1] << 16);
  codes.y = c[2] | (c[3] << 16);
  codes.z = c[4] | (c[5] << 16);
  codes.w = c[6] | (c[7] << 16);
  return s;
}

// Write the scales of one chunk (4 groups) of row r.  Lanes 0, 8, 16, 24
// hold the scales of groups 0..3 of the chunk.
// (status, base_off, n_s: the debug build's bounds check of the scale
// array, base_off = the offset of `scales` within it.)
template <int FMT>
__device__ __forceinline__ void store_chunk_scales(float s, bool gactive, int lane,
                                                   int64_t chunk, int64_t r, void* scales,
                                                   int64_t ld, int* status, int64_t base_off,
                                                   int64_t n_s) {
  if (FMT == BFQ_SCALE_UE8M0_PACKED) {
    uint32_t b = gactive ? ue8m0_byte(s) : 0u;
    uint32_t b0 = __shfl_sync(0xFFFFFFFFu, b, 0);
    uint32_t b1 = __shfl_sync(0xFFFFFFFFu, b, 8);
    uint32_t b2 = __shfl_sync(0xFFFFFFFFu, b, 16);
    uint32_t b3 = __shfl_sync(0xFFFFFFFFu, b, 24);
    if (lane == 0 && in_bounds(status, base_off + chunk * ld + r, 1, n_s))
      ((uint32_t*)scales)[chunk * ld + r] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
  } else {
    const int64_t off = (chunk * 4 + (lane >> 3)) * ld + r;
    if (gactive && (lane & 7) == 0 && in_bounds(status, base_off + off, 1, n_s))
      ((float*)scales)[off] = s;
  }
}

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float (&v)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
}

// ---------------------------------------------------------------------------
// per-token-group quant
// ---------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quant_kernel(const __nv_bfloat16* __restrict__ x, int64_t M, int64_t K, int64_t ld_x,
                 uint8_t* __restrict__ q, void* __restrict__ scales, int64_t scale_ld,
                 int* status, int64_t n_x, int64_t n_s) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t G = K / 128;
  const int64_t chunks = (G + 3) / 4;
  const int64_t units = M * chunks;
  const int64_t warp0 = ((int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5)) * kUnroll;
  const int64_t stride = (int64_t)gridDim.x * kQuantWarps * kUnroll;
  const int gl = lane >> 3;  // group of this lane within the chunk

  for (int64_t u0 = warp0; u0 < units; u0 += stride) {
    uint4 raw[kUnroll][2];
    bool act[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int64_t u = u0 + j;
      const int64_t r = u / chunks, c = u - (u / chunks) * chunks;
      act[j] = (u < units) && (c * 4 + gl < G) &&
               in_bounds(status, r * ld_x + c * 512 + lane * 16, 16, n_x);
      if (act[j]) {
        const __nv_bfloat16* p = x + r * ld_x + c * 512 + lane * 16;
        raw[j][0] = ld_stream_v4(p);
        raw[j][1] = ld_stream_v4(p + 8);
      } else {
        raw[j][0] = make_uint4(0, 0, 0, 0);
        raw[j][1] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int64_t u = u0 + j;
      if (u >= units) break;  // warp-uniform
      const int64_t r = u / chunks, c = u - (u / chunks) * chunks;
      float v[16];
      unpack16(raw[j][0], raw[j][1], v);
      uint4 codes;
      const float s = quant16<FMT>(v, codes);
      if (act[j] && in_bounds(status, r * K + c * 512 + lane * 16, 16, M * K))
        st_v4(q + r * K + c * 512 + lane * 16, codes);
      store_chunk_scales<FMT>(s, act[j], lane, c, r, scales, scale_ld, status, 0, n_s);
    }
  }
}

// ---------------------------------------------------------------------------
// fused silu-and-mul + quant over a masked per-expert batch
// ---------------------------------------------------------------------------
// The gate is a bf16 value, so silu takes one of 65536 inputs: the library
// evaluates bfq_silu for every one of them once per device into this table
// (indexed by the gate's 16 bits), and the kernel looks silu up instead of
// spending ~40 instructions per element on the exp polynomial and the IEEE
// division.  The values are those of bfq_silu bit for bit.
__device__ float g_silu_table[65536];

__global__ void __launch_bounds__(256) silu_table_kernel(float* __restrict__ table) {
  const int i = blockIdx.x * 256 + threadIdx.x;
  table[i] = bfq_silu(__uint_as_float((uint32_t)i << 16));
}

// Two rows per block and one unit in flight per warp: small blocks keep more
// warps resident and spread the valid rows evenly over the SMs.  TABLE:
// silu by table lookup; otherwise computed (the same values).
constexpr int kSiluRowsPerBlock = 2;
constexpr int kSiluUnroll = 1;

template <int FMT, bool TABLE>
__global__ void __launch_bounds__(kQuantWarps * 32)
    silu_mul_quant_kernel(const __nv_bfloat16* __restrict__ x, int T, int I,
                          const int32_t* __restrict__ counts, uint8_t* __restrict__ q,
                          void* __restrict__ scales, int64_t scale_ld,
                          const float* __restrict__ silu_tab, int* status, int64_t n_x,
                          int64_t n_s) {
  griddep_wait();
  griddep_launch_dependents();
  const int e = blockIdx.y;
  int cnt = __ldg(counts + e);
  cnt = cnt < 0 ? 0 : (cnt > T ? T : cnt);
  const int r0 = blockIdx.x * kSiluRowsPerBlock;
  if (r0 >= cnt) return;  // padded rows: nothing is read or written
  const int rows = min(kSiluRowsPerBlock, cnt - r0);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int G = I / 128;
  const int chunks = (G + 3) / 4;
  const int units = rows * chunks;
  const int gl = lane >> 3;
  const int64_t cols = (FMT == BFQ_SCALE_UE8M0_PACKED) ? chunks : G;
  void* sc_e = (FMT == BFQ_SCALE_UE8M0_PACKED)
                   ? (void*)((uint32_t*)scales + (int64_t)e * cols * scale_ld)
                   : (void*)((float*)scales + (int64_t)e * cols * scale_ld);

  for (int u0 = warp * kSiluUnroll; u0 < units; u0 += kQuantWarps * kSiluUnroll) {
    uint4 raw[kSiluUnroll][4];
    bool act[kSiluUnroll];
#pragma unroll
    for (int j = 0; j < kSiluUnroll; ++j) {
      const int u = u0 + j;
      const int r = r0 + u / chunks, c = u % chunks;
      act[j] = (u < units) && (c * 4 + gl < G) &&
               in_bounds(status,
                         ((int64_t)e * T + r) * (2 * (int64_t)I) + c * 512 + lane * 16 + I, 16,
                         n_x);
      if (act[j]) {
        const __nv_bfloat16* p = x + ((int64_t)e * T + r) * (2 * (int64_t)I) + c * 512 + lane * 16;
        raw[j][0] = ld_stream_v4(p);
        raw[j][1] = ld_stream_v4(p + 8);
        raw[j][2] = ld_stream_v4(p + I);
        raw[j][3] = ld_stream_v4(p + I + 8);
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) raw[j][t] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int j = 0; j < kSiluUnroll; ++j) {
      const int u = u0 + j;
      if (u >= units) break;
      const int r = r0 + u / chunks, c = u % chunks;
      float g[16], up[16], y[16];
      unpack16(raw[j][0], raw[j][1], g);
      unpack16(raw[j][2], raw[j][3], up);
      const uint32_t gw[8] = {raw[j][0].x, raw[j][0].y, raw[j][0].z, raw[j][0].w,
                              raw[j][1].x, raw[j][1].y, raw[j][1].z, raw[j][1].w};
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        float2 sg;
        if constexpr (TABLE) {
          sg.x = __ldg(silu_tab + (gw[i / 2] & 0xFFFFu));
          sg.y = __ldg(silu_tab + (gw[i / 2] >> 16));
        } else {
          sg = bfq_silu2(g[i], g[i + 1]);
        }
        const float2 yy = unpack2(mul2_rn(pack2(sg.x, sg.y), pack2(up[i], up[i + 1])));
        y[i] = yy.x;
        y[i + 1] = yy.y;
      }
      uint4 codes;
      const float s = quant16<FMT>(y, codes);
      const int64_t qoff = ((int64_t)e * T + r) * I + c * 512 + lane * 16;
      if (act[j] && in_bounds(status, qoff, 16, n_x / 2)) st_v4(q + qoff, codes);
      store_chunk_scales<FMT>(s, act[j], lane, c, r, sc_e, scale_ld, status,
                              (int64_t)e * cols * scale_ld, n_s);
    }
  }
}

// ---------------------------------------------------------------------------
// 128 x 128 block weight quant: one block of 256 threads per weight block;
// thread t owns row t/2, columns [64 (t%2), 64 (t%2) + 64) of the block.
// ---------------------------------------------------------------------------
template <bool POW2>
__global__ void __launch_bounds__(256)
    weight_quant_kernel(const __nv_bfloat16* __restrict__ w, int64_t N, int64_t K,
                        uint8_t* __restrict__ wq, float* __restrict__ sw, int* status,
                        int64_t n_w, int64_t n_s) {
  __shared__ float red[8];
  griddep_wait();
  griddep_launch_dependents();
  const int64_t NB = (N + 127) / 128, KB = K / 128;
  const int64_t nb = blockIdx.y, kb = blockIdx.x, b = blockIdx.z;
  const int t = threadIdx.x;
  const int64_t n = nb * 128 + (t >> 1);
  const bool row_ok = n < N && in_bounds(status, (b * N + n) * K + kb * 128 + (t & 1) * 64, 64, n_w);
  const __nv_bfloat16* src = w + (b * N + n) * K + kb * 128 + (t & 1) * 64;
  uint4 raw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    raw[i] = row_ok ? ld_stream_v4(src + 8 * i) : make_uint4(0, 0, 0, 0);
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t ww[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      amax = fmaxf(amax, fmaxf(fabsf(bf16lo(ww[k])), fabsf(bf16hi(ww[k]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if ((t & 31) == 0) red[t >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  float s = __fdiv_rn(fmaxf(amax, kEps), kFp8Max);
  if (POW2) s = ceil_pow2(s);
  const float y = __frcp_rn(s);
  if (t == 0 && in_bounds(status, (b * NB + nb) * KB + kb, 1, n_s)) sw[(b * NB + nb) * KB + kb] = s;
  if (!row_ok) return;
  uint8_t* dst = wq + (b * N + n) * K + kb * 128 + (t & 1) * 64;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t c[8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 r = raw[2 * i + h];
      const uint32_t ww[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = bf16lo(ww[k]), hi = bf16hi(ww[k]);
        c[h * 4 + k] = POW2 ? cvt_e4m3x2(__fmul_rn(lo, y), __fmul_rn(hi, y))
                            : cvt_e4m3x2(group_div(lo, s, y), group_div(hi, s, y));
      }
    }
    st_v4(dst + 16 * i, make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16),
                                   c[4] | (c[5] << 16), c[6] | (c[7] << 16)));
  }
}

namespace {

// Whether a grid of `blocks` blocks of `kernel` runs in one wave (all its
// blocks resident at once).  Only such grids are launched with programmatic
// dependent launch: a multi-wave quant grid launched early slowed the
// 36-shape sweep step by ~1.5-3 % (measured with the launch mode split by
// kernel), a multi-wave silu-mul-quant grid the MoE slice by 2 %, while a
// one-wave grid after a GEMM gains its set-up overlap.
template <typename K>
bool one_wave(K kernel, const DeviceInfo& dev, int64_t blocks) {
  static std::map<std::pair<const void*, int>, int> per_sm;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair((const void*)kernel, dev.ordinal);
  auto it = per_sm.find(key);
  if (it == per_sm.end()) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kQuantWarps * 32, 0) !=
        cudaSuccess) {
      cudaGetLastError();
      n = 1;
    }
    it = per_sm.emplace(key, n > 0 ? n : 1).first;
  }
  return blocks <= (int64_t)it->second * dev.sm_count;
}

}  // namespace

}  // namespace bfq

using namespace bfq;

extern "C" bfq_status bfq_quant(const void* x, int64_t M, int64_t K, int64_t ld_x,
                                int32_t group, int32_t fmt, void* q, void* scales,
                                int64_t scale_ld, void* stream) {
  if (M < 0 || K <= 0 || ld_x < K || scale_ld < M || !valid_fmt(fmt))
    return BFQ_ERR_INVALID_ARG;
  if (group != 128 || K % 128 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BFQ_OK;
  if (!x || !q || !scales) return BFQ_ERR_INVALID_ARG;
  // scale_ld % 4: each scale column starts on a 16-byte boundary, the layout
  // the GEMM's activation-scale argument requires
  if (!aligned16(x) || !aligned16(q) || !aligned16(scales) || ld_x % 8 != 0 ||
      scale_ld % 4 != 0)
    return BFQ_ERR_MISALIGNED;
  DeviceInfo dev;
  bfq_status st = current_device(&dev);
  if (st != BFQ_OK) return st;
  const int64_t units = M * cdiv(K / 128, 4);
  const int64_t per_block = (int64_t)kQuantWarps * kUnroll;
  int64_t blocks = cdiv(units, per_block);
  // Up to 32 blocks per SM in the grid: many short-lived warps with one unit
  // each keep more loads in flight than fewer warps looping over two units
  // (2 % less time over the sweep's quant shapes, back to back).
  const int64_t cap = (int64_t)dev.sm_count * 32;
  if (blocks > cap) blocks = cap;
  cudaStream_t s = (cudaStream_t)stream;
  const auto* xb = (const __nv_bfloat16*)x;
  auto* qb = (uint8_t*)q;
  int* status = device_status_ptr();
  if (!status) return BFQ_ERR_CUDA;
  const int64_t n_x = (M - 1) * ld_x + K;           // extents for the debug bounds checks
  const int64_t n_s = scale_cols(K, fmt) * scale_ld;
  switch (fmt) {
    case BFQ_SCALE_F32:
      st = launch_status(launch_kernel(one_wave(quant_kernel<BFQ_SCALE_F32>, dev, blocks),
                                       quant_kernel<BFQ_SCALE_F32>, dim3((unsigned)blocks),
                                    dim3(kQuantWarps * 32), 0, s, 1, xb, M, K, ld_x, qb, scales,
                                    scale_ld, status, n_x, n_s));
      break;
    case BFQ_SCALE_F32_POW2:
      st = launch_status(launch_kernel(one_wave(quant_kernel<BFQ_SCALE_F32_POW2>, dev, blocks),
                                       quant_kernel<BFQ_SCALE_F32_POW2>, dim3((unsigned)blocks),
                                    dim3(kQuantWarps * 32), 0, s, 1, xb, M, K, ld_x, qb, scales,
                                    scale_ld, status, n_x, n_s));
      break;
    default:
      st = launch_status(launch_kernel(one_wave(quant_kernel<BFQ_SCALE_UE8M0_PACKED>, dev, blocks),
                                       quant_kernel<BFQ_SCALE_UE8M0_PACKED>, dim3((unsigned)blocks),
                                    dim3(kQuantWarps * 32), 0, s, 1, xb, M, K, ld_x, qb, scales,
                                    scale_ld, status, n_x, n_s));
      break;
  }
  return st;
}

namespace bfq {
namespace {
std::mutex g_silu_mu;
const float* g_silu_ready[64];  // per device: the built table, or null
}  // namespace

// The device's silu table, built on first use: the build kernel runs on
// `stream` and the stream is synchronized once, so that every later call, on
// any stream, finds the table complete.  Null while the stream is capturing a
// graph and the table has not been built (the caller then computes silu).
const float* silu_table(const DeviceInfo& dev, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_silu_mu);
  if (g_silu_ready[dev.ordinal]) return g_silu_ready[dev.ordinal];
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (cs != cudaStreamCaptureStatusNone) return nullptr;
  void* t = nullptr;
  if (cudaGetSymbolAddress(&t, g_silu_table) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  silu_table_kernel<<<65536 / 256, 256, 0, stream>>>((float*)t);
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  g_silu_ready[dev.ordinal] = (const float*)t;
  return g_silu_ready[dev.ordinal];
}

namespace {

template <int FMT>
bfq_status launch_silu_mul_quant(const DeviceInfo& dev, dim3 grid, cudaStream_t s,
                                 const __nv_bfloat16* x, int T, int I, const int32_t* counts,
                                 uint8_t* q, void* scales, int64_t scale_ld, const float* tab) {
  int* status = device_status_ptr();
  if (!status) return BFQ_ERR_CUDA;
  // extents for the debug bounds checks: x [E][T][2I], scales [E][cols][scale_ld]
  const int64_t E = grid.y;
  const int64_t n_x = E * T * 2 * (int64_t)I;
  const int64_t n_s = E * scale_cols(I, FMT) * scale_ld;
  // programmatic launch only when the whole grid (padded row pairs included)
  // fits in one wave
  const int64_t blocks = (int64_t)grid.x * grid.y;
  if (tab)
    return launch_status(launch_kernel(one_wave(silu_mul_quant_kernel<FMT, true>, dev, blocks),
                                       silu_mul_quant_kernel<FMT, true>, grid,
                                       dim3(kQuantWarps * 32), 0, s, 1, x, T, I, counts, q,
                                       scales, scale_ld, tab, status, n_x, n_s));
  return launch_status(launch_kernel(one_wave(silu_mul_quant_kernel<FMT, false>, dev, blocks),
                                     silu_mul_quant_kernel<FMT, false>, grid,
                                     dim3(kQuantWarps * 32), 0, s, 1, x, T, I, counts, q, scales,
                                     scale_ld, tab, status, n_x, n_s));
}

}  // namespace
}  // namespace bfq

extern "C" bfq_status bfq_silu_mul_quant(const void* x, int32_t E, int32_t T, int32_t I,
                                         const int32_t* valid_counts, int32_t fmt, void* q,
                                         void* scales, int64_t scale_ld, void* stream) {
  if (E < 0 || T < 0 || I <= 0 || scale_ld < T || !valid_fmt(fmt)) return BFQ_ERR_INVALID_ARG;
  if (I % 128 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (E == 0 || T == 0) return BFQ_OK;
  if (!x || !valid_counts || !q || !scales) return BFQ_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(scales) || scale_ld % 4 != 0)
    return BFQ_ERR_MISALIGNED;
  if (E > 65535) return BFQ_ERR_UNSUPPORTED_SHAPE;
  DeviceInfo dev;
  bfq_status st = current_device(&dev);
  if (st != BFQ_OK) return st;
  dim3 grid((unsigned)cdiv(T, kSiluRowsPerBlock), (unsigned)E);
  cudaStream_t s = (cudaStream_t)stream;
  const auto* xb = (const __nv_bfloat16*)x;
  auto* qb = (uint8_t*)q;
  const float* tab = silu_table(dev, s);
  switch (fmt) {
    case BFQ_SCALE_F32:
      return launch_silu_mul_quant<BFQ_SCALE_F32>(dev, grid, s, xb, T, I, valid_counts, qb, scales,
                                                  scale_ld, tab);
    case BFQ_SCALE_F32_POW2:
      return launch_silu_mul_quant<BFQ_SCALE_F32_POW2>(dev, grid, s, xb, T, I, valid_counts, qb,
                                                       scales, scale_ld, tab);
    default:
      return launch_silu_mul_quant<BFQ_SCALE_UE8M0_PACKED>(dev, grid, s, xb, T, I, valid_counts, qb,
                                                           scales, scale_ld, tab);
  }
}

extern "C" bfq_status bfq_weight_block_quant(const void* w, int64_t batch, int64_t N,
                                             int64_t K, int32_t fmt, void* wq, float* sw,
                                             void* stream) {
  if (batch <= 0 || N <= 0 || K <= 0 || !valid_fmt(fmt)) return BFQ_ERR_INVALID_ARG;
  if (!w || !wq || !sw) return BFQ_ERR_INVALID_ARG;
  if (K % 128 != 0) return BFQ_ERR_UNSUPPORTED_SHAPE;
  if (fmt == BFQ_SCALE_UE8M0_PACKED) return BFQ_ERR_FORMAT;
  if (!aligned16(w) || !aligned16(wq)) return BFQ_ERR_MISALIGNED;
  const int64_t NB = cdiv(N, 128), KB = K / 128;
  if (NB > 65535 || batch > 65535 || KB > 0x7FFFFFFF) return BFQ_ERR_UNSUPPORTED_SHAPE;
  DeviceInfo dev;
  bfq_status st = current_device(&dev);
  if (st != BFQ_OK) return st;
  dim3 grid((unsigned)KB, (unsigned)NB, (unsigned)batch);
  cudaStream_t s = (cudaStream_t)stream;
  const auto* wb = (const __nv_bfloat16*)w;
  auto* wqb = (uint8_t*)wq;
  int* status = device_status_ptr();
  if (!status) return BFQ_ERR_CUDA;
  const int64_t n_w = batch * N * K, n_s = batch * NB * KB;  // debug bounds-check extents
  // weight preparation keeps plain stream order (a multi-wave grid; nothing
  // on the inference path waits on it)
  if (fmt == BFQ_SCALE_F32)
    return launch_status(launch_kernel(false, weight_quant_kernel<false>, grid, dim3(256), 0, s,
                                       1, wb, N, K, wqb, sw, status, n_w, n_s));
  return launch_status(launch_kernel(false, weight_quant_kernel<true>, grid, dim3(256), 0, s, 1,
                                     wb, N, K, wqb, sw, status, n_w, n_s));
}
