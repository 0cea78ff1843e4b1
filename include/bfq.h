/*
 * bfq.h — C ABI of the block-scaled FP8 (W8A8) quantization and GEMM library
 * for NVIDIA GB300 (sm_103a).
 *
 * The library computes the data-parallel hot path of DeepSeek-style block-FP8
 * inference:
 *   - per-token-group (1 x 128) FP8 e4m3 activation quantization with fp32,
 *     power-of-two, or UE8M0 scales packed four per 32-bit word directly in
 *     the GEMM's column-major, TMA-aligned scale layout;
 *   - the same quantization fused behind silu(gate) * up over a masked,
 *     per-expert batch whose padded rows are neither read nor written;
 *   - 128 x 128 block quantization of weights;
 *   - the dense block-scaled FP8 GEMM  out = A * W^T  (1 x 128 activation
 *     scales, 128 x 128 weight scales, fp32 accumulation, bf16 output);
 *   - its masked grouped (per-expert) form.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every buffer argument is a DEVICE pointer owned by the caller.  The
 *    library allocates nothing and frees nothing; it keeps no per-call state.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously on it; the function returns as
 *    soon as the launch is enqueued.  GEMM kernels, and quant and
 *    silu-mul-quant grids that fit in one wave, are launched with
 *    programmatic stream serialization: a kernel may be scheduled while the
 *    previous one in the stream is finishing, but it waits for that kernel's
 *    completion (and memory visibility) before it reads or writes any global
 *    memory, so stream order semantics are unchanged.  (Multi-wave quant
 *    and silu-mul-quant grids keep plain stream order: launched early they
 *    slowed the GEMMs around them.  So does bfq_weight_block_quant.)
 *    Launches can be captured in CUDA graphs.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call launches nothing and returns a non-zero bfq_status.  There
 *    is no CPU fallback and no alternative backend.
 *  - Matrices are row-major with 16-byte aligned base pointers.  e4m3 means
 *    the OCP FP8 E4M3 "fn" format (bias 7, max 448, no infinities).
 *  - Scale arrays are COLUMN-MAJOR over rows: element (row r, column c) lives
 *    at c * scale_ld + r, with scale_ld >= rows (pass align4(rows) for the
 *    16-byte TMA alignment the GEMM uses).  Formats:
 *      BFQ_SCALE_F32          float, one per 128-element group, [K/128][ld];
 *      BFQ_SCALE_F32_POW2     float holding the UE8M0 value (a power of two);
 *      BFQ_SCALE_UE8M0_PACKED uint32 words, [ceil(K/512)][ld]; word w of row
 *                             r holds the biased exponents of groups 4w..4w+3,
 *                             group 4w in the least significant byte; the
 *                             scale of a byte b is 2^(b-127).
 *    The format always travels with the scale pointer: the GEMM is told which
 *    format its activation scales are in, so packed exponents can never be
 *    read as floats (the mismatch reported in the review of "[Perf] Deepgemm
 *    fused layout kernel for activations", vLLM PR #29546).
 *
 * Sources (cited by page title and section):
 *  [DG-bench]   "vLLM DeepGEMM FP8 Block GEMM 基准测试" (article on vLLM's
 *               benchmarks/kernels/deepgemm), §4.1-§4.3.
 *  [PR-29546]   "[Perf] Deepgemm fused layout kernel for activations",
 *               Purpose section and review thread.
 *  [PR-19885]   "[EP+DP] Optimize the little operations in the DeepGEMM +
 *               DeepEP low latency case", Summary item 2.
 *  [PR-19111]   "[Kernel] Integrate batched/masked deepgemm kernel",
 *               Summary of Changes and review thread.
 */
#ifndef BFQ_H_
#define BFQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t bfq_status;

enum {
  BFQ_OK = 0,
  BFQ_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum      */
  BFQ_ERR_UNSUPPORTED_SHAPE = 2, /* K % 128, N % 64, group != 128, ...         */
  BFQ_ERR_MISALIGNED = 3,        /* pointer or stride not 16-byte aligned      */
  BFQ_ERR_FORMAT = 4,            /* scale format not allowed for this operand  */
  BFQ_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed          */
  BFQ_ERR_TIMEOUT = 6,           /* a kernel watchdog gave up waiting          */
  BFQ_ERR_WORKSPACE = 7,         /* unused: no current plan needs a workspace  */
  BFQ_ERR_DEVICE = 8,            /* current device is not sm_100 family        */
  BFQ_ERR_DEVICE_BOUNDS = 9      /* debug build: a kernel's bounds check failed
                                    (latched in the device status; the access
                                    was skipped)                              */
};

typedef enum {
  BFQ_SCALE_F32 = 0,
  BFQ_SCALE_F32_POW2 = 1,
  BFQ_SCALE_UE8M0_PACKED = 2
} bfq_scale_fmt;

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t bfq_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* bfq_status_string(bfq_status status);

/*
 * Per-token-group FP8 quantization ([DG-bench] §4.1 per_token_group_quant_fp8
 * with column_major_scales / tma_aligned_scales / use_ue8m0; [PR-29546]
 * Purpose: the UE8M0 scales are packed into uint32 inside this kernel, so no
 * separate layout kernel runs).
 *
 * For every row r < M and group g < K/128 (128 consecutive columns):
 *     amax = max |x[r, 128g .. 128g+127]|
 *     s    = fl32(max(amax, 1e-10) / 448)             (IEEE fp32 division)
 *     s    = smallest power of two >= s               (POW2 and PACKED)
 *     q[r, k] = e4m3_rne_satfinite(fl32(x[r, k] / s))
 *
 *   x        bf16 [M][ld_x], ld_x >= K, ld_x % 8 == 0, 16-byte aligned.
 *   M, K     M >= 0 (M == 0 is a no-op), K > 0, K % 128 == 0.
 *   group    must be 128.
 *   fmt      a bfq_scale_fmt.
 *   q        e4m3 [M][K] (row stride K), 16-byte aligned.
 *   scales   column-major, see the header comment, 16-byte aligned;
 *            scale_ld >= M and scale_ld % 4 == 0 (the TMA-aligned layout the
 *            GEMM takes).  Entries of rows >= M are not written.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
bfq_status bfq_quant(const void* x, int64_t M, int64_t K, int64_t ld_x, int32_t group,
                     int32_t fmt, void* q, void* scales, int64_t scale_ld, void* stream);

/*
 * Fused silu-and-mul + per-token-group quantization over a masked per-expert
 * batch ([PR-19885] Summary item 2: output in the grouped GEMM's layout,
 * padded tokens are neither loaded nor computed; [PR-19111] masked layout).
 *
 * For expert e and row r < valid_counts[e]:
 *     y[k] = silu(x[e, r, k]) * x[e, r, I + k]     (gate first, up second)
 *     silu(g) = g / (1 + exp(-g)), all in fp32, y not rounded to bf16,
 *     exp = the library's fp32 exp (Cody-Waite reduction, degree-7 Taylor
 *           polynomial; within 2 ulp of the exact function);
 * then y is quantized exactly as in bfq_quant.  Rows r >= valid_counts[e]
 * (and all rows of an expert with count <= 0) are neither read nor written,
 * in x, q or scales.
 *
 * The gate is bf16, so silu has 65536 possible inputs: the library evaluates
 * silu (the arithmetic above) for all of them once per device into a 256 KB
 * table in its own device memory, and looks silu up.  The first call on a
 * device that is not being captured into a CUDA graph builds the table on
 * `stream` and synchronizes that stream once; calls made while a graph is
 * being captured before then compute silu in the kernel instead.  Either way
 * the results are the same, bit for bit.
 *
 *   x             bf16 [E][T][2I], 16-byte aligned.
 *   E, T, I       E >= 0, T >= 0, I > 0, I % 128 == 0.
 *   valid_counts  device int32 [E]; values are clamped to [0, T].
 *   fmt           a bfq_scale_fmt.
 *   q             e4m3 [E][T][I], 16-byte aligned.
 *   scales        [E][cols][scale_ld], cols = I/128 (fp32 formats) or
 *                 ceil(I/512) (packed), 16-byte aligned, scale_ld >= T,
 *                 scale_ld % 4 == 0.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
bfq_status bfq_silu_mul_quant(const void* x, int32_t E, int32_t T, int32_t I,
                              const int32_t* valid_counts, int32_t fmt, void* q,
                              void* scales, int64_t scale_ld, void* stream);

/*
 * 128 x 128 block quantization of weights ([DG-bench] §4.1
 * per_block_cast_to_fp8(B, [128, 128], use_ue8m0)): the group rule of
 * bfq_quant applied to each 128 x 128 block (amax over the block).
 *
 *   w       bf16 [batch][N][K], 16-byte aligned.
 *   batch   >= 1 independent matrices (experts); blocks never straddle them.
 *   N, K    N > 0, K > 0, K % 128 == 0.  A partial last row-block uses only
 *           its rows < N.
 *   fmt     BFQ_SCALE_F32 or BFQ_SCALE_F32_POW2 (else BFQ_ERR_FORMAT).
 *   wq      e4m3 [batch][N][K].
 *   sw      float [batch][ceil(N/128)][K/128], row-major.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, FORMAT, CUDA.
 */
bfq_status bfq_weight_block_quant(const void* w, int64_t batch, int64_t N, int64_t K,
                                  int32_t fmt, void* wq, float* sw, void* stream);

/*
 * Bytes of workspace a GEMM problem needs: 0 for every problem.
 *
 *   E == 0     dense bfq_gemm_block_fp8 / bfq_gemm_block_fp8_quant of
 *              M x N x K;
 *   E >= 1     the masked grouped GEMM of E experts with M rows each.
 *
 * Every K split reduces its fp32 partial sums through the distributed shared
 * memory of its thread-block cluster, so no plan uses global scratch.  Kept
 * so that callers written against a workspace-taking interface need not
 * change.
 */
size_t bfq_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t E);

/*
 * Dense block-scaled FP8 GEMM, "NT" ([DG-bench] §4.2 fp8_gemm_nt and the
 * promotion loop of w8a8_triton_block_scaled_mm; eligibility of §4.2 end):
 *
 *   out[m, n] = bf16_rne( sum_b sA[m, b] * sW[n / 128, b]
 *                         * sum_{k in block b} a_q[m, k] * w_q[n, k] )
 *
 * with fp32 accumulation on the tensor cores and the scale product applied
 * to each 128-deep K block ("promotion").  When there are fewer output tiles
 * than SMs, K is split over the CTAs of a thread-block cluster (at most 8);
 * each CTA keeps its fp32 partial sum in shared memory and the cluster adds
 * them in split order through distributed shared memory, so results are
 * deterministic.  With more tiles than SMs, one CTA per SM walks the tiles.
 *
 *   a_q            e4m3 [M][K], 16-byte aligned.
 *   a_scales       column-major activation scales in format a_fmt
 *                  (any bfq_scale_fmt), leading dimension a_scale_ld >= M,
 *                  a_scale_ld % 4 == 0.
 *   w_q            e4m3 [N][K], 16-byte aligned.
 *   w_scales       float [ceil(N/128)][K/128].
 *   M, N, K        M >= 0 (0 = no-op), N > 0, N % 64 == 0, K > 0,
 *                  K % 128 == 0.
 *   out            bf16 [M][N] (preallocated by the caller).
 *   workspace      unused by the current plans (may be NULL / 0); a non-NULL
 *                  workspace must be 16-byte aligned, and workspace_bytes > 0
 *                  with a NULL workspace is INVALID_ARG.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, FORMAT, CUDA, DEVICE.
 */
bfq_status bfq_gemm_block_fp8(const void* a_q, const void* a_scales, int32_t a_fmt,
                              int64_t a_scale_ld, const void* w_q, const float* w_scales,
                              int64_t M, int64_t N, int64_t K, void* out, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Dense block-scaled FP8 GEMM whose epilogue also quantizes its output for
 * the next block-FP8 GEMM: the per-token-group (1 x 128) activation quant of
 * the bf16 result, fused into the GEMM so that the output is not written and
 * read back before it is quantized (the direction of "[Perf] Deepgemm fused
 * layout kernel for activations", Purpose: remove an extra kernel and its
 * memory round trip; [DG-bench] §4.1 for the quant it fuses).
 *
 *   C = bf16_rne(GEMM of bfq_gemm_block_fp8)
 *   q_out, q_scales = bfq_quant(C, group 128, q_fmt, q_scale_ld)
 *
 * bit for bit: q_out and q_scales are exactly what bfq_quant writes for the
 * bf16 output of bfq_gemm_block_fp8 with the same inputs.
 *
 *   a_q .. K       as for bfq_gemm_block_fp8, and N % 128 == 0.
 *   out            bf16 [M][N], or NULL when only the quantized form is
 *                  wanted.
 *   q_fmt          scale format of the output quant (any bfq_scale_fmt).
 *   q_out          e4m3 [M][N], 16-byte aligned.
 *   q_scales       column-major scales as bfq_quant writes them:
 *                  float [N/128][q_scale_ld] or uint32 [ceil(N/512)][q_scale_ld]
 *                  (packed UE8M0, a partial last word with zero bytes for its
 *                  missing groups); q_scale_ld >= M, q_scale_ld % 4 == 0;
 *                  columns M .. q_scale_ld-1 are not written.
 *   workspace      as for bfq_gemm_block_fp8 (unused; same launch plan); with
 *                  K split, the cluster's reduction quantizes whole
 *                  128-column groups, one warp each.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE (also N % 128 != 0), MISALIGNED,
 * FORMAT, CUDA, DEVICE.
 */
bfq_status bfq_gemm_block_fp8_quant(const void* a_q, const void* a_scales, int32_t a_fmt,
                                    int64_t a_scale_ld, const void* w_q, const float* w_scales,
                                    int64_t M, int64_t N, int64_t K, void* out, int32_t q_fmt,
                                    void* q_out, void* q_scales, int64_t q_scale_ld,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * bfq_gemm_block_fp8 for callers that cannot allocate device memory.  (The
 * pages have no counterpart; this is a convenience of this library.)
 *
 * Some callers cannot call cudaMalloc: plugins inside a framework that owns
 * all device memory through its own caching allocator (a raw cudaMalloc
 * would bypass its accounting), and serving loops that forbid allocation
 * after start-up because cudaMalloc can synchronize the device and stall
 * every stream.
 * This entry point takes the same arguments as bfq_gemm_block_fp8 minus the
 * workspace and computes the same result with the same launch plan.  No plan
 * needs scratch (K splits reduce through distributed shared memory), so it
 * allocates nothing, frees nothing and holds no device memory of its own;
 * calls may overlap on the GPU like any other.  Inputs and outputs are the
 * caller's.
 * Errors: those of bfq_gemm_block_fp8.
 */
bfq_status bfq_gemm_block_fp8_noalloc(const void* a_q, const void* a_scales, int32_t a_fmt,
                                      int64_t a_scale_ld, const void* w_q,
                                      const float* w_scales, int64_t M, int64_t N, int64_t K,
                                      void* out, void* stream);

/* Device scratch held by bfq_gemm_block_fp8_noalloc, in bytes: 0. */
size_t bfq_gemm_noalloc_scratch_bytes(void);

/*
 * Masked grouped block-scaled FP8 GEMM ([PR-19111]
 * m_grouped_gemm_fp8_fp8_bf16_nt_masked; per-expert valid-row count):
 *
 *   for e < E, r < valid_counts[e]:   out[e, r, :] = GEMM(a_q[e, r, :], w_q[e])
 *
 * Row tiles that start at or beyond valid_counts[e] are skipped entirely (no
 * loads, no MMA); output rows r >= valid_counts[e] are never written.
 *
 *   a_q            e4m3 [E][T][K].
 *   a_scales       [E][cols][a_scale_ld] in format a_fmt, a_scale_ld >= T,
 *                  a_scale_ld % 4 == 0.
 *   w_q            e4m3 [E][N][K].
 *   w_scales       float [E][ceil(N/128)][K/128].
 *   valid_counts   device int32 [E], clamped to [0, T].
 *   expected_m     hint of the typical count (0 = unknown).  Accepted and
 *                  not used by the current plans, which read the counts on
 *                  the device; it can never change the result.
 *   out            bf16 [E][T][N].
 *   workspace, workspace_bytes   accepted and not used: no plan of the
 *                  masked GEMM needs a workspace (bfq_gemm_workspace_bytes
 *                  with E >= 1 returns 0); may be NULL / 0.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, FORMAT, CUDA, DEVICE.
 */
bfq_status bfq_gemm_block_fp8_masked(const void* a_q, const void* a_scales, int32_t a_fmt,
                                     int64_t a_scale_ld, const void* w_q,
                                     const float* w_scales, const int32_t* valid_counts,
                                     int32_t E, int32_t T, int64_t N, int64_t K,
                                     int32_t expected_m, void* out, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * Dense block-scaled FP8 GEMM for power-of-two (UE8M0) scales, the scales
 * applied by the tensor cores' block scaling instead of promotion ([DG-bench]
 * §4.1–4.2: UE8M0 is the hardware-friendly scale form, each 1 x 128 scale
 * reused by the four K = 32 MMAs of its block).  Same result definition as
 * bfq_gemm_block_fp8: multiplying by a power of two is exact, so the two
 * differ only in fp32 summation order (within the same error bound).
 * tcgen05.mma kind::mxf8f6f4.block_scale scales each K = 32 step's products
 * by 2^(eA + eB) and accumulates the whole K range in TMEM; the scale words
 * are copied into TMEM once per four K blocks.  One CTA per SM walks the
 * 128 x 256 output tiles; there is no K split.  Launch plan: for M <= 128,
 * K < 1024 or fewer output tiles than half the SMs, the call runs
 * bfq_gemm_block_fp8's plan instead (promotion; K split over a cluster),
 * which is faster there and gives the same result for these scales.
 *
 *   a_q, a_scale_ld, w_q, M, N, K, out   as for bfq_gemm_block_fp8.
 *   a_fmt          BFQ_SCALE_UE8M0_PACKED or BFQ_SCALE_F32_POW2 (else FORMAT).
 *   a_scales       column-major, as for bfq_gemm_block_fp8; packed UE8M0
 *                  words 16-byte aligned (they are moved by bulk copies).
 *   w_scales       float [ceil(N/128)][K/128], each a positive power of two
 *                  2^-126 .. 2^127 (as bfq_weight_block_quant writes them with
 *                  fmt = BFQ_SCALE_F32_POW2).
 * A scale that is not a positive power of two cannot be applied: the kernel
 * latches BFQ_ERR_FORMAT in the device status (bfq_poll_device_status) and
 * the output of that call is undefined.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, FORMAT, CUDA, DEVICE.
 */
bfq_status bfq_gemm_block_fp8_ue8m0(const void* a_q, const void* a_scales, int32_t a_fmt,
                                    int64_t a_scale_ld, const void* w_q, const float* w_scales,
                                    int64_t M, int64_t N, int64_t K, void* out, void* stream);

/*
 * Masked grouped form of bfq_gemm_block_fp8_ue8m0 (the per-expert valid-row
 * counts of bfq_gemm_block_fp8_masked, whose argument rules apply, without
 * its unused expected_m and workspace): rows r >= valid_counts[e] are never
 * written; a_fmt and w_scales as for bfq_gemm_block_fp8_ue8m0; E <= 1024.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, FORMAT, CUDA, DEVICE.
 */
bfq_status bfq_gemm_block_fp8_masked_ue8m0(const void* a_q, const void* a_scales, int32_t a_fmt,
                                           int64_t a_scale_ld, const void* w_q,
                                           const float* w_scales, const int32_t* valid_counts,
                                           int32_t E, int32_t T, int64_t N, int64_t K,
                                           void* out, void* stream);

/*
 * Reorders an MoE up-projection weight for the fused form below: each
 * expert's [2I][K] e4m3 weight (gate rows 0..I-1, up rows I..2I-1, the
 * split of "[EP+DP] Optimize the little operations in the DeepGEMM + DeepEP
 * low latency case" silu-and-mul) and its [2I/128][K/128] block scales are
 * copied so that 128-row block 2j is gate block j and block 2j+1 is up
 * block j.  A one-time layout step (as weight quant is), on the GPU.
 *
 *   w_q, w_scales           e4m3 [E][2I][K] (16-byte aligned), float
 *                           [E][2I/128][K/128]
 *   w_q_out, w_scales_out   same shapes, distinct buffers
 *   I % 128 == 0, K % 128 == 0.
 * Errors: INVALID_ARG (also in-place), UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
bfq_status bfq_interleave_gate_up(const void* w_q, const float* w_scales, int32_t E, int64_t I,
                                  int64_t K, void* w_q_out, float* w_scales_out, void* stream);

/*
 * Masked grouped up-projection GEMM with silu-and-mul and its quant fused
 * into the epilogue: for expert e and row r < valid_counts[e],
 *
 *   h[e, r, :]  = bf16(GEMM of bfq_gemm_block_fp8_masked with the
 *                 un-interleaved weight), 2I columns (gate | up)
 *   q_out, q_scales = bfq_silu_mul_quant(h, valid_counts, q_fmt)
 *
 * bit for bit, without writing h: each 256-wide tile holds a gate block and
 * its up block (weights from bfq_interleave_gate_up), so the epilogue forms
 * y = silu(gate) * up for 128 features of a row and quantizes them as one
 * 1 x 128 group (silu from the table described at bfq_silu_mul_quant, built
 * on the same terms).  Rows r >= count are neither computed nor written (only row
 * tiles below the count are scheduled, as in bfq_gemm_block_fp8_masked).
 *
 *   a_q .. a_scale_ld   as for bfq_gemm_block_fp8_masked (K of the up
 *                       projection, E <= 1024).
 *   w_q, w_scales       interleaved (bfq_interleave_gate_up).
 *   I                   features per expert (the down projection's K),
 *                       I % 128 == 0.
 *   q_fmt, q_out, q_scales, q_scale_ld   the output of bfq_silu_mul_quant:
 *                       e4m3 [E][T][I]; scales [E][cols][q_scale_ld] with
 *                       cols = I/128 (fp32, pow2) or ceil(I/512) (packed
 *                       UE8M0); q_scale_ld >= T, % 4 == 0.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE (also E > 1024), MISALIGNED, CUDA,
 * DEVICE.
 */
bfq_status bfq_gemm_block_fp8_masked_silu_quant(const void* a_q, const void* a_scales,
                                                int32_t a_fmt, int64_t a_scale_ld,
                                                const void* w_q, const float* w_scales,
                                                const int32_t* valid_counts, int32_t E,
                                                int32_t T, int64_t I, int64_t K, int32_t q_fmt,
                                                void* q_out, void* q_scales, int64_t q_scale_ld,
                                                void* stream);

/*
 * bfq_gemm_block_fp8_masked_silu_quant on the block-scaled kernel of
 * bfq_gemm_block_fp8_masked_ue8m0 (power-of-two scales on both operands,
 * applied by the MMA): q_out and q_scales equal, bit for bit,
 * bfq_silu_mul_quant of the bf16 output of bfq_gemm_block_fp8_masked_ue8m0
 * with the un-interleaved weight.  Arguments as for
 * bfq_gemm_block_fp8_masked_silu_quant; a_fmt BFQ_SCALE_UE8M0_PACKED or
 * BFQ_SCALE_F32_POW2 (else FORMAT); w_scales powers of two (a scale that is
 * not latches BFQ_ERR_FORMAT in the device status, as for
 * bfq_gemm_block_fp8_ue8m0).
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE (also E > 1024), MISALIGNED, FORMAT,
 * CUDA, DEVICE.
 */
bfq_status bfq_gemm_block_fp8_masked_silu_quant_ue8m0(
    const void* a_q, const void* a_scales, int32_t a_fmt, int64_t a_scale_ld, const void* w_q,
    const float* w_scales, const int32_t* valid_counts, int32_t E, int32_t T, int64_t I,
    int64_t K, int32_t q_fmt, void* q_out, void* q_scales, int64_t q_scale_ld, void* stream);

/*
 * Process-wide switch for programmatic dependent launch ([DG-bench] §4.2: the
 * GEMM wrapper enables PDL so that a kernel's set-up overlaps the tail of the
 * kernel before it).  enable != 0 (the default): kernels are launched with
 * programmatic stream serialization as described in the conventions above.
 * enable == 0: plain stream order for every kernel, each scheduled only after
 * the previous one has finished.  Results are bit-identical either way; the
 * switch exists to measure what the overlap buys.  It applies to launches
 * made (or captured into a graph) after the call.  Returns the previous
 * setting (0 or 1).
 */
int32_t bfq_set_programmatic_launch(int32_t enable);

/*
 * Reads and clears the device-side error latch that kernel watchdogs set when
 * a bounded wait (on a TMA/MMA barrier) gives up.  The read and the clear are
 * one atomic exchange on the device (a one-thread kernel on `stream`), so a
 * timeout latched by a kernel on another stream is reported by this call or
 * the next one, never lost.  Synchronizes `stream`.
 * Returns BFQ_OK or the latched code — BFQ_ERR_TIMEOUT (a watchdog),
 * BFQ_ERR_FORMAT (a block-scaled GEMM met a scale that is not a power of
 * two), BFQ_ERR_DEVICE_BOUNDS (libbfq_debug.so only: a kernel's bounds check
 * failed) — or BFQ_ERR_CUDA.
 */
bfq_status bfq_poll_device_status(void* stream);

/*
 * Watchdog self-test: launches one kernel that waits on a barrier that
 * nothing ever completes, with a limit of timeout_us microseconds, after
 * which the kernel records BFQ_ERR_TIMEOUT in the device latch and returns.
 * The CUDA context stays usable.  Read the result with
 * bfq_poll_device_status().  timeout_us must be in [1, 1000000].
 */
bfq_status bfq_watchdog_selftest(int32_t timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BFQ_H_ */
