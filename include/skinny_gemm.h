/*
 * skinny_gemm.h -- C ABI of the GB300 (sm_103a) bf16 GEMM / skinny-GEMV library.
 *
 * Operation (every GEMM entry point):
 *
 *     C[m, n] = sum_{k < K} A[m, k] * B[n, k]        0 <= m < M, 0 <= n < N
 *
 * with A[m, k] = A[m*lda + k], B[n, k] = B[n*ldb + k], C[m, n] = C[m*ldc + n].
 * All three are bf16 (stored as 16-bit patterns), products are accumulated in
 * fp32 and the result is rounded to bf16 with round-to-nearest-even.  B is laid
 * out like a linear layer's weight [out_features, in_features], so C = A . B^T.
 * This is the bf16 GEMM with fp32 accumulation of spark-kernels ("the bf16 gemm":
 * 4096-cubed, the 7B-model 11008-wide MLP shapes and the decode shapes) and the
 * skinny bf16 GEMV of "The kernels that were there" ("The GEMV": one pass over
 * the weights for all rows of a small M, fp32 accumulation, bf16 store).
 *
 * Conventions shared by all entry points
 *   - Pointers A, B, C are DEVICE pointers on the current CUDA device; the caller
 *     owns them.  The library never frees or retains them.
 *   - Every call only enqueues work on `stream` (never the legacy default stream,
 *     never a device synchronisation), so calls may be captured in a CUDA graph
 *     ("The kernels that were there", "The bench that lied": the launch must
 *     follow the caller's stream).
 *   - Synchronous argument errors return a non-zero sg_status before anything is
 *     launched.  Launch failures return SG_ERR_CUDA (see sg_last_cuda_error).
 *     Kernel-side wait timeouts are reported by sg_check_device_errors.
 *   - Requirements: M, N, K >= 0; lda >= K, ldb >= K, ldc >= N; A, B, C 16-byte
 *     aligned and lda, ldb, ldc multiples of 8 elements (16-byte row pitch), else
 *     SG_ERR_MISALIGNED.  M = 0 or N = 0 is a no-op; K = 0 sets C to zero.
 *   - C must not overlap A or B.
 *   - The library keeps one workspace per device (Stream-K / split-K partial sums
 *     and arrival counters), allocated on the first call that needs it.  That
 *     first call must not happen during stream capture (SG_ERR_INVALID_ARG is
 *     returned instead); make one warm-up call first.  Calls that run
 *     concurrently on different streams of one device share that workspace and
 *     are not supported.
 */
#ifndef SKINNY_GEMM_H
#define SKINNY_GEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define SG_API __attribute__((visibility("default")))
#else
#define SG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *sg_stream_t;

typedef enum {
    SG_OK = 0,
    SG_ERR_INVALID_ARG = 1,        /* null pointer, negative size, ld too small, M > 64 on gemv */
    SG_ERR_MISALIGNED = 2,         /* pointer or leading dimension breaks the 16-byte rule */
    SG_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
    SG_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed */
    SG_ERR_TIMEOUT = 5,            /* a kernel gave up on a bounded wait */
    SG_ERR_OUT_OF_MEMORY = 6       /* workspace allocation failed */
} sg_status;

/* Skinny-path kernels selectable through gemv_bf16_path. */
typedef enum {
    SG_PATH_AUTO = 0,        /* library's choice (see gemv_bf16) */
    SG_PATH_CUDA_CORE = 1,   /* fp32 FMA stream over the weights, no tensor cores */
    SG_PATH_TENSOR_CORE = 2, /* tcgen05 with the weight rows on the MMA's M side */
    SG_PATH_GEMM = 3,        /* tcgen05 GEMM, one CTA per 128 x 256 or 128 x 128 tile */
    SG_PATH_GEMM_PAIR = 4    /* tcgen05 GEMM, a 2-CTA cluster per 256 x 256 tile */
} sg_path;

/*
 * gemm_bf16 -- C = A . B^T for any M, N, K (the main entry point).
 *
 * M > 64 runs the persistent tcgen05 GEMM: a TMA-fed ring of 128-byte-swizzled
 * shared-memory stages, warp-specialised producer / MMA / epilogue roles, fp32
 * accumulators in tensor memory, a Stream-K tail (spark-kernels, "stream-k
 * proper") and a TMA-store epilogue.  Its tiles are 256 x 256 on clusters of two
 * CTAs from M = 256, or 128 x 128 on one CTA each when those fit in one wave of
 * SMs (then K is split into equal pieces, one per CTA, if the tiles still leave
 * SMs idle), or 128 x 256 on one CTA below M = 256 and where at most 32 k-steps
 * of pair tiles would fall short of a wave.  M <= 64 is
 * routed to the skinny path exactly as gemv_bf16 would (spark-kernels, "the
 * decode kernel": the decode shapes get their own kernel).
 *
 * Returns SG_OK or an sg_status code.
 */
SG_API int gemm_bf16(const void *A, const void *B, void *C,
              int64_t M, int64_t N, int64_t K,
              int64_t lda, int64_t ldb, int64_t ldc, sg_stream_t stream);

/*
 * gemv_bf16 -- the skinny path, 1 <= M <= 64 (M > 64 or M < 0: SG_ERR_INVALID_ARG).
 *
 * Each weight byte of B is read from memory once for all M rows of A
 * ("The kernels that were there", "The GEMV": the M = 2 kernel loads each weight
 * once and feeds both rows).  For M <= 2 the kernel is the CUDA-core stream:
 * 16-byte weight loads coalesced along K, fp32 FMAs, warp-shuffle reductions and
 * a K split only when there are too few row groups to keep enough bytes in flight
 * (spark-kernels, "the decode kernel").  For larger M the fp32 FMA rate of the
 * CUDA cores falls below the weight stream, so the tcgen05 kernel with the weight
 * rows on the MMA's M side takes over; it reads the weights once as well.
 */
SG_API int gemv_bf16(const void *A, const void *B, void *C,
              int64_t M, int64_t N, int64_t K,
              int64_t lda, int64_t ldb, int64_t ldc, sg_stream_t stream);

/*
 * gemv_bf16_path -- gemv_bf16 with the kernel chosen by the caller
 * (path = SG_PATH_AUTO, SG_PATH_CUDA_CORE or SG_PATH_TENSOR_CORE).  The CUDA-core
 * kernel holds at most 8 rows of accumulators; larger M is processed in
 * consecutive launches of 8 rows each.  Same arguments and errors as gemv_bf16;
 * an unknown path is SG_ERR_INVALID_ARG.
 */
SG_API int gemv_bf16_path(const void *A, const void *B, void *C,
                   int64_t M, int64_t N, int64_t K,
                   int64_t lda, int64_t ldb, int64_t ldc, int path, sg_stream_t stream);

/*
 * gemm_bf16_swiglu -- the gated MLP's first half in one launch:
 *
 *     C[m, n] = silu(G[m, n]) * U[m, n],   G = A . Wg^T,  U = A . Wu^T,
 *     silu(x) = x / (1 + e^-x),
 *
 * the fused gate/up projection with a SwiGLU epilogue (spark-kernels, "the bf16
 * gemm": the fused MLP kernels; the pages' "fused MLP epilogues" as the next
 * step).  A is M x K (lda), Wg and Wu are N x K weights with one leading
 * dimension ldw, C is M x N (ldc); all bf16, row-major, 16-byte aligned, leading
 * dimensions multiples of 8.  G and U accumulate in fp32; the SiLU and the
 * product are fp32 (expf); C is rounded to bf16 (nearest even).  G and U are
 * never written to memory.
 *
 * Kernels (SG_PATH_AUTO): M <= 2, the CUDA-core stream, each CTA reading the gate
 * and up rows of its outputs once for all M rows (paired FMAs on gate and up);
 * 3 <= M <= 64, the swapped tcgen05 kernel with a gate and an up accumulator
 * side by side in TMEM (64 outputs per tile); M > 64, the tcgen05 GEMM with each
 * tile's 256 B rows made of 128 rows of Wg and 128 of Wu (128 output columns per
 * tile), on CTA pairs from M = 256 as in gemm_bf16.  Same errors as gemm_bf16 (a
 * null or misaligned Wu as for B).  K = 0 gives C = 0.
 */
SG_API int gemm_bf16_swiglu(const void *A, const void *Wg, const void *Wu, void *C,
                     int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldw, int64_t ldc, sg_stream_t stream);

/* gemm_bf16_swiglu with the kernel named: SG_PATH_AUTO, SG_PATH_GEMM or
 * SG_PATH_GEMM_PAIR (any M), or SG_PATH_CUDA_CORE / SG_PATH_TENSOR_CORE (M <= 64);
 * others SG_ERR_INVALID_ARG. */
SG_API int gemm_bf16_swiglu_path(const void *A, const void *Wg, const void *Wu, void *C,
                          int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldw, int64_t ldc, int path, sg_stream_t stream);

/*
 * gemm_bf16_residual -- a projection with its residual added in the epilogue:
 *
 *     C[m, n] = sum_k A[m, k] B[n, k] + R[m, n],
 *
 * the down projection of the MLP block with the residual stream added (the pages'
 * second fused MLP epilogue).  R is M x N bf16 with leading dimension ldr (>= N, a
 * multiple of 8, 16-byte aligned); R may be C itself (in place, then ldr == ldc);
 * any other overlap of R, C, A or B is undefined.  The sum is fp32 (the
 * accumulator plus R's value) and is rounded to bf16 once.  The kernels are
 * gemm_bf16's (the same automatic choice); K = 0 gives C = R.  Errors as
 * gemm_bf16, plus SG_ERR_INVALID_ARG for a null R, ldr < N or ldr != ldc in place,
 * and SG_ERR_MISALIGNED for a misaligned R or ldr.
 */
SG_API int gemm_bf16_residual(const void *A, const void *B, const void *R, void *C,
                       int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldr, int64_t ldc, sg_stream_t stream);

/* gemm_bf16_residual with the kernel named (paths as gemm_bf16_path). */
SG_API int gemm_bf16_residual_path(const void *A, const void *B, const void *R, void *C,
                            int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int64_t ldr, int64_t ldc, int path, sg_stream_t stream);

/*
 * gemv_bf16_batched -- several skinny GEMMs that share their activations, in one
 * launch: for i < count, C_i[m, n] = sum_k A[m, k] B_i[n, k] (1 <= M <= 64).
 *
 * The decode step's projections that read the same input (Q, K and V; several
 * small weights of one layer) then cost one launch and fill the GPU together
 * (the pages' "next" step: amortise the ~2 us a launch costs a decode step).  A is
 * M x K (lda); B[i] is N[i] x K (ldb[i]); C[i] is M x N[i] (ldc[i]); count <= 8; the
 * arrays are host arrays of device pointers and sizes.  path: SG_PATH_AUTO (the
 * CUDA-core stream for M = 1, else tcgen05), SG_PATH_CUDA_CORE (each matrix
 * gets its own run of CTAs, in proportion to its rows) or SG_PATH_TENSOR_CORE.  Each C_i is exactly what gemv_bf16 gives for (A, B_i)
 * with the same kernel, up to the order of the fp32 sums.  Errors as gemv_bf16
 * for each matrix, plus SG_ERR_INVALID_ARG for count outside 1..8 or null arrays.
 */
SG_API int gemv_bf16_batched(const void *A, int64_t M, int64_t K, int64_t lda,
                      const void *const *B, const int64_t *N, const int64_t *ldb,
                      void *const *C, const int64_t *ldc, int count, int path, sg_stream_t stream);

/*
 * gemm_nvfp4 -- dense W4A4 block-scaled GEMM with FP16 output:
 *
 *   C[m, n] = alpha * sum_k a[m, k] sa[m, k/16] b[n, k] sb[n, k/16]
 *
 * the operation the gemm3 benchmarks page times ("Implementations": packed NVFP4
 * operands, E4M3 scales over 16-element blocks, alpha = 1, FP16 output), on the
 * tcgen05 block-scaled MMA.
 *
 * Operands (device pointers):
 *   A    M rows of K/2 bytes, pitch lda bytes: element a[m, k] is the E2M1 code in
 *        byte k/2 of row m, the low nibble for even k (E2M1: sign, 2 exponent bits
 *        with bias 1, 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6).
 *   B    N rows of K/2 bytes, pitch ldb bytes, the same encoding (a weight matrix
 *        [out, in], as for gemm_bf16).
 *   SFA  E4M3 scales of A in scale atoms (below); sa[m, j] scales a[m, 16j .. 16j+15].
 *   SFB  E4M3 scales of B in scale atoms.
 *   C    M x N fp16 (IEEE binary16 bit patterns), pitch ldc elements.
 * A scale atom is 512 bytes holding 128 rows x 4 blocks (64 of K): row r, block j
 * at byte (r % 32) * 16 + (r / 32) * 4 + j.  For a matrix of `rows` rows, atom
 * (row block R, k chunk c) sits at byte (R * ceil(K/64) + c) * 512 of its buffer,
 * nvfp4_scale_bytes(rows, K) bytes in all.  nvfp4_pack_scales builds this layout
 * from plain row-major scales.  Atom bytes past K/16 blocks or past the last row
 * must hold finite scales (nvfp4_pack_scales writes 0): the kernel multiplies them
 * by zero-filled operands, and a NaN scale would make the product NaN.
 *
 * Arithmetic: every product is exact in fp32 (at most 12 significant bits), the
 * sums are fp32 in an unspecified order, then multiplied by alpha and rounded to
 * fp16 (nearest even).  Results are the same on every run.
 *
 * Requirements: K a multiple of 16; lda, ldb >= K/2 and multiples of 16; ldc >= N
 * and a multiple of 8; A, B, SFA, SFB, C 16-byte aligned.  Errors: SG_ERR_INVALID_ARG
 * (negative or too large sizes, K % 16 != 0, short pitches, null pointers),
 * SG_ERR_MISALIGNED, SG_ERR_UNSUPPORTED_DEVICE, SG_ERR_CUDA, SG_ERR_TIMEOUT (on
 * the next sg_check_device_errors).  M = 0 or N = 0: no work.  K = 0: C := 0.
 * Asynchronous on `stream`; graph-capturable after a first call.
 */
SG_API int gemm_nvfp4(const void *A, const void *SFA, const void *B, const void *SFB, void *C,
                      int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                      float alpha, sg_stream_t stream);

/* gemm_nvfp4 with the kernel named: SG_PATH_GEMM (one CTA per 128 x 256 tile),
 * SG_PATH_GEMM_PAIR (a cluster of two CTAs per 256 x 256 tile, tcgen05
 * cta_group::2) or SG_PATH_AUTO (gemm_nvfp4's choice: the one-CTA kernel).  Any
 * other path: SG_ERR_INVALID_ARG.  The two kernels add the fp32 products in
 * different orders, so their results may differ in the last bits; each gives the
 * same bits on every run. */
SG_API int gemm_nvfp4_path(const void *A, const void *SFA, const void *B, const void *SFB, void *C,
                           int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                           float alpha, int path, sg_stream_t stream);

/* Bytes of a scale-atom buffer for `rows` rows and K elements of K (-1 if negative). */
SG_API int64_t nvfp4_scale_bytes(int64_t rows, int64_t K);

/*
 * nvfp4_pack_scales -- the repacking step: plain row-major E4M3 scales (rows x
 * K/16 bytes, pitch ld bytes) to the scale atoms gemm_nvfp4 reads
 * (nvfp4_scale_bytes(rows, K) bytes; padding written as 0).  One kernel on
 * `stream`; device pointers.  Errors: SG_ERR_INVALID_ARG (negative sizes,
 * K % 16 != 0, ld < K/16, null pointers when rows * K > 0), SG_ERR_CUDA.
 */
SG_API int nvfp4_pack_scales(const void *plain, int64_t rows, int64_t K, int64_t ld, void *atoms,
                             sg_stream_t stream);

/*
 * attention_bf16 -- fused scaled dot-product attention (forward), the attention
 * kernel of the spark-kernels page ("attention": flash attention with the online
 * softmax, S = Q K^T and O += P V on the tensor cores, P rounded to bf16 for the
 * second product, causal tiles above the diagonal skipped):
 *
 *   O[b, i, h, :] = sum_j softmax_j(scale * Q[b, i, h, :] . K[b, j, g, :]) V[b, j, g, :]
 *
 * over the keys j visible to query i, with g = h / (heads / kv_heads) (grouped
 * query heads share a key/value head).  Key j is visible when j < seq_k and, if
 * `causal` is non-zero, j <= i + (seq_k - seq_q): the queries are the last seq_q
 * positions of a sequence whose first seq_k positions are the keys (the lower
 * triangle when seq_q = seq_k, a decode step against a cache when seq_q < seq_k).
 * A query that sees no key gets O = 0.
 *
 * Layout (device pointers, bf16 bit patterns, row-major):
 *   Q  batch * seq_q rows (token b * seq_q + i) of heads * head_dim elements:
 *      head h at columns [h * head_dim, (h + 1) * head_dim); row pitch ldq.
 *   K, V  batch * seq_k rows (token b * seq_k + j) of kv_heads * head_dim
 *      elements, pitches ldk and ldv.
 *   O  like Q, pitch ldo (written; Q, K, V only read).
 * The caller owns every buffer; nothing is allocated per call (the library's
 * per-device workspace is allocated on a first call).  K and V must be finite:
 * keys past seq_k inside a tile are masked, but their values are multiplied by 0.
 *
 * Kernels: the tcgen05 kernel above, or, for a decode step whose query rows per
 * key/value head (seq_q * heads / kv_heads) are at most 4, a CUDA-core kernel
 * that streams K and V once with plain 16-byte loads, each CTA taking one key
 * range of one (batch, kv head) for all of that head's query rows; key ranges
 * are merged from fp32 partials (log2-sum-exp weights), as the tcgen05 kernel's
 * key splits are.  attention_bf16 picks the CUDA-core kernel for 1, 3 or 4 rows
 * (measured faster there; 2 rows run faster on the tcgen05 kernel).
 *
 * Arithmetic: scores and the softmax in fp32 (exp2 of log2-scaled scores), the
 * weights rounded to bf16 for the tcgen05 kernel's P V product (kept in fp32 by
 * the CUDA-core kernel), fp32 accumulation, one bf16 rounding of O (nearest
 * even).  Results are the same on every run.
 *
 * Requirements: head_dim = 128; heads a multiple of kv_heads; ldq, ldo >= heads *
 * head_dim and ldk, ldv >= kv_heads * head_dim, all multiples of 8; pointers
 * 16-byte aligned; scale finite.  Errors: SG_ERR_INVALID_ARG (negative sizes,
 * head_dim != 128, heads % kv_heads != 0, short pitches, null pointers, sizes past
 * 32-bit row indices), SG_ERR_MISALIGNED, SG_ERR_UNSUPPORTED_DEVICE, SG_ERR_CUDA,
 * SG_ERR_TIMEOUT (on the next sg_check_device_errors).  batch, seq_q or heads = 0:
 * no work.  seq_k = 0: O := 0.  Asynchronous on `stream`; graph-capturable after
 * a first call.
 */
SG_API int attention_bf16(const void *Q, const void *K, const void *V, void *O, int64_t batch, int64_t seq_q,
                          int64_t seq_k, int64_t heads, int64_t kv_heads, int64_t head_dim, int64_t ldq,
                          int64_t ldk, int64_t ldv, int64_t ldo, int causal, float scale, sg_stream_t stream);

/* attention_bf16 with the kernel named: SG_PATH_AUTO (attention_bf16's choice),
 * SG_PATH_TENSOR_CORE (the tcgen05 kernel, any shape) or SG_PATH_CUDA_CORE (the
 * decode kernel; SG_ERR_INVALID_ARG unless seq_q * heads / kv_heads <= 4).  Any
 * other path: SG_ERR_INVALID_ARG.  Otherwise as attention_bf16. */
SG_API int attention_bf16_path(const void *Q, const void *K, const void *V, void *O, int64_t batch,
                               int64_t seq_q, int64_t seq_k, int64_t heads, int64_t kv_heads, int64_t head_dim,
                               int64_t ldq, int64_t ldk, int64_t ldv, int64_t ldo, int causal, float scale,
                               int path, sg_stream_t stream);

/*
 * gemv_bf16_noalloc -- gemv_bf16 on the CUDA-core kernel (SG_PATH_CUDA_CORE),
 * for callers that cannot allocate device memory.  The pages have no
 * counterpart: this entry point exists for integration, not for the method.
 *
 * Who needs it: gemv_bf16 allocates its split-K workspace with cudaMalloc on
 * the first call.  Some callers cannot allow that: an engine whose device memory
 * belongs to its own pool allocator (where a raw cudaMalloc fails or fragments
 * the pool), a plug-in inside a host framework that forbids raw allocations, or
 * code that must not pay the implicit device synchronisation of cudaMalloc.
 * This call makes no cudaMalloc, cudaFree or other allocating call.  Its scratch
 * (split-K fp32 partial sums and arrival counters) is a fixed array in the
 * library's device image, SG_NOALLOC_PARTIAL_BYTES + 4 * SG_NOALLOC_COUNTERS
 * bytes, which every GPU that loads the library holds until the process exits.
 *
 * Arguments, layout and errors are those of gemv_bf16 (1 <= M <= 64; results
 * equal gemv_bf16_path(..., SG_PATH_CUDA_CORE, ...)).  A call whose K split would
 * need more partial sums or counters than the array holds returns
 * SG_ERR_INVALID_ARG before launching anything.
 *
 * The first call on each device looks up the array's device address (it must be
 * made with that device current), so make that first call before any stream
 * capture.  Every call shares the one array and finds the previous call's
 * contents in it; each call clears the counters it uses before its kernel runs.
 * Calls whose kernels overlap on the GPU (different streams, or different host
 * threads) race on the array and may return wrong results: serialise them.
 */
#define SG_NOALLOC_PARTIAL_BYTES (1u << 20)
#define SG_NOALLOC_COUNTERS 4096u
SG_API int gemv_bf16_noalloc(const void *A, const void *B, void *C,
                             int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, int64_t ldc, sg_stream_t stream);

/*
 * gemm_bf16_path -- gemm_bf16 with the kernel chosen by the caller:
 * SG_PATH_AUTO (gemm_bf16's choice), SG_PATH_GEMM (one CTA per tile: 128 x 128
 * when those tiles fit in one wave of SMs, else 128 x 256),
 * SG_PATH_GEMM_PAIR (a cluster of two CTAs on two SMs per 256 x 256 tile, each
 * CTA loading half of the A rows and half of the B rows of the tile), or, for
 * M <= 64, SG_PATH_CUDA_CORE / SG_PATH_TENSOR_CORE as in gemv_bf16_path.  Any M
 * is accepted by the two GEMM kernels.  Same arguments and errors as gemm_bf16;
 * an unknown path, or a skinny path with M > 64, is SG_ERR_INVALID_ARG.
 */
SG_API int gemm_bf16_path(const void *A, const void *B, void *C,
                          int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int64_t ldc, int path, sg_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
SG_API const char *sg_status_string(int status);

/* The raw cudaError_t of the most recent SG_ERR_CUDA on this host thread (0 if none). */
SG_API int sg_last_cuda_error(void);

/*
 * sg_check_device_errors -- synchronises `stream`, then reads and clears the
 * current device's kernel error word.  Returns SG_OK, SG_ERR_TIMEOUT (a kernel
 * gave up on a bounded wait; its output is undefined and the workspace counters
 * are reset here so later calls are correct), or SG_ERR_CUDA.  If `detail` is not
 * NULL it receives {code, block, warp, where} of the first recorded error.
 */
SG_API int sg_check_device_errors(sg_stream_t stream, uint32_t detail[4]);

/*
 * sg_set_wait_timeout_ns -- upper bound on any single in-kernel wait (mbarrier
 * phases).  Default 2e9 ns.  Values below 1e6 are raised to 1e6.  Applies to
 * launches made after the call, on every device.
 */
SG_API void sg_set_wait_timeout_ns(uint64_t ns);

/*
 * sg_debug_inject_missing_tx -- failure injection for tests of the bounded
 * waits.  The next launch on any device of the tcgen05 GEMM (gemm_bf16 with
 * M > 64), the one-CTA NVFP4 GEMM or the attention kernel arms the first
 * pipeline stage (the first K tile, for attention) of every CTA with `bytes`
 * more than its copies deliver, so the MMA issuer's wait can never complete:
 * the kernel gives up
 * after the wait bound (sg_set_wait_timeout_ns), records the timeout, unwinds
 * and exits, and sg_check_device_errors then returns SG_ERR_TIMEOUT.  The
 * output of that launch is undefined.  bytes = 0 cancels a pending injection.
 * The injection is consumed by one launch.
 */
SG_API void sg_debug_inject_missing_tx(uint32_t bytes);

/* --------------------------------------------------------------------------
 * Planning (host only; no CUDA call is made, usable without a GPU)
 * -------------------------------------------------------------------------- */
typedef struct {
    int32_t path;       /* sg_path the call takes */
    int32_t tile_m;     /* output rows per tile (MMA M side; weight rows if swapped) */
    int32_t tile_n;     /* output columns per tile (MMA N side) */
    int32_t tile_k;     /* K per pipeline stage (64 for tcgen05 paths) */
    int32_t tiles_m, tiles_n, k_steps;
    int32_t grid;       /* CTAs launched */
    int32_t dp_tiles;   /* whole tiles, round-robin over the grid */
    int32_t sk_tiles;   /* tiles split by Stream-K */
    int64_t sk_units;   /* sk_tiles * k_steps */
    int32_t group_m;    /* raster group height */
    int32_t stages;     /* shared-memory ring depth */
    int32_t split_k;    /* CUDA-core path: K slices per row group; tensor-core skinny
                           path and bf16 GEMM paths: k pieces per tile, one CTA (or
                           cluster) each, every one resident at once (0: persistent
                           schedule); else 0 */
    int32_t rows_per_cta; /* CUDA-core path: weight rows per CTA */
    double wave_efficiency; /* of one tile per CTA, (ctas/slots)/ceil(ctas/slots) */
    int32_t cluster_size; /* CTAs per schedule unit: 2 for SG_PATH_GEMM_PAIR, else 1 */
    int32_t ctas_per_sm;  /* CTAs the kernel keeps resident on one SM */
    int32_t prefetch_steps; /* weights each CTA pulls into L2 before it waits for the
                               previous work in the stream (a hint; reads nothing into
                               the result): k-steps on the tensor-core skinny path, row
                               passes (0 or 1) on the CUDA-core path; else 0 */
} sg_plan_info;

/*
 * sg_plan -- the launch plan gemm_bf16_path would use for this shape and `entry`
 * (an sg_path; 0 = gemm_bf16's automatic choice) on a device with `num_sms` SMs.
 * For the paired GEMM, `grid` counts clusters (each of cluster_size CTAs).
 * Returns SG_OK or SG_ERR_INVALID_ARG.
 */
SG_API int sg_plan(int64_t M, int64_t N, int64_t K, int32_t num_sms, int32_t entry, sg_plan_info *out);

/* sg_plan_swiglu -- the launch plan of gemm_bf16_swiglu_path for `entry` (an
 * sg_path it accepts).  GEMM plans: tile_n counts output columns (each from
 * tile_n gate and tile_n up weight rows); tensor-core skinny plans: tile_m
 * counts outputs (each from one gate and one up weight row). */
SG_API int sg_plan_swiglu(int64_t M, int64_t N, int64_t K, int32_t num_sms, int32_t entry, sg_plan_info *out);

/* The plan gemm_nvfp4_path uses for `path` (SG_PATH_AUTO, SG_PATH_GEMM or
 * SG_PATH_GEMM_PAIR): whole tiles round-robin, 256 of K per stage (tile_k counts
 * fp4 elements); 128 x 256 tiles over one CTA per SM (SG_PATH_GEMM), or 256 x 256
 * tiles over clusters of two CTAs (SG_PATH_GEMM_PAIR; `grid` counts clusters).
 * SG_PATH_AUTO takes the one-CTA kernel.  num_sms >= 2. */
SG_API int sg_plan_nvfp4(int64_t M, int64_t N, int64_t K, int32_t num_sms, int32_t path, sg_plan_info *out);

/*
 * sg_plan_item -- work item `index` of CTA `cta` under a tcgen05 plan from sg_plan:
 * out = {tile, k0, k1, piece, npieces, slot, sk_index, tile_row, tile_col}.
 * Returns the CTA's item count, or -1 if cta/index are out of range.
 */
SG_API int sg_plan_item(const sg_plan_info *plan, int32_t cta, int32_t index, int32_t out[9]);

/* Wave efficiency (ctas / slots) / ceil(ctas / slots) (UwULLM kernel-dev, budget 4). */
SG_API double sg_wave_efficiency(int64_t ctas, int64_t slots);

/* --------------------------------------------------------------------------
 * Roofline microbenchmarks (spark-kernels, "how things are measured": the
 * card's own peaks are measured, not quoted).  Each runs on `stream`, times
 * itself with CUDA events and synchronises `stream` before returning.
 * -------------------------------------------------------------------------- */
typedef struct {
    int32_t sm_count;
    int32_t cc_major, cc_minor;
    int32_t smem_optin_bytes;   /* max dynamic shared memory per block */
    int32_t l2_bytes;
    int64_t global_mem_bytes;
    int32_t clock_khz;          /* cudaDevAttrClockRate */
    int32_t mem_clock_khz;
    int32_t mem_bus_bits;
} sg_device_info;

/* Device properties of the current device (the pages' rule: query, never hard-code). */
SG_API int sg_device_query(sg_device_info *out);

/*
 * sg_bench_tcgen05_peak -- every SM runs one CTA issuing back-to-back
 * tcgen05.mma.kind::f16 128x256x16 (bf16 in, fp32 accumulate) from operands
 * resident in shared memory into tensor memory, `iters` MMAs per CTA.
 * Outputs dense TFLOP/s (2*128*256*16 per MMA) and the SM clock in MHz derived
 * from clock64 over %globaltimer during the loop.
 */
SG_API int sg_bench_tcgen05_peak(int64_t iters, double *tflops, double *sm_mhz, sg_stream_t stream);

/*
 * sg_bench_copy -- device-to-device cudaMemcpyAsync of `bytes` from src to dst,
 * `reps` times; *gbps = 2 * bytes / median time (read + write counted).
 */
SG_API int sg_bench_copy(void *dst, const void *src, int64_t bytes, int32_t reps, double *gbps, sg_stream_t stream);

/*
 * sg_bench_read -- a kernel that streams `bytes` (multiple of 16) with 16-byte
 * loads and reduces them to one word (written to sink, 16 bytes of device memory);
 * *gbps = bytes / median time over `reps` launches.
 */
SG_API int sg_bench_read(const void *src, int64_t bytes, int32_t reps, void *sink, double *gbps, sg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SKINNY_GEMM_H */
