/*
 * bsq.h -- C ABI of libbsq: block-scaled quantization of BF16 activations to
 * NVFP4, MXFP4 and MXFP8 with the scale factors written in the 5D TCGEN
 * (tcgen05 block-scaled MMA) layout, for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (Modular "block_scaled_quantization" pages):
 *   - "block_scaled_quantization" module page, function list: quantizers
 *     for the NVFP4, MXFP4 and MXFP8 formats; block_scales_interleave, which
 *     rearranges rank-2 scales to the 5D TCGEN order the tensor cores read;
 *     block_scaled_matmul_with_epilogue: callers allocate the outputs;
 *   - quantize_dynamic_scaled_async_fp4_kernel: per-group scale factors,
 *     packed FP4 elements, FP32 tensor_sf, SF_VECTOR_SIZE;
 *   - grouped_quantize_dynamic_scaled_fp4_async_kernel: per-expert tiles
 *     found by searching row_offsets / scales_offsets with a whole warp
 *     (uint32), expert_ids (int32), per-expert FP32 sf_tensor, optional int32
 *     row_indices, k_tiles_per_block column tiles per block.
 *
 * Formats and conventions (the pages name but do not define them; these are
 * the readings this library implements bit-exactly):
 *   NVFP4  E2M1 elements, one E4M3 scale per 16 elements.  Per block:
 *          s = fl32(fl32(amax/6) * tensor_sf) -> E4M3 (nearest-even, satfinite);
 *          os = (decoded scale == 0) ? 0 : fl32(tensor_sf / decoded scale);
 *          q_i = E2M1(fl32(x_i * os)).
 *   MXFP4  E2M1 elements, one E8M0 scale per 32; MXFP8 E4M3 elements, one E8M0
 *          scale per 32.  Per block: s = fl32(amax/Qmax) (Qmax 6 / 448),
 *          e = ceil(log2 s) clamped to [-127,127] (-127 when s == 0),
 *          scale byte e+127, q_i = encode(fl32(x_i * 2^-e)).
 *   Element encodes round to nearest, ties to the even code, saturate to the
 *   largest finite magnitude and keep the sign bit (also of zero).
 *   FP4 packing: element 2k in the low nibble of byte k.
 *   Packed output: row-major, packed_row_bytes(fmt, K) bytes per row, rows
 *   contiguous (no padding between rows).
 *   5D scale layout, shape (ceil(rows/128), ceil(S/4), 32, 4, 4) bytes with
 *   S = K/SF: the byte of (row m, scale column s) lives at
 *     ((m/128)*Kt + s/4)*512 + (m%32)*16 + ((m%128)/32)*4 + (s%4),
 *   Kt = ceil(S/4).
 *   NaN or Inf inputs are outside the contract (results undefined).
 *
 * Ownership and execution: every pointer argument named *_dev is device
 * memory allocated by the caller; the library allocates nothing and keeps no
 * pointer after a call returns.  Compute calls are asynchronous on `stream`
 * (a cudaStream_t; NULL = the legacy default stream) of the calling thread's
 * current CUDA device; they return after enqueueing.
 *
 * Errors: every function returns a bsq_status and never throws.  Arguments the
 * host can check are checked before anything is enqueued (nothing is launched
 * on error).  Device-resident metadata of the grouped call is bounds-checked
 * on the device: an inconsistent entry skips the affected rows and records
 * BSQ_ERR_VALUE in the per-device error word, readable with
 * bsq_device_error().  Kernels that wait on asynchronous copies bound every
 * wait (about one second); an expired wait records BSQ_ERR_TIMEOUT there.
 */
#ifndef BSQ_H
#define BSQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BSQ_API __attribute__((visibility("default")))
#else
#define BSQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BSQ_NVFP4 = 0, /* E2M1 x16 + E4M3 scale + FP32 tensor_sf */
  BSQ_MXFP4 = 1, /* E2M1 x32 + E8M0 scale */
  BSQ_MXFP8 = 2  /* E4M3 x32 + E8M0 scale */
} bsq_format;

typedef enum {
  BSQ_OK = 0,
  BSQ_ERR_NULL = 1,    /* a required pointer is NULL */
  BSQ_ERR_SHAPE = 2,   /* negative size, K not a multiple of 32, ld too small, ... */
  BSQ_ERR_ALIGN = 3,   /* a pointer or row stride breaks the alignment stated below */
  BSQ_ERR_VALUE = 4,   /* bad scalar (format, tensor_sf, k_tiles_per_block, G) or bad device metadata */
  BSQ_ERR_CUDA = 5,    /* a CUDA runtime / driver call failed */
  BSQ_ERR_TIMEOUT = 6  /* a bounded device-side wait expired */
} bsq_status;

/* Library version, (major << 16) | minor. */
BSQ_API int32_t bsq_version(void);

/* Human-readable name of a status code (static string, never NULL). */
BSQ_API const char* bsq_status_string(int32_t status);

/* Elements covered by one scale factor: 16 (NVFP4) or 32 (MXFP4 / MXFP8);
 * 0 for an unknown format. */
BSQ_API int32_t bsq_block_size(int32_t fmt);

/* Bytes of one packed output row: K/2 for NVFP4 / MXFP4, K for MXFP8;
 * 0 for an unknown format or K < 0. */
BSQ_API int64_t bsq_packed_row_bytes(int32_t fmt, int64_t K);

/* Bytes of a 5D scale buffer for `rows` rows of K elements:
 * ceil(rows/128) * ceil(K/SF/4) * 512; 0 for bad arguments. */
BSQ_API int64_t bsq_scales5d_bytes(int32_t fmt, int64_t rows, int64_t K);

/*
 * Dense quantize: an (M, K) BF16 matrix -> packed elements + 5D scales.
 * (quantize_dynamic_scaled_fp4fp8 / quantize_dynamic_scaled_async_fp4_kernel)
 *
 *   fmt           bsq_format.
 *   in_dev        BF16 input, row r at in_dev + r*ld_in elements; 16-byte aligned.
 *   M, K          rows and columns; M >= 0, K >= 0, K % 32 == 0.  M == 0 or
 *                 K == 0 is a no-op.  M < 2^31.
 *   ld_in         input row stride in elements; ld_in >= K, ld_in % 8 == 0.
 *   out_dev       packed output, M * bsq_packed_row_bytes(fmt, K) bytes;
 *                 16-byte aligned.
 *   scales5d_dev  bsq_scales5d_bytes(fmt, M, K) bytes; every byte is written
 *                 (padding rows / columns of the last tiles get 0x00).
 *   tensor_sf     NVFP4 per-tensor scale (finite, > 0); ignored for MX.
 */
BSQ_API int32_t bsq_quantize(int32_t fmt, const void* in_dev, int64_t M, int64_t K, int64_t ld_in,
                     void* out_dev, void* scales5d_dev, float tensor_sf, void* stream);

/*
 * Grouped per-expert quantize (grouped_quantize_dynamic_scaled_fp4_async_kernel).
 *
 *   in_dev              BF16 source rows (in_rows x K, stride ld_in elements,
 *                       16-byte aligned, ld_in % 8 == 0).
 *   row_offsets_dev     uint32[G+1], non-decreasing, row_offsets[0] == 0:
 *                       group g owns destination rows [row_offsets[g], row_offsets[g+1]).
 *   scales_offsets_dev  uint32[G+1], non-decreasing multiples of 128,
 *                       scales_offsets[0] == 0, scales_offsets[g+1]-scales_offsets[g]
 *                       >= row count of g: first 5D scale row of group g.
 *   expert_ids_dev      int32[G]: expert of group g; a negative id skips the group.
 *   sf_dev              float[num_experts]: NVFP4 tensor_sf per expert
 *                       (may be NULL for MX formats).
 *   num_experts         length of sf_dev (>= 1 for NVFP4; ignored for MX).
 *   row_indices_dev     int32[total_rows] or NULL: destination row d reads source
 *                       row row_indices[d] (NULL: source row d).
 *   G                   number of groups, 0 <= G <= 1<<20 (0 = no-op).
 *   total_rows          destination rows allocated in out_dev; the device
 *                       checks row_offsets[G] <= total_rows.
 *   total_scale_rows    5D scale rows allocated (multiple of 128); the device
 *                       checks scales_offsets[G] <= total_scale_rows.
 *   out_dev             total_rows * packed_row_bytes bytes: row d is written
 *                       iff d belongs to a group with a non-negative expert id.
 *   scales5d_dev        bsq_scales5d_bytes(fmt, total_scale_rows, K) bytes: each
 *                       written row gets all ceil(S/4)*4 scale bytes (padding
 *                       columns 0x00); padding rows are not written.
 *   k_tiles_per_block   1, 2, 4 or 8 column tiles (64 columns for NVFP4, 128
 *                       for MX) handled by one unit of work of the latency
 *                       kernel (a warp), or 0: chosen by the library (the
 *                       fewest that keep the latency kernel's grid within
 *                       four blocks per SM, else 8); the streaming kernel's
 *                       thread blocks take fixed runs of 7168 columns.
 *                       Results do not depend on it.
 * Device checks (error word BSQ_ERR_VALUE, the affected rows are skipped):
 * a source row index outside [0, in_rows); row_offsets[G] > total_rows;
 * scales_offsets[G] > total_scale_rows; scales_offsets[0] != 0; a group with
 * more rows than its padded scale rows; an NVFP4 expert id >= num_experts.
 */
BSQ_API int32_t bsq_grouped_quantize(int32_t fmt, const void* in_dev, int64_t in_rows, int64_t K,
                             int64_t ld_in, const uint32_t* row_offsets_dev,
                             const uint32_t* scales_offsets_dev, const int32_t* expert_ids_dev,
                             const float* sf_dev, int32_t num_experts,
                             const int32_t* row_indices_dev, int32_t G,
                             int64_t total_rows, int64_t total_scale_rows, void* out_dev,
                             void* scales5d_dev, int32_t k_tiles_per_block, void* stream);

/* Kernel of the grouped quantize. */
typedef enum {
  BSQ_GROUPED_AUTO = 0,    /* LATENCY when total_rows <= 16 * G; else TOKEN when row_indices is
                              given, G <= 1024, total_rows >= 2 * in_rows and in_rows <= 8 * K;
                              else STREAM */
  BSQ_GROUPED_STREAM = 1,  /* one thread block per 32 destination rows x a run of scale blocks,
                              a warp per row at a time (groups of many rows) */
  BSQ_GROUPED_LATENCY = 2, /* one warp per 2 destination rows (groups of a few rows) */
  BSQ_GROUPED_TOKEN = 3    /* token-major: each source row read once and quantized into all of
                              its destination rows (gathers that reuse source rows, e.g. top-k
                              routing); one block per SM, each scanning row_indices; needs
                              G <= 1024 and total_rows < 2^32, else STREAM runs */
} bsq_grouped_kernel;

/*
 * bsq_grouped_quantize with an explicit kernel choice (bsq_grouped_kernel);
 * the results are identical whichever kernel runs.  An unknown `kernel`
 * returns BSQ_ERR_VALUE.  The token kernel stores scale bytes with an L2
 * evict_last hint (their 32-byte sectors fill from many rows over the
 * launch); the lines return to normal priority on their next ordinary read,
 * e.g. by the matmul that consumes the scales.
 */
BSQ_API int32_t bsq_grouped_quantize_kernel(int32_t fmt, const void* in_dev, int64_t in_rows,
                                            int64_t K, int64_t ld_in,
                                            const uint32_t* row_offsets_dev,
                                            const uint32_t* scales_offsets_dev,
                                            const int32_t* expert_ids_dev, const float* sf_dev,
                                            int32_t num_experts, const int32_t* row_indices_dev,
                                            int32_t G, int64_t total_rows,
                                            int64_t total_scale_rows, void* out_dev,
                                            void* scales5d_dev, int32_t k_tiles_per_block,
                                            int32_t kernel, void* stream);

/*
 * Workspace bytes of bsq_grouped_quantize_ws: total_scale_rows * ceil(S/4) * 4
 * (one row-major scale row per 5D scale row, the size of the 5D scale
 * buffer) plus 4 bytes per 128-row band, rounded up to 16; 0 for bad
 * arguments.
 */
BSQ_API int64_t bsq_grouped_quantize_workspace_bytes(int32_t fmt, int64_t total_scale_rows, int64_t K);

/*
 * bsq_grouped_quantize_kernel with a caller workspace for the token kernel's
 * NVFP4 scales (an extension; the pages' grouped kernel writes its scales
 * through TMA stores of whole tiles, which a token-major kernel cannot
 * form).  The token kernel (BSQ_GROUPED_TOKEN, or AUTO choosing it)
 * then writes each destination row's scale bytes row-major into the
 * workspace (whole sectors instead of 4 bytes in each of 8 atoms) and a
 * second kernel moves the rows it wrote to their 5D positions with
 * whole-atom stores.  MX formats and the other kernels ignore the
 * workspace.  It pays off when the scale stores dominate (many destination
 * rows per token and long rows, e.g. top-8 routing at K = 7168); with few
 * destination rows per token the second launch costs more than it saves.
 * The bytes of out_dev and scales5d_dev are identical to
 * bsq_grouped_quantize_kernel's (padding scale rows and the rows of skipped
 * groups are not written); on a reported device error the scale bytes of
 * the offending rows are unspecified.
 *
 *   workspace_dev    NULL (then exactly bsq_grouped_quantize_kernel), or
 *                    device memory of at least
 *                    bsq_grouped_quantize_workspace_bytes(fmt, total_scale_rows, K)
 *                    bytes, 16-byte aligned, overlapping no other argument.
 *                    Its contents need no initialisation and are unspecified
 *                    afterwards; it is in use until the call's work on
 *                    `stream` completes (reuse it in stream order).
 *   workspace_bytes  its size.
 * Errors: BSQ_ERR_ALIGN for a misaligned workspace, BSQ_ERR_SHAPE for a
 * smaller one; otherwise as bsq_grouped_quantize_kernel.
 */
BSQ_API int32_t bsq_grouped_quantize_ws(int32_t fmt, const void* in_dev, int64_t in_rows, int64_t K,
                                        int64_t ld_in, const uint32_t* row_offsets_dev,
                                        const uint32_t* scales_offsets_dev, const int32_t* expert_ids_dev,
                                        const float* sf_dev, int32_t num_experts,
                                        const int32_t* row_indices_dev, int32_t G, int64_t total_rows,
                                        int64_t total_scale_rows, void* out_dev, void* scales5d_dev,
                                        int32_t k_tiles_per_block, int32_t kernel, void* workspace_dev,
                                        int64_t workspace_bytes, void* stream);

/*
 * Rank-2 -> 5D scale reinterleave (block_scales_interleave / _fp4 / _fp4_kernel).
 *
 *   scales2d_dev  M rows of S scale bytes, row stride ld bytes (ld >= S).
 *   M, S          M >= 0, S >= 0 (either 0 = no-op).
 *   scales5d_dev  ceil(M/128)*ceil(S/4)*512 bytes, all written (padding 0x00).
 * A pure byte permutation: any 8-bit scale type (E4M3 or E8M0).
 */
BSQ_API int32_t bsq_scales_interleave(const void* scales2d_dev, int64_t M, int64_t S, int64_t ld,
                              void* scales5d_dev, void* stream);

/*
 * Dense quantize with the NVFP4 tensor_sf read from device memory
 * (tensor_sf_dev: one float, e.g. element 1 of bsq_tensor_sf's output), so that
 * computing the scale and quantizing chain on the GPU without a host round
 * trip.  Same arguments and layouts as bsq_quantize otherwise; ignored for MX.
 * A tensor_sf that is not finite and > 0 records BSQ_ERR_VALUE in the device
 * error word and nothing is written.
 */
BSQ_API int32_t bsq_quantize_dynamic(int32_t fmt, const void* in_dev, int64_t M, int64_t K,
                                     int64_t ld_in, void* out_dev, void* scales5d_dev,
                                     const float* tensor_sf_dev, void* stream);

/*
 * NVFP4 per-tensor scale of a BF16 matrix, on the GPU:
 *   amax = max |x| (exact), tensor_sf = fl32(448 * 6 / amax), 1.0 when amax == 0
 *   (+Inf when amax < 2688 / FLT_MAX).
 * (the FP32 tensor_sf of quantize_dynamic_scaled_async_fp4_kernel)
 *   in_dev        BF16, M rows of K elements (K % 8 == 0), row stride ld_in
 *                 elements (multiple of 8), 16-byte aligned.  M == 0 or K == 0:
 *                 amax 0, tensor_sf 1.
 *   out_dev       float[2] = {amax, tensor_sf} (device).
 *   workspace_dev bsq_tensor_sf_workspace_bytes() bytes of caller-allocated
 *                 device scratch, 16-byte aligned, zeroed by the caller once
 *                 before its first use (e.g. cudaMemsetAsync); every call leaves
 *                 it zeroed again, so consecutive calls need no memset.  A
 *                 completion counter that is not zero at launch is reported:
 *                 BSQ_ERR_VALUE in the device error word.  When the stale
 *                 counter is at least the launch's block count nothing is
 *                 written; a smaller stale value can let a block finish the
 *                 reduction before the others have arrived, so the outputs of
 *                 a launch that reported BSQ_ERR_VALUE must be discarded.  A
 *                 stale running maximum under a zero counter is NOT detected
 *                 (it would be folded into amax): a workspace left non-zero
 *                 must be zeroed whole before reuse.
 *                 Calls sharing one workspace must not overlap on the GPU.
 *   The reduction reads in_dev with an L2 evict_last hint, so that a quantize
 *   of the same tensor right after it finds much of it in L2; that quantize
 *   (or any later read with the default policy) returns the lines to normal
 *   priority.
 */
BSQ_API int64_t bsq_tensor_sf_workspace_bytes(void);
BSQ_API int32_t bsq_tensor_sf(const void* in_dev, int64_t M, int64_t K, int64_t ld_in,
                              float* out_dev, void* workspace_dev, int64_t workspace_bytes,
                              void* stream);

/*
 * Per-expert NVFP4 scales of grouped activations, on the GPU: for every
 * expert e, amax_e = max |x| over the source rows of the groups with
 * expert_ids[g] == e (row_indices gather as in bsq_grouped_quantize),
 * sf_dev[e] = fl32(448 * 6 / amax_e), or 1.0 when the expert has no rows.
 * (the per-expert sf_tensor of grouped_quantize_dynamic_scaled_fp4_async_kernel)
 *   num_experts   length of sf_dev (>= 1); expert ids >= num_experts or rows
 *                 outside [0, in_rows) record BSQ_ERR_VALUE and are skipped.
 *   workspace_dev bsq_grouped_tensor_sf_workspace_bytes(num_experts) bytes of
 *                 device scratch, 16-byte aligned, zeroed by the caller once
 *                 before its first use; every call leaves it zeroed again.  A
 *                 stale completion counter is reported as for bsq_tensor_sf
 *                 (BSQ_ERR_VALUE; discard that launch's outputs).  Stale
 *                 per-expert maxima under a zero counter are NOT detected:
 *                 they can only raise an expert's amax, giving a smaller
 *                 scale, so a workspace must be zeroed whole.  Calls sharing
 *                 one workspace must not overlap on the GPU.
 */
BSQ_API int64_t bsq_grouped_tensor_sf_workspace_bytes(int32_t num_experts);
BSQ_API int32_t bsq_grouped_tensor_sf(const void* in_dev, int64_t in_rows, int64_t K,
                                      int64_t ld_in, const uint32_t* row_offsets_dev,
                                      const int32_t* expert_ids_dev,
                                      const int32_t* row_indices_dev, int32_t G,
                                      int64_t total_rows, float* sf_dev, int32_t num_experts,
                                      void* workspace_dev, int64_t workspace_bytes, void* stream);

/*
 * bsq_grouped_tensor_sf without a workspace argument: the same per-expert
 * scales, bit for bit, for callers that cannot allocate device memory where
 * they need them -- a plugin whose C interface hands over only input and
 * output buffers, a host framework that owns all device memory through its
 * own pool and forbids direct cudaMalloc, or a latency-critical loop that
 * cannot take the device-wide synchronization cudaMalloc/cudaFree may cause.
 * The paper has no counterpart of this entry point; it is an addition of this
 * library.
 *   Scratch       a static device array inside this library (16 + 4 *
 *                 BSQ_NOALLOC_MAX_EXPERTS bytes, one copy on every device that
 *                 loads the library, kept until the process exits).  Nothing is
 *                 allocated: no cudaMalloc, cudaFree or allocating library call.
 *   Limit         num_experts <= BSQ_NOALLOC_MAX_EXPERTS; larger returns
 *                 BSQ_ERR_SHAPE before anything is enqueued.  num_experts < 1
 *                 returns BSQ_ERR_VALUE.
 *   First call    on a device looks up the array's device address and the SM
 *                 count (cudaGetSymbolAddress, cudaDeviceGetAttribute) with that
 *                 device current; make it before any stream capture begins.
 *                 The address is kept for the life of the process: after a
 *                 cudaDeviceReset (or any teardown of the device's primary
 *                 context) it belongs to a context that no longer exists, so
 *                 do not call this entry point on that device again.
 *   Sharing       every call on a device uses the same array; each call clears
 *                 the part it uses on `stream` first.  Calls that overlap on the
 *                 GPU (other streams, other host threads, without ordering
 *                 between them) race on the array and give wrong scales.
 * Other arguments, layouts and device-side errors as bsq_grouped_tensor_sf.
 */
#define BSQ_NOALLOC_MAX_EXPERTS 1024
BSQ_API int32_t bsq_grouped_tensor_sf_noalloc(const void* in_dev, int64_t in_rows, int64_t K,
                                              int64_t ld_in, const uint32_t* row_offsets_dev,
                                              const int32_t* expert_ids_dev,
                                              const int32_t* row_indices_dev, int32_t G,
                                              int64_t total_rows, float* sf_dev,
                                              int32_t num_experts, void* stream);

/*
 * Naive block-scaled matmul, a validator of quantized operands (the
 * "block_scaled_quantization" module page lists such a reference matmul,
 * naive_block_scaled_matmul; this is our GPU version of the idea):
 *   c_dev[m*N + n] = sum_k deq(A)[m][k] * deq(B)[n][k]   (FP64, row-major M x N)
 * with deq = decoded element * decoded block scale (/ tensor_sf for NVFP4).
 *   a_packed_dev, b_packed_dev  packed rows of A (M x K) and B (N x K), as
 *                 bsq_quantize writes them (K/2 or K bytes per row).
 *   a_scales5d_dev, b_scales5d_dev  their scales in the 5D layout.
 *   a_tsf, b_tsf  NVFP4 tensor scales (finite, > 0); ignored for MX.
 * K % 32 == 0.  One thread per output, FP64 on the CUDA cores: slow, exact
 * per block, meant for checks, not for throughput.
 */
BSQ_API int32_t bsq_block_scaled_dot(int32_t fmt, const void* a_packed_dev, const void* a_scales5d_dev,
                                     float a_tsf, const void* b_packed_dev, const void* b_scales5d_dev,
                                     float b_tsf, int64_t M, int64_t N, int64_t K, double* c_dev,
                                     void* stream);

/*
 * A producer with the quantize fused into its epilogue: C = A * B^T with BF16
 * operands and FP32 accumulation, C rounded to BF16 (round to nearest even)
 * and quantized block-wise along N exactly as bsq_quantize quantizes a BF16
 * M x N tensor, without storing C.  The block_scaled_quantization module page
 * (function list, block_scaled_matmul_with_epilogue) runs the elementwise
 * epilogues of its block-scaled matmul as a separate kernel; this is the
 * fused form for the quantize.
 *   a_dev         M rows of K BF16 values, row stride lda elements (lda >= K,
 *                 lda % 8 == 0, 16-byte aligned).
 *   b_dev         N rows of K BF16 values (the weight, K-major), row stride
 *                 ldb (ldb >= K, ldb % 8 == 0, 16-byte aligned).
 *   M, N, K       M >= 0 (0 = no-op), N % 128 == 0, K % 32 == 0, K > 0.
 *   tensor_sf     NVFP4 tensor scale (finite, > 0); ignored for MX.
 *   out_dev       M x bsq_packed_row_bytes(fmt, N) packed codes, 16-byte aligned.
 *   scales5d_dev  bsq_scales5d_bytes(fmt, M, N) bytes of 5D scales, all
 *                 written (rows past M in the last 128-row band: 0x00).
 *   c_bf16_dev    optional (NULL = none): M x N BF16 copy of C, row stride N,
 *                 16-byte aligned (for checks: the fused bytes equal
 *                 bsq_quantize applied to it).
 * The mainloop runs on the tcgen05 tensor cores: 128 x 256 tiles, operands
 * staged by TMA, FP32 accumulators in tensor memory, one CTA per SM; a wait
 * that expires records BSQ_ERR_TIMEOUT.  Errors: BSQ_ERR_SHAPE, BSQ_ERR_NULL,
 * BSQ_ERR_ALIGN, BSQ_ERR_VALUE (format or tensor_sf), BSQ_ERR_CUDA (launch).
 */
BSQ_API int32_t bsq_gemm_quantize(int32_t fmt, const void* a_dev, const void* b_dev, int64_t M, int64_t N,
                                  int64_t K, int64_t lda, int64_t ldb, float tensor_sf, void* out_dev,
                                  void* scales5d_dev, void* c_bf16_dev, void* stream);

/*
 * Self-test of the device-side failure path: enqueues a one-warp kernel that
 * waits, with the bounded wait every pipelined kernel here uses, on a
 * barrier nothing will complete.  After about one second the wait gives up
 * and records BSQ_ERR_TIMEOUT in the error word (read it with
 * bsq_device_error); nothing faults or hangs, and the context stays usable.
 */
BSQ_API int32_t bsq_selftest_wait_timeout(void* stream);

/*
 * Synchronize `stream`, then read and clear the current device's error word.
 * *code_out receives BSQ_OK or the first device-side error recorded since the
 * last call (BSQ_ERR_VALUE, BSQ_ERR_TIMEOUT).  Returns BSQ_ERR_CUDA if the
 * synchronization itself fails (e.g. an earlier launch faulted).
 */
BSQ_API int32_t bsq_device_error(void* stream, int32_t* code_out);

#ifdef __cplusplus
}
#endif

#endif /* BSQ_H */
