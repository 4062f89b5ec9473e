/*
 * q4mm.h -- C ABI of libq4mm: weight-only 4-bit quantized matrix multiplies
 *           y = x . dequant(W)^T on one NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers named as device data (x, w, scales, biases, y, out, ids, workspace, ...) are
 *    device pointers in the current CUDA device's address space.  The only host pointers
 *    are the LUT4 codebook (`book`, copied by value into the launch) and output arguments
 *    named `out_*` of the query calls.
 *  - Ownership: the caller owns every buffer, including workspaces.  No call allocates,
 *    frees, or synchronises; every kernel is enqueued on `stream` in call order (a NULL
 *    stream is the legacy default stream).  Calls on one stream see each other's results.
 *  - Layouts are row-major and dense (no strides).  "bf16" arguments are uint16_t bit
 *    patterns of bfloat16 values; "fp16" are IEEE binary16 bit patterns.
 *  - Errors: arguments are checked on the host before anything is enqueued; a failed check
 *    returns a status and launches nothing.  M == 0 (or n_tokens == 0) returns Q4MM_OK
 *    with nothing enqueued.  After enqueueing, a launch failure reported by the CUDA runtime
 *    is returned as Q4MM_ERR_CUDA.  Each call picks one of this library's kernels from the
 *    shape, layout and alignment; none hands work to the CPU or to another library.
 *  - Device-side faults are never raised on purpose: bounded waits that give up, and
 *    routed ids outside [0, n_experts), are recorded in a device error word readable
 *    with q4mm_device_errors().
 *
 * Sources (page title, section) of the operations:
 *   quant_fastkernel.rs  -- onnxruntime-ep-mlx 0.27.4, src/ops/quant_fastkernel.rs: the INT4
 *                           group-32 affine MatMulNBits prefill kernel (module doc "Algorithm",
 *                           kernel source, `eligible`, `try_apply`).
 *   lut4.rs              -- onnxruntime-ep-mlx 0.31.1, src/ops/lut4.rs: `LookupMatMul`, the
 *                           lookup4 kernel source, `execute` and the lookup4 decode kernel.
 *   quantized_matmul_id_ggml.rs -- mlx-native 0.9.0: module doc (routed-matmul definition),
 *                           `quantized_matmul_id_ggml`, `IdMmScratch`, `dispatch_id_mv`,
 *                           `dispatch_id_mm_for_test` (map0 + mm_id stages).
 */
#ifndef Q4MM_H
#define Q4MM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *q4mm_stream_t;

typedef enum q4mm_status {
    Q4MM_OK = 0,
    Q4MM_ERR_INVALID_ARG = 1,  /* null pointer, bad size, size out of range            */
    Q4MM_ERR_UNSUPPORTED = 2,  /* valid request this build does not serve (alignment)   */
    Q4MM_ERR_WORKSPACE = 3,    /* workspace missing or smaller than the size query says */
    Q4MM_ERR_CUDA = 4,         /* the CUDA runtime reported an error                     */
    Q4MM_ERR_DEVICE = 5        /* current device is not compute capability 10.3         */
} q4mm_status;

typedef enum q4mm_dtype { Q4MM_F32 = 0, Q4MM_BF16 = 1, Q4MM_F16 = 2 } q4mm_dtype;

/* Bits of the device error word. */
#define Q4MM_DEVERR_WAIT_TIMEOUT 0x1u  /* a pipeline wait gave up; that output is invalid */
#define Q4MM_DEVERR_BAD_EXPERT 0x2u    /* an id >= n_experts was routed (its row is zero) */
#define Q4MM_DEVERR_F16_RANGE 0x4u     /* a tensor-core mat-mat form (Q4_0, Q8_0), which
                                          forms each weight (q-8)*d or q*d in fp16, met a
                                          block whose |d| could take a weight beyond fp16's
                                          range (|d| >= 8192 for Q4_0, >= 512 for Q8_0).  The
                                          outputs that block feeds are correct if all of its
                                          weights stay below 65520 in magnitude, else not
                                          finite.  x itself is never out of range: each
                                          gathered row is scaled by a power of two. */

/* Static string for a status code (never NULL). */
const char *q4mm_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int q4mm_version(void);

/* Reads the current device's error word into *out_flags (host pointer) and, if clear != 0,
 * resets it.  Synchronises the device (diagnostics only, not for hot loops). */
q4mm_status q4mm_device_errors(uint32_t *out_flags, int clear);

/* Self-test of the bounded waits (diagnostics; the source pages have no counterpart).  Runs
 * one small kernel whose wait on a pipeline barrier that nothing completes gives up after
 * limit_ns nanoseconds (1 .. 10^9), exactly as every pipeline wait of the library gives up
 * after its 2 s limit: it sets Q4MM_DEVERR_WAIT_TIMEOUT, the other waiting warp leaves on the
 * CTA's abort flag, and a bulk copy the kernel started lands before the kernel exits.  src16:
 * device pointer to 16 readable, 16-byte aligned bytes (the copy's source).  Nothing faults
 * or traps; the next calls run normally.  Read the bit with q4mm_device_errors. */
q4mm_status q4mm_selftest_wait_timeout(const void *src16, uint32_t limit_ns, q4mm_stream_t stream);

/* ======================================================================================
 * INT4 group-32 affine MatMulNBits  (quant_fastkernel.rs)
 *   w       uint32 [N, K/8]: element k of row n is bits 4*(k%8)..4*(k%8)+3 of word
 *           w[n][k/8] (low nibble first), an unsigned code q in 0..15.
 *   scales  bf16 [N, K/32], biases bf16 [N, K/32]; bias = -zero_point * scale.
 *   value   W[n][k] = fmaf(q, scales[n][k/32], biases[n][k/32])   (fp32, one rounding)
 *   x       bf16 [M, K];   y bf16 [M, N],  y[m][n] = sum_k x[m][k] * W[n][k].
 * Requirements: N >= 1, K >= 32, K % 32 == 0; w, scales, biases, x, y 16-byte aligned
 * (Q4MM_ERR_UNSUPPORTED otherwise).  Float outputs are fp32-accumulated and rounded to
 * bf16 (nearest even) once.
 * ====================================================================================*/

/* Standalone dequant (the decode-then-GEMM pattern of lut4.rs `decoded_gemm`, for the
 * INT4 format).  out: [N, K] of out_dtype (Q4MM_F32 / Q4MM_BF16 / Q4MM_F16); F32 output is
 * the fmaf value bit for bit, BF16/F16 are that value rounded to nearest even. */
q4mm_status q4_dequant(const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                       int64_t N, int64_t K, void *out, int out_dtype, q4mm_stream_t stream);

/* Decode matmul, 1 <= M <= 16 (tokens).  Streams W once from HBM; split-K partial sums
 * are combined inside a thread-block cluster in a fixed order (deterministic).  Needs no
 * workspace. */
q4mm_status q4_gemv(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                    const uint16_t *biases, uint16_t *y, int64_t M, int64_t N, int64_t K,
                    q4mm_stream_t stream);

/* q4_gemv with launch flags (q4_gemv is q4_gemv_ex with flags = 0).
 *
 * Q4MM_GEMV_STATIC_WEIGHTS: the caller promises that w, scales and biases are not written
 *   by the kernel that precedes this call in the stream.  The call is then launched with
 *   programmatic stream serialization: its CTAs may start while that kernel is still
 *   running and begin streaming W at once; they read x and write y only after that kernel
 *   has completed and its writes are visible, so chaining calls whose x is the previous
 *   call's y (or whose y is the previous call's x) stays correct.  Back-to-back decode
 *   matmuls then overlap one call's weight stream with the previous call's tail.  Results
 *   are bit-identical to flags = 0.  If the preceding kernel does write the weights, the
 *   result is undefined.
 * Unknown flag bits: Q4MM_ERR_INVALID_ARG. */
#define Q4MM_GEMV_STATIC_WEIGHTS 0x1u
q4mm_status q4_gemv_ex(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                       const uint16_t *biases, uint16_t *y, int64_t M, int64_t N, int64_t K,
                       uint32_t flags, q4mm_stream_t stream);

/* Prefill matmul (meant for M > 16; any M >= 1 is served).  Fifth-generation tensor
 * cores: W tiles are dequantised to bf16 in shared memory, x tiles arrive by TMA,
 * fp32 accumulators live in tensor memory. */
q4mm_status q4_gemm(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                    const uint16_t *biases, uint16_t *y, int64_t M, int64_t N, int64_t K,
                    q4mm_stream_t stream);

/* ======================================================================================
 * LUT4: frozen 16-entry codebook, blocked 4-bit  (lut4.rs)
 *   The stored matrix has `rows` x `cols` codes; flat index f = r*cols + c; byte f/2 of
 *   `packed` holds code f: the HIGH nibble for even f, the LOW nibble for odd f.
 *   scales  f32 [ceil(rows*cols / block)], one per `block` consecutive flat elements.
 *   value   W = fl32(book[code] * scales[f / block])  (one fp32 product)
 *   transpose = 1: stored [rows = N, cols = K], W[n][k] at f = n*K + k  (the [N, K/2] layout)
 *   transpose = 0: stored [rows = K, cols = N], W[n][k] at f = k*N + n
 *   book    HOST pointer to 16 floats, copied into the launch.
 *   x bf16 [M, K]  ->  y bf16 [M, N], y[m][n] = sum_k x[m][k] * W[n][k].
 * Requirements: M >= 0, N, K >= 1, block > 0 and even; packed holds ceil(rows*cols/2) bytes;
 * x, y 2-byte aligned, scales 4-byte aligned.  The fast kernels serve transpose = 1 with K % 32 == 0,
 * block % 32 == 0, K % block == 0 and 16-byte aligned x/packed/y (for M <= 16 also 16-byte aligned
 * scales); any other valid layout runs on a general (slower) kernel with the same results.
 * ====================================================================================*/
q4mm_status lut4_matmul(const uint16_t *x, const uint8_t *packed, const float *scales,
                        const float *book, uint16_t *y, int64_t M, int64_t N, int64_t K,
                        int64_t block, int transpose, q4mm_stream_t stream);

/* lut4_matmul with launch flags (lut4_matmul is lut4_matmul_ex with flags = 0).
 * Q4MM_GEMV_STATIC_WEIGHTS: the promise and effect described at q4_gemv_ex, for packed and
 *   scales (the codebook is copied into the launch).  It changes only calls served by the
 *   decode kernels (M <= 16 on the fast layout); other calls launch as with flags = 0.
 *   Results are bit-identical to the same call without this bit.
 * Q4MM_LUT4_ROUND_F16, Q4MM_LUT4_ROUND_BF16 (at most one): the rounded-weight variant of
 *   lut4.rs (`rounded_weight`; the graph casts the decoded weight to half or bfloat16, and for
 *   the adjoint back to float).  Each decoded value W = fl32(book[code] * scale) is rounded to
 *   IEEE binary16 (F16) or bfloat16 (BF16), nearest even, and the matmul multiplies x by that
 *   rounded value: y[m][n] = sum_k x[m][k] * round(W[n][k]), fp32 accumulation, bf16 y.  With
 *   F16, |W| below 2^-25 becomes 0 and |W| of 65520 or more becomes infinity (so y may be
 *   infinite or NaN).  F16 runs on CUDA cores (fp32 FMA); BF16 uses the tensor-core paths
 *   where their operand is exactly the rounded value.  Every layout lut4_matmul accepts is
 *   accepted.  Both bits set: Q4MM_ERR_INVALID_ARG.
 * Unknown flag bits: Q4MM_ERR_INVALID_ARG. */
#define Q4MM_LUT4_ROUND_F16 0x2u
#define Q4MM_LUT4_ROUND_BF16 0x4u
q4mm_status lut4_matmul_ex(const uint16_t *x, const uint8_t *packed, const float *scales,
                           const float *book, uint16_t *y, int64_t M, int64_t N, int64_t K,
                           int64_t block, int transpose, uint32_t flags, q4mm_stream_t stream);

/* Standalone LUT4 decode (lut4.rs lookup4 decode kernel): out [rows, cols] of out_dtype,
 * out[f] = fl32(book[code(f)] * scales[f / block]) (F32 bit for bit; BF16/F16 rounded to
 * nearest even). */
q4mm_status lut4_dequant(const uint8_t *packed, const float *scales, const float *book,
                         int64_t rows, int64_t cols, int64_t block, void *out, int out_dtype,
                         q4mm_stream_t stream);

/* ======================================================================================
 * GGML Q4_0 expert-routed matmul  (quantized_matmul_id_ggml.rs)
 *   x    f32 [n_tokens, K]; one row per token, shared by all of its top_k slots.
 *   w    stacked experts: expert e starts at byte e*expert_stride; within it row n is
 *        K/32 consecutive 18-byte blocks.  Block: fp16 d (little endian), then 16 bytes qs;
 *        element j < 16 is (qs[j] & 15) - 8, element 16+j is (qs[j] >> 4) - 8;
 *        value = (q - 8) * d.
 *   ids  uint32 [n_tokens * top_k]; routed row r = token*top_k + slot uses expert ids[r].
 *   out  f32 [n_tokens * top_k, N]; out[r][n] = sum_k x[r / top_k][k] * W[ids[r]][n][k].
 *        A row whose id is >= n_experts is written as zeros and sets
 *        Q4MM_DEVERR_BAD_EXPERT.
 * ====================================================================================*/

/* Per-expert routed lists (the map0 stage of dispatch_id_mm_for_test).
 *   htpe  uint32 [n_experts]: htpe[e] = number of rows r < n_rows with ids[r] == e.
 *   hids  int32 [n_rows]: expert 0's rows, then expert 1's, ..., each list ascending in r;
 *         expert e's list starts at sum_{e'<e} htpe[e'].  Entries past the total are
 *         left unchanged.
 *   n_invalid  uint32 [1] (device, may be NULL): rows whose id is >= n_experts.
 * Requirements: 1 <= n_rows <= 2^24, 1 <= n_experts <= 1024.  Deterministic. */
q4mm_status q4_0_route(const uint32_t *ids, int64_t n_rows, int64_t n_experts, uint32_t *htpe,
                       int32_t *hids, uint32_t *n_invalid, q4mm_stream_t stream);

/* Bytes of workspace q4_0_matmul_id needs in mat-mat mode (0 in mat-vec mode). */
size_t q4_0_matmul_id_workspace_size(int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                                     int64_t n_experts);

/* Mode: 0 = automatic (mat-mat when n_tokens > Q4MM_MM_ID_THRESHOLD, else mat-vec),
 *       1 = mat-vec (each routed row reads its expert's rows; no workspace),
 *       2 = mat-mat (route, gather each expert's rows, stream each expert's weights once
 *           per 128-row tile through the tensor cores; needs the workspace).
 * The mat-mat form runs on the tensor cores when K % 256 == 0 and w and expert_stride are
 * 16-byte aligned (fp16 operands: each weight (q-8)*d rounded once to fp16, each x row scaled
 * by a power of two and rounded once to fp16; fp32 accumulation), else on the fp32 FMA pipes.
 * Requirements: n_tokens, top_k, N, K, n_experts >= 1; K % 32 == 0; expert_stride >=
 * N*(K/32)*18; x, out 16-byte aligned; workspace (mat-mat) 256-byte aligned and at least
 * q4_0_matmul_id_workspace_size(...) bytes. */
#define Q4MM_MM_ID_THRESHOLD 32
q4mm_status q4_0_matmul_id(const float *x, const void *w, const uint32_t *ids, float *out,
                           int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                           int64_t n_experts, uint64_t expert_stride, int mode,
                           void *workspace, size_t workspace_bytes, q4mm_stream_t stream);

/* Fused SwiGLU + expert-routed Q4_0 mat-vec (quantized_matmul_id_ggml.rs,
 * quantized_matmul_id_swiglu_q4_0 and its doc comment): the down projection of a MoE FFN
 * in one launch, without writing silu(gate) * up to memory.
 *   gate, up  f32 [n_tokens * top_k, K]: one row per ROUTED row r = token*top_k + slot.
 *   w, ids    as for q4_0_matmul_id.
 *   out       f32 [n_tokens * top_k, N];
 *             out[r][n] = sum_k W[ids[r]][n][k] * silu(gate[r][k]) * up[r][k],
 *             silu(z) = z / (1 + exp(-z)), formed in fp32.  A row whose id is >= n_experts
 *             is written as zeros and sets Q4MM_DEVERR_BAD_EXPERT.
 * Every routed row reads its expert's rows (the mat-vec form, as on the page, for every
 * n_tokens); the product runs on the tensor cores when K % 128 == 0 and the expert slabs
 * are 8-byte aligned, else on the fp32 FMA pipes, with the same results to tolerance.
 * Requirements: n_tokens >= 0 (0 is a no-op), top_k, N, K, n_experts >= 1, K % 32 == 0,
 * n_experts <= 1024, n_tokens*top_k <= 2^24, expert_stride >= N*(K/32)*18; gate, up, out
 * 16-byte aligned, ids 4-byte aligned.  No workspace; nothing is allocated. */
q4mm_status q4_0_matmul_id_swiglu(const float *gate, const float *up, const void *w,
                                  const uint32_t *ids, float *out, int64_t n_tokens,
                                  int64_t top_k, int64_t N, int64_t K, int64_t n_experts,
                                  uint64_t expert_stride, q4mm_stream_t stream);

/* ======================================================================================
 * GGML Q8_0 expert-routed matmul  (quantized_matmul_id_ggml.rs names Q8_0 among its routed
 * kernels and its decode records; the page does not print the block, so this is the GGML
 * Q8_0 block:)  34 bytes per 32 values: fp16 d (little endian), then 32 signed bytes qs;
 * value of element j = qs[j] * d.  Row n of expert e is K/32 consecutive blocks at
 * w + e*expert_stride + n*(K/32)*34.  x, ids, out, routing and modes as q4_0_matmul_id:
 *   out[r][n] = sum_k x[r / top_k][k] * W[ids[r]][n][k]   (f32, fp32 accumulation);
 *   an id >= n_experts gives a zero row and sets Q4MM_DEVERR_BAD_EXPERT.
 * Mode 0 (automatic: mat-mat when n_tokens > Q4MM_MM_ID_THRESHOLD), 1 (mat-vec: each routed
 * row in order; on the tensor cores when K % 128 == 0 and w and expert_stride are 8-byte
 * aligned -- x rounded to bf16, the byte products exact, fp32 sums -- else fp32 FMA) or 2
 * (mat-mat: route, then the tensor-core kernel of q4_0_matmul_id with the Q8_0 decode when
 * K % 256 == 0 and w and expert_stride are 16-byte aligned -- weights q*d rounded once to
 * fp16, see Q4MM_DEVERR_F16_RANGE -- else the routed rows expert by expert on the fp32 FMA
 * pipes).  The mat-mat form needs q8_0_matmul_id_workspace_size(...)
 * bytes of 256-byte aligned workspace (the routing lists and the gathered x rows).
 * Requirements: K % 32 == 0, expert_stride >= N*(K/32)*34, x and out 16-byte aligned, ids
 * 4-byte aligned. */
size_t q8_0_matmul_id_workspace_size(int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                                     int64_t n_experts);
q4mm_status q8_0_matmul_id(const float *x, const void *w, const uint32_t *ids, float *out,
                           int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                           int64_t n_experts, uint64_t expert_stride, int mode,
                           void *workspace, size_t workspace_bytes, q4mm_stream_t stream);

/* ======================================================================================
 * Dispatch records: plan a decode call once, replay it with new pointers.
 *
 * The counterpart of the pages' pre-baked decode dispatches (quantized_matmul_id_ggml.rs,
 * `build_q6k_id_nr2_m1_record` and `build_q8_0_id_decode_record`: bake the load-time-
 * immutable parts of a per-token call -- kernel, launch geometry, parameter block -- once,
 * so each token's dispatch only binds buffers).  A record holds the planned kernel, grid,
 * cluster shape, shared-memory size and launch attributes of one call shape; creating it
 * also performs the kernel's one-time attribute set-up, so the first replay may be inside a
 * stream capture.  A replay launches exactly the kernel the direct call would launch, with
 * bit-identical results.
 *
 *   - Creation allocates one small HOST object (no device memory); free it with
 *     q4mm_record_free.  A record may be replayed any number of times, from any host thread,
 *     on any stream of the device that was current at creation (else Q4MM_ERR_DEVICE).
 *   - Replays check pointers (null: Q4MM_ERR_INVALID_ARG; alignment: Q4MM_ERR_UNSUPPORTED)
 *     but not buffer sizes: the buffers must have the recorded shape.
 * ====================================================================================*/
typedef struct q4mm_record q4mm_record;

/* Record q4_gemv_ex(M, N, K, flags): 1 <= M <= 16, K % 32 == 0, flags as for q4_gemv_ex. */
q4mm_status q4_gemv_record(int64_t M, int64_t N, int64_t K, uint32_t flags, q4mm_record **out);
/* Replay: the q4_gemv_ex call the record was made for, on x, w, scales, biases, y (each
 * 16-byte aligned, with the recorded shape). */
q4mm_status q4_gemv_record_launch(const q4mm_record *rec, const uint16_t *x, const uint32_t *w,
                                  const uint16_t *scales, const uint16_t *biases, uint16_t *y,
                                  q4mm_stream_t stream);

/* Replay n gemv records in order on one stream, in one host call (a decode step's sequence
 * of planned calls): record i on x[i], w[i], scales[i], biases[i], y[i] (host arrays of n
 * device pointers, each as q4_gemv_record_launch requires).  Every record and pointer is
 * checked before anything is launched; on a check failure nothing is launched.  A launch
 * error stops the sequence (the launches before it stay enqueued).  0 <= n <= 65536;
 * n = 0 is a no-op. */
q4mm_status q4_gemv_record_launch_n(const q4mm_record *const *recs, const uint16_t *const *x,
                                    const uint32_t *const *w, const uint16_t *const *scales,
                                    const uint16_t *const *biases, uint16_t *const *y, int64_t n,
                                    q4mm_stream_t stream);

/* Record the routed Q4_0 mat-vec: q4_0_matmul_id in mode 1 (swiglu = 0) or
 * q4_0_matmul_id_swiglu (swiglu = 1), with the argument rules of those calls.  The plan
 * assumes the weight pointer of every replay is 16-byte aligned when K % 256 == 0 and
 * expert_stride % 16 == 0, else 8-byte aligned when K % 128 == 0 and expert_stride % 8 == 0;
 * a replay whose w breaks that returns Q4MM_ERR_UNSUPPORTED (the direct calls accept it). */
q4mm_status q4_0_matmul_id_mv_record(int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                                     int64_t n_experts, uint64_t expert_stride, int swiglu,
                                     q4mm_record **out);
/* Replay: x is x [n_tokens, K] (swiglu = 0; up must be NULL) or gate [n_tokens*top_k, K]
 * with up [n_tokens*top_k, K] (swiglu = 1). */
q4mm_status q4_0_matmul_id_mv_record_launch(const q4mm_record *rec, const float *x, const float *up,
                                            const void *w, const uint32_t *ids, float *out,
                                            q4mm_stream_t stream);

/* Release a record (NULL is a no-op).  Launches already enqueued are unaffected. */
void q4mm_record_free(q4mm_record *rec);

/* ======================================================================================
 * Allocation-free variant of the mat-mat form (the source pages have no counterpart).
 *
 * For callers that cannot obtain device memory at the moment of the call -- serving loops
 * that must never wait on or fail in the device allocator, hosts that own all device
 * buffers.  Computes exactly what
 * q4_0_matmul_id computes in mode 2 (mat-mat), with the same argument rules, but takes no
 * workspace: its scratch is a fixed Q4MM_NOALLOC_SCRATCH_BYTES array built into the library,
 * held on every device that loads the library until process exit.
 *   - Returns Q4MM_ERR_WORKSPACE, launching nothing, when
 *     q4_0_matmul_id_workspace_size(n_tokens, top_k, N, K, n_experts) exceeds the array.
 *   - The first call on a device (made with that device current) looks up the array's device
 *     address (cudaGetSymbolAddress; no allocation) and keeps it.  Later calls look it up
 *     again unless their stream reports that it is capturing, so after a device reset
 *     (cudaDeviceReset) the next call picks up the new address.
 *   - All calls on a device share the array.  Calls that overlap on the GPU race on it and
 *     give wrong results: order them (for instance on one stream).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * ====================================================================================*/
#define Q4MM_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
q4mm_status q4_0_matmul_id_noalloc(const float *x, const void *w, const uint32_t *ids, float *out,
                                   int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                                   int64_t n_experts, uint64_t expert_stride, q4mm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4MM_H */
