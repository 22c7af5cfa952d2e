/*
 * tp_api.h -- C ABI of the sharded-GEMM library (libtp.so) for one GB300.
 *
 * The library runs the sharded matrix multiplies behind tensor-parallel
 * linear layers.  The N logical shards (the ranks of a tensor-parallel group)
 * are N separate device buffers on ONE GPU, so the cross-shard reduction of a
 * row-parallel layer is a fixed-order in-GPU sum, not a collective.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Linear weights are (out, in) row-major and a layer computes
 *    y = x @ W^T + b ("MLX tensor parallelism guide", section 2.1/2.2).
 *    SUMMA computes Y = X A with A laid out (K, N) ("ColossalAI 2D tensor
 *    parallel via SUMMA", SUMMA section).  All matrices are row-major; a
 *    leading dimension (ld*) is the distance in ELEMENTS between rows.
 *  - Data pointers are DEVICE pointers owned by the caller; the library never
 *    frees or keeps them.  Arrays of per-shard pointers (w[r], y[r], ...)
 *    live in HOST memory and are read during the call only.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and is asynchronous: the call returns before the GPU finishes.
 *  - Return value: TP_OK (0) or a negative tp_status.  Argument errors are
 *    detected on the host before anything is launched; on error nothing is
 *    launched and tp_last_error() returns a message for the calling thread.
 *  - Bias vectors are float32.  Accumulation is float32 everywhere.
 *  - The device-side waits of the kernels are bounded; a wait that runs out
 *    makes the kernel record TP_ERR_TIMEOUT in a device status word and
 *    return.  tp_query_status() reads (and clears) that word.
 *  - The library allocates one 4-byte device status word per device on
 *    first use and caches host-side TMA descriptors.  Calls whose kernel
 *    splits a sum across CTAs (the row-parallel 4-bit linears, split-K 4-bit
 *    and MXFP8 tiles, and 16-bit linears of at most 16 tokens whose output
 *    has fewer 128-row tiles than the GPU has SMs) use a per-(device, stream)
 *    float32 workspace with zeroed counters, allocated (cudaMalloc) on first
 *    need and grown when a larger call needs more; the counters are back at
 *    zero when each kernel ends.  A workspace that grows keeps its old
 *    buffers allocated (a graph captured earlier still addresses them) until
 *    tp_shutdown(), which frees all of it.
 *    tp_q4_sharded_to_all_noalloc never allocates.  A call may therefore be
 *    captured into a CUDA graph once the same call has run on the capturing
 *    stream outside the capture, and a later, larger call on that stream
 *    does not invalidate the capture.
 *  - Kernels may be launched with programmatic stream serialization: their
 *    set-up can overlap the end of the previous kernel on the stream, but
 *    they read and write no global memory before it has completed.
 */
#ifndef TP_API_H
#define TP_API_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TP_OK = 0,
    TP_ERR_INVALID_ARG = -1,   /* null pointer, bad enum, negative size ...   */
    TP_ERR_NOT_DIVISIBLE = -2, /* a dimension does not split evenly            */
    TP_ERR_ALIGNMENT = -3,     /* pointer / leading dimension misaligned       */
    TP_ERR_UNSUPPORTED = -4,   /* valid request this build does not implement  */
    TP_ERR_CUDA = -5,          /* a CUDA runtime/driver call failed            */
    TP_ERR_TIMEOUT = -6        /* a bounded device-side wait ran out           */
} tp_status;

typedef enum { TP_F32 = 0, TP_BF16 = 1, TP_F16 = 2 } tp_dtype;

/* Kernel selection policy (tp_set_policy). */
typedef enum {
    TP_POLICY_AUTO = 0,      /* tensor-core (tcgen05) kernels where they apply  */
    TP_POLICY_SIMT = 1,      /* plain CUDA-core kernels only (slow cross-check)  */
    TP_POLICY_SINGLE_SM = 2  /* tensor-core kernels, one CTA per output tile    */
} tp_policy;

typedef void *tp_stream_t; /* a cudaStream_t */

/* Library version, major*10000 + minor*100 + patch. */
int tp_version(void);

/* Message describing the last error returned to the calling thread ("" if none). */
const char *tp_last_error(void);

/* Number of kernels this library has launched from the calling thread so far
 * (monotonic; a call may launch several, e.g. a GEMM and its ordered split
 * reduction).  Never fails. */
int64_t tp_launch_count(void);

/* Synchronizes `stream`, copies the current device's status words into
 * *device_status (0 = no error, else a tp_status such as TP_ERR_TIMEOUT)
 * and resets them to 0.  Two words are read: the library's own (written by
 * every entry point but the next) and the one inside the fixed buffer of
 * tp_q4_sharded_to_all_noalloc; the first nonzero one is reported.  After a
 * nonzero word the split counters it concerns are cleared as well.  Allocates
 * nothing (a word that was never created reads as 0).  Returns TP_OK or
 * TP_ERR_CUDA. */
int tp_query_status(tp_stream_t stream, int *device_status);

/* Selects the kernel family for the calling process (default AUTO).  The SIMT
 * policy exists to cross-check the tensor-core kernels; it is slow. */
int tp_set_policy(int policy);

/* Limit, in nanoseconds, of every bounded device-side wait (default 2e9).
 * Values below 1e6 or above 6e10 are rejected with TP_ERR_INVALID_ARG. */
int tp_set_wait_limit_ns(int64_t limit_ns);

/* Role timeline tracing (profiling aid; no counterpart on the pages).  With a
 * non-NULL device buffer of `bytes` bytes (>= 256 KiB + 128 bytes, 16-byte
 * aligned, caller owned), CTA 0 of every later tensor-core q4 decode launch
 * writes the globaltimer value (ns) of event e at stage sequence number s
 * (s < 1024, e < 32) into 64-bit word 16 + e*1024 + s, with plain stores.
 * NULL switches tracing off.
 * 8-bit decode kernel (every part's K a multiple of 512): 1 the codes of the
 * stage were issued; 2 the MMA thread had the stage's operands, 5 it issued
 * the stage's commit; 6 converter warp 2 had the codes and a free A half, 8
 * its tensor-memory stores completed; 9 epilogue warp 6 saw the stage's first
 * accumulator pair, 11 it finished the stage.  Per accumulator pair p of
 * stage s, at word index 4s + p: 17/18 the MMA thread issued / committed it,
 * 12/13/14 epilogue warp 6 saw it / had loaded it / had applied it.  Per CTA
 * b, at index b: 28 the SM id + 1, 30/31 the CTA's start / end, and 29/10
 * the start / end of its share of the activation pre-pass.  The ordered split
 * sum that follows a split launch (4-bit and mxfp8): per block b, 21/22 its
 * start (after the programmatic-launch wait) and end.
 * 16-bit decode kernel (other shapes): 1 producer issued the stage's loads;
 * 2/3/4 the MMA thread saw the stage's data / A operand / free accumulator,
 * 5 it committed the stage; 6/7 converter warp 2 saw the data / a free A
 * slot, 12 finished the x reorder, 13 its tensor-memory stores completed, 8
 * signalled the MMA; 9/10/11 epilogue warp 10 saw the accumulator, released
 * it, finished the stage. */
int tp_set_trace(void *device_buffer, int64_t bytes);

/* Frees the per-device status words and cached descriptors. */
int tp_shutdown(void);

/*
 * a1 -- weight sharding (MLX page, section 3.2, `_shard`; section 3.1
 * `shard_linear` only reads the original layer).
 *
 * Slices a full row-major (rows, cols) array `w` of `elem_bytes`-byte
 * elements into N shard buffers: along `axis` (0 = rows, 1 or -1 = columns)
 * the array is split into `segments` equal contiguous parts, each part into N
 * equal contiguous parts, and shard r receives part r of every segment,
 * concatenated in segment order.  With L the axis length and
 * w_len = L / (segments * N), local index i of shard r is global index
 * (i / w_len) * (L / segments) + r * w_len + (i % w_len).
 *   axis 0 : shards[r] is (rows / N, cols) row-major;
 *   axis 1 : shards[r] is (rows, cols / N) row-major.
 * The copy is bit-exact.  `shards` is a host array of N device pointers to
 * caller-allocated buffers that must not overlap `w` or each other.
 * Errors: TP_ERR_NOT_DIVISIBLE if L % (segments * N) != 0 (message
 * "Cannot shard the output of size L across N devices."); TP_ERR_INVALID_ARG
 * for a bad axis, segments < 1, N < 1 or N > 64, elem_bytes not in
 * {1, 2, 4, 8}, or a null pointer.
 */
int tp_shard_weight(const void *w, int64_t rows, int64_t cols, int elem_bytes, int axis,
                    int segments, int N, void *const *shards, tp_stream_t stream);

/*
 * a2 / a4 -- column-parallel linear, "all-to-sharded" (MLX page, section 2.1
 * AllToShardedLinear; the pages' Linear1D_Col with gather_output=False, and
 * the fused-QKV and vocab-parallel LM head of the EnergonAI page, sections 2
 * and 3).  The contraction dimension is not sharded, so there is no
 * communication ("sharded matrices" notes, case 1).
 *
 * For r = 0..N-1:  y[r] = x @ w[r]^T + bias[r]
 *   x      (T, K) in_dt, row stride ldx (>= K), replicated input;
 *   w[r]   (O/N, K) in_dt contiguous: shard r of the (O, K) weight;
 *   bias   NULL, or a host array of N device pointers to float32 (O/N);
 *   y[r]   (T, O/N) out_dt, row stride ldy (>= O/N).  For a gathered output
 *          (vocab-parallel logits) pass y[r] = base + r*(O/N) and ldy = O.
 * in_dt: TP_BF16 or TP_F16 (tensor cores) or TP_F32 (CUDA cores);
 * out_dt: TP_F32, TP_BF16 or TP_F16.
 * Errors: TP_ERR_NOT_DIVISIBLE if O % N != 0, with the message
 * "Cannot shard the output of size O across N devices."; TP_ERR_INVALID_ARG
 * for null pointers, T < 0, K < 1, N < 1 or N > 64, ldx < K, ldy < O/N;
 * TP_ERR_ALIGNMENT if x, w[r] or y[r] is not aligned to its element size or
 * bias[r] to 4 bytes.  Operands the tensor copies cannot take (a base not
 * 16-byte aligned, a row stride not a multiple of 16 bytes) run on the
 * CUDA-core kernel instead, with the same result.  T = 0 is valid and
 * launches nothing.
 */
int tp_all_to_sharded(int N, const void *x, int64_t T, int64_t K, int64_t ldx,
                      const void *const *w, int64_t O, const void *const *bias,
                      tp_dtype in_dt, void *const *y, int64_t ldy, tp_dtype out_dt,
                      tp_stream_t stream);

/*
 * f2 -- gated FFN input projections, both column-parallel on the same input
 * (MLX tensor parallelism guide, section 5.2: the FFN's gate projection w1
 * and up projection w3 become all-to-sharded, w2 sharded-to-all; section
 * 5.3: the elementwise product between them keeps the sharding, so it runs
 * on each rank's shard with no communication).  The activation of the gate
 * is SiLU, silu(a) = a / (1 + exp(-a)), as in the Llama FFN the guide shards.
 *
 * For r = 0..N-1:
 *   h[r] = silu(x @ w1[r]^T + b1[r]) * (x @ w3[r]^T + b3[r])   (elementwise)
 *   x       (T, K) in_dt, row stride ldx (>= K), replicated input;
 *   w1[r], w3[r]  (F/N, K) in_dt contiguous: shard r of the (F, K) gate and
 *           up weights (axis 0);
 *   b1, b3  NULL, or host arrays of N device pointers to float32 (F/N);
 *   h[r]    (T, F/N) out_dt, row stride ldh (>= F/N): the input of the
 *           row-parallel w2 (tp_sharded_to_all with x[r] = h[r]).
 * Both projections accumulate in float32; the gate, the SiLU and the product
 * are formed in float32 from the two sums and rounded once to out_dt.  The
 * SiLU uses the fast exponential (relative error a few units in the last
 * float32 place for |a| below 80).
 * Errors: TP_ERR_NOT_DIVISIBLE if F % N != 0 ("Cannot shard the output of
 * size F across N devices."); otherwise as tp_all_to_sharded, with ldh
 * checked against F/N.  T = 0 is valid and launches nothing.
 */
int tp_gated_all_to_sharded(int N, const void *x, int64_t T, int64_t K, int64_t ldx,
                            const void *const *w1, const void *const *w3, int64_t F,
                            const void *const *b1, const void *const *b3, tp_dtype in_dt,
                            void *const *h, int64_t ldh, tp_dtype out_dt, tp_stream_t stream);

/*
 * a3 -- row-parallel linear, "sharded-to-all" (MLX page, section 2.2
 * ShardedToAllLinear: local matmul, then all_sum over the group, then the
 * bias; the pages' Linear1D_Row; "sharded matrices" notes, case 3).
 *
 * y = (sum over r = 0..N-1, ascending, of x[r] @ w[r]^T) + bias
 *   x[r]   (T, K/N) in_dt, row stride ldx (>= K/N): shard r of the input;
 *   w[r]   (O, K/N) in_dt contiguous: shard r of the (O, K) weight, split on
 *          its last axis;
 *   bias   NULL or float32 (O), added once, after the sum;
 *   y      (T, O) out_dt, row stride ldy (>= O).
 * Every partial x[r] @ w[r]^T is formed in float32 from zero and the
 * partials are added in ascending r, so the result does not depend on how
 * the GPU schedules the work.  Partials do not go through device memory.
 * Exception, T <= 16 with fewer 128-row output tiles than the GPU has SMs:
 * the contraction over r = 0..N-1 laid end to end is cut into consecutive
 * k-block ranges.  Each range is summed in float32 from zero, across rank
 * boundaries too, and the range sums are added in range order through the
 * float32 workspace.  The order is still ascending r, and it is fixed by the
 * shapes alone.
 * Errors: TP_ERR_NOT_DIVISIBLE if K % N != 0; otherwise as tp_all_to_sharded.
 */
int tp_sharded_to_all(int N, const void *const *x, int64_t T, int64_t K, int64_t ldx,
                      const void *const *w, int64_t O, const void *bias, tp_dtype in_dt,
                      void *y, int64_t ldy, tp_dtype out_dt, tp_stream_t stream);

/*
 * f1 -- row-parallel linear with a reduce-scatter, "sharded-to-sharded"
 * ("sharded matrices" notes, case 3, second option: reduce-scatter the
 * partial sums instead of all-reducing them, so the output stays sharded
 * along its columns; primitive table, ReduceScatter_{X,K}).
 *
 * For c = 0..N-1:
 *   y[c] = (sum over r = 0..N-1, ascending, of x[r] @ W_r[c]^T) + bias[c*O/N ..]
 * where W_r[c] is rows c*O/N .. (c+1)*O/N - 1 of w[r].
 *   x[r]   (T, K/N) in_dt, row stride ldx (>= K/N): shard r of the input;
 *   w[r]   (O, K/N) in_dt contiguous: shard r of the (O, K) weight, split on
 *          its last axis (the same shards as tp_sharded_to_all);
 *   bias   NULL or float32 (O), the layer's replicated bias; rank c adds its
 *          block c*O/N .. once, after the sum;
 *   y[c]   (T, O/N) out_dt, row stride ldy (>= O/N): rank c's block of the
 *          output.  With y[c] = base + c*(O/N) and ldy = O the blocks form
 *          the all-reduced (T, O) output of tp_sharded_to_all.
 * Every partial is formed in float32 from zero and the N partials of a block
 * are added in ascending r, as in tp_sharded_to_all; partials do not go
 * through device memory (with the same small-batch exception).
 * Errors: TP_ERR_NOT_DIVISIBLE if K % N != 0 ("Cannot shard the input of
 * size K across N devices.") or O % N != 0 ("Cannot shard the output ...");
 * TP_ERR_UNSUPPORTED if N * N > 64; otherwise as tp_sharded_to_all, with
 * ldy checked against O/N.  T = 0 is valid and launches nothing.
 */
int tp_sharded_to_sharded(int N, const void *const *x, int64_t T, int64_t K, int64_t ldx,
                          const void *const *w, int64_t O, const void *bias, tp_dtype in_dt,
                          void *const *y, int64_t ldy, tp_dtype out_dt, tp_stream_t stream);

/*
 * f1 -- all-gather then column-parallel linear, "gathered-to-sharded"
 * ("sharded matrices" notes, case 2, standard route: all-gather the input's
 * sharded contraction axis, then the local matmul; the large-batch strategy
 * of the same notes, and the first half of their Transformer FFN with one
 * all-gather and one reduce-scatter).
 *
 * For r = 0..N-1:  y[r] = concat_q(x[q]) @ w[r]^T + bias[r]
 *   x[q]   (T, K/N) in_dt, row stride ldx (>= K/N): block q of the input's
 *          columns (the gathered input is the N blocks side by side);
 *   w[r]   (O/N, K) in_dt contiguous: shard r of the (O, K) weight (axis 0,
 *          as tp_all_to_sharded);
 *   bias   NULL, or a host array of N device pointers to float32 (O/N);
 *   y[r]   (T, O/N) out_dt, row stride ldy (>= O/N).
 * The gather is not materialised: rank r's product reads every block x[q]
 * against columns q*K/N .. of w[r], accumulating in one float32 sum in
 * block order, which is the order of the gathered contraction axis.
 * Errors: as tp_sharded_to_sharded, with bias an array of N pointers.
 */
int tp_gathered_to_sharded(int N, const void *const *x, int64_t T, int64_t K, int64_t ldx,
                           const void *const *w, int64_t O, const void *const *bias,
                           tp_dtype in_dt, void *const *y, int64_t ldy, tp_dtype out_dt,
                           tp_stream_t stream);

/*
 * a5 -- SUMMA on a q x q grid ("ColossalAI 2D tensor parallel via SUMMA",
 * SUMMA section, equations (1) and (2); Matmul_AB_2D).
 *
 * Y = X A with X (M, K) and A (K, Ncols) held as q*q blocks, block (i, j) at
 * index i*q + j:
 *   X[i*q+j]  (M/q, K/q) in_dt contiguous;
 *   A[i*q+j]  (K/q, Ncols/q) in_dt contiguous;
 *   Y[i*q+j]  (M/q, Ncols/q) float32 contiguous, written (not accumulated).
 * Y_ij = sum over t = 0..q-1 of X_it A_tj, accumulated in float32 in step
 * order t.  The per-step row and column broadcasts of the distributed
 * algorithm become reads of the owning block's buffer.
 * in_dt: TP_BF16, TP_F16 or TP_F32.
 * Errors: TP_ERR_NOT_DIVISIBLE if q < 1 or M, K or Ncols is not a multiple of
 * q (the page's grid requires P = q*q processors and block dimensions that
 * divide evenly); TP_ERR_UNSUPPORTED if q > 4 (this build holds at most 16
 * logical processors); TP_ERR_ALIGNMENT if an X or A block is not aligned
 * to its element size or a Y block to 4 bytes; TP_ERR_INVALID_ARG for null
 * pointers, sizes below 1 or a bad dtype.  Blocks the tensor copies cannot
 * take (a base not 16-byte aligned, a block row not a multiple of 16 bytes)
 * run on the CUDA-core kernel instead, with the same result.
 */
int tp_summa(int q, const void *const *X, const void *const *A, void *const *Y, int64_t M,
             int64_t K, int64_t Ncols, tp_dtype in_dt, tp_stream_t stream);

/*
 * f4 -- the "mxfp8" quantization mode of the sharded linears (MLX tensor
 * parallelism guide, section 2.3: mode "mxfp8" is passed through sharding
 * like "affine" and has no per-group biases; section 4's tests check that
 * it propagates).  Format (OCP microscaling FP8): E4M3 codes, one byte per
 * weight (1 sign, 4 exponent bits with bias 7, 3 mantissa bits), and one
 * E8M0 scale byte per 32 consecutive weights of a row, value 2^(s - 127):
 *   W_hat[o][k] = e4m3(codes[o][k]) * 2^(scales[o][k / 32] - 127).
 *
 * tp_mx_quantize: w (rows, K) float32 -> codes uint8 (rows, K) and scales
 *   uint8 (rows, K/32).  Per block: X = floor(log2(max |w|)) - 8 clamped to
 *   [-127, 127] (-127 for an all-zero block), scale byte X + 127, code = E4M3
 *   of w * 2^-X rounded to nearest even, saturated to +-448, sign kept.
 *   Errors: TP_ERR_NOT_DIVISIBLE if K % 32 != 0.
 * tp_mx_all_to_sharded: y[r] = x @ W_hat_r^T + bias[r]; x (T, K) bf16
 *   contiguous; codes[r] (O/N, K), scales[r] (O/N, K/32) (the rows of shard
 *   r); bias NULL or N float32 (O/N); y[r] (T, O/N) out_dt, row stride ldy.
 * tp_mx_sharded_to_all: y = sum over r ascending of x[r] @ W_hat_r^T, then
 *   bias once; x[r] (T, K/N) bf16 contiguous; codes[r] (O, K/N), scales[r]
 *   (O, K/(32 N)) (split on the last axis, whole blocks per shard); y (T, O).
 * x is used as given (bf16); every product x * e4m3 is exact in float32 and
 * the sums are float32.  Errors as the 4-bit linears: TP_ERR_NOT_DIVISIBLE
 * if O % N (all-to-sharded), K % N or (K/N) % 32 (sharded-to-all) or K % 32
 * is not zero.  T = 0 launches nothing.
 */
int tp_mx_quantize(const float *w, int64_t rows, int64_t K, uint8_t *codes, uint8_t *scales,
                   tp_stream_t stream);
int tp_mx_all_to_sharded(int N, const void *x, int64_t T, int64_t K, const uint8_t *const *codes,
                         const uint8_t *const *scales, int64_t O, const void *const *bias,
                         void *const *y, int64_t ldy, tp_dtype out_dt, tp_stream_t stream);
int tp_mx_sharded_to_all(int N, const void *const *x, int64_t T, int64_t K,
                         const uint8_t *const *codes, const uint8_t *const *scales, int64_t O,
                         const void *bias, void *y, int64_t ldy, tp_dtype out_dt,
                         tp_stream_t stream);

/*
 * f3 -- SUMMA with the layer's bias, and the two backward products of the 2-D
 * layer ("ColossalAI 2D tensor parallel via SUMMA", source-level section: in
 * backward the input gradient goes through Matmul_ABT_2D (A B^T) and the
 * weight gradient through Matmul_ATB_2D (A^T B); Linear2D adds its bias
 * after gathering it along the column group, add_bias_2d).
 *
 * All three keep tp_summa's conventions: q*q blocks indexed i*q + j, float32
 * output blocks (M/q, Ncols/q) written, q step products chained in float32
 * in step order t, the row / column broadcasts turned into reads of the
 * owning block.  Errors and limits as tp_summa.
 *
 * tp_summa_linear: Y_ij = sum_t X_it A_tj + bias[j], bias NULL or a host
 *   array of q device pointers to float32 (Ncols/q): column block j's bias,
 *   the gathered piece every block of column j adds.
 * tp_summa_abt: C = A B^T with A (M, K) and B (Ncols, K):
 *   C_ij = sum_t A_it B_jt^T;  A blocks (M/q, K/q), B blocks (Ncols/q, K/q).
 *   (dX = dY W^T: A = dY, B = W.)
 * tp_summa_atb: C = A^T B with A (K, M) and B (K, Ncols):
 *   C_ij = sum_t A_ti^T B_tj;  A blocks (K/q, M/q), B blocks (K/q, Ncols/q).
 *   (dW = X^T dY: A = X, B = dY.)
 */
int tp_summa_linear(int q, const void *const *X, const void *const *A, const void *const *bias,
                    void *const *Y, int64_t M, int64_t K, int64_t Ncols, tp_dtype in_dt,
                    tp_stream_t stream);
int tp_summa_abt(int q, const void *const *A, const void *const *B, void *const *C, int64_t M,
                 int64_t K, int64_t Ncols, tp_dtype in_dt, tp_stream_t stream);
int tp_summa_atb(int q, const void *const *A, const void *const *B, void *const *C, int64_t M,
                 int64_t K, int64_t Ncols, tp_dtype in_dt, tp_stream_t stream);

/*
 * f3 -- backward of the 1-D sharded linears.
 *
 * tp_all_to_sharded_dx: the input gradient of the column-parallel layer.
 *   Its forward wraps x in sum_gradients (MLX tensor parallelism guide,
 *   "gradient aggregation in backward": identity forward, all_sum of the
 *   incoming gradient in backward), so every rank's local dx_r = dy[r] @ w[r]
 *   is all-summed:
 *     dx = sum over r = 0..N-1, ascending, of dy[r] @ w[r]
 *   dy[r]  (T, O/N) in_dt, row stride lddy (>= O/N): gradient of y[r];
 *   w[r]   (O/N, K) in_dt contiguous: the forward's weight shard;
 *   dx     (T, K) out_dt, row stride lddx (>= K).
 *   Every partial is formed in float32 from zero and the partials are added
 *   in ascending r, as in tp_sharded_to_all.
 *   Errors: TP_ERR_NOT_DIVISIBLE if O % N != 0; TP_ERR_INVALID_ARG for null
 *   pointers, T < 0, K < 1, lddy < O/N or lddx < K; T = 0 launches nothing.
 *
 * tp_sharded_to_all_dx: the input gradient of the row-parallel layer.  Its
 *   incoming gradient dy is replicated (the forward ended in an all_sum), so
 *   each rank's slice needs no communication:
 *     dx[r] = dy @ w[r]
 *   dy     (T, O) in_dt, row stride lddy (>= O);
 *   w[r]   (O, K/N) in_dt contiguous; dx[r] (T, K/N) out_dt, stride lddx.
 *   Errors: TP_ERR_NOT_DIVISIBLE if K % N != 0; otherwise as above.
 *
 * tp_sharded_dw: weight gradients of N shards, dw[r] = dy[r]^T @ x[r]:
 *     dw[r][o][k] = sum over tokens t of dy[r][t][o] * x[r][t][k]
 *   dy[r]  (T, O) in_dt, row stride lddy (>= O);
 *   x[r]   (T, K) in_dt, row stride ldx (>= K);
 *   dw[r]  (O, K) out_dt, row stride lddw (>= K).
 *   Column-parallel layer: dy[r] = its output gradient shard, x[r] = x for
 *   every r; row-parallel layer: dy[r] = dy for every r, x[r] = its input
 *   shard.  T = 0 writes zeros (the empty sum).
 *
 * tp_bias_grad: bias gradients, float32 column sums in a fixed order:
 *     db[o][c] = sum over b = 0..nin-1 of sum over rows t of dy[o*nin + b][t*ld + c]
 *   dy     nout*nin device pointers, each (rows, cols) in_dt, row stride ld;
 *   db[o]  float32 (cols).
 *   Column-parallel bias: nout = N, nin = 1; row-parallel bias (added once
 *   after the sum): nout = nin = 1; Linear2D bias of column block j: nin = q
 *   blocks dY_0j .. dY_(q-1)j.  Requires nout <= 64, nout * nin <= 64.
 */
int tp_all_to_sharded_dx(int N, const void *const *dy, int64_t T, int64_t O, int64_t lddy,
                         const void *const *w, int64_t K, tp_dtype in_dt, void *dx, int64_t lddx,
                         tp_dtype out_dt, tp_stream_t stream);
int tp_sharded_to_all_dx(int N, const void *dy, int64_t T, int64_t O, int64_t lddy,
                         const void *const *w, int64_t K, tp_dtype in_dt, void *const *dx,
                         int64_t lddx, tp_dtype out_dt, tp_stream_t stream);
int tp_sharded_dw(int N, const void *const *dy, int64_t lddy, const void *const *x, int64_t ldx,
                  int64_t T, int64_t O, int64_t K, tp_dtype in_dt, void *const *dw, int64_t lddw,
                  tp_dtype out_dt, tp_stream_t stream);
int tp_bias_grad(int nout, int nin, const void *const *dy, int64_t rows, int64_t cols, int64_t ld,
                 tp_dtype in_dt, float *const *db, tp_stream_t stream);

/*
 * a6 -- affine 4-bit quantization of a float32 weight on the device (MLX
 * page, section 2.3: group_size 64, bits 4, mode "affine").  Data
 * preparation, not part of a forward pass.
 *
 *   w       (rows, K) float32 row-major;
 *   wq      (rows, K/8) uint32: 8 codes per word, element k at bits 4*(k%8);
 *   scales  (rows, K/group_size) float16 (raw 16-bit storage);
 *   qbias   (rows, K/group_size) float16.
 * Per group of group_size consecutive elements of a row:
 *   s = (max - min) / 15 in float32, 1 if that is 0; b = min;
 *   s and b rounded to float16 (nearest even), s = 1 if it rounds to 0;
 *   code = clamp(rint((w - b) / s), 0, 15) with float32 operations.
 * Errors: TP_ERR_UNSUPPORTED if group_size != 64; TP_ERR_NOT_DIVISIBLE if
 * K % group_size != 0; TP_ERR_INVALID_ARG for null pointers or sizes < 1.
 */
int tp_q4_quantize(const float *w, int64_t rows, int64_t K, int group_size, uint32_t *wq,
                   void *scales, void *qbias, tp_stream_t stream);

/*
 * a7 -- quantized column-parallel linear (MLX page, section 2.3
 * QuantizedAllToShardedLinear).
 *
 * For r = 0..N-1:  y[r] = x @ What[r]^T + bias[r], where
 * What[r][o][k] = scales[r][o][k/64] * code(wq[r], o, k) + qbias[r][o][k/64].
 *   x          (T, K) bfloat16 contiguous;
 *   wq[r]      (O/N, K/8) uint32;  scales[r], qbias[r] (O/N, K/64) float16;
 *   bias       NULL or host array of N device pointers to float32 (O/N);
 *   y[r]       (T, O/N) out_dt, row stride ldy.
 * Errors: TP_ERR_UNSUPPORTED if group_size != 64; TP_ERR_NOT_DIVISIBLE if
 * O % N != 0 or K % 64 != 0; TP_ERR_INVALID_ARG / TP_ERR_ALIGNMENT as above.
 */
int tp_q4_all_to_sharded(int N, const void *x, int64_t T, int64_t K,
                         const uint32_t *const *wq, const void *const *scales,
                         const void *const *qbias, int group_size, int64_t O,
                         const void *const *bias, void *const *y, int64_t ldy,
                         tp_dtype out_dt, tp_stream_t stream);

/*
 * a7 -- quantized row-parallel linear (MLX page, section 2.3
 * QuantizedShardedToAllLinear: local quantized matmul, then all_sum).
 *
 * y = (sum over r ascending of x[r] @ What[r]^T) + bias
 *   x[r]       (T, K/N) bfloat16 contiguous;
 *   wq[r]      (O, K/N/8) uint32;  scales[r], qbias[r] (O, K/N/64) float16
 *              (each shard holds whole groups);
 *   bias       NULL or float32 (O);   y (T, O) out_dt, row stride ldy.
 * Errors: TP_ERR_NOT_DIVISIBLE if K % N != 0 or (K/N) % 64 != 0; otherwise
 * as tp_q4_all_to_sharded.
 */
int tp_q4_sharded_to_all(int N, const void *const *x, int64_t T, int64_t K,
                         const uint32_t *const *wq, const void *const *scales,
                         const void *const *qbias, int group_size, int64_t O,
                         const void *bias, void *y, int64_t ldy, tp_dtype out_dt,
                         tp_stream_t stream);

/*
 * tp_q4_sharded_to_all without device allocation.  The pages have no
 * counterpart; this exists for callers that cannot call cudaMalloc, such as
 * a serving loop being captured into a CUDA graph, an engine whose device
 * memory belongs to its own pool allocator, or a latency-critical path where
 * cudaMalloc's implicit device synchronization is not acceptable.
 *
 * Arguments, layout, result and errors are those of tp_q4_sharded_to_all.
 * Instead of allocating a workspace it uses one fixed 8 MiB array of device
 * memory that belongs to the library image: the driver creates it on every
 * GPU that loads the library and it lives until the process exits.  Of it,
 * 64 KiB hold the split counters and 8 MiB - 64.25 KiB the float32 split
 * partials; a call whose split needs more (large T or many output rows)
 * returns TP_ERR_UNSUPPORTED with the sizes in the message and launches
 * nothing.  For decode-sized calls (T <= 16) the K split is chosen to fit
 * the array: the down projection of an 8192 x 28672 layer split 8 ways
 * (T = 16) takes 4.64 MB, its prepared activations and 7 partials per
 * 128-row tile.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, no allocation); make that first call before any
 *    stream capture.
 *  - Every call, on every stream, shares the same array, and the array keeps
 *    what the last call left in it.  Each call clears the counters it uses
 *    (an asynchronous memset on `stream`) before its kernel.  Calls that can
 *    overlap on the GPU (on different streams without ordering) race on the
 *    array and give undefined results: order them.
 *  - Device-side wait timeouts of this entry point are recorded in a status
 *    word inside the array; tp_query_status() reads and clears it (without
 *    allocating) together with the library's own word.  After a timeout the
 *    output is unspecified.
 *  - Under TP_POLICY_SIMT it runs the CUDA-core kernel, like every other
 *    entry point; that kernel needs no scratch.
 */
int tp_q4_sharded_to_all_noalloc(int N, const void *const *x, int64_t T, int64_t K,
                                 const uint32_t *const *wq, const void *const *scales,
                                 const void *const *qbias, int group_size, int64_t O,
                                 const void *bias, void *y, int64_t ldy, tp_dtype out_dt,
                                 tp_stream_t stream);

/*
 * Fault check of the bounded waits (no counterpart on the pages): launches a
 * one-block kernel that waits on a shared-memory barrier nothing ever
 * arrives at, with the given limit (1e6 .. 6e10 ns).  The wait runs out,
 * the kernel records TP_ERR_TIMEOUT in the status word and returns; the
 * context stays usable.  Read the result with tp_query_status().
 */
int tp_debug_wait_timeout(int64_t limit_ns, tp_stream_t stream);

/*
 * Check of the 8-bit 4-bit decode's fallback (no counterpart on the pages).
 * With on != 0, every later launch of that kernel (T <= 16, tp_q4_* calls)
 * has each CTA prepare every activation item itself instead of waiting for
 * the launch-wide count of the other CTAs' shares: the path a CTA takes when
 * its peers are not resident.  The prepared values are the same either way,
 * so the outputs are bit-identical.  on = 0 restores the default.  Process
 * wide; returns TP_OK.
 */
int tp_debug_prep_alone(int on);

#ifdef __cplusplus
}
#endif

#endif /* TP_API_H */
