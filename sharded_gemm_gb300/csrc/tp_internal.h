// tp_internal.h -- definitions shared by the translation units of libtp.so.
//
// A request of any entry point is lowered to one `Problem`: a list of output
// matrices ("jobs"), each the sum of one or more matrix products ("parts").
//   C_j[m][n] = bias_j[n] + sum over parts p of job j of
//               sum_k A_p[m][k] * B_p(n, k)
// B_p(n, k) is B_p[n*ldb + k] (layout BL_KMAJOR, a linear weight (out, in)),
// B_p[k*ldb + n] (BL_MNMAJOR, SUMMA's A block (K, N)), or the dequantized
// 4-bit weight s[n][k/64]*code(n, k) + b[n][k/64] (BL_Q4).
// `chain` = 1: the parts of a job accumulate into one float32 sum in part
// order (SUMMA's q steps).  `chain` = 0: every part is a separate float32
// partial formed from zero and the partials are added in part order (the
// row-parallel all_sum over ranks r = 0..N-1).
// `a_mn` = 1: A_p(m, k) is A_p[k*lda + m] (the operand stored K-major by
// rows, as a gradient's dy or x is when the contraction runs over tokens).
// `gated` = 1 (chain mode, BL_KMAJOR only): every part carries a second
// weight B2 and every job a second bias, and the job's output is the gated
// product silu(G + bias) * (U + bias2), G and U the chained sums over its
// parts of A_p B_p^T and A_p B2_p^T (the gate / up projections of a gated FFN).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/tp_api.h"

namespace tp {

constexpr int kMaxShards = 64;
constexpr int kMaxJobs = 64;
constexpr int kMaxParts = 64;

// BL_MX: MXFP8 weights: B = E4M3 codes uint8 (N, K) (ldb = bytes per row),
// scales = E8M0 uint8 (N, K/32); W(n, k) = e4m3(B[n][k]) * 2^(scales[n][k/32] - 127).
enum BLayout { BL_KMAJOR = 0, BL_MNMAJOR = 1, BL_Q4 = 2, BL_MX = 3 };

struct Part {
  const void *A;       // (M, K) row-major, row stride lda
  const void *B;       // see BLayout
  const void *scales;  // BL_Q4: float16 (N, K/64)
  const void *qbias;   // BL_Q4: float16 (N, K/64)
  int64_t K, lda, ldb;
  const void *B2;      // gated problems: the up-projection weight, same layout as B
};

struct Job {
  void *C;             // (M, N) out_dt, row stride ldc
  const float *bias;   // nullable, (N)
  int64_t M, N, ldc;
  int part0, nparts;
  const float *bias2;  // gated problems: nullable up-projection bias, (N)
};

struct Problem {
  Job jobs[kMaxJobs];
  Part parts[kMaxParts];
  int njobs;
  int in_dt, out_dt;   // tp_dtype
  int b_layout;        // BLayout
  int chain;
  int gated;
  int a_mn;
  int *status;         // device status word
  int64_t wait_ns;     // bound of device-side waits
};

#ifdef __CUDACC__
// SiLU, a * sigmoid(a), of the gated FFN.  For a below about -88 the
// exponential overflows to infinity and the quotient is -0, the limit.
__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }
#endif

// ---- shared host state (tp_api.cu)
int *device_status_word();  // per current device; nullptr on failure
int64_t wait_limit_ns();
bool pair_policy_allowed();  // false under TP_POLICY_SINGLE_SM (no pairs, no rank clusters)
bool simt_policy();          // true under TP_POLICY_SIMT (CUDA-core kernel only)
// The status word of the no-allocation entry point's fixed buffer on the
// current device: read into *value and, if nonzero, cleared (with the split
// counters) on `s`.  0 if that entry point has not run on this device.
// Allocates nothing.
int noalloc_status_take(cudaStream_t s, int *value);
void trace_buffer(unsigned long long **buf, int64_t *cap_records);
int set_error(int code, const char *fmt, ...);
void note_launch();  // counts one kernel launch of the calling thread (tp_launch_count)
int cuda_error(cudaError_t e, const char *what);

// Launches `kern` with programmatic stream serialization: it may be scheduled
// while the previous kernel of the stream finishes, so it must call
// griddep_wait() before its first global-memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// ---- launchers (each returns TP_OK or a tp_status, error message set)
int launch_simt(const Problem &p, cudaStream_t s);
int launch_umma(const Problem &p, cudaStream_t s, bool *handled);
int launch_q4(const Problem &p, cudaStream_t s, bool *handled);
// launch_q4 with a caller-provided split workspace instead of the per-stream one;
// fails with TP_ERR_UNSUPPORTED if the launch needs more than it holds.
int launch_q4_fixed_workspace(const Problem &p, cudaStream_t s, bool *handled, float *ws,
                              size_t ws_bytes, int *cnt, size_t ncnt_max);
// Split-reduction workspace supplier: bytes of float32 slots and a count of
// zeroed int counters; returns TP_OK or a tp_status.
typedef int (*GvWorkspaceFn)(void *ctx, size_t bytes, size_t ncounters, float **ws, int **cnt);
// CUDA-core 4-bit GEMV for decode batches of one or two tokens; leaves
// *handled false (and returns TP_OK) for problems it does not take.
int launch_q4_gemv(const Problem &p, cudaStream_t s, bool *handled, GvWorkspaceFn get_ws, void *ctx);
// Tensor-core 4-bit decode with 8-bit operands for up to 16 tokens (k_q4dec.cu);
// leaves *handled false (and returns TP_OK) for problems it does not take.
// ws_cap: the most workspace bytes get_ws can supply (the split is chosen to fit).
int launch_q4_dec8(const Problem &p, cudaStream_t s, bool *handled, GvWorkspaceFn get_ws, void *ctx,
                   size_t ws_cap);
// Debug: every CTA of later 8-bit decode launches prepares all activation
// items itself instead of waiting for the launch-wide count (tp_debug_prep_alone).
void set_dec8_prep_alone(bool on);
int launch_shard(const void *w, int64_t rows, int64_t cols, int elem_bytes, int axis,
                 int segments, int N, void *const *shards, cudaStream_t s);
int launch_quantize(const float *w, int64_t rows, int64_t K, uint32_t *wq, void *scales,
                    void *qbias, cudaStream_t s);
int launch_debug_wait(int64_t limit_ns, int *status, cudaStream_t s);
int launch_mx(const Problem &p, cudaStream_t s, bool *handled);
// Ordered sum of split-K partial tiles (k_split.cu): tiles of 128 rows x BN
// token columns, `splits` float32 slots each, column-major, from ws_base.
struct SplitJob {
  void *C;
  const float *bias;
  int64_t ldc, ws_base;
  int rows, T, tiles, ntiles, splits;
};
int launch_split_reduce(const SplitJob *jobs, int njobs, const float *ws, int BN, int out_dt, cudaStream_t s);
int launch_mx_quantize(const float *w, int64_t rows, int64_t K, uint8_t *codes, uint8_t *scales,
                       cudaStream_t s);
int launch_colsum(int nout, int nin, const void *const *in, int64_t rows, int64_t cols, int64_t ld,
                  int in_dt, float *const *out, cudaStream_t s);
void umma_shutdown();

// ---- shared host helpers (tmap.cu)
int sm_count();
int make_tmap_2d(CUtensorMap *out, const void *ptr, CUtensorMapDataType dt, int elem_bytes,
                 uint64_t inner, uint64_t outer, uint64_t ld_elems, uint32_t box0, uint32_t box1,
                 CUtensorMapSwizzle swz);
// 3-D (chunk, rows, chunks) view of a row-major matrix whose boxes cover
// several consecutive chunks of every row in one tensor copy (tmap.cu).
int make_tmap_3d_chunks(CUtensorMap *out, const void *ptr, CUtensorMapDataType dt, int elem_bytes,
                        uint64_t row_elems, uint64_t rows, uint64_t ld_elems, uint32_t chunk_elems,
                        uint32_t box_rows, uint32_t box_chunks, CUtensorMapSwizzle swz);
void tmap_cache_clear();
// Per-(device, stream) workspace of the split-tile reductions: float partials and
// int arrival counters (zero between calls).  Grows on demand.
int split_workspace(cudaStream_t s, size_t partial_bytes, size_t ncounters, float **partials,
                    int **counters);
void split_workspace_reset();  // clears every counter (after a device-side error)
void split_workspace_free();

}  // namespace tp
