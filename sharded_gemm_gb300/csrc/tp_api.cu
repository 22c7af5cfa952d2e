// tp_api.cu -- the C ABI: argument validation, lowering of each entry point
// to a `Problem`, and dispatch to the kernels.  No kernel lives here.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>

#include "tp_internal.h"

namespace tp {

static thread_local std::string t_last_error;
static thread_local int64_t t_launches = 0;

void note_launch() { ++t_launches; }
static std::atomic<int> g_policy{TP_POLICY_AUTO};
static std::atomic<int64_t> g_wait_ns{2000000000LL};
static std::atomic<unsigned long long *> g_trace{nullptr};
static std::atomic<int64_t> g_trace_cap{0};
static std::mutex g_status_mu;
static int *g_status[64] = {nullptr};

int set_error(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int cuda_error(cudaError_t e, const char *what) {
  return set_error(TP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int64_t wait_limit_ns() { return g_wait_ns.load(); }

bool pair_policy_allowed() { return g_policy.load() != TP_POLICY_SINGLE_SM; }
bool simt_policy() { return g_policy.load() == TP_POLICY_SIMT; }

void trace_buffer(unsigned long long **buf, int64_t *cap_records) {
  *buf = g_trace.load();
  *cap_records = g_trace_cap.load();
}

int *device_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status[dev]) {
    int *p = nullptr;
    if (cudaMalloc(&p, sizeof(int)) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) {
      cudaFree(p);
      return nullptr;
    }
    g_status[dev] = p;
  }
  return g_status[dev];
}

static int elem_size(int dt) { return dt == TP_F32 ? 4 : 2; }
static bool valid_dt(int dt) { return dt == TP_F32 || dt == TP_BF16 || dt == TP_F16; }
static bool aligned(const void *p, int a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }

static int dispatch(Problem &p, cudaStream_t s) {
  p.status = device_status_word();
  if (!p.status) return set_error(TP_ERR_CUDA, "cannot allocate the device status word");
  p.wait_ns = wait_limit_ns();
  bool handled = false;
  if (g_policy.load() != TP_POLICY_SIMT) {
    int rc = p.b_layout == BL_Q4   ? launch_q4(p, s, &handled)
             : p.b_layout == BL_MX ? launch_mx(p, s, &handled)
                                   : launch_umma(p, s, &handled);
    if (rc != TP_OK || handled) return rc;
  }
  return launch_simt(p, s);
}

}  // namespace tp

using namespace tp;

int64_t tp_launch_count(void) { return t_launches; }

extern "C" {

int tp_version(void) { return 100; }

const char *tp_last_error(void) { return t_last_error.c_str(); }

int tp_set_policy(int policy) {
  if (policy != TP_POLICY_AUTO && policy != TP_POLICY_SIMT && policy != TP_POLICY_SINGLE_SM)
    return set_error(TP_ERR_INVALID_ARG, "unknown policy %d", policy);
  g_policy.store(policy);
  return TP_OK;
}

int tp_set_wait_limit_ns(int64_t ns) {
  if (ns < 1000000LL || ns > 60000000000LL)
    return set_error(TP_ERR_INVALID_ARG, "wait limit %lld ns outside [1e6, 6e10]", (long long)ns);
  g_wait_ns.store(ns);
  return TP_OK;
}

int tp_set_trace(void *device_buffer, int64_t bytes) {
  if (!device_buffer) {
    g_trace.store(nullptr);
    g_trace_cap.store(0);
    return TP_OK;
  }
  if (bytes < (int64_t)(16 + 32 * 1024) * 8 || ((uintptr_t)device_buffer & 15))
    return set_error(TP_ERR_INVALID_ARG, "trace buffer must be >= 262272 bytes and 16-byte aligned");
  g_trace_cap.store(bytes / 8);
  g_trace.store((unsigned long long *)device_buffer);
  return TP_OK;
}

int tp_query_status(tp_stream_t stream, int *device_status) {
  if (!device_status) return set_error(TP_ERR_INVALID_ARG, "device_status is NULL");
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  int *w = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (dev >= 0 && dev < 64) w = g_status[dev];  // never allocated here
  }
  int v = 0;
  if (w) {
    e = cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_error(e, "read status word");
    if (v != 0) {
      e = cudaMemset(w, 0, sizeof(int));
      if (e != cudaSuccess) return cuda_error(e, "clear status word");
      split_workspace_reset();  // a kernel may have stopped mid-reduction
    }
  }
  int v2 = 0;
  int rc = noalloc_status_take((cudaStream_t)stream, &v2);
  if (rc) return rc;
  *device_status = v != 0 ? v : v2;
  return TP_OK;
}

int tp_shutdown(void) {
  std::lock_guard<std::mutex> lk(g_status_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (int d = 0; d < 64; ++d) {
    if (g_status[d]) {
      cudaSetDevice(d);
      cudaFree(g_status[d]);
      g_status[d] = nullptr;
    }
  }
  cudaSetDevice(cur);
  umma_shutdown();
  return TP_OK;
}

int tp_shard_weight(const void *w, int64_t rows, int64_t cols, int elem_bytes, int axis,
                    int segments, int N, void *const *shards, tp_stream_t stream) {
  if (!w || !shards) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (rows < 1 || cols < 1) return set_error(TP_ERR_INVALID_ARG, "rows and cols must be >= 1");
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return set_error(TP_ERR_INVALID_ARG, "elem_bytes must be 1, 2, 4 or 8");
  if (axis == -1) axis = 1;
  if (axis != 0 && axis != 1) return set_error(TP_ERR_INVALID_ARG, "axis must be 0, 1 or -1");
  if (segments < 1) return set_error(TP_ERR_INVALID_ARG, "segments must be >= 1");
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  int64_t L = axis == 0 ? rows : cols;
  if (L % ((int64_t)segments * N) != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the output of size %lld across %d devices.",
                     (long long)L, segments * N);
  if (!aligned(w, elem_bytes)) return set_error(TP_ERR_ALIGNMENT, "w not aligned to its element size");
  for (int r = 0; r < N; ++r) {
    if (!shards[r]) return set_error(TP_ERR_INVALID_ARG, "shards[%d] is NULL", r);
    if (!aligned(shards[r], elem_bytes))
      return set_error(TP_ERR_ALIGNMENT, "shards[%d] not aligned to its element size", r);
  }
  return launch_shard(w, rows, cols, elem_bytes, axis, segments, N, shards, (cudaStream_t)stream);
}

int tp_all_to_sharded(int N, const void *x, int64_t T, int64_t K, int64_t ldx,
                      const void *const *w, int64_t O, const void *const *bias, tp_dtype in_dt,
                      void *const *y, int64_t ldy, tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  if (!valid_dt(in_dt) || !valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  if (O % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the output of size %lld across %d devices.",
                     (long long)O, N);
  const int64_t On = O / N;
  if (!x || !w || !y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldx < K) return set_error(TP_ERR_INVALID_ARG, "ldx (%lld) < K (%lld)", (long long)ldx, (long long)K);
  if (ldy < On) return set_error(TP_ERR_INVALID_ARG, "ldy (%lld) < O/N (%lld)", (long long)ldy, (long long)On);
  const int ie = elem_size(in_dt), oe = elem_size(out_dt);
  if (!aligned(x, ie)) return set_error(TP_ERR_ALIGNMENT, "x not aligned to its element size");
  for (int r = 0; r < N; ++r) {
    if (!w[r] || !y[r]) return set_error(TP_ERR_INVALID_ARG, "w[%d] or y[%d] is NULL", r, r);
    if (bias && !bias[r]) return set_error(TP_ERR_INVALID_ARG, "bias[%d] is NULL", r);
    if (!aligned(w[r], ie) || !aligned(y[r], oe) || (bias && !aligned(bias[r], 4)))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = N;
  p.in_dt = in_dt;
  p.out_dt = out_dt;
  p.b_layout = BL_KMAJOR;
  p.chain = 1;
  for (int r = 0; r < N; ++r) {
    p.jobs[r] = Job{y[r], bias ? (const float *)bias[r] : nullptr, T, On, ldy, r, 1};
    p.parts[r] = Part{x, w[r], nullptr, nullptr, K, ldx, K};
  }
  return dispatch(p, (cudaStream_t)stream);
}

int tp_gated_all_to_sharded(int N, const void *x, int64_t T, int64_t K, int64_t ldx,
                            const void *const *w1, const void *const *w3, int64_t F,
                            const void *const *b1, const void *const *b3, tp_dtype in_dt,
                            void *const *h, int64_t ldh, tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  if (!valid_dt(in_dt) || !valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || F < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, F >= 1");
  if (F % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the output of size %lld across %d devices.",
                     (long long)F, N);
  const int64_t Fn = F / N;
  if (!x || !w1 || !w3 || !h) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldx < K) return set_error(TP_ERR_INVALID_ARG, "ldx (%lld) < K (%lld)", (long long)ldx, (long long)K);
  if (ldh < Fn) return set_error(TP_ERR_INVALID_ARG, "ldh (%lld) < F/N (%lld)", (long long)ldh, (long long)Fn);
  const int ie = elem_size(in_dt), oe = elem_size(out_dt);
  if (!aligned(x, ie)) return set_error(TP_ERR_ALIGNMENT, "x not aligned to its element size");
  for (int r = 0; r < N; ++r) {
    if (!w1[r] || !w3[r] || !h[r]) return set_error(TP_ERR_INVALID_ARG, "w1[%d], w3[%d] or h[%d] is NULL", r, r, r);
    if ((b1 && !b1[r]) || (b3 && !b3[r])) return set_error(TP_ERR_INVALID_ARG, "b1[%d] or b3[%d] is NULL", r, r);
    if (!aligned(w1[r], ie) || !aligned(w3[r], ie) || !aligned(h[r], oe) || (b1 && !aligned(b1[r], 4)) ||
        (b3 && !aligned(b3[r], 4)))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = N;
  p.in_dt = in_dt;
  p.out_dt = out_dt;
  p.b_layout = BL_KMAJOR;
  p.chain = 1;
  p.gated = 1;
  for (int r = 0; r < N; ++r) {
    p.jobs[r] = Job{h[r], b1 ? (const float *)b1[r] : nullptr, T, Fn, ldh, r, 1,
                    b3 ? (const float *)b3[r] : nullptr};
    p.parts[r] = Part{x, w1[r], nullptr, nullptr, K, ldx, K, w3[r]};
  }
  return dispatch(p, (cudaStream_t)stream);
}

int tp_sharded_to_all(int N, const void *const *x, int64_t T, int64_t K, int64_t ldx,
                      const void *const *w, int64_t O, const void *bias, tp_dtype in_dt, void *y,
                      int64_t ldy, tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  if (!valid_dt(in_dt) || !valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  if (K % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the input of size %lld across %d devices.",
                     (long long)K, N);
  const int64_t Kn = K / N;
  if (!x || !w || !y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldx < Kn) return set_error(TP_ERR_INVALID_ARG, "ldx (%lld) < K/N (%lld)", (long long)ldx, (long long)Kn);
  if (ldy < O) return set_error(TP_ERR_INVALID_ARG, "ldy (%lld) < O (%lld)", (long long)ldy, (long long)O);
  const int ie = elem_size(in_dt), oe = elem_size(out_dt);
  if (!aligned(y, oe) || (bias && !aligned(bias, 4)))
    return set_error(TP_ERR_ALIGNMENT, "y or bias not aligned to its element size");
  for (int r = 0; r < N; ++r) {
    if (!x[r] || !w[r]) return set_error(TP_ERR_INVALID_ARG, "x[%d] or w[%d] is NULL", r, r);
    if (!aligned(x[r], ie) || !aligned(w[r], ie))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = 1;
  p.in_dt = in_dt;
  p.out_dt = out_dt;
  p.b_layout = BL_KMAJOR;
  p.chain = 0;
  p.jobs[0] = Job{y, (const float *)bias, T, O, ldy, 0, N};
  for (int r = 0; r < N; ++r) p.parts[r] = Part{x[r], w[r], nullptr, nullptr, Kn, ldx, Kn};
  return dispatch(p, (cudaStream_t)stream);
}

int tp_sharded_to_sharded(int N, const void *const *x, int64_t T, int64_t K, int64_t ldx,
                          const void *const *w, int64_t O, const void *bias, tp_dtype in_dt,
                          void *const *y, int64_t ldy, tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  if (N * N > kMaxParts)
    return set_error(TP_ERR_UNSUPPORTED, "reduce-scatter over %d ranks: at most %d partial blocks", N,
                     kMaxParts);
  if (!valid_dt(in_dt) || !valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  if (K % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the input of size %lld across %d devices.",
                     (long long)K, N);
  if (O % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the output of size %lld across %d devices.",
                     (long long)O, N);
  const int64_t Kn = K / N, On = O / N;
  if (!x || !w || !y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldx < Kn) return set_error(TP_ERR_INVALID_ARG, "ldx (%lld) < K/N (%lld)", (long long)ldx, (long long)Kn);
  if (ldy < On) return set_error(TP_ERR_INVALID_ARG, "ldy (%lld) < O/N (%lld)", (long long)ldy, (long long)On);
  const int ie = elem_size(in_dt), oe = elem_size(out_dt);
  if (bias && !aligned(bias, 4)) return set_error(TP_ERR_ALIGNMENT, "bias not aligned to its element size");
  for (int r = 0; r < N; ++r) {
    if (!x[r] || !w[r] || !y[r]) return set_error(TP_ERR_INVALID_ARG, "x[%d], w[%d] or y[%d] is NULL", r, r, r);
    if (!aligned(x[r], ie) || !aligned(w[r], ie) || !aligned(y[r], oe))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  // Job c is output block c; its part r is rank r's partial x[r] @ W_r[c]^T,
  // W_r[c] being rows c*O/N.. of w[r] (a contiguous (O/N, K/N) block).
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = N;
  p.in_dt = in_dt;
  p.out_dt = out_dt;
  p.b_layout = BL_KMAJOR;
  p.chain = 0;
  for (int c = 0; c < N; ++c) {
    p.jobs[c] = Job{y[c], bias ? (const float *)bias + c * On : nullptr, T, On, ldy, c * N, N};
    for (int r = 0; r < N; ++r)
      p.parts[c * N + r] = Part{x[r], (const char *)w[r] + (size_t)(c * On * Kn) * ie, nullptr, nullptr, Kn,
                                ldx, Kn};
  }
  return dispatch(p, (cudaStream_t)stream);
}

int tp_gathered_to_sharded(int N, const void *const *x, int64_t T, int64_t K, int64_t ldx,
                           const void *const *w, int64_t O, const void *const *bias, tp_dtype in_dt,
                           void *const *y, int64_t ldy, tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  if (N * N > kMaxParts)
    return set_error(TP_ERR_UNSUPPORTED, "all-gather over %d ranks: at most %d input blocks", N, kMaxParts);
  if (!valid_dt(in_dt) || !valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  if (K % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the input of size %lld across %d devices.",
                     (long long)K, N);
  if (O % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the output of size %lld across %d devices.",
                     (long long)O, N);
  const int64_t Kn = K / N, On = O / N;
  if (!x || !w || !y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldx < Kn) return set_error(TP_ERR_INVALID_ARG, "ldx (%lld) < K/N (%lld)", (long long)ldx, (long long)Kn);
  if (ldy < On) return set_error(TP_ERR_INVALID_ARG, "ldy (%lld) < O/N (%lld)", (long long)ldy, (long long)On);
  const int ie = elem_size(in_dt), oe = elem_size(out_dt);
  for (int r = 0; r < N; ++r) {
    if (!x[r] || !w[r] || !y[r]) return set_error(TP_ERR_INVALID_ARG, "x[%d], w[%d] or y[%d] is NULL", r, r, r);
    if (bias && !bias[r]) return set_error(TP_ERR_INVALID_ARG, "bias[%d] is NULL", r);
    if (!aligned(x[r], ie) || !aligned(w[r], ie) || !aligned(y[r], oe) || (bias && !aligned(bias[r], 4)))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  // Job r is rank r's column-parallel output; its parts q = 0..N-1 chain the
  // gathered input's column blocks x[q] against columns q*K/N.. of w[r] into
  // one float32 accumulator, in block order (the order of the gathered K).
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = N;
  p.in_dt = in_dt;
  p.out_dt = out_dt;
  p.b_layout = BL_KMAJOR;
  p.chain = 1;
  for (int r = 0; r < N; ++r) {
    p.jobs[r] = Job{y[r], bias ? (const float *)bias[r] : nullptr, T, On, ldy, r * N, N};
    for (int q = 0; q < N; ++q)
      p.parts[r * N + q] = Part{x[q], (const char *)w[r] + (size_t)(q * Kn) * ie, nullptr, nullptr, Kn, ldx, K};
  }
  return dispatch(p, (cudaStream_t)stream);
}

int tp_all_to_sharded_dx(int N, const void *const *dy, int64_t T, int64_t O, int64_t lddy,
                         const void *const *w, int64_t K, tp_dtype in_dt, void *dx, int64_t lddx,
                         tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  if (!valid_dt(in_dt) || !valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  if (O % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the output of size %lld across %d devices.",
                     (long long)O, N);
  const int64_t On = O / N;
  if (!dy || !w || !dx) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (lddy < On) return set_error(TP_ERR_INVALID_ARG, "lddy (%lld) < O/N (%lld)", (long long)lddy, (long long)On);
  if (lddx < K) return set_error(TP_ERR_INVALID_ARG, "lddx (%lld) < K (%lld)", (long long)lddx, (long long)K);
  const int ie = elem_size(in_dt), oe = elem_size(out_dt);
  if (!aligned(dx, oe)) return set_error(TP_ERR_ALIGNMENT, "dx not aligned to its element size");
  for (int r = 0; r < N; ++r) {
    if (!dy[r] || !w[r]) return set_error(TP_ERR_INVALID_ARG, "dy[%d] or w[%d] is NULL", r, r);
    if (!aligned(dy[r], ie) || !aligned(w[r], ie))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  // One output, N partials dy[r] @ w[r] (w[r] is (O/N, K): K-contiguous rows
  // of the contraction), formed from zero and added in ascending r.
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = 1;
  p.in_dt = in_dt;
  p.out_dt = out_dt;
  p.b_layout = BL_MNMAJOR;
  p.chain = 0;
  p.jobs[0] = Job{dx, nullptr, T, K, lddx, 0, N};
  for (int r = 0; r < N; ++r) p.parts[r] = Part{dy[r], w[r], nullptr, nullptr, On, lddy, K};
  return dispatch(p, (cudaStream_t)stream);
}

int tp_sharded_to_all_dx(int N, const void *dy, int64_t T, int64_t O, int64_t lddy, const void *const *w,
                         int64_t K, tp_dtype in_dt, void *const *dx, int64_t lddx, tp_dtype out_dt,
                         tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  if (!valid_dt(in_dt) || !valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  if (K % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the input of size %lld across %d devices.",
                     (long long)K, N);
  const int64_t Kn = K / N;
  if (!dy || !w || !dx) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (lddy < O) return set_error(TP_ERR_INVALID_ARG, "lddy (%lld) < O (%lld)", (long long)lddy, (long long)O);
  if (lddx < Kn) return set_error(TP_ERR_INVALID_ARG, "lddx (%lld) < K/N (%lld)", (long long)lddx, (long long)Kn);
  const int ie = elem_size(in_dt), oe = elem_size(out_dt);
  if (!aligned(dy, ie)) return set_error(TP_ERR_ALIGNMENT, "dy not aligned to its element size");
  for (int r = 0; r < N; ++r) {
    if (!w[r] || !dx[r]) return set_error(TP_ERR_INVALID_ARG, "w[%d] or dx[%d] is NULL", r, r);
    if (!aligned(w[r], ie) || !aligned(dx[r], oe))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = N;
  p.in_dt = in_dt;
  p.out_dt = out_dt;
  p.b_layout = BL_MNMAJOR;
  p.chain = 1;
  for (int r = 0; r < N; ++r) {
    p.jobs[r] = Job{dx[r], nullptr, T, Kn, lddx, r, 1};
    p.parts[r] = Part{dy, w[r], nullptr, nullptr, O, lddy, Kn};
  }
  return dispatch(p, (cudaStream_t)stream);
}

int tp_sharded_dw(int N, const void *const *dy, int64_t lddy, const void *const *x, int64_t ldx, int64_t T,
                  int64_t O, int64_t K, tp_dtype in_dt, void *const *dw, int64_t lddw, tp_dtype out_dt,
                  tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  if (!valid_dt(in_dt) || !valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  if (!dy || !x || !dw) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (lddy < O) return set_error(TP_ERR_INVALID_ARG, "lddy (%lld) < O (%lld)", (long long)lddy, (long long)O);
  if (ldx < K) return set_error(TP_ERR_INVALID_ARG, "ldx (%lld) < K (%lld)", (long long)ldx, (long long)K);
  if (lddw < K) return set_error(TP_ERR_INVALID_ARG, "lddw (%lld) < K (%lld)", (long long)lddw, (long long)K);
  const int ie = elem_size(in_dt), oe = elem_size(out_dt);
  for (int r = 0; r < N; ++r) {
    // an empty batch (T = 0) may come with null operand pointers
    if ((T > 0 && (!dy[r] || !x[r])) || !dw[r])
      return set_error(TP_ERR_INVALID_ARG, "dy[%d], x[%d] or dw[%d] is NULL", r, r, r);
    if (!aligned(dy[r], ie) || !aligned(x[r], ie) || !aligned(dw[r], oe))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) {  // an empty sum over tokens: the gradient is zero
    for (int r = 0; r < N; ++r) {
      cudaError_t e = cudaMemset2DAsync(dw[r], (size_t)(lddw * oe), 0, (size_t)(K * oe), (size_t)O,
                                        (cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_error(e, "cudaMemset2DAsync");
    }
    return TP_OK;
  }
  // dW_r(o, k) = sum over tokens t of dy_r[t][o] * x_r[t][k]: both operands
  // are read token-major (M- and N-major), the contraction runs over T.
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = N;
  p.in_dt = in_dt;
  p.out_dt = out_dt;
  p.b_layout = BL_MNMAJOR;
  p.a_mn = 1;
  p.chain = 1;
  for (int r = 0; r < N; ++r) {
    p.jobs[r] = Job{dw[r], nullptr, O, K, lddw, r, 1};
    p.parts[r] = Part{dy[r], x[r], nullptr, nullptr, T, lddy, ldx};
  }
  return dispatch(p, (cudaStream_t)stream);
}

int tp_bias_grad(int nout, int nin, const void *const *dy, int64_t rows, int64_t cols, int64_t ld,
                 tp_dtype in_dt, float *const *db, tp_stream_t stream) {
  if (nout < 1 || nout > kMaxJobs || nin < 1 || nout * nin > kMaxParts)
    return set_error(TP_ERR_INVALID_ARG, "need 1 <= nout <= %d, nin >= 1, nout * nin <= %d", kMaxJobs,
                     kMaxParts);
  if (!valid_dt(in_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (rows < 0 || cols < 1) return set_error(TP_ERR_INVALID_ARG, "need rows >= 0, cols >= 1");
  if (ld < cols) return set_error(TP_ERR_INVALID_ARG, "ld (%lld) < cols (%lld)", (long long)ld, (long long)cols);
  if (!dy || !db) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  const int ie = elem_size(in_dt);
  for (int i = 0; i < nout * nin; ++i)
    if ((rows > 0 && !dy[i]) || !aligned(dy[i], ie))
      return set_error(TP_ERR_INVALID_ARG, "dy[%d] is NULL or unaligned", i);
  for (int o = 0; o < nout; ++o)
    if (!db[o] || !aligned(db[o], 4)) return set_error(TP_ERR_INVALID_ARG, "db[%d] is NULL or unaligned", o);
  return launch_colsum(nout, nin, dy, rows, cols, ld, in_dt, db, (cudaStream_t)stream);
}

// SUMMA-family lowering: q*q output blocks, each chaining q block products in
// step order t.  kind 0: Y_ij = sum_t X_it A_tj (+ bias_j);  kind 1 (A B^T):
// Y_ij = sum_t X_it A_jt^T;  kind 2 (A^T B): Y_ij = sum_t X_ti^T A_tj.
static int summa_lower(int kind, int q, const void *const *X, const void *const *A,
                       const void *const *bias, void *const *Y, int64_t M, int64_t K, int64_t Ncols,
                       tp_dtype in_dt, tp_stream_t stream) {
  if (q < 1) return set_error(TP_ERR_NOT_DIVISIBLE, "q must be >= 1 (P = q*q processors)");
  if (q > 4) return set_error(TP_ERR_UNSUPPORTED, "q = %d: this build supports q <= 4", q);
  if (!valid_dt(in_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (M < 1 || K < 1 || Ncols < 1) return set_error(TP_ERR_INVALID_ARG, "sizes must be >= 1");
  if (M % q || K % q || Ncols % q)
    return set_error(TP_ERR_NOT_DIVISIBLE, "M=%lld, K=%lld, N=%lld must all be multiples of q=%d",
                     (long long)M, (long long)K, (long long)Ncols, q);
  if (!X || !A || !Y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  const int ie = elem_size(in_dt);
  for (int b = 0; b < q * q; ++b) {
    if (!X[b] || !A[b] || !Y[b]) return set_error(TP_ERR_INVALID_ARG, "block %d pointer is NULL", b);
    if (!aligned(X[b], ie) || !aligned(A[b], ie) || !aligned(Y[b], 4))
      return set_error(TP_ERR_ALIGNMENT, "block %d pointer not aligned to its element size", b);
  }
  if (bias)
    for (int j = 0; j < q; ++j)
      if (!bias[j] || !aligned(bias[j], 4)) return set_error(TP_ERR_INVALID_ARG, "bias[%d] is NULL or unaligned", j);
  const int64_t bm = M / q, bk = K / q, bn = Ncols / q;
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = q * q;
  p.in_dt = in_dt;
  p.out_dt = TP_F32;
  p.b_layout = kind == 1 ? BL_KMAJOR : BL_MNMAJOR;
  p.a_mn = kind == 2;
  p.chain = 1;
  for (int i = 0; i < q; ++i)
    for (int j = 0; j < q; ++j) {
      const int jb = i * q + j;
      p.jobs[jb] = Job{Y[jb], bias ? (const float *)bias[j] : nullptr, bm, bn, bn, jb * q, q};
      for (int t = 0; t < q; ++t) {
        Part &P = p.parts[jb * q + t];
        if (kind == 0)
          P = Part{X[i * q + t], A[t * q + j], nullptr, nullptr, bk, bk, bn};
        else if (kind == 1)
          P = Part{X[i * q + t], A[j * q + t], nullptr, nullptr, bk, bk, bk};
        else
          P = Part{X[t * q + i], A[t * q + j], nullptr, nullptr, bk, bm, bn};
      }
    }
  return dispatch(p, (cudaStream_t)stream);
}

int tp_summa(int q, const void *const *X, const void *const *A, void *const *Y, int64_t M,
             int64_t K, int64_t Ncols, tp_dtype in_dt, tp_stream_t stream) {
  return summa_lower(0, q, X, A, nullptr, Y, M, K, Ncols, in_dt, stream);
}

int tp_summa_linear(int q, const void *const *X, const void *const *A, const void *const *bias,
                    void *const *Y, int64_t M, int64_t K, int64_t Ncols, tp_dtype in_dt,
                    tp_stream_t stream) {
  return summa_lower(0, q, X, A, bias, Y, M, K, Ncols, in_dt, stream);
}

int tp_summa_abt(int q, const void *const *A, const void *const *B, void *const *C, int64_t M,
                 int64_t K, int64_t Ncols, tp_dtype in_dt, tp_stream_t stream) {
  return summa_lower(1, q, A, B, nullptr, C, M, K, Ncols, in_dt, stream);
}

int tp_summa_atb(int q, const void *const *A, const void *const *B, void *const *C, int64_t M,
                 int64_t K, int64_t Ncols, tp_dtype in_dt, tp_stream_t stream) {
  return summa_lower(2, q, A, B, nullptr, C, M, K, Ncols, in_dt, stream);
}

static int mx_check_common(int64_t T, int64_t K, int64_t O, tp_dtype out_dt) {
  if (!valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  return TP_OK;
}

int tp_mx_quantize(const float *w, int64_t rows, int64_t K, uint8_t *codes, uint8_t *scales,
                   tp_stream_t stream) {
  if (!w || !codes || !scales) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (rows < 1 || K < 1) return set_error(TP_ERR_INVALID_ARG, "rows and K must be >= 1");
  if (K % 32) return set_error(TP_ERR_NOT_DIVISIBLE, "K (%lld) not a multiple of 32", (long long)K);
  if (!aligned(w, 4)) return set_error(TP_ERR_ALIGNMENT, "w not aligned to its element size");
  return launch_mx_quantize(w, rows, K, codes, scales, (cudaStream_t)stream);
}

int tp_mx_all_to_sharded(int N, const void *x, int64_t T, int64_t K, const uint8_t *const *codes,
                         const uint8_t *const *scales, int64_t O, const void *const *bias, void *const *y,
                         int64_t ldy, tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  int rc = mx_check_common(T, K, O, out_dt);
  if (rc) return rc;
  if (O % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the output of size %lld across %d devices.",
                     (long long)O, N);
  if (K % 32) return set_error(TP_ERR_NOT_DIVISIBLE, "K (%lld) not a multiple of 32", (long long)K);
  const int64_t On = O / N;
  if (!x || !codes || !scales || !y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldy < On) return set_error(TP_ERR_INVALID_ARG, "ldy < O/N");
  const int oe = elem_size(out_dt);
  if (!aligned(x, 2)) return set_error(TP_ERR_ALIGNMENT, "x not aligned");
  for (int r = 0; r < N; ++r) {
    if (!codes[r] || !scales[r] || !y[r] || (bias && !bias[r]))
      return set_error(TP_ERR_INVALID_ARG, "shard %d pointer is NULL", r);
    if (!aligned(y[r], oe) || (bias && !aligned(bias[r], 4)))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = N;
  p.in_dt = TP_BF16;
  p.out_dt = out_dt;
  p.b_layout = BL_MX;
  p.chain = 1;
  for (int r = 0; r < N; ++r) {
    p.jobs[r] = Job{y[r], bias ? (const float *)bias[r] : nullptr, T, On, ldy, r, 1};
    p.parts[r] = Part{x, codes[r], scales[r], nullptr, K, K, K};
  }
  return dispatch(p, (cudaStream_t)stream);
}

int tp_mx_sharded_to_all(int N, const void *const *x, int64_t T, int64_t K, const uint8_t *const *codes,
                         const uint8_t *const *scales, int64_t O, const void *bias, void *y, int64_t ldy,
                         tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  int rc = mx_check_common(T, K, O, out_dt);
  if (rc) return rc;
  if (K % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the input of size %lld across %d devices.",
                     (long long)K, N);
  const int64_t Kn = K / N;
  if (Kn % 32)
    return set_error(TP_ERR_NOT_DIVISIBLE, "K/N (%lld) must hold whole blocks of 32", (long long)Kn);
  if (!x || !codes || !scales || !y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldy < O) return set_error(TP_ERR_INVALID_ARG, "ldy < O");
  const int oe = elem_size(out_dt);
  if (!aligned(y, oe) || (bias && !aligned(bias, 4))) return set_error(TP_ERR_ALIGNMENT, "y or bias not aligned");
  for (int r = 0; r < N; ++r) {
    if (!x[r] || !codes[r] || !scales[r]) return set_error(TP_ERR_INVALID_ARG, "shard %d pointer is NULL", r);
    if (!aligned(x[r], 2)) return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned", r);
  }
  if (T == 0) return TP_OK;
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = 1;
  p.in_dt = TP_BF16;
  p.out_dt = out_dt;
  p.b_layout = BL_MX;
  p.chain = 0;
  p.jobs[0] = Job{y, (const float *)bias, T, O, ldy, 0, N};
  for (int r = 0; r < N; ++r) p.parts[r] = Part{x[r], codes[r], scales[r], nullptr, Kn, Kn, Kn};
  return dispatch(p, (cudaStream_t)stream);
}

int tp_q4_quantize(const float *w, int64_t rows, int64_t K, int group_size, uint32_t *wq,
                   void *scales, void *qbias, tp_stream_t stream) {
  if (group_size != 64) return set_error(TP_ERR_UNSUPPORTED, "group_size %d: only 64 is supported", group_size);
  if (!w || !wq || !scales || !qbias) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (rows < 1 || K < 1) return set_error(TP_ERR_INVALID_ARG, "rows and K must be >= 1");
  if (K % group_size) return set_error(TP_ERR_NOT_DIVISIBLE, "K (%lld) not a multiple of %d", (long long)K, group_size);
  if (!aligned(w, 4) || !aligned(wq, 4) || !aligned(scales, 2) || !aligned(qbias, 2))
    return set_error(TP_ERR_ALIGNMENT, "pointer not aligned to its element size");
  return launch_quantize(w, rows, K, wq, scales, qbias, (cudaStream_t)stream);
}

static int q4_check_common(int group_size, int64_t T, int64_t K, int64_t O, tp_dtype out_dt) {
  if (group_size != 64) return set_error(TP_ERR_UNSUPPORTED, "group_size %d: only 64 is supported", group_size);
  if (!valid_dt(out_dt)) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  return TP_OK;
}

int tp_q4_all_to_sharded(int N, const void *x, int64_t T, int64_t K, const uint32_t *const *wq,
                         const void *const *scales, const void *const *qbias, int group_size,
                         int64_t O, const void *const *bias, void *const *y, int64_t ldy,
                         tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  int rc = q4_check_common(group_size, T, K, O, out_dt);
  if (rc) return rc;
  if (O % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the output of size %lld across %d devices.",
                     (long long)O, N);
  if (K % group_size) return set_error(TP_ERR_NOT_DIVISIBLE, "K (%lld) not a multiple of %d", (long long)K, group_size);
  const int64_t On = O / N;
  if (!x || !wq || !scales || !qbias || !y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldy < On) return set_error(TP_ERR_INVALID_ARG, "ldy < O/N");
  const int oe = elem_size(out_dt);
  if (!aligned(x, 2)) return set_error(TP_ERR_ALIGNMENT, "x not aligned");
  for (int r = 0; r < N; ++r) {
    if (!wq[r] || !scales[r] || !qbias[r] || !y[r] || (bias && !bias[r]))
      return set_error(TP_ERR_INVALID_ARG, "shard %d pointer is NULL", r);
    if (!aligned(wq[r], 4) || !aligned(scales[r], 2) || !aligned(qbias[r], 2) || !aligned(y[r], oe) ||
        (bias && !aligned(bias[r], 4)))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = N;
  p.in_dt = TP_BF16;
  p.out_dt = out_dt;
  p.b_layout = BL_Q4;
  p.chain = 1;
  for (int r = 0; r < N; ++r) {
    p.jobs[r] = Job{y[r], bias ? (const float *)bias[r] : nullptr, T, On, ldy, r, 1};
    p.parts[r] = Part{x, wq[r], scales[r], qbias[r], K, K, K / 8};
  }
  return dispatch(p, (cudaStream_t)stream);
}

int tp_q4_sharded_to_all(int N, const void *const *x, int64_t T, int64_t K,
                         const uint32_t *const *wq, const void *const *scales,
                         const void *const *qbias, int group_size, int64_t O, const void *bias,
                         void *y, int64_t ldy, tp_dtype out_dt, tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  int rc = q4_check_common(group_size, T, K, O, out_dt);
  if (rc) return rc;
  if (K % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the input of size %lld across %d devices.",
                     (long long)K, N);
  const int64_t Kn = K / N;
  if (Kn % group_size)
    return set_error(TP_ERR_NOT_DIVISIBLE, "K/N (%lld) must hold whole groups of %d", (long long)Kn, group_size);
  if (!x || !wq || !scales || !qbias || !y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldy < O) return set_error(TP_ERR_INVALID_ARG, "ldy < O");
  if (!aligned(y, elem_size(out_dt)) || (bias && !aligned(bias, 4)))
    return set_error(TP_ERR_ALIGNMENT, "y or bias not aligned to its element size");
  for (int r = 0; r < N; ++r) {
    if (!x[r] || !wq[r] || !scales[r] || !qbias[r]) return set_error(TP_ERR_INVALID_ARG, "shard %d pointer is NULL", r);
    if (!aligned(x[r], 2) || !aligned(wq[r], 4) || !aligned(scales[r], 2) || !aligned(qbias[r], 2))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;
  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = 1;
  p.in_dt = TP_BF16;
  p.out_dt = out_dt;
  p.b_layout = BL_Q4;
  p.chain = 0;
  p.jobs[0] = Job{y, (const float *)bias, T, O, ldy, 0, N};
  for (int r = 0; r < N; ++r) p.parts[r] = Part{x[r], wq[r], scales[r], qbias[r], Kn, Kn, Kn / 8};
  return dispatch(p, (cudaStream_t)stream);
}

int tp_debug_prep_alone(int on) {
  set_dec8_prep_alone(on != 0);
  return TP_OK;
}

int tp_debug_wait_timeout(int64_t limit_ns, tp_stream_t stream) {
  if (limit_ns < 1000000LL || limit_ns > 60000000000LL)
    return set_error(TP_ERR_INVALID_ARG, "limit %lld ns outside [1e6, 6e10]", (long long)limit_ns);
  int *st = device_status_word();
  if (!st) return set_error(TP_ERR_CUDA, "cannot allocate the device status word");
  return launch_debug_wait(limit_ns, st, (cudaStream_t)stream);
}

}  // extern "C"
