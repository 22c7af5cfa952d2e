// k_noalloc.cu -- tp_q4_sharded_to_all_noalloc: the quantized row-parallel
// linear for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: a serving loop that is being captured
// into a CUDA graph, an engine whose memory is owned by its own pool allocator,
// or a latency-critical path where cudaMalloc's implicit device synchronization
// is not acceptable.  The regular tp_q4_sharded_to_all allocates its
// split-reduction workspace (and the library's status word) lazily on first
// use; this variant instead uses one fixed array in device memory that is part
// of the library image, so no call ever allocates.
//
// The array below holds, in order: a 4-byte status word (256 bytes reserved),
// the split arrival counters (64 KiB) and the float32 split partials (the
// rest, 8 MiB - 64 KiB - 256 bytes).  It is allocated by the CUDA driver when
// the library's device code is loaded on a GPU and stays until the process
// exits, on every GPU that loads the library.
#include <string.h>

#include <mutex>

#include "tp_internal.h"

namespace tp {
namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr size_t kStatusBytes = 256;
constexpr size_t kCounterBytes = size_t(64) << 10;
constexpr size_t kPartialBytes = kScratchBytes - kStatusBytes - kCounterBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_addr_mu;
void *g_addr[64] = {nullptr};

// Device address of the scratch array on the current device.  The first call
// on a device looks it up with cudaGetSymbolAddress (no allocation).
int scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(TP_ERR_UNSUPPORTED, "device index %d >= 64", dev);
  std::lock_guard<std::mutex> lk(g_addr_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(scratch)");
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return TP_OK;
}

bool aligned(const void *p, int a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }

}  // namespace

int noalloc_status_take(cudaStream_t s, int *value) {
  *value = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  void *base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_addr_mu);
    if (dev >= 0 && dev < 64) base = g_addr[dev];
  }
  if (!base) return TP_OK;  // no call of the entry point on this device yet
  unsigned char *b = static_cast<unsigned char *>(base);
  int v = 0;
  e = cudaMemcpyAsync(&v, b, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_error(e, "read the fixed buffer's status word");
  if (v != 0) {
    // a kernel may have stopped before re-arming its split counters
    e = cudaMemsetAsync(b + kStatusBytes, 0, kCounterBytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(b, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "clear the fixed buffer's status word");
  }
  *value = v;
  return TP_OK;
}

}  // namespace tp

using namespace tp;

extern "C" int tp_q4_sharded_to_all_noalloc(int N, const void *const *x, int64_t T, int64_t K,
                                            const uint32_t *const *wq, const void *const *scales,
                                            const void *const *qbias, int group_size, int64_t O,
                                            const void *bias, void *y, int64_t ldy, tp_dtype out_dt,
                                            tp_stream_t stream) {
  if (N < 1 || N > kMaxShards) return set_error(TP_ERR_INVALID_ARG, "N must be in 1..%d", kMaxShards);
  if (group_size != 64) return set_error(TP_ERR_UNSUPPORTED, "group_size %d: only 64 is supported", group_size);
  if (out_dt != TP_F32 && out_dt != TP_BF16 && out_dt != TP_F16) return set_error(TP_ERR_INVALID_ARG, "bad dtype");
  if (T < 0 || K < 1 || O < 1) return set_error(TP_ERR_INVALID_ARG, "need T >= 0, K >= 1, O >= 1");
  if (K % N != 0)
    return set_error(TP_ERR_NOT_DIVISIBLE, "Cannot shard the input of size %lld across %d devices.",
                     (long long)K, N);
  const int64_t Kn = K / N;
  if (Kn % group_size)
    return set_error(TP_ERR_NOT_DIVISIBLE, "K/N (%lld) must hold whole groups of %d", (long long)Kn, group_size);
  if (!x || !wq || !scales || !qbias || !y) return set_error(TP_ERR_INVALID_ARG, "null pointer");
  if (ldy < O) return set_error(TP_ERR_INVALID_ARG, "ldy < O");
  if (!aligned(y, out_dt == TP_F32 ? 4 : 2) || (bias && !aligned(bias, 4)))
    return set_error(TP_ERR_ALIGNMENT, "y or bias not aligned to its element size");
  for (int r = 0; r < N; ++r) {
    if (!x[r] || !wq[r] || !scales[r] || !qbias[r])
      return set_error(TP_ERR_INVALID_ARG, "shard %d pointer is NULL", r);
    if (!aligned(x[r], 2) || !aligned(wq[r], 4) || !aligned(scales[r], 2) || !aligned(qbias[r], 2))
      return set_error(TP_ERR_ALIGNMENT, "shard %d pointer not aligned to its element size", r);
  }
  if (T == 0) return TP_OK;

  void *base = nullptr;
  int rc = scratch_address(&base);
  if (rc) return rc;
  unsigned char *b = static_cast<unsigned char *>(base);
  int *status = reinterpret_cast<int *>(b);
  int *counters = reinterpret_cast<int *>(b + kStatusBytes);
  float *partials = reinterpret_cast<float *>(b + kStatusBytes + kCounterBytes);

  Problem p;
  memset(&p, 0, sizeof(p));
  p.njobs = 1;
  p.in_dt = TP_BF16;
  p.out_dt = out_dt;
  p.b_layout = BL_Q4;
  p.chain = 0;
  p.jobs[0] = Job{y, (const float *)bias, T, O, ldy, 0, N};
  for (int r = 0; r < N; ++r) p.parts[r] = Part{x[r], wq[r], scales[r], qbias[r], Kn, Kn, Kn / 8};
  p.status = status;
  p.wait_ns = wait_limit_ns();

  bool handled = false;
  if (!simt_policy()) {
    rc = launch_q4_fixed_workspace(p, (cudaStream_t)stream, &handled, partials, kPartialBytes, counters,
                                   kCounterBytes / sizeof(int));
    if (rc != TP_OK || handled) return rc;
  }
  // Shapes the tensor-core kernel does not take run on the CUDA-core kernel,
  // which needs no scratch.
  return launch_simt(p, (cudaStream_t)stream);
}
