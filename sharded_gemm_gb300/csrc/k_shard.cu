// k_shard.cu -- a1: the `_shard` slicing of one parameter into N device
// buffers ("MLX tensor parallelism guide", section 3.2), as one strided copy
// kernel.  Bit-exact: it moves bytes, in the widest unit (1..16 bytes) that
// every row, run and pointer involved is aligned to.
#include "tp_internal.h"

namespace tp {

struct ShardArgs {
  const uint8_t *src;
  uint8_t *dst[kMaxShards];
  int64_t dst_rows;       // rows of every shard
  int64_t dst_row_units;  // units per shard row
  int64_t src_row_units;  // units per source row
  int64_t w_len;          // slice length along the axis (rows for axis 0, units for axis 1)
  int64_t seg_len;        // segment length along the axis (same unit)
  int axis, N;
};

template <typename U>
__global__ void shard_kernel(const __grid_constant__ ShardArgs a) {
  const int64_t per_shard = a.dst_rows * a.dst_row_units;
  const int64_t total = per_shard * a.N;
  const U *src = reinterpret_cast<const U *>(a.src);
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / per_shard);
    const int64_t rem = idx - (int64_t)r * per_shard;
    const int64_t i = rem / a.dst_row_units;  // shard row
    const int64_t u = rem - i * a.dst_row_units;
    int64_t srow, sunit;
    if (a.axis == 0) {
      srow = (i / a.w_len) * a.seg_len + r * a.w_len + (i % a.w_len);
      sunit = u;
    } else {
      srow = i;
      sunit = (u / a.w_len) * a.seg_len + r * a.w_len + (u % a.w_len);
    }
    reinterpret_cast<U *>(a.dst[r])[rem] = src[srow * a.src_row_units + sunit];
  }
}

static int64_t gcd64(int64_t a, int64_t b) {
  while (b) {
    int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

int launch_shard(const void *w, int64_t rows, int64_t cols, int eb, int axis, int segments, int N,
                 void *const *shards, cudaStream_t s) {
  // Widest unit V (bytes) dividing every row pitch, run length and pointer.
  int64_t g = 16;
  const int64_t row_bytes = cols * eb;
  g = gcd64(g, row_bytes);
  if (axis == 1) {
    const int64_t wl = cols / ((int64_t)segments * N);
    g = gcd64(g, wl * eb);
    g = gcd64(g, (cols / N) * eb);
  }
  g = gcd64(g, (int64_t)((uintptr_t)w & 15));
  for (int r = 0; r < N; ++r) g = gcd64(g, (int64_t)((uintptr_t)shards[r] & 15));
  if (g == 0) g = 16;
  const int V = (int)g;  // 1, 2, 4, 8 or 16

  ShardArgs a;
  a.src = (const uint8_t *)w;
  for (int r = 0; r < N; ++r) a.dst[r] = (uint8_t *)shards[r];
  a.axis = axis;
  a.N = N;
  a.src_row_units = row_bytes / V;
  if (axis == 0) {
    a.dst_rows = rows / N;
    a.dst_row_units = row_bytes / V;
    a.w_len = rows / ((int64_t)segments * N);
    a.seg_len = rows / segments;
  } else {
    a.dst_rows = rows;
    a.dst_row_units = (cols / N) * eb / V;
    a.w_len = (cols / ((int64_t)segments * N)) * eb / V;
    a.seg_len = (cols / segments) * eb / V;
  }
  const int64_t total = a.dst_rows * a.dst_row_units * N;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  switch (V) {
    case 16: shard_kernel<uint4><<<(unsigned)blocks, 256, 0, s>>>(a); break;
    case 8: shard_kernel<uint2><<<(unsigned)blocks, 256, 0, s>>>(a); break;
    case 4: shard_kernel<uint32_t><<<(unsigned)blocks, 256, 0, s>>>(a); break;
    case 2: shard_kernel<uint16_t><<<(unsigned)blocks, 256, 0, s>>>(a); break;
    default: shard_kernel<uint8_t><<<(unsigned)blocks, 256, 0, s>>>(a); break;
  }
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "shard_kernel launch");
}

}  // namespace tp
