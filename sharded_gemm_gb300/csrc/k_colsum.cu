// k_colsum.cu -- bias gradients: float32 column sums of one or more row-major
// (rows, cols) matrices.  The bias of a linear layer is added to every row of
// its output, so its gradient is the sum over rows of the output gradient;
// for the 2-D (SUMMA) layer the column group's blocks are summed as well.
//
// out[o][c] = sum over inputs b = 0..nin-1 (in order) of sum over rows t of
// in[o*nin + b][t*ld + c].  HBM-bound: one read of each input.  Every
// partial sum is added in a fixed order, so the result does not depend on
// scheduling.
//
// colsum_cluster_kernel (16-byte aligned rows): a cluster of 8 CTAs owns a
// strip of 32 * VEC columns (VEC = 16 bytes of elements per lane, so a warp
// reads one 512-byte row segment) and splits the rows into 8 chunks, one per
// CTA; inside a CTA warp w adds rows w, w+8, ... of the chunk (8 vector loads
// in flight per lane), the 8 warp sums are added in warp order, and CTA 0
// adds the 8 chunk sums in rank order from its peers' shared memory.
// colsum_kernel (any alignment): a CTA owns 32 columns, one per lane.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include "ptx.cuh"
#include "tp_internal.h"

namespace tp {

struct ColSumArgs {
  const void *in[kMaxParts];
  float *out[kMaxJobs];
  int64_t rows, cols, ld;
  int nin;
};

template <int DT>
__device__ __forceinline__ float col_elem(const void *p, int64_t i) {
  if (DT == TP_F32) return __ldg(static_cast<const float *>(p) + i);
  const uint16_t bits = __ldg(static_cast<const unsigned short *>(p) + i);
  if (DT == TP_BF16) return __uint_as_float((uint32_t)bits << 16);
  return __half2float(__ushort_as_half(bits));
}

template <int DT>
__global__ void __launch_bounds__(256) colsum_kernel(const __grid_constant__ ColSumArgs a) {
  __shared__ float part[8][33];
  const int o = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c = (int64_t)blockIdx.x * 32 + lane;
  float acc = 0.f;
  if (c < a.cols) {
    for (int b = 0; b < a.nin; ++b) {
      const void *p = a.in[o * a.nin + b];
#pragma unroll 4
      for (int64_t t = warp; t < a.rows; t += 8) acc += col_elem<DT>(p, t * a.ld + c);
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && c < a.cols) {
    float s = part[0][lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) s += part[w][lane];
    a.out[o][c] = s;
  }
}

constexpr int kColClu = 8;

template <int DT>
__global__ void __launch_bounds__(256) colsum_cluster_kernel(const __grid_constant__ ColSumArgs a) {
  constexpr int ES = DT == TP_F32 ? 4 : 2;
  constexpr int VEC = 16 / ES;
  constexpr int STRIP = 32 * VEC;
  __shared__ __align__(16) float part[8][STRIP];
  __shared__ __align__(16) float chunk_sum[STRIP];
  const int o = blockIdx.y;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c0 = (int64_t)blockIdx.x * STRIP + lane * VEC;
  const int64_t per = (a.rows + kColClu - 1) / kColClu;
  const int64_t t0 = (int64_t)rank * per, t1 = t0 + per < a.rows ? t0 + per : a.rows;
  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
  const bool full = c0 + VEC <= a.cols;
  for (int b = 0; b < a.nin; ++b) {
    const char *p = static_cast<const char *>(a.in[o * a.nin + b]);
#pragma unroll 8
    for (int64_t t = t0 + warp; t < t1; t += 8) {
      if (full) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(p + (t * a.ld + c0) * ES));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        if (DT == TP_F32) {
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] += __uint_as_float(w[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint16_t lo = (uint16_t)(w[i] & 0xffffu), hi = (uint16_t)(w[i] >> 16);
            acc[2 * i] += DT == TP_BF16 ? __uint_as_float((uint32_t)lo << 16) : __half2float(__ushort_as_half(lo));
            acc[2 * i + 1] += DT == TP_BF16 ? __uint_as_float((uint32_t)hi << 16) : __half2float(__ushort_as_half(hi));
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i)
          if (c0 + i < a.cols) acc[i] += col_elem<DT>(p, t * a.ld + c0 + i);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < VEC; ++i) part[warp][lane * VEC + i] = acc[i];
  __syncthreads();
  for (int c = threadIdx.x; c < STRIP; c += 256) {
    float v = part[0][c];
#pragma unroll
    for (int w = 1; w < 8; ++w) v += part[w][c];
    chunk_sum[c] = v;
  }
  __syncthreads();
  cluster_sync_all();  // every chunk sum is in its CTA's shared memory
  if (rank == 0) {
    const uint32_t base = smem_u32(chunk_sum);
    for (int c4 = threadIdx.x; c4 < STRIP / 4; c4 += 256) {
      float4 v = ld_cluster_f4(mapa_shared(base + c4 * 16, 0));
      for (uint32_t r = 1; r < kColClu; ++r) {
        const float4 u = ld_cluster_f4(mapa_shared(base + c4 * 16, r));
        v.x += u.x;
        v.y += u.y;
        v.z += u.z;
        v.w += u.w;
      }
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t c = (int64_t)blockIdx.x * STRIP + c4 * 4 + i;
        if (c < a.cols) a.out[o][c] = vv[i];
      }
    }
  }
  cluster_sync_all();  // peers keep their shared memory until CTA 0 has read it
}

template <int DT>
static int launch_colsum_cluster(const ColSumArgs &a, int nout, cudaStream_t s) {
  constexpr int STRIP = 32 * (DT == TP_F32 ? 4 : 8);
  const int64_t gx = (a.cols + STRIP - 1) / STRIP;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)gx, (unsigned)nout, kColClu);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = kColClu;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, colsum_cluster_kernel<DT>, a);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "colsum_cluster_kernel launch");
}

int launch_colsum(int nout, int nin, const void *const *in, int64_t rows, int64_t cols, int64_t ld,
                  int in_dt, float *const *out, cudaStream_t s) {
  ColSumArgs a;
  memset(&a, 0, sizeof(a));
  for (int i = 0; i < nout * nin; ++i) a.in[i] = in[i];
  for (int o = 0; o < nout; ++o) a.out[o] = out[o];
  a.rows = rows;
  a.cols = cols;
  a.ld = ld;
  a.nin = nin;
  const int es = in_dt == TP_F32 ? 4 : 2;
  bool vec = ((ld * es) % 16) == 0 && rows > 0;
  for (int i = 0; i < nout * nin; ++i) vec = vec && ((uintptr_t)in[i] % 16) == 0;
  if (vec && cols <= (int64_t)INT32_MAX) {
    if (in_dt == TP_F32) return launch_colsum_cluster<TP_F32>(a, nout, s);
    if (in_dt == TP_BF16) return launch_colsum_cluster<TP_BF16>(a, nout, s);
    return launch_colsum_cluster<TP_F16>(a, nout, s);
  }
  const int64_t gx = (cols + 31) / 32;
  if (gx > INT32_MAX) return set_error(TP_ERR_UNSUPPORTED, "too many columns");
  dim3 grid((unsigned)gx, (unsigned)nout, 1);
  if (in_dt == TP_F32)
    colsum_kernel<TP_F32><<<grid, 256, 0, s>>>(a);
  else if (in_dt == TP_BF16)
    colsum_kernel<TP_BF16><<<grid, 256, 0, s>>>(a);
  else
    colsum_kernel<TP_F16><<<grid, 256, 0, s>>>(a);
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "colsum_kernel launch");
}

}  // namespace tp
