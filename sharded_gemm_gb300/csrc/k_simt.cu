// k_simt.cu -- CUDA-core GEMM for every `Problem` (all layouts and dtypes).
//
// Role: the path for float32 inputs (the MLX worked example), and a slow,
// simple cross-check of the tensor-core kernels (policy TP_POLICY_SIMT).
// 64 x 64 output tile per block, 256 threads, 4 x 4 outputs per thread,
// float32 accumulation with k ascending inside each part; parts either
// continue one accumulator (chain) or are separate partials added in part
// order (row-parallel sum over ranks).  Gated problems carry a second
// accumulator for the up projection and store silu(gate) * up.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "tp_internal.h"

namespace tp {

template <int DT>
__device__ __forceinline__ float load_elem(const void *p, int64_t i) {
  if (DT == TP_F32) return static_cast<const float *>(p)[i];
  const uint16_t bits = static_cast<const uint16_t *>(p)[i];
  if (DT == TP_BF16) return __uint_as_float((uint32_t)bits << 16);
  return __half2float(__ushort_as_half(bits));
}

template <int DT, int BL>
__device__ __forceinline__ float load_b(const Part &pt, int64_t n, int64_t k) {
  if (BL == BL_KMAJOR) return load_elem<DT>(pt.B, n * pt.ldb + k);
  if (BL == BL_MNMAJOR) return load_elem<DT>(pt.B, k * pt.ldb + n);
  if (BL == BL_MX) {  // E4M3 code times the block's power-of-two scale, both exact
    const uint8_t code = static_cast<const uint8_t *>(pt.B)[n * pt.ldb + k];
    const uint32_t sb = static_cast<const uint8_t *>(pt.scales)[n * (pt.K >> 5) + (k >> 5)];
    const float c = __half2float(__half(__nv_cvt_fp8_to_halfraw(code, __NV_E4M3)));
    return c * (sb ? __uint_as_float(sb << 23) : __uint_as_float(0x00400000u));
  }
  // BL_Q4: ldb = words per row; scales / qbias have K/64 entries per row.
  const uint32_t word = static_cast<const uint32_t *>(pt.B)[n * pt.ldb + (k >> 3)];
  const float code = (float)((word >> (4 * (k & 7))) & 15u);
  const int64_t gi = n * (pt.K >> 6) + (k >> 6);
  const float sc = __half2float(__ushort_as_half(static_cast<const uint16_t *>(pt.scales)[gi]));
  const float bq = __half2float(__ushort_as_half(static_cast<const uint16_t *>(pt.qbias)[gi]));
  return fmaf(sc, code, bq);
}

__device__ __forceinline__ void store_out(void *C, int64_t i, float v, int dt) {
  if (dt == TP_F32)
    static_cast<float *>(C)[i] = v;
  else if (dt == TP_BF16)
    static_cast<__nv_bfloat16 *>(C)[i] = __float2bfloat16_rn(v);
  else
    static_cast<__half *>(C)[i] = __float2half_rn(v);
}

template <int DT, int BL, bool GATED>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const __grid_constant__ Problem P) {
  const Job &J = P.jobs[blockIdx.z];
  const int64_t m0 = (int64_t)blockIdx.y * 64, n0 = (int64_t)blockIdx.x * 64;
  if (m0 >= J.M || n0 >= J.N) return;
  __shared__ float As[16][68];
  __shared__ float Bs[16][68];
  __shared__ float Bs2[GATED ? 16 : 1][68];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4], tot[4][4], acc2[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = tot[i][j] = acc2[i][j] = 0.f;

  for (int pi = 0; pi < J.nparts; ++pi) {
    const Part &pt = P.parts[J.part0 + pi];
    if (!P.chain) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    }
    for (int64_t k0 = 0; k0 < pt.K; k0 += 16) {
      for (int e = threadIdx.x; e < 1024; e += 256) {
        const int mm = e >> 4, kk = e & 15;
        const int64_t gm = m0 + mm, gk = k0 + kk;
        As[kk][mm] = (gm < J.M && gk < pt.K)
                         ? load_elem<DT>(pt.A, P.a_mn ? gk * pt.lda + gm : gm * pt.lda + gk)
                         : 0.f;
        const int64_t gn = n0 + mm;
        Bs[kk][mm] = (gn < J.N && gk < pt.K) ? load_b<DT, BL>(pt, gn, gk) : 0.f;
        if constexpr (GATED)
          Bs2[kk][mm] = (gn < J.N && gk < pt.K) ? load_elem<DT>(pt.B2, gn * pt.ldb + gk) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        if constexpr (GATED) {
#pragma unroll
          for (int j = 0; j < 4; ++j) b[j] = Bs2[kk][tx * 4 + j];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc2[i][j] = fmaf(a[i], b[j], acc2[i][j]);
        }
      }
      __syncthreads();
    }
    if (!P.chain) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) tot[i][j] += acc[i][j];
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty * 4 + i;
    if (gm >= J.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gn = n0 + tx * 4 + j;
      if (gn >= J.N) continue;
      float v = P.chain ? acc[i][j] : tot[i][j];
      if (J.bias) v += J.bias[gn];
      if constexpr (GATED) {
        float up = acc2[i][j];
        if (J.bias2) up += J.bias2[gn];
        v = silu_f(v) * up;
      }
      store_out(J.C, gm * J.ldc + gn, v, P.out_dt);
    }
  }
}

int launch_simt(const Problem &p, cudaStream_t s) {
  int64_t maxM = 0, maxN = 0;
  for (int j = 0; j < p.njobs; ++j) {
    if (p.jobs[j].M > maxM) maxM = p.jobs[j].M;
    if (p.jobs[j].N > maxN) maxN = p.jobs[j].N;
  }
  if (maxM == 0 || maxN == 0) return TP_OK;
  const int64_t gx = (maxN + 63) / 64, gy = (maxM + 63) / 64;
  if (gy > 65535) return set_error(TP_ERR_UNSUPPORTED, "M too large for the CUDA-core kernel");
  dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)p.njobs);
  if (p.gated && (p.b_layout != BL_KMAJOR || !p.chain))
    return set_error(TP_ERR_UNSUPPORTED, "gated products need chained K-major weights");
#define TP_SIMT_CASE(DT, BL)                                                      \
  if (p.in_dt == DT && p.b_layout == BL) {                                        \
    if (p.gated)                                                                  \
      simt_gemm_kernel<DT, BL, BL == BL_KMAJOR><<<grid, 256, 0, s>>>(p);          \
    else                                                                          \
      simt_gemm_kernel<DT, BL, false><<<grid, 256, 0, s>>>(p);                    \
    note_launch();                                                                \
    cudaError_t e = cudaGetLastError();                                           \
    return e == cudaSuccess ? TP_OK : cuda_error(e, "simt_gemm_kernel launch");   \
  }
  TP_SIMT_CASE(TP_F32, BL_KMAJOR)
  TP_SIMT_CASE(TP_BF16, BL_KMAJOR)
  TP_SIMT_CASE(TP_F16, BL_KMAJOR)
  TP_SIMT_CASE(TP_F32, BL_MNMAJOR)
  TP_SIMT_CASE(TP_BF16, BL_MNMAJOR)
  TP_SIMT_CASE(TP_F16, BL_MNMAJOR)
  TP_SIMT_CASE(TP_BF16, BL_Q4)
  TP_SIMT_CASE(TP_BF16, BL_MX)
#undef TP_SIMT_CASE
  return set_error(TP_ERR_UNSUPPORTED, "no CUDA-core kernel for dtype %d / layout %d", p.in_dt,
                   p.b_layout);
}

}  // namespace tp
