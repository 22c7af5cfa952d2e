// k_q4.cu -- 4-bit affine (group 64) kernels: a6 device quantizer, and the
// dispatch of the dequant-fused linears (a7).
#include <cuda_fp16.h>

#include "tp_internal.h"

namespace tp {

// a6: one thread per group of 64 consecutive elements of a row.  Every
// floating-point step is a correctly rounded float32 operation (explicit
// _rn intrinsics), so the codes, scales and biases are reproducible
// bit for bit by any IEEE float32 implementation of the same steps.
__global__ void quantize_affine4_kernel(const float *__restrict__ w, int64_t rows, int64_t K,
                                        uint32_t *__restrict__ wq, __half *__restrict__ sc,
                                        __half *__restrict__ qb) {
  const int64_t groups_per_row = K >> 6;
  const int64_t total = rows * groups_per_row;
  for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < total;
       gi += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = gi / groups_per_row, g = gi - row * groups_per_row;
    const float4 *src = reinterpret_cast<const float4 *>(w + row * K + g * 64);
    float v[64];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 f = src[i];
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
    float mn = v[0], mx = v[0];
#pragma unroll
    for (int i = 1; i < 64; ++i) {
      mn = fminf(mn, v[i]);
      mx = fmaxf(mx, v[i]);
    }
    float s = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    if (s == 0.0f) s = 1.0f;
    __half s16 = __float2half_rn(s);
    if (__half2float(s16) == 0.0f) s16 = __float2half_rn(1.0f);
    const __half b16 = __float2half_rn(mn);
    const float sf = __half2float(s16), bf = __half2float(b16);
    uint32_t *out = wq + row * (K >> 3) + g * 8;
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float q = rintf(__fdiv_rn(__fsub_rn(v[wd * 8 + e], bf), sf));
        q = fminf(fmaxf(q, 0.0f), 15.0f);
        word |= ((uint32_t)q) << (4 * e);
      }
      out[wd] = word;
    }
    sc[gi] = s16;
    qb[gi] = b16;
  }
}

int launch_quantize(const float *w, int64_t rows, int64_t K, uint32_t *wq, void *scales,
                    void *qbias, cudaStream_t s) {
  if (((uintptr_t)w & 15) != 0)
    return set_error(TP_ERR_ALIGNMENT, "w must be 16-byte aligned for the quantizer");
  const int64_t total = rows * (K / 64);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (total + 127) / 128;
  if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
  quantize_affine4_kernel<<<(unsigned)blocks, 128, 0, s>>>(w, rows, K, wq, (__half *)scales,
                                                           (__half *)qbias);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "quantize kernel launch");
}

int launch_q4(const Problem &p, cudaStream_t s, bool *handled) {
  (void)p;
  (void)s;
  *handled = false;  // dequant-fused tensor-core kernels not built yet
  return TP_OK;
}

}  // namespace tp
