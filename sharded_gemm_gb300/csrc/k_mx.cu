// k_mx.cu -- MXFP8 weights ("mxfp8" quantization mode of the MLX tensor
// parallelism guide, section 2.3): the device quantizer and the CUDA-core
// decode GEMV of the sharded linears.
//
// Format (OCP microscaling FP8): E4M3 codes, one byte per weight, row-major
// (rows, K); one E8M0 scale byte per 32 consecutive weights of a row, (rows,
// K/32), value 2^(s - 127).  W(o, k) = e4m3(code) * 2^(s - 127); the product
// x (bf16) * e4m3 is exact in float32 and so is the power-of-two scaling.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "tp_internal.h"

namespace tp {

// 2^(s - 127) for an E8M0 scale byte s (0..254): the float32 with exponent
// field s, or the subnormal 2^-127 for s = 0.
__device__ __forceinline__ float e8m0_value(uint32_t s) {
  return s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}

// ------------------------------------------------------------------ quantizer
// One thread per block of 32 consecutive elements of a row:
//   X = floor(log2(max |w|)) - 8 clamped to [-127, 127] (-127 for an all-zero
//   block), scale byte X + 127, code = E4M3(w * 2^-X) rounded to nearest even
//   and saturated to +-448.  w * 2^-X is exact in float32 except where it is
//   below 2^-126, far under E4M3's smallest code, so the codes do not depend
//   on how the product is formed.
__global__ void quantize_mx_kernel(const float *__restrict__ w, int64_t rows, int64_t K,
                                   uint8_t *__restrict__ codes, uint8_t *__restrict__ scales) {
  const int64_t groups = K / 32;
  const int64_t total = rows * groups;
  for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < total;
       gi += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = gi / groups, g = gi - row * groups;
    const float *src = w + row * K + g * 32;
    float amax = 0.f;
#pragma unroll 8
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(src[i]));
    int X = -127;
    if (amax > 0.f) {
      int ex;
      frexpf(amax, &ex);  // amax = f * 2^ex, f in [0.5, 1)
      X = max(-127, min(127, ex - 1 - 8));
    }
    scales[gi] = (uint8_t)(X + 127);
    const float inv = e8m0_value((uint32_t)(127 - X));  // 2^-X, X in [-127, 127]
    uint8_t *dst = codes + row * K + g * 32;
#pragma unroll 8
    for (int i = 0; i < 32; ++i) dst[i] = (uint8_t)__nv_cvt_float_to_fp8(src[i] * inv, __NV_SATFINITE, __NV_E4M3);
  }
}

int launch_mx_quantize(const float *w, int64_t rows, int64_t K, uint8_t *codes, uint8_t *scales,
                       cudaStream_t s) {
  const int64_t total = rows * (K / 32);
  if (total == 0) return TP_OK;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 65535);
  quantize_mx_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, rows, K, codes, scales);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "quantize_mx_kernel launch");
}

// ------------------------------------------------------------------ decode GEMV
// T <= 4 tokens.  The x of every distinct input (one for the column-parallel
// layer, one per rank for the row-parallel one) is staged once per CTA as
// float32 (x[t][k] at xs[xoff + t*K + k]).  A warp task is kRows output rows of
// one job; lane l reads 16 codes (16 bytes) of each row at k = 16*l + 512*i,
// converts them pairwise to f16 (exact) and forms the 16-term dot product
// with x in float32, then adds it times the block's scale.  Each part (rank)
// of a row-parallel job accumulates from zero; the warp sums (fixed butterfly
// order) are added in part order, then the bias.
constexpr int kMxWarps = 16;
constexpr int kMxRows = 4;

struct MxJob {
  void *C;
  const float *bias;
  int64_t ldc;
  int rows, part0, nparts, task0;
};
struct MxPart {
  const uint8_t *codes;
  const uint8_t *scales;
  int64_t K, ldb;
  int xi;  // distinct-input index
};
struct MxArgs {
  MxJob jobs[kMaxJobs];
  MxPart parts[kMaxParts];
  const uint16_t *x[kMaxParts];
  int64_t xK[kMaxParts], xld[kMaxParts], xoff[kMaxParts];
  int njobs, nx, T, ntasks, chain, out_dt, xvec;
};

__device__ __forceinline__ void mx_expand16(const uint4 q, float (&c)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
    const float2 a = __half22float2(__half2(lo));
    const float2 b = __half22float2(__half2(hi));
    c[4 * i] = a.x;
    c[4 * i + 1] = a.y;
    c[4 * i + 2] = b.x;
    c[4 * i + 3] = b.y;
  }
}

template <int TT>
__global__ void __launch_bounds__(kMxWarps * 32, 1) mx_gemv_kernel(const __grid_constant__ MxArgs a) {
  extern __shared__ float xs[];
  // stage every distinct input as float32
  for (int d = 0; d < a.nx; ++d) {
    const int64_t K = a.xK[d], ld = a.xld[d];
    const uint16_t *src = a.x[d];
    float *dst = xs + a.xoff[d];
    if (a.xvec) {  // 16-byte loads of 8 bf16 (rows and bases 16-byte aligned)
      const int64_t K8 = K >> 3;
      for (int64_t i = threadIdx.x; i < (int64_t)TT * K8; i += blockDim.x) {
        const int64_t t = i / K8, k = (i - t * K8) << 3;
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src + t * ld + k));
        float4 *o = reinterpret_cast<float4 *>(dst + t * K + k);
        o[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
        o[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u),
                           __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
      }
    } else {
      for (int64_t i = threadIdx.x; i < (int64_t)TT * K; i += blockDim.x) {
        const int64_t t = i / K, k = i - t * K;
        dst[i] = __uint_as_float((uint32_t)__ldg(src + t * ld + k) << 16);
      }
    }
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int task = blockIdx.x * kMxWarps + warp; task < a.ntasks; task += gridDim.x * kMxWarps) {
    int j = 0;
    while (j + 1 < a.njobs && task >= a.jobs[j + 1].task0) ++j;
    const MxJob &J = a.jobs[j];
    const int row0 = (task - J.task0) * kMxRows;
    float tot[TT][kMxRows];
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
      for (int r = 0; r < kMxRows; ++r) tot[t][r] = 0.f;
    for (int p = 0; p < J.nparts; ++p) {
      const MxPart P = a.parts[J.part0 + p];
      const float *xp = xs + a.xoff[P.xi];
      float acc[TT][kMxRows];
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) acc[t][r] = 0.f;
      const int64_t G = P.K >> 5;
      // The codes and scales of the next 512-code step are loaded before the
      // current step is computed, so one step's loads are always in flight.
      const uint8_t *crow[kMxRows];
      const uint8_t *srow[kMxRows];
#pragma unroll
      for (int r = 0; r < kMxRows; ++r) {
        const int row = row0 + r < J.rows ? row0 + r : J.rows - 1;  // ragged tail: a valid row, result unused
        crow[r] = P.codes + (int64_t)row * P.ldb;
        srow[r] = P.scales + (int64_t)row * G;
      }
      uint4 qn[kMxRows];
      uint32_t sn[kMxRows];
      int64_t k0 = (int64_t)lane * 16;
      if (k0 < P.K) {
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
          qn[r] = __ldcs(reinterpret_cast<const uint4 *>(crow[r] + k0));
          sn[r] = __ldg(srow[r] + (k0 >> 5));
        }
      }
      for (; k0 < P.K; k0 += 512) {
        uint4 q[kMxRows];
        float sc[kMxRows];
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
          q[r] = qn[r];
          sc[r] = e8m0_value(sn[r]);
        }
        if (k0 + 512 < P.K) {
#pragma unroll
          for (int r = 0; r < kMxRows; ++r) {
            qn[r] = __ldcs(reinterpret_cast<const uint4 *>(crow[r] + k0 + 512));
            sn[r] = __ldg(srow[r] + ((k0 + 512) >> 5));
          }
        }
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
          float c[16];
          mx_expand16(q[r], c);  // once per row, shared by the tokens
#pragma unroll
          for (int t = 0; t < TT; ++t) {
            const float4 *xq = reinterpret_cast<const float4 *>(xp + (int64_t)t * P.K + k0);
            float d = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 v = xq[i];
              d = fmaf(v.x, c[4 * i], d);
              d = fmaf(v.y, c[4 * i + 1], d);
              d = fmaf(v.z, c[4 * i + 2], d);
              d = fmaf(v.w, c[4 * i + 3], d);
            }
            acc[t][r] = fmaf(d, sc[r], acc[t][r]);
          }
        }
      }
      // warp sums of this part, added to the total in part order
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
          float v = acc[t][r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          tot[t][r] = (p == 0) ? v : tot[t][r] + v;
        }
    }
    if (lane < TT * kMxRows) {
      const int t = lane / kMxRows, r = lane % kMxRows;
      const int row = row0 + r;
      float v = 0.f;
#pragma unroll
      for (int tt = 0; tt < TT; ++tt)
#pragma unroll
        for (int rr = 0; rr < kMxRows; ++rr)
          if (tt == t && rr == r) v = tot[tt][rr];
      if (t < TT && row < J.rows) {
        if (J.bias) v += J.bias[row];
        const int64_t idx = (int64_t)t * J.ldc + row;
        if (a.out_dt == TP_F32)
          static_cast<float *>(J.C)[idx] = v;
        else if (a.out_dt == TP_BF16)
          static_cast<__nv_bfloat16 *>(J.C)[idx] = __float2bfloat16_rn(v);
        else
          static_cast<__half *>(J.C)[idx] = __float2half_rn(v);
      }
    }
  }
}

int launch_mx(const Problem &p, cudaStream_t s, bool *handled) {
  *handled = false;
  if (p.in_dt != TP_BF16) return TP_OK;
  int64_t maxT = 0;
  for (int j = 0; j < p.njobs; ++j) maxT = std::max<int64_t>(maxT, p.jobs[j].M);
  if (maxT < 1 || maxT > 4) return TP_OK;
  static MxArgs args;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  memset(&args, 0, sizeof(args));
  int64_t floats = 0;
  int ntasks = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    if (J.M != maxT || J.N > INT32_MAX) return TP_OK;
    args.jobs[j] = MxJob{J.C, J.bias, J.ldc, (int)J.N, J.part0, J.nparts, ntasks};
    ntasks += (int)((J.N + kMxRows - 1) / kMxRows);
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      if (((uintptr_t)P.B & 15) || (P.ldb % 16) || (P.K % 32)) return TP_OK;
      int xi = -1;
      for (int d = 0; d < args.nx; ++d)
        if ((const void *)args.x[d] == P.A && args.xK[d] == P.K && args.xld[d] == P.lda) xi = d;
      if (xi < 0) {
        if (args.nx == kMaxParts) return TP_OK;
        xi = args.nx++;
        args.x[xi] = static_cast<const uint16_t *>(P.A);
        args.xK[xi] = P.K;
        args.xld[xi] = P.lda;
        args.xoff[xi] = floats;
        floats += maxT * P.K;
      }
      args.parts[J.part0 + q] = MxPart{static_cast<const uint8_t *>(P.B), static_cast<const uint8_t *>(P.scales),
                                       P.K, P.ldb, xi};
    }
  }
  const size_t smem = (size_t)floats * 4;
  if (smem > 200 * 1024) return TP_OK;  // inputs too large to stage: the CUDA-core GEMM takes it
  args.njobs = p.njobs;
  args.T = (int)maxT;
  args.xvec = 1;
  for (int d = 0; d < args.nx; ++d)
    if (((uintptr_t)args.x[d] & 15) || (args.xld[d] % 8) || (args.xK[d] % 8)) args.xvec = 0;
  args.ntasks = ntasks;
  args.chain = p.chain;
  args.out_dt = p.out_dt;
  const int grid = std::min(sm_count(), (ntasks + kMxWarps - 1) / kMxWarps);
  cudaError_t e = cudaSuccess;
#define TP_MX_CASE(TTV)                                                                                   \
  if (maxT == TTV) {                                                                                      \
    e = cudaFuncSetAttribute(mx_gemv_kernel<TTV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    if (e == cudaSuccess) mx_gemv_kernel<TTV><<<grid, kMxWarps * 32, smem, s>>>(args);                   \
  }
  TP_MX_CASE(1)
  TP_MX_CASE(2)
  TP_MX_CASE(3)
  TP_MX_CASE(4)
#undef TP_MX_CASE
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "mx_gemv_kernel launch");
  *handled = true;
  return TP_OK;
}

}  // namespace tp
