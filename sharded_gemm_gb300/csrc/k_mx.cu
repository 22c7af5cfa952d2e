// k_mx.cu -- MXFP8 weights ("mxfp8" quantization mode of the MLX tensor
// parallelism guide, section 2.3): the device quantizer, the CUDA-core
// decode GEMV (T <= 4) and the tensor-core kernel (T > 4) of the sharded
// linears.
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

#include "ptx.cuh"
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
  note_launch();
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
  griddep_launch_dependents();
  griddep_wait();  // programmatic launch: no global memory before the previous kernel completes
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
      // The codes and scales of the next PD 512-code steps are loaded before
      // the current step is computed (PD = 2 for one or two tokens), so PD
      // steps' loads are always in flight.
      constexpr int PD = TT <= 2 ? 2 : 1;
      const uint8_t *crow[kMxRows];
      const uint8_t *srow[kMxRows];
#pragma unroll
      for (int r = 0; r < kMxRows; ++r) {
        const int row = row0 + r < J.rows ? row0 + r : J.rows - 1;  // ragged tail: a valid row, result unused
        crow[r] = P.codes + (int64_t)row * P.ldb;
        srow[r] = P.scales + (int64_t)row * G;
      }
      uint4 qn[PD][kMxRows];
      uint32_t sn[PD][kMxRows];
      int64_t k0 = (int64_t)lane * 16;
#pragma unroll
      for (int d = 0; d < PD; ++d) {
        const int64_t k = k0 + 512 * d;
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
          qn[d][r] = k < P.K ? __ldcs(reinterpret_cast<const uint4 *>(crow[r] + k)) : make_uint4(0u, 0u, 0u, 0u);
          sn[d][r] = k < P.K ? (uint32_t)__ldg(srow[r] + (k >> 5)) : 0u;
        }
      }
      for (; k0 < P.K; k0 += 512) {
        uint4 q[kMxRows];
        float sc[kMxRows];
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
          q[r] = qn[0][r];
          sc[r] = e8m0_value(sn[0][r]);
        }
#pragma unroll
        for (int d = 0; d + 1 < PD; ++d)
#pragma unroll
          for (int r = 0; r < kMxRows; ++r) {
            qn[d][r] = qn[d + 1][r];
            sn[d][r] = sn[d + 1][r];
          }
        const int64_t kn = k0 + 512 * PD;
        if (kn < P.K) {
#pragma unroll
          for (int r = 0; r < kMxRows; ++r) {
            qn[PD - 1][r] = __ldcs(reinterpret_cast<const uint4 *>(crow[r] + kn));
            sn[PD - 1][r] = __ldg(srow[r] + (kn >> 5));
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

static int launch_mx_gemv(const Problem &p, cudaStream_t s, bool *handled) {
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
    if (e == cudaSuccess) e = launch_pdl(mx_gemv_kernel<TTV>, dim3(grid), dim3(kMxWarps * 32), smem, s, args); \
  }
  TP_MX_CASE(1)
  TP_MX_CASE(2)
  TP_MX_CASE(3)
  TP_MX_CASE(4)
#undef TP_MX_CASE
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "mx_gemv_kernel launch");
  *handled = true;
  return TP_OK;
}

// ------------------------------------------------------------------ tensor cores
// T > 4 tokens (and any shape the GEMV does not take).  Swap-AB tiles: 128
// weight rows fill M, BN tokens fill N.  Per 64-element k-block, TMA brings the
// 128 x 64 code bytes (64-byte swizzle) and the BN x 64 x tile (bf16, 128-byte
// swizzle); 8 converter warps turn the codes into the exact bf16 values
// e4m3 * 2^(s-127) (one row and one 32-element block per thread) and write
// them as the MMA's A operand (K-major, 128-byte swizzle) into the same stage;
// one thread issues tcgen05.mma kind::f16 (bf16 x bf16, float32 in TMEM).
// A unit is (job, 128-row tile, token tile, split); a split is a run of
// k-blocks of one part (rank); the float32 partials of split tiles go to
// workspace slots (column-major, so a warp's 32 rows of one column are one
// 128-byte line) and a second launch adds each tile's slots in split (rank)
// order, then the bias.
namespace {

constexpr int kMtThreads = 14 * 32;  // producer, MMA, 8 converter warps, 4 epilogue warps

struct MtPart {
  const uint8_t *sc;  // scales (rows, G)
  int G;              // K / 32
  int kblocks;        // ceil(K / 64)
  int16_t cmap, xmap;
  int nchunk, chunk_kb;
};
struct MtJob {
  void *C;
  const float *bias;
  int64_t ldc;
  int rows, T;
  int part0, nparts;
  int tiles, ntiles, splits;
  int unit_begin;
  int64_t ws_base;
};
struct MtArgs {
  CUtensorMap cmaps[kMaxParts];
  CUtensorMap xmaps[kMaxParts];
  MtJob jobs[kMaxJobs];
  MtPart parts[kMaxParts];
  int njobs, total_units, out_dt;
  uint32_t idesc;
  float *ws;
  int *status;
  uint64_t wait_ns;
};

struct MtUnit {
  int job, part, tile, ntile, tile_lin, sidx, kb0, kb1;
};

__device__ __forceinline__ void mt_unit(const MtArgs &a, int u, MtUnit &ui) {
  int j = 0;
  while (j + 1 < a.njobs && u >= a.jobs[j + 1].unit_begin) ++j;
  const MtJob &J = a.jobs[j];
  const int local = u - J.unit_begin;
  ui.job = j;
  ui.tile_lin = local / J.splits;
  ui.sidx = local - ui.tile_lin * J.splits;
  ui.tile = ui.tile_lin % J.tiles;
  ui.ntile = ui.tile_lin / J.tiles;
  int p = 0, c = ui.sidx;
  while (p + 1 < J.nparts && c >= a.parts[J.part0 + p].nchunk) {
    c -= a.parts[J.part0 + p].nchunk;
    ++p;
  }
  const MtPart &P = a.parts[J.part0 + p];
  ui.part = J.part0 + p;
  ui.kb0 = c * P.chunk_kb;
  ui.kb1 = min(P.kblocks, ui.kb0 + P.chunk_kb);
}

// Eight E4M3 codes (two 32-bit words) times 2^(s-127) -> eight bf16 (one
// 16-byte chunk, natural order).  The conversions to f16 and float32 are
// exact, so is the power-of-two product, and the values (4 significant bits)
// are exact in bf16.
__device__ __forceinline__ uint32_t mx_pair_bf16(uint32_t pair, float scale) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)pair, __NV_E4M3);
  const float2 f = __half22float2(__half2(h));
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(f.y * scale), "f"(f.x * scale));
  return d;
}
__device__ __forceinline__ uint4 mx_chunk_bf16(uint32_t w0, uint32_t w1, float scale) {
  return make_uint4(mx_pair_bf16(w0 & 0xffffu, scale), mx_pair_bf16(w0 >> 16, scale),
                    mx_pair_bf16(w1 & 0xffffu, scale), mx_pair_bf16(w1 >> 16, scale));
}

// The two scale bytes of k-block kb (blocks 2kb, 2kb+1) of a row; a block
// past the row's end reads as 0.
__device__ __forceinline__ uint32_t mt_scale_pair(const uint8_t *row, int kb, int G) {
  const int b = 2 * kb;
  if (b + 1 < G && ((uintptr_t)(row + b) & 1) == 0) return __ldg(reinterpret_cast<const uint16_t *>(row + b));
  uint32_t v = __ldg(row + b);
  if (b + 1 < G) v |= (uint32_t)__ldg(row + b + 1) << 8;
  return v;
}

// y[t][orow] of an output whose pointer and row stride the caller holds in
// registers (read through the kernel-parameter block, they would be reloaded
// after every store: the compiler cannot tell the output from the parameters).
__device__ __forceinline__ void mt_store(int out_dt, void *C, int64_t ldc, int t, int orow, float v) {
  const int64_t idx = (int64_t)t * ldc + orow;
  if (out_dt == TP_F32)
    static_cast<float *>(C)[idx] = v;
  else if (out_dt == TP_BF16)
    static_cast<__nv_bfloat16 *>(C)[idx] = __float2bfloat16_rn(v);
  else
    static_cast<__half *>(C)[idx] = __float2half_rn(v);
}

#define MT_WAIT_ALL(bar, par, okvar)                                   \
  {                                                                    \
    const bool _r = mbar_wait((bar), (par), lim, a.status, &abort_sh); \
    if (!__all_sync(0xffffffffu, _r)) okvar = false;                   \
  }

__device__ __forceinline__ uint4 mt_lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void mt_sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <int BN>
struct MtCfg {
  static constexpr int A_BYTES = 128 * 128;  // 128 rows x 64 bf16
  static constexpr int X_BYTES = BN * 128;   // BN tokens x 64 bf16
  static constexpr int C_BYTES = 128 * 64;   // 128 rows x 64 codes
  static constexpr int STAGE = A_BYTES + X_BYTES + C_BYTES;
  static constexpr int ND = (512 / BN) < 4 ? (512 / BN) : 4;  // accumulator slots
  static constexpr int COLS = ND * BN <= 32 ? 32 : ND * BN <= 64 ? 64 : ND * BN <= 128 ? 128 : ND * BN <= 256 ? 256 : 512;
  static constexpr int CHK = BN >= 32 ? 32 : 16;
};

// Epilogue role (4 warps): per unit, the 128 x BN float32 tile from TMEM slot
// ds to the output (token t, row) with the bias, or to the unit's split slot.
template <int BN, int ND>
__device__ __forceinline__ void mt_epilogue(const MtArgs &a, uint32_t tmem, uint64_t *dfull_bar,
                                            uint64_t *dempty_bar, int &abort_sh, int warp, int lane) {
  using C = MtCfg<BN>;
  const uint64_t lim = a.wait_ns;
  const int q = warp & 3;
  const int m = q * 32 + lane;
  const uint32_t lane_off = (uint32_t)(q * 32) << 16;
  int ds = 0;
  uint32_t dph = 0;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
    MtUnit ui;
    mt_unit(a, u, ui);
    const MtJob &J = a.jobs[ui.job];
    const int orow = ui.tile * 128 + m;
    const bool valid = orow < J.rows;
    MT_WAIT_ALL(smem_u32(&dfull_bar[ds]), dph, ok);
    if (!ok) break;
    tc_fence_after();
    const float bias = (valid && J.bias) ? __ldg(J.bias + orow) : 0.f;
    const int t0 = ui.ntile * BN;
    const bool split = J.splits > 1;
    void *const oC = J.C;
    const int64_t oldc = J.ldc;
    const int oT = J.T, odt = a.out_dt;
    float *slot = split ? a.ws + (J.ws_base + (int64_t)ui.tile_lin * J.splits + ui.sidx) * 128 * BN + m : nullptr;
#pragma unroll 1
    for (int c = 0; c < BN / C::CHK; ++c) {
      float v[C::CHK];
      if constexpr (C::CHK == 32)
        tmem_ld32(tmem + lane_off + ds * BN + c * 32, v);
      else
        tmem_ld16(tmem + lane_off + ds * BN + c * 16, v);
      tmem_wait_ld();
      if (split) {
#pragma unroll
        for (int i = 0; i < C::CHK; ++i) __stcg(slot + (c * C::CHK + i) * 128, v[i]);
      } else if (valid) {
#pragma unroll
        for (int i = 0; i < C::CHK; ++i) {
          const int t = t0 + c * C::CHK + i;
          if (t < oT) mt_store(odt, oC, oldc, t, orow, v[i] + bias);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&dempty_bar[ds]));
    if (++ds == ND) {
      ds = 0;
      dph ^= 1;
    }
  }
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kMtThreads, 1) mx_umma_kernel(const __grid_constant__ MtArgs a) {
  griddep_launch_dependents();
  griddep_wait();  // programmatic launch: no global memory before the previous kernel completes
  using C = MtCfg<BN>;
  static_assert(STAGES == 1 || STAGES == 2 || STAGES == 4 || STAGES == 8, "8 converter warps share the slots");
  static_assert(C::STAGE % 1024 == 0, "stage alignment");
  constexpr int ND = C::ND;

  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], afull_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t dfull_bar[ND], dempty_bar[ND];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&afull_bar[i]), 8 / STAGES);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < ND; ++i) {
      mbar_init(smem_u32(&dfull_bar[i]), 1);
      mbar_init(smem_u32(&dempty_bar[i]), 4);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_sh), C::COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      bool used[STAGES];
      uint32_t lastph[STAGES];
#pragma unroll
      for (int i = 0; i < STAGES; ++i) used[i] = false;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        MtUnit ui;
        mt_unit(a, u, ui);
        const MtPart &P = a.parts[ui.part];
        for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
          if (!mbar_wait(smem_u32(&empty_bar[st]), ph ^ 1, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          const uint32_t base = sbase + st * C::STAGE;
          const uint32_t fb = smem_u32(&full_bar[st]);
          mbar_arrive_expect_tx(fb, C::X_BYTES + C::C_BYTES);
          tma_load_2d(base + C::A_BYTES, &a.xmaps[P.xmap], fb, kb * 64, ui.ntile * BN);
          // the weights are read once: evicted first, so x and the split partials stay in L2
          tma_load_2d_hint(base + C::A_BYTES + C::X_BYTES, &a.cmaps[P.cmap], fb, kb * 64, ui.tile * 128,
                           l2_policy_evict_first());
          used[st] = true;
          lastph[st] = ph;
          if (++st == STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok)
        for (int i = 0; i < STAGES; ++i)
          if (used[i]) mbar_wait(smem_u32(&full_bar[i]), lastph[i], lim, a.status, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int st = 0, ds = 0;
      uint32_t ph = 0, dph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        MtUnit ui;
        mt_unit(a, u, ui);
        bool first = true;
        for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
          // the x tile has landed and the converters have written A
          if (!mbar_wait(smem_u32(&full_bar[st]), ph, lim, a.status, &abort_sh) ||
              !mbar_wait(smem_u32(&afull_bar[st]), ph, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          if (first && !mbar_wait(smem_u32(&dempty_bar[ds]), dph ^ 1, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t base = sbase + st * C::STAGE;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16(tmem + ds * BN, umma_desc_sw128(base + kk * 32, 16, 1024),
                     umma_desc_sw128(base + C::A_BYTES + kk * 32, 16, 1024), a.idesc,
                     (first && kk == 0) ? 0u : 1u);
          umma_commit(smem_u32(&empty_bar[st]));
          if (++st == STAGES) {
            st = 0;
            ph ^= 1;
          }
          first = false;
        }
        if (!ok) break;
        umma_commit(smem_u32(&dfull_bar[ds]));
        if (++ds == ND) {
          ds = 0;
          dph ^= 1;
        }
      }
      umma_commit(smem_u32(&drain_bar));
      mbar_wait(smem_u32(&drain_bar), 0, lim, a.status, nullptr);
    }
  } else if (warp < 10) {
    // ---------------------------------------------------------- converters
    // Converter warp cw owns ring slots s with s % STAGES == cw % STAGES; the
    // 8 / STAGES warps of a slot split its 128 rows (lane l takes rows
    // r0 + l + 32 i).  Each converts whole stages, so up to 8 stages are in
    // conversion at once.  A row's two scale bytes of a k-block are loaded one
    // round of the ring ahead.
    constexpr int WPS = 8 / STAGES;          // warps per slot
    constexpr int RPL = 128 / (32 * WPS);    // rows per lane
    const int cw = warp - 2;
    const int myslot = cw % STAGES;
    const int rbase = (cw / STAGES) * (128 / WPS);
    int n = 0;  // stage sequence number over all units of this CTA
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
      MtUnit ui;
      mt_unit(a, u, ui);
      const MtPart &P = a.parts[ui.part];
      const MtJob &J = a.jobs[ui.job];
      // first k-block of this unit that is this warp's
      int kb = ui.kb0 + ((myslot - n % STAGES) + STAGES) % STAGES;
      n += ui.kb1 - ui.kb0;
      uint32_t snext[RPL];
      const uint8_t *srow[RPL];
      bool rv[RPL];
#pragma unroll
      for (int i = 0; i < RPL; ++i) {
        const int orow = ui.tile * 128 + rbase + lane + 32 * i;
        rv[i] = orow < J.rows;
        srow[i] = P.sc + (int64_t)(rv[i] ? orow : 0) * P.G;
        snext[i] = (rv[i] && kb < ui.kb1) ? mt_scale_pair(srow[i], kb, P.G) : 0u;
      }
      for (; ok && kb < ui.kb1; kb += STAGES) {
        const int seq = n - (ui.kb1 - ui.kb0) + (kb - ui.kb0);  // stage sequence number of kb
        const uint32_t ph = (uint32_t)((seq / STAGES) & 1);
        uint32_t scur[RPL];
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
          scur[i] = snext[i];
          const int kn = kb + STAGES;
          snext[i] = (rv[i] && kn < ui.kb1) ? mt_scale_pair(srow[i], kn, P.G) : 0u;
        }
        MT_WAIT_ALL(smem_u32(&full_bar[myslot]), ph, ok);
        if (!ok) break;
        const uint32_t base = sbase + myslot * C::STAGE;
        // all of the stage's code loads first (plain shared-memory reads, so
        // they are issued together), then the conversions and A stores
        uint8_t *gbase = dsmem + (base - smem_u32(dsmem));
        uint4 cv[RPL][4];
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
          const int r = rbase + lane + 32 * i;
          const uint8_t *crow = gbase + C::A_BYTES + C::X_BYTES + r * 64;  // 64-byte swizzled code row
#pragma unroll
          for (int c = 0; c < 4; ++c) cv[i][c] = *reinterpret_cast<const uint4 *>(crow + ((c ^ ((r >> 1) & 3)) << 4));
        }
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
          const int r = rbase + lane + 32 * i;
          const float s0 = rv[i] ? e8m0_value(scur[i] & 0xffu) : 0.f;
          const float s1 = (rv[i] && 2 * kb + 1 < P.G) ? e8m0_value(scur[i] >> 8) : 0.f;
          uint4 *arow = reinterpret_cast<uint4 *>(gbase + r * 128);  // 128-byte swizzled A row
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float sc = c < 2 ? s0 : s1;
            arow[(2 * c) ^ (r & 7)] = mx_chunk_bf16(cv[i][c].x, cv[i][c].y, sc);
            arow[(2 * c + 1) ^ (r & 7)] = mx_chunk_bf16(cv[i][c].z, cv[i][c].w, sc);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&afull_bar[myslot]));
      }
    }
  } else {
    mt_epilogue<BN, ND>(a, tmem, dfull_bar, dempty_bar, abort_sh, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::COLS);
  }
}

// Decode form (BN <= 32).  The TMA ring holds only a stage's x tile and
// codes (10-12 KB, so about 15 stages of codes are in flight); stage n is
// converted by converter group n % 2 (4 warps, 32 rows each) into A buffer
// n % NA (bf16 weights + a copy of the x tile), and its ring slot is released
// as soon as it has been read.  The MMA reads only the A buffer.
template <int BN, int STAGES, int NA>
__global__ void __launch_bounds__(kMtThreads, 1) mx_dec_kernel(const __grid_constant__ MtArgs a) {
  griddep_launch_dependents();
  griddep_wait();  // programmatic launch: no global memory before the previous kernel completes
  using C = MtCfg<BN>;
  constexpr int X_BYTES = BN * 128;
  constexpr int C_BYTES = 128 * 64;
  constexpr int RING = X_BYTES + C_BYTES;  // x (128-byte swizzle) then codes (64-byte swizzle)
  constexpr int A_BYTES = 128 * 128;
  constexpr int ABUF = A_BYTES + X_BYTES;  // bf16 weights then the x copy
  constexpr int ND = C::ND;
  static_assert(RING % 1024 == 0 && ABUF % 1024 == 0, "alignment");

  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t afull_bar[NA], aempty_bar[NA];
  __shared__ __align__(8) uint64_t dfull_bar[ND], dempty_bar[ND];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t abase = sbase + STAGES * RING;
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 4);
    }
    for (int i = 0; i < NA; ++i) {
      mbar_init(smem_u32(&afull_bar[i]), 4);
      mbar_init(smem_u32(&aempty_bar[i]), 1);
    }
    for (int i = 0; i < ND; ++i) {
      mbar_init(smem_u32(&dfull_bar[i]), 1);
      mbar_init(smem_u32(&dempty_bar[i]), 4);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_sh), C::COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      bool used[STAGES];
      uint32_t lastph[STAGES];
#pragma unroll
      for (int i = 0; i < STAGES; ++i) used[i] = false;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        MtUnit ui;
        mt_unit(a, u, ui);
        const MtPart &P = a.parts[ui.part];
        for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
          if (!mbar_wait(smem_u32(&empty_bar[st]), ph ^ 1, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          const uint32_t base = sbase + st * RING;
          const uint32_t fb = smem_u32(&full_bar[st]);
          mbar_arrive_expect_tx(fb, RING);
          tma_load_2d(base, &a.xmaps[P.xmap], fb, kb * 64, ui.ntile * BN);
          tma_load_2d(base + X_BYTES, &a.cmaps[P.cmap], fb, kb * 64, ui.tile * 128);
          used[st] = true;
          lastph[st] = ph;
          if (++st == STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok)
        for (int i = 0; i < STAGES; ++i)
          if (used[i]) mbar_wait(smem_u32(&full_bar[i]), lastph[i], lim, a.status, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int n = 0, ds = 0;
      uint32_t dph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        MtUnit ui;
        mt_unit(a, u, ui);
        bool first = true;
        for (int kb = ui.kb0; kb < ui.kb1; ++kb, ++n) {
          const int ab = n % NA;
          if (!mbar_wait(smem_u32(&afull_bar[ab]), (uint32_t)((n / NA) & 1), lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          if (first && !mbar_wait(smem_u32(&dempty_bar[ds]), dph ^ 1, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ba = abase + ab * ABUF;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16(tmem + ds * BN, umma_desc_sw128(ba + kk * 32, 16, 1024),
                     umma_desc_sw128(ba + A_BYTES + kk * 32, 16, 1024), a.idesc, (first && kk == 0) ? 0u : 1u);
          umma_commit(smem_u32(&aempty_bar[ab]));
          first = false;
        }
        if (!ok) break;
        umma_commit(smem_u32(&dfull_bar[ds]));
        if (++ds == ND) {
          ds = 0;
          dph ^= 1;
        }
      }
      umma_commit(smem_u32(&drain_bar));
      mbar_wait(smem_u32(&drain_bar), 0, lim, a.status, nullptr);
    }
  } else if (warp < 10) {
    // ---------------------------------------------------------- converters
    const int g = (warp - 2) >> 2, q = (warp - 2) & 3;
    const int r = q * 32 + lane;  // weight row of the tile
    const int tg = q * 32 + lane; // thread index in the group (x copy)
    int n = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
      MtUnit ui;
      mt_unit(a, u, ui);
      const MtPart &P = a.parts[ui.part];
      const MtJob &J = a.jobs[ui.job];
      const int n0 = n;
      n += ui.kb1 - ui.kb0;
      const int orow = ui.tile * 128 + r;
      const bool rv = orow < J.rows;
      const uint8_t *srow = P.sc + (int64_t)(rv ? orow : 0) * P.G;
      int kb = ui.kb0 + (((g - n0) % 2) + 2) % 2;  // this group's first k-block of the unit
      uint32_t snext = (rv && kb < ui.kb1) ? mt_scale_pair(srow, kb, P.G) : 0u;
      for (; ok && kb < ui.kb1; kb += 2) {
        const int seq = n0 + (kb - ui.kb0);
        const int cs = seq % STAGES, ab = seq % NA;
        const uint32_t scur = snext;
        snext = (rv && kb + 2 < ui.kb1) ? mt_scale_pair(srow, kb + 2, P.G) : 0u;
        MT_WAIT_ALL(smem_u32(&full_bar[cs]), (uint32_t)((seq / STAGES) & 1), ok);
        if (!ok) break;
        MT_WAIT_ALL(smem_u32(&aempty_bar[ab]), (uint32_t)(((seq / NA) & 1) ^ 1), ok);
        if (!ok) break;
        uint8_t *ring = dsmem + (sbase + cs * RING - smem_u32(dsmem));
        uint8_t *abuf = dsmem + (abase + ab * ABUF - smem_u32(dsmem));
        uint4 cv[4];
        const uint8_t *crow = ring + X_BYTES + r * 64;  // 64-byte swizzled code row
#pragma unroll
        for (int c = 0; c < 4; ++c) cv[c] = *reinterpret_cast<const uint4 *>(crow + ((c ^ ((r >> 1) & 3)) << 4));
        uint4 xv[X_BYTES / 16 / 128];
#pragma unroll
        for (int i = 0; i < X_BYTES / 16 / 128; ++i) xv[i] = reinterpret_cast<const uint4 *>(ring)[tg + 128 * i];
        const float s0 = rv ? e8m0_value(scur & 0xffu) : 0.f;
        const float s1 = (rv && 2 * kb + 1 < P.G) ? e8m0_value(scur >> 8) : 0.f;
        uint4 *arow = reinterpret_cast<uint4 *>(abuf + r * 128);  // 128-byte swizzled A row
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float sc = c < 2 ? s0 : s1;
          arow[(2 * c) ^ (r & 7)] = mx_chunk_bf16(cv[c].x, cv[c].y, sc);
          arow[(2 * c + 1) ^ (r & 7)] = mx_chunk_bf16(cv[c].z, cv[c].w, sc);
        }
#pragma unroll
        for (int i = 0; i < X_BYTES / 16 / 128; ++i) reinterpret_cast<uint4 *>(abuf + A_BYTES)[tg + 128 * i] = xv[i];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&empty_bar[cs]));  // the ring slot has been read
          mbar_arrive(smem_u32(&afull_bar[ab]));
        }
      }
    }
  } else {
    mt_epilogue<BN, ND>(a, tmem, dfull_bar, dempty_bar, abort_sh, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::COLS);
  }
}

}  // namespace

namespace {

std::mutex g_mt_mu;

template <int BN, int STAGES, int NA>
int mt_dec_launch(MtArgs &args, int sms, cudaStream_t s) {
  auto kern = mx_dec_kernel<BN, STAGES, NA>;
  constexpr int smem = STAGES * (BN * 128 + 128 * 64) + NA * (128 * 128 + BN * 128) + 1024;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(mx decode)");
    attr_done[dev & 63] = true;
  }
  const int grid = args.total_units < sms ? args.total_units : sms;
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kMtThreads), smem, s, args);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "mx_dec_kernel launch");
}

template <int BN, int STAGES>
int mt_launch(MtArgs &args, int sms, cudaStream_t s) {
  auto kern = mx_umma_kernel<BN, STAGES>;
  constexpr int smem = STAGES * MtCfg<BN>::STAGE + 1024;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(mx)");
    attr_done[dev & 63] = true;
  }
  const int grid = args.total_units < sms ? args.total_units : sms;
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kMtThreads), smem, s, args);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "mx_umma_kernel launch");
}

// Tensor-core launch of `p` (bf16 x, 16-byte aligned codes and x rows).
int launch_mx_tc(const Problem &p, cudaStream_t s, bool *handled) {
  *handled = false;
  int64_t maxT = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    if (J.M > maxT) maxT = J.M;
    if (J.N > INT32_MAX / 2 || J.M > INT32_MAX / 2) return TP_OK;
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      if (((uintptr_t)P.A & 15) || (P.lda % 8) || ((uintptr_t)P.B & 15) || (P.ldb % 16) || (P.K % 32)) return TP_OK;
    }
  }
  const int BN = maxT <= 16 ? 16 : maxT <= 32 ? 32 : maxT <= 64 ? 64 : maxT <= 128 ? 128 : 256;
  std::lock_guard<std::mutex> lk(g_mt_mu);
  const int sms = sm_count();
  static MtArgs args;
  memset(&args, 0, sizeof(args));
  // k-block chunks per part: the same count for every part, chosen to fill
  // the SMs with the fewest k-blocks per unit, plus, for split tiles, the
  // ordered split sum that reads every float32 partial back (measured about
  // 4.3 TB/s) and, where the partials outgrow what L2 keeps beside the
  // streamed weights (about 48 MB), their write to DRAM and read back.
  // Costs in k-block times (about 0.64 us at 256 tokens).
  int64_t tiles_parts = 0;
  int kb_max = 0, parts_max = 1;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    tiles_parts += ((J.N + 127) / 128) * ((J.M + BN - 1) / BN) * J.nparts;
    parts_max = std::max(parts_max, J.nparts);
    for (int q = 0; q < J.nparts; ++q) kb_max = std::max(kb_max, (int)((p.parts[J.part0 + q].K + 63) / 64));
  }
  int chunks = 1;
  double best = 1e300;
  for (int c = 1; c <= 16 && c <= kb_max; ++c) {
    const int ck = (kb_max + c - 1) / c;
    const int64_t units = tiles_parts * ((kb_max + ck - 1) / ck);
    const bool split = c > 1 || parts_max > 1;
    const double slot_mb = split ? (double)units * 128.0 * BN * 4.0 / 1e6 : 0.0;
    const double kb_us = 0.64;
    const double cost = (double)((units + sms - 1) / sms) * (ck + 4.0) +
                        (split ? 2.0 + slot_mb / 4.3 / kb_us + (slot_mb > 48.0 ? 2.0 * slot_mb / 6.8 / kb_us : 0.0)
                               : 0.0);
    if (cost < best - 1e-9) {
      best = cost;
      chunks = c;
    }
  }
  const void *cptr[kMaxParts], *xptr[kMaxParts];
  int ncm = 0, nxm = 0;
  int64_t units = 0, slots = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    MtJob &Q = args.jobs[j];
    Q.C = J.C;
    Q.bias = J.bias;
    Q.ldc = J.ldc;
    Q.rows = (int)J.N;
    Q.T = (int)J.M;
    Q.part0 = J.part0;
    Q.nparts = J.nparts;
    Q.tiles = (Q.rows + 127) / 128;
    Q.ntiles = (Q.T + BN - 1) / BN;
    int splits = 0;
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      MtPart &QP = args.parts[J.part0 + q];
      QP.sc = static_cast<const uint8_t *>(P.scales);
      QP.G = (int)(P.K / 32);
      QP.kblocks = (int)((P.K + 63) / 64);
      QP.chunk_kb = (QP.kblocks + chunks - 1) / chunks;
      QP.nchunk = (QP.kblocks + QP.chunk_kb - 1) / QP.chunk_kb;
      splits += QP.nchunk;
      int ic = -1, ix = -1;
      for (int i = 0; i < ncm; ++i)
        if (cptr[i] == P.B) ic = i;
      for (int i = 0; i < nxm; ++i)
        if (xptr[i] == P.A) ix = i;
      int rc;
      if (ic < 0) {
        rc = make_tmap_2d(&args.cmaps[ncm], P.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)P.K, (uint64_t)Q.rows,
                          (uint64_t)P.ldb, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B);
        if (rc) return rc;
        cptr[ncm] = P.B;
        ic = ncm++;
      }
      if (ix < 0) {
        rc = make_tmap_2d(&args.xmaps[nxm], P.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)P.K, (uint64_t)Q.T,
                          (uint64_t)P.lda, 64, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc) return rc;
        xptr[nxm] = P.A;
        ix = nxm++;
      }
      QP.cmap = (int16_t)ic;
      QP.xmap = (int16_t)ix;
    }
    Q.splits = splits;
    Q.unit_begin = (int)units;
    Q.ws_base = slots;
    const int64_t tl = (int64_t)Q.tiles * Q.ntiles;
    units += tl * splits;
    if (splits > 1) slots += tl * splits;
  }
  if (units == 0) {
    *handled = true;
    return TP_OK;
  }
  if (units > INT32_MAX) return TP_OK;
  if (slots > 0) {
    int *unused_cnt = nullptr;
    int rc = split_workspace(s, (size_t)slots * 128 * BN * sizeof(float), 0, &args.ws, &unused_cnt);
    if (rc) return rc;
  }
  args.njobs = p.njobs;
  args.total_units = (int)units;
  args.out_dt = p.out_dt;
  args.idesc = umma_idesc_f16(1u, 0u, 128u, (uint32_t)BN);
  args.status = p.status;
  args.wait_ns = (uint64_t)p.wait_ns;
  int rc;
  if (BN == 16)
    rc = mt_dec_launch<16, 15, 4>(args, sms, s);
  else if (BN == 32)
    rc = mt_dec_launch<32, 12, 4>(args, sms, s);
  else if (BN == 64)
    rc = mt_launch<64, 4>(args, sms, s);
  else if (BN == 128)
    rc = mt_launch<128, 4>(args, sms, s);
  else
    rc = mt_launch<256, 4>(args, sms, s);
  if (rc != TP_OK) return rc;
  *handled = true;
  if (slots > 0) {  // ordered sums of the split tiles
    SplitJob sj[kMaxJobs];
    for (int j = 0; j < p.njobs; ++j) {
      const MtJob &Q = args.jobs[j];
      sj[j] = SplitJob{Q.C, Q.bias, Q.ldc, Q.ws_base, Q.rows, Q.T, Q.tiles, Q.ntiles, Q.splits};
    }
    return launch_split_reduce(sj, p.njobs, args.ws, BN, p.out_dt, s);
  }
  return TP_OK;
}

}  // namespace

int launch_mx(const Problem &p, cudaStream_t s, bool *handled) {
  *handled = false;
  if (p.in_dt != TP_BF16) return TP_OK;
  int rc = launch_mx_gemv(p, s, handled);
  if (rc != TP_OK || *handled) return rc;
  return launch_mx_tc(p, s, handled);
}

}  // namespace tp
