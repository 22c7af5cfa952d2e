// k_q4.cu -- 4-bit affine (group 64) kernels: the a6 device quantizer and the
// dequant-fused tensor-core linears of a7.
//
// q4_umma_kernel builds the WEIGHT operand of tcgen05.mma in tensor memory:
// converter warps read the packed codes that TMA brought into shared memory,
// expand them in registers and write them to TMEM with tcgen05.st; the MMA
// takes A from TMEM and the activations x (B, K-major, 128B-swizzled) from
// shared memory.  Weight rows fill the M = 128 dimension, tokens the N
// dimension (swap-AB), and the epilogue stores the transpose.
//
// Decode (T <= 16): the codes enter the MMA as the exact integers 0..15
// (bf16), one TMEM partial D_g per 64-element group g, and the epilogue forms
//   y[t][o] = sum_g ( s[o][g] * D_g[o][t] + b[o][g] * X_g[t] ),
//   X_g[t] = sum_{k in g} x[t][k],
// in float32.  Lane 31 of every 32-lane quarter of the tile is a row of ones,
// so the tensor core computes X_g alongside D_g (124 weight rows per tile).
// Prefill (T > 16): the converter writes the dequantized values
// s*q + b (float32, rounded once to bf16) and the groups accumulate in one
// TMEM accumulator.
// Tiles are split over CTAs by K (rank by rank for the row-parallel layer);
// each split's float32 partial goes to a workspace slot.  Decode: the warp
// that arrives last at the tile's counter adds the slots in split order (rank
// order), then the bias once; no CTA ever waits for another.  Prefill: a
// second launch adds each tile's column-major slots in split order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include <mutex>

#include "ptx.cuh"
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
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "quantize kernel launch");
}

// ====================================================================== q4 tcgen05
namespace {

constexpr int kQThreads = 14 * 32;  // producer, MMA, 8 converter warps, 4 epilogue warps

struct Q4Part {
  const uint16_t *sc, *qb;  // float16 bits, (rows, groups)
  int groups;               // K / 64
  int16_t cmap, xmap;
  int nchunk, chunk_groups;
};

struct Q4Job {
  void *C;
  const float *bias;
  int64_t ldc;
  int rows, T;
  int part0, nparts;
  int tiles, ntiles, splits;
  int unit_begin;
  int cnt_base;
  int64_t ws_base;  // first partial slot of this job (slot = 128 x 16 floats)
};

struct Q4Args {
  CUtensorMap cmaps[kMaxParts];
  CUtensorMap xmaps[kMaxParts];
  const float *xfac[kMaxParts];  // prefill: per x map, 2^-c of every token (x was scaled by 2^c)
  Q4Job jobs[kMaxJobs];
  Q4Part parts[kMaxParts];
  int njobs, total_units, ncm, nxm;
  int out_dt;
  int sb_vec;  // scales/biases allow 8-byte loads of 4 groups (groups % 4 == 0, 8B aligned)
  uint32_t idesc;
  float *ws;
  int *cnt;
  int *status;
  uint64_t wait_ns;
  unsigned long long *trace;  // role timeline of CTA 0, or null
  int64_t trace_cap;
};

// Records the time of (event, stage sequence) when tracing CTA 0.
__device__ __forceinline__ void q4_trace(const Q4Args &a, int role, int event, int seq) {
  (void)role;
  if (a.trace != nullptr && blockIdx.x == 0 && seq < 1024) a.trace[16 + event * 1024 + seq] = globaltimer_ns();
}

template <bool DECODE>
struct Q4Cfg;
template <>
struct Q4Cfg<true> {
  static constexpr int BN = 16, GS = 4, STAGES = 8, NA = 8, ND = 8, ROWS = 124;
  static constexpr int CODES_BYTES = 16384, XBOX = 2048, X_BYTES = 4 * 2048;
  static constexpr int CODES_TX = 124 * 128, X_TX = 4 * 2048;
  static constexpr int A_COL0 = 0, D_COL0 = 256;
};
template <>
struct Q4Cfg<false> {
  static constexpr int BN = 256, GS = 1, STAGES = 5, NA = 8, ND = 1, ROWS = 128;
  static constexpr int CODES_BYTES = 4096, XBOX = 32768, X_BYTES = 32768;
  static constexpr int CODES_TX = 4096, X_TX = 32768;
  static constexpr int A_COL0 = 256, D_COL0 = 0;
};

struct UnitInfo {
  int job, part, tile, ntile, tile_lin, sidx, g0, g1;
};

__device__ __forceinline__ void q4_decode_unit(const Q4Args &a, int u, UnitInfo &ui) {
  int j = 0;
  while (j + 1 < a.njobs && u >= a.jobs[j + 1].unit_begin) ++j;
  const Q4Job &J = a.jobs[j];
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
  const Q4Part &P = a.parts[J.part0 + p];
  ui.part = J.part0 + p;
  ui.g0 = c * P.chunk_groups;
  ui.g1 = min(P.groups, ui.g0 + P.chunk_groups);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}


// Eight 4-bit codes (one word, element e at bits 4e) -> four bf16x2 words of
// the exact integers, natural element order (low half = even element).
// 0x4300 | n is the bf16 of 128 + n; one fused multiply-add by (1, 1) and
// (-128, -128) returns n exactly.
__device__ __forceinline__ void codes_to_int_bf16(uint32_t w, uint32_t *o) {
  const uint32_t a = (w & 0x000F000Fu) | 0x43004300u;          // (n0, n4)
  const uint32_t b = ((w >> 4) & 0x000F000Fu) | 0x43004300u;   // (n1, n5)
  const uint32_t c = ((w >> 8) & 0x000F000Fu) | 0x43004300u;   // (n2, n6)
  const uint32_t d = ((w >> 12) & 0x000F000Fu) | 0x43004300u;  // (n3, n7)
  const uint32_t one = 0x3F803F80u, m128 = 0xC300C300u;
  o[0] = fma_bf16x2(prmt(a, b, 0x5410), one, m128);  // (n0, n1)
  o[1] = fma_bf16x2(prmt(c, d, 0x5410), one, m128);  // (n2, n3)
  o[2] = fma_bf16x2(prmt(a, b, 0x7632), one, m128);  // (n4, n5)
  o[3] = fma_bf16x2(prmt(c, d, 0x7632), one, m128);  // (n6, n7)
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Eight codes of one word -> four f16x2 words of s*code + b in the blocked K
// order (n0,n4), (n1,n5), (n2,n6), (n3,n7).  0x6400 | n is the f16 of 1024 + n;
// subtracting 1024 gives n exactly, and one f16 fused multiply-add forms
// s*n + b with a single rounding.  s2, b2 hold the group's f16 s and b twice.
__device__ __forceinline__ void codes_to_values_f16_blocked(uint32_t w, uint32_t s2, uint32_t b2,
                                                            uint32_t *o) {
  const uint32_t m = 0x64006400u;
  o[0] = hfma2_u32(hsub2_u32((w & 0x000F000Fu) | m, m), s2, b2);
  o[1] = hfma2_u32(hsub2_u32(((w >> 4) & 0x000F000Fu) | m, m), s2, b2);
  o[2] = hfma2_u32(hsub2_u32(((w >> 8) & 0x000F000Fu) | m, m), s2, b2);
  o[3] = hfma2_u32(hsub2_u32(((w >> 12) & 0x000F000Fu) | m, m), s2, b2);
}

// A job's output, copied to registers once per unit.  Read through the
// kernel-parameter block instead, every field is reloaded after every store
// (the compiler cannot tell the output from the parameters): one dependent
// load per element, 54 us for a 128 x 256 prefill tile.
struct Q4Out {
  void *C;
  int64_t ldc;
  int T, dt;
};
__device__ __forceinline__ Q4Out q4_out(const Q4Args &a, const Q4Job &J) { return Q4Out{J.C, J.ldc, J.T, a.out_dt}; }

__device__ __forceinline__ void q4_store(const Q4Out &o, int t, int orow, float v) {
  const int64_t idx = (int64_t)t * o.ldc + orow;
  if (o.dt == TP_F32)
    static_cast<float *>(o.C)[idx] = v;
  else if (o.dt == TP_BF16)
    static_cast<uint16_t *>(o.C)[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  else
    static_cast<uint16_t *>(o.C)[idx] = __half_as_ushort(__float2half_rn(v));
}

#define Q4_WAIT_ALL(bar, par, okvar)                                                   \
  {                                                                                    \
    const bool _r = mbar_wait((bar), (par), lim, a.status, &abort_sh);                 \
    if (!__all_sync(0xffffffffu, _r)) {                                                \
      okvar = false;                                                                   \
    }                                                                                  \
  }


// ---------------------------------------------------------------- prefill x pre-pass
// The prefill MMA takes both operands in float16 (the dequantized weights
// s*q + b are formed in f16, one rounding), in the weights' blocked order
// inside every 8-element block of K (0,4,1,5,2,6,3,7; a dot product does not
// depend on the order of its terms).  Each activation row x[t] is
// scaled by a power of two 2^c (its largest |x| lands in [2^14, 2^15)) and
// rounded to f16 once, here, instead of in every CTA that reads it; the
// epilogue multiplies the token's column by 2^-c.  Every bfloat16 x with
// |x 2^c| >= 2^-14 (within 2^28 of its row's largest) keeps all 8 of its
// significant bits; smaller ones become f16 subnormals, off by at most
// 2^-25 in the scaled unit (2^-39 of the row's largest).  So the whole
// bfloat16 range is kept: |x| > 65504 and rows of tiny values included.
struct XsRegion {
  const uint16_t *x;  // bf16 rows, stride lda
  int64_t lda;
  uint16_t *xs;       // f16 rows, stride K
  float *fac;         // 2^-c per row
  int K, row_begin;
};
struct XsArgs {
  XsRegion r[kMaxParts];
  int nregions;
};

__global__ void __launch_bounds__(256) q4_xs_prep_kernel(const __grid_constant__ XsArgs a) {
  griddep_launch_dependents();
  griddep_wait();  // x may be the previous kernel's output
  __shared__ uint32_t red[8];
  const int row = blockIdx.x;
  int ri = 0;
  while (ri + 1 < a.nregions && row >= a.r[ri + 1].row_begin) ++ri;
  const XsRegion &R = a.r[ri];
  const int t = row - R.row_begin;
  const uint4 *src = reinterpret_cast<const uint4 *>(R.x + (int64_t)t * R.lda);
  const int n16 = R.K / 8;
  // the largest |x| of the row, as float32 bits (ordered like the values)
  uint32_t mx = 0;
  for (int i = threadIdx.x; i < n16; i += 256) {
    const uint4 w = src[i];
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      mx = max(mx, (wv[k] & 0x7FFFu) << 16);
      mx = max(mx, wv[k] & 0x7FFF0000u);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) mx = max(mx, red[i]);
  // biased exponent E of the largest |x| (1 for zero or subnormal rows):
  // max * 2^(141 - E) lies in [2^14, 2^15); c is kept where 2^c and 2^-c
  // are normal floats
  const int E = max((int)(mx >> 23), 1);
  const int c = min(max(141 - E, -125), 125);
  const float sc = __uint_as_float((uint32_t)(127 + c) << 23);
  uint4 *dst = reinterpret_cast<uint4 *>(R.xs + (int64_t)t * R.K);
  for (int i = threadIdx.x; i < n16; i += 256) {
    const uint4 w = src[i];
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    float e[8];  // the block's 8 elements, scaled
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      e[2 * k] = __uint_as_float(wv[k] << 16) * sc;
      e[2 * k + 1] = __uint_as_float(wv[k] & 0xFFFF0000u) * sc;
    }
    // the weights' blocked K order inside the block: (0,4), (1,5), (2,6), (3,7)
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 h = __floats2half2_rn(e[k], e[k + 4]);
      o[k] = *reinterpret_cast<const uint32_t *>(&h);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) R.fac[t] = __uint_as_float((uint32_t)(127 - c) << 23);
}

// When tracing, every CTA b (< 1024) records its SM id + 1 (event 28) and its
// start (30) and end (31) times at word index b.
__device__ __forceinline__ void q4_cta_trace(const Q4Args &a, int event) {
  if (a.trace == nullptr || threadIdx.x != 0 || blockIdx.x >= 1024) return;
  if (event == 30) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    a.trace[16 + 28 * 1024 + blockIdx.x] = smid + 1;
  }
  a.trace[16 + event * 1024 + blockIdx.x] = globaltimer_ns();
}

template <bool DECODE>
__global__ void __launch_bounds__(kQThreads, 1) q4_umma_kernel(const __grid_constant__ Q4Args a) {
  q4_cta_trace(a, 30);
  griddep_launch_dependents();
  griddep_wait();  // programmatic launch: no global memory before the previous kernel completes
  using C = Q4Cfg<DECODE>;
  constexpr int STAGE_BYTES = C::CODES_BYTES + C::X_BYTES;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");

  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[C::STAGES], empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t afull_bar[C::NA], aempty_bar[C::NA];
  __shared__ __align__(8) uint64_t dfull_bar[C::ND], dempty_bar[C::ND];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < C::NA; ++i) {
      mbar_init(smem_u32(&afull_bar[i]), 8);
      mbar_init(smem_u32(&aempty_bar[i]), 1);
    }
    for (int i = 0; i < C::ND; ++i) {
      mbar_init(smem_u32(&dfull_bar[i]), 1);
      mbar_init(smem_u32(&dempty_bar[i]), 4);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int st = 0, pseq = 0;
      uint32_t ph = 0;
      bool used[C::STAGES];
      uint32_t lastph[C::STAGES];
#pragma unroll
      for (int i = 0; i < C::STAGES; ++i) used[i] = false;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        UnitInfo ui;
        q4_decode_unit(a, u, ui);
        const Q4Part &P = a.parts[ui.part];
        for (int gs = ui.g0; gs < ui.g1; gs += C::GS) {
          if (!mbar_wait(smem_u32(&empty_bar[st]), ph ^ 1, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          const uint32_t base = sbase + st * STAGE_BYTES;
          const uint32_t fb = smem_u32(&full_bar[st]);
          mbar_arrive_expect_tx(fb, C::CODES_TX + C::X_TX);
          // the codes are read once: evicted first, so x and the split partials stay in L2
          tma_load_2d_hint(base, &a.cmaps[P.cmap], fb, gs * 8, ui.tile * C::ROWS, l2_policy_evict_first());
#pragma unroll
          for (int gi = 0; gi < C::GS; ++gi)
            tma_load_2d(base + C::CODES_BYTES + gi * C::XBOX, &a.xmaps[P.xmap], fb, (gs + gi) * 64,
                        ui.ntile * C::BN);
          q4_trace(a, 1, 1, pseq++);
          used[st] = true;
          lastph[st] = ph;
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok)
        for (int i = 0; i < C::STAGES; ++i)
          if (used[i]) mbar_wait(smem_u32(&full_bar[i]), lastph[i], lim, a.status, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int st = 0, as = 0, ds = 0, mseq = 0;
      uint32_t ph = 0, aph = 0, dph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        UnitInfo ui;
        q4_decode_unit(a, u, ui);
        bool first = true;
        for (int gs = ui.g0; ok && gs < ui.g1; gs += C::GS) {
          if (!mbar_wait(smem_u32(&full_bar[st]), ph, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          q4_trace(a, 2, 2, mseq);
          tc_fence_after();
          const uint32_t base = sbase + st * STAGE_BYTES;
          const int ng = min(C::GS, ui.g1 - gs);
          for (int gi = 0; gi < ng; ++gi) {
            if (!mbar_wait(smem_u32(&afull_bar[as]), aph, lim, a.status, &abort_sh)) {
              ok = false;
              break;
            }
            if (DECODE || first) {
              if (!mbar_wait(smem_u32(&dempty_bar[ds]), dph ^ 1, lim, a.status, &abort_sh)) {
                ok = false;
                break;
              }
            }
            tc_fence_after();
            const uint32_t d = tmem + C::D_COL0 + ds * C::BN;
            const uint32_t xb = base + C::CODES_BYTES + (DECODE ? gi * C::XBOX : 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = DECODE ? (kk > 0 ? 1u : 0u) : ((first && kk == 0) ? 0u : 1u);
              umma_f16_ts(d, tmem + C::A_COL0 + as * 32 + kk * 8,
                          umma_desc_sw128(xb + kk * 32, 16, 1024), a.idesc, acc);
            }
            umma_commit(smem_u32(&aempty_bar[as]));
            if (++as == C::NA) {
              as = 0;
              aph ^= 1;
            }
            if (DECODE) {
              umma_commit(smem_u32(&dfull_bar[ds]));
              if (++ds == C::ND) {
                ds = 0;
                dph ^= 1;
              }
            }
            first = false;
          }
          if (!ok) break;
          umma_commit(smem_u32(&empty_bar[st]));
          q4_trace(a, 2, 5, mseq++);
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!DECODE && ok) {
          umma_commit(smem_u32(&dfull_bar[ds]));
          if (++ds == C::ND) {
            ds = 0;
            dph ^= 1;
          }
        }
      }
      umma_commit(smem_u32(&drain_bar));
      mbar_wait(smem_u32(&drain_bar), 0, lim, a.status, nullptr);
      if (a.trace != nullptr && blockIdx.x < 1024) a.trace[16 + 27 * 1024 + blockIdx.x] = globaltimer_ns();
    }
  } else if (warp < 10) {
    // ---------------------------------------------------------- converters
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const bool ones = DECODE && lane == 31;
    const int srow = DECODE ? quarter * 31 + lane : quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool tr = warp == 2 && lane == 0;
    int st = 0, as = 0, cseq = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
      UnitInfo ui;
      q4_decode_unit(a, u, ui);
      const Q4Part &P = a.parts[ui.part];
      const Q4Job &J = a.jobs[ui.job];
      const int orow = ui.tile * C::ROWS + srow;
      for (int gs = ui.g0; ok && gs < ui.g1; gs += C::GS) {
        Q4_WAIT_ALL(smem_u32(&full_bar[st]), ph, ok);
        if (!ok) break;
        if (tr) q4_trace(a, 3, 6, cseq);
        const uint32_t base = sbase + st * STAGE_BYTES;
        const int ng = min(C::GS, ui.g1 - gs);
        for (int gi = 0; gi < ng; ++gi) {
          Q4_WAIT_ALL(smem_u32(&aempty_bar[as]), aph ^ 1, ok);
          if (!ok) break;
          if (tr) q4_trace(a, 3, 7, cseq);
          tc_fence_after();
          uint32_t out[16];
          if (DECODE) {
            if (ones) {
#pragma unroll
              for (int i = 0; i < 16; ++i) out[i] = 0x3F803F80u;
            } else {
              const int c = gi * 2 + half;
              const uint4 w = lds128(base + srow * 128 + ((c ^ (srow & 7)) << 4));
              codes_to_int_bf16(w.x, out + 0);
              codes_to_int_bf16(w.y, out + 4);
              codes_to_int_bf16(w.z, out + 8);
              codes_to_int_bf16(w.w, out + 12);
            }
          } else {
            // the x tile is already f16 in the blocked K order (pre-pass)
            if (tr) q4_trace(a, 3, 12, cseq);
            uint32_t s2 = 0, b2 = 0;
            if (orow < J.rows) {
              const int64_t gi64 = (int64_t)orow * P.groups + gs + gi;
              const uint32_t sh = __ldg(P.sc + gi64), bh = __ldg(P.qb + gi64);
              s2 = sh | (sh << 16);
              b2 = bh | (bh << 16);
            }
            const uint4 w = lds128(base + srow * 32 + half * 16);
            codes_to_values_f16_blocked(w.x, s2, b2, out + 0);
            codes_to_values_f16_blocked(w.y, s2, b2, out + 4);
            codes_to_values_f16_blocked(w.z, s2, b2, out + 8);
            codes_to_values_f16_blocked(w.w, s2, b2, out + 12);
          }
          tmem_st16(tmem + lane_off + C::A_COL0 + as * 32 + half * 16, out);
          tmem_wait_st();
          if (tr) q4_trace(a, 3, 13, cseq);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&afull_bar[as]));
          if (tr) q4_trace(a, 3, 8, cseq++);
          if (++as == C::NA) {
            as = 0;
            aph ^= 1;
          }
        }
        if (++st == C::STAGES) {
          st = 0;
          ph ^= 1;
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const bool ones = DECODE && lane == 31;
    const int srow = DECODE ? quarter * 31 + lane : m;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int ds = 0, eseq = 0;
    uint32_t dph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
      UnitInfo ui;
      q4_decode_unit(a, u, ui);
      const Q4Part &P = a.parts[ui.part];
      const Q4Job &J = a.jobs[ui.job];
      const Q4Out o = q4_out(a, J);
      const int orow = ui.tile * C::ROWS + srow;
      const bool valid = !ones && orow < J.rows;
      if constexpr (DECODE) {
        float acc[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) acc[t] = 0.f;
        for (int g = ui.g0; g < ui.g1; ++g) {
          Q4_WAIT_ALL(smem_u32(&dfull_bar[ds]), dph, ok);
          if (!ok) break;
          tc_fence_after();
          float v[16];
          tmem_ld16(tmem + lane_off + C::D_COL0 + ds * 16, v);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&dempty_bar[ds]));
          if (++ds == C::ND) {
            ds = 0;
            dph ^= 1;
          }
          float sc = 0.f, bq = 0.f;
          if (valid) {
            const int64_t gi64 = (int64_t)orow * P.groups + g;
            sc = h2f(__ldg(P.sc + gi64));
            bq = h2f(__ldg(P.qb + gi64));
          }
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const float xs = __shfl_sync(0xffffffffu, v[t], 31);
            acc[t] = fmaf(sc, v[t], fmaf(bq, xs, acc[t]));
          }
        }
        if (!ok) break;
        if (J.splits == 1) {
          if (valid) {
            const float bias = J.bias ? __ldg(J.bias + orow) : 0.f;
#pragma unroll
            for (int t = 0; t < 16; ++t)
              if (t < o.T) q4_store(o, t, orow, acc[t] + bias);
          }
        } else {
          // Split tile: every warp owns its 32 rows; the warp that arrives last
          // at its (tile, quarter) counter adds the split partials in order.
          float *slot = a.ws + ((J.ws_base + (int64_t)ui.tile_lin * J.splits + ui.sidx) * 128 + m) * C::BN;
#pragma unroll
          for (int t = 0; t < 16; t += 4)
            __stcg(reinterpret_cast<float4 *>(slot + t), make_float4(acc[t], acc[t + 1], acc[t + 2], acc[t + 3]));
          __threadfence();
          __syncwarp();
          int prev = 0;
          int *cnt = a.cnt + (int64_t)(J.cnt_base + ui.tile_lin) * 4 + quarter;
          if (lane == 0) prev = atomicAdd(cnt, 1);
          prev = __shfl_sync(0xffffffffu, prev, 0);
          if (prev == J.splits - 1) {
            __threadfence();
            float sum[16];
            const float *s0 = a.ws + ((J.ws_base + (int64_t)ui.tile_lin * J.splits) * 128 + m) * C::BN;
#pragma unroll
            for (int t = 0; t < 16; t += 4) {
              const float4 f = __ldcg(reinterpret_cast<const float4 *>(s0 + t));
              sum[t] = f.x;
              sum[t + 1] = f.y;
              sum[t + 2] = f.z;
              sum[t + 3] = f.w;
            }
            for (int j = 1; j < J.splits; ++j) {
              const float *sj = s0 + (int64_t)j * 128 * C::BN;
#pragma unroll
              for (int t = 0; t < 16; t += 4) {
                const float4 f = __ldcg(reinterpret_cast<const float4 *>(sj + t));
                sum[t] += f.x;
                sum[t + 1] += f.y;
                sum[t + 2] += f.z;
                sum[t + 3] += f.w;
              }
            }
            if (valid) {
              const float bias = J.bias ? __ldg(J.bias + orow) : 0.f;
#pragma unroll
              for (int t = 0; t < 16; ++t)
                if (t < o.T) q4_store(o, t, orow, sum[t] + bias);
            }
            __syncwarp();
            if (lane == 0) *cnt = 0;  // ready for the next call
          }
        }
      } else {
        const int t0 = ui.ntile * C::BN;
        // 2^-c of the unit's tokens (lane l: tokens t0 + 32 j + l), loaded
        // before the accumulator is waited on
        const float *fac = a.xfac[P.xmap];
        float fw[C::BN / 32];
#pragma unroll
        for (int j = 0; j < C::BN / 32; ++j) {
          const int t = t0 + 32 * j + lane;
          fw[j] = t < J.T ? __ldg(fac + t) : 0.f;
        }
        const float bias = (valid && J.bias) ? __ldg(J.bias + orow) : 0.f;
        Q4_WAIT_ALL(smem_u32(&dfull_bar[ds]), dph, ok);
        if (!ok) break;
        if (warp == 10 && lane == 0) q4_trace(a, 4, 9, eseq);
        tc_fence_after();
        // split tiles: float32 partials to column-major workspace slots (a
        // warp's 32 rows of one column are one 128-byte line); a second launch
        // adds each tile's slots in split (rank) order, then the bias
        const bool split = J.splits > 1;
        float *slot = split ? a.ws + (J.ws_base + (int64_t)ui.tile_lin * J.splits + ui.sidx) * 128 * C::BN + m
                            : nullptr;
#pragma unroll
        for (int c = 0; c < C::BN / 32; ++c) {
          float v[32];
          tmem_ld32(tmem + lane_off + C::D_COL0 + ds * C::BN + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= __shfl_sync(0xffffffffu, fw[c], i);  // undo the x scaling (exact)
          if (split) {
#pragma unroll
            for (int i = 0; i < 32; ++i) __stcg(slot + (c * 32 + i) * 128, v[i]);
          } else if (valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int t = t0 + c * 32 + i;
              if (t < o.T) q4_store(o, t, orow, v[i] + bias);
            }
          }
          if (warp == 10 && lane == 0) q4_trace(a, 4, 10, eseq * 8 + c);
        }
        ++eseq;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&dempty_bar[ds]));
        if (++ds == C::ND) {
          ds = 0;
          dph ^= 1;
        }
      }
    }
  }

  if (a.trace != nullptr && warp == 10 && lane == 0 && blockIdx.x < 1024)
    a.trace[16 + 26 * 1024 + blockIdx.x] = globaltimer_ns();  // first epilogue warp done
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  q4_cta_trace(a, 31);
}

// ---------------------------------------------------------------- decode kernel
// T <= 16.  Work is handed between roles one stage (4 groups of 64 codes) at a
// time.  Inside every 8-element block of K the weights and x use the same
// order (0,4,1,5,2,6,3,7): a packed code word then expands with one mask per
// output register, and the converters apply the same order to the x tile in
// shared memory (a 16-byte chunk holds one block, so the swizzle is unaffected).
// A dot product does not depend on the order of its terms, so D is unchanged.
struct DecCfg {
  static constexpr int BN = 16, GS = 4, STAGES = 8, ROWS = 124;
  static constexpr int CODES_BYTES = 16384, XBOX = 2048, X_BYTES = 4 * 2048;
  static constexpr int STAGE_BYTES = CODES_BYTES + X_BYTES;
  static constexpr int TX = 124 * 128 + 4 * 2048;
  static constexpr int NA = 2, A_COLS = 128, A_COL0 = 0;  // one A slot = one stage
  static constexpr int ND = 2, D_COLS = 64, D_COL0 = 256;  // one D slot = one stage
};

// Eight codes of one word -> four bf16x2 words of exact integers, blocked order.
__device__ __forceinline__ void codes_to_int_bf16_blocked(uint32_t w, uint32_t *o) {
  const uint32_t one = 0x3F803F80u, m128 = 0xC300C300u;
  o[0] = fma_bf16x2((w & 0x000F000Fu) | 0x43004300u, one, m128);          // (n0, n4)
  o[1] = fma_bf16x2(((w >> 4) & 0x000F000Fu) | 0x43004300u, one, m128);   // (n1, n5)
  o[2] = fma_bf16x2(((w >> 8) & 0x000F000Fu) | 0x43004300u, one, m128);   // (n2, n6)
  o[3] = fma_bf16x2(((w >> 12) & 0x000F000Fu) | 0x43004300u, one, m128);  // (n3, n7)
}

template <int TCAP>
__global__ void __launch_bounds__(kQThreads, 1) q4_decode_kernel(const __grid_constant__ Q4Args a) {
  griddep_launch_dependents();
  griddep_wait();  // programmatic launch: no global memory before the previous kernel completes
  using C = DecCfg;
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[C::STAGES], empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t afull_bar[C::NA], aempty_bar[C::NA];
  __shared__ __align__(8) uint64_t dfull_bar[C::ND], dempty_bar[C::ND];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < C::NA; ++i) {
      mbar_init(smem_u32(&afull_bar[i]), 8);
      mbar_init(smem_u32(&aempty_bar[i]), 1);
    }
    for (int i = 0; i < C::ND; ++i) {
      mbar_init(smem_u32(&dfull_bar[i]), 1);
      mbar_init(smem_u32(&dempty_bar[i]), 4);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int st = 0, pseq = 0;
      uint32_t ph = 0;
      bool used[C::STAGES];
      uint32_t lastph[C::STAGES];
#pragma unroll
      for (int i = 0; i < C::STAGES; ++i) used[i] = false;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        UnitInfo ui;
        q4_decode_unit(a, u, ui);
        const Q4Part &P = a.parts[ui.part];
        for (int gs = ui.g0; gs < ui.g1; gs += C::GS) {
          if (!mbar_wait(smem_u32(&empty_bar[st]), ph ^ 1, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          const uint32_t base = sbase + st * C::STAGE_BYTES;
          const uint32_t fb = smem_u32(&full_bar[st]);
          mbar_arrive_expect_tx(fb, C::TX);
          tma_load_2d(base, &a.cmaps[P.cmap], fb, gs * 8, ui.tile * C::ROWS);
#pragma unroll
          for (int gi = 0; gi < C::GS; ++gi)
            tma_load_2d(base + C::CODES_BYTES + gi * C::XBOX, &a.xmaps[P.xmap], fb, (gs + gi) * 64, 0);
          q4_trace(a, 1, 1, pseq++);
          used[st] = true;
          lastph[st] = ph;
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok)
        for (int i = 0; i < C::STAGES; ++i)
          if (used[i]) mbar_wait(smem_u32(&full_bar[i]), lastph[i], lim, a.status, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int st = 0, as = 0, ds = 0, mseq = 0;
      uint32_t ph = 0, aph = 0, dph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        UnitInfo ui;
        q4_decode_unit(a, u, ui);
        for (int gs = ui.g0; gs < ui.g1; gs += C::GS) {
          if (!mbar_wait(smem_u32(&full_bar[st]), ph, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          q4_trace(a, 2, 2, mseq);
          if (!mbar_wait(smem_u32(&afull_bar[as]), aph, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          q4_trace(a, 2, 3, mseq);
          if (!mbar_wait(smem_u32(&dempty_bar[ds]), dph ^ 1, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          q4_trace(a, 2, 4, mseq);
          tc_fence_after();
          const uint32_t xb = sbase + st * C::STAGE_BYTES + C::CODES_BYTES;
          const int ng = min(C::GS, ui.g1 - gs);
          // k-major order: consecutive MMAs go to different groups' accumulators,
          // so no MMA waits for the one issued just before it.
          // Descriptors and TMEM addresses are formed once per stage; the
          // 4-group case is fully unrolled so each MMA costs one add and the issue.
          const uint64_t bd0 = umma_desc_sw128(xb, 16, 1024);
          const uint32_t d0 = tmem + C::D_COL0 + ds * C::D_COLS;
          const uint32_t a0 = tmem + C::A_COL0 + as * C::A_COLS;
          if (ng == C::GS) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
              for (int gi = 0; gi < C::GS; ++gi)
                umma_f16_ts(d0 + gi * 16, a0 + gi * 32 + kk * 8,
                            bd0 + (uint64_t)((gi * C::XBOX + kk * 32) >> 4), a.idesc, kk > 0 ? 1u : 0u);
          } else {
            for (int kk = 0; kk < 4; ++kk)
              for (int gi = 0; gi < ng; ++gi)
                umma_f16_ts(d0 + gi * 16, a0 + gi * 32 + kk * 8,
                            bd0 + (uint64_t)((gi * C::XBOX + kk * 32) >> 4), a.idesc, kk > 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(&dfull_bar[ds]));
          umma_commit(smem_u32(&aempty_bar[as]));
          umma_commit(smem_u32(&empty_bar[st]));
          q4_trace(a, 2, 5, mseq++);
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1;
          }
          if (++as == C::NA) {
            as = 0;
            aph ^= 1;
          }
          if (++ds == C::ND) {
            ds = 0;
            dph ^= 1;
          }
        }
      }
      umma_commit(smem_u32(&drain_bar));
      mbar_wait(smem_u32(&drain_bar), 0, lim, a.status, nullptr);
    }
  } else if (warp < 10) {
    // ---------------------------------------------------------- converters
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int cid = (warp - 2) * 32 + lane;  // 0..255, for the x reorder
    const bool ones = lane == 31;
    const int srow = quarter * 31 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool tr = (warp == 2 && lane == 0);
    int st = 0, as = 0, cseq = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
      UnitInfo ui;
      q4_decode_unit(a, u, ui);
      for (int gs = ui.g0; gs < ui.g1; gs += C::GS) {
        Q4_WAIT_ALL(smem_u32(&full_bar[st]), ph, ok);
        if (!ok) break;
        if (tr) q4_trace(a, 3, 6, cseq);
        Q4_WAIT_ALL(smem_u32(&aempty_bar[as]), aph ^ 1, ok);
        if (!ok) break;
        if (tr) q4_trace(a, 3, 7, cseq);
        tc_fence_after();
        const uint32_t base = sbase + st * C::STAGE_BYTES;
        // x tile (4 groups x 16 rows x 128 B = 512 chunks): blocked order in place
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t addr = base + C::CODES_BYTES + (cid + k * 256) * 16;
          const uint4 v = lds128(addr);
          uint4 w;
          w.x = prmt(v.x, v.z, 0x5410);
          w.y = prmt(v.x, v.z, 0x7632);
          w.z = prmt(v.y, v.w, 0x5410);
          w.w = prmt(v.y, v.w, 0x7632);
          sts128(addr, w);
        }
        fence_proxy_async_smem();
        if (tr) q4_trace(a, 3, 12, cseq);
        const int ng = min(C::GS, ui.g1 - gs);
        uint4 wv[C::GS];
#pragma unroll
        for (int gi = 0; gi < C::GS; ++gi) {
          const int c = gi * 2 + half;
          wv[gi] = (ones || gi >= ng) ? make_uint4(0, 0, 0, 0)
                                      : lds128(base + srow * 128 + ((c ^ (srow & 7)) << 4));
        }
        uint32_t out[C::GS][16];
#pragma unroll
        for (int gi = 0; gi < C::GS; ++gi) {
          if (ones) {
#pragma unroll
            for (int i = 0; i < 16; ++i) out[gi][i] = 0x3F803F80u;
          } else {
            codes_to_int_bf16_blocked(wv[gi].x, out[gi] + 0);
            codes_to_int_bf16_blocked(wv[gi].y, out[gi] + 4);
            codes_to_int_bf16_blocked(wv[gi].z, out[gi] + 8);
            codes_to_int_bf16_blocked(wv[gi].w, out[gi] + 12);
          }
        }
#pragma unroll
        for (int gi = 0; gi < C::GS; ++gi)
          if (gi < ng) tmem_st16(tmem + lane_off + C::A_COL0 + as * C::A_COLS + gi * 32 + half * 16, out[gi]);
        tmem_wait_st();
        if (tr) q4_trace(a, 3, 13, cseq);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&afull_bar[as]));
        if (tr) q4_trace(a, 3, 8, cseq++);
        if (++st == C::STAGES) {
          st = 0;
          ph ^= 1;
        }
        if (++as == C::NA) {
          as = 0;
          aph ^= 1;
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const bool ones = lane == 31;
    const int srow = quarter * 31 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool tr = (warp == 10 && lane == 0);
    int ds = 0, eseq = 0;
    uint32_t dph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
      UnitInfo ui;
      q4_decode_unit(a, u, ui);
      const Q4Part &P = a.parts[ui.part];
      const Q4Job &J = a.jobs[ui.job];
      const Q4Out o = q4_out(a, J);
      const int orow = ui.tile * C::ROWS + srow;
      const bool valid = !ones && orow < J.rows;
      float acc[TCAP];
#pragma unroll
      for (int t = 0; t < TCAP; ++t) acc[t] = 0.f;
      for (int gs = ui.g0; gs < ui.g1; gs += C::GS) {
        const int ng = min(C::GS, ui.g1 - gs);
        float sc[4] = {0.f, 0.f, 0.f, 0.f}, bq[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid) {
          const int64_t g64 = (int64_t)orow * P.groups + gs;
          if (a.sb_vec && ng == 4) {
            const uint2 s4 = __ldg(reinterpret_cast<const uint2 *>(P.sc + g64));
            const uint2 b4 = __ldg(reinterpret_cast<const uint2 *>(P.qb + g64));
            sc[0] = h2f((uint16_t)(s4.x & 0xFFFF));
            sc[1] = h2f((uint16_t)(s4.x >> 16));
            sc[2] = h2f((uint16_t)(s4.y & 0xFFFF));
            sc[3] = h2f((uint16_t)(s4.y >> 16));
            bq[0] = h2f((uint16_t)(b4.x & 0xFFFF));
            bq[1] = h2f((uint16_t)(b4.x >> 16));
            bq[2] = h2f((uint16_t)(b4.y & 0xFFFF));
            bq[3] = h2f((uint16_t)(b4.y >> 16));
          } else {
#pragma unroll
            for (int gi = 0; gi < 4; ++gi)
              if (gi < ng) {
                sc[gi] = h2f(__ldg(P.sc + g64 + gi));
                bq[gi] = h2f(__ldg(P.qb + g64 + gi));
              }
          }
        }
        Q4_WAIT_ALL(smem_u32(&dfull_bar[ds]), dph, ok);
        if (!ok) break;
        if (tr) q4_trace(a, 4, 9, eseq);
        tc_fence_after();
        float v[64];
        {
          float lo[32], hi[32];
          tmem_ld32(tmem + lane_off + C::D_COL0 + ds * C::D_COLS, lo);
          tmem_ld32(tmem + lane_off + C::D_COL0 + ds * C::D_COLS + 32, hi);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = lo[i];
            v[32 + i] = hi[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&dempty_bar[ds]));
        if (tr) q4_trace(a, 4, 10, eseq);
        if (++ds == C::ND) {
          ds = 0;
          dph ^= 1;
        }
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          if (gi < ng) {
#pragma unroll
            for (int t = 0; t < TCAP; ++t) {
              const float xs = __shfl_sync(0xffffffffu, v[gi * 16 + t], 31);
              acc[t] = fmaf(sc[gi], v[gi * 16 + t], fmaf(bq[gi], xs, acc[t]));
            }
          }
        }
        if (tr) q4_trace(a, 4, 11, eseq++);
      }
      if (!ok) break;
      if (J.splits == 1) {
        if (valid) {
          const float bias = J.bias ? __ldg(J.bias + orow) : 0.f;
#pragma unroll
          for (int t = 0; t < TCAP; ++t)
            if (t < o.T) q4_store(o, t, orow, acc[t] + bias);
        }
      } else {
        float *slot = a.ws + ((J.ws_base + (int64_t)ui.tile_lin * J.splits + ui.sidx) * 128 + m) * 16;
#pragma unroll
        for (int t = 0; t < TCAP; ++t) __stcg(slot + t, acc[t]);
        __threadfence();
        __syncwarp();
        int prev = 0;
        int *cnt = a.cnt + (int64_t)(J.cnt_base + ui.tile_lin) * 4 + quarter;
        if (lane == 0) prev = atomicAdd(cnt, 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == J.splits - 1) {
          __threadfence();
          const float *s0 = a.ws + ((J.ws_base + (int64_t)ui.tile_lin * J.splits) * 128 + m) * 16;
          float sum[TCAP];
#pragma unroll
          for (int t = 0; t < TCAP; ++t) sum[t] = __ldcg(s0 + t);
          for (int j = 1; j < J.splits; ++j) {
            const float *sj = s0 + (int64_t)j * 128 * 16;
#pragma unroll
            for (int t = 0; t < TCAP; ++t) sum[t] += __ldcg(sj + t);
          }
          if (valid) {
            const float bias = J.bias ? __ldg(J.bias + orow) : 0.f;
#pragma unroll
            for (int t = 0; t < TCAP; ++t)
              if (t < o.T) q4_store(o, t, orow, sum[t] + bias);
          }
          __syncwarp();
          if (lane == 0) *cnt = 0;  // ready for the next call
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int TCAP>
int q4_decode_launch(Q4Args &args, int sms, cudaStream_t s) {
  auto kern = q4_decode_kernel<TCAP>;
  constexpr int smem = DecCfg::STAGES * DecCfg::STAGE_BYTES + 1024;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(q4 decode)");
    attr_done[dev & 63] = true;
  }
  const int grid = args.total_units < sms ? args.total_units : sms;
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kQThreads), smem, s, args);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "q4_decode_kernel launch");
}

std::mutex g_q4_mu;

bool al16(const void *p) { return ((uintptr_t)p & 15) == 0; }

template <bool DECODE>
int q4_launch_cfg(Q4Args &args, int sms, cudaStream_t s) {
  using C = Q4Cfg<DECODE>;
  auto kern = q4_umma_kernel<DECODE>;
  constexpr int smem = C::STAGES * (C::CODES_BYTES + C::X_BYTES) + 1024;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(q4)");
    attr_done[dev & 63] = true;
  }
  const int grid = args.total_units < sms ? args.total_units : sms;
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kQThreads), smem, s, args);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "q4_umma_kernel launch");
}

// Chunks per part for the decode split: minimize waves x groups per unit.
int choose_chunks(const Problem &p, int tiles_total_parts, int groups, int sms) {
  int best = 1;
  double best_cost = 1e300;
  for (int c = 1; c <= 8 && c <= groups; ++c) {
    const int cg = ((groups + c - 1) / c + 3) / 4 * 4;
    const int nch = (groups + cg - 1) / cg;
    if (nch != c && c > 1) continue;
    const long units = (long)tiles_total_parts * nch;
    const double waves = (double)((units + sms - 1) / sms);
    const double cost = waves * (cg + 2.0) + (nch > 1 ? 1.0 : 0.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = c;
    }
  }
  (void)p;
  return best;
}

// Builds the launch of `p` and runs it.  `get_ws(bytes, ncounters, &ws, &cnt)`
// supplies the split-reduction workspace when the launch needs one.
template <class WsFn>
int launch_q4_impl(const Problem &p, cudaStream_t s, bool *handled, WsFn get_ws, size_t ws_cap) {
  *handled = false;
  if (p.in_dt != TP_BF16) return TP_OK;
  int64_t maxT = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    if (J.M > maxT) maxT = J.M;
    if (J.N > INT32_MAX / 2 || J.M > INT32_MAX / 2) return TP_OK;
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      if (!al16(P.A) || (P.lda % 8) || !al16(P.B) || (P.ldb % 4) || (P.K % 64)) return TP_OK;
    }
  }
  // One or two tokens: the CUDA-core GEMV (HBM-bound; the tensor-core decode
  // below is bound by its MMA issue rate there).  TP_POLICY_SINGLE_SM keeps
  // the tensor-core decode.
  GvWorkspaceFn thunk = [](void *ctx, size_t bytes, size_t ncnt, float **ws, int **cnt) -> int {
    return (*static_cast<WsFn *>(ctx))(bytes, ncnt, ws, cnt);
  };
  if (maxT <= 2 && pair_policy_allowed()) {
    int rc = launch_q4_gemv(p, s, handled, thunk, &get_ws);
    if (rc != TP_OK || *handled) return rc;
  }
  // Up to 16 tokens: the 8-bit tensor-core decode (k_q4dec.cu) where its
  // shape rules hold, else the 16-bit one below.
  if (maxT <= 16) {
    int rc = launch_q4_dec8(p, s, handled, thunk, &get_ws, ws_cap);
    if (rc != TP_OK || *handled) return rc;
  }
  const bool decode = maxT <= 16;
  const int ROWS = decode ? 124 : 128;
  const int BN = decode ? 16 : 256;
  const int GS = decode ? 4 : 1;

  std::lock_guard<std::mutex> lk(g_q4_mu);
  const int sms = sm_count();
  static Q4Args args;
  memset(&args, 0, sizeof(args));

  // split choice (decode): the same number of chunks for every part
  int64_t tiles_parts = 0;
  int groups_max = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    const int tiles = (int)((J.N + ROWS - 1) / ROWS);
    tiles_parts += (int64_t)tiles * J.nparts;
    for (int q = 0; q < J.nparts; ++q) {
      const int g = (int)(p.parts[J.part0 + q].K / 64);
      if (g > groups_max) groups_max = g;
    }
  }
  const int c = decode ? choose_chunks(p, (int)tiles_parts, groups_max, sms) : 1;

  const void *cptr[kMaxParts], *xptr[kMaxParts];
  int64_t xK[kMaxParts], xlda[kMaxParts], xT[kMaxParts];
  int ncm = 0, nxm = 0;
  int64_t units = 0, slots = 0;
  int counters = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    Q4Job &Q = args.jobs[j];
    Q.C = J.C;
    Q.bias = J.bias;
    Q.ldc = J.ldc;
    Q.rows = (int)J.N;
    Q.T = (int)J.M;
    Q.part0 = J.part0;
    Q.nparts = J.nparts;
    Q.tiles = (Q.rows + ROWS - 1) / ROWS;
    Q.ntiles = decode ? 1 : (Q.T + BN - 1) / BN;
    int splits = 0;
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      Q4Part &QP = args.parts[J.part0 + q];
      QP.sc = (const uint16_t *)P.scales;
      QP.qb = (const uint16_t *)P.qbias;
      QP.groups = (int)(P.K / 64);
      int cg = (QP.groups + c - 1) / c;
      cg = (cg + GS - 1) / GS * GS;
      if (cg > QP.groups) cg = QP.groups;
      QP.chunk_groups = cg;
      QP.nchunk = (QP.groups + cg - 1) / cg;
      splits += QP.nchunk;
      int ic = -1, ix = -1;
      for (int i = 0; i < ncm; ++i)
        if (cptr[i] == P.B) ic = i;
      for (int i = 0; i < nxm; ++i)
        if (xptr[i] == P.A && xK[i] == P.K && xlda[i] == P.lda && xT[i] == J.M) ix = i;
      int rc;
      if (ic < 0) {
        rc = make_tmap_2d(&args.cmaps[ncm], P.B, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, (uint64_t)(P.K / 8),
                          (uint64_t)Q.rows, (uint64_t)P.ldb, (uint32_t)(GS * 8), (uint32_t)ROWS,
                          decode ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc) return rc;
        cptr[ncm] = P.B;
        ic = ncm++;
      }
      if (ix < 0) {
        // prefill: the map is made over the pre-pass's f16 copy, once the workspace is known
        if (decode) {
          rc = make_tmap_2d(&args.xmaps[nxm], P.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)P.K,
                            (uint64_t)Q.T, (uint64_t)P.lda, 64, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B);
          if (rc) return rc;
        }
        xptr[nxm] = P.A;
        xK[nxm] = P.K;
        xlda[nxm] = P.lda;
        xT[nxm] = J.M;
        ix = nxm++;
      }
      QP.cmap = (int16_t)ic;
      QP.xmap = (int16_t)ix;
    }
    Q.splits = splits;
    Q.unit_begin = (int)units;
    Q.cnt_base = counters;
    Q.ws_base = slots;
    const int64_t tl = (int64_t)Q.tiles * Q.ntiles;
    units += tl * splits;
    if (splits > 1) {
      slots += tl * splits;
      counters += (int)tl;
    }
  }
  if (units == 0) {
    *handled = true;
    return TP_OK;
  }
  if (units > INT32_MAX) return TP_OK;
  // workspace: split partial slots, then (prefill) each x region's f16 copy and factors
  const size_t slot_bytes = (size_t)slots * 128 * BN * sizeof(float);
  size_t prep_off[kMaxParts], prep_bytes = 0;
  if (!decode)
    for (int r = 0; r < nxm; ++r) {
      prep_off[r] = slot_bytes + prep_bytes;
      prep_bytes += ((size_t)xT[r] * xK[r] * 2 + (size_t)xT[r] * 4 + 255) / 256 * 256;
    }
  static XsArgs xa;
  memset(&xa, 0, sizeof(xa));
  int xs_rows = 0;
  if (slot_bytes + prep_bytes > 0) {
    int rc = get_ws(slot_bytes + prep_bytes, (size_t)counters * 4, &args.ws, &args.cnt);
    if (rc) return rc;
  }
  if (!decode) {
    uint8_t *wsb = reinterpret_cast<uint8_t *>(args.ws);
    for (int r = 0; r < nxm; ++r) {
      XsRegion &R = xa.r[r];
      R.x = static_cast<const uint16_t *>(xptr[r]);
      R.lda = xlda[r];
      R.K = (int)xK[r];
      R.xs = reinterpret_cast<uint16_t *>(wsb + prep_off[r]);
      R.fac = reinterpret_cast<float *>(wsb + prep_off[r] + (size_t)xT[r] * xK[r] * 2);
      R.row_begin = xs_rows;
      xs_rows += (int)xT[r];
      args.xfac[r] = R.fac;
      int rc = make_tmap_2d(&args.xmaps[r], R.xs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)xK[r],
                            (uint64_t)xT[r], (uint64_t)xK[r], 64, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc) return rc;
    }
    xa.nregions = nxm;
  }
  args.njobs = p.njobs;
  args.total_units = (int)units;
  args.ncm = ncm;
  args.nxm = nxm;
  args.out_dt = p.out_dt;
  // decode: exact integer codes and x in bf16; prefill: f16 values and f16 x
  args.idesc = umma_idesc_f16(decode ? 1u : 0u, 0u, 128u, (uint32_t)BN);
  args.status = p.status;
  args.wait_ns = (uint64_t)p.wait_ns;
  trace_buffer(&args.trace, &args.trace_cap);
  int sbv = 1;
  for (int j = 0; j < p.njobs; ++j)
    for (int q = 0; q < p.jobs[j].nparts; ++q) {
      const Q4Part &QP = args.parts[p.jobs[j].part0 + q];
      if ((QP.groups % 4) || ((uintptr_t)QP.sc & 7) || ((uintptr_t)QP.qb & 7)) sbv = 0;
    }
  args.sb_vec = sbv;
  int rc;
  if (!decode) {
    rc = TP_OK;
    if (xs_rows > 0) {
      cudaError_t e = launch_pdl(q4_xs_prep_kernel, dim3((unsigned)xs_rows), dim3(256), 0, s, xa);
      note_launch();
      if (e == cudaSuccess) e = cudaGetLastError();
      if (e != cudaSuccess) rc = cuda_error(e, "q4_xs_prep_kernel launch");
    }
    if (rc == TP_OK) rc = q4_launch_cfg<false>(args, sms, s);
    if (rc == TP_OK && slots > 0) {  // ordered sums of the split tiles
      SplitJob sj[kMaxJobs];
      for (int j = 0; j < p.njobs; ++j) {
        const Q4Job &Q = args.jobs[j];
        sj[j] = SplitJob{Q.C, Q.bias, Q.ldc, Q.ws_base, Q.rows, Q.T, Q.tiles, Q.ntiles, Q.splits};
      }
      rc = launch_split_reduce(sj, p.njobs, args.ws, BN, p.out_dt, s);
    }
  }
  else if (maxT <= 1)
    rc = q4_decode_launch<1>(args, sms, s);
  else if (maxT <= 4)
    rc = q4_decode_launch<4>(args, sms, s);
  else
    rc = q4_decode_launch<16>(args, sms, s);
  if (rc == TP_OK) *handled = true;
  return rc;
}

}  // namespace

int launch_q4(const Problem &p, cudaStream_t s, bool *handled) {
  return launch_q4_impl(
      p, s, handled,
      [s](size_t bytes, size_t ncnt, float **ws, int **cnt) -> int { return split_workspace(s, bytes, ncnt, ws, cnt); },
      SIZE_MAX);
}

int launch_q4_fixed_workspace(const Problem &p, cudaStream_t s, bool *handled, float *ws,
                              size_t ws_bytes, int *cnt, size_t ncnt_max) {
  return launch_q4_impl(p, s, handled, [&](size_t bytes, size_t ncnt, float **w, int **c) -> int {
    if (bytes > ws_bytes || ncnt > ncnt_max)
      return set_error(TP_ERR_UNSUPPORTED,
                       "this call needs %zu bytes of split scratch and %zu counters; the fixed "
                       "buffer holds %zu bytes and %zu counters",
                       bytes, ncnt, ws_bytes, ncnt_max);
    cudaError_t e = cudaMemsetAsync(cnt, 0, ncnt * sizeof(int), s);
    if (e != cudaSuccess) return cuda_error(e, "clearing the split counters");
    *w = ws;
    *c = cnt;
    return TP_OK;
  }, ws_bytes);
}

}  // namespace tp
