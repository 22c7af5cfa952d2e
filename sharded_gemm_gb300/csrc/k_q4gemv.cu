// k_q4gemv.cu -- 4-bit affine quantized linears on the CUDA cores for decode
// batches of one or two tokens.
//
// What it computes (the quantized variants of the column- and row-parallel
// linears, group size 64): for output row o of a shard and token t,
//   p_q[t][o] = sum over groups g of
//                 s[o][g] * sum_{k in g} code(o, k) * x_q[t][k]
//               + b[o][g] * sum_{k in g} x_q[t][k]
// which is sum_k (s*code + b) * x, the dequantized weight times x, regrouped.
// A column-parallel shard has one part; a row-parallel job has one part per
// rank, and its output is ((p_0 + p_1) + ...) + bias, the partials added in
// ascending rank order, each partial a float32 sum formed from zero.
//
// Why CUDA cores: at one or two tokens every weight is used once or twice, so
// the path is bound by HBM (0.5625 bytes per weight: the 4-bit code plus the
// float16 scale and bias of its group).  A 128-row tensor-core MMA takes
// about as long for 16 tokens as for one, and at one token its issue rate,
// not HBM, sets the pace; here the per-weight work is a quarter of a logic
// operation and half an integer dot-product instruction per token, well under
// the SM's issue rate at full HBM bandwidth.
//
// Integer decode.  Element k of a 32-bit code word sits at bits 4(k%8).  One
// AND with 0x0F0F0F0F leaves the even elements (0, 2, 4, 6) as four bytes,
// one AND with 0xF0F0F0F0 the odd ones (1, 3, 5, 7) times 16, so a word
// costs two logic operations and no shifts.  x is staged once per CTA as
// 16-bit integers: each 64-element group is scaled by 2^(14-emax) (emax =
// exponent of the group's largest |x|) and rounded to the nearest integer,
// so |x_int| < 2^15 and every element within 2^7 of the group's largest keeps
// all eight bits of its bfloat16 significand (smaller ones lose at most half
// a unit of 2^(emax-14)).  Four two-way integer dot products (dp2a: two
// 16-bit x times two code bytes, added to a 32-bit sum) take a word's eight
// products; the even and the odd sums of a group are exact integers, joined
// as 16*even + odd = 16 * sum(code * x_int) (|.| < 2^29), and the group's
// epilogue adds s * that * 2^(emax-18) + b * sum(x) to a float32 sum.  All
// sums run in a fixed order and no atomics touch the values, so repeated runs
// are bit-identical.
//
// Work split.  A warp task is kGvRows output rows of one part; in a step lane
// l takes group 32v+l of those rows (32 bytes of codes per row, a warp
// covering 1 KB of each row), so the scale, bias and exponent epilogue runs
// once per 64 weights; the lanes' sums meet in a warp-shuffle tree.  A
// row-parallel job's parts are separate tasks: each writes its partial to a
// workspace slot and the warp that finishes a row block's last part (an
// arrival counter) adds the slots in part order, adds the bias, stores, and
// resets the counter.
//
// Two kernels share that arithmetic.  The TMA-fed one (the default) gives each
// CTA one x block ("region": the x of one rank of a row-parallel job, or the x
// the column-parallel shards share) and each warp a ring of shared-memory
// slots that its lane 0 fills a few steps ahead with three 2-D tensor copies
// (codes, scales, biases of kGvRows rows x 32 groups), so the bytes in flight
// do not depend on registers.  The load-fed one takes what the tensor copies
// cannot (K not a multiple of 512, bases not 16-byte aligned, more than 32
// parts): each warp keeps its next step's code loads in flight in registers.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include <mutex>

#include "ptx.cuh"
#include "tp_internal.h"

namespace tp {
namespace {

constexpr int kGvRows = 4;  // output rows per warp task

struct GvJob {
  void *C;
  const float *bias;
  int64_t ldc;
  int rows, part0, nparts, nblocks, unit_begin, cnt_base;
  int64_t ws_base;  // first workspace float of this job (row-parallel)
};

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ldg_u16(const uint16_t *p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ldcg_f(const float *p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float bf16_to_f(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }
__device__ __forceinline__ float f16_to_f(uint16_t v) { return __half2float(__ushort_as_half(v)); }
__device__ __forceinline__ uint4 lds_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
// the same at base + OFF (an immediate offset: no address arithmetic)
template <int OFF>
__device__ __forceinline__ uint4 lds_u4_at(uint32_t base) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(base), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint16_t lds_u16_at(uint32_t base) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1+%2];" : "=h"(v) : "r"(base), "n"(OFF));
  return v;
}
__device__ __forceinline__ float lds_f(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint16_t lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
// 2^e as a float, for -126 <= e <= 127
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// Two-way dot products: c + a.lo16 * b.byte[0] + a.hi16 * b.byte[1] (LO) or
// with bytes 2 and 3 (HI); a holds two signed 16-bit x, b four unsigned code
// bytes.
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Staged x layout.  Per token, a block of 32*Gp 32-bit words (Gp = groups
// rounded up to 32; 128 bytes a group): word m = 0..7 of group g (elements
// 8m..8m+7) is one 16-byte chunk at byte ((g>>5)*8 + m)*512 + (g&31)*16, so
// the 32 lanes of a warp reading chunk m of 32 consecutive groups read 512
// contiguous bytes.  A chunk holds the integer x as four pairs of 16-bit
// halves, (x0, x2), (x4, x6), (x1, x3), (x5, x7) (x_j = element 8m+j): the
// even pairs meet the code bytes of (word & 0x0F0F0F0F), the odd pairs those
// of (word & 0xF0F0F0F0).  Then, per token, three arrays of Gp floats: the
// group's plain sum over its 64 bfloat16 elements in ascending order, and
// ra, rb with ra*rb = 2^(emax-18), each in float range.
__device__ __forceinline__ uint32_t chunk_byte(int g, int m) {
  return (uint32_t)((((g >> 5) * 8 + m) * 32 + (g & 31)) * 16);
}
__device__ __forceinline__ uint32_t pack16(int lo, int hi) {
  return ((uint32_t)lo & 0xFFFFu) | ((uint32_t)hi << 16);
}

// The whole CTA stages x: bfloat16 (T, 64*G), row stride lda.  Four
// threads share a group (two words, 16 elements, each); the group's sum adds
// the four quarter sums in order.  Scaling by 2^(14-emax) takes two exact
// multiplies by powers of two (the exponent reaches 147).
// xdst, sums: per-token strides xstride, sstride in 32-bit words.
__device__ __forceinline__ void stage_x(const uint16_t *x, int64_t lda, int G, int T, uint32_t *xdst, int xstride,
                                        float *sums, int sstride) {
  const int n = 4 * G * T;
  const int n_up = (n + 31) & ~31;  // whole warps take part in the shuffles
  for (int e = threadIdx.x; e < n_up; e += blockDim.x) {
    const bool live = e < n;
    const int ee = live ? e : n - 1;
    const int qd = ee & 3, gt = ee >> 2;
    const int tk = gt / G, g = gt % G;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + tk * lda + 64 * (int64_t)g + 16 * qd);
    float v[16];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 r = src[c];
      const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        v[8 * c + 2 * m] = bf16_to_f((uint16_t)(wv[m] & 0xFFFFu));
        v[8 * c + 2 * m + 1] = bf16_to_f((uint16_t)(wv[m] >> 16));
      }
    }
    float sum = 0.f, mx = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      sum += v[m];
      mx = fmaxf(mx, fabsf(v[m]));
    }
    // the four quarters of a group are lanes 4k..4k+3 of this warp
    const float s1 = __shfl_down_sync(0xffffffffu, sum, 1), s2 = __shfl_down_sync(0xffffffffu, sum, 2),
                s3 = __shfl_down_sync(0xffffffffu, sum, 3);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (!live) continue;
    // emax = floor(log2(mx)) for a normal mx (-127 bounds a subnormal one)
    const int emax = mx == 0.f ? 0 : (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127;
    const int t = 14 - emax;  // in [-113, 141]
    const float sa = pow2f(t < 127 ? t : 127), sb = pow2f(t < 127 ? 0 : t - 127);
    int xi[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) xi[m] = __float2int_rn(v[m] * sa * sb);
    uint32_t *dst = xdst + tk * xstride;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int *q = xi + 8 * c;
      *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(dst) + chunk_byte(g, 2 * qd + c)) =
          make_uint4(pack16(q[0], q[2]), pack16(q[4], q[6]), pack16(q[1], q[3]), pack16(q[5], q[7]));
    }
    if (qd == 0) {
      const int e18 = emax - 18;  // in [-145, 109]
      float *sbk = sums + tk * 3 * sstride;
      sbk[g] = ((sum + s1) + s2) + s3;
      sbk[sstride + g] = pow2f(e18 >> 1);
      sbk[2 * sstride + g] = pow2f(e18 - (e18 >> 1));
    }
  }
}

// acc[i][t] += this lane's group g of rows i (code words cw[i][0..1], eight
// words as two uint4; scale and bias s[i], b[i]) against token t's staged x.
// xs, sums: shared-memory addresses of the staged block; strides in 32-bit
// words.
template <int TT>
__device__ __forceinline__ void group_dot(const uint4 (&cw)[kGvRows][2], const float (&s)[kGvRows],
                                          const float (&b)[kGvRows], int g, uint32_t xs, int xstride,
                                          uint32_t sums, int sstride, float (&acc)[kGvRows][TT]) {
  const uint32_t xg = xs + chunk_byte(g, 0);  // chunk m of group g is at xg + 512 m
#pragma unroll
  for (int tk = 0; tk < TT; ++tk) {
    const uint32_t xt = xg + 4u * tk * xstride;
    int ev[kGvRows], od[kGvRows];
#pragma unroll
    for (int i = 0; i < kGvRows; ++i) ev[i] = od[i] = 0;
    uint4 X[8];
    X[0] = lds_u4_at<0 * 512>(xt);
    X[1] = lds_u4_at<1 * 512>(xt);
    X[2] = lds_u4_at<2 * 512>(xt);
    X[3] = lds_u4_at<3 * 512>(xt);
    X[4] = lds_u4_at<4 * 512>(xt);
    X[5] = lds_u4_at<5 * 512>(xt);
    X[6] = lds_u4_at<6 * 512>(xt);
    X[7] = lds_u4_at<7 * 512>(xt);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
#pragma unroll
      for (int i = 0; i < kGvRows; ++i) {
        const uint4 &c4 = cw[i][m >> 2];
        const uint32_t w = (m & 3) == 0 ? c4.x : (m & 3) == 1 ? c4.y : (m & 3) == 2 ? c4.z : c4.w;
        const uint32_t e = w & 0x0F0F0F0Fu, o = w & 0xF0F0F0F0u;
        ev[i] = dp2a_lo(X[m].x, e, ev[i]);
        ev[i] = dp2a_hi(X[m].y, e, ev[i]);
        od[i] = dp2a_lo(X[m].z, o, od[i]);
        od[i] = dp2a_hi(X[m].w, o, od[i]);
      }
    }
    const uint32_t sb = sums + 4u * (tk * 3 * sstride + g);
    const float Xs = lds_f(sb), ra = lds_f(sb + 4u * sstride), rb = lds_f(sb + 8u * sstride);
#pragma unroll
    for (int i = 0; i < kGvRows; ++i) {
      const float D = (float)(16 * ev[i] + od[i]);  // 16 * sum(code * x_int), exact below 2^24
      acc[i][tk] = fmaf(s[i] * ra, D * rb, acc[i][tk]);
      acc[i][tk] = fmaf(b[i], Xs, acc[i][tk]);
    }
  }
}

__device__ __forceinline__ void store_out(void *C, int out_dt, int64_t idx, float v) {
  if (out_dt == TP_F32)
    static_cast<float *>(C)[idx] = v;
  else if (out_dt == TP_BF16)
    static_cast<__nv_bfloat16 *>(C)[idx] = __float2bfloat16_rn(v);
  else
    static_cast<__half *>(C)[idx] = __float2half_rn(v);
}

// Output k (row k/TT, token k%TT) of row block b of job J: its partial slots
// 0..nparts-1 added in part order (loads issued eight at a time, ahead of the
// adds), plus the bias, stored.
template <int TT>
__device__ __forceinline__ void reduce_one(const GvJob &J, int b, int k, int out_dt, const float *ws) {
  const float *slots = ws + J.ws_base + (int64_t)b * J.nparts * (kGvRows * TT) + k;
  const int o = b * kGvRows + k / TT;
  if (o >= J.rows) return;
  float r = 0.f;
  for (int q0 = 0; q0 < J.nparts; q0 += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = q0 + u < J.nparts ? ldcg_f(slots + (q0 + u) * (kGvRows * TT)) : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (q0 + u < J.nparts) r = q0 + u == 0 ? v[u] : r + v[u];
  }
  if (J.bias) r += J.bias[o];
  store_out(J.C, out_dt, (int64_t)(k % TT) * J.ldc + o, r);
}

// The warp reduces row block b of job J (lanes 0..kGvRows*TT-1) and resets its
// counter.
template <int TT>
__device__ __forceinline__ void reduce_parts(const GvJob &J, int b, int lane, int out_dt, const float *ws,
                                             int *cnt) {
  if (lane < kGvRows * TT) reduce_one<TT>(J, b, lane, out_dt, ws);
  if (lane == 0) cnt[J.cnt_base + b] = 0;
}

// Warp-sums the lanes' accumulators for rows b*kGvRows.. of job J, part
// index qi within the job, then stores (one part) or writes the partial's slot
// and, unless DEFER (the caller then runs the arrivals later), runs the
// arrival and the ordered cross-part reduction; clears the accumulators.
template <int TT, bool DEFER>
__device__ __forceinline__ void finish_rows(const GvJob &J, int qi, int b, int lane, int out_dt, float *ws,
                                            int *cnt, float (&acc)[kGvRows][TT]) {
#pragma unroll
  for (int i = 0; i < kGvRows; ++i)
#pragma unroll
    for (int tk = 0; tk < TT; ++tk) {
      float v = acc[i][tk];
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
      acc[i][tk] = v;  // every lane now holds the same total
    }
  // lane k < kGvRows*TT owns (row i, token tk) = (k / TT, k % TT)
  float mine = 0.f;
#pragma unroll
  for (int i = 0; i < kGvRows; ++i)
#pragma unroll
    for (int tk = 0; tk < TT; ++tk)
      if (lane == i * TT + tk) mine = acc[i][tk];
  const int i_me = lane / TT, tk_me = lane % TT;
  const int o = b * kGvRows + i_me;
  const bool owner = lane < kGvRows * TT && o < J.rows;
  if (J.nparts == 1) {
    if (owner) {
      const float r = J.bias ? mine + J.bias[o] : mine;
      store_out(J.C, out_dt, (int64_t)tk_me * J.ldc + o, r);
    }
  } else {
    float *slots = ws + J.ws_base + (int64_t)b * J.nparts * (kGvRows * TT);
    if (lane < kGvRows * TT) slots[qi * (kGvRows * TT) + lane] = mine;
    if (!DEFER) {
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(cnt + J.cnt_base + b, 1) == J.nparts - 1;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        reduce_parts<TT>(J, b, lane, out_dt, ws, cnt);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kGvRows; ++i)
#pragma unroll
    for (int tk = 0; tk < TT; ++tk) acc[i][tk] = 0.f;
}

// ====================================================== load-fed kernel
constexpr int kGvWarps = 8;  // warps per CTA (one CTA per SM)
constexpr int kGvSmemMax = 220 * 1024;

struct GvPart {
  const uint4 *codes;       // (rows, K/32) in 16-byte units
  const uint16_t *sc, *qb;  // float16 (rows, G)
  int64_t ld4;              // code row stride in 16-byte units
  int G;                    // groups (K/64)
  int xoff, soff;           // float offsets of this part's x block and sums
  int xstride, sstride;     // per-token strides of the two
};

struct GvX {  // one distinct x block to stage
  const uint16_t *x;  // bfloat16 (T, K), row stride lda
  int64_t lda;
  int G;
  int xoff, soff, xstride, sstride;
};

struct GvArgs {
  GvJob jobs[kMaxJobs];
  GvPart parts[kMaxParts];
  GvX xs[kMaxParts];
  int njobs, nx, total_units, out_dt, T;
  float *ws;
  int *cnt;
};

// One warp task: rows b*kGvRows .. +kGvRows-1 of job j, part q.
struct Task {
  int u;  // unit id, or -1 past the end
  int j, q, b;
};

__device__ __forceinline__ void task_at(const GvArgs &a, int u, Task &t) {
  t.u = u < a.total_units ? u : -1;
  if (t.u < 0) return;
  int j = 0;
  while (j + 1 < a.njobs && a.jobs[j + 1].unit_begin <= u) ++j;
  const GvJob &J = a.jobs[j];
  const int local = u - J.unit_begin;
  t.j = j;
  t.b = local / J.nparts;
  t.q = J.part0 + local % J.nparts;
}

__device__ __forceinline__ int nsteps(const GvArgs &a, const Task &t) { return (a.parts[t.q].G + 31) / 32; }

struct Buf {
  uint4 c[kGvRows][2];
  uint16_t s[kGvRows], b[kGvRows];
};

__device__ __forceinline__ void load_step(const GvArgs &a, const Task &t, int v, int lane, Buf &B) {
  const GvPart &P = a.parts[t.q];
  const int rows = a.jobs[t.j].rows, o0 = t.b * kGvRows;
  const int g = v * 32 + lane;
#pragma unroll
  for (int i = 0; i < kGvRows; ++i) {
    const int o = o0 + i;
    if (g < P.G && o < rows) {
      const uint4 *row = P.codes + (int64_t)o * P.ld4 + 2 * g;
      B.c[i][0] = ldg_stream(row);
      B.c[i][1] = ldg_stream(row + 1);
      B.s[i] = ldg_u16(P.sc + (int64_t)o * P.G + g);
      B.b[i] = ldg_u16(P.qb + (int64_t)o * P.G + g);
    } else {
      B.c[i][0] = B.c[i][1] = make_uint4(0u, 0u, 0u, 0u);
      B.s[i] = B.b[i] = 0;
    }
  }
}

template <int TT>
__device__ __forceinline__ void compute_step(const GvArgs &a, const Task &t, int v, int lane, const Buf &B,
                                             const float *xsm, float (&acc)[kGvRows][TT]) {
  const GvPart &P = a.parts[t.q];
  const int g = v * 32 + lane;
  if (g >= P.G) return;
  float s[kGvRows], b[kGvRows];
#pragma unroll
  for (int i = 0; i < kGvRows; ++i) {
    s[i] = f16_to_f(B.s[i]);
    b[i] = f16_to_f(B.b[i]);
  }
  group_dot<TT>(B.c, s, b, g, smem_u32(xsm + P.xoff), P.xstride, smem_u32(xsm + P.soff), P.sstride, acc);
}

__device__ __forceinline__ void advance(const GvArgs &a, const Task &cur, int v, int W, Task &nt, int &nv) {
  if (v + 1 < nsteps(a, cur)) {
    nt = cur;
    nv = v + 1;
  } else {
    task_at(a, cur.u + W, nt);
    nv = 0;
  }
}

template <int TT>
__global__ void __launch_bounds__(kGvWarps * 32, 1) q4_gemv_kernel(const __grid_constant__ GvArgs a) {
  griddep_launch_dependents();
  griddep_wait();  // programmatic launch: no global memory before the previous kernel completes
  extern __shared__ __align__(16) float xsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int W = gridDim.x * kGvWarps;

  // The first step's code loads go out before x is staged.
  Task tA, tB;
  int vA = 0, vB = 0;
  Buf bA, bB;
  task_at(a, blockIdx.x * kGvWarps + warp, tA);
  if (tA.u >= 0) load_step(a, tA, 0, lane, bA);
  for (int xi = 0; xi < a.nx; ++xi) {
    const GvX &X = a.xs[xi];
    stage_x(X.x, X.lda, X.G, a.T, reinterpret_cast<uint32_t *>(xsm + X.xoff), X.xstride, xsm + X.soff, X.sstride);
  }
  __syncthreads();

  float acc[kGvRows][TT];
#pragma unroll
  for (int i = 0; i < kGvRows; ++i)
#pragma unroll
    for (int tk = 0; tk < TT; ++tk) acc[i][tk] = 0.f;

  // Ping-pong over steps: the loads of the next step are issued before the
  // current step is computed, except when the current step ends a task whose
  // partial goes through the cross-part reduction: its memory fence would
  // wait for those loads, so they go out after it (their latency is then
  // exposed once per such task; the other warps cover it).
  while (tA.u >= 0) {
    advance(a, tA, vA, W, tB, vB);
    const bool endA = vA + 1 == nsteps(a, tA);
    const bool lateA = endA && a.jobs[tA.j].nparts > 1;
    if (tB.u >= 0 && !lateA) load_step(a, tB, vB, lane, bB);
    compute_step<TT>(a, tA, vA, lane, bA, xsm, acc);
    if (endA) finish_rows<TT, false>(a.jobs[tA.j], tA.q - a.jobs[tA.j].part0, tA.b, lane, a.out_dt, a.ws, a.cnt, acc);
    if (tB.u < 0) break;
    if (lateA) load_step(a, tB, vB, lane, bB);
    advance(a, tB, vB, W, tA, vA);
    const bool endB = vB + 1 == nsteps(a, tB);
    const bool lateB = endB && a.jobs[tB.j].nparts > 1;
    if (tA.u >= 0 && !lateB) load_step(a, tA, vA, lane, bA);
    compute_step<TT>(a, tB, vB, lane, bB, xsm, acc);
    if (endB) finish_rows<TT, false>(a.jobs[tB.j], tB.q - a.jobs[tB.j].part0, tB.b, lane, a.out_dt, a.ws, a.cnt, acc);
    if (tA.u >= 0 && lateB) load_step(a, tA, vA, lane, bA);
  }
}

// ====================================================== TMA-fed kernel
constexpr int kGtWarps = 16;
constexpr int kGtGroups = 32;                           // groups per step
constexpr int kGtCodeBytes = kGvRows * kGtGroups * 32;  // 4096
constexpr int kGtSbBytes = kGvRows * kGtGroups * 2;     // 256 (scales; again biases)
constexpr int kGtSlot = kGtCodeBytes + 2 * kGtSbBytes;  // 4608, a multiple of 128
static_assert(kGvRows == 4 && kGtGroups == 32, "the slot reads below are written out for 4 rows x 32 groups");
constexpr int kGtMaxParts = 32;
constexpr int kGtSmemMax = 227 * 1024;

struct GtPart {
  int G, job;
};
struct GtRPart {  // a part served by a region
  int q, unit_begin;
};
struct GtRegion {
  const uint16_t *x;
  int64_t lda;
  int G, xstride, sstride;  // x block: groups, per-token strides (32-bit words)
  int rp_begin, rp_count, units;
  int cta_begin, cta_count;
};
// MP: the largest part, job and region count the launch holds (8 or 32); the
// kernel's parameter block grows with it (128 bytes of tensor maps per part and
// operand), and a smaller block starts sooner.
template <int MP>
struct GtArgs {
  CUtensorMap maps[3 * MP];  // per part: codes, scales, biases
  GvJob jobs[MP];
  GtPart parts[MP];
  GtRPart rparts[MP];
  GtRegion regions[MP];
  int nregions, out_dt, T, stages;
  float *ws;
  int *cnt;
  int *status;
  uint64_t wait_ns;
};

struct GtCur {
  int u, v, ns, q, b;
};

template <int MP>
__device__ __forceinline__ void gt_set(const GtArgs<MP> &a, const GtRegion &R, int u, GtCur &c) {
  c.u = u < R.units ? u : -1;
  c.v = 0;
  if (c.u < 0) return;
  int r = R.rp_begin;
  while (r + 1 < R.rp_begin + R.rp_count && a.rparts[r + 1].unit_begin <= u) ++r;
  c.q = a.rparts[r].q;
  c.b = u - a.rparts[r].unit_begin;
  c.ns = (a.parts[c.q].G + kGtGroups - 1) / kGtGroups;
}

template <int MP>
__device__ __forceinline__ void gt_next(const GtArgs<MP> &a, const GtRegion &R, int Wr, GtCur &c) {
  if (++c.v < c.ns) return;
  gt_set(a, R, c.u + Wr, c);
}

// lane 0: the three tensor copies of step c into slot `dst` (barrier `bar`)
template <int MP>
__device__ __forceinline__ void gt_issue(const GtArgs<MP> &a, const GtCur &c, uint32_t dst, uint32_t bar) {
  mbar_arrive_expect_tx(bar, kGtSlot);
  const int y = c.b * kGvRows;
  tma_load_2d(dst, &a.maps[3 * c.q], bar, c.v * kGtGroups * 8, y);
  tma_load_2d(dst + kGtCodeBytes, &a.maps[3 * c.q + 1], bar, c.v * kGtGroups, y);
  tma_load_2d(dst + kGtCodeBytes + kGtSbBytes, &a.maps[3 * c.q + 2], bar, c.v * kGtGroups, y);
}

// L2 prefetch of step c's three tiles (no shared memory, no barrier)
template <int MP>
__device__ __forceinline__ void gt_prefetch(const GtArgs<MP> &a, const GtCur &c) {
  const int y = c.b * kGvRows;
  tma_prefetch_l2_2d(&a.maps[3 * c.q], c.v * kGtGroups * 8, y);
  tma_prefetch_l2_2d(&a.maps[3 * c.q + 1], c.v * kGtGroups, y);
  tma_prefetch_l2_2d(&a.maps[3 * c.q + 2], c.v * kGtGroups, y);
}

template <int TT, int MP>
__global__ void __launch_bounds__(kGtWarps * 32, 1) q4_gemv_tma_kernel(const __grid_constant__ GtArgs<MP> a) {
  griddep_launch_dependents();
  extern __shared__ __align__(1024) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = a.stages;
  int ri = 0;
  while (ri + 1 < a.nregions && (int)blockIdx.x >= a.regions[ri].cta_begin + a.regions[ri].cta_count) ++ri;
  const GtRegion &R = a.regions[ri];
  const int Wr = R.cta_count * kGtWarps;
  const int gw = ((int)blockIdx.x - R.cta_begin) * kGtWarps + warp;
  // Before the programmatic-launch wait: L2 prefetches of this warp's first
  // steps.  Weights are not outputs of the previous kernel, and L2 is the
  // point of coherence, so the tensor copies issued after the wait still see
  // any line that kernel writes; the prefetches only start the DRAM reads.
  if (lane == 0) {
    GtCur pc;
    gt_set(a, R, gw, pc);
    for (int k = 0; k < S && pc.u >= 0; ++k) {
      gt_prefetch(a, pc);
      gt_next(a, R, Wr, pc);
    }
  }
  griddep_wait();  // programmatic launch: no global loads before the previous kernel completes

  unsigned char *ring = smem + (size_t)warp * S * kGtSlot;
  const uint32_t bars = smem_u32(smem + (size_t)kGtWarps * S * kGtSlot) + warp * S * 8;
  float *xs = reinterpret_cast<float *>(smem + (size_t)kGtWarps * S * kGtSlot + kGtWarps * S * 8);
  float *sums = xs + TT * R.xstride;
  const uint32_t ring_s = smem_u32(ring), xs_s = smem_u32(xs), sums_s = smem_u32(sums);

  if (lane == 0) {
    for (int k = 0; k < S; ++k) mbar_init(bars + 8 * k, 1);
    fence_mbar_init();
  }
  __syncwarp();

  GtCur ci, cc;
  gt_set(a, R, gw, ci);
  cc = ci;
  // issue and compute cursors walk the same steps; slot indices and the
  // compute phase advance incrementally (S is a launch parameter)
  int ki = 0, si = 0;
  // prologue: the first S-1 steps go out before x is staged
  for (; ki < S - 1 && ci.u >= 0; ++ki) {
    if (lane == 0) gt_issue(a, ci, ring_s + si * kGtSlot, bars + 8 * si);
    si = si + 1 == S ? 0 : si + 1;
    gt_next(a, R, Wr, ci);
  }

  stage_x(R.x, R.lda, R.G, TT, reinterpret_cast<uint32_t *>(xs), R.xstride, sums, R.sstride);
  __syncthreads();

  float acc[kGvRows][TT];
#pragma unroll
  for (int i = 0; i < kGvRows; ++i)
#pragma unroll
    for (int tk = 0; tk < TT; ++tk) acc[i][tk] = 0.f;

  int kc = 0, slot = 0;
  uint32_t phase = 0;
  bool ok = true;
  while (cc.u >= 0) {
    // refill the slot the previous step freed
    if (ci.u >= 0) {
      if (lane == 0) gt_issue(a, ci, ring_s + si * kGtSlot, bars + 8 * si);
      si = si + 1 == S ? 0 : si + 1;
      gt_next(a, R, Wr, ci);
      ++ki;
    }
    ok = mbar_wait(bars + 8 * slot, phase, a.wait_ns, a.status, nullptr);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const int G = a.parts[cc.q].G;
    const int g = cc.v * kGtGroups + lane;
    if (g < G) {
      const uint32_t sl = ring_s + slot * kGtSlot;
      // row i of the slot: 32 groups x 32 code bytes at i * 1024, then the
      // scales (64 bytes a row) and the biases
      uint4 cw[kGvRows][2];
      float s[kGvRows], b[kGvRows];
      const uint32_t cb = sl + lane * 32, sbb = sl + kGtCodeBytes + 2 * lane;
      cw[0][0] = lds_u4_at<0>(cb);
      cw[0][1] = lds_u4_at<16>(cb);
      cw[1][0] = lds_u4_at<1024>(cb);
      cw[1][1] = lds_u4_at<1040>(cb);
      cw[2][0] = lds_u4_at<2048>(cb);
      cw[2][1] = lds_u4_at<2064>(cb);
      cw[3][0] = lds_u4_at<3072>(cb);
      cw[3][1] = lds_u4_at<3088>(cb);
      s[0] = f16_to_f(lds_u16_at<0>(sbb));
      s[1] = f16_to_f(lds_u16_at<64>(sbb));
      s[2] = f16_to_f(lds_u16_at<128>(sbb));
      s[3] = f16_to_f(lds_u16_at<192>(sbb));
      b[0] = f16_to_f(lds_u16_at<kGtSbBytes>(sbb));
      b[1] = f16_to_f(lds_u16_at<kGtSbBytes + 64>(sbb));
      b[2] = f16_to_f(lds_u16_at<kGtSbBytes + 128>(sbb));
      b[3] = f16_to_f(lds_u16_at<kGtSbBytes + 192>(sbb));
      group_dot<TT>(cw, s, b, g, xs_s, R.xstride, sums_s, R.sstride, acc);
    }
    if (cc.v + 1 == cc.ns) {
      const GvJob &J = a.jobs[a.parts[cc.q].job];
      finish_rows<TT, true>(J, cc.q - J.part0, cc.b, lane, a.out_dt, a.ws, a.cnt, acc);
    }
    __syncwarp();
    gt_next(a, R, Wr, cc);
    ++kc;
    if (++slot == S) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (!ok) {
    // a wait ran out: let the copies already issued land (bounded) before
    // the CTA's shared memory goes away
    for (int k = kc; k < ki; ++k) mbar_wait(bars + 8 * (k % S), (k / S) & 1, a.wait_ns, nullptr, nullptr);
    return;
  }
  // Arrivals of this warp's row-parallel partials, one fence for all of
  // them; lane l takes the warp's task base+l.  The last arrival of a row
  // block sums its slots in part order.
  __threadfence();
  for (int base = 0;; base += 32) {
    const int u = gw + (base + lane) * Wr;
    int last = 0, jj = 0, bb = 0;
    if (u < R.units) {
      GtCur c;
      gt_set(a, R, u, c);
      jj = a.parts[c.q].job;
      bb = c.b;
      const GvJob &J = a.jobs[jj];
      if (J.nparts > 1) last = atomicAdd(a.cnt + J.cnt_base + c.b, 1) == J.nparts - 1;
    }
    unsigned m = __ballot_sync(0xffffffffu, last);
    if (m) __threadfence();
    // up to 32/(kGvRows*TT) row blocks at a time, lanes split by (block, output)
    constexpr int kPer = kGvRows * TT, kAtOnce = 32 / kPer;
    while (m) {
      int src = -1;
      unsigned mm = m;
      for (int t = 0; t < kAtOnce && mm; ++t) {
        const int l = __ffs(mm) - 1;
        mm &= mm - 1;
        if (lane / kPer == t) src = l;
      }
      m = mm;
      const int jl = __shfl_sync(0xffffffffu, jj, src < 0 ? 0 : src);
      const int bl = __shfl_sync(0xffffffffu, bb, src < 0 ? 0 : src);
      if (src >= 0) {
        const GvJob &J = a.jobs[jl];
        reduce_one<TT>(J, bl, lane % kPer, a.out_dt, a.ws);
        if (lane % kPer == 0) a.cnt[J.cnt_base + bl] = 0;
      }
    }
    if (!__any_sync(0xffffffffu, gw + (base + 32) * Wr < R.units)) break;
  }
}

// ====================================================== host
std::mutex g_gv_mu;

bool al16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// Staged-x 32-bit words for K = 64*G and T tokens: the integer x block (two
// 16-bit values a word) and the three per-group float arrays; sets the
// per-token strides.
int64_t stage_floats(int G, int T, int *xstride, int *sstride) {
  const int gp = (G + 31) / 32 * 32;
  *xstride = gp * 32;
  *sstride = gp;
  return (int64_t)T * ((int64_t)gp * 32 + 3 * (int64_t)gp);
}

template <typename K, typename A>
int launch_one(K kern, const A &args, int grid, int threads, size_t smem, int smem_max, bool *attr_done,
               cudaStream_t s, const char *what) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (e != cudaSuccess) return cuda_error(e, what);
    attr_done[dev & 63] = true;
  }
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(threads), smem, s, args);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, what);
}

// The TMA-fed launch; leaves *handled false for problems it does not take.
template <int MP>
int launch_gemv_tma(const Problem &p, int T, cudaStream_t s, bool *handled, GvWorkspaceFn get_ws, void *ctx) {
  int nparts = 0;  // one past the highest part index in use
  for (int j = 0; j < p.njobs; ++j)
    if (p.jobs[j].part0 + p.jobs[j].nparts > nparts) nparts = p.jobs[j].part0 + p.jobs[j].nparts;
  if (nparts > MP || p.njobs > MP) return TP_OK;
  for (int j = 0; j < p.njobs; ++j)
    for (int q = 0; q < p.jobs[j].nparts; ++q) {
      const Part &P = p.parts[p.jobs[j].part0 + q];
      if ((P.K % 512) || !al16(P.B) || !al16(P.scales) || !al16(P.qbias) || (P.ldb % 4) || !al16(P.A) ||
          (P.lda % 8))
        return TP_OK;
    }
  static GtArgs<MP> args;
  memset(&args, 0, sizeof(args));
  // regions: distinct (x, K, lda)
  int reg_of[kMaxParts];
  for (int i = 0; i < kMaxParts; ++i) reg_of[i] = -1;
  int nreg = 0;
  int64_t xfloats = 0;
  for (int j = 0; j < p.njobs; ++j)
    for (int q = 0; q < p.jobs[j].nparts; ++q) {
      const int qq = p.jobs[j].part0 + q;
      const Part &P = p.parts[qq];
      const int G = (int)(P.K / 64);
      int r = -1;
      for (int i = 0; i < nreg; ++i)
        if (args.regions[i].x == P.A && args.regions[i].G == G && args.regions[i].lda == P.lda) r = i;
      if (r < 0) {
        r = nreg++;
        GtRegion &R = args.regions[r];
        R.x = static_cast<const uint16_t *>(P.A);
        R.lda = P.lda;
        R.G = G;
        const int64_t f = stage_floats(G, T, &R.xstride, &R.sstride);
        if (f > xfloats) xfloats = f;
      }
      reg_of[qq] = r;
    }
  const int sms = sm_count();
  if (nreg > sms) return TP_OK;
  const int64_t per_stage = (int64_t)kGtWarps * (kGtSlot + 8);
  int S = (int)((kGtSmemMax - xfloats * 4) / per_stage);
  if (S > 4) S = 4;
  if (S < 2) return TP_OK;

  // jobs, parts, maps, workspace layout
  int64_t ws_floats = 0;
  int counters = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    GvJob &GJ = args.jobs[j];
    GJ.C = J.C;
    GJ.bias = J.bias;
    GJ.ldc = J.ldc;
    GJ.rows = (int)J.N;
    GJ.part0 = J.part0;
    GJ.nparts = J.nparts;
    GJ.nblocks = (GJ.rows + kGvRows - 1) / kGvRows;
    if (J.nparts > 1) {
      GJ.cnt_base = counters;
      GJ.ws_base = ws_floats;
      counters += GJ.nblocks;
      ws_floats += (int64_t)GJ.nblocks * J.nparts * kGvRows * T;
    }
    for (int q = 0; q < J.nparts; ++q) {
      const int qq = J.part0 + q;
      const Part &P = p.parts[qq];
      GtPart &GP = args.parts[qq];
      GP.G = (int)(P.K / 64);
      GP.job = j;
      int rc = make_tmap_2d(&args.maps[3 * qq], P.B, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, (uint64_t)(P.K / 8),
                            (uint64_t)J.N, (uint64_t)P.ldb, kGtGroups * 8, kGvRows, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (!rc)
        rc = make_tmap_2d(&args.maps[3 * qq + 1], P.scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)GP.G,
                          (uint64_t)J.N, (uint64_t)GP.G, kGtGroups, kGvRows, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (!rc)
        rc = make_tmap_2d(&args.maps[3 * qq + 2], P.qbias, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)GP.G,
                          (uint64_t)J.N, (uint64_t)GP.G, kGtGroups, kGvRows, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (rc) return rc;
    }
  }
  // each region's parts, in part order, and its units (row blocks)
  int nrp = 0;
  double work[kMaxParts];
  int64_t total_units = 0;
  for (int r = 0; r < nreg; ++r) {
    GtRegion &R = args.regions[r];
    R.rp_begin = nrp;
    int units = 0;
    for (int qq = 0; qq < nparts; ++qq)
      if (reg_of[qq] == r) {
        args.rparts[nrp].q = qq;
        args.rparts[nrp].unit_begin = units;
        units += args.jobs[args.parts[qq].job].nblocks;
        ++nrp;
      }
    R.rp_count = nrp - R.rp_begin;
    R.units = units;
    work[r] = (double)units * R.G;
    total_units += units;
  }
  if (total_units == 0) {
    *handled = true;
    return TP_OK;
  }
  // CTAs per region in proportion to its work: at least one, at most one
  // warp per unit
  double wsum = 0;
  for (int r = 0; r < nreg; ++r) wsum += work[r];
  int given = 0, cap[kMaxParts], cnt[kMaxParts];
  for (int r = 0; r < nreg; ++r) {
    cap[r] = (args.regions[r].units + kGtWarps - 1) / kGtWarps;
    if (cap[r] < 1) cap[r] = 1;
    cnt[r] = (int)(sms * work[r] / wsum);
    if (cnt[r] < 1) cnt[r] = 1;
    if (cnt[r] > cap[r]) cnt[r] = cap[r];
    given += cnt[r];
  }
  while (given > sms) {  // one CTA each can overshoot
    int best = -1;
    for (int r = 0; r < nreg; ++r)
      if (cnt[r] > 1 && (best < 0 || work[r] / cnt[r] < work[best] / cnt[best])) best = r;
    if (best < 0) return TP_OK;
    --cnt[best];
    --given;
  }
  while (given < sms) {
    int best = -1;
    for (int r = 0; r < nreg; ++r)
      if (cnt[r] < cap[r] && (best < 0 || work[r] / cnt[r] > work[best] / cnt[best])) best = r;
    if (best < 0) break;
    ++cnt[best];
    ++given;
  }
  int cta = 0;
  for (int r = 0; r < nreg; ++r) {
    args.regions[r].cta_begin = cta;
    args.regions[r].cta_count = cnt[r];
    cta += cnt[r];
  }
  args.nregions = nreg;
  args.out_dt = p.out_dt;
  args.T = T;
  args.stages = S;
  args.status = p.status;
  args.wait_ns = (uint64_t)p.wait_ns;
  if (counters > 0) {
    int rc = get_ws(ctx, (size_t)ws_floats * sizeof(float), (size_t)counters, &args.ws, &args.cnt);
    if (rc) return rc;
  }
  const size_t smem = (size_t)(per_stage * S + xfloats * 4);
  static bool done1[64] = {false}, done2[64] = {false};
  const int rc = T == 1 ? launch_one(q4_gemv_tma_kernel<1, MP>, args, cta, kGtWarps * 32, smem, kGtSmemMax, done1, s,
                                     "q4_gemv_tma_kernel")
                        : launch_one(q4_gemv_tma_kernel<2, MP>, args, cta, kGtWarps * 32, smem, kGtSmemMax, done2, s,
                                     "q4_gemv_tma_kernel");
  if (rc == TP_OK) *handled = true;
  return rc;
}

// The load-fed launch; leaves *handled false if x does not fit.
int launch_gemv_ldg(const Problem &p, int T, cudaStream_t s, bool *handled, GvWorkspaceFn get_ws, void *ctx) {
  static GvArgs args;
  memset(&args, 0, sizeof(args));
  const void *xptr[kMaxParts];
  int nx = 0;
  int64_t floats = 0;
  int64_t units = 0, ws_floats = 0;
  int counters = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    GvJob &GJ = args.jobs[j];
    GJ.C = J.C;
    GJ.bias = J.bias;
    GJ.ldc = J.ldc;
    GJ.rows = (int)J.N;
    GJ.part0 = J.part0;
    GJ.nparts = J.nparts;
    GJ.nblocks = (GJ.rows + kGvRows - 1) / kGvRows;
    GJ.unit_begin = (int)units;
    units += (int64_t)GJ.nblocks * J.nparts;
    if (J.nparts > 1) {
      GJ.cnt_base = counters;
      GJ.ws_base = ws_floats;
      counters += GJ.nblocks;
      ws_floats += (int64_t)GJ.nblocks * J.nparts * kGvRows * T;
    }
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      GvPart &GP = args.parts[J.part0 + q];
      GP.codes = static_cast<const uint4 *>(P.B);
      GP.sc = static_cast<const uint16_t *>(P.scales);
      GP.qb = static_cast<const uint16_t *>(P.qbias);
      GP.ld4 = P.ldb / 4;
      GP.G = (int)(P.K / 64);
      int xi = -1;
      for (int i = 0; i < nx; ++i)
        if (xptr[i] == P.A && args.xs[i].G == GP.G && args.xs[i].lda == P.lda) xi = i;
      if (xi < 0) {
        GvX &X = args.xs[nx];
        X.x = static_cast<const uint16_t *>(P.A);
        X.lda = P.lda;
        X.G = GP.G;
        X.xoff = (int)floats;
        const int64_t f = stage_floats(X.G, T, &X.xstride, &X.sstride);
        X.soff = (int)(floats + (int64_t)T * X.xstride);
        floats += f;
        if (floats * 4 > kGvSmemMax) return TP_OK;  // x does not fit: tensor-core decode
        xptr[nx] = P.A;
        xi = nx++;
      }
      GP.xoff = args.xs[xi].xoff;
      GP.soff = args.xs[xi].soff;
      GP.xstride = args.xs[xi].xstride;
      GP.sstride = args.xs[xi].sstride;
    }
  }
  if (units == 0) {
    *handled = true;
    return TP_OK;
  }
  if (units > INT32_MAX) return TP_OK;
  args.njobs = p.njobs;
  args.nx = nx;
  args.total_units = (int)units;
  args.out_dt = p.out_dt;
  args.T = T;
  if (counters > 0) {
    int rc = get_ws(ctx, (size_t)ws_floats * sizeof(float), (size_t)counters, &args.ws, &args.cnt);
    if (rc) return rc;
  }
  const int sms = sm_count();
  const int64_t need = (units + kGvWarps - 1) / kGvWarps;
  const int grid = (int)(need < sms ? need : sms);
  const size_t smem = (size_t)floats * 4;
  static bool done1[64] = {false}, done2[64] = {false};
  const int rc = T == 1 ? launch_one(q4_gemv_kernel<1>, args, grid, kGvWarps * 32, smem, kGvSmemMax, done1, s,
                                     "q4_gemv_kernel")
                        : launch_one(q4_gemv_kernel<2>, args, grid, kGvWarps * 32, smem, kGvSmemMax, done2, s,
                                     "q4_gemv_kernel");
  if (rc == TP_OK) *handled = true;
  return rc;
}

}  // namespace

int launch_q4_gemv(const Problem &p, cudaStream_t s, bool *handled, GvWorkspaceFn get_ws, void *ctx) {
  *handled = false;
  if (p.in_dt != TP_BF16 || p.b_layout != BL_Q4 || p.njobs < 1) return TP_OK;
  const int64_t T = p.jobs[0].M;
  if (T < 1 || T > 2) return TP_OK;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    if (J.M != T || J.N > INT32_MAX / 2 || J.nparts < 1) return TP_OK;
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      if (!al16(P.A) || (P.lda % 8) || !al16(P.B) || (P.ldb % 4) || (P.K % 64) || P.K > INT32_MAX / 2)
        return TP_OK;
    }
  }
  std::lock_guard<std::mutex> lk(g_gv_mu);
  int nparts = 0;
  for (int j = 0; j < p.njobs; ++j)
    if (p.jobs[j].part0 + p.jobs[j].nparts > nparts) nparts = p.jobs[j].part0 + p.jobs[j].nparts;
  int rc = nparts <= 8 && p.njobs <= 8 ? launch_gemv_tma<8>(p, (int)T, s, handled, get_ws, ctx)
                                       : launch_gemv_tma<kGtMaxParts>(p, (int)T, s, handled, get_ws, ctx);
  if (rc != TP_OK || *handled) return rc;
  return launch_gemv_ldg(p, (int)T, s, handled, get_ws, ctx);
}

}  // namespace tp
