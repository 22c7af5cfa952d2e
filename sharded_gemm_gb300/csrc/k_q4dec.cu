// k_q4dec.cu -- the 4-bit affine (group 64) linears for decode batches of up
// to 16 tokens on the tensor cores, with 8-bit operands.
//
// What it computes (the quantized column- and row-parallel linears): for
// output row o and token t,
//   y[t][o] = sum over parts p, groups g of
//               s[o][g] * sum_{k in g} code(o, k) * x_p[t][k]
//             + b[o][g] * sum_{k in g} x_p[t][k]
// then the bias.  The groups of all parts, laid end to end in ascending part
// (rank) order, are cut into consecutive ranges of whole stages; each range
// is summed in float32 from zero, across part boundaries too, and the range
// sums are added in range order.  The order is fixed by the shapes alone.
//
// Exact 8-bit operands.  A 4-bit code c, zero-extended to a byte, reads as an
// FP8 E4M3 number equal to c * 2^-9 for every c in 0..15 (c < 8: a subnormal
// c/8 * 2^-6; c >= 8: exponent field 1, (1 + (c-8)/8) * 2^-6).  So a code
// word expands to the MMA's A operand with two masks and a shift:
// (w & 0x0F0F0F0F) holds elements 0, 2, 4, 6 of the word and
// ((w >> 4) & 0x0F0F0F0F) elements 1, 3, 5, 7, as bytes.  The activations
// take the same order along K inside every block of eight (a dot product
// does not depend on the order of its terms).  A pre-pass scales each
// 64-element group of x by a power of two 2^c (its largest |x| lands in
// [128, 256)) and writes it as two E4M3 terms, hi = e4m3(x 2^c) and
// lo = e4m3(x 2^c - hi); every bfloat16 x within 2^9 of the group's largest
// is exactly hi + lo (4 + 4 significant bits cover its 8), smaller ones are
// off by at most 2^-10 of the scaled unit.  hi and lo are the B operand's
// rows t and TP + t.  One MMA group (two tcgen05.mma kind::f8f6f4, K = 32
// each) leaves D_g[o][t] = 2^(c-9) sum code * hi and the same for lo in its
// own TMEM accumulator; the epilogue adds
//   (s[o][g] * 2^(9-c)) * (D_hi + D_lo) + b[o][g] * X_g[t]
// to a float32 sum (X_g: the group's plain sum of x, from the pre-pass).
// Every product is exact; the per-group sums of 64 terms run in the tensor
// core's accumulator and the groups are added in float32 in a fixed order.
//
// Roles (one CTA per SM, persistent over units = (tile of 128 output rows,
// range of stages)).  The pre-pass runs inside this kernel: at the start the
// epilogue warps of every CTA write their share of the prepared activations
// and count themselves done on a launch-wide counter; once it is full (or,
// after a short wait, once this CTA has prepared every item itself) the
// activation stream starts.  The codes stream starts at once with its first
// stage.  Warp 0 issues the tensor copy of a stage's packed
// codes (8 groups) into the codes ring; warp 10 the stage's activation tile,
// scales, biases and per-group factors into the operand ring.  Warps 2-5
// expand a stage's codes into one of two halves of the A operand in TMEM
// (tcgen05.st, one wait per stage), so the next stage is expanded while the
// MMAs read this one.  Warp 1 issues the stage's 16 MMAs (A from TMEM, B
// from shared memory) into 4 accumulator slots of two groups each, with 6
// barrier waits and 3 commits per stage (one per half-stage, one for the
// stage): per-group handshakes cost more than the MMAs they guard.  Warps 6-9 load a slot's accumulators while the
// previous slot's are applied and release it.  At a unit's end a unit that
// covers its whole job stores y; otherwise the epilogue warps store its
// float32 partial to the unit's workspace slot and go on, and a second
// launch (the ordered split sum shared with the prefill kernels) adds each
// tile's slots in range order, then the bias.  A CTA-local ordered sum was
// measured first and dropped: one SM pulling a tile's 14 slots (112 KB)
// from L2 while HBM streams at full rate took 10-20 us per tile, and the
// CTAs doing it fell behind the rest by as much.
// Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "ptx.cuh"
#include "tp_internal.h"

namespace tp {
namespace {

constexpr int kD8Threads = 11 * 32;  // 2 producers, MMA, 4 converter warps, 4 epilogue warps
constexpr int kD8GroupsPerStage = 8;
// Units are dispensed at run time: a CTA's first unit is its block index,
// later ones come from a global counter, so SMs that stream faster take more
// units (measured: CTAs of the same launch finishing equal work at times
// 1.7x apart).  The codes producer takes each unit and passes its index to
// the other roles through a ring in shared memory.
constexpr int kUnitRing = 4;
constexpr int kUnitReaders = 1 + 1 + 4 + 4;  // operand producer, MMA, converters, epilogue
// Codes stages a CTA issues before the prepared activations are ready: the
// first stage's DRAM latency then overlaps the pre-pass, and the pre-pass's
// reads of x still meet short DRAM queues.
constexpr int kD8PreStages = 1;
// How long a CTA waits for the other CTAs' shares of the pre-pass before it
// prepares every item itself (identical values, so the duplicate writes are
// harmless).  The launch does not require all CTAs to be resident together.
constexpr uint64_t kD8PrepAloneNs = 30000;

template <int TP>
struct D8Cfg {
  static constexpr int N = 2 * TP;                    // B rows: TP hi, TP lo
  // Codes ring: a stage's packed codes (8 groups x 128 rows), released by the
  // converters as soon as they have read them, so the DRAM stream runs
  // stages ahead of the MMAs.
  static constexpr int CODES_BOX = 128 * 128;         // 4 groups x 128 rows, 128B-swizzled
  static constexpr int CODES_BYTES = 2 * CODES_BOX;
  static constexpr int CSTAGES = TP == 16 ? 5 : 4;
  // Operand ring: the stage's activation tile (released by the MMA's
  // commit) with its scales, biases and per-group factors and sums
  // (released by the epilogue, which reads them a few groups behind).
  static constexpr int B_BOX = N * 128;               // 2 groups of K (128 bytes) x N rows
  static constexpr int B_OFF = 0;
  static constexpr int S_OFF = 4 * B_BOX;             // scales, 128 rows x 8 groups f16
  static constexpr int Q_OFF = S_OFF + 2048;          // biases
  static constexpr int GX_OFF = Q_OFF + 2048;         // per group: TP factors, TP sums (f32)
  static constexpr int GX_BYTES = kD8GroupsPerStage * 2 * TP * 4;
  static constexpr int OP_BYTES = (GX_OFF + GX_BYTES + 1023) / 1024 * 1024;
  static constexpr int OP_TX = 4 * B_BOX + 4096 + GX_BYTES;
  static constexpr int OSTAGES = TP == 16 ? 3 : 6;
  static constexpr int A_COL0 = 0;                    // A: two halves of 128 columns (a stage's 8 groups each)
  static constexpr int D_COL0 = 256;                  // D: 4 pair slots of 2N columns (2 groups each)
  static constexpr int NDP = 4, DP_COLS = 2 * N;
  static constexpr int SMEM = CSTAGES * CODES_BYTES + OSTAGES * OP_BYTES + 1024;
  static_assert(B_BOX % 1024 == 0 && CODES_BYTES % 1024 == 0, "swizzled boxes on 1024-byte boundaries");
  static_assert(D_COL0 + NDP * DP_COLS <= 512, "TMEM columns");
  static_assert(SMEM <= 227 * 1024 - 1024, "shared memory (dynamic, leaving room for the static barriers)");
};

// A region of the activation pre-pass: one distinct activation block.
struct PrepRegion {
  const uint16_t *x;  // bfloat16 (T, K), row stride lda
  int64_t lda;
  uint8_t *xq;        // (2 TP, K) bytes
  float *gx;          // (groups, 2, TP)
  int K, groups, T, item_begin;
};
struct D8Part {
  int16_t cmap, smap, qmap, region;
  int groups;
  int st0;  // first stage of this part in its job's stages laid end to end
};

struct D8Job {
  void *C;
  const float *bias;
  int64_t ldc;
  int rows, T, part0, nparts, tiles;
  int nst;        // stages of all parts
  int range_len;  // stages per range (the last range may be shorter)
  int splits;     // ranges per tile
  int unit_begin;
  int64_t ws_base;  // first partial slot (slot = TP columns x 128 rows, column-major)
};

template <int MP>
struct D8Args {
  CUtensorMap cmaps[MP], smaps[MP], qmaps[MP];  // per part: codes, scales, biases
  CUtensorMap xmaps[MP];                        // per region: prepared activations
  D8Job jobs[MP];
  D8Part parts[MP];
  const float *gx[MP];                          // per region: [groups][2][TP] floats
  PrepRegion prep[MP];                          // per region: the pre-pass's input and outputs
  int nprep, prep_items;
  uint64_t prep_alone_ns;  // wait for the other CTAs' shares at most this long (0: not at all)
  int njobs, total_units, out_dt;
  uint32_t idesc;
  float *ws;
  int *work, *done;  // unit dispenser and finished-CTA count (zero between launches)
  int *prepped;      // CTAs done with their share of the pre-pass (zero between launches)
  int *status;
  uint64_t wait_ns;
  unsigned long long *trace;  // optional role timeline of CTA 0 (tp_set_trace)
};

// Records the time of (event, stage sequence) when tracing CTA 0.
template <int MP>
__device__ __forceinline__ void d8_trace(const D8Args<MP> &a, int event, int seq) {
  if (a.trace != nullptr && blockIdx.x == 0 && seq < 1024) a.trace[16 + event * 1024 + seq] = globaltimer_ns();
}

struct D8Unit {
  int job, tile, sidx, s0, nst;  // stages s0 .. s0 + nst - 1 of tile `tile`
};

template <int MP>
__device__ __forceinline__ void d8_unit(const D8Args<MP> &a, int u, D8Unit &ui) {
  int j = 0;
  while (j + 1 < a.njobs && u >= a.jobs[j + 1].unit_begin) ++j;
  const D8Job &J = a.jobs[j];
  const int local = u - J.unit_begin;
  ui.job = j;
  ui.tile = local / J.splits;
  ui.sidx = local - ui.tile * J.splits;
  ui.s0 = ui.sidx * J.range_len;
  ui.nst = min(J.range_len, J.nst - ui.s0);
}

// The part holding stage s of job J, and the stage's first group in it.
template <int MP>
__device__ __forceinline__ int d8_stage_part(const D8Args<MP> &a, const D8Job &J, int s, int &gs) {
  int p = J.part0;
  while (p + 1 < J.part0 + J.nparts && s >= a.parts[p + 1].st0) ++p;
  gs = (s - a.parts[p].st0) * kD8GroupsPerStage;
  return p;
}

// ------------------------------------------------------------------ PTX
// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f8f6f4 (8-bit A and B, f32 D).
__device__ __forceinline__ void umma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from registers into TMEM.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 64 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}


// a = b * c + a on two float lanes at once (packed f32x2)
__device__ __forceinline__ void fma2(float &a0, float &a1, float b0, float b1, float c0, float c1) {
  asm("{\n .reg .b64 A, B, C;\n mov.b64 A, {%0, %1};\n mov.b64 B, {%2, %3};\n mov.b64 C, {%4, %5};\n"
      " fma.rn.f32x2 A, B, C, A;\n mov.b64 {%0, %1}, A;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float &a0, float &a1, float b0, float b1) {
  asm("{\n .reg .b64 A, B;\n mov.b64 A, {%0, %1};\n mov.b64 B, {%2, %3};\n"
      " add.rn.f32x2 A, A, B;\n mov.b64 {%0, %1}, A;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul2(float &a0, float &a1, float b0, float b1) {
  asm("{\n .reg .b64 A, B;\n mov.b64 A, {%0, %1};\n mov.b64 B, {%2, %3};\n"
      " mul.rn.f32x2 A, A, B;\n mov.b64 {%0, %1}, A;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// y[t][orow] of an output whose pointer and row stride the caller holds in
// registers (read through the kernel-parameter block, they would be reloaded
// after every store: the compiler cannot tell the output from the parameters).
__device__ __forceinline__ void d8_store(int out_dt, void *C, int64_t ldc, int t, int orow, float v) {
  const int64_t idx = (int64_t)t * ldc + orow;
  if (out_dt == TP_F32)
    static_cast<float *>(C)[idx] = v;
  else if (out_dt == TP_BF16)
    static_cast<uint16_t *>(C)[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  else
    static_cast<uint16_t *>(C)[idx] = __half_as_ushort(__float2half_rn(v));
}

#define D8_WAIT(bar, par, okvar)                                           \
  {                                                                        \
    const bool _r = mbar_wait((bar), (par), lim, a.status, &abort_sh);     \
    if (!__all_sync(0xffffffffu, _r)) okvar = false;                       \
  }

// The next unit index of a role (-1: no more), single-thread roles.
#define D8_NEXT_UNIT_1(u, okvar)                                                       \
  {                                                                                    \
    if (!mbar_wait(smem_u32(&ufull_bar[us]), uph, lim, a.status, &abort_sh)) {         \
      okvar = false;                                                                   \
      u = -1;                                                                          \
    } else {                                                                           \
      u = *(volatile int *)&unit_ring[us];                                             \
      mbar_arrive(smem_u32(&uempty_bar[us]));                                          \
    }                                                                                  \
    if (++us == kUnitRing) {                                                           \
      us = 0;                                                                          \
      uph ^= 1;                                                                        \
    }                                                                                  \
  }
// The same for a whole warp (one arrival per warp).
#define D8_NEXT_UNIT_W(u, okvar)                                                       \
  {                                                                                    \
    D8_WAIT(smem_u32(&ufull_bar[us]), uph, okvar);                                     \
    u = okvar ? *(volatile int *)&unit_ring[us] : -1;                                  \
    __syncwarp();                                                                      \
    if (okvar && lane == 0) mbar_arrive(smem_u32(&uempty_bar[us]));                    \
    if (++us == kUnitRing) {                                                           \
      us = 0;                                                                          \
      uph ^= 1;                                                                        \
    }                                                                                  \
  }

// ------------------------------------------------------------------ pre-pass
// One item per (region, token t < TP, group g): the group's 64 bfloat16 x
// scaled by 2^c, c = 7 - floor(log2 max|x|) (clamped so 2^(9-c) stays a
// normal float), written as E4M3 hi and lo terms into rows t and TP + t of
// the region's (2 TP, K) byte matrix in the K order of the expanded codes,
// and gx[g][0][t] = 2^(9-c), gx[g][1][t] = the group's plain ascending sum.
// Tokens T <= t < TP get zero rows and zero factors.  The decode kernel's
// CTAs share the items out at their start (see the kernel).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {  // lo -> byte 0, hi -> byte 1
  unsigned short d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ void e4m3x2_value(uint32_t v, float &lo, float &hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)v));
  lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
  hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

template <int TP, int MP>
__device__ __forceinline__ void d8_prep_item(const PrepRegion (&regs)[MP], int nregions, int item) {
  int ri = 0;
  while (ri + 1 < nregions && item >= regs[ri + 1].item_begin) ++ri;
  const PrepRegion &R = regs[ri];
  const int local = item - R.item_begin;
  const int t = local / R.groups, g = local - t * R.groups;
  uint32_t hiw[16], low[16];
  float fac = 0.f, sum = 0.f;
  if (t < R.T) {
    const uint4 *src = reinterpret_cast<const uint4 *>(R.x + (int64_t)t * R.lda + 64 * (int64_t)g);
    float v[64];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 w = src[c];
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        v[8 * c + 2 * m] = __uint_as_float(wv[m] << 16);
        v[8 * c + 2 * m + 1] = __uint_as_float(wv[m] & 0xFFFF0000u);
      }
    }
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < 64; ++k) {
      sum += v[k];
      mx = fmaxf(mx, fabsf(v[k]));
    }
    int e = mx == 0.f ? 0 : (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127;  // floor(log2 mx), normal mx
    e = e < -120 ? -120 : (e > 120 ? 120 : e);
    const int c = 7 - e;                                 // in [-113, 127]
    const float scale = __uint_as_float((uint32_t)(c + 127) << 23);
    fac = __uint_as_float((uint32_t)(2 + e + 127) << 23);  // 2^(9-c)
    // K order inside each block of eight: 0, 2, 4, 6, 1, 3, 5, 7
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      uint32_t hp[4], lp[4];  // byte pairs (element ord[2i], element ord[2i+1])
      constexpr int ord[8] = {0, 2, 4, 6, 1, 3, 5, 7};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float x0 = v[8 * m + ord[2 * i]] * scale, x1 = v[8 * m + ord[2 * i + 1]] * scale;
        const uint32_t h = e4m3x2(x0, x1);
        float h0, h1;
        e4m3x2_value(h, h0, h1);
        hp[i] = h;
        lp[i] = e4m3x2(x0 - h0, x1 - h1);
      }
      hiw[2 * m] = hp[0] | (hp[1] << 16);
      hiw[2 * m + 1] = hp[2] | (hp[3] << 16);
      low[2 * m] = lp[0] | (lp[1] << 16);
      low[2 * m + 1] = lp[2] | (lp[3] << 16);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) hiw[i] = low[i] = 0u;
  }
  uint4 *dh = reinterpret_cast<uint4 *>(R.xq + (int64_t)t * R.K + 64 * (int64_t)g);
  uint4 *dl = reinterpret_cast<uint4 *>(R.xq + (int64_t)(TP + t) * R.K + 64 * (int64_t)g);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dh[i] = make_uint4(hiw[4 * i], hiw[4 * i + 1], hiw[4 * i + 2], hiw[4 * i + 3]);
    dl[i] = make_uint4(low[4 * i], low[4 * i + 1], low[4 * i + 2], low[4 * i + 3]);
  }
  R.gx[((int64_t)g * 2) * TP + t] = fac;
  R.gx[((int64_t)g * 2 + 1) * TP + t] = sum;
}


// ------------------------------------------------------------------ kernel
template <int TP, int MP>
__global__ void __launch_bounds__(kD8Threads, 1) q4_dec8_kernel(const __grid_constant__ D8Args<MP> a) {
  griddep_launch_dependents();
  // when tracing: every CTA's start (event 30) and end (event 31) times
  if (a.trace != nullptr && threadIdx.x == 0 && blockIdx.x < 1024) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    a.trace[16 + 28 * 1024 + blockIdx.x] = smid + 1;
    a.trace[16 + 30 * 1024 + blockIdx.x] = globaltimer_ns();
  }
  using C = D8Cfg<TP>;
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t cfull_bar[C::CSTAGES], cempty_bar[C::CSTAGES];  // codes ring
  __shared__ __align__(8) uint64_t ofull_bar[C::OSTAGES], oempty_bar[C::OSTAGES];  // operand ring
  __shared__ __align__(8) uint64_t sdone_bar[C::OSTAGES];  // a stage's MMAs completed (A half, B tile free)
  __shared__ __align__(8) uint64_t afull_bar[2];                                   // A halves
  __shared__ __align__(8) uint64_t dfull_bar[2], dempty_bar[C::NDP];  // D: half-stage ready, pair slot free
  __shared__ __align__(8) uint64_t ufull_bar[kUnitRing], uempty_bar[kUnitRing];  // unit indices to every role
  __shared__ int unit_ring[kUnitRing];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t xready_bar;  // the prepared activations of every region are written
  __shared__ int prep_alone_sh;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t cbase = (smem_u32(dsmem) + 1023u) & ~1023u;  // codes ring
  const uint32_t obase = cbase + C::CSTAGES * C::CODES_BYTES;  // operand ring
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int i = 0; i < C::CSTAGES; ++i) {
      mbar_init(smem_u32(&cfull_bar[i]), 1);
      mbar_init(smem_u32(&cempty_bar[i]), 4);  // the 4 converter warps read it
    }
    for (int i = 0; i < C::OSTAGES; ++i) {
      mbar_init(smem_u32(&ofull_bar[i]), 1);
      mbar_init(smem_u32(&oempty_bar[i]), 4);  // the 4 epilogue warps read the scales, biases, factors
      mbar_init(smem_u32(&sdone_bar[i]), 1);   // the MMA's commit after the stage
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&afull_bar[i]), 4);  // the 4 converter warps
      mbar_init(smem_u32(&dfull_bar[i]), 1);  // the MMA's commit after pairs 2i, 2i+1
    }
    for (int i = 0; i < C::NDP; ++i) {
      mbar_init(smem_u32(&dempty_bar[i]), 4);  // the 4 epilogue warps
    }
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(smem_u32(&ufull_bar[i]), 1);              // the scheduler wrote the slot
      mbar_init(smem_u32(&uempty_bar[i]), kUnitReaders);  // every other role read it
    }
    mbar_init(smem_u32(&drain_bar), 1);
    mbar_init(smem_u32(&xready_bar), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();  // programmatic launch: no global loads before the previous kernel completes
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0 || warp == 10) {
    // ------------------------------------------------------------ producers
    // warp 0: the codes ring; warp 10: the operand ring.  Two threads, so a
    // full operand ring (the epilogue is behind) never holds back the codes.
    if (lane == 0) {
      const bool codes = warp == 0;
      const int NS = codes ? C::CSTAGES : C::OSTAGES;
      uint64_t *fullb = codes ? cfull_bar : ofull_bar;
      uint64_t *emptyb = codes ? cempty_bar : oempty_bar;
      int st = 0, seq = 0;
      uint32_t ph = 0;
      uint32_t usedmask = 0, lastph = 0;  // per stage: issued at least once, parity of its last fill
      bool ok = true;
      int us = 0;
      uint32_t uph = 0;
      int next = (int)blockIdx.x < a.total_units ? (int)blockIdx.x : -1;  // the codes producer's unit to publish
      bool prep_ok = false;
      while (ok) {
        int u;
        if (codes) {
          // scheduler: publish the unit to the other roles, then take the one after
          if (!mbar_wait(smem_u32(&uempty_bar[us]), uph ^ 1, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          unit_ring[us] = next;
          mbar_arrive(smem_u32(&ufull_bar[us]));
          if (++us == kUnitRing) {
            us = 0;
            uph ^= 1;
          }
          u = next;
          next = -2;  // taken while the unit's last stage is issued
        } else {
          D8_NEXT_UNIT_1(u, ok);
        }
        if (u < 0) break;
        D8Unit ui;
        d8_unit(a, u, ui);
        const D8Job &J = a.jobs[ui.job];
        for (int k = 0; k < ui.nst; ++k, ++seq) {
          int gs;
          const D8Part &P = a.parts[d8_stage_part(a, J, ui.s0 + k, gs)];
          const int y = ui.tile * 128;
          if (!mbar_wait(smem_u32(&emptyb[st]), ph ^ 1, lim, a.status, &abort_sh) ||
              (!codes && !mbar_wait(smem_u32(&sdone_bar[st]), ph ^ 1, lim, a.status, &abort_sh))) {
            ok = false;
            break;
          }
          // The codes stream issues its first stages before the prepared
          // activations are ready, then waits for them too.
          if (!prep_ok && codes && seq >= kD8PreStages) {
            if (!mbar_wait(smem_u32(&xready_bar), 0, lim, a.status, &abort_sh)) {
              ok = false;
              break;
            }
            fence_proxy_async_global();  // the tensor copies below read what other threads wrote
            prep_ok = true;
          }
          const uint32_t fb = smem_u32(&fullb[st]);
          if (codes) {
            const uint32_t base = cbase + st * C::CODES_BYTES;
            mbar_arrive_expect_tx(fb, C::CODES_BYTES);
            tma_load_3d(base, &a.cmaps[P.cmap], fb, 0, y, gs / 4);  // chunks gs/4, gs/4 + 1
            d8_trace(a, 1, seq);
            if (k == ui.nst - 1) {  // the next unit, a ring's depth before this one is done
              const int g = (int)gridDim.x + atomicAdd(a.work, 1);
              next = g < a.total_units ? g : -1;
            }
          } else {
            const uint32_t base = obase + st * C::OP_BYTES;
            mbar_arrive_expect_tx(fb, C::OP_TX);
            tma_load_2d(base + C::S_OFF, &a.smaps[P.smap], fb, gs, y);
            tma_load_2d(base + C::Q_OFF, &a.qmaps[P.qmap], fb, gs, y);
            if (!prep_ok) {  // the scales and biases above need no prepared activations
              if (!mbar_wait(smem_u32(&xready_bar), 0, lim, a.status, &abort_sh))
                ok = false;  // the copies below are still issued: the stage completes before teardown
              fence_proxy_async_global();  // the tensor copies below read what other threads wrote
              prep_ok = true;
            }
            tma_load_3d(base + C::B_OFF, &a.xmaps[P.region], fb, 0, 0, gs / 2);  // chunks gs/2 .. gs/2 + 3
            bulk_load(base + C::GX_OFF, a.gx[P.region] + (int64_t)gs * 2 * TP, C::GX_BYTES, fb);
          }
          usedmask |= 1u << st;
          lastph = (lastph & ~(1u << st)) | (ph << st);
          if (++st == NS) {
            st = 0;
            ph ^= 1;
          }
          if (!ok) break;
        }
      }
      if (!ok)  // let the copies in flight land before the CTA's memory goes away
        for (int i = 0; i < NS; ++i)
          if (usedmask & (1u << i)) mbar_wait(smem_u32(&fullb[i]), (lastph >> i) & 1u, lim, a.status, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One stage = A half h (8 groups in TMEM), the stage's activation tile,
    // and the 4 D pair slots: 6 barrier waits and 3 commits for 16 MMAs.
    if (lane == 0) {
      int os = 0, h = 0, seq = 0, us = 0;
      uint32_t oph = 0, hph = 0, dph = 0, uph = 0;
      bool ok = true;
      for (;;) {
        int u;
        D8_NEXT_UNIT_1(u, ok);
        if (u < 0) break;
        D8Unit ui;
        d8_unit(a, u, ui);
        for (int k = 0; ok && k < ui.nst; ++k, ++seq) {
          if (!mbar_wait(smem_u32(&ofull_bar[os]), oph, lim, a.status, &abort_sh) ||
              !mbar_wait(smem_u32(&afull_bar[h]), hph, lim, a.status, &abort_sh)) {
            ok = false;
            break;
          }
          d8_trace(a, 2, seq);
          tc_fence_after();
          const uint32_t base = obase + os * C::OP_BYTES;
          const uint32_t abase = tmem + C::A_COL0 + h * 128;
          // Per half-stage (pairs 2hp, 2hp+1: 4 accumulators), the 4 first K-steps
          // and then the 4 second ones, so that no MMA follows the one it adds to.
          for (int hp = 0; hp < 2; ++hp) {
            if (!mbar_wait(smem_u32(&dempty_bar[2 * hp]), dph ^ 1, lim, a.status, &abort_sh) ||
                !mbar_wait(smem_u32(&dempty_bar[2 * hp + 1]), dph ^ 1, lim, a.status, &abort_sh)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d8_trace(a, 17, seq * 4 + 2 * hp);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
              for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                for (int gg = 0; gg < 2; ++gg) {
                  const int p = 2 * hp + pp;
                  const uint32_t d = tmem + C::D_COL0 + p * C::DP_COLS + gg * C::N;
                  const uint32_t bb = base + C::B_OFF + p * C::B_BOX + gg * 64;
                  umma_f8_ts(d, abase + p * 32 + gg * 16 + kk * 8, umma_desc_sw128(bb + kk * 32, 16, 1024), a.idesc,
                             kk > 0 ? 1u : 0u);
                }
            umma_commit(smem_u32(&dfull_bar[hp]));
            d8_trace(a, 18, seq * 4 + 2 * hp);
          }
          if (!ok) break;
          umma_commit(smem_u32(&sdone_bar[os]));  // frees A half h and the stage's B tile
          d8_trace(a, 5, seq);
          dph ^= 1;
          if (++os == C::OSTAGES) {
            os = 0;
            oph ^= 1;
          }
          if (++h == 2) {
            h = 0;
            hph ^= 1;
          }
        }
        if (!ok) break;
      }
      umma_commit(smem_u32(&drain_bar));
      mbar_wait(smem_u32(&drain_bar), 0, lim, a.status, nullptr);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ converters
    // A stage's 8 groups go to A half h: all four slots' stores, one wait,
    // one arrival.  The halves alternate, so the next stage is expanded
    // while the MMAs read this one; the packed codes are released as soon
    // as they have been read.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // this thread's row of the tile = its TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int cs = 0, h = 0, seq = 0, us = 0;
    uint32_t cph = 0, uph = 0;
    bool ok = true;
    for (;;) {
      int u;
      D8_NEXT_UNIT_W(u, ok);
      if (u < 0) break;
      D8Unit ui;
      d8_unit(a, u, ui);
      for (int k = 0; ok && k < ui.nst; ++k, ++seq) {
        D8_WAIT(smem_u32(&cfull_bar[cs]), cph, ok);
        if (ok && seq >= 2) {  // A half h is free once the MMAs of stage seq - 2 completed
          const int ps = seq - 2;
          D8_WAIT(smem_u32(&sdone_bar[ps % C::OSTAGES]), (uint32_t)(ps / C::OSTAGES) & 1u, ok);
        }
        if (!ok) break;
        if (warp == 2 && lane == 0) d8_trace(a, 6, seq);
        tc_fence_after();
        const uint32_t base = cbase + cs * C::CODES_BYTES;
        uint32_t out[4][32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // slot j: groups 2j, 2j+1
          // row r's 64 code bytes of groups 2j, 2j+1: chunks 4(j%2)..+3 of its
          // 128-byte row in codes box j/2 (16-byte chunk c stored at c ^ (r%8))
          const uint32_t row = base + (j >> 1) * C::CODES_BOX + r * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = (j & 1) * 4 + i;
            const uint4 w = lds128(row + ((c ^ (r & 7)) << 4));
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              out[j][8 * i + 2 * m] = wv[m] & 0x0F0F0F0Fu;             // elements 0, 2, 4, 6
              out[j][8 * i + 2 * m + 1] = (wv[m] >> 4) & 0x0F0F0F0Fu;  // elements 1, 3, 5, 7
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&cempty_bar[cs]));  // the codes are in registers
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_st32(tmem + lane_off + C::A_COL0 + h * 128 + j * 32, out[j]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&afull_bar[h]));
        if (warp == 2 && lane == 0) d8_trace(a, 8, seq);
        if (++cs == C::CSTAGES) {
          cs = 0;
          cph ^= 1;
        }
        h ^= 1;
      }
      if (!ok) break;
    }
    tmem_wait_st();  // no store may still be in flight when the CTA tears down
  } else if (warp < 10) {
    // ------------------------------------------------------------ epilogue
    {
      // First this CTA's share of the activation pre-pass (a contiguous run
      // of items), one arrival on the launch-wide count, and a short wait
      // for the other CTAs' shares; a CTA that waits in vain (the others are
      // not resident) prepares every item itself.  Then the producers go.
      const int per = (a.prep_items + (int)gridDim.x - 1) / (int)gridDim.x;
      const int i0 = (int)blockIdx.x * per;
      const int i1 = min(a.prep_items, i0 + per);
      const int et = (warp - 6) * 32 + lane;
      const bool tr = a.trace != nullptr && warp == 6 && lane == 0 && blockIdx.x < 1024;
      if (tr) a.trace[16 + 29 * 1024 + blockIdx.x] = globaltimer_ns();
      for (int it = i0 + et; it < i1; it += 128) d8_prep_item<TP, MP>(a.prep, a.nprep, it);
      fence_proxy_async_global();  // the tensor copies of every CTA read what this thread wrote
      __threadfence();
      named_barrier(1, 128);
      if (warp == 6 && lane == 0) {
        atomicAdd(a.prepped, 1);
        const uint64_t t0 = globaltimer_ns();
        int all = 0;
        for (; a.prep_alone_ns > 0;) {
          int v;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.prepped) : "memory");
          if (v >= (int)gridDim.x) {
            all = 1;
            break;
          }
          if (globaltimer_ns() - t0 > a.prep_alone_ns || abort_sh) break;
          __nanosleep(64);
        }
        prep_alone_sh = !all;
      }
      named_barrier(1, 128);
      if (prep_alone_sh) {
        for (int it = et; it < a.prep_items; it += 128) d8_prep_item<TP, MP>(a.prep, a.nprep, it);
        fence_proxy_async_global();
        __threadfence();
        named_barrier(1, 128);
      }
      if (warp == 6 && lane == 0) mbar_arrive(smem_u32(&xready_bar));
      if (tr) a.trace[16 + 10 * 1024 + blockIdx.x] = globaltimer_ns();
    }
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int os = 0, seq = 0, us = 0;
    uint32_t oph = 0, dph = 0, uph = 0;
    bool ok = true;
    for (;;) {
      int u;
      D8_NEXT_UNIT_W(u, ok);
      if (u < 0) break;
      D8Unit ui;
      d8_unit(a, u, ui);
      const D8Job &J = a.jobs[ui.job];
      const int orow = ui.tile * 128 + r;
      const bool valid = orow < J.rows;
      float acc[TP];
#pragma unroll
      for (int t = 0; t < TP; ++t) acc[t] = 0.f;
      for (int k = 0; ok && k < ui.nst; ++k, ++seq) {
        D8_WAIT(smem_u32(&ofull_bar[os]), oph, ok);  // the stage's scales, biases, factors
        if (!ok) break;
        const uint32_t sb = obase + os * C::OP_BYTES;
        const uint4 s8 = lds128(sb + C::S_OFF + r * 16), q8 = lds128(sb + C::Q_OFF + r * 16);
        // group gi's accumulator (hi columns 0..TP-1, lo TP..2TP-1 from v + o) into acc
        auto consume = [&](const float *v, int gi) {
          const int hw = gi >> 1;  // the word holding group gi's f16 scale and bias
          const uint32_t sw = hw == 0 ? s8.x : hw == 1 ? s8.y : hw == 2 ? s8.z : s8.w;
          const uint32_t qw = hw == 0 ? q8.x : hw == 1 ? q8.y : hw == 2 ? q8.z : q8.w;
          const uint32_t sh = (gi & 1) ? (sw >> 16) : (sw & 0xFFFFu);
          const uint32_t qh = (gi & 1) ? (qw >> 16) : (qw & 0xFFFFu);
          const float s = __half2float(__ushort_as_half((unsigned short)sh));
          const float b = __half2float(__ushort_as_half((unsigned short)qh));
          const uint32_t gxa = sb + C::GX_OFF + gi * 2 * TP * 4;
          // all of the group's factors and sums first: one load latency per group
          float4 fq[TP / 4], Xq[TP / 4];
#pragma unroll
          for (int q = 0; q < TP / 4; ++q) {
            fq[q] = lds128f(gxa + q * 16);             // 2^(9-c) of tokens 4q..4q+3
            Xq[q] = lds128f(gxa + (TP + 4 * q) * 4);  // sum of x of tokens 4q..4q+3
          }
#pragma unroll
          for (int t = 0; t < TP; t += 4) {
            const float4 f = fq[t / 4];
            const float4 X = Xq[t / 4];
            float d0 = v[t], d1 = v[t + 1], d2 = v[t + 2], d3 = v[t + 3];
            add2(d0, d1, v[TP + t], v[TP + t + 1]);
            add2(d2, d3, v[TP + t + 2], v[TP + t + 3]);
            float m0 = f.x, m1 = f.y, m2 = f.z, m3 = f.w;
            mul2(m0, m1, s, s);
            mul2(m2, m3, s, s);
            fma2(acc[t], acc[t + 1], m0, m1, d0, d1);
            fma2(acc[t + 2], acc[t + 3], m2, m3, d2, d3);
            fma2(acc[t], acc[t + 1], b, b, X.x, X.y);
            fma2(acc[t + 2], acc[t + 3], b, b, X.z, X.w);
          }
        };
        // waits for D pair slot p and starts its load into v (no wait for the data)
        auto fetch = [&](float (&v)[C::DP_COLS], int p) -> bool {
          if ((p & 1) == 0) D8_WAIT(smem_u32(&dfull_bar[p >> 1]), dph, ok);
          if (!ok) return false;
          if (warp == 6 && lane == 0) d8_trace(a, 12, seq * 4 + p);
          tc_fence_after();
          if constexpr (C::DP_COLS == 64) {
            tmem_ld64(tmem + lane_off + C::D_COL0 + p * C::DP_COLS, v);
          } else {
            tmem_ld32(tmem + lane_off + C::D_COL0 + p * C::DP_COLS, v);
          }
          return true;
        };
        // after the loads landed: pair slot p goes back to the MMA
        auto release = [&](int p) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&dempty_bar[p]));
        };
        // Software pipeline over the stage's 4 pairs: the next pair's
        // accumulators load while this pair is being applied.
        float va[C::DP_COLS], vb[C::DP_COLS];
        if (!fetch(va, 0)) break;
        if (warp == 6 && lane == 0) d8_trace(a, 9, seq);
        const bool tr = warp == 6 && lane == 0;
        for (int p = 0; p < C::NDP; p += 2) {
          tmem_wait_ld();
          if (tr) d8_trace(a, 13, seq * 4 + p);
          release(p);
          if (!fetch(vb, p + 1)) break;
          consume(va, 2 * p);
          consume(va + C::N, 2 * p + 1);
          if (tr) d8_trace(a, 14, seq * 4 + p);
          tmem_wait_ld();
          if (tr) d8_trace(a, 13, seq * 4 + p + 1);
          release(p + 1);
          if (p + 2 < C::NDP && !fetch(va, p + 2)) break;
          consume(vb, 2 * p + 2);
          consume(vb + C::N, 2 * p + 3);
          if (tr) d8_trace(a, 14, seq * 4 + p + 1);
        }
        dph ^= 1;
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&oempty_bar[os]));
        if (warp == 6 && lane == 0) d8_trace(a, 11, seq);
        if (++os == C::OSTAGES) {
          os = 0;
          oph ^= 1;
        }
      }
      if (!ok) break;
      if (J.splits == 1) {
        if (valid) {
          const float bias = J.bias ? __ldg(J.bias + orow) : 0.f;
          void *const oC = J.C;
          const int64_t oldc = J.ldc;
          const int oT = J.T, odt = a.out_dt;
#pragma unroll
          for (int t = 0; t < TP; ++t)
            if (t < oT) d8_store(odt, oC, oldc, t, orow, acc[t] + bias);
        }
      } else {
        // A split tile: the partial goes to the unit's workspace slot,
        // column-major (a warp's 32 rows of one token are one 128-byte line),
        // for the ordered split sum that runs after this kernel.
        float *slot = a.ws + (J.ws_base + (int64_t)ui.tile * J.splits + ui.sidx) * 128 * TP + r;
#pragma unroll
        for (int t = 0; t < TP; ++t) __stcg(slot + t * 128, acc[t]);
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
  if (threadIdx.x == 0) {
    // the last CTA to finish re-arms the unit dispenser for the next launch
    // (every CTA has taken its last index: it only exits after a -1)
    __threadfence();
    if (atomicAdd(a.done, 1) == (int)gridDim.x - 1) {
      atomicExch(a.work, 0);
      atomicExch(a.done, 0);
      atomicExch(a.prepped, 0);
    }
  }
  if (a.trace != nullptr && threadIdx.x == 0 && blockIdx.x < 1024) a.trace[16 + 31 * 1024 + blockIdx.x] = globaltimer_ns();
}

// ------------------------------------------------------------------ host
std::mutex g_d8_mu;
std::atomic<bool> g_d8_prep_alone{false};

bool al16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// Ranges per tile.  Units are dispensed at run time, but the SMs stream at
// about the same rate, so the time is about the whole rounds of units the
// SMs run (units / SMs rounded up, times the longest unit plus a per-unit
// cost of 0.3 stage times), or the even share of all stages where that is
// larger; then, with more than one range, the ordered split sum: a fixed
// part and a part that grows with the float32 partials it reads back (about
// 0.39 stage times per MB).  All in stage times (a stage streams 36 KB of
// codes, scales and biases per SM).  Fitted to a sweep of the ranges at
// T = 16: the column layer's 16 stages a tile in 2 ranges took 1.2 us less
// per call than in 4 (3, 6, 8 slower); the row layer's 56 in 7 ranges as
// long as in 14, in 8, 10, 19 or 28 longer (8 ranges: 4 rounds of 7 stages
// against 3 of 8).
struct D8Split {
  int ranges;
  double cost;
};
D8Split d8_ranges(const int64_t *tiles, const int *nst, int njobs, int sms, int c, int TP) {
  double stages = 0, units = 0, slots = 0;
  int longest = 0;
  for (int j = 0; j < njobs; ++j) {
    const int len = (nst[j] + c - 1) / c;
    const int r = (nst[j] + len - 1) / len;
    stages += (double)tiles[j] * nst[j];
    units += (double)tiles[j] * r;
    if (r > 1) slots += (double)tiles[j] * r;
    if (len > longest) longest = len;
  }
  const double share = (stages + 0.3 * units) / sms;
  const double rounds = std::ceil(units / sms) * (longest + 0.3);
  const double slot_mb = slots * 128.0 * TP * 4.0 / 1e6;
  return D8Split{c, std::max(share, rounds) + (c > 1 ? 1.5 + 0.39 * slot_mb : 0.0)};
}

template <typename K, typename A>
int d8_launch(K kern, const A &args, int grid, int threads, int smem, bool *attr_done, cudaStream_t s,
              const char *what) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, what);
    attr_done[dev & 63] = true;
  }
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(threads), (size_t)smem, s, args);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, what);
}

template <int TP, int MP>
int launch_dec8_t(const Problem &p, cudaStream_t s, bool *handled, GvWorkspaceFn get_ws, void *ctx, size_t ws_cap) {
  using C = D8Cfg<TP>;
  static D8Args<MP> args;
  memset(&args, 0, sizeof(args));
  const int sms = sm_count();

  // regions: distinct activation blocks (x, K, lda)
  int nreg = 0;
  int reg_of[kMaxParts];
  int64_t prep_bytes = 0;
  int64_t reg_off[kMaxParts];
  int items = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    for (int q = 0; q < J.nparts; ++q) {
      const int qq = J.part0 + q;
      const Part &P = p.parts[qq];
      const int G = (int)(P.K / 64);
      int r = -1;
      for (int i = 0; i < nreg; ++i)
        if (args.prep[i].x == P.A && args.prep[i].K == (int)P.K && args.prep[i].lda == P.lda) r = i;
      if (r < 0) {
        if (nreg >= MP) return TP_OK;
        r = nreg++;
        PrepRegion &R = args.prep[r];
        R.x = static_cast<const uint16_t *>(P.A);
        R.lda = P.lda;
        R.K = (int)P.K;
        R.groups = G;
        R.T = (int)J.M;
        R.item_begin = items;
        items += TP * G;
        reg_off[r] = prep_bytes;
        prep_bytes += ((int64_t)2 * TP * P.K + (int64_t)G * 2 * TP * 4 + 255) / 256 * 256;
      }
      reg_of[qq] = r;
    }
  }
  // stages per job (parts laid end to end) and the ranges per tile: the
  // cheapest count whose partial slots fit the workspace cap
  int64_t tiles_j[kMaxJobs];
  int nst_j[kMaxJobs];
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    tiles_j[j] = (J.N + 127) / 128;
    nst_j[j] = 0;
    for (int q = 0; q < J.nparts; ++q) nst_j[j] += (int)(p.parts[J.part0 + q].K / 512);
  }
  int c = 1;
  double best = 1e300;
  for (int cc = 1; cc <= 64; ++cc) {
    int64_t sl = 0;
    bool useful = false;
    for (int j = 0; j < p.njobs; ++j) {
      const int len = (nst_j[j] + cc - 1) / cc;
      const int r = (nst_j[j] + len - 1) / len;
      if (r == cc) useful = true;
      if (r > 1) sl += tiles_j[j] * r;
    }
    if (!useful) continue;
    if (cc > 1 && (size_t)prep_bytes + (size_t)sl * 128 * TP * sizeof(float) > ws_cap) continue;
    const D8Split d = d8_ranges(tiles_j, nst_j, p.njobs, sms, cc, TP);
    if (d.cost < best - 1e-9) {
      best = d.cost;
      c = cc;
    }
  }

  // jobs, parts, units, workspace layout (partial slots after the prepared x)
  int64_t units = 0, slots = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    D8Job &Q = args.jobs[j];
    Q.C = J.C;
    Q.bias = J.bias;
    Q.ldc = J.ldc;
    Q.rows = (int)J.N;
    Q.T = (int)J.M;
    Q.part0 = J.part0;
    Q.nparts = J.nparts;
    Q.tiles = (Q.rows + 127) / 128;
    int st = 0;
    for (int q = 0; q < J.nparts; ++q) {
      const int qq = J.part0 + q;
      const Part &P = p.parts[qq];
      D8Part &DP = args.parts[qq];
      DP.groups = (int)(P.K / 64);
      DP.st0 = st;
      st += DP.groups / kD8GroupsPerStage;
      DP.cmap = DP.smap = DP.qmap = (int16_t)qq;
      DP.region = (int16_t)reg_of[qq];
      // codes: one copy per stage, 2 chunks of 128 bytes (4 groups) of 128 rows
      int rc = make_tmap_3d_chunks(&args.cmaps[qq], P.B, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, (uint64_t)(P.K / 8),
                                   (uint64_t)J.N, (uint64_t)P.ldb, 32, 128, 2, CU_TENSOR_MAP_SWIZZLE_128B);
      if (!rc)
        rc = make_tmap_2d(&args.smaps[qq], P.scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)DP.groups,
                          (uint64_t)J.N, (uint64_t)DP.groups, 8, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (!rc)
        rc = make_tmap_2d(&args.qmaps[qq], P.qbias, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)DP.groups,
                          (uint64_t)J.N, (uint64_t)DP.groups, 8, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (rc) return rc;
    }
    Q.nst = st;
    Q.range_len = (st + c - 1) / c;
    Q.splits = (st + Q.range_len - 1) / Q.range_len;
    Q.unit_begin = (int)units;
    Q.ws_base = slots;
    units += (int64_t)Q.tiles * Q.splits;
    if (Q.splits > 1) slots += (int64_t)Q.tiles * Q.splits;
  }
  if (units == 0) {
    *handled = true;
    return TP_OK;
  }
  if (units > INT32_MAX) return TP_OK;
  const int64_t slot_floats = slots * 128 * TP;
  float *ws = nullptr;
  int *cnt = nullptr;
  int rc = get_ws(ctx, (size_t)prep_bytes + (size_t)slot_floats * sizeof(float), 3, &ws, &cnt);
  if (rc) return rc;
  uint8_t *wsb = reinterpret_cast<uint8_t *>(ws);
  for (int r = 0; r < nreg; ++r) {
    PrepRegion &R = args.prep[r];
    R.xq = wsb + reg_off[r];
    R.gx = reinterpret_cast<float *>(wsb + reg_off[r] + (int64_t)2 * TP * R.K);
    args.gx[r] = R.gx;
    // the activation tile: one copy per stage, 4 chunks of 128 bytes (2 groups) of the 2 TP rows
    rc = make_tmap_3d_chunks(&args.xmaps[r], R.xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)R.K,
                             (uint64_t)(2 * TP), (uint64_t)R.K, 128, (uint32_t)(2 * TP), 4,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  int64_t trace_cap = 0;
  trace_buffer(&args.trace, &trace_cap);
  args.nprep = nreg;
  args.prep_alone_ns = g_d8_prep_alone.load() ? 0 : kD8PrepAloneNs;
  args.prep_items = items;
  args.njobs = p.njobs;
  args.total_units = (int)units;
  args.out_dt = p.out_dt;
  args.ws = reinterpret_cast<float *>(wsb + prep_bytes);
  args.work = cnt;
  args.done = cnt + 1;
  args.prepped = cnt + 2;
  args.status = p.status;
  args.wait_ns = (uint64_t)p.wait_ns;
  // kind::f8f6f4 instruction descriptor: D f32, A and B E4M3 (format 0), both
  // K-major, M = 128, N = 2 TP
  args.idesc = (1u << 4) | ((uint32_t)(C::N >> 3) << 17) | ((128u >> 4) << 24);

  static bool kdone[64] = {false};
  const int grid = args.total_units < sms ? args.total_units : sms;
  rc = d8_launch(q4_dec8_kernel<TP, MP>, args, grid, kD8Threads, C::SMEM, kdone, s, "q4_dec8_kernel");
  if (rc == TP_OK && slots > 0) {  // ordered sums of the split tiles
    SplitJob sj[kMaxJobs];
    for (int j = 0; j < p.njobs; ++j) {
      const D8Job &Q = args.jobs[j];
      sj[j] = SplitJob{Q.C, Q.bias, Q.ldc, Q.ws_base, Q.rows, Q.T, Q.tiles, 1, Q.splits};
    }
    rc = launch_split_reduce(sj, p.njobs, args.ws, TP, p.out_dt, s);
  }
  if (rc == TP_OK) *handled = true;
  return rc;
}

}  // namespace

void set_dec8_prep_alone(bool on) { g_d8_prep_alone.store(on); }

int launch_q4_dec8(const Problem &p, cudaStream_t s, bool *handled, GvWorkspaceFn get_ws, void *ctx,
                   size_t ws_cap) {
  *handled = false;
  if (p.in_dt != TP_BF16 || p.b_layout != BL_Q4 || p.njobs < 1) return TP_OK;
  int64_t maxT = 0;
  int nparts = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    if (J.M > maxT) maxT = J.M;
    if (J.M < 1 || J.N > INT32_MAX / 2 || J.nparts < 1) return TP_OK;
    if (J.part0 + J.nparts > nparts) nparts = J.part0 + J.nparts;
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      // whole 8-group stages; 16-byte aligned operands and rows for the tensor
      // copies and the pre-pass's vector loads
      if ((P.K % 512) || P.K > (int64_t)1 << 30 || !al16(P.A) || (P.lda % 8) || !al16(P.B) || (P.ldb % 4) ||
          !al16(P.scales) || !al16(P.qbias))
        return TP_OK;
    }
  }
  if (maxT > 16 || nparts > 32 || p.njobs > 32) return TP_OK;
  std::lock_guard<std::mutex> lk(g_d8_mu);
  const bool small = nparts <= 8 && p.njobs <= 8;
  if (maxT <= 8)
    return small ? launch_dec8_t<8, 8>(p, s, handled, get_ws, ctx, ws_cap)
                 : launch_dec8_t<8, 32>(p, s, handled, get_ws, ctx, ws_cap);
  return small ? launch_dec8_t<16, 8>(p, s, handled, get_ws, ctx, ws_cap)
               : launch_dec8_t<16, 32>(p, s, handled, get_ws, ctx, ws_cap);
}

}  // namespace tp
