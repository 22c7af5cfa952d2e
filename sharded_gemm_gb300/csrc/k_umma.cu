// k_umma.cu -- tcgen05 tensor-core GEMM for sm_103a: the column-parallel
// (all-to-sharded), row-parallel (sharded-to-all) and SUMMA products.
//
// One persistent, warp-specialized kernel, one CTA per SM:
//   warp 0      TMA producer: A tile (128 x 64) and B tile (BN x 64) of bf16/f16
//               per k-block into a ring of STAGES shared-memory stages, 128-byte
//               swizzled, completion tracked by mbarrier transaction counts;
//   warp 1      allocates TMEM; one thread issues tcgen05.mma (M=128, N=BN,
//               K=16) into float32 accumulators in TMEM and commits them to
//               mbarriers;
//   warps 2..9  epilogue: tcgen05.ld of the accumulator, fixed-order sum of
//               partials (row-parallel), bias, conversion, global store.
// A work unit is one output tile of one job.  Within a job, `parts` are the
// matrix products that make the tile:
//   chain (SUMMA, column-parallel): all parts accumulate into one TMEM
//     accumulator in part order (SUMMA's q steps);
//   partials (row-parallel): every part (rank r) is formed from zero in its
//     own TMEM buffer, and the epilogue adds the partials in ascending r in
//     registers, then adds the bias once.  Partials never touch device memory.
// Swap-AB (T <= 16, decode): the weight rows fill the 128-row MMA dimension,
// the tokens the N = 16 dimension, and the epilogue stores the transpose.
// Every mbarrier wait is bounded (see ptx.cuh): a wait that runs out records
// TP_ERR_TIMEOUT in the status word and the CTA drains its in-flight copies and
// MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "ptx.cuh"
#include "tp_internal.h"

namespace tp {

constexpr int kMaxMaps = 64;
// k-blocks of the weight operand the row-parallel cluster kernel pulls into
// L2 beyond its operand ring (cp.async.bulk.prefetch), so its tensor copies
// find their lines in L2 (measured 53.6 -> 52.2 us on the MLP's W2; the same
// prefetch slowed the pair kernels, whose weight tiles are shared by two
// pairs, and is not used there).
constexpr int kPrefetchKb = 6;
constexpr int kMaxCMaps = 16;  // output maps of the TMA-store epilogue
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;

struct UJob {
  void *C;
  const float *bias;
  int64_t ldc;
  int rowsA, rowsB;    // extents of the A-operand rows and B-operand rows
  int part0, nparts;
  int tilesA, tilesB;
  int unit_begin;
  int splits;          // > 1: units are (tile, k-block range) pieces (swap mode)
  const float *bias2;  // gated: the up projection's bias (nullable)
  int64_t ws_base;     // split mode: first float32 slot of this job
  int kb_total;        // split mode: k-blocks of all parts together
  int cnt_base;        // split mode: first tile counter (kEpiWarps per tile)
};

struct UPart {
  int16_t amap, bmap;
  int32_t kblocks;
  int16_t bmap2;  // gated: the up projection's weight map
};

struct UmmaArgs {
  CUtensorMap mapA[kMaxMaps];
  CUtensorMap mapB[kMaxMaps];
  // TMA-store epilogues: float32 outputs in 32 x 32 boxes, 128-byte swizzle
  // (TSTORE), or a warp's 32 rows x its columns, unswizzled (rstore)
  CUtensorMap mapC[kMaxCMaps];
  UJob jobs[kMaxJobs];
  UPart parts[kMaxParts];
  int njobs, total_units, nmapA, nmapB;
  int chain, out_dt, vec_ok;
  int cluster_n;  // ranks per cluster (row-parallel cluster kernel)
  int rstore;     // pair kernel: a CTA's last unit is stored through its drained operand ring
  unsigned long long *trace;  // optional timeline of CTA 0 (tp_set_trace)
  uint32_t idesc;
  int *status;
  uint64_t wait_ns;
  float *ws;  // split mode: float32 slots, 128 x BN per (tile, split), column-major
  int *cnt;   // split mode: arrival counters, zero between calls
};

// Records the time of (event, k-block sequence) for CTA 0 when tracing.
__device__ __forceinline__ void umma_trace(const UmmaArgs &a, int event, int seq) {
  if (a.trace != nullptr && blockIdx.x == 0 && seq < 1024) a.trace[16 + event * 1024 + seq] = globaltimer_ns();
}

// When tracing, every CTA b (< 1024) records its SM id + 1 (event 28) and its
// start (30) and end (31) times at word index b.
__device__ __forceinline__ void umma_cta_trace(const UmmaArgs &a, int event) {
  if (a.trace == nullptr || threadIdx.x != 0 || blockIdx.x >= 1024) return;
  if (event == 30) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    a.trace[16 + 28 * 1024 + blockIdx.x] = smid + 1;
  }
  a.trace[16 + event * 1024 + blockIdx.x] = globaltimer_ns();
}

__device__ __forceinline__ int find_job(const UmmaArgs &a, int u) {
  int j = 0;
  while (j + 1 < a.njobs && u >= a.jobs[j + 1].unit_begin) ++j;
  return j;
}

// Pulls a tile into L2 only (no shared memory, no barrier); parts of the tile
// outside the tensor are skipped.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// Position of a unit within its job: the output tile (ta, tb) and, when the
// job is split, the k-block range [k0, k1) of the concatenated parts and the
// split index sp; else the whole contraction.
struct UnitPos {
  int ta, tb, sp, k0, k1;
};
__device__ __forceinline__ UnitPos unit_pos(const UJob &J, int local) {
  UnitPos q;
  q.ta = local % J.tilesA;
  int rest = local / J.tilesA;
  q.sp = 0;
  q.k0 = 0;
  q.k1 = INT_MAX;
  if (J.splits > 1) {
    q.sp = rest % J.splits;
    rest /= J.splits;
    q.k0 = (int)((int64_t)q.sp * J.kb_total / J.splits);
    q.k1 = (int)((int64_t)(q.sp + 1) * J.kb_total / J.splits);
  }
  q.tb = rest;
  return q;
}

__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float x, float y) {
  __half2 h = __floats2half2_rn(x, y);
  return *reinterpret_cast<uint32_t *>(&h);
}

// The bias of a warp's contiguous output columns [col0, col0 + 32 NW): lane l
// holds columns col0 + 32 j + l.  Loaded before the warp waits for its
// accumulator; loaded per output chunk instead, the bias reads (L1 misses
// behind a full operand stream, about a microsecond each) serialized the
// epilogue: 10 us for a 128 x 320 tile.
template <int NW>
struct WarpBias {
  float v[NW];
  __device__ __forceinline__ void load(const float *bias, int col0, int ncols, int lane) {
#pragma unroll
    for (int j = 0; j < NW; ++j) {
      const int c = col0 + j * 32 + lane;
      v[j] = (bias != nullptr && c < ncols) ? __ldg(bias + c) : 0.f;
    }
  }
  // The bias of column col0 + o (o a compile-time constant after unrolling).
  __device__ __forceinline__ float at(int o) const { return __shfl_sync(0xffffffffu, v[o >> 5], o & 31); }
  // v[i] += bias of column col0 + o0 + i, when the job has a bias.
  template <int CH>
  __device__ __forceinline__ void add(bool has_bias, int o0, float (&x)[CH]) const {
    if (!has_bias) return;
#pragma unroll
    for (int i = 0; i < CH; ++i) x[i] += at(o0 + i);
  }
};

// A job's output, copied to registers once per unit: read through the
// kernel-parameter block, the fields are reloaded after every store and every
// tensor-memory load (the compiler cannot tell the output, or the asm
// statements' memory, from the parameters), a dependent load per chunk.
struct UOut {
  void *C;
  const float *bias;
  int64_t ldc;
  int rowsA, rowsB;
  int out_dt, vec_ok;
};
__device__ __forceinline__ UOut uout(const UmmaArgs &a, const UJob &J) {
  return UOut{J.C, J.bias, J.ldc, J.rowsA, J.rowsB, a.out_dt, a.vec_ok};
}

// Stores CH consecutive output values of one thread (row-major, normal mode).
template <int CH, bool BIAS = true>
__device__ __forceinline__ void store_row_chunk(const UOut &J, int row, int col0, float (&v)[CH]) {
  if (row >= J.rowsA) return;
  if (BIAS && J.bias) {
#pragma unroll
    for (int i = 0; i < CH; ++i)
      if (col0 + i < J.rowsB) v[i] += __ldg(J.bias + col0 + i);
  }
  const int64_t base = (int64_t)row * J.ldc + col0;
  const bool full = J.vec_ok && (col0 + CH <= J.rowsB);
  if (J.out_dt == TP_F32) {
    float *C = static_cast<float *>(J.C) + base;
    if (full && (CH % 4 == 0)) {
#pragma unroll
      for (int i = 0; i < CH; i += 4)
        *reinterpret_cast<float4 *>(C + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < CH; ++i)
        if (col0 + i < J.rowsB) C[i] = v[i];
    }
  } else {
    uint16_t *C = static_cast<uint16_t *>(J.C) + base;
    const bool bf = J.out_dt == TP_BF16;
    if (full && (CH % 8 == 0)) {
#pragma unroll
      for (int i = 0; i < CH; i += 8) {
        uint4 q;
        q.x = bf ? pack_bf16(v[i], v[i + 1]) : pack_f16(v[i], v[i + 1]);
        q.y = bf ? pack_bf16(v[i + 2], v[i + 3]) : pack_f16(v[i + 2], v[i + 3]);
        q.z = bf ? pack_bf16(v[i + 4], v[i + 5]) : pack_f16(v[i + 4], v[i + 5]);
        q.w = bf ? pack_bf16(v[i + 6], v[i + 7]) : pack_f16(v[i + 6], v[i + 7]);
        *reinterpret_cast<uint4 *>(C + i) = q;
      }
    } else {
#pragma unroll
      for (int i = 0; i < CH; ++i)
        if (col0 + i < J.rowsB)
          C[i] = bf ? __bfloat16_as_ushort(__float2bfloat16_rn(v[i]))
                    : __half_as_ushort(__float2half_rn(v[i]));
    }
  }
}

// TMA-store epilogue: a warp's 32 x 32 float32 chunk (lane l holds row
// row0 + l) goes to the warp's 4 KB staging buffer in the 128-byte
// swizzled layout of the output map (row r's 16-byte piece j at position
// j ^ (r % 8): each group of 8 lanes covers all 32 banks), and lane 0 issues
// the tile store.
constexpr int kTsWarpBytes = 4096;
__device__ __forceinline__ void tstore_chunk(const UmmaArgs &a, const UJob &J, int job, int row0, int col0,
                                             float (&v)[32], uint32_t bufs, int &cnt, int lane) {
  // A chunk wholly outside the output (ragged last tile) is skipped outright:
  // it neither stores nor writes the staging buffer, which is rewritten only
  // after the store issued from it has read it.
  if (row0 >= J.rowsA || col0 >= J.rowsB) return;  // the caller has added the bias
  if (cnt >= 1) {  // the previous store has read the buffer
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }
  const uint32_t buf = bufs;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t dst = buf + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) * 16));
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "f"(v[4 * j]), "f"(v[4 * j + 1]),
                 "f"(v[4 * j + 2]), "f"(v[4 * j + 3])
                 : "memory");
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {  // the map clips a partly outside chunk
    tma_store_2d(&a.mapC[job], buf, col0, row0);
    bulk_commit_group();
  }
  ++cnt;
}

// Ring-staged store: CH values of the thread's row go to its row of the
// warp's staging block (32 rows x `pitch` bytes, unswizzled), converted to
// the output type; o0 is the chunk's first column within the block.
template <int CH>
__device__ __forceinline__ void stage_row_chunk(int out_dt, uint32_t rowbuf, int o0, const float (&v)[CH]) {
  if (out_dt == TP_F32) {
#pragma unroll
    for (int i = 0; i < CH; i += 4)
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(rowbuf + (uint32_t)((o0 + i) * 4)), "f"(v[i]),
                   "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3])
                   : "memory");
  } else {
    const bool bf = out_dt == TP_BF16;
#pragma unroll
    for (int i = 0; i < CH; i += 8) {
      uint32_t q[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        q[k] = bf ? pack_bf16(v[i + 2 * k], v[i + 2 * k + 1]) : pack_f16(v[i + 2 * k], v[i + 2 * k + 1]);
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(rowbuf + (uint32_t)((o0 + i) * 2)), "r"(q[0]),
                   "r"(q[1]), "r"(q[2]), "r"(q[3])
                   : "memory");
    }
  }
}

// Swap-AB store: the thread's A row is output column `row`; its values are
// tokens col0.. of that column.
template <int CH>
__device__ __forceinline__ void store_col_chunk(const UOut &J, int row, int col0, const float (&v)[CH], float b) {
  if (row >= J.rowsA) return;
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int t = col0 + i;
    if (t >= J.rowsB) break;
    const int64_t idx = (int64_t)t * J.ldc + row;
    const float x = v[i] + b;
    if (J.out_dt == TP_F32)
      static_cast<float *>(J.C)[idx] = x;
    else if (J.out_dt == TP_BF16)
      static_cast<uint16_t *>(J.C)[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
    else
      static_cast<uint16_t *>(J.C)[idx] = __half_as_ushort(__float2half_rn(x));
  }
}

// Split-mode store (swap): CH token columns cl0.. of output row m of the
// unit's float32 slot (column-major, 128 rows per column); no bias, which the
// tile's ordered finish (split_finish) adds.  Columns past the token count are
// not written.
template <int CH, int BN>
__device__ __forceinline__ void store_slot_chunk(const UmmaArgs &a, const UJob &J, const UnitPos &q, int m,
                                                 int cl0, const float (&v)[CH]) {
  const int64_t slot = J.ws_base + ((int64_t)q.tb * J.tilesA + q.ta) * J.splits + q.sp;
  float *s = a.ws + slot * (BN * 128) + m;
  const int t0 = q.tb * BN + cl0;
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    if (t0 + i >= J.rowsB) break;
    __stcg(s + (cl0 + i) * 128, v[i]);
  }
}

// Split mode, after a warp has stored its slot values: the warp that arrives
// last at its (tile, warp) counter adds the tile's split slots in split order
// for its 32 rows x HALF token columns (so the sum does not depend on which
// unit finishes last), adds the bias, stores the output and re-arms the counter.
template <int BN, int HALF>
__device__ __forceinline__ void split_finish(const UmmaArgs &a, const UJob &J, const UnitPos &q, int ew, int row,
                                             int m, int half, int lane) {
  __threadfence();
  __syncwarp();
  const int64_t tile = (int64_t)q.tb * J.tilesA + q.ta;
  int *cnt = a.cnt + (J.cnt_base + tile) * kEpiWarps + ew;
  int prev = 0;
  if (lane == 0) prev = atomicAdd(cnt, 1);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != J.splits - 1) return;
  __threadfence();
  const int cl0 = half * HALF;
  const int ncol = J.rowsB - q.tb * BN - cl0;  // token columns of this warp that exist
  const float *s0 = a.ws + (J.ws_base + tile * J.splits) * (BN * 128) + m;
  float v[HALF];
#pragma unroll
  for (int i = 0; i < HALF; ++i) v[i] = i < ncol ? __ldcg(s0 + (cl0 + i) * 128) : 0.f;
#pragma unroll 4
  for (int sp = 1; sp < J.splits; ++sp) {
    const float *sj = s0 + (int64_t)sp * (BN * 128);
#pragma unroll
    for (int i = 0; i < HALF; ++i)
      if (i < ncol) v[i] += __ldcg(sj + (cl0 + i) * 128);
  }
  store_col_chunk<HALF>(uout(a, J), row, q.tb * BN + cl0, v, (J.bias && row < J.rowsA) ? __ldg(J.bias + row) : 0.f);
  __syncwarp();
  if (lane == 0) *cnt = 0;
}

// Epilogue chunk width: the widest of 32 / 16 / 8 columns that divides half a tile.
template <int HALF>
struct ChunkOf {
  static constexpr int v = (HALF % 32 == 0) ? 32 : (HALF % 16 == 0) ? 16 : 8;
};

template <int CH>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, float (&v)[CH]) {
  if constexpr (CH == 32) {
    tmem_ld32(taddr, v);
  } else if constexpr (CH == 16) {
    tmem_ld16(taddr, v);
  } else {
    static_assert(CH == 8, "chunk");
    tmem_ld8(taddr, v);
  }
}

template <int N>
struct TmemCols {
  static constexpr int v = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : N <= 256 ? 256 : 512;
};

template <int BN, bool B_MN, bool SWAP, bool PARTIALS, int STAGES, int NACC, bool A_MN = false>
__global__ void __launch_bounds__(kThreads, 1) umma_gemm_kernel(const __grid_constant__ UmmaArgs a) {
  static_assert(!A_MN || !SWAP, "M-major A is not swapped");
  constexpr int A_BYTES = BM * BK * 2;
  constexpr int B_BYTES = BN * BK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int TCOLS = TmemCols<NACC * BN>::v;
  constexpr int HALF = BN / 2;
  constexpr int CH = ChunkOf<HALF>::v;
  constexpr int NCH = HALF / CH;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(NACC * BN <= 512, "TMEM capacity");

  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[NACC], tempty_bar[NACC];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int s = 0; s < NACC; ++s) {
      mbar_init(smem_u32(&tfull_bar[s]), 1);
      mbar_init(smem_u32(&tempty_bar[s]), kEpiWarps);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), TCOLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < a.nmapA && i < 8; ++i) prefetch_tmap(&a.mapA[i]);
    for (int i = 0; i < a.nmapB && i < 8; ++i) prefetch_tmap(&a.mapB[i]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  // The set-up above overlaps the previous kernel's tail (programmatic
  // launch); global memory is read and written only after it has completed.
  griddep_launch_dependents();
  if constexpr (SWAP) {
    // The swapped A operand is the weight matrix: start pulling this CTA's
    // first k-blocks into L2 meanwhile.  L2 is the point of coherence, so a
    // line the previous kernel writes after the prefetch is still what the
    // tensor loads (issued after the wait) see.
    if (warp == 0 && lane == 0 && (int)blockIdx.x < a.total_units) {
      const UJob &J = a.jobs[find_job(a, blockIdx.x)];
      const UnitPos q = unit_pos(J, blockIdx.x - J.unit_begin);
      int off = 0, n = 0;
      for (int p = 0; p < J.nparts && n < STAGES; ++p) {
        const UPart P = a.parts[J.part0 + p];
        const int lo = max(0, q.k0 - off), hi = min(P.kblocks, q.k1 - off);
        off += P.kblocks;
        for (int kb = lo; kb < hi && n < STAGES; ++kb, ++n) tma_prefetch_l2_2d(&a.mapA[P.amap], kb * BK, q.ta * BM);
      }
    }
  }
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t last_phase[STAGES];
      bool used[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) used[s] = false;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        const UJob &J = a.jobs[find_job(a, u)];
        const UnitPos q = unit_pos(J, u - J.unit_begin);
        const int rowA0 = q.ta * BM, rowB0 = q.tb * BN;
        int off = 0;
        for (int p = 0; ok && p < J.nparts; ++p) {
          const UPart P = a.parts[J.part0 + p];
          const int lo = max(0, q.k0 - off), hi = min(P.kblocks, q.k1 - off);
          off += P.kblocks;
          for (int kb = lo; kb < hi; ++kb) {
            if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, lim, a.status, &abort_sh)) {
              ok = false;
              break;
            }
            const uint32_t sa = sbase + stage * STAGE_BYTES, sb = sa + A_BYTES;
            const uint32_t fb = smem_u32(&full_bar[stage]);
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            if constexpr (A_MN) {  // two boxes of 64 rows of M (128 bytes) x BK
              tma_load_2d(sa, &a.mapA[P.amap], fb, rowA0, kb * BK);
              tma_load_2d(sa + 8192, &a.mapA[P.amap], fb, rowA0 + 64, kb * BK);
            } else {
              tma_load_2d(sa, &a.mapA[P.amap], fb, kb * BK, rowA0);
            }
            if constexpr (B_MN) {
#pragma unroll
              for (int c = 0; c < BN / 64; ++c)
                tma_load_2d(sb + c * 8192, &a.mapB[P.bmap], fb, rowB0 + c * 64, kb * BK);
            } else {
              tma_load_2d(sb, &a.mapB[P.bmap], fb, kb * BK, rowB0);
            }
            used[stage] = true;
            last_phase[stage] = phase;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
      if (!ok) {
        // Wait (bounded, ignoring the abort flag) for copies still in flight.
        for (int s = 0; s < STAGES; ++s)
          if (used[s]) mbar_wait(smem_u32(&full_bar[s]), last_phase[s], lim, a.status, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
        const UJob &J = a.jobs[find_job(a, u)];
        const UnitPos q = unit_pos(J, u - J.unit_begin);
        // one accumulator per unit (chained parts, or a split's k-block
        // range), else one per part
        const bool uchain = a.chain || J.splits > 1;
        bool held = false;  // an accumulator is acquired and not yet committed
        uint32_t accum = 0;
        int off = 0;
        for (int p = 0; ok && p < J.nparts; ++p) {
          const UPart P = a.parts[J.part0 + p];
          const int lo = max(0, q.k0 - off), hi = min(P.kblocks, q.k1 - off);
          off += P.kblocks;
          if (lo >= hi) continue;
          if (!held) {
            if (!mbar_wait(smem_u32(&tempty_bar[acc]), acc_phase ^ 1, lim, a.status, &abort_sh)) {
              ok = false;
              break;
            }
            tc_fence_after();
            held = true;
            accum = 0;
          }
          const uint32_t d = tmem_base + (uint32_t)(acc * BN);
          for (int kb = lo; kb < hi; ++kb) {
            if (!mbar_wait(smem_u32(&full_bar[stage]), phase, lim, a.status, &abort_sh)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = sbase + stage * STAGE_BYTES, sb = sa + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = A_MN ? umma_desc_sw128(sa + kk * 2048, 8192, 1024)
                                       : umma_desc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? umma_desc_sw128(sb + kk * 2048, 8192, 1024)
                                       : umma_desc_sw128(sb + kk * 32, 16, 1024);
              umma_f16(d, ad, bd, a.idesc, accum);
              accum = 1u;
            }
            umma_commit(smem_u32(&empty_bar[stage]));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          if (!uchain) {
            umma_commit(smem_u32(&tfull_bar[acc]));
            held = false;
            if (++acc == NACC) {
              acc = 0;
              acc_phase ^= 1;
            }
          }
        }
        if (ok && held) {
          umma_commit(smem_u32(&tfull_bar[acc]));
          if (++acc == NACC) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
      }
      // All MMAs issued by this thread complete before TMEM is released.
      umma_commit(smem_u32(&drain_bar));
      mbar_wait(smem_u32(&drain_bar), 0, lim, a.status, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    float sum[PARTIALS ? HALF : 1];
    for (int u = blockIdx.x; ok && u < a.total_units; u += gridDim.x) {
      const UJob &J = a.jobs[find_job(a, u)];
      const UnitPos q = unit_pos(J, u - J.unit_begin);
      const int row = q.ta * BM + quarter * 32 + lane;
      const int colb = q.tb * BN + half * HALF;
      const bool split = SWAP && J.splits > 1;
      const int nep = (a.chain || split) ? 1 : J.nparts;
      // bias: swap mode, one per thread (its output column); else the warp's columns
      const float rbias = (SWAP && J.bias && row < J.rowsA) ? __ldg(J.bias + row) : 0.f;
      const UOut uo = uout(a, J);
      WarpBias<(HALF + 31) / 32> wb;
      if constexpr (!SWAP && !PARTIALS) wb.load(J.bias, colb, J.rowsB, lane);
      for (int pe = 0; pe < nep; ++pe) {
        // warp-uniform: every lane must take the same path into tcgen05.ld
        const bool got = mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, lim, a.status, &abort_sh);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb_addr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16) +
                                 (uint32_t)(half * HALF);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float v[CH];
          tmem_load_chunk<CH>(tb_addr + c * CH, v);
          tmem_wait_ld();
          if constexpr (PARTIALS) {
#pragma unroll
            for (int i = 0; i < CH; ++i) sum[c * CH + i] = (pe == 0) ? v[i] : sum[c * CH + i] + v[i];
          } else {
            if constexpr (SWAP) {
              if (split)
                store_slot_chunk<CH, BN>(a, J, q, quarter * 32 + lane, half * HALF + c * CH, v);
              else
                store_col_chunk<CH>(uo, row, colb + c * CH, v, rbias);
            } else {
              wb.add<CH>(J.bias != nullptr, c * CH, v);
              store_row_chunk<CH, false>(uo, row, colb + c * CH, v);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
        if (++acc == NACC) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if constexpr (PARTIALS) {
        if (ok) {
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            float v[CH];
#pragma unroll
            for (int i = 0; i < CH; ++i) v[i] = sum[c * CH + i];
            if constexpr (SWAP) {
              if (split)
                store_slot_chunk<CH, BN>(a, J, q, quarter * 32 + lane, half * HALF + c * CH, v);
              else
                store_col_chunk<CH>(uo, row, colb + c * CH, v, rbias);
            } else {
              // bias read per chunk: a preloaded copy beside the partial sums spills
              store_row_chunk<CH>(uo, row, colb + c * CH, v);
            }
          }
        }
      }
      if constexpr (SWAP) {
        if (split && ok) split_finish<BN, HALF>(a, J, q, ew, row, quarter * 32 + lane, half, lane);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TCOLS);
  }
}

// ====================================================================== CTA pairs
// umma_pair_kernel: the chain-mode GEMM on 2-CTA clusters with the pair MMA
// (tcgen05.mma.cta_group::2, M = 256).  Rank 0 of a pair issues the MMAs for
// both CTAs; each CTA stages its own 128 rows of A and its half (BN/2 rows) of
// B, so a CTA holds (128 + BN/2) x 64 operand elements per k-block instead of
// (128 + BN) x 64 and the same shared memory covers more latency.  Every TMA
// load of the pair completes on rank 0's stage barrier; rank 0's commits reach
// both CTAs' barriers; both epilogues release the accumulator on rank 0's
// barrier.  Each CTA's TMEM holds its own 128 rows of the 256 x BN tile.
//
// NSUB = 2: a unit is 256 x 2BN (two accumulators of BN columns) sharing its A
// rows; each k-block stages A once and BN rows of B per CTA, so an SM stages
// 128 + BN rows for 2 x BN columns of MMA work instead of 128 + BN/2 rows for
// BN.  CTA r holds the unit's B rows [r*BN, (r+1)*BN) as one box; MMA s takes
// rows [s*BN/2, (s+1)*BN/2) of each CTA's box, so accumulator s's columns are
// the unit's columns s*BN/2 + [0, BN/2) (from CTA 0) and BN + s*BN/2 + [0, BN/2)
// (from CTA 1).
//
// GATED (NSUB = 2): a unit is 256 x BN output columns; accumulator 0 is the
// gate projection x W1^T and accumulator 1 the up projection x W3^T of the
// same columns (CTA r loads BN/2 rows of each weight as two boxes), and the
// epilogue stores silu(gate + b1) * (up + b3).
template <int BN, bool B_MN, int STAGES, int NACC, int NSUB, bool GATED = false, bool A_MN = false,
          bool TSTORE = false>
__global__ void __launch_bounds__(kThreads, 1) umma_pair_kernel(const __grid_constant__ UmmaArgs a) {
  static_assert(!A_MN || NSUB == 1, "M-major A with one-tile units");
  umma_cta_trace(a, 30);
  static_assert(!TSTORE || (!GATED && ChunkOf<BN / 2>::v == 32), "TMA stores of 32-column float32 chunks");
  static_assert(!GATED || (NSUB == 2 && NACC == 1), "gated units are two accumulators of one tile");
  constexpr int BNH = BN / 2;
  constexpr int A_BYTES = BM * BK * 2;
  constexpr int B_SUB = BNH * BK * 2;  // one tile's B half, a multiple of 1024
  constexpr int B_BYTES = NSUB * B_SUB;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int TCOLS = TmemCols<NACC * NSUB * BN>::v;
  constexpr int HALF = BN / 2;
  constexpr int CH = ChunkOf<HALF>::v;
  constexpr int NCH = HALF / CH;
  static_assert(STAGE_BYTES % 1024 == 0 && B_SUB % 1024 == 0, "stage alignment");
  static_assert(NACC * NSUB * BN <= 512, "TMEM capacity");
  static_assert(!B_MN || BNH % 64 == 0, "MN-major B needs 64-column boxes");

  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[NACC], tempty_bar[NACC];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int s = 0; s < NACC; ++s) {
      mbar_init(smem_u32(&tfull_bar[s]), 1);
      mbar_init(smem_u32(&tempty_bar[s]), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_base_sh), TCOLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < a.nmapA && i < 8; ++i) prefetch_tmap(&a.mapA[i]);
    for (int i = 0; i < a.nmapB && i < 8; ++i) prefetch_tmap(&a.mapB[i]);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote use
  tc_fence_after();
  if (threadIdx.x == 0) umma_trace(a, 8, 0);
  const uint32_t tmem_base = tmem_base_sh;
  griddep_launch_dependents();
  // L2 prefetch of a unit part's B (weight) k-block, the boxes this CTA loads
  auto prefetch_b = [&](const UPart &P, int rowB0, int kb) {
    if (kb >= P.kblocks) return;
    if constexpr (B_MN) {
#pragma unroll
      for (int sub = 0; sub < NSUB; ++sub)
#pragma unroll
        for (int c = 0; c < BNH / 64; ++c)
          tma_prefetch_l2_2d(&a.mapB[P.bmap], rowB0 + sub * BNH + c * 64, kb * BK);
    } else if constexpr (GATED) {
      tma_prefetch_l2_2d(&a.mapB[P.bmap], kb * BK, rowB0);
      tma_prefetch_l2_2d(&a.mapB[P.bmap2], kb * BK, rowB0);
    } else {
      tma_prefetch_l2_2d(&a.mapB[P.bmap], kb * BK, rowB0);
    }
  };
  auto unit_rowB0 = [&](const UJob &J, int u) {
    const int tb = (u - J.unit_begin) / J.tilesA;
    return GATED ? tb * BN + (int)rank * BNH : tb * NSUB * BN + (int)rank * (NSUB == 2 ? BN : BNH);
  };
  // The weights are not outputs of the previous kernel, and L2 is the point
  // of coherence: the first unit's first k-blocks are pulled into L2 before
  // the programmatic-launch wait, which only starts the DRAM reads early.
  // (issued by an epilogue thread, idle until the first accumulator is ready:
  // the prefetch instructions held back the producer's first copies by 2 us)
  if (warp == 2 && lane == 0 && !A_MN && pair < a.total_units) {
    const UJob &J = a.jobs[find_job(a, pair)];
    const UPart P = a.parts[J.part0];
    for (int kb = 0; kb < STAGES; ++kb) prefetch_b(P, unit_rowB0(J, pair), kb);
  }
  griddep_wait();  // programmatic launch: no global memory before the previous kernel completes
  if (threadIdx.x == 0) umma_trace(a, 8, 1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0, pseq = 0;
      uint32_t phase = 0;
      uint32_t last_phase[STAGES];
      bool used[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) used[s] = false;
      bool ok = true;
      for (int u = pair; ok && u < a.total_units; u += npairs) {
        const UJob &J = a.jobs[find_job(a, u)];
        const int local = u - J.unit_begin;
        const int ta = local % J.tilesA, tb = local / J.tilesA;
        const int rowA0 = ta * 2 * BM + (int)rank * BM;
        const int rowB0 = GATED ? tb * BN + (int)rank * BNH : tb * NSUB * BN + (int)rank * (NSUB == 2 ? BN : BNH);
        for (int p = 0; ok && p < J.nparts; ++p) {
          const UPart P = a.parts[J.part0 + p];
          for (int kb = 0; kb < P.kblocks; ++kb) {
            if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, lim, a.status, &abort_sh)) {
              ok = false;
              break;
            }
            const uint32_t sa = sbase + stage * STAGE_BYTES, sb = sa + A_BYTES;
            const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
            if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full_bar[stage]), 2 * STAGE_BYTES);
            if constexpr (A_MN) {  // two boxes of 64 rows of M (128 bytes) x BK
              tma_load_2d_pair(sa, &a.mapA[P.amap], fb, rowA0, kb * BK);
              tma_load_2d_pair(sa + 8192, &a.mapA[P.amap], fb, rowA0 + 64, kb * BK);
            } else {
              tma_load_2d_pair(sa, &a.mapA[P.amap], fb, kb * BK, rowA0);
            }
            if constexpr (B_MN) {  // per sub-tile: BN/2 columns as 64-column boxes
#pragma unroll
              for (int sub = 0; sub < NSUB; ++sub)
#pragma unroll
                for (int c = 0; c < BNH / 64; ++c)
                  tma_load_2d_pair(sb + sub * B_SUB + c * 8192, &a.mapB[P.bmap], fb, rowB0 + sub * BNH + c * 64,
                                   kb * BK);
            } else if constexpr (GATED) {
              tma_load_2d_pair(sb, &a.mapB[P.bmap], fb, kb * BK, rowB0);  // BN/2 rows of W1
              tma_load_2d_pair(sb + B_SUB, &a.mapB[P.bmap2], fb, kb * BK, rowB0);  // and of W3
            } else {
              tma_load_2d_pair(sb, &a.mapB[P.bmap], fb, kb * BK, rowB0);  // NSUB * BN/2 rows
            }
            umma_trace(a, 1, pseq++);
            used[stage] = true;
            last_phase[stage] = phase;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
      if (!ok && rank == 0) {
        for (int s = 0; s < STAGES; ++s)
          if (used[s]) mbar_wait(smem_u32(&full_bar[s]), last_phase[s], lim, a.status, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (lane == 0 && rank == 0) {
      int stage = 0, acc = 0, mseq = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = pair; ok && u < a.total_units; u += npairs) {
        const UJob &J = a.jobs[find_job(a, u)];
        for (int p = 0; ok && p < J.nparts; ++p) {
          const UPart P = a.parts[J.part0 + p];
          if (p == 0) {
            if (!mbar_wait(smem_u32(&tempty_bar[acc]), acc_phase ^ 1, lim, a.status, &abort_sh)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t d = tmem_base + (uint32_t)(acc * NSUB * BN);
          for (int kb = 0; kb < P.kblocks; ++kb) {
            if (!mbar_wait(smem_u32(&full_bar[stage]), phase, lim, a.status, &abort_sh)) {
              ok = false;
              break;
            }
            umma_trace(a, 2, mseq);
            tc_fence_after();
            const uint32_t sa = sbase + stage * STAGE_BYTES, sb = sa + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = A_MN ? umma_desc_sw128(sa + kk * 2048, 8192, 1024)
                                       : umma_desc_sw128(sa + kk * 32, 16, 1024);
#pragma unroll
              for (int sub = 0; sub < NSUB; ++sub) {
                const uint64_t bd = B_MN ? umma_desc_sw128(sb + sub * B_SUB + kk * 2048, 8192, 1024)
                                         : umma_desc_sw128(sb + sub * B_SUB + kk * 32, 16, 1024);
                umma_f16_pair(d + (uint32_t)(sub * BN), ad, bd, a.idesc, (kb > 0 || kk > 0 || p > 0) ? 1u : 0u);
              }
            }
            umma_commit_pair(smem_u32(&empty_bar[stage]), (uint16_t)3);
            umma_trace(a, 3, mseq++);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          if (p == J.nparts - 1) {
            umma_commit_pair(smem_u32(&tfull_bar[acc]), (uint16_t)3);
            if (++acc == NACC) {
              acc = 0;
              acc_phase ^= 1;
            }
          }
        }
      }
      umma_commit_pair(smem_u32(&drain_bar), (uint16_t)1);
      mbar_wait(smem_u32(&drain_bar), 0, lim, a.status, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const uint32_t ts_bufs = sbase + (uint32_t)(STAGES * STAGE_BYTES + ew * kTsWarpBytes);
    int ts_cnt = 0;
    int acc = 0, eseq = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int u = pair; ok && u < a.total_units; u += npairs) {
      const UJob &J = a.jobs[find_job(a, u)];
      const int local = u - J.unit_begin;
      const int ta = local % J.tilesA, tb = local / J.tilesA;
      const int row = ta * 2 * BM + (int)rank * BM + quarter * 32 + lane;
      // the warp's output columns: [wcol0, wcol0 + BN) of the two accumulators
      // (NSUB = 2, not gated), else [wcol0, wcol0 + HALF)
      constexpr int WCOLS = (NSUB == 2 && !GATED) ? BN : HALF;
      const int wcol0 = (NSUB == 2 && !GATED) ? tb * 2 * BN + half * BN : tb * BN + half * HALF;
      const UOut uo = uout(a, J);
      WarpBias<(WCOLS + 31) / 32> wb, wb2;
      wb.load(J.bias, wcol0, J.rowsB, lane);
      if constexpr (GATED) wb2.load(J.bias2, wcol0, J.rowsB, lane);
      // The pair's last unit: its operand ring has drained once the
      // accumulator is complete, so the warp stages its 32 x WCOLS block
      // there and writes it with one tensor store (a warp's row-chunk stores
      // touch 32 rows each: 0.5 us per 16 columns).
      const bool rs = !A_MN && !TSTORE && a.rstore && u + npairs >= a.total_units;
      const int oes = a.out_dt == TP_F32 ? 4 : 2;
      const uint32_t rs_buf = sbase + (uint32_t)(ew * 32 * WCOLS * oes);
      const uint32_t rs_row = rs_buf + (uint32_t)(lane * WCOLS * oes);
      const bool got = mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, lim, a.status, &abort_sh);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      if (ew == 0 && lane == 0) umma_trace(a, 4, eseq);
      tc_fence_after();
      if constexpr (GATED) {
        const int colb = tb * BN + half * HALF;
        const uint32_t g_addr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(half * HALF);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float g[CH], v[CH];
          tmem_load_chunk<CH>(g_addr + c * CH, g);
          tmem_load_chunk<CH>(g_addr + BN + c * CH, v);
          tmem_wait_ld();
          wb.add<CH>(J.bias != nullptr, c * CH, g);
          wb2.add<CH>(J.bias2 != nullptr, c * CH, v);
#pragma unroll
          for (int i = 0; i < CH; ++i) v[i] = silu_f(g[i]) * v[i];
          if (rs)
            stage_row_chunk<CH>(a.out_dt, rs_row, c * CH, v);
          else
            store_row_chunk<CH, false>(uo, row, colb + c * CH, v);
        }
      }
#pragma unroll
      for (int sub = 0; sub < (GATED ? 0 : NSUB); ++sub) {
        const int colb = NSUB == 2 ? tb * 2 * BN + half * BN + sub * BNH : tb * BN + half * HALF;
        const uint32_t tb_addr = tmem_base + (uint32_t)((acc * NSUB + sub) * BN) + ((uint32_t)(quarter * 32) << 16) +
                                 (uint32_t)(half * HALF);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float v[CH];
          tmem_load_chunk<CH>(tb_addr + c * CH, v);
          tmem_wait_ld();
          if (ew == 0 && lane == 0) umma_trace(a, 6, (eseq * NSUB + sub) * 32 + c);
          wb.add<CH>(J.bias != nullptr, (NSUB == 2 ? sub * BNH : 0) + c * CH, v);
          if constexpr (TSTORE)
            tstore_chunk(a, J, find_job(a, u), row - lane, colb + c * CH, v, ts_bufs, ts_cnt, lane);
          else if (rs)
            stage_row_chunk<CH>(a.out_dt, rs_row, (NSUB == 2 && !GATED ? sub * BNH : 0) + c * CH, v);
          else
            store_row_chunk<CH, false>(uo, row, colb + c * CH, v);
          if (ew == 0 && lane == 0) umma_trace(a, 7, (eseq * NSUB + sub) * 32 + c);
        }
      }
      if (rs) {  // the block is staged: one tensor store (the map clips rows and columns outside)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row - lane < J.rowsA && wcol0 < J.rowsB) {
          tma_store_2d(&a.mapC[find_job(a, u)], rs_buf, wcol0, row - lane);
          bulk_commit_group();
        }
      }
      if (ew == 0 && lane == 0) umma_trace(a, 5, eseq);
      ++eseq;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (TSTORE || a.rstore) {
      if (lane == 0) bulk_wait_group_all();  // the tile stores have finished
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still use its memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TCOLS);
  }
  umma_cta_trace(a, 31);
}

// ====================================================================== rank clusters
// umma_row_cluster_kernel: the row-parallel GEMM with one CTA per (output
// tile, rank r), the N CTAs of a tile forming one cluster.  CTA r forms rank
// r's partial x_r W_r^T of the 128 x BN tile from zero in TMEM and parks it in
// its own shared memory; after a cluster barrier CTA r sums column slice r of
// the tile over the N partials in ascending rank order (reading its peers'
// shared memory), adds the bias once and stores.  The partials never leave
// the chip.  One unit per CTA (not persistent).
//
// MSUB = 2: the tile is 256 x BN, two 128-row sub-tiles sharing each k-block's
// B rows (two accumulators), so a k-block stages 256 + BN rows for twice the
// MMA work; the partial is parked and reduced one sub-tile at a time.
// B_MN: the weights are stored N-contiguous (K, N) and staged as BN/64 boxes
// of 64 columns (the input gradient of the column-parallel layer, dy_r W_r).
template <int BN, int STAGES, int MSUB, bool B_MN = false>
__global__ void __launch_bounds__(kThreads, 1) umma_row_cluster_kernel(const __grid_constant__ UmmaArgs a) {
  static_assert(!B_MN || BN % 64 == 0, "M/N-major B needs 64-column boxes");
  umma_cta_trace(a, 30);
  constexpr int A_SUB = BM * BK * 2;
  constexpr int A_BYTES = MSUB * A_SUB;
  constexpr int B_BYTES = BN * BK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int TCOLS = TmemCols<MSUB * BN>::v;
  constexpr int HALF = BN / 2;
  constexpr int CH = ChunkOf<HALF>::v;
  constexpr int NCH = HALF / CH;
  constexpr int RED_LD = BN + 4;  // floats per row of the parked partial
  static_assert(BM * RED_LD * 4 <= STAGES * STAGE_BYTES, "partial must fit the stage memory");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");

  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.cluster_n;
  const uint32_t rank = cluster_ctarank();
  const int tile = blockIdx.x / N;
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint64_t lim = a.wait_ns;
  const UJob &J = a.jobs[find_job(a, tile)];
  const int local = tile - J.unit_begin;
  const int ta = local % J.tilesA, tbn = local / J.tilesA;
  const int rowA0 = ta * MSUB * BM, rowB0 = tbn * BN;
  const UPart P = a.parts[J.part0 + (int)rank];

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&tfull_bar), 1);
    mbar_init(smem_u32(&drain_bar), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  griddep_launch_dependents();
  // The weights (B) are not outputs of the previous kernel, and L2 is the
  // point of coherence: their first k-blocks are pulled into L2 before the
  // programmatic-launch wait, which only starts the DRAM reads early.
  auto prefetch_b = [&](int kb) {
    if (kb >= P.kblocks) return;
    if constexpr (B_MN) {
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) tma_prefetch_l2_2d(&a.mapB[P.bmap], rowB0 + c * 64, kb * BK);
    } else {
      tma_prefetch_l2_2d(&a.mapB[P.bmap], kb * BK, rowB0);
    }
  };
  if (warp == 2 && lane == 0)  // an epilogue thread: the producer starts its copies at once
    for (int kb = 0; kb < STAGES + kPrefetchKb; ++kb) prefetch_b(kb);
  griddep_wait();  // programmatic launch: no global memory before the previous kernel completes
  if (threadIdx.x == 0) umma_trace(a, 8, 1);

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&a.mapA[P.amap]);
      prefetch_tmap(&a.mapB[P.bmap]);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t last_phase[STAGES];
      bool used[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) used[s] = false;
      bool ok = true;
      for (int kb = 0; kb < P.kblocks; ++kb) {
        if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, lim, a.status, &abort_sh)) {
          ok = false;
          break;
        }
        const uint32_t sa = sbase + stage * STAGE_BYTES, sb = sa + A_BYTES;
        const uint32_t fb = smem_u32(&full_bar[stage]);
        mbar_arrive_expect_tx(fb, STAGE_BYTES);
        // A: one box of all MSUB * 128 rows (the map's box height), B: one box
        // (K-major) or BN/64 boxes of 64 columns (N-major)
        tma_load_2d(sa, &a.mapA[P.amap], fb, kb * BK, rowA0);
        if constexpr (B_MN) {
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) tma_load_2d(sb + c * 8192, &a.mapB[P.bmap], fb, rowB0 + c * 64, kb * BK);
        } else {
          tma_load_2d(sb, &a.mapB[P.bmap], fb, kb * BK, rowB0);
        }
        prefetch_b(kb + STAGES + kPrefetchKb);  // keeps the weight stream ahead of the ring
        umma_trace(a, 1, kb);
        used[stage] = true;
        last_phase[stage] = phase;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok)
        for (int s = 0; s < STAGES; ++s)
          if (used[s]) mbar_wait(smem_u32(&full_bar[s]), last_phase[s], lim, a.status, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < P.kblocks; ++kb) {
        if (!mbar_wait(smem_u32(&full_bar[stage]), phase, lim, a.status, &abort_sh)) break;
        umma_trace(a, 2, kb);
        tc_fence_after();
        const uint32_t sa = sbase + stage * STAGE_BYTES, sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
#pragma unroll
          for (int m = 0; m < MSUB; ++m)
            umma_f16(tmem_base + (uint32_t)(m * BN), umma_desc_sw128(sa + m * A_SUB + kk * 32, 16, 1024),
                     B_MN ? umma_desc_sw128(sb + kk * 2048, 8192, 1024) : umma_desc_sw128(sb + kk * 32, 16, 1024),
                     a.idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        umma_commit(smem_u32(&empty_bar[stage]));
        umma_trace(a, 3, kb);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      umma_commit(smem_u32(&tfull_bar));
      umma_commit(smem_u32(&drain_bar));
      mbar_wait(smem_u32(&drain_bar), 0, lim, a.status, nullptr);
    }
  }

  // Per 128-row sub-tile: park this rank's partial in shared memory (row-major,
  // padded rows), cluster barrier, sum column slice `rank` over the ranks in
  // order and store, cluster barrier (peers are done reading before the next
  // sub-tile is parked over it).
  bool got = true;
  // The 4 bias values of the columns an epilogue thread stores: with 256
  // threads over rows of BN / N / 4 items the column is the same for every
  // item of the thread, so they are loaded once, before the wait.
  const int slice = BN / N;
  const int per_row = slice / 4;
  const int tcol = (int)rank * slice + (((int)threadIdx.x - 64) % per_row) * 4;
  float bcol[4] = {0.f, 0.f, 0.f, 0.f};
  const UOut uo = uout(a, J);
  if (warp >= 2 && J.bias) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (rowB0 + tcol + i < J.rowsB) bcol[i] = __ldg(J.bias + rowB0 + tcol + i);
  }
  if (warp >= 2) {
    got = mbar_wait(smem_u32(&tfull_bar), 0, lim, a.status, &abort_sh);
    got = __all_sync(0xffffffffu, got);
  }
  for (int m = 0; m < MSUB; ++m) {
    if (warp == 2 && lane == 0) umma_trace(a, 4, m);
    if (warp >= 2 && got) {
      const int quarter = warp & 3;
      const int half = (warp - 2) >> 2;
      const int row = quarter * 32 + lane;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(m * BN) + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(half * HALF);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        float v[CH];
        tmem_load_chunk<CH>(taddr + c * CH, v);
        tmem_wait_ld();
        const uint32_t dst = sbase + (uint32_t)((row * RED_LD + half * HALF + c * CH) * 4);
#pragma unroll
        for (int i = 0; i < CH; i += 4)
          asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(dst + i * 4), "f"(v[i]),
                       "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3])
                       : "memory");
      }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // every rank's partial of sub-tile m is parked
    if (warp == 2 && lane == 0) umma_trace(a, 9, m);

    if (warp >= 2) {
      // column slice `rank` of the sub-tile: sum over ranks 0..N-1 in order, then bias
      const int t = threadIdx.x - 64;
      for (int idx = t; idx < BM * per_row; idx += 256) {
        const int r = idx / per_row;
        const int c = (int)rank * slice + (idx - r * per_row) * 4;
        const uint32_t off = sbase + (uint32_t)((r * RED_LD + c) * 4);
        float4 acc = ld_cluster_f4(mapa_shared(off, 0));
        for (int q = 1; q < N; ++q) {
          const float4 v = ld_cluster_f4(mapa_shared(off, (uint32_t)q));
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        float o[4] = {acc.x, acc.y, acc.z, acc.w};
        if (J.bias) {
          if (c == tcol) {
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] += bcol[i];
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (rowB0 + c + i < J.rowsB) o[i] += __ldg(J.bias + rowB0 + c + i);
          }
        }
        store_row_chunk<4, false>(uo, rowA0 + m * BM + r, rowB0 + c, o);
      }
      if (warp == 2 && lane == 0) umma_trace(a, 5, m);
    }
    if (m + 1 < MSUB) {
      __syncthreads();
      cluster_sync_all();  // peers are done reading sub-tile m
    }
  }

  __syncthreads();
  cluster_sync_all();  // peers stop reading this CTA's shared memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TCOLS);
  }
  umma_cta_trace(a, 31);
}

// ====================================================================== host
namespace {

std::mutex g_mu;

// 2-D bf16/f16 row-major tensor map, 128B swizzle.
int make_map(CUtensorMap *out, const void *ptr, int dt, uint64_t inner, uint64_t outer, uint64_t ld,
             uint32_t box0, uint32_t box1) {
  return make_tmap_2d(out, ptr,
                      dt == TP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      2, inner, outer, ld, box0, box1, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int BN, bool B_MN, bool SWAP, bool PARTIALS, int STAGES, int NACC, bool A_MN = false>
int launch_config(UmmaArgs &args, int sms, cudaStream_t s) {
  auto kern = umma_gemm_kernel<BN, B_MN, SWAP, PARTIALS, STAGES, NACC, A_MN>;
  constexpr int smem = STAGES * (BM * BK * 2 + BN * BK * 2) + 1024;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
    attr_done[dev & 63] = true;
  }
  const int grid = args.total_units < sms ? args.total_units : sms;
  cudaError_t e = launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, s, args);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "umma_gemm_kernel launch");
}

template <int BN, bool B_MN, int STAGES, int NACC, int NSUB, bool GATED = false, bool A_MN = false,
          bool TSTORE = false>
int launch_pair(UmmaArgs &args, int sms, cudaStream_t s) {
  auto kern = umma_pair_kernel<BN, B_MN, STAGES, NACC, NSUB, GATED, A_MN, TSTORE>;
  constexpr int ring = STAGES * (BM * BK * 2 + NSUB * (BN / 2) * BK * 2);
  constexpr int smem = ring + 1024 + (TSTORE ? kEpiWarps * kTsWarpBytes : 0);
  // Ring-staged tensor stores of each pair's last unit: a warp's block is 32
  // rows x WCOLS columns (the warp's columns, as in the epilogue); every
  // warp's block must fit the ring, and every output's base and rows must
  // allow tensor stores.
  args.rstore = 0;
  if (!A_MN && !TSTORE && args.njobs <= kMaxCMaps) {
    constexpr int WCOLS = (NSUB == 2 && !GATED) ? BN : BN / 2;
    const int oes = args.out_dt == TP_F32 ? 4 : 2;
    bool ok = kEpiWarps * 32 * WCOLS * oes <= ring && (WCOLS * oes) % 16 == 0;
    for (int j = 0; ok && j < args.njobs; ++j)
      ok = ((uintptr_t)args.jobs[j].C % 16) == 0 && (args.jobs[j].ldc * oes) % 16 == 0;
    for (int j = 0; ok && j < args.njobs; ++j) {
      const UJob &J = args.jobs[j];
      const CUtensorMapDataType dt = args.out_dt == TP_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : args.out_dt == TP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
      if (make_tmap_2d(&args.mapC[j], J.C, dt, oes, (uint64_t)J.rowsB, (uint64_t)J.rowsA, (uint64_t)J.ldc,
                       (uint32_t)WCOLS, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        ok = false;
    }
    args.rstore = ok ? 1 : 0;
  }
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(pair)");
    attr_done[dev & 63] = true;
  }
  const int max_pairs = sms / 2;
  const int pairs = args.total_units < max_pairs ? args.total_units : max_pairs;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "umma_pair_kernel launch");
}

template <int BN, int STAGES, int MSUB, bool B_MN = false>
int launch_row_cluster(UmmaArgs &args, cudaStream_t s) {
  auto kern = umma_row_cluster_kernel<BN, STAGES, MSUB, B_MN>;
  constexpr int smem = STAGES * (MSUB * BM * BK * 2 + BN * BK * 2) + 1024;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(row cluster)");
    attr_done[dev & 63] = true;
  }
  const int N = args.cluster_n;
  const int64_t tiles = args.total_units;
  if (tiles * N > INT32_MAX) return set_error(TP_ERR_UNSUPPORTED, "too many tiles");
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)(tiles * N), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)N;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "umma_row_cluster_kernel launch");
}

bool al16(const void *p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

int launch_umma(const Problem &p, cudaStream_t s, bool *handled) {
  *handled = false;
  if (p.in_dt != TP_BF16 && p.in_dt != TP_F16) return TP_OK;
  if (p.b_layout != BL_KMAJOR && p.b_layout != BL_MNMAJOR) return TP_OK;
  // M-major A only with M-major B (weight gradients, SUMMA's A^T B), chained.
  if (p.a_mn && (p.b_layout != BL_MNMAJOR || !p.chain)) return TP_OK;
  // Gated products run only on the CTA-pair kernel.
  if (p.gated && (p.b_layout != BL_KMAJOR || !p.chain || !pair_policy_allowed() || sm_count() < 2))
    return TP_OK;
  // TMA needs 16-byte aligned bases and row strides; else the CUDA-core path.
  int64_t maxM = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    if (J.M > INT32_MAX / 2 || J.N > INT32_MAX / 2) return TP_OK;
    if (J.M > maxM) maxM = J.M;
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      if (!al16(P.A) || !al16(P.B) || (P.lda % 8) || (P.ldb % 8)) return TP_OK;
      if (p.gated && !al16(P.B2)) return TP_OK;
    }
  }
  const bool summa = p.b_layout == BL_MNMAJOR;
  const bool swap = !summa && maxM <= 16 && !p.gated;
  const bool partials = !p.chain;
  // Kernel and tile choice.  Per k-block a tile costs about
  // max(MMA cycles, 2.2 x the operand rows one CTA stages): a CTA can keep
  // only so many bytes in flight, so the staged rows set the pace once the
  // MMA is fast enough.  Rounds of tiles over the SMs multiply that.
  int BN, nsub = 1, msub = 1, splits = 1;
  bool pair = false, rowclu = false;
  if (swap) {
    BN = 16;
    // Small batches: a unit streams a 128-row weight tile through one SM at
    // about 38 GB/s (0.48 us per 64-column k-block, plus about 1.5 us per
    // unit, measured), so with fewer tiles than SMs most of HBM sits idle,
    // and a last round of tiles that covers only part of the SMs leaves the
    // rest idle.
    // Split each tile's contraction into S k-block ranges (float32 slots
    // that the last-arriving unit of the tile adds in order: about 1 us plus
    // the slot traffic) when that shortens the longest SM's queue.
    const int sms0 = sm_count();
    int64_t tiles = 0, kbw = 1;
    for (int j = 0; j < p.njobs; ++j) {
      int64_t kb = 0;
      for (int q = 0; q < p.jobs[j].nparts; ++q) kb += (p.parts[p.jobs[j].part0 + q].K + BK - 1) / BK;
      kbw = std::max(kbw, kb);
      tiles += ((p.jobs[j].N + BM - 1) / BM) * ((p.jobs[j].M + BN - 1) / BN);
    }
    int64_t maxT = 1;
    for (int j = 0; j < p.njobs; ++j) maxT = std::max<int64_t>(maxT, std::min<int64_t>(p.jobs[j].M, BN));
    if (kbw >= 2) {
      double best = 1e300;
      for (int sp = 1; sp <= 16 && sp <= kbw; ++sp) {
        const double rounds = (double)((tiles * sp + sms0 - 1) / sms0);
        const double slot_us = sp > 1 ? 2.0 * (double)(tiles * sp * maxT * BM * 4) / 6.0e6 : 0.0;
        const double cost =
            rounds * ((double)((kbw + sp - 1) / sp) * 0.48 + 1.5) + (sp > 1 ? 1.0 + slot_us : 0.0);
        if (cost < best - 1e-9) {
          best = cost;
          splits = sp;
        }
      }
    }
  } else if (p.gated) {
    // Pair units of 256 x BN outputs with two accumulators (gate, up): per
    // k-block a CTA stages 128 + BN rows for 2 x BN columns of MMA work, and
    // the epilogue (one accumulator set) is exposed once per unit.
    const int sms0 = sm_count();
    int64_t kbw = 1;
    for (int j = 0; j < p.njobs; ++j) {
      int64_t kb = 0;
      for (int q = 0; q < p.jobs[j].nparts; ++q) kb += (p.parts[p.jobs[j].part0 + q].K + BK - 1) / BK;
      if (kb > kbw) kbw = kb;
    }
    double best = 1e300;
    BN = 256;
    for (int bn : {256, 192, 160}) {
      int64_t units = 0;
      for (int j = 0; j < p.njobs; ++j)
        units += ((p.jobs[j].M + 2 * BM - 1) / (2 * BM)) * ((p.jobs[j].N + bn - 1) / bn);
      const double rounds = (double)((units + sms0 / 2 - 1) / (sms0 / 2));
      const double per_kb = std::max(4.0 * bn, 2.2 * (128.0 + bn));
      const double cost = rounds * ((double)kbw * per_kb + 6000.0);
      if (cost < best - 1e-9) {
        best = cost;
        BN = bn;
      }
    }
    pair = true;
    nsub = 2;
  } else if (partials) {
    BN = 128;
    // Rank clusters (one CTA per rank of a 128 x 256 tile) when one CTA per
    // 128 x 128 tile would leave SMs idle; costs in cycles, measured rates.
    const int sms0 = sm_count();
    if (pair_policy_allowed() && !p.a_mn) {
      // Every job (one per output block: several for a reduce-scatter) must
      // have the same rank count and every part the same K.
      const int N = p.jobs[0].nparts;
      const int64_t K0 = p.parts[p.jobs[0].part0].K;
      bool same_k = true;
      int64_t mt = 0, mt2 = 0, t128 = 0;  // 128x256, 256x256 and 128x128 tiles
      for (int j = 0; j < p.njobs; ++j) {
        const Job &J = p.jobs[j];
        same_k = same_k && J.nparts == N;
        for (int q = 0; q < J.nparts; ++q) same_k = same_k && p.parts[J.part0 + q].K == K0;
        const int64_t m1 = (J.M + BM - 1) / BM, m2 = (J.M + 2 * BM - 1) / (2 * BM);
        mt += m1 * ((J.N + 255) / 256);
        mt2 += m2 * ((J.N + 255) / 256);
        t128 += m1 * ((J.N + 127) / 128);
      }
      const double kb = (double)((K0 + BK - 1) / BK);
      // Measured: 4-rank clusters win on long K (MLP 2752 per rank); 8-rank
      // clusters and short K lose to the fixed per-CTA cost of this kernel.
      // msub = 2: 256 x 256 tiles (two row sub-tiles sharing B; 64 KB
      // k-blocks, about 4/3 the time of a 48 KB one, and two reduce rounds).
      // Clusters of four CTAs: 144 of the 152 SMs can hold them at once.
      if (N >= 2 && N <= 4 && kb >= 32 && (256 % N) == 0 && same_k) {
        const int64_t resident = N == 4 ? sms0 / 152.0 * 144 : sms0;
        const double single = (double)((t128 + sms0 - 1) / sms0) * N * kb * 720.0;
        const double clu1 = (double)((mt * N + resident - 1) / resident) * (kb * 850.0 + 12000.0);
        const double clu2 = (double)((mt2 * N + resident - 1) / resident) * (kb * 1133.0 + 24000.0);
        if (std::min(clu1, clu2) < single) {
          rowclu = true;
          BN = 256;
          msub = clu2 < clu1 ? 2 : 1;
        }
      }
    }
  } else {
    // Candidates: one CTA or a CTA pair per unit, a unit one tile or (pairs)
    // two neighbouring tiles sharing A (nsub = 2, one accumulator set, so its
    // epilogue is not hidden behind the next unit's main loop: about 5000
    // cycles).  Cost: rounds x (k-blocks x per-k-block cost + exposed
    // epilogue).
    const int sms0 = sm_count();
    const bool allow_pair = pair_policy_allowed() && sms0 >= 2;
    int64_t kbw = 1;  // k-blocks of one unit (the chained parts together)
    for (int j = 0; j < p.njobs; ++j) {
      int64_t kb = 0;
      for (int q = 0; q < p.jobs[j].nparts; ++q) kb += (p.parts[p.jobs[j].part0 + q].K + BK - 1) / BK;
      if (kb > kbw) kbw = kb;
    }
    double best = 1e300;
    BN = 256;
    for (int pm = 0; pm < (allow_pair ? 2 : 1); ++pm) {
      for (int ns = 1; ns <= 2; ++ns) {
        if (ns == 2 && (!pm || p.a_mn)) continue;
        for (int bn : {256, 192, 160}) {
          if (summa && bn != 256) continue;
          const int64_t mrows = pm ? 2 * BM : BM;
          int64_t units = 0;
          for (int j = 0; j < p.njobs; ++j)
            units += ((p.jobs[j].M + mrows - 1) / mrows) * ((p.jobs[j].N + ns * bn - 1) / (ns * bn));
          const int64_t slots = pm ? sms0 / 2 : sms0;
          const double rounds = (double)((units + slots - 1) / slots);
          const double per_kb = std::max(2.0 * bn * ns, 2.2 * (128.0 + ns * (pm ? bn / 2 : bn)));
          const double epi = 5000.0;
          const double cost = rounds * (double)kbw * per_kb + (ns == 2 ? rounds * epi : epi);
          if (cost < best - 1e-9) {
            best = cost;
            BN = bn;
            pair = pm == 1;
            nsub = ns;
          }
        }
      }
    }
  }

  std::lock_guard<std::mutex> lk(g_mu);
  int rc = TP_OK;
  const int sms = sm_count();

  static UmmaArgs args;  // large; guarded by g_mu
  memset(&args, 0, sizeof(args));
  int nA = 0, nB = 0;
  const void *aptr[kMaxMaps], *bptr[kMaxMaps];
  int64_t units = 0, tiles_so_far = 0;
  for (int j = 0; j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    UJob &U = args.jobs[j];
    U.C = J.C;
    U.bias = J.bias;
    U.ldc = J.ldc;
    U.rowsA = (int)(swap ? J.N : J.M);
    U.rowsB = (int)(swap ? J.M : J.N);
    U.part0 = J.part0;
    U.nparts = J.nparts;
    U.tilesA = (U.rowsA + (pair || msub == 2 ? 2 * BM : BM) - 1) / (pair || msub == 2 ? 2 * BM : BM);
    U.tilesB = p.gated ? (U.rowsB + BN - 1) / BN : (U.rowsB + nsub * BN - 1) / (nsub * BN);
    U.bias2 = J.bias2;
    U.unit_begin = (int)units;
    U.splits = splits;
    U.kb_total = 0;
    for (int q = 0; q < J.nparts; ++q) U.kb_total += (int)((p.parts[J.part0 + q].K + BK - 1) / BK);
    U.ws_base = U.unit_begin;  // split mode: one slot per unit
    U.cnt_base = (int)tiles_so_far;
    tiles_so_far += (int64_t)U.tilesA * U.tilesB;
    units += (int64_t)U.tilesA * U.tilesB * splits;
    for (int q = 0; q < J.nparts; ++q) {
      const Part &P = p.parts[J.part0 + q];
      // operand roles: normal A = activations (M rows), B = weights / SUMMA block
      const void *opA = swap ? P.B : P.A;
      const void *opB = swap ? P.A : P.B;
      const int64_t ldA = swap ? P.ldb : P.lda, ldB = swap ? P.lda : P.ldb;
      int ia = -1, ib = -1, ib2 = -1;
      for (int i = 0; i < nA; ++i)
        if (aptr[i] == opA) ia = i;
      for (int i = 0; i < nB; ++i) {
        if (bptr[i] == opB) ib = i;
        if (p.gated && bptr[i] == P.B2) ib2 = i;
      }
      if (ia < 0) {
        if (nA == kMaxMaps) return TP_OK;
        // the rank clusters with 256-row tiles load A as one 256-row box
        if (p.a_mn)  // A stored (K, M) row-major: inner = M, boxes of 64 x BK
          rc = make_map(&args.mapA[nA], opA, p.in_dt, (uint64_t)U.rowsA, (uint64_t)P.K, (uint64_t)ldA, 64, BK);
        else
          rc = make_map(&args.mapA[nA], opA, p.in_dt, (uint64_t)P.K, (uint64_t)U.rowsA, (uint64_t)ldA, BK,
                        rowclu ? msub * BM : BM);
        if (rc) return rc;
        aptr[nA] = opA;
        ia = nA++;
      }
      if (ib < 0) {
        if (nB == kMaxMaps) return TP_OK;
        if (summa)  // B block (K, Nblk) row-major: inner = N
          rc = make_map(&args.mapB[nB], opB, p.in_dt, (uint64_t)U.rowsB, (uint64_t)P.K, (uint64_t)ldB, 64, BK);
        else
          rc = make_map(&args.mapB[nB], opB, p.in_dt, (uint64_t)P.K, (uint64_t)U.rowsB, (uint64_t)ldB, BK,
                        (uint32_t)(pair ? (p.gated ? BN / 2 : nsub * BN / 2) : BN));
        if (rc) return rc;
        bptr[nB] = opB;
        ib = nB++;
        if (p.gated && P.B2 == opB) ib2 = ib;
      }
      if (p.gated && ib2 < 0) {
        if (nB == kMaxMaps) return TP_OK;
        rc = make_map(&args.mapB[nB], P.B2, p.in_dt, (uint64_t)P.K, (uint64_t)U.rowsB, (uint64_t)ldB, BK,
                      (uint32_t)(BN / 2));
        if (rc) return rc;
        bptr[nB] = P.B2;
        ib2 = nB++;
      }
      args.parts[J.part0 + q] =
          UPart{(int16_t)ia, (int16_t)ib, (int32_t)((P.K + BK - 1) / BK), (int16_t)(ib2 < 0 ? 0 : ib2)};
    }
  }
  if (units == 0) {
    *handled = true;
    return TP_OK;
  }
  if (units > INT32_MAX) return TP_OK;
  args.njobs = p.njobs;
  args.nmapA = nA;
  args.nmapB = nB;
  args.total_units = (int)units;
  args.cluster_n = rowclu ? p.jobs[0].nparts : 1;
  {
    int64_t cap = 0;
    trace_buffer(&args.trace, &cap);
  }
  args.chain = p.chain;
  args.out_dt = p.out_dt;
  const int oe = p.out_dt == TP_F32 ? 4 : 2;
  int vec = 1;
  for (int j = 0; j < p.njobs; ++j)
    if (!al16(p.jobs[j].C) || ((p.jobs[j].ldc * oe) % 16)) vec = 0;
  args.vec_ok = vec;
  // TMA-store epilogue (M-major-A pair units, whose short contraction leaves
  // the float32 output stores as the critical path): float32 outputs with
  // 16-byte aligned bases and rows.
  bool tstore = pair && summa && p.a_mn && p.out_dt == TP_F32 && p.njobs <= kMaxCMaps;
  for (int j = 0; tstore && j < p.njobs; ++j)
    tstore = al16(p.jobs[j].C) && (p.jobs[j].ldc % 4) == 0;
  for (int j = 0; tstore && j < p.njobs; ++j) {
    const Job &J = p.jobs[j];
    rc = make_tmap_2d(&args.mapC[j], J.C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)J.N, (uint64_t)J.M,
                      (uint64_t)J.ldc, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  args.idesc = umma_idesc_f16(p.in_dt == TP_BF16 ? 1u : 0u, summa ? 1u : 0u, pair ? 2 * BM : BM, (uint32_t)BN,
                              p.a_mn ? 1u : 0u);
  args.status = p.status;
  args.wait_ns = (uint64_t)p.wait_ns;
  if (splits > 1) {
    rc = split_workspace(s, (size_t)units * BM * BN * sizeof(float), (size_t)tiles_so_far * kEpiWarps, &args.ws,
                         &args.cnt);
    if (rc) return rc;
  }

  if (p.gated && BN == 160)
    rc = launch_pair<160, false, 6, 1, 2, true>(args, sms, s);
  else if (p.gated && BN == 192)
    rc = launch_pair<192, false, 5, 1, 2, true>(args, sms, s);
  else if (p.gated)
    rc = launch_pair<256, false, 4, 1, 2, true>(args, sms, s);
  else if (rowclu && msub == 2 && summa)
    rc = launch_row_cluster<256, 3, 2, true>(args, s);
  else if (rowclu && summa)
    rc = launch_row_cluster<256, 4, 1, true>(args, s);
  else if (rowclu && msub == 2)
    rc = launch_row_cluster<256, 3, 2>(args, s);
  else if (rowclu)
    rc = launch_row_cluster<256, 4, 1>(args, s);
  else if (pair && summa && p.a_mn && tstore)
    rc = launch_pair<256, true, 6, 2, 1, false, true, true>(args, sms, s);
  else if (pair && summa && p.a_mn)
    rc = launch_pair<256, true, 6, 2, 1, false, true>(args, sms, s);
  else if (pair && summa && nsub == 2)
    rc = launch_pair<256, true, 4, 1, 2>(args, sms, s);
  else if (pair && summa)
    rc = launch_pair<256, true, 7, 2, 1>(args, sms, s);
  else if (pair && nsub == 2 && BN == 160)
    rc = launch_pair<160, false, 6, 1, 2>(args, sms, s);
  else if (pair && nsub == 2 && BN == 192)
    rc = launch_pair<192, false, 5, 1, 2>(args, sms, s);
  else if (pair && nsub == 2)
    rc = launch_pair<256, false, 4, 1, 2>(args, sms, s);
  else if (pair && BN == 160)
    rc = launch_pair<160, false, 8, 2, 1>(args, sms, s);
  else if (pair && BN == 192)
    rc = launch_pair<192, false, 7, 2, 1>(args, sms, s);
  else if (pair)
    rc = launch_pair<256, false, 6, 2, 1>(args, sms, s);
  else if (summa && partials)
    rc = launch_config<128, true, false, true, 6, 4>(args, sms, s);
  else if (summa && p.a_mn)
    rc = launch_config<256, true, false, false, 4, 2, true>(args, sms, s);
  else if (summa)
    rc = launch_config<256, true, false, false, 4, 2>(args, sms, s);
  else if (swap && partials)
    rc = launch_config<16, false, true, true, 8, 4>(args, sms, s);
  else if (swap)
    rc = launch_config<16, false, true, false, 8, 4>(args, sms, s);
  else if (partials)
    rc = launch_config<128, false, false, true, 6, 4>(args, sms, s);
  else if (BN == 160)
    rc = launch_config<160, false, false, false, 6, 2>(args, sms, s);
  else if (BN == 192)
    rc = launch_config<192, false, false, false, 5, 2>(args, sms, s);
  else
    rc = launch_config<256, false, false, false, 4, 2>(args, sms, s);
  if (rc == TP_OK) *handled = true;
  return rc;
}

void umma_shutdown() {
  tmap_cache_clear();
  split_workspace_free();
}

}  // namespace tp
