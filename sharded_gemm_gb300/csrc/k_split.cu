// k_split.cu -- ordered sum of split-K partial tiles, shared by the
// quantized tensor-core kernels.
//
// A split tile is 128 output rows x BN token columns; each of its `splits`
// partials is a float32 slot stored column-major (slot[c][m], so a warp's 32
// rows of one column are one 128-byte line).  out[t][row] = (slot_0 + slot_1
// + ... in split order, which is rank order for the row-parallel layer) +
// bias, one thread per output element.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include <algorithm>

#include "ptx.cuh"
#include "tp_internal.h"

namespace tp {
namespace {

struct SrJob {
  SplitJob j;
  int64_t item0;  // first item of this job
};
struct SrArgs {
  SrJob jobs[kMaxJobs];
  const float *ws;
  int njobs, BN, out_dt;
  int64_t nitems;
  unsigned long long *trace;  // optional: block start (event 21) and end (event 22) times
};

template <int DT, int VW>
__device__ __forceinline__ void sr_store(void *C, int64_t idx, const float (&v)[VW], int n) {
  constexpr int ES = DT == TP_F32 ? 4 : 2;
  // the vector store needs the whole group and its address VW-element aligned
  if (n == VW && (VW == 1 || (reinterpret_cast<uintptr_t>(static_cast<char *>(C) + idx * ES) % (VW * ES)) == 0)) {
    if (DT == TP_F32) {
      if constexpr (VW == 4)
        *reinterpret_cast<float4 *>(static_cast<float *>(C) + idx) = make_float4(v[0], v[1], v[2], v[3]);
      else
        static_cast<float *>(C)[idx] = v[0];
    } else {
      uint16_t h[VW];
#pragma unroll
      for (int i = 0; i < VW; ++i)
        h[i] = DT == TP_BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v[i])) : __half_as_ushort(__float2half_rn(v[i]));
      if constexpr (VW == 4)
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(C) + idx) =
            make_uint2((uint32_t)h[0] | ((uint32_t)h[1] << 16), (uint32_t)h[2] | ((uint32_t)h[3] << 16));
      else
        static_cast<uint16_t *>(C)[idx] = h[0];
    }
    return;
  }
  for (int i = 0; i < n; ++i) {
    if (DT == TP_F32)
      static_cast<float *>(C)[idx + i] = v[i];
    else if (DT == TP_BF16)
      static_cast<__nv_bfloat16 *>(C)[idx + i] = __float2bfloat16_rn(v[i]);
    else
      static_cast<__half *>(C)[idx + i] = __float2half_rn(v[i]);
  }
}

// One item = VW consecutive output rows (VW = 4 or 1) of one token column:
// one VW-float load per split (a warp reads 32 VW floats of a slot column
// at once), the splits added in order, then the bias and one store.  With
// VW = 4 (large sums: many items, high occupancy) the split loop is unrolled
// by 8; with VW = 1 (small sums over many splits) all loads of up to 16
// splits are issued before the adds, so the sum takes one round trip to L2.
template <int DT, int VW>
__global__ void __launch_bounds__(256, VW == 4 ? 6 : 3) split_reduce_kernel(const __grid_constant__ SrArgs a) {
  griddep_launch_dependents();
  griddep_wait();  // the slots are written by the kernel before this one
  if (a.trace != nullptr && threadIdx.x == 0 && blockIdx.x < 1024) a.trace[16 + 21 * 1024 + blockIdx.x] = globaltimer_ns();
  constexpr int LPC = 128 / VW;  // items per column of a tile
  const int per_tile_items = a.BN * LPC;
  const int64_t per_tile = (int64_t)a.BN * 128;
  // Every item count is a multiple of 32 and so is the stride: the 32 lanes
  // of a warp take 32 consecutive items of one column of one tile together.
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < a.nitems;
       it += (int64_t)gridDim.x * blockDim.x) {
    int j = 0;
    while (j + 1 < a.njobs && it >= a.jobs[j + 1].item0) ++j;
    const SplitJob &J = a.jobs[j].j;
    const int64_t local = it - a.jobs[j].item0;
    const int64_t tile_lin = local / per_tile_items;
    const int rem = (int)(local - tile_lin * per_tile_items);
    const int c = rem / LPC, m = (rem % LPC) * VW;
    const int tile = (int)(tile_lin % J.tiles), ntile = (int)(tile_lin / J.tiles);
    const int orow = tile * 128 + m;
    const int t = ntile * a.BN + c;
    const int splits = J.splits;
    const float *s0 = a.ws + (J.ws_base + tile_lin * splits) * per_tile + (int64_t)c * 128 + m;
    // slots past the tokens or rows may be unwritten: not read, not stored
    const bool in = orow < J.rows && t < J.T;
    if (in) {
      float acc[VW];
      if constexpr (VW == 4) {
        // many items at once: one 16-byte load per split, unrolled by 8
        float4 a4 = __ldcg(reinterpret_cast<const float4 *>(s0));
#pragma unroll 8
        for (int sp = 1; sp < splits; ++sp) {
          const float4 f = __ldcg(reinterpret_cast<const float4 *>(s0 + (int64_t)sp * per_tile));
          a4.x += f.x;
          a4.y += f.y;
          a4.z += f.z;
          a4.w += f.w;
        }
        acc[0] = a4.x;
        acc[1] = a4.y;
        acc[2] = a4.z;
        acc[3] = a4.w;
      } else {
        // few items, many splits: every split's load in flight at once
        acc[0] = __ldcg(s0);
        for (int sp0 = 1; sp0 < splits; sp0 += 16) {
          float f[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (sp0 + i < splits) f[i] = __ldcg(s0 + (int64_t)(sp0 + i) * per_tile);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (sp0 + i < splits) acc[0] += f[i];
        }
      }
      const int n = J.rows - orow < VW ? J.rows - orow : VW;
      if (J.bias)
        for (int e = 0; e < n; ++e) acc[e] += __ldg(J.bias + orow + e);
      sr_store<DT, VW>(J.C, (int64_t)t * J.ldc + orow, acc, n);
    }
    // The slots are scratch: once every lane of the warp has read its part,
    // the first lane of each 128-byte line drops it from L2 without a
    // write-back (the partials never need to reach DRAM).
    __syncwarp();
    if ((m & 31) == 0)
      for (int sp = 0; sp < splits; ++sp) l2_discard_line(s0 + (int64_t)sp * per_tile);
  }
  if (a.trace != nullptr && threadIdx.x == 0 && blockIdx.x < 1024) a.trace[16 + 22 * 1024 + blockIdx.x] = globaltimer_ns();
}

}  // namespace

int launch_split_reduce(const SplitJob *jobs, int njobs, const float *ws, int BN, int out_dt, cudaStream_t s) {
  SrArgs a;
  memset(&a, 0, sizeof(a));
  int64_t outs = 0;
  for (int j = 0; j < njobs; ++j)
    if (jobs[j].splits > 1) outs += (int64_t)jobs[j].tiles * jobs[j].ntiles * BN * 128;
  if (outs == 0) return TP_OK;
  // one row per thread for a small sum over more than 8 splits (a decode's
  // long contraction), four rows per thread otherwise
  const int sms = sm_count();
  int max_splits = 0;
  for (int j = 0; j < njobs; ++j) max_splits = std::max(max_splits, jobs[j].splits);
  const int VW = (max_splits > 8 && outs <= ((int64_t)1 << 20)) ? 1 : 4;
  int64_t items = 0;
  for (int j = 0; j < njobs; ++j) {
    a.jobs[j].j = jobs[j];
    a.jobs[j].item0 = items;
    if (jobs[j].splits > 1) items += (int64_t)jobs[j].tiles * jobs[j].ntiles * BN * (128 / VW);
  }
  a.ws = ws;
  a.njobs = njobs;
  a.BN = BN;
  a.out_dt = out_dt;
  a.nitems = items;
  int64_t trace_cap = 0;
  trace_buffer(&a.trace, &trace_cap);
  const int grid = (int)std::min<int64_t>((items + 255) / 256, (int64_t)sms * 16);
  cudaError_t e;
  if (VW == 4) {
    if (out_dt == TP_F32)
      e = launch_pdl(split_reduce_kernel<TP_F32, 4>, dim3(grid), dim3(256), 0, s, a);
    else if (out_dt == TP_BF16)
      e = launch_pdl(split_reduce_kernel<TP_BF16, 4>, dim3(grid), dim3(256), 0, s, a);
    else
      e = launch_pdl(split_reduce_kernel<TP_F16, 4>, dim3(grid), dim3(256), 0, s, a);
  } else {
    if (out_dt == TP_F32)
      e = launch_pdl(split_reduce_kernel<TP_F32, 1>, dim3(grid), dim3(256), 0, s, a);
    else if (out_dt == TP_BF16)
      e = launch_pdl(split_reduce_kernel<TP_BF16, 1>, dim3(grid), dim3(256), 0, s, a);
    else
      e = launch_pdl(split_reduce_kernel<TP_F16, 1>, dim3(grid), dim3(256), 0, s, a);
  }
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "split_reduce_kernel launch");
}

}  // namespace tp
