// k_split.cu -- ordered sum of split-K partial tiles, shared by the
// quantized tensor-core kernels.
//
// A split tile is 128 output rows x BN token columns; each of its `splits`
// partials is a float32 slot stored column-major (slot[c][m], so a warp's 32
// rows of one column are one 128-byte line).  out[t][row] = (slot_0 + slot_1
// + ... in split order, which is rank order for the row-parallel layer) +
// bias, one thread per 4 consecutive rows of one token column.
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
  int njobs, BN, out_dt, vec_out;
  int64_t nitems;
};

template <int DT>
__device__ __forceinline__ void sr_store4(void *C, int64_t idx, const float (&v)[4], int n, bool vec) {
  if (vec && n == 4) {
    if (DT == TP_F32) {
      *reinterpret_cast<float4 *>(static_cast<float *>(C) + idx) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
      uint16_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        h[i] = DT == TP_BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v[i])) : __half_as_ushort(__float2half_rn(v[i]));
      *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(C) + idx) =
          make_uint2((uint32_t)h[0] | ((uint32_t)h[1] << 16), (uint32_t)h[2] | ((uint32_t)h[3] << 16));
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

// One item = 4 consecutive output rows of one token column: one 16-byte load
// per split (a warp reads 512 contiguous bytes of a slot column), the splits
// added in order, then bias and one 8- or 16-byte store.
template <int DT>
__global__ void __launch_bounds__(256) split_reduce_kernel(const __grid_constant__ SrArgs a) {
  griddep_launch_dependents();
  griddep_wait();  // the slots are written by the kernel before this one
  const int per_tile4 = a.BN * 32;  // items per 128 x BN tile
  const int64_t per_tile = (int64_t)a.BN * 128;
  // Every item count is a multiple of 32 and so is the stride: the 32 lanes
  // of a warp take the 32 items of one column of one tile together (its 128
  // rows: four 128-byte slot lines per split, eight lanes per line).
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < a.nitems;
       it += (int64_t)gridDim.x * blockDim.x) {
    int j = 0;
    while (j + 1 < a.njobs && it >= a.jobs[j + 1].item0) ++j;
    const SplitJob &J = a.jobs[j].j;
    const int64_t local = it - a.jobs[j].item0;
    const int64_t tile_lin = local / per_tile4;
    const int rem = (int)(local - tile_lin * per_tile4);
    const int c = rem >> 5, m = (rem & 31) * 4;
    const int tile = (int)(tile_lin % J.tiles), ntile = (int)(tile_lin / J.tiles);
    const int orow = tile * 128 + m;
    const int t = ntile * a.BN + c;
    const int splits = J.splits;
    const float *s0 = a.ws + (J.ws_base + tile_lin * splits) * per_tile + (int64_t)c * 128 + m;
    // slots past the tokens or rows may be unwritten: not read, not stored
    const bool in = orow < J.rows && t < J.T;
    if (in) {
      float4 acc = __ldcg(reinterpret_cast<const float4 *>(s0));
#pragma unroll 8
      for (int sp = 1; sp < splits; ++sp) {
        const float4 f = __ldcg(reinterpret_cast<const float4 *>(s0 + (int64_t)sp * per_tile));
        acc.x += f.x;
        acc.y += f.y;
        acc.z += f.z;
        acc.w += f.w;
      }
      float v[4] = {acc.x, acc.y, acc.z, acc.w};
      const int n = J.rows - orow < 4 ? J.rows - orow : 4;
      if (J.bias) {
        for (int i = 0; i < n; ++i) v[i] += __ldg(J.bias + orow + i);
      }
      sr_store4<DT>(J.C, (int64_t)t * J.ldc + orow, v, n, a.vec_out != 0);
    }
    // The slots are scratch: once every lane of the warp has read its part,
    // the first lane of each line drops the line from L2 without a write-back
    // (the partials never need to reach DRAM).
    __syncwarp();
    if ((m & 31) == 0)
      for (int sp = 0; sp < splits; ++sp) l2_discard_line(s0 + (int64_t)sp * per_tile);
  }
}

}  // namespace

int launch_split_reduce(const SplitJob *jobs, int njobs, const float *ws, int BN, int out_dt, cudaStream_t s) {
  SrArgs a;
  memset(&a, 0, sizeof(a));
  int64_t items = 0;
  const int es = out_dt == TP_F32 ? 4 : 2;
  int vec = 1;
  for (int j = 0; j < njobs; ++j) {
    a.jobs[j].j = jobs[j];
    a.jobs[j].item0 = items;
    if (jobs[j].splits > 1) items += (int64_t)jobs[j].tiles * jobs[j].ntiles * BN * 32;
    // 4-row stores need the row start (a multiple of 4 elements) 4-element aligned
    if (((uintptr_t)jobs[j].C % (4 * es)) || (jobs[j].ldc % 4)) vec = 0;
  }
  if (items == 0) return TP_OK;
  a.ws = ws;
  a.njobs = njobs;
  a.BN = BN;
  a.out_dt = out_dt;
  a.vec_out = vec;
  a.nitems = items;
  const int grid = (int)std::min<int64_t>((items + 255) / 256, (int64_t)sm_count() * 16);
  cudaError_t e;
  if (out_dt == TP_F32)
    e = launch_pdl(split_reduce_kernel<TP_F32>, dim3(grid), dim3(256), 0, s, a);
  else if (out_dt == TP_BF16)
    e = launch_pdl(split_reduce_kernel<TP_BF16>, dim3(grid), dim3(256), 0, s, a);
  else
    e = launch_pdl(split_reduce_kernel<TP_F16>, dim3(grid), dim3(256), 0, s, a);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "split_reduce_kernel launch");
}

}  // namespace tp
