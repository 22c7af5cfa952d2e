// k_split.cu -- ordered sum of split-K partial tiles, shared by the
// quantized tensor-core kernels and the small-batch 16-bit kernel.
//
// A split tile is 128 output rows x BN token columns; each of its `splits`
// partials is a float32 slot stored column-major (slot[c][m], so a warp's 32
// rows of one column are one 128-byte line).  out[t][row] = (slot_0 + slot_1
// + ... in split order, which is rank order for the row-parallel layer) +
// bias, one thread per output element (consecutive threads: consecutive rows).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include <algorithm>

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
};

__global__ void __launch_bounds__(256) split_reduce_kernel(const __grid_constant__ SrArgs a) {
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < a.nitems;
       it += (int64_t)gridDim.x * blockDim.x) {
    int j = 0;
    while (j + 1 < a.njobs && it >= a.jobs[j + 1].item0) ++j;
    const SplitJob &J = a.jobs[j].j;
    const int64_t local = it - a.jobs[j].item0;
    const int64_t per_tile = (int64_t)a.BN * 128;
    const int64_t tile_lin = local / per_tile;
    const int rem = (int)(local - tile_lin * per_tile);
    const int c = rem >> 7, m = rem & 127;
    const int tile = (int)(tile_lin % J.tiles), ntile = (int)(tile_lin / J.tiles);
    const int orow = tile * 128 + m;
    const int t = ntile * a.BN + c;
    if (orow < J.rows && t < J.T) {  // slots past the tokens or rows may be unwritten
      const float *s0 = a.ws + (J.ws_base + tile_lin * J.splits) * per_tile + (int64_t)c * 128 + m;
      float v = __ldcg(s0);
#pragma unroll 8
      for (int sp = 1; sp < J.splits; ++sp) v += __ldcg(s0 + (int64_t)sp * per_tile);
      if (J.bias) v += __ldg(J.bias + orow);
      const int64_t idx = (int64_t)t * J.ldc + orow;
      if (a.out_dt == TP_F32)
        static_cast<float *>(J.C)[idx] = v;
      else if (a.out_dt == TP_BF16)
        static_cast<__nv_bfloat16 *>(J.C)[idx] = __float2bfloat16_rn(v);
      else
        static_cast<__half *>(J.C)[idx] = __float2half_rn(v);
    }
  }
}

}  // namespace

int launch_split_reduce(const SplitJob *jobs, int njobs, const float *ws, int BN, int out_dt, cudaStream_t s) {
  SrArgs a;
  memset(&a, 0, sizeof(a));
  int64_t items = 0;
  for (int j = 0; j < njobs; ++j) {
    a.jobs[j].j = jobs[j];
    a.jobs[j].item0 = items;
    if (jobs[j].splits > 1) items += (int64_t)jobs[j].tiles * jobs[j].ntiles * BN * 128;
  }
  if (items == 0) return TP_OK;
  a.ws = ws;
  a.njobs = njobs;
  a.BN = BN;
  a.out_dt = out_dt;
  a.nitems = items;
  const int grid = (int)std::min<int64_t>((items + 255) / 256, (int64_t)sm_count() * 16);
  split_reduce_kernel<<<grid, 256, 0, s>>>(a);
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "split_reduce_kernel launch");
}

}  // namespace tp
