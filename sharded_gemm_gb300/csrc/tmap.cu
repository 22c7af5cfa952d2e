// tmap.cu -- host helpers shared by the tensor-core launchers: TMA tensor-map
// encoding (resolved from the driver at run time, cached per argument set),
// the SM count, and the per-(device, stream) split-reduction workspace.
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <vector>
#include <unordered_map>

#include "tp_internal.h"

namespace tp {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_map_mu;

struct MapKey {
  uint64_t ptr, inner, outer, stride;
  uint32_t box0, box1, dt, swz;
  bool operator==(const MapKey &o) const {
    return ptr == o.ptr && inner == o.inner && outer == o.outer && stride == o.stride &&
           box0 == o.box0 && box1 == o.box1 && dt == o.dt && swz == o.swz;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey &k) const {
    uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
    h ^= k.inner + 0x7f4a7c15 + (h << 6) + (h >> 2);
    h ^= k.outer + 0x2545F491 + (h << 6) + (h >> 2);
    h ^= k.stride + ((uint64_t)k.box0 << 32 | k.box1) + (h << 6) + (h >> 2);
    return (size_t)(h ^ ((uint64_t)k.dt << 8) ^ k.swz);
  }
};
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

std::mutex g_ws_mu;
struct Workspace {
  float *partials = nullptr;
  size_t pbytes = 0;
  int *counters = nullptr;
  size_t ncnt = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

int g_sms[64] = {0};

}  // namespace

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  dev &= 63;
  if (!g_sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = v > 0 ? v : 1;
  }
  return g_sms[dev];
}

int make_tmap_2d(CUtensorMap *out, const void *ptr, CUtensorMapDataType dt, int elem_bytes,
                 uint64_t inner, uint64_t outer, uint64_t ld_elems, uint32_t box0, uint32_t box1,
                 CUtensorMapSwizzle swz) {
  std::lock_guard<std::mutex> lk(g_map_mu);
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return set_error(TP_ERR_CUDA, "cannot resolve cuTensorMapEncodeTiled");
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  }
  MapKey key{(uint64_t)(uintptr_t)ptr, inner, outer, ld_elems, box0, box1, (uint32_t)dt, (uint32_t)swz};
  auto it = g_maps.find(key);
  if (it != g_maps.end()) {
    *out = it->second;
    return TP_OK;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld_elems * (uint64_t)elem_bytes};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(out, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  if (g_maps.size() > 8192) g_maps.clear();
  g_maps.emplace(key, *out);
  return TP_OK;
}

// 3-D view of a row-major (rows, ld) matrix as (chunk, rows, chunks): dim 0
// the chunk_elems elements of one chunk of a row, dim 1 the rows (stride
// ld_elems), dim 2 the row's chunks (stride chunk_elems); a box of
// (chunk_elems, box_rows, box_chunks) lands in shared memory as box_chunks
// consecutive (box_rows x chunk) tiles -- one tensor copy where 2-D boxes
// would need box_chunks.
int make_tmap_3d_chunks(CUtensorMap *out, const void *ptr, CUtensorMapDataType dt, int elem_bytes,
                        uint64_t row_elems, uint64_t rows, uint64_t ld_elems, uint32_t chunk_elems,
                        uint32_t box_rows, uint32_t box_chunks, CUtensorMapSwizzle swz) {
  std::lock_guard<std::mutex> lk(g_map_mu);
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return set_error(TP_ERR_CUDA, "cannot resolve cuTensorMapEncodeTiled");
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  }
  // cached under a key no 2-D map can have (box1 carries the chunk count in its top bits)
  MapKey key{(uint64_t)(uintptr_t)ptr, row_elems, rows, ld_elems, chunk_elems,
             box_rows | (box_chunks << 16) | 0x80000000u, (uint32_t)dt, (uint32_t)swz};
  auto it = g_maps.find(key);
  if (it != g_maps.end()) {
    *out = it->second;
    return TP_OK;
  }
  cuuint64_t dims[3] = {chunk_elems, rows, row_elems / chunk_elems};
  cuuint64_t strides[2] = {ld_elems * (uint64_t)elem_bytes, (uint64_t)chunk_elems * elem_bytes};
  cuuint32_t box[3] = {chunk_elems, box_rows, box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(out, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(TP_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
  if (g_maps.size() > 8192) g_maps.clear();
  g_maps.emplace(key, *out);
  return TP_OK;
}

void tmap_cache_clear() {
  std::lock_guard<std::mutex> lk(g_map_mu);
  g_maps.clear();
}

// Buffers a workspace outgrew.  A CUDA graph captured from an earlier call
// still holds their addresses, so they stay allocated (and their counters
// stay at zero) until split_workspace_free(): growing a workspace never
// invalidates a capture.
struct Retired {
  int dev;
  void *p;
  size_t counter_bytes;  // > 0: a counter array (cleared by split_workspace_reset)
};
static std::vector<Retired> g_retired;

int split_workspace(cudaStream_t s, size_t partial_bytes, size_t ncounters, float **partials,
                    int **counters) {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_ws_mu);
  Workspace &w = g_ws[{dev, s}];
  if (w.pbytes < partial_bytes) {
    size_t want = partial_bytes + partial_bytes / 4;
    float *np = nullptr;
    cudaError_t e = cudaMalloc(&np, want);
    if (e != cudaSuccess) return cuda_error(e, "workspace allocation");
    if (w.partials) g_retired.push_back(Retired{dev, w.partials, 0});
    w.partials = np;
    w.pbytes = want;
  }
  if (w.ncnt < ncounters) {
    size_t want = ncounters + 1024;
    int *nc = nullptr;
    cudaError_t e = cudaMalloc(&nc, want * sizeof(int));
    if (e != cudaSuccess) return cuda_error(e, "workspace allocation");
    e = cudaMemsetAsync(nc, 0, want * sizeof(int), s);
    if (e != cudaSuccess) {
      cudaFree(nc);
      return cuda_error(e, "workspace clear");
    }
    if (w.counters) g_retired.push_back(Retired{dev, w.counters, w.ncnt * sizeof(int)});
    w.counters = nc;
    w.ncnt = want;
  }
  *partials = w.partials;
  *counters = w.counters;
  return TP_OK;
}

void split_workspace_reset() {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto &kv : g_ws)
    if (kv.second.counters) {
      cudaSetDevice(kv.first.first);
      cudaMemset(kv.second.counters, 0, kv.second.ncnt * sizeof(int));
    }
  for (auto &r : g_retired)
    if (r.counter_bytes) {
      cudaSetDevice(r.dev);
      cudaMemset(r.p, 0, r.counter_bytes);
    }
  cudaSetDevice(cur);
}

void split_workspace_free() {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto &kv : g_ws) {
    cudaSetDevice(kv.first.first);
    if (kv.second.partials) cudaFree(kv.second.partials);
    if (kv.second.counters) cudaFree(kv.second.counters);
  }
  g_ws.clear();
  for (auto &r : g_retired) {
    cudaSetDevice(r.dev);
    cudaFree(r.p);
  }
  g_retired.clear();
  cudaSetDevice(cur);
}

}  // namespace tp
