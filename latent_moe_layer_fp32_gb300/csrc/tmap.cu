// Host-side tensor-map encoding with a small cache (weights rarely move, so
// re-encoding every call would only cost host time).
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "lmoe.h"
#include "tmap.cuh"

namespace lmoe {
namespace {

struct Entry {
  bool used = false;
  CUtensorMapDataType dtype;
  int rank;
  const void* base;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  CUtensorMapSwizzle swz;
  int device;
  CUtensorMap map;
};

constexpr int kCache = 64;
Entry g_cache[kCache];
int g_next = 0;
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool same(const Entry& e, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
          const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swz, int dev) {
  if (!e.used || e.dtype != dtype || e.rank != rank || e.base != base || e.swz != swz || e.device != dev) return false;
  for (int i = 0; i < rank; ++i)
    if (e.dims[i] != dims[i] || e.box[i] != box[i]) return false;
  for (int i = 0; i < rank - 1; ++i)
    if (e.strides[i] != strides[i]) return false;
  return true;
}

}  // namespace

int get_tmap(CUtensorMap* out, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
             const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swz) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMOE_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < kCache; ++i)
    if (same(g_cache[i], dtype, rank, base, dims, strides, box, swz, dev)) {
      *out = g_cache[i].map;
      return LMOE_OK;
    }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return LMOE_ECUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cuuint64_t d[3], s[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides[i];
  CUtensorMap m;
  if (g_encode(&m, dtype, rank, const_cast<void*>(base), d, s, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return LMOE_ECUDA;
  Entry& e = g_cache[g_next];
  g_next = (g_next + 1) % kCache;
  e.used = true;
  e.dtype = dtype;
  e.rank = rank;
  e.base = base;
  e.swz = swz;
  e.device = dev;
  for (int i = 0; i < rank; ++i) {
    e.dims[i] = dims[i];
    e.box[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) e.strides[i] = strides[i];
  e.map = m;
  *out = m;
  return LMOE_OK;
}

}  // namespace lmoe
