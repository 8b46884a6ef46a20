// Routing for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory at the point where they
// run the layer: a plugin called from another runtime's enqueue path, where
// the host framework owns every device allocation and forbids new ones, or
// an embedded runtime with a fixed memory budget fixed at start-up.  They
// cannot size and pass the workspace that lmoe_route needs.
// lmoe_route_noalloc gives them the same routing with its scratch (router
// split partials, group list, status word) in a fixed array inside the
// library instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocScratchBytes, about 1.1 MB) until the process
// exits.  Every call shares it: two calls that overlap on the GPU (different
// streams, or different host threads) race on it and must be serialised by
// the caller.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr int kNoAllocMaxT = 64;
constexpr int kNoAllocMaxE = 256;
constexpr int kNoAllocMaxSplit = 16;
constexpr size_t kStatusBytes = 256;
constexpr size_t kPartBytes = sizeof(float) * kNoAllocMaxSplit * kNoAllocMaxT * kNoAllocMaxE;
constexpr size_t kGroupsBytes = ((sizeof(int4) * (kNoAllocMaxT * 8 + kNoAllocMaxE + 1)) + 255) / 256 * 256;
constexpr size_t kNoAllocScratchBytes = kStatusBytes + kPartBytes + kGroupsBytes;

// The scratch.  In host code this name is only a host-side stand-in for the
// device variable; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {};
int g_sms[64] = {};

// Once per device, with that device current: look up the array's device
// address and the SM count.
int scratch_for_current_device(void** addr, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LMOE_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return LMOE_ECUDA;
    if (major != 10 || minor != 3) return LMOE_EUNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return LMOE_ECUDA;
    g_sms[dev] = n;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  *sms = g_sms[dev];
  return LMOE_OK;
}

bool al16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One launch of `kern` on `s` through cudaLaunchKernelEx (its own return code, not a
// sticky error of an earlier call), counted and named like every other launch.
template <typename... KArgs, typename... Args>
int launch(dim3 grid, dim3 block, cudaStream_t s, const char* name, void (*kern)(KArgs...), Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  lmoe::pre_launch(s, name);
  if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) return LMOE_ECUDA;
  lmoe::launched();
  return LMOE_OK;
}

}  // namespace

extern "C" LMOE_API int lmoe_route_noalloc(const lmoe_dims* d, const uint16_t* x, const float* router_w,
                                           const float* router_bias, int32_t* topk_idx, float* topk_w,
                                           int32_t* expert_offsets, int32_t* sorted_rows, int32_t* row_pos,
                                           lmoe_stream_t stream) {
  using namespace lmoe;
  calls_begin();
  // the same dimension rules as lmoe_route, then the limits of the fixed scratch
  int rc = check_dims(d);
  if (rc != LMOE_OK) return rc;
  if (d->T > kNoAllocMaxT || d->n_experts > kNoAllocMaxE) return LMOE_ENOSCRATCH;
  if (!al16(x) || !al16(router_w) || !topk_idx || !topk_w || !expert_offsets || !sorted_rows || !row_pos ||
      (router_bias && !al16(router_bias)))
    return LMOE_EINVAL;
  void* base = nullptr;
  int sms = 0;
  rc = scratch_for_current_device(&base, &sms);
  if (rc != LMOE_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = d->T, E = d->n_experts, k = d->top_k, H = d->hidden;
  char* scratch = static_cast<char*>(base);
  Status* st = reinterpret_cast<Status*>(scratch);
  int32_t* n_groups = reinterpret_cast<int32_t*>(scratch + 16);
  float* part = reinterpret_cast<float*>(scratch + kStatusBytes);
  int4* groups = reinterpret_cast<int4*>(scratch + kStatusBytes + kPartBytes);
  // the status word and the routing ticket must start at zero; everything else is written before it is read
  if (cudaMemsetAsync(st, 0, 128, s) != cudaSuccess) return LMOE_ECUDA;
  // lmoe_route's router for this T: the one-launch routing up to 16 tokens (its ticket counter
  // sits in the zeroed status region), else the split-K partials (at most 16 splits, which the
  // scratch holds) and the separate top-k and table kernels
  const int KS = fast_route_ks(H);
  if (T <= 16 && KS > 0) {
    rc = launch(dim3((E + 7) / 8, H / KS), dim3(256), s, "route_fast_kernel", route_fast_kernel, x, router_w,
                router_bias, part, T, H, E, k, KS, expert_max_group(T), topk_idx, topk_w, expert_offsets, sorted_rows,
                row_pos, groups, n_groups, reinterpret_cast<int32_t*>(scratch + 64), st, (const uint16_t*)nullptr,
                (const float*)nullptr);
    return rc;
  }
  const int ns = router_splits(T, E, H, sms, kNoAllocMaxSplit);
  rc = launch(dim3((E + 31) / 32, (T + 7) / 8, ns), dim3(256), s, "router_partial_kernel", router_partial_kernel, x,
              router_w, part, T, H, E, H / ns, (const uint16_t*)nullptr);
  if (rc == LMOE_OK)
    rc = launch(dim3(T), dim3(256), s, "topk_kernel", topk_kernel, (const float*)part, ns, router_bias, T, E, k,
                topk_idx, topk_w, (const float*)nullptr);
  if (rc == LMOE_OK)
    rc = launch(dim3(1), dim3(1024), s, "table_kernel", table_kernel, (const int32_t*)topk_idx, T * k, E,
                expert_max_group(T), expert_offsets, sorted_rows, row_pos, groups, n_groups, st);
  return rc;
}
