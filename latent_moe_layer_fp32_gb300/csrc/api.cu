// C ABI of the latent-MoE layer: argument checks, workspace carving and the
// launch sequences.  See include/lmoe.h for the contract of every call.
#include <atomic>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "kernels.cuh"

using namespace lmoe;

namespace lmoe {

thread_local int g_launches = 0;
constexpr int kMaxNamed = 32;
thread_local const char* g_names[kMaxNamed];
thread_local void* const* g_events = nullptr;
thread_local int g_nevents = 0;
thread_local cudaStream_t g_cur_stream = nullptr;  // the stream of the launch being issued

void calls_begin() { g_launches = 0; }

void pre_launch(cudaStream_t s, const char* name) {
  if (g_launches < kMaxNamed) g_names[g_launches] = name;
  g_cur_stream = s;
  if (g_events && 2 * g_launches + 1 < g_nevents)
    cudaEventRecord(static_cast<cudaEvent_t>(g_events[2 * g_launches]), s);
}

void launched() {
  if (g_events && 2 * g_launches + 1 < g_nevents)
    cudaEventRecord(static_cast<cudaEvent_t>(g_events[2 * g_launches + 1]), g_cur_stream);
  ++g_launches;
}

int check_dims(const lmoe_dims* d) {
  if (!d) return LMOE_EINVAL;
  if (d->T < 1 || d->T > 65536 || d->top_k < 1 || d->top_k > 8 || d->n_experts < d->top_k ||
      d->n_experts > 256 || d->hidden < 128 || d->latent < 128 || d->inter < 128 || d->hidden % 128 ||
      d->latent % 128 || d->inter % 128 || !(d->eps >= 0.f))
    return LMOE_EINVAL;
  // expert kernels stream K in 128-byte planes and 2048-element chunks, the
  // projections in 256- or 512-element chunks
  if (d->hidden % 256 || d->latent % 256 || d->inter % 256) return LMOE_EUNSUPPORTED;
  if ((d->latent > 2048 && d->latent % 2048) || (d->inter > 2048 && d->inter % 2048)) return LMOE_EUNSUPPORTED;
  // the decode expert kernels keep a group's activation rows (whole K) in shared memory
  if (d->latent > 8192 || d->inter > 8192) return LMOE_EUNSUPPORTED;
  return LMOE_OK;
}

int fast_route_ks(int H) {
  const int ks = H % 1024 == 0 ? 1024 : (H % 512 == 0 ? 512 : (H % 256 == 0 ? 256 : 0));
  return (ks > 0 && H / ks <= 16) ? ks : 0;
}

int router_splits(int T, int E, int H, int sms, int max_split) {
  const int base = ((E + 31) / 32) * ((T + 7) / 8);
  int ns = 1;
  while (base * ns < 2 * sms && ns < max_split && H % (128 * ns * 2) == 0) ns *= 2;
  return ns;
}

}  // namespace lmoe

namespace {

constexpr int kDenseMinTokensDefault = 64;
// measured crossover on GB300 at the full layer shape: the streaming experts win up to
// about 350 tokens (256: 2.28 against 2.93 ms per step), the grouped GEMMs from there (384: 2.96 against 3.16)
constexpr int kExpertTcMinTokensDefault = 352;
// decode sizes: gate/up and down in one persistent launch up to this many tokens
constexpr int kFusedMaxTokensDefault = 0;
// the post-expert norm and weighted sum inside the down launch up to this many tokens (0: off).
// Measured on GB300 against the separate combine launch it was no faster: 99.7 against 99.0 us
// per T = 1 step and about 2 us slower at T = 4 and 8; a per-kernel timeline of the T = 1 step
// put z 1.3 us later and the unpooler's end 2.5 us later (the down CTAs hold their SMs through
// the z step, and its loads queue behind the unpooler's early weight stream).
constexpr int kDownZMaxTokensDefault = 0;
std::atomic<int> g_dense_min_t{kDenseMinTokensDefault};
std::atomic<int> g_expert_tc_min_t{kExpertTcMinTokensDefault};
std::atomic<int> g_fused_max_t{kFusedMaxTokensDefault};
std::atomic<int> g_downz_max_t{kDownZMaxTokensDefault};
// the options as read once at the start of the current call on this thread, so
// that every decision inside one call sees the same regime
thread_local int t_dense_min_t = kDenseMinTokensDefault;
thread_local int t_expert_tc_min_t = kExpertTcMinTokensDefault;
thread_local int t_fused_max_t = kFusedMaxTokensDefault;
thread_local int t_downz_max_t = kDownZMaxTokensDefault;
void snapshot_options() {
  t_dense_min_t = g_dense_min_t.load(std::memory_order_relaxed);
  t_expert_tc_min_t = g_expert_tc_min_t.load(std::memory_order_relaxed);
  t_fused_max_t = g_fused_max_t.load(std::memory_order_relaxed);
  t_downz_max_t = g_downz_max_t.load(std::memory_order_relaxed);
}

// the router as a tensor-core GEMM: above the fused small-T routing, from the
// dense-projection threshold on, for expert counts that fill whole 32-column chunks
bool router_tc(const lmoe_dims* d) {
  return d->T > 16 && d->T >= t_dense_min_t && d->n_experts % 32 == 0;
}

bool experts_tc(int T) { return T >= t_expert_tc_min_t; }
// the persistent decode experts: MXFP4, at most 8 tokens and 64 route rows
bool experts_fused(const lmoe_dims* d, bool nvfp4) {
  return !nvfp4 && !experts_tc(d->T) && d->T <= t_fused_max_t && d->T <= 8 && d->T * d->top_k <= 64;
}
// the streaming down kernel also forms z: at most 64 route rows
bool down_forms_z(const lmoe_dims* d) { return d->T <= t_downz_max_t && d->T * d->top_k <= 64; }
// rows per group of the routing table: what the expert kernels of this regime consume
int group_rows(int T) { return experts_tc(T) ? kTcExpertGroup : expert_max_group(T); }


struct DevInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

int dev_info(DevInfo* out) {
  static DevInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMOE_ECUDA;
  DevInfo& c = cache[dev & 63];
  if (c.sms == 0) {
    if (cudaDeviceGetAttribute(&c.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return LMOE_ECUDA;
  }
  *out = c;
  if (c.major != 10 || c.minor != 3) return LMOE_EUNSUPPORTED;
  return LMOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A second stream per host thread and device, forked from and joined back to
// the caller's stream with events, so that independent steps of one call run
// side by side (the many-token routing next to the pooler).  Created on first
// use and kept for the life of the thread.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

int side_stream(SideStream** out) {
  thread_local SideStream side[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMOE_ECUDA;
  SideStream& ss = side[dev & 63];
  if (ss.s == nullptr) {
    if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
      return LMOE_ECUDA;
  }
  *out = &ss;
  return LMOE_OK;
}

// The small kernels (routing, combine, helpers) prefer the largest shared-memory
// carveout: an SM configured for them can then also host a CTA of the weight-
// streaming kernel launched behind them (up to ~200 KB of shared memory), which
// starts while they run instead of after.  Once per device.
int set_carveouts() {
  static unsigned long long done = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMOE_ECUDA;
  if (done >> (dev & 63) & 1ull) return LMOE_OK;
  const void* fns[] = {
      reinterpret_cast<const void*>(route_small_kernel), reinterpret_cast<const void*>(router_partial_kernel),
      reinterpret_cast<const void*>(route_fast_kernel),
      reinterpret_cast<const void*>(topk_kernel),        reinterpret_cast<const void*>(table_kernel),
      reinterpret_cast<const void*>(topk_hist_kernel),   reinterpret_cast<const void*>(table_scan_kernel),
      reinterpret_cast<const void*>(table_scatter_kernel), reinterpret_cast<const void*>(table_hist_kernel),
      reinterpret_cast<const void*>(combine_kernel),     reinterpret_cast<const void*>(ssq_kernel),
      reinterpret_cast<const void*>(groups_from_offsets_kernel),
      reinterpret_cast<const void*>(gather_rows_kernel), reinterpret_cast<const void*>(router_split_kernel),
      reinterpret_cast<const void*>(prenorm_kernel),     reinterpret_cast<const void*>(postnorm_residual_kernel)};
  for (const void* f : fns)
    if (cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
        cudaSuccess)
      return LMOE_ECUDA;
  done |= 1ull << (dev & 63);
  return LMOE_OK;
}

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

int router_splits(const lmoe_dims* d, int sms) { return lmoe::router_splits(d->T, d->n_experts, d->hidden, sms, 16); }

struct WsLayout {
  lmoe_ws_layout pub;
  size_t n_groups, route_count, ctr, zero_bytes, groups, part, h, ssq, xs, wr3, rank, chunk;
  // the sandwich block: pre-norm output (bf16), its per-token rinv, the router
  // input split in two bf16 parts (tensor-core router), the layer's output
  size_t nb = 0, rinv = 0, usplit = 0, lout = 0;
  int nsplit;
};

// block: also the sandwich block's buffers (lmoe_block_forward)
int layout(const lmoe_dims* d, int sms, WsLayout* w, bool block = false) {
  int rc = check_dims(d);
  if (rc) return rc;
  const size_t T = d->T, E = d->n_experts, k = d->top_k, R = T * k, L = d->latent, I = d->inter;
  w->nsplit = router_splits(d, sms);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = al(o + bytes);
    return at;
  };
  // zeroed at the start of every call: status word, counters
  w->pub.status = 0;
  w->n_groups = 16;
  w->route_count = 64;  // small-T routing tickets: [0] last block overall, [1 + b] last split of block b (b < 16)
  w->ctr = 256;         // persistent decode experts: per-group completion counters (64) + down-done count
  w->zero_bytes = 768;
  take(w->zero_bytes);
  w->pub.topk_idx = take(4 * R);
  w->pub.topk_w = take(4 * R);
  w->pub.expert_offsets = take(4 * (E + 1));
  w->pub.sorted_rows = take(4 * R);
  w->pub.row_pos = take(4 * R);
  w->groups = take(16 * (R + E + 1));
  w->rank = take(4 * R);                                        // many-token table: row rank in its chunk and expert
  w->chunk = take(4 * ((T + kChunkTok - 1) / kChunkTok) * E);  // per chunk and expert: count, then base position
  w->part = take(4 * (size_t)16 * T * E);
  w->pub.x_lat = take(2 * T * L);
  w->h = take(2 * R * I);
  w->pub.y = take(4 * R * L);
  w->ssq = take(4 * R * (L / 32));
  w->pub.z = take(2 * T * L);
  w->xs = take(2 * R * L);  // x_lat rows in sorted order (grouped tensor-core experts)
  // router weights as three bf16 parts (tensor-core router); the block's router
  // takes each part twice
  w->wr3 = take(2 * E * 3 * (size_t)d->hidden * (block ? 2 : 1));
  if (block) {
    const size_t H = d->hidden;
    w->nb = take(2 * T * H);
    w->rinv = take(4 * T);
    w->usplit = take(2 * T * 2 * H);
    w->lout = take(2 * T * H);
  }
  w->pub.total = o;
  return LMOE_OK;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

cudaLaunchConfig_t pdl_cfg(dim3 grid, dim3 block, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

#define LAUNCH(grid, block, stream, kern, ...)                                   \
  do {                                                                           \
    cudaLaunchAttribute attr_[1];                                                \
    cudaLaunchConfig_t cfg_ = pdl_cfg(grid, block, stream, attr_);               \
    pre_launch(stream, #kern);                                                   \
    if (cudaLaunchKernelEx(&cfg_, kern, __VA_ARGS__) != cudaSuccess) return LMOE_ECUDA; \
    launched();                                                                \
  } while (0)

#define CHECK(x)                 \
  do {                           \
    int rc_ = (x);               \
    if (rc_ != LMOE_OK) return rc_; \
  } while (0)

int prologue(const lmoe_dims* d, void* ws, size_t ws_bytes, DevInfo* di, WsLayout* w, cudaStream_t s,
             bool need_ws = true, bool block = false) {
  calls_begin();
  snapshot_options();
  CHECK(check_dims(d));
  CHECK(dev_info(di));
  CHECK(set_carveouts());
  CHECK(layout(d, di->sms, w, block));
  if (need_ws) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return LMOE_EINVAL;
    if (ws_bytes < w->pub.total) return LMOE_EWORKSPACE;
    // the status word and counters: a kernel, not a memset, so the routing launch can start early
    LAUNCH(dim3(1), dim3(64), s, ws_zero_kernel, static_cast<uint4*>(ws), (int)(w->zero_bytes / 16));
  }
  return LMOE_OK;
}

// pre_g, rinv, usplit (the sandwich block, else null): the router's input is
// x * pre_g with its dot products scaled by rinv per token; usplit holds
// x * pre_g as two bf16 parts for the tensor-core router
int run_route(const lmoe_dims* d, const WsLayout& w, const DevInfo& di, const uint16_t* x, const float* router_w,
              const float* router_bias, int32_t* topk_idx, float* topk_w, int32_t* offsets, int32_t* sorted_rows,
              int32_t* row_pos, void* ws, cudaStream_t s, const uint16_t* pre_g = nullptr,
              const float* rinv = nullptr, const uint16_t* usplit = nullptr) {
  const int T = d->T, E = d->n_experts, k = d->top_k, H = d->hidden;
  Status* st = at<Status>(ws, w.pub.status);
  float* part = at<float>(ws, w.part);
  if (T <= 16) {
    // one launch: router partials with every weight load in flight at once, then the last CTA
    // finishes the routing
    const int KS = fast_route_ks(H);
    if (KS > 0) {
      LAUNCH(dim3((E + 7) / 8, H / KS), dim3(256), s, route_fast_kernel, x, router_w, router_bias, part, T, H, E, k, KS,
             group_rows(T), topk_idx, topk_w, offsets, sorted_rows, row_pos, at<int4>(ws, w.groups),
             at<int32_t>(ws, w.n_groups), at<int32_t>(ws, w.route_count), st, pre_g, rinv);
      return LMOE_OK;
    }
    LAUNCH(dim3((E + 31) / 32, (T + 7) / 8, w.nsplit), dim3(256), s, route_small_kernel, x, router_w, router_bias,
           part, T, H, E, k, H / w.nsplit, group_rows(T), topk_idx, topk_w, offsets, sorted_rows, row_pos,
           at<int4>(ws, w.groups), at<int32_t>(ws, w.n_groups), at<int32_t>(ws, w.route_count), st, pre_g, rinv);
    return LMOE_OK;
  }
  int nsplit = w.nsplit;
  if (router_tc(d)) {
    // logits on the tensor cores: x (bf16) against the three bf16 parts of Wr, split-K
    // partials; the block's input x * g is itself two bf16 parts, against each part of Wr
    uint16_t* w3 = at<uint16_t>(ws, w.wr3);
    const int dup = usplit ? 2 : 1;
    LAUNCH(dim3((H + 1023) / 1024, E), dim3(256), s, router_split_kernel, router_w, E, H, w3, dup);
    // split-K: enough CTAs for the GPU, and at least 4 splits whatever T, so no fp32
    // accumulation chain runs longer than a quarter of K (the logits' rounding error
    // grows with the chain; the top-k weights follow it)
    const int kblocks = 3 * dup * H / 64, tiles_m = (T + 127) / 128;
    nsplit = 1;
    for (int c = 16; c >= 2; --c)
      if (kblocks % c == 0 && (tiles_m * c <= di.sms || c <= 4)) {
        nsplit = c;
        break;
      }
    TcGemmArgs g{};
    g.M = T;
    g.N = E;
    g.K = 3 * dup * H;
    g.st = st;
    g.out_f32 = part;
    g.a_kblocks = dup * H / 64;
    g.n_tile = E;
    g.nsplit = nsplit;
    pre_launch(s, "router_tc_gemm");
    CHECK(launch_tc_gemm_bf16(g, usplit ? usplit : x, w3, s, di.sms));
    launched();
  } else {
    LAUNCH(dim3((E + 31) / 32, (T + 7) / 8, w.nsplit), dim3(256), s, router_partial_kernel, x, router_w, part, T,
           H, E, H / w.nsplit, pre_g);
  }
  const int R = T * k, nchunks = (T + kChunkTok - 1) / kChunkTok;
  int32_t* rank = at<int32_t>(ws, w.rank);
  int32_t* chunk = at<int32_t>(ws, w.chunk);
  LAUNCH(dim3(nchunks), dim3(1024), s, topk_hist_kernel, (const float*)part, nsplit, router_bias, T, E, k, topk_idx,
         topk_w, rank, chunk, rinv);
  LAUNCH(dim3(1), dim3(256), s, table_scan_kernel, chunk, nchunks, E, R, group_rows(T), offsets,
         at<int4>(ws, w.groups), at<int32_t>(ws, w.n_groups));
  LAUNCH(dim3((R + 255) / 256), dim3(256), s, table_scatter_kernel, (const int32_t*)topk_idx, (const int32_t*)rank,
         (const int32_t*)chunk, R, E, k, sorted_rows, row_pos);
  return LMOE_OK;
}

// x_sorted: when set (tensor-core pooler only), x_lat rows are also written in
// expert-sorted order (row_pos = each route row's sorted position)
// wait_mode (decode regime): kWaitAtEnd when nothing earlier in the stream can
// still be writing x (in lmoe_forward it follows the call's own zeroing kernel and routing)
int run_pool(const lmoe_dims* d, const DevInfo& di, const uint16_t* x, const uint16_t* pooler_w, uint16_t* x_lat,
             Status* st, cudaStream_t s, const int32_t* row_pos = nullptr,
             uint16_t* x_sorted = nullptr, int wait_mode = kWaitFirst) {
  const bool dense = x_sorted != nullptr || d->T >= t_dense_min_t;
  pre_launch(s, dense ? "pool_tc_gemm" : "pool_gemv");
  if (dense) {
    TcGemmArgs g{x_lat, d->T, d->latent, d->hidden, st};
    if (x_sorted) {
      g.scatter_pos = row_pos;
      g.scatter_k = d->top_k;
      g.scatter_out = x_sorted;
    }
    CHECK(launch_tc_gemm_bf16(g, x, pooler_w, s, di.sms));
  } else {
    GemvArgs g{pooler_w, x, x_lat, d->latent, d->hidden, d->T, st, wait_mode};
    CHECK(launch_gemv_bf16(g, s, di.sms));
  }
  launched();
  return LMOE_OK;
}

// groups must already be in the workspace
// groups_early: the group list was written by a kernel before the preceding one
// (lmoe_forward: the routing precedes the pooler), so the gate/up kernel may
// stream its first weights before waiting for its predecessor
// nz (the layer's norm and sum, else null): the persistent decode experts then also
// form bf16(z) in the workspace and set *z_ready
struct NormSum {
  const int32_t* topk_idx;
  const float* topk_w;
  const uint16_t* norm_g;
  bool* z_ready;
};

int run_experts(const lmoe_dims* d, const WsLayout& w, const DevInfo& di, const uint16_t* x_lat,
                const int32_t* sorted_rows, const uint8_t* w13_q, const uint8_t* w13_s, const uint8_t* w2_q,
                const uint8_t* w2_s, float* y, void* ws, cudaStream_t s, bool xs_ready = false,
                bool groups_early = false, const float* w13_gs = nullptr, const float* w2_gs = nullptr,
                const NormSum* nz = nullptr) {
  const int T = d->T, k = d->top_k, L = d->latent, I = d->inter;
  Status* st = at<Status>(ws, w.pub.status);
  if (experts_tc(T)) {
    const int R = T * k;
    uint16_t* xs = at<uint16_t>(ws, w.xs);
    if (!xs_ready) LAUNCH(dim3((R + 7) / 8), dim3(256), s, gather_rows_kernel, x_lat, sorted_rows, R, k, L, xs);
    TcExpertArgs t{};
    t.groups = at<int4>(ws, w.groups);
    t.n_groups = at<int32_t>(ws, w.n_groups);
    t.sorted_rows = sorted_rows;
    t.inter = I;
    t.latent = L;
    t.n_experts = d->n_experts;
    t.rows = R;
    t.st = st;
    t.q = w13_q;
    t.s = w13_s;
    t.gs = w13_gs;
    t.K = L;
    t.h_out = at<uint16_t>(ws, w.h);
    pre_launch(s, "expert_gateup_tc");
    CHECK(launch_tc_gateup(t, xs, s, di.sms));
    launched();
    t.q = w2_q;
    t.s = w2_s;
    t.gs = w2_gs;
    t.K = I;
    t.h_out = nullptr;
    t.y_out = y;
    t.ssq_out = at<float>(ws, w.ssq);
    pre_launch(s, "expert_down_tc");
    CHECK(launch_tc_down(t, at<uint16_t>(ws, w.h), s, di.sms));
    launched();
    return LMOE_OK;
  }
  if (experts_fused(d, w13_gs != nullptr)) {
    FusedExpertArgs f{};
    f.w13_q = w13_q;
    f.w13_s = w13_s;
    f.w2_q = w2_q;
    f.w2_s = w2_s;
    f.x_lat = x_lat;
    f.groups = at<int4>(ws, w.groups);
    f.n_groups = at<int32_t>(ws, w.n_groups);
    f.sorted_rows = sorted_rows;
    f.h = f.h_out = at<uint16_t>(ws, w.h);
    f.y_out = y;
    f.ssq_out = at<float>(ws, w.ssq);
    f.ctr = at<int32_t>(ws, w.ctr);
    f.st = st;
    f.T = T;
    f.latent = L;
    f.inter = I;
    f.top_k = k;
    f.n_experts = d->n_experts;
    f.rows = T * k;
    f.early = groups_early ? 1 : 0;
    if (nz) {
      f.topk_idx = nz->topk_idx;
      f.topk_w = nz->topk_w;
      f.norm_g = nz->norm_g;
      f.zb = at<uint16_t>(ws, w.pub.z);
      f.eps = d->eps;
      *nz->z_ready = true;
    }
    pre_launch(s, "expert_fused");
    CHECK(launch_fused_experts(f, s, di.sms));
    launched();
    return LMOE_OK;
  }
  const int G = expert_max_group(T);
  ExpertArgs a{};
  a.groups = at<int4>(ws, w.groups);
  a.n_groups = at<int32_t>(ws, w.n_groups);
  a.sorted_rows = sorted_rows;
  a.inter = I;
  a.latent = L;
  a.top_k = k;
  a.n_experts = d->n_experts;
  a.st = st;
  a.q = w13_q;
  a.s = w13_s;
  a.gs = w13_gs;
  a.act = x_lat;
  a.K = L;
  a.h_out = at<uint16_t>(ws, w.h);
  a.early = groups_early ? 1 : 0;
  a.groups_cap = T * k + d->n_experts + 1;
  a.rows = T * k;
  pre_launch(s, "expert_gateup");
  CHECK(launch_gateup(a, T, G, s, di.sms));
  launched();
  a.q = w2_q;
  a.s = w2_s;
  a.gs = w2_gs;
  a.act = at<uint16_t>(ws, w.h);
  a.K = I;
  a.h_out = nullptr;
  a.y_out = y;
  a.ssq_out = at<float>(ws, w.ssq);
  a.early = 1;  // the gate/up kernel waited for whatever wrote the group list
  if (nz && down_forms_z(d)) {
    a.zb = at<uint16_t>(ws, w.pub.z);
    a.topk_idx = nz->topk_idx;
    a.topk_w = nz->topk_w;
    a.norm_g = nz->norm_g;
    a.zctr = at<int32_t>(ws, w.ctr) + 64;
    a.eps = d->eps;
    a.T = T;
    *nz->z_ready = true;
  }
  pre_launch(s, "expert_down");
  CHECK(launch_down(a, T, G, s, di.sms));
  launched();
  return LMOE_OK;
}

// z_ready: bf16(z) is already in the workspace (the persistent decode experts formed it)
int run_combine_unpool(const lmoe_dims* d, const WsLayout& w, const DevInfo& di, const float* y,
                       const int32_t* topk_idx, const float* topk_w, const uint16_t* norm_g,
                       const uint16_t* unpooler_w, uint16_t* out, void* ws, cudaStream_t s, bool ssq_ready,
                       bool z_ready = false) {
  Status* st = at<Status>(ws, w.pub.status);
  uint16_t* zb = at<uint16_t>(ws, w.pub.z);
  if (z_ready) {
    if (d->T < t_dense_min_t) {
      pre_launch(s, "unpool_gemv");
      GemvArgs g{unpooler_w, zb, out, d->hidden, d->latent, d->T, st, kWaitAfterWeights};
      CHECK(launch_gemv_bf16(g, s, di.sms));
    } else {
      pre_launch(s, "unpool_tc_gemm");
      TcGemmArgs g{out, d->T, d->hidden, d->latent, st};
      CHECK(launch_tc_gemm_bf16(g, zb, unpooler_w, s, di.sms));
    }
    launched();
    return LMOE_OK;
  }
  if (!ssq_ready) {
    const long long n = (long long)d->T * d->top_k * (d->latent / 32);
    LAUNCH(dim3((unsigned)((n + 7) / 8)), dim3(256), s, ssq_kernel, y, d->T * d->top_k, d->latent,
           at<float>(ws, w.ssq));
  }
  int csplit = 1;  // column splits per token: enough CTAs for the GPU at small T
  while (csplit < d->latent / 256 && d->T * csplit < 2 * di.sms) csplit *= 2;
  LAUNCH(dim3(d->T, csplit), dim3(256), s, combine_kernel, y, (const float*)at<float>(ws, w.ssq),
         topk_idx, topk_w, norm_g, d->latent, d->top_k, d->n_experts, d->eps, zb, st);
  if (d->T < t_dense_min_t) {
    // the unpooler weights depend on nothing earlier: they stream while the combine finishes
    pre_launch(s, "unpool_gemv");
    GemvArgs g{unpooler_w, zb, out, d->hidden, d->latent, d->T, st, kWaitAfterWeights};
    CHECK(launch_gemv_bf16(g, s, di.sms));
    launched();
    return LMOE_OK;
  }
  pre_launch(s, "unpool_tc_gemm");
  TcGemmArgs g{out, d->T, d->hidden, d->latent, st};
  CHECK(launch_tc_gemm_bf16(g, zb, unpooler_w, s, di.sms));
  launched();
  return LMOE_OK;
}

int check_weights(const lmoe_weights* wt) {
  if (!wt) return LMOE_EINVAL;
  const void* ptrs[] = {wt->router_w, wt->pooler_w, wt->w13_q, wt->w13_s, wt->w2_q, wt->w2_s, wt->norm_g,
                        wt->unpooler_w};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LMOE_EINVAL;
  if (wt->router_bias && !aligned16(wt->router_bias)) return LMOE_EINVAL;
  return LMOE_OK;
}

// The layer, routed by its own router.  x_route feeds the router (times pre_g
// and rinv when given), x_pool the pooler; in lmoe_forward both are x.
// nv (NVFP4 experts, else null): the global scales; wt->w13_s and w2_s are then E4M3 per 16
int run_layer(const lmoe_dims* d, const lmoe_weights* wt, const WsLayout& w, const DevInfo& di,
              const uint16_t* x_route, const uint16_t* x_pool, const uint16_t* pre_g, const float* rinv,
              const uint16_t* usplit, uint16_t* out, void* ws, cudaStream_t s,
              const lmoe_nvfp4_scales* nv = nullptr) {
  int32_t* idx = at<int32_t>(ws, w.pub.topk_idx);
  float* tw = at<float>(ws, w.pub.topk_w);
  int32_t* srows = at<int32_t>(ws, w.pub.sorted_rows);
  uint16_t* x_lat = at<uint16_t>(ws, w.pub.x_lat);
  float* y = at<float>(ws, w.pub.y);
  Status* st = at<Status>(ws, w.pub.status);
  // The pooler depends only on its input and weights.  Small T: it runs alongside the
  // one-launch routing and waits for it only at its end (programmatic launch).
  // Many tokens: the routing kernels run on a side stream next to it.
  const bool fork = d->T > 16;
  if (fork) {
    SideStream* ss = nullptr;
    CHECK(side_stream(&ss));
    if (cudaEventRecord(ss->fork, s) != cudaSuccess || cudaStreamWaitEvent(ss->s, ss->fork, 0) != cudaSuccess)
      return LMOE_ECUDA;
    CHECK(run_route(d, w, di, x_route, wt->router_w, wt->router_bias, idx, tw, at<int32_t>(ws, w.pub.expert_offsets),
                    srows, at<int32_t>(ws, w.pub.row_pos), ws, ss->s, pre_g, rinv, usplit));
    if (cudaEventRecord(ss->join, ss->s) != cudaSuccess) return LMOE_ECUDA;
    CHECK(run_pool(d, di, x_pool, wt->pooler_w, x_lat, st, s));
    if (cudaStreamWaitEvent(s, ss->join, 0) != cudaSuccess) return LMOE_ECUDA;
  } else {
    // the pooler's input was written before the routing kernel (or is the call's input):
    // it may read it before its wait
    CHECK(run_route(d, w, di, x_route, wt->router_w, wt->router_bias, idx, tw, at<int32_t>(ws, w.pub.expert_offsets),
                    srows, at<int32_t>(ws, w.pub.row_pos), ws, s, pre_g, rinv, usplit));
    CHECK(run_pool(d, di, x_pool, wt->pooler_w, x_lat, st, s, nullptr, nullptr, kWaitAtEnd));
  }
  // (with the fork, the expert kernels follow the join: nothing may stream before their wait)
  bool z_ready = false;
  const NormSum nz{idx, tw, wt->norm_g, &z_ready};
  CHECK(run_experts(d, w, di, x_lat, srows, wt->w13_q, wt->w13_s, wt->w2_q, wt->w2_s, y, ws, s, false, !fork,
                    nv ? nv->w13_gs : nullptr, nv ? nv->w2_gs : nullptr, &nz));
  CHECK(run_combine_unpool(d, w, di, y, idx, tw, wt->norm_g, wt->unpooler_w, out, ws, s, true, z_ready));
  return LMOE_OK;
}

// lmoe_forward_host moves up to this many bytes each way with its own copy kernels (one
// launch latency, no copy-engine round trip: T = 1 e2e 113.7 -> 103.6 us per step); above it,
// with the copy engines (64 MB took 890 us in the upload kernel, loads over the host link)
constexpr size_t kHostIoKernelMaxBytes = 256 * 1024;

// lmoe_forward_host: the layer's workspace, then the token staging buffer and the
// output staging buffer (T x H bf16 each)
struct HostIo {
  size_t xin, xout, total;
};
HostIo host_io_layout(const lmoe_dims* d, const WsLayout& w) {
  HostIo h;
  const size_t rows = (size_t)d->T * d->hidden * 2;
  h.xin = al(w.pub.total);
  h.xout = al(h.xin + rows);
  h.total = al(h.xout + rows);
  return h;
}

// A device-usable address of pinned (page-locked) host memory, or null for any
// other kind of pointer (device, managed, pageable host memory).
const void* pinned_device_ptr(const void* p) {
  if (!p) return nullptr;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // an unregistered pointer can leave an error behind on older runtimes
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  return at.devicePointer;
}

}  // namespace

extern "C" {

size_t lmoe_workspace_bytes(const lmoe_dims* d) {
  DevInfo di;
  int sms = (dev_info(&di) == LMOE_OK) ? di.sms : 148;
  WsLayout w;
  if (layout(d, sms, &w) != LMOE_OK) return 0;
  return w.pub.total;
}

int lmoe_workspace_layout(const lmoe_dims* d, lmoe_ws_layout* out) {
  if (!out) return LMOE_EINVAL;
  DevInfo di;
  int sms = (dev_info(&di) == LMOE_OK) ? di.sms : 148;
  WsLayout w;
  CHECK(layout(d, sms, &w));
  *out = w.pub;
  return LMOE_OK;
}

int lmoe_route(const lmoe_dims* d, const uint16_t* x, const float* router_w, const float* router_bias,
               int32_t* topk_idx, float* topk_w, int32_t* expert_offsets, int32_t* sorted_rows, int32_t* row_pos,
               void* ws, size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s));
  if (!aligned16(x) || !aligned16(router_w) || !topk_idx || !topk_w || !expert_offsets || !sorted_rows ||
      !row_pos || (router_bias && !aligned16(router_bias)))
    return LMOE_EINVAL;
  return run_route(d, w, di, x, router_w, router_bias, topk_idx, topk_w, expert_offsets, sorted_rows,
                                row_pos, ws, s);
}

int lmoe_pool(const lmoe_dims* d, const uint16_t* x, const uint16_t* pooler_w, uint16_t* x_lat, void* ws,
              size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s, ws != nullptr));
  if (!aligned16(x) || !aligned16(pooler_w) || !aligned16(x_lat) || !x || !pooler_w || !x_lat) return LMOE_EINVAL;
  Status* st = ws ? at<Status>(ws, w.pub.status) : nullptr;
  return run_pool(d, di, x, pooler_w, x_lat, st, s);
}

int lmoe_experts_mxfp4(const lmoe_dims* d, const uint16_t* x_lat, const int32_t* expert_offsets,
                       const int32_t* sorted_rows, const uint8_t* w13_q, const uint8_t* w13_s, const uint8_t* w2_q,
                       const uint8_t* w2_s, float* y, void* ws, size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s));
  const void* ptrs[] = {x_lat, expert_offsets, sorted_rows, w13_q, w13_s, w2_q, w2_s, y};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LMOE_EINVAL;
  const int R = d->T * d->top_k;
  LAUNCH(dim3(1), dim3(256), s, groups_from_offsets_kernel, expert_offsets, sorted_rows, d->n_experts, R,
         group_rows(d->T), at<int4>(ws, w.groups), at<int32_t>(ws, w.n_groups), at<Status>(ws, w.pub.status));
  return run_experts(d, w, di, x_lat, sorted_rows, w13_q, w13_s, w2_q, w2_s, y, ws, s);
}

int lmoe_norm_combine_unpool(const lmoe_dims* d, const float* y, const int32_t* topk_idx, const float* topk_w,
                             const uint16_t* norm_g, const uint16_t* unpooler_w, uint16_t* out, void* ws,
                             size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s));
  const void* ptrs[] = {y, topk_idx, topk_w, norm_g, unpooler_w, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LMOE_EINVAL;
  return run_combine_unpool(d, w, di, y, topk_idx, topk_w, norm_g, unpooler_w, out, ws, s, false);
}

int lmoe_forward(const lmoe_dims* d, const lmoe_weights* wt, const uint16_t* x, uint16_t* out, void* ws,
                 size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s));
  if (!x || !out || !aligned16(x) || !aligned16(out)) return LMOE_EINVAL;
  CHECK(check_weights(wt));
  CHECK(run_layer(d, wt, w, di, x, x, nullptr, nullptr, nullptr, out, ws, s));
  return LMOE_OK;
}

size_t lmoe_host_workspace_bytes(const lmoe_dims* d) {
  DevInfo di;
  int sms = (dev_info(&di) == LMOE_OK) ? di.sms : 148;
  WsLayout w;
  if (layout(d, sms, &w) != LMOE_OK) return 0;
  return host_io_layout(d, w).total;
}

int lmoe_forward_host(const lmoe_dims* d, const lmoe_weights* wt, const uint16_t* x_host, uint16_t* out_host,
                      void* ws, size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s, false));
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return LMOE_EINVAL;
  const HostIo h = host_io_layout(d, w);
  if (ws_bytes < h.total) return LMOE_EWORKSPACE;
  const void* xh = pinned_device_ptr(x_host);
  void* oh = const_cast<void*>(pinned_device_ptr(out_host));
  if (!xh || !oh || !aligned16(xh) || !aligned16(oh)) return LMOE_EINVAL;
  CHECK(check_weights(wt));
  const size_t bytes = (size_t)d->T * d->hidden * 2, n16 = bytes / 16;
  uint16_t* xin = at<uint16_t>(ws, h.xin);
  uint16_t* xout = at<uint16_t>(ws, h.xout);
  if (bytes > kHostIoKernelMaxBytes) {
    // many tokens: the copy engines move the rows faster than loads over the host link
    LAUNCH(dim3(1), dim3(64), s, ws_zero_kernel, static_cast<uint4*>(ws), (int)(w.zero_bytes / 16));
    if (cudaMemcpyAsync(xin, xh, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return LMOE_ECUDA;
    CHECK(run_layer(d, wt, w, di, xin, xin, nullptr, nullptr, nullptr, xout, ws, s));
    if (cudaMemcpyAsync(oh, xout, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return LMOE_ECUDA;
    return LMOE_OK;
  }
  // the zeroed region and the tokens in one launch (in place of the zeroing kernel and an upload)
  const size_t blocks = (n16 + 255) / 256, cap = (size_t)di.sms * 4;
  const unsigned gin = (unsigned)(blocks < cap ? blocks : cap);
  LAUNCH(dim3(max(gin, (unsigned)((w.zero_bytes / 16 + 255) / 256))), dim3(256), s, io_in_kernel,
         static_cast<const uint4*>(xh), reinterpret_cast<uint4*>(xin), n16, static_cast<uint4*>(ws),
         (int)(w.zero_bytes / 16));
  CHECK(run_layer(d, wt, w, di, xin, xin, nullptr, nullptr, nullptr, xout, ws, s));
  LAUNCH(dim3(gin), dim3(256), s, io_out_kernel, reinterpret_cast<const uint4*>(xout), static_cast<uint4*>(oh), n16);
  return LMOE_OK;
}

int lmoe_forward_nvfp4(const lmoe_dims* d, const lmoe_weights* wt, const lmoe_nvfp4_scales* nv, const uint16_t* x,
                       uint16_t* out, void* ws, size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s));
  if (!x || !out || !aligned16(x) || !aligned16(out) || !nv || !nv->w13_gs || !nv->w2_gs) return LMOE_EINVAL;
  CHECK(check_weights(wt));
  CHECK(run_layer(d, wt, w, di, x, x, nullptr, nullptr, nullptr, out, ws, s, nv));
  return LMOE_OK;
}

int lmoe_experts_nvfp4(const lmoe_dims* d, const uint16_t* x_lat, const int32_t* expert_offsets,
                       const int32_t* sorted_rows, const uint8_t* w13_q, const uint8_t* w13_s, const float* w13_gs,
                       const uint8_t* w2_q, const uint8_t* w2_s, const float* w2_gs, float* y, void* ws,
                       size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s));
  const void* ptrs[] = {x_lat, expert_offsets, sorted_rows, w13_q, w13_s, w2_q, w2_s, y};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LMOE_EINVAL;
  if (!w13_gs || !w2_gs) return LMOE_EINVAL;
  const int R = d->T * d->top_k;
  LAUNCH(dim3(1), dim3(256), s, groups_from_offsets_kernel, expert_offsets, sorted_rows, d->n_experts, R,
         group_rows(d->T), at<int4>(ws, w.groups), at<int32_t>(ws, w.n_groups), at<Status>(ws, w.pub.status));
  return run_experts(d, w, di, x_lat, sorted_rows, w13_q, w13_s, w2_q, w2_s, y, ws, s, false, false,
                                  w13_gs, w2_gs);
}

size_t lmoe_block_workspace_bytes(const lmoe_dims* d) {
  DevInfo di;
  int sms = (dev_info(&di) == LMOE_OK) ? di.sms : 148;
  WsLayout w;
  if (layout(d, sms, &w, true) != LMOE_OK) return 0;
  return w.pub.total;
}

int lmoe_block_forward(const lmoe_dims* d, const lmoe_weights* wt, const lmoe_block_norms* nm, const uint16_t* x,
                       uint16_t* y, void* ws, size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s, true, true));
  if (!x || !y || !aligned16(x) || !aligned16(y) || !nm || !nm->pre_g || !nm->post_g || !aligned16(nm->pre_g) ||
      !aligned16(nm->post_g) || !(nm->eps >= 0.f))
    return LMOE_EINVAL;
  CHECK(check_weights(wt));
  const int T = d->T, H = d->hidden;
  uint16_t* nb = at<uint16_t>(ws, w.nb);
  float* rinv = at<float>(ws, w.rinv);
  uint16_t* usplit = router_tc(d) ? at<uint16_t>(ws, w.usplit) : nullptr;
  uint16_t* lout = at<uint16_t>(ws, w.lout);
  // pre-norm: the pooler's bf16 input, the router's per-token scale (and split input)
  LAUNCH(dim3(T), dim3(256), s, prenorm_kernel, x, nm->pre_g, nm->eps, H, nb, rinv, usplit);
  CHECK(run_layer(d, wt, w, di, x, nb, nm->pre_g, rinv, usplit, lout, ws, s));
  // post-norm of the layer's output and the residual
  LAUNCH(dim3(T), dim3(256), s, postnorm_residual_kernel, (const uint16_t*)lout, x, nm->post_g, nm->eps, H, y);
  return LMOE_OK;
}

int lmoe_forward_routed(const lmoe_dims* d, const lmoe_weights* wt, const uint16_t* x, const int32_t* topk_idx,
                        const float* topk_w, uint16_t* out, void* ws, size_t ws_bytes, lmoe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevInfo di;
  WsLayout w;
  CHECK(prologue(d, ws, ws_bytes, &di, &w, s));
  if (!wt || !x || !out || !topk_idx || !topk_w || !aligned16(x) || !aligned16(out) || !aligned16(topk_idx) ||
      !aligned16(topk_w))
    return LMOE_EINVAL;
  const void* ptrs[] = {wt->pooler_w, wt->w13_q, wt->w13_s, wt->w2_q, wt->w2_s, wt->norm_g, wt->unpooler_w};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LMOE_EINVAL;
  const int T = d->T, E = d->n_experts, k = d->top_k, R = T * k, nchunks = (T + kChunkTok - 1) / kChunkTok;
  int32_t* srows = at<int32_t>(ws, w.pub.sorted_rows);
  uint16_t* x_lat = at<uint16_t>(ws, w.pub.x_lat);
  float* y = at<float>(ws, w.pub.y);
  Status* st = at<Status>(ws, w.pub.status);
  int32_t* rank = at<int32_t>(ws, w.rank);
  int32_t* chunk = at<int32_t>(ws, w.chunk);
  // the table from the given ids (the router is not run), next to the pooler for many tokens
  const bool fork = T > 16;
  SideStream* ss = nullptr;
  cudaStream_t st_table = s;
  if (fork) {
    CHECK(side_stream(&ss));
    if (cudaEventRecord(ss->fork, s) != cudaSuccess || cudaStreamWaitEvent(ss->s, ss->fork, 0) != cudaSuccess)
      return LMOE_ECUDA;
    st_table = ss->s;
  }
  LAUNCH(dim3(nchunks), dim3(256), st_table, table_hist_kernel, topk_idx, T, E, k, rank, chunk, st);
  LAUNCH(dim3(1), dim3(256), st_table, table_scan_kernel, chunk, nchunks, E, R, group_rows(T),
         at<int32_t>(ws, w.pub.expert_offsets), at<int4>(ws, w.groups), at<int32_t>(ws, w.n_groups));
  LAUNCH(dim3((R + 255) / 256), dim3(256), st_table, table_scatter_kernel, topk_idx, (const int32_t*)rank,
         (const int32_t*)chunk, R, E, k, srows, at<int32_t>(ws, w.pub.row_pos));
  if (fork) {
    if (cudaEventRecord(ss->join, ss->s) != cudaSuccess) return LMOE_ECUDA;
    CHECK(run_pool(d, di, x, wt->pooler_w, x_lat, st, s));
    if (cudaStreamWaitEvent(s, ss->join, 0) != cudaSuccess) return LMOE_ECUDA;
  } else {
    CHECK(run_pool(d, di, x, wt->pooler_w, x_lat, st, s, nullptr, nullptr, kWaitAtEnd));
  }
  bool z_ready = false;
  const NormSum nz{topk_idx, topk_w, wt->norm_g, &z_ready};
  CHECK(run_experts(d, w, di, x_lat, srows, wt->w13_q, wt->w13_s, wt->w2_q, wt->w2_s, y, ws, s, false, !fork,
                    nullptr, nullptr, &nz));
  CHECK(run_combine_unpool(d, w, di, y, topk_idx, topk_w, wt->norm_g, wt->unpooler_w, out, ws, s, true, z_ready));
  return LMOE_OK;
}

int lmoe_status_check(const void* ws, lmoe_stream_t stream) {
  if (!ws) return LMOE_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return LMOE_ECUDA;
  Status h{};
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return LMOE_ECUDA;
  return h.code;
}

const char* lmoe_error_string(int code) {
  switch (code) {
    case LMOE_OK: return "ok";
    case LMOE_EINVAL: return "invalid argument (null or misaligned pointer, or dims out of range)";
    case LMOE_EUNSUPPORTED: return "unsupported dims or device (needs compute capability 10.3)";
    case LMOE_ECUDA: return "CUDA runtime error";
    case LMOE_ETIMEOUT: return "a bounded device-side wait ran out";
    case LMOE_EDEVICE_CHECK: return "device-side input check failed (routing table out of range)";
    case LMOE_EWORKSPACE: return "workspace too small";
    case LMOE_ENOSCRATCH: return "larger than the fixed scratch of lmoe_route_noalloc (T <= 64)";
    default: return "unknown error";
  }
}

int lmoe_last_launch_count(void) { return g_launches; }

const char* lmoe_last_launch_name(int i) {
  return (i >= 0 && i < g_launches && i < kMaxNamed) ? g_names[i] : nullptr;
}

int lmoe_set_option(int key, int value) {
  switch (key) {
    case LMOE_OPT_DENSE_MIN_TOKENS:
      return g_dense_min_t.exchange(value > 0 ? value : kDenseMinTokensDefault);
    case LMOE_OPT_EXPERT_TC_MIN_TOKENS:
      return g_expert_tc_min_t.exchange(value > 0 ? value : kExpertTcMinTokensDefault);
    case LMOE_OPT_FUSED_MAX_TOKENS:
      return g_fused_max_t.exchange(value >= 0 ? value : kFusedMaxTokensDefault);
    case LMOE_OPT_DOWN_Z_MAX_TOKENS:
      return g_downz_max_t.exchange(value >= 0 ? value : kDownZMaxTokensDefault);
    default:
      return LMOE_EINVAL;
  }
}

int lmoe_profile_events(void* const* events, int n) {
  if (n < 0 || (n > 0 && !events)) return LMOE_EINVAL;
  g_events = n > 0 ? events : nullptr;
  g_nevents = n;
  return LMOE_OK;
}

int lmoe_selftest_dequant_bf16(const uint8_t* codes, const uint8_t* scales, int nblocks, uint16_t* out) {
  if (!codes || !scales || !out || nblocks < 1 || !aligned16(codes) || !aligned16(out)) return LMOE_EINVAL;
  DevInfo di;
  CHECK(dev_info(&di));
  dequant_selftest_kernel<<<(nblocks + 127) / 128, 128>>>(codes, scales, nblocks, out);
  if (cudaGetLastError() != cudaSuccess) return LMOE_ECUDA;
  return cudaDeviceSynchronize() == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

int lmoe_selftest_timeout(void* ws, size_t ws_bytes, unsigned limit_us, lmoe_stream_t stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < sizeof(Status) || limit_us == 0 ||
      limit_us > 1000000u)
    return LMOE_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  calls_begin();
  if (cudaMemsetAsync(ws, 0, sizeof(Status), s) != cudaSuccess) return LMOE_ECUDA;
  pre_launch(s, "timeout_selftest_kernel");
  timeout_selftest_kernel<<<1, 32, 0, s>>>(static_cast<Status*>(ws), (unsigned long long)limit_us * 1000ull);
  launched();
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

int lmoe_selftest_e2m1(float* out) {
  if (!out || !aligned16(out)) return LMOE_EINVAL;
  DevInfo di;
  CHECK(dev_info(&di));
  e2m1_selftest_kernel<<<1, 256>>>(out);
  if (cudaGetLastError() != cudaSuccess) return LMOE_ECUDA;
  return cudaDeviceSynchronize() == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

}  // extern "C"
