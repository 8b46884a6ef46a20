// Small kernels around the streaming ones: the group list for caller-supplied
// routing tables, post_expert_norm + weighted sum, the copies between pinned
// host memory and the workspace for lmoe_forward_host, and the E2M1
// conversion self-test.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

// Group list (groups of <= G rows per expert) from a caller-supplied table,
// with the table checked: offsets[0] == 0, monotone, offsets[E] == R, and
// every sorted row id in [0, R).  One CTA of 256 threads.
__global__ void __launch_bounds__(256) groups_from_offsets_kernel(const int32_t* __restrict__ offsets,
                                                                  const int32_t* __restrict__ sorted_rows, int E,
                                                                  int R, int G, int4* __restrict__ groups,
                                                                  int32_t* __restrict__ n_groups, Status* st) {
  pdl_wait();
  pdl_trigger();
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < R; i += 256)
    if (sorted_rows[i] < 0 || sorted_rows[i] >= R) bad = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    // validate the whole table before writing any group
    bool ok = offsets[0] == 0 && offsets[E] == R && !bad;
    for (int e = 0; e < E && ok; ++e)
      if (offsets[e + 1] < offsets[e] || offsets[e + 1] > R) ok = false;
    int ng = 0;
    if (ok) {
      for (int e = 0; e < E; ++e) {
        const int a = offsets[e], n = offsets[e + 1] - a;
        for (int g0 = 0; g0 < n; g0 += G) groups[ng++] = make_int4(e, a + g0, min(G, n - g0), 0);
      }
    } else {
      set_error(st, LMOE_EDEVICE_CHECK, 101);
    }
    *n_groups = ng;
  }
}

// Sum of squares of each route row per 32-column tile: ssq[r][tile] (used when
// y comes from the caller; the down kernel writes the same partials itself).
// One warp per (row, tile), 8 per CTA.
__global__ void __launch_bounds__(256) ssq_kernel(const float* __restrict__ y, int R, int L,
                                                  float* __restrict__ ssq) {
  pdl_wait();
  pdl_trigger();
  const int tiles = L / 32;
  const long long i = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (i >= (long long)R * tiles) return;
  const int r = (int)(i / tiles), tile = (int)(i % tiles), lane = threadIdx.x & 31;
  const float v = y[(size_t)r * L + tile * 32 + lane];
  const float s = warp_sum(v * v);
  if (lane == 0) ssq[i] = s;
}

// post_expert_norm on each route row, then the fp32 weighted sum in route
// order ("Muse Spark Open on Gaudi 2", "The latent MoE: A' with a per-expert
// norm").  Grid (T, ceil(L/256)), 256 threads, 1 column per thread:
//   ss_j  = sum over the row's 32-column tiles of ssq (fixed order)
//   rinv  = 1 / sqrt(ss_j / L + eps)
//   z[l]  = sum_j w[t][j] * ((y * rinv) * g[e_j][l]),  zb = bf16(z)
// Grid (T, S): CTA (t, c) takes columns [c L/S, (c+1) L/S) of token t, four
// consecutive columns per thread and step (16-byte loads of y); S > 1 only
// when T alone would leave SMs idle.  Each CTA recomputes the k factors rinv of
// its token from the k x L/32 partials.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const float* __restrict__ ssq,
                                                      const int32_t* __restrict__ topk_idx,
                                                      const float* __restrict__ topk_w,
                                                      const uint16_t* __restrict__ norm_g, int L, int k, int E,
                                                      float eps, uint16_t* __restrict__ zb, Status* st) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_rinv[8];
  __shared__ int s_e[8];
  __shared__ float s_w[8];
  const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tiles = L / 32;
  if (warp < k) {
    const int r = t * k + warp;
    // every load of the lane first (up to 8 of its tiles), then the sum in tile order
    float s = 0.f;
    for (int i0 = lane; i0 < tiles; i0 += 32 * 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = (i0 + 32 * u < tiles) ? ssq[(size_t)r * tiles + i0 + 32 * u] : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + 32 * u < tiles) s += v[u];
    }
    s = warp_sum(s);
    if (lane == 0) {
      int e = topk_idx[r];
      if (e < 0 || e >= E) {
        set_error(st, LMOE_EDEVICE_CHECK, 102);
        e = 0;
      }
      s_e[warp] = e;
      s_w[warp] = topk_w[r];
      s_rinv[warp] = 1.0f / sqrtf(s / (float)L + eps);
    }
  }
  __syncthreads();
  const int span = L / gridDim.y, c_end = (blockIdx.y + 1) * span;
  for (int l = blockIdx.y * span + 4 * tid; l < c_end; l += 4 * 256) {
    float z[4] = {0.f, 0.f, 0.f, 0.f};
    // every route's y and gain loads first (k <= 8), then the sum in route order
    float4 yv[8];
    uint2 gw[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k) {
        yv[j] = __ldcs(reinterpret_cast<const float4*>(y + ((size_t)t * k + j) * L + l));
        gw[j] = *reinterpret_cast<const uint2*>(norm_g + (size_t)s_e[j] * L + l);
      }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j >= k) break;
      const float yy[4] = {yv[j].x, yv[j].y, yv[j].z, yv[j].w};
      const float gg[4] = {bf16_bits_to_f32(gw[j].x & 0xFFFFu), bf16_bits_to_f32(gw[j].x >> 16),
                           bf16_bits_to_f32(gw[j].y & 0xFFFFu), bf16_bits_to_f32(gw[j].y >> 16)};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float yh = __fmul_rn(__fmul_rn(yy[q], s_rinv[j]), gg[q]);
        z[q] = __fadd_rn(z[q], __fmul_rn(s_w[j], yh));
      }
    }
    uint2 out;
    out.x = (uint32_t)f32_to_bf16_bits(z[0]) | ((uint32_t)f32_to_bf16_bits(z[1]) << 16);
    out.y = (uint32_t)f32_to_bf16_bits(z[2]) | ((uint32_t)f32_to_bf16_bits(z[3]) << 16);
    *reinterpret_cast<uint2*>(zb + (size_t)t * L + l) = out;
  }
}

__global__ void e2m1_selftest_kernel(float* out) {
  const uint32_t b = threadIdx.x;
  uint32_t h0, h1, h2, h3;
  e2m1x8_to_f16x8(b, h0, h1, h2, h3);
  const __half2 v = *reinterpret_cast<const __half2*>(&h0);
  out[2 * b] = __low2float(v);
  out[2 * b + 1] = __high2float(v);
}

// Failure-detection self-test: one thread waits on a shared-memory mbarrier
// that nothing ever completes, with the library's bounded-wait pattern but a
// limit of limit_ns (and an iteration cap, so the kernel ends even if the
// timer stalled), then records LMOE_ETIMEOUT in the status word and returns.
// The context stays usable: nothing faults, nothing is left in flight.
__global__ void __launch_bounds__(32) timeout_selftest_kernel(Status* st, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_test_wait(&bar, 0)) return;  // never: no thread arrives
    if ((it & 255u) == 0 && globaltimer() - t0 > limit_ns) break;
  }
  set_error(st, LMOE_ETIMEOUT, 99);
}

// The workspace's status and counter words, zeroed at the start of a call (a
// programmatic-launch chain can start the next kernel early, which a memset
// would not allow).  One CTA; n16 counts 16-byte units.
__global__ void __launch_bounds__(64) ws_zero_kernel(uint4* __restrict__ p, int n16) {
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < n16; i += blockDim.x) p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Host I/O for lmoe_forward_host.  io_in_kernel zeroes the workspace's zeroed
// region (in place of ws_zero_kernel) and copies the tokens from pinned host
// memory into the device staging buffer; io_out_kernel, after the unpooler,
// copies the output rows back to pinned host memory.  16-byte accesses,
// grid-stride; n16 counts 16-byte units.
__global__ void __launch_bounds__(256) io_in_kernel(const uint4* __restrict__ x_host, uint4* __restrict__ x_dev,
                                                    size_t n16, uint4* __restrict__ zero, int nzero16) {
  pdl_wait();
  pdl_trigger();
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x, step = (size_t)gridDim.x * blockDim.x;
  if (i0 < (size_t)nzero16) zero[i0] = make_uint4(0u, 0u, 0u, 0u);
  for (size_t i = i0; i < n16; i += step) x_dev[i] = __ldcs(x_host + i);
}

__global__ void __launch_bounds__(256) io_out_kernel(const uint4* __restrict__ out_dev, uint4* __restrict__ out_host,
                                                     size_t n16) {
  pdl_wait();
  pdl_trigger();
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x, step = (size_t)gridDim.x * blockDim.x;
  for (size_t i = i0; i < n16; i += step) out_host[i] = __ldcs(out_dev + i);
}

}  // namespace lmoe
