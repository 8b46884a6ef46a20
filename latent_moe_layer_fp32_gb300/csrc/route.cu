// Router, top-k selection and routing table.
//
// "Muse Spark Open on Gaudi 2", section "What was built": the router is fp32
// over 256 experts and picks the top 8.  Section "The latent MoE: A' with a
// per-expert norm": each (token, route) pair becomes its own row, and the
// expert op costs per touched expert slice -- the table below groups rows by
// expert so every touched slice is streamed once per group of rows.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

// ---------------------------------------------------------------------------
// logits partials: part[s][t][e] = sum_{h in split s} x[t][h] * Wr[e][h]
// grid (E/32, ceil(T/8), nsplit), 256 threads: warp w owns 4 experts of the
// CTA's 32, lanes walk h in float4 steps.  fp32 FMA (not TF32).
// ---------------------------------------------------------------------------
constexpr int kRouterTok = 8;

__global__ void __launch_bounds__(256) router_partial_kernel(const uint16_t* __restrict__ x,
                                                             const float* __restrict__ wr,
                                                             float* __restrict__ part, int T, int H, int E,
                                                             int split_len) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * 32 + warp * 4;
  const int t0 = blockIdx.y * kRouterTok;
  const int h_begin = blockIdx.z * split_len;
  float acc[4][kRouterTok];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < kRouterTok; ++j) acc[i][j] = 0.f;
  const int ntok = min(kRouterTok, T - t0);
  for (int h = h_begin + lane * 4; h < h_begin + split_len; h += 128) {
    float4 w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = (e0 + i < E) ? __ldg(reinterpret_cast<const float4*>(wr + (size_t)(e0 + i) * H + h))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kRouterTok; ++j) {
      if (j < ntok) {
        uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t0 + j) * H + h));
        float x0 = bf16_bits_to_f32(xv.x & 0xffffu), x1 = bf16_bits_to_f32(xv.x >> 16);
        float x2 = bf16_bits_to_f32(xv.y & 0xffffu), x3 = bf16_bits_to_f32(xv.y >> 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float a = acc[i][j];
          a = fmaf(x0, w[i].x, a);
          a = fmaf(x1, w[i].y, a);
          a = fmaf(x2, w[i].z, a);
          a = fmaf(x3, w[i].w, a);
          acc[i][j] = a;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < kRouterTok; ++j) acc[i][j] = warp_sum(acc[i][j]);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < kRouterTok; ++j)
        if (j < ntok && e0 + i < E) part[((size_t)blockIdx.z * T + t0 + j) * E + e0 + i] = acc[i][j];
  }
}

// ---------------------------------------------------------------------------
// top-k + softmax-renormalised weights, one warp per token.
// logit[e] = sum over splits in order (+ bias); candidates e = lane + 32*i.
// Ties go to the lower expert index.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ part, int nsplit,
                                                   const float* __restrict__ bias, int T, int E, int k,
                                                   int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  pdl_wait();
  pdl_trigger();
  // one CTA per token: thread e sums its nsplit partials (independent loads,
  // summed in split order), then warp 0 selects the top k
  __shared__ float s_lg[256];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  if (tid < E) {
    float v[16];
#pragma unroll
    for (int sp = 0; sp < 16; ++sp) v[sp] = sp < nsplit ? part[((size_t)sp * T + t) * E + tid] : 0.f;
    float acc = v[0];
#pragma unroll
    for (int sp = 1; sp < 16; ++sp)
      if (sp < nsplit) acc += v[sp];
    if (bias) acc = acc + bias[tid];
    s_lg[tid] = acc;
  }
  __syncthreads();
  if (tid >= 32) return;
  float lg[8];
  bool taken[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? s_lg[e] : -INFINITY;
    taken[i] = (e >= E);
  }
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < 8; ++i) mx = fmaxf(mx, lg[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sel_p[8];
  int sel_e[8];
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sel_p[j] = 0.f;
    sel_e[j] = 0;
    if (j < k) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        if (!taken[i] && (bi == 0x7fffffff || better(lg[i], e, bv, bi))) {
          bv = lg[i];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || better(ov, oi, bv, bi))) {
          bv = ov;
          bi = oi;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (lane + 32 * i == bi) taken[i] = true;
      sel_e[j] = bi;
      sel_p[j] = expf(bv - mx);
      den += sel_p[j];
    }
  }
  float p = 0.f;
  int e = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j == lane) {
      p = sel_p[j];
      e = sel_e[j];
    }
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = e;
    topk_w[(size_t)t * k + lane] = p / den;
  }
}

// ---------------------------------------------------------------------------
// Routing table, one CTA of 1024 threads.  Deterministic stable counting sort
// of the R = T*k row ids by expert; builds the group list used by the expert
// kernels (groups of at most G rows of one expert).
// ---------------------------------------------------------------------------
constexpr int kTableThreads = 1024;

__global__ void __launch_bounds__(kTableThreads) table_kernel(const int32_t* __restrict__ topk_idx, int R, int E,
                                                              int G, int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ sorted_rows,
                                                              int32_t* __restrict__ row_pos,
                                                              int4* __restrict__ groups,
                                                              int32_t* __restrict__ n_groups, Status* st) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_count[256];
  __shared__ int s_fill[256];
  __shared__ int s_off[257];
  __shared__ int s_goff[256];
  __shared__ int s_wcnt[32][256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < 256; e += kTableThreads) s_count[e] = 0;
  __syncthreads();
  for (int r = tid; r < R; r += kTableThreads) {
    int e = topk_idx[r];
    if (e < 0 || e >= E) {
      set_error(st, LMOE_EDEVICE_CHECK, 100);
      e = 0;
    }
    atomicAdd(&s_count[e], 1);
  }
  __syncthreads();
  // exclusive scans (warp 0, 8 experts per lane, lane order = expert order):
  // row offsets and group offsets
  if (warp == 0) {
    int cnt[8], gcnt[8], rs = 0, gs = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      cnt[i] = e < E ? s_count[e] : 0;
      gcnt[i] = (cnt[i] + G - 1) / G;
      rs += cnt[i];
      gs += gcnt[i];
    }
    int rx = rs, gx = gs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ry = __shfl_up_sync(0xffffffffu, rx, o), gy = __shfl_up_sync(0xffffffffu, gx, o);
      if (lane >= o) {
        rx += ry;
        gx += gy;
      }
    }
    int racc = rx - rs, gacc = gx - gs;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) {
        s_off[e] = racc;
        s_goff[e] = gacc;
      }
      racc += cnt[i];
      gacc += gcnt[i];
    }
    if (lane == 31) {
      s_off[E] = racc;
      *n_groups = gacc;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kTableThreads) {
    const int n = s_count[e], a0 = s_off[e];
    int gi = s_goff[e];
    for (int g0 = 0; g0 < n; g0 += G) groups[gi++] = make_int4(e, a0 + g0, min(G, n - g0), 0);
  }
  for (int e = tid; e < 256; e += kTableThreads) s_fill[e] = 0;
  __syncthreads();
  for (int e = tid; e <= E; e += kTableThreads) offsets[e] = s_off[e];

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < R; base += kTableThreads) {
    for (int i = tid; i < 32 * 256; i += kTableThreads) (&s_wcnt[0][0])[i] = 0;
    __syncthreads();
    const int r = base + tid;
    int e = -1, rank = 0;
    if (r < R) {
      e = topk_idx[r];
      if (e < 0 || e >= E) e = 0;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    if (r < R) {
      rank = __popc(same & lt_mask);
      if (rank == 0) s_wcnt[warp][e] = __popc(same);
    }
    __syncthreads();
    // exclusive prefix over warps, per expert (fixed order)
    if (tid < E) {
      int acc = 0;
      for (int w = 0; w < 32; ++w) {
        const int c = s_wcnt[w][tid];
        s_wcnt[w][tid] = acc;
        acc += c;
      }
      s_count[tid] = acc;  // rows of expert tid in this chunk
    }
    __syncthreads();
    if (r < R) {
      const int pos = s_off[e] + s_fill[e] + s_wcnt[warp][e] + rank;
      sorted_rows[pos] = r;
      row_pos[r] = pos;
    }
    __syncthreads();
    if (tid < E) s_fill[tid] += s_count[tid];
    __syncthreads();
  }
}

}  // namespace lmoe
