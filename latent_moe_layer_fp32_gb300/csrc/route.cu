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
// With a gain g (the sandwich block's pre-norm), the input is u = x * g, a
// product of two bf16 values and exact in fp32; the reduction then scales the
// dot product by the token's rinv.
// ---------------------------------------------------------------------------
constexpr int kRouterTok = 8;

__device__ __forceinline__ void router_partial_body(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                                                    float* __restrict__ part, int T, int H, int E, int split_len,
                                                    const uint16_t* __restrict__ g) {
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
    float g0 = 1.f, g1 = 1.f, g2 = 1.f, g3 = 1.f;
    if (g) {
      const uint2 gv = __ldg(reinterpret_cast<const uint2*>(g + h));
      g0 = bf16_bits_to_f32(gv.x & 0xffffu);
      g1 = bf16_bits_to_f32(gv.x >> 16);
      g2 = bf16_bits_to_f32(gv.y & 0xffffu);
      g3 = bf16_bits_to_f32(gv.y >> 16);
    }
#pragma unroll
    for (int j = 0; j < kRouterTok; ++j) {
      if (j < ntok) {
        uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t0 + j) * H + h));
        float x0 = bf16_bits_to_f32(xv.x & 0xffffu), x1 = bf16_bits_to_f32(xv.x >> 16);
        float x2 = bf16_bits_to_f32(xv.y & 0xffffu), x3 = bf16_bits_to_f32(xv.y >> 16);
        if (g) {  // exact products
          x0 = __fmul_rn(x0, g0);
          x1 = __fmul_rn(x1, g1);
          x2 = __fmul_rn(x2, g2);
          x3 = __fmul_rn(x3, g3);
        }
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

__global__ void __launch_bounds__(256) router_partial_kernel(const uint16_t* __restrict__ x,
                                                             const float* __restrict__ wr,
                                                             float* __restrict__ part, int T, int H, int E,
                                                             int split_len, const uint16_t* __restrict__ g) {
  router_partial_body(x, wr, part, T, H, E, split_len, g);
}

// ---------------------------------------------------------------------------
// top-k + softmax-renormalised weights, one warp per token.
// logit[e] = sum over splits in order (+ bias); candidates e = lane + 32*i.
// Ties go to the lower expert index.
// ---------------------------------------------------------------------------
// A 64-bit key per logit whose unsigned order is the selection order: the
// float's bits mapped to an order-preserving unsigned value (sign bit set for
// non-negative values, all bits flipped for negative ones) above the bit-
// inverted expert index, so that equal logits rank the lower index first.
// v + 0 turns -0 into +0 (the two compare equal as floats).  Key 0 marks an
// absent slot; every finite or infinite logit has a larger key.  A NaN logit
// ranks above every number: logits are expected to be finite.
__device__ __forceinline__ unsigned long long topk_key(float v, int e) {
  unsigned u = __float_as_uint(__fadd_rn(v, 0.0f));
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | static_cast<unsigned>(~e);
}

__device__ __forceinline__ float topk_key_value(unsigned hi) {
  return __uint_as_float((hi & 0x80000000u) ? (hi & 0x7fffffffu) : ~hi);
}

__device__ __forceinline__ void key_cx(unsigned long long& a, unsigned long long& b) {
  const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Top-k of one token by one warp, logits lg_s[0..E) in shared memory.
// Writes topk_idx[k], topk_w[k] for the token (softmax over all E,
// renormalised over the k picks; ties to the lower expert index).
// Lane l holds experts l, l+32, ..., l+224, sorts its eight keys (a 19-
// comparator network), and each pick is one warp-wide maximum over the lanes'
// leading keys (the high words, then the low words of the lanes that reach
// the maximum), after which the owning lane drops its leading key.
__device__ __forceinline__ void topk_one_token(const float* lg_s, int E, int k, int32_t* topk_idx, float* topk_w,
                                               int lane, int* s_pick = nullptr) {
  unsigned long long q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    q[i] = e < E ? topk_key(lg_s[e], e) : 0ull;
  }
  key_cx(q[0], q[2]); key_cx(q[1], q[3]); key_cx(q[4], q[6]); key_cx(q[5], q[7]);
  key_cx(q[0], q[4]); key_cx(q[1], q[5]); key_cx(q[2], q[6]); key_cx(q[3], q[7]);
  key_cx(q[0], q[1]); key_cx(q[2], q[3]); key_cx(q[4], q[5]); key_cx(q[6], q[7]);
  key_cx(q[2], q[4]); key_cx(q[3], q[5]);
  key_cx(q[1], q[4]); key_cx(q[3], q[6]);
  key_cx(q[1], q[2]); key_cx(q[3], q[4]); key_cx(q[5], q[6]);
  float mx = 0.f, v = 0.f;
  int e = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      const unsigned hi = static_cast<unsigned>(q[0] >> 32), lo = static_cast<unsigned>(q[0]);
      const unsigned mh = __reduce_max_sync(0xffffffffu, hi);
      const unsigned ml = __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u);
      const int ej = static_cast<int>(~ml);
      const float vj = topk_key_value(mh);
      if (j == 0) mx = vj;  // the largest logit
      if (lane == j) {
        v = vj;
        e = ej;
      }
      if (lane == (ej & 31)) {  // the owner drops its leading key
#pragma unroll
        for (int i = 0; i < 7; ++i) q[i] = q[i + 1];
        q[7] = 0ull;
      }
    }
  }
  // softmax over the picks, summed in pick order
  const float p = lane < k ? expf(v - mx) : 0.f;
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float pj = __shfl_sync(0xffffffffu, p, j);
    if (j < k) den += pj;
  }
  if (lane < k) {
    topk_idx[lane] = e;
    topk_w[lane] = p / den;
    if (s_pick) s_pick[lane] = e;
  }
}

// logit[e] of token t = sum over splits in split order (times rinv[t]) (+ bias)
__device__ __forceinline__ float token_logit(const float* part, int nsplit, const float* bias, int T, int E, int t,
                                             int e, const float* rinv) {
  float v[16];
#pragma unroll
  for (int sp = 0; sp < 16; ++sp) v[sp] = sp < nsplit ? __ldcg(part + ((size_t)sp * T + t) * E + e) : 0.f;
  float acc = v[0];
#pragma unroll
  for (int sp = 1; sp < 16; ++sp)
    if (sp < nsplit) acc += v[sp];
  if (rinv) acc = __fmul_rn(acc, rinv[t]);
  if (bias) acc = acc + bias[e];
  return acc;
}

__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ part, int nsplit,
                                                   const float* __restrict__ bias, int T, int E, int k,
                                                   int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                   const float* __restrict__ rinv) {
  pdl_wait();
  pdl_trigger();
  // one CTA per token: thread e sums its partials, warp 0 selects the top k
  __shared__ float s_lg[256];
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid < E) s_lg[tid] = token_logit(part, nsplit, bias, T, E, t, tid, rinv);
  __syncthreads();
  if (tid < 32) topk_one_token(s_lg, E, k, topk_idx + (size_t)t * k, topk_w + (size_t)t * k, tid);
}

// ---------------------------------------------------------------------------
// Routing table, one CTA of 1024 threads.  Deterministic stable counting sort
// of the R = T*k row ids by expert; builds the group list used by the expert
// kernels (groups of at most G rows of one expert).
// ---------------------------------------------------------------------------
constexpr int kTableThreads = 1024;

// Shared state of the table build for a CTA of NT threads.
template <int NT>
struct TableSmem {
  int count[256], fill[256], off[257], goff[256];
  int wcnt[NT / 32][256];
};

// Stable counting sort of the R row ids by expert (ascending row id within an
// expert) plus the group list, by one CTA of NT threads; idx may be global
// memory written by this CTA before a __syncthreads.
template <int NT>
__device__ void build_table(const int32_t* idx, int R, int E, int G, int32_t* __restrict__ offsets,
                            int32_t* __restrict__ sorted_rows, int32_t* __restrict__ row_pos, int4* __restrict__ groups,
                            int32_t* __restrict__ n_groups, Status* st, TableSmem<NT>& sm) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < 256; e += NT) sm.count[e] = 0;
  __syncthreads();
  for (int r = tid; r < R; r += NT) {
    int e = idx[r];
    if (e < 0 || e >= E) {
      set_error(st, LMOE_EDEVICE_CHECK, 100);
      e = 0;
    }
    atomicAdd(&sm.count[e], 1);
  }
  __syncthreads();
  // exclusive scans (warp 0, 8 experts per lane, lane order = expert order):
  // row offsets and group offsets
  if (warp == 0) {
    int cnt[8], gcnt[8], rs = 0, gs = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      cnt[i] = e < E ? sm.count[e] : 0;
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
        sm.off[e] = racc;
        sm.goff[e] = gacc;
      }
      racc += cnt[i];
      gacc += gcnt[i];
    }
    if (lane == 31) {
      sm.off[E] = racc;
      *n_groups = gacc;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += NT) {
    const int n = sm.count[e], a0 = sm.off[e];
    int gi = sm.goff[e];
    for (int g0 = 0; g0 < n; g0 += G) groups[gi++] = make_int4(e, a0 + g0, min(G, n - g0), 0);
  }
  for (int e = tid; e < 256; e += NT) sm.fill[e] = 0;
  __syncthreads();
  for (int e = tid; e <= E; e += NT) offsets[e] = sm.off[e];

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < R; base += NT) {
    for (int i = tid; i < NW * 256; i += NT) (&sm.wcnt[0][0])[i] = 0;
    __syncthreads();
    const int r = base + tid;
    int e = -1, rank = 0;
    if (r < R) {
      e = idx[r];
      if (e < 0 || e >= E) e = 0;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    if (r < R) {
      rank = __popc(same & lt_mask);
      if (rank == 0) sm.wcnt[warp][e] = __popc(same);
    }
    __syncthreads();
    // exclusive prefix over warps, per expert (fixed order)
    if (tid < E) {
      int acc = 0;
      for (int w = 0; w < NW; ++w) {
        const int c = sm.wcnt[w][tid];
        sm.wcnt[w][tid] = acc;
        acc += c;
      }
      sm.count[tid] = acc;  // rows of expert tid in this chunk
    }
    __syncthreads();
    if (r < R) {
      const int pos = sm.off[e] + sm.fill[e] + sm.wcnt[warp][e] + rank;
      sorted_rows[pos] = r;
      row_pos[r] = pos;
    }
    __syncthreads();
    if (tid < E) sm.fill[tid] += sm.count[tid];
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kTableThreads) table_kernel(const int32_t* __restrict__ topk_idx, int R, int E,
                                                              int G, int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ sorted_rows,
                                                              int32_t* __restrict__ row_pos,
                                                              int4* __restrict__ groups,
                                                              int32_t* __restrict__ n_groups, Status* st) {
  pdl_wait();
  pdl_trigger();
  __shared__ TableSmem<kTableThreads> sm;
  build_table<kTableThreads>(topk_idx, R, E, G, offsets, sorted_rows, row_pos, groups, n_groups, st, sm);
}

// ---------------------------------------------------------------------------
// Small-T routing in one launch: the router partials of router_partial_kernel
// (same grid), then "last CTA finishes":
//  - T <= 2: the last CTA overall sums every (token, expert) logit from its
//    split partials (split order, + bias) itself;
//  - T > 2, two levels: per (32-expert block, 8-token block) the last of its
//    split CTAs sums the block's logits and stores them over split 0 of the
//    partials (it alone reads or writes that block), and the last block to
//    finish reads those;
// then it selects the top k of every token (one warp per token, in turns) and
// builds the table from the picks it holds in shared memory.
// tickets[0] counts the last level, tickets[1 + block] the first; all start at
// zero.  Requires T <= 16 (at most 16 blocks).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) route_small_kernel(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                                                          const float* __restrict__ bias, float* __restrict__ part,
                                                          int T, int H, int E, int k, int split_len, int G,
                                                          int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ sorted_rows,
                                                          int32_t* __restrict__ row_pos, int4* __restrict__ groups,
                                                          int32_t* __restrict__ n_groups, int32_t* tickets,
                                                          Status* st, const uint16_t* __restrict__ g,
                                                          const float* __restrict__ rinv) {
  router_partial_body(x, wr, part, T, H, E, split_len, g);
  __shared__ int s_last;
  const bool one_level = T <= 2;
  const int blk = blockIdx.y * gridDim.x + blockIdx.x;
  __syncthreads();
  if (!one_level) {
    if (threadIdx.x == 0) {
      __threadfence();  // this CTA's partials before its ticket
      s_last = (atomicAdd(&tickets[1 + blk], 1) == (int)gridDim.z - 1);
      if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    // thread (u, el): token blockIdx.y*8 + u, expert blockIdx.x*32 + el
    const int t = blockIdx.y * kRouterTok + (threadIdx.x >> 5), e = blockIdx.x * 32 + (threadIdx.x & 31);
    if (t < T && e < E) {
      const float v = token_logit(part, gridDim.z, bias, T, E, t, e, rinv);
      __stcg(part + (size_t)t * E + e, v);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's partials (or its block's logits) before the ticket
    s_last = (atomicAdd(&tickets[0], 1) == (int)(one_level ? gridDim.x * gridDim.y * gridDim.z
                                                           : gridDim.x * gridDim.y) - 1);
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  __shared__ float s_lg[8][256];
  __shared__ int s_pick[16 * 8];
  __shared__ TableSmem<256> sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t0 = 0; t0 < T; t0 += 8) {
    // thread e: expert e's logit of up to 8 tokens, every load before the stores
    if (threadIdx.x < E) {
      float v[8];
      if (one_level) {
#pragma unroll
        for (int u = 0; u < 2; ++u)
          v[u] = (t0 + u < T) ? token_logit(part, gridDim.z, bias, T, E, t0 + u, threadIdx.x, rinv) : 0.f;
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = (t0 + u < T) ? __ldcg(part + (size_t)(t0 + u) * E + threadIdx.x) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (t0 + u < T && (!one_level || u < 2)) s_lg[u][threadIdx.x] = v[u];
    }
    __syncthreads();
    if (t0 + warp < T)
      topk_one_token(s_lg[warp], E, k, topk_idx + (size_t)(t0 + warp) * k, topk_w + (size_t)(t0 + warp) * k, lane,
                     s_pick + (t0 + warp) * k);
    __syncthreads();
  }
  build_table<256>(s_pick, T * k, E, G, offsets, sorted_rows, row_pos, groups, n_groups, st, sm);
}

// ---------------------------------------------------------------------------
// Small-T routing in one launch, all weight loads in flight at once.
// Grid (ceil(E/8), nsplit): warp w of CTA (b, s) owns expert b*8 + w and the
// K range [s*KS, (s+1)*KS) (KS = H/nsplit, a multiple of 128, at most 1024):
// every lane issues its KS/128 16-byte weight loads before any arithmetic, so
// the whole router matrix is requested in the first microseconds.  The CTA
// stages its K range of up to four tokens at a time in shared memory (bf16)
// and each lane keeps one fp32 FMA chain per token in element order; the warp
// then adds its lanes in a fixed tree and stores the partial.  The last CTA to
// finish (a ticket counter) sums every logit's partials in split order (times
// rinv, + bias), selects the top k of every token (one warp per token) and
// builds the table from the picks it holds in shared memory.
// tickets[0] starts at zero.  Requires T <= 16 and nsplit <= 16.
// ---------------------------------------------------------------------------
constexpr int kFastKS = 1024;  // largest K range per warp: 8 loads of 16 bytes per lane
constexpr int kFastTok = 4;    // tokens staged per pass

struct FastRouteSmem {
  union {
    uint16_t xs[kFastTok][kFastKS];  // the CTA's K range of up to four tokens (bf16 bits)
    struct {
      float lg[16][256];             // last CTA: logits
      int pick[16 * 8];
      TableSmem<256> tab;
    } tail;
  };
};

// Logits of expert ee for every token from the split partials: the partials of
// TC tokens (NS >= nsplit splits each) are all loaded before any is summed;
// each logit sums its splits in split order, then times rinv, then + bias.
template <int TC, int NS>
__device__ __forceinline__ void tail_logits(const float* part, int nsplit, int T, int E, int ee,
                                            const float* bias, const float* rinv, float (*lg)[256]) {
  for (int t0 = 0; t0 < T; t0 += TC) {
    float v[TC][NS];
#pragma unroll
    for (int tt = 0; tt < TC; ++tt)
#pragma unroll
      for (int sp = 0; sp < NS; ++sp)
        v[tt][sp] = (t0 + tt < T && sp < nsplit) ? __ldcg(part + ((size_t)sp * T + t0 + tt) * E + ee) : 0.f;
#pragma unroll
    for (int tt = 0; tt < TC; ++tt) {
      if (t0 + tt < T) {
        float a = v[tt][0];
#pragma unroll
        for (int sp = 1; sp < NS; ++sp)
          if (sp < nsplit) a += v[tt][sp];
        if (rinv) a = __fmul_rn(a, rinv[t0 + tt]);
        if (bias) a = a + bias[ee];
        lg[t0 + tt][ee] = a;
      }
    }
  }
}

__global__ void __launch_bounds__(256) route_fast_kernel(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                                                         const float* __restrict__ bias, float* __restrict__ part,
                                                         int T, int H, int E, int k, int KS, int G,
                                                         int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ sorted_rows,
                                                         int32_t* __restrict__ row_pos, int4* __restrict__ groups,
                                                         int32_t* __restrict__ n_groups, int32_t* tickets,
                                                         Status* st, const uint16_t* __restrict__ g,
                                                         const float* __restrict__ rinv) {
  pdl_wait();
  pdl_trigger();
  __shared__ FastRouteSmem sm;
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp, split = blockIdx.y, k0 = split * KS;
  const int nv = KS / 128;  // 16-byte weight loads per lane
  // every weight load of this warp first
  float4 w[kFastKS / 128];
#pragma unroll
  for (int i = 0; i < kFastKS / 128; ++i)
    w[i] = (i < nv && e < E) ? __ldg(reinterpret_cast<const float4*>(wr + (size_t)e * H + k0 + i * 128 + lane * 4))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int t0 = 0; t0 < T; t0 += kFastTok) {
    const int nt = min(kFastTok, T - t0);
    __syncthreads();  // the previous pass's reads of the staging buffer are done
    for (int u = threadIdx.x; u < nt * (KS / 8); u += blockDim.x) {
      const int tt = u / (KS / 8), c = u % (KS / 8);
      *reinterpret_cast<uint4*>(&sm.xs[tt][c * 8]) =
          __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * H + k0 + c * 8));
    }
    __syncthreads();
    float acc[kFastTok];
#pragma unroll
    for (int tt = 0; tt < kFastTok; ++tt) acc[tt] = 0.f;
#pragma unroll
    for (int i = 0; i < kFastKS / 128; ++i) {
      if (i < nv) {
        const int kk = i * 128 + lane * 4;
        float g4[4] = {1.f, 1.f, 1.f, 1.f};
        if (g) {
          const uint2 gv = __ldg(reinterpret_cast<const uint2*>(g + k0 + kk));
          g4[0] = bf16_bits_to_f32(gv.x & 0xffffu);
          g4[1] = bf16_bits_to_f32(gv.x >> 16);
          g4[2] = bf16_bits_to_f32(gv.y & 0xffffu);
          g4[3] = bf16_bits_to_f32(gv.y >> 16);
        }
#pragma unroll
        for (int tt = 0; tt < kFastTok; ++tt) {
          if (tt < nt) {
            const uint2 xv = *reinterpret_cast<const uint2*>(&sm.xs[tt][kk]);
            float x4[4] = {bf16_bits_to_f32(xv.x & 0xffffu), bf16_bits_to_f32(xv.x >> 16),
                           bf16_bits_to_f32(xv.y & 0xffffu), bf16_bits_to_f32(xv.y >> 16)};
            if (g) {  // exact products
#pragma unroll
              for (int c = 0; c < 4; ++c) x4[c] = __fmul_rn(x4[c], g4[c]);
            }
            float a = acc[tt];
            a = fmaf(x4[0], w[i].x, a);
            a = fmaf(x4[1], w[i].y, a);
            a = fmaf(x4[2], w[i].z, a);
            a = fmaf(x4[3], w[i].w, a);
            acc[tt] = a;
          }
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < kFastTok; ++tt) {
      const float v = warp_sum(acc[tt]);
      if (lane == 0 && tt < nt && e < E) part[((size_t)split * T + t0 + tt) * E + e] = v;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's partials before its ticket
    s_last = (atomicAdd(&tickets[0], 1) == (int)(gridDim.x * gridDim.y) - 1);
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  // last CTA: logits (splits in order, times rinv, + bias), top k, table
  if ((int)threadIdx.x < E) {
    if (gridDim.y <= 8)
      tail_logits<4, 8>(part, gridDim.y, T, E, threadIdx.x, bias, rinv, sm.tail.lg);
    else
      tail_logits<2, 16>(part, gridDim.y, T, E, threadIdx.x, bias, rinv, sm.tail.lg);
  }
  __syncthreads();
  for (int t = warp; t < T; t += 8)
    topk_one_token(sm.tail.lg[t], E, k, topk_idx + (size_t)t * k, topk_w + (size_t)t * k, lane, sm.tail.pick + t * k);
  __syncthreads();
  build_table<256>(sm.tail.pick, T * k, E, G, offsets, sorted_rows, row_pos, groups, n_groups, st, sm.tail.tab);
}

// ---------------------------------------------------------------------------
// Router weights for the tensor-core router: w = w1 + w2 + w3 exactly, each a
// bf16 holding the next 8 significant bits of the fp32 value (w1, w2 by
// truncation, w3 by rounding the last 8 bits, which it holds exactly for any
// |w| >= 2^-110).  Laid out [E][3H] as (w1 | w2 | w3), so that
//   x . w = x . w1 + x . w2 + x . w3
// is one GEMM over K = 3H against x repeated three times.  Products of the bf16
// x with each part are exact in fp32, so the tensor core reproduces an fp32
// dot product up to the order of the fp32 sum.  Finite weights required.
// dup = 2 lays the parts out [E][6H] as (w1 | w1 | w2 | w2 | w3 | w3) for an
// input split in two bf16 parts (u1 | u2) repeated three times:
//   u . w = sum over parts b of (u1 . wb + u2 . wb).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ wr, int E, int H,
                                                           uint16_t* __restrict__ w3, int dup) {
  pdl_wait();
  pdl_trigger();
  // block (x, e): columns [x * 1024, x * 1024 + 1024) of expert row e, four per thread
  const int e = blockIdx.y, h = (blockIdx.x * 256 + threadIdx.x) * 4;
  if (h >= H) return;
  const float4 w4 = *reinterpret_cast<const float4*>(wr + (size_t)e * H + h);
  const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
  uint32_t p1[2], p2[2], p3[2];
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    uint32_t b1[2], b2[2], b3[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float w = wv[i + u];
      b1[u] = __float_as_uint(w) >> 16;
      const float r1 = w - __uint_as_float(b1[u] << 16);
      b2[u] = __float_as_uint(r1) >> 16;
      const float r2 = r1 - __uint_as_float(b2[u] << 16);
      b3[u] = f32_to_bf16_bits(r2);
    }
    p1[i / 2] = b1[0] | (b1[1] << 16);
    p2[i / 2] = b2[0] | (b2[1] << 16);
    p3[i / 2] = b3[0] | (b3[1] << 16);
  }
  uint16_t* row = w3 + (size_t)e * 3 * dup * H;
  for (int r = 0; r < dup; ++r) {
    *reinterpret_cast<uint2*>(row + (size_t)(0 * dup + r) * H + h) = make_uint2(p1[0], p1[1]);
    *reinterpret_cast<uint2*>(row + (size_t)(1 * dup + r) * H + h) = make_uint2(p2[0], p2[1]);
    *reinterpret_cast<uint2*>(row + (size_t)(2 * dup + r) * H + h) = make_uint2(p3[0], p3[1]);
  }
}

// ---------------------------------------------------------------------------
// Routing for many tokens, in three launches (no single-CTA pass over all rows):
//  1. topk_hist_kernel: chunks of 32 tokens (k*32 rows), one warp per token:
//     logits from the split partials (split order, + bias), the top k,
//     then each row's stable rank among the chunk's rows of its expert and the
//     chunk's per-expert counts;
//  2. table_scan_kernel (one CTA): per expert, offsets and the base position of
//     every chunk's rows (counts replaced in place), the group list;
//  3. table_scatter_kernel: sorted_rows[pos] = r, row_pos[r] = pos with
//     pos = base[chunk][expert] + rank.
// Row ids r = t*k + j keep their order inside an expert (the table is the same
// stable counting sort as build_table).
// ---------------------------------------------------------------------------
// Stable rank of each of a chunk's rows among the chunk's rows of its expert
// (row order), and the chunk's per-expert counts.  Threads 0..255 (warps 0-7)
// take local rows 0..255; picks[i] is local row i's expert, rows from
// `row0`; s_wcnt is zeroed shared scratch.  Every thread of the block calls it.
__device__ __forceinline__ void chunk_ranks(const int* picks, int nrow, int E, int row0, int chunk,
                                            int32_t* __restrict__ rank, int32_t* __restrict__ chunk_cnt,
                                            int (&s_wcnt)[8][256]) {
  const int i = threadIdx.x, warp = i >> 5, lane = i & 31;
  int e = 0, rk = 0;
  if (warp < 8) {
    e = i < nrow ? picks[i] : -1 - lane;  // rows past the end match nothing
    const unsigned same = __match_any_sync(0xffffffffu, e);
    rk = __popc(same & ((1u << lane) - 1u));
    if (i < nrow && rk == 0) s_wcnt[warp][e] = __popc(same);
  }
  __syncthreads();
  if (i < E) {
    int acc = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int c = s_wcnt[w][i];
      s_wcnt[w][i] = acc;
      acc += c;
    }
    chunk_cnt[(size_t)chunk * E + i] = acc;
  }
  __syncthreads();
  if (warp < 8 && i < nrow) rank[(size_t)row0 + i] = s_wcnt[warp][e] + rk;
}

__global__ void __launch_bounds__(1024) topk_hist_kernel(const float* __restrict__ part, int nsplit,
                                                         const float* __restrict__ bias, int T, int E, int k,
                                                         int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                         int32_t* __restrict__ rank, int32_t* __restrict__ chunk_cnt,
                                                         const float* __restrict__ rinv) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_lg[kChunkTok][256];
  __shared__ int s_pick[kChunkTok * 8];
  __shared__ int s_wcnt[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kChunkTok;
  const int ntok = min(kChunkTok, T - t0);
  for (int i = threadIdx.x; i < 8 * 256; i += 1024) (&s_wcnt[0][0])[i] = 0;
  if (warp < ntok) {
    // warp w takes token t0 + w; lane takes experts lane + 32 i, every load before the stores
    const int t = t0 + warp;
    float lg[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      lg[i] = e < E ? token_logit(part, nsplit, bias, T, E, t, e, rinv) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i < E) s_lg[warp][lane + 32 * i] = lg[i];
    __syncwarp();
    topk_one_token(s_lg[warp], E, k, topk_idx + (size_t)t * k, topk_w + (size_t)t * k, lane, s_pick + warp * k);
  }
  __syncthreads();
  chunk_ranks(s_pick, ntok * k, E, t0 * k, blockIdx.x, rank, chunk_cnt, s_wcnt);
}

// Routing table from caller-supplied expert ids, first pass: chunks of 32
// tokens as in topk_hist_kernel.  Ids outside [0, E) are reported on the
// device (LMOE_EDEVICE_CHECK) and counted as expert 0 so every index stays in
// range.
__global__ void __launch_bounds__(256) table_hist_kernel(const int32_t* __restrict__ topk_idx, int T, int E, int k,
                                                         int32_t* __restrict__ rank, int32_t* __restrict__ chunk_cnt,
                                                         Status* st) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_pick[kChunkTok * 8];
  __shared__ int s_wcnt[8][256];
  const int t0 = blockIdx.x * kChunkTok;
  const int nrow = min(kChunkTok, T - t0) * k;
  for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) (&s_wcnt[0][0])[i] = 0;
  if ((int)threadIdx.x < nrow) {
    int e = topk_idx[(size_t)t0 * k + threadIdx.x];
    if (e < 0 || e >= E) {
      set_error(st, LMOE_EDEVICE_CHECK, 104);
      e = 0;
    }
    s_pick[threadIdx.x] = e;
  }
  __syncthreads();
  chunk_ranks(s_pick, nrow, E, t0 * k, blockIdx.x, rank, chunk_cnt, s_wcnt);
}

__global__ void __launch_bounds__(256) table_scan_kernel(int32_t* __restrict__ chunk_cnt, int nchunks, int E, int R,
                                                         int G, int32_t* __restrict__ offsets,
                                                         int4* __restrict__ groups, int32_t* __restrict__ n_groups) {
  pdl_wait();
  pdl_trigger();
  const int e = threadIdx.x, warp = e >> 5, lane = e & 31;
  // chunk counts in batches of 8 independent loads
  int total = 0;
  if (e < E)
    for (int c0 = 0; c0 < nchunks; c0 += 8) {
      int v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = c0 + j < nchunks ? __ldcg(chunk_cnt + (size_t)(c0 + j) * E + e) : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) total += v[j];
    }
  const int gcnt = (total + G - 1) / G;
  // exclusive scans over experts (256 threads: warp scans, then warp totals)
  __shared__ int s_wr[8], s_wg[8];
  int rx = total, gx = gcnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ry = __shfl_up_sync(0xffffffffu, rx, o), gy = __shfl_up_sync(0xffffffffu, gx, o);
    if (lane >= o) {
      rx += ry;
      gx += gy;
    }
  }
  if (lane == 31) {
    s_wr[warp] = rx;
    s_wg[warp] = gx;
  }
  __syncthreads();
  int rbase = 0, gbase = 0;
  for (int w = 0; w < warp; ++w) {
    rbase += s_wr[w];
    gbase += s_wg[w];
  }
  const int off = rbase + rx - total, goff = gbase + gx - gcnt;
  if (e < E) {
    offsets[e] = off;
    int acc = off;
    for (int c0 = 0; c0 < nchunks; c0 += 8) {
      int v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = c0 + j < nchunks ? __ldcg(chunk_cnt + (size_t)(c0 + j) * E + e) : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < nchunks) {
          chunk_cnt[(size_t)(c0 + j) * E + e] = acc;  // base position of chunk c's rows of expert e
          acc += v[j];
        }
    }
    int gi = goff;
    for (int g0 = 0; g0 < total; g0 += G) groups[gi++] = make_int4(e, off + g0, min(G, total - g0), 0);
  }
  if (e == E - 1) {
    offsets[E] = off + total;  // = R
    *n_groups = goff + gcnt;
  }
}

__global__ void __launch_bounds__(256) table_scatter_kernel(const int32_t* __restrict__ topk_idx,
                                                            const int32_t* __restrict__ rank,
                                                            const int32_t* __restrict__ chunk_base, int R, int E,
                                                            int k, int32_t* __restrict__ sorted_rows,
                                                            int32_t* __restrict__ row_pos) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * 256 + threadIdx.x;
  if (r >= R) return;
  int e = topk_idx[r];
  if (e < 0 || e >= E) e = 0;  // as the first pass counted it (caller-supplied ids are checked there)
  const int c = (r / k) / kChunkTok;
  const int pos = chunk_base[(size_t)c * E + e] + rank[r];
  sorted_rows[pos] = r;
  row_pos[r] = pos;
}

}  // namespace lmoe
