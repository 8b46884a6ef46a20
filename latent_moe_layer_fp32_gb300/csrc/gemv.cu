// bf16 x bf16 -> bf16 projections for small token counts (pooler and
// unpooler in the decode regime).
//
// "Soporte de dia 0 para Muse Spark Open en vLLM", section "MoE latente": the
// pooler maps each token 8192 -> 4096 and the unpooler 4096 -> 8192, both
// learned matrices shared by all experts.  "Muse Spark Open on Gaudi 2",
// "Correctness": bf16 values with fp32 accumulation.
//
// out[t][n] = bf16_rne(sum_k act[t][k] * W[n][k]).  At small T this is a
// weight stream.  Item = 16 weight rows x all of K for a group of up to 8*NT
// tokens; the W consumer warps of a CTA share an item (chunk c of 512 K
// elements goes to warp c % W) and add their fp32 partials in warp order at
// the end.  Per chunk the producer issues one TMA tensor copy of the weights
// (a 3-D view {64 elements, rows, K/64} with 128-byte swizzle: 16 rows x 512
// elements, 16 KB) and one of the token rows (min(8*NT, T) rows: at one token a
// 1 KB box instead of 8 KB mostly zero-filled; tokens beyond T read as zero);
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) takes both operands by
// ldmatrix from the swizzled boxes.
#include "common.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace lmoe {


// KC: K elements per chunk (KC/64 planes of 64); 512 gives 16 KB weight boxes
template <int NT, int KC>
struct GemvLayout {
  static constexpr int kW = 16 * KC * 2;       // 16 KB at KC = 512
  static constexpr int kA = 8 * NT * KC * 2;   // 8 KB per n-tile at KC = 512
  static constexpr int kSlot = (kW + kA + 1023) / 1024 * 1024;
};

template <int NT, int KC, int W, int D>
__global__ void __launch_bounds__(32 * (W + 1), 1)
    gemv_bf16_kernel(const GemvArgs a, const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x) {
  using Lay = GemvLayout<NT, KC>;
  constexpr int kGemvKC = KC;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red = reinterpret_cast<float*>(smem + W * D * Lay::kSlot);  // [W][NT][4][32]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + W * NT * 4 * 32);
  uint64_t* empty = full + W * D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, nch = K / kGemvKC;
  constexpr int GT = 8 * NT;
  const int ngroups = (a.T + GT - 1) / GT;
  const int mtiles = a.N / 16;
  const int n_items = mtiles * ngroups;
  // token rows per box: the token group (8*NT), or T when fewer -- the MMA's columns past
  // the last token read whatever the slot holds there and are never stored
  const int xrows = min(GT, a.T);
  const uint32_t xbytes = (uint32_t)xrows * kGemvKC * 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < W * D; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int it0 = (int)((long long)n_items * blockIdx.x / gridDim.x);
  const int it1 = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x);
  const int mode = a.wait_mode;

  if (warp == W) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
      const uint64_t pol = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      // Chunk c of an item goes to consumer warp c % W; chunks are issued in
      // (item, chunk) order.  With kWaitAfterWeights the weight copies of the
      // first chunks (while their warps' slots are still unused) go out before
      // the wait and their token rows after it.
      int seq[W];
#pragma unroll
      for (int w = 0; w < W; ++w) seq[w] = 0;
      int npre = 0;
      if (mode == kWaitAfterWeights) {
        bool room = true;
        for (int it = it0; it < it1 && room; ++it)
          for (int c = 0; c < nch; ++c) {
            const int w = c % W;
            if (seq[w] >= D) {
              room = false;
              break;
            }
            const int d = seq[w]++;
            uint8_t* slot = smem + (w * D + d) * Lay::kSlot;
            uint64_t* bar = &full[w * D + d];
            mbar_arrive_expect_tx(bar, Lay::kW + xbytes);  // token rows follow after the wait
            tma_load_3d(slot, &tm_w, 0, (it % mtiles) * 16, c * (kGemvKC / 64), bar, pol);
            ++npre;
          }
#pragma unroll
        for (int w = 0; w < W; ++w) seq[w] = 0;
      }
      if (mode != kWaitAtEnd) {
        pdl_wait();
        pdl_trigger();
      }
      bool ok = true;
      int lin = 0;
      for (int it = it0; it < it1 && ok; ++it) {
        // token group outer, row tile inner: consecutive items share tokens
        const int tg = it / mtiles, mt = it % mtiles;
        for (int c = 0; c < nch; ++c, ++lin) {
          const int w = c % W;
          const int d = seq[w] % D;
          const uint32_t par = ((seq[w] / D) & 1) ^ 1;
          ++seq[w];
          uint8_t* slot = smem + (w * D + d) * Lay::kSlot;
          uint64_t* bar = &full[w * D + d];
          if (lin >= npre) {
            if (!mbar_wait(&empty[w * D + d], par, a.st, 11)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar, Lay::kW + xbytes);  // out-of-range token rows are zero-filled, bytes still count
            tma_load_3d(slot, &tm_w, 0, mt * 16, c * (kGemvKC / 64), bar, pol);
          }
          tma_load_3d(slot + Lay::kW, &tm_x, 0, tg * GT, c * (kGemvKC / 64), bar, pol_x);
        }
      }
#pragma unroll
      for (int w = 0; w < W; ++w)
        for (int s = max(0, seq[w] - D); s < seq[w]; ++s) mbar_wait(&full[w * D + (s % D)], (s / D) & 1, a.st, 12);
    }
    // The other lanes wait for lane 0 here: a lane parked in griddepcontrol.wait
    // would hold the whole warp, lane 0's copies included, until the preceding
    // kernel completes.
    __syncwarp();
    if (mode == kWaitAtEnd) {
      pdl_wait();
      pdl_trigger();
    }
    return;
  }
  // consumers read only shared memory and write outputs nothing earlier in the stream touches
  if (mode != kWaitAtEnd) {
    pdl_wait();
    pdl_trigger();
  }

  const int g = lane >> 2, q = lane & 3;
  const int lm = lane >> 3, rr = lane & 7;
  // A (weights, 16 rows x 16 k) x4: (rows 0-7,k0-7) (rows 8-15,k0-7) (rows 0-7,k8-15) (rows 8-15,k8-15)
  const int a_row = rr + 8 * (lm & 1), a_k8 = lm >> 1;
  // B (tokens, 8 x 16 k) x4 over k-steps s, s+1: (k0-7) (k8-15) (k16-23) (k24-31)
  const int b_k8 = lm;
  int seq = 0;
  bool alive = true;
  for (int it = it0; it < it1; ++it) {
    const int tg = it / mtiles, mt = it % mtiles;
    const int t0 = tg * GT, ntok = min(GT, a.T - t0);
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    for (int c = warp; c < nch && alive; c += W) {
      const int d = seq % D;
      const uint32_t par = (seq / D) & 1;
      ++seq;
      if (!mbar_wait(&full[warp * D + d], par, a.st, 13)) {
        alive = false;
        break;
      }
      const uint32_t base = smem_u32(smem + (warp * D + d) * Lay::kSlot);
      const uint32_t xbase = base + Lay::kW;
#pragma unroll 4
      for (int ks = 0; ks < kGemvKC / 16; ks += 2) {
        // element k of the chunk: plane k/64, 16-byte chunk (k%64)/8
        uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
        {
          const int k8 = ks * 2 + a_k8;  // 8-element column index for k-step ks
          ldmatrix_x4(a0, a1, a2, a3, base + swz128(k8 >> 3, 16, a_row, k8 & 7));
          const int k8b = k8 + 2;        // k-step ks + 1
          ldmatrix_x4(a4, a5, a6, a7, base + swz128(k8b >> 3, 16, a_row, k8b & 7));
        }
        const int bk8 = ks * 2 + b_k8;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          uint32_t b0, b1, b2, b3;
          // line (plane * xrows + row) of the token box; the 128-byte swizzle XORs the 16-byte
          // chunk with the line index (the box base is 1024-byte aligned)
          const int xl = (bk8 >> 3) * xrows + n * 8 + rr;
          ldmatrix_x4(b0, b1, b2, b3, xbase + (uint32_t)((xl << 7) + (((bk8 & 7) ^ (xl & 7)) << 4)));
          mma_bf16(acc[n], a0, a1, a2, a3, b0, b1);
          mma_bf16(acc[n], a4, a5, a6, a7, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[warp * D + d]);
    }
    // cross-warp reduction in warp order (named barrier over the consumers only)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[((warp * NT + n) * 4 + i) * 32 + lane] = acc[n][i];
    asm volatile("bar.sync 1, %0;" ::"r"(W * 32) : "memory");
    if (warp == 0) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[i] = red[((0 * NT + n) * 4 + i) * 32 + lane];
          for (int w = 1; w < W; ++w) v[i] += red[((w * NT + n) * 4 + i) * 32 + lane];
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int tok = n * 8 + 2 * q + i;
          const uint16_t b_lo = f32_to_bf16_bits(v[i]), b_hi = f32_to_bf16_bits(v[2 + i]);
          if (tok < ntok) {
            uint16_t* o = a.out + (size_t)(t0 + tok) * a.N + mt * 16;
            o[g] = b_lo;
            o[g + 8] = b_hi;
          }
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(W * 32) : "memory");
  }
  if (mode == kWaitAtEnd) {
    pdl_wait();
    pdl_trigger();
  }
}

template <int NT, int KC, int W, int D>
static int launch_gemv(const GemvArgs& a, cudaStream_t s, int num_sms) {
  using Lay = GemvLayout<NT, KC>;
  constexpr int kGemvKC = KC;
  auto kern = gemv_bf16_kernel<NT, KC, W, D>;
  constexpr int smem = W * D * Lay::kSlot + W * NT * 4 * 32 * 4 + 2 * W * D * 8 + 1024;
  static_assert(smem <= 232448, "shared memory budget");
  static unsigned long long attr_done = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done >> (dev & 63) & 1ull)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return LMOE_ECUDA;
    attr_done |= 1ull << (dev & 63);
  }
  CUtensorMap tw, tx;
  {
    // {64 elements (128 B), rows, K/64 planes}: plane stride 128 B, row stride 2K B
    const uint64_t dims[3] = {64, (uint64_t)a.N, (uint64_t)a.K / 64};
    const uint64_t strides[2] = {(uint64_t)a.K * 2, 128};
    const uint32_t box[3] = {64, 16, kGemvKC / 64};
    if (get_tmap(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return LMOE_ECUDA;
  }
  {
    const uint64_t dims[3] = {64, (uint64_t)a.T, (uint64_t)a.K / 64};
    const uint64_t strides[2] = {(uint64_t)a.K * 2, 128};
    const uint32_t box[3] = {64, (uint32_t)min(8 * NT, a.T), kGemvKC / 64};
    if (get_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.act, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return LMOE_ECUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(32 * (W + 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, tw, tx) == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

int launch_gemv_bf16(const GemvArgs& a, cudaStream_t s, int num_sms) {
  if (a.K % 512 == 0) {
    if (a.T <= 8) return launch_gemv<1, 512, 4, 2>(a, s, num_sms);
    if (a.T <= 16) return launch_gemv<2, 512, 3, 2>(a, s, num_sms);
    return launch_gemv<4, 512, 2, 2>(a, s, num_sms);
  }
  if (a.T <= 8) return launch_gemv<1, 256, 4, 4>(a, s, num_sms);
  if (a.T <= 16) return launch_gemv<2, 256, 4, 3>(a, s, num_sms);
  return launch_gemv<4, 256, 4, 2>(a, s, num_sms);
}

}  // namespace lmoe
