// bf16 x bf16 -> bf16 projections for small token counts (pooler and
// unpooler in the decode regime).
//
// "Soporte de dia 0 para Muse Spark Open en vLLM", section "MoE latente": the
// pooler maps each token 8192 -> 4096 and the unpooler 4096 -> 8192, both
// learned matrices shared by all experts.  "Muse Spark Open on Gaudi 2",
// "Correctness": bf16 values with fp32 accumulation.
//
// out[t][n] = bf16_rne(sum_k act[t][k] * W[n][k]).  At small T this is a
// weight stream: each item is 16 weight rows x all of K for a group of up to
// 8*NT tokens; weights and the matching activation chunk arrive by TMA bulk
// copies in per-warp mbarrier rings, and mma.sync m16n8k16 (bf16 in, fp32
// accumulate) does the products with both operands fed by ldmatrix.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

template <int NT, int KC>
struct GemvLayout {
  static constexpr int kRow = KC * 2 + 16;  // padded row: ldmatrix phases hit distinct banks
  static constexpr int kW = 16 * kRow;
  static constexpr int kA = 8 * NT * kRow;
  static constexpr int kSlot = (kW + kA + 127) / 128 * 128;
};

template <int NT, int KC, int W, int D>
__global__ void __launch_bounds__(32 * (W + 1), 1) gemv_bf16_kernel(const GemvArgs a) {
  using Lay = GemvLayout<NT, KC>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + W * D * Lay::kSlot);
  uint64_t* empty = full + W * D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, nch = K / KC;
  constexpr int GT = 8 * NT;
  const int ngroups = (a.T + GT - 1) / GT;
  const int n_items = (a.N / 16) * ngroups;

  if (threadIdx.x == 0) {
    for (int i = 0; i < W * D; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  const int it0 = (int)((long long)n_items * blockIdx.x / gridDim.x);
  const int it1 = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x);
  const int nloc = it1 - it0;

  if (warp == W) {
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int seq[W];
#pragma unroll
    for (int w = 0; w < W; ++w) seq[w] = 0;
    bool ok = true;
    for (int base = 0; base < nloc && ok; base += W) {
      const int nw = min(W, nloc - base);
      for (int c = 0; c < nch && ok; ++c) {
        const int k0 = c * KC;
        for (int w = 0; w < nw; ++w) {
          const int it = it0 + base + w;
          // token group outer, row tile inner: consecutive items share tokens
          const int tg = it / (a.N / 16), mt = it % (a.N / 16);
          const int t0 = tg * GT, ntok = min(GT, a.T - t0);
          const int d = seq[w] % D;
          const uint32_t par = ((seq[w] / D) & 1) ^ 1;
          ++seq[w];
          if (!mbar_wait(&empty[w * D + d], par, a.st, 11)) {
            ok = false;
            break;
          }
          uint8_t* slot = smem + (w * D + d) * Lay::kSlot;
          uint64_t* bar = &full[w * D + d];
          mbar_arrive_expect_tx(bar, 16u * KC * 2 + (uint32_t)ntok * KC * 2);
#pragma unroll 4
          for (int i = 0; i < 16; ++i)
            bulk_g2s_stream(slot + i * Lay::kRow, a.w + (size_t)(mt * 16 + i) * K + k0, KC * 2, bar, pol);
          for (int j = 0; j < ntok; ++j)
            bulk_g2s(slot + Lay::kW + j * Lay::kRow, a.act + (size_t)(t0 + j) * K + k0, KC * 2, bar);
        }
      }
    }
#pragma unroll
    for (int w = 0; w < W; ++w)
      for (int s = max(0, seq[w] - D); s < seq[w]; ++s) mbar_wait(&full[w * D + (s % D)], (s / D) & 1, a.st, 12);
    return;
  }

  const int g = lane >> 2, q = lane & 3;
  const int lm_m = lane >> 3, lm_r = lane & 7;
  // A (weights, 16 rows x 16 k): matrices (rows 0-7,k0-7) (rows 8-15,k0-7) (rows 0-7,k8-15) (rows 8-15,k8-15)
  const int a_row = lm_r + 8 * (lm_m & 1), a_col = 16 * (lm_m >> 1);
  // B (tokens, 8 x 16 k) via x4: matrices (tok 0-7,k0-7) (tok 0-7,k8-15) for k-step s and s+1
  const int b_col = 16 * (lm_m & 1) + 32 * (lm_m >> 1);
  int seq = 0;
  for (int j = warp; j < nloc; j += W) {
    const int it = it0 + j;
    const int tg = it / (a.N / 16), mt = it % (a.N / 16);
    const int t0 = tg * GT, ntok = min(GT, a.T - t0);
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    for (int c = 0; c < nch; ++c) {
      const int d = seq % D;
      const uint32_t par = (seq / D) & 1;
      ++seq;
      if (!mbar_wait(&full[warp * D + d], par, a.st, 13)) return;
      const uint32_t base = smem_u32(smem + (warp * D + d) * Lay::kSlot);
      const uint32_t a_addr = base + a_row * Lay::kRow + a_col;
      const uint32_t b_addr = base + Lay::kW + lm_r * Lay::kRow + b_col;
#pragma unroll 4
      for (int ks = 0; ks < KC / 16; ks += 2) {
        uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
        ldmatrix_x4(a0, a1, a2, a3, a_addr + ks * 32);
        ldmatrix_x4(a4, a5, a6, a7, a_addr + ks * 32 + 32);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(b0, b1, b2, b3, b_addr + n * 8 * Lay::kRow + ks * 32);
          mma_bf16(acc[n], a0, a1, a2, a3, b0, b1);
          mma_bf16(acc[n], a4, a5, a6, a7, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[warp * D + d]);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int tok = n * 8 + 2 * q + i;
        if (tok < ntok) {
          uint16_t* o = a.out + (size_t)(t0 + tok) * a.N + mt * 16;
          o[g] = f32_to_bf16_bits(acc[n][i]);
          o[g + 8] = f32_to_bf16_bits(acc[n][2 + i]);
        }
      }
    }
  }
}

template <int NT, int KC, int W, int D>
static int launch_gemv(const GemvArgs& a, cudaStream_t s, int num_sms) {
  using Lay = GemvLayout<NT, KC>;
  auto kern = gemv_bf16_kernel<NT, KC, W, D>;
  constexpr int smem = W * D * Lay::kSlot + 2 * W * D * 8;
  static_assert(smem <= 232448, "shared memory budget");
  static unsigned long long attr_done = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done >> (dev & 63) & 1ull)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return LMOE_ECUDA;
    attr_done |= 1ull << (dev & 63);
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
  return cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

int launch_gemv_bf16(const GemvArgs& a, cudaStream_t s, int num_sms) {
  if (a.K % 512 != 0) {
    // small K (tiny shapes): one chunk of 128
    if (a.T <= 8) return launch_gemv<1, 128, 4, 2>(a, s, num_sms);
    return launch_gemv<4, 128, 4, 2>(a, s, num_sms);
  }
  if (a.T <= 8) return launch_gemv<1, 512, 4, 2>(a, s, num_sms);
  if (a.T <= 16) return launch_gemv<2, 512, 3, 2>(a, s, num_sms);
  return launch_gemv<4, 512, 4, 1>(a, s, num_sms);
}

}  // namespace lmoe
