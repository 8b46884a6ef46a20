// Routed experts, MXFP4 W4A16, decode-regime streaming kernels.
//
// "Muse Spark Open on Gaudi 2": experts run W4A16 ("What was built"), each
// (token, route) pair is its own row and the cost is per touched expert slice
// ("The latent MoE: A' with a per-expert norm"); the checkpoint's packed E2M1
// nibbles and E8M0 scales are read directly ("Why it needed a port").  The
// page's stock op unpacked every touched slice to bf16 in memory ("What it
// taught about Gaudi"); here nothing is unpacked in memory.
//
// Work item = (group of <= G rows of one expert, tile of 16 weight rows).
// gate/up tile: 8 gate rows + the 8 matching up rows (so SwiGLU is local to a
// lane); down tile: 16 consecutive output rows.  Each item streams its 16
// weight rows once (all of K) for every row of the group.
//
// CTA = W consumer warps + 1 producer warp.  The producer issues TMA bulk
// copies (codes, scales and the group's f16 activation rows for one K chunk)
// into per-warp rings of D slots guarded by mbarriers; consumer warp w
// handles items w, w+W, ... of the CTA's contiguous item range.
//
// Consumer inner loop per 32-element scale block: ldmatrix.x4 hands every
// lane 4 code bytes of a gate row and of an up row; cvt.rn.f16x2.e2m1x2 turns
// each byte into two exact f16 values; two mma.sync m16n8k16 (f16 in, fp32
// accumulate) take the K positions of one block in a fixed permutation that
// the activation fragment follows; the fresh block result is scaled by the
// block's E8M0 value and added to the fp32 accumulator.  Activations arrive
// as f16 scaled by a per-row power of two (exact; undone in the epilogue).
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

enum { MODE_GATEUP = 0, MODE_DOWN = 1 };

constexpr int kMaxKs = 128;  // scale bytes per row (K <= 4096)

template <int G, int KCMAX>
struct Layout {
  static constexpr int kCodeRow = KCMAX / 2 + 16;  // padded: 8 rows hit distinct banks for ldmatrix
  static constexpr int kCodes = 16 * kCodeRow;
  static constexpr int kScales = 16 * kMaxKs;
  static constexpr int kActRow = KCMAX * 2 + 64;   // padded: conflict-free 16-byte loads
  static constexpr int kActs = G * kActRow;
  static constexpr int kSlot = ((kCodes + kScales + kActs) + 127) / 128 * 128;
};

template <int MODE, int G, int KCMAX, int W, int D>
__global__ void __launch_bounds__(32 * (W + 1), 1) expert_kernel(const ExpertArgs a) {
  using Lay = Layout<G, KCMAX>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + W * D * Lay::kSlot);
  uint64_t* empty = full + W * D;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, kc = a.kc, Ks = K / 32, nch = K / kc;
  const int kcode_row = kc / 2 + 16;  // runtime row stride when kc < KCMAX keeps the padding rule
  const int kact_row = kc * 2 + 64;
  const int tiles = (MODE == MODE_GATEUP) ? a.inter / 8 : a.latent / 16;
  const int rows_per_expert = (MODE == MODE_GATEUP) ? 2 * a.inter : a.latent;

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

  const int n_items = *a.n_groups * tiles;
  const int it0 = (int)((long long)n_items * blockIdx.x / gridDim.x);
  const int it1 = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x);
  const int nloc = it1 - it0;

  if (warp == W) {
    // ------------------------------ producer ------------------------------
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int seq[W];
#pragma unroll
    for (int w = 0; w < W; ++w) seq[w] = 0;
    bool ok = true;
    for (int base = 0; base < nloc && ok; base += W) {
      const int nw = min(W, nloc - base);
      for (int c = 0; c < nch && ok; ++c) {
        const int k0 = c * kc;
        for (int w = 0; w < nw; ++w) {
          const int it = it0 + base + w;
          const int grp = it / tiles, tile = it % tiles;
          const int4 gi = a.groups[grp];
          const int e = gi.x, p0 = gi.y, ntok = gi.z;
          const int d = seq[w] % D;
          const uint32_t par = ((seq[w] / D) & 1) ^ 1;
          ++seq[w];
          if (!mbar_wait(&empty[w * D + d], par, a.st, 1)) {
            ok = false;
            break;
          }
          uint8_t* slot = smem + (w * D + d) * Lay::kSlot;
          uint64_t* bar = &full[w * D + d];
          const uint32_t bytes = 16u * (kc / 2) + 16u * Ks + (uint32_t)ntok * kc * 2;
          mbar_arrive_expect_tx(bar, bytes);
          // codes: 16 rows of kc/2 bytes
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {
            int row;
            if (MODE == MODE_GATEUP)
              row = e * rows_per_expert + (i < 8 ? tile * 8 + i : a.inter + tile * 8 + i - 8);
            else
              row = e * rows_per_expert + tile * 16 + i;
            bulk_g2s_stream(slot + i * kcode_row, a.q + (size_t)row * (K / 2) + k0 / 2, kc / 2, bar, pol);
          }
          // scales: whole rows (16 x Ks bytes)
          uint8_t* sdst = slot + Lay::kCodes;
          if (MODE == MODE_GATEUP) {
            const size_t g_row = (size_t)e * rows_per_expert + tile * 8;
            bulk_g2s(sdst, a.s + g_row * Ks, 8 * Ks, bar);
            bulk_g2s(sdst + 8 * Ks, a.s + (g_row + a.inter) * Ks, 8 * Ks, bar);
          } else {
            bulk_g2s(sdst, a.s + ((size_t)e * rows_per_expert + tile * 16) * Ks, 16 * Ks, bar);
          }
          // activations: ntok rows of kc f16
          uint8_t* adst = slot + Lay::kCodes + Lay::kScales;
          for (int j = 0; j < ntok; ++j) {
            int arow;
            if (MODE == MODE_GATEUP)
              arow = a.sorted_rows[p0 + j] / a.top_k;
            else
              arow = p0 + j;
            bulk_g2s(adst + j * kact_row, a.act16 + (size_t)arow * K + k0, kc * 2, bar);
          }
        }
      }
    }
    // drain: make sure no copy is still in flight when this thread leaves
#pragma unroll
    for (int w = 0; w < W; ++w) {
      for (int s = max(0, seq[w] - D); s < seq[w]; ++s) {
        mbar_wait(&full[w * D + (s % D)], (s / D) & 1, a.st, 2);
      }
    }
    return;
  }

  // -------------------------------- consumer --------------------------------
  const int g = lane >> 2, q = lane & 3;
  // ldmatrix.x4 source row/column for this lane: matrix m = lane/8
  const int lm_m = lane >> 3, lm_r = lane & 7;
  const int lm_row = lm_r + 8 * (lm_m & 1);
  const int lm_blk = lm_m >> 1;
  int seq = 0;
  for (int j = warp; j < nloc; j += W) {
    const int it = it0 + j;
    const int grp = it / tiles, tile = it % tiles;
    const int4 gi = a.groups[grp];
    const int p0 = gi.y, ntok = gi.z;
    float acc_lo[2] = {0.f, 0.f}, acc_hi[2] = {0.f, 0.f};
    for (int c = 0; c < nch; ++c) {
      const int d = seq % D;
      const uint32_t par = (seq / D) & 1;
      ++seq;
      if (!mbar_wait(&full[warp * D + d], par, a.st, 3)) return;
      const uint8_t* slot = smem + (warp * D + d) * Lay::kSlot;
      const uint32_t codes = smem_u32(slot);
      const uint8_t* sc = slot + Lay::kCodes;
      const uint32_t acts = smem_u32(slot + Lay::kCodes + Lay::kScales);
      const int kb0 = c * (kc / 32);
      const uint32_t lm_addr = codes + lm_row * kcode_row + lm_blk * 16;
      // lanes whose token column is beyond the group's capacity read row 0 (in
      // bounds); their mma columns are never stored
      const uint32_t act_addr = acts + (g < G ? g : 0) * kact_row + q * 16;
#pragma unroll 2
      for (int bb = 0; bb < kc / 32; bb += 2) {
        uint32_t w0, w1, w2, w3;
        ldmatrix_x4(w0, w1, w2, w3, lm_addr + bb * 16);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int blk = bb + half;
          const uint32_t wl = half ? w2 : w0, wh = half ? w3 : w1;
          uint32_t l0, l1, l2, l3, h0, h1, h2, h3;
          e2m1x8_to_f16x8(wl, l0, l1, l2, l3);
          e2m1x8_to_f16x8(wh, h0, h1, h2, h3);
          uint32_t b0, b1, b2, b3;
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                       : "r"(act_addr + blk * 64));
          float dacc[4];
          mma_f16_zero(dacc, l0, h0, l1, h1, b0, b1);
          mma_f16(dacc, l2, h2, l3, h3, b2, b3);
          const float s_lo = e8m0_to_f32(sc[g * Ks + kb0 + blk]);
          const float s_hi = e8m0_to_f32(sc[(8 + g) * Ks + kb0 + blk]);
          acc_lo[0] = fmaf(dacc[0], s_lo, acc_lo[0]);
          acc_lo[1] = fmaf(dacc[1], s_lo, acc_lo[1]);
          acc_hi[0] = fmaf(dacc[2], s_hi, acc_hi[0]);
          acc_hi[1] = fmaf(dacc[3], s_hi, acc_hi[1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[warp * D + d]);
    }
    // ------------------------------ epilogue ------------------------------
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int tok = 2 * q + i;
      if (tok < ntok) {
        const int p = p0 + tok;
        if (MODE == MODE_GATEUP) {
          const int t = a.sorted_rows[p] / a.top_k;
          const float inv = ldexpf(1.0f, -a.act_exp[t]);
          const float gv = acc_lo[i] * inv, uv = acc_hi[i] * inv;
          const float hv = gv / (1.0f + expf(-gv)) * uv;
          a.h_out[(size_t)p * a.inter + tile * 8 + g] = f32_to_bf16_bits(hv);
        } else {
          const int r = a.sorted_rows[p];
          const float inv = ldexpf(1.0f, -a.act_exp[p]);
          float* yr = a.y_out + (size_t)r * a.latent + tile * 16;
          yr[g] = acc_lo[i] * inv;
          yr[g + 8] = acc_hi[i] * inv;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launch configuration
// ---------------------------------------------------------------------------
int expert_max_group(int T) { return T <= 1 ? 1 : 8; }

static int pick_kc(int K, int kcmax) {
  int kc = kcmax;
  while (kc > 128 && (K % kc) != 0) kc >>= 1;
  if (kc > K) kc = K;
  while (K % kc) kc >>= 1;
  return kc;
}

template <int MODE, int G, int KCMAX, int W, int D>
static int launch_one(ExpertArgs a, cudaStream_t s, int num_sms) {
  using Lay = Layout<G, KCMAX>;
  auto kern = expert_kernel<MODE, G, KCMAX, W, D>;
  const int smem = W * D * Lay::kSlot + 2 * W * D * 8;
  static_assert(W * D * Lay::kSlot + 2 * W * D * 8 <= 232448, "shared memory budget");
  static unsigned long long attr_done = 0;  // one bit per device, per template instance
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done >> (dev & 63) & 1ull)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return LMOE_ECUDA;
    attr_done |= 1ull << (dev & 63);
  }
  a.kc = pick_kc(a.K, KCMAX);
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

int launch_gateup(const ExpertArgs& a, int T, int max_group, cudaStream_t s, int num_sms) {
  if (max_group == 1) return launch_one<MODE_GATEUP, 1, 2048, 5, 2>(a, s, num_sms);
  return launch_one<MODE_GATEUP, 8, 1024, 4, 2>(a, s, num_sms);
}

int launch_down(const ExpertArgs& a, int T, int max_group, cudaStream_t s, int num_sms) {
  if (max_group == 1) return launch_one<MODE_DOWN, 1, 2048, 5, 2>(a, s, num_sms);
  return launch_one<MODE_DOWN, 8, 1024, 4, 2>(a, s, num_sms);
}

}  // namespace lmoe
