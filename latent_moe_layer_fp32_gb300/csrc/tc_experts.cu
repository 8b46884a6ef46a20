// Routed experts for many tokens: grouped W4A16 GEMMs on tcgen05.
//
// "Muse Spark Open on Gaudi 2", section "The latent MoE: A' with a per-expert
// norm" and "Soporte de dia 0 para Muse Spark Open en vLLM", section "MoE
// latente": each routed row r = (token, route) of expert e computes
//   h_r = bf16(silu(x_lat . Wg_e^T) * (x_lat . Wu_e^T)),   y_r = h_r . Wd_e^T,
// with MXFP4 weights (OCP MX v1.0: E2M1 codes, one E8M0 scale per 32 K
// elements) and bf16 activations, fp32 accumulation.
//
// One work item = one group of up to 160 rows of one expert (sorted
// positions p0 .. p0+n-1) x output features: one 128-row tile of the gate and
// of the up half (gate/up), or two consecutive 128-row tiles (down), so every
// activation stage feeds two MMAs.
// The weight tile is the MMA's A operand (M = 128), the group's activation
// rows are B (N = n rounded up to 16), so ragged groups cost no padded rows
// of A.  Per CTA (persistent, one per SM, 19 warps):
//   warp 0      TMA: raw MXFP4 codes, 128 rows x 256 K per stage (16 KB per
//               weight matrix), into a ring
//   warp 1      TMA: activation rows (sorted order), 32-row boxes of 64 K
//   warp 2      TMEM owner; one thread issues tcgen05.mma kind::f16 with A
//               read from tensor memory and B from shared memory
//   warps 3-10  dequantise codes to bf16 (E2M1 x 2^(s-127) is exact in
//               bf16); a thread owns one weight row, which is one TMEM lane,
//               and stores its 64 K of a step with tcgen05.st, so the
//               dequantised operand never passes through shared memory
//   warps 11-18 epilogue: tcgen05.ld, SwiGLU -> h (gate/up), or y and the
//               per-32-column sums of squares for post_expert_norm (down);
//               two warps per TMEM lane quarter take alternate 32-column chunks
// NVFP4 weights (FMT = 1): E4M3 scales per 16 elements and an fp32 global
// scale per expert matrix.  E2M1 x E4M3 has at most 6 significant bits and is
// exact in bf16 for every scale byte, so the dequantiser builds each 16-block's
// eight scaled patterns with fp32 products; the epilogue applies the global
// scale to the accumulators.
// Tensor memory (512 columns): accumulators of 160 columns (gate/up: gate at
// 0, up at 160, so SwiGLU pairs are lane-local; down: the item's two 128-row
// output tiles at 0 and 160), and from column 320 the A stages, 32 columns
// (64 K of bf16) per weight matrix.
#include <atomic>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace lmoe {
namespace {

constexpr int kXM = 128;                 // weight rows per matrix tile (MMA M)
constexpr int kXNmax = kTcExpertGroup;   // activation rows per group (MMA N, max): 160
constexpr int kXTile = kXM * 128;        // 16 KB: 128 rows x 128 B of codes (256 K)
constexpr int kXBStage = kXNmax * 128;   // 20 KB: 160 activation rows x 64 K bf16
constexpr int kXAcc = 160;               // TMEM columns per accumulator
constexpr int kXACol = 320;              // first TMEM column of the A stages
static_assert(kXNmax <= kXAcc && kXNmax % 32 == 0, "group rows fit an accumulator");
constexpr int kXBBox = 32 * 128;         // one 32-row activation box
constexpr int kDqWarps = 8, kEpWarps = 8;
constexpr int kXThreads = (3 + kDqWarps + kEpWarps) * 32;

template <int MODE>
struct XCfg;
template <>
struct XCfg<0> {  // gate/up: two weight matrices per item, single accumulator pair
  static constexpr int NMAT = 2, RAW = 3, ST = 3, NACC = 1;
};
template <>
struct XCfg<2> {  // down, two 128-row output tiles per item sharing each activation stage
  static constexpr int NMAT = 2, RAW = 3, ST = 3, NACC = 1;
};
static_assert(kXACol + XCfg<0>::ST * XCfg<0>::NMAT * 32 <= 512 && 2 * kXAcc <= kXACol, "TMEM columns");
static_assert(kXACol + XCfg<2>::ST * XCfg<2>::NMAT * 32 <= 512 && 2 * kXAcc <= kXACol, "TMEM columns");

template <int MODE>
constexpr int xring_bytes() {
  using C = XCfg<MODE>;
  return C::RAW * C::NMAT * kXTile + C::ST * kXBStage;
}
template <int MODE>
constexpr int xsmem_bytes() {
  return xring_bytes<MODE>() + 1024 + 256;
}
static_assert(xsmem_bytes<0>() <= 232448 && xsmem_bytes<2>() <= 232448,
              "shared memory budget");

// ---------------------------------------------------------------------------
// MXFP4 -> bf16.  E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 have bf16 bit
// patterns 0, 3F00, 3F80, 3FC0, 4000, 4040, 4080, 40C0; the E8M0 scale
// 2^(s-127) adds s-127 to the exponent field of every nonzero magnitude,
// exact while the result stays a normal number (2 <= s <= 252).  A block's
// eight scaled patterns are split into low-byte and high-byte tables and
// looked up with byte permutes, 3-bit code magnitudes as selectors.
// ---------------------------------------------------------------------------
struct DqTable {
  uint32_t la, lb, ha, hb;  // low / high bytes of the patterns of magnitudes 0-3 and 4-7
};

__device__ __forceinline__ DqTable dq_table(uint32_t s) {
  const uint32_t d = s * 128u - 127u * 128u;  // (s - 127) << 7, two's complement
  const uint32_t p01 = 0x3F000000u + (d << 16);
  const uint32_t p23 = 0x3FC03F80u + d * 0x10001u;
  const uint32_t p45 = 0x40404000u + d * 0x10001u;
  const uint32_t p67 = 0x40C04080u + d * 0x10001u;
  DqTable t;
  t.la = __byte_perm(p01, p23, 0x6420);
  t.ha = __byte_perm(p01, p23, 0x7531);
  t.lb = __byte_perm(p45, p67, 0x6420);
  t.hb = __byte_perm(p45, p67, 0x7531);
  return t;
}

// Eight codes (one word, element i in nibble i) -> four bf16x2 words.
__device__ __forceinline__ void dq8(uint32_t w, const DqTable& t, uint32_t* o) {
  const uint32_t mags = w & 0x77777777u;
  const uint32_t w4 = w * 16u;  // multiply forms of the shifts run on the FMA pipe, not the integer ALU
  // byte i of sa / sb carries the sign of element i / 4+i in its top bit
  const uint32_t sa = __byte_perm(w4, w, 0x5140);
  const uint32_t sb = __byte_perm(w4, w, 0x7362);
  uint32_t lo = __byte_perm(t.la, t.lb, mags);
  uint32_t hi = __byte_perm(t.ha, t.hb, mags) | (sa & 0x80808080u);
  o[0] = __byte_perm(lo, hi, 0x5140);
  o[1] = __byte_perm(lo, hi, 0x7362);
  const uint32_t mh = __umulhi(mags, 0x10000u);  // mags >> 16
  lo = __byte_perm(t.la, t.lb, mh);
  hi = __byte_perm(t.ha, t.hb, mh) | (sb & 0x80808080u);
  o[2] = __byte_perm(lo, hi, 0x5140);
  o[3] = __byte_perm(lo, hi, 0x7362);
}

// NVFP4: the eight patterns of one 16-element block under E4M3 scale byte s,
// as products in fp32 (exact, with at most 6 significant bits, so the bf16
// pattern is the top half).  E4M3 -> f16 -> f32 is exact.
__device__ __forceinline__ DqTable dq_table_nv(uint32_t s) {
  uint32_t f2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f2) : "h"((uint16_t)s));
  const float sc = __half2float(__ushort_as_half((unsigned short)(f2 & 0xffffu)));
  const float mags[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  uint32_t pat[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) pat[i] = __float_as_uint(__fmul_rn(mags[i], sc)) >> 16;
  const uint32_t p01 = pat[0] | (pat[1] << 16), p23 = pat[2] | (pat[3] << 16);
  const uint32_t p45 = pat[4] | (pat[5] << 16), p67 = pat[6] | (pat[7] << 16);
  DqTable t;
  t.la = __byte_perm(p01, p23, 0x6420);
  t.ha = __byte_perm(p01, p23, 0x7531);
  t.lb = __byte_perm(p45, p67, 0x6420);
  t.hb = __byte_perm(p45, p67, 0x7531);
  return t;
}

// Scales outside the exponent-add range (subnormal, overflowing or NaN
// results): the value in fp32, then bf16 (exact: every finite product is
// representable in bf16).
__device__ __forceinline__ void dq_block_exact(uint4 c, uint32_t s, uint32_t* o) {
  const float sc = e8m0_to_f32(s);
  const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    uint32_t pair = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t code = (wv[i >> 2] >> (8 * (i & 3) + 4 * h)) & 15u;
      const uint32_t m = code & 7u;
      float mag = m < 2 ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)(m & 1u), (int)(m >> 1) - 1);
      if (code & 8u) mag = -mag;
      pair |= (uint32_t)f32_to_bf16_bits(mag * sc) << (16 * h);
    }
    o[i] = pair;
  }
}

// 32 codes (16 bytes) with scale byte s -> 32 bf16 (16 words).  `fast`: the
// caller has checked 2 <= s <= 252.
__device__ __forceinline__ void dq_block(uint4 c, uint32_t s, uint32_t* o, bool fast) {
  if (fast) {
    const DqTable t = dq_table(s);
    dq8(c.x, t, o);
    dq8(c.y, t, o + 4);
    dq8(c.z, t, o + 8);
    dq8(c.w, t, o + 12);
  } else {
    dq_block_exact(c, s, o);
  }
}

}  // namespace

// One group of the item list, checked: false (and an error recorded) for an
// entry the routing table could not have produced.
struct XItem {
  int e, p0, n, ft;
};

// Group entry of item `it` (loaded one item ahead by every role).
__device__ __forceinline__ int4 x_group(const TcExpertArgs& a, int it, int nft, int n_items) {
  return it < n_items ? __ldg(&a.groups[it / nft]) : make_int4(0, 0, 0, 0);
}

__device__ __forceinline__ bool x_item(const TcExpertArgs& a, int4 g, int it, int nft, XItem* x) {
  x->e = g.x;
  x->p0 = g.y;
  x->n = g.z;
  x->ft = it % nft;
  if (g.x < 0 || g.x >= a.n_experts || g.z < 1 || g.z > kXNmax || g.y < 0 || g.y + g.z > a.rows) {
    set_error(a.st, LMOE_EDEVICE_CHECK, 60);
    return false;
  }
  return true;
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(kXThreads, 1)
    tc_expert_kernel(const TcExpertArgs a, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_act) {
  using C = XCfg<MODE>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_raw = smem;                                   // [RAW][NMAT] code tiles
  uint8_t* s_b = s_raw + C::RAW * C::NMAT * kXTile;        // [ST] activation stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_b + C::ST * kXBStage);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + C::RAW;
  // step stage s: A (TMEM columns) and B (shared memory) of one 64-K step.
  // full[s]: the dequant warps' arrivals + the activation TMA's arrival and
  // bytes; empty[s]: one MMA commit frees both halves.
  uint64_t* full = raw_empty + C::RAW;
  uint64_t* empty = full + C::ST;
  uint64_t* acc_full = empty + C::ST;
  uint64_t* acc_empty = acc_full + C::NACC;
  uint64_t* done = acc_empty + C::NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::RAW; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kDqWarps);
    }
    for (int i = 0; i < C::ST; ++i) {
      mbar_init(&full[i], kDqWarps + 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < C::NACC; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpWarps);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 2) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();
  pdl_trigger();

  // rows of the weight matrix per item and matrix tile m: gate/up: tile ft of the gate
  // (m = 0) and up (m = 1) halves; down: the 128-row tiles 2 ft and 2 ft + 1
  constexpr int TPI = MODE == 2 ? 2 : 1;                            // output tiles per item
  const int nft = (MODE == 0 ? a.inter : a.latent) / (kXM * TPI);  // items per group
  const int n_items = *a.n_groups * nft;
  const int K = a.K, nks = K / 64, nkr = K / 256;
  const int rows_pe = MODE == 0 ? 2 * a.inter : a.latent;  // weight rows per expert

  if (warp == 0) {
    // ---------------- raw code producer ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int rs = 0, issued = 0;
      uint32_t rph = 0;
      bool ok = true;
      int4 g_next = x_group(a, blockIdx.x, nft, n_items);
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const int4 g_cur = g_next;
        g_next = x_group(a, it + gridDim.x, nft, n_items);
        XItem x;
        if (!x_item(a, g_cur, it, nft, &x)) continue;
        for (int kr = 0; kr < nkr; ++kr) {
          if (!mbar_wait(&raw_empty[rs], rph ^ 1, a.st, 61)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[rs], C::NMAT * kXTile);
#pragma unroll
          for (int m = 0; m < C::NMAT; ++m)
            tma_load_2d(s_raw + (rs * C::NMAT + m) * kXTile, &tm_q, kr * 128,
                        x.e * rows_pe + (MODE == 0 ? m * a.inter + x.ft * kXM : (x.ft * TPI + m) * kXM),
                        &raw_full[rs], pol);
          ++issued;
          if (++rs == C::RAW) {
            rs = 0;
            rph ^= 1;
          }
        }
      }
      for (int i = 0; i < C::RAW && i < issued; ++i) {  // the last copies land before exit
        if (--rs < 0) {
          rs = C::RAW - 1;
          rph ^= 1;
        }
        mbar_wait(&raw_full[rs], rph, a.st, 62);
      }
    }
  } else if (warp == 1) {
    // ---------------- activation producer ----------------
    const uint64_t pol = policy_evict_last();
    int bs = 0, issued = 0;
    uint32_t bph = 0;
    bool ok = true;
    int4 g_next = x_group(a, blockIdx.x, nft, n_items);
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const int4 g_cur = g_next;
      g_next = x_group(a, it + gridDim.x, nft, n_items);
      XItem x;
      if (!x_item(a, g_cur, it, nft, &x)) continue;
      const int nb = (x.n + 31) >> 5;
      for (int ks = 0; ks < nks; ++ks) {
        int good = 1;
        if (lane == 0) good = mbar_wait(&empty[bs], bph ^ 1, a.st, 63);
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[bs], nb * kXBBox);
        __syncwarp();
        if (lane < nb)
          tma_load_2d(s_b + bs * kXBStage + lane * kXBBox, &tm_act, ks * 64, x.p0 + lane * 32, &full[bs], pol);
        ++issued;
        if (++bs == C::ST) {
          bs = 0;
          bph ^= 1;
        }
      }
    }
    if (lane == 0)  // the last copies land before exit (the stages' empty commits follow them)
      for (int i = 0; i < C::ST && i < issued; ++i) {
        if (--bs < 0) {
          bs = C::ST - 1;
          bph ^= 1;
        }
        mbar_wait(&empty[bs], bph, a.st, 64);
      }
  } else if (warp == 2) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int as = 0, acc = 0;
      uint32_t aph = 0, cph = 0;
      bool ok = true;
      int4 g_next = x_group(a, blockIdx.x, nft, n_items);
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const int4 g_cur = g_next;
        g_next = x_group(a, it + gridDim.x, nft, n_items);
        XItem x;
        if (!x_item(a, g_cur, it, nft, &x)) continue;
        const uint32_t idesc = idesc_bf16_f32(kXM, (x.n + 15) & ~15);
        if (!mbar_wait(&acc_empty[acc], cph ^ 1, a.st, 65)) break;
        tc_fence_after();
        const uint32_t d = tmem;  // one accumulator pair per item (NACC = 1)
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait(&full[as], aph, a.st, 66)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b0 = smem_u32(s_b + as * kXBStage);
          const uint32_t a0 = tmem + kXACol + (uint32_t)(as * C::NMAT) * 32u;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int m = 0; m < C::NMAT; ++m)
              tc_mma_bf16_ts(d + m * kXAcc, a0 + m * 32u + kk * 8u, smem_desc_sw128(b0 + kk * 32), idesc,
                             (ks | kk) != 0);
          tc_commit(&empty[as]);
          if (++as == C::ST) {
            as = 0;
            aph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        if (++acc == C::NACC) {
          acc = 0;
          cph ^= 1;
        }
      }
      tc_commit(done);  // every MMA issued has completed before TMEM is released
      mbar_wait(done, 0, a.st, 68);
    }
  } else if (warp < 3 + kDqWarps) {
    // ---------------- dequantisation: codes -> bf16 A stages in TMEM ----------------
    // A warp may only touch the TMEM lanes of its quarter (warp % 4): warp w
    // handles rows 32 (w % 4) .. +31.  Two tiles per item (gate and up, or two
    // down tiles): warps 3-6 the first tile, 7-10 the second, both 32-blocks of
    // each 64-K step.
    const int dw = warp - 3, q = warp & 3;
    const int m = dw >> 2;
    const int rr = q * 32 + lane;
    const int sw = rr & 7;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    constexpr int NB = 2;  // 32-blocks per 64-K step
    int rs = 0, as = 0;
    uint32_t rph = 0, aph = 0;
    bool ok = true;
    int4 g_next = x_group(a, blockIdx.x, nft, n_items);
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const int4 g_cur = g_next;
      g_next = x_group(a, it + gridDim.x, nft, n_items);
      XItem x;
      if (!x_item(a, g_cur, it, nft, &x)) continue;
      const size_t grow = (size_t)x.e * rows_pe +
                          (MODE == 0 ? (size_t)m * a.inter + (size_t)x.ft * kXM : (size_t)(x.ft * TPI + m) * kXM) + rr;
      constexpr int kSB = FMT == 1 ? 16 : 32;  // elements per scale byte
      const uint8_t* srow = a.s + grow * (size_t)(K / kSB);
      // a stage's scale bytes: 8 E8M0 or 16 E4M3 (in .x, .y or all four words)
      auto load_sc = [&](int kr) -> uint4 {
        if constexpr (FMT == 1) {
          return __ldg(reinterpret_cast<const uint4*>(srow + kr * 16));
        } else {
          const uint2 v = __ldg(reinterpret_cast<const uint2*>(srow + kr * 8));
          return make_uint4(v.x, v.y, 0u, 0u);
        }
      };
      uint4 sc_next = load_sc(0);  // loaded one stage ahead
      for (int kr = 0; kr < nkr && ok; ++kr) {
        const uint4 sc16 = sc_next;
        const uint2 sc8 = make_uint2(sc16.x, sc16.y);
        if (kr + 1 < nkr) sc_next = load_sc(kr + 1);
        // all eight in the exponent-add range [2, 252]: bytewise (s - 2) <= 250
        const bool fast = (__vcmpleu4(__vsub4(sc8.x, 0x02020202u), 0xFAFAFAFAu) &
                           __vcmpleu4(__vsub4(sc8.y, 0x02020202u), 0xFAFAFAFAu)) == 0xFFFFFFFFu;
        if (!mbar_wait(&raw_full[rs], rph, a.st, 70)) {
          ok = false;
          break;
        }
        const uint8_t* rawt = s_raw + (rs * C::NMAT + m) * kXTile + rr * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t o[16 * NB];
#pragma unroll
          for (int bi = 0; bi < NB; ++bi) {
            const int b = bi;
            const int kb = 2 * j + b;  // 32-block within the raw stage
            const uint4 c = *reinterpret_cast<const uint4*>(rawt + ((kb ^ sw) << 4));
            if constexpr (FMT == 1) {
              // 16-blocks 2 kb (codes in c.x, c.y) and 2 kb + 1 (c.z, c.w)
              const uint32_t sword = (kb < 2) ? sc16.x : (kb < 4) ? sc16.y : (kb < 6) ? sc16.z : sc16.w;
              const uint32_t sh = 16 * (kb & 1);
              const DqTable t0 = dq_table_nv((sword >> sh) & 0xFFu), t1 = dq_table_nv((sword >> (sh + 8)) & 0xFFu);
              dq8(c.x, t0, o + 16 * bi);
              dq8(c.y, t0, o + 16 * bi + 4);
              dq8(c.z, t1, o + 16 * bi + 8);
              dq8(c.w, t1, o + 16 * bi + 12);
            } else {
              const uint32_t sword = kb < 4 ? sc8.x : sc8.y;
              const uint32_t sb = (sword >> (8 * (kb & 3))) & 0xFFu;
              dq_block(c, sb, o + 16 * bi, fast || (sb >= 2u && sb <= 252u));
            }
          }
          if (!mbar_wait(&empty[as], aph ^ 1, a.st, 71)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t acol = tmem + lane_base + kXACol + (uint32_t)(as * C::NMAT + m) * 32u;
          tmem_st32(acol, o);
          // the stage is complete once the store lands: arrive at once (deferring the
          // arrival past the next step's dequantisation made the MMAs wait longer)
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[as]);
          if (++as == C::ST) {
            as = 0;
            aph ^= 1;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rs]);
        if (++rs == C::RAW) {
          rs = 0;
          rph ^= 1;
        }
      }
    }
  } else {
    // ---------------- epilogue: TMEM -> h (gate/up) or y, ssq (down) ----------------
    const int q = warp & 3;                      // TMEM lane quarter this warp may read
    const int half = (warp - 3 - kDqWarps) >> 2;  // which alternate 32-column chunks
    int acc = 0;
    uint32_t cph = 0;
    int4 g_next = x_group(a, blockIdx.x, nft, n_items);
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const int4 g_cur = g_next;
      g_next = x_group(a, it + gridDim.x, nft, n_items);
      XItem x;
      if (!x_item(a, g_cur, it, nft, &x)) continue;
      if (!mbar_wait_sleep(&acc_full[acc], cph, a.st, 72, 256)) break;
      tc_fence_after();
      const float gsc = FMT == 1 ? __ldg(a.gs + x.e) : 1.0f;  // NVFP4 global scale of this expert matrix
      for (int m = 0; m < TPI; ++m) {
      const int f = (x.ft * TPI + m) * kXM + q * 32 + lane;  // output feature of this lane
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)m * kXAcc;
      for (int c0 = 32 * half; c0 < x.n; c0 += 64) {
        if (MODE == 0) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c0, g);
          tmem_ld32(tb + kXAcc + c0, u);
          tmem_ld_wait();
          // silu(g) * u with the fast exponential and the approximate reciprocal
          // (relative error ~1e-6, far below the bf16 rounding of h that follows;
          // the correctly rounded reciprocal cost the epilogue ~40% more time, and
          // the MMAs wait for the epilogue at every item)
          float hv[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float gv = __uint_as_float(g[i]), uv = __uint_as_float(u[i]);
            if (FMT == 1) {
              gv *= gsc;
              uv *= gsc;
            }
            float r;
            asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + __expf(-gv)));
            hv[i] = gv * r * uv;
          }
          // Lane l holds feature f (= f0 + l) of columns c0..c0+31.  Per block of 8
          // columns, an 8 x 8 transpose inside each group of 8 lanes (three
          // butterfly exchanges) leaves lane l with features f0 + 8(l/8) .. +7 of
          // column c0 + 8b + l%8: one 16-byte store instead of eight 2-byte ones.
          const int j = lane & 7;
          const int f0 = f - lane + 8 * (lane >> 3);
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = hv[8 * b + k];
#pragma unroll
            for (int sh = 4; sh >= 1; sh >>= 1) {
              const bool hi = (j & sh) != 0;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (k & sh) continue;
                const float recv = __shfl_xor_sync(0xffffffffu, hi ? v[k] : v[k | sh], sh);
                if (hi)
                  v[k] = recv;
                else
                  v[k | sh] = recv;
              }
            }
            const int col = c0 + 8 * b + j;
            if (col < x.n) {
              uint4 pk;
              pk.x = (uint32_t)f32_to_bf16_bits(v[0]) | ((uint32_t)f32_to_bf16_bits(v[1]) << 16);
              pk.y = (uint32_t)f32_to_bf16_bits(v[2]) | ((uint32_t)f32_to_bf16_bits(v[3]) << 16);
              pk.z = (uint32_t)f32_to_bf16_bits(v[4]) | ((uint32_t)f32_to_bf16_bits(v[5]) << 16);
              pk.w = (uint32_t)f32_to_bf16_bits(v[6]) | ((uint32_t)f32_to_bf16_bits(v[7]) << 16);
              *reinterpret_cast<uint4*>(a.h_out + (size_t)(x.p0 + col) * a.inter + f0) = pk;
            }
          }
        } else {
          uint32_t v[32];
          tmem_ld32(tb + c0, v);
          tmem_ld_wait();
          const int my_row = c0 + lane < x.n ? a.sorted_rows[x.p0 + c0 + lane] : 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int rid = __shfl_sync(0xffffffffu, my_row, i);
            if (FMT == 1) v[i] = __float_as_uint(__uint_as_float(v[i]) * gsc);
            if (c0 + i < x.n) a.y_out[(size_t)rid * a.latent + f] = __uint_as_float(v[i]);
          }
          // sum of squares over this warp's 32 features for each of the 32 columns:
          // halve the column set at every step, lane l ends with column l
          float s[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(v[i]) * __uint_as_float(v[i]);
#pragma unroll
          for (int w = 16; w >= 1; w >>= 1) {
            const bool upper = (lane & w) != 0;
#pragma unroll
            for (int i = 0; i < w; ++i) {
              const float send = upper ? s[i] : s[i + w];
              const float keep = upper ? s[i + w] : s[i];
              s[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
            }
          }
          if (c0 + lane < x.n)
            a.ssq_out[(size_t)my_row * (a.latent / 32) + ((x.ft * TPI + m) * kXM + q * 32) / 32] = s[0];
        }
      }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (++acc == C::NACC) {
        acc = 0;
        cph ^= 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int MODE, int FMT>
int launch_tc_expert(const TcExpertArgs& a, const uint16_t* act, cudaStream_t s, int num_sms) {
  const int K = a.K;
  if (K % 256 || a.inter % kXM || a.latent % (MODE == 2 ? 2 * kXM : kXM)) return LMOE_EUNSUPPORTED;
  constexpr int smem = xsmem_bytes<MODE>();
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMOE_ECUDA;
  if (!(attr_done.load() >> (dev & 63) & 1ull)) {
    if (cudaFuncSetAttribute(tc_expert_kernel<MODE, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return LMOE_ECUDA;
    attr_done.fetch_or(1ull << (dev & 63));
  }
  const int rows_pe = MODE == 0 ? 2 * a.inter : a.latent;
  CUtensorMap tq, ta;
  {
    const uint64_t dims[2] = {(uint64_t)K / 2, (uint64_t)a.n_experts * rows_pe};
    const uint64_t strides[1] = {(uint64_t)K / 2};
    const uint32_t box[2] = {128, kXM};
    if (get_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return LMOE_ECUDA;
  }
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)a.rows};
    const uint64_t strides[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {64, 32};
    if (get_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, act, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return LMOE_ECUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kXThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_expert_kernel<MODE, FMT>, a, tq, ta) == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

int launch_tc_gateup(const TcExpertArgs& a, const uint16_t* x_sorted, cudaStream_t s, int num_sms) {
  if (a.gs) return launch_tc_expert<0, 1>(a, x_sorted, s, num_sms);
  return launch_tc_expert<0, 0>(a, x_sorted, s, num_sms);
}

int launch_tc_down(const TcExpertArgs& a, const uint16_t* h, cudaStream_t s, int num_sms) {
  // two output tiles per item halve the activation traffic per MMA
  // two 128-row output tiles per item: every supported latent width is a multiple of 256
  if (a.latent % (2 * kXM)) return LMOE_EUNSUPPORTED;
  if (a.gs) return launch_tc_expert<2, 1>(a, h, s, num_sms);
  return launch_tc_expert<2, 0>(a, h, s, num_sms);
}

// x_sorted[p] = x_lat[sorted_rows[p] / k]: one warp per sorted row, 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x_lat,
                                                          const int32_t* __restrict__ sorted_rows, int R, int k,
                                                          int L, uint16_t* __restrict__ x_sorted) {
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (p >= R) return;
  const int t = sorted_rows[p] / k;
  const uint4* src = reinterpret_cast<const uint4*>(x_lat + (size_t)t * L);
  uint4* dst = reinterpret_cast<uint4*>(x_sorted + (size_t)p * L);
  for (int i = lane; i < L / 8; i += 32) dst[i] = __ldg(src + i);
}

// Device self-check of the expert dequantisation: block b of 32 codes
// (codes[16 b .. 16 b + 15]) with scale byte scales[b] -> out[32 b .. 32 b + 31].
__global__ void dequant_selftest_kernel(const uint8_t* codes, const uint8_t* scales, int nblocks, uint16_t* out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  const uint4 c = *reinterpret_cast<const uint4*>(codes + 16 * (size_t)b);
  uint32_t o[16];
  dq_block(c, scales[b], o, scales[b] >= 2 && scales[b] <= 252);
  uint4* dst = reinterpret_cast<uint4*>(out + 32 * (size_t)b);
#pragma unroll
  for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}

}  // namespace lmoe
