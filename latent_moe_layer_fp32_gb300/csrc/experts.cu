// Routed experts, MXFP4 W4A16, decode-regime streaming kernels.
//
// "Muse Spark Open on Gaudi 2": experts run W4A16 ("What was built"), each
// (token, route) pair is its own row and the cost is per touched expert slice
// ("The latent MoE: A' with a per-expert norm"); the checkpoint's packed E2M1
// nibbles and E8M0 scales are read directly ("Why it needed a port").  The
// page's stock op unpacked every touched slice to bf16 in memory ("What it
// taught about Gaudi"); here nothing is unpacked in memory.
//
// Work item = (group of <= G rows of one expert, tile of 32 weight rows =
// two m16 tiles).  gate/up: 16 gate rows + the matching 16 up rows (an m16
// tile pairs 8 gate rows with their 8 up rows, so SwiGLU is local to a lane);
// down: 32 consecutive output rows.  Each item streams its rows once (all of
// K) for every row of its group.  A CTA takes a contiguous range of items,
// so consecutive items mostly share a group.
//
// CTA = Q consumer warps + 1 producer warp + 1 epilogue warp.
//  - producer: per K chunk, two TMA tensor copies of the codes (16 rows x
//    kc/2 bytes each, a 3-D view {128 B, rows, K/256} with 128-byte swizzle,
//    so each copy is one 16 KB request and ldmatrix reads it without bank
//    conflicts) and two of the E8M0 scales, into a ring of D slots.  When
//    the group changes it loads the group's activation rows (bf16, whole K)
//    into the activation panel, once the consumers released the old one.
//  - consumers: convert a fresh panel once (bf16 -> f16 times a per-row power
//    of two that puts the row's largest magnitude in [2^14, 2^15): exact for
//    every element down to 2^-17 of that scale; undone in the epilogue), then
//    share every slot, warp j taking the chunk's 128-byte planes j, j+Q, ...
//    They hand their fp32 partials to the epilogue warp through a
//    double-buffered exchange and go straight on to the next item.
//  - epilogue: adds the Q partials in warp order (fixed summation order) and
//    finishes the item (SwiGLU -> h, or y plus its sums of squares).
// Every wait is an mbarrier wait bounded in time.
//
// Consumer per 32-element scale block: ldmatrix.x4 hands each lane 4 code
// bytes of two rows; cvt.rn.f16x2.e2m1x2 turns each byte into two exact f16
// values; two mma.sync m16n8k16 (f16 in, fp32 accumulate) cover the block's
// 32 K positions in a fixed permutation that the activation fragment follows;
// the fresh block result is scaled by the block's E8M0 value (expanded once
// per plane into a per-warp fp32 table) and added to the fp32 accumulator.
//
// NVFP4 weights (FMT_NV): one E4M3 scale per 16 elements and an fp32 global
// scale per expert matrix.  A lane's 8 codes of a 32-element block lie in one
// 16-element half, and E2M1 x E4M3 is exact in f16 (at most 6 significant
// bits, magnitudes 2^-10 .. 2688), so each f16x2 pair of codes is multiplied
// by its block scale before the MMA and the MMAs accumulate the whole item in
// fp32; the epilogue applies the global scale.
#include "common.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace lmoe {

enum { MODE_GATEUP = 0, MODE_DOWN = 1 };
enum { FMT_MX = 0, FMT_NV = 1 };  // MXFP4 (E8M0 per 32) or NVFP4 (E4M3 per 16 + global)

constexpr int kRows = 32;  // weight rows per item: two m16 tiles
constexpr int kKC = 2048;  // K elements per chunk when K > 2048 (else the whole K): 16 KB code boxes

// Group header the producer writes next to an activation panel.
struct PanelHdr {
  int p0, ntok, expert, pad1;
  int rows[8];  // per token: sorted_rows[p0 + j] (the original route row id)
};

// Item header a consumer passes to the epilogue warp with the partials.
struct ItemHdr {
  int p0, ntok, tile;
  float gscale;  // NVFP4: the expert matrix's global scale
  int aexp[8];  // per token of the group: power of two mapping its activation row into f16 range
  int rows[8];
};

// One ring slot: codes and scales of a K chunk of one item.
template <int FMT>
struct Layout {
  static constexpr int kSB = (FMT == FMT_NV) ? 16 : 32;  // elements per scale byte
  static constexpr int kBox = 16 * (kKC / 2);  // one code box: 16 rows x kc/2 bytes (16 KB)
  static constexpr int kCodes = 2 * kBox;      // box A (rows 0-15 of the item), box B (rows 16-31)
  static constexpr int kScales = kRows * (kKC / kSB);
  static constexpr int kSlot = (kCodes + kScales + 1023) / 1024 * 1024;  // 1 KB aligned (swizzle atom)
  static constexpr int kTable = 256;  // 4-byte words of a warp's scale table (fp32 E8M0 / f16 E4M3 values)
};

constexpr int kMaxSlots = 8;
constexpr int kMaxK = 8192;  // activation panel: up to G rows of this many elements

// Expand the E8M0 bytes of one 128-byte plane (8 blocks; scale region
// [32 rows][nb], blocks p*8 .. p*8+7) into fp32 2^(s-127) in the warp's table
// [block][mtile][g][lo,hi].  Fast path s << 23 is exact for 1 <= s <= 254; a
// plane holding 0 or 255 takes the exact per-value path.
template <int MODE>
__device__ __forceinline__ void expand_plane_scales(const uint8_t* sc, int nb, int p, float* table, int lane) {
  const int r = lane;  // region row: rows 0-15 from box A, 16-31 from box B
  const int box = r >> 4, rb = r & 15;
  // gate/up: box A = gate (lo), box B = up (hi); m-tile = rb / 8.
  // down: box = m-tile; lo/hi = rb / 8.
  const int mt = (MODE == MODE_GATEUP) ? (rb >> 3) : box;
  const int hi = (MODE == MODE_GATEUP) ? box : (rb >> 3);
  const int g = r & 7;
  const uint32_t* src = reinterpret_cast<const uint32_t*>(sc + r * nb + p * 8);
  const uint32_t w0 = src[0], w1 = src[1];
  bool special = ((__vcmpeq4(w0, 0u) | __vcmpeq4(w0, 0xffffffffu) | __vcmpeq4(w1, 0u) |
                   __vcmpeq4(w1, 0xffffffffu)) != 0u);
  special = __any_sync(0xffffffffu, special);
  float* dst = table + (mt * 8 + g) * 2 + hi;
  if (!special) {
    dst[0 * 32] = __uint_as_float((w0 << 23) & 0x7f800000u);
    dst[1 * 32] = __uint_as_float((w0 << 15) & 0x7f800000u);
    dst[2 * 32] = __uint_as_float((w0 << 7) & 0x7f800000u);
    dst[3 * 32] = __uint_as_float((w0 >> 1) & 0x7f800000u);
    dst[4 * 32] = __uint_as_float((w1 << 23) & 0x7f800000u);
    dst[5 * 32] = __uint_as_float((w1 << 15) & 0x7f800000u);
    dst[6 * 32] = __uint_as_float((w1 << 7) & 0x7f800000u);
    dst[7 * 32] = __uint_as_float((w1 >> 1) & 0x7f800000u);
  } else {
    for (int j = 0; j < 8; ++j) dst[j * 32] = e8m0_to_f32(sc[r * nb + p * 8 + j]);
  }
}

// The 8 blocks of one 128-byte plane p of a chunk.  The four 16-byte chunk
// offsets a lane reads are fixed by the swizzle (chunk ^ (row & 7)), so every
// address is a per-lane base plus an immediate.  `table` holds this plane's
// scales only.
template <int NV>
__device__ __forceinline__ void plane_blocks(uint32_t sbase, uint32_t act_addr, const float* table,
                                             const uint32_t (&box_off)[2], const int (&row_in_box)[2], int lm, int g,
                                             float (&acc)[2][2][NV], int p) {
  const float2* tab2 = reinterpret_cast<const float2*>(table) + g;
  const int rr = row_in_box[0] & 7;  // both m-tiles' rows share row & 7
  const uint32_t pb0 = sbase + box_off[0] + row_in_box[0] * 128 + p * 2048;  // plane stride: 16 rows x 128 B
  const uint32_t pb1 = sbase + box_off[1] + row_in_box[1] * 128 + p * 2048;
  const uint32_t pact = act_addr + p * 512;  // 8 blocks x 64 B
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t coff = static_cast<uint32_t>(((2 * i + (lm >> 1)) ^ rr) << 4);
    uint32_t w[2][4];
    ldmatrix_x4(w[0][0], w[0][1], w[0][2], w[0][3], pb0 + coff);
    ldmatrix_x4(w[1][0], w[1][1], w[1][2], w[1][3], pb1 + coff);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int blk = 2 * i + half;  // block within the plane
      uint32_t b0, b1, b2, b3;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                   : "r"(pact + blk * 64));
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        uint32_t l0, l1, l2, l3, h0, h1, h2, h3;
        e2m1x8_to_f16x8(w[m][2 * half], l0, l1, l2, l3);
        e2m1x8_to_f16x8(w[m][2 * half + 1], h0, h1, h2, h3);
        float dacc[4];
        mma_f16_zero(dacc, l0, h0, l1, h1, b0, b1);
        mma_f16(dacc, l2, h2, l3, h3, b2, b3);
        const float2 sc = tab2[(blk * 2 + m) * 8];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          acc[m][0][v] = fmaf(dacc[v], sc.x, acc[m][0][v]);
          acc[m][1][v] = fmaf(dacc[2 + v], sc.y, acc[m][1][v]);
        }
      }
    }
  }
}

// NVFP4: the 16 E4M3 bytes of one 128-byte plane p (16 blocks of 16, scale
// region [32 rows][nsb]) as f16 values in the warp's table [block j][mtile][g][lo,hi]
// (so one 32-bit word holds a row pair's two scales).  E4M3 -> f16 is exact
// (cvt.rn.f16x2.e4m3x2).
template <int MODE>
__device__ __forceinline__ void expand_plane_scales_nv(const uint8_t* sc, int nsb, int p, uint16_t* table, int lane) {
  const int r = lane;
  const int box = r >> 4, rb = r & 15;
  const int mt = (MODE == MODE_GATEUP) ? (rb >> 3) : box;
  const int hi = (MODE == MODE_GATEUP) ? box : (rb >> 3);
  const int g = r & 7;
  const uint4 v = *reinterpret_cast<const uint4*>(sc + r * nsb + p * 16);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint16_t* dst = table + (mt * 8 + g) * 2 + hi;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
      uint32_t f2;  // f16 pair of blocks 4i + 2hw (low half) and 4i + 2hw + 1 (high half)
      const uint16_t b2 = (uint16_t)(w[i] >> (16 * hw));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f2) : "h"(b2));
      const int j = 4 * i + 2 * hw;
      dst[j * 32] = (uint16_t)(f2 & 0xffffu);
      dst[(j + 1) * 32] = (uint16_t)(f2 >> 16);
    }
  }
}

// NVFP4: the 8 blocks of 32 of plane p.  The lane's codes of a block lie in its
// 16-element half q / 2; their f16 values times that half's scale are exact, so
// the MMAs accumulate straight into acc4 (two chains per m-tile, by block parity).
template <int NV>
__device__ __forceinline__ void plane_blocks_nv(uint32_t sbase, uint32_t act_addr, const uint16_t* table,
                                                const uint32_t (&box_off)[2], const int (&row_in_box)[2], int lm,
                                                int g, int q, float (&acc4)[2][2][4], int p) {
  const uint32_t* tab1 = reinterpret_cast<const uint32_t*>(table) + g;  // (lo, hi) f16 pair per word
  const int rr = row_in_box[0] & 7;
  const uint32_t pb0 = sbase + box_off[0] + row_in_box[0] * 128 + p * 2048;
  const uint32_t pb1 = sbase + box_off[1] + row_in_box[1] * 128 + p * 2048;
  const uint32_t pact = act_addr + p * 512;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t coff = static_cast<uint32_t>(((2 * i + (lm >> 1)) ^ rr) << 4);
    uint32_t w[2][4];
    ldmatrix_x4(w[0][0], w[0][1], w[0][2], w[0][3], pb0 + coff);
    ldmatrix_x4(w[1][0], w[1][1], w[1][2], w[1][3], pb1 + coff);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int blk = 2 * i + half;
      uint32_t b0, b1, b2, b3;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                   : "r"(pact + blk * 64));
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        uint32_t l[4], h[4];
        e2m1x8_to_f16x8(w[m][2 * half], l[0], l[1], l[2], l[3]);
        e2m1x8_to_f16x8(w[m][2 * half + 1], h[0], h[1], h[2], h[3]);
        const uint32_t sp = tab1[((2 * blk + (q >> 1)) * 2 + m) * 8];
        const uint32_t slo = __byte_perm(sp, sp, 0x1010), shi = __byte_perm(sp, sp, 0x3232);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(l[t]) : "r"(slo));
          asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h[t]) : "r"(shi));
        }
        mma_f16(acc4[half][m], l[0], h[0], l[1], h[1], b0, b1);
        mma_f16(acc4[half][m], l[2], h[2], l[3], h[3], b2, b3);
      }
    }
  }
}

// Shared-memory plan of one CTA (bytes), shared by the kernel and the launch.
// NP activation panels: two when one group's rows are small (G = 1), so the
// next group's rows load while the current group is still being consumed.
template <int G, int Q, int FMT>
struct Smem {
  using Lay = Layout<FMT>;
  static constexpr int NP = (G == 1) ? 2 : 1;
  static constexpr int NV = (G == 1) ? 1 : 2;        // token columns per lane that can hold a valid token
  static constexpr int kPart = 2 * 2 * NV * 32;      // floats per warp partial: [mtile][lo/hi][v][lane]
  static __host__ __device__ int panel_row(int K) { return K * 2 + 64; }  // padded: conflict-free 16-byte loads
  static __host__ __device__ int fixed(int K) {
    return NP * G * panel_row(K) + Q * Lay::kTable * 4 + 2 * Q * kPart * 4 + Q * G * 4 + 2 * (int)sizeof(ItemHdr) +
           NP * (int)sizeof(PanelHdr) + (2 * kMaxSlots + 2 * NP + 6) * 8;
  }
  static __host__ __device__ int bytes(int K, int D) { return D * Lay::kSlot + fixed(K) + 1024; }
};

// Down at decode sizes: the post-expert norm and the fp32 weighted sum in the
// same launch ("Muse Spark Open on Gaudi 2", "The latent MoE: A' with a
// per-expert norm").  Once every CTA has counted itself done (its y rows and
// their per-tile sums of squares written; a device-wide counter, bounded
// wait), CTA b forms z for the 32-column slices b, b + gridDim, ... of the
// latent width, one token per calling warp:
//   rinv[r] = 1/sqrt(sum of row r's tile sums (tile order) / L + eps),
//   z[t][l] = sum over j in order of w[t][j] * ((y[t*k+j][l] * rinv) * g[e][l]),
// the same arithmetic in the same order as combine_kernel.  The routes'
// experts, weights and gains (ready since the routing) are read before the
// wait; after it, one round of loads brings the rows' tile sums and y.
// `wid` numbers the calling warps 0..NW-1; `scratch` is shared memory no
// other warp still uses.
template <int NW>
__device__ void down_z_step(const ExpertArgs& a, float* scratch, int wid, int lane) {
  const int L = a.latent, k = a.top_k, tiles = L / kRows, nsl = L / 32;
  if ((int)blockIdx.x >= nsl) return;  // no slice here (CTA-uniform)
  int* s_ok = reinterpret_cast<int*>(scratch);
  // the first token's routes and its gains in the first slice, before the wait
  int er[8];
  float wr[8], g0[8];
  auto routes = [&](int t) {
    int e = 0;
    float wv = 0.f;
    if (lane < k) {
      e = a.topk_idx[t * k + lane];
      if (e < 0 || e >= a.n_experts) {
        set_error(a.st, LMOE_EDEVICE_CHECK, 103);
        e = 0;
      }
      wv = a.topk_w[t * k + lane];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      er[j] = __shfl_sync(0xffffffffu, e, j);
      wr[j] = __shfl_sync(0xffffffffu, wv, j);
    }
  };
  if (wid < a.T) {
    routes(wid);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      g0[j] = j < k ? bf16_bits_to_f32(a.norm_g[(size_t)er[j] * L + blockIdx.x * 32 + lane]) : 0.f;
  }
  named_bar(1, NW * 32);  // every calling warp is past its last use of the scratch
  if (wid == 0 && lane == 0) *s_ok = counter_wait(a.zctr, gridDim.x, a.st, 60) ? 1 : 0;
  named_bar(1, NW * 32);
  if (!*s_ok) return;
  for (int t = wid; t < a.T; t += NW) {
    if (t != wid) routes(t);
    // every tile sum of the token's k rows and their y in the first slice, then the sums
    float v[8][8], yv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = t * k + j;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[j][u] = (j < k && lane + 32 * u < tiles) ? __ldcg(a.ssq_out + (size_t)r * tiles + lane + 32 * u) : 0.f;
      yv[j] = j < k ? __ldcg(a.y_out + (size_t)r * L + blockIdx.x * 32 + lane) : 0.f;
    }
    float rinv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float sq = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (lane + 32 * u < tiles) sq += v[j][u];
      sq = warp_sum(sq);
      rinv[j] = 1.0f / sqrtf(sq / (float)L + a.eps);
    }
    for (int sl = blockIdx.x; sl < nsl; sl += gridDim.x) {
      const int l = sl * 32 + lane;
      float gv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (sl == (int)blockIdx.x && t == wid) {
          gv[j] = g0[j];
        } else {
          gv[j] = j < k ? bf16_bits_to_f32(a.norm_g[(size_t)er[j] * L + l]) : 0.f;
          if (j < k && sl != (int)blockIdx.x) yv[j] = __ldcg(a.y_out + ((size_t)t * k + j) * L + l);
        }
      }
      float z = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= k) break;
        const float yh = __fmul_rn(__fmul_rn(yv[j], rinv[j]), gv[j]);
        z = __fadd_rn(z, __fmul_rn(wr[j], yh));
      }
      a.zb[(size_t)t * L + l] = f32_to_bf16_bits(z);
    }
  }
}

template <int MODE, int G, int Q, int FMT>
__global__ void __launch_bounds__(32 * (Q + 2), 1)
    expert_kernel(const ExpertArgs a, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_s,
                  int D) {
  using Lay = Layout<FMT>;
  using SM = Smem<G, Q, FMT>;
  constexpr int NP = SM::NP;
  constexpr int NV = SM::NV;
  constexpr int kPart = SM::kPart;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1 KB alignment for the swizzled boxes
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int K = a.K, kc = a.kc, nch = K / kc, nb = kc / 32, cbk = kc / 256;  // cbk: 128-byte planes per chunk
  const int nsb = kc / Lay::kSB;  // scale bytes per row and chunk
  const int prow = SM::panel_row(K);
  uint8_t* panels = smem + D * Lay::kSlot;                                 // [NP][G][prow]: activation rows
  float* tables = reinterpret_cast<float*>(panels + NP * G * prow);       // [Q][kTable]: per-warp scale table
  float* red = tables + Q * Lay::kTable;                                  // [2][Q][kPart]: partials
  float* smax = red + 2 * Q * kPart;                                      // [Q][G]: per-warp row maxima
  ItemHdr* ihdr = reinterpret_cast<ItemHdr*>(smax + Q * G);               // [2]
  PanelHdr* phdr = reinterpret_cast<PanelHdr*>(ihdr + 2);                 // [NP]
  uint64_t* full = reinterpret_cast<uint64_t*>(phdr + NP);                // [D] slot loaded (1 + tx)
  uint64_t* empty = full + kMaxSlots;                                     // [D] slot released (Q)
  uint64_t* pfull = empty + kMaxSlots;                                    // [NP] panel loaded (1 + tx)
  uint64_t* pempty = pfull + NP;                                          // [NP] panel released (Q)
  uint64_t* pmaxed = pempty + NP;                                         // row maxima written (Q)
  uint64_t* pready = pmaxed + 1;                                          // panel converted (Q)
  uint64_t* rfull = pready + 1;                                           // [2] partials written (Q)
  uint64_t* rempty = rfull + 2;                                           // [2] partials taken (1)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Ks = K / Lay::kSB;  // scale bytes per weight row
  const int tiles = (MODE == MODE_GATEUP) ? a.inter / 16 : a.latent / kRows;
  const int rows_per_expert = (MODE == MODE_GATEUP) ? 2 * a.inter : a.latent;

  if (threadIdx.x == 0) {
    for (int i = 0; i < D; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], Q);
    }
    for (int i = 0; i < NP; ++i) {
      mbar_init(&pfull[i], 1);
      mbar_init(&pempty[i], Q);
    }
    mbar_init(pmaxed, Q);
    mbar_init(pready, Q);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&rfull[i], Q);
      mbar_init(&rempty[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // Programmatic dependent launch: the routing table and the weights come from
  // kernels that completed before this grid was launched (the preceding kernel
  // waits for its own predecessor before it lets this one start), so the
  // producer streams its first slots of weights before waiting; the activation
  // rows (the preceding kernel's output) are read only after the wait.
  if (warp != Q || !a.early) {
    pdl_wait();
    pdl_trigger();
  }

  // The producer's routing reads in one round trip with the group count: group
  // entries 0..63 and row ids 0..127 read ahead (as far as allocated); a CTA
  // whose groups lie beyond them reads those from memory.
  int4 sg0 = make_int4(0, 0, 0, 0), sg1 = make_int4(0, 0, 0, 0);
  int sr[4] = {0, 0, 0, 0};
  if (warp == Q) {
    if (lane < a.groups_cap) sg0 = a.groups[lane];
    if (lane + 32 < a.groups_cap) sg1 = a.groups[lane + 32];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (lane + 32 * i < a.rows) sr[i] = a.sorted_rows[lane + 32 * i];
  }
  const int n_items = *a.n_groups * tiles;
  const int it0 = (int)((long long)n_items * blockIdx.x / gridDim.x);
  const int it1 = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x);
  const int nloc = it1 - it0;

  if (warp == Q) {
    // ------------------------------ producer ------------------------------
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_s)) : "memory");
    }
    const int4* groups = a.groups;
    auto entry = [sg0, sg1, groups](int grp) -> int4 {  // grp is warp-uniform
      if (grp < 64) {
        const int4 v = grp < 32 ? sg0 : sg1;
        const int src = grp & 31;
        return make_int4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                         __shfl_sync(0xffffffffu, v.z, src), 0);
      }
      return groups[grp];
    };
    int seq = 0, pseq = 0, cur = -1;
    bool ok = true;
    // codes and scales of chunk c of local item j (expert e) into the next ring
    // slot; lane 0 waits for the slot and issues all four copies
    auto issue = [&](int j, int c, int e) -> bool {
      const int tile = (it0 + j) % tiles;
      // first rows of box A and box B
      int rowA, rowB;
      if (MODE == MODE_GATEUP) {
        rowA = e * rows_per_expert + tile * 16;
        rowB = rowA + a.inter;
      } else {
        rowA = e * rows_per_expert + tile * kRows;
        rowB = rowA + 16;
      }
      const int d = seq % D;
      const uint32_t par = ((seq / D) & 1) ^ 1;
      ++seq;
      int good = 1;
      if (lane == 0) {
        good = seq <= D || mbar_wait(&empty[d], par, a.st, 1);  // the first D slots start free
        if (good) {
          uint8_t* slot = smem + d * Lay::kSlot;
          uint64_t* bar = &full[d];
          mbar_arrive_expect_tx(bar, kRows * (kc / 2) + kRows * nsb);
          tma_load_3d(slot, &tm_q, 0, rowA, c * cbk, bar, pol);
          tma_load_3d(slot + 16 * (kc / 2), &tm_q, 0, rowB, c * cbk, bar, pol);
          uint8_t* sdst = slot + Lay::kCodes;
          if (nch > 1) {
            tma_load_2d(sdst, &tm_s, c * nsb, rowA, bar, pol);
            tma_load_2d(sdst + 16 * nsb, &tm_s, c * nsb, rowB, bar, pol);
          } else {  // one chunk: the 16 rows' scales are contiguous
            bulk_g2s(sdst, a.s + (size_t)rowA * Ks, 16 * Ks, bar);
            bulk_g2s(sdst + 16 * nsb, a.s + (size_t)rowB * Ks, 16 * Ks, bar);
          }
        }
      }
      return __shfl_sync(0xffffffffu, good, 0) != 0;
    };
    // two of the ring's free slots before waiting (the activation panel, issued
    // right after the wait, gates the first MMAs; the rest of the ring follows it)
    int issued = 0;
    const int total = nloc * nch;
    while (a.early && ok && issued < total && issued < 2) {
      const int j = issued / nch;
      ok = issue(j, issued % nch, entry((it0 + j) / tiles).x);
      ++issued;
    }
    if (a.early) {
      pdl_wait();
      pdl_trigger();
    }
    for (int j = 0; j < nloc && ok; ++j) {
      const int it = it0 + j, grp = it / tiles;
      const int e_item = entry(grp).x;
      for (int c = 0; c < nch && ok; ++c) {
        if (j * nch + c >= issued) {
          ok = issue(j, c, e_item);
          ++issued;
          if (!ok) break;
        }
        if (c == 0 && grp != cur) {
          // New group: its activation rows go to the next panel once every
          // consumer released what that panel held.  Issued after this item's
          // first chunk, so the ring keeps streaming weights meanwhile; the
          // older groups' chunks are all issued, so the wait cannot close a cycle.
          cur = grp;
          const int4 g4 = entry(grp);
          const int p0 = g4.y, ntok = g4.z;
          const int pb = pseq % NP;
          int pg = 1;
          if (lane == 0) pg = mbar_wait(&pempty[pb], ((pseq / NP) & 1) ^ 1, a.st, 4);
          if (!__shfl_sync(0xffffffffu, pg, 0)) {
            ok = false;
            break;
          }
          int my_row = 0;
          if (p0 + ntok <= 128) {  // from the rows read ahead
            const int idx = (p0 + lane) & 127;
            int v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = __shfl_sync(0xffffffffu, sr[i], idx & 31);
            my_row = v[0];
#pragma unroll
            for (int i = 1; i < 4; ++i)
              if (idx >> 5 == i) my_row = v[i];
          } else if (lane < ntok) {
            my_row = a.sorted_rows[p0 + lane];
          }
          PanelHdr* h = phdr + pb;
          if (lane == 0) {
            h->p0 = p0;
            h->ntok = ntok;
            h->expert = g4.x;
          }
          if (lane < G) h->rows[lane] = my_row;
          __syncwarp();
          if (lane == 0) mbar_arrive_expect_tx(&pfull[pb], (uint32_t)ntok * K * 2);
          __syncwarp();
          if (lane < ntok) {
            const int arow = (MODE == MODE_GATEUP) ? my_row / a.top_k : p0 + lane;
            const uint16_t* src = a.act + (size_t)arow * K;
            uint8_t* dst = panels + (pb * G + lane) * prow;
            for (int k0 = 0; k0 < K; k0 += 8192)  // pieces of at most 16 KB
              bulk_g2s(dst + k0 * 2, src + k0, (uint32_t)min(8192, K - k0) * 2, &pfull[pb]);
          }
          ++pseq;
          __syncwarp();
        }
      }
    }
    // drain: no copy may still be in flight when this warp leaves
    if (lane == 0) {
      for (int s = max(0, seq - D); s < seq; ++s) mbar_wait(&full[s % D], (s / D) & 1, a.st, 2);
      for (int s = max(0, pseq - NP); s < pseq; ++s) mbar_wait(&pfull[s % NP], (s / NP) & 1, a.st, 5);
    }
    return;
  }

  if (warp == Q + 1) {
    // ------------------------------ epilogue ------------------------------
    const int g = lane >> 2, q = lane & 3;
    for (int j = 0; j < nloc; ++j) {
      const int pb = j & 1;
      if (!mbar_wait(&rfull[pb], (j >> 1) & 1, a.st, 6)) break;
      const ItemHdr* h = ihdr + pb;
      const int p0 = h->p0, ntok = h->ntok, tile = h->tile;
      const float gsc = h->gscale;
      int aexp[G], arow_id[G];
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        aexp[jj] = h->aexp[jj];
        arow_id[jj] = h->rows[jj];
      }
      const float* rb = red + pb * Q * kPart;
      float acc[2][2][NV];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            const int o = ((m * 2 + hh) * NV + v) * 32 + lane;
            float t = rb[o];
#pragma unroll
            for (int w = 1; w < Q; ++w) t += rb[w * kPart + o];
            acc[m][hh][v] = t;
          }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[pb]);
      // gate/up m-tile m holds features tile*16 + m*8 + g; down m-tile m holds
      // output rows tile*32 + m*16 + g (+8 for the hi half)
      float ssq[NV];
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int tok = 2 * q + v;
        ssq[v] = 0.f;
        int e_tok = 0, r_tok = 0;
#pragma unroll
        for (int jj = 0; jj < G; ++jj)
          if (jj == tok) {
            e_tok = aexp[jj];
            r_tok = arow_id[jj];
          }
        if (tok < ntok) {
          const int p = p0 + tok;
          float inv = ldexpf(1.0f, -e_tok);
          if (FMT == FMT_NV) inv *= gsc;  // a power of two times the global scale: one rounding
          if (MODE == MODE_GATEUP) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const float gv = acc[m][0][v] * inv, uv = acc[m][1][v] * inv;
              a.h_out[(size_t)p * a.inter + tile * 16 + m * 8 + g] = f32_to_bf16_bits(gv / (1.0f + expf(-gv)) * uv);
            }
          } else {
            float* yr = a.y_out + (size_t)r_tok * a.latent + tile * kRows;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const float y0 = acc[m][0][v] * inv, y1 = acc[m][1][v] * inv;
              yr[m * 16 + g] = y0;
              yr[m * 16 + g + 8] = y1;
              ssq[v] = fmaf(y0, y0, fmaf(y1, y1, ssq[v]));
            }
          }
        }
      }
      if (MODE == MODE_DOWN && a.ssq_out) {
        // sum of squares of the tile's 32 rows per token (fixed tree over g)
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          float sv = ssq[v];
          sv += __shfl_xor_sync(0xffffffffu, sv, 4);
          sv += __shfl_xor_sync(0xffffffffu, sv, 8);
          sv += __shfl_xor_sync(0xffffffffu, sv, 16);
          const int tok = 2 * q + v;
          int r_tok = 0;
#pragma unroll
          for (int jj = 0; jj < G; ++jj)
            if (jj == tok) r_tok = arow_id[jj];
          if (g == 0 && tok < ntok) a.ssq_out[(size_t)r_tok * (a.latent / kRows) + tile] = sv;
        }
      }
    }
    if (MODE == MODE_DOWN && a.zb) {
      // this CTA's y rows and sums of squares are written: count the CTA (release)
      __threadfence();
      __syncwarp();
      if (lane == 0) counter_add_release(a.zctr, 1);
      down_z_step<Q + 1>(a, red, Q, lane);
    }
    return;
  }

  // -------------------------------- consumer --------------------------------
  const int g = lane >> 2, q = lane & 3;
  // ldmatrix.x4 for m-tile m and blocks (b, b+1): matrices (lo rows, b) (hi rows, b) (lo rows, b+1) (hi rows, b+1)
  const int lm = lane >> 3, rr = lane & 7;
  float* table = tables + warp * Lay::kTable;
  // per m-tile: byte offset of this lane's ldmatrix box and its row in the box
  uint32_t box_off[2];
  int row_in_box[2];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    int box, row;
    if (MODE == MODE_GATEUP) {
      box = lm & 1;  // gate box (lo) / up box (hi)
      row = m * 8 + rr;
    } else {
      box = m;
      row = (lm & 1) * 8 + rr;
    }
    box_off[m] = box * 16 * (kc / 2);
    row_in_box[m] = row;
  }
  const int nplanes = nb / 8;
  const int units = K / 8;  // 16-byte units per activation row
  int seq = 0, pseq = 0, cur = -1;
  int p0 = 0, ntok = 0;
  float gscale = 1.f;  // NVFP4: the current group's expert matrix global scale
  uint32_t act_row = 0;  // this lane's activation row (token g) in the current panel
  int aexp[G], arow_id[G];
#pragma unroll
  for (int jj = 0; jj < G; ++jj) aexp[jj] = arow_id[jj] = 0;
  bool alive = true;
  for (int j = 0; j < nloc && alive; ++j) {
    const int it = it0 + j, grp = it / tiles, tile = it % tiles;
    if (grp != cur) {
      // a fresh panel: each row's largest magnitude sets its power of two, then
      // the rows are converted in place (bf16 -> f16 * 2^e), all consumer warps
      cur = grp;
      const int pb = pseq % NP;
      if (!mbar_wait(&pfull[pb], (pseq / NP) & 1, a.st, 7)) break;
      const PanelHdr* h = phdr + pb;
      uint8_t* panel = panels + pb * G * prow;
      p0 = h->p0;
      ntok = h->ntok;
      if constexpr (FMT == FMT_NV) gscale = a.gs[h->expert];
#pragma unroll
      for (int jj = 0; jj < G; ++jj) arow_id[jj] = h->rows[jj];
      for (int r = 0; r < ntok; ++r) {
        float m = 0.f;
        for (int u = warp * 32 + lane; u < units; u += Q * 32) {
          const uint4 v = *reinterpret_cast<const uint4*>(panel + r * prow + u * 16);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int t = 0; t < 4; ++t)
            m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(w4[t] & 0xffffu)), fabsf(bf16_bits_to_f32(w4[t] >> 16))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) smax[warp * G + r] = m;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(pmaxed);
      if (!mbar_wait(pmaxed, pseq & 1, a.st, 10)) break;
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        aexp[jj] = 0;
        if (jj < ntok) {
          float m = smax[jj];
#pragma unroll
          for (int w = 1; w < Q; ++w) m = fmaxf(m, smax[w * G + jj]);
          aexp[jj] = act_exponent(__float_as_uint(m));
        }
      }
      for (int r = 0; r < ntok; ++r) {
        int er = 0;
#pragma unroll
        for (int jj = 0; jj < G; ++jj)
          if (jj == r) er = aexp[jj];
        const float sc = ldexpf(1.0f, er);
        for (int u = warp * 32 + lane; u < units; u += Q * 32) {
          uint4* pa = reinterpret_cast<uint4*>(panel + r * prow + u * 16);
          const uint4 v = *pa;
          const uint32_t in[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            __half2 h2 = __floats2half2_rn(bf16_bits_to_f32(in[t] & 0xffffu) * sc, bf16_bits_to_f32(in[t] >> 16) * sc);
            o[t] = *reinterpret_cast<uint32_t*>(&h2);
          }
          *pa = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(pready);
      if (!mbar_wait(pready, pseq & 1, a.st, 8)) break;
      act_row = smem_u32(panel) + (g < G ? g : 0) * prow + q * 16;
      ++pseq;
    }
    float acc[2][2][NV];  // [mtile][lo/hi row][token column]
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[m][h][v] = 0.f;
    float acc4[2][2][4];  // NVFP4: [block parity][mtile][mma accumulator]
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc4[u][m][i] = 0.f;
    for (int c = 0; c < nch; ++c) {
      const int d = seq % D;
      const uint32_t par = (seq / D) & 1;
      ++seq;
      if (!mbar_wait(&full[d], par, a.st, 3)) {
        alive = false;
        break;
      }
      const uint8_t* slot = smem + d * Lay::kSlot;
      const uint32_t sbase = smem_u32(slot);
      const uint32_t act_addr = act_row + c * kc * 2;
      for (int pl = warp; pl < nplanes; pl += Q) {
        if constexpr (FMT == FMT_NV) {
          uint16_t* tab = reinterpret_cast<uint16_t*>(table);
          expand_plane_scales_nv<MODE>(slot + Lay::kCodes, nsb, pl, tab, lane);
          __syncwarp();
          plane_blocks_nv<NV>(sbase, act_addr, tab, box_off, row_in_box, lm, g, q, acc4, pl);
        } else {
          expand_plane_scales<MODE>(slot + Lay::kCodes, nb, pl, table, lane);
          __syncwarp();
          plane_blocks<NV>(sbase, act_addr, table, box_off, row_in_box, lm, g, acc, pl);
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(&empty[d]);
    }
    if (!alive) break;
    if constexpr (FMT == FMT_NV) {
      // m16n8 accumulator: d0, d1 row g, columns 2q, 2q+1; d2, d3 row g + 8
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int v = 0; v < NV; ++v) acc[m][h][v] = acc4[0][m][2 * h + v] + acc4[1][m][2 * h + v];
    }
    const bool last_of_group = (j + 1 == nloc) || ((it + 1) / tiles != grp);
    if (last_of_group) {
      // panel reads (and this warp's conversion writes) come before the next bulk copy into it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&pempty[(pseq - 1) % NP]);
    }
    // partials to the epilogue warp (double-buffered by item parity)
    const int pb = j & 1;
    if (!mbar_wait(&rempty[pb], ((j >> 1) & 1) ^ 1, a.st, 9)) break;
    float* rbuf = red + (pb * Q + warp) * kPart;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int v = 0; v < NV; ++v) rbuf[((m * 2 + h) * NV + v) * 32 + lane] = acc[m][h][v];
    if (warp == 0) {
      ItemHdr* h = ihdr + pb;
      if (lane == 0) {
        h->p0 = p0;
        h->ntok = ntok;
        h->tile = tile;
        h->gscale = gscale;
      }
      if (lane < G) {
#pragma unroll
        for (int jj = 0; jj < G; ++jj)
          if (jj == lane) {
            h->aexp[lane] = aexp[jj];
            h->rows[lane] = arow_id[jj];
          }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rfull[pb]);
  }
  if (MODE == MODE_DOWN && a.zb) down_z_step<Q + 1>(a, red, warp, lane);
}

// ---------------------------------------------------------------------------
// launch configuration
// ---------------------------------------------------------------------------
int expert_max_group(int T) { return T <= 1 ? 1 : 8; }

template <int MODE, int G, int Q, int FMT>
static int launch_one(ExpertArgs a, cudaStream_t s, int num_sms) {
  using SM = Smem<G, Q, FMT>;
  using Lay = Layout<FMT>;
  auto kern = expert_kernel<MODE, G, Q, FMT>;
  if (FMT == FMT_NV && !a.gs) return LMOE_EINVAL;
  constexpr int kSmemMax = 232448;
  if (a.K > kMaxK) return LMOE_EUNSUPPORTED;
  // as many ring slots as fit next to the panel (at least 2)
  const int D = min(kMaxSlots, (kSmemMax - SM::fixed(a.K) - 1024) / Lay::kSlot);
  if (D < 2) return LMOE_EUNSUPPORTED;
  const int smem = SM::bytes(a.K, D);
  static int attr_done[64] = {};  // per device: largest dynamic shared memory size set so far
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_done[dev & 63] < smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return LMOE_ECUDA;
    attr_done[dev & 63] = smem;
  }
  // K chunk: the whole K when K <= kKC, else kKC (K is a multiple of kKC then)
  a.kc = a.K <= kKC ? a.K : kKC;
  const int rows_per_expert = (MODE == MODE_GATEUP) ? 2 * a.inter : a.latent;
  const uint64_t rows_total = (uint64_t)a.n_experts * rows_per_expert;
  CUtensorMap tq, ts;
  {
    // codes as {128 B, rows, K/256 planes}: plane stride 128 B, row stride K/2 B
    const uint64_t dims[3] = {128, rows_total, (uint64_t)a.K / 256};
    const uint64_t strides[2] = {(uint64_t)a.K / 2, 128};
    const uint32_t box[3] = {128, 16, (uint32_t)(a.kc / 256)};
    if (get_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return LMOE_ECUDA;
  }
  if (a.K > kKC) {
    // scales as {K/SB bytes, rows}: SB = 32 (E8M0) or 16 (E4M3) elements per byte
    const uint64_t dims[2] = {(uint64_t)a.K / Lay::kSB, rows_total};
    const uint64_t strides[1] = {(uint64_t)a.K / Lay::kSB};
    const uint32_t box[2] = {(uint32_t)(a.kc / Lay::kSB), 16};
    if (get_tmap(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.s, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return LMOE_ECUDA;
  } else {
    ts = tq;  // unused: one chunk copies the scales with a bulk copy
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(32 * (Q + 2));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, tq, ts, D) == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

int launch_gateup(const ExpertArgs& a, int T, int max_group, cudaStream_t s, int num_sms) {
  if (a.gs) {
    if (max_group == 1) return launch_one<MODE_GATEUP, 1, 8, FMT_NV>(a, s, num_sms);
    return launch_one<MODE_GATEUP, 8, 8, FMT_NV>(a, s, num_sms);
  }
  if (max_group == 1) return launch_one<MODE_GATEUP, 1, 8, FMT_MX>(a, s, num_sms);
  return launch_one<MODE_GATEUP, 8, 8, FMT_MX>(a, s, num_sms);
}

int launch_down(const ExpertArgs& a, int T, int max_group, cudaStream_t s, int num_sms) {
  if (a.gs) {
    if (max_group == 1) return launch_one<MODE_DOWN, 1, 8, FMT_NV>(a, s, num_sms);
    return launch_one<MODE_DOWN, 8, 8, FMT_NV>(a, s, num_sms);
  }
  if (max_group == 1) return launch_one<MODE_DOWN, 1, 8, FMT_MX>(a, s, num_sms);
  return launch_one<MODE_DOWN, 8, 8, FMT_MX>(a, s, num_sms);
}

}  // namespace lmoe
