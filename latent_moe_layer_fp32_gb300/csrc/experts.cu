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
// K) for every row of its group.
//
// CTA = W consumer warps + 1 producer warp.  Per K chunk the producer issues
// two TMA tensor copies of the codes (16 rows x kc/2 bytes each, a 3-D view
// {128 B, rows, K/256} with 128-byte swizzle, so each copy is one 16 KB
// request and ldmatrix reads it without bank conflicts), two of the E8M0
// scales and one bulk copy per activation row, into per-warp mbarrier rings
// of D slots; consumer warp w takes items w, w+W, ... of the CTA's range.
//
// Consumer per 32-element scale block: ldmatrix.x4 hands each lane 4 code
// bytes of two rows; cvt.rn.f16x2.e2m1x2 turns each byte into two exact f16
// values; two mma.sync m16n8k16 (f16 in, fp32 accumulate) cover the block's
// 32 K positions in a fixed permutation that the activation fragment follows;
// the fresh block result is scaled by the block's E8M0 value (expanded once
// per chunk into a per-warp fp32 table) and added to the fp32 accumulator.
// Activations arrive as bf16 rows; each warp converts its plane's columns to
// f16 times a per-row power of two (exact; undone in the epilogue), the power
// coming from the row's max |value| that the producing kernel recorded.
#include "common.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace lmoe {

enum { MODE_GATEUP = 0, MODE_DOWN = 1 };

constexpr int kRows = 32;  // weight rows per item: two m16 tiles
constexpr int kKC = 2048;  // K elements per chunk when K > 2048 (else the whole K): 16 KB code boxes

// Header the producer writes into the first slot of every item.
struct ItemMeta {
  int p0, ntok, pad0, pad1;
  int aexp[8];  // per token of the group: power of two mapping its activation row into f16 range
  int rows[8];  // per token: sorted_rows[p0 + j] (the original route row id)
};
static_assert(sizeof(ItemMeta) <= 128, "item header");

template <int G>
struct Layout {
  static constexpr int kBox = 16 * (kKC / 2);  // one code box: 16 rows x kc/2 bytes (16 KB)
  static constexpr int kCodes = 2 * kBox;      // box A (rows 0-15 of the item), box B (rows 16-31)
  static constexpr int kScales = kRows * (kKC / 32);
  static constexpr int kActRow = kKC * 2 + 64;  // padded: conflict-free 16-byte loads
  static constexpr int kActs = G * kActRow;
  static constexpr int kMeta = 128;  // item header: p0, ntok, per-token exponent and row id
  static constexpr int kSlot = (kCodes + kScales + kActs + kMeta + 1023) / 1024 * 1024;  // 1 KB aligned (swizzle atom)
};

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

template <int MODE, int G, int NGRP, int Q, int D>
__global__ void __launch_bounds__(32 * (NGRP * Q + 1), 1)
    expert_kernel(const ExpertArgs a, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_s) {
  // NGRP groups of Q consumer warps; group gi owns a ring of D slots and the
  // CTA items gi, gi+NGRP, ...; its Q warps share every slot, member j taking
  // the chunk's 128-byte planes j, j+Q, ...; the members' fp32 partials are
  // added in member order at the end of each item.
  using Lay = Layout<G>;
  constexpr int NW = NGRP * Q;
  constexpr int NV = (G == 1) ? 1 : 2;  // token columns per lane that can hold a valid token
  constexpr int kRed = 2 * 2 * NV * 32;  // floats per member partial (two buffers, by item parity)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1 KB alignment for the swizzled boxes
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* tables = reinterpret_cast<float*>(smem + NGRP * D * Lay::kSlot);      // [NW][8*2*8*2]
  float* red = tables + NW * 256;                                              // [2][NW][kRed]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 2 * NW * kRed);
  uint64_t* empty = full + NGRP * D;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K, kc = a.kc, nch = K / kc, nb = kc / 32, cbk = kc / 256;  // cbk: 128-byte planes per chunk
  const int Ks = K / 32;
  const int tiles = (MODE == MODE_GATEUP) ? a.inter / 16 : a.latent / kRows;
  const int rows_per_expert = (MODE == MODE_GATEUP) ? 2 * a.inter : a.latent;
  const int kact_row = kc * 2 + 64;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NGRP * D; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], Q);
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

  if (warp == NW) {
    // ------------------------------ producer ------------------------------
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_s)) : "memory");
    }
    int seq[NGRP];
#pragma unroll
    for (int gi = 0; gi < NGRP; ++gi) seq[gi] = 0;
    bool ok = true;
    // metadata of 32 items at a time, item (batch + lane) in lane `lane`
    int m_e = 0, m_p0 = 0, m_ntok = 0, m_rows[G], m_exp[G];
    int batch = -1;
    for (int base = 0; base < nloc && ok; base += NGRP) {
      const int ng = min(NGRP, nloc - base);
      if (base / 32 != batch) {
        batch = base / 32;
        const int itl = batch * 32 + lane;
        m_ntok = 0;
        if (itl < nloc) {
          const int4 gq = a.groups[(it0 + itl) / tiles];
          m_e = gq.x;
          m_p0 = gq.y;
          m_ntok = gq.z;
        }
#pragma unroll
        for (int jj = 0; jj < G; ++jj) {
          m_rows[jj] = 0;
          m_exp[jj] = 0;
          if (jj < m_ntok) m_rows[jj] = a.sorted_rows[m_p0 + jj];
        }
#pragma unroll
        for (int jj = 0; jj < G; ++jj)
          if (jj < m_ntok) m_exp[jj] = act_exponent(a.act_max[(MODE == MODE_GATEUP) ? m_rows[jj] / a.top_k : m_p0 + jj]);
      }
      for (int c = 0; c < nch && ok; ++c) {
        for (int gi = 0; gi < ng; ++gi) {
          const int it = it0 + base + gi;
          const int tile = it % tiles;
          const int src = (base + gi) & 31;
          const int e = __shfl_sync(0xffffffffu, m_e, src);
          const int p0 = __shfl_sync(0xffffffffu, m_p0, src);
          const int ntok = __shfl_sync(0xffffffffu, m_ntok, src);
          int my_row = 0, my_exp = 0;  // token `lane` of this item
#pragma unroll
          for (int jj = 0; jj < G; ++jj) {
            const int rv = __shfl_sync(0xffffffffu, m_rows[jj], src);
            const int ev = __shfl_sync(0xffffffffu, m_exp[jj], src);
            if (lane == jj) {
              my_row = rv;
              my_exp = ev;
            }
          }
          const int d = seq[gi] % D;
          const uint32_t par = ((seq[gi] / D) & 1) ^ 1;
          ++seq[gi];
          int got = 1;
          if (lane == 0) got = mbar_wait(&empty[gi * D + d], par, a.st, 1);
          if (!__shfl_sync(0xffffffffu, got, 0)) {
            ok = false;
            break;
          }
          uint8_t* slot = smem + (gi * D + d) * Lay::kSlot;
          uint64_t* bar = &full[gi * D + d];
          // first rows of box A and box B
          int rowA, rowB;
          if (MODE == MODE_GATEUP) {
            rowA = e * rows_per_expert + tile * 16;
            rowB = rowA + a.inter;
          } else {
            rowA = e * rows_per_expert + tile * kRows;
            rowB = rowA + 16;
          }
          if (c == 0) {
            ItemMeta* meta = reinterpret_cast<ItemMeta*>(slot + Lay::kCodes + Lay::kScales + Lay::kActs);
            if (lane == 0) {
              meta->p0 = p0;
              meta->ntok = ntok;
            }
            if (lane < G) {
              meta->aexp[lane] = my_exp;
              meta->rows[lane] = my_row;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_expect_tx(bar, kRows * (kc / 2) + kRows * nb + (uint32_t)ntok * kc * 2);
          __syncwarp();
          if (lane == 0) {
            tma_load_3d(slot, &tm_q, 0, rowA, c * cbk, bar, pol);
            tma_load_3d(slot + 16 * (kc / 2), &tm_q, 0, rowB, c * cbk, bar, pol);
          } else if (lane == 1 || lane == 2) {
            uint8_t* sdst = slot + Lay::kCodes + (lane - 1) * 16 * nb;
            const int srow = lane == 1 ? rowA : rowB;
            if (nch > 1)
              tma_load_2d(sdst, &tm_s, c * nb, srow, bar, pol);
            else  // one chunk: the 16 rows' scales are contiguous
              bulk_g2s(sdst, a.s + (size_t)srow * Ks, 16 * Ks, bar);
          }
          // activation rows: token j's copy from lane j (its row id is in my_row)
          if (lane < ntok) {
            const int j = lane;
            const int arow = (MODE == MODE_GATEUP) ? my_row / a.top_k : p0 + j;
            bulk_g2s(slot + Lay::kCodes + Lay::kScales + j * kact_row, a.act + (size_t)arow * K + c * kc, kc * 2,
                     bar);
          }
          __syncwarp();
        }
      }
    }
    // drain: no copy may still be in flight when this warp leaves
    if (lane == 0) {
#pragma unroll
      for (int gi = 0; gi < NGRP; ++gi)
        for (int s = max(0, seq[gi] - D); s < seq[gi]; ++s)
          mbar_wait(&full[gi * D + (s % D)], (s / D) & 1, a.st, 2);
    }
    return;
  }

  // -------------------------------- consumer --------------------------------
  const int gi = warp / Q, mem = warp % Q;
  const int g = lane >> 2, q = lane & 3;
  // ldmatrix.x4 for m-tile m and blocks (b, b+1): matrices (lo rows, b) (hi rows, b) (lo rows, b+1) (hi rows, b+1)
  const int lm = lane >> 3, rr = lane & 7;
  float* table = tables + warp * 256;
  int item_count = 0;
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
  int seq = 0;
  bool alive = true;
  for (int j = gi; j < nloc; j += NGRP) {
    const int it = it0 + j;
    const int tile = it % tiles;
    int p0 = 0, ntok = 0;
    int aexp[G], arow_id[G];  // from the item header (first chunk's slot)
    float acc[2][2][NV];  // [mtile][lo/hi row][token column]
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[m][h][v] = 0.f;
    for (int c = 0; c < nch && alive; ++c) {
      const int d = seq % D;
      const uint32_t par = (seq / D) & 1;
      ++seq;
      if (!mbar_wait(&full[gi * D + d], par, a.st, 3)) {
        alive = false;
        break;
      }
      const uint8_t* slot = smem + (gi * D + d) * Lay::kSlot;
      if (c == 0) {
        const ItemMeta* meta = reinterpret_cast<const ItemMeta*>(slot + Lay::kCodes + Lay::kScales + Lay::kActs);
        p0 = meta->p0;
        ntok = meta->ntok;
#pragma unroll
        for (int jj = 0; jj < G; ++jj) {
          aexp[jj] = meta->aexp[jj];
          arow_id[jj] = meta->rows[jj];
        }
      }
      const uint32_t sbase = smem_u32(slot);
      const uint32_t act_addr = smem_u32(slot + Lay::kCodes + Lay::kScales) + (g < G ? g : 0) * kact_row + q * 16;
      for (int pl = mem; pl < nplanes; pl += Q) {
        expand_plane_scales<MODE>(slot + Lay::kCodes, nb, pl, table, lane);
        // this plane's activation columns (256 per token): bf16 -> f16 * 2^e in place
#pragma unroll
        for (int jj = 0; jj < G; ++jj) {
          if (jj < ntok) {
            uint4* pa = reinterpret_cast<uint4*>(const_cast<uint8_t*>(slot) + Lay::kCodes + Lay::kScales +
                                                 jj * kact_row + pl * 512) + lane;
            const uint4 v = *pa;
            const float sc = ldexpf(1.0f, aexp[jj]);
            const uint32_t in[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              __half2 h2 = __floats2half2_rn(bf16_bits_to_f32(in[u] & 0xffffu) * sc, bf16_bits_to_f32(in[u] >> 16) * sc);
              o[u] = *reinterpret_cast<uint32_t*>(&h2);
            }
            *pa = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        __syncwarp();
        plane_blocks<NV>(sbase, act_addr, table, box_off, row_in_box, lm, g, acc, pl);
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(&empty[gi * D + d]);
    }
    // ------------------- member partials, added in member order -------------------
    // Two buffers by item parity: a member may write item i+1's partials while
    // member 0 still reads item i's, so one barrier per item suffices (a member
    // reaches item i+2's write only after the barrier of item i+1, which member
    // 0 passes after finishing item i).
    float* rbuf = red + (item_count & 1) * NW * kRed;
    ++item_count;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int v = 0; v < NV; ++v) rbuf[warp * kRed + ((m * 2 + h) * NV + v) * 32 + lane] = acc[m][h][v];
    asm volatile("bar.sync %0, %1;" ::"r"(1 + gi), "r"(Q * 32) : "memory");
    if (mem == 0) {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            float t = rbuf[(gi * Q) * kRed + ((m * 2 + h) * NV + v) * 32 + lane];
            for (int o = 1; o < Q; ++o) t += rbuf[(gi * Q + o) * kRed + ((m * 2 + h) * NV + v) * 32 + lane];
            acc[m][h][v] = t;
          }
      // ------------------------------ epilogue ------------------------------
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
          const float inv = ldexpf(1.0f, -e_tok);
          if (MODE == MODE_GATEUP) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const float gv = acc[m][0][v] * inv, uv = acc[m][1][v] * inv;
              const uint16_t hb = f32_to_bf16_bits(gv / (1.0f + expf(-gv)) * uv);
              a.h_out[(size_t)p * a.inter + tile * 16 + m * 8 + g] = hb;
              ssq[v] = fmaxf(ssq[v], fabsf(bf16_bits_to_f32(hb)));  // gate/up: running max |h|
            }
          } else {
            const int r = r_tok;
            float* yr = a.y_out + (size_t)r * a.latent + tile * kRows;
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
      if (MODE == MODE_GATEUP) {
        // row max of |h| over this tile's 16 features, folded into the row's max word
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          float mv = ssq[v];
          mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, 4));
          mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, 8));
          mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, 16));
          const int tok = 2 * q + v;
          if (g == 0 && tok < ntok) atomicMax(&a.h_max[p0 + tok], __float_as_uint(mv));
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
  }
}

// ---------------------------------------------------------------------------
// launch configuration
// ---------------------------------------------------------------------------
int expert_max_group(int T) { return T <= 1 ? 1 : 8; }

template <int MODE, int G, int NGRP, int Q, int D>
static int launch_one(ExpertArgs a, cudaStream_t s, int num_sms) {
  using Lay = Layout<G>;
  auto kern = expert_kernel<MODE, G, NGRP, Q, D>;
  constexpr int NV = (G == 1) ? 1 : 2;
  constexpr int smem = NGRP * D * Lay::kSlot + NGRP * Q * (256 + 2 * 2 * 2 * NV * 32) * 4 + 2 * NGRP * D * 8 +
                       1024;  // +1 KB alignment slack
  static_assert(smem <= 232448, "shared memory budget");
  static unsigned long long attr_done = 0;  // one bit per device, per template instance
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done >> (dev & 63) & 1ull)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return LMOE_ECUDA;
    attr_done |= 1ull << (dev & 63);
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
    const uint64_t dims[2] = {(uint64_t)a.K / 32, rows_total};
    const uint64_t strides[1] = {(uint64_t)a.K / 32};
    const uint32_t box[2] = {(uint32_t)(a.kc / 32), 16};
    if (get_tmap(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.s, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return LMOE_ECUDA;
  } else {
    ts = tq;  // unused: one chunk copies the scales with a bulk copy
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(32 * (NGRP * Q + 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, tq, ts) == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

int launch_gateup(const ExpertArgs& a, int T, int max_group, cudaStream_t s, int num_sms) {
  if (max_group == 1) return launch_one<MODE_GATEUP, 1, 1, 8, 5>(a, s, num_sms);
  return launch_one<MODE_GATEUP, 8, 1, 8, 3>(a, s, num_sms);
}

int launch_down(const ExpertArgs& a, int T, int max_group, cudaStream_t s, int num_sms) {
  if (max_group == 1) return launch_one<MODE_DOWN, 1, 1, 8, 5>(a, s, num_sms);
  return launch_one<MODE_DOWN, 8, 1, 8, 3>(a, s, num_sms);
}

}  // namespace lmoe
