// Routed experts at decode sizes (a routing table of at most 64 rows), MXFP4
// W4A16: gate/up + SwiGLU and then down, in ONE persistent launch.
//
// "Muse Spark Open on Gaudi 2": experts run W4A16 ("What was built"), each
// (token, route) pair is its own row and the cost is per touched expert slice
// ("The latent MoE: A' with a per-expert norm"); the packed E2M1 nibbles and
// E8M0 scales are read directly ("Why it needed a port").  "RadixArk team
// serves Meta's Muse Spark Open on one TPU host", "A single program": the weight
// stream is kept going from one stage to the next instead of draining and
// ramping up again at every kernel boundary.
//
// One CTA per SM; every CTA takes a contiguous range of the gate/up work items
// and then a contiguous range of the down items.  A work item is one group of
// rows of one expert (sorted positions p0 .. p0+n-1, n <= G) together with a
// tile of 32 weight rows: 16 gate rows and the matching 16 up rows, or 32
// down rows.  Each slot of the weight ring holds one K chunk (up to 2048) of
// one item: two 16-row code boxes (a 3-D view {128 B, rows, K/256} with
// 128-byte swizzle) and their two E8M0 scale boxes (a 3-D view {16 B, rows,
// K/512}, so that the scales of 16 blocks of one row are 16 contiguous bytes
// and the eight rows a warp reads at once fall on eight distinct bank groups).
//
// Warps:
//  - 0 .. 7   consumers: every slot is shared, warp j taking 128-byte planes
//             j, j+8, ... of the chunk.  Per 32-element block, ldmatrix hands
//             each lane code bytes of two rows, cvt.rn.f16x2.e2m1x2 makes exact
//             f16 pairs, two mma.sync m16n8k16 (fp32 accumulate) take the
//             block, and the block result is scaled by the block's E8M0 value
//             (2^(s-127) built in registers from the scale byte) and added to
//             the fp32 accumulator.  Partials go to the epilogue warp.
//  - 8        weight producer: the routing table (<= 64 groups and rows) is
//             read once into registers; one lane issues the four copies of
//             every slot.  It never waits on data, only on free slots, so the
//             down weights stream while the gate/up results are still being
//             completed elsewhere on the GPU.
//  - 9        activation producer: all T rows of x_lat at once for gate/up
//             (each group picks its tokens' rows); then the h rows of each
//             down group, into one of NPd panels, once that group's h rows
//             are complete (a device-wide counter per group).
//  - 10       epilogue: adds the 8 partials of an item in warp order, then
//             SwiGLU -> h (bf16), or y (fp32, by original row id) plus its
//             sums of squares per 32-column tile; after each gate/up item it
//             raises its group's counter.
// With a workspace for the layer's norm and sum (lmoe_forward), the consumer
// warps then form z = sum_j w_j * (y_j * rinv_j) * g_j for a 32-column slice
// of the latent width once every CTA has written its down rows (a device-wide
// counter), so no separate launch sits between the experts and the unpooler.
// Activations are converted once per panel: bf16 -> f16 times the power of
// two that puts the row's largest magnitude in [2^14, 2^15) (exact for every
// element down to 2^-17 of that scale), undone in the epilogue.
// Every wait is bounded (LMOE_ETIMEOUT in the status word).  The device-wide
// counter needs every CTA resident at once: the grid is one CTA per SM and
// the launch is cooperative.
#include "common.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace lmoe {
namespace {

constexpr int kQ = 8;                  // consumer warps
constexpr int kWProd = kQ, kAProd = kQ + 1, kEpi = kQ + 2;
constexpr int kThreads = 32 * (kQ + 3);
constexpr int kRows = 32;              // weight rows per item
constexpr int kKC = 2048;              // K chunk (whole K when K <= 2048)
constexpr int kSlot = 17 * kKC;        // codes 16*kc + scales kc bytes: 34 KB
constexpr int kMaxSlots = 6;
constexpr int kMaxTab = 64;            // routing-table rows / groups held in registers
enum { PH_GATEUP = 0, PH_DOWN = 1 };

// What the weight producer tells the consumers about the item of a slot.
struct SlotHdr {
  int p0, ntok, tile, phase;
  int rows[8];  // sorted_rows[p0 + i]: the original route row ids
};

// What consumer warp 0 hands the epilogue with an item's partials.
struct ItemHdr {
  int p0, ntok, tile, phase, grp, pad[3];
  int aexp[8];
  int rows[8];
};

struct Plan {
  int D, NPd, prow_x, prow_h, region, G, NV;
  __host__ __device__ int kpart() const { return 2 * 2 * NV * 32; }
};

__device__ __forceinline__ float e8m0_fast(uint32_t w, int j) {
  // byte j of w as the exponent field: 2^(s-127) for 1 <= s <= 254
  const uint32_t b = j == 0 ? (w << 23) : j == 1 ? (w << 15) : j == 2 ? (w << 7) : (w >> 1);
  return __uint_as_float(b & 0x7f800000u);
}

__device__ __forceinline__ bool has_special_byte(uint32_t w) {
  // some byte is 0 (2^-127) or 255 (NaN): take the exact per-value path
  return __vcmpltu4(__vadd4(w, 0x01010101u), 0x02020202u) != 0u;
}

// The codes of 128-byte plane p of a slot, for m-tiles 0 and 1, into registers
// (w[i][m][4]: ldmatrix.x4 of blocks 2i, 2i+1), so that the slot can be
// released before the arithmetic: the ring refills while the plane is computed.
__device__ __forceinline__ void plane_load(uint32_t cbase, const uint32_t (&box_off)[2], const int (&row_in_box)[2],
                                           int lm, int p, uint32_t (&w)[4][2][4]) {
  const int rr = row_in_box[0] & 7;  // both m-tiles' rows share row & 7
  const uint32_t pb0 = cbase + box_off[0] + row_in_box[0] * 128 + p * 2048;
  const uint32_t pb1 = cbase + box_off[1] + row_in_box[1] * 128 + p * 2048;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t coff = static_cast<uint32_t>(((2 * i + (lm >> 1)) ^ rr) << 4);
    ldmatrix_x4(w[i][0][0], w[i][0][1], w[i][0][2], w[i][0][3], pb0 + coff);
    ldmatrix_x4(w[i][1][0], w[i][1][1], w[i][1][2], w[i][1][3], pb1 + coff);
  }
}

// The 8 blocks of a plane from its codes in registers.  sw[m][h]: the 8
// scale bytes of this lane's lo (h = 0) / hi (h = 1) row of m-tile m.
template <int NV, bool SPECIAL>
__device__ __forceinline__ void plane_mx(const uint32_t (&w)[4][2][4], uint32_t act_addr, const uint2 (&sw)[2][2],
                                         float (&acc)[2][2][NV], int p) {
  const uint32_t pact = act_addr + p * 512;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int blk = 2 * i + half;
      uint32_t b0, b1, b2, b3;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                   : "r"(pact + blk * 64));
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        uint32_t l0, l1, l2, l3, h0, h1, h2, h3;
        e2m1x8_to_f16x8(w[i][m][2 * half], l0, l1, l2, l3);
        e2m1x8_to_f16x8(w[i][m][2 * half + 1], h0, h1, h2, h3);
        float dacc[4];
        mma_f16_zero(dacc, l0, h0, l1, h1, b0, b1);
        mma_f16(dacc, l2, h2, l3, h3, b2, b3);
        const uint32_t wlo = (blk < 4) ? sw[m][0].x : sw[m][0].y;
        const uint32_t whi = (blk < 4) ? sw[m][1].x : sw[m][1].y;
        float slo, shi;
        if (SPECIAL) {
          slo = e8m0_to_f32((wlo >> (8 * (blk & 3))) & 0xffu);
          shi = e8m0_to_f32((whi >> (8 * (blk & 3))) & 0xffu);
        } else {
          slo = e8m0_fast(wlo, blk & 3);
          shi = e8m0_fast(whi, blk & 3);
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          acc[m][0][v] = fmaf(dacc[v], slo, acc[m][0][v]);
          acc[m][1][v] = fmaf(dacc[2 + v], shi, acc[m][1][v]);
        }
      }
    }
  }
}

// The 8 consumer warps meet at `cbar` (count kQ; nsync counts the meetings so
// far, the same in every consumer warp).  Bounded like every other wait.
__device__ __forceinline__ bool consumers_meet(uint64_t* cbar, int& nsync, Status* st, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(cbar);
  const bool ok = mbar_wait(cbar, nsync & 1, st, 53);
  ++nsync;
  return ok;
}

// Convert `nrows` activation rows of a panel in place, by the 8 consumer warps:
// bf16 -> f16 * 2^e with e per row.  Row r's exponent goes to exps[r].
__device__ __forceinline__ bool convert_rows(uint8_t* panel, int prow, int nrows, int K, float* smax, int* exps,
                                             int warp, int lane, uint64_t* cbar, int& nsync, Status* st) {
  const int units = K / 8;  // 16-byte units per row
  for (int r = 0; r < nrows; ++r) {
    float m = 0.f;
    for (int u = warp * 32 + lane; u < units; u += kQ * 32) {
      const uint4 v = *reinterpret_cast<const uint4*>(panel + r * prow + u * 16);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; ++t)
        m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(w4[t] & 0xffffu)), fabsf(bf16_bits_to_f32(w4[t] >> 16))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) smax[warp * 8 + r] = m;
  }
  if (!consumers_meet(cbar, nsync, st, lane)) return false;
  if (warp == 0 && lane < nrows) {
    float m = smax[lane];
#pragma unroll
    for (int w = 1; w < kQ; ++w) m = fmaxf(m, smax[w * 8 + lane]);
    exps[lane] = act_exponent(__float_as_uint(m));
  }
  if (!consumers_meet(cbar, nsync, st, lane)) return false;
  for (int r = 0; r < nrows; ++r) {
    const float sc = ldexpf(1.0f, exps[r]);
    for (int u = warp * 32 + lane; u < units; u += kQ * 32) {
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
  return consumers_meet(cbar, nsync, st, lane);
}

// The items of one stage this CTA takes, in order: it = first, first + step, ... < end
// (a contiguous range: the CTA's gate/up and down items belong to the same one
// or two groups, so each down group waits only for the CTAs that share it).
struct Seq {
  int first, step, end;
  __device__ __forceinline__ int count() const { return first < end ? (end - first + step - 1) / step : 0; }
};

__device__ __forceinline__ Seq stage_seq(int n) {
  return {(int)((long long)n * blockIdx.x / gridDim.x), 1, (int)((long long)n * (blockIdx.x + 1) / gridDim.x)};
}

template <int G, int NV>
__global__ void __launch_bounds__(kThreads, 1)
    fused_experts_kernel(const FusedExpertArgs a, const __grid_constant__ CUtensorMap tq_gu,
                         const __grid_constant__ CUtensorMap ts_gu, const __grid_constant__ CUtensorMap tq_dn,
                         const __grid_constant__ CUtensorMap ts_dn, const Plan pl) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int D = pl.D, NPd = pl.NPd;
  constexpr int kPart = 2 * 2 * NV * 32;
  uint8_t* region = smem + D * kSlot;                                       // x_lat rows, later the h panels
  float* red = reinterpret_cast<float*>(region + pl.region);                // [2][kQ][kPart]
  float* smax = red + 2 * kQ * kPart;                                       // [kQ][8]
  int* texp = reinterpret_cast<int*>(smax + kQ * 8);                        // [8] x_lat row exponents
  int* pexp = texp + 8;                                                     // [2][8] h panel row exponents
  SlotHdr* shdr = reinterpret_cast<SlotHdr*>(pexp + 16);                    // [kMaxSlots]
  ItemHdr* ihdr = reinterpret_cast<ItemHdr*>(shdr + kMaxSlots);             // [2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ihdr + 2);
  uint64_t* full = bars;                     // [kMaxSlots] slot loaded (1 + tx)
  uint64_t* empty = full + kMaxSlots;        // [kMaxSlots] slot released (kQ)
  uint64_t* xfull = empty + kMaxSlots;       // x_lat rows loaded (1 + tx)
  uint64_t* xempty = xfull + 1;              // x_lat region released (kQ)
  uint64_t* pfull = xempty + 1;              // [2] h panel loaded (1 + tx)
  uint64_t* pempty = pfull + 2;              // [2] h panel released (kQ)
  uint64_t* rfull = pempty + 2;              // [2] partials written (kQ)
  uint64_t* rempty = rfull + 2;              // [2] partials taken (1)
  uint64_t* cbar = rempty + 2;               // consumer warps meet (kQ)
  uint64_t* gudone = cbar + 1;               // this CTA's gate/up items are written (1)
  float* s_rinv = reinterpret_cast<float*>(gudone + 1);  // [64] per route row: 1/rms of y (the z step)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = a.latent, I = a.inter, k = a.top_k;
  const int tiles_gu = I / 16, tiles_dn = L / kRows;

  if (threadIdx.x == 0) {
    for (int i = 0; i < D; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kQ);
    }
    mbar_init(xfull, 1);
    mbar_init(xempty, kQ);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull[i], 1);
      mbar_init(&pempty[i], kQ);
      mbar_init(&rfull[i], kQ);
      mbar_init(&rempty[i], 1);
    }
    mbar_init(cbar, kQ);
    mbar_init(gudone, 1);
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWProd) {
    // ------------------------------ weight producer ------------------------------
    if (!a.early) {
      pdl_wait();
      pdl_trigger();
    }
    // the routing table (written before the preceding kernel ran) in registers
    const int ng = min(*a.n_groups, kMaxTab);
    int4 g0 = make_int4(0, 0, 0, 0), g1 = g0;
    if (lane < ng) g0 = a.groups[lane];
    if (lane + 32 < ng) g1 = a.groups[lane + 32];
    auto entry = [&](int grp) -> int4 {
      const int4 v = grp < 32 ? g0 : g1;
      const int src = grp & 31;
      return make_int4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                       __shfl_sync(0xffffffffu, v.z, src), 0);
    };
    int r0 = 0, r1 = 0;
    if (lane < a.rows) r0 = a.sorted_rows[lane];
    if (lane + 32 < a.rows) r1 = a.sorted_rows[lane + 32];
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tq_gu)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tq_dn)) : "memory");
    }
    int seq = 0;
    bool ok = true, waited = !a.early;
    for (int ph = 0; ph < 2 && ok; ++ph) {
      const int tiles = ph == PH_GATEUP ? tiles_gu : tiles_dn;
      const int K = ph == PH_GATEUP ? L : I;
      const int kc = K <= kKC ? K : kKC, nch = K / kc;
      const int rows_per_expert = ph == PH_GATEUP ? 2 * I : L;
      const bool scale_tma = (kc % 512) == 0;
      const CUtensorMap* tq = ph == PH_GATEUP ? &tq_gu : &tq_dn;
      const CUtensorMap* ts = ph == PH_GATEUP ? &ts_gu : &ts_dn;
      const uint8_t* sbase = ph == PH_GATEUP ? a.w13_s : a.w2_s;
      const Seq sq = ph == PH_GATEUP ? stage_seq(ng * tiles) : stage_seq(ng * tiles);
      int cur = -1;
      int4 g4 = make_int4(0, 0, 0, 0);
      int my_row = 0;
      for (int it = sq.first; it < sq.end && ok; it += sq.step) {
        const int grp = it / tiles, tile = it % tiles;
        if (grp != cur) {
          cur = grp;
          g4 = entry(grp);
          const int idx = (g4.y + lane) & 63;
          const int v0 = __shfl_sync(0xffffffffu, r0, idx & 31), v1 = __shfl_sync(0xffffffffu, r1, idx & 31);
          my_row = idx < 32 ? v0 : v1;
        }
        int rowA, rowB;
        if (ph == PH_GATEUP) {
          rowA = g4.x * rows_per_expert + tile * 16;
          rowB = rowA + I;
        } else {
          rowA = g4.x * rows_per_expert + tile * kRows;
          rowB = rowA + 16;
        }
        for (int c = 0; c < nch && ok; ++c) {
          const int d = seq % D;
          const uint32_t par = ((seq / D) & 1) ^ 1;
          int good = 1;
          if (lane == 0) good = seq < D || mbar_wait(&empty[d], par, a.st, 41);
          ok = __shfl_sync(0xffffffffu, good, 0) != 0;
          if (!ok) break;
          if (c == 0) {
            SlotHdr* h = shdr + d;
            if (lane == 0) {
              h->p0 = g4.y;
              h->ntok = g4.z;
              h->tile = tile;
              h->phase = ph;
            }
            if (lane < 8) h->rows[lane] = my_row;
          }
          __syncwarp();
          if (lane == 0) {
            uint8_t* slot = smem + d * kSlot;
            mbar_arrive_expect_tx(&full[d], 17 * kc);
            tma_load_3d(slot, tq, 0, rowA, c * (kc / 256), &full[d], pol);
            tma_load_3d(slot + 16 * (kc / 2), tq, 0, rowB, c * (kc / 256), &full[d], pol);
            uint8_t* sdst = slot + 16 * kc;
            if (scale_tma) {
              tma_load_3d(sdst, ts, 0, rowA, c * (kc / 512), &full[d], pol);
              tma_load_3d(sdst + kc / 2, ts, 0, rowB, c * (kc / 512), &full[d], pol);
            } else {  // one chunk: 16 rows' scales are contiguous
              bulk_g2s(sdst, sbase + (size_t)rowA * (K / 32), kc / 2, &full[d]);
              bulk_g2s(sdst + kc / 2, sbase + (size_t)rowB * (K / 32), kc / 2, &full[d]);
            }
          }
          ++seq;
          if (!waited && seq >= D) {
            pdl_wait();
            pdl_trigger();
            waited = true;
          }
        }
      }
    }
    if (!waited) {
      pdl_wait();
      pdl_trigger();
    }
    // drain: no copy may still be in flight when this warp leaves
    if (lane == 0)
      for (int s = max(0, seq - D); s < seq; ++s) mbar_wait(&full[s % D], (s / D) & 1, a.st, 42);
    return;
  }

  pdl_wait();
  pdl_trigger();
  const int ng = min(*a.n_groups, kMaxTab);
  const int n_gu = ng * tiles_gu, n_dn = ng * tiles_dn;

  if (warp == kAProd) {
    // ------------------------------ activation producer ------------------------------
    int4 g0 = make_int4(0, 0, 0, 0), g1 = g0;
    if (lane < ng) g0 = a.groups[lane];
    if (lane + 32 < ng) g1 = a.groups[lane + 32];
    const Seq sg = stage_seq(n_gu), sd = stage_seq(n_dn);
    const bool has_gu = sg.count() > 0;
    bool ok = true;
    // x_lat: all T rows, once
    if (has_gu) {
      if (lane == 0) mbar_arrive_expect_tx(xfull, (uint32_t)a.T * L * 2);
      __syncwarp();
      if (lane < a.T)
        for (int k0 = 0; k0 < L; k0 += 8192)
          bulk_g2s(region + lane * pl.prow_x + k0 * 2, a.x_lat + (size_t)lane * L + k0, min(8192, L - k0) * 2, xfull);
    }
    // h panels of the down groups, each once every CTA has written that group's h rows
    int dseq = 0;
    {
      int cur = -1;
      for (int it = sd.first; it < sd.end && ok; it += sd.step) {
        const int grp = it / tiles_dn;
        if (grp == cur) continue;
        cur = grp;
        const int4 v = grp < 32 ? g0 : g1;
        const int p0 = __shfl_sync(0xffffffffu, v.y, grp & 31), ntok = __shfl_sync(0xffffffffu, v.z, grp & 31);
        const int pb = dseq % NPd;
        int good = 1;
        if (lane == 0) {
          // this CTA's own gate/up items first (no device-memory polling meanwhile), then the group's
          if (dseq == 0 && has_gu) good = mbar_wait_sleep(gudone, 0, a.st, 54, 256);
          if (good) good = counter_wait(a.ctr + grp, tiles_gu, a.st, 43);
          fence_proxy_async_global();
          // the x_lat rows share the region: the first panel waits until the consumers released them
          if (good && dseq == 0 && has_gu) good = mbar_wait(xempty, 0, a.st, 44);
          if (good && dseq >= NPd) good = mbar_wait(&pempty[pb], ((dseq / NPd) & 1) ^ 1, a.st, 45);
        }
        ok = __shfl_sync(0xffffffffu, good, 0) != 0;
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&pfull[pb], (uint32_t)ntok * I * 2);
        __syncwarp();
        uint8_t* panel = region + pb * G * pl.prow_h;
        if (lane < ntok)
          for (int k0 = 0; k0 < I; k0 += 8192)
            bulk_g2s(panel + lane * pl.prow_h + k0 * 2, a.h + (size_t)(p0 + lane) * I + k0, min(8192, I - k0) * 2,
                     &pfull[pb]);
        ++dseq;
      }
    }
    if (lane == 0) {
      if (has_gu) mbar_wait(xfull, 0, a.st, 46);
      for (int s = max(0, dseq - NPd); s < dseq; ++s) mbar_wait(&pfull[s % NPd], (s / NPd) & 1, a.st, 47);
    }
    return;
  }

  if (warp == kEpi) {
    // ------------------------------ epilogue ------------------------------
    const int g = lane >> 2, q = lane & 3;
    const Seq eg = stage_seq(n_gu);
    const int n_my_gu = eg.count();
    const int nitems = n_my_gu + stage_seq(n_dn).count();
    // group of this CTA's gate/up item j + 1 (for the per-group counts)
    auto next_grp = [&](int jj) { return (eg.first + (jj + 1) * eg.step) / tiles_gu; };
    int gcount = 0;
    for (int j = 0; j < nitems; ++j) {
      const int pb = j & 1;
      if (!mbar_wait(&rfull[pb], (j >> 1) & 1, a.st, 48)) break;
      const ItemHdr* h = ihdr + pb;
      const int p0 = h->p0, ntok = h->ntok, tile = h->tile, ph = h->phase, grp = h->grp;
      if (ph == PH_GATEUP) ++gcount;
      int aexp[G], arow[G];
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        aexp[jj] = h->aexp[jj];
        arow[jj] = h->rows[jj];
      }
      const float* rb = red + pb * kQ * kPart;
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
            for (int w = 1; w < kQ; ++w) t += rb[w * kPart + o];
            acc[m][hh][v] = t;
          }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[pb]);
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
            r_tok = arow[jj];
          }
        if (tok < ntok) {
          const float inv = ldexpf(1.0f, -e_tok);
          if (ph == PH_GATEUP) {
            const int p = p0 + tok;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const float gv = acc[m][0][v] * inv, uv = acc[m][1][v] * inv;
              a.h_out[(size_t)p * I + tile * 16 + m * 8 + g] = f32_to_bf16_bits(gv / (1.0f + expf(-gv)) * uv);
            }
          } else {
            float* yr = a.y_out + (size_t)r_tok * L + tile * kRows;
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
      if (ph == PH_DOWN) {
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
            if (jj == tok) r_tok = arow[jj];
          if (g == 0 && tok < ntok) a.ssq_out[(size_t)r_tok * (L / kRows) + tile] = sv;
        }
      }
      if (ph == PH_GATEUP && (j + 1 == n_my_gu || grp != next_grp(j))) {
        // this CTA's h rows of the group are written: count them for the group (release)
        __threadfence();
        __syncwarp();
        if (lane == 0) counter_add_release(a.ctr + grp, gcount);
        gcount = 0;
      }
      if (ph == PH_GATEUP && j + 1 == n_my_gu && lane == 0) mbar_arrive(gudone);

    }
    if (a.zb) {
      // this CTA's down rows (if any) are written: count the CTA for the z step (release)
      __threadfence();
      __syncwarp();
      if (lane == 0) counter_add_release(a.ctr + 64, 1);
    }
    return;
  }

  // -------------------------------- consumers --------------------------------
  const int g = lane >> 2, q = lane & 3;
  const int lm = lane >> 3, rr = lane & 7;
  const Seq sg = stage_seq(n_gu), sd = stage_seq(n_dn);
  int seq = 0, j = 0, dseq = 0, nsync = 0;
  bool alive = true;
  for (int ph = 0; ph < 2 && alive; ++ph) {
    const Seq r = ph == PH_GATEUP ? sg : sd;
    if (r.count() == 0) continue;
    const int tiles = ph == PH_GATEUP ? tiles_gu : tiles_dn;
    const int K = ph == PH_GATEUP ? L : I;
    const int kc = K <= kKC ? K : kKC, nch = K / kc, nplanes = kc / 256;
    const bool scale_tma = (kc % 512) == 0;
    // per m-tile: byte offset of this lane's ldmatrix box and its row in the box
    uint32_t box_off[2];
    int row_in_box[2];
    // scale rows of this lane: [m][lo/hi] = (box, row)
    int sbox[2][2], srow[2][2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      if (ph == PH_GATEUP) {
        box_off[m] = (lm & 1) * 16 * (kc / 2);  // gate box (lo) / up box (hi)
        row_in_box[m] = m * 8 + rr;
        sbox[m][0] = 0;
        sbox[m][1] = 1;
        srow[m][0] = srow[m][1] = m * 8 + g;
      } else {
        box_off[m] = m * 16 * (kc / 2);
        row_in_box[m] = (lm & 1) * 8 + rr;
        sbox[m][0] = sbox[m][1] = m;
        srow[m][0] = g;
        srow[m][1] = g + 8;
      }
    }
    if (ph == PH_GATEUP) {
      // all T rows of x_lat, converted once
      if (!mbar_wait(xfull, 0, a.st, 49)) break;
      if (!convert_rows(region, pl.prow_x, a.T, L, smax, texp, warp, lane, cbar, nsync, a.st)) break;
    }
    int cur = -1, pbuf = 0;
    int p0 = 0, ntok = 0, tile = 0;
    int arow[G], aexp[G];
#pragma unroll
    for (int jj = 0; jj < G; ++jj) arow[jj] = aexp[jj] = 0;
    uint32_t act_row = 0;
    for (int it = r.first; it < r.end && alive; it += r.step, ++j) {
      const int grp = it / tiles;
      float acc[2][2][NV];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int v = 0; v < NV; ++v) acc[m][h][v] = 0.f;
      for (int c = 0; c < nch; ++c) {
        const int d = seq % D;
        const uint32_t par = (seq / D) & 1;
        ++seq;
        if (!mbar_wait(&full[d], par, a.st, 50)) {
          alive = false;
          break;
        }
        if (c == 0) {
          const SlotHdr* hd = shdr + d;
          p0 = hd->p0;
          ntok = hd->ntok;
          tile = hd->tile;
#pragma unroll
          for (int jj = 0; jj < G; ++jj) arow[jj] = hd->rows[jj];
          if (grp != cur) {
            cur = grp;
            if (ph == PH_GATEUP) {
              // this lane's token column g: x_lat row of route row arow[g]
              int tok = 0, e = 0;
#pragma unroll
              for (int jj = 0; jj < G; ++jj)
                if (jj == (g < ntok ? g : 0)) tok = arow[jj] / k;
              act_row = smem_u32(region) + tok * pl.prow_x + q * 16;
#pragma unroll
              for (int jj = 0; jj < G; ++jj) {
                e = jj < ntok ? texp[arow[jj] / k] : 0;
                aexp[jj] = e;
              }
            } else {
              pbuf = dseq % NPd;
              if (!mbar_wait(&pfull[pbuf], (dseq / NPd) & 1, a.st, 51)) {
                alive = false;
                break;
              }
              uint8_t* panel = region + pbuf * G * pl.prow_h;
              if (!convert_rows(panel, pl.prow_h, ntok, I, smax, pexp + pbuf * 8, warp, lane, cbar, nsync, a.st)) {
                alive = false;
                break;
              }
#pragma unroll
              for (int jj = 0; jj < G; ++jj) aexp[jj] = jj < ntok ? pexp[pbuf * 8 + jj] : 0;
              act_row = smem_u32(panel) + (g < ntok ? g : 0) * pl.prow_h + q * 16;
              ++dseq;
            }
          }
        }
        const uint8_t* slot = smem + d * kSlot;
        const uint32_t cbase = smem_u32(slot);
        const uint8_t* sreg = slot + 16 * kc;
        const uint32_t act_addr = act_row + c * kc * 2;
        // a chunk has at most 8 planes: warp p takes plane p
        const int p = warp;
        const bool mine = p < nplanes;
        uint32_t wq[4][2][4];
        uint2 sw[2][2];
        bool special = false;
        if (mine) {
          plane_load(cbase, box_off, row_in_box, lm, p, wq);
#pragma unroll
          for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint8_t* src = scale_tma
                                       ? sreg + sbox[m][hh] * (kc / 2) + ((p >> 1) * 16 + srow[m][hh]) * 16 + (p & 1) * 8
                                       : sreg + sbox[m][hh] * (kc / 2) + srow[m][hh] * (kc / 32) + p * 8;
              sw[m][hh] = *reinterpret_cast<const uint2*>(src);
              special |= has_special_byte(sw[m][hh].x) | has_special_byte(sw[m][hh].y);
            }
        }
        // the slot's bytes are in registers: release it before the arithmetic
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[d]);
        if (mine) {
          if (__any_sync(0xffffffffu, special))
            plane_mx<NV, true>(wq, act_addr, sw, acc, p);
          else
            plane_mx<NV, false>(wq, act_addr, sw, acc, p);
        }
      }
      if (!alive) break;
      const bool last_of_group = (it + r.step >= r.end) || ((it + r.step) / tiles != grp);
      if (ph == PH_DOWN && last_of_group) {
        // panel reads and this warp's conversion writes come before the next bulk copy into it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[pbuf]);
      }
      // partials to the epilogue warp (double-buffered by item parity)
      const int pb = j & 1;
      if (!mbar_wait(&rempty[pb], ((j >> 1) & 1) ^ 1, a.st, 52)) {
        alive = false;
        break;
      }
      float* rbuf = red + (pb * kQ + warp) * kPart;
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
          h->phase = ph;
          h->grp = grp;
        }
        if (lane < G) {
#pragma unroll
          for (int jj = 0; jj < G; ++jj)
            if (jj == lane) {
              h->aexp[lane] = aexp[jj];
              h->rows[lane] = arow[jj];
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull[pb]);
    }
    if (ph == PH_GATEUP) {
      // the x_lat rows (and this warp's conversion writes) come before the h panels loaded over them
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(xempty);
    }
  }
  if (!alive || !a.zb) return;
  // ---------------- post_expert_norm per route row and the fp32 weighted sum ----------------
  // z[t][l] = sum_j w[t][j] * ((y[t*k+j][l] * rinv[t*k+j]) * g[e][l]), j in order, for this CTA's
  // 32-column slices of the latent width, once every CTA has written its down rows.
  const int nsl = L / 32;
  if ((int)blockIdx.x >= nsl) return;
  {
    int good = 1;
    if (lane == 0) good = counter_wait(a.ctr + 64, gridDim.x, a.st, 55);
    if (!__shfl_sync(0xffffffffu, good, 0)) return;
  }
  const int R = a.rows, tiles = L / 32;
  // 1/rms of every route row from its per-tile sums of squares (lanes over tiles, then a tree)
  for (int r = warp; r < R; r += kQ) {
    float sq = 0.f;
    for (int i = lane; i < tiles; i += 32) sq += __ldcg(a.ssq_out + (size_t)r * tiles + i);
    sq = warp_sum(sq);
    if (lane == 0) s_rinv[r] = 1.0f / sqrtf(sq / (float)L + a.eps);
  }
  if (!consumers_meet(cbar, nsync, a.st, lane)) return;
  const int tid = warp * 32 + lane;
  for (int sl = blockIdx.x; sl < nsl; sl += gridDim.x) {
    const int l = sl * 32 + (tid & 31);
    for (int t = tid >> 5; t < a.T; t += kQ) {
      float z = 0.f;
      for (int jj = 0; jj < k; ++jj) {
        const int r = t * k + jj;
        int e = a.topk_idx[r];
        if (e < 0 || e >= a.n_experts) {
          set_error(a.st, LMOE_EDEVICE_CHECK, 102);
          e = 0;
        }
        const float yv = __ldcg(a.y_out + (size_t)r * L + l);
        const float gv = bf16_bits_to_f32(a.norm_g[(size_t)e * L + l]);
        const float yh = __fmul_rn(__fmul_rn(yv, s_rinv[r]), gv);
        z = __fadd_rn(z, __fmul_rn(a.topk_w[r], yh));
      }
      a.zb[(size_t)t * L + l] = f32_to_bf16_bits(z);
    }
  }
}

template <int G, int NV>
int launch_fused(const FusedExpertArgs& a, cudaStream_t s, int num_sms) {
  auto kern = fused_experts_kernel<G, NV>;
  constexpr int kSmemMax = 232448;
  const int L = a.latent, I = a.inter;
  Plan pl{};
  pl.G = G;
  pl.NV = NV;
  pl.prow_x = L * 2 + 64;  // padded rows: conflict-free 16-byte loads
  pl.prow_h = I * 2 + 64;
  const int rows_h = min(G, a.T);  // a token picks an expert once: at most T rows per group
  const int fixed = 2 * kQ * pl.kpart() * 4 + kQ * 8 * 4 + 24 * 4 + kMaxSlots * (int)sizeof(SlotHdr) +
                    2 * (int)sizeof(ItemHdr) + (2 * kMaxSlots + 12) * 8 + 64 * 4 + 1024 + 256;
  auto region_for = [&](int npd) { return ((max(a.T * pl.prow_x, npd * G * pl.prow_h) + 127) / 128) * 128; };
  (void)rows_h;
  pl.NPd = 2;
  pl.region = region_for(2);
  pl.D = min(kMaxSlots, (kSmemMax - fixed - pl.region) / kSlot);
  if (pl.D < 4) {
    pl.NPd = 1;
    pl.region = region_for(1);
    pl.D = min(kMaxSlots, (kSmemMax - fixed - pl.region) / kSlot);
  }
  if (pl.D < 2) return LMOE_EUNSUPPORTED;
  const int smem = pl.D * kSlot + pl.region + fixed;
  static int attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_done[dev & 63] < smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return LMOE_ECUDA;
    attr_done[dev & 63] = smem;
  }
  CUtensorMap tq[2], ts[2];
  for (int ph = 0; ph < 2; ++ph) {
    const int K = ph == 0 ? L : I;
    const int kc = K <= kKC ? K : kKC;
    const uint64_t rows_total = (uint64_t)a.n_experts * (ph == 0 ? 2 * I : L);
    const uint8_t* q = ph == 0 ? a.w13_q : a.w2_q;
    const uint8_t* sc = ph == 0 ? a.w13_s : a.w2_s;
    {
      const uint64_t dims[3] = {128, rows_total, (uint64_t)K / 256};
      const uint64_t strides[2] = {(uint64_t)K / 2, 128};
      const uint32_t box[3] = {128, 16, (uint32_t)(kc / 256)};
      if (get_tmap(&tq[ph], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return LMOE_ECUDA;
    }
    if (kc % 512 == 0) {
      // scales as {16 B, rows, K/512}: 16 blocks of one row per 16-byte line
      const uint64_t dims[3] = {16, rows_total, (uint64_t)K / 512};
      const uint64_t strides[2] = {(uint64_t)K / 32, 16};
      const uint32_t box[3] = {16, 16, (uint32_t)(kc / 512)};
      if (get_tmap(&ts[ph], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, sc, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
        return LMOE_ECUDA;
    } else {
      ts[ph] = tq[ph];  // unused: one chunk copies the scales with a bulk copy
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.early ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, tq[0], ts[0], tq[1], ts[1], pl);
  if (e != cudaSuccess && cfg.numAttrs == 2) {
    // no programmatic overlap for a cooperative launch here: launch it after its predecessor
    (void)cudaGetLastError();
    FusedExpertArgs b = a;
    b.early = 0;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, b, tq[0], ts[0], tq[1], ts[1], pl);
  }
  return e == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

}  // namespace

int launch_fused_experts(const FusedExpertArgs& a, cudaStream_t s, int num_sms) {
  if (a.rows > kMaxTab || a.T > 8 || a.T < 1) return LMOE_EUNSUPPORTED;
  if (a.latent > 8192 || a.inter > 8192) return LMOE_EUNSUPPORTED;
  if (a.T == 1) return launch_fused<1, 1>(a, s, num_sms);
  return launch_fused<8, 2>(a, s, num_sms);
}

}  // namespace lmoe
