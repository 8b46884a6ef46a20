// bf16 x bf16 -> bf16 GEMM on tcgen05 for large token counts (pooler and
// unpooler in the prefill regime): C[M][N] = bf16_rne(A[M][K] . B[N][K]^T),
// fp32 accumulation in tensor memory.
//
// "Soporte de dia 0 para Muse Spark Open en vLLM", section "MoE latente": the
// pooler (8192 -> 4096) and unpooler (4096 -> 8192) are learned projections;
// "Muse Spark Open on Gaudi 2", "Correctness": bf16 values, fp32 accumulation.
//
// Persistent CTAs walk 128 x 256 output tiles (m fastest, so CTAs in flight
// share weight tiles through L2).  Warp 0 streams 128x64 A and 256x64 B tiles
// with TMA (128-byte swizzle, K-major) into a 4-stage ring; one thread of
// warp 1 issues tcgen05.mma kind::f16 (M=128, N=256, K=16) into one of two
// TMEM accumulators (2 x 256 fp32 columns) and commits each stage back to the
// producer; warps 4-7 read the finished accumulator with tcgen05.ld (each its
// 32-lane quarter: one output row per thread), round to bf16 and store.
#include <atomic>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace lmoe {

constexpr int kTM = 128, kTN = kTcGemmN, kTK = kTcGemmK, kTStages = 4;
constexpr int kTAbytes = kTM * kTK * 2;  // 16 KB
constexpr int kTBbytes = kTN * kTK * 2;  // 32 KB

__global__ void __launch_bounds__(256, 1)
    tc_gemm_bf16_kernel(const TcGemmArgs a, const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kTStages * kTAbytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kTStages * kTBbytes);
  uint64_t* empty = full + kTStages;
  uint64_t* accf = empty + kTStages;  // accumulator ready for the epilogue
  uint64_t* acce = accf + 2;          // accumulator drained by the epilogue
  uint64_t* done = acce + 2;          // every MMA of this CTA has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 4);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();
  pdl_trigger();

  const int n_tile = a.n_tile > 0 ? a.n_tile : kTN;
  const int nsplit = a.nsplit > 1 ? a.nsplit : 1;
  const int tiles_m = (a.M + kTM - 1) / kTM, tiles_n = a.N / n_tile, tiles_mn = tiles_m * tiles_n;
  const int ntiles = tiles_mn * nsplit;
  const int nk = a.K / kTK / nsplit;  // k-blocks per tile

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    const uint64_t pol_b = policy_evict_last();
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    int issued = 0;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const int mt = t % tiles_m, nt = (t / tiles_m) % tiles_n, ks = t / tiles_mn;
      for (int kb = ks * nk; kb < (ks + 1) * nk; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1, a.st, 21)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kTAbytes + n_tile * kTK * 2);
        tma_load_2d(sA + s * kTAbytes, &tmA, (a.a_kblocks > 0 ? kb % a.a_kblocks : kb) * kTK, mt * kTM, &full[s],
                    pol_b);
        tma_load_2d(sB + s * kTBbytes, &tmB, kb * kTK, nt * n_tile, &full[s], pol_b);
        ++issued;
        if (++s == kTStages) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    // drain: the last stages' copies must land before the CTA can finish
    for (int i = 0; i < kTStages && i < issued; ++i) {
      if (--s < 0) {
        s = kTStages - 1;
        ph ^= 1;
      }
      mbar_wait(&full[s], ph, a.st, 22);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = idesc_bf16_f32(kTM, n_tile);
    int s = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      if (!mbar_wait(&acce[acc], aph ^ 1, a.st, 23)) break;
      tc_fence_after();
      const uint32_t d = tmem + acc * kTN;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(&full[s], ph, a.st, 24)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * kTAbytes), b0 = smem_u32(sB + s * kTBbytes);
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk)
          tc_mma_bf16(d, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc, (kb | kk) != 0);
        tc_commit(&empty[s]);
        if (++s == kTStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
      tc_commit(&accf[acc]);
      if (++acc == 2) {
        acc = 0;
        aph ^= 1;
      }
    }
    // every MMA issued (also those of a tile abandoned after a timeout) must
    // complete before TMEM is released
    tc_commit(done);
    mbar_wait(done, 0, a.st, 25);
  } else if (warp >= 4) {
    // ---------------- epilogue: TMEM -> bf16 -> global ----------------
    const int wq = warp - 4;  // TMEM lane quarter of this warp
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const int mt = t % tiles_m, nt = (t / tiles_m) % tiles_n, ks = t / tiles_mn;
      if (!mbar_wait(&accf[acc], aph, a.st, 26)) break;
      tc_fence_after();
      const int row = mt * kTM + wq * 32 + lane;
#pragma unroll 1
      for (int ch = 0; ch < n_tile / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(wq * 32) << 16) + acc * kTN + ch * 32, r);
        tmem_ld_wait();
        if (a.out_f32) {
          if (row < a.M) {
            float4* dst = reinterpret_cast<float4*>(a.out_f32 + ((size_t)ks * a.M + row) * a.N + nt * n_tile + ch * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                   __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
          }
          continue;
        }
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint16_t lo = f32_to_bf16_bits(__uint_as_float(r[2 * i]));
          const uint16_t hi = f32_to_bf16_bits(__uint_as_float(r[2 * i + 1]));
          o[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        if (row < a.M) {
          uint4* dst = reinterpret_cast<uint4*>(a.out + (size_t)row * a.N + nt * n_tile + ch * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          for (int j = 0; j < a.scatter_k; ++j) {
            const int p = __ldg(a.scatter_pos + (size_t)row * a.scatter_k + j);
            uint4* sd = reinterpret_cast<uint4*>(a.scatter_out + (size_t)p * a.N + nt * n_tile + ch * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) sd[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[acc]);
      if (++acc == 2) {
        acc = 0;
        aph ^= 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int launch_tc_gemm_bf16(const TcGemmArgs& a, const uint16_t* A, const uint16_t* B, cudaStream_t s, int num_sms) {
  const int n_tile = a.n_tile > 0 ? a.n_tile : kTN;
  const int nsplit = a.nsplit > 1 ? a.nsplit : 1;
  if (n_tile % 32 || n_tile > kTN || a.N % n_tile || a.K % (kTK * nsplit) || a.M < 1) return LMOE_EUNSUPPORTED;
  if (a.a_kblocks > 0 && (a.K / kTK) % a.a_kblocks) return LMOE_EUNSUPPORTED;
  constexpr int smem = kTStages * (kTAbytes + kTBbytes) + 1024 + 256;
  static_assert(smem <= 232448, "shared memory budget");
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LMOE_ECUDA;
  if (!(attr_done.load() >> (dev & 63) & 1ull)) {
    if (cudaFuncSetAttribute(tc_gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return LMOE_ECUDA;
    attr_done.fetch_or(1ull << (dev & 63));
  }
  CUtensorMap ta, tb;
  {
    const uint64_t ka = a.a_kblocks > 0 ? (uint64_t)a.a_kblocks * kTK : (uint64_t)a.K;  // A's own width
    const uint64_t dims[2] = {ka, (uint64_t)a.M};
    const uint64_t strides[1] = {ka * 2};
    const uint32_t box[2] = {kTK, kTM};
    if (get_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return LMOE_ECUDA;
  }
  {
    const uint64_t dims[2] = {(uint64_t)a.K, (uint64_t)a.N};
    const uint64_t strides[1] = {(uint64_t)a.K * 2};
    const uint32_t box[2] = {kTK, (uint32_t)n_tile};
    if (get_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return LMOE_ECUDA;
  }
  const int ntiles = ((a.M + kTM - 1) / kTM) * (a.N / n_tile) * nsplit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntiles < num_sms ? ntiles : num_sms);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_bf16_kernel, a, ta, tb) == cudaSuccess ? LMOE_OK : LMOE_ECUDA;
}

}  // namespace lmoe
