// The sandwich block around the layer: y = x + post_norm(F(pre_norm(x))).
//
// "Soporte de dia 0 para Muse Spark Open en vLLM", section "Normalizacion en
// sandwich": a norm before the mixture-of-experts block and one after it.
// Section "Nvidia" of the same page: the router GEMM is fed by the fp32
// output of the pre-norm, and norm, gating and residual work is fused.
//
// Both norms are RMSNorm over the hidden width: rinv = 1/sqrt(sum(x^2)/H +
// eps), out = (x * rinv) * g with a bf16 gain per column (the same form as
// post_expert_norm).  Products and sums use the _rn intrinsics so that no
// multiply-add is contracted: each value is rounded exactly where the plain
// fp32 expression rounds it.
#include "common.cuh"
#include "kernels.cuh"

namespace lmoe {

namespace {

// Sum of squares of one bf16 row of width H (a multiple of 8) by 256 threads:
// each thread adds its 8-element pieces in order, then a fixed tree over
// lanes and warps.  Every thread gets the total.
__device__ __forceinline__ float row_sumsq(const uint16_t* __restrict__ row, int H, float* s_red) {
  float ss = 0.f;
  for (int c = threadIdx.x * 8; c < H; c += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = bf16_bits_to_f32(w[i] & 0xffffu), b = bf16_bits_to_f32(w[i] >> 16);
      ss = __fadd_rn(ss, __fmul_rn(a, a));
      ss = __fadd_rn(ss, __fmul_rn(b, b));
    }
  }
  ss = warp_sum(ss);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_red[warp] = ss;
  __syncthreads();
  float t = s_red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) t += s_red[w];
  return t;
}

__device__ __forceinline__ float rms_inv(float ss, int H, float eps) {
  return __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps)));
}

}  // namespace

// Pre-norm, one CTA of 256 threads per token:
//   n_bf16[t][c] = bf16((x * rinv) * g)     the pooler's input
//   rinv[t]                                  the router scales its dot products by it
//   u_split[t] = (u1 | u2), u = x * g        when the router runs on the tensor cores:
// u is a product of two bf16 values, exact in fp32 with at most 16 significant
// bits, so u1 (its top 8 bits, by truncation) and u2 = u - u1 are both exact
// bf16 values.  The router then computes rinv * (u . w), which differs from
// n . w only by the rounding of n.
__global__ void __launch_bounds__(256) prenorm_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ g,
                                                      float eps, int H, uint16_t* __restrict__ n_bf16,
                                                      float* __restrict__ rinv_out,
                                                      uint16_t* __restrict__ u_split) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_red[8];
  const int t = blockIdx.x;
  const uint16_t* xr = x + (size_t)t * H;
  const float rinv = rms_inv(row_sumsq(xr, H, s_red), H, eps);
  if (threadIdx.x == 0) rinv_out[t] = rinv;
  for (int c = threadIdx.x * 8; c < H; c += 256 * 8) {
    const uint4 xv = *reinterpret_cast<const uint4*>(xr + c);
    const uint4 gv = *reinterpret_cast<const uint4*>(g + c);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t nb[4], hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t packn = 0, packh = 0, packl = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float xv1 = bf16_bits_to_f32((xw[i] >> (16 * h)) & 0xffffu);
        const float gv1 = bf16_bits_to_f32((gw[i] >> (16 * h)) & 0xffffu);
        packn |= (uint32_t)f32_to_bf16_bits(__fmul_rn(__fmul_rn(xv1, rinv), gv1)) << (16 * h);
        const float u = __fmul_rn(xv1, gv1);
        const uint32_t u1 = __float_as_uint(u) >> 16;
        packh |= u1 << (16 * h);
        packl |= (uint32_t)f32_to_bf16_bits(__fsub_rn(u, __uint_as_float(u1 << 16))) << (16 * h);
      }
      nb[i] = packn;
      hi[i] = packh;
      lo[i] = packl;
    }
    *reinterpret_cast<uint4*>(n_bf16 + (size_t)t * H + c) = make_uint4(nb[0], nb[1], nb[2], nb[3]);
    if (u_split) {
      uint16_t* ur = u_split + (size_t)t * 2 * H;
      *reinterpret_cast<uint4*>(ur + c) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(ur + H + c) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
}

// Post-norm and residual, one CTA of 256 threads per token:
//   y[t][c] = bf16(x[t][c] + (out[t][c] * rinv) * g[c]),  rinv from out's row.
// y may alias x (an in-place update of the residual stream): each element is
// read before the same thread writes it, and no other thread touches it.
__global__ void __launch_bounds__(256) postnorm_residual_kernel(const uint16_t* __restrict__ out,
                                                                const uint16_t* x, const uint16_t* __restrict__ g,
                                                                float eps, int H, uint16_t* y) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_red[8];
  const int t = blockIdx.x;
  const uint16_t* orow = out + (size_t)t * H;
  const float rinv = rms_inv(row_sumsq(orow, H, s_red), H, eps);
  for (int c = threadIdx.x * 8; c < H; c += 256 * 8) {
    const uint4 ov = *reinterpret_cast<const uint4*>(orow + c);
    const uint4 xv = *reinterpret_cast<const uint4*>(x + (size_t)t * H + c);
    const uint4 gv = *reinterpret_cast<const uint4*>(g + c);
    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w},
                   gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t yw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t pack = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float o1 = bf16_bits_to_f32((ow[i] >> (16 * h)) & 0xffffu);
        const float x1 = bf16_bits_to_f32((xw[i] >> (16 * h)) & 0xffffu);
        const float g1 = bf16_bits_to_f32((gw[i] >> (16 * h)) & 0xffffu);
        pack |= (uint32_t)f32_to_bf16_bits(__fadd_rn(x1, __fmul_rn(__fmul_rn(o1, rinv), g1))) << (16 * h);
      }
      yw[i] = pack;
    }
    *reinterpret_cast<uint4*>(y + (size_t)t * H + c) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
  }
}

}  // namespace lmoe
