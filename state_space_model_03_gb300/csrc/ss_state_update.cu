// One decode step of the selective scan (section 4.4 of the page "PaddleNLP
// Kernel 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南" lists the
// operator as "selective_state_update"; its operands are the section 4.1 scan
// at a single time step): for every (batch, channel, state)
//   dt = softplus(delta + delta_bias); state = exp(dt A) state + dt B u;
//   out = (sum_n C state + D u) silu(z).
//
// The step is bound by HBM traffic: the fp32 state is read and written once
// (8 bytes per (batch, channel, state)); everything else is a few bytes per
// (batch, channel) or per (batch, group). LPC adjacent lanes own one channel,
// 4 * Q states each (16-byte state and A accesses, so a warp streams 32/LPC
// contiguous state rows), and reduce y with shuffles. The grid
// is (channel tiles, batch rows): no integer division in the index math, which
// measured as the limit of a flat-index version.
#include "ss_dispatch.h"
#include "ss_fwd_kernel.cuh"

namespace ssk {

namespace {

// Four 16-bit (or fp32) values of one lane as floats.
template <typename BCT>
__device__ __forceinline__ void load4(const BCT *src, bool vec, int valid, float (&v)[4]) {
  if constexpr (sizeof(BCT) == 4) {
    if (vec && valid == 4) {
      const float4 q = *reinterpret_cast<const float4 *>(src);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
      return;
    }
  } else {
    if (vec && valid == 4) {
      const uint2 q = *reinterpret_cast<const uint2 *>(src);
      const float2 a = unpack2<BCT>(q.x), b = unpack2<BCT>(q.y);
      v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
      return;
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = k < valid ? to_f<BCT>(src[k]) : 0.f;
}

// state' = exp(dt A) state + dt B u for the lane's 4 states; returns its part of y.
__device__ __forceinline__ float step4(float dt, float w, const float (&a)[4], const float (&bv)[4],
                                       const float (&cv)[4], float (&x)[4]) {
  float yp = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[k] = fmaf(ex2(dt * (a[k] * kLog2e)), x[k], w * bv[k]);
    yp = fmaf(cv[k], x[k], yp);
  }
  return yp;
}

// ---------------------------------------------------------------------------
// General kernel
// ---------------------------------------------------------------------------
template <typename T, typename BCT, int LPC, int Q>  // LPC lanes per channel, 4 * Q states per lane
__global__ void __launch_bounds__(256) ss_state_update_kernel(const __grid_constant__ SUParams p) {
  constexpr int CPB = 256 / LPC;  // channels per CTA
  const int j = threadIdx.x % LPC;
  const int n0 = 4 * Q * j;
  // grid: (channel tiles, batch rows, batch rows / 65535); no integer division
  const int dc = blockIdx.x * CPB + threadIdx.x / LPC;
  const int bc = blockIdx.y + gridDim.y * blockIdx.z;
  const bool active = dc < p.dim && bc < p.batch;
  const int b = active ? bc : 0, d = active ? dc : 0;
  float uu = 0.f, dt = 0.f, zz = 0.f;
  if (active) {
    uu = to_f<T>(static_cast<const T *>(p.u)[b * p.su[0] + d * p.su[1]]);
    const float v = to_f<T>(static_cast<const T *>(p.delta)[b * p.sd[0] + d * p.sd[1]]) +
                    (p.has_bias ? p.bias[d] : 0.f);
    dt = p.softplus ? softplus_t<T>(v) : v;
    if (p.has_z) zz = to_f<T>(static_cast<const T *>(p.z)[b * p.sz[0] + d * p.sz[1]]);
  }
  float *srow = p.state + b * p.sst[0] + (long long)d * p.sst[1] + n0;
  const float *arow = p.A + (long long)d * p.sA[0] + n0;
  const BCT *brow, *crow;
  if (p.fixed) {
    brow = static_cast<const BCT *>(p.B) + (long long)d * p.sB[0] + n0;
    crow = static_cast<const BCT *>(p.C) + (long long)d * p.sC[0] + n0;
  } else {
    const int g = p.dpg == p.dim ? 0 : d / p.dpg;
    brow = static_cast<const BCT *>(p.B) + b * p.sB[0] + (long long)g * p.sB[1] + n0;
    crow = static_cast<const BCT *>(p.C) + b * p.sC[0] + (long long)g * p.sC[1] + n0;
  }
  float x[Q][4], a[Q][4], bv[Q][4], cv[Q][4];
  int valid[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int r = p.dstate - n0 - 4 * q;
    valid[q] = !active ? 0 : (r < 0 ? 0 : (r > 4 ? 4 : r));
    load4<float>(srow + 4 * q, p.vec != 0, valid[q], x[q]);
    load4<float>(arow + 4 * q, p.avec != 0, valid[q], a[q]);
    load4<BCT>(brow + 4 * q, p.bcvec != 0, valid[q], bv[q]);
    load4<BCT>(crow + 4 * q, p.bcvec != 0, valid[q], cv[q]);
  }
  float yp = 0.f;
#pragma unroll
  for (int q = 0; q < Q; ++q) yp += step4(dt, dt * uu, a[q], bv[q], cv[q], x[q]);
#pragma unroll
  for (int o = LPC / 2; o > 0; o >>= 1) yp += __shfl_xor_sync(0xffffffffu, yp, o);
  if (!active) return;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    if (p.vec && valid[q] == 4) {
      *reinterpret_cast<float4 *>(srow + 4 * q) = make_float4(x[q][0], x[q][1], x[q][2], x[q][3]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (k < valid[q]) srow[4 * q + k] = x[q][k];
    }
  }
  if (j == 0) {
    float y = yp + (p.has_D ? p.D[d] : 0.f) * uu;
    if (p.has_z) y *= silu_t<T>(zz);
    static_cast<T *>(p.out)[b * p.so[0] + d * p.so[1]] = from_f<T>(y);
  }
}

template <typename T, typename BCT>
const void *pick(int lpc, int q) {
  if (q == 4) {
    switch (lpc) {
      case 1: return (const void *)&ss_state_update_kernel<T, BCT, 1, 4>;
      case 2: return (const void *)&ss_state_update_kernel<T, BCT, 2, 4>;
      default: return (const void *)&ss_state_update_kernel<T, BCT, 4, 4>;
    }
  }
  if (q == 2) {
    switch (lpc) {
      case 1: return (const void *)&ss_state_update_kernel<T, BCT, 1, 2>;
      case 2: return (const void *)&ss_state_update_kernel<T, BCT, 2, 2>;
      case 4: return (const void *)&ss_state_update_kernel<T, BCT, 4, 2>;
      default: return (const void *)&ss_state_update_kernel<T, BCT, 8, 2>;
    }
  }
  switch (lpc) {
    case 1: return (const void *)&ss_state_update_kernel<T, BCT, 1, 1>;
    case 2: return (const void *)&ss_state_update_kernel<T, BCT, 2, 1>;
    case 4: return (const void *)&ss_state_update_kernel<T, BCT, 4, 1>;
    case 8: return (const void *)&ss_state_update_kernel<T, BCT, 8, 1>;
    default: return (const void *)&ss_state_update_kernel<T, BCT, 16, 1>;
  }
}

}  // namespace

const void *state_update_kernel(int in_dtype, bool bc_f32, int lpc, int q) {
  switch (in_dtype) {
    case 0: return pick<float, float>(lpc, q);
    case 1: return bc_f32 ? pick<__half, float>(lpc, q) : pick<__half, __half>(lpc, q);
    default: return bc_f32 ? pick<__nv_bfloat16, float>(lpc, q) : pick<__nv_bfloat16, __nv_bfloat16>(lpc, q);
  }
}

}  // namespace ssk
