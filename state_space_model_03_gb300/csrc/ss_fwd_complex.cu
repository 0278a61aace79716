// Complex-A selective-scan forward (section 4.1 of the page "PaddleNLP Kernel
// 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南": A "real or complex").
// Per (batch b, channel d, state n, step t), with complex A and state x:
//   a = exp(dt A) = e^{dt Re A} (cos(dt Im A) + i sin(dt Im A))
//   x = a x + dt B u,   y = Re(sum_n C x) + D u,   out = y silu(z)
//
// Schedule. A thread owns one (batch, channel, state) recurrence (two fp32
// registers); the 16 lanes of a half-warp hold the states of one channel (with
// more than 16 states a lane loops over n = j, j + 16, ...). The row is walked
// in segments of kT steps: lane j prepares step t0 + j of the channel (dt,
// dt u, the gate) into shared memory, every lane walks the segment for its
// state(s) accumulating its part of y per step, and the 16 lanes' terms pass
// through shared memory so that lane j sums step t0 + j's, gates and stores it.
// The lane's global inputs of the next segment are fetched before the current
// one is walked.
// There is no cross-warp communication, so warps run independently.
#include "ss_dispatch.h"
#include "ss_fwd_kernel.cuh"

namespace ssk {

namespace {

constexpr int kW = 8;         // warps per CTA
constexpr int kT = 16;        // steps per segment
constexpr int kCPC = 2 * kW;  // channels per CTA

constexpr int kYRow = kT + 4;  // padded row of the per-state y terms (conflict-free 16-byte stores)

// sin and cos of th + lo: th = k pi/2 + r (Cody-Waite reduction with fused
// multiply-adds against a three-part split of pi/2), r += lo, |r| <= pi/4 + |lo|,
// then the Taylor series of sin r to r^9 and of cos r to r^8 (truncation below
// 4e-8) and the quadrant k mod 4. lo is the rounding error of the angle's
// product (th + lo = dt Im A exactly), so the phase keeps fp32 accuracy at
// large angles; accurate to a few fp32 ulps for |th| up to ~1e5.
// FAST (16-bit inputs, whose outputs are rounded to 8 or 11 bits): the reduced
// sin and cos come from the MUFU approximations instead of the series
// (absolute error ~1e-6 on |r| <= pi/4).
__device__ __forceinline__ float sin_approx(float x) {
  float y;
  asm("sin.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float cos_approx(float x) {
  float y;
  asm("cos.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
template <bool FAST>
__device__ __forceinline__ void sincos_rr(float th, float lo, float &sn, float &cs) {
  if constexpr (FAST) {
    // sin.approx / cos.approx keep an absolute error near 2^-21 for |x| up to
    // 100 pi on their own, so angles in that range skip the reduction
    if (fabsf(th + lo) <= 314.0f) {
      sn = sin_approx(th + lo);
      cs = cos_approx(th + lo);
      return;
    }
  }
  const float k = rintf(th * 0.636619772367581343f);  // 2 / pi
  float r = fmaf(-k, 1.5707963705062866f, th);
  r = fmaf(-k, -4.371138828673793e-08f, r);
  r = fmaf(-k, -1.7763568394002505e-15f, r);
  r += lo;
  float s, c;
  if constexpr (FAST) {
    s = sin_approx(r);
    c = cos_approx(r);
  } else {
    const float r2 = r * r;
    s = r * fmaf(r2, fmaf(r2, fmaf(r2, fmaf(r2, 2.7557319223985893e-06f, -1.984126984126984e-04f),
                                   8.333333333333333e-03f), -1.6666666666666666e-01f), 1.f);
    c = fmaf(r2, fmaf(r2, fmaf(r2, fmaf(r2, 2.48015873015873e-05f, -1.388888888888889e-03f),
                               4.1666666666666664e-02f), -0.5f), 1.f);
  }
  const int q = static_cast<int>(k) & 3;  // two's complement: k = -1 gives quadrant 3
  const float s1 = (q & 1) ? c : s, c1 = (q & 1) ? s : c;
  sn = (q & 2) ? -s1 : s1;
  cs = ((q + 1) & 2) ? -c1 : c1;
}

// The step of the complex path. A rotation of dt Im A radians per step turns
// a relative error of dt into a phase error that grows with |Im A|, so fp32
// inputs take softplus from the library exponential and log1p (each within a
// few ulps, against ~5e-7 for the one-MUFU form the real forward uses). 16-bit
// inputs, whose outputs are rounded to 8 or 11 bits, keep the MUFU form.
template <typename T>
__device__ __forceinline__ float softplus_cx(float v) {
  if constexpr (sizeof(T) == 4) return fmaxf(v, 0.f) + log1pf(expf(-fabsf(v)));
  else return softplus_f(v);
}

// kT values of one B/C row starting at step t: 16-byte loads when vec (the
// row is aligned and the segment complete), else element by element with
// zeros past the end.
template <typename BCT>
struct Row {
  static constexpr int kWords = kT * (int)sizeof(BCT) / 16;  // 16-byte words per segment
  uint4 w[kWords];
};
template <typename BCT>
__device__ __forceinline__ void fetch_row(const BCT *src, int t, int L, bool vec, Row<BCT> &r) {
  if (vec && t + kT <= L) {
#pragma unroll
    for (int q = 0; q < Row<BCT>::kWords; ++q) r.w[q] = reinterpret_cast<const uint4 *>(src + t)[q];
  } else {
    BCT tmp[kT];
#pragma unroll
    for (int i = 0; i < kT; ++i) tmp[i] = t + i < L ? src[t + i] : from_f<BCT>(0.f);
    memcpy(&r.w[0], tmp, sizeof(tmp));
  }
}
template <typename BCT>
__device__ __forceinline__ void unpack_row(const Row<BCT> &r, float (&v)[kT]) {
  if constexpr (sizeof(BCT) == 4) {
#pragma unroll
    for (int q = 0; q < Row<BCT>::kWords; ++q) {
      v[4 * q] = __uint_as_float(r.w[q].x);
      v[4 * q + 1] = __uint_as_float(r.w[q].y);
      v[4 * q + 2] = __uint_as_float(r.w[q].z);
      v[4 * q + 3] = __uint_as_float(r.w[q].w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < Row<BCT>::kWords; ++q) {
      const uint32_t wd[4] = {r.w[q].x, r.w[q].y, r.w[q].z, r.w[q].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = unpack2<BCT>(wd[k]);
        v[8 * q + 2 * k] = f.x;
        v[8 * q + 2 * k + 1] = f.y;
      }
    }
  }
}

template <typename T, typename BCT, bool FIXED, int SPL>
__global__ void __launch_bounds__(kW * 32, 2) ss_fwd_complex_kernel(const __grid_constant__ CxParams p) {
  __shared__ __align__(16) float s_ch[kCPC][2][kT];        // dt, dt*u per channel and step
  __shared__ __align__(16) float s_y[kCPC][16][kYRow];     // per-state y terms of the segment

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, j = lane & 15;
  const int chl = warp * 2 + half;
  const int N = p.dstate, L = p.seqlen;
  const int g = blockIdx.x / p.tiles;
  const int dl = (blockIdx.x - g * p.tiles) * kCPC + chl;
  const bool active = dl < p.dpg;
  const int d = g * p.dpg + (active ? dl : 0);
  const int b = blockIdx.y + gridDim.y * blockIdx.z;
  if (b >= p.batch) return;  // the last batch slab of a folded grid (whole CTA)

  const T *u_row = static_cast<const T *>(p.u) + b * p.su[0] + d * p.su[1];
  const T *dl_row = static_cast<const T *>(p.delta) + b * p.sd[0] + d * p.sd[1];
  const T *z_row = p.has_z ? static_cast<const T *>(p.z) + b * p.sz[0] + d * p.sz[1] : nullptr;
  T *o_row = static_cast<T *>(p.out) + b * p.so[0] + d * p.so[1];
  const float bias = p.bias ? p.bias[d] : 0.f;
  const float Dd = p.D ? p.D[d] : 0.f;
  const BCT *B_base = FIXED ? static_cast<const BCT *>(p.B) + d * p.sB[0]
                            : static_cast<const BCT *>(p.B) + b * p.sB[0] + g * p.sB[1];
  const BCT *C_base = FIXED ? static_cast<const BCT *>(p.C) + d * p.sC[0]
                            : static_cast<const BCT *>(p.C) + b * p.sC[0] + g * p.sC[1];

  float Ar2[SPL], Ai[SPL], xr[SPL], xi[SPL], Bf[SPL], Cf[SPL];
#pragma unroll
  for (int s = 0; s < SPL; ++s) {
    const int n = 16 * s + j;
    const bool ok = n < N;
    Ar2[s] = ok ? p.A[2 * (d * p.sA + n)] * kLog2e : 0.f;
    Ai[s] = ok ? p.A[2 * (d * p.sA + n) + 1] : 0.f;
    const long long ii = 2 * (b * p.si[0] + d * p.si[1] + n);
    xr[s] = (ok && active && p.init) ? p.init[ii] : 0.f;
    xi[s] = (ok && active && p.init) ? p.init[ii + 1] : 0.f;
    Bf[s] = (FIXED && ok) ? to_f<BCT>(B_base[n]) : 0.f;
    Cf[s] = (FIXED && ok) ? to_f<BCT>(C_base[n]) : 0.f;
  }
  float *const ch = &s_ch[chl][0][0];
  float *const sy = &s_y[chl][0][0];

  // the lane's inputs of a segment, fetched one segment ahead (one state group:
  // B/C rows too)
  const T zero_t = from_f<T>(0.f);
  T raw[3], nraw[3];
  Row<BCT> rb, rc, nrb, nrc;
  auto fetch = [&](int t0, T (&r)[3], Row<BCT> &fb, Row<BCT> &fc) {
    const bool vj = active && t0 + j < L;
    r[0] = vj ? u_row[t0 + j] : zero_t;
    r[1] = vj ? dl_row[t0 + j] : zero_t;
    r[2] = (vj && p.has_z) ? z_row[t0 + j] : zero_t;
    if constexpr (!FIXED && SPL == 1) {
      const bool ok = active && j < N;
      fetch_row<BCT>(B_base + j * p.sB[2], t0, ok ? L : 0, p.bcvec != 0, fb);
      fetch_row<BCT>(C_base + j * p.sC[2], t0, ok ? L : 0, p.bcvec != 0, fc);
    }
  };
  fetch(0, raw, rb, rc);

  for (int t0 = 0; t0 < L; t0 += kT) {
    if (t0 + kT < L) fetch(t0 + kT, nraw, nrb, nrc);
    // lane j prepares step t0 + j
    const bool vj = active && t0 + j < L;
    float uj = 0.f, dtj = 0.f, gate = 1.f;
    if (vj) {
      uj = to_f<T>(raw[0]);
      const float v = to_f<T>(raw[1]) + bias;
      dtj = p.softplus ? softplus_cx<T>(v) : v;
      if (p.has_z) gate = silu_f(to_f<T>(raw[2]));
    }
    ch[j] = dtj;
    ch[kT + j] = dtj * uj;
    __syncwarp();

    float yv[kT];
#pragma unroll
    for (int i = 0; i < kT; ++i) yv[i] = 0.f;
#pragma unroll
    for (int s = 0; s < SPL; ++s) {
      const int n = 16 * s + j;
      float Bv[kT], Cv[kT];
      if constexpr (FIXED) {
#pragma unroll
        for (int i = 0; i < kT; ++i) {
          Bv[i] = Bf[s];
          Cv[i] = Cf[s];
        }
      } else if constexpr (SPL == 1) {
        unpack_row<BCT>(rb, Bv);
        unpack_row<BCT>(rc, Cv);
      } else {
        const bool ok = active && n < N;
        Row<BCT> tb, tc;
        fetch_row<BCT>(B_base + n * p.sB[2], t0, ok ? L : 0, p.bcvec != 0, tb);
        fetch_row<BCT>(C_base + n * p.sC[2], t0, ok ? L : 0, p.bcvec != 0, tc);
        unpack_row<BCT>(tb, Bv);
        unpack_row<BCT>(tc, Cv);
      }
      float r = xr[s], im = xi[s];
#pragma unroll
      for (int i = 0; i < kT; i += 4) {
        const float4 dt4 = *reinterpret_cast<const float4 *>(ch + i);
        const float4 du4 = *reinterpret_cast<const float4 *>(ch + kT + i);
        const float dtv[4] = {dt4.x, dt4.y, dt4.z, dt4.w}, duv[4] = {du4.x, du4.y, du4.z, du4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float e = ex2(dtv[q] * Ar2[s]);
          float sn, cs;
          const float th = dtv[q] * Ai[s];
          // fp32 inputs: the product's rounding error joins the reduced angle
          const float lo = (sizeof(T) < 4) ? 0.f : fmaf(dtv[q], Ai[s], -th);
          sincos_rr<(sizeof(T) < 4)>(th, lo, sn, cs);
          const float ar = e * cs, ai = e * sn;
          const float nr = fmaf(ar, r, fmaf(-ai, im, duv[q] * Bv[i + q]));
          im = fmaf(ar, im, ai * r);
          r = nr;
          yv[i + q] = fmaf(Cv[i + q], r, yv[i + q]);
        }
      }
      xr[s] = r;
      xi[s] = im;
    }
    // y of step t0 + j = sum over the channel's 16 lanes of their term j
#pragma unroll
    for (int i = 0; i < kT; i += 4)
      *reinterpret_cast<float4 *>(sy + j * kYRow + i) = make_float4(yv[i], yv[i + 1], yv[i + 2], yv[i + 3]);
    __syncwarp();
    float y = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) y += sy[k * kYRow + j];
    if (vj) o_row[t0 + j] = from_f<T>(fmaf(Dd, uj, y) * gate);
    __syncwarp();  // the channel's step values and terms are read before the next segment overwrites them
#pragma unroll
    for (int q = 0; q < 3; ++q) raw[q] = nraw[q];
    rb = nrb;
    rc = nrc;
  }

  if (!active || !p.last) return;
#pragma unroll
  for (int s = 0; s < SPL; ++s) {
    const int n = 16 * s + j;
    if (n >= N) continue;
    const long long li = 2 * (b * p.sl[0] + d * p.sl[1] + n);
    p.last[li] = xr[s];
    p.last[li + 1] = xi[s];
  }
}

template <typename T, typename BCT, bool FIXED>
const void *by_states(int spl) {
  switch (spl) {
    case 1: return (const void *)&ss_fwd_complex_kernel<T, BCT, FIXED, 1>;
    case 2: return (const void *)&ss_fwd_complex_kernel<T, BCT, FIXED, 2>;
    case 3: return (const void *)&ss_fwd_complex_kernel<T, BCT, FIXED, 3>;
    default: return (const void *)&ss_fwd_complex_kernel<T, BCT, FIXED, 4>;
  }
}

template <typename T, typename BCT>
const void *pick(bool fixed, int spl) {
  if constexpr (sizeof(BCT) == 4) {
    if (fixed) return by_states<T, float, true>(spl);
  }
  return by_states<T, BCT, false>(spl);
}

}  // namespace

int cx_segment_steps() { return kT; }
int cx_channels_per_cta() { return kCPC; }
int cx_threads() { return kW * 32; }

const void *cx_kernel(int in_dtype, bool bc_f32, bool fixed, int dstate) {
  const int spl = (dstate + 15) / 16;
  switch (in_dtype) {
    case 0: return pick<float, float>(fixed, spl);
    case 1: return bc_f32 ? pick<__half, float>(fixed, spl) : pick<__half, __half>(false, spl);
    default: return bc_f32 ? pick<__nv_bfloat16, float>(fixed, spl) : pick<__nv_bfloat16, __nv_bfloat16>(false, spl);
  }
}

}  // namespace ssk
