// Backward of the selective scan (section 4.1 of the page "PaddleNLP Kernel
// 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南" routes the backward of
// selective_scan_fn to a CUDA kernel returning every input's gradient). For
// L = sum(dout * out), per (batch b, channel d, state n, step t):
//   lam_t = dy_t C_t + a_{t+1} lam_{t+1},  a_t = exp(dt_t A), dy_t = dout_t silu(z_t)
//   du_t  = dy_t D + sum_n lam_t dt_t B_t,  ddt_t = sum_n lam_t (A a_t x_{t-1} + B_t u_t)
//   dA += lam_t a_t x_{t-1} dt_t,  dB_t += lam_t dt_t u_t,  dC_t += dy_t x_t
//   dz_t = dout_t y_t silu'(z_t),  ddelta_t = ddt_t sigmoid(v_t),  dD += dy_t u_t
//
// Schedule. A warp owns one (b, d) row; a CTA holds kBwdWarps rows of the same
// batch row and B/C group, so their dB/dC terms (which sum over the group's
// channels) are added in shared memory before one atomic per CTA. The row is
// cut into chunks of 32 x kE steps, lane j owning kE consecutive steps.
//   1. Forward over the chunks, state by state: each lane composes its steps'
//      affine maps x -> a x + dt B u, a warp scan composes the lanes, and the
//      state at every chunk start is kept in the workspace.
//   2. Backward over the chunks (last first), state by state: the lane's
//      states are recomputed from the chunk-start checkpoint (warp scan of the
//      same maps), the adjoint lam runs right to left through the chunk by the
//      mirrored warp scan of the maps mu -> a (mu + g), and each step adds its
//      gradient terms. dt, dy, du, ddt and y live in registers across the
//      state loop; the per-state carries live in shared memory.
// All arithmetic is fp32; the reductions over batch and steps are fp32
// atomics into zero-filled outputs.
#include "ss_dispatch.h"
#include "ss_fwd_kernel.cuh"

namespace ssk {

namespace {

#ifndef SSB_WARPS
#define SSB_WARPS 8
#endif
constexpr int kBwdWarps = SSB_WARPS;  // rows (warps) per CTA
constexpr int kE = 8;          // steps per lane
constexpr int kCH = 32 * kE;   // steps per chunk
static_assert(kE == 8, "the dB/dC reduction splits a lane's run into two quads");
constexpr int kMaxN = 64;
constexpr int kLaneRow = kE + 4;   // a lane's padded run of dB/dC terms (conflict-free 16-byte accesses)
constexpr int kRedRow = 32 * kLaneRow;  // one row's dB (or dC) terms of a chunk
constexpr unsigned kFull = 0xffffffffu;

template <typename T>
__device__ __forceinline__ void load_steps(const T *src, bool vec, int valid, float (&v)[kE]) {
  if (vec && valid == kE) {
    if constexpr (sizeof(T) == 4) {
      const float4 a = reinterpret_cast<const float4 *>(src)[0];
      const float4 b = reinterpret_cast<const float4 *>(src)[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
      const uint4 q = *reinterpret_cast<const uint4 *>(src);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2<T>(w[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < kE; ++i) v[i] = i < valid ? to_f<T>(src[i]) : 0.f;
}

template <typename T>
__device__ __forceinline__ void store_steps(T *dst, bool vec, int valid, const float (&v)[kE]) {
  if (vec && valid == kE) {
    if constexpr (sizeof(T) == 4) {
      reinterpret_cast<float4 *>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<float4 *>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      *reinterpret_cast<uint4 *>(dst) =
          make_uint4(pack2<T>(v[0], v[1]), pack2<T>(v[2], v[3]), pack2<T>(v[4], v[5]), pack2<T>(v[6], v[7]));
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < kE; ++i)
    if (i < valid) dst[i] = from_f<T>(v[i]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Inclusive scan of affine maps x -> P x + Q over lanes, lower lanes applied first.
__device__ __forceinline__ void scan_up(float &P, float &Q, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float Pp = __shfl_up_sync(kFull, P, o), Qp = __shfl_up_sync(kFull, Q, o);
    if (lane >= o) {
      Q = fmaf(P, Qp, Q);
      P *= Pp;
    }
  }
}
// Inclusive scan over lanes, higher lanes applied first.
__device__ __forceinline__ void scan_down(float &P, float &Q, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float Pn = __shfl_down_sync(kFull, P, o), Qn = __shfl_down_sync(kFull, Q, o);
    if (lane + o < 32) {
      Q = fmaf(P, Qn, Q);
      P *= Pn;
    }
  }
}

constexpr int kNB = 16;  // states of variable B/C staged in shared memory at a time

// Shared-memory carve-up (bytes), per instantiation.
template <typename BCT, bool FIXED>
struct BwdSmem {
  static constexpr int kRows = kBwdWarps * kMaxN;                     // per-row, per-state floats
  static constexpr int kRed = FIXED ? 0 : 2 * 2 * kBwdWarps * kRedRow;  // dB/dC terms, double-buffered
  static constexpr int kStage = FIXED ? 0 : 2 * kNB * kCH * (int)sizeof(BCT);  // B, C of kNB states
  static constexpr int kSmall = (FIXED ? 7 : 3) * kRows;             // carry, dA, A (+ dB, dC sums, B, C values)
  static constexpr int kBytes = kRed * 4 + kStage + kSmall * 4;
};

template <typename T, typename BCT, bool FIXED>
__global__ void __launch_bounds__(kBwdWarps * 32, 2) ss_bwd_kernel(const __grid_constant__ BwdParams p) {
  using SM = BwdSmem<BCT, FIXED>;
  extern __shared__ __align__(16) unsigned char smem[];
  float *sred = reinterpret_cast<float *>(smem);                                  // [2][2][K][32][kLaneRow]
  BCT *sbc = reinterpret_cast<BCT *>(smem + SM::kRed * 4);                          // [2][kNB][kCH]
  float *small = reinterpret_cast<float *>(smem + SM::kRed * 4 + SM::kStage);
  float *scar = small;                      // [K][kMaxN] state / adjoint carry
  float *sdA = small + SM::kRows;           // [K][kMaxN]
  float *sAr = small + 2 * SM::kRows;       // [K][kMaxN] A of the row
  float *sdB = small + 3 * SM::kRows;       // fixed: [K][kMaxN] dB, dC sums and B, C values
  float *sdC = small + 4 * SM::kRows;
  float *sBf = small + 5 * SM::kRows;       // fixed: [2][K][kMaxN] B then C values of the rows

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.dstate, L = p.seqlen, nch = p.nch;
  const int g = blockIdx.x / p.tiles;
  const int dl = (blockIdx.x - g * p.tiles) * kBwdWarps + warp;  // channel within the group
  const bool active = dl < p.dpg;
  const int d = g * p.dpg + (active ? dl : 0);
  const int b = blockIdx.y + gridDim.y * blockIdx.z;
  if (b >= p.batch) return;  // the last batch slab of a folded grid (whole CTA)
  const long long row = (long long)b * p.dim + d;

  const T *u_row = static_cast<const T *>(p.u) + b * p.su[0] + d * p.su[1];
  const T *dl_row = static_cast<const T *>(p.delta) + b * p.sd[0] + d * p.sd[1];
  const T *z_row = p.has_z ? static_cast<const T *>(p.z) + b * p.sz[0] + d * p.sz[1] : nullptr;
  const T *g_row = static_cast<const T *>(p.dout) + b * p.sg[0] + d * p.sg[1];
  const float bias = p.bias ? p.bias[d] : 0.f;
  const float Dd = p.D ? p.D[d] : 0.f;
  float *ws_row = p.ws + row * nch * N;
  const BCT *B_base = FIXED ? static_cast<const BCT *>(p.B) + d * p.sB[0]
                            : static_cast<const BCT *>(p.B) + b * p.sB[0] + g * p.sB[1];
  const BCT *C_base = FIXED ? static_cast<const BCT *>(p.C) + d * p.sC[0]
                            : static_cast<const BCT *>(p.C) + b * p.sC[0] + g * p.sC[1];
  float *const my_car = scar + warp * kMaxN;
  float *const my_dA = sdA + warp * kMaxN;
  float *const my_A = sAr + warp * kMaxN;

  for (int n = lane; n < N; n += 32) {
    my_car[n] = (p.init && active) ? p.init[b * p.si[0] + d * p.si[1] + n] : 0.f;
    my_dA[n] = 0.f;
    my_A[n] = p.A[d * p.sA + n];
    if constexpr (FIXED) {
      sdB[warp * kMaxN + n] = 0.f;
      sdC[warp * kMaxN + n] = 0.f;
      sBf[warp * kMaxN + n] = to_f<BCT>(B_base[n]);
      sBf[kBwdWarps * kMaxN + warp * kMaxN + n] = to_f<BCT>(C_base[n]);  // C values follow B's
    }
  }
  __syncwarp();

  // Variable B/C: copy states [n0, n0 + nb) of chunk c into shared memory
  // (B only when !with_c); zeros past the end of the row. Whole CTA.
  auto stage = [&](int c, int n0, int nb, bool with_c) {
    __syncthreads();  // earlier readers of the stage are done
    constexpr int G = 16 / (int)sizeof(BCT);  // elements per 16-byte group
    const int per_mat = nb * (kCH / G);
    const int total = (with_c ? 2 : 1) * per_mat;
    for (int e = threadIdx.x; e < total; e += kBwdWarps * 32) {
      const int which = e >= per_mat;
      const int rem = e - which * per_mat;
      const int nn = rem / (kCH / G), tg = (rem - nn * (kCH / G)) * G;
      const int t = c * kCH + tg;
      const BCT *src = (which ? C_base + (n0 + nn) * p.sC[2] : B_base + (n0 + nn) * p.sB[2]) + t;
      BCT *dst = sbc + (which * kNB + nn) * kCH + tg;
      if (p.bcvec && t + G <= L) {
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
      } else {
#pragma unroll
        for (int j = 0; j < G; ++j) dst[j] = t + j < L ? src[j] : from_f<BCT>(0.f);
      }
    }
    __syncthreads();
  };
  // the lane's kE values of state n (relative to the staged block) of B (which 0) or C (1)
  auto staged = [&](int which, int nn, float (&v)[kE]) {
    load_steps<BCT>(sbc + (which * kNB + nn) * kCH + lane * kE, true, kE, v);
  };

  // dt and dt*u of this lane's steps of chunk c (0 past the end of the row)
  auto load_dt = [&](int c, float (&dt)[kE], float (&uu)[kE], float (&v)[kE], int &valid, int &t0) {
    t0 = c * kCH + lane * kE;
    valid = active ? min(max(L - t0, 0), kE) : 0;
    load_steps<T>(u_row + t0, p.vec, valid, uu);
    load_steps<T>(dl_row + t0, p.vec, valid, v);
#pragma unroll
    for (int i = 0; i < kE; ++i) {
      v[i] += bias;
      dt[i] = i < valid ? (p.softplus ? softplus_f(v[i]) : v[i]) : 0.f;
    }
  };

  // ---- 1. forward: chunk-start states into the workspace -------------------
  for (int c = 0; c < nch; ++c) {
    float dt[kE], uu[kE], v[kE];
    int valid, t0;
    load_dt(c, dt, uu, v, valid, t0);
    for (int n0 = 0; n0 < N; n0 += kNB) {
      const int nb = min(kNB, N - n0);
      if constexpr (!FIXED) stage(c, n0, nb, false);
      for (int nn = 0; nn < nb; ++nn) {
        const int n = n0 + nn;
        const float A2 = my_A[n] * kLog2e;
        float Bv[kE];
        if constexpr (FIXED) {
          const float bf = sBf[warp * kMaxN + n];
#pragma unroll
          for (int i = 0; i < kE; ++i) Bv[i] = bf;
        } else {
          staged(0, nn, Bv);
        }
        float P = 1.f, Q = 0.f;
#pragma unroll
        for (int i = 0; i < kE; ++i) {
          const float a = ex2(dt[i] * A2);
          Q = fmaf(a, Q, dt[i] * uu[i] * Bv[i]);
          P *= a;
        }
        // the chunk's map: the lanes' maps composed in order by a tree that ends in lane 0
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float Pn = __shfl_down_sync(kFull, P, o), Qn = __shfl_down_sync(kFull, Q, o);
          Q = fmaf(Pn, Q, Qn);  // this lane's steps first, then lane + o's
          P *= Pn;
        }
        if (lane == 0) {
          const float h = my_car[n];
          if (active) ws_row[(long long)c * N + n] = h;
          my_car[n] = fmaf(P, h, Q);
        }
      }
    }
    __syncwarp();
  }

  // ---- 2. backward, last chunk first ---------------------------------------
  for (int n = lane; n < N; n += 32) my_car[n] = 0.f;  // adjoint entering the row's end
  __syncwarp();
  float dD_acc = 0.f, dbias_acc = 0.f;
  int it = 0;  // state-loop iterations so far: parity of the dB/dC buffer
  for (int c = nch - 1; c >= 0; --c) {
    float dt[kE], uu[kE], v[kE], dy[kE], gz[kE];
    int valid, t0;
    load_dt(c, dt, uu, v, valid, t0);
    load_steps<T>(g_row + t0, p.vec, valid, dy);  // dout
    if (p.has_z) {
      load_steps<T>(z_row + t0, p.vec, valid, gz);
#pragma unroll
      for (int i = 0; i < kE; ++i) {
        const float s = rcp(1.f + ex2(-gz[i] * kLog2e));
        const float go = dy[i];
        dy[i] = go * gz[i] * s;                      // dout silu(z)
        gz[i] = go * s * fmaf(gz[i], 1.f - s, 1.f);  // dout silu'(z)
      }
    }
    float du[kE], ddt[kE], yv[kE];
#pragma unroll
    for (int i = 0; i < kE; ++i) {
      if (i >= valid) dy[i] = 0.f;
      v[i] = p.softplus ? rcp(1.f + ex2(-v[i] * kLog2e)) : 1.f;  // d dt / d delta
      du[i] = dy[i] * Dd;
      ddt[i] = 0.f;
      yv[i] = 0.f;
    }
    // chunk-start states of this row: state n in lane n % 32 (n < 32) / (n >= 32)
    const float hcA = (active && lane < N) ? ws_row[(long long)c * N + lane] : 0.f;
    const float hcB = (active && lane + 32 < N) ? ws_row[(long long)c * N + lane + 32] : 0.f;

    for (int n0 = 0; n0 < N; n0 += kNB) {
      const int nb = min(kNB, N - n0);
      if constexpr (!FIXED) stage(c, n0, nb, true);
      for (int nn = 0; nn < nb; ++nn, ++it) {
        const int n = n0 + nn;
        const float An = my_A[n], A2 = An * kLog2e;
        float Bv[kE], Cv[kE], a[kE], h[kE];
        if constexpr (FIXED) {
          const float bf = sBf[warp * kMaxN + n], cf = sBf[kBwdWarps * kMaxN + warp * kMaxN + n];
#pragma unroll
          for (int i = 0; i < kE; ++i) {
            Bv[i] = bf;
            Cv[i] = cf;
          }
        } else {
          staged(0, nn, Bv);
          staged(1, nn, Cv);
        }
        // the lane's affine map x -> P x + Q over its steps
        float P = 1.f, Q = 0.f;
#pragma unroll
        for (int i = 0; i < kE; ++i) {
          a[i] = ex2(dt[i] * A2);
          Q = fmaf(a[i], Q, dt[i] * uu[i] * Bv[i]);
          P *= a[i];
        }
        const float Plane = P;
        // states: chunk-start checkpoint through the lanes up to this one
        scan_up(P, Q, lane);
        const float hc = __shfl_sync(kFull, n < 32 ? hcA : hcB, n & 31);
        float h0 = __shfl_up_sync(kFull, fmaf(P, hc, Q), 1);  // state before the lane's first step
        if (lane == 0) h0 = hc;
        float hp = h0;
#pragma unroll
        for (int i = 0; i < kE; ++i) {
          h[i] = fmaf(a[i], hp, dt[i] * uu[i] * Bv[i]);
          hp = h[i];
          yv[i] = fmaf(Cv[i], h[i], yv[i]);
        }
        // adjoint: the lane's map mu -> Plane mu + Qr (mu = a lam, passed to the left)
        float Qr = 0.f;
#pragma unroll
        for (int i = kE - 1; i >= 0; --i) Qr = a[i] * fmaf(dy[i], Cv[i], Qr);
        float Pr = Plane;
        scan_down(Pr, Qr, lane);
        const float mc = my_car[n];
        float mu = __shfl_down_sync(kFull, fmaf(Pr, mc, Qr), 1);  // adjoint entering the lane's last step
        if (lane == 31) mu = mc;
        float dA_acc = 0.f, dBs = 0.f, dCs = 0.f;
        // dB/dC terms: each lane's run of kE steps, padded rows (16-byte stores)
        float *rb = sred + (((it & 1) * 2 + 0) * kBwdWarps + warp) * kRedRow + lane * kLaneRow;
        float *rc = sred + (((it & 1) * 2 + 1) * kBwdWarps + warp) * kRedRow + lane * kLaneRow;
        float tb[4], tc[4];
#pragma unroll
        for (int i = kE - 1; i >= 0; --i) {
          const float lam = fmaf(dy[i], Cv[i], mu);
          const float ah = a[i] * (i > 0 ? h[i - 1] : h0);
          const float ld = lam * dt[i];
          du[i] = fmaf(ld, Bv[i], du[i]);
          ddt[i] = fmaf(lam, fmaf(An, ah, Bv[i] * uu[i]), ddt[i]);
          dA_acc = fmaf(ld, ah, dA_acc);
          if constexpr (FIXED) {
            dBs = fmaf(ld, uu[i], dBs);
            dCs = fmaf(dy[i], h[i], dCs);
          } else {
            tb[i & 3] = ld * uu[i];
            tc[i & 3] = dy[i] * h[i];
            if ((i & 3) == 0) {
              *reinterpret_cast<float4 *>(rb + i) = make_float4(tb[0], tb[1], tb[2], tb[3]);
              *reinterpret_cast<float4 *>(rc + i) = make_float4(tc[0], tc[1], tc[2], tc[3]);
            }
          }
          mu = a[i] * lam;
        }
        __syncwarp();
        if (lane == 0) my_car[n] = mu;  // leaves the chunk to the left
        dA_acc = warp_sum(dA_acc);
        if (lane == 0) my_dA[n] += dA_acc;
        if constexpr (FIXED) {
          dBs = warp_sum(dBs);
          dCs = warp_sum(dCs);
          if (lane == 0) {
            sdB[warp * kMaxN + n] += dBs;
            sdC[warp * kMaxN + n] += dCs;
          }
        } else {
          // group sum over the CTA's rows, then one atomic per step and state
          __syncthreads();
          if (threadIdx.x < 2 * kCH / 4) {
            // thread: B or C, steps 4q .. 4q+3 of lane l's run of kE steps
            const int which = threadIdx.x / (kCH / 4);
            const int r = threadIdx.x % (kCH / 4);
            const int l = r & 31, i0 = (r >> 5) * 4;
            const float *src = sred + ((it & 1) * 2 + which) * kBwdWarps * kRedRow + l * kLaneRow + i0;
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kBwdWarps; ++k) {
              const float4 q = *reinterpret_cast<const float4 *>(src + k * kRedRow);
              s.x += q.x;
              s.y += q.y;
              s.z += q.z;
              s.w += q.w;
            }
            const int t = c * kCH + l * kE + i0;
            float *dst = (which ? p.dC : p.dB) + (((long long)b * p.ngroups + g) * N + n) * L + t;
            if (p.dbvec && t + 4 <= L) {
              atomicAdd(reinterpret_cast<float4 *>(dst), s);
            } else {
              const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (t + j < L) atomicAdd(dst + j, sv[j]);
            }
          }
        }
      }
    }
    __syncwarp();

    // per-step outputs of the chunk
#pragma unroll
    for (int i = 0; i < kE; ++i) {
      if (p.has_z) gz[i] *= fmaf(Dd, uu[i], yv[i]);  // dz = dout y silu'(z)
      ddt[i] = i < valid ? ddt[i] * v[i] : 0.f;      // ddelta
      dD_acc = fmaf(dy[i], uu[i], dD_acc);
      dbias_acc += ddt[i];
    }
    if (valid > 0) {
      store_steps<T>(static_cast<T *>(p.du) + b * p.sdu[0] + d * p.sdu[1] + t0, p.vec, valid, du);
      store_steps<T>(static_cast<T *>(p.ddelta) + b * p.sdd[0] + d * p.sdd[1] + t0, p.vec, valid, ddt);
      if (p.has_z) store_steps<T>(static_cast<T *>(p.dz) + b * p.sdz[0] + d * p.sdz[1] + t0, p.vec, valid, gz);
    }
  }

  // ---- per-row results ----------------------------------------------------
  dD_acc = warp_sum(dD_acc);
  dbias_acc = warp_sum(dbias_acc);
  if (!active) return;
  if (lane == 0) {
    if (p.dD) atomicAdd(p.dD + d, dD_acc);
    if (p.dbias) atomicAdd(p.dbias + d, dbias_acc);
  }
  for (int n = lane; n < N; n += 32) {
    atomicAdd(p.dA + (long long)d * N + n, my_dA[n]);
    if constexpr (FIXED) {
      atomicAdd(p.dB + (long long)d * N + n, sdB[warp * kMaxN + n]);
      atomicAdd(p.dC + (long long)d * N + n, sdC[warp * kMaxN + n]);
    }
    if (p.dx0) p.dx0[row * N + n] = my_car[n];
  }
}

template <typename T, typename BCT, bool FIXED>
BwdKernel info() {
  return {(const void *)&ss_bwd_kernel<T, BCT, FIXED>, BwdSmem<BCT, FIXED>::kBytes};
}

template <typename T, typename BCT>
BwdKernel pick(bool fixed) {
  if constexpr (sizeof(BCT) == 4) {
    if (fixed) return info<T, float, true>();
  }
  return info<T, BCT, false>();
}

}  // namespace

int bwd_chunk_steps() { return kCH; }
int bwd_rows_per_cta() { return kBwdWarps; }
int bwd_threads() { return kBwdWarps * 32; }

BwdKernel bwd_kernel(int in_dtype, bool bc_f32, bool fixed, int /*dstate: one kernel serves 1..64 states*/) {
  switch (in_dtype) {
    case 0: return pick<float, float>(fixed);
    case 1: return bc_f32 ? pick<__half, float>(fixed) : pick<__half, __half>(false);
    default: return bc_f32 ? pick<__nv_bfloat16, float>(fixed) : pick<__nv_bfloat16, __nv_bfloat16>(false);
  }
}

}  // namespace ssk
