// Selective-scan forward for fixed B/C (dim, dstate), one lane per channel.
//
// Operation (operands of `selective_scan_fn`, page "PaddleNLP Kernel 算子库：
// CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南", section 4.1): per batch b,
// channel d, state n and step t
//   dt = softplus(delta + delta_bias); x_n = exp(dt A_n) x_n + dt B_n u_t;
//   y = sum_n C_n x_n + D u_t; out = y silu(z_t); last_state = final x.
//
// With fixed B and C nothing but (u, delta, z) varies along the sequence, so a
// lane can own a whole channel: its NS states live in its registers, and the
// lane itself evaluates softplus, the gate, the D skip and the output, which
// leaves no per-element hand-off between warps and no cross-lane reduction of
// y. Each CTA is one warp: 32 consecutive channels of one batch row over one
// sequence segment. Lane 0 streams 128-byte rows of u, delta and z (32 steps
// of fp32, 64 of 16-bit types) by TMA into a two-stage ring guarded by
// mbarriers; the lane reads its own row 16 bytes at a time (the 128-byte
// swizzle keeps the 32 rows' reads conflict-free) and writes its outputs
// straight to global memory, 16 bytes per store.
//
// The state is carried as xi = x / B (x = B xi: exact algebra, and B = 0
// still gives x = 0), which removes the dt u B product: per (state, step)
// pair, one exponent product, one ex2, one FMA for xi and one FMA for y
// (packed in fp32x2 state pairs). A start state cannot be expressed as x / B
// where B = 0, so with one the lanes run the plain update instead (GEN).
//
// Parallelism across the sequence comes from segments (blockIdx.y): a summary
// pass records each segment's end state from zero (in xi form) and its step
// sum, and the forward folds the summaries of the earlier segments into its
// start state, as the 32-channel forward kernel does, with the same workspace
// layout.
#include "ss_dispatch.h"
#include "ss_fwd_kernel.cuh"

namespace ssk {

namespace {

constexpr int kLaneStages = 2;

template <typename T>
struct LaneCfg {
  static constexpr int L = 128 / (int)sizeof(T);  // steps per chunk (one 128-byte row per channel)
  static constexpr int G = 16 / (int)sizeof(T);   // steps per 16-byte shared read and output store
  static constexpr int TILE = 32 * 128;           // one tensor's tile: 32 channels x 128 bytes
};

template <typename T, int NS, bool SUMMARY, bool GEN>
__global__ void __launch_bounds__(32, 12)
ss_fwd_lane_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tm_u,
                   const __grid_constant__ CUtensorMap tm_dl, const __grid_constant__ CUtensorMap tm_z) {
  using CF = LaneCfg<T>;
  constexpr int L = CF::L, G = CF::G, NP2 = NS / 2;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int ntile = p.has_z && !SUMMARY ? 3 : 2;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kLaneStages * ntile * CF::TILE);
  const int lane = threadIdx.x;
  const int tiles = (p.dim + 31) / 32;
  const int b = blockIdx.x / tiles;
  const int d0 = (blockIdx.x - b * tiles) * 32;
  const int d = d0 + lane;
  const bool ok = d < p.dim;
  const int dc = ok ? d : p.dim - 1;
  const int seg = blockIdx.y;
  const int tseg0 = seg * p.seg_len;
  const int tseg1 = min(p.seqlen, tseg0 + p.seg_len);
  const int nchunks = (tseg1 - tseg0 + L - 1) / L;
  const int nsum = p.nseg - 1;

  if (lane == 0) {
    for (int s = 0; s < kLaneStages; ++s) mbar_init(&bar[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  auto tile = [&](int s, int k) -> unsigned char * { return smem + (s * ntile + k) * CF::TILE; };
  auto issue = [&](int ci) {
    if (ci == p.stall_chunk) return;  // test hook: this chunk never lands
    const int s = ci % kLaneStages;
    const int t0 = tseg0 + ci * L;
    fence_proxy_async();  // the stage's previous contents were read through the generic proxy
    mbar_arrive_expect_tx(&bar[s], ntile * CF::TILE);
    tma_load_3d(tile(s, 0), &tm_u, &bar[s], t0, d0, b);
    tma_load_3d(tile(s, 1), &tm_dl, &bar[s], t0, d0, b);
    if (ntile == 3) tma_load_3d(tile(s, 2), &tm_z, &bar[s], t0, d0, b);
  };
  int issued = 0;
  if (lane == 0)
    for (; issued < kLaneStages && issued < nchunks; ++issued) issue(issued);

  // per-channel constants
  f2 a2p[NP2], cb2[NP2], bb2[NP2], cc2[NP2], x2[NP2];
#pragma unroll
  for (int k = 0; k < NP2; ++k) {
    float a[2], bv[2], cv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = 2 * k + h;
      const bool in = n < p.dstate;
      a[h] = in ? p.A[(long long)dc * p.sA[0] + n] * kLog2e : 0.f;
      bv[h] = in ? static_cast<const float *>(p.B)[(long long)dc * p.sB[0] + n] : 0.f;
      cv[h] = in ? static_cast<const float *>(p.C)[(long long)dc * p.sC[0] + n] : 0.f;
    }
    a2p[k] = pk(a[0], a[1]);
    if constexpr (GEN) {  // the plain update keeps B and C; the x / B form only C * B
      bb2[k] = pk(bv[0], bv[1]);
      cc2[k] = pk(cv[0], cv[1]);
    } else {
      cb2[k] = pk(cv[0] * bv[0], cv[1] * bv[1]);
    }
    x2[k] = pk(0.f, 0.f);
    if (!SUMMARY && GEN && ok) {  // x itself (the plain update)
      const float *xr = p.init + (long long)b * p.si[0] + (long long)dc * p.si[1];
      x2[k] = pk(2 * k < p.dstate ? xr[2 * k] : 0.f, 2 * k + 1 < p.dstate ? xr[2 * k + 1] : 0.f);
    }
  }
  const float bias = p.has_bias ? p.bias[dc] : 0.f;
  const float Dd = p.has_D ? p.D[dc] : 0.f;

  if (!SUMMARY && seg > 0) {
    // carry-in: fold the summaries of segments 0..seg-1 (the state after
    // segment k from state x is exp(A sum dt_k) x + end_k, end_k from zero)
    const long long row_bd = (long long)b * p.dim + dc;
    const float *wsx = p.ws + row_bd * nsum * NS;
    const float *wsl = p.ws + (long long)nsum * NS * p.batch * p.dim + row_bd * nsum;
    for (int ks = 0; ks < seg; ++ks) {
      const float lk = wsl[ks];
      const f2 l2 = pk(lk, lk);
#pragma unroll
      for (int k = 0; k < NP2; ++k) {
        const float2 e = upk(mul2(l2, a2p[k]));
        const f2 dec = pk(ex2(e.x), ex2(e.y));
        const float2 xe = *reinterpret_cast<const float2 *>(wsx + ks * NS + 2 * k);
        f2 end = pk(xe.x, xe.y);
        if constexpr (GEN) end = mul2(bb2[k], end);  // summaries are x / B; the plain update carries x
        x2[k] = fma2(dec, x2[k], end);
      }
    }
  }

  T *gout = static_cast<T *>(p.out);
  const long long orow = (long long)b * p.so[0] + (long long)dc * p.so[1];
  const bool out_vec = p.out_vec != 0;
  float lam = 0.f, lam_c = 0.f;  // compensated step sum (summary pass)
  const int softplus = p.softplus;
  int ci = 0;
  for (; ci < nchunks; ++ci) {
    const int s = ci % kLaneStages;
    // every lane polls; the outcome is made warp-uniform before anyone acts on it
    const bool landed = mbar_wait(&bar[s], (ci / kLaneStages) & 1, p.err, kErrWaitFull, p.wait_limit);
    if (!__all_sync(0xffffffffu, landed)) break;
    const unsigned char *tu = tile(s, 0), *td = tile(s, 1), *tz = tile(s, ntile - 1);
    const int tc0 = tseg0 + ci * L;
    // four groups per loop body, so that one group's loads and softplus
    // overlap another's recurrence (long_fixed_fp32, groups per body 1 / 2 /
    // 4 / 8: 834 / 811 / 805 / 835 us)
#pragma unroll 4
    for (int g = 0; g < L / G; ++g) {
      const int tg = tc0 + g * G;
      float uv[G], dv[G], dt[G], yv[G];
      lds_row<T, G>(tu, lane, g * G, uv);
      lds_row<T, G>(td, lane, g * G, dv);
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const float v = dv[k] + bias;
        dt[k] = softplus ? softplus_t<T>(v) : v;
        if (tg + k >= tseg1) dt[k] = 0.f;  // steps past the end leave x unchanged
      }
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const float w = (tg + k < tseg1) ? dt[k] * uv[k] : 0.f;
        const f2 w2 = pk(w, w), d2 = pk(dt[k], dt[k]);
        f2 y2 = pk(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < NP2; ++q) {
          const float2 e = upk(mul2(d2, a2p[q]));
          const f2 a = pk(ex2(e.x), ex2(e.y));
          if constexpr (GEN) {
            x2[q] = fma2(a, x2[q], mul2(w2, bb2[q]));
            y2 = fma2(cc2[q], x2[q], y2);
          } else {
            x2[q] = fma2(a, x2[q], w2);
            if constexpr (!SUMMARY) y2 = fma2(cb2[q], x2[q], y2);
          }
        }
        if constexpr (SUMMARY) {
          const float yk = dt[k] - lam_c;
          const float tk = lam + yk;
          lam_c = (tk - lam) - yk;
          lam = tk;
        } else {
          const float2 yy = upk(y2);
          yv[k] = fmaf(Dd, uv[k], yy.x + yy.y);
        }
      }
      if constexpr (!SUMMARY) {
        if (p.has_z) {
          float zv[G];
          lds_row<T, G>(tz, lane, g * G, zv);
#pragma unroll
          for (int k = 0; k < G; ++k) yv[k] *= silu_t<T>(zv[k]);
        }
        if (out_vec) {
          // y replaces the u values just read (same lane, same 16 bytes); the
          // warp stores the chunk's rows whole below
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if constexpr (sizeof(T) == 4) w[i] = __float_as_uint(yv[i]);
            else w[i] = pack2<T>(yv[2 * i], yv[2 * i + 1]);
          }
          *reinterpret_cast<uint4 *>(tile(s, 0) + swz(lane, g * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
        } else if (ok && tg < tseg1) {
          stg_row<T, G>(gout + orow + tg, yv, false, tseg1 - tg);
        }
      }
    }
    if constexpr (!SUMMARY) {
      if (out_vec) {
        // the chunk's outputs, row by row: 8 lanes store one row's 128
        // contiguous bytes, 4 rows per warp store (instead of each lane
        // storing 16 bytes into each of 32 rows); only steps of this segment
        __syncwarp();
        const int tv = min(L, tseg1 - tc0);
        constexpr int EPC = 16 / (int)sizeof(T);  // elements per 16-byte piece
#pragma unroll 2
        for (int it = 0; it < 8; ++it) {
          const int r = it * 4 + (lane >> 3), c16 = lane & 7, e0 = c16 * EPC;
          const int dr = d0 + r;
          if (dr < p.dim && e0 < tv) {
            const uint4 v = *reinterpret_cast<const uint4 *>(tile(s, 0) + swz(r, 16 * c16));
            T *dst = gout + (long long)b * p.so[0] + (long long)dr * p.so[1] + tc0 + e0;
            if (e0 + EPC <= tv) {
              *reinterpret_cast<uint4 *>(dst) = v;
            } else {  // the sequence's last, partial chunk: element by element
              const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int e = 0; e < EPC; ++e) {
                if (e >= tv - e0) break;
                if constexpr (sizeof(T) == 4)
                  reinterpret_cast<uint32_t *>(dst)[e] = wv[e];
                else
                  reinterpret_cast<uint16_t *>(dst)[e] = static_cast<uint16_t>(wv[e / 2] >> (16 * (e & 1)));
              }
            }
          }
        }
      }
    }
    __syncwarp();  // every lane is done with stage s
    if (lane == 0 && issued < nchunks) issue(issued++);
  }
  if (ci < nchunks) {
    // a wait gave up: let the copies still in flight land before the CTA exits
    if (lane == 0)
      for (int cj = ci; cj < issued; ++cj)
        (void)mbar_wait(&bar[cj % kLaneStages], (cj / kLaneStages) & 1, p.err, kErrWaitFull, p.wait_limit);
    __syncwarp();
    return;
  }

  if constexpr (SUMMARY) {
    if (ok) {
      float *wsx = p.ws + (((long long)b * p.dim + d) * nsum + seg) * NS;
#pragma unroll
      for (int k = 0; k < NP2; ++k) *reinterpret_cast<float2 *>(wsx + 2 * k) = upk(x2[k]);
      p.ws[(long long)nsum * NS * p.batch * p.dim + ((long long)b * p.dim + d) * nsum + seg] = lam - lam_c;
    }
    return;
  }
  if (ok && p.want_last && seg == p.nseg - 1) {
    float *lr = p.last + (long long)b * p.sl[0] + (long long)d * p.sl[1];
#pragma unroll
    const float *br = static_cast<const float *>(p.B) + (long long)d * p.sB[0];
    for (int k = 0; k < NP2; ++k) {
      f2 xv = x2[k];
      if constexpr (!GEN)  // x = B xi
        xv = mul2(pk(2 * k < p.dstate ? br[2 * k] : 0.f, 2 * k + 1 < p.dstate ? br[2 * k + 1] : 0.f), xv);
      const float2 v = upk(xv);
      if (2 * k < p.dstate) lr[(2 * k) * p.sl[2]] = v.x;
      if (2 * k + 1 < p.dstate) lr[(2 * k + 1) * p.sl[2]] = v.y;
    }
  }
}

template <typename T, int NS>
LaneKernel pick_t(bool summary, bool gen) {
  // dynamic shared memory for two streamed tensors; add lane_tile_bytes() per
  // stage when z is streamed too
  const int smem = kLaneStages * 2 * LaneCfg<T>::TILE + 1024 + 64;
  const void *fn = summary ? (const void *)&ss_fwd_lane_kernel<T, NS, true, false>
                   : gen   ? (const void *)&ss_fwd_lane_kernel<T, NS, false, true>
                           : (const void *)&ss_fwd_lane_kernel<T, NS, false, false>;
  return LaneKernel{fn, smem, LaneCfg<T>::L};
}

template <typename T>
LaneKernel pick_ns(int ns, bool summary, bool gen) {
  switch (ns) {
    case 4: return pick_t<T, 4>(summary, gen);
    case 8: return pick_t<T, 8>(summary, gen);
    default: return pick_t<T, 16>(summary, gen);
  }
}

}  // namespace

int lane_tile_bytes() { return 32 * 128; }
int lane_stages() { return kLaneStages; }

LaneKernel lane_kernel(int in_dtype, int ns, bool summary, bool gen) {
  switch (in_dtype) {
    case 0: return pick_ns<float>(ns, summary, gen);
    case 1: return pick_ns<__half>(ns, summary, gen);
    default: return pick_ns<__nv_bfloat16>(ns, summary, gen);
  }
}

}  // namespace ssk
