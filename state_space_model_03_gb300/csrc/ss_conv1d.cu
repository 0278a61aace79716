// Causal depthwise 1-D convolution: the causal_conv1d_fn operator of the page
// "PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南",
// section 4.2, and its one-step decode update. Per (batch b, channel d, step t):
//   out[b,d,t] = act(bias[d] + sum_{k<W} weight[d,k] * x[b,d,t-(W-1)+k])
// with x before step 0 taken from initial_states (else 0), with positions of
// another packed sequence (seq_idx) counting as 0, act = identity or silu, and
// final_states = the last W-1 inputs of each row.
//
// The forward streams each row once: a thread owns EPT consecutive steps
// (16-byte loads and stores when the row allows), gets the W-1 inputs to its
// left from the neighbouring lane by shuffles (lane 0 loads them), and writes
// its EPT outputs. The operator is bound by HBM traffic (x in, out out).
#include "ss_dispatch.h"
#include "ss_fwd_kernel.cuh"

namespace ssk {

namespace {

constexpr int kConvThreads = 256;

template <typename T>
__device__ __forceinline__ float act_f(float v, int act) {
  if (!act) return v;
  // fp32 I/O: ex2 + rcp; 16-bit I/O: the tanh form (one MUFU op, rel. error ~1e-4)
  return silu_t<T>(v);
}

// x row value at step t of (b, d): x itself for t >= 0, else the initial state
// (or 0).
template <typename T>
__device__ __forceinline__ float left_value(const ConvParams &p, const T *xrow, int b, int d, int t) {
  if (t >= 0) return to_f<T>(xrow[t]);
  if (!p.init) return 0.f;
  const int k = p.width - 1 + t;  // 0 .. W-2
  return to_f<T>(static_cast<const T *>(p.init)[b * p.si[0] + (long long)d * p.si[1] + k * p.si[2]]);
}

// W: kernel width (2..4); SEQ: packed sequences (seq_idx) present.
template <typename T, int EPT, int W, bool SEQ>
__global__ void __launch_bounds__(kConvThreads) ss_conv1d_kernel(const __grid_constant__ ConvParams p) {
  constexpr int H = W - 1;
  const int d = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31;
  const int seqlen = (int)p.seqlen;  // < 2^31 (checked by the host)
  const int t0 = (blockIdx.x * kConvThreads + threadIdx.x) * EPT;
  const T *xrow = static_cast<const T *>(p.x) + b * p.sx[0] + (long long)d * p.sx[1];
  T *orow = static_cast<T *>(p.out) + b * p.so[0] + (long long)d * p.so[1];
  float w[W];
#pragma unroll
  for (int k = 0; k < W; ++k) w[k] = p.weight[(long long)d * p.sw[0] + k];
  const float bias = p.bias ? p.bias[d] : 0.f;

  // this thread's inputs (zeros past the end of the row)
  float v[EPT];
  const bool full = t0 + EPT <= seqlen;
  if (full && p.xvec) {
    constexpr int NW = EPT * (int)sizeof(T) / 16;  // 16-byte words
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const uint4 r = reinterpret_cast<const uint4 *>(xrow + t0)[q];
      const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (sizeof(T) == 4) {
          v[q * 4 + i] = __uint_as_float(wd[i]);
        } else {
          const float2 f = unpack2<T>(wd[i]);
          v[q * 8 + 2 * i] = f.x;
          v[q * 8 + 2 * i + 1] = f.y;
        }
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPT; ++i) v[i] = t0 + i < seqlen ? to_f<T>(xrow[t0 + i]) : 0.f;
  }
  // the H (<= 3) inputs to the left: from the previous lane's last values,
  // lane 0 (or the row start) reads them itself
  float h[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const float up = __shfl_up_sync(0xffffffffu, v[EPT - 3 + k], 1);
    h[k] = (lane > 0) ? up : (t0 < seqlen ? left_value<T>(p, xrow, b, d, t0 - 3 + k) : 0.f);
  }
  // sequence ids of the EPT positions and the 3 to the left
  int sid[EPT], hs[3];
  if constexpr (SEQ) {
    const int *srow = p.seq + b * p.sq[0];
#pragma unroll
    for (int i = 0; i < EPT; ++i) sid[i] = t0 + i < seqlen ? srow[t0 + i] : -1;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int up = __shfl_up_sync(0xffffffffu, sid[EPT - 3 + k], 1);
      const int t = t0 - 3 + k;
      hs[k] = (lane > 0) ? up : (t >= 0 && t0 < seqlen ? srow[t] : -2);
    }
  }
  if (t0 >= seqlen) return;

  // window e[j] = x[t0 - 3 + j], j = 0 .. EPT + 2
  float y[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    float acc = bias;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const int j = i + 3 - H + k;  // window index of x[t0 + i - H + k]
      const float xv = j < 3 ? h[j] : v[j - 3];
      if constexpr (SEQ) {
        const int s = j < 3 ? hs[j] : sid[j - 3];
        if (s == sid[i]) acc = fmaf(w[k], xv, acc);
      } else {
        acc = fmaf(w[k], xv, acc);
      }
    }
    y[i] = act_f<T>(acc, p.act);
  }
  if (full && p.ovec) {
    constexpr int NW = EPT * (int)sizeof(T) / 16;
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      uint32_t wd[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (sizeof(T) == 4) wd[i] = __float_as_uint(y[q * 4 + i]);
        else wd[i] = pack2<T>(y[q * 8 + 2 * i], y[q * 8 + 2 * i + 1]);
      }
      reinterpret_cast<uint4 *>(orow + t0)[q] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPT; ++i)
      if (t0 + i < seqlen) orow[t0 + i] = from_f<T>(y[i]);
  }
  // final states: the last H inputs of the row (initial states to their left)
  if (p.fin && t0 <= seqlen - 1 && seqlen - 1 < t0 + EPT) {
    T *frow = static_cast<T *>(p.fin) + b * p.sf[0] + (long long)d * p.sf[1];
#pragma unroll
    for (int k = 0; k < H; ++k) frow[k * p.sf[2]] = from_f<T>(left_value<T>(p, xrow, b, d, seqlen - H + k));
  }
}

// One decode step per (batch, channel): window = [conv_state, x], oldest first.
// grid: (channel tiles, batch rows)
template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads) ss_conv1d_update_kernel(const __grid_constant__ ConvUpdateParams p) {
  const int d = blockIdx.x * kConvThreads + threadIdx.x;
  const int b = blockIdx.y;
  if (d >= p.dim) return;
  T *st = static_cast<T *>(p.state) + b * p.ss[0] + (long long)d * p.ss[1];
  T raw[W];  // window, oldest first: the W-1 states, then the new input
#pragma unroll
  for (int k = 0; k < W - 1; ++k) raw[k] = st[k * p.ss[2]];
  raw[W - 1] = static_cast<const T *>(p.x)[b * p.sx[0] + (long long)d * p.sx[1]];
  float acc = p.bias ? p.bias[d] : 0.f;
#pragma unroll
  for (int k = 0; k < W; ++k) acc += p.weight[(long long)d * p.sw[0] + k] * to_f<T>(raw[k]);
  static_cast<T *>(p.out)[b * p.so[0] + (long long)d * p.so[1]] = from_f<T>(act_f<T>(acc, p.act));
  // shift the window left by one: the newest input becomes the last state entry
#pragma unroll
  for (int k = 0; k < W - 1; ++k) st[k * p.ss[2]] = raw[k + 1];
}

template <typename T, int EPT, bool SEQ>
const void *fwd_width(int width) {
  return width == 2 ? (const void *)&ss_conv1d_kernel<T, EPT, 2, SEQ>
       : width == 3 ? (const void *)&ss_conv1d_kernel<T, EPT, 3, SEQ>
                    : (const void *)&ss_conv1d_kernel<T, EPT, 4, SEQ>;
}

template <typename T>
const void *fwd_kernel(int ept, int width, bool seq) {
  if (ept != 8) return nullptr;
  return seq ? fwd_width<T, 8, true>(width) : fwd_width<T, 8, false>(width);
}

template <typename T>
const void *upd_kernel(int width) {
  return width == 2 ? (const void *)&ss_conv1d_update_kernel<T, 2>
       : width == 3 ? (const void *)&ss_conv1d_update_kernel<T, 3>
                    : (const void *)&ss_conv1d_update_kernel<T, 4>;
}

}  // namespace

const void *conv1d_kernel(int dtype, int ept, int width, bool seq) {
  switch (dtype) {
    case 0: return fwd_kernel<float>(ept, width, seq);
    case 1: return fwd_kernel<__half>(ept, width, seq);
    default: return fwd_kernel<__nv_bfloat16>(ept, width, seq);
  }
}

const void *conv1d_update_kernel(int dtype, int width) {
  switch (dtype) {
    case 0: return upd_kernel<float>(width);
    case 1: return upd_kernel<__half>(width);
    default: return upd_kernel<__nv_bfloat16>(width);
  }
}

}  // namespace ssk
