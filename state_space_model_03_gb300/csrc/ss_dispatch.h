// Kernel registry shared by the per-dtype translation units and the C ABI.
#pragma once

namespace ssk {

struct KernelInfo {
  const void *fn;  // __global__ function (launch with cudaLaunchKernel)
  int smem;        // dynamic shared memory bytes
  int threads;     // threads per CTA
  int ch;          // channels per CTA
  int L;           // steps per chunk (TMA box width)
};

// np in {4, 8, 16, 32, 64}; bc_f32: variable B/C stored as fp32 (else in the
// input dtype); summary: the segment-summary pass instead of the forward;
// sub8: 8-step hand-offs (instantiated for the TMA forward only); ch16:
// 16-channel CTAs (TMA forward, np == 16 only); ys: y summed by the scan
// warps (TMA forward, np == 16, 16-step hand-offs, 32-channel CTAs only).
// Returns fn == nullptr if not instantiated.
KernelInfo lookup_f32(int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8, bool ch16, bool ys);
KernelInfo lookup_f16(int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8, bool ch16, bool ys);
KernelInfo lookup_bf16(int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8, bool ch16, bool ys);

// Decode step (ss_state_update): launch parameters and kernel lookup.
// lpc: lanes per channel, 4 * q states per lane (q 1: lpc 1..16; q 2: lpc
// 1..8; q 4: lpc 1..4), 256 threads.
struct SUParams {
  int batch, dim, dstate, dpg;
  int fixed, has_z, has_D, has_bias, softplus;
  int vec, avec, bcvec;  // 16-byte state / A / B-C row accesses allowed
  float *state;
  const void *u, *delta, *z, *B, *C;
  const float *A, *D, *bias;
  void *out;
  long long sst[3], su[2], sd[2], sz[2], so[2], sB[3], sC[3], sA[2];
};
const void *state_update_kernel(int in_dtype, bool bc_f32, int lpc, int q);

// Causal depthwise conv1d (ss_causal_conv1d / ss_causal_conv1d_update).
struct ConvParams {
  int batch, dim, width;
  long long seqlen;
  int act;         // 0 identity, 1 silu
  int xvec, ovec;  // 16-byte x loads / out stores allowed (aligned rows)
  const void *x;
  const float *weight, *bias;
  const int *seq;  // seq_idx (batch, seqlen) or NULL
  const void *init;  // (batch, dim, width-1) or NULL
  void *fin;         // (batch, dim, width-1) or NULL
  void *out;
  long long sx[3], so[3], sw[2], sq[2], si[3], sf[3];
};
struct ConvUpdateParams {
  int batch, dim, width, act;
  const void *x;
  void *state;
  const float *weight, *bias;
  void *out;
  long long sx[2], ss[3], sw[2], so[2];
};
// ept: steps per thread of the forward (8); width 2..4.
const void *conv1d_kernel(int dtype, int ept, int width, bool seq);
const void *conv1d_update_kernel(int dtype, int width);

// Selective-scan backward (ss_bwd).
struct BwdParams {
  int batch, dim, dstate, ngroups, dpg;
  int tiles;        // CTAs per group along the channels
  int seqlen, nch;  // steps; chunks of bwd_chunk_steps() steps
  int has_z, softplus;
  int vec;          // 16-byte row accesses of u, delta, z, dout, du, ddelta, dz allowed
  int bcvec;        // 16-byte B/C row accesses allowed (variable B/C)
  int dbvec;        // 16-byte atomics into dB/dC allowed
  const void *u, *delta, *z, *B, *C, *dout;
  const float *A, *D, *bias, *init;
  void *du, *ddelta, *dz;
  float *dA, *dB, *dC, *dD, *dbias, *dx0;
  float *ws;        // chunk-start states (batch, dim, nch, dstate)
  long long su[2], sd[2], sz[2], sg[2], sdu[2], sdd[2], sdz[2], sB[3], sC[3], sA, si[2];
};
int bwd_chunk_steps();   // steps per chunk (checkpoint interval)
int bwd_rows_per_cta();  // channels per CTA
int bwd_threads();       // threads per CTA
struct BwdKernel {
  const void *fn;
  int smem;  // dynamic shared memory bytes
};
BwdKernel bwd_kernel(int in_dtype, bool bc_f32, bool fixed, int dstate);

// Fixed-B/C forward with one lane per channel (ss_fwd_lane.cu): the forward
// (gen: plain update, for a start state) or the segment-summary pass, for
// padded state counts 4, 8 or 16. Launch with 32 threads per CTA, grid
// (batch * ceil(dim / 32), segments), the KParams of the 32-channel kernel and
// three 3-D tensor maps (u, delta, z) with boxes of L steps x 32 channels.
// smem is for two streamed tensors; add lane_stages() * lane_tile_bytes()
// when z is streamed.
struct LaneKernel {
  const void *fn;
  int smem;  // dynamic shared memory bytes
  int L;     // steps per chunk (the box width)
};
LaneKernel lane_kernel(int in_dtype, int ns, bool summary, bool gen);
int lane_tile_bytes();
int lane_stages();

// Complex-A forward (ss_fwd_complex).
struct CxParams {
  int batch, dim, dstate, ngroups, dpg, tiles;  // tiles: CTAs per group along the channels
  int seqlen, nseg;                             // steps; segments of cx_segment_steps() steps
  int has_z, softplus;
  int bcvec;                         // 16-byte B/C row accesses allowed (variable B/C)
  const void *u, *delta, *z, *B, *C;
  const float *A, *D, *bias, *init;  // A, init: complex64 interleaved
  void *out;
  float *last;                       // complex64 interleaved
  long long su[2], sd[2], sz[2], so[2], sB[3], sC[3], sA, si[2], sl[2];
};
int cx_segment_steps();
int cx_channels_per_cta();
int cx_threads();
const void *cx_kernel(int in_dtype, bool bc_f32, bool fixed, int dstate);

}  // namespace ssk
