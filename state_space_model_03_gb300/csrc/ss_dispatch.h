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
// 16-channel CTAs (TMA forward, np == 16 only).
// Returns fn == nullptr if not instantiated.
KernelInfo lookup_f32(int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8, bool ch16);
KernelInfo lookup_f16(int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8, bool ch16);
KernelInfo lookup_bf16(int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8, bool ch16);

// Decode step (ss_state_update): launch parameters and kernel lookup.
// lpc: lanes per channel (1, 2, 4, 8, 16), 4 states per lane, 256 threads.
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
const void *state_update_kernel(int in_dtype, bool bc_f32, int lpc);

}  // namespace ssk
