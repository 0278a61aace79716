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

}  // namespace ssk
