// Kernel registry of the selective-scan forward for one input type T (u,
// delta, z, out): which ss_fwd_kernel instance serves a (padded dstate, B/C
// form, producer, pass, hand-off size, CTA width, y summed by the scan warps)
// choice. Each of
// ss_fwd_f32.cu / ss_fwd_f16.cu / ss_fwd_bf16.cu instantiates it for its type,
// so the three compile in parallel.
#pragma once

#include "ss_dispatch.h"
#include "ss_fwd_kernel.cuh"

namespace ssk {
namespace reg {

template <typename T, int NP, int K, bool FIXED, bool BCF32, bool TMA, bool SUMMARY, int SUB, int CHN = 32, bool YS = false>
KernelInfo info() {
  using CF = Cfg<T, NP, K, FIXED, BCF32, SUB, CHN, !TMA, YS>;
  return KernelInfo{reinterpret_cast<const void *>(&ss_fwd_kernel<T, NP, K, FIXED, BCF32, TMA, SUMMARY, SUB, CHN, YS>),
                    CF::SMEM_ALLOC, CF::THREADS, CF::CH, CF::L};
}

template <typename T, int NP, int K, bool FIXED, bool BCF32, bool TMA>
KernelInfo pick3(bool summary, bool sub8, bool ch16, bool ys) {
  constexpr KernelInfo none{nullptr, 0, 0, 0, 0};
  if (summary) return (ch16 || ys) ? none : info<T, NP, K, FIXED, BCF32, TMA, true, 16>();
  if constexpr (TMA) {
    if constexpr (NP == 16) {  // the common state size only
      if (ch16 && !sub8 && !ys) return info<T, NP, K, FIXED, BCF32, TMA, false, 16, 16>();  // 16-channel CTAs
      if (ys && !sub8 && !ch16) return info<T, NP, K, FIXED, BCF32, TMA, false, 16, 32, true>();
    }
    if (ch16 || ys) return none;
    if (sub8) return info<T, NP, K, FIXED, BCF32, TMA, false, 8>();
  }
  if (sub8 || ch16 || ys) return none;
  return info<T, NP, K, FIXED, BCF32, TMA, false, 16>();
}

template <typename T, int NP, int K, bool FIXED, bool BCF32>
KernelInfo pick2(bool tma, bool summary, bool sub8, bool ch16, bool ys) {
  return tma ? pick3<T, NP, K, FIXED, BCF32, true>(summary, sub8, ch16, ys)
             : pick3<T, NP, K, FIXED, BCF32, false>(summary, sub8, ch16, ys);
}

template <typename T, int NP, int K>
KernelInfo pick(bool fixed, bool bc_f32, bool tma, bool summary, bool sub8, bool ch16, bool ys) {
  // fixed B/C live in registers (fp32); BCF32 only selects the variable tile type
  if (fixed) return pick2<T, NP, K, true, false>(tma, summary, sub8, ch16, ys);
  return bc_f32 ? pick2<T, NP, K, false, true>(tma, summary, sub8, ch16, ys)
                : pick2<T, NP, K, false, false>(tma, summary, sub8, ch16, ys);
}

template <typename T>
KernelInfo lookup(int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8, bool ch16, bool ys) {
  switch (np) {
    case 4: return pick<T, 4, 4>(fixed, bc_f32, tma, summary, sub8, ch16, ys);
    case 8: return pick<T, 8, 4>(fixed, bc_f32, tma, summary, sub8, ch16, ys);
    case 16: return pick<T, 16, 4>(fixed, bc_f32, tma, summary, sub8, ch16, ys);
    case 32: return pick<T, 32, 8>(fixed, bc_f32, tma, summary, sub8, ch16, ys);
    case 64: return pick<T, 64, 8>(fixed, bc_f32, tma, summary, sub8, ch16, ys);
    default: return KernelInfo{nullptr, 0, 0, 0, 0};
  }
}

}  // namespace reg
}  // namespace ssk
