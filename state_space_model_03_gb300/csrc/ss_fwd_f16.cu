// Kernel instances for __half inputs (u, delta, z, out).
#include "ss_dispatch.h"
#include "ss_fwd_kernel.cuh"

namespace ssk {

template <int NP, int K, bool FIXED, bool BCF32, bool TMA, bool SUMMARY>
static KernelInfo info() {
  using CF = Cfg<__half, NP, K, FIXED, BCF32>;
  return KernelInfo{reinterpret_cast<const void *>(&ss_fwd_kernel<__half, NP, K, FIXED, BCF32, TMA, SUMMARY>),
                    CF::SMEM_ALLOC, CF::THREADS, CF::CH, CF::L};
}

template <int NP, int K, bool FIXED, bool BCF32, bool TMA>
static KernelInfo pick3(bool summary) {
  return summary ? info<NP, K, FIXED, BCF32, TMA, true>() : info<NP, K, FIXED, BCF32, TMA, false>();
}

template <int NP, int K, bool FIXED, bool BCF32>
static KernelInfo pick2(bool tma, bool summary) {
  return tma ? pick3<NP, K, FIXED, BCF32, true>(summary) : pick3<NP, K, FIXED, BCF32, false>(summary);
}

template <int NP, int K>
static KernelInfo pick(bool fixed, bool bc_f32, bool tma, bool summary) {
  // fixed B/C live in registers (fp32); BCF32 only selects the variable tile type
  if (fixed) return pick2<NP, K, true, false>(tma, summary);
  return bc_f32 ? pick2<NP, K, false, true>(tma, summary) : pick2<NP, K, false, false>(tma, summary);
}

KernelInfo lookup_f16(int np, bool fixed, bool bc_f32, bool tma, bool summary) {
  switch (np) {
    case 4: return pick<4, 4>(fixed, bc_f32, tma, summary);
    case 8: return pick<8, 4>(fixed, bc_f32, tma, summary);
    case 16: return pick<16, 4>(fixed, bc_f32, tma, summary);
    case 32: return pick<32, 8>(fixed, bc_f32, tma, summary);
    case 64: return pick<64, 8>(fixed, bc_f32, tma, summary);
    default: return KernelInfo{nullptr, 0, 0, 0, 0};
  }
}

}  // namespace ssk
