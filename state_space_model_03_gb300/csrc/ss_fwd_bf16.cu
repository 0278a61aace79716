// Kernel instances for __nv_bfloat16 inputs (u, delta, z, out).
#include "ss_dispatch.h"
#include "ss_fwd_kernel.cuh"

namespace ssk {

template <int NP, int K, bool FIXED, bool BCF32, bool TMA, bool SUMMARY, int SUB>
static KernelInfo info() {
  using CF = Cfg<__nv_bfloat16, NP, K, FIXED, BCF32, SUB>;
  return KernelInfo{reinterpret_cast<const void *>(&ss_fwd_kernel<__nv_bfloat16, NP, K, FIXED, BCF32, TMA, SUMMARY, SUB>),
                    CF::SMEM_ALLOC, CF::THREADS, CF::CH, CF::L};
}

template <int NP, int K, bool FIXED, bool BCF32, bool TMA>
static KernelInfo pick3(bool summary, bool sub8) {
  if (summary) return info<NP, K, FIXED, BCF32, TMA, true, 16>();
  if constexpr (TMA) {
    if (sub8) return info<NP, K, FIXED, BCF32, TMA, false, 8>();
  }
  if (sub8) return KernelInfo{nullptr, 0, 0, 0, 0};
  return info<NP, K, FIXED, BCF32, TMA, false, 16>();
}

template <int NP, int K, bool FIXED, bool BCF32>
static KernelInfo pick2(bool tma, bool summary, bool sub8) {
  return tma ? pick3<NP, K, FIXED, BCF32, true>(summary, sub8) : pick3<NP, K, FIXED, BCF32, false>(summary, sub8);
}

template <int NP, int K>
static KernelInfo pick(bool fixed, bool bc_f32, bool tma, bool summary, bool sub8) {
  // fixed B/C live in registers (fp32); BCF32 only selects the variable tile type
  if (fixed) return pick2<NP, K, true, false>(tma, summary, sub8);
  return bc_f32 ? pick2<NP, K, false, true>(tma, summary, sub8) : pick2<NP, K, false, false>(tma, summary, sub8);
}

KernelInfo lookup_bf16(int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8) {
  switch (np) {
    case 4: return pick<4, 4>(fixed, bc_f32, tma, summary, sub8);
    case 8: return pick<8, 4>(fixed, bc_f32, tma, summary, sub8);
    case 16: return pick<16, 4>(fixed, bc_f32, tma, summary, sub8);
    case 32: return pick<32, 8>(fixed, bc_f32, tma, summary, sub8);
    case 64: return pick<64, 8>(fixed, bc_f32, tma, summary, sub8);
    default: return KernelInfo{nullptr, 0, 0, 0, 0};
  }
}

}  // namespace ssk
