// Kernel instances of the selective-scan forward for __nv_bfloat16 inputs.
#include "ss_fwd_instances.cuh"

namespace ssk {
KernelInfo lookup_bf16(int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8, bool ch16, bool ys) {
  return reg::lookup<__nv_bfloat16>(np, fixed, bc_f32, tma, summary, sub8, ch16, ys);
}
}  // namespace ssk
