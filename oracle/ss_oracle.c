/*
 * Selective-scan forward: plain, slow, sequential fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only the tests, the package's smoke check and the bench's CPU
 * baseline leg use it. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (one (batch, channel) row at a time, no blocking, no fusion,
 * no reordering beyond the definition):
 *
 *   Operands and shapes follow the page "PaddleNLP Kernel 算子库：CUDA 与 Triton
 *   双实现的高性能 NLP GPU 算子实战指南", section 4.1 "CUDA 算子 selective_scan":
 *   u, delta, z are (batch, dim, seqlen); A is (dim, dstate), real here;
 *   B, C are fixed (dim, dstate) or vary over the sequence as
 *   (batch, groups, dstate, seqlen) (the 3-D (batch, dstate, seqlen) form is
 *   groups = 1); D and delta_bias are (dim,); last_state is (batch, dim, dstate).
 *
 *   The page names the operator but prints no formula. The recurrence is the
 *   Mamba-1 selective scan with an Euler input term:
 *     v    = delta[t] + delta_bias                (bias first, then softplus)
 *     dt   = softplus(v) if delta_softplus else v
 *     x_k  = exp(dt * A[k]) * x_k + dt * B[k,t] * u[t]   for every state k
 *     y    = sum_k C[k,t] * x_k  (x after the step-t update) + D * u[t]
 *     out  = y * silu(z[t]) = y * z / (1 + exp(-z))  when z is given, else y
 *   with x = initial_state before t = 0 when one is given, else x = 0 (the
 *   page's signature has no initial-state argument; the optional initial
 *   state is the chaining input of a decode step, one of the operators the
 *   same page lists next to the scan: "selective_state_update"), and
 *   last_state = x after the final step.
 *
 *   Channel d of a grouped B/C uses group d / (dim / groups) (each group serves
 *   dim/groups contiguous channels).
 *
 *   softplus(v) = log(1 + e^v), evaluated as max(v, 0) + log1p(exp(-|v|)),
 *   which is the same function without overflow for large v.
 *
 * All operands are fp64 here; callers widen the stored (already rounded)
 * fp32/fp16/bf16 values exactly before the call.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

static double oracle_softplus(double v) {
  double m = v > 0.0 ? v : 0.0;
  return m + log1p(exp(-fabs(v)));
}

/* One row: the recurrence over t for one (batch, channel).
 * Bk(k, t) = B_row[k * b_kstride + t * b_tstride]; fixed B/C pass b_tstride = 0. */
static void oracle_row(int64_t seqlen, int64_t dstate,
                       const double *u_row, const double *delta_row, const double *z_row,
                       const double *A_row,
                       const double *B_row, int64_t b_kstride, int64_t b_tstride,
                       const double *C_row, int64_t c_kstride, int64_t c_tstride,
                       double D_d, double bias_d, int delta_softplus, const double *x0_row,
                       double *out_row, double *last_row, double *x) {
  for (int64_t k = 0; k < dstate; ++k) x[k] = x0_row ? x0_row[k] : 0.0;
  for (int64_t t = 0; t < seqlen; ++t) {
    double uu = u_row[t];
    double v = delta_row[t] + bias_d;
    double dt = delta_softplus ? oracle_softplus(v) : v;
    double y = 0.0;
    for (int64_t k = 0; k < dstate; ++k) {
      double Bk = B_row[k * b_kstride + t * b_tstride];
      double Ck = C_row[k * c_kstride + t * c_tstride];
      x[k] = exp(dt * A_row[k]) * x[k] + dt * Bk * uu;
      y += Ck * x[k];
    }
    y += D_d * uu;
    if (z_row) {
      double zz = z_row[t];
      y = y * (zz / (1.0 + exp(-zz)));
    }
    out_row[t] = y;
  }
  if (last_row)
    for (int64_t k = 0; k < dstate; ++k) last_row[k] = x[k];
}

/*
 * Rows r in [row_begin, row_end) of the problem, r = b * dim + d.
 *   u, delta, z, out : (batch, dim, seqlen), contiguous; z may be NULL.
 *   A                : (dim, dstate), contiguous.
 *   B, C             : bc_fixed ? (dim, dstate) : (batch, ngroups, dstate, seqlen), contiguous.
 *   D, delta_bias    : (dim,) or NULL (absent = 0).
 *   initial_state    : (batch, dim, dstate) or NULL (absent = 0).
 *   last_state       : (batch, dim, dstate) or NULL.
 *   scratch          : dstate doubles owned by the caller (one per thread).
 * Returns 0, or -1 on a shape error (dim % ngroups != 0, non-positive sizes).
 */
int ss_oracle_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int64_t ngroups,
                  int bc_fixed,
                  const double *u, const double *delta, const double *z,
                  const double *A, const double *B, const double *C,
                  const double *D, const double *delta_bias, int delta_softplus,
                  const double *initial_state, double *out, double *last_state,
                  int64_t row_begin, int64_t row_end, double *scratch) {
  if (batch < 0 || dim <= 0 || seqlen < 0 || dstate <= 0) return -1;
  if (!bc_fixed && (ngroups <= 0 || dim % ngroups != 0)) return -1;
  if (row_begin < 0 || row_end > batch * dim || row_begin > row_end) return -1;
  int64_t dpg = bc_fixed ? dim : dim / ngroups;
  for (int64_t r = row_begin; r < row_end; ++r) {
    int64_t b = r / dim, d = r % dim;
    const double *B_row, *C_row;
    int64_t kstride, tstride;
    if (bc_fixed) {
      B_row = B + d * dstate;
      C_row = C + d * dstate;
      kstride = 1;
      tstride = 0;
    } else {
      int64_t g = d / dpg;
      B_row = B + (b * ngroups + g) * dstate * seqlen;
      C_row = C + (b * ngroups + g) * dstate * seqlen;
      kstride = seqlen;
      tstride = 1;
    }
    oracle_row(seqlen, dstate,
               u + r * seqlen, delta + r * seqlen, z ? z + r * seqlen : NULL,
               A + d * dstate,
               B_row, kstride, tstride, C_row, kstride, tstride,
               D ? D[d] : 0.0, delta_bias ? delta_bias[d] : 0.0, delta_softplus,
               initial_state ? initial_state + r * dstate : NULL, out + r * seqlen, last_state ? last_state + r * dstate : NULL, scratch);
  }
  return 0;
}
