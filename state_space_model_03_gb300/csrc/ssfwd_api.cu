// C ABI of libssfwd.so: validation, TMA descriptors, dispatch and launch for
// the selective-scan forward (declarations and contract in include/ssfwd.h).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ss_dispatch.h"
#include "ss_fwd_kernel.cuh"
#include "ssfwd.h"

namespace {

// Device error word written by kernels that give up on a bounded wait. Host
// code obtains its device address once per device (cudaGetSymbolAddress).
__device__ int32_t g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t *g_err_ptr[kMaxDevices] = {};
bool g_attr_done[kMaxDevices][3][5][2][2][2][2][2][2][2] = {};
int g_occupancy[kMaxDevices][3][5][2][2][4] = {};  // CTAs/SM of the TMA forward variants 0 .. 3
bool g_bwd_attr_done[kMaxDevices][3][2][2] = {};     // dynamic shared memory attribute set for ss_bwd

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

int elem_size(int dt) { return dt == SS_F32 ? 4 : 2; }

bool fault_injected(const char *what) {
  // Host-side fault injection for tests: SSFWD_FAULT=<what> makes the named
  // step report a CUDA failure before anything is enqueued.
  const char *f = std::getenv("SSFWD_FAULT");
  return f && std::strcmp(f, what) == 0;
}

struct Range {
  uintptr_t lo, hi;  // [lo, hi) in bytes; empty if lo == hi
};

Range span(const void *ptr, int esize, const int64_t *sizes, const int64_t *strides, int nd) {
  if (!ptr) return {0, 0};
  int64_t last = 0;
  for (int i = 0; i < nd; ++i) {
    if (sizes[i] == 0) return {0, 0};
    last += (sizes[i] - 1) * strides[i];
  }
  uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
  return {lo, lo + static_cast<uintptr_t>((last + 1) * esize)};
}

bool overlap(Range a, Range b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

bool aligned(const void *p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int validate(const ss_fwd_params *p) {
  if (!p) return SS_ERR_NULL;
  if (p->abi_version != SS_ABI_VERSION) return SS_ERR_VERSION;
  if (p->in_dtype < SS_F32 || p->in_dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->bc_dtype < SS_F32 || p->bc_dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->bc_mode != SS_BC_FIXED && p->bc_mode != SS_BC_VARIABLE) return SS_ERR_SHAPE;
  const bool fixed = p->bc_mode == SS_BC_FIXED;
  if (fixed && p->bc_dtype != SS_F32) return SS_ERR_DTYPE;
  if (!fixed && p->bc_dtype != p->in_dtype && p->bc_dtype != SS_F32) return SS_ERR_DTYPE;
  if (p->batch < 0 || p->dim < 0 || p->seqlen < 0) return SS_ERR_SHAPE;
  if (p->dstate < 1) return SS_ERR_SHAPE;
  if (p->dstate > 64) return SS_ERR_UNSUPPORTED;
  if (!fixed && (p->ngroups < 1 || (p->dim > 0 && p->dim % p->ngroups != 0))) return SS_ERR_SHAPE;
  if (p->batch > 65535 || p->dim > (1 << 30) || p->seqlen > (int64_t(1) << 31) - 1024) return SS_ERR_UNSUPPORTED;
  if (p->error_word && !aligned(p->error_word, 4)) return SS_ERR_ALIGN;
  if (p->batch * p->dim == 0) return SS_OK;
  if (p->last_state && p->last_state_stride[2] != 1) return SS_ERR_STRIDE;
  for (int i = 0; i < 3; ++i)
    if (p->last_state && p->last_state_stride[i] < 0) return SS_ERR_STRIDE;
  const int64_t szl[3] = {p->batch, p->dim, p->dstate};
  Range last = p->last_state ? span(p->last_state, 4, szl, p->last_state_stride, 3) : Range{0, 0};
  Range init{0, 0};
  if (p->initial_state) {
    if (p->initial_state_stride[2] != 1) return SS_ERR_STRIDE;
    for (int i = 0; i < 3; ++i)
      if (p->initial_state_stride[i] < 0) return SS_ERR_STRIDE;
    if (!aligned(p->initial_state, 4)) return SS_ERR_ALIGN;
    init = span(p->initial_state, 4, szl, p->initial_state_stride, 3);
    // the start state may be last_state itself (same buffer and strides)
    const bool same = p->last_state == p->initial_state && p->last_state_stride[0] == p->initial_state_stride[0] &&
                      p->last_state_stride[1] == p->initial_state_stride[1];
    if (!same && overlap(init, last)) return SS_ERR_ALIAS;
  }
  if (p->seqlen == 0) return SS_OK;
  if (!p->u || !p->delta || !p->A || !p->B || !p->C || !p->out) return SS_ERR_NULL;
  const int64_t *st3[4] = {p->u_stride, p->delta_stride, p->z ? p->z_stride : p->u_stride, p->out_stride};
  for (auto s : st3) {
    if (s[2] != 1) return SS_ERR_STRIDE;
    if (s[0] < 0 || s[1] < 0) return SS_ERR_STRIDE;
  }
  if (p->A_stride[1] != 1 || p->A_stride[0] < 0) return SS_ERR_STRIDE;
  if (fixed) {
    if (p->B_stride[1] != 1 || p->C_stride[1] != 1 || p->B_stride[0] < 0 || p->C_stride[0] < 0) return SS_ERR_STRIDE;
  } else {
    for (int i = 0; i < 4; ++i)
      if (p->B_stride[i] < 0 || p->C_stride[i] < 0) return SS_ERR_STRIDE;
    if (p->B_stride[3] != 1 || p->C_stride[3] != 1) return SS_ERR_STRIDE;
  }
  const int es = elem_size(p->in_dtype), bs = elem_size(p->bc_dtype);
  if (!aligned(p->u, es) || !aligned(p->delta, es) || !aligned(p->out, es) || (p->z && !aligned(p->z, es)))
    return SS_ERR_ALIGN;
  if (!aligned(p->B, bs) || !aligned(p->C, bs) || !aligned(p->A, 4)) return SS_ERR_ALIGN;
  if ((p->D && !aligned(p->D, 4)) || (p->delta_bias && !aligned(p->delta_bias, 4)) ||
      (p->last_state && !aligned(p->last_state, 4)))
    return SS_ERR_ALIGN;
  // outputs must not overlap inputs or each other
  const int64_t sz3[3] = {p->batch, p->dim, p->seqlen};
  Range out = span(p->out, es, sz3, p->out_stride, 3);
  Range ins[9];
  int ni = 0;
  ins[ni++] = span(p->u, es, sz3, p->u_stride, 3);
  ins[ni++] = span(p->delta, es, sz3, p->delta_stride, 3);
  if (p->z) ins[ni++] = span(p->z, es, sz3, p->z_stride, 3);
  const int64_t sza[2] = {p->dim, p->dstate};
  ins[ni++] = span(p->A, 4, sza, p->A_stride, 2);
  if (fixed) {
    ins[ni++] = span(p->B, 4, sza, p->B_stride, 2);
    ins[ni++] = span(p->C, 4, sza, p->C_stride, 2);
  } else {
    const int64_t szb[4] = {p->batch, p->ngroups, p->dstate, p->seqlen};
    ins[ni++] = span(p->B, bs, szb, p->B_stride, 4);
    ins[ni++] = span(p->C, bs, szb, p->C_stride, 4);
  }
  const int64_t one[1] = {p->dim}, unit[1] = {1};
  if (p->D) ins[ni++] = span(p->D, 4, one, unit, 1);
  if (p->delta_bias) ins[ni++] = span(p->delta_bias, 4, one, unit, 1);
  for (int i = 0; i < ni; ++i)
    if (overlap(out, ins[i]) || overlap(last, ins[i])) return SS_ERR_ALIAS;
  if (overlap(out, last) || overlap(out, init)) return SS_ERR_ALIAS;
  if (p->initial_state) ins[ni++] = init;  // the workspace must not overlap it either
  if (p->workspace_bytes < 0) return SS_ERR_SHAPE;
  Range ws{0, 0};
  if (p->workspace && p->workspace_bytes > 0) {
    ws = Range{reinterpret_cast<uintptr_t>(p->workspace),
               reinterpret_cast<uintptr_t>(p->workspace) + static_cast<uintptr_t>(p->workspace_bytes)};
    for (int i = 0; i < ni; ++i)
      if (overlap(ws, ins[i])) return SS_ERR_ALIAS;
    if (overlap(ws, out) || overlap(ws, last)) return SS_ERR_ALIAS;
  }
  if (p->error_word) {  // written by the kernels on failure: it must not alias anything they touch
    const Range ew{reinterpret_cast<uintptr_t>(p->error_word), reinterpret_cast<uintptr_t>(p->error_word) + 4};
    for (int i = 0; i < ni; ++i)
      if (overlap(ew, ins[i])) return SS_ERR_ALIAS;
    if (overlap(ew, out) || overlap(ew, last) || overlap(ew, ws)) return SS_ERR_ALIAS;
  }
  return SS_OK;
}

int padded_states(int64_t n) {
  if (n <= 4) return 4;
  if (n <= 8) return 8;
  if (n <= 16) return 16;
  if (n <= 32) return 32;
  return 64;
}

int np_index(int np) { return np == 4 ? 0 : np == 8 ? 1 : np == 16 ? 2 : np == 32 ? 3 : 4; }

ssk::KernelInfo lookup(int dt, int np, bool fixed, bool bc_f32, bool tma, bool summary, bool sub8 = false,
                       bool ch16 = false, bool ys = false) {
  switch (dt) {
    case SS_F32: return ssk::lookup_f32(np, fixed, bc_f32, tma, summary, sub8, ch16, ys);
    case SS_F16: return ssk::lookup_f16(np, fixed, bc_f32, tma, summary, sub8, ch16, ys);
    default: return ssk::lookup_bf16(np, fixed, bc_f32, tma, summary, sub8, ch16, ys);
  }
}

// Stride as used by a TMA descriptor: a dimension of extent 1 may carry any
// stride, so give it a legal one.
uint64_t tma_stride(int64_t extent, int64_t stride_elems, int esize, uint64_t fallback) {
  if (extent <= 1) return fallback;
  return static_cast<uint64_t>(stride_elems) * esize;
}

bool tma_ok_stride(uint64_t s) { return s % 16 == 0 && s > 0 && s < (uint64_t(1) << 40); }

// 3-D (seqlen, dim, batch) descriptor for u / delta / z: box {L, CH, 1}.
bool make_map3(CUtensorMap *m, const void *base, int es, const ss_fwd_params *p, const int64_t *st, int L, int CH) {
  if (!aligned(base, 16)) return false;
  const uint64_t row = static_cast<uint64_t>(p->seqlen) * es;
  const uint64_t s1 = tma_stride(p->dim, st[1], es, (row + 15) / 16 * 16);
  const uint64_t s2 = tma_stride(p->batch, st[0], es, s1 * static_cast<uint64_t>(p->dim));
  if (!tma_ok_stride(s1) || !tma_ok_stride(s2)) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(p->seqlen), static_cast<cuuint64_t>(p->dim),
                        static_cast<cuuint64_t>(p->batch)};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(L), static_cast<cuuint32_t>(CH), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                        const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D (seqlen, dstate, groups, batch) descriptor for variable B / C: box {L, dstate, 1, 1}.
bool make_map4(CUtensorMap *m, const void *base, int bs, const ss_fwd_params *p, const int64_t *st, int L) {
  if (!aligned(base, 16)) return false;
  const uint64_t row = static_cast<uint64_t>(p->seqlen) * bs;
  const uint64_t s1 = tma_stride(p->dstate, st[2], bs, (row + 15) / 16 * 16);
  const uint64_t s2 = tma_stride(p->ngroups, st[1], bs, s1 * static_cast<uint64_t>(p->dstate));
  const uint64_t s3 = tma_stride(p->batch, st[0], bs, s2 * static_cast<uint64_t>(p->ngroups));
  if (!tma_ok_stride(s1) || !tma_ok_stride(s2) || !tma_ok_stride(s3)) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(p->seqlen), static_cast<cuuint64_t>(p->dstate),
                        static_cast<cuuint64_t>(p->ngroups), static_cast<cuuint64_t>(p->batch)};
  cuuint64_t strides[3] = {s1, s2, s3};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(L), static_cast<cuuint32_t>(p->dstate), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const bool swz = (L * bs == 128);
  CUresult r = g_encode(m, bs == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                        const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int32_t *error_word_ptr(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!g_err_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int32_t *>(ptr);
  }
  return g_err_ptr[dev];
}

// seqlen == 0: last_state is the start state (or zero).
__global__ void empty_sequence_state(float *last, const float *init, int64_t batch, int64_t dim, int64_t dstate,
                                     int64_t s0, int64_t s1, int64_t s2, int64_t i0, int64_t i1) {
  const int64_t total = batch * dim * dstate;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i % dstate, r = i / dstate, d = r % dim, b = r / dim;
    last[b * s0 + d * s1 + n * s2] = init ? init[b * i0 + d * i1 + n] : 0.f;
  }
}

int num_sms(int dev) {
  static int cache[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return 0;
  if (!cache[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = v;
  }
  return cache[dev];
}

// Sequence segmentation: when the (batch, group, channel-tile) CTAs cannot
// fill the GPU, the sequence is cut into segments processed by separate CTAs.
// A summary pass records, for every segment but the last, the state it reaches
// from zero and the sum of its steps; the forward pass folds the summaries of
// the preceding segments into its starting state.
constexpr int64_t kSegMinSteps = 2048;  // shortest segment worth a summary pass
constexpr int kMaxSegments = 64;

struct SegPlan {
  int nseg = 1;
  int seg_len = 0;
  int64_t ws_bytes = 0;
};

SegPlan plan_segments(const ss_fwd_params *p, int np, int L, int ch, int nsm) {
  SegPlan sp;
  sp.seg_len = static_cast<int>(p->seqlen);
  const int64_t groups = p->bc_mode == SS_BC_FIXED ? 1 : p->ngroups;
  const int64_t dpg = p->dim / groups;
  const int64_t base = (dpg + ch - 1) / ch * groups * p->batch;
  if (nsm <= 0 || base >= 2 * nsm || p->seqlen < 2 * kSegMinSteps) return sp;
  int64_t want = (3 * nsm + base - 1) / base;
  want = std::min<int64_t>(want, p->seqlen / kSegMinSteps);
  want = std::min<int64_t>(want, kMaxSegments);
  if (want < 2) return sp;
  int64_t len = (p->seqlen + want - 1) / want;
  len = (len + L - 1) / L * L;
  sp.nseg = static_cast<int>((p->seqlen + len - 1) / len);
  sp.seg_len = static_cast<int>(len);
  if (sp.nseg < 2) { sp.nseg = 1; sp.seg_len = static_cast<int>(p->seqlen); return sp; }
  sp.ws_bytes = p->batch * p->dim * (sp.nseg - 1) * (np + 1) * int64_t(sizeof(float));
  return sp;
}

// Fixed-B/C forward with one lane per channel (ss_fwd_lane.cu). It serves
// fixed B/C with dstate <= 16 whenever u, delta (and z) have legal TMA
// descriptors with 32-channel boxes; everything else runs the 32-channel
// kernel. Its warps (one per 32 channels per segment) saturate at about eight
// per SM, and a segmented schedule costs a summary pass (~0.8x of the
// forward), so the sequence is split only when the unsplit grid gives fewer
// than three warps per SM, into as many segments as one wave of resident CTAs
// holds (at most 12 per SM), each at least kLaneMinSeg steps. `cap` bounds the
// workspace (the caller's, or the static buffer of ss_fwd_noalloc): the plan
// drops segments until it fits.
constexpr int64_t kLaneMinSeg = 512;

struct LanePlan {
  bool use = false;
  ssk::LaneKernel fwd{}, sum{};
  int smem = 0, nseg = 1, seg_len = 0;
  int64_t ws_bytes = 0;
  CUtensorMap tm[3];
};

int g_lane_occ[kMaxDevices][3][3][2] = {};  // CTAs/SM of the lane forward by (dtype, ns, z)

bool lane_setup(const ss_fwd_params *p, int dev, int64_t cap, LanePlan *lp) {
  lp->use = false;
  if (p->bc_mode != SS_BC_FIXED || p->dstate > 16 || std::getenv("SSFWD_NO_LANE") || std::getenv("SSFWD_NO_TMA"))
    return false;
  std::call_once(g_encode_once, load_encode);
  if (!g_encode || dev < 0 || dev >= kMaxDevices) return false;
  const int np = padded_states(p->dstate);
  const int es = elem_size(p->in_dtype);
  lp->fwd = ssk::lane_kernel(p->in_dtype, np, false, p->initial_state != nullptr);
  lp->sum = ssk::lane_kernel(p->in_dtype, np, true, false);
  if (!lp->fwd.fn || !lp->sum.fn) return false;
  std::memset(lp->tm, 0, sizeof(lp->tm));
  if (!make_map3(&lp->tm[0], p->u, es, p, p->u_stride, lp->fwd.L, 32) ||
      !make_map3(&lp->tm[1], p->delta, es, p, p->delta_stride, lp->fwd.L, 32) ||
      (p->z && !make_map3(&lp->tm[2], p->z, es, p, p->z_stride, lp->fwd.L, 32)))
    return false;
  lp->smem = lp->fwd.smem + (p->z ? ssk::lane_stages() * ssk::lane_tile_bytes() : 0);
  int occ = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    int &slot = g_lane_occ[dev][p->in_dtype][np == 4 ? 0 : np == 8 ? 1 : 2][p->z ? 1 : 0];
    if (!slot && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&slot, lp->fwd.fn, 32, lp->smem) != cudaSuccess)
      slot = 0;
    occ = slot;
  }
  const int nsm = num_sms(dev);
  if (occ <= 0 || nsm <= 0) return false;
  const int64_t warps = p->batch * ((p->dim + 31) / 32);  // warps of one segment
  lp->nseg = 1;
  lp->seg_len = static_cast<int>(p->seqlen);
  if (warps < 3 * int64_t(nsm)) {
    int64_t want = std::min<int64_t>(occ, 12) * nsm / warps;
    want = std::min<int64_t>(want, p->seqlen / kLaneMinSeg);
    want = std::min<int64_t>(want, kMaxSegments);
    const int64_t per_seg = p->batch * p->dim * (np + 1) * int64_t(sizeof(float));
    if (per_seg > 0) want = std::min<int64_t>(want, cap / per_seg + 1);  // workspace for want - 1 summaries
    if (want >= 2) {
      int64_t len = (p->seqlen + want - 1) / want;
      len = (len + lp->fwd.L - 1) / lp->fwd.L * lp->fwd.L;
      const int64_t nseg = (p->seqlen + len - 1) / len;
      if (nseg >= 2) {
        lp->nseg = static_cast<int>(nseg);
        lp->seg_len = static_cast<int>(len);
        lp->ws_bytes = (nseg - 1) * per_seg;
      }
    }
  }
  lp->use = true;
  return true;
}

bool set_smem_attr(int dev, const ssk::KernelInfo &ki, int dt, int np, bool fixed, bool bc_f32, bool tma, bool summary,
                   bool sub8 = false, bool ch16 = false, bool ys = false) {
  std::lock_guard<std::mutex> lk(g_mu);
  bool &done = g_attr_done[dev][dt][np_index(np)][fixed][bc_f32 && !fixed][tma][summary][sub8][ch16][ys];
  if (!done) {
    if (cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem) != cudaSuccess)
      return false;
    done = true;
  }
  return true;
}

// Bytes of workspace the fastest path wants for p (0 if it needs none), with
// at most `cap` bytes for the one-lane-per-channel schedule.
int workspace_bytes(const ss_fwd_params *p, int64_t *bytes, int64_t cap = INT64_MAX) {
  *bytes = 0;
  if (p->batch * p->dim == 0 || p->seqlen == 0) return SS_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
  {
    LanePlan lp;
    if (lane_setup(p, dev, cap, &lp)) {
      *bytes = lp.ws_bytes;
      return SS_OK;
    }
  }
  const bool fixed = p->bc_mode == SS_BC_FIXED;
  const int np = padded_states(p->dstate);
  ssk::KernelInfo ki = lookup(p->in_dtype, np, fixed, p->bc_dtype == SS_F32, true, false);
  if (!ki.fn) return SS_ERR_UNSUPPORTED;
  *bytes = plan_segments(p, np, ki.L, ki.ch, num_sms(dev)).ws_bytes;
  return SS_OK;
}

// Enqueue the forward. ws/ws_bytes: workspace for sequence segmentation
// (device memory, may be NULL/0: the single-pass path is used then).
int launch(const ss_fwd_params *p, cudaStream_t stream, void *ws, int64_t ws_bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
  if (p->batch * p->dim == 0) return SS_OK;
  if (p->seqlen == 0) {
    if (!p->last_state) return SS_OK;
    if (fault_injected("launch")) return SS_ERR_CUDA;
    const int64_t total = p->batch * p->dim * p->dstate;
    const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 4096));
    if (p->initial_state == p->last_state && p->initial_state_stride[0] == p->last_state_stride[0] &&
        p->initial_state_stride[1] == p->last_state_stride[1])
      return SS_OK;  // in place: the start state already is the result
    empty_sequence_state<<<blocks, 256, 0, stream>>>(p->last_state, p->initial_state, p->batch, p->dim, p->dstate,
                                                     p->last_state_stride[0], p->last_state_stride[1],
                                                     p->last_state_stride[2], p->initial_state_stride[0],
                                                     p->initial_state_stride[1]);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
  }
  int32_t *err = p->error_word ? p->error_word : error_word_ptr(dev);
  if (!err) return SS_ERR_CUDA;
  std::call_once(g_encode_once, load_encode);

  const bool fixed = p->bc_mode == SS_BC_FIXED;
  const int np = padded_states(p->dstate);
  const int es = elem_size(p->in_dtype), bs = elem_size(p->bc_dtype);
  const bool bc_f32 = p->bc_dtype == SS_F32;
  ssk::KernelInfo ki = lookup(p->in_dtype, np, fixed, bc_f32, true, false);
  if (!ki.fn) return SS_ERR_UNSUPPORTED;

  ssk::KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.batch = static_cast<int>(p->batch);
  kp.dim = static_cast<int>(p->dim);
  kp.seqlen = static_cast<int>(p->seqlen);
  kp.dstate = static_cast<int>(p->dstate);
  kp.ngroups = fixed ? 1 : static_cast<int>(p->ngroups);
  kp.dpg = kp.dim / kp.ngroups;
  kp.tiles_per_group = (kp.dpg + ki.ch - 1) / ki.ch;
  kp.has_z = p->z != nullptr;
  kp.has_D = p->D != nullptr;
  kp.has_bias = p->delta_bias != nullptr;
  kp.softplus = p->delta_softplus != 0;
  kp.want_last = p->last_state != nullptr;
  kp.out_vec = aligned(p->out, 16) && (p->batch <= 1 || (p->out_stride[0] * es) % 16 == 0) &&
               (p->dim <= 1 || (p->out_stride[1] * es) % 16 == 0);
  kp.u = p->u; kp.delta = p->delta; kp.z = p->z; kp.B = p->B; kp.C = p->C;
  kp.A = p->A; kp.D = p->D; kp.bias = p->delta_bias;
  kp.out = p->out; kp.last = p->last_state;
  for (int i = 0; i < 3; ++i) {
    kp.su[i] = p->u_stride[i]; kp.sd[i] = p->delta_stride[i]; kp.sz[i] = p->z_stride[i];
    kp.so[i] = p->out_stride[i]; kp.sl[i] = p->last_state_stride[i];
  }
  for (int i = 0; i < 4; ++i) { kp.sB[i] = p->B_stride[i]; kp.sC[i] = p->C_stride[i]; }
  kp.sA[0] = p->A_stride[0]; kp.sA[1] = p->A_stride[1];
  kp.init = p->initial_state;
  for (int i = 0; i < 3; ++i) kp.si[i] = p->initial_state ? p->initial_state_stride[i] : 0;
  kp.err = err;
  kp.wait_limit = ssk::kMaxWaitIters;
  kp.stall_chunk = -1;
  if (const char *st = std::getenv("SSFWD_TEST_STALL")) {
    // Test hook: the producer never issues chunk `st` of each CTA and every
    // wait gives up after a short limit, so the bounded-wait exits and the
    // error word can be checked without a hang.
    kp.stall_chunk = std::atoi(st);
    kp.wait_limit = 1u << 10;
  }

  const int nsm = num_sms(dev);
  {
    // fixed B/C, dstate <= 16: one lane per channel when the descriptors allow
    LanePlan lp;
    const bool ws_ok = ws && aligned(ws, 16) && !std::getenv("SSFWD_NO_SEGMENTS");
    if (lane_setup(p, dev, ws_ok ? ws_bytes : 0, &lp)) {
      kp.nseg = lp.nseg;
      kp.seg_len = lp.seg_len;
      kp.ws = lp.nseg > 1 ? static_cast<float *>(ws) : nullptr;
      const unsigned gx = static_cast<unsigned>(p->batch * ((p->dim + 31) / 32));
      if (std::getenv("SSFWD_DEBUG"))
        std::fprintf(stderr, "ssfwd: lane np=%d L=%d grid=%ux%d seg_len=%d smem=%d\n", np, lp.fwd.L, gx,
                     lp.nseg, lp.seg_len, lp.smem);
      if (fault_injected("launch")) return SS_ERR_CUDA;
      void *args[4] = {&kp, &lp.tm[0], &lp.tm[1], &lp.tm[2]};
      if (lp.nseg > 1) {
        const int ssm = lp.sum.smem;  // the summary pass streams u and delta only
        if (cudaLaunchKernel(lp.sum.fn, dim3(gx, lp.nseg - 1), dim3(32), args, static_cast<size_t>(ssm), stream) !=
            cudaSuccess)
          return SS_ERR_CUDA;
      }
      return cudaLaunchKernel(lp.fwd.fn, dim3(gx, lp.nseg), dim3(32), args, static_cast<size_t>(lp.smem), stream) ==
                     cudaSuccess
                 ? SS_OK
                 : SS_ERR_CUDA;
    }
  }
  SegPlan sp = plan_segments(p, np, ki.L, ki.ch, nsm);
  if (sp.nseg > 1 && (!ws || ws_bytes < sp.ws_bytes || !aligned(ws, 16) || std::getenv("SSFWD_NO_SEGMENTS"))) {
    sp.nseg = 1;  // no (or too small a) workspace: single pass over the whole sequence
    sp.seg_len = kp.seqlen;
  }
  kp.nseg = sp.nseg;
  kp.seg_len = sp.seg_len;
  kp.ws = sp.nseg > 1 ? static_cast<float *>(ws) : nullptr;

  // TMA when every streamed tensor has a legal descriptor; else the instance
  // without tensor maps (rows copied as their covering 16-byte blocks), with
  // the same compute path.
  auto encode = [&](CUtensorMap *tm, int ch) -> bool {
    std::memset(tm, 0, 5 * sizeof(CUtensorMap));
    bool ok = make_map3(&tm[0], p->u, es, p, p->u_stride, ki.L, ch);
    if (ok) ok = make_map3(&tm[1], p->delta, es, p, p->delta_stride, ki.L, ch);
    if (ok && p->z) ok = make_map3(&tm[2], p->z, es, p, p->z_stride, ki.L, ch);
    if (ok && !fixed) ok = make_map4(&tm[3], p->B, bs, p, p->B_stride, ki.L);
    if (ok && !fixed) ok = make_map4(&tm[4], p->C, bs, p, p->C_stride, ki.L);
    return ok;
  };
  CUtensorMap tm[5], tm_sum[5];
  bool tma = g_encode != nullptr && !std::getenv("SSFWD_NO_TMA") && encode(tm_sum, ki.ch);
  const int groups = kp.ngroups;
  // Forward variant: 32-channel CTAs with 16-step hand-offs (0), the same
  // with 8-step hand-offs (1: smaller buffers, one more resident CTA per SM,
  // about 1.36x the time per CTA), 16-channel CTAs (2), or the scan warps
  // summing y over their lanes (3: a smaller y slot, so a fourth 16-step CTA
  // fits per SM; about 7% slower than variant 0 per CTA, 20% faster than
  // variant 1). A CTA's time grows only mildly with the CTAs that share its SM
  // (the recurrence is latency-bound), so the variant that runs the grid in
  // the fewest waves of resident CTAs wins. Among equals: 16-channel CTAs when
  // the 32-channel grid leaves no SM more than two CTAs (about 5% faster
  // there), else variant 0, then 3.
  bool sub8 = false, ch16 = false, ys = false;
  if (tma) {
    ssk::KernelInfo kv[4] = {};
    int64_t waves[4] = {0, 0, 0, 0}, ctas[4] = {0, 0, 0, 0};
    const char *force = std::getenv("SSFWD_VARIANT");  // diagnostics: one variant only
    for (int v = 0; v < 4; ++v) {
      const bool v8 = v == 1, v16 = v == 2, vys = v == 3;
      if (v16 && std::getenv("SSFWD_NO_CH16")) continue;
      if (v8 && std::getenv("SSFWD_NO_SUB8")) continue;
      if (vys && std::getenv("SSFWD_NO_YSUM")) continue;
      if (force && std::atoi(force) != v) continue;
      ssk::KernelInfo k = lookup(p->in_dtype, np, fixed, bc_f32, true, false, v8, v16, vys);
      if (!k.fn) continue;
      if (!set_smem_attr(dev, k, p->in_dtype, np, fixed, bc_f32, true, false, v8, v16, vys)) return SS_ERR_CUDA;
      int occ = 0;
      {
        std::lock_guard<std::mutex> lk(g_mu);
        int &slot = g_occupancy[dev][p->in_dtype][np_index(np)][fixed][bc_f32 && !fixed][v];
        if (!slot && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&slot, k.fn, k.threads, k.smem) != cudaSuccess)
          slot = 0;
        occ = slot;
      }
      if (occ <= 0 || nsm <= 0) continue;
      kv[v] = k;
      ctas[v] = int64_t((kp.dpg + k.ch - 1) / k.ch) * groups * kp.batch * sp.nseg;
      waves[v] = (ctas[v] + int64_t(occ) * nsm - 1) / (int64_t(occ) * nsm);
    }
    const int64_t ctas32 = int64_t((kp.dpg + 31) / 32) * groups * kp.batch * sp.nseg;
    const int order_small[4] = {2, 0, 3, 1}, order[4] = {0, 2, 3, 1};
    const int *pref = ctas32 <= 2 * int64_t(nsm) ? order_small : order;
    int best = -1;
    for (int i = 0; i < 4; ++i) {
      const int v = pref[i];
      if (kv[v].fn && (best < 0 || waves[v] < waves[best])) best = v;
    }
    ssk::KernelInfo bestk = ki;
    if (best >= 0) {
      bestk = kv[best];
      sub8 = best == 1;
      ch16 = best == 2;
      ys = best == 3;
    }
    ki = bestk;
    if (ch16 && !encode(tm, ki.ch)) return SS_ERR_INTERNAL;
    if (!ch16) std::memcpy(tm, tm_sum, sizeof(tm));
  } else {
    ki = lookup(p->in_dtype, np, fixed, bc_f32, false, false);
    if (!ki.fn) return SS_ERR_UNSUPPORTED;
    if (!set_smem_attr(dev, ki, p->in_dtype, np, fixed, bc_f32, false, false)) return SS_ERR_CUDA;
    std::memset(tm, 0, sizeof(tm));
    std::memset(tm_sum, 0, sizeof(tm_sum));
  }
  kp.tiles_per_group = (kp.dpg + ki.ch - 1) / ki.ch;
  // rows TMA cannot describe: the producer copies the 16-byte blocks that
  // cover each row (SSFWD_NO_BULK: plain loads into the same layout, for
  // comparison)
  kp.rows_bulk = !tma && !std::getenv("SSFWD_NO_BULK");
  ssk::KParams kps = kp;  // summary pass: 32-channel CTAs
  ssk::KernelInfo ks{};
  if (sp.nseg > 1) {
    ks = lookup(p->in_dtype, np, fixed, bc_f32, tma, true);
    if (!ks.fn) return SS_ERR_UNSUPPORTED;
    if (!set_smem_attr(dev, ks, p->in_dtype, np, fixed, bc_f32, tma, true)) return SS_ERR_CUDA;
    kps.tiles_per_group = (kp.dpg + ks.ch - 1) / ks.ch;
  }
  if (fault_injected("launch")) return SS_ERR_CUDA;
  const unsigned gx = static_cast<unsigned>(kp.tiles_per_group * kp.ngroups), gy = static_cast<unsigned>(kp.batch);
  if (std::getenv("SSFWD_DEBUG"))  // opt-in launch report on stderr
    std::fprintf(stderr,
                 "ssfwd: %s np=%d fixed=%d bc_f32=%d ch=%d L=%d grid=%ux%ux%d seg_len=%d sub=%d ysum=%d threads=%d smem=%d\n",
                 tma ? "tma" : (kp.rows_bulk ? "generic-bulk" : "generic"), np, (int)fixed, (int)bc_f32, ki.ch, ki.L, gx, gy, sp.nseg, sp.seg_len,
                 sub8 ? 8 : 16, (int)ys, ki.threads, ki.smem);
  if (sp.nseg > 1) {
    void *sargs[6] = {&kps, &tm_sum[0], &tm_sum[1], &tm_sum[2], &tm_sum[3], &tm_sum[4]};
    const unsigned sx = static_cast<unsigned>(kps.tiles_per_group * kps.ngroups);
    cudaError_t e = cudaLaunchKernel(ks.fn, dim3(sx, gy, sp.nseg - 1), dim3(ks.threads), sargs,
                                     static_cast<size_t>(ks.smem), stream);
    if (e != cudaSuccess) return SS_ERR_CUDA;
  }
  void *args[6] = {&kp, &tm[0], &tm[1], &tm[2], &tm[3], &tm[4]};
  cudaError_t e = cudaLaunchKernel(ki.fn, dim3(gx, gy, sp.nseg), dim3(ki.threads), args,
                                   static_cast<size_t>(ki.smem), stream);
  return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Allocation-free entry point (ss_fwd_noalloc)
// ---------------------------------------------------------------------------
// Scratch for callers that cannot allocate device memory: a fixed buffer that
// is part of the loaded library image on every device (held until exit). Only
// the segment summaries of the split-sequence schedule live here.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SS_NOALLOC_MAX_SCRATCH];
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on `dev` (which must be current): the
// name itself is only a host-side stand-in, so the address is looked up once
// per device and cached.
void *noalloc_scratch(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!g_noalloc_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_noalloc_ptr[dev] = ptr;
  }
  return g_noalloc_ptr[dev];
}

// The host-staged entry point copies whole tensors, so the device buffers must
// be laid out contiguously (a dimension of extent 1 may carry any stride).
bool contiguous(const int64_t *sizes, const int64_t *strides, int nd) {
  int64_t expect = 1;
  for (int i = nd - 1; i >= 0; --i) {
    if (sizes[i] > 1 && strides[i] != expect) return false;
    expect *= sizes[i];
  }
  return true;
}

bool host_layout_ok(const ss_fwd_params *p) {
  const int64_t sz3[3] = {p->batch, p->dim, p->seqlen};
  if (!contiguous(sz3, p->u_stride, 3) || !contiguous(sz3, p->delta_stride, 3) || !contiguous(sz3, p->out_stride, 3))
    return false;
  if (p->z && !contiguous(sz3, p->z_stride, 3)) return false;
  const int64_t sza[2] = {p->dim, p->dstate};
  if (!contiguous(sza, p->A_stride, 2)) return false;
  if (p->bc_mode == SS_BC_FIXED) {
    if (!contiguous(sza, p->B_stride, 2) || !contiguous(sza, p->C_stride, 2)) return false;
  } else {
    const int64_t szb[4] = {p->batch, p->ngroups, p->dstate, p->seqlen};
    if (!contiguous(szb, p->B_stride, 4) || !contiguous(szb, p->C_stride, 4)) return false;
  }
  const int64_t szl[3] = {p->batch, p->dim, p->dstate};
  if (p->last_state && !contiguous(szl, p->last_state_stride, 3)) return false;
  return true;
}

// ---------------------------------------------------------------------------
// Host-staged forward (ss_fwd_host): the copies overlap the kernels
// ---------------------------------------------------------------------------
// The problem is cut into row blocks, each whole batch rows or a range of
// channels inside one batch row (group-aligned for grouped B/C), so that each
// block's u, delta, z, out and last_state are contiguous in memory. Block i's
// inputs go host-to-device on one internal stream, its kernel runs on the
// caller's stream, and its outputs go device-to-host on a second internal
// stream, so the two copy directions and the kernels of neighbouring blocks
// run at the same time. Events fork the internal streams from the caller's
// stream and join them back, so the call keeps the caller's stream ordering.
// The streams and events are created once per device and kept until exit.
constexpr int kHostBlocksMax = 8;
constexpr int64_t kHostBlockBytes = int64_t(32) << 20;  // input bytes per block, at least

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, in_done[kHostBlocksMax] = {}, k_done[kHostBlocksMax] = {};
  std::mutex mu;  // one enqueue sequence at a time per device (the events are reused)
};
HostPipe g_pipe[kMaxDevices];

HostPipe *host_pipe(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  HostPipe &hp = g_pipe[dev];
  std::lock_guard<std::mutex> lk(g_mu);
  if (!hp.ready) {
    const unsigned ev = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.fork, ev) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.join, ev) == cudaSuccess;
    for (int i = 0; ok && i < kHostBlocksMax; ++i)
      ok = cudaEventCreateWithFlags(&hp.in_done[i], ev) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.k_done[i], ev) == cudaSuccess;
    if (!ok) return nullptr;
    hp.ready = true;
  }
  return &hp;
}

struct HostBlock {
  int64_t b0, b1, d0, d1;
};

// Row blocks of about kHostBlockBytes of inputs each (at most kHostBlocksMax).
int host_blocks(const ss_fwd_params *p, HostBlock *blk) {
  const int64_t es = elem_size(p->in_dtype);
  const int64_t in_bytes = p->batch * p->dim * p->seqlen * es * (p->z ? 3 : 2);
  int want = static_cast<int>(std::min<int64_t>(kHostBlocksMax, std::max<int64_t>(1, in_bytes / kHostBlockBytes)));
  if (std::getenv("SSFWD_HOST_SERIAL")) want = 1;
  if (const char *nb = std::getenv("SSFWD_HOST_BLOCKS"))  // diagnostics: a fixed block count
    want = std::max(1, std::min(kHostBlocksMax, std::atoi(nb)));
  if (want <= 1 || p->batch * p->dim <= 1) {
    blk[0] = {0, p->batch, 0, p->dim};
    return 1;
  }
  int n = 0;
  if (p->batch >= want) {  // whole batch rows
    for (int i = 0; i < want; ++i) {
      const int64_t a = p->batch * i / want, c = p->batch * (i + 1) / want;
      if (c > a) blk[n++] = {a, c, 0, p->dim};
    }
    return n;
  }
  // channel ranges inside each batch row, on a unit that keeps groups whole
  const int per_b = (want + static_cast<int>(p->batch) - 1) / static_cast<int>(p->batch);
  const int64_t unit = (p->bc_mode == SS_BC_VARIABLE && p->ngroups > 1) ? p->dim / p->ngroups : 32;
  const int64_t units = (p->dim + unit - 1) / unit;
  const int parts = static_cast<int>(std::min<int64_t>(per_b, units));
  for (int64_t b = 0; b < p->batch; ++b)
    for (int i = 0; i < parts && n < kHostBlocksMax; ++i) {
      const int64_t a = std::min(p->dim, units * i / parts * unit), c = std::min(p->dim, units * (i + 1) / parts * unit);
      if (c > a) blk[n++] = {b, b + 1, a, c};
    }
  return n;
}

// The sub-problem of one block (device pointers offset into the full buffers).
ss_fwd_params host_block_params(const ss_fwd_params *p, const HostBlock &k) {
  ss_fwd_params q = *p;
  const int64_t es = elem_size(p->in_dtype), bs = elem_size(p->bc_dtype);
  const int64_t row0 = k.b0 * p->dim + k.d0;  // first (batch, channel) row of the block
  auto off = [&](const void *ptr, int64_t elems, int64_t size) -> const void * {
    return ptr ? static_cast<const char *>(ptr) + elems * size : nullptr;
  };
  q.batch = k.b1 - k.b0;
  q.dim = k.d1 - k.d0;
  q.u = off(p->u, row0 * p->seqlen, es);
  q.delta = off(p->delta, row0 * p->seqlen, es);
  q.z = off(p->z, row0 * p->seqlen, es);
  q.out = const_cast<void *>(off(p->out, row0 * p->seqlen, es));
  q.last_state = static_cast<float *>(const_cast<void *>(off(p->last_state, row0 * p->dstate, 4)));
  q.A = static_cast<const float *>(off(p->A, k.d0 * p->A_stride[0], 4));
  q.D = static_cast<const float *>(off(p->D, k.d0, 4));
  q.delta_bias = static_cast<const float *>(off(p->delta_bias, k.d0, 4));
  if (p->initial_state)
    q.initial_state = static_cast<const float *>(
        off(p->initial_state, k.b0 * p->initial_state_stride[0] + k.d0 * p->initial_state_stride[1], 4));
  if (p->bc_mode == SS_BC_FIXED) {
    q.B = off(p->B, k.d0 * p->B_stride[0], 4);
    q.C = off(p->C, k.d0 * p->C_stride[0], 4);
  } else {
    const int64_t dpg = p->dim / p->ngroups;
    const int64_t g0 = k.d0 / dpg, g1 = (k.d1 - 1) / dpg + 1;
    q.ngroups = g1 - g0;
    q.B = off(p->B, k.b0 * p->B_stride[0] + g0 * p->B_stride[1], bs);
    q.C = off(p->C, k.b0 * p->C_stride[0] + g0 * p->C_stride[1], bs);
  }
  return q;
}

// ---------------------------------------------------------------------------
// Decode step (ss_state_update)
// ---------------------------------------------------------------------------
int validate_su(const ss_state_update_params *p) {
  if (!p) return SS_ERR_NULL;
  if (p->abi_version != SS_ABI_VERSION) return SS_ERR_VERSION;
  if (p->in_dtype < SS_F32 || p->in_dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->bc_dtype < SS_F32 || p->bc_dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->bc_mode != SS_BC_FIXED && p->bc_mode != SS_BC_VARIABLE) return SS_ERR_SHAPE;
  const bool fixed = p->bc_mode == SS_BC_FIXED;
  if (fixed && p->bc_dtype != SS_F32) return SS_ERR_DTYPE;
  if (!fixed && p->bc_dtype != p->in_dtype && p->bc_dtype != SS_F32) return SS_ERR_DTYPE;
  if (p->batch < 0 || p->dim < 0) return SS_ERR_SHAPE;
  if (p->dstate < 1) return SS_ERR_SHAPE;
  if (p->dstate > 64) return SS_ERR_UNSUPPORTED;
  if (!fixed && (p->ngroups < 1 || (p->dim > 0 && p->dim % p->ngroups != 0))) return SS_ERR_SHAPE;
  if (p->batch > (int64_t(1) << 30) || p->dim > (int64_t(1) << 30) || p->batch * p->dim > (int64_t(1) << 40))
    return SS_ERR_UNSUPPORTED;
  if (p->batch * p->dim == 0) return SS_OK;
  if (!p->state || !p->u || !p->delta || !p->A || !p->B || !p->C || !p->out) return SS_ERR_NULL;
  if (p->state_stride[2] != 1 || p->state_stride[0] < 0 || p->state_stride[1] < 0) return SS_ERR_STRIDE;
  const int64_t *st2[4] = {p->u_stride, p->delta_stride, p->z ? p->z_stride : p->u_stride, p->out_stride};
  for (auto st : st2)
    if (st[0] < 0 || st[1] < 0) return SS_ERR_STRIDE;
  if (p->A_stride[1] != 1 || p->A_stride[0] < 0) return SS_ERR_STRIDE;
  if (fixed) {
    if (p->B_stride[1] != 1 || p->C_stride[1] != 1 || p->B_stride[0] < 0 || p->C_stride[0] < 0) return SS_ERR_STRIDE;
  } else {
    for (int i = 0; i < 3; ++i)
      if (p->B_stride[i] < 0 || p->C_stride[i] < 0) return SS_ERR_STRIDE;
    if (p->B_stride[2] != 1 || p->C_stride[2] != 1) return SS_ERR_STRIDE;
  }
  const int es = elem_size(p->in_dtype), bs = elem_size(p->bc_dtype);
  if (!aligned(p->u, es) || !aligned(p->delta, es) || !aligned(p->out, es) || (p->z && !aligned(p->z, es)))
    return SS_ERR_ALIGN;
  if (!aligned(p->B, bs) || !aligned(p->C, bs) || !aligned(p->A, 4) || !aligned(p->state, 4)) return SS_ERR_ALIGN;
  if ((p->D && !aligned(p->D, 4)) || (p->delta_bias && !aligned(p->delta_bias, 4))) return SS_ERR_ALIGN;
  const int64_t sz2[2] = {p->batch, p->dim};
  const int64_t szs[3] = {p->batch, p->dim, p->dstate};
  Range out = span(p->out, es, sz2, p->out_stride, 2);
  Range state = span(p->state, 4, szs, p->state_stride, 3);
  Range ins[8];
  int ni = 0;
  ins[ni++] = span(p->u, es, sz2, p->u_stride, 2);
  ins[ni++] = span(p->delta, es, sz2, p->delta_stride, 2);
  if (p->z) ins[ni++] = span(p->z, es, sz2, p->z_stride, 2);
  const int64_t sza[2] = {p->dim, p->dstate};
  ins[ni++] = span(p->A, 4, sza, p->A_stride, 2);
  if (fixed) {
    ins[ni++] = span(p->B, 4, sza, p->B_stride, 2);
    ins[ni++] = span(p->C, 4, sza, p->C_stride, 2);
  } else {
    const int64_t szb[3] = {p->batch, p->ngroups, p->dstate};
    ins[ni++] = span(p->B, bs, szb, p->B_stride, 3);
    ins[ni++] = span(p->C, bs, szb, p->C_stride, 3);
  }
  const int64_t one[1] = {p->dim}, unit[1] = {1};
  if (p->D) ins[ni++] = span(p->D, 4, one, unit, 1);
  if (p->delta_bias) ins[ni++] = span(p->delta_bias, 4, one, unit, 1);
  for (int i = 0; i < ni; ++i)
    if (overlap(out, ins[i]) || overlap(state, ins[i])) return SS_ERR_ALIAS;
  if (overlap(out, state)) return SS_ERR_ALIAS;
  return SS_OK;
}

int launch_su(const ss_state_update_params *p, cudaStream_t stream) {
  if (p->batch * p->dim == 0) return SS_OK;
  const bool fixed = p->bc_mode == SS_BC_FIXED;
  ssk::SUParams k{};
  k.batch = static_cast<int>(p->batch);
  k.dim = static_cast<int>(p->dim);
  k.dstate = static_cast<int>(p->dstate);
  k.dpg = fixed ? k.dim : static_cast<int>(p->dim / p->ngroups);
  k.fixed = fixed;
  k.has_z = p->z != nullptr;
  k.has_D = p->D != nullptr;
  k.has_bias = p->delta_bias != nullptr;
  k.softplus = p->delta_softplus != 0;
  k.state = p->state;
  k.u = p->u; k.delta = p->delta; k.z = p->z; k.B = p->B; k.C = p->C;
  k.A = p->A; k.D = p->D; k.bias = p->delta_bias;
  k.out = p->out;
  for (int i = 0; i < 3; ++i) k.sst[i] = p->state_stride[i];
  for (int i = 0; i < 2; ++i) {
    k.su[i] = p->u_stride[i]; k.sd[i] = p->delta_stride[i];
    k.sz[i] = p->z ? p->z_stride[i] : 0; k.so[i] = p->out_stride[i]; k.sA[i] = p->A_stride[i];
  }
  for (int i = 0; i < 3; ++i) { k.sB[i] = p->B_stride[i]; k.sC[i] = p->C_stride[i]; }
  // 16-byte state accesses when every row start is 16-byte aligned
  k.vec = aligned(p->state, 16) && (p->state_stride[0] % 4 == 0 || p->batch == 1) &&
          (p->state_stride[1] % 4 == 0 || p->dim == 1);
  k.avec = aligned(p->A, 16) && (p->A_stride[0] % 4 == 0 || p->dim == 1);
  {
    // B/C rows: 4 values of the lane = 16 (fp32) or 8 (16-bit) bytes
    const int bsz = elem_size(p->bc_dtype), need = 4 * bsz;
    auto row_ok = [&](const void *base, const int64_t *st) {
      if (!aligned(base, need)) return false;
      if (fixed) return p->dim == 1 || (st[0] * bsz) % need == 0;
      return (p->batch == 1 || (st[0] * bsz) % need == 0) && (p->ngroups == 1 || (st[1] * bsz) % need == 0);
    };
    k.bcvec = row_ok(p->B, p->B_stride) && row_ok(p->C, p->C_stride);
  }
  // groups of 4 states, rounded up to a power of two, split into lpc lanes
  // per channel of q groups each: 8 states a lane (q = 2) measured fastest on
  // decode130m_bf16 (18.9 us, against 20.5-21.2 with 4 and 23.3-23.8 with
  // 16), fewer lanes repeating the per-channel work; SSFWD_SU_Q overrides
  const int lanes = static_cast<int>((p->dstate + 3) / 4);
  const int l2 = lanes <= 1 ? 1 : lanes <= 2 ? 2 : lanes <= 4 ? 4 : lanes <= 8 ? 8 : 16;
  int q = 2;
  if (const char *e = std::getenv("SSFWD_SU_Q")) q = std::atoi(e) >= 4 ? 4 : (std::atoi(e) >= 2 ? 2 : 1);
  q = std::min(q, l2);
  const int lpc = l2 / q;
  const bool bc_f32 = fixed || p->bc_dtype == SS_F32;
  if (fault_injected("launch")) return SS_ERR_CUDA;
  void *args[1] = {&k};
  // grid: (channel tiles, batch rows [, batch rows beyond 65535])
  const void *fn = ssk::state_update_kernel(p->in_dtype, bc_f32, lpc, q);
  const int64_t gx = (p->dim + 256 / lpc - 1) / (256 / lpc);
  const int64_t gy = std::min<int64_t>(p->batch, 65535), gz = (p->batch + gy - 1) / gy;
  if (gx > 0x7fffffff || gz > 65535) return SS_ERR_UNSUPPORTED;
  return cudaLaunchKernel(fn, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(gz)),
                          dim3(256), args, 0, stream) == cudaSuccess
             ? SS_OK
             : SS_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Causal depthwise conv1d (ss_causal_conv1d, ss_causal_conv1d_update)
// ---------------------------------------------------------------------------
int validate_conv(const ss_conv1d_params *p) {
  if (!p) return SS_ERR_NULL;
  if (p->abi_version != SS_ABI_VERSION) return SS_ERR_VERSION;
  if (p->dtype < SS_F32 || p->dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->activation != SS_ACT_NONE && p->activation != SS_ACT_SILU) return SS_ERR_UNSUPPORTED;
  if (p->batch < 0 || p->dim < 0 || p->seqlen < 0 || p->width < 1) return SS_ERR_SHAPE;
  if (p->width < 2 || p->width > 4) return SS_ERR_UNSUPPORTED;
  if (p->batch > 65535 || p->dim > 65535 || p->seqlen > (int64_t(1) << 31) - 4096) return SS_ERR_UNSUPPORTED;
  if (p->seq_idx && (p->initial_states || p->final_states)) return SS_ERR_UNSUPPORTED;
  if (p->batch * p->dim == 0) return SS_OK;
  if (!p->weight || (p->seqlen > 0 && (!p->out || !p->x))) return SS_ERR_NULL;
  const int es = elem_size(p->dtype);
  if (p->x_stride[2] != 1 || p->out_stride[2] != 1 || p->weight_stride[1] != 1) return SS_ERR_STRIDE;
  for (int i = 0; i < 3; ++i)
    if (p->x_stride[i] < 0 || p->out_stride[i] < 0 || (p->initial_states && p->initial_states_stride[i] < 0) ||
        (p->final_states && p->final_states_stride[i] < 0))
      return SS_ERR_STRIDE;
  if (p->weight_stride[0] < 0 || (p->seq_idx && p->seq_idx_stride[0] < 0)) return SS_ERR_STRIDE;
  if (p->seq_idx && p->seq_idx_stride[1] != 1) return SS_ERR_STRIDE;
  if (!aligned(p->x, es) || !aligned(p->out, es) || !aligned(p->weight, 4) || (p->bias && !aligned(p->bias, 4)) ||
      (p->seq_idx && !aligned(p->seq_idx, 4)) || (p->initial_states && !aligned(p->initial_states, es)) ||
      (p->final_states && !aligned(p->final_states, es)))
    return SS_ERR_ALIGN;
  const int64_t sz3[3] = {p->batch, p->dim, p->seqlen}, szs[3] = {p->batch, p->dim, p->width - 1};
  const int64_t szw[2] = {p->dim, p->width}, szq[2] = {p->batch, p->seqlen}, one[1] = {p->dim}, unit[1] = {1};
  const Range out = span(p->out, es, sz3, p->out_stride, 3);
  const Range fin = p->final_states ? span(p->final_states, es, szs, p->final_states_stride, 3) : Range{0, 0};
  Range ins[5];
  int ni = 0;
  ins[ni++] = span(p->x, es, sz3, p->x_stride, 3);
  ins[ni++] = span(p->weight, 4, szw, p->weight_stride, 2);
  if (p->bias) ins[ni++] = span(p->bias, 4, one, unit, 1);
  if (p->seq_idx) ins[ni++] = span(p->seq_idx, 4, szq, p->seq_idx_stride, 2);
  if (p->initial_states) ins[ni++] = span(p->initial_states, es, szs, p->initial_states_stride, 3);
  for (int i = 0; i < ni; ++i)
    if (overlap(out, ins[i]) || overlap(fin, ins[i])) return SS_ERR_ALIAS;
  if (overlap(out, fin)) return SS_ERR_ALIAS;
  return SS_OK;
}

__global__ void conv_empty_final(ssk::ConvParams p, int es) {
  // seqlen == 0: final states are the initial states (or zeros)
  const int64_t total = (int64_t)p.batch * p.dim * (p.width - 1);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = i % (p.width - 1), r = i / (p.width - 1), d = r % p.dim, b = r / p.dim;
    unsigned char *dst = static_cast<unsigned char *>(p.fin) + (b * p.sf[0] + d * p.sf[1] + k * p.sf[2]) * es;
    const unsigned char *src = p.init ? static_cast<const unsigned char *>(p.init) + (b * p.si[0] + d * p.si[1] + k * p.si[2]) * es : nullptr;
    for (int j = 0; j < es; ++j) dst[j] = src ? src[j] : 0;
  }
}

int launch_conv(const ss_conv1d_params *p, cudaStream_t stream) {
  if (p->batch * p->dim == 0) return SS_OK;
  ssk::ConvParams k{};
  k.batch = static_cast<int>(p->batch);
  k.dim = static_cast<int>(p->dim);
  k.width = static_cast<int>(p->width);
  k.seqlen = p->seqlen;
  k.act = p->activation == SS_ACT_SILU;
  k.x = p->x; k.weight = p->weight; k.bias = p->bias; k.seq = p->seq_idx;
  k.init = p->initial_states; k.fin = p->final_states; k.out = p->out;
  for (int i = 0; i < 3; ++i) {
    k.sx[i] = p->x_stride[i]; k.so[i] = p->out_stride[i];
    k.si[i] = p->initial_states_stride[i]; k.sf[i] = p->final_states_stride[i];
  }
  for (int i = 0; i < 2; ++i) { k.sw[i] = p->weight_stride[i]; k.sq[i] = p->seq_idx_stride[i]; }
  const int es = elem_size(p->dtype);
  auto rows16 = [&](const void *base, const int64_t *st) {
    return aligned(base, 16) && (p->batch == 1 || (st[0] * es) % 16 == 0) && (p->dim == 1 || (st[1] * es) % 16 == 0);
  };
  k.xvec = rows16(p->x, p->x_stride);
  k.ovec = rows16(p->out, p->out_stride);
  if (fault_injected("launch")) return SS_ERR_CUDA;
  void *args[1] = {&k};
  if (p->seqlen == 0) {
    if (!p->final_states) return SS_OK;
    const int64_t total = p->batch * p->dim * (p->width - 1);
    const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 4096));
    void *a2[2] = {&k, const_cast<int *>(&es)};
    return cudaLaunchKernel(reinterpret_cast<const void *>(&conv_empty_final), dim3(blocks), dim3(256), a2, 0,
                            stream) == cudaSuccess
               ? SS_OK
               : SS_ERR_CUDA;
  }
  // 8 steps per thread (16 steps measured the same on 8192-step rows and
  // 18% slower on 2048-step rows)
  const int ept = 8;
  const void *fn = ssk::conv1d_kernel(p->dtype, ept, static_cast<int>(p->width), p->seq_idx != nullptr);
  const int64_t gx = (p->seqlen + 256 * ept - 1) / (256 * ept);
  if (gx > 0x7fffffff) return SS_ERR_UNSUPPORTED;
  return cudaLaunchKernel(fn, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(p->dim),
                                   static_cast<unsigned>(p->batch)),
                          dim3(256), args, 0, stream) == cudaSuccess
             ? SS_OK
             : SS_ERR_CUDA;
}

int validate_conv_update(const ss_conv1d_update_params *p) {
  if (!p) return SS_ERR_NULL;
  if (p->abi_version != SS_ABI_VERSION) return SS_ERR_VERSION;
  if (p->dtype < SS_F32 || p->dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->activation != SS_ACT_NONE && p->activation != SS_ACT_SILU) return SS_ERR_UNSUPPORTED;
  if (p->batch < 0 || p->dim < 0 || p->width < 1) return SS_ERR_SHAPE;
  if (p->width < 2 || p->width > 4) return SS_ERR_UNSUPPORTED;
  if (p->batch > 65535 || p->dim > (int64_t(1) << 30)) return SS_ERR_UNSUPPORTED;
  if (p->batch * p->dim == 0) return SS_OK;
  if (!p->x || !p->conv_state || !p->weight || !p->out) return SS_ERR_NULL;
  if (p->weight_stride[1] != 1) return SS_ERR_STRIDE;
  for (int i = 0; i < 2; ++i)
    if (p->x_stride[i] < 0 || p->out_stride[i] < 0 || p->weight_stride[i] < 0) return SS_ERR_STRIDE;
  for (int i = 0; i < 3; ++i)
    if (p->conv_state_stride[i] < 0) return SS_ERR_STRIDE;
  const int es = elem_size(p->dtype);
  if (!aligned(p->x, es) || !aligned(p->out, es) || !aligned(p->conv_state, es) || !aligned(p->weight, 4) ||
      (p->bias && !aligned(p->bias, 4)))
    return SS_ERR_ALIGN;
  const int64_t sz2[2] = {p->batch, p->dim}, szs[3] = {p->batch, p->dim, p->width - 1};
  const int64_t szw[2] = {p->dim, p->width}, one[1] = {p->dim}, unit[1] = {1};
  const Range out = span(p->out, es, sz2, p->out_stride, 2);
  const Range st = span(p->conv_state, es, szs, p->conv_state_stride, 3);
  Range ins[3];
  int ni = 0;
  ins[ni++] = span(p->x, es, sz2, p->x_stride, 2);
  ins[ni++] = span(p->weight, 4, szw, p->weight_stride, 2);
  if (p->bias) ins[ni++] = span(p->bias, 4, one, unit, 1);
  for (int i = 0; i < ni; ++i)
    if (overlap(out, ins[i]) || overlap(st, ins[i])) return SS_ERR_ALIAS;
  if (overlap(out, st)) return SS_ERR_ALIAS;
  return SS_OK;
}

int launch_conv_update(const ss_conv1d_update_params *p, cudaStream_t stream) {
  if (p->batch * p->dim == 0) return SS_OK;
  ssk::ConvUpdateParams k{};
  k.batch = static_cast<int>(p->batch);
  k.dim = static_cast<int>(p->dim);
  k.width = static_cast<int>(p->width);
  k.act = p->activation == SS_ACT_SILU;
  k.x = p->x; k.state = p->conv_state; k.weight = p->weight; k.bias = p->bias; k.out = p->out;
  for (int i = 0; i < 2; ++i) { k.sx[i] = p->x_stride[i]; k.sw[i] = p->weight_stride[i]; k.so[i] = p->out_stride[i]; }
  for (int i = 0; i < 3; ++i) k.ss[i] = p->conv_state_stride[i];
  if (fault_injected("launch")) return SS_ERR_CUDA;
  void *args[1] = {&k};
  const void *fn = ssk::conv1d_update_kernel(p->dtype, static_cast<int>(p->width));
  const int64_t gx = (p->dim + 255) / 256;
  return cudaLaunchKernel(fn, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(p->batch)), dim3(256), args, 0,
                          stream) == cudaSuccess
             ? SS_OK
             : SS_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Backward (ss_bwd)
// ---------------------------------------------------------------------------
int64_t bwd_chunks(int64_t seqlen) { return (seqlen + ssk::bwd_chunk_steps() - 1) / ssk::bwd_chunk_steps(); }

int64_t bwd_ws_bytes(const ss_bwd_params *p) {
  return p->batch * p->dim * bwd_chunks(p->seqlen) * p->dstate * 4;
}

// Everything except the workspace.
int validate_bwd_operands(const ss_bwd_params *p) {
  if (!p) return SS_ERR_NULL;
  if (p->abi_version != SS_ABI_VERSION) return SS_ERR_VERSION;
  if (p->in_dtype < SS_F32 || p->in_dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->bc_dtype < SS_F32 || p->bc_dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->bc_mode != SS_BC_FIXED && p->bc_mode != SS_BC_VARIABLE) return SS_ERR_SHAPE;
  const bool fixed = p->bc_mode == SS_BC_FIXED;
  if (fixed && p->bc_dtype != SS_F32) return SS_ERR_DTYPE;
  if (!fixed && p->bc_dtype != p->in_dtype && p->bc_dtype != SS_F32) return SS_ERR_DTYPE;
  if (p->batch < 0 || p->dim < 0 || p->seqlen < 0) return SS_ERR_SHAPE;
  if (p->dstate < 1) return SS_ERR_SHAPE;
  if (p->dstate > 64) return SS_ERR_UNSUPPORTED;
  if (!fixed && (p->ngroups < 1 || (p->dim > 0 && p->dim % p->ngroups != 0))) return SS_ERR_SHAPE;
  if (p->batch > (int64_t(1) << 24) || p->dim > (1 << 30) || p->seqlen > (int64_t(1) << 31) - 1024)
    return SS_ERR_UNSUPPORTED;
  if (p->batch * p->dim == 0) return SS_OK;
  if (!p->A || !p->dA) return SS_ERR_NULL;
  if ((fixed || p->seqlen > 0) && (!p->dB || !p->dC)) return SS_ERR_NULL;  // variable dB/dC are empty at seqlen 0
  if (p->A_stride[1] != 1 || p->A_stride[0] < 0) return SS_ERR_STRIDE;
  if (p->initial_state) {
    if (p->initial_state_stride[2] != 1 || p->initial_state_stride[0] < 0 || p->initial_state_stride[1] < 0)
      return SS_ERR_STRIDE;
    if (!aligned(p->initial_state, 4)) return SS_ERR_ALIGN;
  }
  const int es = elem_size(p->in_dtype), bs = elem_size(p->bc_dtype);
  const int64_t sz3[3] = {p->batch, p->dim, p->seqlen};
  const int64_t sza[2] = {p->dim, p->dstate};
  const int64_t szs[3] = {p->batch, p->dim, p->dstate};
  const int64_t one[1] = {p->dim}, unit[1] = {1};
  if (!aligned(p->A, 4) || !aligned(p->dA, 4) || !aligned(p->dB, 4) || !aligned(p->dC, 4)) return SS_ERR_ALIGN;
  if ((p->D && !aligned(p->D, 4)) || (p->delta_bias && !aligned(p->delta_bias, 4)) ||
      (p->dD && !aligned(p->dD, 4)) || (p->ddelta_bias && !aligned(p->ddelta_bias, 4)) ||
      (p->dinitial_state && !aligned(p->dinitial_state, 4)))
    return SS_ERR_ALIGN;
  if (p->seqlen > 0) {
    if (!p->u || !p->delta || !p->B || !p->C || !p->dout || !p->du || !p->ddelta) return SS_ERR_NULL;
    if (p->z && !p->dz) return SS_ERR_NULL;
    const int64_t *st3[7] = {p->u_stride, p->delta_stride, p->z ? p->z_stride : p->u_stride, p->dout_stride,
                             p->du_stride, p->ddelta_stride, p->z ? p->dz_stride : p->u_stride};
    for (auto st : st3)
      if (st[2] != 1 || st[0] < 0 || st[1] < 0) return SS_ERR_STRIDE;
    if (fixed) {
      if (p->B_stride[1] != 1 || p->C_stride[1] != 1 || p->B_stride[0] < 0 || p->C_stride[0] < 0)
        return SS_ERR_STRIDE;
    } else {
      for (int i = 0; i < 4; ++i)
        if (p->B_stride[i] < 0 || p->C_stride[i] < 0) return SS_ERR_STRIDE;
      if (p->B_stride[3] != 1 || p->C_stride[3] != 1) return SS_ERR_STRIDE;
    }
    if (!aligned(p->u, es) || !aligned(p->delta, es) || !aligned(p->dout, es) || !aligned(p->du, es) ||
        !aligned(p->ddelta, es) || (p->z && (!aligned(p->z, es) || !aligned(p->dz, es))))
      return SS_ERR_ALIGN;
    if (!aligned(p->B, bs) || !aligned(p->C, bs)) return SS_ERR_ALIGN;
  }
  // outputs must not overlap inputs, the workspace or each other
  Range ins[12], outs[10];
  int ni = 0, no = 0;
  const int64_t c2[2] = {p->dstate, 1};
  const int64_t c3[3] = {p->dim * p->dstate, p->dstate, 1};
  ins[ni++] = span(p->A, 4, sza, p->A_stride, 2);
  if (p->D) ins[ni++] = span(p->D, 4, one, unit, 1);
  if (p->delta_bias) ins[ni++] = span(p->delta_bias, 4, one, unit, 1);
  if (p->initial_state) ins[ni++] = span(p->initial_state, 4, szs, p->initial_state_stride, 3);
  outs[no++] = span(p->dA, 4, sza, c2, 2);
  if (p->dD) outs[no++] = span(p->dD, 4, one, unit, 1);
  if (p->ddelta_bias) outs[no++] = span(p->ddelta_bias, 4, one, unit, 1);
  if (p->dinitial_state) outs[no++] = span(p->dinitial_state, 4, szs, c3, 3);
  if (fixed) {
    if (p->seqlen > 0) {
      ins[ni++] = span(p->B, 4, sza, p->B_stride, 2);
      ins[ni++] = span(p->C, 4, sza, p->C_stride, 2);
    }
    outs[no++] = span(p->dB, 4, sza, c2, 2);
    outs[no++] = span(p->dC, 4, sza, c2, 2);
  } else {
    const int64_t szb[4] = {p->batch, p->ngroups, p->dstate, p->seqlen};
    const int64_t cb[4] = {p->ngroups * p->dstate * p->seqlen, p->dstate * p->seqlen, p->seqlen, 1};
    if (p->seqlen > 0) {
      ins[ni++] = span(p->B, bs, szb, p->B_stride, 4);
      ins[ni++] = span(p->C, bs, szb, p->C_stride, 4);
    }
    outs[no++] = span(p->dB, 4, szb, cb, 4);
    outs[no++] = span(p->dC, 4, szb, cb, 4);
  }
  if (p->seqlen > 0) {
    ins[ni++] = span(p->u, es, sz3, p->u_stride, 3);
    ins[ni++] = span(p->delta, es, sz3, p->delta_stride, 3);
    ins[ni++] = span(p->dout, es, sz3, p->dout_stride, 3);
    if (p->z) ins[ni++] = span(p->z, es, sz3, p->z_stride, 3);
    outs[no++] = span(p->du, es, sz3, p->du_stride, 3);
    outs[no++] = span(p->ddelta, es, sz3, p->ddelta_stride, 3);
    if (p->z) outs[no++] = span(p->dz, es, sz3, p->dz_stride, 3);
  }
  for (int o = 0; o < no; ++o) {
    for (int i = 0; i < ni; ++i)
      if (overlap(outs[o], ins[i])) return SS_ERR_ALIAS;
    for (int q = o + 1; q < no; ++q)
      if (overlap(outs[o], outs[q])) return SS_ERR_ALIAS;
  }
  if (p->workspace && p->workspace_bytes > 0) {
    const Range ws{reinterpret_cast<uintptr_t>(p->workspace),
                   reinterpret_cast<uintptr_t>(p->workspace) + static_cast<uintptr_t>(p->workspace_bytes)};
    for (int i = 0; i < ni; ++i)
      if (overlap(ws, ins[i])) return SS_ERR_ALIAS;
    for (int o = 0; o < no; ++o)
      if (overlap(ws, outs[o])) return SS_ERR_ALIAS;
  }
  return SS_OK;
}

int validate_bwd(const ss_bwd_params *p) {
  const int st = validate_bwd_operands(p);
  if (st != SS_OK) return st;
  if (p->workspace_bytes < 0) return SS_ERR_SHAPE;
  if (p->batch * p->dim == 0 || p->seqlen == 0) return SS_OK;
  if (!p->workspace || p->workspace_bytes < bwd_ws_bytes(p)) return SS_ERR_SCRATCH;
  if (!aligned(p->workspace, 16)) return SS_ERR_ALIGN;
  return SS_OK;
}

int launch_bwd(const ss_bwd_params *p, cudaStream_t stream) {
  if (p->batch * p->dim == 0) return SS_OK;
  const bool fixed = p->bc_mode == SS_BC_FIXED;
  if (fault_injected("launch")) return SS_ERR_CUDA;
  // the reduced gradients are sums of atomic additions: start from zero
  const int64_t nbc = fixed ? p->dim * p->dstate : p->batch * p->ngroups * p->dstate * p->seqlen;
  bool ok = cudaMemsetAsync(p->dA, 0, p->dim * p->dstate * 4, stream) == cudaSuccess;
  if (ok && nbc > 0)
    ok = cudaMemsetAsync(p->dB, 0, nbc * 4, stream) == cudaSuccess &&
         cudaMemsetAsync(p->dC, 0, nbc * 4, stream) == cudaSuccess;
  if (ok && p->dD) ok = cudaMemsetAsync(p->dD, 0, p->dim * 4, stream) == cudaSuccess;
  if (ok && p->ddelta_bias) ok = cudaMemsetAsync(p->ddelta_bias, 0, p->dim * 4, stream) == cudaSuccess;
  if (!ok) return SS_ERR_CUDA;
  if (p->seqlen == 0) {
    if (p->dinitial_state &&
        cudaMemsetAsync(p->dinitial_state, 0, p->batch * p->dim * p->dstate * 4, stream) != cudaSuccess)
      return SS_ERR_CUDA;
    return SS_OK;
  }
  ssk::BwdParams k{};
  k.batch = static_cast<int>(p->batch);
  k.dim = static_cast<int>(p->dim);
  k.dstate = static_cast<int>(p->dstate);
  k.ngroups = fixed ? 1 : static_cast<int>(p->ngroups);
  k.dpg = k.dim / k.ngroups;
  const int rows = ssk::bwd_rows_per_cta();
  k.tiles = (k.dpg + rows - 1) / rows;
  k.seqlen = static_cast<int>(p->seqlen);
  k.nch = static_cast<int>(bwd_chunks(p->seqlen));
  k.has_z = p->z != nullptr;
  k.softplus = p->delta_softplus != 0;
  k.u = p->u; k.delta = p->delta; k.z = p->z; k.B = p->B; k.C = p->C; k.dout = p->dout;
  k.A = p->A; k.D = p->D; k.bias = p->delta_bias; k.init = p->initial_state;
  k.du = p->du; k.ddelta = p->ddelta; k.dz = p->dz;
  k.dA = p->dA; k.dB = p->dB; k.dC = p->dC; k.dD = p->dD; k.dbias = p->ddelta_bias; k.dx0 = p->dinitial_state;
  k.ws = static_cast<float *>(p->workspace);
  for (int i = 0; i < 2; ++i) {
    k.su[i] = p->u_stride[i]; k.sd[i] = p->delta_stride[i]; k.sg[i] = p->dout_stride[i];
    k.sz[i] = p->z ? p->z_stride[i] : 0; k.sdz[i] = p->z ? p->dz_stride[i] : 0;
    k.sdu[i] = p->du_stride[i]; k.sdd[i] = p->ddelta_stride[i];
    k.si[i] = p->initial_state ? p->initial_state_stride[i] : 0;
  }
  for (int i = 0; i < 3; ++i) { k.sB[i] = p->B_stride[i]; k.sC[i] = p->C_stride[i]; }
  k.sA = p->A_stride[0];
  // 16-byte accesses of 8 steps: every row start 16-byte aligned
  const int es = elem_size(p->in_dtype), bs = elem_size(p->bc_dtype);
  auto rows_ok = [&](const void *ptr, const int64_t *st, int esz) {
    return aligned(ptr, 16) && (p->batch == 1 || (st[0] * esz) % 16 == 0) && (p->dim == 1 || (st[1] * esz) % 16 == 0);
  };
  k.vec = rows_ok(p->u, p->u_stride, es) && rows_ok(p->delta, p->delta_stride, es) &&
          rows_ok(p->dout, p->dout_stride, es) && rows_ok(p->du, p->du_stride, es) &&
          rows_ok(p->ddelta, p->ddelta_stride, es) &&
          (!p->z || (rows_ok(p->z, p->z_stride, es) && rows_ok(p->dz, p->dz_stride, es)));
  k.bcvec = !fixed && aligned(p->B, 16) && aligned(p->C, 16);
  for (int i = 0; i < 3 && k.bcvec; ++i)
    k.bcvec = (p->B_stride[i] * bs) % 16 == 0 && (p->C_stride[i] * bs) % 16 == 0;
  k.dbvec = !fixed && aligned(p->dB, 16) && aligned(p->dC, 16) && p->seqlen % 4 == 0;
  const bool bc_f32 = fixed || p->bc_dtype == SS_F32;
  const ssk::BwdKernel ki = ssk::bwd_kernel(p->in_dtype, bc_f32, fixed, k.dstate);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SS_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    bool &done = g_bwd_attr_done[dev][p->in_dtype][bc_f32][fixed];
    if (!done && ki.smem > 0) {
      if (cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem) != cudaSuccess)
        return SS_ERR_CUDA;
      done = true;
    }
  }
  const int64_t gx = static_cast<int64_t>(k.ngroups) * k.tiles;
  const int64_t gy = std::min<int64_t>(p->batch, 65535), gz = (p->batch + gy - 1) / gy;
  if (gx > 0x7fffffff || gz > 65535) return SS_ERR_UNSUPPORTED;
  void *args[1] = {&k};
  return cudaLaunchKernel(ki.fn, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(gz)),
                          dim3(ssk::bwd_threads()), args, ki.smem, stream) == cudaSuccess
             ? SS_OK
             : SS_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Complex-A forward (ss_fwd_complex)
// ---------------------------------------------------------------------------
int validate_cx(const ss_fwd_complex_params *p) {
  if (!p) return SS_ERR_NULL;
  if (p->abi_version != SS_ABI_VERSION) return SS_ERR_VERSION;
  if (p->in_dtype < SS_F32 || p->in_dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->bc_dtype < SS_F32 || p->bc_dtype > SS_BF16) return SS_ERR_DTYPE;
  if (p->bc_mode != SS_BC_FIXED && p->bc_mode != SS_BC_VARIABLE) return SS_ERR_SHAPE;
  const bool fixed = p->bc_mode == SS_BC_FIXED;
  if (fixed && p->bc_dtype != SS_F32) return SS_ERR_DTYPE;
  if (!fixed && p->bc_dtype != p->in_dtype && p->bc_dtype != SS_F32) return SS_ERR_DTYPE;
  if (p->batch < 0 || p->dim < 0 || p->seqlen < 0) return SS_ERR_SHAPE;
  if (p->dstate < 1) return SS_ERR_SHAPE;
  if (p->dstate > 64) return SS_ERR_UNSUPPORTED;
  if (!fixed && (p->ngroups < 1 || (p->dim > 0 && p->dim % p->ngroups != 0))) return SS_ERR_SHAPE;
  if (p->batch > (int64_t(1) << 24) || p->dim > (1 << 30) || p->seqlen > (int64_t(1) << 31) - 1024)
    return SS_ERR_UNSUPPORTED;
  if (p->batch * p->dim == 0) return SS_OK;
  const int64_t szl[3] = {p->batch, p->dim, p->dstate};
  Range last{0, 0}, init{0, 0};
  if (p->last_state) {
    if (p->last_state_stride[2] != 1 || p->last_state_stride[0] < 0 || p->last_state_stride[1] < 0)
      return SS_ERR_STRIDE;
    if (!aligned(p->last_state, 8)) return SS_ERR_ALIGN;
    last = span(p->last_state, 8, szl, p->last_state_stride, 3);
  }
  if (p->initial_state) {
    if (p->initial_state_stride[2] != 1 || p->initial_state_stride[0] < 0 || p->initial_state_stride[1] < 0)
      return SS_ERR_STRIDE;
    if (!aligned(p->initial_state, 8)) return SS_ERR_ALIGN;
    init = span(p->initial_state, 8, szl, p->initial_state_stride, 3);
    const bool same = p->last_state == p->initial_state && p->last_state_stride[0] == p->initial_state_stride[0] &&
                      p->last_state_stride[1] == p->initial_state_stride[1];
    if (!same && overlap(init, last)) return SS_ERR_ALIAS;
  }
  if (p->seqlen == 0) return SS_OK;
  if (!p->u || !p->delta || !p->A || !p->B || !p->C || !p->out) return SS_ERR_NULL;
  const int64_t *st3[4] = {p->u_stride, p->delta_stride, p->z ? p->z_stride : p->u_stride, p->out_stride};
  for (auto st : st3)
    if (st[2] != 1 || st[0] < 0 || st[1] < 0) return SS_ERR_STRIDE;
  if (p->A_stride[1] != 1 || p->A_stride[0] < 0) return SS_ERR_STRIDE;
  if (fixed) {
    if (p->B_stride[1] != 1 || p->C_stride[1] != 1 || p->B_stride[0] < 0 || p->C_stride[0] < 0) return SS_ERR_STRIDE;
  } else {
    for (int i = 0; i < 4; ++i)
      if (p->B_stride[i] < 0 || p->C_stride[i] < 0) return SS_ERR_STRIDE;
    if (p->B_stride[3] != 1 || p->C_stride[3] != 1) return SS_ERR_STRIDE;
  }
  const int es = elem_size(p->in_dtype), bs = elem_size(p->bc_dtype);
  if (!aligned(p->u, es) || !aligned(p->delta, es) || !aligned(p->out, es) || (p->z && !aligned(p->z, es)))
    return SS_ERR_ALIGN;
  if (!aligned(p->B, bs) || !aligned(p->C, bs) || !aligned(p->A, 8)) return SS_ERR_ALIGN;
  if ((p->D && !aligned(p->D, 4)) || (p->delta_bias && !aligned(p->delta_bias, 4))) return SS_ERR_ALIGN;
  const int64_t sz3[3] = {p->batch, p->dim, p->seqlen};
  Range out = span(p->out, es, sz3, p->out_stride, 3);
  Range ins[9];
  int ni = 0;
  ins[ni++] = span(p->u, es, sz3, p->u_stride, 3);
  ins[ni++] = span(p->delta, es, sz3, p->delta_stride, 3);
  if (p->z) ins[ni++] = span(p->z, es, sz3, p->z_stride, 3);
  const int64_t sza[2] = {p->dim, p->dstate};
  ins[ni++] = span(p->A, 8, sza, p->A_stride, 2);
  if (fixed) {
    ins[ni++] = span(p->B, 4, sza, p->B_stride, 2);
    ins[ni++] = span(p->C, 4, sza, p->C_stride, 2);
  } else {
    const int64_t szb[4] = {p->batch, p->ngroups, p->dstate, p->seqlen};
    ins[ni++] = span(p->B, bs, szb, p->B_stride, 4);
    ins[ni++] = span(p->C, bs, szb, p->C_stride, 4);
  }
  const int64_t one[1] = {p->dim}, unit[1] = {1};
  if (p->D) ins[ni++] = span(p->D, 4, one, unit, 1);
  if (p->delta_bias) ins[ni++] = span(p->delta_bias, 4, one, unit, 1);
  for (int i = 0; i < ni; ++i)
    if (overlap(out, ins[i]) || overlap(last, ins[i])) return SS_ERR_ALIAS;
  if (overlap(out, last) || overlap(out, init)) return SS_ERR_ALIAS;
  return SS_OK;
}

__global__ void complex_empty_state(float *last, const float *init, long long s0, long long s1, long long s2i0,
                                    long long s2i1, int batch, int dim, int dstate) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= (long long)batch * dim * dstate) return;
  const int n = i % dstate, d = (i / dstate) % dim, b = i / ((long long)dstate * dim);
  const long long o = 2 * (b * s0 + d * s1 + n);
  const long long q = 2 * (b * s2i0 + d * s2i1 + n);
  last[o] = init ? init[q] : 0.f;
  last[o + 1] = init ? init[q + 1] : 0.f;
}

int launch_cx(const ss_fwd_complex_params *p, cudaStream_t stream) {
  if (p->batch * p->dim == 0) return SS_OK;
  if (fault_injected("launch")) return SS_ERR_CUDA;
  if (p->seqlen == 0) {
    if (!p->last_state || p->last_state == p->initial_state) return SS_OK;
    const long long n = p->batch * p->dim * p->dstate;
    complex_empty_state<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
        p->last_state, p->initial_state, p->last_state_stride[0], p->last_state_stride[1],
        p->initial_state ? p->initial_state_stride[0] : 0, p->initial_state ? p->initial_state_stride[1] : 0,
        static_cast<int>(p->batch), static_cast<int>(p->dim), static_cast<int>(p->dstate));
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
  }
  const bool fixed = p->bc_mode == SS_BC_FIXED;
  ssk::CxParams k{};
  k.batch = static_cast<int>(p->batch);
  k.dim = static_cast<int>(p->dim);
  k.dstate = static_cast<int>(p->dstate);
  k.ngroups = fixed ? 1 : static_cast<int>(p->ngroups);
  k.dpg = k.dim / k.ngroups;
  const int cpc = ssk::cx_channels_per_cta();
  k.tiles = (k.dpg + cpc - 1) / cpc;
  k.seqlen = static_cast<int>(p->seqlen);
  k.nseg = static_cast<int>((p->seqlen + ssk::cx_segment_steps() - 1) / ssk::cx_segment_steps());
  k.has_z = p->z != nullptr;
  k.softplus = p->delta_softplus != 0;
  k.u = p->u; k.delta = p->delta; k.z = p->z; k.B = p->B; k.C = p->C;
  k.A = p->A; k.D = p->D; k.bias = p->delta_bias; k.init = p->initial_state;
  k.out = p->out; k.last = p->last_state;
  for (int i = 0; i < 2; ++i) {
    k.su[i] = p->u_stride[i]; k.sd[i] = p->delta_stride[i]; k.so[i] = p->out_stride[i];
    k.sz[i] = p->z ? p->z_stride[i] : 0;
    k.si[i] = p->initial_state ? p->initial_state_stride[i] : 0;
    k.sl[i] = p->last_state ? p->last_state_stride[i] : 0;
  }
  for (int i = 0; i < 3; ++i) { k.sB[i] = p->B_stride[i]; k.sC[i] = p->C_stride[i]; }
  k.sA = p->A_stride[0];
  {
    const int bs = elem_size(p->bc_dtype);
    k.bcvec = !fixed && aligned(p->B, 16) && aligned(p->C, 16);
    for (int i = 0; i < 3 && k.bcvec; ++i) k.bcvec = (p->B_stride[i] * bs) % 16 == 0 && (p->C_stride[i] * bs) % 16 == 0;
  }
  const bool bc_f32 = fixed || p->bc_dtype == SS_F32;
  const void *fn = ssk::cx_kernel(p->in_dtype, bc_f32, fixed, k.dstate);
  const int64_t gx = static_cast<int64_t>(k.ngroups) * k.tiles;
  const int64_t gy = std::min<int64_t>(p->batch, 65535), gz = (p->batch + gy - 1) / gy;
  if (gx > 0x7fffffff || gz > 65535) return SS_ERR_UNSUPPORTED;
  void *args[1] = {&k};
  return cudaLaunchKernel(fn, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(gz)),
                          dim3(ssk::cx_threads()), args, 0, stream) == cudaSuccess
             ? SS_OK
             : SS_ERR_CUDA;
}

}  // namespace

extern "C" {

int ss_abi_version(void) { return SS_ABI_VERSION; }

const char *ss_status_string(int s) {
  switch (s) {
    case SS_OK: return "ok";
    case SS_ERR_NULL: return "a required pointer is NULL";
    case SS_ERR_SHAPE: return "invalid shape (negative size, dstate < 1, or dim not divisible by ngroups)";
    case SS_ERR_DTYPE: return "unsupported dtype or dtype combination";
    case SS_ERR_STRIDE: return "unsupported stride (the seqlen/state stride must be 1; strides must be >= 0)";
    case SS_ERR_ALIGN: return "pointer not aligned to its element size";
    case SS_ERR_ALIAS: return "an output overlaps an input or the other output";
    case SS_ERR_UNSUPPORTED: return "unsupported size (dstate > 64, batch > 65535, or too large)";
    case SS_ERR_CUDA: return "a CUDA call failed";
    case SS_ERR_INTERNAL: return "a device-side self-check failed";
    case SS_ERR_VERSION: return "ABI version mismatch";
    case SS_ERR_SCRATCH:
      return "not enough scratch: ss_fwd_noalloc's static buffer (SS_NOALLOC_MAX_SCRATCH bytes) is too "
             "small for the problem (call ss_fwd with a workspace), or ss_bwd's workspace is missing or "
             "smaller than ss_bwd_workspace_size";
    default: return "unknown status";
  }
}

int ss_fwd_validate(const ss_fwd_params *p) { return validate(p); }

int ss_fwd_workspace_size(const ss_fwd_params *p, int64_t *bytes) {
  if (!bytes) return SS_ERR_NULL;
  *bytes = 0;
  int st = validate(p);
  if (st != SS_OK) return st;
  return workspace_bytes(p, bytes);
}

int ss_fwd(const ss_fwd_params *p, void *stream) {
  int st = validate(p);
  if (st != SS_OK) return st;
  return launch(p, static_cast<cudaStream_t>(stream), p->workspace, p->workspace_bytes);
}

int ss_fwd_noalloc(const ss_fwd_params *p, void *stream) {
  if (!p) return SS_ERR_NULL;
  if (p->abi_version != SS_ABI_VERSION) return SS_ERR_VERSION;
  // The caller's workspace fields play no part here: validate and run a copy
  // without them, so a stale pointer left there cannot cause an alias error.
  ss_fwd_params q = *p;
  q.workspace = nullptr;
  q.workspace_bytes = 0;
  int st = validate(&q);
  if (st != SS_OK) return st;
  // Every call looks the scratch address up (cached after the first on each
  // device), so any first call, even an empty one, prepares the device.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
  void *scratch = noalloc_scratch(dev);
  if (!scratch) return SS_ERR_CUDA;
  int64_t need = 0;
  st = workspace_bytes(&q, &need, SS_NOALLOC_MAX_SCRATCH);
  if (st != SS_OK) return st;
  if (need > SS_NOALLOC_MAX_SCRATCH) return SS_ERR_SCRATCH;
  // The summaries are fully written by the summary pass before the forward
  // pass reads them, so the buffer needs no clearing between calls.
  return launch(&q, static_cast<cudaStream_t>(stream), need > 0 ? scratch : nullptr, need);
}

int ss_fwd_host(const ss_fwd_params *p, const void *h_u, const void *h_delta, const void *h_z, const void *h_B,
                const void *h_C, const float *h_A, const float *h_D, const float *h_delta_bias, void *h_out,
                float *h_last_state, void *stream) {
  int st = validate(p);
  if (st != SS_OK) return st;
  if (!host_layout_ok(p)) return SS_ERR_STRIDE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t es = elem_size(p->in_dtype), bs = elem_size(p->bc_dtype);
  const size_t nbc = p->bc_mode == SS_BC_FIXED ? static_cast<size_t>(p->dim * p->dstate)
                                               : static_cast<size_t>(p->batch * p->ngroups * p->dstate * p->seqlen);
  struct Copy {
    void *dst;
    const void *src;
    size_t bytes;
  };
  // inputs that every block reads whole: B, C, A, D, delta_bias
  const Copy shared_in[5] = {{const_cast<void *>(p->B), h_B, nbc * bs},
                             {const_cast<void *>(p->C), h_C, nbc * bs},
                             {const_cast<float *>(p->A), h_A, static_cast<size_t>(p->dim * p->dstate) * 4},
                             {const_cast<float *>(p->D), h_D, static_cast<size_t>(p->dim) * 4},
                             {const_cast<float *>(p->delta_bias), h_delta_bias, static_cast<size_t>(p->dim) * 4}};
  for (const Copy &c : shared_in)
    if (c.src && c.bytes && !c.dst) return SS_ERR_NULL;
  if (h_z && !p->z) return SS_ERR_NULL;
  if (fault_injected("h2d")) return SS_ERR_CUDA;
  if (p->batch * p->dim == 0) return SS_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
  HostPipe *hp = host_pipe(dev);
  if (!hp) return SS_ERR_CUDA;
  HostBlock blk[kHostBlocksMax];
  const int nblk = host_blocks(p, blk);
  std::lock_guard<std::mutex> lk(hp->mu);
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // on a failure after the fork, the caller's stream still waits for whatever
  // the copy streams already hold, so no copy outlives the call's ordering
  auto fail = [&](int code) -> int {
    if (ok(cudaEventRecord(hp->join, hp->in))) (void)cudaStreamWaitEvent(s, hp->join, 0);
    if (ok(cudaEventRecord(hp->join, hp->out))) (void)cudaStreamWaitEvent(s, hp->join, 0);
    return code;
  };
  // fork: the copy streams start after the work already on the caller's stream
  if (!ok(cudaEventRecord(hp->fork, s)) || !ok(cudaStreamWaitEvent(hp->in, hp->fork, 0)) ||
      !ok(cudaStreamWaitEvent(hp->out, hp->fork, 0)))
    return SS_ERR_CUDA;
  for (const Copy &c : shared_in)
    if (c.src && c.bytes && !ok(cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyHostToDevice, hp->in)))
      return fail(SS_ERR_CUDA);
  const char *hin[3] = {static_cast<const char *>(h_u), static_cast<const char *>(h_delta),
                        static_cast<const char *>(h_z)};
  const void *din[3] = {p->u, p->delta, p->z};
  for (int i = 0; i < nblk; ++i) {
    const HostBlock &k = blk[i];
    const size_t row0 = static_cast<size_t>(k.b0 * p->dim + k.d0);
    const size_t rows = static_cast<size_t>((k.b1 - k.b0) * (k.d1 - k.d0));
    const size_t o = row0 * p->seqlen * es, n = rows * p->seqlen * es;
    for (int t = 0; t < 3; ++t) {
      if (!hin[t] || n == 0) continue;
      if (!ok(cudaMemcpyAsync(static_cast<char *>(const_cast<void *>(din[t])) + o, hin[t] + o, n,
                              cudaMemcpyHostToDevice, hp->in)))
        return fail(SS_ERR_CUDA);
    }
    if (!ok(cudaEventRecord(hp->in_done[i], hp->in)) || !ok(cudaStreamWaitEvent(s, hp->in_done[i], 0)))
      return fail(SS_ERR_CUDA);
    const ss_fwd_params q = host_block_params(p, k);
    st = launch(&q, s, p->workspace, p->workspace_bytes);
    if (st != SS_OK) return fail(st);
    if (!ok(cudaEventRecord(hp->k_done[i], s)) || !ok(cudaStreamWaitEvent(hp->out, hp->k_done[i], 0)))
      return fail(SS_ERR_CUDA);
    if (h_out && n && !ok(cudaMemcpyAsync(static_cast<char *>(h_out) + o, static_cast<const char *>(p->out) + o, n,
                                          cudaMemcpyDeviceToHost, hp->out)))
      return fail(SS_ERR_CUDA);
    if (h_last_state && p->last_state) {
      const size_t lo = row0 * p->dstate * 4, ln = rows * p->dstate * 4;
      if (ln && !ok(cudaMemcpyAsync(reinterpret_cast<char *>(h_last_state) + lo,
                                    reinterpret_cast<const char *>(p->last_state) + lo, ln, cudaMemcpyDeviceToHost,
                                    hp->out)))
        return fail(SS_ERR_CUDA);
    }
  }
  // join: the caller's stream completes after the last copy back
  if (!ok(cudaEventRecord(hp->join, hp->out)) || !ok(cudaStreamWaitEvent(s, hp->join, 0))) return SS_ERR_CUDA;
  return SS_OK;
}

int ss_state_update_validate(const ss_state_update_params *p) { return validate_su(p); }

int ss_state_update(const ss_state_update_params *p, void *stream) {
  int st = validate_su(p);
  if (st != SS_OK) return st;
  return launch_su(p, static_cast<cudaStream_t>(stream));
}

int ss_causal_conv1d_validate(const ss_conv1d_params *p) { return validate_conv(p); }

int ss_causal_conv1d(const ss_conv1d_params *p, void *stream) {
  int st = validate_conv(p);
  if (st != SS_OK) return st;
  return launch_conv(p, static_cast<cudaStream_t>(stream));
}

int ss_causal_conv1d_update_validate(const ss_conv1d_update_params *p) { return validate_conv_update(p); }

int ss_causal_conv1d_update(const ss_conv1d_update_params *p, void *stream) {
  int st = validate_conv_update(p);
  if (st != SS_OK) return st;
  return launch_conv_update(p, static_cast<cudaStream_t>(stream));
}

int ss_bwd_validate(const ss_bwd_params *p) { return validate_bwd(p); }

int ss_bwd_workspace_size(const ss_bwd_params *p, int64_t *bytes) {
  if (!bytes) return SS_ERR_NULL;
  const int st = validate_bwd_operands(p);
  if (st != SS_OK) return st;
  *bytes = bwd_ws_bytes(p);
  return SS_OK;
}

int ss_bwd(const ss_bwd_params *p, void *stream) {
  const int st = validate_bwd(p);
  if (st != SS_OK) return st;
  return launch_bwd(p, static_cast<cudaStream_t>(stream));
}

int ss_fwd_complex_validate(const ss_fwd_complex_params *p) { return validate_cx(p); }

int ss_fwd_complex(const ss_fwd_complex_params *p, void *stream) {
  const int st = validate_cx(p);
  if (st != SS_OK) return st;
  return launch_cx(p, static_cast<cudaStream_t>(stream));
}

int ss_device_error(int32_t *out_word, int clear) {
  if (!out_word) return SS_ERR_NULL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
  int32_t *ptr = error_word_ptr(dev);
  if (!ptr) return SS_ERR_CUDA;
  if (cudaMemcpy(out_word, ptr, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return SS_ERR_CUDA;
  if (clear && cudaMemset(ptr, 0, sizeof(int32_t)) != cudaSuccess) return SS_ERR_CUDA;
  return SS_OK;
}

}  // extern "C"
