// K4: the delayed-scaling state update, one CTA per FP8 tensor slot.
//
// After a step, each tensor's running amax joins the front of its rolling
// history, the window is reduced by "max" and the next step's scale is
// fp8_max / that max (TE tutorial, code block 1: DelayedScaling with
// amax_history_len and amax_compute_algo="max"; code block 4 prints
// amax_history[0] as the newest row). A zero or non-finite window, or a scale
// that overflows, keeps the previous scale. fp32 division is IEEE
// round-to-nearest (the library is built without fast-math), so scale and
// scale_inv are reproducible bit for bit.
#include "common.cuh"
#include "internal.h"
#include "state_update.cuh"

namespace lnfp8 {
namespace {

constexpr int kThreads = 256;

struct UpdateSet {
  float* scale;
  float* scale_inv;
  float* hist;
  float* cur;
  float* sinv_before;
  uint64_t e5m2_mask;
  int n, L;
};
struct UpdateTable {
  UpdateSet set[kMaxUpdateSets];
  int first[kMaxUpdateSets];  // first CTA of each set
  int count, margin;
};

__global__ void __launch_bounds__(kThreads)
update_kernel(float* __restrict__ scale, float* __restrict__ scale_inv, float* __restrict__ hist,
              float* __restrict__ cur, int n, int L, uint64_t e5m2_mask, int margin,
              float* __restrict__ sinv_before) {
  extern __shared__ float shist[];  // the new window of this slot, L floats
  __shared__ uint32_t red[kThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x;
  update_slot(scale, scale_inv, hist, cur, n, L, i, (e5m2_mask >> i) & 1ull, margin, sinv_before, shist, red);
}

// Several tensor sets (e.g. every layer of a model, updated after the step) in
// one launch: CTA b updates slot b - first[s] of set s.
__global__ void __launch_bounds__(kThreads) update_many_kernel(const UpdateTable tab) {
  extern __shared__ float shist[];
  __shared__ uint32_t red[kThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  int s = 0;
  while (s + 1 < tab.count && (int)blockIdx.x >= tab.first[s + 1]) ++s;
  const UpdateSet& u = tab.set[s];
  const int i = blockIdx.x - tab.first[s];
  update_slot(u.scale, u.scale_inv, u.hist, u.cur, u.n, u.L, i, (u.e5m2_mask >> i) & 1ull, tab.margin,
              u.sinv_before, shist, red);
}

__global__ void init_kernel(float* scale, float* scale_inv, float* hist, float* cur, int n, int L) {
  const int64_t total = (int64_t)n * L;
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < total; k += (int64_t)gridDim.x * blockDim.x) {
    hist[k] = 0.f;
    if (k < n) {
      scale[k] = 1.f;
      scale_inv[k] = 1.f;
      cur[k] = 0.f;
    }
  }
}

}  // namespace

lnfp8_status validate_meta(const lnfp8_meta* m, int expect_n, const char* who) {
  if (!m) return set_error(LNFP8_ERR_INVALID_ARG, "%s: meta is NULL", who);
  if (m->n < 1 || m->n > 64 || (expect_n > 0 && m->n != expect_n))
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: meta.n = %d (expected %d)", who, m->n, expect_n);
  if (m->history_len < 1 || m->history_len > 16384)
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: meta.history_len = %d (1..16384)", who, m->history_len);
  if (!m->scale || !m->scale_inv || !m->amax_history || !m->amax_cur)
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: a meta pointer is NULL", who);
  return LNFP8_OK;
}

lnfp8_status meta_init_launch(const lnfp8_meta* m, cudaStream_t st) {
  const int64_t total = (int64_t)m->n * m->history_len;
  const int blocks = (int)min64((total + 255) / 256, 1024);
  LaunchScope ls("state_init", st);
  init_kernel<<<blocks, 256, 0, st>>>(m->scale, m->scale_inv, m->amax_history, m->amax_cur, m->n, m->history_len);
  return check_launch("lnfp8_meta_init");
}

UpdateJob update_job(const lnfp8_meta* m, uint64_t e5m2_mask, int margin) {
  return UpdateJob{m->scale, m->scale_inv, m->amax_history, m->amax_cur, e5m2_mask, m->n, m->history_len, margin};
}

lnfp8_status update_launch(const lnfp8_meta* m, uint64_t e5m2_mask, int margin, float* sinv_before,
                           cudaStream_t st) {
  const size_t smem = (size_t)m->history_len * sizeof(float);
  if (smem + 1024 > 48 * 1024) {
    if (cudaFuncSetAttribute(update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return check_launch("amax_history_update: smem attribute");
  }
  LaunchScope ls("state_update", st);
  if (launch_pdl(update_kernel, dim3(m->n), dim3(kThreads), smem, st, m->scale, m->scale_inv, m->amax_history,
                 m->amax_cur, m->n, m->history_len, e5m2_mask, margin, sinv_before) != cudaSuccess)
    return check_launch("amax_history_update launch");
  return check_launch("amax_history_update");
}

lnfp8_status update_many_launch(const lnfp8_meta* const* metas, const uint64_t* e5m2_masks, float* const* sinv_before,
                                int count, int margin, cudaStream_t st) {
  UpdateTable tab = {};
  int slots = 0, maxL = 1;
  for (int k = 0; k < count; ++k) {
    const lnfp8_meta* m = metas[k];
    tab.set[k] = UpdateSet{m->scale, m->scale_inv, m->amax_history, m->amax_cur, sinv_before ? sinv_before[k] : nullptr,
                           e5m2_masks[k], m->n, m->history_len};
    tab.first[k] = slots;
    slots += m->n;
    maxL = m->history_len > maxL ? m->history_len : maxL;
  }
  tab.count = count;
  tab.margin = margin;
  if (!slots) return LNFP8_OK;
  const size_t smem = (size_t)maxL * sizeof(float);
  if (smem + 1024 > 48 * 1024) {
    if (cudaFuncSetAttribute(update_many_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return check_launch("amax_history_update_many: smem attribute");
  }
  LaunchScope ls("state_update_many", st);
  if (launch_pdl(update_many_kernel, dim3(slots), dim3(kThreads), smem, st, tab) != cudaSuccess)
    return check_launch("amax_history_update_many launch");
  return check_launch("amax_history_update_many");
}

}  // namespace lnfp8
