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

namespace lnfp8 {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
update_kernel(float* __restrict__ scale, float* __restrict__ scale_inv, float* __restrict__ hist,
              float* __restrict__ cur, int n, int L, uint64_t e5m2_mask, int margin,
              float* __restrict__ sinv_before) {
  extern __shared__ float shist[];  // the new window of this slot, L floats
  __shared__ uint32_t red[kThreads / 32];
  const int i = blockIdx.x;
  const int t = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  const float c = cur[i];
  // read phase: the new row j is the old row j-1, the new row 0 is cur
  uint32_t m = 0;
  for (int j = t; j < L; j += kThreads) {
    const float v = (j == 0) ? c : hist[(int64_t)(j - 1) * n + i];
    shist[j] = v;
    m = max(m, abs_bits(v));
  }
  __syncthreads();
  for (int j = t; j < L; j += kThreads) hist[(int64_t)j * n + i] = shist[j];
  m = warp_max_u32(m);
  if ((t & 31) == 0) red[t >> 5] = m;
  __syncthreads();
  if (t == 0) {
    uint32_t a_bits = 0;
    for (int w = 0; w < kThreads / 32; ++w) a_bits = max(a_bits, red[w]);
    const float a = __uint_as_float(a_bits);
    if (sinv_before) sinv_before[i] = scale_inv[i];
    cur[i] = 0.f;
    const float fmax = ((e5m2_mask >> i) & 1ull) ? 57344.0f : 448.0f;
    if (isfinite(a) && a > 0.f) {
      float s = fmax / a;
      if (margin > 0) s = s / (float)(1u << margin);
      if (isfinite(s)) {
        scale[i] = s;
        scale_inv[i] = 1.0f / s;
      }
    }
  }
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

lnfp8_status update_launch(const lnfp8_meta* m, uint64_t e5m2_mask, int margin, float* sinv_before,
                           cudaStream_t st) {
  const size_t smem = (size_t)m->history_len * sizeof(float);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return check_launch("amax_history_update: smem attribute");
  }
  LaunchScope ls("state_update", st);
  if (launch_pdl(update_kernel, dim3(m->n), dim3(kThreads), smem, st, m->scale, m->scale_inv, m->amax_history,
                 m->amax_cur, m->n, m->history_len, e5m2_mask, margin, sinv_before) != cudaSuccess)
    return check_launch("amax_history_update launch");
  return check_launch("amax_history_update");
}

}  // namespace lnfp8
