// The per-slot delayed-scaling update (K4), shared by the state-update kernels
// (state.cu) and by the launches that run it in extra CTAs of their own grid
// (layernorm.cu: the LayerNorm backward, the last kernel of a backward call;
// gemm.cu: FC2, the last GEMM of a LayerNormMLP forward).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace lnfp8 {

constexpr int kUpdateThreads = 256;  // the block size of the update kernels

// Slot i of one tensor set: roll its history, insert cur, reduce, rescale. NT
// is the block size; `red` holds NT / 32 words, `shist` L floats.
template <int NT = kUpdateThreads>
__device__ inline void update_slot(float* __restrict__ scale, float* __restrict__ scale_inv, float* __restrict__ hist,
                            float* __restrict__ cur, int n, int L, int i, bool e5m2, int margin,
                            float* __restrict__ sinv_before, float* shist, uint32_t* red) {
  const int t = threadIdx.x;
  const float c = cur[i];
  // read phase: the new row j is the old row j-1, the new row 0 is cur
  uint32_t m = 0;
  for (int j = t; j < L; j += NT) {
    const float v = (j == 0) ? c : hist[(int64_t)(j - 1) * n + i];
    shist[j] = v;
    m = max(m, abs_bits(v));
  }
  __syncthreads();
  for (int j = t; j < L; j += NT) hist[(int64_t)j * n + i] = shist[j];
  m = warp_max_u32(m);
  if ((t & 31) == 0) red[t >> 5] = m;
  __syncthreads();
  if (t == 0) {
    uint32_t a_bits = 0;
    for (int w = 0; w < NT / 32; ++w) a_bits = max(a_bits, red[w]);
    const float a = __uint_as_float(a_bits);
    if (sinv_before) sinv_before[i] = scale_inv[i];
    cur[i] = 0.f;
    const float fmax = e5m2 ? 57344.0f : 448.0f;
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


// The extra CTAs' share of a kernel carrying an UpdateJob: CTA b < job.n
// updates slot b. The caller has passed its programmatic-dependency wait.
__device__ inline void run_update_job(const UpdateJob& job, float* shist, uint32_t* red) {
  const int i = blockIdx.x;
  update_slot(job.scale, job.scale_inv, job.hist, job.cur, job.n, job.L, i, (job.e5m2_mask >> i) & 1ull, job.margin,
              nullptr, shist, red);
}

// Every slot of the job, one after another, by one CTA of NT threads (a kernel
// that carries the update in a single extra CTA). The caller has passed its
// programmatic-dependency wait.
template <int NT>
__device__ inline void run_update_all(const UpdateJob& job, float* shist, uint32_t* red) {
  for (int i = 0; i < job.n; ++i)
    update_slot<NT>(job.scale, job.scale_inv, job.hist, job.cur, job.n, job.L, i, (job.e5m2_mask >> i) & 1ull,
                    job.margin, nullptr, shist, red);
}

}  // namespace lnfp8
