// K1: row LayerNorm + amax + FP8 cast, and K5: LayerNorm backward.
//
// LayerNormLinear / LayerNormMLP open with a LayerNorm over each token row
// (TE tutorial, code block 1: te.LayerNormLinear, te.LayerNormMLP; Turbo-charging
// guide, "The building blocks: fused modules you'll use"). The forward kernel
// fuses the normalisation with the delayed-scaling cast of its output: y is
// formed in fp32, its max |y| folds into the tensor's running amax, and
// fp8(y * scale) is written with the scale decided before the step, so the
// fp32/bf16 LayerNorm output never reaches HBM.
//
// Both kernels are HBM-bound. A group of TPR threads owns one row (TPR = 32 is
// a warp per row; wider rows use 64..256 threads so that a thread holds at most
// 4 x 16-byte vectors of the row). Consecutive threads read consecutive 16-byte
// chunks, and row sums are warp shuffles (plus one shared-memory exchange when
// TPR > 32). The loads run ahead of the arithmetic through a per-thread ring
// in shared memory: each thread copies (cp.async, 16 bytes) the chunks of the
// rows it will normalise RING - 2 iterations later, so the bytes in flight per
// SM no longer depend on registers. A thread only ever reads the ring slots it
// filled itself, and refills a slot two iterations after it last read it.
#include "common.cuh"
#include "internal.h"
#include "state_update.cuh"
#include "weight_cast.cuh"

#include <algorithm>

namespace lnfp8 {
namespace {

constexpr int kThreads = 256;
static_assert(kThreads == kUpdateThreads, "the LayerNorm backward carries state updates");
static_assert(kThreads == kWThreads, "the LayerNorm forward carries weight casts");

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Ring depth (slots) per thread: deeper for short per-thread chunks of a row.
__host__ __device__ constexpr int fwd_ring(int nv) { return nv <= 2 ? 6 : 4; }
__host__ __device__ constexpr int bwd_ring(int nv) { return nv <= 2 ? 5 : (nv == 3 ? 4 : 3); }

// Packed fp32 pairs: two values in one 64-bit register, for the f32x2 add,
// sub, mul and fma of the sm_100-family cores (one instruction per pair).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 up2(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// bf16 pair (low, high halves of a 32-bit word) -> fp32 pair
__device__ __forceinline__ uint64_t bf2(uint32_t w) {
  return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// max(m, |y|) with NaN winning (the amax order: NaN > Inf > finite)
__device__ __forceinline__ float absmax_nan(float m, float y) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(y)));
  return r;
}

// Sum over the TPR threads of a row group. `xch` holds kThreads/32 floats.
template <int TPR>
__device__ __forceinline__ float group_sum(float v, float* xch) {
  v = warp_sum(v);
  if constexpr (TPR == 32) {
    return v;
  } else {
    const int warp = threadIdx.x >> 5;
    const int group = threadIdx.x / TPR;
    constexpr int WPG = TPR / 32;
    if ((threadIdx.x & 31) == 0) xch[warp] = v;
    asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "r"(TPR) : "memory");
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < WPG; ++w) s += xch[group * WPG + w];
    asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "r"(TPR) : "memory");
    return s;
  }
}

// Two independent sums over the TPR threads of a row group in one exchange round
// (each added in the same order as group_sum would). `xch` holds 2 * kThreads/32 floats.
template <int TPR>
__device__ __forceinline__ float2 group_sum2(float a, float b, float* xch) {
  a = warp_sum(a);
  b = warp_sum(b);
  if constexpr (TPR == 32) {
    return make_float2(a, b);
  } else {
    const int warp = threadIdx.x >> 5;
    const int group = threadIdx.x / TPR;
    constexpr int WPG = TPR / 32;
    if ((threadIdx.x & 31) == 0) {
      xch[2 * warp] = a;
      xch[2 * warp + 1] = b;
    }
    asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "r"(TPR) : "memory");
    float sa = 0.f, sb = 0.f;
#pragma unroll
    for (int w = 0; w < WPG; ++w) {
      sa += xch[2 * (group * WPG + w)];
      sb += xch[2 * (group * WPG + w) + 1];
    }
    asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "r"(TPR) : "memory");
    return make_float2(sa, sb);
  }
}

// RES: the row is h = bf16(x + resid) (a residual add fused ahead of the
// LayerNorm); h is written to hsum (the new residual stream, which the backward
// reads as its x) and normalised.
template <int TPR, int NV, int DT, bool RES>
__global__ void __launch_bounds__(kThreads)
ln_fwd_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma,
              const uint16_t* __restrict__ beta, float eps, int64_t M, int D,
              const float* __restrict__ scale_p, float* amax_cur, uint8_t* __restrict__ out,
              float* __restrict__ mu_out, float* __restrict__ rs_out, float* __restrict__ ydbg,
              const uint16_t* __restrict__ resid, uint16_t* __restrict__ hsum, const WeightCastJob wc,
              const SinvSnapshot snap) {
  constexpr int NVR = RES ? 2 * NV : NV;  // 16-byte chunks per row and thread in the ring
  constexpr int RING = fwd_ring(NVR);
  constexpr int P = RING - 2;  // rows in flight ahead of the one being normalised
  __shared__ float xch[kThreads / 32];
  __shared__ uint32_t ared[kThreads / 32];
  // gamma then beta as bf16 (D/8 16-byte vectors each: a warp's loads of consecutive vectors
  // are conflict-free), then the ring
  extern __shared__ uint4 sgb[];
  constexpr int GPB = kThreads / TPR;  // row groups per block
  const int g = threadIdx.x / TPR;
  const int gt = threadIdx.x % TPR;
  const int nvec = D >> 3;
  uint4* ring = sgb + 2 * nvec;  // [RING][NVR][kThreads]: x chunks, then (RES) residual chunks
  pdl_wait();
  pdl_launch_dependents();
  const float s = *scale_p;
  const float inv_d = 1.0f / (float)D;
  const int64_t stride = (int64_t)gridDim.x * GPB;
  float amf = 0.f;

  // one commit group per iteration (empty past the last row) keeps the group count regular
  auto issue = [&](int64_t r, int slot) {
    if (r < M) {
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int c = (gt + TPR * j) * 8;
        if (c < D) {
          cp_async16(&ring[(slot * NVR + j) * kThreads + threadIdx.x], x + r * D + c);
          if (RES) cp_async16(&ring[(slot * NVR + NV + j) * kThreads + threadIdx.x], resid + r * D + c);
        }
      }
    }
    cp_async_commit();
  };

  int64_t row = (int64_t)blockIdx.x * GPB + g;
#pragma unroll
  for (int k = 0; k < P; ++k) issue(row + k * stride, k);
  // while the first rows' loads are in flight: the call's scale_inv snapshot (selects, not a
  // runtime index), the counters it clears, gamma and beta into shared memory, the weight casts
  if (blockIdx.x == 0 && (int)threadIdx.x < snap.n) {
    const int k = threadIdx.x;
    snap.dst[k] = *(k == 0 ? snap.src[0] : k == 1 ? snap.src[1] : k == 2 ? snap.src[2] : snap.src[3]);
  }
  if (wc.zero && blockIdx.x == 0)
    for (int64_t i = threadIdx.x; i < wc.zero_n; i += kThreads) wc.zero[i] = 0u;
  for (int i = threadIdx.x; i < nvec; i += kThreads) {
    sgb[i] = reinterpret_cast<const uint4*>(gamma)[i];
    sgb[nvec + i] = reinterpret_cast<const uint4*>(beta)[i];
  }
  if (wc.tiles[0] + wc.tiles[1] > 0) weight_cast_tiles<DT>(wc);
  __syncthreads();
  int slot = 0;
  // every thread of the block runs the same trip count (group_sum may use barriers)
  for (; row - g < M; row += stride) {
    issue(row + P * stride, slot + P < RING ? slot + P : slot + P - RING);
    cp_async_wait<P>();  // this iteration's group has landed
    // each chunk of 8 values unpacked once into four fp32 pairs
    uint64_t v2[NV][4];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c = (gt + TPR * j) * 8;
      const bool ok = row < M && c < D;
      uint4 u = ok ? ring[(slot * NVR + j) * kThreads + threadIdx.x] : make_uint4(0, 0, 0, 0);
      if (RES) {
        const uint4 ur = ok ? ring[(slot * NVR + NV + j) * kThreads + threadIdx.x] : make_uint4(0, 0, 0, 0);
        const uint32_t wx[4] = {u.x, u.y, u.z, u.w}, wr[4] = {ur.x, ur.y, ur.z, ur.w};
        uint32_t wh[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 hv = up2(add2(bf2(wx[q]), bf2(wr[q])));
          wh[q] = pack_bf16x2(hv.x, hv.y);
        }
        u = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        if (ok) *reinterpret_cast<uint4*>(hsum + row * D + c) = u;
      }
      v2[j][0] = bf2(u.x);
      v2[j][1] = bf2(u.y);
      v2[j][2] = bf2(u.z);
      v2[j][3] = bf2(u.w);
    }
    slot = slot + 1 == RING ? 0 : slot + 1;
    const bool active = row < M;
    uint64_t s2 = 0;  // (0.f, 0.f)
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) s2 = add2(s2, v2[j][q]);
    const float2 sp = up2(s2);
    const float mu = group_sum<TPR>(sp.x + sp.y, xch) * inv_d;
    const uint64_t mu2 = pk2(mu, mu);
    uint64_t q2 = 0;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if ((gt + TPR * j) * 8 < D) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t d = sub2(v2[j][q], mu2);
          q2 = fma2(d, d, q2);
        }
      }
    }
    const float2 qp = up2(q2);
    const float var = group_sum<TPR>(qp.x + qp.y, xch) * inv_d;
    const float rs = 1.0f / sqrtf(var + eps);
    if (active) {
      const uint64_t rs2 = pk2(rs, rs), sc2 = pk2(s, s);
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int c = (gt + TPR * j) * 8;
        if (c >= D) continue;
        const uint4 gu = sgb[gt + TPR * j], bu = sgb[nvec + gt + TPR * j];
        const uint64_t gq[4] = {bf2(gu.x), bf2(gu.y), bf2(gu.z), bf2(gu.w)};
        const uint64_t bq[4] = {bf2(bu.x), bf2(bu.y), bf2(bu.z), bf2(bu.w)};
        float y[8];
        uint32_t c16[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // y = (x - mu) * rsigma * gamma + beta, the same rounded steps as one value at a time
          const uint64_t y2 = fma2(mul2(sub2(v2[j][q], mu2), rs2), gq[q], bq[q]);
          const float2 yv = up2(y2);
          y[2 * q] = yv.x;
          y[2 * q + 1] = yv.y;
          amf = absmax_nan(absmax_nan(amf, yv.x), yv.y);
          const float2 z = up2(mul2(y2, sc2));
          c16[q] = cvt_fp8x2<DT>(z.x, z.y);
        }
        *reinterpret_cast<uint2*>(out + row * D + c) = make_uint2(c16[0] | (c16[1] << 16), c16[2] | (c16[3] << 16));
        if (ydbg) {
          float4* d4 = reinterpret_cast<float4*>(ydbg + row * D + c);
          d4[0] = make_float4(y[0], y[1], y[2], y[3]);
          d4[1] = make_float4(y[4], y[5], y[6], y[7]);
        }
      }
      if (gt == 0) {
        mu_out[row] = mu;
        rs_out[row] = rs;
      }
    }
  }
  cp_async_wait<0>();
  block_amax_commit(__float_as_uint(amf) & 0x7FFFFFFFu, ared, amax_cur);
}

template <int TPR, int NV>
__global__ void __launch_bounds__(kThreads, 2)
ln_bwd_kernel(const uint16_t* __restrict__ dy, const uint16_t* __restrict__ x,
              const uint16_t* __restrict__ gamma, const float* __restrict__ mu_in,
              const float* __restrict__ rs_in, int64_t M, int D, uint16_t* __restrict__ dx,
              float* dgamma, float* dbeta, const UpdateJob job) {
  constexpr int RING = bwd_ring(NV);
  constexpr int P = RING - 2;  // rows in flight ahead of the one being processed
  __shared__ float xch[2 * (kThreads / 32)];
  // [2][D] block partials of dgamma, dbeta; gamma [D/8 uint4] bf16; the ring of x and dY chunks
  // [RING][2 NV][kThreads] uint4; then the ring of mu, rsigma [RING][2][kThreads] fp32
  extern __shared__ float colred[];
  uint4* sg = reinterpret_cast<uint4*>(colred + 2 * D);
  constexpr int GPB = kThreads / TPR;
  const int g = threadIdx.x / TPR;
  const int gt = threadIdx.x % TPR;
  const float inv_d = 1.0f / (float)D;
  const int nvec = D >> 3;
  uint4* ring = sg + nvec;
  float* rstat = reinterpret_cast<float*>(ring + RING * 2 * NV * kThreads);
  pdl_wait();
  pdl_launch_dependents();
  if ((int)blockIdx.x < job.n) {  // an extra CTA: one slot of the call's state update
    run_update_job(job, colred, reinterpret_cast<uint32_t*>(xch));
    return;
  }
  const int64_t bid = (int64_t)blockIdx.x - job.n;
  const int64_t stride = (int64_t)(gridDim.x - job.n) * GPB;

  auto issue = [&](int64_t r, int slot) {
    if (r < M) {
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int c = (gt + TPR * j) * 8;
        if (c < D) {
          cp_async16(&ring[(slot * 2 * NV + j) * kThreads + threadIdx.x], x + r * D + c);
          cp_async16(&ring[(slot * 2 * NV + NV + j) * kThreads + threadIdx.x], dy + r * D + c);
        }
      }
      cp_async4(&rstat[(slot * 2 + 0) * kThreads + threadIdx.x], mu_in + r);
      cp_async4(&rstat[(slot * 2 + 1) * kThreads + threadIdx.x], rs_in + r);
    }
    cp_async_commit();
  };

  // dgamma, dbeta partials of this thread's columns as fp32 pairs
  uint64_t accg[NV][4], accb[NV][4];
#pragma unroll
  for (int j = 0; j < NV; ++j)
#pragma unroll
    for (int q = 0; q < 4; ++q) accg[j][q] = accb[j][q] = 0;

  int64_t row = bid * GPB + g;
#pragma unroll
  for (int k = 0; k < P; ++k) issue(row + k * stride, k);
  // while the first rows' loads are in flight: clear the column partials, gamma into shared memory
  for (int c = threadIdx.x; c < 2 * D; c += kThreads) colred[c] = 0.f;
  for (int i = threadIdx.x; i < nvec; i += kThreads) sg[i] = reinterpret_cast<const uint4*>(gamma)[i];
  __syncthreads();
  int slot = 0;
  for (; row - g < M; row += stride) {
    issue(row + P * stride, slot + P < RING ? slot + P : slot + P - RING);
    cp_async_wait<P>();  // this iteration's group has landed
    const bool active = row < M;
    const float mu = active ? rstat[(slot * 2 + 0) * kThreads + threadIdx.x] : 0.f;
    const float rs = active ? rstat[(slot * 2 + 1) * kThreads + threadIdx.x] : 0.f;
    const uint64_t mu2 = pk2(mu, mu), rs2 = pk2(rs, rs);
    // xhat = (x - mu) * rsigma and g = dy * gamma, kept for the second pass
    uint64_t xh[NV][4], gg[NV][4];
    uint64_t s1 = 0, s2 = 0;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c = (gt + TPR * j) * 8;
      const bool ok = active && c < D;
      const uint4 ux = ok ? ring[(slot * 2 * NV + j) * kThreads + threadIdx.x] : make_uint4(0, 0, 0, 0);
      const uint4 ud = ok ? ring[(slot * 2 * NV + NV + j) * kThreads + threadIdx.x] : make_uint4(0, 0, 0, 0);
      const uint4 ug = c < D ? sg[gt + TPR * j] : make_uint4(0, 0, 0, 0);
      const uint32_t wx[4] = {ux.x, ux.y, ux.z, ux.w}, wd[4] = {ud.x, ud.y, ud.z, ud.w};
      const uint64_t gq[4] = {bf2(ug.x), bf2(ug.y), bf2(ug.z), bf2(ug.w)};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint64_t xv = bf2(wx[q]), dv = bf2(wd[q]);
        xh[j][q] = mul2(sub2(xv, mu2), rs2);
        gg[j][q] = mul2(dv, gq[q]);
        s1 = add2(s1, gg[j][q]);
        s2 = fma2(gg[j][q], xh[j][q], s2);
        accg[j][q] = fma2(dv, xh[j][q], accg[j][q]);
        accb[j][q] = add2(accb[j][q], dv);
      }
    }
    slot = slot + 1 == RING ? 0 : slot + 1;
    const float2 s1p = up2(s1), s2p = up2(s2);
    const float2 sums = group_sum2<TPR>(s1p.x + s1p.y, s2p.x + s2p.y, xch);
    const float mean_g = sums.x * inv_d;
    const float mean_gx = sums.y * inv_d;
    if (!active) continue;
    const uint64_t mg2 = pk2(mean_g, mean_g), nmgx2 = pk2(-mean_gx, -mean_gx);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c = (gt + TPR * j) * 8;
      if (c >= D) continue;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // dx = rsigma * (g - mean(g) - xhat * mean(g * xhat))
        const float2 o = up2(mul2(fma2(xh[j][q], nmgx2, sub2(gg[j][q], mg2)), rs2));
        w[q] = pack_bf16x2(o.x, o.y);
      }
      *reinterpret_cast<uint4*>(dx + row * D + c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }

  cp_async_wait<0>();
  // block reduction of the column partials: the row groups add their partials
  // into shared memory one group at a time (plain 16-byte accesses, no bank
  // conflicts), then one atomic per column per block
  for (int turn = 0; turn < GPB; ++turn) {
    __syncthreads();
    if (g != turn) continue;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c = (gt + TPR * j) * 8;
      if (c >= D) continue;
      float4* pg = reinterpret_cast<float4*>(colred + c);
      float4* pb = reinterpret_cast<float4*>(colred + D + c);
      const float4 g0 = pg[0], g1 = pg[1], b0 = pb[0], b1 = pb[1];
      const float2 a0 = up2(accg[j][0]), a1 = up2(accg[j][1]), a2 = up2(accg[j][2]), a3 = up2(accg[j][3]);
      const float2 e0 = up2(accb[j][0]), e1 = up2(accb[j][1]), e2 = up2(accb[j][2]), e3 = up2(accb[j][3]);
      pg[0] = make_float4(g0.x + a0.x, g0.y + a0.y, g0.z + a1.x, g0.w + a1.y);
      pg[1] = make_float4(g1.x + a2.x, g1.y + a2.y, g1.z + a3.x, g1.w + a3.y);
      pb[0] = make_float4(b0.x + e0.x, b0.y + e0.y, b0.z + e1.x, b0.w + e1.y);
      pb[1] = make_float4(b1.x + e2.x, b1.y + e2.y, b1.z + e3.x, b1.w + e3.y);
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += kThreads) {
    atomicAdd(dgamma + c, colred[c]);
    atomicAdd(dbeta + c, colred[D + c]);
  }
}

// Threads per row and 16-byte vectors per thread for a row of D bf16.
struct RowShape { int tpr, nv; };
RowShape row_shape(int64_t D, int max_nv) {
  const int64_t vecs = (D + 7) / 8;
  for (int tpr = 32; tpr <= 256; tpr *= 2) {
    const int64_t nv = (vecs + tpr - 1) / tpr;
    if (nv <= max_nv || tpr == 256) return nv <= 4 ? RowShape{tpr, (int)nv} : RowShape{0, 0};
  }
  return {0, 0};
}

// Resident blocks per SM for a kernel at kThreads threads and `smem` bytes.
template <typename K>
int64_t resident_blocks(K kernel, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, smem) != cudaSuccess || n < 1) n = 1;
  return (int64_t)n * num_sms();
}

template <int DT, bool RES>
lnfp8_status ln_fwd_dispatch(RowShape rsh, cudaStream_t st, const uint16_t* x,
                             const uint16_t* gamma, const uint16_t* beta, float eps, int64_t M, int D,
                             const float* scale, float* amax_cur, uint8_t* out, float* mu, float* rsigma,
                             float* ydbg, const uint16_t* resid, uint16_t* hsum, const WeightCastJob& wc,
                             const SinvSnapshot& snap) {
  const int nvr = RES ? 2 * rsh.nv : rsh.nv;
  const size_t smem = (size_t)D * 2 * sizeof(uint16_t) + (size_t)fwd_ring(nvr) * nvr * kThreads * 16;
  const int64_t gpb = kThreads / rsh.tpr;
#define LNF(TPR, NV)                                                                                    \
  do {                                                                                                  \
    auto k = ln_fwd_kernel<TPR, NV, DT, RES>;                                                           \
    if (smem + 1024 > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    /* the weight tiles are shared by at least as many CTAs as the rows need, up to a full wave */     \
    const int64_t blocks = min64(max64((M + gpb - 1) / gpb, wc.tiles[0] + wc.tiles[1]), resident_blocks(k, smem)); \
    if (launch_pdl(k, dim3((unsigned)max64(blocks, 1)), dim3(kThreads), smem, st, x, gamma, beta, eps, M, D, scale, amax_cur, out, mu, rsigma, ydbg, resid, hsum, wc, snap) != cudaSuccess) \
      return check_launch("ln_fwd_cast launch");                                                        \
  } while (0)
  switch (rsh.tpr * 10 + rsh.nv) {
    case 321: LNF(32, 1); break;
    case 322: LNF(32, 2); break;
    case 323: LNF(32, 3); break;
    case 324: LNF(32, 4); break;
    case 642: LNF(64, 2); break;
    case 643: LNF(64, 3); break;
    case 644: LNF(64, 4); break;
    case 1282: LNF(128, 2); break;
    case 1283: LNF(128, 3); break;
    case 1284: LNF(128, 4); break;
    case 2562: LNF(256, 2); break;
    case 2563: LNF(256, 3); break;
    case 2564: LNF(256, 4); break;
    default: return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "ln_fwd_cast: unsupported D");
  }
#undef LNF
  return check_launch("ln_fwd_cast");
}

}  // namespace

void weight_cast_add(WeightCastJob& j, int k, const uint16_t* in, int64_t rows, int64_t cols, const float* scale,
                     float* amax, uint8_t* out) {
  j.in[k] = in;
  j.rows[k] = rows;
  j.cols[k] = cols;
  j.scale[k] = scale;
  j.amax[k] = amax;
  j.out[k] = out;
  j.tiles[k] = rows > 0 && cols > 0 ? ((rows + kWTileRows - 1) / kWTileRows) * ((cols + kWTileCols - 1) / kWTileCols) : 0;
}

lnfp8_status ln_fwd_launch(const uint16_t* x, const uint16_t* gamma, const uint16_t* beta, float eps,
                           int64_t M, int64_t D, int dtype, const float* scale, float* amax_cur,
                           uint8_t* out, float* mu, float* rsigma, float* ydbg, cudaStream_t st,
                           const uint16_t* resid, uint16_t* hsum, const WeightCastJob* wcp, const SinvSnapshot* snp) {
  const WeightCastJob nojob = {};
  const WeightCastJob& wc = wcp ? *wcp : nojob;
  const SinvSnapshot nosnap = {};
  const SinvSnapshot& snap = snp ? *snp : nosnap;
  if (M == 0 && wc.tiles[0] + wc.tiles[1] == 0 && !(wc.zero && wc.zero_n > 0) && snap.n == 0) return LNFP8_OK;
  const RowShape rsh = row_shape(D, 4);
  if (rsh.tpr == 0 || D > 8192) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "ln_fwd_cast: D = %lld > 8192", (long long)D);
  LaunchScope ls("ln_fwd_cast", st);
  const bool res = resid != nullptr;
  if (dtype == LNFP8_E4M3)
    return res ? ln_fwd_dispatch<LNFP8_E4M3, true>(rsh, st, x, gamma, beta, eps, M, (int)D, scale, amax_cur, out, mu,
                                                   rsigma, ydbg, resid, hsum, wc, snap)
               : ln_fwd_dispatch<LNFP8_E4M3, false>(rsh, st, x, gamma, beta, eps, M, (int)D, scale, amax_cur, out, mu,
                                                    rsigma, ydbg, nullptr, nullptr, wc, snap);
  return res ? ln_fwd_dispatch<LNFP8_E5M2, true>(rsh, st, x, gamma, beta, eps, M, (int)D, scale, amax_cur, out, mu,
                                                 rsigma, ydbg, resid, hsum, wc, snap)
             : ln_fwd_dispatch<LNFP8_E5M2, false>(rsh, st, x, gamma, beta, eps, M, (int)D, scale, amax_cur, out, mu,
                                                  rsigma, ydbg, nullptr, nullptr, wc, snap);
}

lnfp8_status ln_bwd_launch(const uint16_t* dy, const uint16_t* x, const uint16_t* gamma, const float* mu,
                           const float* rsigma, int64_t M, int64_t D, uint16_t* dx, float* dgamma,
                           float* dbeta, cudaStream_t st, bool clear, const UpdateJob* job, bool* job_done) {
  if (job_done) *job_done = false;
  if (clear && D > 0) {
    if (cudaMemsetAsync(dgamma, 0, D * sizeof(float), st) != cudaSuccess ||
        cudaMemsetAsync(dbeta, 0, D * sizeof(float), st) != cudaSuccess)
      return check_launch("ln_bwd: clearing dgamma/dbeta");
  }
  if (M == 0) return LNFP8_OK;
  const RowShape rsh = row_shape(D, 3);
  if (rsh.tpr == 0 || D > 8192) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "ln_bwd: D = %lld > 8192", (long long)D);
  const int64_t gpb = kThreads / rsh.tpr;
  // the extra CTAs of an UpdateJob keep their history window in the same shared memory
  const UpdateJob nojob = {};
  const UpdateJob& uj = job ? *job : nojob;
  const size_t smem = std::max<size_t>(2 * D * sizeof(float) + D * sizeof(uint16_t) +
                                           (size_t)bwd_ring(rsh.nv) * (2 * rsh.nv * 16 + 2 * 4) * kThreads,
                                       (size_t)uj.L * sizeof(float));
  LaunchScope ls("ln_bwd", st);
#define LNB(TPR, NV)                                                                                   \
  do {                                                                                                 \
    auto k = ln_bwd_kernel<TPR, NV>;                                                                   \
    if (smem + 1024 > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    const int64_t blocks = min64((M + gpb - 1) / gpb, resident_blocks(k, smem)) + uj.n;                \
    if (launch_pdl(k, dim3((unsigned)blocks), dim3(kThreads), smem, st, dy, x, gamma, mu, rsigma, M, (int)D, dx, dgamma, dbeta, uj) != cudaSuccess) \
      return check_launch("ln_bwd launch");                                                            \
  } while (0)
  switch (rsh.tpr * 10 + rsh.nv) {
    case 321: LNB(32, 1); break;
    case 322: LNB(32, 2); break;
    case 323: LNB(32, 3); break;
    case 324: LNB(32, 4); break;
    case 642: LNB(64, 2); break;
    case 643: LNB(64, 3); break;
    case 644: LNB(64, 4); break;
    case 1282: LNB(128, 2); break;
    case 1283: LNB(128, 3); break;
    case 1284: LNB(128, 4); break;
    case 2562: LNB(256, 2); break;
    case 2563: LNB(256, 3); break;
    case 2564: LNB(256, 4); break;
    default: return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "ln_bwd: unsupported D");
  }
#undef LNB
  if (job_done) *job_done = uj.n > 0;
  return check_launch("ln_bwd");
}

}  // namespace lnfp8
