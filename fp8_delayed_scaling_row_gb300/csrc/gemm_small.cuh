// K6: the LayerNormLinear / Linear forward of a few tokens in one launch.
//
// For a handful of tokens (the pages' 8 x 32-token forward through
// te.LayerNormLinear(H, 3H), TE tutorial code block 1) the separate launches
// of the weight cast, the LayerNorm + cast and the GEMM each cost more in
// launch and ramp latency than in work. Here each CTA computes one 128 x 128
// output tile and produces both of its operands itself, straight into the
// shared-memory layout the tensor cores read (K-major, 128-byte swizzle):
//   A: the LayerNorm of its 128 token rows (or, for te.Linear, the rows
//      themselves), amax, E4M3/E5M2 cast with the delayed scale;
//   B: the cast of its 128 weight rows (or the FP8-stored codes as they are).
// One thread then issues the tcgen05 MMAs over the whole K range into tensor
// memory, and all warps dequantise, add the bias and store bf16. The CTAs of
// the first N tile also write the saved LayerNorm codes, mu and rsigma, and
// record the input amax; those of the first M tile write the weight codes and
// record the weight amax. Every arithmetic step is the separate kernels' own
// (the LayerNorm's per-lane chunk order and warp reductions, the scaled casts,
// the single-SM GEMM's K order and epilogue), so the results are theirs bit for
// bit. The state update stays a launch of its own after this one.
//
// Part of gemm.cu's translation unit (PTX wrappers, descriptor helpers).

constexpr int kSmallThreads = 512;  // 16 warps
constexpr int kSmallBN = 128;
constexpr int kSmallMaxK = 768;     // A and B panels of 128 x K codes in shared memory

struct SmallParams {
  int M, N, K;
  const uint16_t* x;
  const uint16_t* gamma;  // NULL: te.Linear (no LayerNorm)
  const uint16_t* beta;
  float eps;
  const uint16_t* w;      // bf16 weight [N, K], cast here; or NULL with wq_in
  const uint8_t* wq_in;   // FP8-stored weight codes [N, K] (used as they are)
  const uint16_t* bias;
  uint16_t* y;
  uint8_t* xq;            // saved codes of the input [M, K]
  uint8_t* wq;            // saved weight codes [N, K] (bf16 weight only)
  float* mu;
  float* rsigma;
  float* ydbg;            // optional fp32 LayerNorm output [M, K]
  const float* scale;     // state: slot 0 input, slot 1 weight
  const float* scale_inv;
  const float* w_scale_inv;  // FP8-stored weight's scale_inv, or NULL
  float* amax_cur;
  uint32_t idesc;
};

// max(m, |y|) with NaN winning: the amax order NaN > Inf > finite, non-negative
__device__ __forceinline__ float nanmax_abs(float m, float y) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(y)));
  return r;
}
__device__ __forceinline__ float nanmax(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Byte offset of code column c of row r inside a [kbs][128 rows][128 B] panel
// laid out as TMA's 128-byte swizzle would write it: the 16-byte chunk index
// within the row is XORed with the row's position in its 8-row group.
__device__ __forceinline__ uint32_t panel_off(int r, int c) {
  const int kb = c >> 7, cb = c & 127;
  return (uint32_t)(kb * 16384 + r * 128 + ((((cb >> 4) ^ (r & 7))) << 4) + (cb & 8));
}

// One row of A (LayerNorm + cast, or the plain cast) or B (the weight cast): each
// lane takes the 8-element chunks lane, lane + 32, ... (the LayerNorm kernel's
// warp-per-row order), writes its codes into the panel, and returns its amax.
template <int NV>
__device__ __forceinline__ void small_load(uint4 (&raw)[NV], const uint16_t* __restrict__ src, bool row_ok, int K,
                                           int lane) {
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c = (lane + 32 * j) * 8;
    raw[j] = row_ok && c < K ? __ldg(reinterpret_cast<const uint4*>(src + c)) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// processes a row whose chunks small_load fetched
template <int NV, int DT, bool LN>
__device__ __forceinline__ float small_row(const uint4 (&raw)[NV], bool row_ok, int K, int kpad,
                                           const uint4* sgb, int nvec, float eps, float inv_k, float s,
                                           uint8_t* panel, int r, uint8_t* gcodes, float* ydbg, float* mu_out,
                                           float* rs_out, int lane) {
  uint64_t v2[NV][4];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    v2[j][0] = bf2_to_f2(raw[j].x);
    v2[j][1] = bf2_to_f2(raw[j].y);
    v2[j][2] = bf2_to_f2(raw[j].z);
    v2[j][3] = bf2_to_f2(raw[j].w);
  }
  uint64_t mu2 = 0, rs2 = 0;
  float mu = 0.f, rs = 0.f;
  if constexpr (LN) {
    uint64_t s2 = 0;
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) s2 = add2(s2, v2[j][q]);
    mu = warp_sum(lo(s2) + hi(s2)) * inv_k;
    mu2 = f2(mu, mu);
    uint64_t q2 = 0;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if ((lane + 32 * j) * 8 < K) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t d = sub2(v2[j][q], mu2);
          q2 = fma2(d, d, q2);
        }
      }
    }
    const float var = warp_sum(lo(q2) + hi(q2)) * inv_k;
    rs = 1.0f / sqrtf(var + eps);
    rs2 = f2(rs, rs);
  }
  float am = 0.f;
  const uint64_t sc2 = f2(s, s);
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c = (lane + 32 * j) * 8;
    if (c >= kpad) continue;
    const bool ok = row_ok && c < K;
    uint32_t c16[4] = {0u, 0u, 0u, 0u};
    if (ok) {
      float y[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint64_t y2 = v2[j][q];
        if constexpr (LN) {
          const uint4 gu = sgb[lane + 32 * j], bu = sgb[nvec + lane + 32 * j];
          const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w}, bw[4] = {bu.x, bu.y, bu.z, bu.w};
          y2 = fma2(mul2(sub2(v2[j][q], mu2), rs2), bf2_to_f2(gw[q]), bf2_to_f2(bw[q]));
        }
        y[2 * q] = lo(y2);
        y[2 * q + 1] = hi(y2);
        am = nanmax_abs(nanmax_abs(am, y[2 * q]), y[2 * q + 1]);
        c16[q] = cvt_pair<DT>(mul2(y2, sc2));
      }
      if (gcodes) *reinterpret_cast<uint2*>(gcodes + c) = make_uint2(c16[0] | (c16[1] << 16), c16[2] | (c16[3] << 16));
      if (ydbg) {
        float4* d4 = reinterpret_cast<float4*>(ydbg + c);
        d4[0] = make_float4(y[0], y[1], y[2], y[3]);
        d4[1] = make_float4(y[4], y[5], y[6], y[7]);
      }
    }
    *reinterpret_cast<uint2*>(panel + panel_off(r, c)) = make_uint2(c16[0] | (c16[1] << 16), c16[2] | (c16[3] << 16));
  }
  if (LN && row_ok && lane == 0 && mu_out) {
    *mu_out = mu;
    *rs_out = rs;
  }
  return am;
}

template <int NV, int DT, bool LN>
__global__ void __launch_bounds__(kSmallThreads, 1) ln_linear_small_kernel(const SmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int kbs = (p.K + 127) >> 7;
  const int kpad = kbs * 128;
  uint8_t* sa = smem;                 // A panel [kbs][128][128 B]
  uint8_t* sb = smem + kbs * 16384;   // B panel
  uint4* sgb = reinterpret_cast<uint4*>(sb + kbs * 16384);  // gamma, beta (bf16)
  const int nvec = p.K >> 3;
  uint64_t* bar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sgb) + 2 * nvec * 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  __shared__ uint32_t ared[kSmallThreads / 32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_blk = blockIdx.x, m_blk = blockIdx.y;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(bar), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kSmallBN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  if (LN)
    for (int i = threadIdx.x; i < nvec; i += kSmallThreads) {
      sgb[i] = reinterpret_cast<const uint4*>(p.gamma)[i];
      sgb[nvec + i] = reinterpret_cast<const uint4*>(p.beta)[i];
    }
  __syncthreads();
  const float inv_k = 1.0f / (float)p.K;
  const bool first_n = n_blk == 0, first_m = m_blk == 0;
  const bool w8 = p.wq_in != nullptr;

  // ---- A (this tile's 128 token rows) and B (its 128 weight rows, cast or stored codes):
  // warp w takes rows w, w + 16, ... of each; every iteration has two A rows and two B
  // rows in flight before any is reduced, so the loads' latency overlaps
  float am_a = 0.f, am_w = 0.f;
  const float sx = p.scale[0], sw = p.scale[1];
  constexpr int kWarps = kSmallThreads / 32;
  for (int r0 = warp; r0 < 128; r0 += 2 * kWarps) {
    uint4 ra[2][NV], rb[2][NV];
    int64_t ma[2], nb[2];
    bool oka[2], okb[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = r0 + i * kWarps;
      ma[i] = (int64_t)m_blk * 128 + r;
      oka[i] = ma[i] < p.M;
      if (!oka[i]) ma[i] = 0;
      small_load<NV>(ra[i], p.x + ma[i] * p.K, oka[i], p.K, lane);
      nb[i] = (int64_t)n_blk * kSmallBN + r;
      okb[i] = nb[i] < p.N;
      if (!okb[i]) nb[i] = 0;
      if (!w8) small_load<NV>(rb[i], p.w + nb[i] * p.K, okb[i], p.K, lane);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = r0 + i * kWarps;
      const int64_t m = ma[i];
      am_a = nanmax(am_a, small_row<NV, DT, LN>(ra[i], oka[i], p.K, kpad, sgb, nvec, p.eps, inv_k, sx, sa, r,
                                                first_n && oka[i] ? p.xq + m * p.K : nullptr,
                                                first_n && oka[i] && p.ydbg ? p.ydbg + m * p.K : nullptr,
                                                first_n && LN ? p.mu + m : nullptr,
                                                first_n && LN ? p.rsigma + m : nullptr, lane));
      if (!w8) {
        am_w = nanmax(am_w, small_row<NV, DT, false>(rb[i], okb[i], p.K, kpad, sgb, nvec, p.eps, inv_k, sw, sb, r,
                                                     first_m && okb[i] ? p.wq + nb[i] * p.K : nullptr, nullptr,
                                                     nullptr, nullptr, lane));
      } else {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          const int c = (lane + 32 * j) * 8;
          if (c >= kpad) continue;
          uint2 q = make_uint2(0u, 0u);
          if (okb[i] && c < p.K) q = __ldg(reinterpret_cast<const uint2*>(p.wq_in + nb[i] * p.K + c));
          *reinterpret_cast<uint2*>(sb + panel_off(r, c)) = q;
        }
      }
    }
  }
  // the amaxes: the input's by the first N tile, the weight's by the first M tile
  block_amax_commit(__float_as_uint(am_a) & 0x7FFFFFFFu, ared, first_n ? p.amax_cur : nullptr);
  __syncthreads();
  block_amax_commit(__float_as_uint(am_w) & 0x7FFFFFFFu, ared, first_m && !w8 ? p.amax_cur + 1 : nullptr);
  // the panels were written by ordinary stores: make them visible to the tensor cores
  fence_async_smem();
  __syncthreads();

  // ---- MMAs over the whole K range (one thread), then the epilogue
  if (threadIdx.x == 0) {
    tc_fence_after();
    const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
    for (int kb = 0; kb < kbs; ++kb) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t off = (uint32_t)(kb * 16384 + kk * 32);
        mma_f8(tmem_base, make_desc(a0 + off, 16, 1024), make_desc(b0 + off, 16, 1024), p.idesc, (kb | kk) != 0);
      }
    }
    mma_commit(smem_u32(bar));
  }
  // the outcome is made warp-uniform: tcgen05.ld below needs the whole warp
  const bool done = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(bar), 0, abort_flag));
  if (!done) {
    uint32_t dummy_flag = 0;  // a late commit must land before the tensor memory is freed
    mbar_wait(smem_u32(bar), 0, &dummy_flag, 100000000ull);
  } else {
    tc_fence_after();
    const int quarter = warp & 3, slice = warp >> 2;  // TMEM lanes 32*quarter.., columns 32*slice..
    const int64_t m = (int64_t)m_blk * 128 + quarter * 32 + lane;
    const int col0 = slice * 32;
    const int64_t n0 = (int64_t)n_blk * kSmallBN + col0;
    uint4 bias8[4];
#pragma unroll
    for (int g = 0; g < 4; ++g)
      bias8[g] = p.bias && n0 + g * 8 < p.N ? __ldg(reinterpret_cast<const uint4*>(p.bias + n0 + g * 8))
                                            : make_uint4(0u, 0u, 0u, 0u);
    uint32_t rr[32];
    tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col0, rr);
    const float s = __fmul_rn(p.scale_inv[0], p.w_scale_inv ? *p.w_scale_inv : p.scale_inv[1]);
    const uint64_t s2 = f2(s, s);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint4 bu = bias8[g];
      const uint64_t b2[4] = {bf2_to_f2(bu.x), bf2_to_f2(bu.y), bf2_to_f2(bu.z), bf2_to_f2(bu.w)};
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t e2 = f2(__uint_as_float(rr[g * 8 + 2 * i]), __uint_as_float(rr[g * 8 + 2 * i + 1]));
        const uint64_t yv = fma2(e2, s2, b2[i]);
        w[i] = pack_bf16x2(lo(yv), hi(yv));
      }
      if (m < p.M && n0 + g * 8 < p.N)
        *reinterpret_cast<uint4*>(p.y + m * p.N + n0 + g * 8) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kSmallBN) : "memory");
  }
}

template <int NV, int DT, bool LN>
lnfp8_status small_launch_t(const SmallParams& sp, cudaStream_t st) {
  auto k = ln_linear_small_kernel<NV, DT, LN>;
  const int kbs = (sp.K + 127) / 128;
  const size_t smem = 1024 + 2 * (size_t)kbs * 16384 + 2 * (size_t)(sp.K / 8) * 16 + 64;
  static bool smem_set = false;
  if (!smem_set) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(1024 + 2 * (kSmallMaxK / 128) * 16384 + 2 * (kSmallMaxK / 8) * 16 + 64)) != cudaSuccess)
      return check_launch("ln_linear small: shared memory attribute");
    smem_set = true;
  }
  const dim3 grid((unsigned)((sp.N + kSmallBN - 1) / kSmallBN), (unsigned)((sp.M + 127) / 128));
  LaunchScope ls("ln_linear_small", st);
  if (launch_pdl(k, grid, dim3(kSmallThreads), smem, st, sp) != cudaSuccess) return check_launch("ln_linear small launch");
  return check_launch("ln_linear small");
}
