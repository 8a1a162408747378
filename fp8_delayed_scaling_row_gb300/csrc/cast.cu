// K2: scaled FP8 cast with amax, optional transposed copy and column sums.
//
// The cast of delayed scaling (Turbo-charging guide, "Playing with
// lower-precision formats: BF16 vs FP8": the recipe tracks the amax of each
// tensor and rescales it): code = fp8(x * scale) with the scale decided before
// the step, while max|x| is folded into the tensor's running amax. Used for
// the weights every step, for the upstream gradient dY (with its column sums,
// the bias gradient) and for a Linear layer's un-normalised input.
//
// HBM-bound: each element is read once (2 or 4 bytes) and written once
// (1 byte, plus 1 for the transpose). A CTA walks one 64-column strip over a
// range of rows, 64 x 64 tiles at a time, with 16-byte loads.
#include "common.cuh"
#include "internal.h"

#define TRY_CAST(x)                    \
  do {                                 \
    const lnfp8_status _s = (x);       \
    if (_s != LNFP8_OK) return _s;     \
  } while (0)

namespace lnfp8 {
namespace {

constexpr int kTC = 64;   // tile columns
constexpr int kTR = 128;  // tile rows per iteration (8 x 16-byte loads in flight per thread)
constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ void load8(const T* p, float* v);

template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* p, float* v) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float* v) {
  float4 a = reinterpret_cast<const float4*>(p)[0];
  float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// The tensor of a strip-form cast launch.
struct CastT {
  const void* in;
  int64_t rows, cols, rows_per_cta;
  const float* scale;
  float* amax_cur;
  uint8_t* out;
  uint8_t* out_t;
  float* colsum;
};

template <typename T, int DT, int TR>
__global__ void __launch_bounds__(kThreads)
cast_kernel(const CastT ct) {
  pdl_wait();
  pdl_launch_dependents();
  const T* __restrict__ in = static_cast<const T*>(ct.in);
  const int64_t rows = ct.rows, cols = ct.cols, rows_per_cta = ct.rows_per_cta;
  const float* __restrict__ scale_p = ct.scale;
  float* amax_cur = ct.amax_cur;
  uint8_t* __restrict__ out = ct.out;
  uint8_t* __restrict__ out_t = ct.out_t;
  float* colsum = ct.colsum;
  if ((int64_t)blockIdx.x * kTC >= cols || (int64_t)blockIdx.y * rows_per_cta >= rows) return;
  // TR rows x 64 columns per iteration; each thread owns one 8-column vector
  // of TR/32 rows and issues all of their loads before converting any.
  constexpr int RPT = TR / 32;
  __shared__ __align__(16) uint8_t tq[kTC][TR + 16];
  __shared__ float red[32][kTC + 1];
  __shared__ uint32_t ared[kThreads / 32];

  const int t = threadIdx.x;
  const int cv = t & 7;          // which 8-column vector of the strip
  const int rr = t >> 3;         // 0..31
  const int64_t c0 = (int64_t)blockIdx.x * kTC;
  const int64_t cc = c0 + cv * 8;
  const bool col_ok = cc < cols;
  const int64_t r_begin = (int64_t)blockIdx.y * rows_per_cta;
  const int64_t r_end = min(rows, r_begin + rows_per_cta);
  const float s = *scale_p;
  const bool t_vec = (rows % 16) == 0;

  uint32_t am = 0;
  float csum[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) csum[i] = 0.f;

  for (int64_t r0 = r_begin; r0 < r_end; r0 += TR) {
    float v[RPT][8];
#pragma unroll
    for (int h = 0; h < RPT; ++h) {
      const int64_t r = r0 + rr + 32 * h;
      if (r < r_end && col_ok) {
        load8<T>(in + r * cols + cc, v[h]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[h][i] = 0.f;
      }
    }
#pragma unroll
    for (int h = 0; h < RPT; ++h) {
      const int rl = rr + 32 * h;
      const int64_t r = r0 + rl;
      uint2 q = make_uint2(0, 0);
      if (r < r_end && col_ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          am = max(am, abs_bits(v[h][i]));
          csum[i] += v[h][i];
        }
        q = cvt_fp8x8<DT>(v[h], s);
        if (out) *reinterpret_cast<uint2*>(out + r * cols + cc) = q;
      }
      if (out_t) {
        const uint32_t w[2] = {q.x, q.y};
#pragma unroll
        for (int i = 0; i < 8; ++i) tq[cv * 8 + i][rl] = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
      }
    }
    if (out_t) {
      __syncthreads();
      // TR rows x 64 columns of codes leave as 16-byte runs along the rows
      for (int idx = t; idx < kTC * (TR / 16); idx += kThreads) {
        const int col = idx / (TR / 16), chunk = (idx % (TR / 16)) * 16;
        const int64_t c = c0 + col;
        if (c < cols) {
          uint8_t* dst = out_t + c * rows + r0 + chunk;
          const int64_t nvalid = min64(16, r_end - (r0 + chunk));
          if (nvalid == 16 && t_vec) {
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&tq[col][chunk]);
          } else {
            for (int i = 0; i < nvalid; ++i) dst[i] = tq[col][chunk + i];
          }
        }
      }
      __syncthreads();
    }
  }

  if (colsum) {
#pragma unroll
    for (int i = 0; i < 8; ++i) red[rr][cv * 8 + i] = csum[i];
    __syncthreads();
    if (t < kTC) {
      float acc = 0.f;
      for (int j = 0; j < 32; ++j) acc += red[j][t];
      if (c0 + t < cols) atomicAdd(colsum + c0 + t, acc);
    }
  }
  block_amax_commit(am, ared, amax_cur);
}

// ------------------------------------------------------------------ row-streaming form
// For bf16 input without a transposed copy: TPR threads per row, each owning NV
// 16-byte column chunks of every row it visits, rows taken by a persistent
// grid stride. Each thread copies the chunks of the rows it will convert
// RING - 2 iterations ahead into its own slots of a shared-memory ring
// (cp.async) and reads only its own slots. Column sums stay in registers
// (fp32 pairs) until the end, then the row groups add them into shared memory
// in turn and the block adds one partial per column to `colsum`.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
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
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t bf2(uint32_t w) {
  return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ float absmax_nan(float m, float y) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(y)));
  return r;
}
__host__ __device__ constexpr int rows_ring(int nv) { return nv <= 2 ? 6 : 4; }
constexpr int64_t kRowsMinElems = 1ll << 24;  // smallest tensor the row form takes

template <int TPR, int NV, int DT>
__global__ void __launch_bounds__(kThreads)
cast_rows_kernel(const uint16_t* __restrict__ in, int64_t rows, int cols, const float* __restrict__ scale_p,
                 float* amax_cur, uint8_t* __restrict__ out, float* colsum) {
  constexpr int RING = rows_ring(NV);
  constexpr int P = RING - 2;
  constexpr int GPB = kThreads / TPR;
  extern __shared__ uint4 rring[];  // [RING][NV][kThreads], then (column sums) [cols] fp32
  __shared__ uint32_t ared[kThreads / 32];
  float* colred = reinterpret_cast<float*>(rring + RING * NV * kThreads);
  const int g = threadIdx.x / TPR;
  const int gt = threadIdx.x % TPR;
  pdl_wait();
  pdl_launch_dependents();
  if (colsum) {
    for (int c = threadIdx.x; c < cols; c += kThreads) colred[c] = 0.f;
  }
  const float s = *scale_p;
  const uint64_t s2 = pk2(s, s);
  const int64_t stride = (int64_t)gridDim.x * GPB;
  float am = 0.f;
  uint64_t cs[NV][4];
#pragma unroll
  for (int j = 0; j < NV; ++j)
#pragma unroll
    for (int q = 0; q < 4; ++q) cs[j][q] = 0;

  auto issue = [&](int64_t r, int slot) {
    if (r < rows) {
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int c = (gt + TPR * j) * 8;
        if (c < cols) cp_async16(&rring[(slot * NV + j) * kThreads + threadIdx.x], in + r * cols + c);
      }
    }
    cp_async_commit();
  };
  int64_t row = (int64_t)blockIdx.x * GPB + g;
#pragma unroll
  for (int k = 0; k < P; ++k) issue(row + k * stride, k);
  int slot = 0;
  for (; row < rows; row += stride) {
    issue(row + P * stride, slot + P < RING ? slot + P : slot + P - RING);
    cp_async_wait<P>();
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c = (gt + TPR * j) * 8;
      if (c >= cols) continue;
      const uint4 u = rring[(slot * NV + j) * kThreads + threadIdx.x];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t c16[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint64_t v = bf2(w[q]);
        cs[j][q] = add2(cs[j][q], v);
        const float2 vv = up2(v);
        am = absmax_nan(absmax_nan(am, vv.x), vv.y);
        const float2 z = up2(mul2(v, s2));
        c16[q] = cvt_fp8x2<DT>(z.x, z.y);
      }
      *reinterpret_cast<uint2*>(out + row * cols + c) = make_uint2(c16[0] | (c16[1] << 16), c16[2] | (c16[3] << 16));
    }
    slot = slot + 1 == RING ? 0 : slot + 1;
  }
  cp_async_wait<0>();
  if (colsum) {
    for (int turn = 0; turn < GPB; ++turn) {
      __syncthreads();
      if (g != turn) continue;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int c = (gt + TPR * j) * 8;
        if (c >= cols) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 v = up2(cs[j][q]);
          colred[c + 2 * q] += v.x;
          colred[c + 2 * q + 1] += v.y;
        }
      }
    }
    __syncthreads();
    for (int c = threadIdx.x; c < cols; c += kThreads) atomicAdd(colsum + c, colred[c]);
  }
  block_amax_commit(__float_as_uint(am) & 0x7FFFFFFFu, ared, amax_cur);
}

}  // namespace

namespace {

struct Grid2 {
  int64_t strips, ysplit, rows_per_cta;
};

Grid2 cast_grid(int64_t rows, int64_t cols, int64_t want) {
  Grid2 g;
  g.strips = (cols + kTC - 1) / kTC;
  const int64_t row_tiles = (rows + kTR - 1) / kTR;
  int64_t ys = (want + g.strips - 1) / g.strips;
  ys = max64(1, min64(ys, row_tiles));
  g.rows_per_cta = ((row_tiles + ys - 1) / ys) * kTR;
  g.ysplit = (rows + g.rows_per_cta - 1) / g.rows_per_cta;
  return g;
}

template <typename T>
lnfp8_status cast_dispatch(dim3 grid, int dtype, const CastT& a, cudaStream_t st) {
  const cudaError_t e = dtype == LNFP8_E4M3 ? launch_pdl(cast_kernel<T, LNFP8_E4M3, kTR>, grid, dim3(kThreads), 0, st, a)
                                             : launch_pdl(cast_kernel<T, LNFP8_E5M2, kTR>, grid, dim3(kThreads), 0, st, a);
  if (e != cudaSuccess) return set_error(LNFP8_ERR_CUDA, "fp8_quantize launch: %s", cudaGetErrorString(e));
  return check_launch("fp8_quantize");
}

}  // namespace

namespace {
// Threads per row and 16-byte chunks per thread of the row-streaming form, or {0, 0}.
struct RowsShape { int tpr, nv; };
RowsShape rows_shape(int64_t cols) {
  if (cols > 8192) return {0, 0};
  const int64_t vecs = (cols + 7) / 8;
  for (int tpr = 32; tpr <= 256; tpr *= 2) {
    const int64_t nv = (vecs + tpr - 1) / tpr;
    if (nv <= 4 || tpr == 256) return nv <= 4 ? RowsShape{tpr, (int)nv} : RowsShape{0, 0};
  }
  return {0, 0};
}

template <int DT>
lnfp8_status rows_dispatch(RowsShape rs, const uint16_t* in, int64_t rows, int64_t cols, const float* scale,
                           float* amax_cur, uint8_t* out, float* colsum, cudaStream_t st) {
  const size_t smem = (size_t)rows_ring(rs.nv) * rs.nv * kThreads * 16 + (colsum ? (size_t)cols * 4 : 0);
  const int64_t gpb = kThreads / rs.tpr;
#define CRK(TPR, NV)                                                                                   \
  do {                                                                                                 \
    auto k = cast_rows_kernel<TPR, NV, DT>;                                                            \
    if (smem + 1024 > 48 * 1024 &&                                                                            \
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) \
      return check_launch("fp8_quantize: smem attribute");                                             \
    int nb = 0;                                                                                        \
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k, kThreads, smem) != cudaSuccess || nb < 1) nb = 1; \
    const int64_t blocks = min64((rows + gpb - 1) / gpb, (int64_t)nb * num_sms());                     \
    if (launch_pdl(k, dim3((unsigned)blocks), dim3(kThreads), smem, st, in, rows, (int)cols, scale, amax_cur, out, colsum) != cudaSuccess) \
      return check_launch("fp8_quantize launch");                                                      \
  } while (0)
  switch (rs.tpr * 10 + rs.nv) {
    case 321: CRK(32, 1); break;
    case 322: CRK(32, 2); break;
    case 323: CRK(32, 3); break;
    case 324: CRK(32, 4); break;
    case 642: CRK(64, 2); break;
    case 643: CRK(64, 3); break;
    case 644: CRK(64, 4); break;
    case 1282: CRK(128, 2); break;
    case 1283: CRK(128, 3); break;
    case 1284: CRK(128, 4); break;
    case 2562: CRK(256, 2); break;
    case 2563: CRK(256, 3); break;
    case 2564: CRK(256, 4); break;
    default: return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "fp8_quantize: unsupported row width");
  }
#undef CRK
  return check_launch("fp8_quantize");
}
}  // namespace

bool cast_streams_rows(int64_t rows, int64_t cols) { return rows_shape(cols).tpr && rows * cols >= kRowsMinElems; }

lnfp8_status cast_launch(const void* in, bool in_fp32, int64_t rows, int64_t cols, int dtype,
                         const float* scale, float* amax_cur, uint8_t* out, uint8_t* out_t,
                         float* colsum, cudaStream_t st, bool clear_colsum) {
  if (clear_colsum && colsum && cols > 0 && cudaMemsetAsync(colsum, 0, cols * sizeof(float), st) != cudaSuccess)
    return check_launch("fp8_quantize: clearing colsum");
  if (rows == 0 || cols == 0) return LNFP8_OK;
  // large bf16 tensors without a transposed copy stream through the row form (on small ones
  // its per-block column reduction costs more than it saves)
  const RowsShape rs = rows_shape(cols);
  if (!in_fp32 && !out_t && out && cast_streams_rows(rows, cols)) {
    LaunchScope ls(colsum ? "cast_colsum" : "cast", st);
    return dtype == LNFP8_E4M3
               ? rows_dispatch<LNFP8_E4M3>(rs, static_cast<const uint16_t*>(in), rows, cols, scale, amax_cur, out, colsum, st)
               : rows_dispatch<LNFP8_E5M2>(rs, static_cast<const uint16_t*>(in), rows, cols, scale, amax_cur, out, colsum, st);
  }
  // enough CTAs that each SM keeps several row tiles of loads in flight
  const Grid2 g = cast_grid(rows, cols, 8LL * num_sms());
  if (g.strips > 0x7FFFFFFF || g.ysplit > 65535)
    return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "fp8_quantize: tensor too large");
  const CastT t{in, rows, cols, g.rows_per_cta, scale, amax_cur, out, out_t, colsum};
  LaunchScope ls(colsum ? "cast_colsum" : "cast", st);
  const dim3 grid((unsigned)g.strips, (unsigned)g.ysplit, 1);
  return in_fp32 ? cast_dispatch<float>(grid, dtype, t, st) : cast_dispatch<uint16_t>(grid, dtype, t, st);
}

namespace {
// Zeroes up to kZeroSpans word ranges in one launch (the accumulated outputs
// and split-K flags a backward call starts from).
constexpr int kZeroSpans = 6;
struct ZeroSpans {
  uint32_t* p[kZeroSpans];
  int64_t n[kZeroSpans];  // 32-bit words
};

__global__ void __launch_bounds__(256) zero_kernel(ZeroSpans z) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = 0; i < kZeroSpans; ++i) {
    uint32_t* p = z.p[i];
    const int64_t n = z.n[i];
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += (int64_t)gridDim.x * blockDim.x) p[j] = 0u;
  }
}
}  // namespace

lnfp8_status zero_launch(std::initializer_list<std::pair<void*, int64_t>> spans, cudaStream_t st) {
  ZeroSpans z = {};
  int k = 0;
  int64_t most = 0;
  for (const auto& sp : spans) {
    if (!sp.first || sp.second <= 0) continue;
    if (k == kZeroSpans) return set_error(LNFP8_ERR_INVALID_ARG, "zero_launch: more than %d spans", kZeroSpans);
    z.p[k] = static_cast<uint32_t*>(sp.first);
    z.n[k] = (sp.second + 3) / 4;
    most = z.n[k] > most ? z.n[k] : most;
    ++k;
  }
  if (!k) return LNFP8_OK;
  const int64_t blocks = (most + 255) / 256 < 152 ? (most + 255) / 256 : 152;
  LaunchScope ls("zero", st);
  if (launch_pdl(zero_kernel, dim3((unsigned)blocks), dim3(256), 0, st, z) != cudaSuccess)
    return check_launch("zero launch");
  return check_launch("zero");
}

}  // namespace lnfp8
