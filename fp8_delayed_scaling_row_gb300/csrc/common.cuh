// Shared device helpers of liblnfp8 (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <utility>
#include <cuda_fp8.h>
#include <stdint.h>

#include "lnfp8.h"

namespace lnfp8 {

// ---------------------------------------------------------------- host side
// Error bookkeeping (implemented in api.cu).
lnfp8_status set_error(lnfp8_status st, const char* fmt, ...);
lnfp8_status check_launch(const char* what);
void clear_error();
int num_sms();

// Launch accounting (api.cu): every kernel the library launches is counted,
// and, while the profiler is on, bracketed by CUDA events on its stream.
void launch_begin(const char* kind, cudaStream_t st);
void launch_end(cudaStream_t st);
struct LaunchScope {
  cudaStream_t st;
  LaunchScope(const char* kind, cudaStream_t s) : st(s) { launch_begin(kind, s); }
  ~LaunchScope() { launch_end(st); }
};

// Sticky device status word (defined next to the kernels that set it, in
// gemm.cu): bit 0 = a bounded wait gave up. Read and cleared from the host.
constexpr unsigned int kStatusTimeout = 1u;
lnfp8_status status_read_clear(cudaStream_t st, unsigned int* word);

// Programmatic dependent launch: every kernel of the library is launched so
// that it may start while the previous kernel on the stream finishes; each
// kernel runs only set-up that reads no data before pdl_wait(), which returns
// once the previous grid has completed and its writes are visible. Because
// every kernel waits before it completes, the ordering is transitive.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

bool pdl_enabled();  // off when the environment sets LNFP8_NO_PDL

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- numerics
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// Two fp32 -> two bf16 (nearest even), packed low = a, high = b.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two fp32 -> two FP8 codes (nearest even, saturating to the largest finite
// value), packed low byte = a, high byte = b.
template <int DT>
__device__ __forceinline__ uint16_t cvt_fp8x2(float a, float b) {
  __nv_fp8x2_storage_t r = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE,
                                                    DT == LNFP8_E4M3 ? __NV_E4M3 : __NV_E5M2);
  return (uint16_t)r;
}

// Eight scaled values -> eight codes in a uint2 (byte i = value i).
template <int DT>
__device__ __forceinline__ uint2 cvt_fp8x8(const float* v, float s) {
  uint2 r;
  r.x = (uint32_t)cvt_fp8x2<DT>(__fmul_rn(v[0], s), __fmul_rn(v[1], s)) |
        ((uint32_t)cvt_fp8x2<DT>(__fmul_rn(v[2], s), __fmul_rn(v[3], s)) << 16);
  r.y = (uint32_t)cvt_fp8x2<DT>(__fmul_rn(v[4], s), __fmul_rn(v[5], s)) |
        ((uint32_t)cvt_fp8x2<DT>(__fmul_rn(v[6], s), __fmul_rn(v[7], s)) << 16);
  return r;
}

// |x| as the ordered bit pattern used for amax: NaN > Inf > finite.
__device__ __forceinline__ uint32_t abs_bits(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// amax_cur holds a non-negative fp32 (or NaN); its bit pattern orders like the value.
__device__ __forceinline__ void atomic_max_amax(float* amax_cur, uint32_t bits) {
  atomicMax(reinterpret_cast<unsigned int*>(amax_cur), bits);
}

// Block-wide max of a per-thread amax, then one atomic per block.
// `red` must hold blockDim.x / 32 words.
__device__ __forceinline__ void block_amax_commit(uint32_t v, uint32_t* red, float* amax_cur) {
  v = warp_max_u32(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    uint32_t m = l < nw ? red[l] : 0u;
    m = warp_max_u32(m);
    if (l == 0 && m != 0u && amax_cur != nullptr) atomic_max_amax(amax_cur, m);
  }
}

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__host__ __device__ constexpr float fp8_max(int dt) { return dt == LNFP8_E4M3 ? 448.0f : 57344.0f; }

}  // namespace lnfp8
