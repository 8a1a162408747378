// ln_linear_bwd_noalloc: the LayerNormLinear / Linear backward for callers that
// cannot allocate device memory.
//
// ln_linear_bwd needs two scratch buffers besides its inputs and outputs: the
// E5M2 codes of dY and the bf16 gradient of the LayerNorm output. Its caller
// allocates them. Some callers cannot: code that runs where cudaMalloc is not
// allowed or not available to it (for instance a plug-in handed only the
// tensors of one layer by a host framework that owns all device memory, or an
// embedded runtime with a fixed memory budget decided before start-up). This
// entry point takes the same arguments without those two buffers and keeps
// them in one file-scope device array instead, of a fixed maximum size
// (kScratchBytes). The array is part of the library's device image: every GPU
// that loads the library holds it until the process exits.
//
// The pages have no counterpart of this entry point; it changes no numerics:
// it runs exactly the kernels of ln_linear_bwd on the same stream.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace lnfp8 {
namespace {

// 16 MiB: room for dY codes (M*N bytes, rounded up to 256) plus the bf16
// LayerNorm-output gradient (2*M*K bytes), e.g. M = 4096 tokens with
// K = 768 -> N = 2304.
constexpr size_t kScratchBytes = size_t(16) << 20;

__device__ __align__(256) unsigned char g_linear_bwd_scratch[kScratchBytes];

// The driver's cuCtxGetCurrent, looked up through the runtime (the library
// links no driver library at build time).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(ptr);
    return static_cast<CtxGetCurrentFn>(nullptr);
  }();
  return fn;
}

CUcontext current_context() {
  CUcontext c = nullptr;
  const CtxGetCurrentFn fn = ctx_get_current();
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  CUcontext ctx;  // the context the address belongs to
  void* addr;
};
std::mutex g_scratch_mu;
ScratchSlot g_scratch[kMaxDevices] = {};

// Device address of the scratch array in the current device's current
// context. In host code the array's name is only a host-side stand-in, so the
// address is looked up with that device current: once per device, and again
// whenever the current context is not the one the address was taken in (a
// caller that runs its own context on the device).
lnfp8_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_launch("ln_linear_bwd_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(LNFP8_ERR_UNSUPPORTED, "ln_linear_bwd_noalloc: device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchSlot& slot = g_scratch[dev];
  const CUcontext ctx = current_context();
  if (!slot.addr || ctx == nullptr || ctx != slot.ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_linear_bwd_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(LNFP8_ERR_CUDA, "ln_linear_bwd_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    slot.addr = p;
    slot.ctx = current_context();  // the lookup made the device's context current if none was
  }
  *out = slot.addr;
  return LNFP8_OK;
}

}  // namespace
}  // namespace lnfp8

using namespace lnfp8;

extern "C" lnfp8_status ln_linear_bwd_noalloc(const lnfp8_ln_linear_bwd_args* args, lnfp8_stream stream) {
  const char* who = "ln_linear_bwd_noalloc";
  clear_error();
  if (!args) return set_error(LNFP8_ERR_INVALID_ARG, "%s: args is NULL", who);
  if (args->M < 0 || args->K <= 0 || args->N <= 0)
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: bad sizes", who);
  const bool ln = args->gamma != nullptr;
  const size_t dyq_bytes = (size_t)args->M * (size_t)args->N;
  const size_t dyq_span = (dyq_bytes + 255) & ~size_t(255);
  const size_t dln_bytes = ln ? (size_t)args->M * (size_t)args->K * 2 : 0;
  if ((args->M > 0 && (size_t)args->M > kScratchBytes) || dyq_span + dln_bytes > kScratchBytes)
    return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE,
                     "%s: needs %zu bytes of scratch (M*N + 2*M*K) but the built-in scratch holds %zu", who,
                     dyq_span + dln_bytes, kScratchBytes);
  void* base = nullptr;
  const lnfp8_status st = scratch_address(&base);
  if (st != LNFP8_OK) return st;
  lnfp8_ln_linear_bwd_args a = *args;
  a.dyq = static_cast<uint8_t*>(base);
  a.dln = ln ? reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(base) + dyq_span) : nullptr;
  return ln_linear_bwd(&a, stream);
}
