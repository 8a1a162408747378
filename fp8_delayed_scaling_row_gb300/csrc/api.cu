// The C ABI of liblnfp8: argument validation, error reporting and the
// LayerNormLinear / LayerNormMLP forward and backward sequences.
//
// Each module call is a fixed sequence of the library's kernels on the
// caller's stream (TE tutorial, code blocks 1 and 3: te.LayerNormLinear /
// te.LayerNormMLP under fp8_autocast with the DelayedScaling recipe):
//   forward  : weight casts (K2) -> LayerNorm + cast (K1) -> FP8 GEMMs (K3,
//              GELU and the next cast fused into FC1's epilogue) -> state update (K4)
//   backward : dY cast + bias gradient (K2) -> dgrad GEMM with dGELU + dH cast
//              fused (K3) -> wgrad / dgrad GEMMs (K3) -> LayerNorm backward (K5)
//              -> state update (K4)
// The casts of a step all use the scales decided before the step (delayed
// scaling); the forward's scale_inv is saved for the backward because the
// update at the end of the forward replaces it.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace lnfp8 {

static thread_local char g_msg[512] = "";

lnfp8_status set_error(lnfp8_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_msg[0] = 0; }

lnfp8_status check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(LNFP8_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return LNFP8_OK;
}

bool pdl_enabled() {
  static const bool on = getenv("LNFP8_NO_PDL") == nullptr;
  return on;
}

// Token counts up to which ln_linear_fwd's automatic choice takes the one-launch
// fused path (when its other conditions hold).
constexpr int64_t kFusedAutoMaxTokens = 0;

// LNFP8_NO_PAIR=1 runs the FC2 data and weight gradients as two launches (for comparison)
bool pair_disabled() {
  static const bool off = getenv("LNFP8_NO_PAIR") != nullptr;
  return off;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

// ------------------------------------------------------------ launch accounting
namespace {
struct ProfRec {
  const char* kind;
  cudaEvent_t a, b;
  bool sampled;  // its time already went into the rows (a graph replay sample)
};
struct ProfRow {
  std::string kind;
  double ms;
  long long launches;
};
std::atomic<long long> g_launches{0};
std::atomic<bool> g_prof_on{false};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof_open;      // recorded, not yet collected
std::vector<cudaEvent_t> g_event_pool;  // reusable events
std::vector<ProfRow> g_prof_rows;      // totals since profiling was switched on
thread_local int g_open_idx = -1;

// external records become event nodes when the stream is being captured into a graph;
// outside a capture the flag is not accepted
unsigned record_flags(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();
    return cudaEventRecordDefault;
  }
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
}

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

void launch_begin(const char* kind, cudaStream_t st) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  ProfRec r{kind, pool_event(), pool_event(), false};
  cudaEventRecordWithFlags(r.a, st, record_flags(st));
  g_prof_open.push_back(r);
  g_open_idx = (int)g_prof_open.size() - 1;
}

void launch_end(cudaStream_t st) {
  if (!g_prof_on.load(std::memory_order_relaxed) || g_open_idx < 0) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_open_idx < (int)g_prof_open.size()) cudaEventRecordWithFlags(g_prof_open[g_open_idx].b, st, record_flags(st));
  g_open_idx = -1;
}

namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQ(p, who)                                                                       \
  do {                                                                                    \
    if (!(p)) return set_error(LNFP8_ERR_INVALID_ARG, "%s: %s is NULL", who, #p);          \
    if (!al16(p)) return set_error(LNFP8_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", who, #p); \
  } while (0)
#define OPT(p, who)                                                                       \
  do {                                                                                    \
    if ((p) && !al16(p)) return set_error(LNFP8_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", who, #p); \
  } while (0)
#define TRY(x)                             \
  do {                                     \
    const lnfp8_status _s = (x);           \
    if (_s != LNFP8_OK) return _s;         \
  } while (0)

lnfp8_status feat(int64_t v, const char* name, const char* who) {
  if (v <= 0 || v % 16 != 0)
    return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: %s = %lld must be a positive multiple of 16", who, name,
                     (long long)v);
  if (v > (1LL << 30)) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: %s = %lld too large", who, name, (long long)v);
  return LNFP8_OK;
}

lnfp8_status tokens(int64_t M, const char* who) {
  if (M < 0) return set_error(LNFP8_ERR_INVALID_ARG, "%s: M = %lld < 0", who, (long long)M);
  if (M > (1LL << 31) - 1) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: M = %lld too large", who, (long long)M);
  return LNFP8_OK;
}

lnfp8_status check_dtype(int dt, const char* who) {
  if (dt != LNFP8_E4M3 && dt != LNFP8_E5M2) return set_error(LNFP8_ERR_INVALID_ARG, "%s: bad FP8 dtype %d", who, dt);
  return LNFP8_OK;
}

lnfp8_status check_recipe(const lnfp8_recipe* r, const lnfp8_meta* m, const char* who) {
  if (!r) return set_error(LNFP8_ERR_INVALID_ARG, "%s: recipe is NULL", who);
  if (r->format < LNFP8_FORMAT_E4M3 || r->format > LNFP8_FORMAT_E5M2)
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: bad recipe format %d", who, r->format);
  if (r->algo != 0) return set_error(LNFP8_ERR_UNSUPPORTED, "%s: amax_compute_algo %d (only 0 = max)", who, r->algo);
  if (r->margin < 0 || r->margin > 30) return set_error(LNFP8_ERR_INVALID_ARG, "%s: margin %d", who, r->margin);
  if (m && r->history_len != m->history_len)
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: recipe.history_len %d != meta.history_len %d", who, r->history_len,
                     m->history_len);
  return LNFP8_OK;
}

int fwd_dtype(const lnfp8_recipe* r) { return r->format == LNFP8_FORMAT_E5M2 ? LNFP8_E5M2 : LNFP8_E4M3; }
int bwd_dtype(const lnfp8_recipe* r) { return r->format == LNFP8_FORMAT_E4M3 ? LNFP8_E4M3 : LNFP8_E5M2; }
uint64_t mask_all(int n, int dt) { return dt == LNFP8_E5M2 ? (n >= 64 ? ~0ull : ((1ull << n) - 1)) : 0ull; }

// End of a forward/backward: either the state update (which also saves the
// pre-update scale_inv) or, when deferred, only the snapshot.
lnfp8_status finish_state(const lnfp8_meta* m, const lnfp8_recipe* r, int dt, float* sinv_saved, int defer,
                          cudaStream_t st) {
  if (!defer) return update_launch(m, mask_all(m->n, dt), r->margin, sinv_saved, st);
  if (sinv_saved && cudaMemcpyAsync(sinv_saved, m->scale_inv, m->n * sizeof(float), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return check_launch("saving scale_inv");
  return LNFP8_OK;
}

// The split-K workspace shared by the GEMMs of one call (they run one after
// another): one flag area, as large as the largest any of them needs, then one
// slot area. Each GEMM takes it only if its own plan fits. Returns the flag
// span the call zeroes before its first kernel.
std::pair<void*, int64_t> share_split_ws(std::initializer_list<GemmArgs*> gs, void* ws, int64_t bytes,
                                         int64_t extra_flag_bytes = 0) {
  if (!ws || bytes <= 0) return {nullptr, 0};
  int64_t flags = extra_flag_bytes;
  for (const GemmArgs* g : gs) {
    const GemmPlan pl = gemm_plan(g->M, g->N, g->K, g->epi, true);
    if (pl.splits > 1 && pl.flag_bytes > flags) flags = pl.flag_bytes;
  }
  for (GemmArgs* g : gs) {
    g->ws = ws;
    g->ws_bytes = bytes;
    g->ws_flag_bytes = flags;
  }
  return {ws, flags < bytes ? flags : bytes};
}

// Workspace bytes that let every GEMM of a call split as planned.
int64_t shared_split_bytes(std::initializer_list<GemmPlan> pls) {
  int64_t flags = 0, slots = 0;
  for (const GemmPlan& pl : pls) {
    flags = pl.flag_bytes > flags ? pl.flag_bytes : flags;
    slots = pl.slot_bytes > slots ? pl.slot_bytes : slots;
  }
  return slots ? flags + slots : 0;
}

GemmArgs gemm_args(const uint8_t* a, int al, int adt, const uint8_t* b, int bl, int bdt, int64_t M, int64_t N,
                   int64_t K, const float* sa, const float* sb) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.a = a; g.a_layout = al; g.a_dtype = adt;
  g.b = b; g.b_layout = bl; g.b_dtype = bdt;
  g.M = M; g.N = N; g.K = K;
  g.sinv_a = sa; g.sinv_b = sb;
  g.epi = EPI_STORE;
  return g;
}

// A weight-gradient GEMM contracts over the tokens; with no tokens it is zero.
lnfp8_status wgrad(const GemmArgs& g, uint16_t* out, cudaStream_t st) {
  if (g.K == 0) {
    if (cudaMemsetAsync(out, 0, g.M * g.N * sizeof(uint16_t), st) != cudaSuccess) return check_launch("zero wgrad");
    return LNFP8_OK;
  }
  return gemm_launch(g, st);
}

}  // namespace
}  // namespace lnfp8

using namespace lnfp8;

extern "C" {

const char* lnfp8_last_error(void) { return g_msg; }

int lnfp8_version(void) { return 400; }

long long lnfp8_launch_count(void) { return g_launches.load(); }

lnfp8_status lnfp8_profile_enable(int on) {
  clear_error();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof_open) {
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof_open.clear();
  g_prof_rows.clear();
  g_prof_on.store(on != 0);
  return LNFP8_OK;
}

namespace {
// adds the elapsed time of every open record to the rows; caller holds g_prof_mu
void prof_add_open(bool only_unsampled) {
  for (auto& r : g_prof_open) {
    if (only_unsampled && r.sampled) continue;
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    r.sampled = true;
    bool found = false;
    for (auto& row : g_prof_rows)
      if (row.kind == r.kind) {
        row.ms += ms;
        row.launches += 1;
        found = true;
        break;
      }
    if (!found) g_prof_rows.push_back({r.kind, (double)ms, 1});
  }
}
}  // namespace

lnfp8_status lnfp8_profile_sample(void) {
  clear_error();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  prof_add_open(false);
  return LNFP8_OK;
}

int lnfp8_profile_collect(void) {
  clear_error();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  prof_add_open(true);
  for (auto& r : g_prof_open) {
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof_open.clear();
  return (int)g_prof_rows.size();
}

lnfp8_status lnfp8_profile_get(int i, const char** kind, double* total_ms, long long* launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (i < 0 || i >= (int)g_prof_rows.size() || !kind || !total_ms || !launches)
    return set_error(LNFP8_ERR_INVALID_ARG, "lnfp8_profile_get: bad index or NULL output");
  *kind = g_prof_rows[i].kind.c_str();
  *total_ms = g_prof_rows[i].ms;
  *launches = g_prof_rows[i].launches;
  return LNFP8_OK;
}

lnfp8_status lnfp8_sync_status(lnfp8_stream stream) {
  clear_error();
  unsigned int word = 0;
  TRY(status_read_clear((cudaStream_t)stream, &word));
  if (word & kStatusTimeout) return set_error(LNFP8_ERR_TIMEOUT, "a bounded device wait gave up");
  return LNFP8_OK;
}

lnfp8_status lnfp8_selftest_timeout(int64_t limit_ns, lnfp8_stream stream) {
  clear_error();
  if (limit_ns < 1000 || limit_ns > 1000000000LL)
    return set_error(LNFP8_ERR_INVALID_ARG, "lnfp8_selftest_timeout: limit_ns must be in [1e3, 1e9]");
  return selftest_timeout_launch(limit_ns, (cudaStream_t)stream);
}

lnfp8_status lnfp8_meta_init(const lnfp8_meta* meta, lnfp8_stream stream) {
  clear_error();
  TRY(validate_meta(meta, 0, "lnfp8_meta_init"));
  return meta_init_launch(meta, (cudaStream_t)stream);
}

lnfp8_status amax_history_update(const lnfp8_meta* meta, const lnfp8_recipe* recipe, const int* dtype_per_tensor,
                                 float* scale_inv_before, lnfp8_stream stream) {
  const char* who = "amax_history_update";
  clear_error();
  TRY(validate_meta(meta, 0, who));
  TRY(check_recipe(recipe, meta, who));
  if (!dtype_per_tensor) return set_error(LNFP8_ERR_INVALID_ARG, "%s: dtype_per_tensor is NULL", who);
  uint64_t mask = 0;
  for (int i = 0; i < meta->n; ++i) {
    TRY(check_dtype(dtype_per_tensor[i], who));
    if (dtype_per_tensor[i] == LNFP8_E5M2) mask |= 1ull << i;
  }
  return update_launch(meta, mask, recipe->margin, scale_inv_before, (cudaStream_t)stream);
}

lnfp8_status amax_history_update_many(const lnfp8_meta* metas, int count, const lnfp8_recipe* recipe,
                                      const int* dtypes, float* const* scale_inv_before, lnfp8_stream stream) {
  const char* who = "amax_history_update_many";
  clear_error();
  if (count < 0 || count > kMaxUpdateSets)
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: count = %d (0..%d)", who, count, kMaxUpdateSets);
  if (count == 0) return LNFP8_OK;
  if (!metas || !dtypes) return set_error(LNFP8_ERR_INVALID_ARG, "%s: metas or dtypes is NULL", who);
  const lnfp8_meta* ptrs[kMaxUpdateSets];
  uint64_t masks[kMaxUpdateSets];
  int off = 0;
  for (int k = 0; k < count; ++k) {
    TRY(validate_meta(&metas[k], 0, who));
    TRY(check_recipe(recipe, &metas[k], who));
    uint64_t mask = 0;
    for (int i = 0; i < metas[k].n; ++i, ++off) {
      TRY(check_dtype(dtypes[off], who));
      if (dtypes[off] == LNFP8_E5M2) mask |= 1ull << i;
    }
    ptrs[k] = &metas[k];
    masks[k] = mask;
  }
  // one CTA per slot updates it in place: a set listed twice (or two sets sharing state) would race
  for (int k = 0; k < count; ++k)
    for (int q = k + 1; q < count; ++q) {
      const lnfp8_meta &a = metas[k], &b = metas[q];
      const uintptr_t pa = reinterpret_cast<uintptr_t>(a.amax_cur), pb = reinterpret_cast<uintptr_t>(b.amax_cur);
      const bool overlap = pa < pb + 4u * (uintptr_t)b.n && pb < pa + 4u * (uintptr_t)a.n;
      if (overlap || a.scale == b.scale || a.amax_history == b.amax_history)
        return set_error(LNFP8_ERR_INVALID_ARG, "%s: sets %d and %d share state", who, k, q);
    }
  return update_many_launch(ptrs, masks, scale_inv_before, count, recipe->margin, (cudaStream_t)stream);
}

lnfp8_status fp8_quantize(const void* in, int in_is_fp32, int64_t rows, int64_t cols, int dtype, const float* scale,
                          float* amax_cur, uint8_t* out, uint8_t* out_t, float* colsum, lnfp8_stream stream) {
  const char* who = "fp8_quantize";
  clear_error();
  TRY(tokens(rows, who));
  TRY(feat(cols, "cols", who));
  TRY(check_dtype(dtype, who));
  if (rows > 0) REQ(in, who);
  if (!scale || !amax_cur) return set_error(LNFP8_ERR_INVALID_ARG, "%s: scale and amax_cur are required", who);
  OPT(out, who);
  OPT(out_t, who);
  OPT(colsum, who);
  return cast_launch(in, in_is_fp32 != 0, rows, cols, dtype, scale, amax_cur, out, out_t, colsum, (cudaStream_t)stream);
}

lnfp8_status fp8_weight_quantize(const uint16_t* w, int64_t rows, int64_t cols, const lnfp8_meta* meta,
                                 const lnfp8_recipe* recipe, int dtype, uint8_t* codes, lnfp8_stream stream) {
  const char* who = "fp8_weight_quantize";
  clear_error();
  TRY(tokens(rows, who));
  TRY(feat(cols, "cols", who));
  TRY(check_dtype(dtype, who));
  if (!meta || !recipe) return set_error(LNFP8_ERR_INVALID_ARG, "%s: meta and recipe are required", who);
  TRY(validate_meta(meta, 1, who));
  TRY(check_recipe(recipe, nullptr, who));  // the weight's own history length is its own
  if (rows > 0) {
    REQ(w, who);
    REQ(codes, who);
  }
  cudaStream_t st = (cudaStream_t)stream;
  TRY(cast_launch(w, false, rows, cols, dtype, meta->scale, meta->amax_cur, nullptr, nullptr, nullptr, st));
  TRY(update_launch(meta, mask_all(1, dtype), recipe->margin, nullptr, st));
  return cast_launch(w, false, rows, cols, dtype, meta->scale, meta->amax_cur, codes, nullptr, nullptr, st);
}

// Copies a weight's stored scale_inv into the forward's saved snapshot (after the state step wrote it).
static lnfp8_status save_weight_sinv(float* sinv_saved_slot, const float* w_scale_inv, cudaStream_t st) {
  if (cudaMemcpyAsync(sinv_saved_slot, w_scale_inv, sizeof(float), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return check_launch("saving the weight's scale_inv");
  return LNFP8_OK;
}

lnfp8_status ln_fwd_cast(const uint16_t* x, const uint16_t* gamma, const uint16_t* beta, float eps, int64_t M, int64_t D,
                         int dtype, const float* scale, float* amax_cur, uint8_t* out, float* mu, float* rsigma,
                         float* y_debug, lnfp8_stream stream) {
  const char* who = "ln_fwd_cast";
  clear_error();
  TRY(tokens(M, who));
  TRY(feat(D, "D", who));
  TRY(check_dtype(dtype, who));
  if (D > 8192) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: D = %lld > 8192", who, (long long)D);
  if (!(eps >= 0.f)) return set_error(LNFP8_ERR_INVALID_ARG, "%s: eps must be >= 0", who);
  REQ(gamma, who);
  REQ(beta, who);
  if (!scale || !amax_cur) return set_error(LNFP8_ERR_INVALID_ARG, "%s: scale and amax_cur are required", who);
  if (M > 0) {
    REQ(x, who);
    REQ(out, who);
    REQ(mu, who);
    REQ(rsigma, who);
  }
  OPT(y_debug, who);
  return ln_fwd_launch(x, gamma, beta, eps, M, D, dtype, scale, amax_cur, out, mu, rsigma, y_debug, (cudaStream_t)stream);
}

lnfp8_status ln_bwd(const uint16_t* dy, const uint16_t* x, const uint16_t* gamma, const float* mu, const float* rsigma,
                    int64_t M, int64_t D, uint16_t* dx, float* dgamma, float* dbeta, lnfp8_stream stream) {
  const char* who = "ln_bwd";
  clear_error();
  TRY(tokens(M, who));
  TRY(feat(D, "D", who));
  if (D > 8192) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: D = %lld > 8192", who, (long long)D);
  REQ(gamma, who);
  REQ(dgamma, who);
  REQ(dbeta, who);
  if (M > 0) {
    REQ(dy, who);
    REQ(x, who);
    REQ(mu, who);
    REQ(rsigma, who);
    REQ(dx, who);
  }
  return ln_bwd_launch(dy, x, gamma, mu, rsigma, M, D, dx, dgamma, dbeta, (cudaStream_t)stream);
}

lnfp8_status fp8_gemm(const uint8_t* A, int a_layout, int a_dtype, const uint8_t* B, int b_layout, int b_dtype, int64_t M,
                      int64_t N, int64_t K, const float* sinv_a, const float* sinv_b, const uint16_t* bias,
                      uint16_t* out, void* workspace, int64_t workspace_bytes, lnfp8_stream stream) {
  const char* who = "fp8_gemm";
  clear_error();
  TRY(tokens(M, who));
  TRY(feat(N, "N", who));
  TRY(feat(K, "K", who));
  TRY(check_dtype(a_dtype, who));
  TRY(check_dtype(b_dtype, who));
  if ((a_layout != 0 && a_layout != 1) || (b_layout != 0 && b_layout != 1))
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: layouts must be 0 or 1", who);
  if (a_layout == 1 && M % 16 != 0)
    return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: M must be a multiple of 16 when A is stored [K, M]", who);
  if (!sinv_a || !sinv_b) return set_error(LNFP8_ERR_INVALID_ARG, "%s: sinv_a and sinv_b are required", who);
  OPT(bias, who);
  if (M > 0) {
    REQ(A, who);
    REQ(out, who);
  }
  REQ(B, who);
  OPT(workspace, who);
  if (workspace && workspace_bytes < 0) return set_error(LNFP8_ERR_INVALID_ARG, "%s: workspace_bytes < 0", who);
  GemmArgs g = gemm_args(A, a_layout, a_dtype, B, b_layout, b_dtype, M, N, K, sinv_a, sinv_b);
  g.bias = bias;
  g.out = out;
  TRY(zero_launch({share_split_ws({&g}, workspace, workspace_bytes)}, (cudaStream_t)stream));
  return gemm_launch(g, (cudaStream_t)stream);
}

int64_t lnfp8_ln_mlp_fwd_workspace_size(int64_t M, int64_t D, int64_t F) {
  if (M < 0 || D < 0 || F < 0) return -1;
  if (M == 0 || D == 0 || F == 0) return 0;
  const int64_t num_m2 = ((M + 127) / 128 + 1) / 2;  // one counter per 256-row block
  return ((num_m2 * 4 + 255) / 256) * 256;
}

int64_t lnfp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return -1;
  return gemm_plan(M, N, K, EPI_STORE, true).ws_bytes;
}

int64_t lnfp8_ln_linear_bwd_workspace_size(int64_t M, int64_t K, int64_t N) {
  if (M < 0 || N < 0 || K < 0) return -1;
  GemmArgs wg;
  memset(&wg, 0, sizeof(wg));
  wg.M = N;
  wg.N = K;
  wg.K = M;
  return shared_split_bytes({pair_plan(wg), gemm_plan(M, K, N, EPI_STORE, true), gemm_plan(N, K, M, EPI_STORE, true)});
}

int64_t lnfp8_ln_mlp_bwd_workspace_size(int64_t M, int64_t D, int64_t F) {
  if (M < 0 || D < 0 || F < 0) return -1;
  GemmArgs w2;
  memset(&w2, 0, sizeof(w2));
  w2.M = D;
  w2.N = F;
  w2.K = M;
  // dW2 runs in one launch with the FC2 data gradient (its own exchange plan), dLN and dW1 alone
  GemmArgs w1 = w2;
  w1.M = F;
  w1.N = D;
  // the weight gradients run paired with the data gradients (their own exchange plan); without pairing the GEMMs' own
  return shared_split_bytes({pair_plan(w2), pair_plan(w1), gemm_plan(D, F, M, EPI_STORE, true),
                             gemm_plan(M, D, F, EPI_STORE, true), gemm_plan(F, D, M, EPI_STORE, true)});
}

int lnfp8_ctx_offsets(int op, int64_t M, int64_t D, int64_t F, int64_t* offsets, int max_offsets) {
  if (M < 0 || D < 0 || F < 0 || !offsets) return -1;
  int64_t sizes[8];
  int n = 0;
  if (op == LNFP8_OP_LN_LINEAR || op == LNFP8_OP_LINEAR) {
    sizes[n++] = M * D;  // xq
    sizes[n++] = F * D;  // wq
    if (op == LNFP8_OP_LN_LINEAR) {
      sizes[n++] = 4 * M;  // mu
      sizes[n++] = 4 * M;  // rsigma
    }
    sizes[n++] = 4 * 2;  // sinv_saved
  } else if (op == LNFP8_OP_LN_MLP) {
    sizes[n++] = M * D;      // lnq
    sizes[n++] = F * D;      // w1q
    sizes[n++] = D * F;      // w2q
    sizes[n++] = 2 * M * F;  // h
    sizes[n++] = M * F;      // aq
    sizes[n++] = 4 * M;      // mu
    sizes[n++] = 4 * M;      // rsigma
    sizes[n++] = 4 * 4;      // sinv_saved
  } else {
    return -1;
  }
  if (max_offsets < n + 1) return -1;
  int64_t off = 0;
  for (int i = 0; i < n; ++i) {
    offsets[i] = off;
    off += (sizes[i] + 255) / 256 * 256;
  }
  offsets[n] = off;
  return n;
}

int64_t lnfp8_ctx_bytes(int op, int64_t M, int64_t D, int64_t F) {
  int64_t off[9];
  const int n = lnfp8_ctx_offsets(op, M, D, F, off, 9);
  return n < 0 ? -1 : off[n];
}

lnfp8_status ln_linear_fwd(const lnfp8_ln_linear_fwd_args* a, lnfp8_stream stream) {
  const char* who = "ln_linear_fwd";
  clear_error();
  if (!a) return set_error(LNFP8_ERR_INVALID_ARG, "%s: args is NULL", who);
  cudaStream_t st = (cudaStream_t)stream;
  TRY(tokens(a->M, who));
  TRY(feat(a->K, "K", who));
  TRY(feat(a->N, "N", who));
  TRY(validate_meta(&a->meta, 2, who));
  TRY(check_recipe(&a->recipe, &a->meta, who));
  const bool ln = a->gamma != nullptr;
  if (ln) {
    REQ(a->beta, who);
    if (a->K > 8192) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: K > 8192 with LayerNorm", who);
  }
  const bool w8 = a->w_scale_inv != nullptr;  // weight stored as FP8 codes
  OPT(a->residual, who);
  if (a->residual) {
    if (!ln) return set_error(LNFP8_ERR_INVALID_ARG, "%s: residual needs the LayerNorm (gamma)", who);
    if (a->M > 0) REQ(a->x_sum, who);
  }
  if (!w8) REQ(a->w, who);
  REQ(a->wq, who);
  OPT(a->bias, who);
  OPT(a->ln_out_debug, who);
  if (!a->sinv_saved) return set_error(LNFP8_ERR_INVALID_ARG, "%s: sinv_saved is NULL", who);
  if (a->M > 0) {
    REQ(a->x, who);
    REQ(a->y, who);
    REQ(a->xq, who);
    if (ln) {
      REQ(a->mu, who);
      REQ(a->rsigma, who);
    }
  }
  const int fdt = fwd_dtype(&a->recipe);
  const lnfp8_meta& m = a->meta;
  if (a->path < LNFP8_PATH_AUTO || a->path > LNFP8_PATH_SEPARATE)
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: path = %d", who, a->path);
  const bool fused_ok = a->residual == nullptr && ln_linear_small_fits(a->M, a->K, a->N);
  if (a->path == LNFP8_PATH_FUSED && !fused_ok)
    return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: the fused path needs 1 <= M, K <= 768 and no residual", who);
  if (a->path == LNFP8_PATH_FUSED || (a->path == LNFP8_PATH_AUTO && fused_ok && a->M <= kFusedAutoMaxTokens)) {
    SmallLinearArgs sa;
    sa.M = a->M;
    sa.N = a->N;
    sa.K = a->K;
    sa.x = a->x;
    sa.gamma = a->gamma;
    sa.beta = a->beta;
    sa.eps = a->eps;
    sa.w = w8 ? nullptr : a->w;
    sa.wq_in = w8 ? a->wq : nullptr;
    sa.bias = a->bias;
    sa.y = a->y;
    sa.xq = a->xq;
    sa.wq = w8 ? nullptr : a->wq;
    sa.mu = a->mu;
    sa.rsigma = a->rsigma;
    sa.ydbg = a->ln_out_debug;
    sa.scale = m.scale;
    sa.scale_inv = m.scale_inv;
    sa.w_scale_inv = w8 ? a->w_scale_inv : nullptr;
    sa.amax_cur = m.amax_cur;
    TRY(ln_linear_small_launch(sa, fdt, st));
    TRY(finish_state(&m, &a->recipe, fdt, a->sinv_saved, a->defer_update, st));
    return w8 ? save_weight_sinv(a->sinv_saved + 1, a->w_scale_inv, st) : LNFP8_OK;
  }
  if (ln) {
    // a small weight cast rides in the LayerNorm launch, a large one streams through its own
    WeightCastJob wc = {};
    if (!w8 && cast_streams_rows(a->N, a->K))
      TRY(cast_launch(a->w, false, a->N, a->K, fdt, m.scale + 1, m.amax_cur + 1, a->wq, nullptr, nullptr, st));
    else if (!w8)
      weight_cast_add(wc, 0, a->w, a->N, a->K, m.scale + 1, m.amax_cur + 1, a->wq);
    // the LayerNorm launch also saves the scale_inv this forward casts with (for the GEMM and the backward)
    const SinvSnapshot snap = {a->sinv_saved, {m.scale_inv + 0, w8 ? a->w_scale_inv : m.scale_inv + 1}, 2};
    TRY(ln_fwd_launch(a->x, a->gamma, a->beta, a->eps, a->M, a->K, fdt, m.scale + 0, m.amax_cur + 0, a->xq, a->mu,
                      a->rsigma, a->ln_out_debug, st, a->residual, a->x_sum, &wc, &snap));
    // the GEMM dequantises with the saved scale_inv, so it can carry the state update: both
    // amaxes are final when it starts
    GemmArgs g = gemm_args(a->xq, 0, fdt, a->wq, 0, fdt, a->M, a->N, a->K, a->sinv_saved + 0, a->sinv_saved + 1);
    g.bias = a->bias;
    g.out = a->y;
    if (a->M > 0 && !a->defer_update) g.upd = update_job(&m, mask_all(m.n, fdt), a->recipe.margin);
    TRY(gemm_launch(g, st));
    if (g.upd.n > 0) return LNFP8_OK;
    // the snapshot is taken: only the update remains (none when deferred)
    return finish_state(&m, &a->recipe, fdt, nullptr, a->defer_update, st);
  }
  if (!w8) TRY(cast_launch(a->w, false, a->N, a->K, fdt, m.scale + 1, m.amax_cur + 1, a->wq, nullptr, nullptr, st));
  TRY(cast_launch(a->x, false, a->M, a->K, fdt, m.scale + 0, m.amax_cur + 0, a->xq, nullptr, nullptr, st));
  GemmArgs g = gemm_args(a->xq, 0, fdt, a->wq, 0, fdt, a->M, a->N, a->K, m.scale_inv + 0,
                         w8 ? a->w_scale_inv : m.scale_inv + 1);
  g.bias = a->bias;
  g.out = a->y;
  TRY(gemm_launch(g, st));
  TRY(finish_state(&m, &a->recipe, fdt, a->sinv_saved, a->defer_update, st));
  return w8 ? save_weight_sinv(a->sinv_saved + 1, a->w_scale_inv, st) : LNFP8_OK;
}

lnfp8_status ln_linear_bwd(const lnfp8_ln_linear_bwd_args* a, lnfp8_stream stream) {
  const char* who = "ln_linear_bwd";
  clear_error();
  if (!a) return set_error(LNFP8_ERR_INVALID_ARG, "%s: args is NULL", who);
  cudaStream_t st = (cudaStream_t)stream;
  TRY(tokens(a->M, who));
  TRY(feat(a->K, "K", who));
  TRY(feat(a->N, "N", who));
  TRY(validate_meta(&a->meta, 1, who));
  TRY(check_recipe(&a->recipe, &a->meta, who));
  const bool ln = a->gamma != nullptr;
  REQ(a->wq, who);
  REQ(a->dw, who);
  OPT(a->dbias, who);
  if (!a->sinv_saved) return set_error(LNFP8_ERR_INVALID_ARG, "%s: sinv_saved is NULL", who);
  if (ln) {
    if (a->K > 8192) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: K > 8192 with LayerNorm", who);
    REQ(a->dgamma, who);
    REQ(a->dbeta, who);
  }
  if (a->M > 0) {
    REQ(a->dy, who);
    REQ(a->xq, who);
    REQ(a->dx, who);
    REQ(a->dyq, who);
    if (ln) {
      REQ(a->x, who);
      REQ(a->mu, who);
      REQ(a->rsigma, who);
      REQ(a->dln, who);
    }
  }
  const int fdt = fwd_dtype(&a->recipe), bdt = bwd_dtype(&a->recipe);
  const lnfp8_meta& m = a->meta;
  OPT(a->gemm_ws, who);
  uint16_t* dln = ln ? a->dln : a->dx;
  if (a->gemm_ws && a->gemm_ws_bytes < 0) return set_error(LNFP8_ERR_INVALID_ARG, "%s: gemm_ws_bytes < 0", who);
  GemmArgs dg = gemm_args(a->dyq, 0, bdt, a->wq, 1, fdt, a->M, a->K, a->N, m.scale_inv + 0, a->sinv_saved + 1);
  dg.out = dln;
  GemmArgs wg = gemm_args(a->dyq, 1, bdt, a->xq, 1, fdt, a->N, a->K, a->M, m.scale_inv + 0, a->sinv_saved + 0);
  wg.out = a->dw;
  // the data and weight gradients share one persistent launch when both are non-empty
  const bool paired = a->M > 0 && a->K > 0 && a->N > 0 && !pair_disabled();
  const auto flags = share_split_ws({&dg, &wg}, a->gemm_ws, a->gemm_ws_bytes, paired ? pair_plan(wg).flag_bytes : 0);
  // the accumulated outputs and the split-K flags are cleared first (one launch)
  TRY(zero_launch({{a->dbias, a->N * 4}, {ln ? a->dgamma : nullptr, a->K * 4}, {ln ? a->dbeta : nullptr, a->K * 4},
                   flags},
                  st));
  TRY(cast_launch(a->dy, false, a->M, a->N, bdt, m.scale + 0, m.amax_cur + 0, a->dyq, nullptr, a->dbias, st, false));
  if (paired) {
    TRY(gemm_pair_launch(dg, wg, st));
  } else {
    TRY(gemm_launch(dg, st));
    TRY(wgrad(wg, a->dw, st));
  }
  bool updated = false;
  if (ln) {
    const UpdateJob job = update_job(&m, mask_all(m.n, bdt), a->recipe.margin);
    TRY(ln_bwd_launch(dln, a->x, a->gamma, a->mu, a->rsigma, a->M, a->K, a->dx, a->dgamma, a->dbeta, st, false,
                      a->defer_update ? nullptr : &job, &updated));
  }
  return updated ? LNFP8_OK : finish_state(&m, &a->recipe, bdt, nullptr, a->defer_update, st);
}

lnfp8_status ln_mlp_fwd(const lnfp8_ln_mlp_fwd_args* a, lnfp8_stream stream) {
  const char* who = "ln_mlp_fwd";
  clear_error();
  if (!a) return set_error(LNFP8_ERR_INVALID_ARG, "%s: args is NULL", who);
  cudaStream_t st = (cudaStream_t)stream;
  TRY(tokens(a->M, who));
  TRY(feat(a->D, "D", who));
  TRY(feat(a->F, "F", who));
  if (a->D > 8192) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: D > 8192", who);
  TRY(validate_meta(&a->meta, 4, who));
  TRY(check_recipe(&a->recipe, &a->meta, who));
  REQ(a->gamma, who);
  REQ(a->beta, who);
  OPT(a->residual, who);
  if (a->residual && a->M > 0) REQ(a->x_sum, who);
  const bool w8 = a->w1_scale_inv != nullptr;  // weights stored as FP8 codes
  if (w8 != (a->w2_scale_inv != nullptr))
    return set_error(LNFP8_ERR_INVALID_ARG, "%s: w1_scale_inv and w2_scale_inv must be given together", who);
  if (!w8) {
    REQ(a->w1, who);
    REQ(a->w2, who);
  }
  REQ(a->w1q, who);
  REQ(a->w2q, who);
  OPT(a->b1, who);
  OPT(a->b2, who);
  OPT(a->ln_out_debug, who);
  OPT(a->act_debug, who);
  if (!a->sinv_saved) return set_error(LNFP8_ERR_INVALID_ARG, "%s: sinv_saved is NULL", who);
  if (a->M > 0) {
    REQ(a->x, who);
    REQ(a->y, who);
    REQ(a->lnq, who);
    REQ(a->mu, who);
    REQ(a->rsigma, who);
    REQ(a->h, who);
    REQ(a->aq, who);
  }
  OPT(a->gemm_ws, who);
  const int fdt = fwd_dtype(&a->recipe);
  const lnfp8_meta& m = a->meta;
  // FC1 and FC2 in one launch when the caller gave room for the FC1 tiles' readiness counters
  const int64_t ready_bytes = lnfp8_ln_mlp_fwd_workspace_size(a->M, a->D, a->F);
  const bool fused = a->M > 0 && a->gemm_ws && ready_bytes > 0 && a->gemm_ws_bytes >= ready_bytes && !pair_disabled();
  // small weight casts (and the FC1 tiles' readiness counters) ride in the LayerNorm launch,
  // large ones stream through their own launches
  WeightCastJob wc = {};
  if (!w8) {
    if (cast_streams_rows(a->F, a->D))
      TRY(cast_launch(a->w1, false, a->F, a->D, fdt, m.scale + 1, m.amax_cur + 1, a->w1q, nullptr, nullptr, st));
    else
      weight_cast_add(wc, 0, a->w1, a->F, a->D, m.scale + 1, m.amax_cur + 1, a->w1q);
    if (cast_streams_rows(a->D, a->F))
      TRY(cast_launch(a->w2, false, a->D, a->F, fdt, m.scale + 3, m.amax_cur + 3, a->w2q, nullptr, nullptr, st));
    else
      weight_cast_add(wc, 1, a->w2, a->D, a->F, m.scale + 3, m.amax_cur + 3, a->w2q);
  }
  if (fused) {
    wc.zero = static_cast<uint32_t*>(a->gemm_ws);
    wc.zero_n = (ready_bytes + 3) / 4;
  }
  // the LayerNorm launch also saves the scale_inv this forward casts with (for FC2 and the backward)
  const SinvSnapshot snap = {a->sinv_saved, {m.scale_inv + 0, w8 ? a->w1_scale_inv : m.scale_inv + 1, m.scale_inv + 2,
                                             w8 ? a->w2_scale_inv : m.scale_inv + 3}, 4};
  TRY(ln_fwd_launch(a->x, a->gamma, a->beta, a->eps, a->M, a->D, fdt, m.scale + 0, m.amax_cur + 0, a->lnq, a->mu,
                    a->rsigma, a->ln_out_debug, st, a->residual, a->x_sum, &wc, &snap));
  GemmArgs f1 = gemm_args(a->lnq, 0, fdt, a->w1q, 0, fdt, a->M, a->F, a->D, m.scale_inv + 0,
                          w8 ? a->w1_scale_inv : m.scale_inv + 1);
  f1.epi = EPI_GELU;
  f1.bias = a->b1;
  f1.out = a->h;
  f1.out_q = a->aq;
  f1.q_dtype = fdt;
  f1.scale_q = m.scale + 2;
  f1.amax_q = m.amax_cur + 2;
  f1.dbg = a->act_debug;
  // FC2 dequantises with the saved scale_inv: the state update may run while it does
  GemmArgs f2 = gemm_args(a->aq, 0, fdt, a->w2q, 0, fdt, a->M, a->D, a->F, a->sinv_saved + 2, a->sinv_saved + 3);
  f2.bias = a->b2;
  f2.out = a->y;
  if (fused) {
    f1.ws = a->gemm_ws;
    f1.ws_bytes = a->gemm_ws_bytes;
    TRY(gemm_pair_launch(f1, f2, st));
  } else {
    // every amax of the forward is final when FC2 starts: it carries the state update
    if (a->M > 0 && !a->defer_update) f2.upd = update_job(&m, mask_all(m.n, fdt), a->recipe.margin);
    TRY(gemm_launch(f1, st));
    TRY(gemm_launch(f2, st));
    if (f2.upd.n > 0) return LNFP8_OK;
  }
  // the snapshot is taken: only the update remains (none when deferred)
  return finish_state(&m, &a->recipe, fdt, nullptr, a->defer_update, st);
}

lnfp8_status ln_mlp_bwd(const lnfp8_ln_mlp_bwd_args* a, lnfp8_stream stream) {
  const char* who = "ln_mlp_bwd";
  clear_error();
  if (!a) return set_error(LNFP8_ERR_INVALID_ARG, "%s: args is NULL", who);
  cudaStream_t st = (cudaStream_t)stream;
  TRY(tokens(a->M, who));
  TRY(feat(a->D, "D", who));
  TRY(feat(a->F, "F", who));
  if (a->D > 8192) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "%s: D > 8192", who);
  TRY(validate_meta(&a->meta, 2, who));
  TRY(check_recipe(&a->recipe, &a->meta, who));
  REQ(a->gamma, who);
  REQ(a->w1q, who);
  REQ(a->w2q, who);
  REQ(a->dw1, who);
  REQ(a->dw2, who);
  REQ(a->dgamma, who);
  REQ(a->dbeta, who);
  OPT(a->db1, who);
  OPT(a->db2, who);
  OPT(a->dh_debug, who);
  if (!a->sinv_saved) return set_error(LNFP8_ERR_INVALID_ARG, "%s: sinv_saved is NULL", who);
  if (a->M > 0) {
    REQ(a->dy, who);
    REQ(a->x, who);
    REQ(a->lnq, who);
    REQ(a->mu, who);
    REQ(a->rsigma, who);
    REQ(a->h, who);
    REQ(a->aq, who);
    REQ(a->dx, who);
    REQ(a->dyq, who);
    REQ(a->dhq, who);
    REQ(a->dln, who);
  }
  const int fdt = fwd_dtype(&a->recipe), bdt = bwd_dtype(&a->recipe);
  const lnfp8_meta& m = a->meta;
  OPT(a->gemm_ws, who);
  if (a->gemm_ws && a->gemm_ws_bytes < 0) return set_error(LNFP8_ERR_INVALID_ARG, "%s: gemm_ws_bytes < 0", who);
  // FC2 wgrad: dW2 = dYq^T . Aq
  GemmArgs w2 = gemm_args(a->dyq, 1, bdt, a->aq, 1, fdt, a->D, a->F, a->M, m.scale_inv + 0, a->sinv_saved + 2);
  w2.out = a->dw2;
  // FC1 dgrad: dLN = dHq . W1q
  GemmArgs d1 = gemm_args(a->dhq, 0, bdt, a->w1q, 1, fdt, a->M, a->D, a->F, m.scale_inv + 1, a->sinv_saved + 1);
  d1.out = a->dln;
  // FC1 wgrad: dW1 = dHq^T . LNq
  GemmArgs w1 = gemm_args(a->dhq, 1, bdt, a->lnq, 1, fdt, a->F, a->D, a->M, m.scale_inv + 1, a->sinv_saved + 0);
  w1.out = a->dw1;
  // dW2 shares one launch with the FC2 data gradient when both are non-empty
  // (and dW1 with dLN): each data gradient shares one persistent launch with its weight gradient
  const bool paired = a->M > 0 && a->F > 0 && a->D > 0 && !pair_disabled();
  const auto flags = share_split_ws({&w2, &d1, &w1}, a->gemm_ws, a->gemm_ws_bytes,
                                    paired ? std::max(pair_plan(w2).flag_bytes, pair_plan(w1).flag_bytes) : 0);
  // the accumulated outputs and the split-K flags are cleared first (one launch)
  TRY(zero_launch({{a->db2, a->D * 4}, {a->db1, a->F * 4}, {a->dgamma, a->D * 4}, {a->dbeta, a->D * 4}, flags}, st));
  TRY(cast_launch(a->dy, false, a->M, a->D, bdt, m.scale + 0, m.amax_cur + 0, a->dyq, nullptr, a->db2, st, false));
  // FC2 dgrad with the GELU derivative and the dH cast fused: dH = (dYq . W2q) * s * gelu'(H)
  GemmArgs d2 = gemm_args(a->dyq, 0, bdt, a->w2q, 1, fdt, a->M, a->F, a->D, m.scale_inv + 0, a->sinv_saved + 3);
  d2.epi = EPI_DGELU;
  d2.h_in = a->h;
  d2.out_q = a->dhq;
  d2.q_dtype = bdt;
  d2.scale_q = m.scale + 1;
  d2.amax_q = m.amax_cur + 1;
  d2.colsum = a->db1;
  d2.dbg = a->dh_debug;
  if (paired) {
    TRY(gemm_pair_launch(d2, w2, st));
  } else {
    TRY(gemm_launch(d2, st));
    TRY(wgrad(w2, a->dw2, st));
  }
  if (paired) {
    TRY(gemm_pair_launch(d1, w1, st));
  } else {
    TRY(gemm_launch(d1, st));
    TRY(wgrad(w1, a->dw1, st));
  }
  // the state update rides in extra CTAs of the LayerNorm backward, the last kernel
  const UpdateJob job = update_job(&m, mask_all(m.n, bdt), a->recipe.margin);
  bool updated = false;
  TRY(ln_bwd_launch(a->dln, a->x, a->gamma, a->mu, a->rsigma, a->M, a->D, a->dx, a->dgamma, a->dbeta, st, false,
                    a->defer_update ? nullptr : &job, &updated));
  return updated ? LNFP8_OK : finish_state(&m, &a->recipe, bdt, nullptr, a->defer_update, st);
}

}  // extern "C"
