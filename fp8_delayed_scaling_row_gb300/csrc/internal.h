// Internal launchers of liblnfp8 (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>
#include <utility>

#include "lnfp8.h"

namespace lnfp8 {

lnfp8_status validate_meta(const lnfp8_meta* m, int expect_n, const char* who);
lnfp8_status meta_init_launch(const lnfp8_meta* m, cudaStream_t st);
// one state-update launch for up to kMaxUpdateSets tensor sets (each validated by the caller)
constexpr int kMaxUpdateSets = 128;  // the table travels as a ~7.7 KB kernel parameter
lnfp8_status update_many_launch(const lnfp8_meta* const* metas, const uint64_t* e5m2_masks, float* const* sinv_before,
                                int count, int margin, cudaStream_t st);
lnfp8_status update_launch(const lnfp8_meta* m, uint64_t e5m2_mask, int margin, float* sinv_before,
                           cudaStream_t st);

// One tensor set's state update carried by `n` extra CTAs at the front of the
// grid of a call's last kernel (n = 0: none). Those CTAs start after every
// earlier kernel of the stream has finished, so the amaxes are final and no
// later kernel of the call reads the scales they write.
struct UpdateJob {
  float* scale;
  float* scale_inv;
  float* hist;
  float* cur;
  uint64_t e5m2_mask;
  int n, L, margin;
};
UpdateJob update_job(const lnfp8_meta* m, uint64_t e5m2_mask, int margin);

// Whether a bf16 cast of this shape (no transposed copy) takes the row-streaming
// form, which reaches a larger share of HBM on large tensors.
bool cast_streams_rows(int64_t rows, int64_t cols);
lnfp8_status cast_launch(const void* in, bool in_fp32, int64_t rows, int64_t cols, int dtype,
                         const float* scale, float* amax_cur, uint8_t* out, uint8_t* out_t,
                         float* colsum, cudaStream_t st, bool clear_colsum = true);

// Zeroes each (pointer, bytes) span (bytes a multiple of 4; NULL or 0 skipped), one launch.
lnfp8_status zero_launch(std::initializer_list<std::pair<void*, int64_t>> spans, cudaStream_t st);

// Up to two bf16 weight tensors cast to FP8 (the forward dtype) inside the
// LayerNorm forward launch: tensor k is [rows[k], cols[k]] row-major with cols a
// multiple of 8; tiles[k] = 0 skips it. `zero` (optional) names words that
// the launch clears (counters that a later kernel of the call uses). The
// forward calls put a weight here when it is small enough that its own launch
// would be latency-bound (below the row-streaming cast's size); a larger one
// gets its own row-streaming cast launch.
struct WeightCastJob {
  const uint16_t* in[2];
  int64_t rows[2], cols[2];
  const float* scale[2];
  float* amax[2];
  uint8_t* out[2];
  int64_t tiles[2];
  uint32_t* zero;
  int64_t zero_n;
};
// Adds tensor k to the job (rows or cols 0: nothing to cast).
void weight_cast_add(WeightCastJob& j, int k, const uint16_t* in, int64_t rows, int64_t cols, const float* scale,
                     float* amax, uint8_t* out);

// The scale_inv a forward casts with, saved by its first kernel for the rest of
// the call and the backward: dst[k] = *src[k] for k < n (n <= 4; a slot whose
// weight is stored in FP8 takes that weight's own scale_inv).
struct SinvSnapshot {
  float* dst;
  const float* src[4];
  int n;
};

lnfp8_status ln_fwd_launch(const uint16_t* x, const uint16_t* gamma, const uint16_t* beta, float eps,
                           int64_t M, int64_t D, int dtype, const float* scale, float* amax_cur,
                           uint8_t* out, float* mu, float* rsigma, float* ydbg, cudaStream_t st,
                           const uint16_t* resid = nullptr, uint16_t* hsum = nullptr,
                           const WeightCastJob* wc = nullptr, const SinvSnapshot* snap = nullptr);
lnfp8_status ln_bwd_launch(const uint16_t* dy, const uint16_t* x, const uint16_t* gamma, const float* mu,
                           const float* rsigma, int64_t M, int64_t D, uint16_t* dx, float* dgamma,
                           float* dbeta, cudaStream_t st, bool clear = true,
                           const UpdateJob* job = nullptr, bool* job_done = nullptr);

// Epilogues of the FP8 GEMM.
enum GemmEpilogue {
  EPI_STORE = 0,  // out = acc * sinv_a * sinv_b (+ bias) -> bf16
  EPI_GELU = 1,   // h = bf16(acc * s + bias) -> out; a = gelu(h) -> fp8(a * scale_q) + amax
  EPI_DGELU = 2,  // dh = acc * s * gelu'(h_in) -> fp8(dh * scale_q) + amax + column sums
};

struct GemmArgs {
  // operands: layout 0 = [rows, K] K-contiguous, 1 = [K, rows] rows-contiguous
  const uint8_t* a;
  int a_layout, a_dtype;
  const uint8_t* b;
  int b_layout, b_dtype;
  int64_t M, N, K;
  const float* sinv_a;
  const float* sinv_b;
  int epi;
  const uint16_t* bias;  // [N] bf16 or NULL
  uint16_t* out;         // [M, N] bf16 (STORE, GELU)
  // GELU / DGELU
  const uint16_t* h_in;  // [M, N] bf16 (DGELU)
  uint8_t* out_q;        // [M, N] codes
  int q_dtype;
  const float* scale_q;
  float* amax_q;
  float* colsum;         // [N] fp32 (DGELU), accumulated: the caller clears it
  float* dbg;            // optional [M, N] fp32 pre-cast value
  // optional split-K workspace (bf16-store epilogue): a flag area of
  // ws_flag_bytes (0: the plan's own flag_bytes; a multiple of 256 at least
  // that large), which must be zero at launch and is left zero, then the
  // partial-product slots
  void* ws = nullptr;
  int64_t ws_bytes = 0;
  int64_t ws_flag_bytes = 0;
  // optional: a state update the launch carries in an extra cluster (upd.n = 0: none); the
  // GEMM itself must read none of the state it writes
  UpdateJob upd = {};
};

struct GemmPlan {
  int bn;             // tile width (256: 2-SM pair tiles; 128: single-SM)
  int splits;         // K pieces per tile
  int kb_per_split;   // K blocks of 128 per piece
  int64_t flag_bytes; // flag words this GEMM needs at the start of the workspace
  int64_t slot_bytes; // partial-product slots after the flag area
  int64_t ws_bytes;   // flag_bytes + slot_bytes (0 without a split)
};
// kmajor: both operands K-major (the only layout the 192-wide tiles are built for)
GemmPlan gemm_plan(int64_t M, int64_t N, int64_t K, int epi, bool may_split, bool kmajor = false);

// One persistent launch of the FC2 data gradient with the dGELU epilogue (g0:
// A [M, K] K-major, B [K, N]) and a bf16-store GEMM (g1, both operands
// [K, rows]): the second GEMM's MMAs fill the first one's epilogue time.
// g1.ws (with g1.ws_flag_bytes) is its split-K exchange area; pair_plan gives
// the sizes it needs.
lnfp8_status gemm_pair_launch(const GemmArgs& g0, const GemmArgs& g1, cudaStream_t st);
GemmPlan pair_plan(const GemmArgs& g1);

lnfp8_status gemm_launch(const GemmArgs& g, cudaStream_t st);

// The LayerNormLinear / Linear forward of few tokens as one launch (K6,
// gemm_small.cuh): LayerNorm (gamma non-NULL) or plain cast of x, the weight
// cast (or FP8-stored codes wq_in), the GEMM, dequantisation and bias. Results
// equal the separate launches' bit for bit; the state update is not included.
struct SmallLinearArgs {
  int64_t M, N, K;
  const uint16_t* x;
  const uint16_t* gamma;
  const uint16_t* beta;
  float eps;
  const uint16_t* w;
  const uint8_t* wq_in;
  const uint16_t* bias;
  uint16_t* y;
  uint8_t* xq;
  uint8_t* wq;
  float* mu;
  float* rsigma;
  float* ydbg;
  const float* scale;
  const float* scale_inv;
  const float* w_scale_inv;
  float* amax_cur;
};
bool ln_linear_small_fits(int64_t M, int64_t K, int64_t N);
lnfp8_status ln_linear_small_launch(const SmallLinearArgs& a, int dtype, cudaStream_t st);
lnfp8_status selftest_timeout_launch(int64_t limit_ns, cudaStream_t st);

}  // namespace lnfp8
