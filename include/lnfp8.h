/*
 * lnfp8.h - C ABI of the GB300 (sm_103a) FP8 delayed-scaling LayerNormLinear /
 * LayerNormMLP library (liblnfp8.so).
 *
 * What the library computes (sources cited by page title and section):
 *   - "Accelerating Transformer Training with NVIDIA Transformer Engine, Fused
 *     Kernels, BF16, FP8, and GPU Benchmarking" (the TE tutorial), code blocks
 *     1-5: te.LayerNormLinear(H, 3H), te.LayerNormMLP(H, 4H), te.Linear, the
 *     DelayedScaling(HYBRID, amax_history_len=16, amax_compute_algo="max")
 *     recipe, fp8_autocast around forward/backward, and the fp8_meta state
 *     (scale, amax_history with row 0 the most recent).
 *   - "Turbo-charging your transformer training: a hands-on guide" (the
 *     Turbo-charging guide), sections "The building blocks: fused modules
 *     you'll use" and "Playing with lower-precision formats: BF16 vs FP8":
 *     LayerNormMLP = layer-norm, two linear layers, GELU; delayed scaling
 *     tracks each tensor's amax and rescales it; HYBRID mixes E4M3 and E5M2;
 *     gradients come back in BF16/FP32.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates no memory and keeps no per-call state between calls. Host
 *     pointers are named as such.
 *   - Row-major layout. bf16 tensors are passed as uint16_t bit patterns, FP8
 *     tensors as uint8_t codes (OCP E4M3 "fn" or E5M2), state as fp32.
 *     Weights are [out_features, in_features] (the nn.Linear layout).
 *   - Every tensor pointer must be 16-byte aligned. Feature sizes (K, N, D, F)
 *     must be multiples of 16; the token count M may be any value >= 0.
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and runs
 *     asynchronously. Argument errors are detected before anything is
 *     enqueued and returned synchronously. Asynchronous CUDA errors are
 *     returned by the call that observes them. A device-side wait that gives
 *     up (bounded, about a second) sets a sticky device status word that
 *     lnfp8_sync_status() returns as LNFP8_ERR_TIMEOUT.
 *   - No entry point aborts or throws; lnfp8_last_error() gives a message for
 *     the last failing call on the calling thread.
 */
#ifndef LNFP8_H
#define LNFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* lnfp8_stream; /* a cudaStream_t */

typedef enum {
  LNFP8_OK = 0,
  LNFP8_ERR_INVALID_ARG = 1,       /* null / misaligned pointer, bad enum, negative size */
  LNFP8_ERR_UNSUPPORTED_SHAPE = 2, /* a feature size that is not a multiple of 16, or too large */
  LNFP8_ERR_CUDA = 3,              /* a CUDA runtime error (launch or asynchronous) */
  LNFP8_ERR_TIMEOUT = 4,           /* a bounded device-side wait gave up */
  LNFP8_ERR_UNSUPPORTED = 5        /* a mode the library does not implement */
} lnfp8_status;

/* FP8 element formats (OCP 8-bit floating point): E4M3 max 448, no Inf;
 * E5M2 max 57344. Casts round to nearest even and saturate to +-max. */
typedef enum { LNFP8_E4M3 = 0, LNFP8_E5M2 = 1 } lnfp8_dtype;

/* Recipe formats (TE tutorial code block 1 / code block 5 "Format.E4M3 vs
 * HYBRID"; Turbo-charging guide "Common pitfalls": Format.E5M2).
 * HYBRID: E4M3 for forward tensors, E5M2 for gradients. */
typedef enum { LNFP8_FORMAT_E4M3 = 0, LNFP8_FORMAT_HYBRID = 1, LNFP8_FORMAT_E5M2 = 2 } lnfp8_format;

/* DelayedScaling(fp8_format, amax_history_len, amax_compute_algo) of the TE
 * tutorial, code block 1. algo 0 = "max", the only algorithm the pages name.
 * margin >= 0 divides the scale by 2^margin (0 in every workload). */
typedef struct {
  int format;      /* lnfp8_format */
  int history_len; /* >= 1 */
  int algo;        /* 0 = max */
  int margin;      /* >= 0 */
} lnfp8_recipe;

/* The delayed-scaling state of n FP8 tensors (one fp8_meta direction, e.g.
 * "scaling_fwd" in the TE tutorial, code block 4). All device pointers.
 *   scale[n], scale_inv[n]     current cast scale and its fp32 reciprocal
 *   amax_history[history_len*n] row-major [history_len][n], row 0 = newest
 *   amax_cur[n]                running max |x| of the step in progress
 * Cast of tensor i: code = fp8(x * scale[i]); amax_cur[i] = max(amax_cur[i], max|x|).
 * Slot order: LayerNormLinear fwd {0 input, 1 weight}, bwd {0 dY};
 *             LayerNormMLP    fwd {0 LN output, 1 W1, 2 GELU output, 3 W2},
 *                             bwd {0 dY, 1 dH}. */
typedef struct {
  float* scale;
  float* scale_inv;
  float* amax_history;
  float* amax_cur;
  int n;           /* 1..64 */
  int history_len; /* >= 1, equal to the recipe's */
} lnfp8_meta;

/* Status and diagnostics ------------------------------------------------- */

/* Message for the last failing call on this thread ("" if none). */
const char* lnfp8_last_error(void);

/* Synchronises `stream`, then reads and clears the sticky device status word.
 * Returns LNFP8_ERR_TIMEOUT if a bounded device wait gave up since the last
 * call, LNFP8_ERR_CUDA on an asynchronous CUDA error, else LNFP8_OK. */
lnfp8_status lnfp8_sync_status(lnfp8_stream stream);

/* Library version, as major*10000 + minor*100 + patch (400: the saved-context
 * layout queries lnfp8_ctx_bytes / lnfp8_ctx_offsets). */
int lnfp8_version(void);

/* Diagnostic of the failure path: enqueues one kernel whose bounded mbarrier
 * wait can never complete (nothing arrives on it). After limit_ns (1e3..1e9)
 * it gives up, sets the sticky status word and exits cleanly, so the next
 * lnfp8_sync_status() returns LNFP8_ERR_TIMEOUT and the context stays usable.
 * The pipeline waits of the GEMM use the same bounded wait (limit 1 s). */
lnfp8_status lnfp8_selftest_timeout(int64_t limit_ns, lnfp8_stream stream);

/* Launch accounting and per-kernel timing ------------------------------- */

/* Number of kernels this library has launched in this process. */
long long lnfp8_launch_count(void);

/* Switches per-kernel timing on (1) or off (0) and discards earlier records
 * and totals. While on, every kernel launch is bracketed by two CUDA events
 * recorded on the launch's own stream (host-side cost only; no device
 * memory). Inside a stream capture the two records become event nodes of the
 * graph, so each replay of the graph re-records them. */
lnfp8_status lnfp8_profile_enable(int on);

/* For a captured graph: waits for the open records, adds their times to the
 * totals and keeps the records, so that it can be called after every replay. */
lnfp8_status lnfp8_profile_sample(void);

/* Waits for the open records that no sample has counted yet, adds them to the
 * totals, releases all records and returns the number of kernel kinds in the
 * totals (which accumulate until the next lnfp8_profile_enable). */
int lnfp8_profile_collect(void);

/* Kind i (0 <= i < the count lnfp8_profile_collect returned): its name (owned
 * by the library, valid until the next collect), total milliseconds and
 * number of launches. */
lnfp8_status lnfp8_profile_get(int i, const char** kind, double* total_ms, long long* launches);

/* Delayed-scaling state -------------------------------------------------- */

/* Initial state (TE tutorial code block 1 recipe; step 1 casts with scale 1):
 * scale = scale_inv = 1, amax_history = 0, amax_cur = 0. */
lnfp8_status lnfp8_meta_init(const lnfp8_meta* meta, lnfp8_stream stream);

/* End-of-step update of every slot of `meta` (Turbo-charging guide, "Playing
 * with lower-precision formats": the scale comes from the tracked amax history):
 *   1. history rows move down one (row j <- row j-1), row 0 <- amax_cur;
 *   2. amax_cur <- 0;
 *   3. a = max over the history_len rows (NaN > Inf > finite);
 *   4. if a is finite and > 0 and s = fp8_max(dtype[i]) / a / 2^margin is finite:
 *      scale = s, scale_inv = 1/s (IEEE fp32 division); otherwise both are kept.
 * dtype_per_tensor: HOST array [n] of lnfp8_dtype giving fp8_max per slot
 *                   (448 for E4M3, 57344 for E5M2).
 * scale_inv_before: optional device [n]; receives scale_inv as it was before
 *                   this update (the snapshot a backward needs). May be NULL. */
lnfp8_status amax_history_update(const lnfp8_meta* meta, const lnfp8_recipe* recipe,
                                 const int* dtype_per_tensor, float* scale_inv_before,
                                 lnfp8_stream stream);

/* The same update for `count` tensor sets (0..128; e.g. every layer of a model
 * after the step, its module calls having run with defer_update) in ONE kernel
 * launch. metas: HOST array [count]; dtypes: HOST array, the sets' per-slot
 * lnfp8_dtype values one after another (sum of the n's entries);
 * scale_inv_before: HOST array [count] of optional device pointers (each [n] or
 * NULL), or NULL. The sets must not share state (a set listed twice, or two
 * sets whose amax_cur ranges overlap, is refused with LNFP8_ERR_INVALID_ARG).
 * The results equal count separate amax_history_update calls bit for bit. */
lnfp8_status amax_history_update_many(const lnfp8_meta* metas, int count, const lnfp8_recipe* recipe,
                                      const int* dtypes, float* const* scale_inv_before,
                                      lnfp8_stream stream);

/* Scaled cast (K2) --------------------------------------------------------- */

/* code = fp8(x * (*scale)), round to nearest even, saturating; *amax_cur =
 * max(*amax_cur, max|x|) (Turbo-charging guide, "Playing with lower-precision
 * formats": amax of each tensor, rescale before the cast).
 *   in        [rows, cols] bf16 (in_is_fp32 = 0) or fp32 (in_is_fp32 = 1)
 *   dtype     lnfp8_dtype of the output codes
 *   scale     device fp32 scalar; amax_cur device fp32 scalar (max-accumulated)
 *   out       [rows, cols] codes, or NULL
 *   out_t     [cols, rows] codes (the transpose), or NULL
 *   colsum    [cols] fp32, or NULL: receives sum over rows of x (overwritten)
 * cols must be a multiple of 16; rows >= 0. */
lnfp8_status fp8_quantize(const void* in, int in_is_fp32, int64_t rows, int64_t cols, int dtype,
                          const float* scale, float* amax_cur, uint8_t* out, uint8_t* out_t,
                          float* colsum, lnfp8_stream stream);

/* One-time conversion of a weight to FP8 storage (TE tutorial closing list:
 * fp8_model_init stores the weights themselves in FP8). Three kernels on
 * `stream`, all on the device:
 *   1. amax_cur[0] = max(amax_cur[0], max|w|);
 *   2. the state update of `meta` (amax_history_update with dtype) - with a
 *      freshly initialised meta of any history length this gives
 *      scale = fp8_max / max|w| / 2^margin (kept at its old value when the
 *      weight is all zeros or not finite);
 *   3. codes = fp8(w * scale[0]) (round to nearest even, saturating), and the
 *      cast's own amax of w is recorded into amax_cur[0] again.
 * meta: n = 1, the weight's own state (any history length; the recipe gives
 * only the margin); afterwards meta->scale_inv[0] is the codes' scale_inv
 * (pass it as the forward's w_scale_inv). dtype: lnfp8_dtype of the codes (the
 * forward format of the recipe the forward will run with).
 * w [rows, cols] bf16; codes [rows, cols]; cols a multiple of 16. */
lnfp8_status fp8_weight_quantize(const uint16_t* w, int64_t rows, int64_t cols, const lnfp8_meta* meta,
                                 const lnfp8_recipe* recipe, int dtype, uint8_t* codes, lnfp8_stream stream);

/* LayerNorm + amax + cast (K1) and LayerNorm backward (K5) --------------- */

/* Per row of x [M, D] bf16: mu = mean, var = biased variance,
 * rsigma = 1/sqrt(var + eps), y = (x - mu) * rsigma * gamma + beta (fp32);
 * *amax_cur = max(*amax_cur, max|y|); out = fp8(y * (*scale)).
 * gamma, beta: [D] bf16. mu, rsigma: [M] fp32 outputs. y_debug: optional
 * [M, D] fp32 copy of y (for verification), may be NULL. */
lnfp8_status ln_fwd_cast(const uint16_t* x, const uint16_t* gamma, const uint16_t* beta, float eps,
                         int64_t M, int64_t D, int dtype, const float* scale, float* amax_cur,
                         uint8_t* out, float* mu, float* rsigma, float* y_debug, lnfp8_stream stream);

/* Gradient of the LayerNorm above: with xhat = (x - mu) * rsigma, g = dy * gamma:
 * dx = rsigma * (g - mean(g) - xhat * mean(g * xhat)) (bf16 [M, D]);
 * dgamma = sum_rows dy * xhat, dbeta = sum_rows dy (fp32 [D], overwritten). */
lnfp8_status ln_bwd(const uint16_t* dy, const uint16_t* x, const uint16_t* gamma, const float* mu,
                    const float* rsigma, int64_t M, int64_t D, uint16_t* dx, float* dgamma,
                    float* dbeta, lnfp8_stream stream);

/* FP8 tensor-core GEMM (K3) ----------------------------------------------- */

/* out[M, N] (bf16) = (sum_k A[m, k] * B[n, k]) * (*sinv_a * *sinv_b) + bias[n]
 * with fp32 accumulation on the tcgen05 tensor cores (TE tutorial, code block 1
 * prose: FP8 tensor cores).
 *   a_layout 0: A stored [M, K] (K contiguous); 1: A stored [K, M].
 *   b_layout 0: B stored [N, K] (K contiguous); 1: B stored [K, N].
 *   a_dtype, b_dtype: lnfp8_dtype. bias: [N] bf16 or NULL.
 * N and K must be multiples of 16, and M too when a_layout = 1.
 * workspace: optional device buffer of workspace_bytes (16-byte aligned), or
 * NULL. When it holds at least lnfp8_gemm_workspace_size(M, N, K) bytes and
 * that size is not 0, the GEMM cuts K into pieces that run on separate SMs
 * (split K) and adds the pieces' fp32 partial products in a fixed order, so
 * the result is deterministic. The library zeroes the part it needs at the
 * start of the call; the buffer is the caller's and must not be used by
 * anything else until the call has completed on the stream. */
lnfp8_status fp8_gemm(const uint8_t* A, int a_layout, int a_dtype, const uint8_t* B, int b_layout,
                      int b_dtype, int64_t M, int64_t N, int64_t K, const float* sinv_a,
                      const float* sinv_b, const uint16_t* bias, uint16_t* out, void* workspace,
                      int64_t workspace_bytes, lnfp8_stream stream);

/* Bytes of workspace with which fp8_gemm would split K for this shape on the
 * current device; 0 when it would not split (then no workspace is used), -1
 * for negative sizes. */
int64_t lnfp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/* LayerNormLinear / Linear ---------------------------------------------- */

typedef struct {
  int64_t M, K, N;        /* tokens, in_features, out_features */
  const uint16_t* x;      /* [M, K] bf16 */
  const uint16_t* gamma;  /* [K] bf16, or NULL: no LayerNorm (te.Linear) */
  const uint16_t* beta;   /* [K] bf16 (required with gamma) */
  float eps;              /* LayerNorm eps (1e-5) */
  const uint16_t* w;      /* [N, K] bf16 */
  const uint16_t* bias;   /* [N] bf16 or NULL */
  uint16_t* y;            /* out [M, N] bf16 */
  /* saved for the backward (caller-owned) */
  uint8_t* xq;            /* [M, K] codes of the LN output (of x without LN) */
  uint8_t* wq;            /* [N, K] codes of w */
  float* mu;              /* [M] (with gamma) */
  float* rsigma;          /* [M] (with gamma) */
  float* sinv_saved;      /* [2] scale_inv of (input, weight) this forward cast with */
  lnfp8_meta meta;        /* forward state, n = 2 */
  lnfp8_recipe recipe;
  int defer_update;       /* 1: accumulate amax_cur only; the caller runs amax_history_update */
  float* ln_out_debug;    /* optional [M, K] fp32 pre-cast input, may be NULL */
  /* FP8-stored weight (fp8_model_init): NULL, or device [1] scale_inv of a
   * weight kept as codes. When set, wq is an INPUT (the weight's [N, K] codes
   * in the recipe's forward format, read only), w is ignored and may be NULL,
   * the forward casts no weight and records no weight amax, the GEMM uses
   * w_scale_inv[0] for the weight and sinv_saved[1] receives it. */
  const float* w_scale_inv;
  /* Residual add fused ahead of the LayerNorm (requires gamma): NULL, or [M, K]
   * bf16 r; then the module's input is h = bf16(x + r) (fp32 add, round to
   * nearest even), which the call writes to x_sum ([M, K] bf16, required with
   * residual) and normalises. The backward takes x_sum as its x. */
  const uint16_t* residual;
  uint16_t* x_sum;
  /* How the forward runs (results are the same bit for bit):
   *   LNFP8_PATH_AUTO      the library's choice (the fused launch for few tokens)
   *   LNFP8_PATH_FUSED     one launch computing the LayerNorm (or the input cast),
   *                        the weight cast, the GEMM and the bias into its output
   *                        tiles, the LayerNorm / cast fused into the GEMM's
   *                        A-operand producer; then the state update. Needs
   *                        M >= 1, K <= 768 and no residual, else
   *                        LNFP8_ERR_UNSUPPORTED_SHAPE.
   *   LNFP8_PATH_SEPARATE  the LayerNorm + cast (which also casts a small
   *                        weight; a large one gets a launch of its own), then
   *                        the GEMM, whose launch also runs the state update.
   *                        Without the LayerNorm: the input cast, the weight
   *                        cast, the GEMM and the state update as launches of
   *                        their own. */
  int path;
} lnfp8_ln_linear_fwd_args;

enum { LNFP8_PATH_AUTO = 0, LNFP8_PATH_FUSED = 1, LNFP8_PATH_SEPARATE = 2 };

typedef struct {
  int64_t M, K, N;
  const uint16_t* dy;         /* [M, N] bf16 upstream gradient */
  const uint16_t* x;          /* [M, K] bf16 forward input */
  const uint16_t* gamma;      /* as in the forward (NULL: no LayerNorm) */
  const uint8_t* xq;          /* saved by the forward */
  const uint8_t* wq;
  const float* mu;
  const float* rsigma;
  const float* sinv_saved;    /* [2] */
  uint16_t* dx;               /* out [M, K] bf16 */
  uint16_t* dw;               /* out [N, K] bf16 */
  float* dbias;               /* out [N] fp32, or NULL */
  float* dgamma;              /* out [K] fp32 (with gamma) */
  float* dbeta;               /* out [K] fp32 (with gamma) */
  uint8_t* dyq;               /* workspace [M, N] codes of dY */
  uint16_t* dln;              /* workspace [M, K] bf16 (with gamma) */
  lnfp8_meta meta;            /* backward state, n = 1 */
  lnfp8_recipe recipe;
  int defer_update;
  void* gemm_ws;              /* optional split-K workspace (see lnfp8_ln_linear_bwd_workspace_size), or NULL */
  int64_t gemm_ws_bytes;
} lnfp8_ln_linear_bwd_args;

/* LayerNormLinear forward (TE tutorial code block 1: te.LayerNormLinear(H, 3H);
 * te.Linear when gamma is NULL):
 *   y = LN(x); xq = fp8(y * scale[0]); wq = fp8(w * scale[1]);
 *   out = (xq . wq^T) * (scale_inv[0] * scale_inv[1]) + bias  (bf16);
 * then the forward state update unless defer_update. With w_scale_inv set
 * (weights stored in FP8, TE tutorial closing list: fp8_model_init), wq is the
 * given codes and w_scale_inv[0] takes the place of scale_inv[1]. With
 * residual set, x is first replaced by h = bf16(x + residual) (the residual
 * connection ahead of the block's LayerNorm, TE tutorial code block 2), fused
 * into the LayerNorm kernel and written to x_sum. */
lnfp8_status ln_linear_fwd(const lnfp8_ln_linear_fwd_args* args, lnfp8_stream stream);

/* LayerNormLinear backward (TE tutorial, code block 3: loss.backward() through
 * the modules under fp8_autocast; Turbo-charging guide, "Playing with
 * lower-precision formats: BF16 vs FP8": gradients go back to BF16/FP32 for
 * the optimizer): dyq = fp8(dy * gscale[0]) (E5M2 under HYBRID);
 * dbias = sum_rows dy; dln = (dyq . wq) * (gscale_inv[0] * sinv_saved[1]);
 * dw = (dyq^T . xq) * (gscale_inv[0] * sinv_saved[0]); dx = LN backward of dln
 * (dx = dln without LayerNorm); then the backward state update. */
lnfp8_status ln_linear_bwd(const lnfp8_ln_linear_bwd_args* args, lnfp8_stream stream);

/* Bytes of args->gemm_ws with which ln_linear_bwd splits K in its GEMMs
 * (the dgrad [M, K] and the wgrad [N, K] over M tokens); 0 when neither
 * would split, -1 for negative sizes. A smaller or NULL workspace is valid
 * and runs the GEMMs unsplit. The library zeroes what it uses at the start
 * of each call; the results are the same with and without it up to fp32
 * summation order. */
int64_t lnfp8_ln_linear_bwd_workspace_size(int64_t M, int64_t K, int64_t N);

/* LayerNormLinear backward without caller-provided scratch. The pages have no
 * counterpart of this entry point. It is for callers that cannot allocate
 * device memory (they may not call cudaMalloc, for example a plug-in that a
 * host framework hands only the tensors of one layer, or a runtime whose
 * device memory is fixed before start-up). It takes the same arguments as
 * ln_linear_bwd; args->dyq and args->dln are ignored. Those two scratch
 * buffers live instead in one fixed device array inside the library, 16 MiB
 * (the dY codes, M*N bytes rounded up to 256, then the bf16 LayerNorm-output
 * gradient, 2*M*K bytes, when gamma is given); every GPU that loads the
 * library holds that array until the process exits. Sizes beyond it return
 * LNFP8_ERR_UNSUPPORTED_SHAPE before anything is enqueued. It allocates
 * nothing and runs the same kernels as ln_linear_bwd.
 *   - The first call on each device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture. A call made under another CUDA context on the same
 *     device than the one of the previous calls looks the address up again
 *     (also before any capture). After cudaDeviceReset the library may still
 *     hold the old address: do not call this entry point again in a process
 *     that has reset the device.
 *   - All calls share the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero (both buffers are fully written
 *     before they are read). Calls whose work overlaps on the GPU (other
 *     streams, or other host threads) race on it: serialise them. */
lnfp8_status ln_linear_bwd_noalloc(const lnfp8_ln_linear_bwd_args* args, lnfp8_stream stream);

/* LayerNormMLP ----------------------------------------------------------- */

typedef struct {
  int64_t M, D, F;        /* tokens, hidden, FFN width */
  const uint16_t* x;      /* [M, D] bf16 */
  const uint16_t* gamma;  /* [D] bf16 */
  const uint16_t* beta;   /* [D] bf16 */
  float eps;
  const uint16_t* w1;     /* [F, D] bf16 */
  const uint16_t* b1;     /* [F] bf16 or NULL */
  const uint16_t* w2;     /* [D, F] bf16 */
  const uint16_t* b2;     /* [D] bf16 or NULL */
  uint16_t* y;            /* out [M, D] bf16 */
  /* saved for the backward (caller-owned) */
  uint8_t* lnq;           /* [M, D] codes of the LN output */
  float* mu;              /* [M] */
  float* rsigma;          /* [M] */
  uint8_t* w1q;           /* [F, D] */
  uint8_t* w2q;           /* [D, F] */
  uint16_t* h;            /* [M, F] bf16 pre-activation */
  uint8_t* aq;            /* [M, F] codes of gelu(h) */
  float* sinv_saved;      /* [4] scale_inv this forward cast with */
  lnfp8_meta meta;        /* forward state, n = 4 */
  lnfp8_recipe recipe;
  int defer_update;
  float* ln_out_debug;    /* optional [M, D] fp32 pre-cast LN output */
  float* act_debug;       /* optional [M, F] fp32 pre-cast GELU output */
  void* gemm_ws;          /* optional, lnfp8_ln_mlp_fwd_workspace_size bytes: FC1 and FC2 run as one launch */
  int64_t gemm_ws_bytes;
  /* FP8-stored weights (fp8_model_init): both NULL, or device [1] scale_inv of
   * W1 and of W2 kept as codes. When set, w1q and w2q are INPUTS (codes in the
   * recipe's forward format, read only), w1 and w2 are ignored and may be NULL,
   * the forward casts no weight and records no weight amax (slots 1 and 3),
   * and sinv_saved[1], sinv_saved[3] receive these values. */
  const float* w1_scale_inv;
  const float* w2_scale_inv;
  /* Residual add fused ahead of the LayerNorm: NULL, or [M, D] bf16 r; then the
   * input is h = bf16(x + r), written to x_sum ([M, D] bf16, required with
   * residual) and normalised; the backward takes x_sum as its x. */
  const uint16_t* residual;
  uint16_t* x_sum;
} lnfp8_ln_mlp_fwd_args;

typedef struct {
  int64_t M, D, F;
  const uint16_t* dy;     /* [M, D] bf16 */
  const uint16_t* x;      /* [M, D] forward input */
  const uint16_t* gamma;
  const uint8_t* lnq;
  const float* mu;
  const float* rsigma;
  const uint8_t* w1q;
  const uint8_t* w2q;
  const uint16_t* h;
  const uint8_t* aq;
  const float* sinv_saved; /* [4] */
  uint16_t* dx;           /* out [M, D] bf16 */
  float* dgamma;          /* out [D] fp32 */
  float* dbeta;           /* out [D] fp32 */
  uint16_t* dw1;          /* out [F, D] bf16 */
  float* db1;             /* out [F] fp32, or NULL */
  uint16_t* dw2;          /* out [D, F] bf16 */
  float* db2;             /* out [D] fp32, or NULL */
  uint8_t* dyq;           /* workspace [M, D] */
  uint8_t* dhq;           /* workspace [M, F] */
  uint16_t* dln;          /* workspace [M, D] bf16 */
  lnfp8_meta meta;        /* backward state, n = 2 */
  lnfp8_recipe recipe;
  int defer_update;
  float* dh_debug;        /* optional [M, F] fp32 pre-cast dH */
  void* gemm_ws;          /* optional split-K workspace (see lnfp8_ln_mlp_bwd_workspace_size), or NULL */
  int64_t gemm_ws_bytes;
} lnfp8_ln_mlp_bwd_args;

/* LayerNormMLP forward (TE tutorial code block 1: te.LayerNormMLP(H, 4H);
 * Turbo-charging guide: layer-norm, two linear layers, GELU):
 *   y = LN(x) -> lnq = fp8(y*scale[0]); w1q = fp8(W1*scale[1]); w2q = fp8(W2*scale[3]);
 *   h = bf16((lnq . w1q^T) * sinv[0]*sinv[1] + b1);
 *   a = gelu_tanh(h) (fp32); aq = fp8(a * scale[2]);
 *   out = bf16((aq . w2q^T) * sinv[2]*sinv[3] + b2); then the state update.
 * With residual set, x is first replaced by h = bf16(x + residual) (fused into
 * the LayerNorm kernel, written to x_sum), as in ln_linear_fwd. */
lnfp8_status ln_mlp_fwd(const lnfp8_ln_mlp_fwd_args* args, lnfp8_stream stream);

/* Bytes of args->gemm_ws with which ln_mlp_fwd runs FC1 (+GELU) and FC2 as one
 * persistent launch: FC2's tiles start as soon as the FC1 tiles of their rows
 * are written, tracked by one counter per 256-row block in the workspace (cleared
 * by the call's first kernel). 0 when M is 0, -1 for negative sizes. With a
 * NULL or smaller workspace the two GEMMs run as separate launches; the
 * results are identical. */
int64_t lnfp8_ln_mlp_fwd_workspace_size(int64_t M, int64_t D, int64_t F);

/* LayerNormMLP backward (TE tutorial, code block 3: loss.backward() through
 * te.LayerNormMLP under fp8_autocast; Turbo-charging guide, "Playing with
 * lower-precision formats: BF16 vs FP8": HYBRID mixes E4M3 and E5M2, so the
 * gradients are cast to E5M2, and they come back in BF16/FP32):
 *   dyq = fp8(dy * gscale[0]); db2 = sum_rows dy;
 *   dh = (dyq . w2q) * gsinv[0]*sinv[3] * gelu'(h) (fp32); dhq = fp8(dh * gscale[1]);
 *   db1 = sum_rows dh; dw2 = (dyq^T . aq) * gsinv[0]*sinv[2];
 *   dln = (dhq . w1q) * gsinv[1]*sinv[1]; dw1 = (dhq^T . lnq) * gsinv[1]*sinv[0];
 *   dx, dgamma, dbeta = LN backward of dln; then the backward state update. */
lnfp8_status ln_mlp_bwd(const lnfp8_ln_mlp_bwd_args* args, lnfp8_stream stream);

/* Bytes of args->gemm_ws with which ln_mlp_bwd splits K in its plain-store
 * GEMMs (dW2 [D, F] and dW1 [F, D] over M tokens, dLN [M, D] over F); 0 when
 * none would split, -1 for negative sizes. As for ln_linear_bwd, a smaller or
 * NULL workspace runs them unsplit. */
int64_t lnfp8_ln_mlp_bwd_workspace_size(int64_t M, int64_t D, int64_t F);

/* The saved context ---------------------------------------------------------
 * What a forward keeps for its backward: the state of the module between
 * `m(x)` and `loss.backward()` (TE tutorial, code blocks 1 and 3: the module
 * call and the backward under fp8_autocast; code block 4: the FP8 codes are
 * cast with the scales kept in fp8_meta). The caller owns it; these queries
 * give one layout for it, so that it can live in a single allocation: the
 * buffers in the order listed, each starting at a multiple of 256 bytes.
 *   LNFP8_OP_LN_LINEAR (in features D, out features F; ln_linear_* with gamma)
 *     0 xq [M, D] u8, 1 wq [F, D] u8, 2 mu [M] f32, 3 rsigma [M] f32,
 *     4 sinv_saved [2] f32
 *   LNFP8_OP_LINEAR (ln_linear_* without LayerNorm)
 *     0 xq [M, D] u8, 1 wq [F, D] u8, 2 sinv_saved [2] f32
 *   LNFP8_OP_LN_MLP (hidden D, FFN width F)
 *     0 lnq [M, D] u8, 1 w1q [F, D] u8, 2 w2q [D, F] u8, 3 h [M, F] bf16,
 *     4 aq [M, F] u8, 5 mu [M] f32, 6 rsigma [M] f32, 7 sinv_saved [4] f32
 * (x, or x_sum after a fused residual add, is the caller's input tensor and
 * is not part of it; nor are the backward's workspaces dyq, dhq, dln.) */
typedef enum { LNFP8_OP_LN_LINEAR = 0, LNFP8_OP_LINEAR = 1, LNFP8_OP_LN_MLP = 2 } lnfp8_op;

/* Total bytes of the saved context of `op` (the end of its last buffer,
 * rounded up to 256);
 * -1 for an unknown op or a negative size. */
int64_t lnfp8_ctx_bytes(int op, int64_t M, int64_t D, int64_t F);

/* Byte offsets of the saved context's buffers: offsets (host array of
 * max_offsets entries) receives the start of each buffer in the order above,
 * then the total. Returns the number of buffers (5, 3 or 8), or -1 for an
 * unknown op, a negative size, a NULL offsets or max_offsets smaller than
 * that number plus one. */
int lnfp8_ctx_offsets(int op, int64_t M, int64_t D, int64_t F, int64_t* offsets, int max_offsets);

#ifdef __cplusplus
}
#endif
#endif /* LNFP8_H */
