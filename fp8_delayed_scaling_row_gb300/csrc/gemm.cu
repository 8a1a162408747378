// K3: FP8 GEMM on the 5th-generation tensor cores (tcgen05, kind::f8f6f4),
// operands staged by TMA, fp32 accumulators in tensor memory, fused epilogues.
//
// The linear layers of LayerNormLinear / LayerNormMLP run on "FP8 tensor
// cores" (TE tutorial, code block 1 prose) with per-tensor scales: the codes
// of both operands are multiplied with fp32 accumulation and the product is
// dequantised by sinv_a * sinv_b (the recorded reciprocals of the two cast
// scales). Three epilogues cover the MLP:
//   EPI_STORE  out = bf16(acc * s + bias)                       (FC2, dgrad, wgrad, Linear)
//   EPI_GELU   h = bf16(acc * s + b1) saved; a = gelu_tanh(h);
//              amax(a); aq = fp8(a * scale_a)                   (FC1 forward)
//   EPI_DGELU  dh = acc * s * gelu_tanh'(h); amax(dh);
//              dhq = fp8(dh * scale_dh); db1 += column sums     (FC2 dgrad)
// so the GELU output and the gradient dH are written only as FP8 codes.
//
// Kernel shape (persistent, one CTA per SM, 640 threads, 96 registers each):
//   warp 0      TMA producer (one elected thread), STAGES-deep smem ring
//   warp 1      tensor-memory allocator (2 x BN fp32 columns: double-buffered
//               accumulator so the epilogue of tile i overlaps the MMAs of
//               i+1), then MMA issuer (one thread): 128 x BN x 32
//               tcgen05.mma per K step
//   warps 2-3   idle (registers are handed out per four warps, so a
//               smaller block would not give the epilogue more of them)
//   warps 4-19  epilogue, two groups of 8: group g drains accumulator buffer g
//               (every other tile), so two tiles' epilogues run at once; warp
//               w reads TMEM lanes 32*(w%4).. (its 32 rows) and one half of
//               the tile's columns with tcgen05.ld
// Operands may be K-major ([rows, K]) or MN-major ([K, rows]); FP8 MN-major
// operands are native to tcgen05, so the backward GEMMs read dY, A, dH and the
// LN output in the layout the forward wrote them, with no transposed copies.
// Split K (bf16-store epilogue only, when the caller provides a workspace):
// a tile's K range is cut into two halves run as separate work units. Each
// half owns half of the tile's 32-column chunks: it writes its raw fp32
// accumulators of the other half's chunks to the workspace and raises a flag,
// waits (bounded) for the other half's flag, and finishes its own chunks as
// part_0 + part_1. The result does not depend on which unit finishes first,
// and both halves share the epilogue work.
// Every mbarrier wait is bounded: on a timeout the CTA records it in the
// library's status word, drains its in-flight copies and MMAs, frees its
// tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "state_update.cuh"

namespace lnfp8 {

__device__ unsigned int g_status = 0;

lnfp8_status status_read_clear(cudaStream_t st, unsigned int* word) {
  *word = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return check_launch("lnfp8_sync_status");
  if (cudaMemcpyFromSymbol(word, g_status, sizeof(unsigned int)) != cudaSuccess)
    return check_launch("lnfp8_sync_status: reading the status word");
  const unsigned int zero = 0;
  if (*word && cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int)) != cudaSuccess)
    return check_launch("lnfp8_sync_status: clearing the status word");
  return LNFP8_OK;
}

namespace {

constexpr int BM = 128;
constexpr int BK = 128;  // bytes (= FP8 elements) of K per pipeline stage
constexpr int kEpiWarps = 16;  // two groups of 8, one per accumulator buffer
// CTAs per cluster: a pair of CTAs works on two M tiles of the same N tile.
// With the 2-SM MMA each CTA loads its own A rows and half of the B tile;
// otherwise each CTA loads its own A rows and the whole B tile. No load
// writes into the peer's shared memory.
constexpr int CL = 2;
constexpr int kThreads = 128 + 32 * kEpiWarps;  // warpgroup 0 (producer, MMA, two idle warps), 16 epilogue warps

template <int BN, bool TWO>
struct Cfg {
  // TWO: 2-SM MMA (cta_group::2): the pair computes a 256 x BN tile and each
  // CTA keeps only its half of the B tile; otherwise each CTA keeps all of B.
  static constexpr int STAGES = TWO ? 5 : (BN == 256 ? 3 : 5);
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = (TWO ? BN / 2 : BN) * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // per epilogue warp: a 32 x 32 bf16 box (2 KB, 64-byte swizzle) and a
  // 32 x 32 FP8 box (1 KB, 32-byte swizzle) staged for TMA stores / loads
  static constexpr int EPI_OUT_OFF = STAGES * STAGE_BYTES;
  static constexpr int EPI_Q_OFF = EPI_OUT_OFF + kEpiWarps * 2048;
  static constexpr int CSUM_OFF = EPI_Q_OFF + kEpiWarps * 1024;
  static constexpr int CSUM_BYTES = 2 * 4 * BN * 4;  // [acc buffer][row quarter][BN] fp32
  static constexpr int BAR_OFF = CSUM_OFF + CSUM_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM = 1024 + BAR_OFF + BAR_BYTES;
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;  // a power of two holding both accumulators
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct KParams {
  int M, N, K;
  int num_m, num_n, num_kb;
  uint32_t idesc;  // instruction descriptor of one MMA
  const float* sinv_a;
  const float* sinv_b;
  const uint16_t* bias;
  uint16_t* out;
  const uint16_t* h_in;
  uint8_t* out_q;
  const float* scale_q;
  float* amax_q;
  float* colsum;
  float* dbg;
  // split K: S (1 or 2) units per tile, kb_per_split K blocks each; ws holds
  // [num_m2 * 2][num_n] tiles of 128 x BN fp32 (the exchanged chunks); flags
  // one word per (piece, tile, epilogue warp of a group), zero at launch
  int splits, kb_per_split;
  float* ws;
  unsigned* flags;
  int group_m;  // M pairs per raster group (see tile_mn)
  // A state update carried by the launch (upd.n > 0): the grid's first cluster runs it
  // (its leader CTA, every slot) while the others compute the GEMM.
  UpdateJob upd;
};

// Output tile t of a [num_m2 x num_n] grid of CTA-pair tiles in grouped raster
// order: M pairs fastest within a group of G pairs, then N, then the next
// group. The clusters in flight at any time then touch about G panels of A
// and ncl / G panels of B, so a G chosen to keep G A-panels in L2 reads A from
// DRAM once and B num_m2 / G times (G = num_m2 is plain M-fastest order).
__device__ __forceinline__ int2 tile_mn(int t, int num_m2, int num_n, int G) {
  const int span = G * num_n;
  const int grp = t / span, r = t - grp * span;
  const int m0 = grp * G;
  const int gs = min(G, num_m2 - m0);
  return make_int2(m0 + r % gs, r / gs);
}

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after ~limit_ns or when another role has aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                       uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(&g_status, kStatusTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 2-SM forms: the load may signal a barrier in the peer CTA; the MMA / commit
// are issued by the pair's leader for both CTAs.
__device__ __forceinline__ void tma_load_2d_cg2(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
// Arrive on a barrier of the pair's leader CTA: an epilogue warp hands an
// accumulator back to the MMA issuer. Its tensor-memory loads have completed
// (tcgen05.wait::ld) and tcgen05.fence::before_thread_sync orders them before
// this arrive; no generic-proxy data is handed over, so the release is
// CTA-scoped. A cluster-scoped release here waits for the warp's earlier
// global traffic to become visible to the peer SM (about 1.5K cycles per tile
// on every epilogue warp, 6% of the d 768 LayerNormMLP step).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Row r of a 32 x 32 box staged for TMA with the 64-byte (bf16) or 32-byte
// (FP8) swizzle: the 16-byte chunk index is XORed with address bits 7..8
// (resp. bit 7) of the row's offset, as the tensor map's swizzle mode expects.
__device__ __forceinline__ uint32_t sw64(int r, int j) { return (uint32_t)(r * 64 + ((j ^ ((r >> 1) & 3)) << 4)); }
__device__ __forceinline__ uint32_t sw32(int r, int j) { return (uint32_t)(r * 32 + ((j ^ ((r >> 2) & 1)) << 4)); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 layout type 2,
// descriptor version 1 in bits 46-47). Both byte offsets are 1024 for
// MN-major tiles (one 128-byte atom wide, 8-row groups 1024 B apart); for
// K-major tiles the stride offset is the 1024 B between 8-row groups and the
// leading offset is unused.
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mma_f8_cg2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit_cg2_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kGeluK = 0.7978845608028654f;  // sqrt(2/pi)
constexpr float kGeluC = 0.044715f;

// Packed fp32 pairs (one 64-bit register pair) and the sm_100+ paired FMA /
// MUL / SUB: two independent IEEE round-to-nearest results per instruction.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float lo(uint64_t r) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
  return a;
}
__device__ __forceinline__ float hi(uint64_t r) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
  return b;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
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
// bf16 pair (low, high halves of a 32-bit word) -> fp32 pair
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// running max of |x| in the fp32 magnitude order, NaN-propagating
__device__ __forceinline__ float maxabs(float m, float x) {
  float r;
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(x));
  return r;
}
template <int DT>
__device__ __forceinline__ uint16_t cvt_pair(uint64_t scaled) {
  return cvt_fp8x2<DT>(lo(scaled), hi(scaled));
}

// Column sums of a 32 x 32 block held one row per lane: after the exchange,
// lane c holds the sum over the 32 rows of column c (31 shuffles).
__device__ __forceinline__ float transpose_reduce32(float* v, int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, w);
    }
  }
  return v[0];
}

// ------------------------------------------------------------ the kernel
template <int BN, bool A_MN, bool B_MN, int EPI, int QDT, bool TWO>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmQ,
            const __grid_constant__ CUtensorMap tmH, const KParams p) {
  using C = Cfg<BN, TWO>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, csum[2 acc][2 halves], hload[kEpiWarps]
  uint32_t* misc = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 9 + kEpiWarps);
  uint32_t* tmem_slot = misc;
  volatile uint32_t* abort_flag = misc + 1;
  float* csred = reinterpret_cast<float*>(smem + C::CSUM_OFF);  // [2][4][BN]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  auto csum_bar = [&](int a, int h) { return bar0 + 8u * (2 * STAGES + 5 + 2 * a + h); };
  auto hload_bar = [&](int w) { return bar0 + 8u * (2 * STAGES + 9 + w); };

  // the first cluster of a launch that carries a state update runs it and leaves: its leader
  // updates every slot (all amaxes it reads were final when the launch started; the GEMM
  // itself reads none of the state it writes)
  const bool has_upd = p.upd.n > 0;
  if (has_upd && (int)blockIdx.x < CL) {
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0) {
      __shared__ uint32_t ured[kThreads / 32];
      run_update_all<kThreads>(p.upd, reinterpret_cast<float*>(smem), ured);
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      // released once: by this CTA's own MMAs (1-SM), or by the pair's leader for both CTAs (2-SM)
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      // the 8 warps of the group that drains buffer a (in both CTAs with the 2-SM MMA)
      mbar_init(tempty_bar(a), (TWO ? 2 : 1) * (kEpiWarps / 2));
    }
    mbar_init(drain_bar, 1);
    for (int a = 0; a < 2; ++a)
      for (int h = 0; h < 2; ++h) mbar_init(csum_bar(a, h), 4);
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(hload_bar(w), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // with the 2-SM MMA the peer's loads and commits signal this CTA's barriers:
  // both CTAs' barriers must be initialised first
  cluster_sync();
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    if constexpr (TWO) {  // one warp of each CTA of the pair allocates collectively
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(C::TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(C::TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // set-up above touches no data; from here on the previous kernel's outputs are read
  pdl_wait();
  pdl_launch_dependents();

  // Work units: one N tile and CL consecutive M tiles, one per CTA of a cluster.
  const int rank = CL == 2 ? (int)cluster_rank() : 0;
  const int cid = blockIdx.x / CL - (has_upd ? 1 : 0), ncl = gridDim.x / CL - (has_upd ? 1 : 0);
  const int num_m2 = (p.num_m + CL - 1) / CL;
  const int S = p.splits;
  const int num_units = num_m2 * p.num_n * S;
  // unit u: tile u / S (grouped raster order), K piece u % S
  auto unit_m = [&](int u) { return tile_mn(u / S, num_m2, p.num_n, p.group_m).x * CL + rank; };
  auto unit_n = [&](int u) { return tile_mn(u / S, num_m2, p.num_n, p.group_m).y; };
  auto unit_kb0 = [&](int u) { return (u % S) * p.kb_per_split; };
  auto unit_kb1 = [&](int u) { return min(p.num_kb, (u % S + 1) * p.kb_per_split); };
  constexpr uint16_t kPair = (1u << CL) - 1u;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int u = cid; u < num_units && ok; u += ncl) {
        const int m_blk = unit_m(u), n_blk = unit_n(u);
        const int kb_end = unit_kb1(u);
        for (int kb = unit_kb0(u); kb < kb_end; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t fb = full_bar(stage);
          const uint32_t a_dst = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_dst = a_dst + C::A_BYTES;
          if constexpr (TWO) {
            // both CTAs load their A rows and their half of B into their own
            // shared memory and signal the leader's barrier, which expects both
            const uint32_t fl = map_to_rank(fb, 0);
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * C::STAGE_BYTES);
            if (!A_MN) tma_load_2d_cg2(a_dst, &tmA, kb * BK, m_blk * BM, fl);
            else       tma_load_2d_cg2(a_dst, &tmA, m_blk * BM, kb * BK, fl);
            if (!B_MN) tma_load_2d_cg2(b_dst, &tmB, kb * BK, n_blk * BN + rank * (BN / 2), fl);
            else       tma_load_2d_cg2(b_dst, &tmB, n_blk * BN + rank * (BN / 2), kb * BK, fl);
          } else {
            mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
            if (!A_MN) tma_load_2d(a_dst, &tmA, kb * BK, m_blk * BM, fb);
            else       tma_load_2d(a_dst, &tmA, m_blk * BM, kb * BK, fb);
            // the whole B tile into this CTA's own ring, as the two half boxes of
            // the B tensor map ([BN/2 rows] K-major; [128 n] x [BK/2 k] MN-major)
#pragma unroll
            for (int h = 0; h < CL; ++h) {
              if (!B_MN)          tma_load_2d(b_dst + h * (BN / CL) * BK, &tmB, kb * BK, n_blk * BN + h * (BN / CL), fb);
              else if (BN == 256) tma_load_2d(b_dst + h * 128 * BK, &tmB, n_blk * BN + h * 128, kb * BK, fb);
              else                tma_load_2d(b_dst + h * (BK / CL) * 128, &tmB, n_blk * BN, kb * BK + h * (BK / CL), fb);
            }
          }
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok && (!TWO || rank == 0)) {
        // drain: wait (bounded) for the copies of the last armed stages to land
        const int64_t pending = issued < STAGES ? issued : STAGES;
        int s = stage;
        uint32_t ph = phase;
        for (int64_t i = 0; i < pending; ++i) {
          if (--s < 0) { s = STAGES - 1; ph ^= 1; }
          uint32_t dummy_flag = 0;
          mbar_wait(full_bar(s), ph, &dummy_flag, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // (with the 2-SM MMA only the pair's leader issues, for both CTAs)
    if (lane == 0 && (!TWO || rank == 0)) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = cid; u < num_units && ok; u += ncl) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int kb_beg = unit_kb0(u), kb_end = unit_kb1(u);
        for (int kb = kb_beg; kb < kb_end; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_base = a_base + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint32_t accum = (kb != kb_beg) || kk != 0;
            const uint64_t ad = A_MN ? make_desc(a_base + kk * 32 * 128, 1024, 1024) : make_desc(a_base + kk * 32, 16, 1024);
            if constexpr (TWO) {
              // 256 x BN x 32 over the pair: A rows and B halves from both CTAs
              const uint64_t bd = B_MN ? make_desc(b_base + kk * 32 * 128, 1024, 1024) : make_desc(b_base + kk * 32, 16, 1024);
              mma_f8_cg2(d_tmem, ad, bd, p.idesc, accum);
            } else if (!B_MN) {
              mma_f8(d_tmem, ad, make_desc(b_base + kk * 32, 16, 1024), p.idesc, accum);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 128; ++j)
                mma_f8(d_tmem + j * 128, ad, make_desc(b_base + j * 128 * BK + kk * 32 * 128, 1024, 1024), p.idesc, accum);
            }
          }
          if constexpr (TWO) mma_commit_cg2_mc(empty_bar(stage), kPair);  // frees the stage in both CTAs
          else mma_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if constexpr (TWO) mma_commit_cg2_mc(tfull_bar(acc), kPair);  // both CTAs' accumulators are ready
        else mma_commit(tfull_bar(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      if (!ok) {
        // make sure no MMA still writes tensor memory before it is freed
        if constexpr (TWO) mma_commit_cg2_mc(drain_bar, 1);
        else mma_commit(drain_bar);
        uint32_t dummy_flag = 0;
        mbar_wait(drain_bar, 0, &dummy_flag, 100000000ull);
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - 4;
    const int grp = ew >> 3;               // accumulator buffer (and tile parity) this warp drains
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. (this warp's 32 rows)
    const int half = (ew >> 2) & 1;        // column half of the tile
    const int r = lane;                    // row within the warp's 32 x 32 box
    constexpr int HALF_COLS = BN / 2;
    constexpr int CHUNKS = HALF_COLS / 32;
    uint8_t* so = smem + C::EPI_OUT_OFF + ew * 2048;  // bf16 box: output (STORE, GELU) or H input (DGELU)
    uint8_t* sq = smem + C::EPI_Q_OFF + ew * 1024;    // FP8 box: codes output (GELU, DGELU)
    const uint32_t so_a = smem_u32(so), sq_a = smem_u32(sq);
    const uint32_t hbar = hload_bar(ew);
    uint32_t hphase = 0;
    bool h_pending = false;
    const float s = __fmul_rn(*p.sinv_a, *p.sinv_b);
    float scale_q = 0.f;
    if constexpr (EPI != EPI_STORE) scale_q = *p.scale_q;
    float am_f = 0.f;  // running max |x| of the cast values (GELU / dGELU epilogues)
    const int acc = grp;
    uint32_t acc_phase = 0;
    // With column sums, warp quarter 0 of each half combines the four 32-row
    // partials of the tile; it releases the accumulator only after reading
    // them, which keeps the partial buffer of this parity from being reused early.
    const bool combiner = EPI == EPI_DGELU && p.colsum != nullptr && quarter == 0;
    auto issue_h = [&](int u, int ch) {
      // prefetch the 32 x 32 block of H this warp needs for (unit, chunk)
      const int m_blk = unit_m(u), n_blk = unit_n(u);
      if (lane == 0) {
        mbar_arrive_expect_tx(hbar, 2048);
        tma_load_2d(so_a, &tmH, n_blk * BN + half * HALF_COLS + ch * 32, m_blk * BM + quarter * 32, hbar);
      }
      h_pending = true;
    };
    // the accumulator is released to the CTA whose MMA reuses it (the leader with the 2-SM MMA)
    const uint32_t tempty_target = TWO ? map_to_rank(tempty_bar(acc), 0) : tempty_bar(acc);
    auto release_acc = [&]() {
      if constexpr (TWO) mbar_arrive_remote(tempty_target);
      else mbar_arrive(tempty_target);
    };
    const int u0 = cid + grp * ncl;  // this group's first unit; then every second one
    if constexpr (EPI == EPI_DGELU) {
      if (u0 < num_units) issue_h(u0, 0);
    }
    // Split K (two pieces): piece q of a tile owns the chunks ch with ch % 2 == q.
    // Each piece spills the chunks the other owns to the workspace and raises
    // its flag, then waits for the other's flag and finishes its own chunks as
    // part_0 + part_1. A chunk is one warp's 32 x 32 fp32 block, stored
    // lane-contiguous (coalesced); each (tile, chunk) is written once.
    const int gw = ew & 7;  // warp within its group
    auto slot_ptr = [&](int m_blk, int n_blk, int ch) {
      const int64_t t = (int64_t)m_blk * p.num_n + n_blk;
      return reinterpret_cast<uint4*>(p.ws + t * (int64_t)(BM * BN)) + ((gw * CHUNKS + ch) * 8) * 32 + lane;
    };
    // flag of the piece q's spill of this warp's chunks of a tile
    auto flag_ptr = [&](int q, int m_blk, int n_blk) {
      return p.flags + (((int64_t)q * (num_m2 * CL) + m_blk) * p.num_n + n_blk) * 8 + gw;
    };
    for (int u = u0; u < num_units; u += 2 * ncl) {
      const int m_blk = unit_m(u), n_blk = unit_n(u);
      const int sp = u % S;
      // this warp's half of the tile's bias, 4 columns per lane, requested before the
      // accumulator wait so that its latency is hidden; chunks take it by shuffles
      uint2 btile = make_uint2(0u, 0u);
      if constexpr (EPI != EPI_DGELU) {
        const int64_t c = (int64_t)n_blk * BN + half * HALF_COLS + lane * 4;
        if (p.bias && lane * 4 < HALF_COLS && c < p.N) btile = __ldg(reinterpret_cast<const uint2*>(p.bias + c));
      }
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) break;
      tc_fence_after();
      const int64_t m = (int64_t)m_blk * BM + quarter * 32 + r;
      const bool row_ok = m < p.M;
      bool aborted = false;
      if constexpr (EPI == EPI_STORE) {
        if (S > 1) {
#pragma unroll 1
          for (int ch = 1 - sp; ch < CHUNKS; ch += 2) {
            uint32_t rr[32];
            tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + half * HALF_COLS + ch * 32), rr);
            uint4* dst = slot_ptr(m_blk, n_blk, ch);
#pragma unroll
            for (int j = 0; j < 8; ++j) __stcg(dst + j * 32, make_uint4(rr[4 * j], rr[4 * j + 1], rr[4 * j + 2], rr[4 * j + 3]));
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) atomicExch(flag_ptr(sp, m_blk, n_blk), 1u);
          // wait (lane 0, bounded) for the other piece's spill of this warp's chunks
          const unsigned* f = flag_ptr(1 - sp, m_blk, n_blk);
          int ready = 1;
          if (lane == 0) {
            const uint64_t t0 = globaltimer();
            for (uint32_t it = 0;; ++it) {
              unsigned v;
              asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
              if (v) break;
              if ((it & 15) == 15) {
                if (*abort_flag) { ready = 0; break; }
                if (globaltimer() - t0 > 1000000000ull) {
                  *abort_flag = 1;
                  atomicOr(&g_status, kStatusTimeout);
                  ready = 0;
                  break;
                }
              }
            }
          }
          ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
          if (!ready) break;
          // every lane acquires the flag (already set); lane 0 then leaves it
          // zero for the next GEMM that uses this workspace
          {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
          }
          __syncwarp();
          if (lane == 0) *const_cast<unsigned*>(f) = 0u;
        }
      }
      // with two K pieces this unit finishes the chunks it owns, the last of them being CHUNKS - 2 + sp
      const int ch_step = S > 1 ? 2 : 1;
      const int ch_last = S > 1 ? CHUNKS - 2 + sp : CHUNKS - 1;
#pragma unroll 1
      for (int ch = S > 1 ? sp : 0; ch < CHUNKS; ch += ch_step) {
        const int col0 = half * HALF_COLS + ch * 32;
        const int64_t n0 = (int64_t)n_blk * BN + col0;
        uint32_t rr[32];
        if (p.num_kb > 0) {
          tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + col0), rr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (ch == ch_last && !combiner) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release_acc();
        }
        if constexpr (EPI == EPI_STORE) {
          if (S > 1) {  // part_0 + part_1 (fp32 addition commutes: either piece gets the same bits)
            const uint4* src = slot_ptr(m_blk, n_blk, ch);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint4 w = __ldcg(src + j * 32);
              rr[4 * j] = __float_as_uint(__uint_as_float(rr[4 * j]) + __uint_as_float(w.x));
              rr[4 * j + 1] = __float_as_uint(__uint_as_float(rr[4 * j + 1]) + __uint_as_float(w.y));
              rr[4 * j + 2] = __float_as_uint(__uint_as_float(rr[4 * j + 2]) + __uint_as_float(w.z));
              rr[4 * j + 3] = __float_as_uint(__uint_as_float(rr[4 * j + 3]) + __uint_as_float(w.w));
            }
          }
        }
        uint4 hin[4];
        if constexpr (EPI == EPI_DGELU) {
          if (!mbar_wait(hbar, hphase, abort_flag)) { aborted = true; break; }
          hphase ^= 1;
          h_pending = false;
#pragma unroll
          for (int j = 0; j < 4; ++j) hin[j] = *reinterpret_cast<const uint4*>(so + sw64(r, j));
          // the box is free again: prefetch the next one this warp will need
          fence_async_smem();
          __syncwarp();
          if (ch + 1 < CHUNKS) issue_h(u, ch + 1);
          else if (u + 2 * ncl < num_units) issue_h(u + 2 * ncl, 0);
        }
        // the previous chunk's TMA stores have read the staging boxes: each 8-column group
        // below writes its results into them as soon as they are computed
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        float v[32];
        const bool full = row_ok && n0 + 32 <= p.N;  // every element of this chunk is inside the tensor
        const uint64_t s2 = f2(s, s);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int64_t n = n0 + g * 8;
          const bool ok = row_ok && n < p.N;
          uint64_t e2[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) e2[i] = f2(__uint_as_float(rr[g * 8 + 2 * i]), __uint_as_float(rr[g * 8 + 2 * i + 1]));
          uint64_t b2[4] = {0ull, 0ull, 0ull, 0ull};
          if constexpr (EPI != EPI_DGELU) {
            // this group's bias: columns 8g..8g+7 of the chunk sit in lanes 8ch + 2g and 8ch + 2g + 1
            const int l0 = ch * 8 + 2 * g;
            b2[0] = bf2_to_f2(__shfl_sync(0xFFFFFFFFu, btile.x, l0));
            b2[1] = bf2_to_f2(__shfl_sync(0xFFFFFFFFu, btile.y, l0));
            b2[2] = bf2_to_f2(__shfl_sync(0xFFFFFFFFu, btile.x, l0 + 1));
            b2[3] = bf2_to_f2(__shfl_sync(0xFFFFFFFFu, btile.y, l0 + 1));
          }
          if constexpr (EPI == EPI_STORE) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint64_t y = fma2(e2[i], s2, b2[i]);
              w[i] = pack_bf16x2(lo(y), hi(y));
            }
            *reinterpret_cast<uint4*>(so + sw64(r, g)) = make_uint4(w[0], w[1], w[2], w[3]);
          } else if constexpr (EPI == EPI_GELU) {
            // h = bf16(acc * s + b); a = h/2 * (1 + tanh(h * (k + k c h^2)))
            const uint64_t K2 = f2(kGeluK, kGeluK), KC2 = f2(kGeluK * kGeluC, kGeluK * kGeluC), H2 = f2(0.5f, 0.5f);
            uint32_t hw[4];
            uint64_t a2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint64_t hf = fma2(e2[i], s2, b2[i]);
              hw[i] = pack_bf16x2(lo(hf), hi(hf));
              const uint64_t h = bf2_to_f2(hw[i]);
              const uint64_t u = mul2(h, fma2(mul2(h, h), KC2, K2));
              const uint64_t t = f2(tanh_fast(lo(u)), tanh_fast(hi(u)));
              a2[i] = fma2(h, t, h);  // 2a: a = h/2 (1 + t) is exactly half of the rounded h + h t
            }
            if (full || ok) {
#pragma unroll
              for (int i = 0; i < 4; ++i) am_f = maxabs(maxabs(am_f, lo(a2[i])), hi(a2[i]));  // 2 amax, halved at the end
              if (p.dbg) {
                const uint64_t o0 = mul2(a2[0], H2), o1 = mul2(a2[1], H2), o2 = mul2(a2[2], H2), o3 = mul2(a2[3], H2);
                float4* d4 = reinterpret_cast<float4*>(p.dbg + m * p.N + n);
                d4[0] = make_float4(lo(o0), hi(o0), lo(o1), hi(o1));
                d4[1] = make_float4(lo(o2), hi(o2), lo(o3), hi(o3));
              }
            }
            *reinterpret_cast<uint4*>(so + sw64(r, g)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            const uint64_t q2 = f2(0.5f * scale_q, 0.5f * scale_q);  // (2a)(scale/2) rounds as a * scale
            *reinterpret_cast<uint2*>(sq + sw32(r, g >> 1) + (g & 1) * 8) =
                make_uint2((uint32_t)cvt_pair<QDT>(mul2(a2[0], q2)) | ((uint32_t)cvt_pair<QDT>(mul2(a2[1], q2)) << 16),
                           (uint32_t)cvt_pair<QDT>(mul2(a2[2], q2)) | ((uint32_t)cvt_pair<QDT>(mul2(a2[3], q2)) << 16));
          } else {  // EPI_DGELU
            // dh = acc * s * gelu'(h) with the dequant scale s folded into the constants:
            // s gelu'(h) = s/2 (1 + t) + h (1 - t^2) (s/2)(k + 3 k c h^2), t = tanh(h (k + k c h^2))
            const uint64_t K2 = f2(kGeluK, kGeluK), KC2 = f2(kGeluK * kGeluC, kGeluK * kGeluC), O2 = f2(1.0f, 1.0f);
            const uint64_t SH2 = f2(0.5f * s, 0.5f * s), SK2 = f2(0.5f * kGeluK * s, 0.5f * kGeluK * s);
            const uint64_t SKC32 = f2(1.5f * kGeluK * kGeluC * s, 1.5f * kGeluK * kGeluC * s);
            const uint32_t hw[4] = {hin[g].x, hin[g].y, hin[g].z, hin[g].w};
            uint64_t d2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint64_t h = bf2_to_f2(hw[i]);
              const uint64_t hsq = mul2(h, h);
              const uint64_t u = mul2(h, fma2(hsq, KC2, K2));
              const uint64_t t = f2(tanh_fast(lo(u)), tanh_fast(hi(u)));
              const uint64_t sdudh = fma2(hsq, SKC32, SK2);
              const uint64_t sech2 = sub2(O2, mul2(t, t));
              d2[i] = mul2(e2[i], fma2(mul2(h, sech2), sdudh, fma2(t, SH2, SH2)));
            }
            const uint64_t q2 = f2(scale_q, scale_q);
            *reinterpret_cast<uint2*>(sq + sw32(r, g >> 1) + (g & 1) * 8) =
                make_uint2((uint32_t)cvt_pair<QDT>(mul2(d2[0], q2)) | ((uint32_t)cvt_pair<QDT>(mul2(d2[1], q2)) << 16),
                           (uint32_t)cvt_pair<QDT>(mul2(d2[2], q2)) | ((uint32_t)cvt_pair<QDT>(mul2(d2[3], q2)) << 16));
            // elements past M or N need no mask in the amax and the column sums: TMA fills their
            // operand rows and H with zeros, so their dh is exactly 0 (the saturating FP8 codes are
            // never Inf, and a NaN operand that makes one NaN makes an in-range element NaN too)
#pragma unroll
            for (int i = 0; i < 4; ++i) am_f = maxabs(maxabs(am_f, lo(d2[i])), hi(d2[i]));
            if (p.dbg && ok) {
              float4* d4 = reinterpret_cast<float4*>(p.dbg + m * p.N + n);
              d4[0] = make_float4(lo(d2[0]), hi(d2[0]), lo(d2[1]), hi(d2[1]));
              d4[1] = make_float4(lo(d2[2]), hi(d2[2]), lo(d2[3]), hi(d2[3]));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[g * 8 + 2 * i] = lo(d2[i]);
              v[g * 8 + 2 * i + 1] = hi(d2[i]);
            }
          }
        }
        // one TMA store per box (rows past M and columns past N are clipped by TMA)
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int y = m_blk * BM + quarter * 32;
          if (y < p.M) {  // boxes wholly below the last row (the pair's spare tile) are skipped
            if constexpr (EPI != EPI_DGELU) tma_store_2d(&tmO, so_a, (int)n0, y);
            if constexpr (EPI != EPI_STORE) tma_store_2d(&tmQ, sq_a, (int)n0, y);
          }
          bulk_commit();
        }
        if constexpr (EPI == EPI_DGELU) {
          if (p.colsum) csred[(acc * 4 + quarter) * BN + col0 + lane] = transpose_reduce32(v, lane);
        }
      }
      if (aborted) break;
      if constexpr (EPI == EPI_DGELU) {
        if (p.colsum) {
          __syncwarp();
          if (lane == 0) mbar_arrive(csum_bar(acc, half));
          if (combiner) {
            if (!mbar_wait(csum_bar(acc, half), acc_phase, abort_flag)) break;
            for (int c = lane; c < HALF_COLS; c += 32) {
              const int col = half * HALF_COLS + c;
              const int64_t n = (int64_t)n_blk * BN + col;
              const float* cs = csred + acc * 4 * BN + col;
              const float tot = (cs[0] + cs[BN]) + (cs[2 * BN] + cs[3 * BN]);
              if (n < p.N) atomicAdd(p.colsum + n, tot);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release_acc();
          }
        }
      }
      acc_phase ^= 1;
    }
    if constexpr (EPI == EPI_DGELU) {
      if (h_pending) {  // an abort left a prefetch in flight: let it land first
        uint32_t dummy_flag = 0;
        if (lane == 0) mbar_wait(hbar, hphase, &dummy_flag, 100000000ull);
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
    if constexpr (EPI != EPI_STORE) {
      if constexpr (EPI == EPI_GELU) am_f *= 0.5f;  // the GELU epilogue tracked 2a (halving is exact)
      const uint32_t am = warp_max_u32(abs_bits(am_f));
      if (lane == 0 && am != 0u) atomic_max_amax(p.amax_q, am);
    }
  }

  tc_fence_before();
  __syncthreads();
  // both CTAs are done with the pair's tensor memory before it is freed
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (TWO)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::TMEM_COLS) : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::TMEM_COLS) : "memory");
  }
  // neither CTA leaves while its peer may still arrive on its barriers (2-SM MMA)
  cluster_sync();
}

// Diagnostic: one bounded wait on an mbarrier that nothing arrives on. It
// gives up after limit_ns, sets the status word and returns, which is how the
// timeout path of every pipeline wait above is exercised without a hang.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &flag, limit_ns);
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D tensor map over a row-major [outer, inner] tensor of 1- or 2-byte
// elements: box {box_inner, box_outer}, the given swizzle, zero fill outside.
bool make_map(CUtensorMap* tm, const void* base, int elem_bytes, int64_t inner, int64_t outer, int box_inner,
              int box_outer, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)(inner * elem_bytes)};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1u, 1u};
  const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8 operand tile: 128-byte rows, 128-byte swizzle.
bool make_operand_map(CUtensorMap* tm, const void* base, int64_t inner, int64_t outer, int box_outer) {
  return make_map(tm, base, 1, inner, outer, 128, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

struct EpiMaps {
  CUtensorMap o, q, h;
};

uint32_t make_idesc(int m_mma, int n_mma, int a_dt, int b_dt, bool a_mn, bool b_mn) {
  return (1u << 4) |                       // accumulator fp32
         ((uint32_t)a_dt << 7) |           // A: 0 E4M3, 1 E5M2
         ((uint32_t)b_dt << 10) |          // B
         ((a_mn ? 1u : 0u) << 15) |        // A major (1 = MN)
         ((b_mn ? 1u : 0u) << 16) |        // B major
         ((uint32_t)(n_mma >> 3) << 17) |  // N / 8
         ((uint32_t)(m_mma >> 4) << 24);   // M / 16
}

template <int BN, bool A_MN, bool B_MN, int EPI, int QDT, bool TWO = (BN >= 192)>
lnfp8_status launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const EpiMaps& em, const KParams& kp,
                      cudaStream_t st) {
  auto k = gemm_kernel<BN, A_MN, B_MN, EPI, QDT, TWO>;
  using C = Cfg<BN, TWO>;
  static bool smem_set = false;
  if (!smem_set) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return check_launch("fp8 gemm: shared memory attribute");
    smem_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent: as many clusters as can be resident at once, at most one per work unit
  static int max_clusters = 0;
  if (!max_clusters) {
    cfg.gridDim = dim3(CL * num_sms() / CL);
    if (cudaOccupancyMaxActiveClusters(&max_clusters, k, &cfg) != cudaSuccess || max_clusters < 1) {
      cudaGetLastError();
      max_clusters = num_sms() / CL;
    }
  }
  const int units = ((kp.num_m + CL - 1) / CL) * kp.num_n * kp.splits;
  const int clusters = units < max_clusters ? units : max_clusters;
  // a split-K reducer waits for the tile's later pieces, which must not queue behind it
  if (kp.splits > clusters) return set_error(LNFP8_ERR_UNSUPPORTED, "fp8 gemm: %d K splits on %d clusters", kp.splits, clusters);
  if (kp.upd.n > 0 && kp.splits > 1) return set_error(LNFP8_ERR_UNSUPPORTED, "fp8 gemm: a state update with split K");
  // one more cluster, the first, when the launch carries a state update
  cfg.gridDim = dim3((clusters + (kp.upd.n > 0 ? 1 : 0)) * CL);
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  static const char* kind = EPI == EPI_GELU ? "gemm_gelu" : EPI == EPI_DGELU ? "gemm_dgelu" :
                            (A_MN ? (B_MN ? "gemm_mn_mn" : "gemm_mn_k") : (B_MN ? "gemm_k_mn" : "gemm_k_k"));
  LaunchScope ls(kind, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, ta, tb, em.o, em.q, em.h, kp);
  if (e != cudaSuccess) return set_error(LNFP8_ERR_CUDA, "fp8 gemm launch: %s", cudaGetErrorString(e));
  return check_launch("fp8 gemm");
}

#include "gemm_pair.cuh"
#include "gemm_small.cuh"

template <int BN, int EPI, int QDT>
lnfp8_status launch_layouts(bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const EpiMaps& em,
                            const KParams& kp, cudaStream_t st) {
  if (!a_mn && !b_mn) return launch_t<BN, false, false, EPI, QDT>(ta, tb, em, kp, st);
  if (!a_mn && b_mn) return launch_t<BN, false, true, EPI, QDT>(ta, tb, em, kp, st);
  if (a_mn && b_mn) return launch_t<BN, true, true, EPI, QDT>(ta, tb, em, kp, st);
  return launch_t<BN, true, false, EPI, QDT>(ta, tb, em, kp, st);
}

}  // namespace

bool ln_linear_small_fits(int64_t M, int64_t K, int64_t N) {
  return M > 0 && M <= 0x7FFFFFFF && N > 0 && N <= 0x7FFFFFFF && K > 0 && K <= kSmallMaxK;
}

lnfp8_status ln_linear_small_launch(const SmallLinearArgs& a, int dtype, cudaStream_t st) {
  if (!ln_linear_small_fits(a.M, a.K, a.N))
    return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "ln_linear small path: M, N > 0 and K <= %d", kSmallMaxK);
  SmallParams sp;
  sp.M = (int)a.M;
  sp.N = (int)a.N;
  sp.K = (int)a.K;
  sp.x = a.x;
  sp.gamma = a.gamma;
  sp.beta = a.beta;
  sp.eps = a.eps;
  sp.w = a.w;
  sp.wq_in = a.wq_in;
  sp.bias = a.bias;
  sp.y = a.y;
  sp.xq = a.xq;
  sp.wq = a.wq;
  sp.mu = a.mu;
  sp.rsigma = a.rsigma;
  sp.ydbg = a.ydbg;
  sp.scale = a.scale;
  sp.scale_inv = a.scale_inv;
  sp.w_scale_inv = a.w_scale_inv;
  sp.amax_cur = a.amax_cur;
  sp.idesc = make_idesc(128, kSmallBN, dtype, dtype, false, false);
  const int nv = (int)((a.K + 255) / 256);
  const bool ln = a.gamma != nullptr;
#define SMALL(NV)                                                                                  \
  if (nv == NV) {                                                                                  \
    if (dtype == LNFP8_E4M3) return ln ? small_launch_t<NV, LNFP8_E4M3, true>(sp, st) : small_launch_t<NV, LNFP8_E4M3, false>(sp, st); \
    return ln ? small_launch_t<NV, LNFP8_E5M2, true>(sp, st) : small_launch_t<NV, LNFP8_E5M2, false>(sp, st); \
  }
  SMALL(1)
  SMALL(2)
  SMALL(3)
#undef SMALL
  return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "ln_linear small path: K = %lld", (long long)a.K);
}

lnfp8_status selftest_timeout_launch(int64_t limit_ns, cudaStream_t st) {
  LaunchScope ls("selftest_wait", st);
  selftest_wait_kernel<<<1, 32, 0, st>>>((uint64_t)limit_ns);
  return check_launch("lnfp8_selftest_timeout");
}

// Tile width and K splits for one GEMM. Costs are counted in K blocks of one
// 2-SM tile: ceil(units / clusters) rounds of K/S blocks each, plus for S > 1
// about four blocks' time for the exchange of the halves' partial products.
// Splitting is considered for the bf16-store epilogue with a workspace only,
// when all units fit in one round (the exchange then overlaps no other
// tile's work, so it is paid once), and taken when it saves more than a tenth.
// M pairs per raster group (tile_mn): as many A panels (tile rows x K codes) as
// fit in 48 MB of the L2 cache; the rest holds the B panels in flight and the
// outputs. Small problems get one group, which is plain M-fastest order.
int raster_group(int64_t num_m2, int64_t panel_bytes) {
  constexpr int64_t kBudget = 48ll << 20;
  const int64_t g = panel_bytes > 0 ? kBudget / panel_bytes : num_m2;
  return (int)max64(1, min64(g, max64(num_m2, 1)));
}

GemmPlan gemm_plan(int64_t M, int64_t N, int64_t K, int epi, bool may_split, bool kmajor) {
  GemmPlan pl;
  const int64_t num_m = (M + BM - 1) / BM;
  const int64_t num_m2 = (num_m + CL - 1) / CL;
  const int64_t num_kb = (K + BK - 1) / BK;
  const int64_t clusters = num_sms() / CL > 0 ? num_sms() / CL : 1;
  const int64_t tiles = num_m2 * ((N + 255) / 256);
  pl.bn = 256;
  pl.splits = 1;
  if (epi == EPI_STORE && may_split && tiles > 0 && num_kb >= 8) {
    auto cost = [&](int64_t sp) {
      const int64_t kbs = (num_kb + sp - 1) / sp;
      return ((tiles * sp + clusters - 1) / clusters) * kbs + 4 * (sp - 1);
    };
    int best = 1;
    for (int sp = 2; sp <= 2; ++sp) {  // the epilogue exchanges chunks between two pieces
      const int64_t kbs = (num_kb + sp - 1) / sp;
      if (kbs < 4 || (sp - 1) * kbs >= num_kb || tiles * sp > clusters) continue;  // non-empty pieces, one round
      if (cost(sp) < cost(best)) best = sp;
    }
    if (best > 1 && 10 * cost(best) < 9 * cost(1)) pl.splits = best;
  }
  // without a split, 128-wide single-SM tiles when 256-wide ones leave most SMs idle
  if (pl.splits == 1 && epi == EPI_STORE && num_m * ((N + 255) / 256) < (int64_t)num_sms()) pl.bn = 128;
  // 192-wide pair tiles (A and B K-major, N a multiple of 192) when their rounds of 3/4-size tiles take less
  // time: e.g. 8192 x 3072 has 384 tiles of 256 x 256 on 76 pairs (six rounds, the last with four tiles) and
  // 512 of 256 x 192 (seven rounds of 3/4 the work each)
  if (pl.splits == 1 && pl.bn == 256 && (epi == EPI_STORE || epi == EPI_GELU) && kmajor && N % 192 == 0) {
    const int64_t r256 = (tiles + clusters - 1) / clusters, r192 = (num_m2 * (N / 192) + clusters - 1) / clusters;
    if (4 * 3 * r192 < 4 * 4 * r256 * 9 / 10) pl.bn = 192;
  }
  pl.kb_per_split = (int)((num_kb + pl.splits - 1) / pl.splits);
  const int64_t rows = num_m2 * CL, cols = (N + pl.bn - 1) / pl.bn;
  pl.flag_bytes = pl.splits > 1 ? ((pl.splits * rows * cols * 8 * 4 + 255) / 256) * 256 : 0;
  pl.slot_bytes = pl.splits > 1 ? rows * cols * (int64_t)(BM * pl.bn) * 4 : 0;
  pl.ws_bytes = pl.flag_bytes + pl.slot_bytes;
  return pl;
}

lnfp8_status gemm_launch(const GemmArgs& g, cudaStream_t st) {
  if (g.M == 0 || g.N == 0) return LNFP8_OK;
  if (g.M > 0x7FFFFFFF || g.N > 0x7FFFFFFF || g.K > 0x7FFFFFFF)
    return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "fp8 gemm: dimension above 2^31");
  const bool a_mn = g.a_layout == 1, b_mn = g.b_layout == 1;
  const int64_t num_m = (g.M + BM - 1) / BM;
  // the 192-wide tiles are built for K-major A and B only
  GemmPlan pl = gemm_plan(g.M, g.N, g.K, g.epi, g.ws != nullptr, !a_mn && !b_mn);
  // the slots start after the flag area, which the caller may size for several GEMMs
  const int64_t flag_off = g.ws_flag_bytes > 0 ? g.ws_flag_bytes : pl.flag_bytes;
  if (pl.splits > 1 && (flag_off < pl.flag_bytes || flag_off % 256 || g.ws_bytes < flag_off + pl.slot_bytes))
    pl = gemm_plan(g.M, g.N, g.K, g.epi, false, !a_mn && !b_mn);
  const int bn = pl.bn;
  const int64_t num_n = (g.N + bn - 1) / bn;
  if (num_m * num_n > 0x7FFFFFFF) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "fp8 gemm: too many tiles");

  CUtensorMap ta, tb;
  const int64_t K = g.K > 0 ? g.K : 1;  // a zero-K product never loads; keep the map valid
  bool ok = a_mn ? make_operand_map(&ta, g.a, g.M, K, BK) : make_operand_map(&ta, g.a, K, g.M, BM);
  // the B box is half of the B tile ([bn/2 rows] K-major, [128 n] or [BK/2 k rows] MN-major): a CTA of a
  // 2-SM pair loads one half, a single-SM CTA both
  ok = ok && (b_mn ? make_operand_map(&tb, g.b, g.N, K, bn == 256 ? BK : BK / CL)
                   : make_operand_map(&tb, g.b, K, g.N, bn / CL));  // 128 or 96 rows per CTA of a pair
  // epilogue boxes: 32 x 32 per warp; unused maps are copies of a valid one
  EpiMaps em;
  em.o = em.q = em.h = ta;
  if (ok && g.epi != EPI_DGELU) ok = make_map(&em.o, g.out, 2, g.N, g.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (ok && g.epi != EPI_STORE) ok = make_map(&em.q, g.out_q, 1, g.N, g.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_32B);
  if (ok && g.epi == EPI_DGELU) ok = make_map(&em.h, g.h_in, 2, g.N, g.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) return set_error(LNFP8_ERR_CUDA, "fp8 gemm: cuTensorMapEncodeTiled failed (driver entry point or arguments)");

  KParams kp;
  kp.M = (int)g.M;
  kp.N = (int)g.N;
  kp.K = (int)g.K;
  kp.num_m = (int)num_m;
  kp.num_n = (int)num_n;
  kp.num_kb = (int)((g.K + BK - 1) / BK);
  kp.group_m = raster_group((num_m + (bn >= 192 ? 1 : 0)) / (bn >= 192 ? 2 : 1), (bn >= 192 ? 256 : 128) * g.K);
  // 256-wide tiles run the 2-SM MMA (M = 256 over the CTA pair, N = 256);
  // 128-wide tiles the 1-SM MMA (M = 128; N = 128 per instruction for MN-major B)
  kp.idesc = bn >= 192 ? make_idesc(256, bn, g.a_dtype, g.b_dtype, a_mn, b_mn)
                       : make_idesc(128, b_mn ? 128 : bn, g.a_dtype, g.b_dtype, a_mn, b_mn);
  kp.sinv_a = g.sinv_a;
  kp.sinv_b = g.sinv_b;
  kp.bias = g.bias;
  kp.out = g.out;
  kp.h_in = g.h_in;
  kp.out_q = g.out_q;
  kp.scale_q = g.scale_q;
  kp.amax_q = g.amax_q;
  kp.colsum = g.colsum;
  kp.dbg = g.dbg;
  kp.splits = pl.splits;
  kp.kb_per_split = pl.kb_per_split;
  kp.flags = pl.splits > 1 ? reinterpret_cast<unsigned*>(g.ws) : nullptr;
  kp.upd = g.upd;
  // the update keeps its history window in the operand ring's shared memory (at least 140 KB in
  // every configuration; a validated history holds at most 16384 floats)
  static_assert(16384 * sizeof(float) <= (size_t)Cfg<192, true>::EPI_OUT_OFF, "history window in the ring");
  if (kp.upd.n > 0 && (pl.splits > 1 || kp.upd.L > 16384 || kp.upd.n > 64))
    return set_error(LNFP8_ERR_UNSUPPORTED, "fp8 gemm: a carried state update needs an unsplit GEMM and a validated state");
  kp.ws = pl.splits > 1 ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(g.ws) + flag_off) : nullptr;

  if (g.epi == EPI_STORE) {
    if (bn == 256) return launch_layouts<256, EPI_STORE, LNFP8_E4M3>(a_mn, b_mn, ta, tb, em, kp, st);
    if (bn == 192) {
      if (!a_mn && !b_mn) return launch_t<192, false, false, EPI_STORE, LNFP8_E4M3>(ta, tb, em, kp, st);
      return set_error(LNFP8_ERR_UNSUPPORTED, "fp8 gemm: 192-wide tiles with layouts (%d, %d) are not built",
                       g.a_layout, g.b_layout);
    }
    return launch_layouts<128, EPI_STORE, LNFP8_E4M3>(a_mn, b_mn, ta, tb, em, kp, st);
  }
  if (g.epi == EPI_GELU && !a_mn && !b_mn) {
    if (bn == 192) {
      if (g.q_dtype == LNFP8_E4M3) return launch_t<192, false, false, EPI_GELU, LNFP8_E4M3>(ta, tb, em, kp, st);
      return launch_t<192, false, false, EPI_GELU, LNFP8_E5M2>(ta, tb, em, kp, st);
    }
    if (g.q_dtype == LNFP8_E4M3) return launch_t<256, false, false, EPI_GELU, LNFP8_E4M3>(ta, tb, em, kp, st);
    return launch_t<256, false, false, EPI_GELU, LNFP8_E5M2>(ta, tb, em, kp, st);
  }
  if (g.epi == EPI_DGELU && !a_mn && b_mn) {
    if (g.q_dtype == LNFP8_E4M3) return launch_t<256, false, true, EPI_DGELU, LNFP8_E4M3>(ta, tb, em, kp, st);
    return launch_t<256, false, true, EPI_DGELU, LNFP8_E5M2>(ta, tb, em, kp, st);
  }
  return set_error(LNFP8_ERR_UNSUPPORTED, "fp8 gemm: epilogue %d with layouts (%d, %d) is not built", g.epi,
                   g.a_layout, g.b_layout);
}

// The split exchange area a paired launch may need for its secondary GEMM
// (flag words and partial-product slots), zero when it cannot split. The launch
// still runs whole tiles where that measured faster (gemm_pair_launch), so this
// is what the workspace must hold, not what every launch uses.
GemmPlan pair_plan(const GemmArgs& sec) {
  GemmPlan pl;
  pl.bn = 256;
  const int64_t num_m2 = ((sec.M + BM - 1) / BM + CL - 1) / CL;
  const int64_t num_n = (sec.N + 255) / 256;
  const int64_t num_kb = (sec.K + BK - 1) / BK;
  pl.splits = num_kb >= 8 ? 2 : 1;
  pl.kb_per_split = (int)((num_kb + pl.splits - 1) / pl.splits);
  const int64_t tiles = num_m2 * CL * num_n;
  pl.flag_bytes = pl.splits > 1 ? ((tiles * 2 * kEpiWarps * 4 + 255) / 256) * 256 : 0;
  pl.slot_bytes = pl.splits > 1 ? tiles * (int64_t)(BM * 256) * 4 : 0;
  pl.ws_bytes = pl.flag_bytes + pl.slot_bytes;
  return pl;
}

lnfp8_status gemm_pair_launch(const GemmArgs& g0, const GemmArgs& g1, cudaStream_t st) {
  const bool fwd = g0.epi == EPI_GELU;  // FC1 (B [N, K]) with FC2 (both operands K-major)
  if (g0.a_layout != 0 || g1.epi != EPI_STORE || (fwd ? g0.b_layout != 0 : (g0.b_layout != 1 || (g0.epi != EPI_DGELU && g0.epi != EPI_STORE))))
    return set_error(LNFP8_ERR_UNSUPPORTED, "fp8 gemm pair: unsupported primary epilogue or layouts");
  for (const GemmArgs* g : {&g0, &g1})
    if (g->M > 0x7FFFFFFF || g->N > 0x7FFFFFFF || g->K > 0x7FFFFFFF)
      return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "fp8 gemm pair: dimension above 2^31");
  if (g0.M == 0 || g0.N == 0 || g0.K == 0 || g1.M == 0 || g1.N == 0 || g1.K == 0)
    return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "fp8 gemm pair: empty operand (run the GEMMs separately)");
  const bool a1_mn = g1.a_layout == 1, b1_mn = g1.b_layout == 1;
  GemmPlan pl = pair_plan(g1);
  const int64_t flag_off = g1.ws_flag_bytes > 0 ? g1.ws_flag_bytes : pl.flag_bytes;
  // Two K pieces per weight-gradient tile spread the weight gradient over more clusters while
  // its tiles are fewer than the clusters. With at least as many tiles as clusters the dGELU
  // pair (its weight gradient's MMAs hidden under the primary epilogue) runs whole tiles: the
  // exchange of partial products only costs. The MMA-bound bf16-store pair runs whole tiles
  // only up to 64 K blocks: the exchange costs the same per tile at any K, while whole tiles
  // leave the clusters' MMA work less even as K grows. Measured on the d 2048 backward: whole
  // dGELU tiles 3-12% faster per step at 2048 to 16384 tokens, even at 32768 and 65536; whole
  // FC1 tiles 8% / 4% faster per step at 2048 / 8192 tokens, about 1% slower at 16384; at d 768
  // (36 tiles on 76 clusters) the dGELU launch runs 5% faster in two pieces.
  const int64_t sec_tiles = (((g1.M + BM - 1) / BM + CL - 1) / CL) * ((g1.N + 255) / 256);
  const int64_t sec_kb = (g1.K + BK - 1) / BK;
  const bool whole_sec = sec_tiles >= num_sms() / CL && (g0.epi == EPI_DGELU || sec_kb <= 64);
  if (pl.splits > 1 &&
      (whole_sec || !g1.ws || flag_off < pl.flag_bytes || flag_off % 256 || g1.ws_bytes < flag_off + pl.slot_bytes)) {
    pl.splits = 1;
    pl.kb_per_split = (int)((g1.K + BK - 1) / BK);
  }

  CUtensorMap maps[7];
  bool ok = make_operand_map(&maps[0], g0.a, g0.K, g0.M, BM);
  ok = ok && (fwd ? make_operand_map(&maps[1], g0.b, g0.K, g0.N, 128) : make_operand_map(&maps[1], g0.b, g0.N, g0.K, BK));
  if (fwd) {
    ok = ok && make_map(&maps[2], g0.out_q, 1, g0.N, g0.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_32B);
    ok = ok && make_map(&maps[3], g0.out, 2, g0.N, g0.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  } else if (g0.epi == EPI_DGELU) {
    ok = ok && make_map(&maps[2], g0.out_q, 1, g0.N, g0.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_32B);
    ok = ok && make_map(&maps[3], g0.h_in, 2, g0.N, g0.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  } else {
    ok = ok && make_map(&maps[2], g0.out, 2, g0.N, g0.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    maps[3] = maps[2];  // no H
  }
  ok = ok && (a1_mn ? make_operand_map(&maps[4], g1.a, g1.M, g1.K, BK) : make_operand_map(&maps[4], g1.a, g1.K, g1.M, BM));
  ok = ok && (b1_mn ? make_operand_map(&maps[5], g1.b, g1.N, g1.K, BK) : make_operand_map(&maps[5], g1.b, g1.K, g1.N, 128));
  ok = ok && make_map(&maps[6], g1.out, 2, g1.N, g1.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) return set_error(LNFP8_ERR_CUDA, "fp8 gemm pair: cuTensorMapEncodeTiled failed");

  PairParams pp;
  auto prob = [&](const GemmArgs& g, bool a_mn, bool b_mn, int splits) {
    PairProb pr;
    pr.M = (int)g.M;
    pr.N = (int)g.N;
    pr.num_m2 = (int)(((g.M + BM - 1) / BM + CL - 1) / CL);
    pr.num_n = (int)((g.N + 255) / 256);
    pr.num_kb = (int)((g.K + BK - 1) / BK);
    pr.units = pr.num_m2 * pr.num_n * splits;
    pr.group_m = fwd ? pr.num_m2 : raster_group(pr.num_m2, 256 * g.K);  // the forward keeps its N-fastest order
    pr.idesc = make_idesc(256, 256, g.a_dtype, g.b_dtype, a_mn, b_mn);
    pr.sinv_a = g.sinv_a;
    pr.sinv_b = g.sinv_b;
    return pr;
  };
  pp.p0 = prob(g0, false, !fwd, 1);
  pp.bias0 = g0.bias;
  pp.p1 = prob(g1, a1_mn, b1_mn, pl.splits);
  pp.scale_q = g0.scale_q;
  pp.amax_q = g0.amax_q;
  pp.colsum = g0.colsum;
  pp.dbg = g0.dbg;
  pp.bias1 = g1.bias;
  pp.splits1 = pl.splits;
  pp.kbs1 = pl.kb_per_split;
  pp.flags = pl.splits > 1 ? reinterpret_cast<unsigned*>(g1.ws) : nullptr;
  pp.ready = nullptr;
  if (fwd) {  // per row block readiness counters in g0's workspace (zeroed by the caller)
    if (pl.splits != 1 || !g0.ws || g0.ws_bytes < (int64_t)pp.p0.num_m2 * 4)
      return set_error(LNFP8_ERR_INVALID_ARG, "fp8 gemm pair: the forward needs its readiness counters and no K split");
    pp.ready = reinterpret_cast<unsigned*>(g0.ws);
  }
  pp.ws = pl.splits > 1 ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(g1.ws) + flag_off) : nullptr;
  if ((int64_t)pp.p0.units + pp.p1.units > 0x7FFFFFFF) return set_error(LNFP8_ERR_UNSUPPORTED_SHAPE, "fp8 gemm pair: too many tiles");
  if (fwd && !a1_mn && !b1_mn) {
    if (g0.q_dtype == LNFP8_E4M3) return pair_launch_t<EPI_GELU, false, false, false, LNFP8_E4M3>(maps, pp, st);
    return pair_launch_t<EPI_GELU, false, false, false, LNFP8_E5M2>(maps, pp, st);
  }
  if (!fwd && a1_mn && b1_mn) {
    if (g0.epi == EPI_STORE) return pair_launch_t<EPI_STORE, true, true, true, LNFP8_E4M3>(maps, pp, st);
    if (g0.q_dtype == LNFP8_E4M3) return pair_launch_t<EPI_DGELU, true, true, true, LNFP8_E4M3>(maps, pp, st);
    return pair_launch_t<EPI_DGELU, true, true, true, LNFP8_E5M2>(maps, pp, st);
  }
  return set_error(LNFP8_ERR_UNSUPPORTED, "fp8 gemm pair: secondary layouts (%d, %d) are not built", g1.a_layout,
                   g1.b_layout);
}

}  // namespace lnfp8
