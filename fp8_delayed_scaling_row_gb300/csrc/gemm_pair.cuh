// Paired persistent GEMM: two independent GEMMs share every CTA pair of one
// launch. In the backward the "primary" is a data gradient (A [M, K] K-major,
// B [K, N]) with either the fused dGELU epilogue (FC2) or a bf16 store (FC1),
// and the "secondary" the matching weight gradient, a bf16 store with both
// operands [K, rows]. In the forward the primary is FC1 with the GELU epilogue
// on one half of the token rows and the secondary FC2 (both operands K-major)
// on the same rows: FC2 tile (rows r, columns n) reads the GELU codes that the
// FC1 tiles of rows r write in this launch, so the launch orders its work by
// row blocks and FC2's loads wait (bounded) on per-tile readiness counters.
//
// The dGELU epilogue (GELU derivative, E5M2 cast, amax, column sums, the
// read of H) takes several times longer per 256 x 256 tile than the tile's
// MMAs (K = d_model), so alone its tensor cores idle most of the time. The
// weight gradient is the opposite: long MMAs (K = tokens) and a short
// epilogue. Here each CTA pair walks one schedule: a primary tile, then a
// slice of its secondary tiles' K blocks, then the next primary tile, ... so
// the MMAs of the secondary run while the epilogue warps work on the primary.
// With a bf16-store primary the pairing evens out the two GEMMs' tile counts
// over the SMs instead (neither fills a whole number of waves alone).
// Tensor memory holds one primary accumulator (columns 0-255) and one
// secondary accumulator (256-511); all 16 epilogue warps drain each tile
// (warp quarter q reads TMEM lanes 32q.., warp slice s the tile's columns
// 64s..64s+63, two 32-column chunks).
//
// This file is part of gemm.cu's translation unit (it uses its PTX wrappers,
// tile constants and status word).

// Shared memory of a paired launch. The dGELU and GELU primaries stage H and
// FP8 codes per epilogue warp and (dGELU) column-sum partials, which leaves room
// for a 4-stage operand ring; a bf16-store primary needs none of them and runs
// 6 stages (its MMAs, not its epilogue, set the launch's time).
template <int PEPI>
struct PairCfg {
  static constexpr bool STORE = PEPI == EPI_STORE;
  static constexpr int STAGES = STORE ? 6 : 4;
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = 128 * BK;  // this CTA's half of the 256-wide B tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int OUT_OFF = STAGES * STAGE_BYTES;                           // bf16 staging box per warp (bf16 stores)
  static constexpr int H_OFF = OUT_OFF + kEpiWarps * 2048;                       // bf16 H box per warp (primary loads)
  static constexpr int Q_OFF = H_OFF + (STORE ? 0 : kEpiWarps * 2048);           // FP8 staging box per warp (primary stores)
  static constexpr int CSUM_OFF = Q_OFF + (STORE ? 0 : kEpiWarps * 1024);        // [tile parity][row quarter][256] fp32 column-sum partials
  static constexpr int BAR_OFF = CSUM_OFF + (STORE ? 0 : 2 * 4 * 256 * 4);
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM = 1024 + BAR_OFF + BAR_BYTES;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(2 * STAGES + 5 + 4 + kEpiWarps + 1 <= BAR_BYTES / 8, "barrier area");
};

struct PairProb {
  int M, N, num_m2, num_n, num_kb, units;
  int group_m;  // M pairs per raster group (tile_mn); the forward (DEP) order is N fastest
  uint32_t idesc;
  const float* sinv_a;
  const float* sinv_b;
};

struct PairParams {
  PairProb p0, p1;  // primary (dGELU or bf16 store), secondary (bf16 store)
  const uint16_t* bias0;  // primary bias (bf16-store primary)
  // primary epilogue
  const float* scale_q;
  float* amax_q;
  float* colsum;
  float* dbg;
  // secondary epilogue
  const uint16_t* bias1;
  int splits1, kbs1;  // K pieces per secondary tile (1 or 2) and K blocks per piece
  // Uneven pieces (bf16-store primary): the first s_tail secondary positions hold the long
  // pieces (K blocks s_small..) of tiles 0..s_tail-1, the last s_tail positions their short
  // pieces (K blocks 0..s_small-1), the positions between both halves of the other tiles.
  // The last positions fall on the clusters with one primary tile more (see pair_launch_t).
  int s_tail, s_small;
  float* ws;          // split exchange: [tile][warp][chunk][8][32] x 16 B
  unsigned* flags;    // [tile][piece][warp]
  unsigned* ready;    // forward: per row block, the epilogue warps (both CTAs, every FC1 tile) done with its codes; zero at launch
};

// Forward dependency order (GELU primary): primary tiles run row block by row
// block (N fastest) and secondary (FC2) tiles row block major. A secondary tile
// may start in the gap one round after the round in which the last FC1 tile of
// its row block runs: every wait then points at work earlier in every CTA
// pair's schedule (no cycles), and by the time a producer gets there those
// tiles' epilogues have usually finished on all SMs, so the wait rarely holds
// up the next FC1 tile's loads.
// Secondary position v -> its tile and K piece.
__device__ __forceinline__ int s_tile(const PairParams& p, int v) {
  if (p.splits1 == 1) return v;
  if (v < p.s_tail) return v;
  if (v >= p.p1.units - p.s_tail) return v - (p.p1.units - p.s_tail);
  return p.s_tail + (v - p.s_tail) / 2;
}
__device__ __forceinline__ int s_piece(const PairParams& p, int v) {
  if (p.splits1 == 1) return 0;
  if (v < p.s_tail) return 1;
  if (v >= p.p1.units - p.s_tail) return 0;
  return (v - p.s_tail) & 1;
}

__device__ __forceinline__ int fwd_release_round(const PairParams& p, int v, int ncl) {
  const int m2 = s_tile(p, v) / p.p1.num_n;
  return (p.p0.num_n * (m2 + 1) - 1) / ncl + 1;
}

// The schedule of one cluster. Its work units are the global units c, c + ncl,
// ... where global units 0..U0-1 are the primary tiles and the rest the
// secondary units (tile, K piece). The cluster runs its primary units in
// order and spreads the K blocks of its secondary units evenly over the gaps
// after them.
struct PairSched {
  int c, ncl, U0, U1, nP;
  int64_t KS;
  __device__ void init(const PairParams& p, int cid, int ncl_) {
    c = cid;
    ncl = ncl_;
    U0 = p.p0.units;
    U1 = p.p1.units;
    nP = U0 > c ? (U0 - c + ncl - 1) / ncl : 0;
    KS = 0;
    for (int g = c + nP * ncl; g < U0 + U1; g += ncl) KS += s_len(p, g - U0);
  }
  __device__ int p_unit(int i) const { return c + i * ncl; }
  __device__ int s_unit(int j) const { return c + (nP + j) * ncl - U0; }  // j-th secondary unit of the cluster
  __device__ static int s_kb0(const PairParams& p, int v) {
    return s_piece(p, v) == 0 ? 0 : (s_tile(p, v) < p.s_tail ? p.s_small : p.kbs1);
  }
  __device__ static int s_len(const PairParams& p, int v) {
    const int k0 = s_kb0(p, v);
    if (s_piece(p, v) == 1 || p.splits1 == 1) return p.p1.num_kb - k0;
    return s_tile(p, v) < p.s_tail ? p.s_small : min(p.p1.num_kb, p.kbs1);
  }
  __device__ int gaps() const { return nP > 0 ? nP : 1; }
  __device__ int64_t gap_end(int i) const { return nP > 0 ? KS * (i + 1) / nP : KS; }
};

// Walks the secondary K blocks of a cluster's schedule: segment = one unit's
// consecutive K blocks inside one gap.
struct SecCursor {
  int j = 0;         // local index of the current secondary unit
  int64_t jo = 0;    // schedule offset where it starts
  int64_t off = 0;   // next offset to run
  // gap: the gap index (for the forward's release rule); dep: forward dependency order
  template <class F>
  __device__ bool run_gap(const PairSched& sc, const PairParams& p, int64_t end, F&& seg, int gap = 0, bool dep = false) {
    const bool last_gap = gap == sc.gaps() - 1;
    if (dep && last_gap) end = sc.KS;
    while (off < end) {
      const int v = sc.s_unit(j);
      if (dep && off == jo && !last_gap && fwd_release_round(p, v, sc.ncl) > gap) break;  // not released yet
      const int len = PairSched::s_len(p, v);
      const int64_t seg_end = min(end, jo + len);
      const int k0 = PairSched::s_kb0(p, v);
      const bool first = off == jo, last = seg_end == jo + len;
      if (!seg(v, k0 + (int)(off - jo), k0 + (int)(seg_end - jo), first, last)) return false;
      off = seg_end;
      if (last) {
        jo += len;
        ++j;
      }
    }
    return true;
  }
};

template <int PEPI, bool B0_MN, bool A1_MN, bool B1_MN, int QDT>
__global__ void __launch_bounds__(kThreads, 1)
pair_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
            const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmH0,
            const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
            const __grid_constant__ CUtensorMap tmO1, const PairParams p) {
  using C = PairCfg<PEPI>;
  constexpr int STAGES = C::STAGES;
  constexpr int BN = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, csum[4 slices], hload[kEpiWarps]
  uint32_t* misc = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5 + 4 + kEpiWarps);
  uint32_t* tmem_slot = misc;
  volatile uint32_t* abort_flag = misc + 1;
  float* csred2 = reinterpret_cast<float*>(smem + C::CSUM_OFF);  // [2 tile parities][4 quarters][256]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  auto csum_bar = [&](int sl) { return bar0 + 8u * (2 * STAGES + 5 + sl); };
  auto hload_bar = [&](int w) { return bar0 + 8u * (2 * STAGES + 9 + w); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);  // released once by the pair's leader MMA
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * kEpiWarps);  // every epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    for (int sl = 0; sl < 4; ++sl) mbar_init(csum_bar(sl), 4);
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(hload_bar(w), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster_sync();
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA0)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB0)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA1)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB1)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)), "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  const int rank = (int)cluster_rank();
  const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
  constexpr uint16_t kPair = 3;
  PairSched sc;
  sc.init(p, cid, ncl);
  // tile coordinates: primary unit u = tile; secondary position v -> s_tile, s_piece
  constexpr bool DEP = PEPI == EPI_GELU;  // forward: FC2 depends on this launch's FC1 output
  auto p_m = [&](int u) {
    return (DEP ? u / p.p0.num_n : tile_mn(u, p.p0.num_m2, p.p0.num_n, p.p0.group_m).x) * CL + rank;
  };
  auto p_n = [&](int u) { return DEP ? u % p.p0.num_n : tile_mn(u, p.p0.num_m2, p.p0.num_n, p.p0.group_m).y; };
  auto s_m = [&](int v) {
    const int t = s_tile(p, v);
    return (DEP ? t / p.p1.num_n : tile_mn(t, p.p1.num_m2, p.p1.num_n, p.p1.group_m).x) * CL + rank;
  };
  auto s_n = [&](int v) {
    const int t = s_tile(p, v);
    return DEP ? t % p.p1.num_n : tile_mn(t, p.p1.num_m2, p.p1.num_n, p.p1.group_m).y;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      auto load = [&](bool prim, int m_blk, int n_blk, int kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) return false;
        const uint32_t fb = full_bar(stage);
        const uint32_t fl = map_to_rank(fb, 0);
        const uint32_t a_dst = smem_u32(smem + stage * C::STAGE_BYTES);
        const uint32_t b_dst = a_dst + C::A_BYTES;
        if (rank == 0) mbar_arrive_expect_tx(fb, 2 * C::STAGE_BYTES);
        if (prim) {  // A [M, K] K-major; B [K, N] (backward) or [N, K] (forward FC1)
          tma_load_2d_cg2(a_dst, &tmA0, kb * BK, m_blk * BM, fl);
          if (B0_MN) tma_load_2d_cg2(b_dst, &tmB0, n_blk * BN + rank * 128, kb * BK, fl);
          else       tma_load_2d_cg2(b_dst, &tmB0, kb * BK, n_blk * BN + rank * 128, fl);
        } else {
          if (!A1_MN) tma_load_2d_cg2(a_dst, &tmA1, kb * BK, m_blk * BM, fl);
          else        tma_load_2d_cg2(a_dst, &tmA1, m_blk * BM, kb * BK, fl);
          if (!B1_MN) tma_load_2d_cg2(b_dst, &tmB1, kb * BK, n_blk * BN + rank * 128, fl);
          else        tma_load_2d_cg2(b_dst, &tmB1, n_blk * BN + rank * 128, kb * BK, fl);
        }
        ++issued;
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
        return true;
      };
      // forward: wait (bounded) until every FC1 tile of the row block has written its GELU codes
      int dep_ok = -1;
      auto wait_ready = [&](int u_dep) {
        if (u_dep == dep_ok) return true;
        const unsigned* f = p.ready + u_dep;
        const uint64_t t0 = globaltimer();
        for (uint32_t it = 0;; ++it) {
          unsigned v;
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
          if (v >= 2u * kEpiWarps * (unsigned)p.p0.num_n) break;
          if ((it & 15) == 15) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > 1000000000ull) {
              *abort_flag = 1;
              atomicOr(&g_status, kStatusTimeout);
              return false;
            }
          }
        }
        // the codes were written by TMA stores: order the acquire before this thread's TMA loads
        asm volatile("fence.proxy.async.global;" ::: "memory");
        dep_ok = u_dep;
        return true;
      };
      SecCursor cur;
      for (int i = 0; i < sc.gaps() && ok; ++i) {
        if (i < sc.nP) {
          const int u = sc.p_unit(i);
          for (int kb = 0; kb < p.p0.num_kb && ok; ++kb) ok = load(true, p_m(u), p_n(u), kb);
        }
        if (ok)
          ok = cur.run_gap(sc, p, sc.gap_end(i), [&](int v, int k0, int k1, bool, bool) {
            for (int kb = k0; kb < k1; ++kb) {
              if (DEP && !wait_ready(s_tile(p, v) / p.p1.num_n)) return false;
              if (!load(false, s_m(v), s_n(v), kb)) return false;
            }
            return true;
          }, i, DEP);
      }
      if (!ok && rank == 0) {
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
    // ---------------------------------------------------------------- MMA issuer (pair leader)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase[2] = {0u, 0u};
      bool ok = true;
      auto mma_blocks = [&](bool prim, int k0, int k1, bool fresh) {
        const uint32_t d_tmem = tmem_base + (prim ? 0u : 256u);
        const uint32_t idesc = prim ? p.p0.idesc : p.p1.idesc;
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) return false;
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_base = a_base + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint32_t accum = !(fresh && kb == k0 && kk == 0);
            const bool a_mn = prim ? false : A1_MN, b_mn = prim ? B0_MN : B1_MN;
            const uint64_t ad = a_mn ? make_desc(a_base + kk * 32 * 128, 1024, 1024) : make_desc(a_base + kk * 32, 16, 1024);
            const uint64_t bd = b_mn ? make_desc(b_base + kk * 32 * 128, 1024, 1024) : make_desc(b_base + kk * 32, 16, 1024);
            mma_f8_cg2(d_tmem, ad, bd, idesc, accum);
          }
          mma_commit_cg2_mc(empty_bar(stage), kPair);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        return true;
      };
      SecCursor cur;
      for (int i = 0; i < sc.gaps() && ok; ++i) {
        if (i < sc.nP) {
          if (!mbar_wait(tempty_bar(0), acc_phase[0] ^ 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          if (!mma_blocks(true, 0, p.p0.num_kb, true)) { ok = false; break; }
          mma_commit_cg2_mc(tfull_bar(0), kPair);
          acc_phase[0] ^= 1;
        }
        ok = cur.run_gap(sc, p, sc.gap_end(i), [&](int, int k0, int k1, bool first, bool last) {
          if (first) {
            if (!mbar_wait(tempty_bar(1), acc_phase[1] ^ 1, abort_flag)) return false;
            tc_fence_after();
          }
          if (!mma_blocks(false, k0, k1, first)) return false;
          if (last) {
            mma_commit_cg2_mc(tfull_bar(1), kPair);
            acc_phase[1] ^= 1;
          }
          return true;
        }, i, DEP);
      }
      if (!ok) {
        mma_commit_cg2_mc(drain_bar, 1);
        uint32_t dummy_flag = 0;
        mbar_wait(drain_bar, 0, &dummy_flag, 100000000ull);
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue (16 warps per tile)
    const int ew = warp - 4;
    const int quarter = warp & 3;  // TMEM lanes 32*quarter..
    const int slice = ew >> 2;     // columns 64*slice .. 64*slice+63 of the tile
    const int r = lane;
    uint8_t* so = smem + C::OUT_OFF + ew * 2048;
    uint8_t* sh = smem + C::H_OFF + ew * 2048;
    uint8_t* sq = smem + C::Q_OFF + ew * 1024;
    const uint32_t so_a = smem_u32(so), sh_a = smem_u32(sh), sq_a = smem_u32(sq);
    const uint32_t hbar = hload_bar(ew);
    uint32_t hphase = 0;
    bool h_pending = false;
    const float s0 = __fmul_rn(*p.p0.sinv_a, *p.p0.sinv_b);
    const float s1 = __fmul_rn(*p.p1.sinv_a, *p.p1.sinv_b);
    const float scale_q = PEPI != EPI_STORE ? *p.scale_q : 0.f;
    float am_f = 0.f;
    uint32_t acc_phase[2] = {0u, 0u};
    const bool combiner = p.colsum != nullptr && quarter == 0;
    const uint32_t tempty0 = map_to_rank(tempty_bar(0), 0), tempty1 = map_to_rank(tempty_bar(1), 0);
    // H prefetch: this warp's two chunks of each of the cluster's primary tiles, one chunk ahead
    int h_i = 0, h_ch = 0;
    auto issue_h = [&]() {
      if (PEPI != EPI_DGELU || h_i >= sc.nP) return;
      const int u = sc.p_unit(h_i);
      if (lane == 0) {
        mbar_arrive_expect_tx(hbar, 2048);
        tma_load_2d(sh_a, &tmH0, p_n(u) * BN + slice * 64 + h_ch * 32, p_m(u) * BM + quarter * 32, hbar);
      }
      h_pending = true;
      if (++h_ch == 2) { h_ch = 0; ++h_i; }
    };
    issue_h();

    // Every warp releases the primary accumulator after its last tensor-memory
    // load, so the next primary tile's MMAs overlap the rest of this epilogue.
    // The column-sum partials alternate between two buffers by tile parity: a
    // combiner reads this tile's buffer before it touches the next tile, and
    // the tile after next cannot start before every warp, the combiner too,
    // has released the next one.
    auto prim_tile = [&](int u) -> bool {
      const int m_blk = p_m(u), n_blk = p_n(u);
      float* csred = csred2 + acc_phase[0] * 4 * BN;
      if (!mbar_wait(tfull_bar(0), acc_phase[0], abort_flag)) return false;
      tc_fence_after();
      const int64_t m = (int64_t)m_blk * BM + quarter * 32 + r;
      const bool row_ok = m < p.p0.M;
#pragma unroll 1
      for (int ch = 0; ch < 2; ++ch) {
        const int col0 = slice * 64 + ch * 32;
        const int64_t n0 = (int64_t)n_blk * BN + col0;
        uint32_t rr[32];
        tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col0, rr);
        if (ch == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(tempty0);
        }
        if (!mbar_wait(hbar, hphase, abort_flag)) return false;
        hphase ^= 1;
        h_pending = false;
        uint4 hin[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) hin[j] = *reinterpret_cast<const uint4*>(sh + sw64(r, j));
        fence_async_smem();
        __syncwarp();
        issue_h();
        float v[32];
        uint2 oq[4];
        // dh = acc * s * gelu'(h) with the dequant scale s folded into per-launch constants:
        // s gelu'(h) = s/2 (1 + t) + h (1 - t^2) (s/2)(k + 3 k c h^2), t = tanh(h (k + k c h^2))
        const uint64_t K2 = f2(kGeluK, kGeluK), KC2 = f2(kGeluK * kGeluC, kGeluK * kGeluC), O2 = f2(1.0f, 1.0f);
        const uint64_t SH2 = f2(0.5f * s0, 0.5f * s0), SK2 = f2(0.5f * kGeluK * s0, 0.5f * kGeluK * s0);
        const uint64_t SKC32 = f2(1.5f * kGeluK * kGeluC * s0, 1.5f * kGeluK * kGeluC * s0);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int64_t n = n0 + g * 8;
          const uint32_t hw[4] = {hin[g].x, hin[g].y, hin[g].z, hin[g].w};
          uint64_t d2[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint64_t e2 = f2(__uint_as_float(rr[g * 8 + 2 * i]), __uint_as_float(rr[g * 8 + 2 * i + 1]));
            const uint64_t h = bf2_to_f2(hw[i]);
            const uint64_t hsq = mul2(h, h);
            const uint64_t uu = mul2(h, fma2(hsq, KC2, K2));
            const uint64_t t = f2(tanh_fast(lo(uu)), tanh_fast(hi(uu)));
            const uint64_t sdudh = fma2(hsq, SKC32, SK2);
            const uint64_t sech2 = sub2(O2, mul2(t, t));
            d2[i] = mul2(e2, fma2(mul2(h, sech2), sdudh, fma2(t, SH2, SH2)));
          }
          const uint64_t q2 = f2(scale_q, scale_q);
          oq[g].x = (uint32_t)cvt_pair<QDT>(mul2(d2[0], q2)) | ((uint32_t)cvt_pair<QDT>(mul2(d2[1], q2)) << 16);
          oq[g].y = (uint32_t)cvt_pair<QDT>(mul2(d2[2], q2)) | ((uint32_t)cvt_pair<QDT>(mul2(d2[3], q2)) << 16);
          // Elements past M or N need no mask in the amax and the column sums: TMA fills their
          // operand rows and H with zeros, so their accumulators and dh are exactly 0 (the
          // saturating FP8 codes are never Inf, and a NaN operand that makes one NaN makes an
          // in-range element of the same row or column NaN too).
#pragma unroll
          for (int i = 0; i < 4; ++i) am_f = maxabs(maxabs(am_f, lo(d2[i])), hi(d2[i]));
          if (p.dbg && row_ok && n < p.p0.N) {
            float4* d4 = reinterpret_cast<float4*>(p.dbg + m * p.p0.N + n);
            d4[0] = make_float4(lo(d2[0]), hi(d2[0]), lo(d2[1]), hi(d2[1]));
            d4[1] = make_float4(lo(d2[2]), hi(d2[2]), lo(d2[3]), hi(d2[3]));
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[g * 8 + 2 * i] = lo(d2[i]);
            v[g * 8 + 2 * i + 1] = hi(d2[i]);
          }
        }
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        *reinterpret_cast<uint4*>(sq + sw32(r, 0)) = make_uint4(oq[0].x, oq[0].y, oq[1].x, oq[1].y);
        *reinterpret_cast<uint4*>(sq + sw32(r, 1)) = make_uint4(oq[2].x, oq[2].y, oq[3].x, oq[3].y);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int y = m_blk * BM + quarter * 32;
          if (y < p.p0.M) tma_store_2d(&tmX0, sq_a, (int)n0, y);
          bulk_commit();
        }
        if (p.colsum) csred[quarter * BN + col0 + lane] = transpose_reduce32(v, lane);
      }
      if (p.colsum) {
        __syncwarp();
        if (lane == 0) mbar_arrive(csum_bar(slice));
        if (combiner) {
          if (!mbar_wait(csum_bar(slice), acc_phase[0], abort_flag)) return false;
          for (int c = lane; c < 64; c += 32) {
            const int col = slice * 64 + c;
            const int64_t n = (int64_t)n_blk * BN + col;
            const float tot = (csred[col] + csred[BN + col]) + (csred[2 * BN + col] + csred[3 * BN + col]);
            if (n < p.p0.N) atomicAdd(p.colsum + n, tot);
          }
        }
      }
      acc_phase[0] ^= 1;
      return true;
    };

    // FC1 tile with the GELU epilogue: h = bf16(acc * s + b1) leaves through
    // tmH0, a = gelu_tanh(h) folds into the amax and leaves as codes through tmX0
    auto gelu_tile = [&](int u) -> bool {
      const int m_blk = p_m(u), n_blk = p_n(u);
      if (!mbar_wait(tfull_bar(0), acc_phase[0], abort_flag)) return false;
      tc_fence_after();
      const int64_t m = (int64_t)m_blk * BM + quarter * 32 + r;
      const bool row_ok = m < p.p0.M;
#pragma unroll 1
      for (int ch = 0; ch < 2; ++ch) {
        const int col0 = slice * 64 + ch * 32;
        const int64_t n0 = (int64_t)n_blk * BN + col0;
        uint4 bias8[4];
#pragma unroll
        for (int g = 0; g < 4; ++g)
          bias8[g] = p.bias0 && n0 + g * 8 < p.p0.N ? __ldg(reinterpret_cast<const uint4*>(p.bias0 + n0 + g * 8))
                                                    : make_uint4(0u, 0u, 0u, 0u);
        uint32_t rr[32];
        tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col0, rr);
        if (ch == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(tempty0);
        }
        uint4 ob[4];
        uint2 oq[4];
        const uint64_t s2 = f2(s0, s0);
        const uint64_t K2 = f2(kGeluK, kGeluK), KC2 = f2(kGeluK * kGeluC, kGeluK * kGeluC), H2 = f2(0.5f, 0.5f);
        const uint64_t q2 = f2(0.5f * scale_q, 0.5f * scale_q);  // (2a)(scale/2) rounds as a * scale
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int64_t n = n0 + g * 8;
          const bool ok = row_ok && n < p.p0.N;
          const uint4 bu = bias8[g];
          const uint64_t b2[4] = {bf2_to_f2(bu.x), bf2_to_f2(bu.y), bf2_to_f2(bu.z), bf2_to_f2(bu.w)};
          uint32_t hw[4];
          uint64_t a2[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint64_t e2 = f2(__uint_as_float(rr[g * 8 + 2 * i]), __uint_as_float(rr[g * 8 + 2 * i + 1]));
            const uint64_t hf = fma2(e2, s2, b2[i]);
            hw[i] = pack_bf16x2(lo(hf), hi(hf));
            const uint64_t h = bf2_to_f2(hw[i]);
            const uint64_t uu = mul2(h, fma2(mul2(h, h), KC2, K2));
            const uint64_t t = f2(tanh_fast(lo(uu)), tanh_fast(hi(uu)));
            a2[i] = fma2(h, t, h);  // 2a: a = h/2 (1 + t) is exactly half of the rounded h + h t
          }
          if (ok) {
#pragma unroll
            for (int i = 0; i < 4; ++i) am_f = maxabs(maxabs(am_f, lo(a2[i])), hi(a2[i]));  // 2 amax, halved at the end
            if (p.dbg) {
              const uint64_t o0 = mul2(a2[0], H2), o1 = mul2(a2[1], H2), o2 = mul2(a2[2], H2), o3 = mul2(a2[3], H2);
              float4* d4 = reinterpret_cast<float4*>(p.dbg + m * p.p0.N + n);
              d4[0] = make_float4(lo(o0), hi(o0), lo(o1), hi(o1));
              d4[1] = make_float4(lo(o2), hi(o2), lo(o3), hi(o3));
            }
          }
          ob[g] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          oq[g].x = (uint32_t)cvt_pair<QDT>(mul2(a2[0], q2)) | ((uint32_t)cvt_pair<QDT>(mul2(a2[1], q2)) << 16);
          oq[g].y = (uint32_t)cvt_pair<QDT>(mul2(a2[2], q2)) | ((uint32_t)cvt_pair<QDT>(mul2(a2[3], q2)) << 16);
        }
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(so + sw64(r, j)) = ob[j];
        *reinterpret_cast<uint4*>(sq + sw32(r, 0)) = make_uint4(oq[0].x, oq[0].y, oq[1].x, oq[1].y);
        *reinterpret_cast<uint4*>(sq + sw32(r, 1)) = make_uint4(oq[2].x, oq[2].y, oq[3].x, oq[3].y);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int y = m_blk * BM + quarter * 32;
          if (y < p.p0.M) {
            tma_store_2d(&tmH0, so_a, (int)n0, y);
            tma_store_2d(&tmX0, sq_a, (int)n0, y);
          }
          bulk_commit();
        }
      }
      // this warp's codes of the tile are written: count it towards the tile's readiness
      if (lane == 0) {
        bulk_wait0();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.ready + u / p.p0.num_n) : "memory");
      }
      __syncwarp();
      acc_phase[0] ^= 1;
      return true;
    };

    // bf16-store tile in accumulator buffer b; with two K pieces (secondary
    // only) the halves exchange chunks: piece q finishes chunk q of every
    // warp's pair and spills the other
    auto slot_ptr = [&](int m_blk, int n_blk, int ch) {
      const int64_t t = (int64_t)m_blk * p.p1.num_n + n_blk;
      return reinterpret_cast<uint4*>(p.ws + t * (int64_t)(BM * BN)) + ((ew * 2 + ch) * 8) * 32 + lane;
    };
    auto flag_ptr = [&](int m_blk, int n_blk, int q) {
      return p.flags + (((int64_t)m_blk * p.p1.num_n + n_blk) * 2 + q) * kEpiWarps + ew;
    };
    auto store_tile = [&](int b, int m_blk, int n_blk, int sp, int splits, const CUtensorMap* tmO,
                          const uint16_t* bias, int N, int M, float sc_ab) -> bool {
      if (!mbar_wait(tfull_bar(b), acc_phase[b], abort_flag)) return false;
      tc_fence_after();
      const uint32_t col_base = (uint32_t)(b * 256);
      if (splits > 1) {
        const int ch = 1 - sp;
        uint32_t rr[32];
        tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + col_base + (uint32_t)(slice * 64 + ch * 32), rr);
        uint4* dst = slot_ptr(m_blk, n_blk, ch);
#pragma unroll
        for (int j = 0; j < 8; ++j) __stcg(dst + j * 32, make_uint4(rr[4 * j], rr[4 * j + 1], rr[4 * j + 2], rr[4 * j + 3]));
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicExch(flag_ptr(m_blk, n_blk, sp), 1u);
        const unsigned* f = flag_ptr(m_blk, n_blk, 1 - sp);
        int ready = 1;
        if (lane == 0) {
          const uint64_t t0 = globaltimer();
          for (uint32_t it = 0;; ++it) {
            unsigned fv;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(fv) : "l"(f) : "memory");
            if (fv) break;
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
        if (!ready) return false;
        {
          unsigned fv;
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(fv) : "l"(f) : "memory");
        }
        __syncwarp();
        if (lane == 0) *const_cast<unsigned*>(f) = 0u;
      }
      const int ch_first = splits > 1 ? sp : 0, ch_step = splits > 1 ? 2 : 1;
#pragma unroll 1
      for (int ch = ch_first; ch < 2; ch += ch_step) {
        const int col0 = slice * 64 + ch * 32;
        const int64_t n0 = (int64_t)n_blk * BN + col0;
        uint4 bias8[4];
#pragma unroll
        for (int g = 0; g < 4; ++g)
          bias8[g] = bias && n0 + g * 8 < N ? __ldg(reinterpret_cast<const uint4*>(bias + n0 + g * 8))
                                            : make_uint4(0u, 0u, 0u, 0u);
        uint32_t rr[32];
        tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + col_base + (uint32_t)col0, rr);
        if (ch + ch_step >= 2) {  // the last load of this warp: release the accumulator
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(b ? tempty1 : tempty0);
        }
        if (splits > 1) {  // part_0 + part_1 (fp32 addition commutes)
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
        uint4 ob[4];
        const uint64_t s2 = f2(sc_ab, sc_ab);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint4 bu = bias8[g];
          const uint64_t b2[4] = {bf2_to_f2(bu.x), bf2_to_f2(bu.y), bf2_to_f2(bu.z), bf2_to_f2(bu.w)};
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint64_t e2 = f2(__uint_as_float(rr[g * 8 + 2 * i]), __uint_as_float(rr[g * 8 + 2 * i + 1]));
            const uint64_t y = fma2(e2, s2, b2[i]);
            w[i] = pack_bf16x2(lo(y), hi(y));
          }
          ob[g] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(so + sw64(r, j)) = ob[j];
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int y = m_blk * BM + quarter * 32;
          if (y < M) tma_store_2d(tmO, so_a, (int)n0, y);
          bulk_commit();
        }
      }
      acc_phase[b] ^= 1;
      return true;
    };

    SecCursor cur;
    bool ok = true;
    for (int i = 0; i < sc.gaps() && ok; ++i) {
      if (i < sc.nP) {
        const int u = sc.p_unit(i);
        if constexpr (PEPI == EPI_DGELU) ok = prim_tile(u);
        else if constexpr (PEPI == EPI_GELU) ok = gelu_tile(u);
        else ok = store_tile(0, p_m(u), p_n(u), 0, 1, &tmX0, p.bias0, p.p0.N, p.p0.M, s0);
      }
      if (ok)
        ok = cur.run_gap(sc, p, sc.gap_end(i), [&](int v, int, int, bool, bool last) {
          return last ? store_tile(1, s_m(v), s_n(v), s_piece(p, v), p.splits1, &tmO1, p.bias1,
                                   p.p1.N, p.p1.M, s1)
                      : true;
        }, i, DEP);
    }
    if (h_pending) {  // a prefetch may be in flight (the last one, or after an abort)
      uint32_t dummy_flag = 0;
      if (lane == 0) mbar_wait(hbar, hphase, &dummy_flag, 100000000ull);
      __syncwarp();
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
    if constexpr (PEPI == EPI_GELU) am_f *= 0.5f;  // the GELU epilogue tracked 2a (halving is exact)
    const uint32_t am = warp_max_u32(abs_bits(am_f));
    if (lane == 0 && am != 0u) atomic_max_amax(p.amax_q, am);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
  }
  cluster_sync();
}

template <int PEPI, bool B0_MN, bool A1_MN, bool B1_MN, int QDT>
lnfp8_status pair_launch_t(const CUtensorMap* maps, const PairParams& pp, cudaStream_t st) {
  auto k = pair_kernel<PEPI, B0_MN, A1_MN, B1_MN, QDT>;
  static bool smem_set = false;
  if (!smem_set) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg<PEPI>::SMEM) != cudaSuccess)
      return check_launch("fp8 gemm pair: shared memory attribute");
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
  cfg.dynamicSmemBytes = PairCfg<PEPI>::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters = 0;
  if (!max_clusters) {
    cfg.gridDim = dim3(num_sms());
    if (cudaOccupancyMaxActiveClusters(&max_clusters, k, &cfg) != cudaSuccess || max_clusters < 1) {
      cudaGetLastError();
      max_clusters = num_sms() / CL;
    }
  }
  const int units = pp.p0.units + pp.p1.units;
  const int clusters = units < max_clusters ? units : max_clusters;
  // the two K pieces of a secondary tile exchange partials: they must run on different clusters
  if (pp.splits1 > 1 && clusters < 2) return set_error(LNFP8_ERR_UNSUPPORTED, "fp8 gemm pair: split on one cluster");
  // With a bf16-store primary the launch is MMA-bound: the first U0 % clusters clusters run one
  // primary tile more, and when the secondary positions wrap onto those clusters once, the
  // tiles whose pieces land there are cut unevenly (a short piece there, the long one on a
  // cluster with fewer primaries), evening out the clusters' K blocks.
  PairParams pq = pp;
  pq.s_tail = pq.s_small = 0;
  if (PEPI == EPI_STORE && pq.splits1 == 2) {
    const int U0 = pq.p0.units, U1 = pq.p1.units, c0 = U0 % clusters, tail = U1 - (clusters - c0);
    const int lo = U0 / clusters, kb0 = pq.p0.num_kb, kb1 = pq.p1.num_kb;
    if (c0 > 0 && tail > 0 && tail <= c0 && U1 >= 2 * tail && U1 <= clusters) {
      const int small = max(1, min(kb1 / 2, (kb1 - kb0) / 2));
      const int before = (lo + 1) * kb0 + pq.kbs1;
      const int after = max((lo + 1) * kb0 + small, lo * kb0 + kb1 - small);
      if (after < before) {
        pq.s_tail = tail;
        pq.s_small = small;
      }
    }
  }
  cfg.gridDim = dim3(clusters * CL);
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  static const char* kind = PEPI == EPI_DGELU ? "gemm_dgelu_wgrad" : PEPI == EPI_GELU ? "gemm_gelu_fc2" : "gemm_dgrad_wgrad";
  LaunchScope ls(kind, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], pq);
  if (e != cudaSuccess) return set_error(LNFP8_ERR_CUDA, "fp8 gemm pair launch: %s", cudaGetErrorString(e));
  return check_launch("fp8 gemm pair");
}
