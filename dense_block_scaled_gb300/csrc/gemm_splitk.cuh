// gemm_splitk.cuh -- split-K GEMM for problems with few output tiles (skinny M).
//
// A GEMM with M = 16 or 128 and N = K = 8192 has only 64 output tiles of
// 128 x 128, fewer than half the SMs, and is bound by HBM reads of B.  Here a
// cluster of SPLIT CTAs works on one 128 x 128 tile, each CTA on its own
// stretch of K, so SPLIT times as many SMs stream B.  The partial
// accumulators meet in shared memory (distributed shared memory, no global
// scratch): each 32-row quadrant of the tile belongs to one CTA of the
// cluster; once a CTA's MMAs are done, the others write their FP32 partials of
// its quadrants into its now idle stage buffers, and it adds them, scales by
// alpha, rounds to BF16 and stores those rows of D.
//
// Same operand formats, layouts, roles and bounded waits as gemm_kernel.cuh;
// single-CTA MMAs (M = 128, N = 128) and one tile per cluster.
//
// For M <= 32 the A tile is loaded AROWS = 32 rows high: the MMA still reads
// 128 rows, but rows 32..127 of its accumulator are never stored, so whatever
// shared memory it reads there does not matter, and the freed 12 KB per stage
// buys a deeper pipeline for the B stream.
//
// The partials move with st.async, which counts its bytes on an mbarrier in
// the receiving CTA; each CTA tells the others that its stage buffers are free
// by a relaxed remote arrive.  No cluster-wide barrier sits on the path.
#pragma once
#include "gemm_kernel.cuh"

namespace tkg {

// 16-byte store into another CTA's shared memory that completes `bytes` of
// transaction count on an mbarrier there.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(cluster_addr), "r"(a), "r"(b), "r"(c), "r"(d), "r"(cluster_bar)
               : "memory");
}

template <int FMT, int SPLIT, int STAGES, int AROWS = 128>
struct SplitKConfig {
  using T = FmtTraits<FMT>;
  static constexpr bool kScaled = FMT != FMT_BF16;
  static constexpr int kThreads = 384;
  static constexpr int kEpiWarps = 8;
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int kRowBytes = 128;
  static constexpr int kABytes = AROWS * kRowBytes;   // rows loaded; the MMA reads BM
  static constexpr int kBBytes = BN * kRowBytes;
  static constexpr int kSfaBytes = T::kSfAtoms * 512;
  static constexpr int kSfbBytes = T::kSfAtoms * 512;   // one 128-row scale block
  static constexpr int kStageBytes = ((kABytes + kBBytes + kSfaBytes + kSfbBytes + 1023) / 1024) * 1024;
  static constexpr int kMmasPerStage = T::kStageK / T::kMmaK;
  static constexpr int kEpiBufBytes = 32 * 64;
  static constexpr int kEpiBytes = kEpiWarps * 2 * kEpiBufBytes;
  static constexpr int kPartialBytes = BM * BN * 4;   // one CTA's FP32 accumulator
  // D's staging boxes live in the stage buffers, past the partials that land in
  // this CTA: by the store every stage load has been consumed.  The 32 KB that
  // a separate staging area took went to deeper rings.
  static constexpr int kEpiOffset = (SPLIT - 1) * kPartialBytes;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kSmemBytes = kBarOffset + kNumBars * 8 + 16 + 1024;
  // bytes per stage for A boxes of a_rows rows (at most AROWS) and B boxes of b_rows rows (at most BN)
  static constexpr uint32_t tx_bytes(int a_rows, int b_rows) {
    return uint32_t(a_rows * kRowBytes + b_rows * kRowBytes + (kScaled ? kSfaBytes + kSfbBytes : 0));
  }
  static constexpr int kAccCols = BN;
  static constexpr int kScaleBase = BN;
  static constexpr int kRegionCols = 8;                  // 4 columns of A scales, 4 of B scales
  static constexpr int kRegions = (512 - BN) / kRegionCols;
  static constexpr int kTmemCols = 512;
  static constexpr int kPrefetchStages = 4;   // L2 prefetch ahead of the dependency wait (deeper delays the real loads)
  static_assert(SPLIT >= 1 && SPLIT <= 4, "split factor");
  static_assert(AROWS == 128 || AROWS == 32, "A tile height");
  // the MMA's 128-row read of a short A tile stays inside its stage
  static_assert(BM * kRowBytes <= kStageBytes, "A read past the stage");
  static_assert(kEpiOffset + kEpiBytes <= STAGES * kStageBytes,
                "partials and D's staging boxes must fit the stage buffers");
  static_assert(kSmemBytes <= 232448, "shared memory overflow");
  static constexpr uint32_t kIdesc =
      FMT == FMT_BF16 ? idesc_f16(BM, BN)
                      : idesc_bs(BM, BN, FMT == FMT_NVFP4 ? 1u : 0u, FMT == FMT_MXFP8 ? 1u : 0u, 0u, 0u);
};

template <int FMT, int SPLIT, int STAGES, int AROWS>
__global__ void __launch_bounds__(384, 1)
    gemm_splitk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                       const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  using C = SplitKConfig<FMT, SPLIT, STAGES, AROWS>;
  using T = FmtTraits<FMT>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  // Programmatic dependent launch: the next kernel may be scheduled onto free
  // SMs from here on (its own dependency wait still holds it until this grid
  // has completed); measured 1-1.5% faster on launch-bound skinny GEMMs than
  // releasing after the set-up.
  ptx::pdl_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (SPLIT > 1) ? ptx::cluster_ctarank() : 0u;

  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  auto stage_a = [&](int s) { return base + uint32_t(s * C::kStageBytes); };
  auto stage_b = [&](int s) { return base + uint32_t(s * C::kStageBytes + C::kABytes); };
  auto stage_sfa = [&](int s) { return base + uint32_t(s * C::kStageBytes + C::kABytes + C::kBBytes); };
  auto stage_sfb = [&](int s) {
    return base + uint32_t(s * C::kStageBytes + C::kABytes + C::kBBytes + C::kSfaBytes);
  };
  const uint32_t epi_base = base + uint32_t(C::kEpiOffset);   // D's staging boxes (stage buffers, past the partials)
  const uint32_t bars = base + uint32_t(C::kBarOffset);
  auto full_bar = [&](int s) { return bars + uint32_t(8 * s); };
  auto empty_bar = [&](int s) { return bars + uint32_t(8 * (STAGES + s)); };
  const uint32_t accf_bar = bars + uint32_t(8 * (2 * STAGES));
  const uint32_t drain_bar = accf_bar + 8;
  const uint32_t never_bar = drain_bar + 8;
  const uint32_t go_bar = never_bar + 8;     // every other CTA's stage buffers are free
  const uint32_t part_bar = go_bar + 8;      // all partial bytes for this CTA's quadrants have landed

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    ptx::mbar_init(accf_bar, 1);
    ptx::mbar_init(drain_bar, 1);
    ptx::mbar_init(never_bar, 1);
    ptx::mbar_init(go_bar, SPLIT > 1 ? SPLIT - 1 : 1);
    ptx::mbar_init(part_bar, 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmD);
    if (C::kScaled) {
      ptx::prefetch_tmap(&tmSFA);
      ptx::prefetch_tmap(&tmSFB);
    }
  }
  if (warp == 2) {
    ptx::tmem_alloc<1>(ptx::smem_u32(&s_tmem_base), C::kTmemCols);
    ptx::tmem_relinquish<1>();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // barrier initialisations are published by fence.mbarrier_init (release,
  // cluster scope), so the arrive is relaxed; the abort flag a peer may write
  // is written only after a wait has run out its time limit
  if (SPLIT > 1) ptx::cluster_sync_relaxed();
  ptx::tc_fence_after();
  const uint32_t tmem = s_tmem_base;

  int mb, nb;
  tile_coords(int(blockIdx.x) / SPLIT, p.tiles_m, p.tiles_n, p.raster_group, mb, nb);
  // this CTA's stretch of K (in stages); the host keeps every stretch non-empty
  const int per = (p.num_kstages + SPLIT - 1) / SPLIT;
  const int ks0 = int(rank) * per;
  const int ks1 = min(ks0 + per, p.num_kstages);

  // Warm L2 with the first stages of this CTA's stretch while the previous
  // kernel may still be running (prefetches read nothing back; see
  // ptx::tma_prefetch_2d).
  if (warp == 0) {
    if (ptx::elect_one()) {
      const int npf = min(ks1 - ks0, C::kPrefetchStages);
#pragma unroll 1
      for (int ks = ks0; ks < ks0 + npf; ++ks) {
        const int kx = ks * C::kRowBytes / (FMT == FMT_BF16 ? 2 : 1);
        ptx::tma_prefetch_2d(&tmB, kx, nb * C::BN);
        ptx::tma_prefetch_2d(&tmA, kx, mb * C::BM);
        if constexpr (C::kScaled) {
          ptx::tma_prefetch_3d(&tmSFB, 0, ks * T::kSfAtoms, nb);
          ptx::tma_prefetch_3d(&tmSFA, 0, ks * T::kSfAtoms, mb);
        }
      }
    }
    __syncwarp();
  }
  // Programmatic dependent launch: the set-up above overlapped the previous
  // kernel's tail.  Only the roles that read global memory wait for the
  // previous grid to complete (griddepcontrol.wait): the producer right before
  // its first load and the storing epilogue before it reads the tensor scales.
  // The MMA issuer and the partial exchange touch only shared and tensor
  // memory, and every store of D follows the producer's first load.

  Ctl ctl;
  ctl.abort_flag = &s_abort;
  ctl.abort_smem = ptx::smem_u32(&s_abort);
  ctl.rank = rank;
  ctl.ncta = SPLIT;
  ctl.status = p.status;
  ctl.timeout_ns = p.timeout_ns;

  // ------------------------------------------------------------------ producer
  if (warp == 0) {
    if (ptx::elect_one()) {
      const uint64_t pol_a = ptx::policy_evict_last();    // A is read by every N tile
      const uint64_t pol_b = ptx::policy_evict_first();   // B is read once
      uint32_t stage = 0, phase = 0, armed = 0, armed_par = 0;
      bool ok = true, waited = false;
#pragma unroll 1
      for (int ks = ks0; ks < ks1; ++ks) {
        if (!wait_bar<false>(empty_bar(stage), phase ^ 1u, ctl)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(full_bar(stage), p.tx_bytes);
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        const int kx = ks * C::kRowBytes / (FMT == FMT_BF16 ? 2 : 1);
        // a ring slot, a K stage of this launch, a 16-byte aligned x (TMA's rule)
        if (!invariant(stage < uint32_t(STAGES) && ks >= 0 && ks < p.num_kstages &&
                           (kx * (FMT == FMT_BF16 ? 2 : 1)) % 16 == 0,
                       p.status)) {
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        if (!waited) {
          ptx::pdl_wait();
          waited = true;
        }
        ptx::tma_load_2d<1>(stage_a(stage), &tmA, kx, mb * C::BM, full_bar(stage), pol_a);
        ptx::tma_load_2d<1>(stage_b(stage), &tmB, kx, nb * C::BN, full_bar(stage), pol_b);
        if constexpr (C::kScaled) {
          ptx::tma_load_3d<1>(stage_sfa(stage), &tmSFA, 0, ks * T::kSfAtoms, mb, full_bar(stage), pol_a);
          ptx::tma_load_3d<1>(stage_sfb(stage), &tmSFB, 0, ks * T::kSfAtoms, nb, full_bar(stage), pol_b);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        Ctl quiet = ctl;
        int dummy = 0;
        quiet.abort_flag = &dummy;
#pragma unroll 1
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) wait_bar<false>(full_bar(s), (armed_par >> s) & 1u, quiet);
      }
    }
    __syncwarp();
  }
  // ------------------------------------------------------------------ MMA issuer
  else if (warp == 1) {
    if (ptx::elect_one()) {
      uint32_t stage = 0, phase = 0, region = 0;
      bool ok = true;
      if (p.inject_stall) ok = wait_bar<false>(never_bar, 0u, ctl);
#pragma unroll 1
      for (int ks = ks0; ks < ks1 && ok; ++ks) {
        if (!wait_bar<false>(full_bar(stage), phase, ctl)) {
          ok = false;
          break;
        }
        const uint64_t adesc = sdesc_sw128(stage_a(stage));
        const uint64_t bdesc = sdesc_sw128(stage_b(stage));
        // the accumulator and the scale region lie inside the allocation
        const uint32_t n_mma = ((p.idesc >> 17) & 0x3Fu) << 3;
        const bool stage_ok = invariant(stage < uint32_t(STAGES) && n_mma <= uint32_t(C::kAccCols), p.status);
#pragma unroll
        for (int j = 0; j < C::kMmasPerStage; ++j) {
          const int k0 = ks * T::kStageK + j * T::kMmaK;
          if (k0 >= p.k || !stage_ok) break;
          const uint64_t koff = uint64_t((j * 32) >> 4);
          const uint32_t accum = (ks > ks0 || j > 0) ? 1u : 0u;
          if constexpr (FMT == FMT_BF16) {
            ptx::mma_f16<1>(tmem, adesc + koff, bdesc + koff, p.idesc, accum);
          } else {
            const int g = (FMT == FMT_NVFP4) ? j : 0;
            if (!invariant(region < uint32_t(C::kRegions) &&
                               uint32_t(C::kScaleBase) + (region + 1u) * uint32_t(C::kRegionCols) <=
                                   uint32_t(C::kTmemCols),
                           p.status))
              break;
            const uint32_t reg = tmem + uint32_t(C::kScaleBase + region * C::kRegionCols);
            if (FMT == FMT_NVFP4 || j == 0) {
              ptx::tmem_cp_32x128b_x4<1>(reg, sdesc_sf(stage_sfa(stage) + uint32_t(512 * g)));
              ptx::tmem_cp_32x128b_x4<1>(reg + 4u, sdesc_sf(stage_sfb(stage) + uint32_t(512 * g)));
            }
            if constexpr (FMT == FMT_MXFP8) {
              const uint32_t idesc = p.idesc | (uint32_t(j) << 29) | (uint32_t(j) << 4);
              ptx::mma_mxf8<1>(tmem, adesc + koff, bdesc + koff, idesc, reg, reg + 4u, accum);
            } else {
              ptx::mma_nvf4<1>(tmem, adesc + koff, bdesc + koff, p.idesc, reg, reg + 4u, accum);
            }
            if (FMT == FMT_NVFP4 || j == C::kMmasPerStage - 1 || k0 + T::kMmaK >= p.k) {
              if (++region == uint32_t(C::kRegions)) region = 0;
            }
          }
        }
        ptx::tc_commit<1>(empty_bar(stage), 1);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) ptx::tc_commit<1>(accf_bar, 1);
      ptx::tc_commit<1>(drain_bar, 1);
      Ctl quiet = ctl;
      int dummy = 0;
      quiet.abort_flag = &dummy;
      wait_bar<false>(drain_bar, 0u, quiet);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------------ epilogue: own partial into registers
  const bool epi = warp >= 4;
  const int e = warp - 4;
  const int q = warp & 3;              // accumulator lane quadrant
  const int h = e >> 2;                // column half: [0, 64) or [64, 128)
  const int row = q * 32 + lane;       // tile row this thread holds
  uint32_t v[2][32];
  uint32_t have = 0;
  // a quadrant whose 32 rows all lie beyond M (M = 16 leaves three of four
  // idle) has nothing to reduce or store
  const bool live = mb * C::BM + q * 32 < p.m;
  if (epi && live) {
    // whole-warp waits, converged (as in the persistent kernel's epilogue)
    have = wait_bar_warp<false>(accf_bar, 0u, ctl) ? 1u : 0u;
    if constexpr (SPLIT > 1) {
      if (warp == 4 && lane == 0 && have) {
        // every MMA of this CTA has completed, so its stage buffers may take
        // partials: arm the partial barrier and tell the other CTAs
        const int rows_left = p.m - mb * C::BM;
        const int live_q = rows_left >= C::BM ? 4 : (rows_left + 31) / 32;
        int my_live = 0;   // quadrants with rows below M that this CTA owns
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) my_live += (qq < live_q && (qq * SPLIT) / 4 == int(rank)) ? 1 : 0;
        ptx::mbar_arrive_expect_tx(part_bar, uint32_t((SPLIT - 1) * my_live * 2) * uint32_t(32 * 64 * 4));
#pragma unroll 1
        for (uint32_t r = 0; r < uint32_t(SPLIT); ++r)
          if (r != rank) ptx::mbar_arrive_relaxed_cluster(ptx::map_to_rank(go_bar, r));
      }
    }
    if (have) {
      ptx::tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t(q * 32) << 16) + uint32_t(h * 64);
      ptx::tmem_ld_32x32b_x32(taddr, v[0]);
      ptx::tmem_ld_32x32b_x32(taddr + 32u, v[1]);
      ptx::tmem_ld_wait();
    }
  }
  // 16-byte chunk c (of 32 per 512-byte row) of a partial row, XOR-swizzled by row
  auto partial_addr = [&](uint32_t region_base, int c) {
    return region_base + uint32_t(row * 512) + uint32_t(((c ^ row) & 31) * 16);
  };

  // ------------------------------------------------------------------ split-K reduction
  // Quadrant q of the tile is summed and stored by CTA q * SPLIT / 4 (with two
  // CTAs: rows 0-63 by the first, 64-127 by the second), so the partial traffic
  // and the final epilogue are spread over the cluster.
  const int owner = (q * SPLIT) / 4;
  const bool mine = owner == int(rank);
  if constexpr (SPLIT > 1) {
    if (epi && have && !mine) {
      if (wait_bar_warp<false>(go_bar, 0u, ctl)) {
        const int slot = int(rank) < owner ? int(rank) : int(rank) - 1;   // this CTA's place among the senders
        const uint32_t dst = ptx::map_to_rank(base + uint32_t(slot * C::kPartialBytes), uint32_t(owner));
        const uint32_t rbar = ptx::map_to_rank(part_bar, uint32_t(owner));
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t a = dst + uint32_t(row * 512) + uint32_t((((h * 16 + c * 8 + j) ^ row) & 31) * 16);
            st_async_v4(a, v[c][4 * j], v[c][4 * j + 1], v[c][4 * j + 2], v[c][4 * j + 3], rbar);
          }
      }
    }
    if (epi && have && mine) {
      have = wait_bar_warp<false>(part_bar, 0u, ctl) ? 1u : 0u;
      if (have) {
#pragma unroll 1
        for (int r = 0; r < SPLIT - 1; ++r) {
          const uint32_t src = base + uint32_t(r * C::kPartialBytes);
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t w0, w1, w2, w3;
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                           : "r"(partial_addr(src, h * 16 + c * 8 + j)));
              v[c][4 * j] = __float_as_uint(__uint_as_float(v[c][4 * j]) + __uint_as_float(w0));
              v[c][4 * j + 1] = __float_as_uint(__uint_as_float(v[c][4 * j + 1]) + __uint_as_float(w1));
              v[c][4 * j + 2] = __float_as_uint(__uint_as_float(v[c][4 * j + 2]) + __uint_as_float(w2));
              v[c][4 * j + 3] = __float_as_uint(__uint_as_float(v[c][4 * j + 3]) + __uint_as_float(w3));
            }
        }
      }
    }
  }

  // ------------------------------------------------------------------ epilogue: the owner stores D
  if (epi && mine && have && !s_abort) {
    ptx::pdl_wait();
    float alpha = p.alpha;
    if (p.ta) alpha = alpha * __ldg(p.ta);
    if (p.tb) alpha = alpha * __ldg(p.tb);
    const uint32_t my_buf0 = epi_base + uint32_t(e * 2 * C::kEpiBufBytes);
    const int row0 = mb * C::BM + q * 32;
    const int col0 = nb * C::BN + h * 64;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint32_t buf = my_buf0 + uint32_t(c * C::kEpiBufBytes);
      const uint32_t row_addr = buf + uint32_t(lane * 64);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
          w[x] = ptx::pack_bf16x2(__uint_as_float(v[c][8 * j + 2 * x]) * alpha,
                                  __uint_as_float(v[c][8 * j + 2 * x + 1]) * alpha);
        ptx::st_shared_v4(row_addr + ((uint32_t(j) ^ ((uint32_t(lane) >> 1) & 3u)) * 16u), w[0], w[1], w[2], w[3]);
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(&tmD, buf, col0 + c * 32, row0);
        ptx::bulk_commit_group();
      }
    }
    // the stores need only have read their shared memory before this CTA goes;
    // their global writes are part of the grid's work the next kernel waits for
    if (lane == 0) ptx::bulk_wait_group_read<0>();
    __syncwarp();
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (s_abort && threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 50000ull) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // By now no CTA touches another's shared memory (the partials have all
  // landed, the go arrivals were waited for), so the exit barrier needs no
  // memory ordering.
  if (SPLIT > 1) ptx::cluster_sync_relaxed();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<1>(tmem, C::kTmemCols);
  }
}

}  // namespace tkg
