// Grouped GEMM on CTA pairs (tcgen05 cta_group::2), bf16 and MXFP8, for the large-M regime.
//
// Same computation as the 1-CTA kernel in gemm_tc.cu ("Efficient MoE training for
// biological foundation models", section "GroupedLinear Optimizes Expert Computation":
// grouped per-expert GEMMs with ScaledSwiGLU fused after the first), but a cluster of two
// CTAs on one TPC computes a 256 x 256 tile with one MMA stream:
//   * CTA r of the pair stages rows [128 r, 128 r + 128) of the tile's A (token rows of
//     one expert) and rows [128 r, 128 r + 128) of the 256-row B tile (packed weights);
//     both TMA loads count on the leader's (rank 0) full barrier;
//   * the leader's single MMA thread issues tcgen05.mma.cta_group::2 (M = 256, N = 256,
//     K = 16); the accumulator rows of each CTA land in that CTA's own TMEM;
//   * the leader's commits arrive on the empty / accumulator-full barriers of both CTAs
//     (multicast); both CTAs' epilogue warps drain their own TMEM rows and arrive on the
//     leader's accumulator-empty barrier.
// Per SM and 64-wide K step this stages 32 KB instead of the 48 KB of a 1-CTA 128 x 256
// tile, so the same shared memory holds a 6-deep ring (more bytes in flight per FLOP)
// and each weight byte fetched from L2 feeds two SMs.  Rows of a 256-row tile past the
// expert's segment are computed and discarded, so the pair pays more padding on small
// segments; the host picks it only when experts hold many rows.
// Row-gather mode (GEMM1): A is not loaded by TMA from a permuted copy; 4 extra warps in
// each CTA copy that CTA's 128 token rows of the stage straight from x (cp.async into the
// 128-byte swizzled layout).  The leader's gather threads arrive on the leader's full
// barrier when their copies land; the peer's arrive on a barrier of their own, and the
// peer's MMA warp (idle otherwise) relays each completed stage to the leader's full barrier
// after a proxy fence, so the leader's MMA sees both halves of A.
// MXFP8 ("MXFP8 Precision Reduces Memory Footprint": E4M3 values with one E8M0 scale per 32
// along K, Blackwell block-scaled MMAs): 128 K values (128 bytes) per stage, block-scaled
// MMAs (M = 256, N = 256, K = 32).  Each CTA stages its own scale atoms by TMA (its 128 rows'
// A scales; B's scales as the pair MMA reads them), the leader copies them into both CTAs'
// TMEM (tcgen05.cp.cta_group::2) before the stage's MMAs.  TMEM holds one 256-column
// accumulator and two sets of scale columns, so the epilogue of a tile does not overlap the
// next tile's main loop (as in the 1-CTA MXFP8 kernel at 256-wide tiles).
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"

namespace moe {

// B's scales in each CTA's TMEM: all 256 columns of the pair tile (true), or the CTA's own
// 128 (false).
constexpr bool kPairSfbFull = true;

template <bool MX>
struct PairSmemT {
  static constexpr int STAGES = 6;
  static constexpr int A_BYTES = 128 * kRowBytes;  // this CTA's 128 rows of A
  static constexpr int B_BYTES = 128 * kRowBytes;  // this CTA's half of the 256 B rows
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BK = MX ? 128 : 64;         // K elements per stage (128 bytes per row)
  static constexpr int SFA_BYTES = MX ? 512 : 0;   // one scale atom (128 rows x 128 K)
  static constexpr int SFB_BYTES = MX ? (kPairSfbFull ? 1024 : 512) : 0;
  static constexpr int SF_STAGE = SFA_BYTES + SFB_BYTES;
  static constexpr int OFF_SF = STAGES * STAGE_BYTES;
  static constexpr int OFF_EPI = OFF_SF + STAGES * SF_STAGE;
  // bf16 outputs leave by TMA stores; MXFP8 keeps the padded staging of plain stores
  static constexpr int EPI_WARP_BYTES = MX ? kEpiWarpBytes : kEpiTmaWarpBytes;
  static constexpr int OFF_BAR = OFF_EPI + 4 * EPI_WARP_BYTES;
  // full, empty, tmem_full[2], tmem_empty[2], drain, gathered (row-gather mode, peer CTA)
  static constexpr int NUM_BARS = 3 * STAGES + 5;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_TAB = OFF_MISC + 16;
  // s_off, s_mtp (256-row m-tiles), s_mtp128 (128-row m-tiles: the scale layout's)
  static constexpr int SMEM_BYTES = OFF_TAB + 3 * (kMaxEloc + 1) * 4 + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};
constexpr int kPairBM = 256;  // rows of a pair tile (128 per CTA)
constexpr int kPairBN = 256;  // columns of a pair tile

// Scale-factor maps (MXFP8): the 512-byte atoms of A's and B's SF tile layouts as rows of
// 128 uint32 (box: one atom of A; one or two consecutive atoms of B).
struct SfMaps {
  CUtensorMap sfa, sfb;
};

// Threads beyond the 6 GEMM warps: A-gather warps (row gather) or zero-row warps (combine).
template <int EPI, bool GATHER>
constexpr int pair_extra_threads() {
  return GATHER ? kGatherThreads : EPI == EPI_COMBINE ? kZeroThreads : 0;
}

template <bool MX, int EPI, bool GATHER>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads + pair_extra_threads<EPI, GATHER>(), 1)
    tc_grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                const __grid_constant__ SfMaps tmS, const __grid_constant__ OutMaps tmO,
                                const GemmArgs g) {
  static_assert(!(MX && GATHER), "the MXFP8 pair kernel reads A by TMA");
  using C = PairSmemT<MX>;
  constexpr int NUM_ACC = MX ? 1 : 2;  // accumulators in TMEM (MXFP8: + scale columns)
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 4);
  auto gath_bar = [&](int s) { return bar0 + 8u * (2 * C::STAGES + 5 + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* s_off = reinterpret_cast<int*>(smem + C::OFF_TAB);
  int* s_mtp = s_off + g.E_loc + 1;
  int* s_mtp128 = s_mtp + g.E_loc + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // row gather: the leader's expect-tx arrival, its own 128 gather threads and the
      // peer's relay
      ptx::mbar_init(full_bar(s), GATHER ? 1 + kGatherThreads + 1 : 1);
      ptx::mbar_init(empty_bar(s), 1);
      if (GATHER) ptx::mbar_init(gath_bar(s), kGatherThreads);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 8);  // 4 epilogue warps in each CTA of the pair
    }
    ptx::mbar_init(drain_bar, 1);
    *s_abort = 0;
    ptx::fence_mbar_init();
    if (!GATHER) ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if (MX) {
      ptx::prefetch_tmap(&tmS.sfa);
      ptx::prefetch_tmap(&tmS.sfb);
    }
  }
  if (warp == 1) {  // one warp in each CTA of the pair allocates the pair's TMEM
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish_pair();
  }
  pdl_wait();  // offsets, row data and scales come from the previous kernels
  if (warp == 2) {
    build_mtile_prefix(g.offsets, g.E_loc, kPairBM, s_off, s_mtp);
    if (MX) build_mtile_prefix(g.offsets, g.E_loc, 128, s_off, s_mtp128);
  }
  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync();  // barrier inits of both CTAs visible before any cross-CTA signal
  ptx::tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int n_tiles_n = (g.n_out + kPairBN - 1) / kPairBN;
  const int total = s_mtp[g.E_loc] * n_tiles_n;
  const int num_kb = (g.K + C::BK - 1) / C::BK;
  // 128-row m-tile of the scale layout holding this CTA's rows of tile tl
  auto mtile128 = [&](const Tile& tl) {
    return s_mtp128[tl.e] + (tl.row0 + 128 * static_cast<int>(rank) - s_off[tl.e]) / 128;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer (both CTAs)
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        const Tile tl = decode_tile(t, n_tiles_n, kPairBN, s_off, s_mtp, g.E_loc, kPairBM);
        const int a_row = tl.row0 + 128 * static_cast<int>(rank);
        const int b_row = tl.n0 + 128 * static_cast<int>(rank);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (*s_abort) { ok = false; break; }
          if (!ptx::mbar_wait(empty_bar(s), ph ^ 1u, g.timeout_ns)) { gemm_abort(g, s_abort); ok = false; break; }
          const uint32_t fb_leader = ptx::mapa_shared(full_bar(s), 0);
          // in row-gather mode the gather warps fill A themselves
          if (leader)
            ptx::mbar_arrive_expect_tx(full_bar(s), GATHER ? 2 * C::B_BYTES : 2 * (C::STAGE_BYTES + C::SF_STAGE));
          const uint32_t st_addr = sbase + s * C::STAGE_BYTES;
          if (!GATHER) ptx::tma_load_3d_pair(st_addr, &tmA, fb_leader, kb * C::BK, a_row, 0);
          ptx::tma_load_3d_pair(st_addr + C::A_BYTES, &tmB, fb_leader, kb * C::BK, b_row, tl.e);
          if constexpr (MX) {
            const int kg = g.K / 128;
            const uint32_t sf_addr = sbase + C::OFF_SF + s * C::SF_STAGE;
            ptx::tma_load_2d_pair(sf_addr, &tmS.sfa, fb_leader, 0, mtile128(tl) * kg + kb);
            const int b_atom = (tl.e * kg + kb) * (g.n_out / 128) + tl.n0 / 128 + (kPairSfbFull ? 0 : static_cast<int>(rank));
            ptx::tma_load_2d_pair(sf_addr + C::SFA_BYTES, &tmS.sfb, fb_leader, 0, b_atom);
          }
          ++issued;
          if (++s == C::STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok && leader) {  // let the copies already issued land before the pair exits
        for (int64_t i = issued - 1; i >= 0 && i >= issued - C::STAGES; --i)
          ptx::mbar_wait(full_bar(static_cast<int>(i % C::STAGES)), static_cast<uint32_t>((i / C::STAGES) & 1),
                         g.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------------ MMA issuer (leader)
      const uint32_t idesc = MX ? ptx::idesc_mxf8(kPairBM, kPairBN) : ptx::idesc_bf16(kPairBM, kPairBN);
      constexpr int SF_COLS = 4 + (kPairSfbFull ? 8 : 4);  // A's scales + B's, per stage
      int s = 0;
      uint32_t ph = 0, kbg = 0;
      int it = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs, ++it) {
        const int acc = NUM_ACC == 2 ? (it & 1) : 0;
        const uint32_t acc_ph = NUM_ACC == 2 ? static_cast<uint32_t>((it >> 1) & 1) : static_cast<uint32_t>(it & 1);
        if (!ptx::mbar_wait(tempty_bar(acc), acc_ph ^ 1u, g.timeout_ns)) { gemm_abort(g, s_abort); break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kPairBN);
        for (int kb = 0; kb < num_kb; ++kb) {
          // row gather: the peer's rows were released at cluster scope by its relay
          const bool got = GATHER ? ptx::mbar_wait_cluster(full_bar(s), ph, g.timeout_ns)
                                  : ptx::mbar_wait(full_bar(s), ph, g.timeout_ns);
          if (!got) { gemm_abort(g, s_abort); ok = false; break; }
          if (GATHER) ptx::fence_proxy_async_smem();  // the leader's gathered rows were written by cp.async
          ptx::tc_fence_after();
          const uint32_t a_addr = sbase + s * C::STAGE_BYTES;
          const uint32_t b_addr = a_addr + C::A_BYTES;
          if constexpr (MX) {
            const uint32_t sf_addr = sbase + C::OFF_SF + s * C::SF_STAGE;
            const uint32_t sf_col = tmem_base + NUM_ACC * kPairBN + (kbg & 1u) * SF_COLS;
            ptx::tmem_cp_32x128b_x4_pair(sf_col, ptx::sdesc_sf(sf_addr));
            ptx::tmem_cp_32x128b_x4_pair(sf_col + 4, ptx::sdesc_sf(sf_addr + C::SFA_BYTES));
            if (kPairSfbFull) ptx::tmem_cp_32x128b_x4_pair(sf_col + 8, ptx::sdesc_sf(sf_addr + C::SFA_BYTES + 512));
#pragma unroll
            for (int k = 0; k < C::BK / 32; ++k)
              ptx::mma_mxf8_pair(d_tmem, ptx::sdesc_sw128(a_addr + k * 32), ptx::sdesc_sw128(b_addr + k * 32),
                                 ptx::idesc_sf_id(idesc, k), sf_col, sf_col + 4, (kb | k) != 0);
            ++kbg;
          } else {
#pragma unroll
            for (int k = 0; k < C::BK / 16; ++k)
              ptx::mma_bf16_pair(d_tmem, ptx::sdesc_sw128(a_addr + k * 32), ptx::sdesc_sw128(b_addr + k * 32), idesc,
                                 (kb | k) != 0);
          }
          ptx::mma_commit_pair(empty_bar(s), 0x3);  // frees the stage in both CTAs
          if (++s == C::STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit_pair(tfull_bar(acc), 0x3);  // accumulator rows ready in both CTAs
      }
      ptx::mma_commit_pair(drain_bar, 0x1);  // every MMA issued by the pair has completed
      ptx::mbar_wait(drain_bar, 0, g.timeout_ns);
    } else if (GATHER && lane == 0 && !leader) {
      // ------------------------------------------------------------------ gather relay (peer)
      // Each stage this CTA's gather threads completed: make their cp.async rows (already in
      // this CTA's shared memory) visible to the async proxy that the pair MMA reads them
      // through, then arrive on the leader's full barrier.  The arrival is a CTA-scope
      // release: a cluster-scope one measured ~1 us per stage on B300 (GEMM1 241 vs 97 us at
      // T = 8192, d = 7168, 4 experts).
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        for (int kb = 0; kb < num_kb; ++kb) {
          if (*s_abort) { ok = false; break; }
          if (!ptx::mbar_wait(gath_bar(s), ph, g.timeout_ns)) { gemm_abort(g, s_abort); ok = false; break; }
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive_remote(ptx::mapa_shared(full_bar(s), 0));
          if (++s == C::STAGES) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    EpiStage est{smem + C::OFF_EPI + (warp - 2) * C::EPI_WARP_BYTES,
                 sbase + static_cast<uint32_t>(C::OFF_EPI + (warp - 2) * C::EPI_WARP_BYTES), 0, -1};
    int it = 0;
    for (int t = pair; t < total; t += npairs, ++it) {
      if (*s_abort) break;
      Tile tl = decode_tile(t, n_tiles_n, kPairBN, s_off, s_mtp, g.E_loc, kPairBM);
      if (MX) tl.mt = mtile128(tl);                        // the scale layout's m-tile of this CTA's rows
      tl.row0 += 128 * static_cast<int>(rank);             // this CTA's rows of the tile
      tl.rows = max(0, min(128, tl.rows - 128 * static_cast<int>(rank)));
      const int acc = NUM_ACC == 2 ? (it & 1) : 0;
      const uint32_t acc_ph = NUM_ACC == 2 ? static_cast<uint32_t>((it >> 1) & 1) : static_cast<uint32_t>(it & 1);
      int okw = 0;
      if (lane == 0) okw = ptx::mbar_wait(tfull_bar(acc), acc_ph, g.timeout_ns) ? 1 : 0;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      if (!okw) { if (lane == 0) gemm_abort(g, s_abort); break; }
      (void)ptx::mbar_try_wait(tfull_bar(acc), acc_ph);  // completed phase: acquire for every lane
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kPairBN);
      auto release = [&]() {  // the accumulator may be overwritten by the next tile's MMAs
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(acc), 0));
      };
      epilogue_warp<EPI, !MX>(g, tmO, tl, tbase, kPairBN, q, lane, est, release);
    }
    if (lane == 0) ptx::bulk_wait_all();  // this warp's TMA stores have completed

  } else if constexpr (GATHER) {
    // ------------------------------------------------------------------ A gather (both CTAs)
    // Thread gt copies 16-byte chunk (gt % 8) of rows gt / 8 + 16 i (i < 8) of this CTA's
    // 128 rows of each stage's A straight from the token rows, into the 128-byte swizzled
    // layout a TMA load would produce; its copies of a stage arrive (when they land) on the
    // leader's full barrier in the leader, on the relayed barrier in the peer.
    const int gt = threadIdx.x - kGemmThreads;
    const int chunk = gt & 7, rbase = gt >> 3;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = pair; t < total && ok; t += npairs) {
      Tile tl = decode_tile(t, n_tiles_n, kPairBN, s_off, s_mtp, g.E_loc, kPairBM);
      tl.row0 += 128 * static_cast<int>(rank);  // this CTA's rows of the tile
      tl.rows = max(0, min(128, tl.rows - 128 * static_cast<int>(rank)));
      const uint8_t* src[8];
      uint32_t live = 0;  // bit i: row rbase + 16 i lies in the tile
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rbase + 16 * i;
        const bool v = r < tl.rows;
        const int64_t tok = v ? __ldg(g.row_token + tl.row0 + r) : 0;
        src[i] = g.gx + tok * g.gx_ld + chunk * 16;
        live |= static_cast<uint32_t>(v) << i;
      }
      for (int kb = 0; kb < num_kb; ++kb) {
        int okw = 0;
        if (lane == 0) okw = *s_abort ? 0 : (ptx::mbar_wait(empty_bar(s), ph ^ 1u, g.timeout_ns) ? 1 : 2);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (okw != 1) {
          if (okw == 2 && lane == 0) gemm_abort(g, s_abort);
          ok = false;
          break;
        }
        (void)ptx::mbar_try_wait(empty_bar(s), ph ^ 1u);  // completed phase: acquire for every lane
        const uint32_t a_addr = sbase + s * C::STAGE_BYTES;
        const int64_t kbyte = static_cast<int64_t>(kb) * C::BK * 2 + chunk * 16;
        const bool kin = kbyte < static_cast<int64_t>(g.K) * 2;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = rbase + 16 * i;
          const bool v = kin && ((live >> i) & 1u);
          ptx::cp_async_16(a_addr + r * kRowBytes + ((chunk ^ (r & 7)) << 4), v ? src[i] + kb * C::BK * 2 : g.gx,
                           v ? 16u : 0u);
        }
        ptx::cp_async_arrive_noinc(leader ? full_bar(s) : gath_bar(s));
        if (++s == C::STAGES) { s = 0; ph ^= 1u; }
      }
    }
    ptx::cp_async_wait_all();  // nothing of ours may still be landing when the CTA exits
  } else if constexpr (EPI == EPI_COMBINE) {
    // ------------------------------------------------------------------ combine + zero rows of y
    zero_rows(g, blockIdx.x * 4 + (warp - 6), gridDim.x * 4, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync();  // neither CTA leaves while its peer may still signal or read it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, 512);
  }
}

bool make_sf_map(CUtensorMap* m, const void* base, uint64_t n_atoms, uint32_t atoms_per_box) {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!enc) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  const cuuint64_t dims[2] = {128, n_atoms};
  const cuuint64_t strides[1] = {512};
  const cuuint32_t box[2] = {128, atoms_per_box};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A: the permuted rows [a_rows, K] (TMA), or unused (nullptr) in row-gather mode.
template <bool MX, int EPI, bool GATHER = false>
static cudaError_t launch_pair_inst(const void* A, int64_t a_rows, const void* B, const GemmArgs& g, cudaStream_t st) {
  using C = PairSmemT<MX>;
  CUtensorMap ta = {}, tb;
  if (!GATHER && !make_operand_map(&ta, A, MX, g.K, a_rows, 1, 128)) return cudaErrorInvalidValue;
  if (!make_operand_map(&tb, B, MX, g.K, g.n_out, g.E_loc, 128)) return cudaErrorInvalidValue;
  SfMaps ts;
  memset(&ts, 0, sizeof(ts));
  if (MX) {
    const uint64_t kg = static_cast<uint64_t>(g.K / 128);
    if (!make_sf_map(&ts.sfa, g.a_sf, static_cast<uint64_t>(mx_tiles_cap(a_rows, g.E_loc)) * kg, 1))
      return cudaErrorInvalidValue;
    if (!make_sf_map(&ts.sfb, g.b_sf, static_cast<uint64_t>(g.E_loc) * kg * (g.n_out / 128), kPairSfbFull ? 2 : 1))
      return cudaErrorInvalidValue;
  }
  OutMaps tmo;
  memset(&tmo, 0, sizeof(tmo));
  if (!MX && !make_out_maps(&tmo, g)) return cudaErrorInvalidValue;
  auto kern = tc_grouped_gemm_pair_kernel<MX, EPI, GATHER>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int grid = num_sms() & ~1;  // whole pairs
  const int threads = kGemmThreads + pair_extra_threads<EPI, GATHER>();
  return launch_pdl(kern, dim3(grid), dim3(threads), C::SMEM_BYTES, st, ta, tb, ts, tmo, g);
}

// swiglu: GEMM1 (+ scaled SwiGLU, MXFP8: + requantisation of h), else GEMM2 (bf16 store).
cudaError_t launch_pair_gemm(const void* A, int64_t a_rows, const void* B, const GemmArgs& g, bool swiglu, bool mx,
                             cudaStream_t st) {
  if (mx)
    return swiglu ? launch_pair_inst<true, EPI_SWIGLU_MX>(A, a_rows, B, g, st)
                  : launch_pair_inst<true, EPI_STORE_BF16>(A, a_rows, B, g, st);
  return swiglu ? launch_pair_inst<false, EPI_SWIGLU_BF16>(A, a_rows, B, g, st)
                : launch_pair_inst<false, EPI_STORE_BF16>(A, a_rows, B, g, st);
}

cudaError_t launch_pair_gemm_combine(const void* A, int64_t a_rows, const void* B, const GemmArgs& g, bool mx,
                                     cudaStream_t st) {
  return mx ? launch_pair_inst<true, EPI_COMBINE>(A, a_rows, B, g, st)
            : launch_pair_inst<false, EPI_COMBINE>(A, a_rows, B, g, st);
}

// GEMM1 + scaled SwiGLU on CTA pairs with A gathered from the token rows (g.gx, g.row_token).
cudaError_t launch_pair_gemm1_gather(const void* B, const GemmArgs& g, cudaStream_t st) {
  return launch_pair_inst<false, EPI_SWIGLU_BF16, true>(nullptr, 0, B, g, st);
}

}  // namespace moe
