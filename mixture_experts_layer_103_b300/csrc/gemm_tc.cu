// Steps 3-4: grouped GEMMs of the expert MLP on the 5th-generation tensor cores.
//
// "Efficient MoE training for biological foundation models" (BioNeMo), section
// "GroupedLinear Optimizes Expert Computation": every expert keeps its own matrices but
// all experts run as one grouped operation; GroupedLinear -> ScaledSwiGLU -> GroupedLinear
// is fused so the gate/up pre-activation is never materialised, and ScaledSwiGLU applies
// the routing probabilities inside the activation.  Section "MXFP8 Precision Reduces
// Memory Footprint": 8-bit values with one scale per 32 along K on Blackwell tensor-core
// instructions, with quantisation fused into the same kernel.
//
// One persistent kernel per GEMM, one CTA per SM, 6 warps:
//   warp 0      TMA producer: per pipeline stage one 128 x 128-byte tile of A (the
//               expert's token rows) and one BN x 128-byte tile of B (the expert's packed
//               weights), 128-byte swizzled; MXFP8 adds the two scale-factor atoms (plain
//               bulk copies; the SF tile layout makes each one contiguous)
//   warp 1      TMEM allocator + MMA issuer (one thread): tcgen05.mma 128 x BN x 16 (bf16)
//               or block-scaled 128 x BN x 32 (E4M3 x E4M3 with E8M0 scales copied to TMEM
//               by tcgen05.cp), fp32 accumulators in TMEM, double-buffered when they fit
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (one TMEM lane = one row per
//               thread), then either bf16 store (GEMM2) or the fused scaled SwiGLU
//               h = p * silu(gate) * up with bf16 or MXFP8 (32 values = one block per
//               thread) output (GEMM1)
// CTAs run in clusters of two.  The static scheduler hands out units of two tiles, one
// per CTA of a cluster: while an expert has two m-tiles left, a unit is the pair of
// m-tiles (m, m + 1) against one n-tile, so both CTAs stream the same weight tile at the
// same time (the second read of each weight box is an L2 hit); an expert's odd last
// m-tile forms units of two n-tiles.  Every CTA loads all of its own operands with plain
// TMA loads into its own shared memory (no cross-CTA copies, so the kernel is the same on
// any number of GPUs).  m-tiles are 128-row slices of each expert's segment
// [offsets[e], offsets[e+1]), numbered in expert order, so experts with no tokens cost
// nothing and their weights are never read.  Rows of a tile past its expert's segment are
// computed and discarded.  Both CTAs of a cluster consume the same sequence of pipeline
// stages in lockstep: a stage is refilled only when both have finished with it (each MMA
// issuer's commit arrives on the empty barriers of both CTAs), which keeps the two weight
// streams of a unit within a few k-blocks of each other.
// Every wait is bounded; on a timeout the kernel records MOE_ERR_TIMEOUT in the device
// error word, drains its own copies and MMAs and exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "gemm_tc.cuh"

namespace moe {

// Shared-memory plan.  The A/B pipeline is a ring of variable-size stages inside a fixed
// byte budget: a stage holds one 128-row A tile and one BN-row B tile (128 bytes per
// row), so the depth is 4 stages at BN = 256, 6 at BN = 128 and 8 at BN = 64.  The MXFP8
// scale atoms of each stage live in a separate ring.
template <bool MX>
struct GemmSmem {
  static constexpr int MAX_STAGES = MX ? 6 : 8;            // MXFP8 tiles are 256 or 128 wide
  static constexpr int A_BYTES = kBM * kRowBytes;           // 16 KB
  static constexpr int PIPE_BYTES = 192 * 1024;             // A + B ring
  static constexpr int SF_STAGE_BYTES = MX ? 512 + 1024 : 0; // SFA atom + up to two SFB atoms
  static constexpr int BK = MX ? 128 : 64;                  // K elements per stage
  static constexpr int UMMA_K = MX ? 32 : 16;               // K elements per MMA
  static constexpr int OFF_PIPE = 0;
  static constexpr int OFF_SF = OFF_PIPE + PIPE_BYTES;
  static constexpr int OFF_EPI = OFF_SF + MAX_STAGES * SF_STAGE_BYTES;  // epilogue staging
  // bf16 outputs leave by TMA stores (two swizzled buffers per warp); MXFP8 kernels keep
  // the padded staging of plain stores (their scale rings leave no room for more)
  static constexpr int EPI_WARP_BYTES = MX ? kEpiWarpBytes : kEpiTmaWarpBytes;
  static constexpr int OFF_BAR = OFF_EPI + 4 * EPI_WARP_BYTES;
  static constexpr int NUM_BARS = 2 * MAX_STAGES + 5;       // full, empty, tmem_full[2], tmem_empty[2], drain
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_TAB = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = OFF_TAB + 3 * (kMaxEloc + 1) * 4 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// Units (tile pairs) of a launch with n-tile count nt: an expert with M m-tiles gives
// (M / 2) * nt shared-weight units plus ceil(nt / 2) units for an odd last m-tile.
// mt_total = total m-tiles, odd = experts with an odd m-tile count.
__device__ __forceinline__ long unit_count(int mt_total, int odd, int nt) {
  return static_cast<long>((mt_total - odd) / 2) * nt + static_cast<long>(odd) * ((nt + 1) / 2);
}

// Tile width of a launch, identical in every CTA: the candidate with the fewest
// cost-weighted waves of units over the clusters.  The relative costs of a 128 x BN tile
// (1.0 / 0.72 / 0.5 for BN = 256 / 128 / 64) are measured per-wave times on B300 at
// these shapes; a narrower tile does less work but feeds the tensor core less
// efficiently.  MXFP8 uses 256 or 128 (its scale-factor atoms cover 128 rows of B).
__device__ __forceinline__ int choose_bn(int mt_total, int odd, int n_out, int clusters, bool mx) {
  const int cand[3] = {256, 128, 64};
  const float cost[3] = {1.0f, 0.72f, 0.5f};
  int best = 256;
  float best_cost = 3.0e38f;
  for (int i = 0; i < (mx ? 2 : 3); ++i) {
    const long units = unit_count(mt_total, odd, (n_out + cand[i] - 1) / cand[i]);
    const long waves = (units + clusters - 1) / clusters;
    const float c = static_cast<float>(waves) * cost[i];
    if (c < best_cost) {
      best_cost = c;
      best = cand[i];
    }
  }
  return best;
}

// Per-expert tables in shared memory (one warp): s_off[e] = offsets[e], s_mtp[e] = m-tiles
// of the experts before e, s_odd[e] = experts before e with an odd m-tile count; entry
// E_loc holds the totals.
__device__ __forceinline__ void build_unit_tables(const int32_t* __restrict__ offsets, int E_loc, int* s_off,
                                                  int* s_mtp, int* s_odd) {
  const int lane = threadIdx.x & 31;
  const int per = (E_loc + 31) / 32;
  const int e_begin = lane * per, e_end = min(E_loc, e_begin + per);
  int sum = 0, odd = 0;
  for (int e = e_begin; e < e_end; ++e) {
    const int o0 = __ldg(offsets + e), o1 = __ldg(offsets + e + 1);
    const int m = (o1 - o0 + kBM - 1) / kBM;
    s_off[e] = o0;
    sum += m;
    odd += m & 1;
  }
  int incl = sum, incl_odd = odd;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    const int z = __shfl_up_sync(0xffffffffu, incl_odd, off);
    if (lane >= off) {
      incl += y;
      incl_odd += z;
    }
  }
  int run = incl - sum, run_odd = incl_odd - odd;
  for (int e = e_begin; e < e_end; ++e) {
    s_mtp[e] = run;
    s_odd[e] = run_odd;
    const int m = (__ldg(offsets + e + 1) - __ldg(offsets + e) + kBM - 1) / kBM;
    run += m;
    run_odd += m & 1;
  }
  if (lane == 31) {
    s_mtp[E_loc] = incl;
    s_odd[E_loc] = incl_odd;
    s_off[E_loc] = __ldg(offsets + E_loc);
  }
}

// The tile CTA `rank` of a cluster computes in unit u.  shared_b: both CTAs use the same
// weight tile; valid = false only for the idle half of a unit whose
// expert has an odd m-tile and an odd n-tile count: that CTA recomputes its partner's tile
// and stores nothing.
struct UnitTile {
  Tile t;
  bool shared_b, valid;
};

__device__ __forceinline__ UnitTile decode_unit(int u, int rank, int nt, int bn, const int* s_off, const int* s_mtp,
                                                const int* s_odd, int E_loc) {
  const int hnt = (nt + 1) / 2;
  auto first_unit = [&](int e) { return nt * ((s_mtp[e] - s_odd[e]) >> 1) + hnt * s_odd[e]; };
  int lo = 0, hi = E_loc - 1;  // last expert whose first unit is <= u (skips empty experts)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (first_unit(mid) <= u) lo = mid;
    else hi = mid - 1;
  }
  const int e = lo, i = u - first_unit(e);
  const int m_e = s_mtp[e + 1] - s_mtp[e];
  const int pairs = m_e >> 1;
  int mloc, n;
  UnitTile r;
  r.valid = true;
  if (i < pairs * nt) {
    mloc = 2 * (i / nt) + rank;
    n = i % nt;
    r.shared_b = true;
  } else {
    const int j = i - pairs * nt;
    mloc = m_e - 1;
    n = 2 * j + rank;
    r.shared_b = false;
    if (n >= nt) {
      n = 2 * j;
      r.valid = false;
    }
  }
  r.t.e = e;
  r.t.mt = s_mtp[e] + mloc;
  r.t.row0 = s_off[e] + mloc * kBM;
  r.t.rows = min(kBM, s_off[e + 1] - r.t.row0);
  r.t.n0 = n * bn;
  return r;
}

// B operand maps with box heights 256, 128 and 64 rows: a full tile of each width.
struct BMaps {
  CUtensorMap b256, b128, b64;
};

// Threads beyond the 6 GEMM warps: A-gather warps (row gather) or zero-row warps (combine).
template <int EPI, bool GATHER>
constexpr int extra_threads() {
  return GATHER ? kGatherThreads : EPI == EPI_COMBINE ? kZeroThreads : 0;
}

template <bool MX, int EPI, bool GATHER>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads + extra_threads<EPI, GATHER>(), 1)
    tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ BMaps tmB,
                           const __grid_constant__ OutMaps tmO, const GemmArgs g) {
  using C = GemmSmem<MX>;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::MAX_STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::MAX_STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::MAX_STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::MAX_STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* s_off = reinterpret_cast<int*>(smem + C::OFF_TAB);
  int* s_mtp = s_off + g.E_loc + 1;
  int* s_odd = s_mtp + g.E_loc + 1;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const int cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
  const uint16_t both = 0x3;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::MAX_STAGES; ++s) {
      ptx::mbar_init(full_bar(s), GATHER ? 1 + kGatherThreads : 1);  // + every gather thread
      ptx::mbar_init(empty_bar(s), 2);  // the MMA issuers of both CTAs
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 4);
    }
    ptx::mbar_init(drain_bar, 1);
    *s_abort = 0;
    ptx::fence_mbar_init();
    if (!GATHER) ptx::prefetch_tmap(&tmA);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  pdl_wait();  // offsets, row data and scales come from the previous kernels
  if (warp == 2) build_unit_tables(g.offsets, g.E_loc, s_off, s_mtp, s_odd);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer's barriers exist before any remote commit
  ptx::tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int BN = choose_bn(s_mtp[g.E_loc], s_odd[g.E_loc], g.n_out, clusters, MX);
  const CUtensorMap* tmb = BN == 256 ? &tmB.b256 : BN == 128 ? &tmB.b128 : &tmB.b64;
  const int stage_bytes = C::A_BYTES + BN * kRowBytes;  // multiple of 1024
  const int stages = min(C::MAX_STAGES, C::PIPE_BYTES / stage_bytes);
  const int sf_cols = MX ? (BN / 128 + 1) * 4 : 0;       // SFA 4 columns + SFB 4 per 128 rows
  const int num_acc = (2 * BN + 2 * sf_cols <= 512) ? 2 : 1;
  const uint32_t sf_base_col = static_cast<uint32_t>(num_acc * BN);
  const int n_tiles_n = (g.n_out + BN - 1) / BN;
  const int units = static_cast<int>(unit_count(s_mtp[g.E_loc], s_odd[g.E_loc], n_tiles_n));
  const int num_kb = (g.K + C::BK - 1) / C::BK;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer
      ptx::prefetch_tmap(tmb);
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int u = cluster; u < units && ok; u += clusters) {
        const UnitTile ut = decode_unit(u, rank, n_tiles_n, BN, s_off, s_mtp, s_odd, g.E_loc);
        const Tile& tl = ut.t;
        const int sfb_bytes = MX ? min(BN, g.n_out - tl.n0) / 128 * 512 : 0;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (*s_abort) { ok = false; break; }
          if (!ptx::mbar_wait(empty_bar(s), ph ^ 1u, g.timeout_ns)) { gemm_abort(g, s_abort); ok = false; break; }
          const uint32_t fb = full_bar(s);
          const uint32_t st_addr = sbase + C::OFF_PIPE + s * stage_bytes;
          // in row-gather mode the gather warps fill A (and its scales) themselves
          ptx::mbar_arrive_expect_tx(fb, (GATHER ? BN * kRowBytes : stage_bytes) + (MX ? (GATHER ? 0 : 512) + sfb_bytes : 0));
          if (!GATHER) ptx::tma_load_3d(st_addr, &tmA, fb, kb * C::BK, tl.row0, 0);
          ptx::tma_load_3d(st_addr + C::A_BYTES, tmb, fb, kb * C::BK, tl.n0, tl.e);
          if constexpr (MX) {
            const int kg = g.K / 128;
            const uint32_t sf_addr = sbase + C::OFF_SF + s * C::SF_STAGE_BYTES;
            if (!GATHER) ptx::bulk_load(sf_addr, g.a_sf + (static_cast<int64_t>(tl.mt) * kg + kb) * 512, 512, fb);
            ptx::bulk_load(sf_addr + 512,
                           g.b_sf + ((static_cast<int64_t>(tl.e) * kg + kb) * (g.n_out / 128) + tl.n0 / 128) * 512,
                           sfb_bytes, fb);
          }
          ++issued;
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {  // let the copies already issued land before the CTA exits
        for (int64_t i = issued - 1; i >= 0 && i >= issued - stages; --i)
          ptx::mbar_wait(full_bar(static_cast<int>(i % stages)), static_cast<uint32_t>((i / stages) & 1),
                         g.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------------ MMA issuer
      const uint32_t idesc = MX ? ptx::idesc_mxf8(kBM, BN) : ptx::idesc_bf16(kBM, BN);
      int s = 0;
      uint32_t ph = 0, kbg = 0;
      int it = 0;
      bool ok = true;
      for (int u = cluster; u < units && ok; u += clusters, ++it) {
        const int acc = num_acc == 2 ? (it & 1) : 0;
        const uint32_t acc_ph = num_acc == 2 ? static_cast<uint32_t>((it >> 1) & 1) : static_cast<uint32_t>(it & 1);
        if (!ptx::mbar_wait(tempty_bar(acc), acc_ph ^ 1u, g.timeout_ns)) { gemm_abort(g, s_abort); break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait(full_bar(s), ph, g.timeout_ns)) { gemm_abort(g, s_abort); ok = false; break; }
          if (GATHER) ptx::fence_proxy_async_smem();  // gathered rows were written by cp.async
          ptx::tc_fence_after();
          const uint32_t a_addr = sbase + C::OFF_PIPE + s * stage_bytes;
          const uint32_t b_addr = a_addr + C::A_BYTES;
          if constexpr (MX) {
            const uint32_t sf_addr = sbase + C::OFF_SF + s * C::SF_STAGE_BYTES;
            const uint32_t sf_col = tmem_base + sf_base_col + (kbg & 1u) * static_cast<uint32_t>(sf_cols);
            ptx::tmem_cp_32x128b_x4(sf_col, ptx::sdesc_sf(sf_addr));
            for (int i = 0; i < BN / 128; ++i)
              ptx::tmem_cp_32x128b_x4(sf_col + 4 + 4 * i, ptx::sdesc_sf(sf_addr + 512 + i * 512));
#pragma unroll
            for (int k = 0; k < C::BK / C::UMMA_K; ++k)
              ptx::mma_mxf8(d_tmem, ptx::sdesc_sw128(a_addr + k * 32), ptx::sdesc_sw128(b_addr + k * 32),
                            ptx::idesc_sf_id(idesc, k), sf_col, sf_col + 4, (kb | k) != 0);
            ++kbg;
          } else {
#pragma unroll
            for (int k = 0; k < C::BK / C::UMMA_K; ++k)
              ptx::mma_bf16(d_tmem, ptx::sdesc_sw128(a_addr + k * 32), ptx::sdesc_sw128(b_addr + k * 32), idesc,
                            (kb | k) != 0);
          }
          ptx::mma_commit_mc(empty_bar(s), both);  // frees the stage in both CTAs (lockstep) once read
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit(tfull_bar(acc));  // accumulator ready for the epilogue
      }
      ptx::mma_commit(drain_bar);  // every MMA issued by this thread has completed
      ptx::mbar_wait(drain_bar, 0, g.timeout_ns);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    EpiStage est{smem + C::OFF_EPI + (warp - 2) * C::EPI_WARP_BYTES,
                 sbase + static_cast<uint32_t>(C::OFF_EPI + (warp - 2) * C::EPI_WARP_BYTES), 0, -1};
    int it = 0;
    for (int u = cluster; u < units; u += clusters, ++it) {
      if (*s_abort) break;
      const UnitTile ut = decode_unit(u, rank, n_tiles_n, BN, s_off, s_mtp, s_odd, g.E_loc);
      const Tile& tl = ut.t;
      const int acc = num_acc == 2 ? (it & 1) : 0;
      const uint32_t acc_ph = num_acc == 2 ? static_cast<uint32_t>((it >> 1) & 1) : static_cast<uint32_t>(it & 1);
      int okw = 0;
      if (lane == 0) okw = ptx::mbar_wait(tfull_bar(acc), acc_ph, g.timeout_ns) ? 1 : 0;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      if (!okw) { if (lane == 0) gemm_abort(g, s_abort); break; }
      (void)ptx::mbar_try_wait(tfull_bar(acc), acc_ph);  // completed phase: acquire for every lane
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      // TMA stores for the bf16 outputs except the ScaledSwiGLU backward's three per block,
      // which measured faster with plain stores (two staging buffers serialise them)
      auto release = [&]() {  // the accumulator may be overwritten by the next tile's MMAs
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty_bar(acc));
      };
      if (ut.valid)
        epilogue_warp<EPI, !MX && EPI != EPI_DSWIGLU>(g, tmO, tl, tbase, BN, q, lane, est, release);
      else
        release();
    }
    if (lane == 0) ptx::bulk_wait_all();  // this warp's TMA stores have completed

  } else if constexpr (GATHER) {
    // ------------------------------------------------------------------ A gather
    // Thread gt copies 16-byte chunk (gt % 8) of the rows gt / 8 + 16 i (i < 8) of each
    // stage's 128 x 128-byte A tile straight from the source rows (cp.async), into the
    // 128-byte swizzled layout a TMA load would produce (chunk c of row r at
    // r * 128 + (c ^ r % 8) * 16), and in MXFP8 mode the 4 scale bytes of row gt into the
    // stage's SF atom.  Each thread's copies of a stage arrive on the stage's full barrier
    // when they land (cp.async.mbarrier.arrive), so the gather runs as far ahead as the
    // ring allows; the MMA issuer fences to the async proxy after its full-barrier wait.
    constexpr int elt = MX ? 1 : 2;
    const int gt = threadIdx.x - kGemmThreads;
    const int chunk = gt & 7, rbase = gt >> 3;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int u = cluster; u < units && ok; u += clusters) {
      const UnitTile ut = decode_unit(u, rank, n_tiles_n, BN, s_off, s_mtp, s_odd, g.E_loc);
      const Tile& tl = ut.t;
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
      const uint8_t* sf_src = nullptr;
      if constexpr (MX) {
        const int64_t tok = gt < tl.rows ? __ldg(g.row_token + tl.row0 + gt) : 0;
        sf_src = g.gx_sf + tok * g.gx_sf_ld;
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
        const uint32_t a_addr = sbase + C::OFF_PIPE + s * stage_bytes;
        const int64_t kbyte = static_cast<int64_t>(kb) * C::BK * elt + chunk * 16;
        const bool kin = kbyte < static_cast<int64_t>(g.K) * elt;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = rbase + 16 * i;
          const bool v = kin && ((live >> i) & 1u);
          ptx::cp_async_16(a_addr + r * kRowBytes + ((chunk ^ (r & 7)) << 4), v ? src[i] + kb * C::BK * elt : g.gx,
                           v ? 16u : 0u);
        }
        if constexpr (MX) {
          const uint32_t sf_addr = sbase + C::OFF_SF + s * C::SF_STAGE_BYTES + (gt & 31) * 16 + (gt >> 5) * 4;
          const bool v = gt < tl.rows;
          ptx::cp_async_4(sf_addr, v ? sf_src + kb * 4 : g.gx_sf, v ? 4u : 0u);
        }
        ptx::cp_async_arrive_noinc(full_bar(s));
        if (++s == stages) { s = 0; ph ^= 1u; }
      }
    }
    ptx::cp_async_wait_all();  // nothing of ours may still be landing when the CTA exits
  } else if constexpr (EPI == EPI_COMBINE) {
    // ------------------------------------------------------------------ combine + zero rows of y
    zero_rows(g, blockIdx.x * 4 + (warp - 6), gridDim.x * 4, lane);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while its peer may still write or arrive into it
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D K-major operand [outer, rows, K] (outer = 1 for a plain matrix), box [1, box_rows, 128 bytes].
bool make_operand_map(CUtensorMap* m, const void* base, bool fp8, uint64_t K, uint64_t rows, uint64_t outer,
                             uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const uint32_t elt = fp8 ? 1 : 2;
  const cuuint64_t dims[3] = {K, rows, outer};
  const cuuint64_t strides[2] = {K * elt, rows * K * elt};
  const cuuint32_t box[3] = {kRowBytes / elt, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_store_map(CUtensorMap* m, void* base, int elt, uint64_t cols, uint64_t rows, uint32_t box_cols,
                    uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc || (elt != 2 && elt != 4)) return false;
  const uint32_t box_bytes = box_cols * static_cast<uint32_t>(elt);
  const CUtensorMapSwizzle sw = box_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : box_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                  : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (sw == CU_TENSOR_MAP_SWIZZLE_NONE) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * static_cast<uint64_t>(elt)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, elt == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base,
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_out_maps(OutMaps* m, const GemmArgs& g) {
  const uint64_t rows = static_cast<uint64_t>(std::max<int64_t>(g.out_rows, 1));
  if (g.out && !make_store_map(&m->out, g.out, 2, static_cast<uint64_t>(g.ld_out), rows, 32, 32)) return false;
  if (g.out2 && !make_store_map(&m->out2, g.out2, 2, static_cast<uint64_t>(g.n_out), rows, 32, 32)) return false;
  return true;
}

// A: the permuted rows [a_rows, K] (TMA), or unused (nullptr) in row-gather mode.
template <bool MX, int EPI, bool GATHER = false>
static cudaError_t launch_gemm_inst(const void* A, int64_t a_rows, const void* B, const GemmArgs& g,
                                    cudaStream_t st) {
  using C = GemmSmem<MX>;
  constexpr int threads = kGemmThreads + extra_threads<EPI, GATHER>();
  CUtensorMap ta = {};
  BMaps tb;
  if (!GATHER && !make_operand_map(&ta, A, MX, g.K, a_rows, 1, kBM)) return cudaErrorInvalidValue;
  if (!make_operand_map(&tb.b256, B, MX, g.K, g.n_out, g.E_loc, 256)) return cudaErrorInvalidValue;
  if (!make_operand_map(&tb.b128, B, MX, g.K, g.n_out, g.E_loc, 128)) return cudaErrorInvalidValue;
  if (!make_operand_map(&tb.b64, B, MX, g.K, g.n_out, g.E_loc, 64)) return cudaErrorInvalidValue;
  OutMaps tmo;
  memset(&tmo, 0, sizeof(tmo));
  if (!MX && !make_out_maps(&tmo, g)) return cudaErrorInvalidValue;
  auto kern = tc_grouped_gemm_kernel<MX, EPI, GATHER>;
  // Once per device: opt in to > 48 KB of dynamic shared memory and size the grid to the
  // clusters of two that can be resident at once (keeps later launches, including ones
  // recorded into a CUDA graph, free of non-launch API calls).
  static int grid_of[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int grid = (dev >= 0 && dev < 64) ? grid_of[dev] : 0;
  if (grid == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms()));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) {
      (void)cudaGetLastError();
      clusters = num_sms() / 2;
    }
    grid = 2 * std::min(clusters, num_sms() / 2);
    if (dev >= 0 && dev < 64) grid_of[dev] = grid;
  }
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(threads), C::SMEM_BYTES, st, ta, tb, tmo, g);
}

static GemmArgs base_args(const int32_t* offsets, int E_loc, int32_t* err, uint64_t timeout_ns) {
  GemmArgs g{};
  g.offsets = offsets;
  g.E_loc = E_loc;
  g.err = err;
  g.timeout_ns = timeout_ns;
  return g;
}

cudaError_t launch_pair_gemm(const void* A, int64_t a_rows, const void* B, const GemmArgs& g, bool swiglu, bool mx,
                             cudaStream_t st);
cudaError_t launch_pair_gemm_combine(const void* A, int64_t a_rows, const void* B, const GemmArgs& g, bool mx,
                                     cudaStream_t st);
cudaError_t launch_pair_gemm1_gather(const void* B, const GemmArgs& g, cudaStream_t st);
cudaError_t launch_swap_gemm1(const void* perm_x, int64_t rows, const void* Wgu, const GemmArgs& g, bool mx, int nt_max,
                              cudaStream_t st);
cudaError_t launch_swap_gemm1_gather(const void* Wgu, const GemmArgs& g, int nt_max, cudaStream_t st);
cudaError_t launch_swap_gemm2(const void* h, int64_t rows, const void* Wd, const GemmArgs& g, bool mx, bool combine,
                              int nt_max, cudaStream_t st);

// Kernel shape of the grouped GEMM launchers below: 0 = 1-CTA kernel (gemm_tc.cu), 1 =
// token-major CTA pairs (gemm_tc_pair.cu), kShapeSwapMin and above = the swapped-operand
// pair kernel (gemm_tc_swap.cu) with that many tokens per tile.
constexpr int kShapeSwapMin = 64;

// GEMM1 + fused scaled SwiGLU on the tensor cores.
//   bf16:  perm_x bf16 [N_cap, d] -> h bf16 [N_cap, f]
//   mxfp8: perm_x E4M3 [N_cap, d] + SF -> h E4M3 [N_cap, f] + SF
// The swapped-operand kernel does not write g/u (gu_save): with gu_save the token-major
// kernels run.
cudaError_t launch_tc_gemm1(const void* perm_x, const uint8_t* perm_sf, const int32_t* offsets, const float* row_prob,
                            int64_t N_cap, int E_loc, int d, int f, bool mx, int shape, const void* Wgu,
                            const uint8_t* Wgu_sf, void* h, uint8_t* h_sf, int32_t* err, uint64_t timeout_ns,
                            void* gu_save, cudaStream_t st) {
  GemmArgs g = base_args(offsets, E_loc, err, timeout_ns);
  g.out2 = mx ? nullptr : gu_save;
  g.n_out = 2 * f;
  g.K = d;
  g.out = h;
  g.ld_out = f;
  g.out_rows = N_cap;
  g.out_sf = h_sf;
  g.row_prob = row_prob;
  g.a_sf = perm_sf;
  g.b_sf = Wgu_sf;
  if (shape >= kShapeSwapMin && !g.out2) return launch_swap_gemm1(perm_x, N_cap, Wgu, g, mx, shape, st);
  if (shape == 1) return launch_pair_gemm(perm_x, N_cap, Wgu, g, true, mx, st);
  if (mx) return launch_gemm_inst<true, EPI_SWIGLU_MX>(perm_x, N_cap, Wgu, g, st);
  return launch_gemm_inst<false, EPI_SWIGLU_BF16>(perm_x, N_cap, Wgu, g, st);
}

// Per-tensor FP8 GEMM1: the block-scaled mainloop (x rows and weights in the MXFP8
// layouts, every scale of a tensor equal) with the bf16 scaled-SwiGLU epilogue, which also
// accumulates the largest |h| into *h_amax (fp32 bits; zeroed by the caller) for the
// per-tensor quantisation of h that GEMM2 reads.
cudaError_t launch_tc_gemm1_fp8(const void* perm_x, const uint8_t* perm_sf, const int32_t* offsets,
                                const float* row_prob, int64_t N_cap, int E_loc, int d, int f, const void* Wgu,
                                const uint8_t* Wgu_sf, void* h_bf16, uint32_t* h_amax, int32_t* err,
                                uint64_t timeout_ns, cudaStream_t st) {
  GemmArgs g = base_args(offsets, E_loc, err, timeout_ns);
  g.n_out = 2 * f;
  g.K = d;
  g.out = h_bf16;
  g.ld_out = f;
  g.out_rows = N_cap;
  g.row_prob = row_prob;
  g.a_sf = perm_sf;
  g.b_sf = Wgu_sf;
  g.amax = h_amax;
  return launch_gemm_inst<true, EPI_SWIGLU_BF16>(perm_x, N_cap, Wgu, g, st);
}

// GEMM1 + fused scaled SwiGLU with A gathered from the token rows: row r of the
// expert-ordered operand is x row row_src_token[r] (bf16 [T, d]; MXFP8: E4M3 [T, d] with
// E8M0 scales x_sf [T, d / 32]), so no permuted copy of x is ever written.
// shape (bf16 only): the token-major CTA-pair kernel (1) or the swapped-operand one (>=
// kShapeSwapMin) instead of the 1-CTA kernel (0).
cudaError_t launch_tc_gemm1_gather(const void* x, const uint8_t* x_sf, const int32_t* row_src_token,
                                   const int32_t* offsets, const float* row_prob, int64_t N_cap, int E_loc, int d,
                                   int f, bool mx, int shape, const void* Wgu, const uint8_t* Wgu_sf, void* h,
                                   uint8_t* h_sf, int32_t* err, uint64_t timeout_ns, void* gu_save, cudaStream_t st) {
  GemmArgs g = base_args(offsets, E_loc, err, timeout_ns);
  g.out2 = mx ? nullptr : gu_save;
  g.n_out = 2 * f;
  g.K = d;
  g.out = h;
  g.ld_out = f;
  g.out_rows = N_cap;
  g.out_sf = h_sf;
  g.row_prob = row_prob;
  g.b_sf = Wgu_sf;
  g.gx = static_cast<const uint8_t*>(x);
  g.gx_ld = static_cast<int64_t>(d) * (mx ? 1 : 2);
  g.row_token = row_src_token;
  g.gx_sf = x_sf;
  g.gx_sf_ld = d / 32;
  if (mx) return launch_gemm_inst<true, EPI_SWIGLU_MX, true>(nullptr, 0, Wgu, g, st);
  if (shape >= kShapeSwapMin && !g.out2) return launch_swap_gemm1_gather(Wgu, g, shape, st);
  if (shape == 1) return launch_pair_gemm1_gather(Wgu, g, st);
  return launch_gemm_inst<false, EPI_SWIGLU_BF16, true>(nullptr, 0, Wgu, g, st);
}

// Backward, bf16: dh = dy_row W_down^T for every routed row (dy_rows = dy in routed-row
// order [N_cap, d], loaded by TMA; B = W_down in the user layout [E_loc, f, d], K-major
// over d) with the ScaledSwiGLU backward fused into the epilogue (dg/du, h and partial dp).
cudaError_t launch_tc_dswiglu(const void* dy_rows, const int32_t* offsets, const float* row_prob, int64_t N_cap,
                              int E_loc, int d, int f, const void* W_down, const void* gu, void* dgu, void* h,
                              float* dp_part, int32_t* err, uint64_t timeout_ns, cudaStream_t st) {
  GemmArgs g = base_args(offsets, E_loc, err, timeout_ns);
  g.n_out = f;
  g.K = d;
  g.out = dgu;
  g.ld_out = 2 * f;
  g.out_rows = N_cap;
  g.out2 = h;
  g.dp_part = dp_part;
  g.aux = static_cast<const uint16_t*>(gu);
  g.row_prob = row_prob;
  return launch_gemm_inst<false, EPI_DSWIGLU>(dy_rows, N_cap, W_down, g, st);
}

// Backward, MXFP8: dh = dy_row W_down^T on the block-scaled tensor cores (dy rows E4M3 [N_cap,
// d] with scales in the activation SF tile layout, K = d; W_down E4M3 [E_loc, f, d] with its
// weight SF tile layout), the ScaledSwiGLU backward fused into the epilogue as in bf16.
cudaError_t launch_tc_dswiglu_mx(const void* dy_q, const uint8_t* dy_sf, const int32_t* offsets,
                                 const float* row_prob, int64_t N_cap, int E_loc, int d, int f, const void* Wd_q,
                                 const uint8_t* Wd_sf, const void* gu, void* dgu, void* h, float* dp_part, int32_t* err,
                                 uint64_t timeout_ns, cudaStream_t st) {
  GemmArgs g = base_args(offsets, E_loc, err, timeout_ns);
  g.n_out = f;
  g.K = d;
  g.out = dgu;
  g.ld_out = 2 * f;
  g.out_rows = N_cap;
  g.out2 = h;
  g.dp_part = dp_part;
  g.aux = static_cast<const uint16_t*>(gu);
  g.row_prob = row_prob;
  g.a_sf = dy_sf;
  g.b_sf = Wd_sf;
  return launch_gemm_inst<true, EPI_DSWIGLU>(dy_q, N_cap, Wd_q, g, st);
}

// MXFP8 grouped GEMM with a bf16 store: out [a_rows, n_out] = A [rows, K] (E4M3, activation SF
// tile layout) times B^T per expert (E4M3 [E_loc, n_out, K], weight SF tile layout).
cudaError_t launch_tc_gemm_store_mx(const void* A, const uint8_t* a_sf, int64_t a_rows, const int32_t* offsets,
                                    int E_loc, int K, int n_out, const void* B, const uint8_t* b_sf, void* out,
                                    int32_t* err, uint64_t timeout_ns, cudaStream_t st) {
  GemmArgs g = base_args(offsets, E_loc, err, timeout_ns);
  g.n_out = n_out;
  g.K = K;
  g.out = out;
  g.ld_out = n_out;
  g.out_rows = a_rows;
  g.a_sf = a_sf;
  g.b_sf = b_sf;
  return launch_gemm_inst<true, EPI_STORE_BF16>(A, a_rows, B, g, st);
}

// Backward, bf16: dx rows = dg/du [N_cap, 2f] (packed order) times the transposed gate/up
// weights WguT [E_loc, d, 2f] (same packed order along K) -> [N_cap, d].
cudaError_t launch_tc_gemm_store(const void* A, int64_t a_rows, const int32_t* offsets, int E_loc, int K, int n_out,
                                 const void* B, void* out, int32_t* err, uint64_t timeout_ns, cudaStream_t st) {
  GemmArgs g = base_args(offsets, E_loc, err, timeout_ns);
  g.n_out = n_out;
  g.K = K;
  g.out = out;
  g.ld_out = n_out;
  g.out_rows = a_rows;
  return launch_gemm_inst<false, EPI_STORE_BF16>(A, a_rows, B, g, st);
}

// GEMM2 with the direct part of the unpermute + combine: h [N_cap, f] (bf16, or E4M3 +
// SF) -> y rows of the tokens with at most one local slot (their row, or zeros), Y2
// [N_cap, d] rows of the tokens with several (summed afterwards by the combine kernel).
cudaError_t launch_tc_gemm2_combine(const void* h, const uint8_t* h_sf, const int32_t* offsets, int64_t N_cap,
                                    int E_loc, int d, int f, bool mx, int shape, const void* Wd, const uint8_t* Wd_sf,
                                    void* Y2, const int32_t* row_src_token, const int32_t* tok_nloc, int T, void* y,
                                    int32_t* err, uint64_t timeout_ns, cudaStream_t st) {
  GemmArgs g = base_args(offsets, E_loc, err, timeout_ns);
  g.n_out = d;
  g.K = f;
  g.out = Y2;
  g.ld_out = d;
  g.out_rows = N_cap;
  g.a_sf = h_sf;
  g.b_sf = Wd_sf;
  g.row_token = row_src_token;
  g.tok_nloc = tok_nloc;
  g.y = y;
  g.T = T;
  if (shape >= kShapeSwapMin) return launch_swap_gemm2(h, N_cap, Wd, g, mx, true, shape, st);
  if (shape == 1) return launch_pair_gemm_combine(h, N_cap, Wd, g, mx, st);
  if (mx) return launch_gemm_inst<true, EPI_COMBINE>(h, N_cap, Wd, g, st);
  return launch_gemm_inst<false, EPI_COMBINE>(h, N_cap, Wd, g, st);
}

// GEMM2 on the tensor cores: h [N_cap, f] (bf16, or E4M3 + SF) -> Y2 bf16 [N_cap, d].
cudaError_t launch_tc_gemm2(const void* h, const uint8_t* h_sf, const int32_t* offsets, int64_t N_cap, int E_loc, int d,
                            int f, bool mx, int shape, const void* Wd, const uint8_t* Wd_sf, void* Y2, int32_t* err,
                            uint64_t timeout_ns, cudaStream_t st) {
  GemmArgs g = base_args(offsets, E_loc, err, timeout_ns);
  g.n_out = d;
  g.K = f;
  g.out = Y2;
  g.ld_out = d;
  g.out_rows = N_cap;
  g.a_sf = h_sf;
  g.b_sf = Wd_sf;
  if (shape >= kShapeSwapMin) return launch_swap_gemm2(h, N_cap, Wd, g, mx, false, shape, st);
  if (shape == 1) return launch_pair_gemm(h, N_cap, Wd, g, false, mx, st);
  if (mx) return launch_gemm_inst<true, EPI_STORE_BF16>(h, N_cap, Wd, g, st);
  return launch_gemm_inst<false, EPI_STORE_BF16>(h, N_cap, Wd, g, st);
}

}  // namespace moe
