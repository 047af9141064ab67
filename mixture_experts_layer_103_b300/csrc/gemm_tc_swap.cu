// Grouped GEMM with swapped operands on CTA pairs, for experts that hold few rows.
//
// Same computation as the kernels in gemm_tc.cu and gemm_tc_pair.cu ("Efficient MoE
// training for biological foundation models", section "GroupedLinear Optimizes Expert
// Computation": per-expert GEMMs run as one grouped operation, ScaledSwiGLU fused after
// the first), with the roles of the operands exchanged: the MMA's M side is the expert's
// packed weight rows and its N side the expert's tokens, so the accumulator holds the
// transposed tile (one TMEM lane per output feature, one column per token).
//   * A tile is (expert, chunk of up to nt_max of its tokens, 256 weight rows).  CTA r of
//     the pair stages weight rows [128 r, 128 r + 128) of the tile and its half of the
//     chunk's token rows; the leader issues tcgen05.mma.cta_group::2 with M = 256 and
//     N = the chunk's token count rounded up to 16 (two MMAs, N = 256 and the rest, when
//     the chunk holds more than 256 tokens).
//   * Why: on expert slices that hold a few hundred rows per expert (the pages' EP64
//     workloads, "Wide-EP ... NVIDIA" explainer, section on arithmetic intensity and
//     tokens per expert) the weights dominate the bytes.  A token-major tile pads each
//     expert's rows to 128 or 256 and re-streams the weights for every such tile; here an
//     expert's tokens are padded to 16, one tile covers up to nt_max of them, and each SM
//     lands 128 weight rows plus half the chunk's token rows per K step.
//   * GEMM1 epilogue: packed weight rows interleave 32 gate and 32 up rows, so in each CTA
//     TMEM lane quarters 0 / 1 hold the gate / up values of 32 features and quarters 2 / 3
//     those of the next 32.  The two warps of a quarter pair swap half of each 32-token
//     block through shared memory (named barrier of the two warps) and each finishes
//     h = p * silu(g) * u for 16 tokens; bf16 h, or MXFP8 h with the 32-feature block's
//     scale from a warp-wide max (the 32 lanes of a warp are the block).
//   * GEMM2 epilogue: bf16 rows of Y2, or (combine mode) the token's y row when the token
//     has a single local slot, with zero rows of y from 4 extra warps.
//   * Outputs leave through a per-warp shared-memory transpose so that every store
//     instruction writes whole 64-byte (bf16) or 32-byte (E4M3) row segments.
//   * The token rows come by TMA (permuted copy, in boxes of 128 / 64 / 32 / 16 / 8 rows
//     so that only the chunk's rows are read), or, for the bf16 GEMM1, by 4 gather warps
//     straight from x (cp.async into the 128-byte swizzled layout, relayed to the leader
//     as in the token-major pair kernel).
//   * Two accumulators in TMEM when a tile holds at most 256 tokens (MXFP8: 128), so the
//     epilogue of a tile overlaps the next tile's MMAs; one (up to 384 columns, MXFP8 scales
//     beside it) for larger tiles, whose epilogue only the TMA ring overlaps.
// Every wait is bounded; on a timeout the kernel records MOE_ERR_TIMEOUT and exits.
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"

namespace moe {

constexpr int kSwapBM = 256;                     // weight rows of a tile (128 per CTA)
constexpr int kSwapMaxStages = 8;
constexpr int kSwapMaxEloc = 256;                // experts of a launch (shared-memory tables)
constexpr int kSwapMaxTokens = 384;              // tokens of a tile (MMA N: 256 + 128)
constexpr int kSwapABytes = 128 * kRowBytes;     // this CTA's 128 weight rows per stage
constexpr int kSwapXchFloats = 2 * 16 * 32;      // one exchange buffer: (g | u) x 16 tokens x 32 lanes
constexpr int kSwapXchBytes = 2 * 2 * kSwapXchFloats * 4;  // 2 quarter pairs x 2 buffers
constexpr int kSwapEpiWarp = 32 * 64;            // transpose staging: 32 tokens x 64 bytes
constexpr int kSwapSfStage = 512 + 3 * 512;      // MXFP8: A's scale atom + up to 3 of B's

struct SwapLayout {
  static constexpr int OFF_XCH = 0;
  static constexpr int OFF_EPI = OFF_XCH + kSwapXchBytes;
  static constexpr int OFF_BAR = OFF_EPI + 4 * kSwapEpiWarp;
  // full, empty, gathered (per stage); tmem_full[2], tmem_empty[2], drain
  static constexpr int NUM_BARS = 3 * kSwapMaxStages + 5;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_TAB = OFF_MISC + 16;
  static constexpr int TAB_BYTES = 3 * (kSwapMaxEloc + 1) * 4;  // s_off, s_ctp, s_mtp128
  static constexpr int FIXED = (OFF_TAB + TAB_BYTES + 1023) / 1024 * 1024;
};
constexpr int kSwapSmemMax = 232448;

// The token-row maps: boxes of 128, 64, 32, 16 and 8 rows of 128 bytes.
struct SwapBMaps {
  CUtensorMap m[5];
};
struct SwapSfMaps {
  CUtensorMap w, act;  // weight SF atoms (A's scales), activation SF atoms (B's)
};

template <int EPI, bool GATHER>
constexpr int swap_extra_threads() {
  return GATHER ? kGatherThreads : EPI == EPI_COMBINE ? kZeroThreads : 0;
}

// Token counts of a tile: N (MMA columns), N1 / N2 of the two MMAs, and each CTA's share
// b1 / b2 of their B rows.
struct SwapGeo {
  int N, N1, N2, b1, b2;
};
__device__ __forceinline__ SwapGeo swap_geo(int rows) {
  SwapGeo q;
  q.N = (rows + 15) & ~15;
  q.N1 = min(q.N, 256);
  q.N2 = q.N - q.N1;
  q.b1 = q.N1 / 2;
  q.b2 = q.N2 / 2;
  return q;
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Ties the 32 registers of a TMEM load to the point after tcgen05.wait::ld, so that no use
// of them is scheduled before the wait.
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                    "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                    "+r"(r[15]));
  asm volatile("" : "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]),
                    "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                    "+r"(r[30]), "+r"(r[31]));
}

// Runs body(c, v, pre(c)) over the tile's 32-column blocks c = 0, 32, ... < N of this
// warp's TMEM lanes, with the next block's TMEM load (and pre, e.g. a global load) in flight
// while body works on the current one; release() right after the last block's load.
template <typename Pre, typename Body, typename Release>
__device__ __forceinline__ void swap_tmem_blocks(uint32_t tb, int N, Pre&& pre, Body&& body, Release&& release) {
  uint32_t va[32], vb[32];
  ptx::tmem_ld32(tb, va);
  auto pa = pre(0);
  auto pb = pa;
  ptx::tmem_ld_wait();
  reg_fence32(va);
#pragma unroll 1
  for (int c = 0;; c += 64) {
    if (c + 32 < N) {
      ptx::tmem_ld32(tb + c + 32, vb);
      pb = pre(c + 32);
    } else {
      release();
    }
    body(c, va, pa);
    if (c + 32 >= N) break;
    ptx::tmem_ld_wait();
    reg_fence32(vb);
    if (c + 64 < N) {
      ptx::tmem_ld32(tb + c + 64, va);
      pa = pre(c + 64);
    } else {
      release();
    }
    body(c + 32, vb, pb);
    if (c + 64 >= N) break;
    ptx::tmem_ld_wait();
    reg_fence32(va);
  }
}

// GEMM1 epilogue of one warp: 32 features (lanes) of either the gate (q even) or the up
// (q odd) half of a quarter pair, over the tile's N token columns.
template <bool MXOUT, typename Release>
__device__ __forceinline__ void swap_epi_swiglu(const GemmArgs& g, const Tile& tl, int N, uint32_t tb, int q, int lane,
                                                int rank, float* xch, uint8_t* est, const int* s_off,
                                                const int* s_mtp128, Release&& release) {
  const bool up = q & 1;
  const int pi = q >> 1;
  const int fdim = g.n_out / 2;
  const int fbase = (tl.n0 + 128 * rank) / 2 + 32 * pi;  // first h column of this warp's lanes
  const bool fvalid = fbase < fdim;                        // fdim is a multiple of 32
  // routing probability of token tok0 + lane (lane < 16) of the block at c
  auto prob = [&](int c) {
    const int tok = c + (up ? 16 : 0) + lane;
    return (lane < 16 && tok < tl.rows) ? __ldg(g.row_prob + tl.row0 + tok) : 0.0f;
  };
  auto body = [&](int c, const uint32_t (&v)[32], float pl) {
    float* X = xch + ((c >> 5) & 1) * kSwapXchFloats;  // [0]: gate of tokens 16..31, [1]: up of tokens 0..15
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (!up) X[j * 32 + lane] = __uint_as_float(v[16 + j]);
      else X[(16 + j) * 32 + lane] = __uint_as_float(v[j]);
    }
    named_bar_sync(1 + pi, 64);
    const int tok0 = c + (up ? 16 : 0);  // this warp's 16 tokens
    const int nvalid = tl.rows - tok0;   // tokens of them inside the chunk (may be <= 0)
    float h[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float gg = up ? X[j * 32 + lane] : __uint_as_float(v[j]);
      const float uu = up ? __uint_as_float(v[16 + j]) : X[(16 + j) * 32 + lane];
      const float p = __shfl_sync(0xffffffffu, pl, j);
      h[j] = p * __fdividef(gg, 1.0f + __expf(-gg)) * uu;
    }
    if constexpr (!MXOUT) {
      uint16_t* s16 = reinterpret_cast<uint16_t*>(est);
#pragma unroll
      for (int j = 0; j < 16; ++j) s16[j * 32 + lane] = static_cast<uint16_t>(pack_bf16x2(h[j], 0.0f) & 0xFFFFu);
      __syncwarp();
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int j = it * 8 + lane / 4, ch = lane % 4;
        if (j < nvalid && fvalid) {
          const uint4 val = *reinterpret_cast<const uint4*>(est + j * 64 + ch * 16);
          *reinterpret_cast<uint4*>(static_cast<uint8_t*>(g.out) + (static_cast<int64_t>(tl.row0) + tok0 + j) * g.ld_out * 2 +
                                    static_cast<int64_t>(fbase) * 2 + ch * 16) = val;
        }
      }
      __syncwarp();
    } else {
      int xs = 0;  // lane j keeps the scale exponent of token j
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float amax = fabsf(h[j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int Xe = mx_exponent(amax);
        est[j * 32 + lane] = static_cast<uint8_t>(e4m3x2(h[j] * mx_inv_scale(Xe), 0.0f) & 0xFFu);
        if (lane == j) xs = Xe;
      }
      __syncwarp();
      {
        const int j = lane / 2, ch = lane % 2;
        if (j < nvalid && fvalid) {
          const uint4 val = *reinterpret_cast<const uint4*>(est + j * 32 + ch * 16);
          *reinterpret_cast<uint4*>(static_cast<uint8_t*>(g.out) + (static_cast<int64_t>(tl.row0) + tok0 + j) * g.ld_out +
                                    fbase + ch * 16) = val;
        }
      }
      if (lane < 16 && lane < nvalid && fvalid) {
        const int srow = tl.row0 + tok0 + lane - s_off[tl.e];  // row within the expert's segment
        g.out_sf[sf_act_offset(s_mtp128[tl.e] + srow / 128, srow % 128, fbase, fdim)] = static_cast<uint8_t>(xs + 127);
      }
      __syncwarp();
    }
  };
  swap_tmem_blocks(tb, N, prob, body, release);
}

// GEMM2 epilogue of one warp: output columns n0w .. n0w + 31 (lanes) over N token columns,
// to Y2 rows, or (COMBINE) to the token's y row when it has a single local slot.
template <bool COMBINE, typename Release>
__device__ __forceinline__ void swap_epi_store(const GemmArgs& g, const Tile& tl, int N, uint32_t tb, int n0w, int lane,
                                               uint8_t* est, Release&& release) {
  uint16_t* s16 = reinterpret_cast<uint16_t*>(est);
  const int64_t ld2 = g.ld_out * 2;
  const int ch = lane % 4;
  const bool col_ok = n0w + ch * 8 < g.n_out;
  // COMBINE: token of each row this lane stores in the block at c (rows c + it * 8 + lane / 4)
  auto tokens = [&](int c) {
    int4 t = make_int4(-1, -1, -1, -1);
    if constexpr (COMBINE) {
      const int r0 = c + lane / 4;
      if (r0 < tl.rows) t.x = __ldg(g.row_token + tl.row0 + r0);
      if (r0 + 8 < tl.rows) t.y = __ldg(g.row_token + tl.row0 + r0 + 8);
      if (r0 + 16 < tl.rows) t.z = __ldg(g.row_token + tl.row0 + r0 + 16);
      if (r0 + 24 < tl.rows) t.w = __ldg(g.row_token + tl.row0 + r0 + 24);
    }
    return t;
  };
  auto body = [&](int c, const uint32_t (&v)[32], int4 tk) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      s16[j * 32 + lane] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(v[j]), 0.0f) & 0xFFFFu);
    __syncwarp();
    const int tok[4] = {tk.x, tk.y, tk.z, tk.w};
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int j = it * 8 + lane / 4;
      if (c + j < tl.rows && col_ok) {
        const int64_t row = static_cast<int64_t>(tl.row0) + c + j;
        uint8_t* dst = static_cast<uint8_t*>(g.out) + row * ld2;
        if constexpr (COMBINE) {
          if (__ldg(g.tok_nloc + tok[it]) == 1)
            dst = static_cast<uint8_t*>(g.y) + static_cast<int64_t>(tok[it]) * g.n_out * 2;
        }
        *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(n0w + ch * 8) * 2) =
            *reinterpret_cast<const uint4*>(est + j * 64 + ch * 16);
      }
    }
    __syncwarp();
  };
  swap_tmem_blocks(tb, N, tokens, body, release);
}

template <bool MX, int EPI, bool GATHER>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads + swap_extra_threads<EPI, GATHER>(), 1)
    tc_swap_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ SwapBMaps tmB,
                        const __grid_constant__ SwapSfMaps tmS, const GemmArgs g) {
  static_assert(!(MX && GATHER), "the MXFP8 token rows come by TMA");
  using L = SwapLayout;
  constexpr int BK = MX ? 128 : 64;  // K elements per stage (128 bytes per row)
  constexpr bool SWIGLU = EPI == EPI_SWIGLU_BF16 || EPI == EPI_SWIGLU_MX;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int S = g.sw_stages;
  const uint32_t SB = static_cast<uint32_t>(g.sw_stage_bytes);
  const uint32_t ring = sbase + L::FIXED;
  const uint32_t sfring = ring + static_cast<uint32_t>(S) * SB;
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kSwapMaxStages + s); };
  auto gath_bar = [&](int s) { return bar0 + 8u * (2 * kSwapMaxStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (3 * kSwapMaxStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (3 * kSwapMaxStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (3 * kSwapMaxStages + 4);
  // accumulators in TMEM: two (columns 0 and 256, double-buffered: the epilogue of a tile
  // overlaps the next tile's MMAs) when a tile holds at most 256 tokens (MXFP8: 128, the
  // scale columns sit at 384), else one of up to 384 columns
  const int nacc = g.nt_max <= (MX ? 128 : 256) ? 2 : 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  int* s_off = reinterpret_cast<int*>(smem + L::OFF_TAB);
  int* s_ctp = s_off + kSwapMaxEloc + 1;
  int* s_mtp128 = s_ctp + kSwapMaxEloc + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
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
    ptx::prefetch_tmap(&tmA);
    if (!GATHER)
      for (int i = 0; i < 5; ++i) ptx::prefetch_tmap(&tmB.m[i]);
    if (MX) {
      ptx::prefetch_tmap(&tmS.w);
      ptx::prefetch_tmap(&tmS.act);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish_pair();
  }
  pdl_wait();  // offsets, token rows and scales come from the previous kernels
  if (warp == 2) {
    build_mtile_prefix(g.offsets, g.E_loc, g.nt_max, s_off, s_ctp);
    if (MX) build_mtile_prefix(g.offsets, g.E_loc, 128, s_off, s_mtp128);
  }
  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int n_fblk = (g.n_out + kSwapBM - 1) / kSwapBM;
  const int total = s_ctp[g.E_loc] * n_fblk;
  const int num_kb = (g.K + BK - 1) / BK;
  auto tile_at = [&](int t) { return decode_tile(t, n_fblk, kSwapBM, s_off, s_ctp, g.E_loc, g.nt_max); };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer (both CTAs)
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      const int kg = g.K / 128;
      const uint32_t fb0 = ptx::mapa_shared(full_bar(0), 0);  // the leader's full barriers, cluster addresses
      for (int t = pair; t < total && ok; t += npairs) {
        const Tile tl = tile_at(t);
        const SwapGeo q = swap_geo(tl.rows);
        const int a_row = tl.n0 + 128 * rank;
        const int r1 = tl.row0 + rank * q.b1;        // this CTA's token rows of the first MMA
        const int r2 = tl.row0 + 256 + rank * q.b2;  // and of the second
        const int nsfb = (q.N + 127) / 128;
        const int mt128 = MX ? s_mtp128[tl.e] + (tl.row0 - s_off[tl.e]) / 128 : 0;
        const uint32_t bytes = 2u * kSwapABytes + (GATHER ? 0u : static_cast<uint32_t>(q.N) * kRowBytes) +
                               (MX ? 2u * 512u * static_cast<uint32_t>(1 + nsfb) : 0u);
        // this CTA's token rows as boxes: bit j of plan = one box of 8 << j rows (b1, b2 are
        // multiples of 8, b1 <= 128, b2 <= 64); a full 128-row first part is one box
        const uint32_t plan1 = static_cast<uint32_t>(q.b1) >> 3, plan2 = static_cast<uint32_t>(q.b2) >> 3;
        const bool one_box = plan1 == 16u && plan2 == 0u;
        if (*s_abort) { ok = false; break; }  // another role gave up: stop at a tile boundary
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait(empty_bar(s), ph ^ 1u, g.timeout_ns)) { gemm_abort(g, s_abort); ok = false; break; }
          const uint32_t fb = fb0 + 8u * static_cast<uint32_t>(s);
          if (leader) ptx::mbar_arrive_expect_tx(full_bar(s), bytes);
          const uint32_t st_a = ring + static_cast<uint32_t>(s) * SB;
          ptx::tma_load_3d_pair(st_a, &tmA, fb, kb * BK, a_row, tl.e);
          if constexpr (!GATHER) {
            const uint32_t dst0 = st_a + kSwapABytes;
            if (one_box) {
              ptx::tma_load_3d_pair(dst0, &tmB.m[0], fb, kb * BK, r1, 0);
            } else {
              uint32_t dst = dst0;
              int row = r1;
#pragma unroll
              for (int j = 4; j >= 0; --j)
                if ((plan1 >> j) & 1u) {
                  ptx::tma_load_3d_pair(dst, &tmB.m[4 - j], fb, kb * BK, row, 0);
                  dst += (8u << j) * kRowBytes;
                  row += 8 << j;
                }
              row = r2;
#pragma unroll
              for (int j = 3; j >= 0; --j)
                if ((plan2 >> j) & 1u) {
                  ptx::tma_load_3d_pair(dst, &tmB.m[4 - j], fb, kb * BK, row, 0);
                  dst += (8u << j) * kRowBytes;
                  row += 8 << j;
                }
            }
          }
          if constexpr (MX) {
            const uint32_t sf = sfring + static_cast<uint32_t>(s) * kSwapSfStage;
            ptx::tma_load_2d_pair(sf, &tmS.w, fb, 0, (tl.e * kg + kb) * (g.n_out / 128) + tl.n0 / 128 + rank);
            for (int a = 0; a < nsfb; ++a)
              ptx::tma_load_2d_pair(sf + 512u * (1 + a), &tmS.act, fb, 0, (mt128 + a) * kg + kb);
          }
          ++issued;
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok && leader) {  // let the copies already issued land before the pair exits
        for (int64_t i = issued - 1; i >= 0 && i >= issued - S; --i)
          ptx::mbar_wait(full_bar(static_cast<int>(i % S)), static_cast<uint32_t>((i / S) & 1), g.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------------ MMA issuer (leader)
      int s = 0;
      uint32_t ph = 0, kbg = 0;
      int it = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs, ++it) {
        const Tile tl = tile_at(t);
        const SwapGeo q = swap_geo(tl.rows);
        const int nsfb = (q.N + 127) / 128;
        const uint32_t id1 = MX ? ptx::idesc_mxf8(kSwapBM, q.N1) : ptx::idesc_bf16(kSwapBM, q.N1);
        const uint32_t id2 = MX ? ptx::idesc_mxf8(kSwapBM, q.N2 > 0 ? q.N2 : 16) : ptx::idesc_bf16(kSwapBM, q.N2 > 0 ? q.N2 : 16);
        const int acc = nacc == 2 ? (it & 1) : 0;
        const uint32_t acc_ph = static_cast<uint32_t>(nacc == 2 ? (it >> 1) & 1 : it & 1);
        if (!ptx::mbar_wait(tempty_bar(acc), acc_ph ^ 1u, g.timeout_ns)) { gemm_abort(g, s_abort); break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
        for (int kb = 0; kb < num_kb; ++kb) {
          const bool got = GATHER ? ptx::mbar_wait_cluster(full_bar(s), ph, g.timeout_ns)
                                  : ptx::mbar_wait(full_bar(s), ph, g.timeout_ns);
          if (!got) { gemm_abort(g, s_abort); ok = false; break; }
          if (GATHER) ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint32_t a_addr = ring + static_cast<uint32_t>(s) * SB;
          const uint32_t b_addr = a_addr + kSwapABytes;
          const uint32_t b2_addr = b_addr + static_cast<uint32_t>(q.b1) * kRowBytes;
          if constexpr (MX) {
            const uint32_t sf = sfring + static_cast<uint32_t>(s) * kSwapSfStage;
            const uint32_t sf_col = tmem_base + kSwapMaxTokens + (kbg & 1u) * 16u;
            ptx::tmem_cp_32x128b_x4_pair(sf_col, ptx::sdesc_sf(sf));
            for (int a = 0; a < nsfb; ++a)
              ptx::tmem_cp_32x128b_x4_pair(sf_col + 4u * (1 + a), ptx::sdesc_sf(sf + 512u * (1 + a)));
#pragma unroll
            for (int k = 0; k < BK / 32; ++k) {
              ptx::mma_mxf8_pair(d_tmem, ptx::sdesc_sw128(a_addr + k * 32), ptx::sdesc_sw128(b_addr + k * 32),
                                 ptx::idesc_sf_id(id1, k), sf_col, sf_col + 4, (kb | k) != 0);
              if (q.N2 > 0)
                ptx::mma_mxf8_pair(d_tmem + 256, ptx::sdesc_sw128(a_addr + k * 32),
                                   ptx::sdesc_sw128(b2_addr + k * 32), ptx::idesc_sf_id(id2, k), sf_col, sf_col + 12,
                                   (kb | k) != 0);
            }
            ++kbg;
          } else if (q.N2 == 0) {  // one MMA per K step (the usual case: up to 256 tokens)
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              ptx::mma_bf16_pair(d_tmem, ptx::sdesc_sw128(a_addr + k * 32), ptx::sdesc_sw128(b_addr + k * 32), id1,
                                 (kb | k) != 0);
          } else {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              ptx::mma_bf16_pair(d_tmem, ptx::sdesc_sw128(a_addr + k * 32), ptx::sdesc_sw128(b_addr + k * 32), id1,
                                 (kb | k) != 0);
              ptx::mma_bf16_pair(d_tmem + 256, ptx::sdesc_sw128(a_addr + k * 32), ptx::sdesc_sw128(b2_addr + k * 32),
                                 id2, (kb | k) != 0);
            }
          }
          ptx::mma_commit_pair(empty_bar(s), 0x3);
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit_pair(tfull_bar(acc), 0x3);
      }
      ptx::mma_commit_pair(drain_bar, 0x1);
      ptx::mbar_wait(drain_bar, 0, g.timeout_ns);
    } else if (GATHER && lane == 0 && !leader) {
      // ------------------------------------------------------------------ gather relay (peer)
      // As in the token-major pair kernel: make this CTA's gathered rows visible to the async
      // proxy, then arrive (CTA-scope release) on the leader's full barrier.
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        if (*s_abort) break;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait(gath_bar(s), ph, g.timeout_ns)) { gemm_abort(g, s_abort); ok = false; break; }
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive_remote(ptx::mapa_shared(full_bar(s), 0));
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    uint8_t* est = smem + L::OFF_EPI + (warp - 2) * kSwapEpiWarp;
    float* xch = reinterpret_cast<float*>(smem + L::OFF_XCH) + (q >> 1) * 2 * kSwapXchFloats;
    int* s_vote = reinterpret_cast<int*>(smem + L::OFF_MISC + 8);  // [2]: one word per quarter pair
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int it = 0;
    for (int t = pair; t < total; t += npairs, ++it) {
      const Tile tl = tile_at(t);
      const SwapGeo gq = swap_geo(tl.rows);
      const int acc = nacc == 2 ? (it & 1) : 0;
      const uint32_t acc_ph = static_cast<uint32_t>(nacc == 2 ? (it >> 1) & 1 : it & 1);
      int okw = 0;
      if (lane == 0) okw = (*s_abort == 0 && ptx::mbar_wait(tfull_bar(acc), acc_ph, g.timeout_ns)) ? 1 : 0;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      if (SWIGLU) {
        // both warps of a quarter pair take the same decision, so their named barriers pair up
        if (lane == 0 && !(q & 1)) s_vote[q >> 1] = 1;
        named_bar_sync(1 + (q >> 1), 64);
        if (lane == 0 && !okw) atomicAnd(&s_vote[q >> 1], 0);
        named_bar_sync(1 + (q >> 1), 64);
        const int both = *reinterpret_cast<volatile int*>(&s_vote[q >> 1]);
        named_bar_sync(1 + (q >> 1), 64);
        if (!both) {
          if (lane == 0 && !okw) gemm_abort(g, s_abort);
          break;
        }
      } else if (!okw) {
        if (lane == 0) gemm_abort(g, s_abort);
        break;
      }
      (void)ptx::mbar_try_wait(tfull_bar(acc), acc_ph);  // completed phase: acquire for every lane
      ptx::tc_fence_after();
      auto release = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(acc), 0));
      };
      const uint32_t tba = tb + static_cast<uint32_t>(acc * 256);
      if constexpr (SWIGLU)
        swap_epi_swiglu<EPI == EPI_SWIGLU_MX>(g, tl, gq.N, tba, q, lane, rank, xch, est, s_off, s_mtp128, release);
      else
        swap_epi_store<EPI == EPI_COMBINE>(g, tl, gq.N, tba, tl.n0 + 128 * rank + 32 * q, lane, est, release);
    }
  } else if constexpr (GATHER) {
    // ------------------------------------------------------------------ token-row gather (both CTAs)
    // Thread gt copies 16-byte chunk (gt % 8) of this CTA's B rows gt / 8 + 16 i of each
    // stage straight from x, into the 128-byte swizzled layout a TMA load would produce.
    const int gt = threadIdx.x - kGemmThreads;
    const int chunk = gt & 7, rbase = gt >> 3;
    constexpr int MAXI = kSwapMaxTokens / 2 / 16;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = pair; t < total && ok; t += npairs) {
      const Tile tl = tile_at(t);
      const SwapGeo q = swap_geo(tl.rows);
      const int nrows = q.b1 + q.b2;  // this CTA's B rows (a multiple of 8)
      const uint8_t* src[MAXI];
      uint32_t live = 0;              // bit i: row rbase + 16 i holds a token of the chunk
#pragma unroll
      for (int i = 0; i < MAXI; ++i) {
        const int sr = rbase + 16 * i;
        const int cr = sr < q.b1 ? rank * q.b1 + sr : 256 + rank * q.b2 + (sr - q.b1);  // row within the chunk
        const bool v = sr < nrows && cr < tl.rows;
        const int64_t tok = v ? __ldg(g.row_token + tl.row0 + cr) : 0;
        src[i] = g.gx + tok * g.gx_ld + chunk * 16;
        live |= static_cast<uint32_t>(v) << i;
      }
      if (*s_abort) break;
      for (int kb = 0; kb < num_kb; ++kb) {
        int okw = 0;
        if (lane == 0) okw = ptx::mbar_wait(empty_bar(s), ph ^ 1u, g.timeout_ns) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          if (lane == 0) gemm_abort(g, s_abort);
          ok = false;
          break;
        }
        (void)ptx::mbar_try_wait(empty_bar(s), ph ^ 1u);
        const uint32_t b_addr = ring + static_cast<uint32_t>(s) * SB + kSwapABytes;
        const int64_t kbyte = static_cast<int64_t>(kb) * BK * 2 + chunk * 16;
        const bool kin = kbyte < static_cast<int64_t>(g.K) * 2;
#pragma unroll
        for (int i = 0; i < MAXI; ++i) {
          const int sr = rbase + 16 * i;
          if (sr < nrows) {
            const bool v = kin && ((live >> i) & 1u);
            ptx::cp_async_16(b_addr + sr * kRowBytes + ((chunk ^ (sr & 7)) << 4), v ? src[i] + kb * BK * 2 : g.gx,
                             v ? 16u : 0u);
          }
        }
        ptx::cp_async_arrive_noinc(leader ? full_bar(s) : gath_bar(s));
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    ptx::cp_async_wait_all();
  } else if constexpr (EPI == EPI_COMBINE) {
    // ------------------------------------------------------------------ zero rows of y
    zero_rows(g, blockIdx.x * 4 + (warp - 6), gridDim.x * 4, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, 512);
  }
}

// B: the token rows [b_rows, K] (permuted copy; nullptr in row-gather mode); A: the packed
// weights [E_loc, n_out, K].  nt_max: tokens per tile (a multiple of 32, 64..384; MXFP8: of
// 128).
template <bool MX, int EPI, bool GATHER = false>
static cudaError_t launch_swap_inst(const void* B, int64_t b_rows, const void* A, const GemmArgs& g0, int nt_max,
                                    cudaStream_t st) {
  if (g0.E_loc > kSwapMaxEloc || nt_max < 64 || nt_max > kSwapMaxTokens || nt_max % 32 != 0 ||
      (MX && nt_max % 128 != 0))
    return cudaErrorInvalidValue;
  GemmArgs g = g0;
  g.nt_max = nt_max;
  g.sw_stage_bytes = kSwapABytes + (nt_max / 2) * kRowBytes;
  const int per_stage = g.sw_stage_bytes + (MX ? kSwapSfStage : 0);
  g.sw_stages = std::min(kSwapMaxStages, (kSwapSmemMax - 1024 - SwapLayout::FIXED) / per_stage);
  const int smem = SwapLayout::FIXED + g.sw_stages * per_stage + 1024;
  CUtensorMap ta;
  if (!make_operand_map(&ta, A, MX, g.K, g.n_out, g.E_loc, 128)) return cudaErrorInvalidValue;
  SwapBMaps tb;
  memset(&tb, 0, sizeof(tb));
  if (!GATHER)
    for (int i = 0; i < 5; ++i)
      if (!make_operand_map(&tb.m[i], B, MX, g.K, b_rows, 1, 128u >> i)) return cudaErrorInvalidValue;
  SwapSfMaps ts;
  memset(&ts, 0, sizeof(ts));
  if (MX) {
    const uint64_t kg = static_cast<uint64_t>(g.K / 128);
    if (!make_sf_map(&ts.w, g.b_sf, static_cast<uint64_t>(g.E_loc) * kg * (g.n_out / 128), 1))
      return cudaErrorInvalidValue;
    if (!make_sf_map(&ts.act, g.a_sf, static_cast<uint64_t>(mx_tiles_cap(b_rows, g.E_loc)) * kg, 1))
      return cudaErrorInvalidValue;
  }
  auto kern = tc_swap_gemm_kernel<MX, EPI, GATHER>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSwapSmemMax);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int grid = num_sms() & ~1;
  const int threads = kGemmThreads + swap_extra_threads<EPI, GATHER>();
  return launch_pdl(kern, dim3(grid), dim3(threads), smem, st, ta, tb, ts, g);
}

// GEMM1 + scaled SwiGLU (MXFP8: + requantisation of h), token rows from a permuted copy.
cudaError_t launch_swap_gemm1(const void* perm_x, int64_t rows, const void* Wgu, const GemmArgs& g, bool mx, int nt_max,
                              cudaStream_t st) {
  return mx ? launch_swap_inst<true, EPI_SWIGLU_MX>(perm_x, rows, Wgu, g, nt_max, st)
            : launch_swap_inst<false, EPI_SWIGLU_BF16>(perm_x, rows, Wgu, g, nt_max, st);
}
// bf16 GEMM1 + scaled SwiGLU with the token rows gathered from x (g.gx, g.row_token).
cudaError_t launch_swap_gemm1_gather(const void* Wgu, const GemmArgs& g, int nt_max, cudaStream_t st) {
  return launch_swap_inst<false, EPI_SWIGLU_BF16, true>(nullptr, 0, Wgu, g, nt_max, st);
}
// GEMM2 to Y2 (combine: the direct rows of y, zero rows, Y2 rows of multi-slot tokens).
cudaError_t launch_swap_gemm2(const void* h, int64_t rows, const void* Wd, const GemmArgs& g, bool mx, bool combine,
                              int nt_max, cudaStream_t st) {
  if (combine)
    return mx ? launch_swap_inst<true, EPI_COMBINE>(h, rows, Wd, g, nt_max, st)
              : launch_swap_inst<false, EPI_COMBINE>(h, rows, Wd, g, nt_max, st);
  return mx ? launch_swap_inst<true, EPI_STORE_BF16>(h, rows, Wd, g, nt_max, st)
            : launch_swap_inst<false, EPI_STORE_BF16>(h, rows, Wd, g, nt_max, st);
}

}  // namespace moe
