// Shared pieces of the tcgen05 grouped GEMM kernels (1-CTA and 2-CTA variants): launch
// arguments, tile decoding over the ragged per-expert segments, the fused epilogue and
// the TMA tensor-map helper.
#pragma once

#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "moe_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

constexpr int kBM = 128;
constexpr int kRowBytes = 128;  // bytes of one operand row per pipeline stage
constexpr int kGemmThreads = 192;        // producer, MMA, 4 epilogue warps
constexpr int kGatherThreads = 128;      // + 4 A-gather warps in row-gather mode
constexpr int kZeroThreads = 128;        // + 4 zero-row warps in combine mode (GEMM2)
constexpr int kMaxEloc = 1024;

// EPI_COMBINE: GEMM2 with the unpermute + combine fused into its epilogue (bf16 y).
enum { EPI_STORE_BF16 = 0, EPI_SWIGLU_BF16 = 1, EPI_SWIGLU_MX = 2, EPI_DSWIGLU = 3, EPI_COMBINE = 4 };


struct GemmArgs {
  const int32_t* offsets;  // [E_loc + 1]
  int E_loc;
  int n_out;               // output columns (GEMM1: packed 2f; GEMM2: d)
  int K;                   // contraction length in elements
  void* out;               // bf16 [rows, ld_out] or E4M3 bytes [rows, ld_out]
  int64_t ld_out;          // elements per output row
  uint8_t* out_sf;         // EPI_SWIGLU_MX: scales of h (activation SF tile layout, K = n_out / 2)
  const float* row_prob;   // GEMM1: routing probability per permuted row
  const uint8_t* a_sf;     // MXFP8: scales of A (activation SF tile layout)
  const uint8_t* b_sf;     // MXFP8: scales of B (weight SF tile layout)
  int32_t* err;            // device error word
  uint64_t timeout_ns;
  // Row-gather mode (GEMM1 only): A row r of the tile is row row_token[r] of gx
  // (gx_ld bytes per row) instead of row r of a permuted copy; MXFP8 takes its scales
  // from gx_sf (gx_sf_ld bytes per row, one E8M0 byte per 32 values).
  const uint8_t* gx;
  int64_t gx_ld;
  const int32_t* row_token;
  const uint8_t* gx_sf;
  int64_t gx_sf_ld;
  // EPI_DSWIGLU (backward, bf16): the accumulator is dh [rows, f]; aux = the forward
  // pre-activations g/u [N_cap, 2f] bf16 in the packed column order; out = dg/du in the
  // same order (ld_out = 2f); out2 = h [N_cap, f] bf16; dp_part [N_cap, f / 32] fp32 =
  // per-32-column partial sums of dh * silu(g) * u.
  // EPI_SWIGLU_BF16 with out2 set (training forward): out2 receives g/u [N_cap, 2f] bf16 in
  // the packed column order, as the backward's aux.
  const uint16_t* aux;
  void* out2;
  float* dp_part;
  int64_t out_rows;        // rows of out / out2 (the extent of their TMA store maps)
  // EPI_COMBINE: y [T, n_out] bf16.  row_token [N_cap] = token of each routed row;
  // tok_nloc [T] = local slots per token.  Rows of tokens with one local slot go straight
  // to y, tokens without one get a zero row (zero-row warps), rows of tokens with several
  // go to out (Y2) for the slot-ordered sum that follows.
  void* y;
  const int32_t* tok_nloc;
  int T;
  // Swapped-operand kernel (gemm_tc_swap.cu): tokens per tile, pipeline depth and bytes
  // per stage (set by its launcher).
  int nt_max;
  int sw_stages;
  int sw_stage_bytes;
  // EPI_SWIGLU_BF16, per-tensor FP8 GEMM1: largest |h| of the bf16 h written (fp32 bits,
  // atomicMax), the scale of h's quantisation for GEMM2; nullptr otherwise.
  uint32_t* amax;
};

// TMA store maps of the bf16 outputs: 32 x 32 boxes over out [out_rows, ld_out] and out2
// [out_rows, n_out] (64-byte swizzle); unused ones are left zero.
struct OutMaps {
  CUtensorMap out, out2;
};

struct Tile {
  int e, mt, row0, rows, n0;
};

// Tile t of a launch whose m-tiles are `bm`-row slices of each expert segment, numbered
// in expert order (s_mtp = prefix of ceil(count / bm)), and n-tiles are `bn` columns.
__device__ __forceinline__ Tile decode_tile(int t, int n_tiles_n, int bn, const int* s_off, const int* s_mtp,
                                            int E_loc, int bm = kBM) {
  const int gm = t / n_tiles_n;
  int lo = 0, hi = E_loc - 1;  // last expert whose first m-tile is <= gm (skips empty experts)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_mtp[mid] <= gm) lo = mid;
    else hi = mid - 1;
  }
  Tile r;
  r.e = lo;
  r.mt = gm;
  r.row0 = s_off[lo] + (gm - s_mtp[lo]) * bm;
  r.rows = min(bm, s_off[lo + 1] - r.row0);
  r.n0 = (t - gm * n_tiles_n) * bn;
  return r;
}

__device__ __forceinline__ void gemm_abort(const GemmArgs& g, volatile int* s_abort) {
  *s_abort = 1;
  set_device_error(g.err, MOE_ERR_TIMEOUT);
}

// Epilogue staging: each epilogue warp owns 32 rows x 80 bytes of shared memory (64 data
// bytes per row + 16 bytes of padding to spread the banks).  A warp's 32 threads each hold
// one output row of a 32-column block in registers; they write it to the staging rows and
// read it back column-chunk-major, so each global store instruction covers whole 64-byte
// (or 32-byte) row segments of 8 (or 16) rows instead of 32 scattered 16-byte pieces.
constexpr int kEpiRowBytes = 80;
constexpr int kEpiWarpBytes = 32 * kEpiRowBytes;
constexpr int kEpiBytes = 4 * kEpiWarpBytes;  // 4 epilogue warps

// v: this lane's row, CHUNKS x 16 bytes.  g0: global address of the warp's first row at
// the block's first column; ld: bytes between rows.  Rows >= rows_valid and 16-byte
// chunks >= chunks_valid are not written.
template <int CHUNKS>
__device__ __forceinline__ void warp_store_rows(uint8_t* stage, const uint4 (&v)[CHUNKS], int lane, uint8_t* g0,
                                                int64_t ld, int rows_valid, int chunks_valid) {
  uint4* mine = reinterpret_cast<uint4*>(stage + lane * kEpiRowBytes);
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) mine[c] = v[c];
  __syncwarp();
  constexpr int kRowsPerStore = 32 / CHUNKS;
#pragma unroll
  for (int j = 0; j < CHUNKS; ++j) {
    const int r = j * kRowsPerStore + lane / CHUNKS;
    const int c = lane % CHUNKS;
    const uint4 val = *reinterpret_cast<const uint4*>(stage + r * kEpiRowBytes + c * 16);
    if (r < rows_valid && c < chunks_valid) *reinterpret_cast<uint4*>(g0 + r * ld + c * 16) = val;
  }
  __syncwarp();
}

// Same staging, but each lane's row goes to its own destination: dst = this lane's
// row at the block's first column (nullptr: nothing stored for that row).  Each store
// instruction covers whole 64-byte row segments (4 lanes per row).
__device__ __forceinline__ void warp_store_rows_to(uint8_t* stage, const uint4 (&v)[4], int lane, uint8_t* dst,
                                                   int chunks_valid) {
  uint4* mine = reinterpret_cast<uint4*>(stage + lane * kEpiRowBytes);
#pragma unroll
  for (int c = 0; c < 4; ++c) mine[c] = v[c];
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = j * 8 + lane / 4;
    const int c = lane % 4;
    uint8_t* row_dst = reinterpret_cast<uint8_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(dst), r));
    const uint4 val = *reinterpret_cast<const uint4*>(stage + r * kEpiRowBytes + c * 16);
    if (row_dst != nullptr && c < chunks_valid) *reinterpret_cast<uint4*>(row_dst + c * 16) = val;
  }
  __syncwarp();
}

// TMA-store staging of the bf16 epilogues: each epilogue warp owns two 2 KB buffers, each
// one 32-row x 64-byte block in the 64-byte swizzle of the store maps (16-byte chunk c of
// row r at c ^ ((r >> 1) & 3)).  The two alternate; a buffer is refilled once the TMA store
// that read it has finished reading.
constexpr int kEpiTmaBuf = 32 * 64;
constexpr int kEpiTmaWarpBytes = 2 * kEpiTmaBuf;
constexpr int kEpiTmaBytes = 4 * kEpiTmaWarpBytes;
static_assert(kEpiTmaWarpBytes >= kEpiWarpBytes, "a TMA staging area also serves the padded staging");

struct EpiStage {
  uint8_t* buf;    // this warp's staging (generic address)
  uint32_t buf_s;  // the same in the shared window
  int next, last;  // buffer to fill next; buffer of the most recent TMA store (-1: none)
};

// One 32 x 32 bf16 block of the warp's rows (v = this lane's row, 4 x 16 bytes).  TMA: a
// whole block (32 valid rows, 4 valid chunks) leaves by one TMA store at (col, row) of
// `map`; a block cut by a segment or matrix edge is written from the staging buffer with
// plain stores (g0 = global address of the warp's first row at the block's first column,
// ld = bytes between rows).  Without TMA the padded staging of warp_store_rows is used
// (st.buf then holds at least kEpiWarpBytes).
template <bool TMA>
__device__ __forceinline__ void warp_store_block(EpiStage& st, const uint4 (&v)[4], int lane, const CUtensorMap* map,
                                                 int col, int64_t row, uint8_t* g0, int64_t ld, int rows_valid,
                                                 int chunks_valid) {
  if constexpr (!TMA) {
    (void)map; (void)col; (void)row;
    warp_store_rows<4>(st.buf, v, lane, g0, ld, rows_valid, chunks_valid);
  } else {
    const int b = st.next;
    if (lane == 0) {
      if (st.last == (b ^ 1)) ptx::bulk_wait_read<1>();
      else ptx::bulk_wait_read<0>();
    }
    __syncwarp();
    uint8_t* buf = st.buf + b * kEpiTmaBuf;
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(buf + lane * 64 + ((c ^ sw) << 4)) = v[c];
    if (rows_valid == 32 && chunks_valid == 4) {
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(map, st.buf_s + b * kEpiTmaBuf, col, static_cast<int>(row));
        ptx::bulk_commit();
      }
      st.last = b;
    } else {
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // 8 rows x 64 bytes per store instruction
        const int r = j * 8 + lane / 4, c = lane % 4;
        const uint4 val = *reinterpret_cast<const uint4*>(buf + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
        if (r < rows_valid && c < chunks_valid) *reinterpret_cast<uint4*>(g0 + r * ld + c * 16) = val;
      }
      __syncwarp();
    }
    st.next = b ^ 1;
  }
}

// ---- combine fused into GEMM2: zero rows of y, written by the zero-row warps

// Zero row of token t (no local slot), streaming stores.
__device__ __forceinline__ void zero_row(const GemmArgs& g, int t, int lane) {
  const int64_t row_vecs = static_cast<int64_t>(g.n_out) * 2 / 16;
  uint4* dst = static_cast<uint4*>(g.y) + static_cast<int64_t>(t) * row_vecs;
  for (int64_t c = lane; c < row_vecs; c += 32) __stcs(dst + c, make_uint4(0u, 0u, 0u, 0u));
}

// Zero-row warp zw of nzw over the grid: the tokens t = zw, zw + nzw, ... without a local
// slot get a zero row, written as early as possible, alongside the GEMM.  (Spreading the
// writes over the GEMM's tiles instead measured slower on B300: the GEMM's operands are
// mostly L2 hits, and the early writes overlap its start-up.)
__device__ __forceinline__ void zero_rows(const GemmArgs& g, int zw, int nzw, int lane) {
  for (int t = zw; t < g.T; t += nzw)
    if (__ldg(g.tok_nloc + t) == 0) zero_row(g, t, lane);
}

// Epilogue of one 32-row slab of an accumulator tile (one warp, one TMEM lane per thread):
// bf16 store of BN columns (GEMM2), or the fused scaled SwiGLU on BN/64 blocks of 32 gate
// + 32 up columns with bf16 or MXFP8 (one 32-value block per thread) output (GEMM1).
// tbase = TMEM address of this warp's lane quarter and accumulator; q = lane quarter;
// tl.row0/tl.rows describe the 128-row tile the slab belongs to.
// release(): called by every lane once this warp's last TMEM read of the tile is done (it
// frees the accumulator for the next tile's MMAs); the MXFP8 SwiGLU epilogue calls it
// before its global stores, the others at the end.
template <int EPI, bool TMA, typename Release>
__device__ __forceinline__ void epilogue_warp(const GemmArgs& g, const OutMaps& om, const Tile& tl, uint32_t tbase,
                                              int BN, int q, int lane, EpiStage& st, Release&& release) {
  const int r = q * 32 + lane;                         // row within the tile
  const int rows_valid = max(0, min(32, tl.rows - q * 32));
  const int64_t row_first = static_cast<int64_t>(tl.row0) + q * 32;
  if constexpr (EPI == EPI_STORE_BF16) {
    uint8_t* out = static_cast<uint8_t*>(g.out);
    const int64_t ld = g.ld_out * 2;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(tbase + c, v);
      ptx::tmem_ld_wait();
      const int n = tl.n0 + c;
      uint4 pk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        pk[j] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
      const int chunks = max(0, min(4, (g.n_out - n) / 8));
      warp_store_block<TMA>(st, pk, lane, &om.out, n, row_first, out + row_first * ld + static_cast<int64_t>(n) * 2, ld,
                            rows_valid, chunks);
    }
  } else if constexpr (EPI == EPI_COMBINE) {
    // GEMM2 + the direct part of the unpermute + combine ("Wide-EP ... NVIDIA" explainer,
    // section "MoE basics": the chosen experts' results are summed per token).  A token
    // with one local slot has y = its row (the slot sum of one bf16 value rounds to
    // itself), so that row goes straight to y; rows of tokens with several local slots go
    // to Y2 for the slot-ordered sum of the follow-up combine pass.  A slab whose rows all
    // go to Y2 leaves by the ordinary (TMA) store path.
    const bool live = r < tl.rows;
    const int64_t row = row_first + lane;
    const int t = live ? __ldg(g.row_token + row) : 0;
    const int nloc = live ? __ldg(g.tok_nloc + t) : 0;
    const bool direct = __any_sync(0xffffffffu, live && nloc == 1);
    uint8_t* Y2 = static_cast<uint8_t*>(g.out);
    const int64_t ld2 = g.ld_out * 2;
    uint8_t* dst = !live ? nullptr
                         : nloc == 1 ? static_cast<uint8_t*>(g.y) + t * (static_cast<int64_t>(g.n_out) * 2)
                                     : Y2 + row * ld2;
    if (TMA && direct && lane == 0) ptx::bulk_wait_read<0>();  // the padded staging reuses the TMA buffers
    if (TMA && direct) st.last = -1;
    __syncwarp();
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(tbase + c, v);
      ptx::tmem_ld_wait();
      const int n = tl.n0 + c;
      uint4 pk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        pk[j] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
      const int chunks = max(0, min(4, (g.n_out - n) / 8));
      if (direct)
        warp_store_rows_to(st.buf, pk, lane, dst == nullptr ? nullptr : dst + static_cast<int64_t>(n) * 2, chunks);
      else
        warp_store_block<TMA>(st, pk, lane, &om.out, n, row_first, Y2 + row_first * ld2 + static_cast<int64_t>(n) * 2,
                              ld2, rows_valid, chunks);
    }
  } else if constexpr (EPI == EPI_DSWIGLU) {
    // ScaledSwiGLU backward for h = p * silu(g) * u, from dh and the saved g, u:
    //   du = p dh silu(g),  dg = p dh u s (1 + g (1 - s)) with s = sigmoid(g),
    //   dp = sum over the row of dh silu(g) u (partial sums per 32 columns)
    // Eight columns at a time, packed to bf16 at once (the kernel's register budget is
    // 168 per thread); the next block's g/u loads are in flight during this block's stores.
    const float p = r < tl.rows ? __ldg(g.row_prob + row_first + lane) : 0.0f;
    const int fdim = g.n_out;
    const int64_t row = row_first + lane;
    const int64_t ld2 = static_cast<int64_t>(2 * fdim) * 2, ldh = static_cast<int64_t>(fdim) * 2;
    const bool live = r < tl.rows;
    auto load_gu = [&](int fc, uint4 (&a)[4], uint4 (&b)[4]) {  // 32 gate + 32 up values of block fc
      if (live && fc < fdim) {
        const uint4* src = reinterpret_cast<const uint4*>(g.aux + row * 2 * fdim + 2 * fc);
#pragma unroll
        for (int j = 0; j < 4; ++j) { a[j] = __ldg(src + j); b[j] = __ldg(src + 4 + j); }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = b[j] = make_uint4(0u, 0u, 0u, 0u);
      }
    };
    uint4 ga[4], ub[4];
    load_gu(tl.n0, ga, ub);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int fc = tl.n0 + c;  // first f column of this block (a multiple of 32)
      if (fc >= fdim) break;
      uint32_t v[32];
      ptx::tmem_ld32(tbase + c, v);
      ptx::tmem_ld_wait();
      uint4 pdg[4], pdu[4], ph[4];
      float dp = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t gw[4] = {ga[j].x, ga[j].y, ga[j].z, ga[j].w};
        const uint32_t uw[4] = {ub[j].x, ub[j].y, ub[j].z, ub[j].w};
        uint32_t odg[4], odu[4], oh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float rdg[2], rdu[2], rh[2];
#pragma unroll
          for (int hl = 0; hl < 2; ++hl) {
            const float gg = hl ? bf16_hi(gw[e]) : bf16_lo(gw[e]);
            const float uu = hl ? bf16_hi(uw[e]) : bf16_lo(uw[e]);
            const float dh = __uint_as_float(v[8 * j + 2 * e + hl]);
            const float sg = __fdividef(1.0f, 1.0f + __expf(-gg));
            const float a = gg * sg;
            rh[hl] = p * a * uu;
            dp += dh * a * uu;
            rdu[hl] = p * dh * a;
            rdg[hl] = p * dh * uu * sg * (1.0f + gg * (1.0f - sg));
          }
          odg[e] = pack_bf16x2(rdg[0], rdg[1]);
          odu[e] = pack_bf16x2(rdu[0], rdu[1]);
          oh[e] = pack_bf16x2(rh[0], rh[1]);
        }
        pdg[j] = make_uint4(odg[0], odg[1], odg[2], odg[3]);
        pdu[j] = make_uint4(odu[0], odu[1], odu[2], odu[3]);
        ph[j] = make_uint4(oh[0], oh[1], oh[2], oh[3]);
      }
      load_gu(c + 32 < BN ? fc + 32 : fdim, ga, ub);
      uint8_t* gbase = static_cast<uint8_t*>(g.out) + row_first * ld2 + static_cast<int64_t>(2 * fc) * 2;
      warp_store_block<TMA>(st, pdg, lane, &om.out, 2 * fc, row_first, gbase, ld2, rows_valid, 4);
      warp_store_block<TMA>(st, pdu, lane, &om.out, 2 * fc + 32, row_first, gbase + 64, ld2, rows_valid, 4);
      warp_store_block<TMA>(st, ph, lane, &om.out2, fc, row_first,
                            static_cast<uint8_t*>(g.out2) + row_first * ldh + static_cast<int64_t>(fc) * 2, ldh,
                            rows_valid, 4);
      if (live) g.dp_part[row * (fdim / 32) + fc / 32] = dp;
    }
  } else if constexpr (EPI == EPI_SWIGLU_MX) {
    // The whole tile's h is computed and quantised into registers first (4 blocks of 32
    // values: 8 words of E4M3 codes and one E8M0 byte each), the accumulator is released,
    // and only then are the codes and scales stored: with one accumulator in TMEM (256-wide
    // MXFP8 tiles) the next tile's MMAs overlap these stores.
    const float p = r < tl.rows ? __ldg(g.row_prob + row_first + lane) : 0.0f;
    const int fdim = g.n_out / 2;
    constexpr int MAXB = 4;  // BN / 64 <= 4
    const int nb = BN / 64;
    uint32_t W[MAXB][8];
    int XS[MAXB];
#pragma unroll
    for (int sb = 0; sb < MAXB; ++sb) {
      XS[sb] = 0;
      if (sb < nb) {
        uint32_t gv[32], uv[32];
        ptx::tmem_ld32(tbase + sb * 64, gv);       // 32 gate columns
        ptx::tmem_ld32(tbase + sb * 64 + 32, uv);  // the matching 32 up columns
        ptx::tmem_ld_wait();
        float h[32];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float gg = __uint_as_float(gv[i]);
          h[i] = p * __fdividef(gg, 1.0f + __expf(-gg)) * __uint_as_float(uv[i]);
          amax = fmaxf(amax, fabsf(h[i]));
        }
        const int X = mx_exponent(amax);
        const float inv = mx_inv_scale(X);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          W[sb][j] = static_cast<uint32_t>(e4m3x2(h[4 * j] * inv, h[4 * j + 1] * inv)) |
                     (static_cast<uint32_t>(e4m3x2(h[4 * j + 2] * inv, h[4 * j + 3] * inv)) << 16);
        XS[sb] = X;
      }
    }
    release();
#pragma unroll
    for (int sb = 0; sb < MAXB; ++sb) {
      if (sb < nb) {
        const int fc = tl.n0 / 2 + sb * 32;  // first h column of this block
        const uint4 pk[2] = {make_uint4(W[sb][0], W[sb][1], W[sb][2], W[sb][3]),
                             make_uint4(W[sb][4], W[sb][5], W[sb][6], W[sb][7])};
        warp_store_rows<2>(st.buf, pk, lane, static_cast<uint8_t*>(g.out) + row_first * g.ld_out + fc, g.ld_out,
                           rows_valid, fc < fdim ? 2 : 0);
        if (r < tl.rows && fc < fdim)
          g.out_sf[sf_act_offset(tl.mt, r, fc, fdim)] = static_cast<uint8_t>(XS[sb] + 127);
      }
    }
    return;
  } else {
    const float p = r < tl.rows ? __ldg(g.row_prob + row_first + lane) : 0.0f;
    const int fdim = g.n_out / 2;
    float hmax = 0.0f;  // largest |h| as stored (bf16), per-tensor FP8 only
#pragma unroll 1
    for (int sb = 0; sb < BN / 64; ++sb) {
      uint32_t gv[32], uv[32];
      ptx::tmem_ld32(tbase + sb * 64, gv);       // 32 gate columns
      ptx::tmem_ld32(tbase + sb * 64 + 32, uv);  // the matching 32 up columns
      ptx::tmem_ld_wait();
      const int fc = tl.n0 / 2 + sb * 32;  // first h column of this block
      float h[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float gg = __uint_as_float(gv[i]);
        // silu(g) = g / (1 + e^-g) with the fast exponential and division intrinsics:
        // a few ulp of fp32 error, far below the bf16 / E4M3 rounding of h
        h[i] = p * __fdividef(gg, 1.0f + __expf(-gg)) * __uint_as_float(uv[i]);
      }
      if constexpr (EPI == EPI_SWIGLU_BF16) {
        uint4 pk[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          pk[j] = make_uint4(pack_bf16x2(h[8 * j + 0], h[8 * j + 1]), pack_bf16x2(h[8 * j + 2], h[8 * j + 3]),
                             pack_bf16x2(h[8 * j + 4], h[8 * j + 5]), pack_bf16x2(h[8 * j + 6], h[8 * j + 7]));
        const int64_t ld = g.ld_out * 2;
        if (g.amax && r < tl.rows && fc < fdim) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t w4[4] = {pk[j].x, pk[j].y, pk[j].z, pk[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) hmax = fmaxf(hmax, fmaxf(fabsf(bf16_lo(w4[e])), fabsf(bf16_hi(w4[e]))));
          }
        }
        if (fc < fdim)
          warp_store_block<TMA>(st, pk, lane, &om.out, fc, row_first,
                                static_cast<uint8_t*>(g.out) + row_first * ld + static_cast<int64_t>(fc) * 2, ld,
                                rows_valid, 4);
        if (g.out2 && fc < fdim) {  // training forward: keep g and u (bf16, packed order) for the backward
          const int64_t ld2 = static_cast<int64_t>(g.n_out) * 2;
          uint8_t* gbase = static_cast<uint8_t*>(g.out2) + row_first * ld2 + static_cast<int64_t>(2 * fc) * 2;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            pk[j] = make_uint4(pack_bf16x2(__uint_as_float(gv[8 * j + 0]), __uint_as_float(gv[8 * j + 1])),
                               pack_bf16x2(__uint_as_float(gv[8 * j + 2]), __uint_as_float(gv[8 * j + 3])),
                               pack_bf16x2(__uint_as_float(gv[8 * j + 4]), __uint_as_float(gv[8 * j + 5])),
                               pack_bf16x2(__uint_as_float(gv[8 * j + 6]), __uint_as_float(gv[8 * j + 7])));
          warp_store_block<TMA>(st, pk, lane, &om.out2, 2 * fc, row_first, gbase, ld2, rows_valid, 4);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            pk[j] = make_uint4(pack_bf16x2(__uint_as_float(uv[8 * j + 0]), __uint_as_float(uv[8 * j + 1])),
                               pack_bf16x2(__uint_as_float(uv[8 * j + 2]), __uint_as_float(uv[8 * j + 3])),
                               pack_bf16x2(__uint_as_float(uv[8 * j + 4]), __uint_as_float(uv[8 * j + 5])),
                               pack_bf16x2(__uint_as_float(uv[8 * j + 6]), __uint_as_float(uv[8 * j + 7])));
          warp_store_block<TMA>(st, pk, lane, &om.out2, 2 * fc + 32, row_first, gbase + 64, ld2, rows_valid, 4);
        }
      } else {
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
        const int X = mx_exponent(amax);
        const float inv = mx_inv_scale(X);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          w[j] = static_cast<uint32_t>(e4m3x2(h[4 * j] * inv, h[4 * j + 1] * inv)) |
                 (static_cast<uint32_t>(e4m3x2(h[4 * j + 2] * inv, h[4 * j + 3] * inv)) << 16);
        const uint4 pk[2] = {make_uint4(w[0], w[1], w[2], w[3]), make_uint4(w[4], w[5], w[6], w[7])};
        warp_store_rows<2>(st.buf, pk, lane, static_cast<uint8_t*>(g.out) + row_first * g.ld_out + fc, g.ld_out,
                           rows_valid, fc < fdim ? 2 : 0);
        if (r < tl.rows && fc < fdim) g.out_sf[sf_act_offset(tl.mt, r, fc, fdim)] = static_cast<uint8_t>(X + 127);
      }
    }
    if constexpr (EPI == EPI_SWIGLU_BF16) {
      if (g.amax) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, o));
        if (lane == 0 && hmax > 0.0f) atomicMax(g.amax, __float_as_uint(hmax));
      }
    }
  }
  release();
}

// 3-D K-major operand map [outer, rows, K], box [1, box_rows, 128 bytes], 128-byte swizzle.
bool make_operand_map(CUtensorMap* m, const void* base, bool fp8, uint64_t K, uint64_t rows, uint64_t outer,
                      uint32_t box_rows);
// 2-D row-major output map [rows, cols] of elt-byte elements (2 = bf16, 4 = fp32) for TMA
// stores of box_rows x box_cols boxes; box_cols * elt must be 32, 64 or 128 bytes and
// selects the matching swizzle (a row's 16-byte chunk c sits at c ^ ((row >> s) & m)).
bool make_store_map(CUtensorMap* m, void* base, int elt, uint64_t cols, uint64_t rows, uint32_t box_cols,
                    uint32_t box_rows);
int num_sms();
// 2-D map over an SF tile layout buffer of n_atoms 512-byte atoms (rows of 128 uint32),
// box = atoms_per_box consecutive atoms.
bool make_sf_map(CUtensorMap* m, const void* base, uint64_t n_atoms, uint32_t atoms_per_box);
// Store maps of g.out (bf16 [out_rows, ld_out]) and g.out2 (bf16 [out_rows, n_out]) where set.
bool make_out_maps(OutMaps* m, const GemmArgs& g);

}  // namespace moe
