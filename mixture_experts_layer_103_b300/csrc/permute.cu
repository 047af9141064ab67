// Step 2: stable permute of token rows into expert-contiguous order (the single-GPU
// analogue of the dispatch step described in the "Wide-EP ... NVIDIA" explainer, section
// "Prerequisite: fast GPU-to-GPU links": each token goes to the experts it was routed to).
//
// Row offsets[e] + r holds the r-th token (ascending token id) routed to local expert e.
// Positions are fixed without atomics so the result is deterministic:
//   count   per tile of 64 or 256 tokens, per-expert counts (shared-memory counters;
//           order-free)
//   scan    one CTA: exclusive scan over (expert, tile) in expert-major order gives each
//           (expert, tile) its first row; offsets and the MXFP8 m-tile bases fall out
//   scatter per tile, the rank of token t among the tile's tokens routed to e is the
//           popcount of a per-expert token bitmask below t
//   gather  one warp per permuted row copies x[t] with 16-byte vector loads/stores (HBM
//           bound); in MXFP8 mode it quantises each 32-value block while copying ("MXFP8
//           Precision Reduces Memory Footprint": one scale per 32 consecutive values).
//           Skipped when no permuted copy is asked for (the row-gather GEMM1 reads x
//           through row_src_token instead); MXFP8 then quantises x once per token.
#include <algorithm>

#include "moe_common.cuh"

namespace moe {

cudaError_t launch_amax(const void* src, moe_dtype dt, int64_t n_per_seg, int n_seg, uint32_t* amax_bits,
                        cudaStream_t st);

int num_sms();

// Tokens per tile of the count and scatter kernels: 64 while the (expert, tile) count
// table stays small (more CTAs for these latency-bound kernels), else 256 (a shorter
// one-CTA scan).
constexpr int kPermTileSmall = 64, kPermTileLarge = 256;
constexpr int64_t kSmallTileTable = 16384;  // max E_loc * tiles for the 64-token tiles

static int perm_tile(int T, int E_loc) {
  const int64_t n = ceil_div(T > 0 ? T : 1, kPermTileSmall) * static_cast<int64_t>(E_loc);
  return n <= kSmallTileTable ? kPermTileSmall : kPermTileLarge;
}

template <int TILE>
__global__ void __launch_bounds__(TILE) perm_count_kernel(const int32_t* __restrict__ ids, int T, int k, int e0,
                                                               int E_loc, int n_tiles, int32_t* __restrict__ tile_counts) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ int s_cnt[];
  for (int e = threadIdx.x; e < E_loc; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * TILE + threadIdx.x;
  if (t < T)
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(ids + t * k + j) - e0;
      if (static_cast<unsigned>(e) < static_cast<unsigned>(E_loc)) atomicAdd(&s_cnt[e], 1);
    }
  __syncthreads();
  for (int e = threadIdx.x; e < E_loc; e += blockDim.x)
    tile_counts[static_cast<int64_t>(e) * n_tiles + blockIdx.x] = s_cnt[e];
}

// Exclusive scan over a 1024-thread block; returns the prefix of v and the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int prefix = warp > 0 ? s_warp[warp - 1] : 0;
  total = s_warp[nwarps - 1];
  __syncthreads();
  return prefix + x - v;
}

__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ tile_counts, int n_tiles, int E_loc,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ mtile_base) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int s_warp[32];
  __shared__ int s_off[1025];
  const int n = E_loc * n_tiles;
  int carry = 0;
  // 4 consecutive entries per thread: 4096 entries per pass
  for (int base = 0; base < n; base += 4 * blockDim.x) {
    const int i0 = base + 4 * threadIdx.x;
    int v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = i0 + q < n ? tile_counts[i0 + q] : 0;
    int total;
    int run = carry + block_exclusive_scan(v[0] + v[1] + v[2] + v[3], s_warp, total);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + q;
      if (i < n) {
        tile_counts[i] = run;  // first row of (expert i / n_tiles, tile i % n_tiles)
        if (i % n_tiles == 0) s_off[i / n_tiles] = run;
      }
      run += v[q];
    }
    carry += total;
  }
  if (threadIdx.x == 0) s_off[E_loc] = carry;
  __syncthreads();
  const int e = threadIdx.x;
  int mt = 0;
  if (e < E_loc) {
    const int c = s_off[e + 1] - s_off[e];
    counts[e] = c;
    offsets[e] = s_off[e];
    mt = (c + 127) / 128;
  }
  if (e == 0) offsets[E_loc] = s_off[E_loc];
  int total;
  const int ex = block_exclusive_scan(mt, s_warp, total);
  if (mtile_base) {
    if (e < E_loc) mtile_base[e] = ex;
    if (e == 0) mtile_base[E_loc] = total;
  }
}

template <int TILE>
__global__ void __launch_bounds__(TILE) perm_scatter_kernel(const int32_t* __restrict__ ids,
                                                                 const float* __restrict__ probs, int T, int k, int e0,
                                                                 int E_loc, int n_tiles,
                                                                 const int32_t* __restrict__ tile_base,
                                                                 int32_t* __restrict__ pair_to_row,
                                                                 int32_t* __restrict__ row_src_token,
                                                                 float* __restrict__ row_prob,
                                                                 int32_t* __restrict__ tok_nloc) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ uint32_t s_mask[];  // [E_loc][TILE / 32] token bitmasks
  constexpr int W = TILE / 32;
  for (int i = threadIdx.x; i < E_loc * W; i += blockDim.x) s_mask[i] = 0u;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * TILE + threadIdx.x;
  if (t < T)
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(ids + t * k + j) - e0;
      if (static_cast<unsigned>(e) < static_cast<unsigned>(E_loc)) atomicOr(&s_mask[e * W + warp], 1u << lane);
    }
  __syncthreads();
  if (t >= T) return;
  int nloc = 0;
  for (int j = 0; j < k; ++j) {
    const int e = __ldg(ids + t * k + j) - e0;
    int32_t row = -1;
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E_loc)) {
      int rank = __popc(s_mask[e * W + warp] & ((1u << lane) - 1u));
      for (int w = 0; w < warp; ++w) rank += __popc(s_mask[e * W + w]);
      row = tile_base[static_cast<int64_t>(e) * n_tiles + blockIdx.x] + rank;
      row_src_token[row] = static_cast<int32_t>(t);
      row_prob[row] = __ldg(probs + t * k + j);
      ++nloc;
    }
    pair_to_row[t * k + j] = row;
  }
  if (tok_nloc) tok_nloc[t] = nloc;  // local slots per token, for the GEMM2 that combines
}

// The same per-token slot count for a GEMM2 + combine call on maps made elsewhere.
__global__ void __launch_bounds__(256) combine_prep_kernel(const int32_t* __restrict__ pair_to_row, int T, int k,
                                                           int32_t* __restrict__ tok_nloc) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int nloc = 0;
  for (int j = 0; j < k; ++j) nloc += __ldg(pair_to_row + t * k + j) >= 0;
  tok_nloc[t] = nloc;
}

cudaError_t launch_combine_prep(const int32_t* pair_to_row, int T, int k, int32_t* tok_nloc, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(combine_prep_kernel, dim3(static_cast<unsigned>(ceil_div(T, 256))), dim3(256), 0, st, pair_to_row,
                    T, k, tok_nloc);
}

// ------------------------------------------------------------------------------ gather
// Plain copy of rows (fp32 -> fp32 or bf16 -> bf16), 16-byte vectors.
__global__ void __launch_bounds__(256) perm_gather_copy_kernel(const uint4* __restrict__ x, int64_t row_vecs,
                                                               const int32_t* __restrict__ offsets, int E_loc,
                                                               const int32_t* __restrict__ row_src_token,
                                                               uint4* __restrict__ perm_x) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int N = __ldg(offsets + E_loc);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < N; r += warps) {
    const int64_t t = __ldg(row_src_token + r);
    const uint4* src = x + t * row_vecs;
    uint4* dst = perm_x + r * row_vecs;
    int64_t c = lane;
    for (; c + 96 < row_vecs; c += 128) {
      const uint4 a = __ldg(src + c), b = __ldg(src + c + 32), cc = __ldg(src + c + 64), d = __ldg(src + c + 96);
      dst[c] = a;
      dst[c + 32] = b;
      dst[c + 64] = cc;
      dst[c + 96] = d;
    }
    for (; c < row_vecs; c += 32) dst[c] = __ldg(src + c);
  }
}

// MXFP8 quantisation of 16-byte vectors [v0, v1) of one row by one warp (blocks of 32
// along d; v0 and v1 on block boundaries).  IN_BF16 = 1: bf16 input (8 values per 16-byte
// vector, 4 lanes per block); 0: fp32 input (4 per vector, 8 lanes).  E4M3 codes go to
// dst (the row's start); the E8M0 byte of the block holding column col is passed to
// put_sf(col, byte) by the first lane of the block.
template <int IN_BF16>
struct MxRow {
  static constexpr int VPV = IN_BF16 ? 8 : 4;  // values per 16-byte vector
  static constexpr int U = IN_BF16 ? 4 : 8;    // 16-byte loads in flight per lane
  static constexpr int SLICE = 32 * U;         // vectors one warp pass covers
};
// tensor_amax (per-tensor FP8): when set, every block uses the one exponent of the whole
// tensor (fp8_tensor_exponent of the tensor's amax) instead of its own.
template <int IN_BF16, typename PutSf>
__device__ __forceinline__ void quantize_row_mx(const uint4* __restrict__ src, int v0, int v1, int lane,
                                                uint8_t* __restrict__ dst, PutSf put_sf,
                                                const uint32_t* __restrict__ tensor_amax = nullptr) {
  const int Xt = tensor_amax ? fp8_tensor_exponent(__ldg(tensor_amax)) : 0;
  constexpr int VPV = MxRow<IN_BF16>::VPV;
  constexpr int LPB = 32 / VPV;  // lanes per 32-value block
  constexpr int U = MxRow<IN_BF16>::U;
  const int row_vecs = v1;
  for (int base = v0; base < row_vecs; base += 32 * U) {
    uint4 q[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = base + 32 * u + lane;
      q[u] = c < row_vecs ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = base + 32 * u + lane;
      const bool act = c < row_vecs;       // whole blocks: row_vecs is a multiple of LPB
      float v[VPV];
      if (IN_BF16) {
        v[0] = bf16_lo(q[u].x); v[1] = bf16_hi(q[u].x); v[2] = bf16_lo(q[u].y); v[3] = bf16_hi(q[u].y);
        v[4] = bf16_lo(q[u].z); v[5] = bf16_hi(q[u].z); v[6] = bf16_lo(q[u].w); v[7] = bf16_hi(q[u].w);
      } else {
        v[0] = __uint_as_float(q[u].x); v[1] = __uint_as_float(q[u].y);
        v[2] = __uint_as_float(q[u].z); v[3] = __uint_as_float(q[u].w);
      }
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < VPV; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
      for (int off = 1; off < LPB; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const int X = tensor_amax ? Xt : mx_exponent(amax);
      const float inv = mx_inv_scale(X);
      if (act) {
        if (IN_BF16) {
          uint2 o;
          o.x = static_cast<uint32_t>(e4m3x2(v[0] * inv, v[1] * inv)) |
                (static_cast<uint32_t>(e4m3x2(v[2] * inv, v[3] * inv)) << 16);
          o.y = static_cast<uint32_t>(e4m3x2(v[4] * inv, v[5] * inv)) |
                (static_cast<uint32_t>(e4m3x2(v[6] * inv, v[7] * inv)) << 16);
          *reinterpret_cast<uint2*>(dst + static_cast<int64_t>(c) * 8) = o;
        } else {
          const uint32_t o = static_cast<uint32_t>(e4m3x2(v[0] * inv, v[1] * inv)) |
                             (static_cast<uint32_t>(e4m3x2(v[2] * inv, v[3] * inv)) << 16);
          *reinterpret_cast<uint32_t*>(dst + static_cast<int64_t>(c) * 4) = o;
        }
        if ((lane % LPB) == 0) put_sf(c * VPV, static_cast<uint8_t>(X + 127));
      }
    }
  }
}

// Row copy with MXFP8 quantisation into the permuted order (scales in the activation SF
// tile layout of the expert m-tiles).  Work items are (row, slice of MxRow::SLICE vectors),
// so short permutations still spread over every SM.  row_src_token == nullptr: the source
// rows are already in routed order (row r from source row r).  mtile_base == nullptr: the
// m-tile table is built from offsets.  tensor_amax: per-tensor FP8 (one exponent for all).
template <int IN_BF16>
__global__ void __launch_bounds__(256) perm_gather_mx_kernel(const uint4* __restrict__ x, int d,
                                                             const int32_t* __restrict__ offsets, int E_loc,
                                                             const int32_t* __restrict__ mtile_base,
                                                             const int32_t* __restrict__ row_src_token,
                                                             uint8_t* __restrict__ perm_x, uint8_t* __restrict__ perm_sf,
                                                             const uint32_t* __restrict__ tensor_amax) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int VPV = IN_BF16 ? 8 : 4;
  extern __shared__ int32_t s_tab[];    // offsets [E_loc+1], mtile_base [E_loc+1]
  if (mtile_base) {
    for (int i = threadIdx.x; i <= E_loc; i += blockDim.x) {
      s_tab[i] = offsets[i];
      s_tab[E_loc + 1 + i] = mtile_base[i];
    }
  } else if (threadIdx.x < 32) {  // no table given: the 128-row m-tile prefix from offsets
    build_mtile_prefix(offsets, E_loc, 128, s_tab, s_tab + E_loc + 1);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int N = s_tab[E_loc];
  const int row_vecs = d / VPV;
  constexpr int SL = MxRow<IN_BF16>::SLICE;
  const int slices = (row_vecs + SL - 1) / SL;
  const int64_t items = static_cast<int64_t>(N) * slices;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items;
       it += warps) {
    const int64_t r = it / slices;
    const int sl = static_cast<int>(it - r * slices);
    // expert of row r: the last e with offsets[e] <= r
    int lo = 0, hi = E_loc - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tab[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    const int il = static_cast<int>(r - s_tab[lo]);
    const int64_t tile = s_tab[E_loc + 1 + lo] + il / 128;
    const int i = il % 128;
    const int64_t t = row_src_token ? __ldg(row_src_token + r) : r;
    quantize_row_mx<IN_BF16>(x + t * row_vecs, sl * SL, min(row_vecs, (sl + 1) * SL), lane, perm_x + r * d,
                             [&](int col, uint8_t b) { perm_sf[sf_act_offset(tile, i, col, d)] = b; }, tensor_amax);
  }
}

// MXFP8 quantisation of token rows in place order: xq [T, d] E4M3 and row-major scales
// x_sf [T, d / 32] (the source of the row-gather GEMM1).  With pair_to_row [T, k], only
// tokens routed to at least one local expert are quantised (the others are never read).
template <int IN_BF16>
__global__ void __launch_bounds__(256) quant_rows_mx_kernel(const uint4* __restrict__ x, int T, int d,
                                                            const int32_t* __restrict__ pair_to_row, int k,
                                                            uint8_t* __restrict__ xq, uint8_t* __restrict__ x_sf) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int VPV = IN_BF16 ? 8 : 4;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int row_vecs = d / VPV;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
    if (pair_to_row) {
      const bool local = lane < k && __ldg(pair_to_row + t * k + lane) >= 0;
      if (!__any_sync(0xffffffffu, local)) continue;
    }
    uint8_t* sf_row = x_sf + t * (d / 32);
    quantize_row_mx<IN_BF16>(x + t * row_vecs, 0, row_vecs, lane, xq + t * d,
                             [&](int col, uint8_t b) { sf_row[col / 32] = b; });
  }
}

cudaError_t launch_quant_rows_mx(const void* x, moe_dtype x_dtype, int T, int d, const int32_t* pair_to_row, int k,
                                 uint8_t* xq, uint8_t* x_sf, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(ceil_div(T, 8), static_cast<int64_t>(num_sms()) * 8));
  cudaError_t e = launch_pdl(x_dtype == MOE_BF16 ? quant_rows_mx_kernel<1> : quant_rows_mx_kernel<0>, dim3(grid),
                             dim3(256), 0, st, static_cast<const uint4*>(x), T, d, pair_to_row, k, xq, x_sf);
  return e != cudaSuccess ? e : cudaGetLastError();
}

struct PermuteWs {
  int32_t* tile_counts;  // [E_loc][n_tiles]
  int32_t* mtile_base;   // [E_loc + 1]
  uint32_t* x_amax;      // per-tensor FP8: largest |x| (fp32 bits)
};

size_t permute_ws_bytes(int T, int E_loc) {
  const int64_t n_tiles = ceil_div(T > 0 ? T : 1, perm_tile(T, E_loc));
  return align_up(static_cast<size_t>(n_tiles) * E_loc * 4, kAlign) + align_up((E_loc + 1) * 4, kAlign) + kAlign;
}

static PermuteWs carve_permute_ws(uint8_t* base, int T, int E_loc) {
  const int64_t n_tiles = ceil_div(T > 0 ? T : 1, perm_tile(T, E_loc));
  PermuteWs w;
  w.tile_counts = reinterpret_cast<int32_t*>(base);
  w.mtile_base = reinterpret_cast<int32_t*>(base + align_up(static_cast<size_t>(n_tiles) * E_loc * 4, kAlign));
  w.x_amax = reinterpret_cast<uint32_t*>(base + align_up(static_cast<size_t>(n_tiles) * E_loc * 4, kAlign) +
                                         align_up((E_loc + 1) * 4, kAlign));
  return w;
}

// m-tile bases [E_loc + 1] (128-row m-tiles of the expert segments, expert order) that the
// permute's scan leaves in its scratch.
int32_t* permute_mtile_base(uint8_t* ws, int T, int E_loc) { return carve_permute_ws(ws, T, E_loc).mtile_base; }

int gather_grid(cudaStream_t st);
// bf16 rows [*, K] into routed order with MXFP8 quantisation (32-blocks along K): dst row r
// = src row row_src_token[r] (or src row r when row_src_token is null) for r <
// offsets[E_loc], E4M3 codes [N_cap, K] and scales in the activation SF tile layout
// (mtile_base from the permute).  K % 128 == 0.
cudaError_t launch_gather_rows_mx(const void* src, int K, const int32_t* offsets, int E_loc,
                                  const int32_t* mtile_base, const int32_t* row_src_token, uint8_t* dst,
                                  uint8_t* dst_sf, cudaStream_t st, const uint32_t* tensor_amax) {
  const size_t sm = static_cast<size_t>(2 * (E_loc + 1)) * 4;
  return launch_pdl(perm_gather_mx_kernel<1>, dim3(gather_grid(st)), dim3(256), sm, st, static_cast<const uint4*>(src),
                    K, offsets, E_loc, mtile_base, row_src_token, dst, dst_sf, tensor_amax);
}

// Rows of src (row_bytes each, a multiple of 16) into routed order: dst row r = src row
// row_src_token[r] for r < offsets[E_loc] (the permute's gather on its own).
cudaError_t launch_gather_rows(const void* src, int64_t row_bytes, const int32_t* offsets, int E_loc,
                               const int32_t* row_src_token, void* dst, cudaStream_t st) {
  return launch_pdl(perm_gather_copy_kernel, dim3(gather_grid(st)), dim3(256), 0, st, static_cast<const uint4*>(src),
                    row_bytes / 16, offsets, E_loc, row_src_token, static_cast<uint4*>(dst));
}

// perm_dtype: MOE_F32 / MOE_BF16 (copy in x's type) or MOE_MXFP8 (quantise).  tok_nloc
// (optional): per-token local slot counts, for the GEMM2 that combines in its epilogue.
cudaError_t launch_permute(const void* x, moe_dtype x_dtype, moe_dtype perm_dtype, int T, int d,
                           const int32_t* ids, const float* probs, int k, int e0, int E_loc, void* perm_x,
                           uint8_t* perm_sf, int32_t* counts, int32_t* offsets, int32_t* row_src_token,
                           float* row_prob, int32_t* pair_to_row, uint8_t* ws, cudaStream_t st,
                           int32_t* tok_nloc) {
  const int tile = perm_tile(T, E_loc);
  const int n_tiles = static_cast<int>(ceil_div(T > 0 ? T : 1, tile));
  PermuteWs w = carve_permute_ws(ws, T, E_loc);
  if (T > 0) {
    cudaError_t e = launch_pdl(tile == kPermTileSmall ? perm_count_kernel<kPermTileSmall>
                                                      : perm_count_kernel<kPermTileLarge>,
                               dim3(n_tiles), dim3(tile), E_loc * 4, st, ids, T, k, e0, E_loc, n_tiles, w.tile_counts);
    if (e != cudaSuccess) return e;
  } else {  // an empty batch: the scan still writes zero counts and offsets
    cudaError_t e = cudaMemsetAsync(w.tile_counts, 0, static_cast<size_t>(n_tiles) * E_loc * 4, st);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, st, w.tile_counts, n_tiles, E_loc, counts,
                             offsets, w.mtile_base);
  if (e != cudaSuccess) return e;
  if (T > 0) {
    e = launch_pdl(tile == kPermTileSmall ? perm_scatter_kernel<kPermTileSmall> : perm_scatter_kernel<kPermTileLarge>,
                   dim3(n_tiles), dim3(tile), E_loc * (tile / 32) * 4, st, ids, probs,
                   T, k, e0, E_loc, n_tiles, static_cast<const int32_t*>(w.tile_counts), pair_to_row, row_src_token,
                   row_prob, tok_nloc);
    if (e != cudaSuccess) return e;
    const int grid = gather_grid(st);
    if (perm_x == nullptr) {
      // maps only: the row-gather GEMM reads x through row_src_token
    } else if (perm_dtype == MOE_MXFP8 || perm_dtype == MOE_FP8) {
      // per-tensor FP8: one exponent for the whole of x [T, d], from its largest magnitude
      if (perm_dtype == MOE_FP8) e = launch_amax(x, x_dtype, static_cast<int64_t>(T) * d, 1, w.x_amax, st);
      if (e != cudaSuccess) return e;
      const size_t sm = static_cast<size_t>(2 * (E_loc + 1)) * 4;
      e = launch_pdl(x_dtype == MOE_BF16 ? perm_gather_mx_kernel<1> : perm_gather_mx_kernel<0>, dim3(grid), dim3(256),
                     sm, st, static_cast<const uint4*>(x), d, static_cast<const int32_t*>(offsets), E_loc,
                     static_cast<const int32_t*>(w.mtile_base), static_cast<const int32_t*>(row_src_token),
                     static_cast<uint8_t*>(perm_x), perm_sf,
                     perm_dtype == MOE_FP8 ? static_cast<const uint32_t*>(w.x_amax) : nullptr);
    } else {
      const int64_t row_vecs = static_cast<int64_t>(d) * (x_dtype == MOE_F32 ? 4 : 2) / 16;
      e = launch_pdl(perm_gather_copy_kernel, dim3(grid), dim3(256), 0, st, static_cast<const uint4*>(x), row_vecs,
                     static_cast<const int32_t*>(offsets), E_loc, static_cast<const int32_t*>(row_src_token),
                     static_cast<uint4*>(perm_x));
    }
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
