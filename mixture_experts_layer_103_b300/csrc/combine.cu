// Step 5: unpermute + combine ("Wide-EP ... NVIDIA" explainer, section "MoE basics": the
// chosen experts' results are summed; section "Prerequisite ...": combine returns expert
// outputs to their tokens).  One warp per token: the token's k row indices are read once
// and broadcast, the rows of Y2 are summed in slot order in fp32 with 16-byte vector
// loads, and the row of y is written once (zeros when no slot is local).  The routing
// probability was applied inside the SwiGLU, so this is an unweighted sum.
//
// Work item = (token, slice of kCombineSlice 16-byte vectors of its row), grid-strided
// over a persistent grid: a wide row (d = 7168) is spread over several warps, and each
// lane issues the loads of its 4 vectors for up to 4 slots at once, so even a token with
// one local slot keeps several loads in flight.
#include <algorithm>

#include "moe_common.cuh"

namespace moe {

int num_sms();

constexpr int kCombineGroup = 4;    // slots whose loads are in flight together
constexpr int kCombineSlice = 128;  // 16-byte vectors per work item (4 per lane)

// Slot-ordered sum of one token's 16-byte vectors [c_begin, c_end) by one warp: rows
// my_row (this lane's slot j = lane, -1 if not local), up to kCombineGroup slots' loads of
// S vectors per lane in flight at once, fp32 accumulation from zero in slot order, one
// rounding; written to dst (the token's row of y).
template <bool F32>
__device__ __forceinline__ void sum_token_slice(const uint4* __restrict__ Y2, int64_t row_vecs, int32_t my_row,
                                                int64_t c_begin, int64_t c_end, int lane, uint4* __restrict__ dst) {
  constexpr int V = F32 ? 4 : 8;                // values per 16-byte vector
  constexpr int S = kCombineSlice / 32;         // vectors per lane per item
  constexpr int G = kCombineGroup;
  const uint32_t valid = __ballot_sync(0xffffffffu, my_row >= 0);  // local slots, ascending j
  const int nv = __popc(valid);
  float acc[S][V];
#pragma unroll
  for (int s = 0; s < S; ++s)
#pragma unroll
    for (int u = 0; u < V; ++u) acc[s][u] = 0.0f;
  uint32_t m = valid;
  for (int g = 0; g < nv; g += G) {
    // the loads of up to G slots x S vectors are issued together, then added in slot order
    uint4 q[G][S];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      int64_t row = 0;
      if (g + j < nv) {  // warp-uniform
        const int src = __ffs(m) - 1;
        m &= m - 1;
        row = __shfl_sync(0xffffffffu, my_row, src);
      }
#pragma unroll
      for (int s = 0; s < S; ++s) {
        const int64_t c = c_begin + lane + 32 * s;
        q[j][s] = (g + j < nv && c < c_end) ? __ldg(Y2 + row * row_vecs + c) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
      if (g + j < nv) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
          if (F32) {
            acc[s][0] += __uint_as_float(q[j][s].x); acc[s][1] += __uint_as_float(q[j][s].y);
            acc[s][2] += __uint_as_float(q[j][s].z); acc[s][3] += __uint_as_float(q[j][s].w);
          } else {
            acc[s][0] += bf16_lo(q[j][s].x); acc[s][1] += bf16_hi(q[j][s].x);
            acc[s][2] += bf16_lo(q[j][s].y); acc[s][3] += bf16_hi(q[j][s].y);
            acc[s][4] += bf16_lo(q[j][s].z); acc[s][5] += bf16_hi(q[j][s].z);
            acc[s][6] += bf16_lo(q[j][s].w); acc[s][7] += bf16_hi(q[j][s].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int64_t c = c_begin + lane + 32 * s;
    uint4 o;
    if (F32) {
      o = make_uint4(__float_as_uint(acc[s][0]), __float_as_uint(acc[s][1]), __float_as_uint(acc[s][2]),
                     __float_as_uint(acc[s][3]));
    } else {
      o = make_uint4(pack_bf16x2(acc[s][0], acc[s][1]), pack_bf16x2(acc[s][2], acc[s][3]),
                     pack_bf16x2(acc[s][4], acc[s][5]), pack_bf16x2(acc[s][6], acc[s][7]));
    }
    if (c < c_end) __stcs(dst + c, o);  // y is written once and not re-read: streaming store
  }
}

// MULTI_ONLY: only tokens with two or more local slots (GEMM2 wrote the others' rows).
template <bool F32, bool MULTI_ONLY>
__global__ void __launch_bounds__(256, 2) combine_kernel(const uint4* __restrict__ Y2, const int32_t* __restrict__ p2r,
                                                      int T, int k, int64_t row_vecs, int slices,
                                                      uint4* __restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t items = static_cast<int64_t>(T) * slices;
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items;
       item += warps) {
    const int64_t t = item / slices;
    const int64_t c_begin = (item - t * slices) * kCombineSlice;
    const int64_t c_end = std::min<int64_t>(row_vecs, c_begin + kCombineSlice);
    const int32_t my_row = lane < k ? __ldg(p2r + t * k + lane) : -1;
    if (MULTI_ONLY && __popc(__ballot_sync(0xffffffffu, my_row >= 0)) < 2) continue;  // warp-uniform
    sum_token_slice<F32>(Y2, row_vecs, my_row, c_begin, c_end, lane, y + t * row_vecs);
  }
}

// Sparse multi-slot combine: few tokens have two or more local slots (the expert slices of
// a wide layer).  Work items are (32 consecutive tokens, one 128-vector slice of the row):
// a warp reads the 32 tokens' slot counts with one load and sums its slice of those with
// two or more; every other row of y was written by GEMM2.
__global__ void __launch_bounds__(256) combine_sparse_kernel(const uint4* __restrict__ Y2,
                                                             const int32_t* __restrict__ p2r,
                                                             const int32_t* __restrict__ tok_nloc, int T, int k,
                                                             int64_t row_vecs, int slices, uint4* __restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t items = (static_cast<int64_t>(T) + 31) / 32 * slices;
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); item < items;
       item += warps) {
    const int64_t ch = item / slices;
    const int64_t c_begin = (item - ch * slices) * kCombineSlice;
    const int64_t c_end = std::min<int64_t>(row_vecs, c_begin + kCombineSlice);
    const int64_t t0 = ch * 32;
    const int nl = t0 + lane < T ? __ldg(tok_nloc + t0 + lane) : 0;
    uint32_t mt = __ballot_sync(0xffffffffu, nl >= 2);
    while (mt != 0u) {
      const int64_t t = t0 + __ffs(mt) - 1;
      mt &= mt - 1;
      const int32_t my_row = lane < k ? __ldg(p2r + t * k + lane) : -1;
      sum_token_slice<false>(Y2, row_vecs, my_row, c_begin, c_end, lane, y + t * row_vecs);
    }
  }
}

// Sum of the tokens with two or more local slots only, bf16 (GEMM2 wrote every other row
// of y): the sparse kernel when tokens average under one local slot, else the (token,
// slice) kernel skipping the tokens with fewer than two.
cudaError_t launch_combine(const void* Y2, const int32_t* p2r, int T, int k, int d, moe_dtype dtype, void* y,
                           cudaStream_t st, bool multi_only);

cudaError_t launch_combine_multi(const void* Y2, const int32_t* p2r, const int32_t* tok_nloc, int T, int k, int d,
                                 void* y, double slots_per_token, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (slots_per_token >= 1.0) return launch_combine(Y2, p2r, T, k, d, MOE_BF16, y, st, /*multi_only=*/true);
  const int64_t row_vecs = static_cast<int64_t>(d) * 2 / 16;
  const int slices = static_cast<int>(ceil_div(row_vecs, kCombineSlice));
  const int64_t items = ceil_div(T, 32) * slices;
  const dim3 grid(static_cast<unsigned>(std::min<int64_t>(ceil_div(items, 8), static_cast<int64_t>(num_sms()) * 4)));
  return launch_pdl(combine_sparse_kernel, grid, dim3(256), 0, st, static_cast<const uint4*>(Y2), p2r, tok_nloc, T, k,
                    row_vecs, slices, static_cast<uint4*>(y));
}

cudaError_t launch_combine(const void* Y2, const int32_t* p2r, int T, int k, int d, moe_dtype dtype, void* y,
                           cudaStream_t st, bool multi_only) {
  if (T == 0) return cudaSuccess;
  const bool f32 = dtype == MOE_F32;
  const int64_t row_vecs = static_cast<int64_t>(d) * (f32 ? 4 : 2) / 16;
  const int slices = static_cast<int>(ceil_div(row_vecs, kCombineSlice));
  const int64_t items = static_cast<int64_t>(T) * slices;
  const dim3 grid(static_cast<unsigned>(std::min<int64_t>(ceil_div(items, 8), static_cast<int64_t>(num_sms()) * 4))),
      block(256);
  auto kern = f32 ? (multi_only ? combine_kernel<true, true> : combine_kernel<true, false>)
                  : (multi_only ? combine_kernel<false, true> : combine_kernel<false, false>);
  return launch_pdl(kern, grid, block, 0, st, static_cast<const uint4*>(Y2), p2r, T, k, row_vecs, slices,
                    static_cast<uint4*>(y));
}

}  // namespace moe
