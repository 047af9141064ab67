// Step 5: unpermute + combine ("Wide-EP ... NVIDIA" explainer, section "MoE basics": the
// chosen experts' results are summed; section "Prerequisite ...": combine returns expert
// outputs to their tokens).  One warp per token: the token's k row indices are read once
// and broadcast, the rows of Y2 are summed in slot order in fp32 with 16-byte vector
// loads, and the row of y is written once (zeros when no slot is local).  The routing
// probability was applied inside the SwiGLU, so this is an unweighted sum.
#include "moe_common.cuh"

namespace moe {

template <bool F32>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ Y2, const int32_t* __restrict__ p2r,
                                                      int T, int k, int64_t row_vecs, uint4* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int32_t my_row = lane < k ? __ldg(p2r + t * k + lane) : -1;
  const uint32_t valid = __ballot_sync(0xffffffffu, my_row >= 0);
  uint4* dst = y + t * row_vecs;
  for (int64_t c = lane; c < row_vecs; c += 32) {
    float acc[F32 ? 4 : 8];
#pragma unroll
    for (int u = 0; u < (F32 ? 4 : 8); ++u) acc[u] = 0.0f;
    uint32_t m = valid;
    while (m) {  // slots in ascending order j = 0..k-1
      const int j = __ffs(m) - 1;
      m &= m - 1;
      const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
      const uint4 q = __ldg(Y2 + row * row_vecs + c);
      if (F32) {
        acc[0] += __uint_as_float(q.x); acc[1] += __uint_as_float(q.y);
        acc[2] += __uint_as_float(q.z); acc[3] += __uint_as_float(q.w);
      } else {
        acc[0] += bf16_lo(q.x); acc[1] += bf16_hi(q.x); acc[2] += bf16_lo(q.y); acc[3] += bf16_hi(q.y);
        acc[4] += bf16_lo(q.z); acc[5] += bf16_hi(q.z); acc[6] += bf16_lo(q.w); acc[7] += bf16_hi(q.w);
      }
    }
    uint4 o;
    if (F32) {
      o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                     __float_as_uint(acc[3]));
    } else {
      o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                     pack_bf16x2(acc[6], acc[7]));
    }
    dst[c] = o;
  }
}

cudaError_t launch_combine(const void* Y2, const int32_t* p2r, int T, int k, int d, moe_dtype dtype, void* y,
                           cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const bool f32 = dtype == MOE_F32;
  const int64_t row_vecs = static_cast<int64_t>(d) * (f32 ? 4 : 2) / 16;
  const dim3 grid(static_cast<unsigned>(ceil_div(T, 8))), block(256);
  if (f32)
    combine_kernel<true><<<grid, block, 0, st>>>(static_cast<const uint4*>(Y2), p2r, T, k, row_vecs,
                                                 static_cast<uint4*>(y));
  else
    combine_kernel<false><<<grid, block, 0, st>>>(static_cast<const uint4*>(Y2), p2r, T, k, row_vecs,
                                                  static_cast<uint4*>(y));
  return cudaGetLastError();
}

}  // namespace moe
