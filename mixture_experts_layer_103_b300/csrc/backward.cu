// Backward of the expert layer (bf16): the gradient of L = sum_t dy_t . y_t with respect to
// x, the three expert weight tensors and the router logits ("Efficient MoE training for
// biological foundation models", section "GroupedLinear Optimizes Expert Computation":
// the fused GroupedMLP has a matching backward, with the ScaledSwiGLU backward producing
// the scale (routing-probability) gradient).  Per routed row (token t, expert e, prob p),
// with x and dy first copied into routed-row order (TMA-loadable operands):
//   g, u = x W_gate_e, x W_up_e        kept by the training forward, else recomputed (bf16
//                                       store GEMM on the x rows)
//   dh = dy_t W_down_e^T                grouped GEMM on the dy rows with the ScaledSwiGLU
//                                       backward in its epilogue: dg, du (packed order), h,
//                                       partial dp
//   dx_row = [dg du] [W_gate W_up]^T    grouped GEMM on the packed transposed weights
//   dx_t = sum over the token's slots   (the forward's combine kernel)
//   dlogits: softmax-over-top-k backward of the local dp (non-local slots count as 0)
//   dW_down_e = h^T dy,  dW_gate/up_e = x^T dg / x^T du   (sums over the expert's rows;
//                                       tensor-core kernel in wgrad_tc.cu)
#include <algorithm>

#include "moe_common.cuh"

namespace moe {

int num_sms();

// ---------------------------------------------------------------------- weight pack
// WguT [E_loc, d, 2f]: row c is row c of W_gate and of W_up interleaved in 32-column
// blocks (packed column 64b + i = gate column 32b + i, 64b + 32 + i = up column 32b + i),
// so dx = [dg du] WguT^T contracts over the packed order dg/du are stored in.
template <typename TIn>
__global__ void __launch_bounds__(256) pack_gu_t_kernel(const TIn* __restrict__ Wg, const TIn* __restrict__ Wu,
                                                        int64_t rows, int f, __nv_bfloat16* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // output element
  const int64_t n2 = 2 * static_cast<int64_t>(f);
  if (i >= rows * n2) return;
  const int64_t row = i / n2;
  const int pc = static_cast<int>(i - row * n2);
  const int col = (pc / 64) * 32 + pc % 32;
  const TIn* src = (pc % 64) < 32 ? Wg : Wu;
  float v;
  if constexpr (sizeof(TIn) == 4) v = __ldg(reinterpret_cast<const float*>(src) + row * f + col);
  else v = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(src) + row * f + col)) << 16);
  out[i] = __float2bfloat16_rn(v);
}

cudaError_t launch_pack_gu_t(const void* Wg, const void* Wu, moe_dtype src, int E_loc, int d, int f, void* WguT,
                             cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(E_loc) * d;
  const int64_t n = rows * 2 * f;
  const dim3 grid(static_cast<unsigned>(ceil_div(n, 256))), block(256);
  if (src == MOE_F32)
    pack_gu_t_kernel<float><<<grid, block, 0, st>>>(static_cast<const float*>(Wg), static_cast<const float*>(Wu),
                                                     rows, f, static_cast<__nv_bfloat16*>(WguT));
  else
    pack_gu_t_kernel<uint16_t><<<grid, block, 0, st>>>(static_cast<const uint16_t*>(Wg),
                                                        static_cast<const uint16_t*>(Wu), rows, f,
                                                        static_cast<__nv_bfloat16*>(WguT));
  return cudaGetLastError();
}

// ---------------------------------------------------------------------- router gradient
// One warp per token.  Lane j < k: dp_j = sum over the f / 32 partial sums of its row (in
// order) when slot j is local, else 0; then dlogit_{id_j} = p_j (dp_j - sum_i p_i dp_i), the
// other E - k logits 0.  The sum over slots is a fixed butterfly (deterministic).
__global__ void __launch_bounds__(256) dlogits_kernel(const int32_t* __restrict__ ids, const float* __restrict__ probs,
                                                      const int32_t* __restrict__ p2r,
                                                      const float* __restrict__ dp_part, int nparts, int T, int E,
                                                      int k, float* __restrict__ dlogits) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float p = 0.0f, dp = 0.0f;
  int id = 0;
  if (lane < k) {
    p = __ldg(probs + t * k + lane);
    id = __ldg(ids + t * k + lane);
    const int32_t row = __ldg(p2r + t * k + lane);
    if (row >= 0)
      for (int b = 0; b < nparts; ++b) dp += __ldg(dp_part + static_cast<int64_t>(row) * nparts + b);
  }
  float s = p * dp;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  float* out = dlogits + t * E;
  for (int q = lane; q < E; q += 32) out[q] = 0.0f;
  __syncwarp();
  if (lane < k) out[id] = p * (dp - s);
}

cudaError_t launch_dlogits(const int32_t* ids, const float* probs, const int32_t* p2r, const float* dp_part,
                           int nparts, int T, int E, int k, float* dlogits, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(dlogits_kernel, dim3(static_cast<unsigned>(ceil_div(T, 8))), dim3(256), 0, st, ids, probs, p2r,
                    dp_part, nparts, T, E, k, dlogits);
}

}  // namespace moe
