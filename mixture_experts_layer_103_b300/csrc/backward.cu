// Backward of the expert layer (bf16): the gradient of L = sum_t dy_t . y_t with respect to
// x, the three expert weight tensors and the router logits ("Efficient MoE training for
// biological foundation models", section "GroupedLinear Optimizes Expert Computation":
// the fused GroupedMLP has a matching backward, with the ScaledSwiGLU backward producing
// the scale (routing-probability) gradient).  Per routed row (token t, expert e, prob p):
//   g, u = x W_gate_e, x W_up_e        recomputed (row-gather GEMM, bf16 store)
//   dh = dy_t W_down_e^T                row-gather GEMM on dy with the ScaledSwiGLU backward in
//                                       its epilogue: dg, du (packed order), h, partial dp
//   dx_row = [dg du] [W_gate W_up]^T    grouped GEMM on the packed transposed weights
//   dx_t = sum over the token's slots   (the forward's combine kernel)
//   dlogits: softmax-over-top-k backward of the local dp (non-local slots count as 0)
//   dW_down_e = h^T dy,  dW_gate/up_e = x^T dg / x^T du   (sums over the expert's rows)
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

// ---------------------------------------------------------------------- weight gradients
// C_e = sum over the rows r of expert e's segment of A_r^T B_r (fp32 accumulate), one
// 64 x 64 tile of C per CTA, rows staged 32 at a time through shared memory.
//   MODE 0: dW_down_e [f, d]: A = h rows (direct), B = dy rows (gathered by token)
//   MODE 1: dW_gate_e / dW_up_e [d, f]: A = x rows (gathered), B = dg/du rows (packed
//           order; columns are split back into gate and up on store)
constexpr int kWgTile = 64, kWgRows = 32, kWgPad = 4;

template <int MODE>
__global__ void __launch_bounds__(256) wgrad_kernel(const uint16_t* __restrict__ A, int64_t lda,
                                                    const uint16_t* __restrict__ B, int64_t ldb,
                                                    const int32_t* __restrict__ row_token,
                                                    const int32_t* __restrict__ offsets, int M, int N,
                                                    float* __restrict__ out0, float* __restrict__ out1) {
  pdl_launch_dependents();
  __shared__ __align__(16) float As[kWgRows][kWgTile + kWgPad];
  __shared__ __align__(16) float Bs[kWgRows][kWgTile + kWgPad];
  pdl_wait();
  const int e = blockIdx.z;
  const int m0 = blockIdx.y * kWgTile, n0 = blockIdx.x * kWgTile;
  const int r_begin = __ldg(offsets + e), r_end = __ldg(offsets + e + 1);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  // loader: thread -> (row lr = tid / 8, 8 consecutive columns (tid % 8) * 8)
  const int lr = threadIdx.x >> 3, lc = (threadIdx.x & 7) * 8;
  for (int r0 = r_begin; r0 < r_end; r0 += kWgRows) {
    const int r = r0 + lr;
    float va[8], vb[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) va[q] = vb[q] = 0.0f;
    if (r < r_end) {
      const int64_t ra = MODE == 1 ? __ldg(row_token + r) : r;
      const int64_t rb = MODE == 0 ? __ldg(row_token + r) : r;
      if (m0 + lc < M) {  // M, N are multiples of 8
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(A + ra * lda + m0 + lc));
        va[0] = bf16_lo(a.x); va[1] = bf16_hi(a.x); va[2] = bf16_lo(a.y); va[3] = bf16_hi(a.y);
        va[4] = bf16_lo(a.z); va[5] = bf16_hi(a.z); va[6] = bf16_lo(a.w); va[7] = bf16_hi(a.w);
      }
      if (n0 + lc < N) {
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(B + rb * ldb + n0 + lc));
        vb[0] = bf16_lo(b.x); vb[1] = bf16_hi(b.x); vb[2] = bf16_lo(b.y); vb[3] = bf16_hi(b.y);
        vb[4] = bf16_lo(b.z); vb[5] = bf16_hi(b.z); vb[6] = bf16_lo(b.w); vb[7] = bf16_hi(b.w);
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      As[lr][lc + q] = va[q];
      Bs[lr][lc + q] = vb[q];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kWgRows; ++kk) {
      const float4 a4 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w}, b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      if (MODE == 0) {
        out0[(static_cast<int64_t>(e) * M + m) * N + n] = acc[i][j];
      } else {  // packed column n -> gate or up column
        const int f = N / 2;
        const int col = (n / 64) * 32 + n % 32;
        float* dst = (n % 64) < 32 ? out0 : out1;
        dst[(static_cast<int64_t>(e) * M + m) * f + col] = acc[i][j];
      }
    }
  }
}

cudaError_t launch_dlogits(const int32_t* ids, const float* probs, const int32_t* p2r, const float* dp_part,
                           int nparts, int T, int E, int k, float* dlogits, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(dlogits_kernel, dim3(static_cast<unsigned>(ceil_div(T, 8))), dim3(256), 0, st, ids, probs, p2r,
                    dp_part, nparts, T, E, k, dlogits);
}

cudaError_t launch_wgrad_down(const void* h, const void* dy, const int32_t* row_token, const int32_t* offsets,
                              int E_loc, int d, int f, float* dWd, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(ceil_div(d, kWgTile)), static_cast<unsigned>(ceil_div(f, kWgTile)),
                  static_cast<unsigned>(E_loc));
  return launch_pdl(wgrad_kernel<0>, grid, dim3(256), 0, st, static_cast<const uint16_t*>(h),
                    static_cast<int64_t>(f), static_cast<const uint16_t*>(dy), static_cast<int64_t>(d), row_token,
                    offsets, f, d, dWd, static_cast<float*>(nullptr));
}

cudaError_t launch_wgrad_gate_up(const void* x, const void* dgu, const int32_t* row_token, const int32_t* offsets,
                                 int E_loc, int d, int f, float* dWg, float* dWu, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(ceil_div(2 * f, kWgTile)), static_cast<unsigned>(ceil_div(d, kWgTile)),
                  static_cast<unsigned>(E_loc));
  return launch_pdl(wgrad_kernel<1>, grid, dim3(256), 0, st, static_cast<const uint16_t*>(x),
                    static_cast<int64_t>(d), static_cast<const uint16_t*>(dgu), static_cast<int64_t>(2 * f),
                    row_token, offsets, d, 2 * f, dWg, dWu);
}

}  // namespace moe
