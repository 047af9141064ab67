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

// ---------------------------------------------------------------------- MXFP8 backward
// "MXFP8 Precision Reduces Memory Footprint" (8-bit values, one E8M0 scale per 32
// consecutive values, Blackwell MXFP8 GEMMs): every backward GEMM reads its two operands
// quantised in 32-blocks along that GEMM's own contraction axis.

// Weight operands of the two row-wise backward GEMMs, quantised along their K:
//   mode 0: Wd_q [E_loc, f, d] = W_down quantised along d  (B of dh = dy W_down^T, rows f)
//   mode 1: WguT_q [E_loc, d, 2f] = [W_gate W_up] in the packed column order, quantised
//           along f (B of dx = [dg du] [W_gate W_up]^T, rows d); a 32-block of the packed
//           order is 32 consecutive gate (or up) columns of one row
// One thread per (row, 32-block): 64 contiguous source bytes in, 32 codes and one scale
// byte (weight SF tile layout) out.  tensor_exp [3][E_loc] (per-tensor FP8, optional): the
// exponents of each expert's W_gate, W_up, W_down, used for every block of that matrix.
template <typename TIn>
__global__ void __launch_bounds__(256) pack_rows_mx_kernel(const TIn* __restrict__ src0, const TIn* __restrict__ src1,
                                                           int mode, int E_loc, int rows, int K, int f,
                                                           uint8_t* __restrict__ dst, uint8_t* __restrict__ dst_sf,
                                                           const int32_t* __restrict__ tensor_exp) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int nkb = K / 32;
  if (i >= static_cast<int64_t>(E_loc) * rows * nkb) return;
  const int kb = static_cast<int>(i % nkb);
  const int64_t er = i / nkb;  // e * rows + row
  const TIn* s;
  if (mode == 0) s = src0 + er * K + kb * 32;
  else s = ((kb & 1) ? src1 : src0) + er * f + (kb >> 1) * 32;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if constexpr (sizeof(TIn) == 4) v[j] = __ldg(reinterpret_cast<const float*>(s) + j);
    else v[j] = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(s) + j)) << 16);
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const int e_ = static_cast<int>(er / rows);
  const int X = tensor_exp ? __ldg(tensor_exp + (mode == 0 ? 2 : (kb & 1)) * E_loc + e_) : mx_exponent(amax);
  const float inv = mx_inv_scale(X);
  uint32_t w[8];
#pragma unroll
  for (int q = 0; q < 8; ++q)
    w[q] = static_cast<uint32_t>(e4m3x2(v[4 * q] * inv, v[4 * q + 1] * inv)) |
           (static_cast<uint32_t>(e4m3x2(v[4 * q + 2] * inv, v[4 * q + 3] * inv)) << 16);
  uint4* d = reinterpret_cast<uint4*>(dst + er * K + kb * 32);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  const int e = static_cast<int>(er / rows), row = static_cast<int>(er % rows);
  dst_sf[sf_w_offset(e, rows, row, kb * 32, K)] = static_cast<uint8_t>(X + 127);
}

// tensor_exp: nullptr (MXFP8) or the per-tensor FP8 exponents [3][E_loc] of moe_pack_weights_fp8.
cudaError_t launch_pack_backward_mx(const void* Wg, const void* Wu, const void* Wdn, moe_dtype src, int E_loc, int d,
                                    int f, uint8_t* WguT_q, uint8_t* WguT_sf, uint8_t* Wd_q, uint8_t* Wd_sf,
                                    cudaStream_t st, const int32_t* tensor_exp) {
  const int64_t n_d = static_cast<int64_t>(E_loc) * f * (d / 32);
  const int64_t n_gu = static_cast<int64_t>(E_loc) * d * (2 * f / 32);
  const dim3 block(256);
  if (src == MOE_F32) {
    pack_rows_mx_kernel<float><<<dim3(static_cast<unsigned>(ceil_div(n_d, 256))), block, 0, st>>>(
        static_cast<const float*>(Wdn), nullptr, 0, E_loc, f, d, f, Wd_q, Wd_sf, tensor_exp);
    pack_rows_mx_kernel<float><<<dim3(static_cast<unsigned>(ceil_div(n_gu, 256))), block, 0, st>>>(
        static_cast<const float*>(Wg), static_cast<const float*>(Wu), 1, E_loc, d, 2 * f, f, WguT_q, WguT_sf,
        tensor_exp);
  } else {
    pack_rows_mx_kernel<uint16_t><<<dim3(static_cast<unsigned>(ceil_div(n_d, 256))), block, 0, st>>>(
        static_cast<const uint16_t*>(Wdn), nullptr, 0, E_loc, f, d, f, Wd_q, Wd_sf, tensor_exp);
    pack_rows_mx_kernel<uint16_t><<<dim3(static_cast<unsigned>(ceil_div(n_gu, 256))), block, 0, st>>>(
        static_cast<const uint16_t*>(Wg), static_cast<const uint16_t*>(Wu), 1, E_loc, d, 2 * f, f, WguT_q, WguT_sf,
        tensor_exp);
  }
  return cudaGetLastError();
}

// Column-wise MXFP8 quantisation for the weight-gradient GEMMs, which contract over an
// expert's routed rows: each column of buf [rows, C] (bf16, routed order) is quantised in
// blocks of 32 rows counted from the start of its expert's segment (a segment's last
// block is padded with zeros, which never raise a block's amax), and replaced in place by
// the dequantised values code * 2^X.  Those are exactly bf16 values (4 significant bits,
// a power-of-two scale), so the bf16 tensor-core weight-gradient kernel reading them
// forms exactly the products a block-scaled MMA of the E4M3 codes would.  Thread = (32-row
// block, column pair); a CTA row of the grid per expert.
__global__ void __launch_bounds__(128) colquant_mx_kernel(uint32_t* __restrict__ buf, int C,
                                                          const int32_t* __restrict__ offsets) {
  pdl_launch_dependents();
  pdl_wait();
  const int e = blockIdx.y;
  const int r0 = __ldg(offsets + e), cnt = __ldg(offsets + e + 1) - r0;
  const int cpairs = C / 2;
  const int nrb = (cnt + 31) / 32;
  const int ncc = (cpairs + blockDim.x - 1) / blockDim.x;
  for (int item = blockIdx.x; item < nrb * ncc; item += gridDim.x) {
    const int rb = item / ncc, cc = item - rb * ncc;
    const int cp = cc * blockDim.x + threadIdx.x;
    if (cp >= cpairs) continue;
    const int rows = min(32, cnt - rb * 32);
    uint32_t* base = buf + static_cast<int64_t>(r0 + rb * 32) * cpairs + cp;
    float lo[32], hi[32];
    float alo = 0.0f, ahi = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t w = i < rows ? base[static_cast<int64_t>(i) * cpairs] : 0u;
      lo[i] = bf16_lo(w);
      hi[i] = bf16_hi(w);
      alo = fmaxf(alo, fabsf(lo[i]));
      ahi = fmaxf(ahi, fabsf(hi[i]));
    }
    const int Xl = mx_exponent(alo), Xh = mx_exponent(ahi);
    const float il = mx_inv_scale(Xl), ih = mx_inv_scale(Xh);
    const float sl = ldexpf(1.0f, Xl), sh = ldexpf(1.0f, Xh);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < rows) {
        const __nv_fp8x2_storage_t q = e4m3x2(lo[i] * il, hi[i] * ih);
        const float2 dq = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(q, __NV_E4M3)));
        base[static_cast<int64_t>(i) * cpairs] = pack_bf16x2(dq.x * sl, dq.y * sh);
      }
    }
  }
}

// MXFP8 backward, the x or dy rows in one pass: each warp takes a 32-row block of an
// expert's segment (rows in routed order, row r = source row row_src_token[r]) by 32
// columns and writes, from one read, both forms the backward uses:
//   q, q_sf  E4M3 codes with one E8M0 scale per 32 values along the row (the row-wise
//            GEMMs' operand, scales in the activation SF tile layout): what
//            launch_gather_rows_mx writes
//   deq      the bf16 values quantised column-wise (one scale per 32 rows of a column
//            within the segment) and dequantised: what launch_gather_rows followed by
//            launch_colquant_mx leaves
// Lane = row: a row block's scale comes from the lane's own 32 values, a column block's
// from one warp max (redux) per column.  Same arithmetic as those kernels, so the same
// bits.  d % 32 == 0.
__global__ void __launch_bounds__(256) rows_mx_both_kernel(const uint16_t* __restrict__ src, int d,
                                                           const int32_t* __restrict__ offsets, int E_loc,
                                                           const int32_t* __restrict__ mtile_base,
                                                           const int32_t* __restrict__ row_src_token,
                                                           uint8_t* __restrict__ q, uint8_t* __restrict__ q_sf,
                                                           uint16_t* __restrict__ deq) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ int32_t s_tab[];
  int32_t* s_off = s_tab;               // [E_loc + 1] segment starts
  int32_t* s_rbp = s_off + E_loc + 1;   // [E_loc + 1] 32-row blocks before each expert
  int32_t* s_mtb = s_rbp + E_loc + 1;   // [E_loc + 1] 128-row m-tiles before each expert
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const int per = (E_loc + 31) / 32, e_begin = lane * per, e_end = min(E_loc, e_begin + per);
    int sum = 0;
    for (int e = e_begin; e < e_end; ++e) sum += (__ldg(offsets + e + 1) - __ldg(offsets + e) + 31) / 32;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
    for (int e = e_begin; e < e_end; ++e) {
      s_off[e] = __ldg(offsets + e);
      s_rbp[e] = run;
      s_mtb[e] = __ldg(mtile_base + e);
      run += (__ldg(offsets + e + 1) - __ldg(offsets + e) + 31) / 32;
    }
    if (lane == 31) {
      s_off[E_loc] = __ldg(offsets + E_loc);
      s_rbp[E_loc] = incl;
    }
  }
  __syncthreads();
  const int ncb = d / 32;
  const int64_t items = static_cast<int64_t>(s_rbp[E_loc]) * ncb;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items;
       it += nwarps) {
    const int cb = static_cast<int>(it % ncb);
    const int rbg = static_cast<int>(it / ncb);
    int lo = 0, hi = E_loc - 1;  // expert: the last e with s_rbp[e] <= rbg
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_rbp[mid] <= rbg) lo = mid;
      else hi = mid - 1;
    }
    const int e = lo;
    const int il = (rbg - s_rbp[e]) * 32 + lane;  // row within the expert's segment
    const bool valid = il < s_off[e + 1] - s_off[e];
    const int64_t r = static_cast<int64_t>(s_off[e]) + il;
    uint4 a[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                  make_uint4(0u, 0u, 0u, 0u)};
    if (valid) {
      const uint4* p = reinterpret_cast<const uint4*>(src + static_cast<int64_t>(__ldg(row_src_token + r)) * d + cb * 32);
#pragma unroll
      for (int j = 0; j < 4; ++j) a[j] = __ldg(p + j);
    }
    float v[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * j + 0] = bf16_lo(a[j].x); v[8 * j + 1] = bf16_hi(a[j].x);
      v[8 * j + 2] = bf16_lo(a[j].y); v[8 * j + 3] = bf16_hi(a[j].y);
      v[8 * j + 4] = bf16_lo(a[j].z); v[8 * j + 5] = bf16_hi(a[j].z);
      v[8 * j + 6] = bf16_lo(a[j].w); v[8 * j + 7] = bf16_hi(a[j].w);
    }
    // along the row: one block of 32 values
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(v[i]));
    const int X = mx_exponent(am);
    const float inv = mx_inv_scale(X);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      w[j] = static_cast<uint32_t>(e4m3x2(v[4 * j] * inv, v[4 * j + 1] * inv)) |
             (static_cast<uint32_t>(e4m3x2(v[4 * j + 2] * inv, v[4 * j + 3] * inv)) << 16);
    if (valid) {
      uint4* dq = reinterpret_cast<uint4*>(q + r * d + cb * 32);
      dq[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dq[1] = make_uint4(w[4], w[5], w[6], w[7]);
      q_sf[sf_act_offset(s_mtb[e] + il / 128, il % 128, cb * 32, d)] = static_cast<uint8_t>(X + 127);
    }
    // down the columns: a block of the segment's 32 rows per column, from the warp's max
    uint32_t o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float m0 = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[2 * j]))));
      const float m1 = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[2 * j + 1]))));
      const int X0 = mx_exponent(m0), X1 = mx_exponent(m1);
      const __nv_fp8x2_storage_t c = e4m3x2(v[2 * j] * mx_inv_scale(X0), v[2 * j + 1] * mx_inv_scale(X1));
      const float2 f2 = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3)));
      o[j] = pack_bf16x2(f2.x * ldexpf(1.0f, X0), f2.y * ldexpf(1.0f, X1));
    }
    if (valid) {
      uint4* dd = reinterpret_cast<uint4*>(deq + r * d + cb * 32);
#pragma unroll
      for (int j = 0; j < 4; ++j) dd[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
    }
  }
}

cudaError_t launch_rows_mx_both(const void* src, int d, const int32_t* offsets, int E_loc, const int32_t* mtile_base,
                                const int32_t* row_src_token, uint8_t* q, uint8_t* q_sf, void* deq, cudaStream_t st) {
  const size_t sm = static_cast<size_t>(3 * (E_loc + 1)) * 4;
  return launch_pdl(rows_mx_both_kernel, dim3(static_cast<unsigned>(num_sms() * 8)), dim3(256), sm, st,
                    static_cast<const uint16_t*>(src), d, offsets, E_loc, mtile_base, row_src_token, q, q_sf,
                    static_cast<uint16_t*>(deq));
}

cudaError_t launch_colquant_mx(void* buf, int C, const int32_t* offsets, int E_loc, cudaStream_t st) {
  // at least four CTAs per SM over all experts (few local experts: many CTAs per expert)
  const int gx = std::max(32, 4 * num_sms() / E_loc);
  return launch_pdl(colquant_mx_kernel, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(E_loc)), dim3(128), 0,
                    st, static_cast<uint32_t*>(buf), C, offsets);
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
