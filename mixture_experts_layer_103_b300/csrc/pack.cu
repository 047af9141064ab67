// One-off weight packing (untimed).  From the user layout W_gate, W_up [E_loc, d, f] and
// W_down [E_loc, f, d] to K-major packed matrices for the grouped GEMMs:
//   Wgu [E_loc, 2f, d]: packed row 64*b + i is gate column 32*b + i (i < 32) or up column
//                       32*b + i - 32 (i >= 32), so every 64 packed rows hold a matching
//                       gate/up pair for 32 h columns;
//   Wd  [E_loc, d, f]:  row n is output column n of the down projection.
// In MXFP8 mode each packed row is quantised in blocks of 32 along K ("Efficient MoE
// training for biological foundation models", section "MXFP8 Precision Reduces Memory
// Footprint": one scale per block of 32 consecutive values) and the E8M0 scales go to the
// weight SF tile layout read by the block-scaled MMA.
//
// One lane per source column: for a fixed k the 32 lanes read 32 consecutive columns
// (coalesced), and each lane then owns 32 consecutive K values of its packed row.
#include "moe_common.cuh"

namespace moe {

// OUT: 0 = fp32, 1 = bf16, 2 = MXFP8, 3 = per-tensor FP8 (MXFP8 layout; every block of
// expert e takes the exponent of tensor_amax[e], the amax of that expert's matrix)
template <typename TIn, int OUT>
__global__ void __launch_bounds__(256) pack_kernel(const TIn* __restrict__ src, int K, int ncols, int map_kind,
                                                   int64_t rows_out, void* __restrict__ dst, uint8_t* __restrict__ dst_sf,
                                                   const uint32_t* __restrict__ tensor_amax) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = blockIdx.x * 32 + lane;
  const int e = blockIdx.z;
  const int k0 = (blockIdx.y * 8 + warp) * 32;
  if (k0 >= K) return;
  const bool col_ok = n < ncols;
  // packed row of source column n: 0 = identity, 1 = gate, 2 = up
  const int64_t prow = map_kind == 0 ? n : (static_cast<int64_t>(n / 32) * 64 + (map_kind == 2 ? 32 : 0) + n % 32);
  const TIn* s = src + static_cast<int64_t>(e) * K * ncols;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int k = k0 + i;
    float a = 0.0f;
    if (col_ok && k < K) {
      if constexpr (sizeof(TIn) == 4) a = __ldg(reinterpret_cast<const float*>(s) + static_cast<int64_t>(k) * ncols + n);
      else a = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(s) +
                                                           static_cast<int64_t>(k) * ncols + n)) << 16);
    }
    v[i] = a;
  }
  if (!col_ok) return;
  const int64_t drow = static_cast<int64_t>(e) * rows_out + prow;
  if (OUT == 0) {
    float* d = static_cast<float*>(dst) + drow * K;
    for (int i = 0; i < 32 && k0 + i < K; ++i) d[k0 + i] = v[i];
  } else if (OUT == 1) {
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(dst) + drow * K;
    for (int i = 0; i < 32 && k0 + i < K; ++i) d[k0 + i] = __float2bfloat16_rn(v[i]);
  } else {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int X = OUT == 3 ? fp8_tensor_exponent(__ldg(tensor_amax + e)) : mx_exponent(amax);
    const float inv = mx_inv_scale(X);
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      w[q] = static_cast<uint32_t>(e4m3x2(v[4 * q] * inv, v[4 * q + 1] * inv)) |
             (static_cast<uint32_t>(e4m3x2(v[4 * q + 2] * inv, v[4 * q + 3] * inv)) << 16);
    uint4* d = reinterpret_cast<uint4*>(static_cast<uint8_t*>(dst) + drow * K + k0);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    dst_sf[sf_w_offset(e, rows_out, prow, k0, K)] = static_cast<uint8_t>(X + 127);
  }
}

template <typename TIn, int OUT>
static void pack_one(const void* src, int E_loc, int K, int ncols, int map_kind, int64_t rows_out, void* dst,
                     uint8_t* sf, cudaStream_t st, const uint32_t* tensor_amax = nullptr) {
  const dim3 grid(static_cast<unsigned>(ceil_div(ncols, 32)), static_cast<unsigned>(ceil_div(K, 256)), E_loc);
  pack_kernel<TIn, OUT><<<grid, 256, 0, st>>>(static_cast<const TIn*>(src), K, ncols, map_kind, rows_out, dst, sf,
                                              tensor_amax);
}

cudaError_t launch_pack(const void* Wg, const void* Wu, const void* Wdn, moe_dtype src, moe_dtype dst, int E_loc, int d,
                        int f, void* Wgu_p, void* Wd_p, uint8_t* Wgu_sf, uint8_t* Wd_sf, cudaStream_t st) {
  const int64_t gu_rows = 2LL * f;
#define MOE_PACK3(TIN, OUT)                                                    \
  do {                                                                         \
    pack_one<TIN, OUT>(Wg, E_loc, d, f, 1, gu_rows, Wgu_p, Wgu_sf, st);        \
    pack_one<TIN, OUT>(Wu, E_loc, d, f, 2, gu_rows, Wgu_p, Wgu_sf, st);        \
    pack_one<TIN, OUT>(Wdn, E_loc, f, d, 0, d, Wd_p, Wd_sf, st);               \
  } while (0)
  if (dst == MOE_F32) MOE_PACK3(float, 0);
  else if (dst == MOE_BF16) MOE_PACK3(uint16_t, 1);
  else if (src == MOE_BF16) MOE_PACK3(uint16_t, 2);
  else MOE_PACK3(float, 2);
#undef MOE_PACK3
  return cudaGetLastError();
}

cudaError_t launch_amax(const void* src, moe_dtype dt, int64_t n_per_seg, int n_seg, uint32_t* amax_bits,
                        cudaStream_t st);
cudaError_t launch_fp8_exponents(int32_t* v, int n, cudaStream_t st);

// Per-tensor FP8 packing: w_exp [3, E_loc] receives the amax of each expert's W_gate, W_up
// and W_down (first pass), the matrices are quantised with their exponent into the MXFP8
// packed layouts (every scale byte of a matrix the same), and w_exp is turned into the
// exponents X in place.
cudaError_t launch_pack_fp8(const void* Wg, const void* Wu, const void* Wdn, moe_dtype src, int E_loc, int d, int f,
                            void* Wgu_p, void* Wd_p, uint8_t* Wgu_sf, uint8_t* Wd_sf, int32_t* w_exp,
                            cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(d) * f;
  uint32_t* amax = reinterpret_cast<uint32_t*>(w_exp);
  cudaError_t e = launch_amax(Wg, src, n, E_loc, amax, st);
  if (e == cudaSuccess) e = launch_amax(Wu, src, n, E_loc, amax + E_loc, st);
  if (e == cudaSuccess) e = launch_amax(Wdn, src, n, E_loc, amax + 2 * E_loc, st);
  if (e != cudaSuccess) return e;
  const int64_t gu_rows = 2LL * f;
  if (src == MOE_BF16) {
    pack_one<uint16_t, 3>(Wg, E_loc, d, f, 1, gu_rows, Wgu_p, Wgu_sf, st, amax);
    pack_one<uint16_t, 3>(Wu, E_loc, d, f, 2, gu_rows, Wgu_p, Wgu_sf, st, amax + E_loc);
    pack_one<uint16_t, 3>(Wdn, E_loc, f, d, 0, d, Wd_p, Wd_sf, st, amax + 2 * E_loc);
  } else {
    pack_one<float, 3>(Wg, E_loc, d, f, 1, gu_rows, Wgu_p, Wgu_sf, st, amax);
    pack_one<float, 3>(Wu, E_loc, d, f, 2, gu_rows, Wgu_p, Wgu_sf, st, amax + E_loc);
    pack_one<float, 3>(Wdn, E_loc, f, d, 0, d, Wd_p, Wd_sf, st, amax + 2 * E_loc);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_fp8_exponents(w_exp, 3 * E_loc, st);
}

}  // namespace moe
