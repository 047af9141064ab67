// fp32 grouped expert MLP on the SIMT FMA pipes (the fp32 layer: tf32 tensor cores cannot
// hold a 1e-5 relative error).  Same packed weights and the same fused epilogue as the
// tensor-core path ("Efficient MoE training for biological foundation models", section
// "GroupedLinear Optimizes Expert Computation": GroupedLinear -> ScaledSwiGLU ->
// GroupedLinear, probabilities applied inside the activation).
//
// Tile: 64 rows of one expert's segment x 64 packed output columns, K in chunks of 32
// staged through shared memory; 256 threads, 4 x 4 fp32 accumulators each.  In the
// GEMM1 tile the 64 packed columns are 32 gate + 32 up columns of the same f-range, so
// each thread holds matching gate/up pairs and writes h directly.
#include "moe_common.cuh"

namespace moe {

constexpr int kSimtBM = 64, kSimtBN = 64, kSimtBK = 32;

template <bool SWIGLU>
__global__ void __launch_bounds__(256) simt_grouped_gemm_kernel(const float* __restrict__ A, int K,
                                                                const int32_t* __restrict__ offsets, int E_loc,
                                                                const float* __restrict__ B, int n_out,
                                                                const float* __restrict__ row_prob,
                                                                float* __restrict__ out, int64_t ld_out) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ int s_tab[];  // s_off [E_loc+1], s_mtp [E_loc+1]
  __shared__ float As[kSimtBK][kSimtBM + 4];
  __shared__ float Bs[kSimtBK][kSimtBN + 4];
  int* s_off = s_tab;
  int* s_mtp = s_tab + E_loc + 1;
  if (threadIdx.x < 32) build_mtile_prefix(offsets, E_loc, kSimtBM, s_off, s_mtp);
  __syncthreads();
  const int gm = blockIdx.x;
  if (gm >= s_mtp[E_loc]) return;
  int lo = 0, hi = E_loc - 1;  // expert of m-tile gm: last e with s_mtp[e] <= gm
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_mtp[mid] <= gm) lo = mid;
    else hi = mid - 1;
  }
  const int e = lo;
  const int row0 = s_off[e] + (gm - s_mtp[e]) * kSimtBM;
  const int rows = min(kSimtBM, s_off[e + 1] - row0);
  const int n0 = blockIdx.y * kSimtBN;  // packed output column
  const float* Be = B + static_cast<int64_t>(e) * n_out * K;

  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  int col[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) col[q] = SWIGLU ? ((q >> 1) * 32 + tx * 2 + (q & 1)) : (tx * 4 + q);
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kSimtBK) {
    for (int i = threadIdx.x; i < kSimtBM * kSimtBK; i += 256) {
      const int r = i / kSimtBK, kk = i % kSimtBK;
      As[kk][r] = (r < rows && k0 + kk < K) ? __ldg(A + static_cast<int64_t>(row0 + r) * K + k0 + kk) : 0.0f;
      const int n = n0 + r;
      Bs[kk][r] = (n < n_out && k0 + kk < K) ? __ldg(Be + static_cast<int64_t>(n) * K + k0 + kk) : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kSimtBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int q = 0; q < 4; ++q) b[q] = Bs[kk][col[q]];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(a[i], b[q], acc[i][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= rows) continue;
    const int64_t grow = row0 + r;
    if (SWIGLU) {
      const float p = __ldg(row_prob + grow);
      const int f0 = n0 / 2;  // packed block of 64 columns -> 32 h columns
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float g = acc[i][q], u = acc[i][q + 2];
        const int fc = f0 + tx * 2 + q;
        if (fc < n_out / 2) out[grow * ld_out + fc] = p * (g / (1.0f + expf(-g))) * u;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = n0 + col[q];
        if (n < n_out) out[grow * ld_out + n] = acc[i][q];
      }
    }
  }
}

// GEMM1 (+ scaled SwiGLU), fp32: perm_x [N_cap, d] -> h [N_cap, f].
cudaError_t launch_simt_gemm1(const float* perm_x, const int32_t* offsets, const float* row_prob, int64_t N_cap,
                              int E_loc, int d, int f, const float* Wgu, float* h, cudaStream_t st) {
  const unsigned mt = static_cast<unsigned>(ceil_div(N_cap, kSimtBM) + E_loc);
  const size_t sm = static_cast<size_t>(2 * (E_loc + 1)) * 4;
  return launch_pdl(simt_grouped_gemm_kernel<true>, dim3(mt, static_cast<unsigned>(ceil_div(2 * f, kSimtBN))),
                    dim3(256), sm, st, perm_x, d, offsets, E_loc, Wgu, 2 * f, row_prob, h, static_cast<int64_t>(f));
}

// GEMM2, fp32: h [N_cap, f] -> Y2 [N_cap, d].
cudaError_t launch_simt_gemm2(const float* h, const int32_t* offsets, int64_t N_cap, int E_loc, int d, int f,
                              const float* Wd, float* Y2, cudaStream_t st) {
  const unsigned mt = static_cast<unsigned>(ceil_div(N_cap, kSimtBM) + E_loc);
  const size_t sm = static_cast<size_t>(2 * (E_loc + 1)) * 4;
  return launch_pdl(simt_grouped_gemm_kernel<false>, dim3(mt, static_cast<unsigned>(ceil_div(d, kSimtBN))), dim3(256),
                    sm, st, h, f, offsets, E_loc, Wd, d, static_cast<const float*>(nullptr), Y2,
                    static_cast<int64_t>(d));
}

}  // namespace moe
