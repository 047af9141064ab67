// fp32 grouped expert MLP on the SIMT FMA pipes (the fp32 layer: tf32 tensor cores cannot
// hold a 1e-5 relative error).  Same packed weights and the same fused epilogue as the
// tensor-core path ("Efficient MoE training for biological foundation models", section
// "GroupedLinear Optimizes Expert Computation": GroupedLinear -> ScaledSwiGLU ->
// GroupedLinear, probabilities applied inside the activation).
//
// Tile: 16 rows of one expert's segment x 64 packed output columns; K is staged through
// shared memory in chunks of up to 256 with every load of a chunk in flight at once
// (16-byte vectors), so a small layer costs one or two memory round trips per GEMM.
// 256 threads: thread (row = tid / 16, column group = tid % 16) holds 4 accumulators.  In
// GEMM1 the 64 packed columns are 32 gate + 32 up columns of one f-range, so each thread
// holds matching gate/up pairs and writes h directly.
#include "moe_common.cuh"

namespace moe {

constexpr int kSimtBM = 16, kSimtBN = 64, kSimtBK = 256, kSimtPad = 1;
constexpr int kStageIters = (kSimtBM + kSimtBN) * (kSimtBK / 4) / 256;  // float4 loads per thread per chunk
static_assert((kSimtBM + kSimtBN) * (kSimtBK / 4) % 256 == 0, "staging covers the chunk exactly");

template <bool SWIGLU>
__global__ void __launch_bounds__(256) simt_grouped_gemm_kernel(const float* __restrict__ A, int K,
                                                                const int32_t* __restrict__ offsets, int E_loc,
                                                                const float* __restrict__ B, int n_out,
                                                                const float* __restrict__ row_prob,
                                                                float* __restrict__ out, int64_t ld_out) {
  pdl_launch_dependents();
  extern __shared__ float s_dyn[];
  int* s_off = reinterpret_cast<int*>(s_dyn);     // [E_loc + 1]
  int* s_mtp = s_off + E_loc + 1;                 // [E_loc + 1]
  float* As = s_dyn + align_up(2 * (E_loc + 1), 4);  // [kSimtBM][kSimtBK + pad]
  float* Bs = As + kSimtBM * (kSimtBK + kSimtPad);   // [kSimtBN][kSimtBK + pad]
  constexpr int LD = kSimtBK + kSimtPad;
  pdl_wait();
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

  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // ty = row in the tile
  int col[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) col[q] = SWIGLU ? ((q >> 1) * 32 + tx * 2 + (q & 1)) : (tx * 4 + q);
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const bool vec = (K % 4) == 0;  // rows 16-byte aligned
  for (int k0 = 0; k0 < K; k0 += kSimtBK) {
    const int kc = min(kSimtBK, K - k0);
    // stage A [16 x kc] and B [64 x kc]: every load of the chunk into registers first,
    // then into shared memory
    float4 buf[kStageIters];
#pragma unroll
    for (int it = 0; it < kStageIters; ++it) {
      const int i = threadIdx.x + it * 256;
      const int r = i / (kSimtBK / 4), c4 = (i % (kSimtBK / 4)) * 4;
      const bool is_a = r < kSimtBM;
      const int rr = is_a ? r : r - kSimtBM;
      const bool ok = c4 < kc && (is_a ? rr < rows : n0 + rr < n_out);
      const float* src = is_a ? A + static_cast<int64_t>(row0 + rr) * K + k0 + c4
                              : Be + static_cast<int64_t>(n0 + rr) * K + k0 + c4;
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (ok) {
        if (vec && c4 + 4 <= kc) {
          v = __ldg(reinterpret_cast<const float4*>(src));
        } else {
          v.x = __ldg(src);
          if (c4 + 1 < kc) v.y = __ldg(src + 1);
          if (c4 + 2 < kc) v.z = __ldg(src + 2);
          if (c4 + 3 < kc) v.w = __ldg(src + 3);
        }
      }
      buf[it] = v;
    }
#pragma unroll
    for (int it = 0; it < kStageIters; ++it) {
      const int i = threadIdx.x + it * 256;
      const int r = i / (kSimtBK / 4), c4 = (i % (kSimtBK / 4)) * 4;
      float* dst = (r < kSimtBM ? As + r * LD : Bs + (r - kSimtBM) * LD) + c4;
      dst[0] = buf[it].x;
      dst[1] = buf[it].y;
      dst[2] = buf[it].z;
      dst[3] = buf[it].w;
    }
    __syncthreads();
    const float* a = As + ty * LD;
#pragma unroll 8
    for (int kk = 0; kk < kc; ++kk) {
      const float av = a[kk];
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] = fmaf(av, Bs[col[q] * LD + kk], acc[q]);
    }
    __syncthreads();
  }
  if (ty >= rows) return;
  const int64_t grow = row0 + ty;
  if (SWIGLU) {
    const float p = __ldg(row_prob + grow);
    const int f0 = n0 / 2;  // packed block of 64 columns -> 32 h columns
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float g = acc[q], u = acc[q + 2];
      const int fc = f0 + tx * 2 + q;
      if (fc < n_out / 2) out[grow * ld_out + fc] = p * (g / (1.0f + expf(-g))) * u;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + col[q];
      if (n < n_out) out[grow * ld_out + n] = acc[q];
    }
  }
}

static size_t simt_smem_bytes(int E_loc) {
  return align_up(2 * (E_loc + 1), 4) * 4 + static_cast<size_t>(kSimtBM + kSimtBN) * (kSimtBK + kSimtPad) * 4;
}

// Opt the kernel into its largest dynamic shared memory (E_loc = 1024) once per device,
// outside any stream capture that may come later.
template <bool SWIGLU>
static cudaError_t simt_attr() {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && attr_set[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(simt_grouped_gemm_kernel<SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(simt_smem_bytes(1024)));
  if (e == cudaSuccess && dev >= 0 && dev < 64) attr_set[dev] = true;
  return e;
}

// GEMM1 (+ scaled SwiGLU), fp32: perm_x [N_cap, d] -> h [N_cap, f].
cudaError_t launch_simt_gemm1(const float* perm_x, const int32_t* offsets, const float* row_prob, int64_t N_cap,
                              int E_loc, int d, int f, const float* Wgu, float* h, cudaStream_t st) {
  const unsigned mt = static_cast<unsigned>(ceil_div(N_cap, kSimtBM) + E_loc);
  const size_t sm = simt_smem_bytes(E_loc);
  cudaError_t e = simt_attr<true>();
  if (e != cudaSuccess) return e;
  return launch_pdl(simt_grouped_gemm_kernel<true>, dim3(mt, static_cast<unsigned>(ceil_div(2 * f, kSimtBN))),
                    dim3(256), sm, st, perm_x, d, offsets, E_loc, Wgu, 2 * f, row_prob, h, static_cast<int64_t>(f));
}

// GEMM2, fp32: h [N_cap, f] -> Y2 [N_cap, d].
cudaError_t launch_simt_gemm2(const float* h, const int32_t* offsets, int64_t N_cap, int E_loc, int d, int f,
                              const float* Wd, float* Y2, cudaStream_t st) {
  const unsigned mt = static_cast<unsigned>(ceil_div(N_cap, kSimtBM) + E_loc);
  const size_t sm = simt_smem_bytes(E_loc);
  cudaError_t e = simt_attr<false>();
  if (e != cudaSuccess) return e;
  return launch_pdl(simt_grouped_gemm_kernel<false>, dim3(mt, static_cast<unsigned>(ceil_div(d, kSimtBN))), dim3(256),
                    sm, st, h, f, offsets, E_loc, Wd, d, static_cast<const float*>(nullptr), Y2,
                    static_cast<int64_t>(d));
}

}  // namespace moe
