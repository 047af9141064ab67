// Per-tensor FP8 support: largest magnitude of a tensor (the scale of per-tensor current
// scaling) and its conversion into the tensor's exponent.
//
// "Efficient MoE training for biological foundation models", section "MXFP8 Precision
// Reduces Memory Footprint": the layer runs in FP8 as well as MXFP8.  Per-tensor FP8 gives
// a whole tensor one scale; here it is a power of two, 2^X with X the smallest integer
// such that amax <= 448 * 2^X (fp8_tensor_exponent), so the E4M3 codes of v / 2^X never
// saturate and the block-scaled MMAs run the tensor with every block scale set to X.
#include <algorithm>

#include "moe_common.cuh"

namespace moe {

// Largest |value| of one 16-byte vector (8 bf16 or 4 fp32 values).
template <int IN_BF16>
__device__ __forceinline__ float vec_amax(const uint4 q) {
  if (IN_BF16)
    return fmaxf(fmaxf(fmaxf(fabsf(bf16_lo(q.x)), fabsf(bf16_hi(q.x))), fmaxf(fabsf(bf16_lo(q.y)), fabsf(bf16_hi(q.y)))),
                 fmaxf(fmaxf(fabsf(bf16_lo(q.z)), fabsf(bf16_hi(q.z))), fmaxf(fabsf(bf16_lo(q.w)), fabsf(bf16_hi(q.w)))));
  return fmaxf(fmaxf(fabsf(__uint_as_float(q.x)), fabsf(__uint_as_float(q.y))),
               fmaxf(fabsf(__uint_as_float(q.z)), fabsf(__uint_as_float(q.w))));
}

// amax of n_seg segments of n values each (segment s at src + s * n): blockIdx.y = segment,
// grid-stride over 16-byte vectors with four independent loads in flight per thread, one
// atomicMax per block on the fp32 bits (non-negative floats order like their bit
// patterns).  n is a multiple of 8 (bf16) or 4 (fp32).  n_rows (optional, device): the
// segment is its first *n_rows rows of row_vecs vectors.
template <int IN_BF16>
__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ src, int64_t nvec, uint32_t* amax_bits,
                                                   const int32_t* __restrict__ n_rows, int64_t row_vecs) {
  pdl_launch_dependents();
  pdl_wait();
  if (n_rows) nvec = min(nvec, static_cast<int64_t>(__ldg(n_rows)) * row_vecs);
  const uint4* s = src + static_cast<int64_t>(blockIdx.y) * nvec;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  float m = 0.0f;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    const uint4 q0 = __ldg(s + i), q1 = __ldg(s + i + stride), q2 = __ldg(s + i + 2 * stride),
                q3 = __ldg(s + i + 3 * stride);
    m = fmaxf(m, fmaxf(fmaxf(vec_amax<IN_BF16>(q0), vec_amax<IN_BF16>(q1)),
                       fmaxf(vec_amax<IN_BF16>(q2), vec_amax<IN_BF16>(q3))));
  }
  for (; i < nvec; i += stride) m = fmaxf(m, vec_amax<IN_BF16>(__ldg(s + i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float s_m[8];
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, s_m[w]);
    atomicMax(amax_bits + blockIdx.y, __float_as_uint(m));
  }
}

// amax_bits[s] = largest |value| of segment s (fp32 bits), zeroed first.
cudaError_t launch_amax(const void* src, moe_dtype dt, int64_t n_per_seg, int n_seg, uint32_t* amax_bits,
                        cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, static_cast<size_t>(n_seg) * 4, st);
  if (e != cudaSuccess || n_per_seg == 0 || n_seg == 0) return e;
  const int vpv = dt == MOE_BF16 ? 8 : 4;
  const int64_t nvec = n_per_seg / vpv;
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = ceil_div(nvec, 256 * 8);  // ~8 vectors per thread
  const int gx = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, std::max(1, 4 * sms / n_seg))));
  return launch_pdl(dt == MOE_BF16 ? amax_kernel<1> : amax_kernel<0>, dim3(gx, n_seg), dim3(256), 0, st,
                    static_cast<const uint4*>(src), nvec, amax_bits, static_cast<const int32_t*>(nullptr),
                    static_cast<int64_t>(0));
}

// *amax_bits = largest |value| of the first *n_rows rows (device count, at most max_rows)
// of a bf16 [rows, row_elems] buffer, zeroed first.
cudaError_t launch_amax_rows(const void* src, int row_elems, const int32_t* n_rows, int64_t max_rows,
                             uint32_t* amax_bits, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, 4, st);
  if (e != cudaSuccess || max_rows == 0) return e;
  const int64_t row_vecs = row_elems / 8;
  const int64_t nvec = max_rows * row_vecs;
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int gx = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(nvec, 256 * 8), 4 * sms)));
  return launch_pdl(amax_kernel<1>, dim3(gx, 1), dim3(256), 0, st, static_cast<const uint4*>(src), nvec, amax_bits,
                    n_rows, row_vecs);
}

// In place on the first *n_rows rows of a bf16 [rows, row_elems] buffer: each value v
// becomes its per-tensor FP8 value code(v / 2^X) * 2^X, X from the tensor's amax (exactly
// a bf16: an E4M3 code times a power of two), the operand values of a per-tensor FP8 GEMM
// that a bf16 tensor-core kernel then multiplies exactly.
__global__ void __launch_bounds__(256) qdq_fp8_kernel(uint4* __restrict__ buf, int64_t nvec,
                                                      const int32_t* __restrict__ n_rows, int64_t row_vecs,
                                                      const uint32_t* __restrict__ amax_bits) {
  pdl_launch_dependents();
  pdl_wait();
  nvec = min(nvec, static_cast<int64_t>(__ldg(n_rows)) * row_vecs);
  const int X = fp8_tensor_exponent(__ldg(amax_bits));
  const float inv = mx_inv_scale(X), sc = ldexpf(1.0f, X);
  auto qdq = [&](uint4& q) {
    uint32_t* w = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_fp8x2_storage_t c = e4m3x2(bf16_lo(w[j]) * inv, bf16_hi(w[j]) * inv);
      const float2 dq = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3)));
      w[j] = pack_bf16x2(dq.x * sc, dq.y * sc);
    }
  };
  // two independent vectors in flight per thread
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + stride < nvec; i += 2 * stride) {
    uint4 q0 = buf[i], q1 = buf[i + stride];
    qdq(q0);
    qdq(q1);
    buf[i] = q0;
    buf[i + stride] = q1;
  }
  if (i < nvec) {
    uint4 q = buf[i];
    qdq(q);
    buf[i] = q;
  }
}

cudaError_t launch_qdq_fp8_rows(void* buf, int row_elems, const int32_t* n_rows, int64_t max_rows,
                                const uint32_t* amax_bits, cudaStream_t st) {
  if (max_rows == 0) return cudaSuccess;
  const int64_t row_vecs = row_elems / 8;
  const int64_t nvec = max_rows * row_vecs;
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int gx = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(nvec, 256 * 4), 8 * sms)));
  return launch_pdl(qdq_fp8_kernel, dim3(gx), dim3(256), 0, st, static_cast<uint4*>(buf), nvec, n_rows, row_vecs,
                    amax_bits);
}

__global__ void fp8_exponents_kernel(int32_t* v, int n) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) v[i] = fp8_tensor_exponent(static_cast<uint32_t>(v[i]));
}

// In place: amax bits -> the tensors' exponents X.
cudaError_t launch_fp8_exponents(int32_t* v, int n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(fp8_exponents_kernel, dim3(static_cast<unsigned>(ceil_div(n, 256))), dim3(256), 0, st, v, n);
}

}  // namespace moe
