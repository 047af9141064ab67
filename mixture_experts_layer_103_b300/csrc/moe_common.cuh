// Shared definitions of the CUDA library (device side and host launch helpers).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Workspace header: the first 256 bytes of every workspace.
//   [0]  int32 device error word (0 = none)
struct WsHeader {
  int32_t error;
  int32_t pad[63];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kAlign = 256;
__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Rows of the permutation buffers: at most min(k, E_loc) local slots per token.
__host__ __device__ inline int64_t n_cap_of(int T, int k, int E_loc) {
  return static_cast<int64_t>(T) * (k < E_loc ? k : E_loc);
}

// Gate/up interleave block of the packed GEMM1 weights.
__host__ __device__ inline int gu_block_of(int f) {
  return (f % 128 == 0) ? 128 : (f % 64 == 0) ? 64 : (f % 32 == 0) ? 32 : 0;
}

// Number of 128-row m-tiles of the activation SF layout, upper bound.
__host__ __device__ inline int64_t mx_tiles_cap(int64_t n_cap, int E_loc) { return ceil_div(n_cap, 128) + E_loc; }

// The device error word is sticky: kernels only ever move it from 0 to an error code;
// moe_get_device_error() reads and clears it.
__device__ __forceinline__ void set_device_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// Programmatic dependent launch.  Every kernel of the layer lets the next kernel on the
// stream be scheduled early (launch_dependents) and waits for the previous kernel to
// finish and flush (wait) before it touches any data the pipeline produces; only
// kernel-local set-up (shared memory, barriers, TMEM) may come before the wait.  On a
// launch without the attribute both are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kern` with programmatic stream serialization allowed (see pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Host-side argument checks of moe_permute, shared by its workspace-free variant.
moe_status check_permute(const void* x, moe_dtype x_dtype, moe_dtype perm_dtype, int T, int d, const void* ids,
                         const void* probs, int k, int e0, int E_loc, const void* perm_x, const void* perm_sf,
                         const void* counts, const void* offsets, const void* rst, const void* rp, const void* p2r);

// ---- bf16 / fp32 helpers --------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---- MXFP8 (E4M3 + E8M0 per 32) ---------------------------------------------------------
// Shared exponent X = floor(log2(amax)) - 8 clamped to [-127, 127]; amax == 0 -> X = 0.
// amax is a non-negative finite fp32; floor(log2) comes from the exponent field.  A
// subnormal amax (< 2^-126) always clamps to X = -127.
__device__ __forceinline__ int mx_exponent(float amax) {
  if (amax == 0.0f) return 0;
  const int biased = (__float_as_uint(amax) >> 23) & 0xFF;
  if (biased == 0) return -127;
  const int X = biased - 127 - 8;
  return X < -127 ? -127 : X;
}
// 2^-X as an exact fp32 (X in [-127, 119]).
__device__ __forceinline__ float mx_inv_scale(int X) { return __uint_as_float(static_cast<uint32_t>(127 - X) << 23); }

// Two fp32 -> two E4M3 codes (round to nearest even, saturate to +-448), low byte = a.
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Per-tensor FP8 (E4M3 with one power-of-two scale per tensor): the smallest X with
// amax <= 448 * 2^X, from the fp32 bit fields of amax (a non-negative float given as its
// bits, the form atomicMax accumulates): amax = (1.m / 2) * 2^(b - 126) and 448 = 0.875 *
// 2^9, so X = b - 135, plus 1 when the significand 1.m exceeds 1.75; clamped to [-127,
// 127]; 0 for amax == 0, -127 for a subnormal amax.
__device__ __forceinline__ int fp8_tensor_exponent(uint32_t amax_bits) {
  if (amax_bits == 0) return 0;
  const int b = static_cast<int>((amax_bits >> 23) & 0xFFu);
  if (b == 0) return -127;
  const int X = b - 135 + ((amax_bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// Byte offset of (row i of m-tile `tile`, K index k) in the activation SF tile layout.
__host__ __device__ inline int64_t sf_act_offset(int64_t tile, int i, int k, int K) {
  return (tile * (K / 128) + k / 128) * 512 + (i % 32) * 16 + (i / 32) * 4 + (k % 128) / 32;
}
// Byte offset of (packed row r of expert e, K index k) in the weight SF tile layout.
__host__ __device__ inline int64_t sf_w_offset(int e, int64_t rows, int64_t r, int k, int K) {
  return ((static_cast<int64_t>(e) * (K / 128) + k / 128) * (rows / 128) + r / 128) * 512 +
         (r % 32) * 16 + ((r % 128) / 32) * 4 + (k % 128) / 32;
}

// m-tile prefix over experts for tiles of `bm` rows: s_mtp[e] = sum_{e'<e} ceil(cnt/bm).
// Executed by one warp.
__device__ __forceinline__ void build_mtile_prefix(const int32_t* __restrict__ offsets, int E_loc, int bm, int* s_off, int* s_mtp) {
  const int lane = threadIdx.x & 31;
  const int per = (E_loc + 31) / 32;
  const int e_begin = lane * per, e_end = min(E_loc, e_begin + per);
  int sum = 0;
  for (int e = e_begin; e < e_end; ++e) {
    const int o0 = __ldg(offsets + e), o1 = __ldg(offsets + e + 1);
    s_off[e] = o0;
    sum += (o1 - o0 + bm - 1) / bm;
  }
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  int run = incl - sum;
  for (int e = e_begin; e < e_end; ++e) {
    s_mtp[e] = run;
    run += (__ldg(offsets + e + 1) - __ldg(offsets + e) + bm - 1) / bm;
  }
  if (lane == 31) {
    s_mtp[E_loc] = incl;
    s_off[E_loc] = __ldg(offsets + E_loc);
  }
}

}  // namespace moe
