// moe_permute_noalloc: the permute with its scratch in a library-owned static device
// array instead of a caller-supplied workspace.
//
// Who needs it: callers that cannot call cudaMalloc when they run the permute, e.g. a
// serving engine that hands all free device memory to its KV-cache pool at start-up and
// plans every later buffer by hand, or a host application that is recording a CUDA graph
// and must not allocate while recording.  They still pass all inputs and outputs; only
// the permute's internal scratch (per-tile expert counts, m-tile bases, error word) moves
// into a fixed array that every device holding this library keeps until the process exits.
//
// The permute kernels themselves are unchanged: this entry point fetches the device
// address of the static array and hands it to moe_permute() as the workspace.
#include <mutex>

#include "moe_common.cuh"

namespace moe {

// Largest scratch the static array can serve (see moe.h for what it means in T / E_loc).
constexpr size_t kStaticPermuteScratchBytes = size_t(1) << 20;  // 1 MiB

static __device__ __align__(256) uint8_t g_permute_scratch[kStaticPermuteScratchBytes];

constexpr int kMaxScratchDevices = 64;
static std::mutex g_scratch_mutex;
static void* g_scratch_address[kMaxScratchDevices];  // device address of the array, per device

// Device address of g_permute_scratch on the current device.  In host code the array's
// name is only a host-side stand-in, so the address comes from cudaGetSymbolAddress, once
// per device, with that device current.
static cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_address[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_address[dev] = p;
  }
  *out = g_scratch_address[dev];
  return cudaSuccess;
}

}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const void* x, moe_dtype x_dtype, moe_dtype perm_dtype, int T, int d,
                                          const int32_t* topk_ids, const float* topk_probs, int k, int e0, int E_loc,
                                          void* perm_x, uint8_t* perm_x_scale, int32_t* counts, int32_t* offsets,
                                          int32_t* row_src_token, float* row_prob, int32_t* pair_to_row,
                                          moe_stream_t stream) {
  // the arguments first, so an out-of-range size is reported as such and never reaches
  // the workspace arithmetic
  const moe_status s = moe::check_permute(x, x_dtype, perm_dtype, T, d, topk_ids, topk_probs, k, e0, E_loc, perm_x,
                                          perm_x_scale, counts, offsets, row_src_token, row_prob, pair_to_row);
  if (s != MOE_OK) return s;
  const size_t need = moe_permute_workspace_size(T, k, E_loc);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > moe::kStaticPermuteScratchBytes) return MOE_ERR_WORKSPACE;  // beyond the static array
  void* scratch = nullptr;
  if (moe::static_scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_permute(x, x_dtype, perm_dtype, T, d, topk_ids, topk_probs, k, e0, E_loc, perm_x, perm_x_scale, counts,
                     offsets, row_src_token, row_prob, pair_to_row, scratch, moe::kStaticPermuteScratchBytes, stream);
}
