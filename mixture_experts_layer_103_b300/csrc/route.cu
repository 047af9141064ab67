// Step 1: top-k routing over fp32 router logits ("Wide-EP ... NVIDIA" explainer, section
// "MoE basics": the router chooses, per token, the experts it uses; DeepSeek-R1 picks 8 of
// 256).  One warp per token; each lane holds E/32 logits as 32-bit order-preserving keys,
// sorted per lane; each of the k rounds takes the largest lane head (ties go to the lower
// expert id) and pops it.  The softmax over the k chosen logits gives the probabilities.
// The logits are read once, coalesced.
#include "moe_common.cuh"

namespace moe {

constexpr int kRouteWarps = 8;

// Order-preserving map of a non-NaN fp32 to a non-zero uint32 (-0.0 folded onto +0.0);
// 0 marks an empty or already chosen slot.
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0) u = 0;  // +-0.0 -> +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Each lane first sorts its VPL keys (with their expert ids) in descending key order,
// ties to the lower id (a bitonic network over registers), so a round only compares the
// lanes' heads: one redux for the largest head; when several lanes hold it (equal
// logits), a second redux picks the lowest id.  The winning lane pops its head.
template <int VPL>
__device__ __forceinline__ void sort_desc(uint32_t (&key)[VPL], uint32_t (&id)[VPL]) {
#pragma unroll
  for (int k = 2; k <= VPL; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int l = i ^ j;
        if (l > i) {
          // (key desc, id asc) order; ascending run where (i & k) != 0
          const bool i_first = key[i] > key[l] || (key[i] == key[l] && id[i] < id[l]);
          const bool want_i_first = (i & k) == 0;
          if (i_first != want_i_first) {
            const uint32_t tk = key[i], ti = id[i];
            key[i] = key[l]; id[i] = id[l];
            key[l] = tk; id[l] = ti;
          }
        }
      }
}

template <int VPL>  // values per lane = ceil(E / 32), a power of two
__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                                       int k, int32_t* __restrict__ ids,
                                                                       float* __restrict__ probs) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + t * E;
  uint32_t key[VPL], id[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? ordered_bits(__ldg(row + e)) : 0u;
    id[i] = static_cast<uint32_t>(e);
  }
  if (VPL > 1) sort_desc<VPL>(key, id);
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, key[0]);
    const bool mine = key[0] == mx;
    const uint32_t holders = __ballot_sync(0xffffffffu, mine);
    int win_lane;
    if ((holders & (holders - 1u)) == 0u) {  // one lane holds the maximum
      win_lane = __ffs(holders) - 1;
    } else {  // equal logits in several lanes: the lowest expert id
      const uint32_t w = __reduce_min_sync(0xffffffffu, mine ? id[0] : 0xffffffffu);
      win_lane = __ffs(__ballot_sync(0xffffffffu, mine && id[0] == w)) - 1;
    }
    const int win = static_cast<int>(__shfl_sync(0xffffffffu, id[0], win_lane));
    if (lane == win_lane) {  // pop the head
#pragma unroll
      for (int i = 0; i + 1 < VPL; ++i) {
        key[i] = key[i + 1];
        id[i] = id[i + 1];
      }
      key[VPL - 1] = 0u;
    }
    // win < E for every non-NaN row; the clamp keeps NaN rows (unspecified result) in bounds
    if (lane == j) my_id = min(win, E - 1);
  }
  // softmax over the k chosen logits; lane 0 holds the largest one
  const float my_val = lane < k ? __ldg(row + my_id) : 0.0f;
  const float l0 = __shfl_sync(0xffffffffu, my_val, 0);
  const float w = (lane < k) ? expf(my_val - l0) : 0.0f;
  float s = w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane < k) {
    ids[t * k + lane] = my_id;
    probs[t * k + lane] = w / s;
  }
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* probs,
                              cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(ceil_div(T, kRouteWarps))), block(kRouteWarps * 32);
  const int vpl = static_cast<int>(ceil_div(E, 32));
  cudaError_t e = cudaSuccess;
#define MOE_ROUTE_CASE(V) \
  case V: e = launch_pdl(route_topk_kernel<V>, grid, block, 0, st, logits, T, E, k, ids, probs); break;
  switch (vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : vpl <= 16 ? 16 : 32) {
    MOE_ROUTE_CASE(2)
    MOE_ROUTE_CASE(4)
    MOE_ROUTE_CASE(8)
    MOE_ROUTE_CASE(16)
    MOE_ROUTE_CASE(32)
  }
#undef MOE_ROUTE_CASE
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
