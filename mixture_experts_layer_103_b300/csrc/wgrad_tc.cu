// Weight gradients of the expert layer on the 5th-generation tensor cores:
//   C_e[M, N] = sum over the rows r of expert e's segment [offsets[e], offsets[e+1]) of
//               A[r, 0:M]^T B[r, 0:N]                     (fp32 accumulate, fp32 out)
// The contraction runs over the expert's routed rows, so K is ragged per expert while
// M and N are the same for every expert.  Both operands are row-major [rows, M or N] in
// routed-row order (the token-indexed operand is first copied into that order): each row
// is one K index holding M (or N) contiguous values, i.e. MN-major tiles.  One thread
// loads every full 64-row block of a segment by TMA (64 x 64 boxes, 128-byte swizzle);
// a segment's last, partial block is loaded by eight warps with cp.async, zero-filling
// the rows past the segment end (TMA cannot stop there) and the columns past M / N, and
// counted on the stage's full barrier as it lands (cp.async.mbarrier.arrive).  One
// thread issues tcgen05.mma (both operands MN-major) into a double-buffered TMEM
// accumulator; four warps move the fp32 tiles out through shared memory, one TMA store per
// 32 x 32 block (plain stores for blocks cut by the matrix edge).  Persistent: one CTA per
// SM, tiles (expert, m-tile, n-tile) round-robin.  Experts without rows get zero tiles.
//   MODE 0: dW_down_e [f, d] = h^T dy   (A = h, B = dy in routed order)
//   MODE 1: dW_gate_e, dW_up_e [d, f] = x^T dg, x^T du (A = x in routed order, B = dg/du in
//           the packed order, stored back to the gate and up matrices)
// ("Efficient MoE training for biological foundation models", section "GroupedLinear
// Optimizes Expert Computation": the GroupedMLP backward's weight-gradient GEMMs.)
#include <algorithm>

#include "gemm_tc.cuh"

namespace moe {

constexpr int kWBM = 128, kWBN = 256, kWBK = 64;      // tile M x N, K rows per stage
constexpr int kWStages = 4;
constexpr int kWA = kWBM * kWBK * 2;                   // 16 KB
constexpr int kWB = kWBN * kWBK * 2;                   // 32 KB
constexpr int kWStage = kWA + kWB;
constexpr int kWGather = 256;                          // partial-block copy threads (8 warps)
constexpr int kWThreads = 32 + 128 + kWGather + 32;    // MMA warp, 4 epilogue, 8 copy, TMA warp
constexpr int kWEpiBuf = 32 * 128;                     // one staged 32 x 32 fp32 block (128-byte swizzle)
constexpr int kWOffEpi = kWStages * kWStage;           // 2 staging buffers per epilogue warp
constexpr int kWOffBar = kWOffEpi + 4 * 2 * kWEpiBuf;
constexpr int kWSmem = kWOffBar + 16 * 8 + 16 + 1024;
static_assert(kWSmem <= 232448, "shared memory per CTA");

struct WgradArgs {
  const uint16_t* A;  // [rows, M] routed-row order
  int64_t lda;
  const uint16_t* B;  // [rows, N] routed-row order
  int64_t ldb;
  const int32_t* offsets;
  int E_loc, M, N;
  float* out0;
  float* out1;
  int32_t* err;
  uint64_t timeout_ns;
};

template <int MODE>
__global__ void __launch_bounds__(kWThreads, 1) wgrad_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                const __grid_constant__ CUtensorMap tmB,
                                                                const __grid_constant__ CUtensorMap tmO0,
                                                                const __grid_constant__ CUtensorMap tmO1,
                                                                const WgradArgs g) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar0 = sbase + kWOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kWStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kWStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kWStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kWStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kWOffBar + 16 * 8);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kWOffBar + 16 * 8 + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      ptx::mbar_init(full_bar(s), kWGather + 1);  // copy threads + the TMA thread
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 4);
    }
    ptx::mbar_init(drain_bar, 1);
    *s_abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  pdl_wait();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int mt_n = (g.M + kWBM - 1) / kWBM, nt_n = (g.N + kWBN - 1) / kWBN;
  const int per_e = mt_n * nt_n;
  const int total = g.E_loc * per_e;
  auto kblocks = [&](int e) {
    const int rows = __ldg(g.offsets + e + 1) - __ldg(g.offsets + e);
    return (rows + kWBK - 1) / kWBK;
  };
  GemmArgs abort_args{};
  abort_args.err = g.err;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16_mn(kWBM, kWBN);
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int nkb = kblocks(t / per_e);
        if (nkb == 0) continue;  // zero tile: the epilogue writes zeros without TMEM
        const int acc = it & 1;
        const uint32_t acc_ph = static_cast<uint32_t>((it >> 1) & 1);
        ++it;
        if (!ptx::mbar_wait(tempty_bar(acc), acc_ph ^ 1u, g.timeout_ns)) { gemm_abort(abort_args, s_abort); break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kWBN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(full_bar(s), ph, g.timeout_ns)) { gemm_abort(abort_args, s_abort); ok = false; break; }
          ptx::fence_proxy_async_smem();  // the stage was written by cp.async
          ptx::tc_fence_after();
          const uint32_t a_addr = sbase + s * kWStage;
          const uint32_t b_addr = a_addr + kWA;
#pragma unroll
          for (int k = 0; k < kWBK / 16; ++k)  // 16 K rows of 128 bytes per MMA
            ptx::mma_bf16(d_tmem, ptx::sdesc_sw128_mn(a_addr + k * 2048, 8192),
                          ptx::sdesc_sw128_mn(b_addr + k * 2048, 8192), idesc, (kb | k) != 0);
          ptx::mma_commit(empty_bar(s));
          if (++s == kWStages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit(tfull_bar(acc));
      }
      ptx::mma_commit(drain_bar);
      ptx::mbar_wait(drain_bar, 0, g.timeout_ns);
    }
  } else if (warp < 5) {
    // ------------------------------------------------------------------ epilogue
    // Each 32-column block of the warp's 32 rows is written to a staging buffer (thread =
    // row, 16-byte chunk c of row r at c ^ (r & 7): the 128-byte swizzle of the store map)
    // and leaves by one TMA store; two buffers alternate, a buffer is rewritten once the
    // store that read it is done reading.
    const int q = warp & 3;  // TMEM lane quarter
    uint8_t* stage = smem + kWOffEpi + (warp - 1) * 2 * kWEpiBuf;
    const uint32_t stage_s = sbase + static_cast<uint32_t>(kWOffEpi + (warp - 1) * 2 * kWEpiBuf);
    int it = 0, sb = 0, last_sb = -1;  // last_sb: buffer of the most recent TMA store
    const int ncols_out = MODE == 0 ? g.N : g.N / 2;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      if (*s_abort) break;
      const int e = t / per_e, rem = t - e * per_e;
      const int m0 = (rem / nt_n) * kWBM, n0 = (rem % nt_n) * kWBN;
      const int nkb = kblocks(e);
      const int acc = it & 1;
      const uint32_t acc_ph = static_cast<uint32_t>((it >> 1) & 1);
      if (nkb > 0) {
        ++it;
        int okw = 0;
        if (lane == 0) okw = ptx::mbar_wait(tfull_bar(acc), acc_ph, g.timeout_ns) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) { if (lane == 0) gemm_abort(abort_args, s_abort); break; }
        (void)ptx::mbar_try_wait(tfull_bar(acc), acc_ph);
        ptx::tc_fence_after();
      }
      const int rows_valid = max(0, min(32, g.M - (m0 + q * 32)));
      const int row_g = e * g.M + m0 + q * 32;  // first output row of the warp's slab
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kWBN);
#pragma unroll 1
      for (int c = 0; c < kWBN; c += 32) {
        const int n = n0 + c;
        if (n >= g.N) break;
        uint32_t v[32];
        if (nkb > 0) {
          ptx::tmem_ld32(tbase + c, v);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        // destination of this 32-column block: dW_down, or the gate / up matrix
        const bool to_up = MODE == 1 && ((n / 32) % 2 == 1);
        const int col = MODE == 0 ? n : (n / 64) * 32;
        const int chunks_valid = max(0, min(8, (g.N - n) / 4));
        const bool whole = rows_valid == 32 && chunks_valid == 8;
        if (lane == 0) {
          if (last_sb == (sb ^ 1)) ptx::bulk_wait_read<1>();
          else ptx::bulk_wait_read<0>();
        }
        __syncwarp();
        uint8_t* buf = stage + sb * kWEpiBuf;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
              make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        if (whole) {
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(to_up ? &tmO1 : &tmO0, stage_s + sb * kWEpiBuf, col, row_g);
            ptx::bulk_commit();
          }
          last_sb = sb;
        } else {  // block cut by the matrix edge: plain stores of the valid part
          __syncwarp();
          float* dst = to_up ? g.out1 : g.out0;
          uint8_t* g0 = reinterpret_cast<uint8_t*>(dst + static_cast<int64_t>(row_g) * ncols_out + col);
#pragma unroll
          for (int j = 0; j < 8; ++j) {  // 4 rows x 128 bytes per store instruction
            const int r = j * 4 + lane / 8, ch = lane % 8;
            const uint4 val = *reinterpret_cast<const uint4*>(buf + r * 128 + ((ch ^ (r & 7)) << 4));
            if (r < rows_valid && ch < chunks_valid)
              *reinterpret_cast<uint4*>(g0 + static_cast<int64_t>(r) * ncols_out * 4 + ch * 16) = val;
          }
          __syncwarp();
        }
        sb ^= 1;
      }
      if (nkb > 0) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty_bar(acc));
      }
    }
    if (lane == 0) ptx::bulk_wait_all();  // the stores have completed before the CTA exits
  } else if (warp == 13) {
    // ------------------------------------------------------------------ TMA (full blocks)
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB);
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      constexpr int kStageBytes = kWA + kWB;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int e = t / per_e, rem = t - e * per_e;
        const int m0 = (rem / nt_n) * kWBM, n0 = (rem % nt_n) * kWBN;
        const int r_begin = __ldg(g.offsets + e), r_end = __ldg(g.offsets + e + 1);
        const int nkb = (r_end - r_begin + kWBK - 1) / kWBK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (*s_abort) { ok = false; break; }
          if (!ptx::mbar_wait(empty_bar(s), ph ^ 1u, g.timeout_ns)) { gemm_abort(abort_args, s_abort); ok = false; break; }
          const int r0 = r_begin + kb * kWBK;
          if (r0 + kWBK <= r_end) {
            const uint32_t a_addr = sbase + s * kWStage;
            ptx::mbar_arrive_expect_tx(full_bar(s), kStageBytes);
            for (int a = 0; a < kWBM / 64; ++a) ptx::tma_load_3d(a_addr + a * 8192, &tmA, full_bar(s), m0 + 64 * a, r0, 0);
            for (int a = 0; a < kWBN / 64; ++a)
              ptx::tma_load_3d(a_addr + kWA + a * 8192, &tmB, full_bar(s), n0 + 64 * a, r0, 0);
            ++issued;
          } else {
            ptx::mbar_arrive(full_bar(s));  // the copy warps load this partial block
          }
          if (++s == kWStages) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {  // let the issued copies land before the CTA exits
        for (int i = 0; i < kWStages; ++i) ptx::mbar_wait(full_bar(i), 0, 1000000ull);
      }
      (void)issued;
    }
  } else {
    // ------------------------------------------------------------------ partial blocks
    const int gt = threadIdx.x - 160;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const int e = t / per_e, rem = t - e * per_e;
      const int m0 = (rem / nt_n) * kWBM, n0 = (rem % nt_n) * kWBN;
      const int r_begin = __ldg(g.offsets + e), r_end = __ldg(g.offsets + e + 1);
      const int nkb = (r_end - r_begin + kWBK - 1) / kWBK;
      for (int kb = 0; kb < nkb; ++kb) {
        int okw = 0;
        if (lane == 0) okw = *s_abort ? 0 : (ptx::mbar_wait(empty_bar(s), ph ^ 1u, g.timeout_ns) ? 1 : 2);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (okw != 1) {
          if (okw == 2 && lane == 0) gemm_abort(abort_args, s_abort);
          ok = false;
          break;
        }
        (void)ptx::mbar_try_wait(empty_bar(s), ph ^ 1u);
        if (r_begin + (kb + 1) * kWBK > r_end) {  // the segment's last, partial block
          const uint32_t a_addr = sbase + s * kWStage, b_addr = a_addr + kWA;
          // thread -> K row kr = gt / 4: 4 of its 16 A chunks (two 64-column atoms) and 8 of
          // its 32 B chunks (four atoms), in the swizzled layout TMA would produce
          const int kr = gt >> 2, sub = gt & 3;
          const int64_t r = r_begin + kb * kWBK + kr;
          const bool rv = r < r_end;
          const uint32_t swz = static_cast<uint32_t>(kr & 7);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int cc = sub + 4 * j, atom = cc >> 3, c = cc & 7;
            const int m = m0 + atom * 64 + c * 8;
            const bool v = rv && m < g.M;
            ptx::cp_async_16(a_addr + atom * 8192 + kr * 128 + ((c ^ swz) << 4),
                             v ? static_cast<const void*>(g.A + r * g.lda + m) : g.A, v ? 16u : 0u);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int cc = sub + 4 * j, atom = cc >> 3, c = cc & 7;
            const int n = n0 + atom * 64 + c * 8;
            const bool v = rv && n < g.N;
            ptx::cp_async_16(b_addr + atom * 8192 + kr * 128 + ((c ^ swz) << 4),
                             v ? static_cast<const void*>(g.B + r * g.ldb + n) : g.B, v ? 16u : 0u);
          }
        }
        ptx::cp_async_arrive_noinc(full_bar(s));  // every stage: the barrier counts all copy threads
        if (++s == kWStages) { s = 0; ph ^= 1u; }
      }
    }
    ptx::cp_async_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

template <int MODE>
static cudaError_t launch_wgrad_tc(const WgradArgs& g, int64_t n_rows, cudaStream_t st) {
  CUtensorMap tmA, tmB, tmO0, tmO1;  // 64 x 64 operand boxes over [n_rows, M] and [n_rows, N]
  if (!make_operand_map(&tmA, g.A, false, static_cast<uint64_t>(g.M), static_cast<uint64_t>(n_rows), 1, 64) ||
      !make_operand_map(&tmB, g.B, false, static_cast<uint64_t>(g.N), static_cast<uint64_t>(n_rows), 1, 64))
    return cudaErrorInvalidValue;
  // outputs [E_loc * M, N or N / 2] fp32, 32 x 32 store boxes
  const uint64_t out_rows = static_cast<uint64_t>(g.E_loc) * g.M, out_cols = MODE == 0 ? g.N : g.N / 2;
  if (!make_store_map(&tmO0, g.out0, 4, out_cols, out_rows, 32, 32) ||
      !make_store_map(&tmO1, MODE == 0 ? g.out0 : g.out1, 4, out_cols, out_rows, 32, 32))
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(wgrad_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  return launch_pdl(wgrad_tc_kernel<MODE>, dim3(static_cast<unsigned>(num_sms())), dim3(kWThreads), kWSmem, st, tmA,
                    tmB, tmO0, tmO1, g);
}

// dW_down [E_loc, f, d] from h [n_rows, f] and dy_rows [n_rows, d] (routed order).
cudaError_t launch_wgrad_down_tc(const void* h, const void* dy_rows, const int32_t* offsets, int64_t n_rows,
                                 int E_loc, int d, int f, float* dWd, int32_t* err, uint64_t timeout_ns,
                                 cudaStream_t st) {
  WgradArgs g{static_cast<const uint16_t*>(h), f, static_cast<const uint16_t*>(dy_rows), d, offsets,
              E_loc, f, d, dWd, nullptr, err, timeout_ns};
  return launch_wgrad_tc<0>(g, n_rows, st);
}

// dW_gate, dW_up [E_loc, d, f] from x_rows [n_rows, d] (routed order) and dg/du [n_rows, 2f].
cudaError_t launch_wgrad_gate_up_tc(const void* x_rows, const void* dgu, const int32_t* offsets, int64_t n_rows,
                                    int E_loc, int d, int f, float* dWg, float* dWu, int32_t* err,
                                    uint64_t timeout_ns, cudaStream_t st) {
  WgradArgs g{static_cast<const uint16_t*>(x_rows), d, static_cast<const uint16_t*>(dgu), 2 * f, offsets,
              E_loc, d, 2 * f, dWg, dWu, err, timeout_ns};
  return launch_wgrad_tc<1>(g, n_rows, st);
}

}  // namespace moe
