// C ABI of the MoE expert-layer library: argument validation, workspace layout and the
// launch sequence of each entry point (declared and documented in include/moe.h).
#include <algorithm>
#include <cstring>
#include <mutex>

#include "moe_common.cuh"

namespace moe {

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* probs, cudaStream_t st);
cudaError_t launch_permute(const void* x, moe_dtype x_dtype, moe_dtype perm_dtype, int T, int d, const int32_t* ids,
                           const float* probs, int k, int e0, int E_loc, void* perm_x, uint8_t* perm_sf,
                           int32_t* counts, int32_t* offsets, int32_t* row_src_token, float* row_prob,
                           int32_t* pair_to_row, uint8_t* ws, cudaStream_t st, int32_t* tok_nloc = nullptr);
size_t permute_ws_bytes(int T, int E_loc);
cudaError_t launch_combine_prep(const int32_t* pair_to_row, int T, int k, int32_t* tok_nloc, cudaStream_t st);
cudaError_t launch_tc_gemm2_combine(const void* h, const uint8_t* h_sf, const int32_t* offsets, int64_t N_cap,
                                    int E_loc, int d, int f, bool mx, int shape, const void* Wd, const uint8_t* Wd_sf,
                                    void* Y2, const int32_t* row_src_token, const int32_t* tok_nloc, int T, void* y,
                                    int32_t* err, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_combine(const void* Y2, const int32_t* p2r, int T, int k, int d, moe_dtype dtype, void* y,
                           cudaStream_t st, bool multi_only = false);
cudaError_t launch_combine_multi(const void* Y2, const int32_t* p2r, const int32_t* tok_nloc, int T, int k, int d,
                                 void* y, double slots_per_token, cudaStream_t st);
cudaError_t launch_simt_gemm1(const float* perm_x, const int32_t* offsets, const float* row_prob, int64_t N_cap,
                              int E_loc, int d, int f, const float* Wgu, float* h, cudaStream_t st);
cudaError_t launch_simt_gemm2(const float* h, const int32_t* offsets, int64_t N_cap, int E_loc, int d, int f,
                              const float* Wd, float* Y2, cudaStream_t st);
cudaError_t launch_tc_gemm1(const void* perm_x, const uint8_t* perm_sf, const int32_t* offsets, const float* row_prob,
                            int64_t N_cap, int E_loc, int d, int f, bool mx, int shape, const void* Wgu,
                            const uint8_t* Wgu_sf, void* h, uint8_t* h_sf, int32_t* err, uint64_t timeout_ns,
                            void* gu_save, cudaStream_t st);
cudaError_t launch_tc_gemm2(const void* h, const uint8_t* h_sf, const int32_t* offsets, int64_t N_cap, int E_loc, int d,
                            int f, bool mx, int shape, const void* Wd, const uint8_t* Wd_sf, void* Y2, int32_t* err,
                            uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_tc_gemm1_gather(const void* x, const uint8_t* x_sf, const int32_t* row_src_token,
                                   const int32_t* offsets, const float* row_prob, int64_t N_cap, int E_loc, int d,
                                   int f, bool mx, int shape, const void* Wgu, const uint8_t* Wgu_sf, void* h,
                                   uint8_t* h_sf, int32_t* err, uint64_t timeout_ns, void* gu_save, cudaStream_t st);
cudaError_t launch_quant_rows_mx(const void* x, moe_dtype x_dtype, int T, int d, const int32_t* pair_to_row, int k,
                                 uint8_t* xq, uint8_t* x_sf, cudaStream_t st);
cudaError_t launch_tc_dswiglu(const void* dy_rows, const int32_t* offsets, const float* row_prob, int64_t N_cap,
                              int E_loc, int d, int f, const void* W_down, const void* gu, void* dgu, void* h,
                              float* dp_part, int32_t* err, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_tc_gemm_store(const void* A, int64_t a_rows, const int32_t* offsets, int E_loc, int K, int n_out,
                                 const void* B, void* out, int32_t* err, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_pack_gu_t(const void* Wg, const void* Wu, moe_dtype src, int E_loc, int d, int f, void* WguT,
                             cudaStream_t st);
cudaError_t launch_dlogits(const int32_t* ids, const float* probs, const int32_t* p2r, const float* dp_part,
                           int nparts, int T, int E, int k, float* dlogits, cudaStream_t st);
cudaError_t launch_wgrad_down_tc(const void* h, const void* dy_rows, const int32_t* offsets, int64_t n_rows,
                                 int E_loc, int d, int f, float* dWd, int32_t* err, uint64_t timeout_ns,
                                 cudaStream_t st);
cudaError_t launch_wgrad_gate_up_tc(const void* x_rows, const void* dgu, const int32_t* offsets, int64_t n_rows,
                                    int E_loc, int d, int f, float* dWg, float* dWu, int32_t* err,
                                    uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_gather_rows(const void* src, int64_t row_bytes, const int32_t* offsets, int E_loc,
                               const int32_t* row_src_token, void* dst, cudaStream_t st);
cudaError_t launch_wait_timeout(int32_t* err, uint64_t timeout_ns, cudaStream_t st);
int32_t* permute_mtile_base(uint8_t* ws, int T, int E_loc);
cudaError_t launch_gather_rows_mx(const void* src, int K, const int32_t* offsets, int E_loc,
                                  const int32_t* mtile_base, const int32_t* row_src_token, uint8_t* dst,
                                  uint8_t* dst_sf, cudaStream_t st, const uint32_t* tensor_amax = nullptr);
cudaError_t launch_tc_gemm1_fp8(const void* perm_x, const uint8_t* perm_sf, const int32_t* offsets,
                                const float* row_prob, int64_t N_cap, int E_loc, int d, int f, const void* Wgu,
                                const uint8_t* Wgu_sf, void* h_bf16, uint32_t* h_amax, int32_t* err,
                                uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_pack_fp8(const void* Wg, const void* Wu, const void* Wdn, moe_dtype src, int E_loc, int d, int f,
                            void* Wgu_p, void* Wd_p, uint8_t* Wgu_sf, uint8_t* Wd_sf, int32_t* w_exp,
                            cudaStream_t st);
cudaError_t launch_pack_backward_mx(const void* Wg, const void* Wu, const void* Wdn, moe_dtype src, int E_loc, int d,
                                    int f, uint8_t* WguT_q, uint8_t* WguT_sf, uint8_t* Wd_q, uint8_t* Wd_sf,
                                    cudaStream_t st, const int32_t* tensor_exp = nullptr);
cudaError_t launch_colquant_mx(void* buf, int C, const int32_t* offsets, int E_loc, cudaStream_t st);
cudaError_t launch_rows_mx_both(const void* src, int d, const int32_t* offsets, int E_loc, const int32_t* mtile_base,
                                const int32_t* row_src_token, uint8_t* q, uint8_t* q_sf, void* deq, cudaStream_t st);
cudaError_t launch_tc_dswiglu_mx(const void* dy_q, const uint8_t* dy_sf, const int32_t* offsets,
                                 const float* row_prob, int64_t N_cap, int E_loc, int d, int f, const void* Wd_q,
                                 const uint8_t* Wd_sf, const void* gu, void* dgu, void* h, float* dp_part, int32_t* err,
                                 uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_tc_gemm_store_mx(const void* A, const uint8_t* a_sf, int64_t a_rows, const int32_t* offsets,
                                    int E_loc, int K, int n_out, const void* B, const uint8_t* b_sf, void* out,
                                    int32_t* err, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_pack(const void* Wg, const void* Wu, const void* Wdn, moe_dtype src, moe_dtype dst, int E_loc, int d,
                        int f, void* Wgu_p, void* Wd_p, uint8_t* Wgu_sf, uint8_t* Wd_sf, cudaStream_t st);

cudaError_t launch_amax(const void* src, moe_dtype dt, int64_t n_per_seg, int n_seg, uint32_t* amax_bits,
                        cudaStream_t st);
cudaError_t launch_amax_rows(const void* src, int row_elems, const int32_t* n_rows, int64_t max_rows,
                             uint32_t* amax_bits, cudaStream_t st);
cudaError_t launch_qdq_fp8_rows(void* buf, int row_elems, const int32_t* n_rows, int64_t max_rows,
                                const uint32_t* amax_bits, cudaStream_t st);

constexpr uint64_t kTimeoutNs = 2000000000ull;  // bounded device waits: 2 s
constexpr int kShapeSwapMin = 64;  // GEMM kernel shapes >= this: swapped operands (gemm_tc.cu)
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;  // routed rows are int32 indices
constexpr int kMaxDevices = 64;
constexpr int kMaxExpertId = 65535;  // e0 + E_loc <= 65536 (moe_permute's contract)

int num_sms() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

int gather_grid(cudaStream_t) { return num_sms() * 6; }

static int elt_bytes(moe_dtype dt) { return dt == MOE_F32 ? 4 : dt == MOE_BF16 ? 2 : 1; }
// E4M3 codes with scales in the SF tile layouts: MXFP8, and per-tensor FP8 (every scale of
// a tensor equal), which runs on the same block-scaled kernels.
static bool is_fp8(moe_dtype dt) { return dt == MOE_MXFP8 || dt == MOE_FP8; }
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
static moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static size_t mx_act_sf_bytes(int64_t n_cap, int K, int E_loc) {
  return static_cast<size_t>(mx_tiles_cap(n_cap, E_loc)) * (K / 128) * 512;
}

// ---- grouped MLP scratch: h (+ its scales; per-tensor FP8: + bf16 h and its amax) ----
struct MlpScratch {
  void* h;
  uint8_t* h_sf;
  void* h16;          // per-tensor FP8: GEMM1's bf16 h, quantised once its amax is known
  uint32_t* h_amax;   // per-tensor FP8: largest |h| (fp32 bits)
};
static size_t mlp_scratch_bytes(int64_t n_cap, int E_loc, int f, moe_dtype dt) {
  size_t b = align_up(static_cast<size_t>(n_cap) * f * elt_bytes(dt), kAlign);
  if (is_fp8(dt)) b += align_up(mx_act_sf_bytes(n_cap, f, E_loc), kAlign);
  if (dt == MOE_FP8) b += align_up(static_cast<size_t>(n_cap) * f * 2, kAlign) + kAlign;
  return b;
}
static MlpScratch carve_mlp(uint8_t* p, int64_t n_cap, int f, moe_dtype dt, int E_loc) {
  MlpScratch s{};
  s.h = p;
  const size_t hb = align_up(static_cast<size_t>(n_cap) * f * elt_bytes(dt), kAlign);
  s.h_sf = is_fp8(dt) ? p + hb : nullptr;
  if (dt == MOE_FP8) {
    uint8_t* q = p + hb + align_up(mx_act_sf_bytes(n_cap, f, E_loc), kAlign);
    s.h16 = q;
    s.h_amax = reinterpret_cast<uint32_t*>(q + align_up(static_cast<size_t>(n_cap) * f * 2, kAlign));
  }
  return s;
}

static moe_status check_mlp_shape(int d, int f, int E_loc, moe_dtype dt) {
  if (d <= 0 || f <= 0 || E_loc < 1 || E_loc > 1024) return MOE_ERR_INVALID_ARG;
  if (f % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if (dt == MOE_BF16 && d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (is_fp8(dt) && (d % 128 != 0 || f % 128 != 0)) return MOE_ERR_UNSUPPORTED;
  if (dt != MOE_F32 && dt != MOE_BF16 && !is_fp8(dt)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// When bf16 GEMM1 runs on CTA pairs (256-row tiles), from the expected rows per local
// expert and K = d.  Measured on B300 (each against the 1-CTA kernel):
//   * from 2048 rows: the pairs win (dense segments, little padding);
//   * 256-1023 rows with K >= 4096 (weight-streaming slices, tiles mostly full): the
//     pairs' lower per-SM shared-memory fill wins (layer step at T = 8192 / 16384, d = 7168,
//     4 of 256 experts: 192 -> 184 / 278 -> 263 us);
//   * otherwise the 1-CTA kernel: at 512 rows with K = 2048 and skewed segments, or a
//     Zipf-skewed 128-row average, the 256-row tiles pad too much (+20 / +28 us).
// Callers of the single GEMMs can force either with rows_hint.
constexpr int kPairRowsThreshold = 2048;

// MXFP8 on CTA pairs (block-scaled cta_group::2 MMAs): correct, but measured slower than
// the 1-CTA kernel at every shape tried on B300 (dense 16384 rows, d = 7168: GEMM1 388 vs
// 373 us, GEMM2 256 vs 237; EP64 slice GEMM2 70 vs 58; Zipf EP8 slice GEMM1 186 vs 158):
// the per-stage scale copies into TMEM cost ~13 % of the main loop and two 256-column
// accumulators do not fit beside the scales.  Taken only from this many expected rows per
// expert (no workload here comes near it).
constexpr int kPairRowsThresholdMx = 1 << 16;

static int64_t expected_rows(int64_t n_cap, int E_loc, int rows_hint) {
  return rows_hint > 0 ? rows_hint : n_cap / (E_loc > 0 ? E_loc : 1);
}

static bool use_pair(moe_dtype dt, int64_t n_cap, int E_loc, int rows_hint, int K) {
  const int64_t rows = expected_rows(n_cap, E_loc, rows_hint);
  if (dt == MOE_MXFP8) return rows >= kPairRowsThresholdMx;
  return dt == MOE_BF16 && (rows >= kPairRowsThreshold || (rows >= 256 && rows < 1024 && K >= 4096));
}

// GEMM2 (K = f, output d) on CTA pairs from 128 expected rows per expert: measured on B300
// inside the layer step the pair kernel's halved per-SM weight traffic outweighs its
// coarser row padding there (bf16_e64 at 512 rows: 127.3 -> 119.9 us; EP64 slice at 256
// rows: 49.3 -> 45.0; at 1024 rows: even) but not for short segments (EP64 slice at 64
// rows: 30.9 -> 34.9; Zipf EP8 slice at 16 rows: 49.6 -> 55.7 in isolation).
constexpr int kPairRowsThresholdGemm2 = 128;

static bool use_pair_gemm2(moe_dtype dt, int64_t n_cap, int E_loc, int rows_hint) {
  const int64_t rows = expected_rows(n_cap, E_loc, rows_hint);
  if (dt == MOE_MXFP8) return rows >= kPairRowsThresholdMx;
  return dt == MOE_BF16 && rows >= kPairRowsThresholdGemm2;
}

// The swapped-operand kernel (gemm_tc_swap.cu: weight rows on the MMA's M side, an
// expert's tokens on N, padded to 16).  Measured on B300 against the token-major kernels
// (graph-replayed layer steps, 2032 MHz):
//   * it wins for bf16 GEMM1 where one tile of up to 384 tokens covers an expert that the
//     token-major tiles split into two 256-row or three 128-row m-tiles, each re-streaming
//     the expert's weights: the EP64 slice at T = 8192 (269 rows per expert, d = 7168):
//     GEMM1 96.6 -> 82-86 us;
//   * it loses elsewhere: with a few dozen tokens per expert every tile still streams its
//     256 weight rows and issues its K / 16 MMAs, now for 128 weight rows per SM instead of
//     256 (EP64 slice at T = 2048: GEMM1 54 -> 62-75 us; Zipf EP8 slice: 95 -> 198), and an
//     expert's short last chunk costs a full weight pass (T = 32768: GEMM1 189 -> 265); its
//     GEMM2 (K = f) and its MXFP8 tiles lost at every shape tried (EP64 slice: GEMM2 67 ->
//     89 us bf16, 57 -> 72 MXFP8; MXFP8 GEMM1 69 -> 74-86).
// Tokens per tile: 1.2 x the expected rows, rounded up to 32 (MXFP8: to 128, the scale
// layout's row tiles), within [64, 384] (MXFP8 [128, 384]); experts above it take more
// tiles.  MOE_KERNEL_SWAP forces it for either GEMM and dtype.
constexpr int kSwapRowsMin = 256;
constexpr int kSwapRowsMax = 320;
constexpr int kSwapElocMax = 256;

static int swap_tokens(moe_dtype dt, int64_t rows) {
  const int gran = dt == MOE_MXFP8 ? 128 : 32;
  const int64_t nt = ((rows * 6 + 4) / 5 + gran - 1) / gran * gran;
  return static_cast<int>(std::min<int64_t>(384, std::max<int64_t>(nt, dt == MOE_MXFP8 ? 128 : 64)));
}

// Kernel shape of a grouped GEMM (0 = 1-CTA, 1 = token-major CTA pairs, >= 64 = swapped
// operands with that many tokens per tile).  rows_hint > 0: expected rows per expert; 0:
// N_cap / E_loc; MOE_KERNEL_* (negative): that kernel.  keeps_gu: GEMM1 must also write
// the gate/up pre-activations (the swapped kernel does not).
static int gemm_shape(bool gemm1, moe_dtype dt, int64_t n_cap, int E_loc, int rows_hint, int K, bool keeps_gu) {
  if (dt == MOE_FP8) return 0;  // per-tensor FP8: the 1-CTA block-scaled kernel, whatever the hint
  const int64_t rows = expected_rows(n_cap, E_loc, rows_hint > 0 ? rows_hint : 0);
  const bool swap_ok = dt != MOE_F32 && E_loc <= kSwapElocMax && !(gemm1 && keeps_gu);
  if (rows_hint == MOE_KERNEL_CTA) return 0;
  if (rows_hint == MOE_KERNEL_PAIR) return dt == MOE_F32 ? 0 : 1;
  if (rows_hint == MOE_KERNEL_SWAP) return swap_ok ? swap_tokens(dt, std::max<int64_t>(rows, 1)) : 0;
  if (swap_ok && gemm1 && dt == MOE_BF16 && K >= 4096 && rows >= kSwapRowsMin && rows <= kSwapRowsMax)
    return swap_tokens(dt, rows);
  return (gemm1 ? use_pair(dt, n_cap, E_loc, rows_hint, K) : use_pair_gemm2(dt, n_cap, E_loc, rows_hint)) ? 1 : 0;
}

static cudaError_t run_gemm1(const void* perm_x, const uint8_t* perm_sf, const int32_t* offsets,
                             const float* row_prob, int64_t n_cap, int E_loc, int d, int f, moe_dtype dt,
                             const void* Wgu, const uint8_t* Wgu_sf, void* h, uint8_t* h_sf, int32_t* err,
                             int rows_hint, cudaStream_t st, void* gu_save = nullptr, void* h16 = nullptr,
                             uint32_t* h_amax = nullptr) {
  if (n_cap == 0) return cudaSuccess;
  if (dt == MOE_FP8) {
    // per-tensor FP8: bf16 h and its largest magnitude first, then h as one E4M3 tensor
    // (one exponent, rows in place order) for GEMM2
    if (!h16 || !h_amax) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(h_amax, 0, 4, st);
    if (e == cudaSuccess)
      e = launch_tc_gemm1_fp8(perm_x, perm_sf, offsets, row_prob, n_cap, E_loc, d, f, Wgu, Wgu_sf, h16, h_amax, err,
                              kTimeoutNs, st);
    if (e == cudaSuccess)
      e = launch_gather_rows_mx(h16, f, offsets, E_loc, nullptr, nullptr, static_cast<uint8_t*>(h), h_sf, st, h_amax);
    return e;
  }
  if (dt == MOE_F32)
    return launch_simt_gemm1(static_cast<const float*>(perm_x), offsets, row_prob, n_cap, E_loc, d, f,
                             static_cast<const float*>(Wgu), static_cast<float*>(h), st);
  return launch_tc_gemm1(perm_x, perm_sf, offsets, row_prob, n_cap, E_loc, d, f, is_fp8(dt),
                         gemm_shape(true, dt, n_cap, E_loc, rows_hint, d, gu_save != nullptr), Wgu, Wgu_sf, h, h_sf,
                         err, kTimeoutNs, gu_save, st);
}

static cudaError_t run_gemm2(const void* h, const uint8_t* h_sf, const int32_t* offsets, int64_t n_cap, int E_loc,
                             int d, int f, moe_dtype dt, const void* Wd, const uint8_t* Wd_sf, void* Y2, int32_t* err,
                             int rows_hint, cudaStream_t st) {
  if (n_cap == 0) return cudaSuccess;
  if (dt == MOE_F32)
    return launch_simt_gemm2(static_cast<const float*>(h), offsets, n_cap, E_loc, d, f, static_cast<const float*>(Wd),
                             static_cast<float*>(Y2), st);
  return launch_tc_gemm2(h, h_sf, offsets, n_cap, E_loc, d, f, is_fp8(dt),
                         gemm_shape(false, dt, n_cap, E_loc, rows_hint, f, false), Wd, Wd_sf, Y2, err, kTimeoutNs, st);
}

static cudaError_t run_mlp(const void* perm_x, const uint8_t* perm_sf, const int32_t* offsets, const float* row_prob,
                           int64_t n_cap, int E_loc, int d, int f, moe_dtype dt, const void* Wgu, const uint8_t* Wgu_sf,
                           const void* Wd, const uint8_t* Wd_sf, void* Y2, uint8_t* scratch, int32_t* err,
                           int rows_hint, cudaStream_t st, void* gu_save = nullptr) {
  MlpScratch s = carve_mlp(scratch, n_cap, f, dt, E_loc);
  cudaError_t e = run_gemm1(perm_x, perm_sf, offsets, row_prob, n_cap, E_loc, d, f, dt, Wgu, Wgu_sf, s.h, s.h_sf, err,
                            rows_hint, st, gu_save, s.h16, s.h_amax);
  if (e != cudaSuccess) return e;
  return run_gemm2(s.h, s.h_sf, offsets, n_cap, E_loc, d, f, dt, Wd, Wd_sf, Y2, err, rows_hint, st);
}

// The bf16 layer reads x rows straight into GEMM1 (row gather), on CTA pairs or the 1-CTA
// kernel; fp32 (SIMT) and MXFP8 take a permuted copy.  Measured on B300, the MXFP8
// row-gather GEMM1 was 7-10 % slower than the TMA-fed one and quantising per token saved
// nothing over quantising while copying, while bf16 gains: the permuted copy costs 27 us
// at T = 4096, d = 2048, k = 8 and the gather adds less than that to GEMM1.
static bool layer_gathers(moe_dtype dt, int T, int d, int k, int E, int E_loc) {
  (void)T; (void)d; (void)k; (void)E; (void)E_loc;
  return dt == MOE_BF16;
}

// The layer folds the combine into GEMM2 (direct rows for tokens with one local slot, zero
// rows from the GEMM's extra warps, a sparse pass for the few with several) when tokens
// average under one local slot, k E_loc < E: measured on B300 the EP64-shaped slices gain
// (GEMM2 + combine 196 -> 162 us at T = 32768, 74 -> 68 at T = 8192, MXFP8 66 -> 57),
// while with one or more local slots per token (all experts local, or the Zipf EP8 slice)
// GEMM2 with its TMA-store epilogue followed by the combine kernel is faster (148 vs 158 us
// at T = 4096, d = 2048, 64 of 64 experts).
static bool fuses_combine(moe_dtype dt, int k, int E_loc, int E) {
  return dt != MOE_F32 && static_cast<int64_t>(k) * E_loc < E;
}

// ---- whole-layer workspace -------------------------------------------------------------
struct LayerWs {
  int32_t* err;
  int32_t* topk_ids;
  float* topk_probs;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_src_token;
  float* row_prob;
  int32_t* pair_to_row;
  uint8_t* perm_ws;
  void* perm_x;      // permuted copy (no row gather) or, MXFP8 row gather, E4M3 x [T, d]
  uint8_t* perm_sf;  // its scales (SF tile layout, or row-major [T, d / 32] for the row gather)
  uint8_t* mlp;
  void* Y2;
  int32_t* tok_nloc;  // bf16 / MXFP8: local slots per token (combine in GEMM2)
  size_t total;
};
static LayerWs layer_layout(uint8_t* base, int T, int d, int f, int E, int k, int E_loc, moe_dtype dt) {
  const int64_t n_cap = n_cap_of(T, k, E_loc);
  const bool gather = layer_gathers(dt, T, d, k, E, E_loc);
  LayerWs w{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + o : nullptr;
    o += align_up(bytes, kAlign);
    return p;
  };
  w.err = reinterpret_cast<int32_t*>(take(sizeof(WsHeader)));
  w.topk_ids = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * k * 4));
  w.topk_probs = reinterpret_cast<float*>(take(static_cast<size_t>(T) * k * 4));
  w.counts = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E_loc) * 4));
  w.offsets = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E_loc + 1) * 4));
  w.row_src_token = reinterpret_cast<int32_t*>(take(static_cast<size_t>(n_cap) * 4));
  w.row_prob = reinterpret_cast<float*>(take(static_cast<size_t>(n_cap) * 4));
  w.pair_to_row = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * k * 4));
  w.perm_ws = take(permute_ws_bytes(T, E_loc));
  if (!gather) {
    w.perm_x = take(static_cast<size_t>(n_cap) * d * elt_bytes(dt));
    w.perm_sf = is_fp8(dt) ? take(mx_act_sf_bytes(n_cap, d, E_loc)) : nullptr;
  } else if (dt == MOE_MXFP8) {
    w.perm_x = take(static_cast<size_t>(T) * d);
    w.perm_sf = take(static_cast<size_t>(T) * (d / 32));
  }
  w.mlp = take(mlp_scratch_bytes(n_cap, E_loc, f, dt));
  w.Y2 = take(static_cast<size_t>(n_cap) * d * (dt == MOE_F32 ? 4 : 2));
  if (fuses_combine(dt, k, E_loc, E)) w.tok_nloc = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * 4));
  w.total = o;
  return w;
}

// ---- backward workspace ------------------------------------------------------------------
struct BackwardWs {
  int32_t* err;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_src_token;
  float* row_prob;
  int32_t* pair_to_row;
  uint8_t* perm_ws;
  void* gu;        // [N_cap, 2f] bf16, packed order
  void* dgu;       // [N_cap, 2f] bf16, packed order
  void* h;         // [N_cap, f] bf16
  float* dp_part;  // [N_cap, f / 32]
  void* dxp;       // [N_cap, d] bf16
  void* x_rows;    // [N_cap, d] bf16: x and dy in routed-row order, the GEMM operands
  void* dy_rows;   //   (TMA-loadable, unlike token-indexed rows)
  // MXFP8 backward: x and dy rows quantised along d, dg/du rows along f (E4M3 + scales in
  // the activation SF tile layout)
  uint8_t *x_q, *x_sf, *dy_q, *dy_sf, *dgu_q, *dgu_sf;
  uint32_t* amax;  // per-tensor FP8: largest |x|, |dy|, |h|, |[dg du]| (fp32 bits)
  int32_t* tok_nloc;  // [T] local slots per token (the dx GEMM that combines)
  size_t total;
};
static BackwardWs backward_layout(uint8_t* base, int T, int d, int f, int k, int E_loc, bool mx = false) {
  const int64_t n_cap = n_cap_of(T, k, E_loc);
  BackwardWs w{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + o : nullptr;
    o += align_up(bytes, kAlign);
    return p;
  };
  w.err = reinterpret_cast<int32_t*>(take(sizeof(WsHeader)));
  w.counts = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E_loc) * 4));
  w.offsets = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E_loc + 1) * 4));
  w.row_src_token = reinterpret_cast<int32_t*>(take(static_cast<size_t>(n_cap) * 4));
  w.row_prob = reinterpret_cast<float*>(take(static_cast<size_t>(n_cap) * 4));
  w.pair_to_row = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * k * 4));
  w.perm_ws = take(permute_ws_bytes(T, E_loc));
  w.gu = take(static_cast<size_t>(n_cap) * 2 * f * 2);
  w.dgu = take(static_cast<size_t>(n_cap) * 2 * f * 2);
  w.h = take(static_cast<size_t>(n_cap) * f * 2);
  w.dp_part = reinterpret_cast<float*>(take(static_cast<size_t>(n_cap) * (f / 32) * 4));
  w.dxp = take(static_cast<size_t>(n_cap) * d * 2);
  w.x_rows = take(static_cast<size_t>(n_cap) * d * 2);
  w.dy_rows = take(static_cast<size_t>(n_cap) * d * 2);
  w.tok_nloc = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * 4));
  if (mx) {  // MXFP8 operands of the row-wise GEMMs (recompute, dh, dx)
    w.x_q = take(static_cast<size_t>(n_cap) * d);
    w.x_sf = take(mx_act_sf_bytes(n_cap, d, E_loc));
    w.dy_q = take(static_cast<size_t>(n_cap) * d);
    w.dy_sf = take(mx_act_sf_bytes(n_cap, d, E_loc));
    w.dgu_q = take(static_cast<size_t>(n_cap) * 2 * f);
    w.dgu_sf = take(mx_act_sf_bytes(n_cap, 2 * f, E_loc));
    w.amax = reinterpret_cast<uint32_t*>(take(16));
  }
  w.total = o;
  return w;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_gu_block(int f) { return f > 0 && f % 32 == 0 ? 32 : 0; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_supported(void) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return 0;
  return (major == 10 && minor == 3) ? 1 : 0;
}

size_t moe_mx_act_scale_bytes(int64_t N_cap, int K, int E_loc) {
  if (N_cap < 0 || K <= 0 || K % 128 != 0 || E_loc < 1) return 0;
  return mx_act_sf_bytes(N_cap, K, E_loc);
}

size_t moe_mx_weight_scale_bytes(int E_loc, int rows, int K) {
  if (E_loc < 1 || rows <= 0 || rows % 128 != 0 || K <= 0 || K % 128 != 0) return 0;
  return static_cast<size_t>(E_loc) * (rows / 128) * (K / 128) * 512;
}

moe_status moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_probs,
                          moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 32) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_ids || !topk_probs)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_route_topk(logits, T, E, k, topk_ids, topk_probs, stream));
}

size_t moe_permute_workspace_size(int T, int k, int E_loc) {
  (void)k;
  if (T < 0 || E_loc < 1 || E_loc > 1024) return 0;
  return sizeof(WsHeader) + permute_ws_bytes(T, E_loc);
}

}  // extern "C"

// Argument checks of moe_permute (also run first by moe_permute_noalloc).
moe_status moe::check_permute(const void* x, moe_dtype x_dtype, moe_dtype perm_dtype, int T, int d, const void* ids,
                              const void* probs, int k, int e0, int E_loc, const void* perm_x, const void* perm_sf,
                              const void* counts, const void* offsets, const void* rst, const void* rp,
                              const void* p2r) {
  if (T < 0 || d <= 0 || k < 1 || k > 32 || e0 < 0 || E_loc < 1 || E_loc > 1024 || e0 > kMaxExpertId + 1 - E_loc)
    return MOE_ERR_INVALID_ARG;
  if (n_cap_of(T, k, E_loc) > kMaxRows) return MOE_ERR_INVALID_ARG;  // int32 rows and offsets
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !ids || !probs || !rst || !rp || !p2r)) return MOE_ERR_INVALID_ARG;
  const bool ok_types = (x_dtype == MOE_F32 && perm_dtype == MOE_F32) || (x_dtype == MOE_BF16 && perm_dtype == MOE_BF16) ||
                        ((x_dtype == MOE_BF16 || x_dtype == MOE_F32) && is_fp8(perm_dtype));
  if (!ok_types) return MOE_ERR_UNSUPPORTED;
  if ((x_dtype == MOE_BF16 && d % 8 != 0) || (x_dtype == MOE_F32 && d % 4 != 0)) return MOE_ERR_UNSUPPORTED;
  // perm_x == NULL: maps only (no permuted copy, so no scales either)
  if (is_fp8(perm_dtype) && (d % 128 != 0 || (T > 0 && perm_x && !perm_sf)))
    return (T > 0 && perm_x && !perm_sf) ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!aligned16(x) || (perm_x && !aligned16(perm_x)))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// dx = the slot sum of the dx rows [N_cap, d] = [dg du] (K = 2f) x WguT per expert.  On
// expert slices with under one local slot per token (k E_loc < E) the GEMM writes the dx
// rows of single-slot tokens straight to dx and zero rows for tokens with none, and a
// sparse pass sums the others (the forward GEMM2's combine mode); otherwise a store GEMM
// and the combine kernel.  a / a_sf: the [dg du] rows (bf16, or E4M3 + SF when mx).
static cudaError_t backward_dx(bool mx, const void* a, const uint8_t* a_sf, const BackwardWs& w, int64_t n_cap, int T,
                               int E, int k, int E_loc, int d, int f, const void* B, const uint8_t* b_sf, void* dx,
                               cudaStream_t st) {
  const moe_dtype dt = mx ? MOE_MXFP8 : MOE_BF16;
  if (n_cap > 0 && fuses_combine(dt, k, E_loc, E)) {
    const int shape = gemm_shape(false, dt, n_cap, E_loc, moe_rows_hint(T, k, E), 2 * f, false);
    cudaError_t e = launch_tc_gemm2_combine(a, a_sf, w.offsets, n_cap, E_loc, d, 2 * f, mx, shape, B, b_sf, w.dxp,
                                            w.row_src_token, w.tok_nloc, T, dx, w.err, kTimeoutNs, st);
    if (e == cudaSuccess)
      e = launch_combine_multi(w.dxp, w.pair_to_row, w.tok_nloc, T, k, d, dx, static_cast<double>(k) * E_loc / E, st);
    return e;
  }
  cudaError_t e = cudaSuccess;
  if (n_cap > 0)
    e = mx ? launch_tc_gemm_store_mx(a, a_sf, n_cap, w.offsets, E_loc, 2 * f, d, B, b_sf, w.dxp, w.err, kTimeoutNs, st)
           : launch_tc_gemm_store(a, n_cap, w.offsets, E_loc, 2 * f, d, B, w.dxp, w.err, kTimeoutNs, st);
  if (e == cudaSuccess) e = launch_combine(w.dxp, w.pair_to_row, T, k, d, MOE_BF16, dx, st);
  return e;
}

extern "C" {

moe_status moe_permute(const void* x, moe_dtype x_dtype, moe_dtype perm_dtype, int T, int d, const int32_t* topk_ids,
                       const float* topk_probs, int k, int e0, int E_loc, void* perm_x, uint8_t* perm_x_scale,
                       int32_t* counts, int32_t* offsets, int32_t* row_src_token, float* row_prob,
                       int32_t* pair_to_row, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  moe_status s = check_permute(x, x_dtype, perm_dtype, T, d, topk_ids, topk_probs, k, e0, E_loc, perm_x, perm_x_scale,
                               counts, offsets, row_src_token, row_prob, pair_to_row);
  if (s != MOE_OK) return s;
  if (!workspace || !aligned256(workspace) || workspace_bytes < moe_permute_workspace_size(T, k, E_loc))
    return MOE_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return cuda_status(launch_permute(x, x_dtype, perm_dtype, T, d, topk_ids, topk_probs, k, e0, E_loc, perm_x,
                                    perm_x_scale, counts, offsets, row_src_token, row_prob, pair_to_row,
                                    ws + sizeof(WsHeader), stream));
}

moe_status moe_pack_weights(const void* W_gate, const void* W_up, const void* W_down, moe_dtype src_dtype,
                            moe_dtype dst_dtype, int E_loc, int d, int f, void* Wgu_packed, void* Wd_packed,
                            uint8_t* Wgu_scale, uint8_t* Wd_scale, moe_stream_t stream) {
  if (!W_gate || !W_up || !W_down || !Wgu_packed || !Wd_packed) return MOE_ERR_INVALID_ARG;
  moe_status s = check_mlp_shape(d, f, E_loc, dst_dtype);
  if (s != MOE_OK) return s;
  const bool ok_types = (src_dtype == MOE_F32 && dst_dtype == MOE_F32) ||
                        (src_dtype == MOE_BF16 && dst_dtype == MOE_BF16) ||
                        ((src_dtype == MOE_BF16 || src_dtype == MOE_F32) && dst_dtype == MOE_MXFP8);
  if (!ok_types) return MOE_ERR_UNSUPPORTED;
  if (dst_dtype == MOE_MXFP8 && (!Wgu_scale || !Wd_scale)) return MOE_ERR_INVALID_ARG;
  if (dst_dtype == MOE_MXFP8 && (!aligned16(Wgu_packed) || !aligned16(Wd_packed))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack(W_gate, W_up, W_down, src_dtype, dst_dtype, E_loc, d, f, Wgu_packed, Wd_packed,
                                 Wgu_scale, Wd_scale, stream));
}

moe_status moe_pack_weights_fp8(const void* W_gate, const void* W_up, const void* W_down, moe_dtype src_dtype,
                                int E_loc, int d, int f, void* Wgu_packed, void* Wd_packed, uint8_t* Wgu_scale,
                                uint8_t* Wd_scale, int32_t* w_exp, moe_stream_t stream) {
  if (!W_gate || !W_up || !W_down || !Wgu_packed || !Wd_packed || !Wgu_scale || !Wd_scale || !w_exp)
    return MOE_ERR_INVALID_ARG;
  moe_status s = check_mlp_shape(d, f, E_loc, MOE_FP8);
  if (s != MOE_OK) return s;
  if (src_dtype != MOE_BF16 && src_dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(W_gate) || !aligned16(W_up) || !aligned16(W_down) || !aligned16(Wgu_packed) || !aligned16(Wd_packed))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack_fp8(W_gate, W_up, W_down, src_dtype, E_loc, d, f, Wgu_packed, Wd_packed, Wgu_scale,
                                     Wd_scale, w_exp, stream));
}

size_t moe_grouped_mlp_workspace_size(int64_t N_cap, int E_loc, int d, int f, moe_dtype dtype) {
  (void)d;
  if (N_cap < 0 || E_loc < 1 || f <= 0) return 0;
  return sizeof(WsHeader) + mlp_scratch_bytes(N_cap, E_loc, f, dtype);
}

moe_status moe_grouped_mlp(const void* perm_x, const uint8_t* perm_x_scale, const int32_t* offsets,
                           const float* row_prob, int64_t N_cap, int E_loc, int d, int f, moe_dtype dtype,
                           const void* Wgu_packed, const uint8_t* Wgu_scale, const void* Wd_packed,
                           const uint8_t* Wd_scale, void* Y2, int rows_hint, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream) {
  moe_status s = check_mlp_shape(d, f, E_loc, dtype);
  if (s != MOE_OK) return s;
  if (N_cap < 0 || N_cap > (int64_t(1) << 31) - 1) return MOE_ERR_INVALID_ARG;
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (N_cap > 0 && (!perm_x || !row_prob || !Wgu_packed || !Wd_packed || !Y2)) return MOE_ERR_INVALID_ARG;
  if (is_fp8(dtype) && N_cap > 0 && (!perm_x_scale || !Wgu_scale || !Wd_scale)) return MOE_ERR_INVALID_ARG;
  if (N_cap > 0 && (!aligned16(perm_x) || !aligned16(Wgu_packed) || !aligned16(Wd_packed) || !aligned16(Y2) ||
                    (perm_x_scale && !aligned16(perm_x_scale)) || (Wgu_scale && !aligned16(Wgu_scale)) ||
                    (Wd_scale && !aligned16(Wd_scale))))
    return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < moe_grouped_mlp_workspace_size(N_cap, E_loc, d, f, dtype))
    return MOE_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return cuda_status(run_mlp(perm_x, perm_x_scale, offsets, row_prob, N_cap, E_loc, d, f, dtype, Wgu_packed, Wgu_scale,
                             Wd_packed, Wd_scale, Y2, ws + sizeof(WsHeader), reinterpret_cast<int32_t*>(ws), rows_hint,
                             stream));
}

size_t moe_expert_gemm_workspace_size(void) { return sizeof(WsHeader); }

int moe_rows_hint(int T, int k, int E) {
  if (T <= 0 || k <= 0 || E <= 0) return 0;
  return static_cast<int>(static_cast<int64_t>(T) * k / E);
}

int moe_layer_fused_combine(int k, int E, int E_loc, moe_dtype dtype) {
  if (k <= 0 || E <= 0 || E_loc <= 0 || E_loc > E) return -1;
  return fuses_combine(dtype, k, E_loc, E) ? 1 : 0;
}

int moe_layer_gemm1_pairs(int T, int d, int k, int E, int E_loc, moe_dtype dtype) {
  if (T < 0 || d <= 0 || k <= 0 || E <= 0 || E_loc <= 0 || E_loc > E) return -1;
  return gemm_shape(true, dtype, n_cap_of(T, k, E_loc), E_loc, moe_rows_hint(T, k, E), d, false) == 1 ? 1 : 0;
}

int moe_layer_gemm_kernel(int T, int d, int f, int k, int E, int E_loc, moe_dtype dtype, int gemm) {
  if (T < 0 || d <= 0 || f <= 0 || k <= 0 || E <= 0 || E_loc <= 0 || E_loc > E || (gemm != 1 && gemm != 2))
    return 0;
  if (dtype != MOE_F32 && dtype != MOE_BF16 && !is_fp8(dtype)) return 0;
  const int s = gemm_shape(gemm == 1, dtype, n_cap_of(T, k, E_loc), E_loc, moe_rows_hint(T, k, E), gemm == 1 ? d : f,
                           false);
  return s >= kShapeSwapMin ? MOE_KERNEL_SWAP : s == 1 ? MOE_KERNEL_PAIR : MOE_KERNEL_CTA;
}

static moe_status check_gemm_common(int64_t N_cap, int E_loc, int d, int f, moe_dtype dtype, const void* offsets,
                                    const void* a, const void* a_sf, const void* w, const void* w_sf, const void* out,
                                    const void* out_sf) {
  moe_status s = check_mlp_shape(d, f, E_loc, dtype);
  if (s != MOE_OK) return s;
  if (N_cap < 0 || N_cap > (int64_t(1) << 31) - 1 || !offsets) return MOE_ERR_INVALID_ARG;
  if (N_cap == 0) return MOE_OK;
  if (!a || !w || !out || !aligned16(a) || !aligned16(w) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (is_fp8(dtype) && (!a_sf || !w_sf || !aligned16(a_sf) || !aligned16(w_sf))) return MOE_ERR_INVALID_ARG;
  (void)out_sf;
  return MOE_OK;
}

moe_status moe_expert_gemm1_swiglu(const void* perm_x, const uint8_t* perm_x_scale, const int32_t* offsets,
                                   const float* row_prob, int64_t N_cap, int E_loc, int d, int f, moe_dtype dtype,
                                   const void* Wgu_packed, const uint8_t* Wgu_scale, void* h, uint8_t* h_scale,
                                   int rows_hint, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  moe_status s = check_gemm_common(N_cap, E_loc, d, f, dtype, offsets, perm_x, perm_x_scale, Wgu_packed, Wgu_scale, h,
                                   h_scale);
  if (s != MOE_OK) return s;
  if (N_cap > 0 && (!row_prob || (is_fp8(dtype) && !h_scale))) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < moe_expert_gemm1_workspace_size(N_cap, f, dtype))
    return MOE_ERR_WORKSPACE;
  int32_t* err = static_cast<int32_t*>(workspace);
  // per-tensor FP8: GEMM1's bf16 h and its amax live in the workspace after the error word
  uint8_t* h16 = static_cast<uint8_t*>(workspace) + sizeof(WsHeader);
  uint32_t* h_amax = reinterpret_cast<uint32_t*>(h16 + align_up(static_cast<size_t>(N_cap) * f * 2, kAlign));
  return cuda_status(run_gemm1(perm_x, perm_x_scale, offsets, row_prob, N_cap, E_loc, d, f, dtype, Wgu_packed,
                               Wgu_scale, h, h_scale, err, rows_hint, stream, nullptr,
                               dtype == MOE_FP8 ? h16 : nullptr, dtype == MOE_FP8 ? h_amax : nullptr));
}

size_t moe_expert_gemm1_workspace_size(int64_t N_cap, int f, moe_dtype dtype) {
  if (N_cap < 0 || f <= 0) return 0;
  if (dtype != MOE_FP8) return sizeof(WsHeader);
  return sizeof(WsHeader) + align_up(static_cast<size_t>(N_cap) * f * 2, kAlign) + kAlign;
}

moe_status moe_expert_gemm1_swiglu_gather(const void* x, const uint8_t* x_scale, const int32_t* row_src_token,
                                          const int32_t* offsets, const float* row_prob, int64_t N_cap, int E_loc,
                                          int d, int f, moe_dtype dtype, const void* Wgu_packed,
                                          const uint8_t* Wgu_scale, void* h, uint8_t* h_scale, int rows_hint,
                                          void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (dtype == MOE_F32 || dtype == MOE_FP8) return MOE_ERR_UNSUPPORTED;
  moe_status s = check_gemm_common(N_cap, E_loc, d, f, dtype, offsets, x, x_scale, Wgu_packed, Wgu_scale, h, h_scale);
  if (s != MOE_OK) return s;
  if (N_cap > 0 && (!row_src_token || !row_prob || (dtype == MOE_MXFP8 && !h_scale))) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
  if (N_cap == 0) return MOE_OK;
  return cuda_status(launch_tc_gemm1_gather(x, x_scale, row_src_token, offsets, row_prob, N_cap, E_loc, d, f,
                                            dtype == MOE_MXFP8,
                                            dtype == MOE_MXFP8 ? 0 : gemm_shape(true, dtype, N_cap, E_loc, rows_hint, d, false),
                                            Wgu_packed, Wgu_scale, h, h_scale, static_cast<int32_t*>(workspace),
                                            kTimeoutNs, nullptr, stream));
}

moe_status moe_quantize_mx_rows(const void* x, moe_dtype x_dtype, int T, int d, const int32_t* pair_to_row, int k,
                                uint8_t* xq, uint8_t* x_scale, moe_stream_t stream) {
  if (T < 0 || d <= 0 || (pair_to_row && (k < 1 || k > 32))) return MOE_ERR_INVALID_ARG;
  if ((x_dtype != MOE_BF16 && x_dtype != MOE_F32) || d % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!x || !xq || !x_scale || !aligned16(x) || !aligned16(xq))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quant_rows_mx(x, x_dtype, T, d, pair_to_row, k, xq, x_scale, stream));
}

moe_status moe_expert_gemm2(const void* h, const uint8_t* h_scale, const int32_t* offsets, int64_t N_cap, int E_loc,
                            int d, int f, moe_dtype dtype, const void* Wd_packed, const uint8_t* Wd_scale, void* Y2,
                            int rows_hint, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  moe_status s = check_gemm_common(N_cap, E_loc, d, f, dtype, offsets, h, h_scale, Wd_packed, Wd_scale, Y2, nullptr);
  if (s != MOE_OK) return s;
  if (!workspace || !aligned256(workspace) || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
  int32_t* err = static_cast<int32_t*>(workspace);
  return cuda_status(
      run_gemm2(h, h_scale, offsets, N_cap, E_loc, d, f, dtype, Wd_packed, Wd_scale, Y2, err, rows_hint, stream));
}

moe_status moe_unpermute_combine(const void* Y2, const int32_t* pair_to_row, int T, int k, int d, moe_dtype dtype,
                                 void* y, moe_stream_t stream) {
  if (T < 0 || k < 1 || k > 32 || d <= 0) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F32 && dtype != MOE_BF16 && !is_fp8(dtype)) return MOE_ERR_UNSUPPORTED;
  if ((dtype == MOE_F32 && d % 4 != 0) || (dtype != MOE_F32 && d % 8 != 0)) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!Y2 || !pair_to_row || !y || !aligned16(Y2) || !aligned16(y))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(Y2, pair_to_row, T, k, d, dtype, y, stream));
}

// Scratch of moe_expert_gemm2_combine: header, Y2 rows, per-token slot counts.
struct Gemm2CombineWs {
  int32_t* err;
  void* Y2;
  int32_t* tok_nloc;
  size_t total;
};
static Gemm2CombineWs gemm2_combine_layout(uint8_t* base, int64_t n_cap, int T, int d) {
  Gemm2CombineWs w{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + o : nullptr;
    o += align_up(bytes, kAlign);
    return p;
  };
  w.err = reinterpret_cast<int32_t*>(take(sizeof(WsHeader)));
  w.Y2 = take(static_cast<size_t>(n_cap) * d * 2);
  w.tok_nloc = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * 4));
  w.total = o;
  return w;
}

size_t moe_expert_gemm2_combine_workspace_size(int64_t N_cap, int T, int d) {
  if (N_cap < 0 || T < 0 || d <= 0) return 0;
  return gemm2_combine_layout(nullptr, N_cap, T, d).total;
}

moe_status moe_expert_gemm2_combine(const void* h, const uint8_t* h_scale, const int32_t* offsets,
                                    const int32_t* row_src_token, const int32_t* pair_to_row, int T, int k,
                                    int64_t N_cap, int E_loc, int d, int f, moe_dtype dtype, const void* Wd_packed,
                                    const uint8_t* Wd_scale, void* y, int rows_hint, void* workspace,
                                    size_t workspace_bytes, moe_stream_t stream) {
  if (dtype == MOE_F32) return MOE_ERR_UNSUPPORTED;
  moe_status s = check_gemm_common(N_cap, E_loc, d, f, dtype, offsets, h, h_scale, Wd_packed, Wd_scale, y, nullptr);
  if (s != MOE_OK) return s;
  if (T < 0 || k < 1 || k > 32) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!row_src_token || !pair_to_row || !y || !aligned16(y))) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < moe_expert_gemm2_combine_workspace_size(N_cap, T, d))
    return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  // no routed rows at all: every token's row is zero (the combine kernel reads no Y2 then)
  if (N_cap == 0) return cuda_status(launch_combine(nullptr, pair_to_row, T, k, d, MOE_BF16, y, stream));
  Gemm2CombineWs w = gemm2_combine_layout(static_cast<uint8_t*>(workspace), N_cap, T, d);
  cudaError_t e = launch_combine_prep(pair_to_row, T, k, w.tok_nloc, stream);
  if (e == cudaSuccess)
    e = launch_tc_gemm2_combine(h, h_scale, offsets, N_cap, E_loc, d, f, is_fp8(dtype),
                                gemm_shape(false, dtype, N_cap, E_loc, rows_hint, f, false), Wd_packed, Wd_scale, w.Y2,
                                row_src_token, w.tok_nloc, T, y, static_cast<int32_t*>(workspace), kTimeoutNs, stream);
  // expected local slots per token (rows_hint rows per expert), which picks the sparse or
  // dense pass for the tokens with several local slots (same result either way)
  const double slots = rows_hint > 0 ? static_cast<double>(rows_hint) * E_loc / T : static_cast<double>(N_cap) / T;
  if (e == cudaSuccess) e = launch_combine_multi(w.Y2, pair_to_row, w.tok_nloc, T, k, d, y, slots, stream);
  return cuda_status(e);
}

size_t moe_layer_workspace_size(int T, int d, int f, int E, int k, int E_loc, moe_dtype dtype) {
  if (T < 0 || d <= 0 || f <= 0 || E < 1 || k < 1 || E_loc < 1) return 0;
  (void)E;
  return layer_layout(nullptr, T, d, f, E, k, E_loc, dtype).total;
}

// Layer forward behind moe_layer_forward and moe_layer_forward_train: ids/probs (when not
// null) receive the routing instead of the workspace; gu_save (bf16 only) keeps the gate/up
// pre-activations for the backward.
static moe_status layer_forward_impl(const void* x, const float* logits, int T, int d, int f, int E, int k, int e0,
                                     int E_loc, moe_dtype dtype, const void* Wgu_packed, const uint8_t* Wgu_scale,
                                     const void* Wd_packed, const uint8_t* Wd_scale, void* y, int32_t* ids,
                                     float* probs, void* gu_save, void* workspace, size_t workspace_bytes,
                                     moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 32) return MOE_ERR_INVALID_ARG;
  if (e0 < 0 || E_loc < 1 || e0 + E_loc > E) return MOE_ERR_INVALID_ARG;
  if (n_cap_of(T, k, E_loc) > kMaxRows) return MOE_ERR_INVALID_ARG;  // int32 rows and offsets
  moe_status s = check_mlp_shape(d, f, E_loc, dtype);
  if (s != MOE_OK) return s;
  if (!Wgu_packed || !Wd_packed) return MOE_ERR_INVALID_ARG;
  if (is_fp8(dtype) && (!Wgu_scale || !Wd_scale)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !logits || !y || !aligned16(x) || !aligned16(y))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(Wgu_packed) || !aligned16(Wd_packed)) return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_F32 && d % 4 != 0) return MOE_ERR_UNSUPPORTED;
  const size_t need = moe_layer_workspace_size(T, d, f, E, k, E_loc, dtype);
  if (!workspace || !aligned256(workspace) || workspace_bytes < need) return MOE_ERR_WORKSPACE;
  LayerWs w = layer_layout(static_cast<uint8_t*>(workspace), T, d, f, E, k, E_loc, dtype);
  if (ids) w.topk_ids = ids;
  if (probs) w.topk_probs = probs;
  const int64_t n_cap = n_cap_of(T, k, E_loc);
  const moe_dtype x_dtype = dtype == MOE_F32 ? MOE_F32 : MOE_BF16;
  const int hint = moe_rows_hint(T, k, E);
  if (T == 0) return MOE_OK;  // nothing to route, compute or write
  // expert slices with under one local slot per token (bf16 / MXFP8): GEMM2 writes y for
  // the tokens with at most one local slot (the permute counts each token's slots) and a
  // sparse pass sums the others; otherwise GEMM2 and the combine kernel (fp32: SIMT GEMMs)
  const bool fused_combine = fuses_combine(dtype, k, E_loc, E);
  cudaError_t e = launch_route_topk(logits, T, E, k, w.topk_ids, w.topk_probs, stream);
  const bool gathers = layer_gathers(dtype, T, d, k, E, E_loc);
  if (e == cudaSuccess)  // maps only when GEMM1 reads the token rows itself
    e = launch_permute(x, x_dtype, dtype, T, d, w.topk_ids, w.topk_probs, k, e0, E_loc, gathers ? nullptr : w.perm_x,
                       gathers ? nullptr : w.perm_sf, w.counts, w.offsets, w.row_src_token, w.row_prob, w.pair_to_row,
                       w.perm_ws, stream, fused_combine ? w.tok_nloc : nullptr);
  MlpScratch ms = carve_mlp(w.mlp, n_cap, f, dtype, E_loc);
  if (gathers) {
    // GEMM1 reads the token rows (quantised once per token for MXFP8)
    const bool mx = dtype == MOE_MXFP8;
    if (e == cudaSuccess && mx)
      e = launch_quant_rows_mx(x, x_dtype, T, d, w.pair_to_row, k, static_cast<uint8_t*>(w.perm_x), w.perm_sf, stream);
    if (e == cudaSuccess)
      e = launch_tc_gemm1_gather(mx ? w.perm_x : x, w.perm_sf, w.row_src_token, w.offsets, w.row_prob, n_cap, E_loc,
                                 d, f, mx, mx ? 0 : gemm_shape(true, dtype, n_cap, E_loc, hint, d, gu_save != nullptr),
                                 Wgu_packed, Wgu_scale, ms.h, ms.h_sf, w.err, kTimeoutNs, gu_save, stream);
  } else if (e == cudaSuccess) {
    e = run_gemm1(w.perm_x, w.perm_sf, w.offsets, w.row_prob, n_cap, E_loc, d, f, dtype, Wgu_packed, Wgu_scale, ms.h,
                  ms.h_sf, w.err, hint, stream, gu_save, ms.h16, ms.h_amax);
  }
  if (fused_combine) {
    if (e == cudaSuccess)
      e = launch_tc_gemm2_combine(ms.h, ms.h_sf, w.offsets, n_cap, E_loc, d, f, is_fp8(dtype),
                                  gemm_shape(false, dtype, n_cap, E_loc, hint, f, false), Wd_packed, Wd_scale, w.Y2,
                                  w.row_src_token, w.tok_nloc, T, y, w.err, kTimeoutNs, stream);
    if (e == cudaSuccess)  // expected local slots per token: k E_loc / E
      e = launch_combine_multi(w.Y2, w.pair_to_row, w.tok_nloc, T, k, d, y,
                               static_cast<double>(k) * E_loc / E, stream);
  } else {
    if (e == cudaSuccess)
      e = run_gemm2(ms.h, ms.h_sf, w.offsets, n_cap, E_loc, d, f, dtype, Wd_packed, Wd_scale, w.Y2, w.err, hint, stream);
    if (e == cudaSuccess) e = launch_combine(w.Y2, w.pair_to_row, T, k, d, dtype, y, stream);
  }
  return cuda_status(e);
}

moe_status moe_layer_forward(const void* x, const float* logits, int T, int d, int f, int E, int k, int e0, int E_loc,
                             moe_dtype dtype, const void* Wgu_packed, const uint8_t* Wgu_scale, const void* Wd_packed,
                             const uint8_t* Wd_scale, void* y, void* workspace, size_t workspace_bytes,
                             moe_stream_t stream) {
  return layer_forward_impl(x, logits, T, d, f, E, k, e0, E_loc, dtype, Wgu_packed, Wgu_scale, Wd_packed, Wd_scale, y,
                            nullptr, nullptr, nullptr, workspace, workspace_bytes, stream);
}

moe_status moe_layer_forward_train(const void* x, const float* logits, int T, int d, int f, int E, int k, int e0,
                                   int E_loc, const void* Wgu_packed, const void* Wd_packed, void* y,
                                   int32_t* topk_ids, float* topk_probs, void* gu_saved, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream) {
  if (T > 0 && (!topk_ids || !topk_probs || !gu_saved || !aligned16(gu_saved))) return MOE_ERR_INVALID_ARG;
  return layer_forward_impl(x, logits, T, d, f, E, k, e0, E_loc, MOE_BF16, Wgu_packed, nullptr, Wd_packed, nullptr, y,
                            topk_ids, topk_probs, gu_saved, workspace, workspace_bytes, stream);
}

moe_status moe_pack_weights_backward(const void* W_gate, const void* W_up, moe_dtype src_dtype, int E_loc, int d,
                                     int f, void* WguT_packed, moe_stream_t stream) {
  if (!W_gate || !W_up || !WguT_packed || E_loc < 1 || E_loc > 1024 || d <= 0 || f <= 0) return MOE_ERR_INVALID_ARG;
  if ((src_dtype != MOE_BF16 && src_dtype != MOE_F32) || f % 32 != 0 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_pack_gu_t(W_gate, W_up, src_dtype, E_loc, d, f, WguT_packed, stream));
}

size_t moe_layer_backward_workspace_size(int T, int d, int f, int k, int E_loc) {
  if (T < 0 || d <= 0 || f <= 0 || k < 1 || E_loc < 1) return 0;
  return backward_layout(nullptr, T, d, f, k, E_loc).total;
}

moe_status moe_layer_backward(const void* x, const void* dy, const int32_t* topk_ids, const float* topk_probs, int T,
                              int d, int f, int E, int k, int e0, int E_loc, const void* Wgu_packed,
                              const void* W_down, const void* WguT_packed, const void* gu_saved, void* dx,
                              float* dlogits, float* dW_gate, float* dW_up, float* dW_down, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 32 || e0 < 0 || E_loc < 1 || e0 + E_loc > E)
    return MOE_ERR_INVALID_ARG;
  if (n_cap_of(T, k, E_loc) > kMaxRows) return MOE_ERR_INVALID_ARG;  // int32 rows and offsets
  moe_status s = check_mlp_shape(d, f, E_loc, MOE_BF16);
  if (s != MOE_OK) return s;
  if (!Wgu_packed || !W_down || !WguT_packed || !dW_gate || !dW_up || !dW_down) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !dy || !topk_ids || !topk_probs || !dx || !dlogits)) return MOE_ERR_INVALID_ARG;
  if (gu_saved && !aligned16(gu_saved)) return MOE_ERR_INVALID_ARG;
  if ((T > 0 && (!aligned16(x) || !aligned16(dy) || !aligned16(dx))) || !aligned16(Wgu_packed) ||
      !aligned16(W_down) || !aligned16(WguT_packed) || !aligned16(dW_gate) || !aligned16(dW_up) ||
      !aligned16(dW_down))
    return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < moe_layer_backward_workspace_size(T, d, f, k, E_loc))
    return MOE_ERR_WORKSPACE;
  BackwardWs w = backward_layout(static_cast<uint8_t*>(workspace), T, d, f, k, E_loc);
  const int64_t n_cap = n_cap_of(T, k, E_loc);
  cudaError_t e = cudaSuccess;
  if (T > 0)
    e = launch_permute(x, MOE_BF16, MOE_BF16, T, d, topk_ids, topk_probs, k, e0, E_loc, nullptr, nullptr, w.counts,
                       w.offsets, w.row_src_token, w.row_prob, w.pair_to_row, w.perm_ws, stream,
                       fuses_combine(MOE_BF16, k, E_loc, E) ? w.tok_nloc : nullptr);
  else
    e = cudaMemsetAsync(w.offsets, 0, static_cast<size_t>(E_loc + 1) * 4, stream);
  // dy and x rows in routed order: the A operands of the recompute and dh GEMMs and of
  // the weight gradients, all loaded by TMA
  if (e == cudaSuccess)
    e = launch_gather_rows(dy, static_cast<int64_t>(d) * 2, w.offsets, E_loc, w.row_src_token, w.dy_rows, stream);
  if (e == cudaSuccess)
    e = launch_gather_rows(x, static_cast<int64_t>(d) * 2, w.offsets, E_loc, w.row_src_token, w.x_rows, stream);
  if (e == cudaSuccess && n_cap > 0 && !gu_saved)  // recompute g, u unless the forward kept them
    e = launch_tc_gemm_store(w.x_rows, n_cap, w.offsets, E_loc, d, 2 * f, Wgu_packed, w.gu, w.err, kTimeoutNs, stream);
  if (e == cudaSuccess && n_cap > 0)
    e = launch_tc_dswiglu(w.dy_rows, w.offsets, w.row_prob, n_cap, E_loc, d, f, W_down, gu_saved ? gu_saved : w.gu,
                          w.dgu, w.h, w.dp_part, w.err, kTimeoutNs, stream);
  if (e == cudaSuccess)
    e = backward_dx(false, w.dgu, nullptr, w, n_cap, T, E, k, E_loc, d, f, WguT_packed, nullptr, dx, stream);
  if (e == cudaSuccess)
    e = launch_dlogits(topk_ids, topk_probs, w.pair_to_row, w.dp_part, f / 32, T, E, k, dlogits, stream);
  if (e == cudaSuccess)
    e = launch_wgrad_down_tc(w.h, w.dy_rows, w.offsets, std::max<int64_t>(n_cap, 1), E_loc, d, f, dW_down, w.err,
                             kTimeoutNs, stream);
  if (e == cudaSuccess)
    e = launch_wgrad_gate_up_tc(w.x_rows, w.dgu, w.offsets, std::max<int64_t>(n_cap, 1), E_loc, d, f, dW_gate, dW_up,
                                w.err, kTimeoutNs, stream);
  return cuda_status(e);
}

moe_status moe_pack_weights_backward_mx(const void* W_gate, const void* W_up, const void* W_down, moe_dtype src_dtype,
                                        int E_loc, int d, int f, uint8_t* WguT_q, uint8_t* WguT_scale, uint8_t* Wd_q,
                                        uint8_t* Wd_scale, moe_stream_t stream) {
  if (!W_gate || !W_up || !W_down || !WguT_q || !WguT_scale || !Wd_q || !Wd_scale || E_loc < 1 || E_loc > 1024 ||
      d <= 0 || f <= 0)
    return MOE_ERR_INVALID_ARG;
  if ((src_dtype != MOE_BF16 && src_dtype != MOE_F32) || d % 128 != 0 || f % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(WguT_q) || !aligned16(Wd_q)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack_backward_mx(W_gate, W_up, W_down, src_dtype, E_loc, d, f, WguT_q, WguT_scale, Wd_q,
                                             Wd_scale, stream));
}

moe_status moe_pack_weights_backward_fp8(const void* W_gate, const void* W_up, const void* W_down,
                                         moe_dtype src_dtype, int E_loc, int d, int f, const int32_t* w_exp,
                                         uint8_t* WguT_q, uint8_t* WguT_scale, uint8_t* Wd_q, uint8_t* Wd_scale,
                                         moe_stream_t stream) {
  if (!w_exp) return MOE_ERR_INVALID_ARG;
  if (!W_gate || !W_up || !W_down || !WguT_q || !WguT_scale || !Wd_q || !Wd_scale || E_loc < 1 || E_loc > 1024 ||
      d <= 0 || f <= 0)
    return MOE_ERR_INVALID_ARG;
  if ((src_dtype != MOE_BF16 && src_dtype != MOE_F32) || d % 128 != 0 || f % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(WguT_q) || !aligned16(Wd_q)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack_backward_mx(W_gate, W_up, W_down, src_dtype, E_loc, d, f, WguT_q, WguT_scale, Wd_q,
                                             Wd_scale, stream, w_exp));
}

size_t moe_layer_backward_fp8_workspace_size(int T, int d, int f, int k, int E_loc) {
  return moe_layer_backward_mx_workspace_size(T, d, f, k, E_loc);
}

size_t moe_layer_backward_mx_workspace_size(int T, int d, int f, int k, int E_loc) {
  if (T < 0 || d <= 0 || f <= 0 || k < 1 || E_loc < 1) return 0;
  return backward_layout(nullptr, T, d, f, k, E_loc, true).total;
}

}  // extern "C"

// The 8-bit layer backward: MXFP8 (per_tensor = false: operands quantised in 32-blocks along
// each GEMM's contraction axis) or per-tensor FP8 (every operand one tensor with one
// power-of-two scale, axis-independent, on the same block-scaled kernels with uniform
// scales; the weight-gradient operands quantised and dequantised in place).
static moe_status layer_backward_8bit(bool per_tensor, const void* x, const void* dy, const int32_t* topk_ids,
                                      const float* topk_probs, int T, int d, int f, int E, int k, int e0, int E_loc,
                                      const void* Wgu_packed, const uint8_t* Wgu_scale, const uint8_t* Wd_q,
                                      const uint8_t* Wd_scale, const uint8_t* WguT_q, const uint8_t* WguT_scale,
                                      void* dx, float* dlogits, float* dW_gate, float* dW_up, float* dW_down,
                                      void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 32 || e0 < 0 || E_loc < 1 || e0 + E_loc > E)
    return MOE_ERR_INVALID_ARG;
  if (n_cap_of(T, k, E_loc) > kMaxRows) return MOE_ERR_INVALID_ARG;  // int32 rows and offsets
  moe_status s = check_mlp_shape(d, f, E_loc, MOE_MXFP8);
  if (s != MOE_OK) return s;
  if (!Wgu_packed || !Wgu_scale || !Wd_q || !Wd_scale || !WguT_q || !WguT_scale || !dW_gate || !dW_up || !dW_down)
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !dy || !topk_ids || !topk_probs || !dx || !dlogits)) return MOE_ERR_INVALID_ARG;
  if ((T > 0 && (!aligned16(x) || !aligned16(dy) || !aligned16(dx))) || !aligned16(Wgu_packed) || !aligned16(Wd_q) ||
      !aligned16(WguT_q) || !aligned16(Wgu_scale) || !aligned16(Wd_scale) || !aligned16(WguT_scale) ||
      !aligned16(dW_gate) || !aligned16(dW_up) || !aligned16(dW_down))
    return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) ||
      workspace_bytes < moe_layer_backward_mx_workspace_size(T, d, f, k, E_loc))
    return MOE_ERR_WORKSPACE;
  BackwardWs w = backward_layout(static_cast<uint8_t*>(workspace), T, d, f, k, E_loc, true);
  const int64_t n_cap = n_cap_of(T, k, E_loc);
  cudaError_t e = cudaSuccess;
  if (T > 0)
    e = launch_permute(x, MOE_BF16, MOE_BF16, T, d, topk_ids, topk_probs, k, e0, E_loc, nullptr, nullptr, w.counts,
                       w.offsets, w.row_src_token, w.row_prob, w.pair_to_row, w.perm_ws, stream,
                       fuses_combine(MOE_MXFP8, k, E_loc, E) ? w.tok_nloc : nullptr);
  else
    e = cudaMemsetAsync(w.offsets, 0, static_cast<size_t>(E_loc + 1) * 4, stream);
  const int32_t* mtb = permute_mtile_base(w.perm_ws, T, E_loc);
  uint32_t* ax = per_tensor ? w.amax : nullptr;  // x, dy, h, [dg du]
  const int32_t* n_rows = w.offsets + E_loc;     // N on the device
  if (e == cudaSuccess && n_cap > 0 && per_tensor) {
    e = launch_amax(x, MOE_BF16, static_cast<int64_t>(T) * d, 1, ax, stream);
    if (e == cudaSuccess) e = launch_amax(dy, MOE_BF16, static_cast<int64_t>(T) * d, 1, ax + 1, stream);
  }
  if (e == cudaSuccess && n_cap > 0) {
    // x and dy rows in routed order: 8-bit along d (the row-wise GEMMs' A operands) and bf16
    // (the weight gradients' operands; MXFP8: quantised column-wise in the same pass,
    // per-tensor FP8: quantised below)
    if (per_tensor) {
      e = launch_gather_rows_mx(x, d, w.offsets, E_loc, mtb, w.row_src_token, w.x_q, w.x_sf, stream, ax);
      if (e == cudaSuccess)
        e = launch_gather_rows_mx(dy, d, w.offsets, E_loc, mtb, w.row_src_token, w.dy_q, w.dy_sf, stream, ax + 1);
      if (e == cudaSuccess)
        e = launch_gather_rows(dy, static_cast<int64_t>(d) * 2, w.offsets, E_loc, w.row_src_token, w.dy_rows,
                               stream);
      if (e == cudaSuccess)
        e = launch_gather_rows(x, static_cast<int64_t>(d) * 2, w.offsets, E_loc, w.row_src_token, w.x_rows, stream);
    } else {
      e = launch_rows_mx_both(x, d, w.offsets, E_loc, mtb, w.row_src_token, w.x_q, w.x_sf, w.x_rows, stream);
      if (e == cudaSuccess)
        e = launch_rows_mx_both(dy, d, w.offsets, E_loc, mtb, w.row_src_token, w.dy_q, w.dy_sf, w.dy_rows, stream);
    }
    // g, u of the MXFP8 forward (x and the gate/up weights along d), kept in bf16
    if (e == cudaSuccess)
      e = launch_tc_gemm_store_mx(w.x_q, w.x_sf, n_cap, w.offsets, E_loc, d, 2 * f, Wgu_packed, Wgu_scale, w.gu,
                                  w.err, kTimeoutNs, stream);
    // dh = dy W_down^T (both along d) with the ScaledSwiGLU backward: dg/du, h, partial dp
    if (e == cudaSuccess)
      e = launch_tc_dswiglu_mx(w.dy_q, w.dy_sf, w.offsets, w.row_prob, n_cap, E_loc, d, f, Wd_q, Wd_scale, w.gu, w.dgu,
                               w.h, w.dp_part, w.err, kTimeoutNs, stream);
    // dx rows = [dg du] [W_gate W_up]^T, both along f (per-tensor: [dg du] as one tensor)
    if (e == cudaSuccess && per_tensor) e = launch_amax_rows(w.dgu, 2 * f, n_rows, n_cap, ax + 3, stream);
    if (e == cudaSuccess)
      e = launch_gather_rows_mx(w.dgu, 2 * f, w.offsets, E_loc, mtb, nullptr, w.dgu_q, w.dgu_sf, stream,
                                per_tensor ? ax + 3 : nullptr);
  }
  if (e == cudaSuccess)
    e = backward_dx(true, w.dgu_q, w.dgu_sf, w, n_cap, T, E, k, E_loc, d, f, WguT_q, WguT_scale, dx, stream);
  if (e == cudaSuccess)
    e = launch_dlogits(topk_ids, topk_probs, w.pair_to_row, w.dp_part, f / 32, T, E, k, dlogits, stream);
  // weight gradients: operands quantised (MXFP8: column-wise, 32-row blocks of each
  // expert's segment; per-tensor FP8: with the tensor's one exponent), the dequantised
  // values in place, then the tensor-core weight-gradient GEMMs
  if (per_tensor) {
    if (e == cudaSuccess && n_cap > 0) e = launch_amax_rows(w.h, f, n_rows, n_cap, ax + 2, stream);
    if (e == cudaSuccess && n_cap > 0) e = launch_qdq_fp8_rows(w.x_rows, d, n_rows, n_cap, ax, stream);
    if (e == cudaSuccess && n_cap > 0) e = launch_qdq_fp8_rows(w.dy_rows, d, n_rows, n_cap, ax + 1, stream);
    if (e == cudaSuccess && n_cap > 0) e = launch_qdq_fp8_rows(w.h, f, n_rows, n_cap, ax + 2, stream);
    if (e == cudaSuccess && n_cap > 0) e = launch_qdq_fp8_rows(w.dgu, 2 * f, n_rows, n_cap, ax + 3, stream);
  } else {  // (x and dy rows: quantised column-wise while gathered)
    if (e == cudaSuccess && n_cap > 0) e = launch_colquant_mx(w.h, f, w.offsets, E_loc, stream);
    if (e == cudaSuccess && n_cap > 0) e = launch_colquant_mx(w.dgu, 2 * f, w.offsets, E_loc, stream);
  }
  if (e == cudaSuccess)
    e = launch_wgrad_down_tc(w.h, w.dy_rows, w.offsets, std::max<int64_t>(n_cap, 1), E_loc, d, f, dW_down, w.err,
                             kTimeoutNs, stream);
  if (e == cudaSuccess)
    e = launch_wgrad_gate_up_tc(w.x_rows, w.dgu, w.offsets, std::max<int64_t>(n_cap, 1), E_loc, d, f, dW_gate, dW_up,
                                w.err, kTimeoutNs, stream);
  return cuda_status(e);
}

extern "C" {

moe_status moe_layer_backward_mx(const void* x, const void* dy, const int32_t* topk_ids, const float* topk_probs, int T,
                                 int d, int f, int E, int k, int e0, int E_loc, const void* Wgu_packed,
                                 const uint8_t* Wgu_scale, const uint8_t* Wd_q, const uint8_t* Wd_scale,
                                 const uint8_t* WguT_q, const uint8_t* WguT_scale, void* dx, float* dlogits,
                                 float* dW_gate, float* dW_up, float* dW_down, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream) {
  return layer_backward_8bit(false, x, dy, topk_ids, topk_probs, T, d, f, E, k, e0, E_loc, Wgu_packed, Wgu_scale, Wd_q,
                             Wd_scale, WguT_q, WguT_scale, dx, dlogits, dW_gate, dW_up, dW_down, workspace,
                             workspace_bytes, stream);
}

moe_status moe_layer_backward_fp8(const void* x, const void* dy, const int32_t* topk_ids, const float* topk_probs,
                                  int T, int d, int f, int E, int k, int e0, int E_loc, const void* Wgu_packed,
                                  const uint8_t* Wgu_scale, const uint8_t* Wd_q, const uint8_t* Wd_scale,
                                  const uint8_t* WguT_q, const uint8_t* WguT_scale, void* dx, float* dlogits,
                                  float* dW_gate, float* dW_up, float* dW_down, void* workspace,
                                  size_t workspace_bytes, moe_stream_t stream) {
  return layer_backward_8bit(true, x, dy, topk_ids, topk_probs, T, d, f, E, k, e0, E_loc, Wgu_packed, Wgu_scale, Wd_q,
                             Wd_scale, WguT_q, WguT_scale, dx, dlogits, dW_gate, dW_up, dW_down, workspace,
                             workspace_bytes, stream);
}

moe_status moe_selftest_wait_timeout(uint64_t timeout_ns, void* workspace, size_t workspace_bytes,
                                     moe_stream_t stream) {
  if (timeout_ns < 1000000ull || timeout_ns > 2000000000ull) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned256(workspace) || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_wait_timeout(static_cast<int32_t*>(workspace), timeout_ns, stream));
}

moe_status moe_workspace_init(void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (!workspace || !aligned256(workspace) || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
  return cudaMemsetAsync(workspace, 0, sizeof(WsHeader), stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_get_device_error(void* workspace, moe_stream_t stream, int32_t* device_error) {
  if (!workspace || !device_error) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(workspace, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
  *device_error = v;
  return MOE_OK;
}

}  // extern "C"
