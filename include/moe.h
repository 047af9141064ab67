/*
 * moe.h -- C ABI of the B300 (sm_103a) MoE expert-layer library (libmoe.so).
 *
 * The library runs the forward pass of a Mixture-of-Experts expert layer on the experts
 * one GPU holds: top-k routing over router logits, a stable permute of token rows into
 * expert-contiguous order, a grouped GEMM1 (gate and up projections) with the scaled
 * SwiGLU fused into its epilogue, a grouped GEMM2 (down projection), and the combine
 * back to token order.
 *
 * Sources for the operations (page titles of the source material):
 *   [WEP]  "Wide-EP ... MoE ... NVIDIA" explainer, section "MoE basics": a router picks,
 *          per token, the experts it uses (DeepSeek-R1: 256 experts, 8 chosen); only those
 *          experts compute and their results are summed.  Section "Wide-EP": under EP8
 *          one GPU holds 32 experts per layer, under EP64 it holds 4.  Section
 *          "Prerequisite: fast GPU-to-GPU links": dispatch sends each token to its
 *          experts, combine brings the results back (on one GPU: permute / unpermute).
 *   [BIO]  "Efficient MoE training for biological foundation models" (BioNeMo), section
 *          "GroupedLinear Optimizes Expert Computation": per-expert matrices submitted as
 *          one grouped operation; GroupedLinear -> ScaledSwiGLU -> GroupedLinear fused
 *          with no intermediate materialised; ScaledSwiGLU applies the routing
 *          probabilities ("scales") inside the activation.  Section "MXFP8 Precision
 *          Reduces Memory Footprint": 8-bit values with one scale per block of 32
 *          consecutive values, run on Blackwell tensor-core instructions, with
 *          quantisation, SwiGLU and routing-weight scaling fused in one kernel.
 *
 * Common conventions
 *   - Every pointer argument named *device* below is a CUDA device pointer owned by the
 *     caller; the library never allocates, never frees and keeps no state between calls
 *     (scratch lives in the caller's workspace).  Calls are re-entrant.
 *   - Every call is asynchronous on the given stream and never synchronises the host,
 *     except moe_get_device_error().  Arguments are validated on the host before any
 *     launch; the first failed check returns an error and launches nothing.  A failed
 *     launch returns MOE_ERR_CUDA.
 *   - Matrices are dense, row-major and contiguous.  "bf16" means IEEE bfloat16 bits.
 *   - Device-detected errors (a bounded wait in a kernel that gave up) are written to
 *     the first 4 bytes of the workspace (the "error word").  The word is sticky: kernels
 *     only move it from 0 to an error code, moe_get_device_error() reads and clears it,
 *     and calls never reset it (so a call adds no memset to the stream).  Initialise a
 *     new workspace once with moe_workspace_init().
 *   - Kernels are launched with programmatic dependent launch: each one lets the next
 *     kernel on the stream start its set-up early and waits for the previous kernel's
 *     results before touching them, so back-to-back calls (and CUDA graphs of them)
 *     overlap kernel boundaries.
 *   - Only compute capability 10.3 (B300, sm_103a) is supported; there is no CPU path.
 */
#ifndef MOE_B300_MOE_H_
#define MOE_B300_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef int32_t moe_status;
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1 /* null pointer, out-of-range size, k > E, ...            */
#define MOE_ERR_UNSUPPORTED 2 /* dtype / shape / device the kernels do not handle      */
#define MOE_ERR_WORKSPACE 3   /* workspace pointer NULL, misaligned or too small        */
#define MOE_ERR_CUDA 4        /* a CUDA runtime call or a kernel launch failed          */
#define MOE_ERR_TIMEOUT 5     /* a bounded device-side wait gave up (device error word) */

typedef int32_t moe_dtype;
#define MOE_F32 0   /* fp32 inputs and outputs; expert GEMMs in fp32 FMA                  */
#define MOE_BF16 1  /* bf16 inputs/weights/outputs; tcgen05 bf16 MMA, fp32 accumulate   */
#define MOE_MXFP8 2 /* E4M3 values + E8M0 scale per 32 along K; tcgen05 block-scaled MMA */
#define MOE_FP8 3   /* per-tensor FP8: E4M3 values, one power-of-two scale per tensor (x, each */
                    /* expert weight matrix, h); stored in the MXFP8 layouts with every block  */
                    /* scale equal to the tensor's, run by the same block-scaled MMAs          */

/* Grouped-GEMM kernel shapes.  Passed as rows_hint (negative values), they force that
 * kernel; moe_layer_gemm_kernel reports the one moe_layer_forward picks.
 *   MOE_KERNEL_CTA   token-major 128-row tiles on one CTA
 *   MOE_KERNEL_PAIR  token-major 256-row tiles on a CTA pair (cta_group::2); fp32: CTA
 *   MOE_KERNEL_SWAP  swapped operands on a CTA pair: 256 packed weight rows on the MMA's M
 *                    side, up to 384 of an expert's tokens (padded to 16) on N; fp32 and
 *                    GEMM1 calls that keep g/u: CTA */
#define MOE_KERNEL_CTA (-1)
#define MOE_KERNEL_PAIR (-2)
#define MOE_KERNEL_SWAP (-3)

/* MXFP8 quantisation rule (both for x, the weights and the intermediate h): blocks of 32
 * consecutive values along the contraction dimension K; amax = max |v| over the block;
 * shared exponent X = floor(log2(amax)) - 8, clamped to [-127, 127] (X = 0 for an
 * all-zero block); scale byte = X + 127 (E8M0); element = E4M3 (OCP "E4M3FN": bias 7,
 * max 448, no infinities) of v * 2^-X, round to nearest even, saturating to +-448. */

/* Layout of MXFP8 scale factors ("SF tile layout").  A matrix with rows grouped in tiles
 * of 128 rows and K a multiple of 128 stores its scales in 512-byte atoms, one per
 * (row tile, 128-wide K group): inside an atom the scale of row i (0..127 within the
 * tile) and K block kk (0..3 within the group) sits at byte (i % 32) * 16 + (i / 32) * 4
 * + kk.  Rows of a tile past the end of its segment hold unspecified bytes.
 *   - activations (perm_x, h): row tiles are the per-expert m-tiles: expert e's segment
 *     [offsets[e], offsets[e+1]) is cut into ceil(count_e / 128) tiles, numbered
 *     globally in expert order (tile base of expert e = sum over e' < e of
 *     ceil(count_e' / 128)); atom (tile, g) is at byte (tile * (K / 128) + g) * 512.
 *     Capacity: moe_mx_act_scale_bytes().
 *   - packed weights: row tiles are 128 consecutive packed output rows of one expert;
 *     atom (e, g, n_tile) is at byte ((e * (K / 128) + g) * (rows / 128) + n_tile) * 512. */

/* Packed weight layout (output of moe_pack_weights, input of the grouped GEMMs).
 *   Wgu_packed [E_loc, 2f, d]  K-major (row = one output column of GEMM1, contiguous
 *              over d).  Gate and up columns are interleaved in blocks of G =
 *              moe_gu_block(f) columns: packed rows [2G*b, 2G*b + G) are gate columns
 *              [G*b, G*b + G) and packed rows [2G*b + G, 2G*b + 2G) are the up columns
 *              of the same range.
 *   Wd_packed  [E_loc, d, f]   K-major (row = one output column of GEMM2, contiguous over f).
 *   Element type: fp32 (MOE_F32), bf16 (MOE_BF16) or E4M3 bytes (MOE_MXFP8, with the
 *   scales in Wgu_scale / Wd_scale in the SF tile layout, see above). */
int moe_gu_block(int f);

/* Route (step 1) [WEP "MoE basics"].
 * For each token t, the k experts with the largest logits logits[t, :], in descending
 * order; equal logits go to the lower expert id (+0.0 and -0.0 are equal); then
 * topk_probs[t, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k chosen logits.
 *   logits     device fp32 [T, E]    (NaN logits: unspecified result; +-inf order normally)
 *   topk_ids   device int32 [T, k]   out
 *   topk_probs device fp32  [T, k]   out
 * Requires 1 <= k <= E <= 1024 and k <= 32, T >= 0.  T == 0 launches nothing. */
moe_status moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_probs,
                          moe_stream_t stream);

/* Permute (step 2) [WEP "Prerequisite ...": dispatch, here as a local permute].
 * Local experts are the ids [e0, e0 + E_loc); pairs (t, j) whose expert is not local are
 * skipped.  counts[e] = number of pairs routed to local expert e0+e; offsets = exclusive
 * prefix sum of counts (offsets[E_loc] = N, the number of local pairs).  Row offsets[e]+r
 * of the permuted buffers holds the r-th token, in ascending token order, that chose
 * expert e0+e: row_src_token[row] = t, row_prob[row] = topk_probs[t, j],
 * pair_to_row[t, j] = row (or -1 if not local), perm_x[row, :] = x[t, :].  The result is
 * deterministic (no atomics decide a position).
 *   x            device [T, d]  x_dtype MOE_F32 or MOE_BF16
 *   perm_dtype   element type of perm_x: MOE_F32 (x fp32), MOE_BF16 (x bf16), MOE_MXFP8
 *                (x bf16 or fp32; rows quantised while copied, scales to perm_x_scale) or
 *                MOE_FP8 (the same layouts; x quantised as one tensor: an amax pass over
 *                all of x [T, d] first, then every scale byte = its exponent + 127)
 *   perm_x       device [N_cap, d], N_cap = T * min(k, E_loc); rows >= N untouched.
 *                NULL: maps only -- counts, offsets, row_src_token, row_prob and
 *                pair_to_row are written, no rows are copied (the input of
 *                moe_expert_gemm1_swiglu_gather); perm_x_scale is then ignored
 *   perm_x_scale device, MOE_MXFP8 / MOE_FP8 with perm_x only (else NULL): SF tile layout, K = d,
 *                moe_mx_act_scale_bytes(N_cap, d, E_loc) bytes
 *   counts [E_loc], offsets [E_loc+1], row_src_token [N_cap], row_prob [N_cap] (fp32),
 *   pair_to_row [T, k]: device int32 outputs
 *   workspace    device, >= moe_permute_workspace_size(T, k, E_loc) bytes, 256-aligned
 * Requires 0 <= e0, 1 <= E_loc <= 1024, e0 + E_loc <= 65536, 1 <= k <= 32; d % 8 == 0 (bf16),
 * d % 4 == 0 (fp32), d % 128 == 0 (MXFP8); N_cap = T * min(k, E_loc) <= 2^31 - 1 (int32
 * row indices), else MOE_ERR_INVALID_ARG. */
moe_status moe_permute(const void* x, moe_dtype x_dtype, moe_dtype perm_dtype, int T, int d,
                       const int32_t* topk_ids, const float* topk_probs, int k, int e0, int E_loc,
                       void* perm_x, uint8_t* perm_x_scale, int32_t* counts, int32_t* offsets,
                       int32_t* row_src_token, float* row_prob, int32_t* pair_to_row, void* workspace,
                       size_t workspace_bytes, moe_stream_t stream);
size_t moe_permute_workspace_size(int T, int k, int E_loc);

/* moe_permute without a workspace argument.  (The source pages have no counterpart; this
 * entry point exists for callers of the library, not for the layer's definition.)
 * For callers that cannot call cudaMalloc at the time they permute -- e.g. a serving
 * engine that has given all free device memory to its KV-cache pool and plans every
 * buffer up front, or a host that is recording a CUDA graph and must not allocate.  It
 * computes exactly what moe_permute computes, with the same arguments minus the
 * workspace; the caller still passes every input and output buffer.  The scratch (error
 * word, per-tile expert counts, m-tile bases) lives in a 1 MiB file-scope device array
 * that every device using this library keeps until the process exits; nothing is
 * allocated or freed.
 *   Limit: moe_permute_workspace_size(T, k, E_loc) <= 1 MiB, i.e. ceil(T / 256) * E_loc
 *   <= about 260,000 (T <= 65,024 tokens at E_loc = 1024, T <= 260,864 at E_loc <= 256);
 *   larger inputs return MOE_ERR_WORKSPACE and launch nothing.  Arguments are checked as
 *   in moe_permute first (MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED before the size).
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call before any
 *   stream capture.  Every call shares the one array: calls whose kernels may overlap on
 *   the GPU (different streams, or different host threads on one device) race on it and
 *   must be serialised by the caller.  Everything the kernels need zeroed is cleared by
 *   the call itself. */
moe_status moe_permute_noalloc(const void* x, moe_dtype x_dtype, moe_dtype perm_dtype, int T, int d,
                               const int32_t* topk_ids, const float* topk_probs, int k, int e0, int E_loc,
                               void* perm_x, uint8_t* perm_x_scale, int32_t* counts, int32_t* offsets,
                               int32_t* row_src_token, float* row_prob, int32_t* pair_to_row, moe_stream_t stream);

/* Bytes of an activation scale buffer in the SF tile layout for N_cap rows, K columns. */
size_t moe_mx_act_scale_bytes(int64_t N_cap, int K, int E_loc);

/* Pack weights (one-off, untimed) [BIO "GroupedLinear ..."].
 * From the user layout W_gate, W_up [E_loc, d, f] and W_down [E_loc, f, d] (src_dtype
 * MOE_F32 or MOE_BF16) to the packed layout above in dst_dtype: MOE_F32 (src fp32),
 * MOE_BF16 (src bf16) or MOE_MXFP8 (src bf16 or fp32; quantised per output column in
 * blocks of 32 along K, scales to Wgu_scale / Wd_scale, sizes moe_mx_weight_scale_bytes).
 * All pointers device.  MXFP8 requires d % 128 == 0 and f % 128 == 0.  Per-tensor FP8
 * (MOE_FP8) is packed by moe_pack_weights_fp8 (MOE_ERR_UNSUPPORTED here). */
moe_status moe_pack_weights(const void* W_gate, const void* W_up, const void* W_down, moe_dtype src_dtype,
                            moe_dtype dst_dtype, int E_loc, int d, int f, void* Wgu_packed, void* Wd_packed,
                            uint8_t* Wgu_scale, uint8_t* Wd_scale, moe_stream_t stream);
size_t moe_mx_weight_scale_bytes(int E_loc, int rows, int K);
/* Per-tensor FP8 packing [BIO "MXFP8 Precision Reduces Memory Footprint": the layer runs
 * in FP8 as well as MXFP8].  Each expert's W_gate, W_up and W_down is one E4M3 tensor
 * with one power-of-two scale 2^X, X the smallest integer with amax <= 448 * 2^X (amax:
 * the matrix's largest magnitude; X clamped to [-127, 127], 0 for an all-zero matrix), so
 * the codes RNE(v / 2^X) never saturate.  Output: the MXFP8 packed layouts (codes as for
 * moe_pack_weights, every scale byte of a matrix X + 127), and w_exp [3][E_loc] int32 =
 * X of W_gate, W_up, W_down per expert.  src_dtype MOE_BF16 or MOE_FP32; d % 128 == 0,
 * f % 128 == 0; all pointers device, 16-byte aligned matrices.  Four kernel passes: the
 * three amax reductions (into w_exp), the quantisation, the exponents (in place). */
moe_status moe_pack_weights_fp8(const void* W_gate, const void* W_up, const void* W_down, moe_dtype src_dtype,
                                int E_loc, int d, int f, void* Wgu_packed, void* Wd_packed, uint8_t* Wgu_scale,
                                uint8_t* Wd_scale, int32_t* w_exp, moe_stream_t stream);

/* Grouped expert MLP (steps 3-4) [BIO "GroupedLinear ...", "MXFP8 Precision ..."].
 * For each local expert e and each row i of its segment [offsets[e], offsets[e+1]):
 *   g = perm_x[i] W_gate_e,  u = perm_x[i] W_up_e          (grouped GEMM1, fp32 accumulate)
 *   h = row_prob[i] * silu(g) * u,  silu(a) = a / (1 + e^-a)  (fused GEMM1 epilogue; h is
 *       stored once, as bf16 (MOE_BF16), fp32 (MOE_F32) or MXFP8 codes + scales
 *       (MOE_MXFP8, quantised in blocks of 32 along f); the 2f-wide pre-activation is never
 *       stored)
 *   Y2[i] = h W_down_e                                      (grouped GEMM2, fp32 accumulate)
 * N = offsets[E_loc] is read on the device; rows [N, N_cap) of Y2 are not written.
 *   perm_x, perm_x_scale   as produced by moe_permute (perm_x_scale NULL unless MXFP8)
 *   offsets [E_loc+1], row_prob [N_cap]   device
 *   Wgu_packed, Wgu_scale, Wd_packed, Wd_scale   packed weights (scales NULL unless MXFP8)
 *   Y2      device [N_cap, d]: fp32 for MOE_F32, bf16 otherwise
 *   workspace device >= moe_grouped_mlp_workspace_size(...) bytes, 256-byte aligned
 *   rows_hint  expected rows per local expert (e.g. moe_rows_hint(T, k, E)); it only picks
 *              the kernel shape, never the result's meaning: bf16 GEMM1 runs on the
 *              swapped-operand kernel (MOE_KERNEL_SWAP, 1.2 x the expected rows per tile)
 *              from 256 to 320 expected rows when d >= 4096 and E_loc <= 256, on
 *              token-major CTA pairs from 2048 expected rows up and from 321 to 1023 when
 *              d >= 4096; bf16 GEMM2 on token-major pairs from 128; MXFP8 GEMMs on pairs
 *              only from 65536 (the block-scaled pair kernel measured slower than the 1-CTA
 *              one on every shape tried); everything else on the 1-CTA kernel.  0 uses
 *              N_cap / E_loc; MOE_KERNEL_* forces a kernel.  MOE_FP8 always runs on the
 *              1-CTA kernel: GEMM1 writes bf16 h and its amax into the workspace, h is
 *              quantised as one tensor, GEMM2 reads it like MXFP8.
 * Requires d % 8 == 0 and f % 32 == 0 (bf16); d % 128 == 0 and f % 128 == 0 (MXFP8, FP8). */
moe_status moe_grouped_mlp(const void* perm_x, const uint8_t* perm_x_scale, const int32_t* offsets,
                           const float* row_prob, int64_t N_cap, int E_loc, int d, int f, moe_dtype dtype,
                           const void* Wgu_packed, const uint8_t* Wgu_scale, const void* Wd_packed,
                           const uint8_t* Wd_scale, void* Y2, int rows_hint, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream);
/* Expected rows per local expert under uniform routing, T * k / E (the hint
 * moe_layer_forward uses). */
int moe_rows_hint(int T, int k, int E);
/* The GEMM1 kernel moe_layer_forward picks for this problem (host only, no launch): 1 if
 * GEMM1 runs on token-major CTA pairs (256-row tiles), else 0 (the 1-CTA or the
 * swapped-operand kernel; moe_layer_gemm_kernel tells which).  Returns -1 for invalid
 * sizes. */
int moe_layer_gemm1_pairs(int T, int d, int k, int E, int E_loc, moe_dtype dtype);
/* The kernel moe_layer_forward runs for GEMM `gemm` (1 or 2) of this problem, as a
 * MOE_KERNEL_* value (host only, no launch); 0 for invalid arguments. */
int moe_layer_gemm_kernel(int T, int d, int f, int k, int E, int E_loc, moe_dtype dtype, int gemm);

/* Whether moe_layer_forward folds the combine into GEMM2 (moe_expert_gemm2_combine's
 * path) for this routing shape: 1 when tokens average under one local slot (k * E_loc <
 * E, bf16 or MXFP8), else 0 (GEMM2, then moe_unpermute_combine's kernel); -1 for invalid
 * sizes.  The result is the same either way; only the kernels differ. */
int moe_layer_fused_combine(int k, int E, int E_loc, moe_dtype dtype);
size_t moe_grouped_mlp_workspace_size(int64_t N_cap, int E_loc, int d, int f, moe_dtype dtype);

/* The two halves of moe_grouped_mlp, for callers that keep h themselves (same
 * preconditions; N = offsets[E_loc] on the device).
 *   moe_expert_gemm1_swiglu: perm_x (+ scales) -> h [N_cap, f] (fp32 / bf16 / E4M3 bytes;
 *       MOE_FP8: GEMM1 writes bf16 h and its amax into the workspace, then h is quantised
 *       as one tensor into h / h_scale; workspace >= moe_expert_gemm1_workspace_size())
 *       and, for MOE_MXFP8, h_scale in the SF tile layout with K = f
 *       (moe_mx_act_scale_bytes(N_cap, f, E_loc) bytes) [BIO "GroupedLinear ...":
 *       GroupedLinear + ScaledSwiGLU (+ quantisation) in one kernel].
 *   moe_expert_gemm2: h (+ h_scale) -> Y2 [N_cap, d] (fp32 for MOE_F32, else bf16)
 *       [BIO: the second GroupedLinear].
 *   rows_hint: as for moe_grouped_mlp.
 *   workspace: >= moe_expert_gemm_workspace_size() bytes, 256-byte aligned (error word). */
/* Workspace of moe_expert_gemm1_swiglu: the error word, plus for MOE_FP8 bf16 h [N_cap, f]
 * and its amax. */
size_t moe_expert_gemm1_workspace_size(int64_t N_cap, int f, moe_dtype dtype);
moe_status moe_expert_gemm1_swiglu(const void* perm_x, const uint8_t* perm_x_scale, const int32_t* offsets,
                                   const float* row_prob, int64_t N_cap, int E_loc, int d, int f, moe_dtype dtype,
                                   const void* Wgu_packed, const uint8_t* Wgu_scale, void* h, uint8_t* h_scale,
                                   int rows_hint, void* workspace, size_t workspace_bytes, moe_stream_t stream);
moe_status moe_expert_gemm2(const void* h, const uint8_t* h_scale, const int32_t* offsets, int64_t N_cap, int E_loc,
                            int d, int f, moe_dtype dtype, const void* Wd_packed, const uint8_t* Wd_scale, void* Y2,
                            int rows_hint, void* workspace, size_t workspace_bytes, moe_stream_t stream);
size_t moe_expert_gemm_workspace_size(void);

/* GEMM1 + scaled SwiGLU reading the token rows directly ("row gather") [BIO "GroupedLinear
 * ...": the grouped op consumes the routed tokens; here no permuted copy of x exists].
 * Computes exactly what moe_expert_gemm1_swiglu computes on moe_permute's perm_x, with
 * perm_x[row] = x[row_src_token[row]]: the kernel copies each 128-row x 128-byte operand
 * tile from the token rows into shared memory itself.
 *   x        MOE_BF16: device bf16 [T, d].  MOE_MXFP8: device E4M3 bytes [T, d] with
 *            x_scale device E8M0 [T, d / 32] row-major (from moe_quantize_mx_rows).
 *            (MOE_F32 and MOE_FP8 are not supported: MOE_ERR_UNSUPPORTED.)
 *   row_src_token [N_cap], offsets [E_loc+1], row_prob [N_cap]: device, from moe_permute
 *            (which may be called with perm_x == NULL)
 *   h, h_scale, Wgu_*, rows_hint, workspace: as for moe_expert_gemm1_swiglu (bf16: the
 *   CTA-pair kernel copies its 256-row tiles' rows the same way, each CTA its own 128).
 *   16-byte aligned x, h and packed weights; d % 8 == 0 (bf16), d % 128 == 0 and f % 128 ==
 *   0 (MXFP8). */
moe_status moe_expert_gemm1_swiglu_gather(const void* x, const uint8_t* x_scale, const int32_t* row_src_token,
                                          const int32_t* offsets, const float* row_prob, int64_t N_cap, int E_loc,
                                          int d, int f, moe_dtype dtype, const void* Wgu_packed,
                                          const uint8_t* Wgu_scale, void* h, uint8_t* h_scale, int rows_hint, void* workspace,
                                          size_t workspace_bytes, moe_stream_t stream);

/* MXFP8 quantisation of token rows [BIO "MXFP8 Precision ..."]: the quantisation rule
 * above, per 32 consecutive values of a row -- the same rule moe_permute applies while
 * copying.
 *   x  device [T, d], x_dtype MOE_BF16 or MOE_F32, 16-byte aligned
 *   pair_to_row  device int32 [T, k] from moe_permute, or NULL: when given, only rows of
 *      tokens with at least one local expert (some pair_to_row[t, j] >= 0) are written --
 *      the only rows the row-gather GEMM1 reads; requires 1 <= k <= 32
 *   xq device E4M3 [T, d] out (16-byte aligned); x_scale device E8M0 [T, d / 32] out.
 * Requires d % 32 == 0. */
moe_status moe_quantize_mx_rows(const void* x, moe_dtype x_dtype, int T, int d, const int32_t* pair_to_row, int k,
                                uint8_t* xq, uint8_t* x_scale, moe_stream_t stream);

/* Unpermute + combine (step 5) [WEP "MoE basics": results of the chosen experts are
 * summed; "Prerequisite ...": combine].
 * y[t] = sum over j = 0..k-1 with pair_to_row[t, j] >= 0 of Y2[pair_to_row[t, j]], summed
 * in slot order in fp32 and rounded once; tokens with no local expert get a zero row.
 * (The routing probability was already applied inside the SwiGLU.)
 *   Y2 device [N_cap, d] (fp32 if dtype == MOE_F32, else bf16); pair_to_row device [T, k];
 *   y  device [T, d] (fp32 if dtype == MOE_F32, else bf16), fully written.
 * Requires d % 8 == 0 (bf16) / d % 4 == 0 (fp32). */
moe_status moe_unpermute_combine(const void* Y2, const int32_t* pair_to_row, int T, int k, int d,
                                 moe_dtype dtype, void* y, moe_stream_t stream);

/* GEMM2 with the unpermute + combine folded into it (steps 4-5) [BIO "GroupedLinear ...":
 * the grouped down projection; WEP "MoE basics": the chosen experts' results are summed
 * per token].  y equals, bit for bit, moe_expert_gemm2 followed by moe_unpermute_combine
 * on the same inputs: each token's local rows (h W_down_e, rounded to bf16) are added in
 * slot order in fp32 from zero and rounded once; tokens with no local expert get a zero
 * row.  The GEMM2 kernel writes y itself for every token with at most one local slot (its
 * row unchanged, which is that sum; or zeros, from extra warps running alongside the
 * GEMM), and stores only the rows of tokens with several local slots to a scratch Y2,
 * which a combine pass over those tokens alone then sums.  moe_layer_forward runs this path for MOE_BF16 and MOE_MXFP8.
 *   h, h_scale, offsets, Wd_packed, Wd_scale   as for moe_expert_gemm2 (dtype MOE_BF16 or
 *                                              MOE_MXFP8; MOE_F32 is MOE_ERR_UNSUPPORTED)
 *   row_src_token [N_cap], pair_to_row [T, k]   device, from moe_permute
 *   y         device bf16 [T, d], fully written (16-byte aligned)
 *   rows_hint  as for moe_expert_gemm2; it also tells the expected local slots per token
 *             (rows_hint * E_loc / T: under one picks the pass built for few multi-slot
 *             tokens); <= 0 assumes min(k, E_loc).  It never changes the result.
 *   workspace device, >= moe_expert_gemm2_combine_workspace_size(N_cap, T, d) bytes,
 *             256-aligned (scratch Y2 and per-token slot counts, set by a small kernel)
 * Requires 1 <= k <= 32 and the shape rules of moe_expert_gemm2. */
moe_status moe_expert_gemm2_combine(const void* h, const uint8_t* h_scale, const int32_t* offsets,
                                    const int32_t* row_src_token, const int32_t* pair_to_row, int T, int k,
                                    int64_t N_cap, int E_loc, int d, int f, moe_dtype dtype, const void* Wd_packed,
                                    const uint8_t* Wd_scale, void* y, int rows_hint, void* workspace,
                                    size_t workspace_bytes, moe_stream_t stream);
size_t moe_expert_gemm2_combine_workspace_size(int64_t N_cap, int T, int d);

/* Whole layer (steps 1-5 in one call) on the local experts [e0, e0 + E_loc).
 *   x [T, d] (fp32 for MOE_F32, else bf16), logits [T, E] fp32, packed weights as above,
 *   y [T, d] (fp32 for MOE_F32, else bf16): device pointers.
 *   workspace device >= moe_layer_workspace_size(...) bytes, 256-byte aligned; it holds
 *   the routing table, the permutation maps, h and Y2, plus the permuted rows where a
 *   copy is made: bf16 layers feed GEMM1 by row gather, except when the CTA-pair GEMM1
 *   is chosen (moe_layer_gemm1_pairs), which reads a permuted copy; fp32 and MXFP8
 *   layers copy (MXFP8 quantises while copying).
 *   MOE_FP8 (per-tensor FP8, weights from moe_pack_weights_fp8): x is one E4M3 tensor (its
 *   amax over all T x d values gives X as for the weights), quantised while copying; GEMM1
 *   writes bf16 h and its amax, h is then quantised as one tensor (all local rows), and
 *   GEMM2 and the combine run as for MXFP8 (the block-scaled kernels with every scale of
 *   a tensor equal).
 * Requires T * min(k, E_loc) <= 2^31 - 1 (int32 row indices), else MOE_ERR_INVALID_ARG. */
moe_status moe_layer_forward(const void* x, const float* logits, int T, int d, int f, int E, int k, int e0,
                             int E_loc, moe_dtype dtype, const void* Wgu_packed, const uint8_t* Wgu_scale,
                             const void* Wd_packed, const uint8_t* Wd_scale, void* y, void* workspace,
                             size_t workspace_bytes, moe_stream_t stream);
size_t moe_layer_workspace_size(int T, int d, int f, int E, int k, int E_loc, moe_dtype dtype);

/* Zeroes the 256-byte header of a new workspace (the device error word), asynchronously on
 * `stream`.  Call once before a workspace's first use. */
moe_status moe_workspace_init(void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Synchronises `stream`, then reads and clears the device error word at the start of
 * `workspace`.  Writes MOE_OK or the error code a kernel stored (MOE_ERR_TIMEOUT) to
 * *device_error.  Returns MOE_ERR_CUDA if the synchronisation fails. */
moe_status moe_get_device_error(void* workspace, moe_stream_t stream, int32_t* device_error);

/* Layer backward (bf16) ["Efficient MoE training for biological foundation models",
 * "GroupedLinear Optimizes Expert Computation": the fused GroupedMLP has a matching
 * backward whose ScaledSwiGLU part also yields the gradient of the routing scales].
 * Gradients of L = sum_t dy_t . y_t for the layer of moe_layer_forward (same x, routing and
 * weights).  Per routed row (token t, local expert e, probability p), with s = sigmoid(g):
 *   g, u = x W_gate_e, x W_up_e (saved or recomputed);  h = p silu(g) u;  dh = W_down_e dy_t
 *   du = p dh silu(g);  dg = p dh u s (1 + g (1 - s));  dp = sum_n dh_n silu(g_n) u_n
 *   dx_t = sum over the token's local slots of W_gate_e dg + W_up_e du
 *   dW_down_e = sum_rows h^T dy_t;  dW_gate_e = sum_rows x_t^T dg;  dW_up_e = sum_rows x_t^T du
 *   dlogits[t, id_j] = p_j (dp_j - sum_i p_i dp_i) over the k selected logits (softmax over
 *   the top k), dp = 0 for slots whose expert is not local; other logits 0.  With experts
 *   split over GPUs, summing every GPU's dx and dlogits gives the full gradients.
 *   x, dy              device bf16 [T, d]
 *   topk_ids/probs     device [T, k] from moe_route_topk on the forward's logits
 *   Wgu_packed         the forward's packed gate/up weights (moe_pack_weights, bf16)
 *   W_down             device bf16 [E_loc, f, d], the user layout
 *   WguT_packed        device bf16 [E_loc, d, 2f] from moe_pack_weights_backward
 *   gu_saved           device bf16 [N_cap, 2f] from moe_layer_forward_train on the same
 *                      inputs (the gate/up pre-activations), or NULL to recompute them
 *   dx                 device bf16 [T, d] out (zero rows for tokens with no local expert)
 *   dlogits            device fp32 [T, E] out
 *   dW_gate, dW_up     device fp32 [E_loc, d, f] out;  dW_down device fp32 [E_loc, f, d] out
 *                      (zero for experts that received no token)
 *   workspace          device >= moe_layer_backward_workspace_size(T, d, f, k, E_loc) bytes,
 *                      256-byte aligned, error word initialised (moe_workspace_init)
 * Requires d % 8 == 0, f % 32 == 0; 16-byte aligned x, dy, dx, weights and gradients;
 * T * min(k, E_loc) <= 2^31 - 1.  bf16 only. */
moe_status moe_layer_backward(const void* x, const void* dy, const int32_t* topk_ids, const float* topk_probs, int T,
                              int d, int f, int E, int k, int e0, int E_loc, const void* Wgu_packed,
                              const void* W_down, const void* WguT_packed, const void* gu_saved, void* dx,
                              float* dlogits, float* dW_gate, float* dW_up, float* dW_down, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream);
size_t moe_layer_backward_workspace_size(int T, int d, int f, int k, int E_loc);

/* Training forward: moe_layer_forward (bf16) that also returns what the backward needs.
 *   topk_ids, topk_probs  device [T, k] out: the routing (as moe_route_topk)
 *   gu_saved              device bf16 [N_cap, 2f] out, N_cap = T * min(k, E_loc): row r holds
 *                         g = x W_gate and u = x W_up of permuted row r (moe_permute's order)
 *                         in the packed column order (columns 64b..64b+31 gate, the next 32
 *                         up, of h columns 32b..32b+31), rounded to bf16; rows >= N unused
 * The other arguments and the workspace are those of moe_layer_forward with dtype bf16;
 * y is bit-identical to moe_layer_forward's. */
moe_status moe_layer_forward_train(const void* x, const float* logits, int T, int d, int f, int E, int k, int e0,
                                   int E_loc, const void* Wgu_packed, const void* Wd_packed, void* y,
                                   int32_t* topk_ids, float* topk_probs, void* gu_saved, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream);

/* Backward weight pack (one-off): WguT [E_loc, d, 2f] bf16, row c = rows c of W_gate and W_up
 * ([E_loc, d, f], src_dtype MOE_BF16 or MOE_F32) interleaved in 32-column blocks (packed
 * column 64b + i = gate column 32b + i, 64b + 32 + i = up column 32b + i) -- the order
 * the backward stores dg/du in.  Requires f % 32 == 0, d % 8 == 0. */
moe_status moe_pack_weights_backward(const void* W_gate, const void* W_up, moe_dtype src_dtype, int E_loc, int d,
                                     int f, void* WguT_packed, moe_stream_t stream);

/* Layer backward, MXFP8 [BIO "GroupedLinear ...": the fused GroupedMLP's backward; "MXFP8
 * Precision Reduces Memory Footprint": 8-bit values with one E8M0 scale per 32 consecutive
 * values, Blackwell MXFP8 GEMMs].  The gradients of L = sum_t dy_t . y_t for the MXFP8 layer
 * of moe_layer_forward (x rows and W_gate, W_up quantised along d), every backward GEMM
 * reading its two operands quantised in 32-blocks along that GEMM's own contraction axis
 * (the rule of moe_pack_weights):
 *   g, u = x W_gate, x W_up            recomputed on the block-scaled tensor cores
 *   dh = dy W_down^T                   dy rows and W_down along d; block-scaled MMAs, the
 *                                      ScaledSwiGLU backward (exact, fp32) in the epilogue
 *   dx_row = dg W_gate^T + du W_up^T   dg, du rows and W_gate, W_up along f; block-scaled
 *   dW_down_e = h^T dy, dW_gate_e = x^T dg, dW_up_e = x^T du
 *                                      h, dy, x, dg, du quantised column-wise in 32-row
 *                                      blocks of each expert's segment (the last block
 *                                      padded with zeros); the dequantised values (code *
 *                                      2^X, exact in bf16) feed the bf16 tensor-core
 *                                      weight-gradient kernel, fp32 accumulate and output
 *   dlogits as moe_layer_backward.
 * g, u, dg, du and h are rounded to bf16 once before their quantisation.
 *   x, dy              device bf16 [T, d]
 *   topk_ids/probs     the forward's routing [T, k]
 *   Wgu_packed, Wgu_scale   moe_pack_weights(..., MOE_MXFP8): the forward's gate/up codes
 *   Wd_q, Wd_scale, WguT_q, WguT_scale   moe_pack_weights_backward_mx
 *   dx (bf16 [T, d]), dlogits (fp32 [T, E]), dW_gate, dW_up (fp32 [E_loc, d, f]),
 *   dW_down (fp32 [E_loc, f, d])   device outputs, fully written
 *   workspace          device >= moe_layer_backward_mx_workspace_size(T, d, f, k, E_loc)
 *                      bytes, 256-byte aligned
 * Requires d % 128 == 0 and f % 128 == 0; other rules as moe_layer_backward. */
moe_status moe_layer_backward_mx(const void* x, const void* dy, const int32_t* topk_ids, const float* topk_probs, int T,
                                 int d, int f, int E, int k, int e0, int E_loc, const void* Wgu_packed,
                                 const uint8_t* Wgu_scale, const uint8_t* Wd_q, const uint8_t* Wd_scale,
                                 const uint8_t* WguT_q, const uint8_t* WguT_scale, void* dx, float* dlogits,
                                 float* dW_gate, float* dW_up, float* dW_down, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream);
size_t moe_layer_backward_mx_workspace_size(int T, int d, int f, int k, int E_loc);

/* Backward weight operands in MXFP8 (one-off): Wd_q [E_loc, f, d] = W_down quantised along d
 * (scales Wd_scale in the weight SF tile layout, rows f, K = d: moe_mx_weight_scale_bytes(
 * E_loc, f, d) bytes) and WguT_q [E_loc, d, 2f] = W_gate, W_up in the packed column order of
 * moe_pack_weights_backward quantised along f (WguT_scale: rows d, K = 2f).  Sources in the
 * user layouts (bf16 or fp32).  Requires d % 128 == 0 and f % 128 == 0. */
moe_status moe_pack_weights_backward_mx(const void* W_gate, const void* W_up, const void* W_down, moe_dtype src_dtype,
                                        int E_loc, int d, int f, uint8_t* WguT_q, uint8_t* WguT_scale, uint8_t* Wd_q,
                                        uint8_t* Wd_scale, moe_stream_t stream);

/* Per-tensor FP8 layer backward ["Efficient MoE training ...", "MXFP8 Precision Reduces
 * Memory Footprint": the layer trains in FP8 as well as MXFP8].  Same arguments, outputs
 * and workspace as moe_layer_backward_mx, with the weights packed by moe_pack_weights_fp8
 * (forward) and moe_pack_weights_backward_fp8 (backward layouts).  Every GEMM operand is
 * one E4M3 tensor with one power-of-two scale (the rule of moe_pack_weights_fp8): x and dy
 * as wholes (an amax pass over each), each expert weight matrix, h and the gradient of the
 * gate/up pre-activation [dg du] over the local routed rows; axis-independent, so the
 * weight gradients read the same values as the row-wise GEMMs (quantised and dequantised
 * in place, exact in bf16).  moe_layer_backward_fp8_workspace_size equals the MXFP8 one. */
moe_status moe_layer_backward_fp8(const void* x, const void* dy, const int32_t* topk_ids, const float* topk_probs,
                                  int T, int d, int f, int E, int k, int e0, int E_loc, const void* Wgu_packed,
                                  const uint8_t* Wgu_scale, const uint8_t* Wd_q, const uint8_t* Wd_scale,
                                  const uint8_t* WguT_q, const uint8_t* WguT_scale, void* dx, float* dlogits,
                                  float* dW_gate, float* dW_up, float* dW_down, void* workspace,
                                  size_t workspace_bytes, moe_stream_t stream);
size_t moe_layer_backward_fp8_workspace_size(int T, int d, int f, int k, int E_loc);
/* The backward weight layouts of moe_pack_weights_backward_mx for per-tensor FP8: each
 * matrix quantised with its exponent from w_exp [3][E_loc] (moe_pack_weights_fp8's output:
 * W_gate, W_up, W_down per expert), every scale byte of a matrix that exponent + 127. */
moe_status moe_pack_weights_backward_fp8(const void* W_gate, const void* W_up, const void* W_down,
                                         moe_dtype src_dtype, int E_loc, int d, int f, const int32_t* w_exp,
                                         uint8_t* WguT_q, uint8_t* WguT_scale, uint8_t* Wd_q, uint8_t* Wd_scale,
                                         moe_stream_t stream);

/* Expert placement and replication plan (host function, no GPU) ["Wide-EP ... MoE ...
 * NVIDIA" explainer, "Load imbalance: EPLB": per-expert load decides placement, and the
 * most loaded experts get copies on several GPUs].  The page gives no algorithm; this is
 * the plain greedy reading:
 *   1. every expert gets one copy; while free slots remain, one more copy goes to the
 *      expert with the largest load per copy (ties: lower id), at most G copies each;
 *   2. copies (load / copies each) in descending load (ties: lower expert id, then
 *      copy index) go to the least loaded GPU with a free slot that holds no copy of
 *      that expert (ties: lower GPU id); an extra copy no GPU can take is dropped.
 *   load         host int64 [E]: tokens routed to each expert (e.g. summed counts from
 *                moe_permute over recent steps), >= 0
 *   E, G, S      experts, GPUs, slots per GPU; requires E <= G * S <= 2^24
 *   slot_expert  host int32 [G * S] out: expert held by slot s of GPU g at g * S + s,
 *                filled from s = 0 up, -1 for an empty slot
 *   replicas     host int32 [E] out: copies placed per expert (>= 1)
 *   gpu_load     host double [G] out: sum over the GPU's copies of load / replicas
 * Deterministic; MOE_ERR_INVALID_ARG on a bad size or negative load. */
moe_status moe_eplb_plan(const int64_t* load, int E, int G, int S, int32_t* slot_expert, int32_t* replicas,
                         double* gpu_load);

/* Self-test of the bounded device waits every pipelined kernel uses (failure detection):
 * launches one thread that waits on an mbarrier nothing arrives on, for timeout_ns
 * (1 ms .. 2 s); the wait gives up, MOE_ERR_TIMEOUT is stored in the (initialised) error
 * word at the start of `workspace` (>= 256 bytes, 256-byte aligned) and the kernel
 * returns, leaving the context usable.  Read the result with moe_get_device_error(). */
moe_status moe_selftest_wait_timeout(uint64_t timeout_ns, void* workspace, size_t workspace_bytes,
                                     moe_stream_t stream);

/* 1 if the current CUDA device is compute capability 10.3 (sm_103a), else 0. */
int moe_supported(void);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_MOE_H_ */
