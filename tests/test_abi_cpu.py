"""The C ABI without a GPU: libmoe.so builds for sm_103a, loads, exports every function
include/moe.h declares, and its host-side logic (sizes, validation) answers correctly.
No call here reaches a kernel: every validation case fails before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_103_b300 import build
    build.build()
    import mixture_experts_layer_103_b300 as m
    return m


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, missing


def test_binding_covers_the_header(lib):
    import mixture_experts_layer_103_b300 as m
    for n in declared_functions():
        assert n in m._SIGS, n


def test_status_strings(lib):
    L = lib.lib()
    assert L.moe_status_string(0) == b"MOE_OK"
    assert L.moe_status_string(5) == b"MOE_ERR_TIMEOUT"
    assert L.moe_status_string(99) == b"MOE_ERR_UNKNOWN"


def test_sizes(lib):
    L = lib.lib()
    assert L.moe_gu_block(2048) == 32 and L.moe_gu_block(48) == 0
    # weight scales: E_loc * (rows/128) * (K/128) atoms of 512 bytes
    assert L.moe_mx_weight_scale_bytes(32, 4096, 7168) == 32 * 32 * 56 * 512
    assert L.moe_mx_weight_scale_bytes(1, 100, 128) == 0
    # activation scales: (ceil(N_cap/128) + E_loc) tiles x (K/128) atoms
    assert L.moe_mx_act_scale_bytes(1000, 256, 8) == (8 + 8) * 2 * 512
    assert L.moe_permute_workspace_size(4096, 8, 64) > 256
    big = L.moe_layer_workspace_size(4096, 2048, 1024, 64, 8, 64, 1)
    # bf16 rows are gathered into GEMM1, so Y2 (bf16) + h dominate (N_cap = 32768) and no
    # permuted copy of x is held
    assert 32768 * 2048 * 2 + 32768 * 1024 * 2 <= big < 2 * 32768 * 2048 * 2 + 32768 * 1024 * 2
    # fp32 copies the rows: perm_x + Y2 + h
    f32 = L.moe_layer_workspace_size(4096, 2048, 1024, 64, 8, 64, 0)
    assert f32 >= 32768 * 2048 * 4 * 2 + 32768 * 1024 * 4
    # tall segments (T * k / E >= 2048) pick the CTA-pair GEMMs, which gather the token
    # rows as well: Y2 + h, no permuted copy
    tall = L.moe_layer_workspace_size(2048, 256, 256, 8, 8, 8, 1)
    assert 16384 * 256 * 2 + 16384 * 256 * 2 <= tall < 2 * 16384 * 256 * 2 + 16384 * 256 * 2
    # MXFP8 copies while quantising: E4M3 perm_x + Y2 (bf16) + E4M3 h
    mx = L.moe_layer_workspace_size(4096, 2048, 1024, 64, 8, 64, 2)
    assert mx >= 32768 * 2048 + 32768 * 2048 * 2 + 32768 * 1024
    assert L.moe_expert_gemm_workspace_size() == 256


def _null():
    return ctypes.c_void_p(0)


def test_validation_before_any_launch(lib):
    L = lib.lib()
    P = ctypes.c_void_p(256)  # never dereferenced: every case below fails validation first
    s = _null()
    # route: k > E, k > 32, E > 1024, null pointers
    assert L.moe_route_topk(P, 4, 8, 9, P, P, s) == 1
    assert L.moe_route_topk(P, 4, 64, 33, P, P, s) == 1
    assert L.moe_route_topk(P, 4, 1025, 8, P, P, s) == 1
    assert L.moe_route_topk(_null(), 4, 8, 2, P, P, s) == 1
    # pack: f not a multiple of 32 / MXFP8 d not a multiple of 128 / bad dtype pairs
    assert L.moe_pack_weights(P, P, P, 1, 1, 2, 64, 48, P, P, None, None, s) == 2
    assert L.moe_pack_weights(P, P, P, 1, 2, 2, 96, 128, P, P, P, P, s) == 2
    assert L.moe_pack_weights(P, P, P, 0, 1, 2, 64, 64, P, P, None, None, s) == 2
    assert L.moe_pack_weights(P, P, P, 1, 2, 2, 128, 128, P, P, None, None, s) == 1
    # permute: workspace too small / misaligned
    assert L.moe_permute(P, 1, 1, 16, 64, P, P, 2, 0, 8, P, None, P, P, P, P, P, P, 0, s) == 3
    assert L.moe_permute(P, 1, 1, 16, 64, P, P, 2, 0, 8, P, None, P, P, P, P, P, ctypes.c_void_p(272), 1 << 20,
                         s) == 3
    assert L.moe_permute(P, 1, 1, 16, 60, P, P, 2, 0, 8, P, None, P, P, P, P, P, P, 1 << 20, s) == 2
    assert L.moe_permute(P, 1, 2, 16, 64, P, P, 2, 0, 8, P, None, P, P, P, P, P, P, 1 << 20, s) == 1
    # permute: local expert ids beyond 65535 (e0 + E_loc > 65536), E_loc > 1024
    assert L.moe_permute(P, 1, 1, 16, 64, P, P, 2, 65536 - 7, 8, P, None, P, P, P, P, P, P, 1 << 20, s) == 1
    assert L.moe_permute(P, 1, 1, 16, 64, P, P, 2, 65536 - 8, 8, P, None, P, P, P, P, P, _null(), 0, s) == 3
    assert L.moe_permute(P, 1, 1, 16, 64, P, P, 2, 0, 2048, P, None, P, P, P, P, P, P, 1 << 20, s) == 1
    assert L.moe_permute_workspace_size(16, 2, 2048) == 0
    # workspace-free permute: the arguments are checked before its scratch size, so an
    # out-of-range E_loc or e0 is an invalid argument, not a workspace overflow
    assert L.moe_permute_noalloc(P, 1, 1, 16, 64, P, P, 2, 0, 2048, P, None, P, P, P, P, P, s) == 1
    assert L.moe_permute_noalloc(P, 1, 1, 16, 64, P, P, 2, 65530, 8, P, None, P, P, P, P, P, s) == 1
    assert L.moe_permute_noalloc(P, 1, 1, 16, 64, P, P, 33, 0, 8, P, None, P, P, P, P, P, s) == 1
    assert L.moe_permute_noalloc(P, 1, 1, 1 << 20, 64, P, P, 8, 0, 1024, P, None, P, P, P, P, P, s) == 3
    # grouped MLP: E_loc out of range, unsupported dtype, workspace too small
    assert L.moe_grouped_mlp(P, None, P, P, 64, 0, 64, 64, 1, P, None, P, None, P, 0, P, 1 << 20, s) == 1
    assert L.moe_grouped_mlp(P, None, P, P, 64, 4, 64, 64, 7, P, None, P, None, P, 0, P, 1 << 20, s) == 2
    assert L.moe_grouped_mlp(P, None, P, P, 64, 4, 64, 64, 1, P, None, P, None, P, 0, P, 16, s) == 3
    # MXFP8 without scales
    assert L.moe_grouped_mlp(P, None, P, P, 64, 4, 128, 128, 2, P, None, P, None, P, 0, P, 1 << 20, s) == 1
    # combine: k > 32, bf16 d not a multiple of 8
    assert L.moe_unpermute_combine(P, P, 4, 33, 64, 1, P, s) == 1
    assert L.moe_unpermute_combine(P, P, 4, 2, 60, 1, P, s) == 2
    # layer: e0 + E_loc > E, workspace too small
    assert L.moe_layer_forward(P, P, 8, 64, 64, 8, 2, 4, 8, 1, P, None, P, None, P, P, 1 << 30, s) == 1
    # more routed rows than int32 indices hold (T * min(k, E_loc) > 2^31 - 1)
    big_T = (1 << 28) + 1
    assert L.moe_layer_forward(P, P, big_T, 64, 64, 8, 8, 0, 8, 1, P, None, P, None, P, P, 1 << 30, s) == 1
    assert L.moe_permute(P, 1, 1, big_T, 64, P, P, 8, 0, 8, P, None, P, P, P, P, P, P, 1 << 20, s) == 1
    assert L.moe_layer_forward(P, P, 8, 64, 64, 8, 2, 0, 8, 1, P, None, P, None, P, P, 64, s) == 3
    # expert GEMMs: workspace missing
    assert L.moe_expert_gemm2(P, None, P, 64, 4, 64, 64, 1, P, None, P, 0, _null(), 256, s) == 3
    assert L.moe_rows_hint(4096, 8, 64) == 512 and L.moe_rows_hint(0, 8, 64) == 0
    # bounded-wait self-test: timeout outside [1 ms, 2 s], missing workspace
    assert L.moe_selftest_wait_timeout(10, P, 256, s) == 1
    assert L.moe_selftest_wait_timeout(5_000_000_000, P, 256, s) == 1
    assert L.moe_selftest_wait_timeout(10_000_000, _null(), 256, s) == 3
    # workspace init: null / misaligned / too small
    assert L.moe_workspace_init(_null(), 256, s) == 3
    assert L.moe_workspace_init(ctypes.c_void_p(272), 256, s) == 3
    assert L.moe_workspace_init(P, 16, s) == 3
    # row-gather GEMM1: fp32 unsupported, null row map, bf16 d % 8
    assert L.moe_expert_gemm1_swiglu_gather(P, None, P, P, P, 64, 4, 64, 64, 0, P, None, P, None, 0, P, 256, s) == 2
    assert L.moe_expert_gemm1_swiglu_gather(P, None, None, P, P, 64, 4, 64, 64, 1, P, None, P, None, 0, P, 256,
                                            s) == 1
    assert L.moe_expert_gemm1_swiglu_gather(P, None, P, P, P, 64, 4, 60, 64, 1, P, None, P, None, 0, P, 256, s) == 2
    assert L.moe_expert_gemm1_swiglu_gather(P, None, P, P, P, 64, 4, 64, 64, 1, P, None, P, None, 0, _null(), 256,
                                            s) == 3
    # MXFP8 row quantiser: d % 32, negative T, wrong source type
    assert L.moe_quantize_mx_rows(P, 1, 4, 48, None, 0, P, P, s) == 2
    assert L.moe_quantize_mx_rows(P, 1, -1, 64, None, 0, P, P, s) == 1
    assert L.moe_quantize_mx_rows(P, 2, 4, 64, None, 0, P, P, s) == 2
    assert L.moe_quantize_mx_rows(P, 1, 4, 64, P, 33, P, P, s) == 1
    # training forward: missing routing / pre-activation outputs
    assert L.moe_layer_forward_train(P, P, 8, 64, 64, 8, 2, 0, 8, P, P, P, None, P, P, P, 1 << 30, s) == 1
    assert L.moe_layer_forward_train(P, P, 8, 64, 64, 8, 2, 0, 8, P, P, P, P, P, None, P, 1 << 30, s) == 1
    # backward: misaligned saved pre-activations
    assert L.moe_layer_backward(P, P, P, P, 8, 64, 64, 8, 2, 0, 8, P, P, P, ctypes.c_void_p(264), P, P, P, P, P, P,
                                1 << 30, s) == 1
    # device error read: null output
    assert L.moe_get_device_error(P, s, None) == 1


def test_8bit_entries_validate_before_any_launch(lib):
    """Per-tensor FP8 and MXFP8 packing / backward entries: argument and shape checks on the
    host, the workspace sizes they quote."""
    L = lib.lib()
    P = ctypes.c_void_p(256)  # never dereferenced
    s = _null()
    MX, FP8 = 2, 3
    # per-tensor FP8 pack: no exponent output, d or f not a multiple of 128, 8-bit source
    assert L.moe_pack_weights_fp8(P, P, P, 1, 4, 128, 128, P, P, P, P, None, s) == 1
    assert L.moe_pack_weights_fp8(P, P, P, 1, 4, 96, 128, P, P, P, P, P, s) == 2
    assert L.moe_pack_weights_fp8(P, P, P, 1, 4, 128, 96, P, P, P, P, P, s) == 2
    assert L.moe_pack_weights_fp8(P, P, P, MX, 4, 128, 128, P, P, P, P, P, s) == 2
    assert L.moe_pack_weights_fp8(P, P, P, 1, 2048, 128, 128, P, P, P, P, P, s) == 1  # E_loc > 1024
    # backward weight layouts: no exponents (FP8), d % 128, misaligned output
    assert L.moe_pack_weights_backward_fp8(P, P, P, 1, 4, 128, 128, None, P, P, P, P, s) == 1
    assert L.moe_pack_weights_backward_fp8(P, P, P, 1, 4, 96, 128, P, P, P, P, P, s) == 2
    assert L.moe_pack_weights_backward_mx(P, P, P, 1, 4, 128, 128, ctypes.c_void_p(264), P, P, P, s) == 1
    # 8-bit layer backward: e0 + E_loc > E, d % 128, workspace too small (both entry points)
    for fn in (L.moe_layer_backward_mx, L.moe_layer_backward_fp8):
        assert fn(P, P, P, P, 8, 128, 128, 8, 2, 4, 8, P, P, P, P, P, P, P, P, P, P, P, P, 1 << 30, s) == 1
        assert fn(P, P, P, P, 8, 96, 128, 8, 2, 0, 8, P, P, P, P, P, P, P, P, P, P, P, P, 1 << 30, s) == 2
        assert fn(P, P, P, P, 8, 128, 128, 8, 2, 0, 8, P, P, P, P, P, P, P, P, P, P, P, P, 64, s) == 3
    # the per-tensor FP8 backward uses the MXFP8 backward's workspace
    for args in ((4096, 2048, 1024, 8, 64), (8192, 7168, 2048, 8, 4), (0, 128, 128, 2, 1)):
        assert L.moe_layer_backward_fp8_workspace_size(*args) == L.moe_layer_backward_mx_workspace_size(*args) > 0
    # GEMM1's own workspace: the error word, plus bf16 h and its amax for per-tensor FP8
    assert L.moe_expert_gemm1_workspace_size(1000, 256, 1) == L.moe_expert_gemm1_workspace_size(1000, 256, MX) == 256
    assert L.moe_expert_gemm1_workspace_size(1000, 256, FP8) >= 256 + 1000 * 256 * 2 + 4
    # per-tensor FP8 GEMMs always run on the 1-CTA block-scaled kernel
    for g in (1, 2):
        assert lib.moe_layer_gemm_kernel(8192, 7168, 2048, 8, 256, 4, "fp8", g) == "cta"
        assert lib.moe_layer_gemm_kernel(4096, 2048, 1024, 8, 64, 64, "fp8", g) == "cta"


def test_gemm1_kernel_choice(lib):
    """The host-side rule behind moe_layer_forward's GEMM1 kernel: CTA pairs from 2048
    expected rows per expert, or 256-1023 rows when d >= 4096 (bf16 only); the 1-CTA
    kernel otherwise (measured per shape on B300)."""
    pairs = lib.moe_layer_gemm1_pairs
    assert not pairs(4096, 2048, 8, 64, 64, "bf16")      # 512 rows, d = 2048
    assert not pairs(8192, 7168, 8, 256, 4, "bf16")      # 256 rows, d = 7168: swapped operands
    assert pairs(16384, 7168, 8, 256, 4, "bf16")         # 512 rows
    assert not pairs(32768, 7168, 8, 256, 4, "bf16")     # 1024 rows
    assert not pairs(2048, 7168, 8, 256, 4, "bf16")      # 64 rows
    assert not pairs(8192, 2048, 8, 256, 4, "bf16")      # 256 rows but d < 4096
    assert pairs(16384, 7168, 1, 1, 1, "bf16")           # dense: 16384 rows
    assert pairs(4096, 1024, 8, 16, 16, "bf16")          # 2048 rows
    assert not pairs(8192, 7168, 8, 256, 4, "mxfp8")     # MXFP8 pairs only from 65536 rows per expert
    assert not pairs(16384, 7168, 1, 1, 1, "mxfp8")
    assert not pairs(8192, 7168, 8, 256, 4, "f32")
    with pytest.raises(ValueError):
        pairs(8192, 7168, 8, 256, 512, "bf16")            # E_loc > E


def test_gemm_kernel_choice(lib):
    """Which grouped-GEMM kernel moe_layer_forward runs (each rule measured on B300): bf16
    GEMM1 on the swapped-operand pair kernel from 256 to 320 expected rows per expert when
    d >= 4096 (E_loc <= 256), on token-major pairs from 321 to 1023 rows (d >= 4096) or from
    2048; bf16 GEMM2 on pairs from 128 rows; MXFP8 on the 1-CTA kernel; fp32 on its own."""
    kern = lib.moe_layer_gemm_kernel
    assert kern(8192, 7168, 2048, 8, 256, 4, "bf16", 1) == "swap"     # 256 rows (EP64, T = 8192)
    assert kern(10240, 7168, 2048, 8, 256, 4, "bf16", 1) == "swap"    # 320 rows
    assert kern(10272, 7168, 2048, 8, 256, 4, "bf16", 1) == "pair"    # 321 rows
    assert kern(8160, 7168, 2048, 8, 256, 4, "bf16", 1) == "cta"      # 255 rows
    assert kern(8192, 2048, 2048, 8, 256, 4, "bf16", 1) == "cta"      # 256 rows, d < 4096
    assert kern(8192, 7168, 2048, 8, 256, 4, "bf16", 2) == "pair"     # GEMM2: token-major pairs
    assert kern(2048, 7168, 2048, 8, 256, 4, "bf16", 1) == "cta"      # 64 rows
    assert kern(2048, 7168, 2048, 8, 256, 4, "bf16", 2) == "cta"
    assert kern(8192, 7168, 2048, 8, 256, 4, "mxfp8", 1) == "cta"
    assert kern(8192, 7168, 2048, 8, 256, 4, "mxfp8", 2) == "cta"
    assert kern(4096, 2048, 1024, 8, 64, 64, "bf16", 1) == "cta"      # bf16_e64: 512 rows
    assert kern(4096, 2048, 1024, 8, 64, 64, "bf16", 2) == "pair"
    assert kern(19200, 7168, 2048, 8, 512, 512, "bf16", 1) == "pair"  # 300 rows, but E_loc > 256
    assert kern(64, 128, 256, 2, 8, 8, "f32", 1) == "cta"
    with pytest.raises(ValueError):
        kern(8192, 7168, 2048, 8, 256, 4, "bf16", 3)


def test_combine_fusion_choice(lib):
    """moe_layer_forward folds the combine into GEMM2 when tokens average under one local
    slot (k * E_loc < E), for bf16 and MXFP8 (measured per shape on B300)."""
    fused = lib.moe_layer_fused_combine
    assert fused(8, 256, 4, "bf16") and fused(8, 256, 4, "mxfp8")   # EP64 slice: 0.125 slots
    assert not fused(8, 256, 32, "bf16")                             # EP8 slice: 1 slot
    assert not fused(8, 64, 64, "bf16")                              # all experts local
    assert not fused(8, 256, 4, "f32")                               # fp32: SIMT GEMMs + combine
    with pytest.raises(ValueError):
        fused(8, 4, 8, "bf16")
