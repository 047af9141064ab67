"""Shared helpers of the tests (no test cases here).

Conversions between the numpy storage of the synthetic inputs and torch device tensors,
the relative L2 error, and the decoders of the library's MXFP8 scale-factor tile layout
(used to compare device scales with the oracle's plain [rows, K/32] scales).
"""
from __future__ import annotations

import numpy as np
import torch

# relative L2 vs the fp64 oracle; per-tensor FP8 takes the MXFP8 bound (same E4M3 codes and
# rounding points on both sides; the GPU rounds h to bf16 before quantising it)
TOL = {"f32": 1e-5, "bf16": 2e-2, "mxfp8": 5e-2, "fp8": 5e-2}


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def to_dev(a: np.ndarray, dev="cuda") -> torch.Tensor:
    """numpy storage -> device tensor (uint16 arrays are bf16 bit patterns)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def to_np(t: torch.Tensor) -> np.ndarray:
    """device tensor -> numpy (bf16 -> fp64 values, others as is)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    return t.numpy()


def bf16_bits_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def mtile_prefix(offsets: np.ndarray) -> np.ndarray:
    cnt = np.diff(offsets.astype(np.int64))
    mt = (cnt + 127) // 128
    return np.concatenate([[0], np.cumsum(mt)])


def unpack_act_sf(sf: np.ndarray, offsets: np.ndarray, K: int, N: int) -> np.ndarray:
    """Activation SF tile layout -> plain scales [N, K/32]."""
    offsets = offsets.astype(np.int64)
    mtp = mtile_prefix(offsets)
    rows = np.arange(N)
    e = np.searchsorted(offsets, rows, side="right") - 1
    il = rows - offsets[e]
    tile = mtp[e] + il // 128
    i = il % 128
    kb = np.arange(K // 32)
    off = ((tile[:, None] * (K // 128) + kb[None, :] // 4) * 512 + (i[:, None] % 32) * 16 + (i[:, None] // 32) * 4
           + kb[None, :] % 4)
    return sf[off]


def unpack_w_sf(sf: np.ndarray, E_loc: int, rows: int, K: int) -> np.ndarray:
    """Weight SF tile layout -> plain scales [E_loc, rows, K/32]."""
    e = np.arange(E_loc)[:, None, None]
    r = np.arange(rows)[None, :, None]
    kb = np.arange(K // 32)[None, None, :]
    off = (((e * (K // 128) + kb // 4) * (rows // 128) + r // 128) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4
           + kb % 4)
    return sf[off]


def gate_up_rows(f: int):
    """Packed GEMM1 row index of gate column n and of up column n (32-column interleave)."""
    n = np.arange(f)
    g = (n // 32) * 64 + n % 32
    return g, g + 32
