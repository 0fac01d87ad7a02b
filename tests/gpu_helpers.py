"""Shared helpers for the GPU parity tests (test-side index bookkeeping only).

`mx_tiles_to_logical_*` undo the tile order in which the library stores MX
scales (documented in include/attn.h) so they can be compared byte for byte
with the oracle's logical scale arrays.
"""
import math

import numpy as np
import torch

import oracle
import workloads

TOL_REL_RMSE = 1e-3
TOL_MAX_ABS = 2e-3
TOL_LSE = 1e-3


def doc_bounds(cu, T):
    return np.array([0, T], dtype=np.int64) if cu is None else np.asarray(cu, dtype=np.int64)


def mx_row_tiles_to_logical(tiles: np.ndarray, cu, T: int, H: int) -> np.ndarray:
    """[H, nt_cap, 512] -> [T, H, 4] (row r of a tile, group g at (r%32)*16 + (r//32)*4 + g)."""
    b = doc_bounds(cu, T)
    out = np.zeros((T, H, 4), dtype=np.uint8)
    toff = 0
    for i in range(len(b) - 1):
        s, L = int(b[i]), int(b[i + 1] - b[i])
        lt = np.arange(L)
        tile = toff + lt // 128
        r = lt % 128
        for g in range(4):
            off = (r % 32) * 16 + (r // 32) * 4 + g
            out[s:s + L, :, g] = tiles[:, tile, off].T
        toff += (L + 127) // 128
    return out


def mx_row_pad_bytes(tiles: np.ndarray, cu, T: int) -> np.ndarray:
    """All scale bytes of rows past the end of their document (must be 127)."""
    b = doc_bounds(cu, T)
    vals = []
    toff = 0
    for i in range(len(b) - 1):
        L = int(b[i + 1] - b[i])
        nt = (L + 127) // 128
        for r in range(L - (nt - 1) * 128, 128):
            for g in range(4):
                vals.append(tiles[:, toff + nt - 1, (r % 32) * 16 + (r // 32) * 4 + g])
        toff += nt
    return np.concatenate(vals) if vals else np.zeros(0, np.uint8)


def mx_col_tiles_to_logical(tiles: np.ndarray, cu, T: int, H: int, d: int) -> np.ndarray:
    """[H, nt_cap, 512] -> [H, NG, d] (channel c, group gi of a tile at (c%32)*16 + (c//32)*4 + gi)."""
    b = doc_bounds(cu, T)
    ng_tot = sum((int(b[i + 1] - b[i]) + 31) // 32 for i in range(len(b) - 1))
    out = np.zeros((H, ng_tot, d), dtype=np.uint8)
    c = np.arange(d)
    toff = goff = 0
    for i in range(len(b) - 1):
        L = int(b[i + 1] - b[i])
        for G in range((L + 31) // 32):
            tile, gi = toff + G // 4, G % 4
            out[:, goff + G, :] = tiles[:, tile, (c % 32) * 16 + (c // 32) * 4 + gi]
        toff += (L + 127) // 128
        goff += (L + 31) // 32
    return out


def mx_col_pad_bytes(tiles: np.ndarray, cu, T: int, d: int) -> np.ndarray:
    b = doc_bounds(cu, T)
    c = np.arange(d)
    vals = []
    toff = 0
    for i in range(len(b) - 1):
        L = int(b[i + 1] - b[i])
        nt = (L + 127) // 128
        for G in range((L + 31) // 32, nt * 4):
            vals.append(tiles[:, toff + G // 4, (c % 32) * 16 + (c // 32) * 4 + G % 4].ravel())
        toff += nt
    return np.concatenate(vals) if vals else np.zeros(0, np.uint8)


def to_device(inp: workloads.Inputs, dtype=None):
    dt = dtype or (torch.float32 if inp.in_dtype == "f32" else torch.bfloat16)
    q, k, v = (torch.from_numpy(np.ascontiguousarray(a)).to(dt).cuda() for a in (inp.q, inp.k, inp.v))
    cu = torch.from_numpy(inp.cu_seqlens.astype(np.int32)).cuda()
    return q, k, v, cu


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def compare_outputs(o_gpu_bf16: torch.Tensor, lse_gpu: torch.Tensor, o_emu_bf16_bits: np.ndarray,
                    lse_emu: np.ndarray, rows=None, ties=None, lse_ties=None):
    """Parity of the GPU output with the oracle's quantised-operand emulation.

    Criteria (the stated accuracy bounds, read for a BF16 output): relative RMSE of
    the BF16 outputs <= 1e-3; per element |diff| <= max(2e-3, one BF16 ulp of
    the emulated value) -- one ulp is what a rounding flip of nearly equal fp32
    values costs, and it exceeds 2e-3 wherever |O| >= 0.5; lse within 1e-3
    (plus, under the log-domain P, `lse_ties`: what tied codes move the row sum).
    `ties` is the emulation's tie allowance: the part of an element that E4M3
    probability codes lying within fp32 rounding of a code boundary may move
    (either neighbouring code is a faithful result); it widens the bound of
    those elements only, and the count of elements that needed it is returned.
    With ties the relative RMSE is taken over what the ties cannot explain,
    max(0, |diff| - allowance) per element (the distance to the nearest result
    the tied codes allow); the plain relative RMSE is reported beside it.
    Returns a dict of the measured figures.
    """
    og = o_gpu_bf16.float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        og = og[rows]
        lg = lg[:, rows]
    oe = oracle.bf16_bits_to_f32(o_emu_bf16_bits).astype(np.float64)
    diff = np.abs(og - oe)
    rel = float(np.linalg.norm(og - oe) / max(np.linalg.norm(oe), 1e-30))
    base = np.maximum(TOL_MAX_ABS, bf16_ulp(oe))
    if ties is None:
        bound = base
        n_ties = 0
        rel_u = rel
    else:
        t = ties.astype(np.float64)
        bound = np.maximum(TOL_MAX_ABS, bf16_ulp(np.abs(oe) + t)) + t
        n_ties = int(np.count_nonzero((diff > base) & (diff <= bound)))
        rel_u = float(np.linalg.norm(np.maximum(diff - t, 0.0)) / max(np.linalg.norm(oe), 1e-30))
    ratio = diff / bound
    worst = float(ratio.max()) if diff.size else 0.0
    at = tuple(int(i) for i in np.unravel_index(int(np.argmax(ratio)), ratio.shape)) if diff.size else ()
    dlse = np.abs(lg - lse_emu)
    if lse_ties is not None:
        dlse = np.maximum(dlse - lse_ties.astype(np.float64), 0.0)
    dl = float(dlse.max()) if lg.size else 0.0
    return {"rel_rmse": rel, "rel_rmse_unexplained": rel_u, "max_abs": float(diff.max()) if diff.size else 0.0,
            "worst_over_bound": worst,
            "lse_max": dl, "tie_explained": n_ties, "worst_at": at,
            "worst_gpu_emu_tie": (float(og[at]), float(oe[at]), 0.0 if ties is None else float(ties[at])) if at else (),
            "ok": rel_u <= TOL_REL_RMSE and worst <= 1.0 and dl <= TOL_LSE}
