"""GPU quantiser parity: codes and scales bit-exact to the oracle (O-2).

Inputs are the seeded workload recipes at reduced sizes that still span
several blocks and tiles, with ragged documents.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import (mx_col_pad_bytes, mx_col_tiles_to_logical, mx_row_pad_bytes, mx_row_tiles_to_logical,
                         to_device)

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu

E4M3, ROW, COL = 0, 1, 2
SEED = 0x5EED0002


def gpu_quant(x_dev, cu_dev, layout, block, rotate, seed=SEED, rule=0):
    T, H, d = x_dev.shape
    nd = cu_dev.numel() - 1
    ws = pa.workspace(T, H, d, nd)
    qt = pa.attn_quantize(x_dev, cu_dev, layout, block, rotate, seed, rule, ws=ws)
    st, flags = pa.attn_read_device_status(ws)
    return qt, st


@pytest.mark.parametrize("wid,lengths,H,block,rotate", [
    (1, [256], 2, 64, True),            # the tiny fp32 workload, d = 64
    (1, [200, 56, 129], 2, 64, False),
    (2, [300, 77, 129], 3, 128, True),  # outlier recipe, bf16
    (2, [300, 77], 2, 32, True),
    (3, [257, 31], 2, 1, True),         # per-token scales (causal-exact layout)
])
def test_e4m3_tokblock_bit_exact(oracle_mod, wid, lengths, H, block, rotate):
    inp = workloads.make(wid, heads=H, lengths=lengths)
    q, k, v, cu = to_device(inp)
    for x_np, x_dev in ((inp.q, q), (inp.v, v)):
        qt, st = gpu_quant(x_dev, cu, E4M3, block, rotate)
        assert st == 0
        codes, scales, ost = oracle_mod.quantize(x_np, inp.cu_seqlens, E4M3, block, rotate, SEED)
        assert ost == 0
        nb = scales.shape[1]
        g_codes = qt.codes.cpu().numpy()
        g_scales = qt.scales.cpu().numpy()[:, :nb]
        assert np.array_equal(g_codes, codes), f"{np.sum(g_codes != codes)} code mismatches"
        assert np.array_equal(g_scales.view(np.uint32), scales.view(np.uint32))
        assert qt.rotated == int(rotate)


@pytest.mark.parametrize("lengths,H,rotate,rule", [
    ([256], 2, True, 0),
    ([300, 77, 129], 2, True, 0),
    ([130, 1, 255], 2, False, 1),
])
def test_mx_bit_exact(oracle_mod, lengths, H, rotate, rule):
    inp = workloads.make(4, heads=H, lengths=lengths)
    q, k, v, cu = to_device(inp)
    T, d = inp.T, 128
    qt, st = gpu_quant(q, cu, ROW, 32, rotate, rule=rule)
    assert st == 0
    codes, su, _ = oracle_mod.quantize(inp.q, inp.cu_seqlens, ROW, 32, rotate, SEED, rule)
    tiles = qt.scales.cpu().numpy()
    assert np.array_equal(qt.codes.cpu().numpy(), codes)
    assert np.array_equal(mx_row_tiles_to_logical(tiles, inp.cu_seqlens, T, H), su)
    assert np.all(mx_row_pad_bytes(tiles, inp.cu_seqlens, T) == 127)

    vt, st = gpu_quant(v, cu, COL, 32, False, rule=rule)
    assert st == 0
    vcodes, vsu, _ = oracle_mod.quantize(inp.v, inp.cu_seqlens, COL, 32, False, 0, rule)
    vtiles = vt.scales.cpu().numpy()
    assert np.array_equal(vt.codes.cpu().numpy(), vcodes)
    assert np.array_equal(mx_col_tiles_to_logical(vtiles, inp.cu_seqlens, T, H, d), vsu)
    assert np.all(mx_col_pad_bytes(vtiles, inp.cu_seqlens, T, d) == 127)


def test_nonfinite_input_flags_status():
    x = torch.randn(64, 2, 128, device="cuda", dtype=torch.bfloat16)
    x[10, 1, 5] = float("inf")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    for layout, block in ((E4M3, 128), (E4M3, 1), (ROW, 32), (COL, 32)):
        _, st = gpu_quant(x, cu, layout, block, True)
        assert st == pa.ATTN_ERR_NONFINITE, (layout, block)


def test_bad_seqlens_flags_status():
    x = torch.randn(64, 2, 128, device="cuda", dtype=torch.bfloat16)
    cu = torch.tensor([0, 40, 30, 64], dtype=torch.int32, device="cuda")   # not monotone
    _, st = gpu_quant(x, cu, E4M3, 128, True)
    assert st == pa.ATTN_ERR_BAD_SEQLENS


def test_strided_input_matches_contiguous(oracle_mod):
    inp = workloads.make(2, heads=4, lengths=[200])
    full = torch.from_numpy(inp.q).to(torch.bfloat16).cuda()
    sub = full[:, 1:3, :]                        # head stride d, token stride 4d
    cu = torch.tensor([0, 200], dtype=torch.int32, device="cuda")
    qt, st = gpu_quant(sub, cu, E4M3, 128, True)
    codes, scales, _ = oracle_mod.quantize(np.ascontiguousarray(inp.q[:, 1:3, :]), inp.cu_seqlens, E4M3, 128,
                                           True, SEED)
    assert st == 0 and np.array_equal(qt.codes.cpu().numpy(), codes)


@pytest.mark.parametrize("lengths,H,rule", [([300, 77, 129], 2, 0), ([130, 1, 255], 3, 1), ([256], 2, 0)])
def test_mx_token_bit_exact(oracle_mod, lengths, H, rule):
    """The MX token layout (V of the causal-exact MX mode): codes and the one
    exponent per (token, head) bit-exact to the oracle, packed documents."""
    inp = workloads.make(5, heads=H, lengths=lengths)
    q, k, v, cu = to_device(inp)
    qt, st = gpu_quant(v, cu, pa.ATTN_MX_TOKEN, 1, False, 0, rule)
    assert st == 0
    codes, su, ost = oracle_mod.quantize(inp.v, inp.cu_seqlens, oracle_mod.MX_TOKEN, 1, False, 0, rule)
    assert ost == 0
    assert np.array_equal(qt.codes.cpu().numpy(), codes)
    assert np.array_equal(qt.scales.cpu().numpy()[:, :inp.T], su)


@pytest.mark.parametrize("wid,lengths,H,rotate", [
    (2, [300, 77, 129], 2, True),       # outlier recipe, ragged documents, rotated
    (4, [256, 1, 130], 2, True),        # outlier channels, a one-token document
    (2, [384], 1, False),
])
def test_nvfp4_bit_exact(oracle_mod, wid, lengths, H, rotate):
    """NVFP4 Q/K operands (FLAMIA sections 1 and 2): E2M1 codes, the fp32 scale of
    each 128-token block and every 16-channel E4M3 scale in the MMA-ready tiles
    equal the oracle's; scale bytes of rows past a document end are 0."""
    inp = workloads.make(wid, heads=H, lengths=lengths)
    q, k, v, cu = to_device(inp)
    T = inp.T
    nd = len(inp.cu_seqlens) - 1
    for x_np, x_dev in ((inp.q, q), (inp.k, k)):
        qt, st = gpu_quant(x_dev, cu, pa.ATTN_NVFP4, 128, rotate)
        assert st == 0
        codes, (sf32, su), ost = oracle_mod.quantize(x_np, inp.cu_seqlens, oracle_mod.NVFP4, 128, rotate, SEED)
        assert ost == 0
        g_st, g_sf = (t.cpu().numpy() for t in pa.nvfp4_scales(qt, nd))
        assert np.array_equal(qt.codes.cpu().numpy(), codes), f"{np.sum(qt.codes.cpu().numpy() != codes)} code bytes differ"
        nb = sf32.shape[1]
        assert np.array_equal(g_st[:, :nb].view(np.uint32), sf32.view(np.uint32))
        lo = mx_row_tiles_to_logical(g_sf[:, :, :512], inp.cu_seqlens, T, H)
        hi = mx_row_tiles_to_logical(g_sf[:, :, 512:], inp.cu_seqlens, T, H)
        assert np.array_equal(np.concatenate([lo, hi], axis=2), su)
        assert np.all(mx_row_pad_bytes(g_sf[:, :, :512], inp.cu_seqlens, T) == 0)
        assert np.all(mx_row_pad_bytes(g_sf[:, :, 512:], inp.cu_seqlens, T) == 0)
