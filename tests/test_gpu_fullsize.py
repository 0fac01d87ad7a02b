"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (quantise Q, K, V, then the FP8 forward, one workspace): codes and scales
of every tensor bit-exact to the oracle's quantiser over the whole tensor, and
the output on sampled rows (the first, tile-boundary and last rows of every
document plus seeded random rows, all heads) within the parity bounds against
the oracle's quantised-operand emulation, with its tie allowance.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import compare_outputs, mx_col_tiles_to_logical, mx_row_tiles_to_logical, to_device

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu

E4M3, ROW, COL = 0, 1, 2


def sample_rows(cu, T, seed, n_random=384):
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        L = e - s
        for r in (0, 1, 2, 127, 128, 129, 255, 256, L - 3, L - 2, L - 1):
            if 0 <= r < L:
                rows.append(s + r)
    rows.extend(rng.choice(T, size=min(n_random, T), replace=False).tolist())
    return np.unique(np.asarray(rows, dtype=np.int32))


@pytest.mark.parametrize("wid,exact", [(2, False), (3, False), (3, True), (4, False), (5, False)])
def test_full_size_codes_and_sampled_rows(oracle_mod, wid, exact):
    """exact: the causal configuration's causal-exact mode (one E4M3 scale per
    token, V ratios against the running maximum of earlier tokens' scales)."""
    w = workloads.WORKLOADS[wid]
    inp = workloads.make(wid)
    T, H, d = inp.q.shape
    cu = inp.cu_seqlens
    q, k, v, cu_d = to_device(inp)
    ws = pa.workspace(T, H, d, len(cu) - 1)
    seed = w.hadamard_seed
    if w.mx:
        lq, lk, lv, blk = ROW, ROW, COL, 32
    else:
        lq = lk = lv = E4M3
        blk = 1 if exact else w.block
    Q = pa.attn_quantize(q, cu_d, lq, blk, True, seed, ws=ws)
    K = pa.attn_quantize(k, cu_d, lk, blk, True, seed, ws=ws)
    V = pa.attn_quantize(v, cu_d, lv, blk, False, 0, ws=ws)
    o, lse = pa.attn_fp8_fwd(Q, K, V, cu_d, w.causal, exact, 0.0, ws=ws)
    st, flags = pa.attn_read_device_status(ws)
    assert st == 0, (st, flags)

    Qo = oracle.quantize_tensor(inp.q, cu, lq, blk, True, seed)
    Ko = oracle.quantize_tensor(inp.k, cu, lk, blk, True, seed)
    Vo = oracle.quantize_tensor(inp.v, cu, lv, blk, False, 0)
    for name, g, c in (("Q", Q, Qo), ("K", K, Ko), ("V", V, Vo)):
        gc = g.codes.cpu().numpy()
        assert np.array_equal(gc, c.codes), f"{name}: {np.count_nonzero(gc != c.codes)} code mismatches"
        gs = g.scales.cpu().numpy()
        if not w.mx:
            nb = c.scales.shape[1]
            assert np.array_equal(gs[:, :nb].view(np.uint32), c.scales.view(np.uint32)), f"{name} scales"
        elif name == "V":
            assert np.array_equal(mx_col_tiles_to_logical(gs, cu, T, H, d), c.scales), f"{name} scales"
        else:
            assert np.array_equal(mx_row_tiles_to_logical(gs, cu, T, H), c.scales), f"{name} scales"

    rows = sample_rows(cu, T, seed=wid)
    _, ob, le, amb = oracle.attention_emulate(Qo, Ko, Vo, cu, w.causal, exact, None, rows=rows, ties=True,
                                              rescale_tau=pa.rescale_threshold(inp.q.shape[2]))
    res = compare_outputs(o, lse, ob, le, rows=rows, ties=amb)
    print(f"workload {wid}{' exact' if exact else ''}: {len(rows)} rows x {H} heads:", res)
    assert res["ok"], res


@pytest.mark.parametrize("wid,exp_mode", [(2, 0), (3, 0), (2, 1), (3, 2)])
def test_full_size_nvfp4_qk_and_bit_level_exponentials(oracle_mod, wid, exp_mode):
    """The mixed NVFP4/FP8 path at the fa3 configurations' full size (NVFP4 Q, K codes
    and both scale levels bit-exact, sampled rows within the parity bounds), with the
    hardware exp2 and with the bit-level exponentials (Schraudolph, log-domain P)."""
    w = workloads.WORKLOADS[wid]
    inp = workloads.make(wid)
    T, H, d = inp.q.shape
    cu = inp.cu_seqlens
    nd = len(cu) - 1
    q, k, v, cu_d = to_device(inp)
    ws = pa.workspace(T, H, d, nd)
    seed = w.hadamard_seed
    Q = pa.attn_quantize(q, cu_d, pa.ATTN_NVFP4, 128, True, seed, ws=ws)
    K = pa.attn_quantize(k, cu_d, pa.ATTN_NVFP4, 128, True, seed, ws=ws)
    V = pa.attn_quantize(v, cu_d, E4M3, 128, False, 0, ws=ws)
    o, lse = pa.attn_fp8_fwd_ex(Q, K, V, cu_d, w.causal, False, 0.0, exp_mode, ws=ws)
    st, flags = pa.attn_read_device_status(ws)
    assert st == 0, (st, flags)
    Qo = oracle.quantize_tensor(inp.q, cu, oracle.NVFP4, 128, True, seed)
    Ko = oracle.quantize_tensor(inp.k, cu, oracle.NVFP4, 128, True, seed)
    Vo = oracle.quantize_tensor(inp.v, cu, E4M3, 128, False, 0)
    for name, g, c in (("Q", Q, Qo), ("K", K, Ko)):
        assert np.array_equal(g.codes.cpu().numpy(), c.codes), name
        g_st, g_sf = (t.cpu().numpy() for t in pa.nvfp4_scales(g, nd))
        nb = c.scales[0].shape[1]
        assert np.array_equal(g_st[:, :nb].view(np.uint32), c.scales[0].view(np.uint32)), name
        both = np.concatenate([mx_row_tiles_to_logical(g_sf[:, :, :512], cu, T, H),
                               mx_row_tiles_to_logical(g_sf[:, :, 512:], cu, T, H)], axis=2)
        assert np.array_equal(both, c.scales[1]), name
    assert np.array_equal(V.codes.cpu().numpy(), Vo.codes)
    rows = sample_rows(cu, T, seed=100 + wid)
    _, ob, le, amb, lamb = oracle.attention_emulate(Qo, Ko, Vo, cu, w.causal, False, None, rows=rows, ties=True,
                                                    rescale_tau=pa.rescale_threshold(d), exp_mode=exp_mode,
                                                    lse_ties=True)
    res = compare_outputs(o, lse, ob, le, rows=rows, ties=amb, lse_ties=lamb)
    res["lse_tie_max"] = float(lamb.max())
    print(f"workload {wid} NVFP4 Q K^T, exp mode {exp_mode}: {len(rows)} rows x {H} heads:", res)
    assert res["ok"], res
