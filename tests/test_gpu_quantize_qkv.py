"""The one-launch Q/K/V quantiser (FLAMIA section 4.3: the forward's quantisation
fused into one launch): attn_quantize_qkv writes the same bytes as three
attn_quantize calls, which the other quantiser tests pin to the oracle; one case
here goes to the oracle directly.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import to_device

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu

E4M3, ROW, COL, TOK, NV = 0, 1, 2, 3, 4
SEED = 0x5EED0009


def _bytes(qt):
    return qt.codes.cpu().numpy().tobytes(), qt.scales.cpu().numpy().tobytes()


def _fill(qt):
    # both sides start from the same garbage so that bytes neither writes compare equal
    qt.codes.fill_(0xA5)
    qt.scales.view(torch.uint8).fill_(0xA5)
    return qt


def _separate_and_fused(q, k, v, cu, lq, bq, lv, bv, rotate, rule=0):
    T, H, d = q.shape
    nd = cu.numel() - 1
    ws = pa.workspace(T, H, d, nd)
    sep = [_fill(pa.empty_qtensor(T, H, d, nd, L, b, rule)) for L, b in ((lq, bq), (lq, bq), (lv, bv))]
    for x, o, r in zip((q, k, v), sep, (rotate, rotate, False)):
        pa.attn_quantize(x, cu, o.layout, o.block, r, SEED, rule, ws=ws, out=o)
    st_sep, _ = pa.attn_read_device_status(ws)
    ws2 = pa.workspace(T, H, d, nd)
    fus = tuple(_fill(pa.empty_qtensor(T, H, d, nd, L, b, rule)) for L, b in ((lq, bq), (lq, bq), (lv, bv)))
    pa.attn_quantize_qkv(q, k, v, cu, lq, bq, lv, bv, rotate, SEED, rule, ws=ws2, outs=fus)
    st_fus, _ = pa.attn_read_device_status(ws2)
    return sep, fus, st_sep, st_fus


@pytest.mark.parametrize("wid,lengths,H,lq,bq,lv,bv,rotate,rule", [
    (2, [300, 77, 129], 3, E4M3, 128, E4M3, 128, True, 0),    # the headline layout, ragged documents
    (1, [200, 56, 129], 2, E4M3, 64, E4M3, 64, True, 0),      # fp32 input, head_dim 64
    (2, [300, 77], 2, E4M3, 32, E4M3, 32, False, 0),
    (3, [257, 31], 2, E4M3, 1, E4M3, 1, True, 0),             # per-token scales (causal-exact operands)
    (4, [300, 77, 129], 2, ROW, 32, COL, 32, True, 0),        # MXFP8
    (4, [130, 1, 255], 2, ROW, 32, COL, 32, False, 1),        # MXFP8, OCP floor rule
    (5, [300, 77, 129], 2, ROW, 32, TOK, 1, True, 0),         # MXFP8, per-token V
    (2, [300, 77, 129], 2, NV, 128, E4M3, 128, True, 0),      # NVFP4 Q, K with E4M3 V
    (4, [256, 1, 130], 2, NV, 128, E4M3, 128, False, 0),
])
def test_fused_equals_three_launches(wid, lengths, H, lq, bq, lv, bv, rotate, rule):
    inp = workloads.make(wid, heads=H, lengths=lengths)
    q, k, v, cu = to_device(inp)
    sep, fus, st_sep, st_fus = _separate_and_fused(q, k, v, cu, lq, bq, lv, bv, rotate, rule)
    assert st_sep == 0 and st_fus == 0
    for name, a, b in zip("QKV", sep, fus):
        ca, sa = _bytes(a)
        cb, sb = _bytes(b)
        assert ca == cb, f"{name} codes differ"
        assert sa == sb, f"{name} scales differ"
        assert (a.rotated, a.hadamard_seed) == (b.rotated, b.hadamard_seed), name
    assert fus[2].rotated == 0 and fus[0].rotated == int(rotate)


@pytest.mark.parametrize("lq,bq,lv,bv", [(E4M3, 128, E4M3, 128), (ROW, 32, COL, 32), (NV, 128, E4M3, 128)])
def test_fused_fp32_input_head_dim_128(lq, bq, lv, bv):
    """fp32 rows of 128 channels: 64 KB stages, one CTA per SM (the bf16 cases run two)."""
    inp = workloads.make(2, heads=2, lengths=[300, 77, 129])
    q, k, v, cu = to_device(inp, dtype=torch.float32)
    sep, fus, st_sep, st_fus = _separate_and_fused(q, k, v, cu, lq, bq, lv, bv, True)
    assert st_sep == 0 and st_fus == 0
    for name, a, b in zip("QKV", sep, fus):
        assert _bytes(a) == _bytes(b), name


def test_fused_matches_oracle(oracle_mod):
    """Q, K and V of one fused launch against the oracle directly (E4M3, 128-token blocks)."""
    inp = workloads.make(2, heads=2, lengths=[300, 77, 129])
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    ws = pa.workspace(T, H, d, 3)
    Q, K, V = pa.attn_quantize_qkv(q, k, v, cu, E4M3, 128, rotate=True, hadamard_seed=SEED, ws=ws)
    assert pa.attn_read_device_status(ws)[0] == 0
    for x_np, qt, r in ((inp.q, Q, True), (inp.k, K, True), (inp.v, V, False)):
        codes, scales, ost = oracle_mod.quantize(x_np, inp.cu_seqlens, E4M3, 128, r, SEED if r else 0)
        assert ost == 0
        assert np.array_equal(qt.codes.cpu().numpy(), codes)
        nb = scales.shape[1]
        assert np.array_equal(qt.scales.cpu().numpy()[:, :nb].view(np.uint32), scales.view(np.uint32))


def test_packed_qkv_views_and_many_documents():
    """Q, K, V as views of one packed [T, 3, H, d] tensor (token stride 3 H d), and
    more documents than fit a CTA's own table (the table kernel runs first)."""
    lens = workloads.doc_lengths(40000, 1, 50, seed=11)
    assert len(lens) > 1024
    inp = workloads.make(2, heads=2, lengths=list(lens))
    q, k, v, cu = to_device(inp)
    qkv = torch.stack([q, k, v], dim=1).contiguous()
    qv, kv, vv = qkv[:, 0], qkv[:, 1], qkv[:, 2]
    assert qv.stride(0) == 3 * 2 * 128
    for lq, bq, lv, bv in ((E4M3, 128, E4M3, 128), (NV, 128, E4M3, 128), (ROW, 32, COL, 32)):
        sep, fus, st_sep, st_fus = _separate_and_fused(qv, kv, vv, cu, lq, bq, lv, bv, True)
        assert st_sep == 0 and st_fus == 0
        for name, a, b in zip("QKV", sep, fus):
            assert _bytes(a) == _bytes(b), (name, lq)


def test_nonfinite_in_any_tensor_flags_the_one_status():
    T, H, d = 200, 2, 128
    cu = torch.tensor([0, 120, 200], dtype=torch.int32, device="cuda")
    for bad in range(3):
        xs = [torch.randn(T, H, d, device="cuda", dtype=torch.bfloat16) for _ in range(3)]
        xs[bad][150, 1, 7] = float("nan")
        ws = pa.workspace(T, H, d, 2)
        pa.attn_quantize_qkv(*xs, cu, E4M3, 128, rotate=True, hadamard_seed=SEED, ws=ws)
        assert pa.attn_read_device_status(ws)[0] == pa.ATTN_ERR_NONFINITE, bad


def test_fused_in_a_cuda_graph_replays_bitwise():
    """The fused launch captures in a CUDA graph; a replay writes the eager bytes."""
    inp = workloads.make(2, heads=2, lengths=[300, 77, 129])
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    ws = pa.workspace(T, H, d, 3)
    outs = tuple(_fill(pa.empty_qtensor(T, H, d, 3, L, 128)) for L in (NV, NV, E4M3))
    pa.attn_quantize_qkv(q, k, v, cu, NV, 128, E4M3, 128, True, SEED, ws=ws, outs=outs)
    torch.cuda.synchronize()
    eager = [_bytes(o) for o in outs]
    for o in outs:
        _fill(o)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pa.attn_quantize_qkv(q, k, v, cu, NV, 128, E4M3, 128, True, SEED, ws=ws, outs=outs, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert [_bytes(o) for o in outs] == eager
