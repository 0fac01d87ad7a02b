"""GPU edge cases of the forward: empty documents inside the packed batch (at
its start, middle and end), all-zero inputs (every block maximum 0: scale 0,
zero codes, every score 0) against the closed form, and a single head."""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import compare_outputs, to_device
from test_gpu_attention import run_emu, run_gpu

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu

EMPTY_DOCS = [0, 150, 0, 0, 257, 1, 0]


@pytest.mark.parametrize("wid,mx,block,causal", [
    (1, False, 64, True),      # d = 64, one-tile kernel
    (2, False, 128, False),    # E4M3 tile scales
    (3, False, 32, True),      # E4M3 per-column scales
    (4, True, 32, False),      # MXFP8
    (5, True, 32, True),
])
def test_zero_length_documents(oracle_mod, wid, mx, block, causal):
    inp = workloads.make(wid, heads=2, lengths=EMPTY_DOCS)
    o, lse = run_gpu(inp, mx, block, causal)
    _, ob, le, amb = run_emu(inp, mx, block, causal)
    res = compare_outputs(o, lse, ob, le, ties=amb)
    assert res["ok"], res


def visible_keys(cu, causal):
    """Keys each row sees: its document's length, or its position + 1 (causal)."""
    n = []
    for a, b in zip(cu[:-1], cu[1:]):
        L = int(b - a)
        n.append(np.arange(1, L + 1) if causal else np.full(L, L))
    return np.concatenate(n).astype(np.float64)


@pytest.mark.parametrize("wid,mx,block,causal", [
    (1, False, 64, False),
    (2, False, 128, False),
    (3, False, 128, True),
    (3, False, 1, True),       # one scale per token (causal-exact layout)
    (4, True, 32, False),
    (5, True, 32, True),
])
def test_all_zero_inputs_closed_form(wid, mx, block, causal):
    """Q = K = V = 0: every score is 0, so each row's probabilities are uniform
    over the keys it sees, O = 0 exactly and lse = ln(number of visible keys)."""
    inp = workloads.make(wid, heads=2, lengths=[200, 77, 129])
    inp.q[:] = 0.0
    inp.k[:] = 0.0
    inp.v[:] = 0.0
    o, lse = run_gpu(inp, mx, block, causal, exact=(block == 1))
    assert int(torch.count_nonzero(o.float())) == 0
    want = np.log(visible_keys(inp.cu_seqlens, causal))
    got = lse.double().cpu().numpy()
    assert got.shape == (2, inp.T)
    assert np.abs(got - want[None, :]).max() <= 1e-5 * np.maximum(1.0, want).max()


@pytest.mark.parametrize("wid,mx,block,causal", [(2, False, 128, False), (3, False, 128, True), (5, True, 32, True)])
def test_single_head(oracle_mod, wid, mx, block, causal):
    inp = workloads.make(wid, heads=1, lengths=[300, 77])
    o, lse = run_gpu(inp, mx, block, causal)
    _, ob, le, amb = run_emu(inp, mx, block, causal)
    res = compare_outputs(o, lse, ob, le, ties=amb)
    assert res["ok"], res


@pytest.mark.parametrize("ndocs", [1024, 3000])
@pytest.mark.parametrize("wid,mx,block,causal", [(3, False, 128, True), (2, False, 32, False), (4, True, 32, False),
                                                 (3, False, 1, True)])
def test_many_documents(oracle_mod, ndocs, wid, mx, block, causal):
    """Many short packed documents, lengths 1 .. 40 drawn from a seed: 1,024
    (the most the quantiser keeps its document table for in shared memory) and
    3,000 (the table built in the workspace by one extra launch); codes and
    scales bit-exact, the forward against the emulation."""
    lengths = np.random.default_rng(ndocs + wid).integers(1, 41, size=ndocs).tolist()
    inp = workloads.make(wid, heads=2, lengths=lengths)
    exact = block == 1
    o, lse = run_gpu(inp, mx, block, causal, exact)
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    ws = pa.workspace(T, H, d, cu.numel() - 1)
    if not mx:   # the quantiser against the oracle's on the same packed batch
        qt = pa.attn_quantize(q, cu, pa.ATTN_E4M3_TOKBLOCK, block, True, 0x5EED0000 + wid, ws=ws)
        codes, scales, _ = oracle_mod.quantize(inp.q, inp.cu_seqlens, 0, block, True, 0x5EED0000 + wid)
        assert np.array_equal(qt.codes.cpu().numpy(), codes)
        assert np.array_equal(qt.scales.cpu().numpy()[:, :scales.shape[1]].view(np.uint32), scales.view(np.uint32))
    _, ob, le, amb = run_emu(inp, mx, block, causal, exact)
    res = compare_outputs(o, lse, ob, le, ties=amb)
    assert res["ok"], res


@pytest.mark.parametrize("block", [128, 1])
def test_valid_forward_after_bad_seqlens_on_same_workspace(oracle_mod, block):
    """A quantise call with malformed cu_seqlens leaves ATTN_ERR_BAD_SEQLENS in
    the workspace's status word; a later, valid forward on the same workspace
    (the status not read in between) must still compute its own schedule and V
    references, and match the emulation."""
    causal = block == 1
    inp = workloads.make(3, heads=2, lengths=[300, 77, 129])
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    ws = pa.workspace(T, H, d, cu.numel() - 1)
    bad = cu.clone()
    bad[1], bad[2] = bad[2].clone(), bad[1].clone()            # offsets out of order
    pa.attn_quantize(q, bad, pa.ATTN_E4M3_TOKBLOCK, block, True, 0x5EED0003, ws=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) & (1 << pa.ATTN_ERR_BAD_SEQLENS)
    seed = 0x5EED0003
    Q = pa.attn_quantize(q, cu, pa.ATTN_E4M3_TOKBLOCK, block, True, seed, ws=ws)
    K = pa.attn_quantize(k, cu, pa.ATTN_E4M3_TOKBLOCK, block, True, seed, ws=ws)
    V = pa.attn_quantize(v, cu, pa.ATTN_E4M3_TOKBLOCK, block, False, 0, ws=ws)
    o, lse = pa.attn_fp8_fwd(Q, K, V, cu, causal, causal, 0.0, ws=ws)
    torch.cuda.synchronize()
    _, ob, le, amb = run_emu(inp, False, block, causal, exact=causal)
    res = compare_outputs(o, lse, ob, le, ties=amb)
    assert res["ok"], res
    st, flags = pa.attn_read_device_status(ws)
    assert st == pa.ATTN_ERR_BAD_SEQLENS and flags == (1 << pa.ATTN_ERR_BAD_SEQLENS)


@pytest.mark.parametrize("causal", [False, True])
def test_nvfp4_empty_and_many_documents(oracle_mod, causal):
    """The mixed NVFP4/FP8 path on zero-length documents inside the batch and on
    1,500 documents of 1 .. 40 tokens: every device probability code checked
    against the emulation, the output under the plain bounds."""
    from test_gpu_ties import check_given_codes
    wid = 3 if causal else 2
    check_given_codes(workloads.make(wid, heads=2, lengths=EMPTY_DOCS), False, 128, causal, nv=True)
    lengths = np.random.default_rng(77 + wid).integers(1, 41, size=1500).tolist()
    check_given_codes(workloads.make(wid, heads=2, lengths=lengths), False, 128, causal, nv=True)


@pytest.mark.parametrize("causal", [False, True])
def test_nvfp4_all_zero_inputs_closed_form(causal):
    """Q = K = V = 0 through NVFP4 Q, K: zero block scales and codes, every score 0:
    O = 0 exactly and lse = ln(visible keys)."""
    inp = workloads.make(2, heads=2, lengths=[200, 77, 129])
    q, k, v, cu = to_device(inp)
    q.zero_()
    k.zero_()
    v.zero_()
    T, H, d = q.shape
    ws = pa.workspace(T, H, d, cu.numel() - 1)
    Q = pa.attn_quantize(q, cu, pa.ATTN_NVFP4, 128, True, 5, ws=ws)
    K = pa.attn_quantize(k, cu, pa.ATTN_NVFP4, 128, True, 5, ws=ws)
    V = pa.attn_quantize(v, cu, pa.ATTN_E4M3_TOKBLOCK, 128, False, 0, ws=ws)
    o, lse = pa.attn_fp8_fwd(Q, K, V, cu, causal, False, 0.0, ws=ws)
    st, _ = pa.attn_read_device_status(ws)
    assert st == 0
    assert int(torch.count_nonzero(o.float())) == 0
    want = np.log(visible_keys(inp.cu_seqlens, causal))
    assert np.abs(lse.double().cpu().numpy() - want[None, :]).max() <= 1e-5 * np.maximum(1.0, want).max()
