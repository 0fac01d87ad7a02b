"""BF16 attention backward (attn_bf16_bwd) against the oracle's FP64 gradients.

The gradients are the plain derivative of the forward's definition ("Fused
attention kernel", Overview; FLAMIA section 1: the training call's backward
over the same document-local token blocks; section 4.5: the causal case).
The oracle's FP64 backward is pinned on its own by finite differences and
closed forms (test_oracle_backward.py).

Tolerances, from the arithmetic. Q, K, V and dO are bf16 values, exact in the
oracle's fp64. The kernel rounds P and dS to bf16 as MMA operands and rounds
its outputs to bf16 (unit roundoff u = 2^-8; a relative error of RMS
u / sqrt(3) = 2.3e-3 for values spread over a binade), and accumulates in fp32.
It takes D = rowsum(dO o O) from the forward's stored bf16 O, as its contract
says; in a row whose softmax is nearly one-hot, dP - D nearly cancels, and O's
rounding then leaves an absolute error of about scale x 2.3e-3 |dO| |V| in dQ
and dK that no relative bound on that row can hold.
  1. Against the exact FP64 gradients: relative RMSE <= 1e-2 per tensor (the
     expected 2.3e-3 to 3e-3, a margin of three; a missed term -- the scale,
     D, a mask, a transposed operand -- moves it by O(1)).
  2. Against the oracle's gradients with D from the same stored O: every
     (token, head) row within 2e-2 of its own norm plus 1e-2 of the tensor's
     RMS (rows measure 2e-3 to 6e-3 relative). This catches errors confined to
     a few rows, such as a wrong causal diagonal or a document boundary, that
     an RMSE over the whole tensor would dilute.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import to_device

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu

REL_RMSE = 1e-2
ROW_REL = 2e-2
ROW_ABS_OF_RMS = 1e-2


def _make(wid, heads, lengths):
    """Seeded inputs of workload `wid` as bf16 values (workload 1, head_dim 64, is
    fp32 in the forward's tests; the backward takes bf16)."""
    inp = workloads.make(wid, heads=heads, lengths=lengths)
    if inp.in_dtype != "bf16":
        inp = dataclasses.replace(inp, q=workloads.bf16_round(inp.q), k=workloads.bf16_round(inp.k),
                                  v=workloads.bf16_round(inp.v), in_dtype="bf16")
    return inp


def _dout(T, H, d, seed=77):
    return workloads.bf16_round(workloads.draw((T, H, d), "normal", seed))


def _run(inp, causal, dout_np, scale=0.0, o_lse=None):
    """The GPU gradients and the bf16 O they used, as fp64 numpy arrays."""
    q, k, v, cu = to_device(inp)
    do = torch.from_numpy(dout_np).to(torch.bfloat16).cuda()
    T, H, d = q.shape
    nd = cu.numel() - 1
    if o_lse is None:
        o, lse = pa.attn_bf16_fwd(q, k, v, cu, causal, scale)
    else:
        o, lse = o_lse
    ws = pa.bwd_workspace(T, H, d, nd)
    dq, dk, dv = pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, causal, scale, ws=ws)
    st, flags = pa.attn_read_device_status(ws)
    assert st == 0, (st, flags)
    grads = [x.float().cpu().numpy().astype(np.float64) for x in (dq, dk, dv)]
    return grads, o.float().cpu().numpy().astype(np.float64)


def _check_all(inp, do, causal, scale, got, o_used):
    sc = None if scale <= 0 else scale
    exact = oracle.attention_fp64_backward(inp.q, inp.k, inp.v, do, inp.cu_seqlens, causal, sc)
    stored = oracle.attention_fp64_backward(inp.q, inp.k, inp.v, do, inp.cu_seqlens, causal, sc, o=o_used)
    for name, g, r, rs in zip(("dq", "dk", "dv"), got, exact, stored):
        assert np.isfinite(g).all(), name
        e = g - r
        rms = float(np.sqrt(np.mean(r * r)))
        rel = float(np.sqrt(np.mean(e * e))) / rms
        assert rel <= REL_RMSE, f"{name}: relative RMSE {rel:.3e} > {REL_RMSE}"
        es = g - rs
        row_err = np.sqrt(np.sum(es * es, axis=2))
        row_ref = np.sqrt(np.sum(rs * rs, axis=2))
        bound = ROW_REL * row_ref + ROW_ABS_OF_RMS * rms * np.sqrt(g.shape[2])
        worst = float(np.max(row_err / bound))
        assert worst <= 1.0, f"{name}: row error {worst:.2f} x its bound at {np.unravel_index(np.argmax(row_err / bound), row_err.shape)}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("wid,lengths", [(2, [700, 129, 1000]), (2, [1, 128, 129, 255]),
                                         (1, [700, 129, 1000]), (1, [1, 64, 65, 255])])
def test_backward_against_fp64(causal, wid, lengths):
    """The chain a caller runs: attn_bf16_fwd, then attn_bf16_bwd on its o and lse
    (head_dim 128: workload 2's normal inputs; head_dim 64: workload 1's)."""
    inp = _make(wid, 2, lengths)
    T, H, d = inp.q.shape
    do = _dout(T, H, d)
    got, o_used = _run(inp, causal, do)
    _check_all(inp, do, causal, 0.0, got, o_used)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_on_oracle_forward(causal):
    """The backward alone: o and lse from the oracle's FP64 forward (o rounded to
    bf16, lse to fp32), with a softmax scale other than 1/sqrt(d)."""
    inp = workloads.make(2, heads=3, lengths=[300, 77, 513])
    T, H, d = inp.q.shape
    do = _dout(T, H, d, seed=78)
    scale = 0.05
    o64, lse64 = oracle.attention_fp64(inp.q, inp.k, inp.v, inp.cu_seqlens, causal, scale)
    o = torch.from_numpy(o64.astype(np.float32)).to(torch.bfloat16).cuda()
    lse = torch.from_numpy(np.ascontiguousarray(lse64.astype(np.float32))).cuda()
    got, o_used = _run(inp, causal, do, scale, (o, lse))
    _check_all(inp, do, causal, scale, got, o_used)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("wid", [2, 1])
def test_backward_deterministic_and_packed_equals_documents(causal, wid):
    """Two calls give the same bits; each document of a packed batch gets the
    bits it gets alone (every tile is document-local, every sum has one order)."""
    lengths = [300, 0, 77, 129]
    inp = _make(wid, 2, lengths)
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    do = torch.from_numpy(_dout(T, H, d)).to(torch.bfloat16).cuda()
    o, lse = pa.attn_bf16_fwd(q, k, v, cu, causal)
    a = pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, causal)
    b = pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, causal)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    bounds = np.concatenate([[0], np.cumsum(lengths)])
    for i in range(len(lengths)):
        s, e = int(bounds[i]), int(bounds[i + 1])
        if e == s:
            continue
        sl = lambda x: x[s:e].contiguous()
        one = pa.attn_bf16_bwd(sl(q), sl(k), sl(v), sl(o), sl(do), lse[:, s:e].contiguous(), None, causal)
        for x, y in zip(a, one):
            assert torch.equal(x[s:e].view(torch.int16), y.view(torch.int16)), i


def test_backward_sum_rules_at_full_length():
    """Properties that hold at any size (softmax rows sum to one; a shift shared
    by every key of a document leaves its softmax unchanged): per document and
    head the dV rows sum to the dO rows and the dK rows sum to zero. Checked on
    one 8192-token causal document with 32 heads, the headline length."""
    lengths = [8192]
    inp = workloads.make(3, heads=32, lengths=lengths)
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    do_np = _dout(T, H, d, seed=79)
    do = torch.from_numpy(do_np).to(torch.bfloat16).cuda()
    o, lse = pa.attn_bf16_fwd(q, k, v, cu, True)
    dq, dk, dv = pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, True)
    # a correct kernel leaves each row with an independent rounding error of about
    # 4e-3 of its size, so a column sum misses its exact value by about 4e-3 of the
    # column's l2 norm; a missing term (D, a mask) leaves O(1) of it
    dv64, dk64 = dv.double(), dk.double()
    dv_err = np.abs(dv64.sum(0).cpu().numpy() - do_np.astype(np.float64).sum(0))
    dk_err = np.abs(dk64.sum(0).cpu().numpy())
    dv_l2 = dv64.square().sum(0).sqrt().cpu().numpy()
    dk_l2 = dk64.square().sum(0).sqrt().cpu().numpy()
    assert np.all(dv_err <= 0.05 * dv_l2), float(np.max(dv_err / dv_l2))
    assert np.all(dk_err <= 0.05 * dk_l2), float(np.max(dk_err / dk_l2))
    assert torch.isfinite(dq.float()).all()


def test_backward_malformed_seqlens_writes_status():
    T, H, d = 256, 2, 128
    q, k, v, o, do = (torch.randn(T, H, d, device="cuda").to(torch.bfloat16) for _ in range(5))
    lse = torch.zeros(H, T, device="cuda")
    cu = torch.tensor([0, 200, 100, 256], dtype=torch.int32, device="cuda")
    ws = pa.bwd_workspace(T, H, d, 3)
    pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, False, ws=ws)
    assert pa.attn_read_device_status(ws)[0] == pa.ATTN_ERR_BAD_SEQLENS


def test_backward_short_wait_limit_then_context_usable():
    """Failure detection without a fault: under a 100-cycle wait limit the
    gradient kernel either completes or gives up with ATTN_ERR_DEVICE_TIMEOUT
    (letting its copies and MMAs finish and freeing TMEM first); either way the
    next call in the same context, default limit, gives the bits of a clean call.
    Each bounded wait starts with mbarrier.try_wait, which suspends until the
    phase completes or a hardware window passes, so a limit is reached only by a
    wait longer than two such windows; the backward's steps are shorter, and the
    forward's failure test (test_gpu_failure.py) is the one whose wait runs out."""
    inp = workloads.make(2, heads=2, lengths=[300, 77, 129])
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    do = torch.from_numpy(_dout(T, H, d)).to(torch.bfloat16).cuda()
    o, lse = pa.attn_bf16_fwd(q, k, v, cu, True)
    clean = pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, True)
    ws = pa.bwd_workspace(T, H, d, 3)
    try:
        pa.attn_set_wait_limit(100)   # SM cycles: no copy or MMA completes that fast
        pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, True, ws=ws)
        st, flags = pa.attn_read_device_status(ws)
    finally:
        pa.attn_set_wait_limit(0)
    assert st in (pa.ATTN_OK, pa.ATTN_ERR_DEVICE_TIMEOUT), (st, flags)
    again = pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, True, ws=ws)
    assert pa.attn_read_device_status(ws)[0] == 0
    for a, b in zip(clean, again):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_backward_many_small_documents():
    """About a thousand documents of 1 to 12 tokens (one partial tile each, the
    prep kernel's document search over a long table), causal, against FP64."""
    lens = workloads.doc_lengths(6000, 1, 12, seed=21)
    assert len(lens) > 800
    inp = workloads.make(2, heads=2, lengths=list(lens))
    T, H, d = inp.q.shape
    do = _dout(T, H, d, seed=80)
    got, o_used = _run(inp, True, do)
    _check_all(inp, do, True, 0.0, got, o_used)
