"""attn_fp8_fwd_noalloc: the forward for callers that cannot allocate device
memory (its scratch is the library's fixed 16 MiB device array instead of a
caller workspace). Checked through the C ABI against attn_fp8_fwd on two calls
in a row with different shapes and layouts, so that the second call also shows
that what the first left in the shared array does not leak into its result.

Collected last on purpose: a run that stops at the first failure has run every
other test before this one.
"""
import numpy as np
import pytest
import torch

import oracle  # noqa: F401  (keeps the import order of the other GPU tests)
import workloads
from gpu_helpers import TOL_LSE, TOL_MAX_ABS, TOL_REL_RMSE, bf16_ulp, to_device

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu

E4M3, ROW, COL = 0, 1, 2


def quantised(inp, mx, block):
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    ws = pa.workspace(T, H, d, cu.numel() - 1)
    seed = 0x5EED0000 + inp.wid
    if mx:
        Q = pa.attn_quantize(q, cu, ROW, 32, True, seed, ws=ws)
        K = pa.attn_quantize(k, cu, ROW, 32, True, seed, ws=ws)
        V = pa.attn_quantize(v, cu, COL, 32, False, 0, ws=ws)
    else:
        Q = pa.attn_quantize(q, cu, E4M3, block, True, seed, ws=ws)
        K = pa.attn_quantize(k, cu, E4M3, block, True, seed, ws=ws)
        V = pa.attn_quantize(v, cu, E4M3, block, False, 0, ws=ws)
    return Q, K, V, cu, ws


def within_tolerance(o_a, l_a, o_b, l_b):
    a = o_a.float().cpu().numpy().astype(np.float64)
    b = o_b.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    worst = (np.abs(a - b) / np.maximum(TOL_MAX_ABS, bf16_ulp(b))).max()
    dl = np.abs(l_a.cpu().numpy() - l_b.cpu().numpy()).max()
    return rel <= TOL_REL_RMSE and worst <= 1.0 and dl <= TOL_LSE


def test_noalloc_forward_matches_workspace_forward_twice():
    cases = [
        (workloads.make(2, heads=2, lengths=[300, 77, 129]), False, 128, False),   # E4M3, non-causal
        (workloads.make(5, heads=3, lengths=[260, 31, 200]), True, 32, True),      # MXFP8, causal, packed
    ]
    for inp, mx, block, causal in cases:
        Q, K, V, cu, ws = quantised(inp, mx, block)
        o_ref, l_ref = pa.attn_fp8_fwd(Q, K, V, cu, causal, False, 0.0, ws=ws)
        st, _ = pa.attn_read_device_status(ws)
        assert st == pa.ATTN_OK
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        o, l = pa.attn_fp8_fwd_noalloc(Q, K, V, cu, causal, False, 0.0, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert within_tolerance(o, l, o_ref, l_ref)
        # the same kernels run on the same inputs: the results are in fact identical
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)) and torch.equal(l, l_ref)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    inp = workloads.make(2, heads=2, lengths=[256])
    Q, K, V, cu, ws = quantised(inp, False, 128)
    big = pa._Shape(1 << 21, 32, 128, 1, None)      # needs far more than 16 MiB of scratch
    cq, ck, cv = Q._c(), K._c(), V._c()
    o = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = pa.lib().attn_fp8_fwd_noalloc(*(pa.ctypes.byref(x) for x in (cq, ck, cv)), pa.ctypes.byref(big), 0, 0,
                                       0.0, o.data_ptr(), o.data_ptr(), None,
                                       torch.cuda.current_stream().cuda_stream)
    assert st == pa.ATTN_ERR_UNSUPPORTED
