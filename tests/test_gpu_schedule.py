"""The just-in-time (ticket) work order of the pair kernel against the static
longest-first rounds (FLAMIA section 4.3: just-in-time work acquisition). Only
which CTA computes which item changes, so O and lse must be bitwise equal, with
several items per CTA so that the tickets past the first round are taken from
the counter, on every pair-kernel mode, causal and not, packed documents
included."""
import pytest
import torch

import workloads
from gpu_helpers import to_device

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu

E4M3, ROW, COL, TOK, NV = 0, 1, 2, 3, 4


def _run(inp, layouts, causal, exact, schedule):
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    nd = cu.numel() - 1
    lq, bq, lv, bv = layouts
    ws = pa.workspace(T, H, d, nd)
    Q = pa.attn_quantize(q, cu, lq, bq, True, 0x5EED0101, ws=ws)
    K = pa.attn_quantize(k, cu, lq, bq, True, 0x5EED0101, ws=ws)
    V = pa.attn_quantize(v, cu, lv, bv, False, 0, ws=ws)
    pa.attn_set_schedule(schedule)
    try:
        o, lse = pa.attn_fp8_fwd(Q, K, V, cu, causal, exact, 0.0, ws=ws)
        torch.cuda.synchronize()
    finally:
        pa.attn_set_schedule(pa.ATTN_SCHED_STATIC)
    st, flags = pa.attn_read_device_status(ws)
    assert st == 0, (st, flags)
    return o, lse


@pytest.mark.parametrize("wid,lengths,H,layouts,causal,exact", [
    (2, [4096, 4096], 16, (E4M3, 128, E4M3, 128), False, False),   # 256 items on 148-152 CTAs
    (3, [4096, 2000, 3000], 16, (E4M3, 128, E4M3, 128), True, False),
    (3, [3000, 2500], 8, (E4M3, 1, E4M3, 1), True, True),          # per-column scales, causal-exact
    (4, [4224, 4224], 8, (ROW, 32, COL, 32), False, False),         # MXFP8
    (5, [5000, 300, 129, 2600], 16, (ROW, 32, TOK, 1), True, True), # MX causal-exact, packed
    (2, [4096, 3000], 16, (NV, 128, E4M3, 128), True, False),       # NVFP4 Q K^T
])
def test_ticket_schedule_equals_static(wid, lengths, H, layouts, causal, exact):
    inp = workloads.make(wid, heads=H, lengths=lengths)
    o0, l0 = _run(inp, layouts, causal, exact, pa.ATTN_SCHED_STATIC)
    o1, l1 = _run(inp, layouts, causal, exact, pa.ATTN_SCHED_TICKET)
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0.view(torch.int32), l1.view(torch.int32))
    # and a second ticket run (the counter restarts with every call)
    o2, l2 = _run(inp, layouts, causal, exact, pa.ATTN_SCHED_TICKET)
    assert torch.equal(o2.view(torch.int16), o0.view(torch.int16))
