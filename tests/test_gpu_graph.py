"""The whole forward captured in a CUDA graph (FLAMIA appendix F: scales and work
lists stay on the GPU, no host synchronisation, graph capture, replay bitwise
equal to eager). The quantiser launch and the forward's work-list, V-reference
and attention kernels (the last three launched as programmatic dependents)
are captured on one stream; replays on new inputs copied into the captured
buffers give O and lse bit for bit equal to eager calls on the same inputs,
under the static and the ticket work order.
"""
import pytest
import torch

import workloads
from gpu_helpers import to_device

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu

E4M3, ROW, COL, NV = 0, 1, 2, 4


def _forward(q, k, v, cu, outs, o, lse, ws, layouts, causal, seed, stream=None):
    lq, blk, lv = layouts
    Q, K, V = pa.attn_quantize_qkv(q, k, v, cu, lq, blk, lv, blk, True, seed, ws=ws, outs=outs, stream=stream)
    pa.attn_fp8_fwd(Q, K, V, cu, causal, False, 0.0, ws=ws, out=o, lse=lse, stream=stream)


@pytest.mark.parametrize("schedule", [0, 1])   # static rounds; tickets (the counter restarts with every replay)
@pytest.mark.parametrize("wid,layouts,causal", [
    (2, (E4M3, 128, E4M3), False),   # E4M3 tile scales (with the V-reference pass)
    (3, (E4M3, 128, E4M3), True),
    (4, (ROW, 32, COL), False),      # MXFP8 (no V-reference pass)
    (2, (NV, 128, E4M3), True),      # NVFP4 Q K^T
])
def test_forward_graph_replay_bitwise(wid, layouts, causal, schedule):
    pa.attn_set_schedule(schedule)
    try:
        _graph_replay(wid, layouts, causal)
    finally:
        pa.attn_set_schedule(pa.ATTN_SCHED_STATIC)


def _graph_replay(wid, layouts, causal):
    lengths = [700, 129, 1000]
    inp = workloads.make(wid, heads=4, lengths=lengths)
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    nd = cu.numel() - 1
    seed = 0x5EED0077
    lq, blk, lv = layouts
    ws = pa.workspace(T, H, d, nd)
    outs = (pa.empty_qtensor(T, H, d, nd, lq, blk), pa.empty_qtensor(T, H, d, nd, lq, blk),
            pa.empty_qtensor(T, H, d, nd, lv, blk))
    o = torch.empty((T, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((H, T), dtype=torch.float32, device="cuda")
    qb, kb, vb = (x.clone() for x in (q, k, v))     # the graph's input buffers

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _forward(qb, kb, vb, cu, outs, o, lse, ws, layouts, causal, seed, stream=s)   # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _forward(qb, kb, vb, cu, outs, o, lse, ws, layouts, causal, seed, stream=s)
    torch.cuda.synchronize()

    gen = torch.Generator(device="cuda").manual_seed(11)
    for rep in range(3):
        # new inputs each replay (the first replay reuses the warm-up's)
        if rep:
            for b in (qb, kb, vb):
                b.copy_(torch.randn(b.shape, device="cuda", generator=gen).to(b.dtype) * (1 + rep))
        g.replay()
        torch.cuda.synchronize()
        st, flags = pa.attn_read_device_status(ws)
        assert st == 0, (st, flags)
        o_g, lse_g = o.clone(), lse.clone()
        ws2 = pa.workspace(T, H, d, nd)
        o_e = torch.empty_like(o)
        lse_e = torch.empty_like(lse)
        outs_e = (pa.empty_qtensor(T, H, d, nd, lq, blk), pa.empty_qtensor(T, H, d, nd, lq, blk),
                  pa.empty_qtensor(T, H, d, nd, lv, blk))
        _forward(qb, kb, vb, cu, outs_e, o_e, lse_e, ws2, layouts, causal, seed)
        torch.cuda.synchronize()
        assert torch.equal(o_g.view(torch.int16), o_e.view(torch.int16)), rep
        assert torch.equal(lse_g.view(torch.int32), lse_e.view(torch.int32)), rep
        assert torch.isfinite(o_g.float()).all()


@pytest.mark.parametrize("causal", [False, True])
def test_backward_graph_replay_bitwise(causal):
    """The BF16 forward and backward (work list, per-row vectors, gradient kernel)
    captured in one graph; replays on new inputs equal eager calls bit for bit."""
    lengths = [700, 129, 1000]
    inp = workloads.make(2, heads=2, lengths=lengths)
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    nd = cu.numel() - 1
    qb, kb, vb = (x.clone() for x in (q, k, v))
    dob = torch.randn_like(qb)
    o = torch.empty_like(qb)
    lse = torch.empty((H, T), dtype=torch.float32, device="cuda")
    outs = tuple(torch.empty_like(qb) for _ in range(3))
    wsf = pa.workspace(T, H, d, nd)
    wsb = pa.bwd_workspace(T, H, d, nd)

    def run(stream=None):
        pa.attn_bf16_fwd(qb, kb, vb, cu, causal, ws=wsf, out=o, lse=lse, stream=stream)
        pa.attn_bf16_bwd(qb, kb, vb, o, dob, lse, cu, causal, ws=wsb, outs=outs, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run(s)
    torch.cuda.synchronize()
    gen = torch.Generator(device="cuda").manual_seed(5)
    for rep in range(2):
        for b in (qb, kb, vb, dob):
            b.copy_(torch.randn(b.shape, device="cuda", generator=gen).to(b.dtype))
        g.replay()
        torch.cuda.synchronize()
        assert pa.attn_read_device_status(wsb)[0] == 0
        got = [x.clone() for x in outs]
        oe, le = pa.attn_bf16_fwd(qb, kb, vb, cu, causal)
        eager = pa.attn_bf16_bwd(qb, kb, vb, oe, dob, le, cu, causal)
        torch.cuda.synchronize()
        for a, b in zip(got, eager):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), rep
