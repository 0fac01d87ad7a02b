"""Failure detection on the GPU without a fault: with a bounded-wait limit far
shorter than a tile's copy, the forward gives up, lets what is in flight
finish, frees what it holds and reports ATTN_ERR_DEVICE_TIMEOUT in the status
word; the context stays usable and the next call is correct. (The quantiser
waits only for its own tile copies, each of which lands within one
mbarrier.try_wait, so no limit makes it time out; its wait is the same bounded
loop.)"""
import pytest

import workloads
from gpu_helpers import compare_outputs, to_device
from test_gpu_attention import run_emu, run_gpu

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wid,mx,block,causal", [(2, False, 128, False), (5, True, 32, True), (1, False, 64, False)])
def test_wait_runs_out_then_context_usable(oracle_mod, wid, mx, block, causal):
    inp = workloads.make(wid, heads=2, lengths=[512, 200])
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    ws = pa.workspace(T, H, d, cu.numel() - 1)
    seed = 0x5EED0000 + wid
    if mx:
        Q = pa.attn_quantize(q, cu, 1, 32, True, seed, ws=ws)
        K = pa.attn_quantize(k, cu, 1, 32, True, seed, ws=ws)
        V = pa.attn_quantize(v, cu, 2, 32, False, 0, ws=ws)
    else:
        Q = pa.attn_quantize(q, cu, 0, block, True, seed, ws=ws)
        K = pa.attn_quantize(k, cu, 0, block, True, seed, ws=ws)
        V = pa.attn_quantize(v, cu, 0, block, False, 0, ws=ws)
    assert pa.attn_read_device_status(ws)[0] == pa.ATTN_OK
    try:
        pa.attn_set_wait_limit(100)   # SM cycles: no copy or MMA completes that fast
        pa.attn_fp8_fwd(Q, K, V, cu, causal, False, 0.0, ws=ws)
        st, flags = pa.attn_read_device_status(ws)
    finally:
        pa.attn_set_wait_limit(0)
    assert st == pa.ATTN_ERR_DEVICE_TIMEOUT, (st, flags)
    # the same context, default limit: a correct forward
    o, lse = run_gpu(inp, mx, block, causal)
    _, ob, le, amb = run_emu(inp, mx, block, causal)
    res = compare_outputs(o, lse, ob, le, ties=amb)
    assert res["ok"], res
