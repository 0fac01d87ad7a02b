"""Where several results are correct, check the one the device chose.

A probability within fp32 rounding of an E4M3 rounding boundary has two
faithful codes: the device forms each score in its own fp32 summation order
and takes 2^x with an fp32 approximation, the oracle's emulation sums in fp64
and rounds once. The test build of the library (include/attn_pdump.h) reports
every probability code the FP8 kernels hand to the P V product; here each one
is checked against the emulation key by key -- it must be the emulation's own
code, or, where the emulation's probability lies inside its tie band, the
code on the other side of that boundary; keys a row does not see must hold 0
-- and the output is then compared with the emulation recomputed from the
device's codes under the plain bounds, with no tie allowance: relative RMSE
<= 1e-3, per element |diff| <= max(2e-3, one BF16 ulp), lse within 1e-3.
The same check covers the bit-level exponentials (Schraudolph's form and the
log-domain P codes), whose emulation mirrors the codes they define.

Sources: "Fused attention kernel", Implementation sketch (the running softmax)
and 8-bit forward pass (P cast to e4m3 before the P V product);
"FP8 attention that keeps FlashAttention-3 throughput at BF16-level accuracy",
How it gets verified.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import compare_outputs, to_device

pa = pytest.importorskip("precision_attention_gb300")

pytestmark = pytest.mark.gpu

E4M3, ROW, COL = 0, 1, 2


def quantise_both(inp, mx, block, rotate=True, nv=False):
    seed = 0x5EED0000 + inp.wid
    q, k, v, cu = to_device(inp)
    T, H, d = q.shape
    ws = pa.workspace(T, H, d, cu.numel() - 1)
    ocu = inp.cu_seqlens
    if nv:    # mixed NVFP4 / FP8: NVFP4 Q, K; E4M3 V in 128-token blocks
        lay = (pa.ATTN_NVFP4, pa.ATTN_NVFP4, E4M3)
        blk = 128
    elif mx:
        lay = (ROW, ROW, pa.ATTN_MX_TOKEN if block == 1 else COL)
        blk = 32
    else:
        lay = (E4M3, E4M3, E4M3)
        blk = block
    rot = (rotate, rotate, False)
    sd = (seed, seed, 0)
    G = [pa.attn_quantize(x, cu, L, blk, r, s_, ws=ws) for x, L, r, s_ in zip((q, k, v), lay, rot, sd)]
    olay = tuple(oracle.MX_TOKEN if L == pa.ATTN_MX_TOKEN else oracle.NVFP4 if L == pa.ATTN_NVFP4 else L
                 for L in lay)
    O = [oracle.quantize_tensor(x, ocu, L, blk, r, s_) for x, L, r, s_ in zip((inp.q, inp.k, inp.v), olay, rot, sd)]
    for g_, o_ in zip(G, O):
        assert np.array_equal(g_.codes.cpu().numpy(), o_.codes)
    return G, O, cu


def key_stride(cu):
    L = int(np.max(np.diff(np.asarray(cu))))
    return max(128, (L + 127) // 128 * 128)


def check_given_codes(inp, mx, block, causal, exact=False, rows=None, exp_mode=0, nv=False):
    (Q, K, V), (Qo, Ko, Vo), cu = quantise_both(inp, mx, block, nv=nv)
    o_ref, l_ref = pa.attn_fp8_fwd_ex(Q, K, V, cu, causal, exact, 0.0, exp_mode)
    ks = key_stride(inp.cu_seqlens)
    o, lse, codes = pa.attn_fp8_fwd_pdump(Q, K, V, cu, ks, causal, exact, exp_mode=exp_mode)
    torch.cuda.synchronize()
    # the test build computes the same output bit for bit
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)) and torch.equal(lse, l_ref)
    _, ob, le, counts = oracle.attention_emulate_given_p(Qo, Ko, Vo, codes.cpu().numpy(), inp.cu_seqlens, causal,
                                                         exact, None, rows=rows,
                                                         rescale_tau=pa.rescale_threshold(inp.q.shape[2]),
                                                         exp_mode=exp_mode)
    assert counts["wrong"] == 0 and counts["masked_nonzero"] == 0, counts
    res = compare_outputs(o, lse, ob, le, rows=rows)
    assert res["ok"], (res, counts)
    return res, counts


CASES = [
    # wid, lengths, heads, mx, block, causal, exact
    (1, [256], 2, False, 64, False, False),          # d = 64 (one-tile kernel), fp32 input
    (1, [200, 56, 129], 2, False, 64, True, False),
    (2, [300, 77, 129], 2, False, 128, False, False),
    (3, [300, 77, 129], 2, False, 128, True, False),
    (3, [260, 31], 2, False, 1, True, True),         # causal-exact
    (2, [384], 2, False, 32, False, False),          # per-key scales
    (4, [300, 77, 129], 2, True, 32, False, False),  # MXFP8
    (5, [300, 77, 129, 1], 2, True, 32, True, False),
    (5, [300, 77, 129, 1], 2, True, 1, True, True),  # MXFP8 causal-exact
]


@pytest.mark.parametrize("wid,lengths,H,mx,block,causal,exact", CASES)
def test_device_codes_are_faithful_and_output_meets_plain_bounds(oracle_mod, wid, lengths, H, mx, block, causal,
                                                                 exact):
    inp = workloads.make(wid, heads=H, lengths=lengths)
    check_given_codes(inp, mx, block, causal, exact)


@pytest.mark.parametrize("wid,mx,causal,exact", [(2, False, False, False), (3, False, True, False),
                                                  (3, False, True, True), (4, True, False, False),
                                                  (5, True, True, False), (5, True, True, True)])
def test_long_documents_with_causal_first_rows(oracle_mod, wid, mx, causal, exact):
    """Two 2,048-token documents, four heads: many items per CTA; rows: the
    first 160 of each document (causal rows that see one to a few keys, where a
    single tied code moves the whole row), tile edges and seeded random rows."""
    inp = workloads.make(wid, heads=4, lengths=[2048, 2048])
    rng = np.random.default_rng(100 + wid)
    T = inp.T
    rows = np.unique(np.concatenate([np.arange(0, 160), np.arange(2048, 2208), np.array([127, 128, 2047, T - 1]),
                                     rng.choice(T, 160, replace=False)])).astype(np.int32)
    block = (1 if exact else 32) if mx else (1 if exact else 128)
    check_given_codes(inp, mx, block, causal, exact, rows=rows)


# the bit-level exponentials (FLAMIA sections 1, 4.3, 4.4): Schraudolph's fp32
# form and the log-domain P codes, on the E4M3 tile and MX paths
BITEXP_CASES = [
    (2, [300, 77, 129], False, 128, False),
    (3, [300, 77, 129], False, 128, True),
    (4, [300, 77, 129], True, 32, False),
    (5, [300, 77, 129, 1], True, 32, True),
]


@pytest.mark.parametrize("exp_mode", [1, 2], ids=["schraudolph", "mitchell_p"])
@pytest.mark.parametrize("wid,lengths,mx,block,causal", BITEXP_CASES)
def test_bit_level_exponentials_codes_and_output(oracle_mod, wid, lengths, mx, block, causal, exp_mode):
    inp = workloads.make(wid, heads=2, lengths=lengths)
    res, counts = check_given_codes(inp, mx, block, causal, exp_mode=exp_mode)
    assert counts["same"] > 0.99 * (counts["same"] + counts["tie_other"])


@pytest.mark.parametrize("exp_mode", [1, 2], ids=["schraudolph", "mitchell_p"])
@pytest.mark.parametrize("wid,mx,causal", [(2, False, False), (5, True, True)])
def test_bit_level_exponentials_long_documents(oracle_mod, wid, mx, causal, exp_mode):
    inp = workloads.make(wid, heads=4, lengths=[2048, 2048])
    rng = np.random.default_rng(200 + wid)
    T = inp.T
    rows = np.unique(np.concatenate([np.arange(0, 96), np.arange(2048, 2144), np.array([127, 128, 2047, T - 1]),
                                     rng.choice(T, 160, replace=False)])).astype(np.int32)
    check_given_codes(inp, mx, 32 if mx else 128, causal, rows=rows, exp_mode=exp_mode)


# mixed NVFP4 / FP8 (FLAMIA sections 1 and 2): S from NVFP4 Q and K through the
# block-scaled FP4 MMA, P V in E4M3
NV_CASES = [
    (2, [300, 77, 129], False, 0),
    (3, [300, 77, 129], True, 0),
    (4, [256, 1, 130], False, 0),
    (5, [300, 77, 129, 1], True, 0),
    (2, [300, 77, 129], False, 1),     # with Schraudolph's exponential
    (3, [300, 77, 129], True, 2),      # with log-domain P (Mitchell-P over NVFP4)
]


@pytest.mark.parametrize("wid,lengths,causal,exp_mode", NV_CASES)
def test_nvfp4_qk_codes_and_output(oracle_mod, wid, lengths, causal, exp_mode):
    inp = workloads.make(wid, heads=2, lengths=lengths)
    check_given_codes(inp, False, 128, causal, exp_mode=exp_mode, nv=True)


@pytest.mark.parametrize("wid,causal", [(2, False), (3, True)])
def test_nvfp4_qk_long_documents(oracle_mod, wid, causal):
    inp = workloads.make(wid, heads=4, lengths=[2048, 2048])
    rng = np.random.default_rng(300 + wid)
    T = inp.T
    rows = np.unique(np.concatenate([np.arange(0, 96), np.arange(2048, 2144), np.array([127, 128, 2047, T - 1]),
                                     rng.choice(T, 160, replace=False)])).astype(np.int32)
    check_given_codes(inp, False, 128, causal, rows=rows, nv=True)
