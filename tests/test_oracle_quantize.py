"""Pins for the oracle's quantiser (O-2), CPU only.

The checks use what the pages and the formats fix: the scale rules' defining
properties, the E4M3 rounding error bound relative to a rotation computed with
a dense Hadamard matrix in fp64, document locality of every block, and cases
whose codes follow by hand from the format definition.
"""
import numpy as np
import pytest

import workloads
from test_oracle_formats import rotation_matrix

E4M3, ROW, COL = 0, 1, 2


def rotate_ref(oracle_mod, x, seed):
    d = x.shape[-1]
    return x.astype(np.float64) @ rotation_matrix(oracle_mod, d, seed).T


def e4m3_err_bound(y, unit):
    """|dequant - y| bound for E4M3 round-to-nearest of y/unit: half a mantissa
    step (2^-4 relative) in the normal range, half the subnormal step below."""
    return 2.0 ** -4 * np.abs(y) + 2.0 ** -10 * unit


def test_tokblock_codes_by_hand(oracle_mod):
    # one token, block 1, no rotation, amax = 448 -> inv = 1, scale = 1: codes are E4M3(x)
    vals = np.array([448, 224, 1, 0.5, 3, -2, 17, 19] + [0] * 24, dtype=np.float32)
    codes, sc, st = oracle_mod.quantize(vals.reshape(1, 1, 32), layout=E4M3, block=1)
    assert st == 0 and sc[0, 0] == 1.0
    assert list(codes.ravel()[:8]) == [0x7E, 0x76, 0x38, 0x30, 0x44, 0xC0, 0x58, 0x5A]
    assert not codes.ravel()[8:].any()


@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("block", [1, 64, 128])
def test_tokblock_scale_rule_and_error_bound(oracle_mod, rotate, block):
    lens = [100, 37, 300]
    cu = workloads.cu_from_lengths(lens)
    T, H, d = int(cu[-1]), 3, 64
    x = workloads.draw((T, H, d), "outlier", 11)
    seed = 0x1234
    codes, sc, st = oracle_mod.quantize(x, cu, E4M3, block, rotate, seed)
    assert st == 0
    y = rotate_ref(oracle_mod, x, seed) if rotate else x.astype(np.float64)
    # the fp32 transform (pinned against the dense matrix elsewhere) fixes the exact scales
    y32 = oracle_mod.rotate(x, seed) if rotate else x
    qt = oracle_mod.QTensor(codes, sc, E4M3, block, rotate, seed)
    deq = oracle_mod.dequantize(qt, cu)
    # blocks are document-local and start at the document start
    nb = 0
    for i in range(len(lens)):
        s, L = int(cu[i]), lens[i]
        for b in range(0, L, block):
            blk = y32[s + b:s + min(b + block, L)]
            for h in range(H):
                amax = np.float32(np.abs(blk[:, h, :]).max())
                assert sc[h, nb] == np.float32(amax / np.float32(448.0))
                # the block's largest element lands on +-448
                j = np.unravel_index(np.argmax(np.abs(blk[:, h, :])), blk[:, h, :].shape)
                assert codes[s + b + j[0], h, j[1]] & 0x7F == 0x7E
            nb += 1
    assert nb == oracle_mod.num_blocks(cu, T, block)
    # every element within the E4M3 rounding bound of the dense-rotated value
    fwht_err = (np.log2(d) * 2.0 ** -22 * np.abs(x).sum(-1, keepdims=True)) if rotate else 0.0
    # per-token block scale from the dequantised block bookkeeping
    scale_tok = np.zeros((T, H))
    off = 0
    for i in range(len(lens)):
        s, L = int(cu[i]), lens[i]
        for t in range(L):
            scale_tok[s + t] = sc[:, off + t // block]
        off += (L + block - 1) // block
    err = np.abs(deq - y)
    assert np.all(err <= e4m3_err_bound(y, scale_tok[:, :, None]) * (1 + 1e-6) + fwht_err + 1e-30)


def test_tokblock_document_locality(oracle_mod):
    lens = [130, 70]
    cu = workloads.cu_from_lengths(lens)
    x = workloads.draw((200, 2, 64), "normal", 3)
    c1, s1, _ = oracle_mod.quantize(x, cu, E4M3, 128, True, 9)
    x2 = x.copy()
    x2[130:] *= 50.0      # change only the second document
    c2, s2, _ = oracle_mod.quantize(x2, cu, E4M3, 128, True, 9)
    assert np.array_equal(c1[:130], c2[:130])
    assert np.array_equal(s1[:, :2], s2[:, :2])     # doc 0 has blocks [0,128) and [128,130)
    assert not np.array_equal(s1[:, 2], s2[:, 2])


def test_tokblock_zero_and_nonfinite(oracle_mod):
    x = np.zeros((4, 1, 32), dtype=np.float32)
    codes, sc, st = oracle_mod.quantize(x, None, E4M3, 4, False, 0)
    assert st == 0 and sc[0, 0] == 0.0 and not codes.any()
    x[2, 0, 5] = np.inf
    _, _, st = oracle_mod.quantize(x, None, E4M3, 4, False, 0)
    assert st == 5


@pytest.mark.parametrize("rotate", [False, True])
def test_mx_row32_rule_and_error_bound(oracle_mod, rotate):
    T, H, d = 50, 2, 128
    x = workloads.draw((T, H, d), "outlier_channels", 21, channels_seed=4)
    codes, su, st = oracle_mod.quantize(x, None, ROW, 32, rotate, 55)
    assert st == 0 and su.shape == (T, H, d // 32)
    y = rotate_ref(oracle_mod, x, 55) if rotate else x.astype(np.float64)
    X = su.astype(np.int64) - 127
    y32 = oracle_mod.rotate(x, 55) if rotate else x
    yg = y32.astype(np.float64).reshape(T, H, d // 32, 32)
    amax = np.abs(yg).max(-1)
    assert np.all(amax <= 448.0 * 2.0 ** X)                   # nothing saturates
    assert np.all(amax > 448.0 * 2.0 ** (X - 1))              # and X is the smallest such
    deq = oracle_mod.dequantize(oracle_mod.QTensor(codes, su, ROW, 32, rotate, 55))
    unit = np.repeat(2.0 ** X, 32, axis=2)
    fwht_err = (np.log2(d) * 2.0 ** -22 * np.abs(x).sum(-1, keepdims=True)) if rotate else 0.0
    assert np.all(np.abs(deq - y) <= e4m3_err_bound(y, unit) + fwht_err)


def test_mx_row32_codes_by_hand(oracle_mod):
    # amax 449 -> X = 1 (default) so 449 / 2 = 224.5 -> 224 (0x76); OCP X = 0 saturates to 448
    x = np.zeros((1, 1, 32), dtype=np.float32)
    x[0, 0, 0], x[0, 0, 1] = 449.0, 2.0
    c, s, _ = oracle_mod.quantize(x, None, ROW, 32, False, 0)
    assert s[0, 0, 0] == 128 and c[0, 0, 0] == 0x76 and c[0, 0, 1] == 0x38
    c, s, _ = oracle_mod.quantize(x, None, ROW, 32, False, 0, oracle_mod.MX_RULE_OCP_FLOOR)
    assert s[0, 0, 0] == 127 and c[0, 0, 0] == 0x7E and c[0, 0, 1] == 0x40
    z = np.zeros((1, 1, 32), dtype=np.float32)
    c, s, _ = oracle_mod.quantize(z, None, ROW, 32, False, 0)
    assert s[0, 0, 0] == 0 and not c.any()


def test_mx_col32_groups_along_tokens_doc_local(oracle_mod):
    lens = [45, 64, 20]
    cu = workloads.cu_from_lengths(lens)
    T, H, d = int(cu[-1]), 2, 64
    x = workloads.draw((T, H, d), "outlier", 8)
    codes, su, st = oracle_mod.quantize(x, cu, COL, 32, False, 0)
    ng = sum((L + 31) // 32 for L in lens)
    assert st == 0 and su.shape == (H, ng, d)
    g = 0
    for i, L in enumerate(lens):
        s = int(cu[i])
        for b in range(0, L, 32):
            blk = x[s + b:s + min(b + 32, L)].astype(np.float64)      # [n, H, d]
            amax = np.abs(blk).max(0)                                 # [H, d]
            X = su[:, g, :].astype(np.int64) - 127
            assert np.all(amax <= 448.0 * 2.0 ** X) and np.all(amax > 448.0 * 2.0 ** (X - 1))
            g += 1
    deq = oracle_mod.dequantize(oracle_mod.QTensor(codes, su, COL, 32), cu)
    xd = x.astype(np.float64)
    # unit of the block each element belongs to
    unit = np.zeros_like(xd)
    g = 0
    for i, L in enumerate(lens):
        s = int(cu[i])
        for b in range(0, L, 32):
            unit[s + b:s + min(b + 32, L)] = 2.0 ** (su[:, g, :].astype(np.int64) - 127)[None]
            g += 1
    assert np.all(np.abs(deq - xd) <= e4m3_err_bound(xd, unit))


def test_quantise_rotation_uses_same_signs_for_q_and_k(oracle_mod):
    x = workloads.draw((10, 1, 128), "normal", 2)
    c1, s1, _ = oracle_mod.quantize(x, None, E4M3, 1, True, 42)
    c2, s2, _ = oracle_mod.quantize(x, None, E4M3, 1, True, 43)
    assert not np.array_equal(c1, c2)            # the seed matters
    c3, s3, _ = oracle_mod.quantize(x, None, E4M3, 1, True, 42)
    assert np.array_equal(c1, c3) and np.array_equal(s1, s3)


def test_mx_token_rule_error_bound_and_locality(oracle_mod):
    """MX token layout (V of the causal-exact MX mode): one E8M0 exponent per
    (token, head) over all channels -- the smallest X with amax <= 448 2^X -- so a
    token's codes and scale depend on that token alone."""
    T, H, d = 70, 2, 128
    x = workloads.draw((T, H, d), "outlier", 31)
    codes, su, st = oracle_mod.quantize(x, None, oracle_mod.MX_TOKEN, 1, False, 0)
    assert st == 0 and su.shape == (H, T)
    X = su.T.astype(np.int64) - 127                          # [T, H]
    amax = np.abs(x.astype(np.float64)).max(-1)
    assert np.all(amax <= 448.0 * 2.0 ** X)
    assert np.all(amax > 448.0 * 2.0 ** (X - 1))
    deq = oracle_mod.dequantize(oracle_mod.QTensor(codes, su, oracle_mod.MX_TOKEN, 1))
    unit = np.broadcast_to((2.0 ** X)[:, :, None], x.shape)
    assert np.all(np.abs(deq - x) <= e4m3_err_bound(x.astype(np.float64), unit))
    # locality: changing token 40 changes nothing of any other token
    y = x.copy()
    y[40] *= 37.0
    c2, s2, _ = oracle_mod.quantize(y, None, oracle_mod.MX_TOKEN, 1, False, 0)
    keep = np.arange(T) != 40
    assert np.array_equal(c2[keep], codes[keep]) and np.array_equal(s2[:, keep], su[:, keep])
    assert not np.array_equal(s2[:, 40], su[:, 40])
    # an all-zero token: exponent -127 (byte 0), zero codes
    z = np.zeros((1, 1, d), dtype=np.float32)
    c, s, _ = oracle_mod.quantize(z, None, oracle_mod.MX_TOKEN, 1, False, 0)
    assert s[0, 0] == 0 and not c.any()
