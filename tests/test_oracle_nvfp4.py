"""Pins for the oracle's NVFP4 operands (the mixed NVFP4/FP8 path), CPU only.

Sources: FLAMIA section 1 (NVFP4 for Q K^T, 8-bit operands elsewhere) and
section 2 (NVFP4: 16-element blocks with a shared scale plus a tensor-level
scale; Blackwell's block-scaled MMA consumes them directly).

E2M1 against hand-derived codes (tests/golden/e2m1_codes.txt) and its
embedding in E4M3; the quantiser against the dense-matrix rotation and an
error bound that follows from the two scale levels, the closed form of a
block's largest element and of an exactly representable group, document
locality and the zero block; the emulation on NVFP4 operands against O-1 on
their dequantised values.
"""
import math
import os

import numpy as np
import pytest

import workloads
from conftest import ROOT

E4M3 = 0


def read_golden(name):
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", name)):
        line = line.split("#")[0].strip()
        if line:
            a, b, *rest = line.split()
            rows.append((float(a), int(b, 16)))
    return rows


def test_e2m1_hand_codes(oracle_mod):
    rows = read_golden("e2m1_codes.txt")
    assert len(rows) >= 20
    got = oracle_mod.e2m1_encode([v for v, _ in rows])
    assert [int(g) for g in got] == [c for _, c in rows]


def test_e2m1_values_are_e4m3_values_and_round_trip(oracle_mod):
    dec2 = oracle_mod.e2m1_decode_table()
    dec8 = oracle_mod.e4m3_decode_table()
    assert list(dec2[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    for c in range(16):
        v = dec2[c]
        assert oracle_mod.e2m1_encode([v])[0] == c or (v == 0 and c in (0, 8))
        assert dec8[oracle_mod.e4m3_encode(np.float32(v))] == v     # E2M1 is a subset of E4M3
    # nearest: on a dense grid no magnitude is closer than the chosen code's
    x = np.linspace(-7, 7, 2801).astype(np.float32)
    e = oracle_mod.e2m1_encode(x)
    err = np.abs(dec2[e] - np.clip(x, -6, 6))
    assert np.all(err <= np.min(np.abs(dec2[None, :8] - np.abs(np.clip(x, -6, 6))[:, None]), axis=1) + 1e-12)


def _dense_rot(x, seed, oracle_mod):
    from test_oracle_formats import rotation_matrix
    d = x.shape[-1]
    R = rotation_matrix(oracle_mod, d, seed)
    return (x.astype(np.float64) @ R.T)


@pytest.mark.parametrize("rotate", [True, False])
def test_nvfp4_error_bound_against_dense_rotation(oracle_mod, rotate):
    """|x_hat - y| <= (1/6)(1 + 2^-4) max|y| over the element's 16-channel group
    (+ fp32 slack): the E2M1 step is at most 1 on the [-6, 6] grid the group's
    E4M3 scale maps it to, and that scale is within 2^-4 of the group maximum."""
    inp = workloads.make(2, heads=2, lengths=[300, 77, 129])
    cu = inp.cu_seqlens
    Q = oracle_mod.quantize_tensor(inp.q, cu, oracle_mod.NVFP4, 128, rotate, 9)
    y = _dense_rot(inp.q, 9, oracle_mod) if rotate else inp.q.astype(np.float64)
    xh = oracle_mod.dequantize(Q, cu)
    g = np.abs(y).reshape(*y.shape[:2], -1, 16).max(-1)
    bound = np.repeat(g, 16, axis=2) * (1 / 6) * (1 + 2.0 ** -4) * (1 + 1e-5) + 1e-30
    assert np.all(np.abs(xh - y) <= bound)
    assert np.abs(xh - y).max() > 0.3 * bound.max() * 0.1    # the bound is not vacuous


def test_nvfp4_block_scale_and_largest_element(oracle_mod):
    """s_t = amax / 2688 for each 128-token block (document-local), and each block's
    largest element comes back within fp32 rounding (it maps to E4M3 448 and E2M1 6)."""
    inp = workloads.make(2, heads=2, lengths=[200, 128, 5])
    cu = inp.cu_seqlens
    codes, (st, sf), s = oracle_mod.quantize(inp.k, cu, oracle_mod.NVFP4, 128, False, 0)
    assert s == 0
    Q = oracle_mod.QTensor(codes, (st, sf), oracle_mod.NVFP4, 128)
    xh = oracle_mod.dequantize(Q, cu)
    b = 0
    for i in range(len(cu) - 1):
        for t0 in range(cu[i], cu[i + 1], 128):
            t1 = min(t0 + 128, cu[i + 1])
            for h in range(2):
                blk = inp.k[t0:t1, h].astype(np.float64)
                amax = np.abs(blk).max()
                assert st[h, b] == np.float32(np.float32(amax) / np.float32(2688.0))
                t, c = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
                assert abs(xh[t0 + t, h, c] - blk[t, c]) <= 4e-7 * amax
            b += 1
    assert b == st.shape[1]


def test_nvfp4_exact_group_and_zero_block(oracle_mod):
    """A block with amax 448 (inverse scale 1) and a group whose largest value is
    48 = 6 * 2^3 (an E4M3 value, so the group's step is exactly 8): values that
    are 8 x E2M1 come back exactly (up to s_t's fp32 rounding); an all-zero block
    gives zero codes and scales."""
    T, H, d = 130, 1, 32
    x = np.zeros((T, H, d), dtype=np.float32)
    x[0, 0, 0] = 448.0
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -6, -4, -3, -2, -1.5, -1, -0.5, 6], dtype=np.float32) * 8
    x[1, 0, 16:32] = vals
    codes, (st, sf), s = oracle_mod.quantize(x, None, oracle_mod.NVFP4, 128, False, 0)
    assert s == 0
    xh = oracle_mod.dequantize(oracle_mod.QTensor(codes, (st, sf), oracle_mod.NVFP4, 128))
    assert sf[1, 0, 1] == 0x64                        # E4M3 48 = 1.5 * 2^5: e = 5 + 7 = 12, m = 4
    assert np.allclose(xh[1, 0, 16:32], vals, rtol=1e-6, atol=0)
    assert abs(xh[0, 0, 0] - 448.0) <= 448.0 * 1e-6
    # tokens 128, 129: the second block is all zero
    assert st[0, 1] == 0 and np.all(codes[128:] == 0) and np.all(sf[128:] == 0)


def test_nvfp4_is_document_local(oracle_mod):
    inp = workloads.make(3, heads=2, lengths=[100, 260, 33])
    cu = inp.cu_seqlens
    whole = oracle_mod.quantize(inp.q, cu, oracle_mod.NVFP4, 128, True, 4)
    parts = [oracle_mod.quantize(inp.q[cu[i]:cu[i + 1]], None, oracle_mod.NVFP4, 128, True, 4)
             for i in range(len(cu) - 1)]
    assert np.array_equal(whole[0], np.concatenate([p[0] for p in parts]))
    assert np.array_equal(whole[1][1], np.concatenate([p[1][1] for p in parts]))
    assert np.array_equal(whole[1][0], np.concatenate([p[1][0] for p in parts], axis=1))


@pytest.mark.parametrize("causal", [False, True])
def test_emulation_on_nvfp4_operands_matches_fp64_on_dequantised(oracle_mod, causal):
    """With P unquantised, the emulation over NVFP4 Q, K and E4M3 V equals O-1 on
    the dequantised operands (the score multiplier carries both s_t, the MMA the
    16-channel scales)."""
    inp = workloads.make(2, heads=2, lengths=[300, 77])
    cu = inp.cu_seqlens
    Q = oracle_mod.quantize_tensor(inp.q, cu, oracle_mod.NVFP4, 128, True, 21)
    K = oracle_mod.quantize_tensor(inp.k, cu, oracle_mod.NVFP4, 128, True, 21)
    V = oracle_mod.quantize_tensor(inp.v, cu, E4M3, 128, False, 0)
    scale = 1.0 / math.sqrt(128)
    o3, _, l3 = oracle_mod.attention_emulate(Q, K, V, cu, causal, False, scale, quantize_p=False)
    qd, kd, vd = (oracle_mod.dequantize(x, cu) for x in (Q, K, V))
    o1, l1 = oracle_mod.attention_fp64(qd, kd, vd, cu, causal, scale / 128)
    assert np.linalg.norm(o3 - o1) / np.linalg.norm(o1) < 2e-6
    assert np.max(np.abs(l3 - l1)) < 1e-4


def test_nvfp4_emulation_rules(oracle_mod):
    inp = workloads.make(2, heads=1, lengths=[200])
    cu = inp.cu_seqlens
    Q = oracle_mod.quantize_tensor(inp.q, cu, oracle_mod.NVFP4, 128, True, 2)
    K8 = oracle_mod.quantize_tensor(inp.k, cu, E4M3, 128, True, 2)
    V = oracle_mod.quantize_tensor(inp.v, cu, E4M3, 128, False, 0)
    with pytest.raises(ValueError):     # Q and K must both be NVFP4
        oracle_mod.attention_emulate(Q, K8, V, cu, False, False, None)
    K = oracle_mod.quantize_tensor(inp.k, cu, oracle_mod.NVFP4, 128, True, 2)
    with pytest.raises(ValueError):     # no causal-exact mode with 128-token s_t
        oracle_mod.attention_emulate(Q, K, V, cu, True, True, None)
    with pytest.raises(ValueError):     # block 128 only
        oracle_mod.quantize_tensor(inp.q, cu, oracle_mod.NVFP4, 64, True, 2)
