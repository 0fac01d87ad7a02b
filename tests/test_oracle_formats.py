"""Pins for the oracle's number formats and rotation (CPU only).

Each check compares the oracle with something other than itself: hand-derived
codes from the OCP E4M3 definition, an exhaustive brute-force nearest-value
search, the E8M0 rule's defining inequality, torch's bf16 conversion, a
published SplitMix64 test vector, and a dense Sylvester Hadamard matrix built
by Kronecker products.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

from conftest import ROOT, read_golden


def test_e4m3_decode_table_properties(oracle_mod):
    t = oracle_mod.e4m3_decode_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0            # largest finite
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])            # the only NaN codes
    assert t[0x01] == 2.0 ** -9                               # smallest subnormal
    assert t[0x08] == 2.0 ** -6 and t[0x07] == 7 * 2.0 ** -9  # normal / subnormal boundary
    assert t[0x38] == 1.0
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)                           # monotone over 0x00..0x7E
    assert np.array_equal(t[0x80:0xFF], -pos)                 # sign-magnitude
    assert np.isfinite(t).sum() == 254


def test_e4m3_encode_golden(oracle_mod):
    for val, code, *_ in read_golden("e4m3_codes.txt"):
        got = oracle_mod.lib().or_e4m3_encode(float(val))
        assert got == int(code, 16), (val, hex(got), code)


def test_e4m3_encode_nan_and_inf(oracle_mod):
    L = oracle_mod.lib()
    assert L.or_e4m3_encode(float("nan")) == 0x7F
    assert L.or_e4m3_encode(float("inf")) == 0x7E
    assert L.or_e4m3_encode(float("-inf")) == 0xFE


@pytest.mark.timeout(600)
def test_e4m3_encode_exhaustive_vs_bruteforce(oracle_mod, tmp_path):
    """All 2^32 fp32 inputs: encoder == nearest decoded value (ties to even)."""
    exe = tmp_path / "bf"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-pthread",
                           "-I", os.path.join(ROOT, "oracle"), "-o", str(exe),
                           os.path.join(ROOT, "tests", "c", "e4m3_bruteforce.c"),
                           os.path.join(ROOT, "oracle", "attn_oracle.c"), "-lm"])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "mismatches 0" in out.stdout


def test_e8m0_golden(oracle_mod):
    for amax, xd, xo in read_golden("e8m0_exponents.txt"):
        assert oracle_mod.e8m0_exponent(float(amax), oracle_mod.MX_RULE_NOSAT) == int(xd), amax
        assert oracle_mod.e8m0_exponent(float(amax), oracle_mod.MX_RULE_OCP_FLOOR) == int(xo), amax


def test_e8m0_defining_inequalities(oracle_mod):
    """Every binade: the default X is the smallest with amax <= 448 * 2^X; the
    OCP X satisfies 2^(X+8) <= amax < 2^(X+9)."""
    rng = np.random.default_rng(5)
    for E in range(-135, 128):
        for m in [1.0, 1.25, 1.5, 1.75, np.nextafter(np.float32(1.75), np.float32(2)), 1.999, *rng.uniform(1, 2, 4)]:
            amax = np.float32(np.ldexp(np.float64(np.float32(m)), E))
            if not np.isfinite(amax) or amax == 0:
                continue
            a = float(amax)
            X = oracle_mod.e8m0_exponent(a, oracle_mod.MX_RULE_NOSAT)
            if -127 < X < 127:
                assert a <= 448.0 * 2.0 ** X and not (a <= 448.0 * 2.0 ** (X - 1)), (a, X)
            Xo = oracle_mod.e8m0_exponent(a, oracle_mod.MX_RULE_OCP_FLOOR)
            if -127 < Xo < 127:
                assert 2.0 ** (Xo + 8) <= a < 2.0 ** (Xo + 9), (a, Xo)
    assert oracle_mod.e8m0_exponent(0.0) == -127


def test_bf16_rne_matches_torch(oracle_mod):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.bf16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_splitmix64_published_vector(oracle_mod):
    rows = read_golden("splitmix64_seed1234567.txt")
    seed = int(rows[0][1])
    want = [int(r[0]) for r in rows[1:]]
    assert oracle_mod.splitmix64_stream(seed, len(want)) == want


def test_signs_are_top_bits_and_balanced(oracle_mod):
    s = oracle_mod.signs(1234567, 5)
    want = [int(r[0]) for r in read_golden("splitmix64_seed1234567.txt")[1:]]
    assert list(s) == [-1.0 if (w >> 63) else 1.0 for w in want]
    big = oracle_mod.signs(0x5EED0002, 4096)
    assert set(np.unique(big)) == {-1.0, 1.0}
    assert abs(big.sum()) < 5 * np.sqrt(4096)


def sylvester(d):
    H = np.array([[1.0]])
    while H.shape[0] < d:
        H = np.kron(H, np.array([[1.0, 1.0], [1.0, -1.0]]))
    return H


def stored_order(d):
    """The channel order the rotation stores at head_dim 128, bit by bit: stored
    channel p (bits p6..p0) holds the transform's output channel with bits
    (p3 p2 p1 p6 p5 p4 p0)."""
    if d != 128:
        return np.arange(d)
    out = []
    for p in range(d):
        bit = [(p >> i) & 1 for i in range(7)]
        out.append(bit[0] | bit[4] << 1 | bit[5] << 2 | bit[6] << 3 | bit[1] << 4 | bit[2] << 5 | bit[3] << 6)
    return np.array(out)


def rotation_matrix(oracle_mod, d, seed):
    """R = P H D: the Sylvester rows in the stored order times the sign diagonal."""
    return sylvester(d)[stored_order(d)] * oracle_mod.signs(seed, d)[None, :]


def test_rotation_stored_order(oracle_mod):
    """At head_dim 128 the rotation stores the transform's outputs with the 3-bit
    fields at bits 1-3 and 4-6 of the channel index swapped (the order the device
    transform leaves them in); R = P H is still a Hadamard matrix, so the rotation
    still cancels in Q K^T. At 64 the order is the natural one."""
    pi = oracle_mod.rotation_channels(128)
    assert np.array_equal(pi, stored_order(128))
    assert sorted(pi) == list(range(128)) and np.array_equal(pi[pi], np.arange(128))   # an involution
    assert [pi[p] for p in (0, 1, 2, 16, 0x0E, 0x70, 0x7F, 0x55)] == [0, 1, 16, 2, 0x70, 0x0E, 0x7F, 0x2B]
    assert np.array_equal(oracle_mod.rotation_channels(64), np.arange(64))
    R = rotation_matrix(oracle_mod, 128, 3)
    assert np.array_equal(R @ R.T, 128 * np.eye(128))
    rng = np.random.default_rng(3)
    xi = rng.integers(-50, 50, size=(6, 128)).astype(np.float32)    # exact in fp32
    assert np.array_equal(oracle_mod.rotate(xi, 3).astype(np.float64), xi.astype(np.float64) @ R.T)


@pytest.mark.parametrize("d", [2, 8, 32, 64, 128])
def test_fwht_equals_dense_hadamard(oracle_mod, d):
    H = sylvester(d)
    assert np.array_equal(H @ H.T, d * np.eye(d))                 # H H^T = d I
    rng = np.random.default_rng(d)
    xi = rng.integers(-50, 50, size=(6, d)).astype(np.float32)    # exact in fp32
    assert np.array_equal(oracle_mod.fwht(xi).astype(np.float64), xi.astype(np.float64) @ H.T)
    xf = rng.standard_normal((6, d)).astype(np.float32)
    y = oracle_mod.fwht(xf).astype(np.float64)
    ref = xf.astype(np.float64) @ H.T
    bound = np.log2(d) * 2.0 ** -23 * np.abs(xf).sum(axis=1, keepdims=True) * 2
    assert np.all(np.abs(y - ref) <= bound)


def test_rotation_cancels_in_qk(oracle_mod):
    """(H D x) . (H D y) = d (x . y): the rotation cancels in Q K^T."""
    d = 128
    s = oracle_mod.signs(77, d)
    rng = np.random.default_rng(1)
    x = rng.integers(-20, 20, size=(5, d)).astype(np.float32)
    y = rng.integers(-20, 20, size=(5, d)).astype(np.float32)
    rx = oracle_mod.fwht(x * s).astype(np.float64)
    ry = oracle_mod.fwht(y * s).astype(np.float64)
    assert np.array_equal(rx @ ry.T, d * (x.astype(np.float64) @ y.astype(np.float64).T))
