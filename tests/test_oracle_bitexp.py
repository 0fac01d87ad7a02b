"""Pins for the oracle's bit-level exponentials (CPU only).

Sources: FLAMIA section 1 (two bit-level exponential approximations for
inference), section 4.3 (log-domain probability quantisation) and section 4.4
"Bit-Level Exponentials at Inference" (Schraudolph's approximation,
Mitchell-P).

The two forms are pinned to what fixes them independently of the oracle's
code: the IEEE-754 binary32 and OCP E4M3 bit layouts (a float whose bits are
2^23 (u + 127) is 2^floor(u) (1 + frac(u)); an E4M3 code 8 (k + 7) + j is
2^k (1 + j / 8)), the shift delta found by numerically minimising the mean
square relative error (not by its closed form), the error range that shift
gives, and the running-softmax emulation against a direct global evaluation
of the same weights on rows whose reference maximum never moves.
"""
import math

import numpy as np
import pytest

import workloads

E4M3, ROW, COL = 0, 1, 2


def test_delta_minimises_the_mean_square_relative_error(oracle_mod):
    from scipy.optimize import minimize_scalar
    f = (np.arange(200000) + 0.5) / 200000
    g = (1.0 + f) * 2.0 ** -f

    def mse(dl):
        return float(np.mean((g * 2.0 ** -dl - 1.0) ** 2))

    res = minimize_scalar(mse, bounds=(0.0, 0.2), method="bounded", options={"xatol": 1e-10})
    assert abs(res.x - oracle_mod.SCHRAUDOLPH_DELTA) < 1e-6
    assert abs(math.sqrt(res.fun) - 0.0177) < 2e-4


def test_schraudolph_is_the_float_with_bits_2_23_u_plus_127(oracle_mod):
    """On u = k + j / 2^14 (exactly representable), the value is the binary32
    whose bit pattern is (k + 127) 2^23 + 2^9 j."""
    rng = np.random.default_rng(11)
    k = rng.integers(-120, 9, 400)
    j = rng.integers(0, 1 << 14, 400)
    u = k + j / 16384.0
    got = oracle_mod.exp2_schraudolph(u + oracle_mod.SCHRAUDOLPH_DELTA)
    want = (((k + 127) << 23) + (j << 9)).astype(np.uint32).view(np.float32)
    # x - delta recovers u to far below 2^-15, so the rounding to 2^-14 lands on it
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # integers exactly: powers of two
    assert np.array_equal(oracle_mod.exp2_schraudolph(np.arange(-20, 9) + oracle_mod.SCHRAUDOLPH_DELTA),
                          np.ldexp(1.0, np.arange(-20, 9)).astype(np.float32))


def test_schraudolph_relative_error_range(oracle_mod):
    """Relative to 2^x the form is 2^-delta g(f), g(f) = (1 + f) 2^-f, f = frac(u):
    between 2^-delta min g - 1 and 2^-delta max g - 1 (about -3.94% and
    +1.97%; the extremes of g on [0, 1] taken numerically), both reached."""
    f = np.linspace(0, 1, 100001)
    g = (1.0 + f) * 2.0 ** -f
    K = 2.0 ** -oracle_mod.SCHRAUDOLPH_DELTA
    lo, hi = K * g.min() - 1.0, K * g.max() - 1.0
    rng = np.random.default_rng(12)
    x = rng.uniform(-30.0, 8.75, 4000)
    rel = oracle_mod.exp2_schraudolph(x).astype(np.float64) / np.exp2(x) - 1.0
    slack = 2.0 ** -13          # u resolved to 2^-14
    assert rel.min() >= lo - slack and rel.max() <= hi + slack
    assert rel.min() < lo + 0.005 and rel.max() > hi - 0.005     # both ends are reached
    assert abs(math.sqrt(np.mean(rel ** 2)) - 0.0177) < 1.5e-3


def test_schraudolph_lower_limit(oracle_mod):
    tiny = np.float32(2.0 ** -126)
    out = oracle_mod.exp2_schraudolph([-126.0, -200.0, -np.inf, np.nan])
    assert np.all(out == tiny)
    assert np.all(oracle_mod.e4m3_encode(out) == 0)         # code 0: masked keys carry no weight


def test_mitchell_code_is_the_fixed_point_log2(oracle_mod):
    """u = k + j / 8 exactly: code 8 (k + 7) + j, whose E4M3 value is 2^k (1 + j / 8)."""
    dec = oracle_mod.e4m3_decode_table()
    k = np.repeat(np.arange(-6, 9), 8)
    j = np.tile(np.arange(8), 15)
    keep = 8 * (k + 7) + j <= 126
    k, j = k[keep], j[keep]
    codes = oracle_mod.exp2_mitchell_code(k + j / 8.0 + oracle_mod.SCHRAUDOLPH_DELTA)
    assert np.array_equal(codes, (8 * (k + 7) + j).astype(np.uint8))
    assert np.allclose(dec[codes], np.ldexp(1.0 + j / 8.0, k), rtol=0, atol=0)


def test_mitchell_code_rounding_monotone_and_limits(oracle_mod):
    d = oracle_mod.SCHRAUDOLPH_DELTA
    # halfway between codes 64 and 65 (u = 1 + 1/16): to even (64); slightly above: 65
    assert oracle_mod.exp2_mitchell_code(1.0 + 1 / 16 + d) == 64
    assert oracle_mod.exp2_mitchell_code(1.0 + 1 / 16 + 1e-9 + d) == 65
    assert oracle_mod.exp2_mitchell_code(1.0 + 3 / 16 + d) == 66      # 65.5 -> 66
    x = np.linspace(-12.0, 8.75, 3001)
    c = oracle_mod.exp2_mitchell_code(x).astype(int)
    assert np.all(np.diff(c) >= 0) and c[0] == 0 and c[-1] <= 126
    assert np.all(oracle_mod.exp2_mitchell_code([-7.1, -50.0, -np.inf, np.nan]) == 0)
    # relative to 2^x the code's value stays within the interpolation error and one half code step
    dec = oracle_mod.e4m3_decode_table()
    x = np.random.default_rng(13).uniform(-5.0, 8.75, 4000)
    rel = dec[oracle_mod.exp2_mitchell_code(x)] / np.exp2(x) - 1.0
    assert rel.min() > 2.0 ** -d * 2.0 ** (-1 / 16) - 1.0 - 1e-9
    assert rel.max() < 2.0 ** -d * 1.0615 * 2.0 ** (1 / 16) - 1.0


def _quant(oracle_mod, inp, mx, rotate=True, seed=0x5EED0011):
    cu = inp.cu_seqlens
    if mx:
        return (oracle_mod.quantize_tensor(inp.q, cu, ROW, 32, rotate, seed),
                oracle_mod.quantize_tensor(inp.k, cu, ROW, 32, rotate, seed),
                oracle_mod.quantize_tensor(inp.v, cu, COL, 32, False, 0))
    return (oracle_mod.quantize_tensor(inp.q, cu, E4M3, 128, rotate, seed),
            oracle_mod.quantize_tensor(inp.k, cu, E4M3, 128, rotate, seed),
            oracle_mod.quantize_tensor(inp.v, cu, E4M3, 128, False, 0))


def _direct(oracle_mod, Q, K, V, mx, exp_mode, causal, tau):
    """Global evaluation of one document: per row the scores s'_t (the emulation's
    fp32 formation), the reference M0 = the maximum over the first key tile, and
    the weights of the chosen exponential at x_t = s'_t - M0 + 8 + log2 r_t over
    all keys at once. Rows where a later key tile exceeds M0 + tau (the reference
    would move) are returned as NaN."""
    dec = oracle_mod.e4m3_decode_table()
    T, H, d = Q.codes.shape
    Cd = (1.0 / math.sqrt(d)) * 1.4426950408889634 / d
    C = np.float32(Cd)
    dl = oracle_mod.SCHRAUDOLPH_DELTA
    if mx:
        qd, kd, vd = (oracle_mod.dequantize(x) for x in (Q, K, V))
    else:
        qd, kd, vd = dec[Q.codes], dec[K.codes], dec[V.codes]
    out = np.full((T, H, d), np.nan)
    lse = np.full((H, T), np.nan)
    for h in range(H):
        S = (qd[:, h] @ kd[:, h].T).astype(np.float32)          # fp64 sums rounded once
        if mx:
            sp = (S * C).astype(np.float32)
            r = np.ones(T)
            ref = 1.0
        else:
            qs, ks, vs = Q.scales[h], K.scales[h], V.scales[h]
            cf = qs[np.arange(T) // 128, None].astype(np.float64) * ks[None, np.arange(T) // 128] * Cd
            sp = (S * cf.astype(np.float32)).astype(np.float32)
            ref = float(vs[: (T + 127) // 128].max())
            inv = np.float32(1.0) / np.float32(ref)
            r = np.array([float(np.float32(vs[t // 128]) * inv) if vs[t // 128] > 0 else 1.0 for t in range(T)])
        for i in range(T):
            n = i + 1 if causal else T
            row = sp[i, :n].astype(np.float64)
            M0 = row[:128].max()
            if n > 128 and row[128:].max() > np.float32(M0 + tau):
                continue
            x = row - M0 + 8.0 + np.log2(r[:n])
            u = x - dl
            if exp_mode == oracle_mod.EXP_MITCHELL_P:
                code = np.clip(np.rint(8.0 * u + 56.0), 0, 126).astype(np.uint8)
                P = dec[code]
                w = P / r[:n]
            else:
                uu = np.maximum(u, -126.0)
                nn = np.rint(np.ldexp(uu + 126.0, 14))
                p = np.ldexp(1.0 + np.mod(nn, 16384) / 16384.0, (np.floor(nn / 16384) - 126).astype(int))
                p = p.astype(np.float32)
                P = dec[oracle_mod.e4m3_encode(p)]
                w = p.astype(np.float64) / r[:n]
            l = w.sum()
            vv = vd[:n, h]
            out[i, h] = ref * (P @ vv) / l
            lse[h, i] = math.log(2.0) * (M0 + math.log2(l) - 8.0)
    return out, lse


@pytest.mark.parametrize("mx", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("exp_name", ["EXP_SCHRAUDOLPH", "EXP_MITCHELL_P"])
def test_emulation_equals_direct_weights(oracle_mod, mx, causal, exp_name):
    """One 300-token document: three key tiles with their own V block scales
    (E4M3: the ratios r_t differ per tile, so a dropped 1/r or a wrong sign of
    log2 r fails), tau = 0.75."""
    exp_mode = getattr(oracle_mod, exp_name)
    inp = workloads.make(2, heads=2, lengths=[300])
    inp.v = inp.v * np.repeat(np.array([1.0, 0.3, 2.5]), [128, 128, 44])[:, None, None].astype(np.float32)
    Q, K, V = _quant(oracle_mod, inp, mx)
    tau = 0.75
    o, _, lse = oracle_mod.attention_emulate(Q, K, V, inp.cu_seqlens, causal, False, None, rescale_tau=tau,
                                             exp_mode=exp_mode)
    od, ld = _direct(oracle_mod, Q, K, V, mx, exp_mode, causal, tau)
    ok = ~np.isnan(ld)
    assert ok.mean() > 0.3
    rows_h = np.argwhere(ok)
    a = np.stack([o[t, h] for h, t in rows_h])
    b = np.stack([od[t, h] for h, t in rows_h])
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-5
    assert np.max(np.abs(lse[ok] - ld[ok])) < 1e-5


def test_bit_level_outputs_stay_close_to_the_exact_exponential(oracle_mod):
    """Against the FP64 attention of the same input, the bit-level forms move the
    output by about what E4M3 P itself costs (output cosine within 1e-4 of the
    exact exponential's on an MX workload, FLAMIA 4.4)."""
    inp = workloads.make(4, heads=2, lengths=[512, 256])
    Q, K, V = _quant(oracle_mod, inp, True)
    ref, _ = oracle_mod.attention_fp64(inp.q.astype(np.float64), inp.k.astype(np.float64),
                                       inp.v.astype(np.float64), inp.cu_seqlens, False, 1 / math.sqrt(128))

    def cos(o):
        return float(np.sum(o * ref) / (np.linalg.norm(o) * np.linalg.norm(ref)))

    base = cos(oracle_mod.attention_emulate(Q, K, V, inp.cu_seqlens, False, False, None, rescale_tau=0.75)[0])
    for mode in (oracle_mod.EXP_SCHRAUDOLPH, oracle_mod.EXP_MITCHELL_P):
        o = oracle_mod.attention_emulate(Q, K, V, inp.cu_seqlens, False, False, None, rescale_tau=0.75,
                                         exp_mode=mode)[0]
        assert abs(cos(o) - base) < 1e-4, (mode, cos(o), base)


def test_bit_level_modes_reject_exact_and_per_token_v(oracle_mod):
    inp = workloads.make(3, heads=1, lengths=[200])
    cu = inp.cu_seqlens
    Q = oracle_mod.quantize_tensor(inp.q, cu, E4M3, 1, True, 3)
    K = oracle_mod.quantize_tensor(inp.k, cu, E4M3, 1, True, 3)
    V = oracle_mod.quantize_tensor(inp.v, cu, E4M3, 1, False, 0)
    with pytest.raises(ValueError):
        oracle_mod.attention_emulate(Q, K, V, cu, True, True, None, exp_mode=oracle_mod.EXP_SCHRAUDOLPH)
    with pytest.raises(ValueError):   # V blocks shorter than a key tile
        oracle_mod.attention_emulate(Q, K, V, cu, True, False, None, exp_mode=oracle_mod.EXP_MITCHELL_P)


def test_log_domain_lse_tie_allowance_explains_score_rounding(oracle_mod):
    """Under the log-domain P the row sum adds the codes' values, so a code that
    sits within fp32 rounding of a boundary moves lse too. A relative change of
    2^-21 in the score scale (the size of an fp32 rounding difference) flips some
    codes; every lse change it causes lies within the emulation's lse allowance
    (plus the continuous part, the running maximum's own shift), which is zero
    under the hardware and Schraudolph exponentials (their row sums add
    unquantised probabilities)."""
    inp = workloads.make(2, heads=2, lengths=[1024, 300])
    cu = inp.cu_seqlens
    Q, K, V = _quant(oracle_mod, inp, False)
    scale = 1 / math.sqrt(128)
    mode = oracle_mod.EXP_MITCHELL_P
    _, _, la, _, lt = oracle_mod.attention_emulate(Q, K, V, cu, False, False, scale, ties=True, exp_mode=mode,
                                                   rescale_tau=0.75, lse_ties=True)
    _, _, lb = oracle_mod.attention_emulate(Q, K, V, cu, False, False, scale * (1 + 2.0 ** -21), exp_mode=mode,
                                            rescale_tau=0.75)
    diff = np.abs(la.astype(np.float64) - lb)
    cont = 2.0 ** -19 * (np.abs(la.astype(np.float64)) + 16.0)
    assert np.all(lt >= 0) and np.count_nonzero(lt) > 0
    assert np.all(diff <= lt + cont)
    assert np.count_nonzero(diff > cont) > 0                  # some row sums did move by a flip
    for other in (oracle_mod.EXP_HW, oracle_mod.EXP_SCHRAUDOLPH):
        _, _, _, _, l0 = oracle_mod.attention_emulate(Q, K, V, cu, False, False, scale, ties=True,
                                                      exp_mode=other, rescale_tau=0.75, lse_ties=True)
        assert not l0.any()
