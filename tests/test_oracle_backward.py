"""Pins for the oracle's FP64 attention backward (dQ, dK, dV for an upstream
dO), CPU only. Independent of its formula: central finite differences of the
FP64 forward on tiny inputs; closed forms (the dV rows of a document sum to its
dO rows, the dK rows sum to zero, a one-key document passes dO to dV and
nothing to dQ, dK); causal structure (a gradient at row i reaches no key after
i); packed documents equal the documents one by one."""
import numpy as np
import pytest

import oracle


def _inputs(lengths, H=2, d=4, seed=7):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    q, k, v, do = (rng.standard_normal((T, H, d)) for _ in range(4))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, do, cu


def _loss(q, k, v, do, cu, causal, scale):
    o, _ = oracle.attention_fp64(q, k, v, cu, causal, scale)
    return float(np.sum(o * do))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(oracle_mod, causal):
    q, k, v, do, cu = _inputs([4, 2, 3])
    scale = 0.7
    dq, dk, dv = oracle.attention_fp64_backward(q, k, v, do, cu, causal, scale)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = dict(q=q, k=k, v=v)
            args_m = dict(q=q, k=k, v=v)
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (_loss(do=do, cu=cu, causal=causal, scale=scale, **args_p) -
                       _loss(do=do, cu=cu, causal=causal, scale=scale, **args_m)) / (2 * eps)
        assert np.abs(g - fd).max() < 1e-7 * max(1.0, np.abs(fd).max()), name


@pytest.mark.parametrize("causal", [False, True])
def test_backward_closed_forms(oracle_mod, causal):
    q, k, v, do, cu = _inputs([5, 1, 7], H=3, d=8, seed=11)
    dq, dk, dv = oracle.attention_fp64_backward(q, k, v, do, cu, causal, 0.4)
    for a, b in zip(cu[:-1], cu[1:]):
        # every row's probabilities sum to one, and every row of dS to zero
        assert np.allclose(dv[a:b].sum(axis=0), do[a:b].sum(axis=0), atol=1e-12)
        assert np.allclose(dk[a:b].sum(axis=0), 0.0, atol=1e-12)
    # the one-key document (tokens 5): P = 1, dS = 0
    assert np.allclose(dv[5], do[5], atol=1e-15)
    assert np.abs(dq[5]).max() < 1e-15 and np.abs(dk[5]).max() < 1e-15


def test_backward_causal_reaches_no_later_key(oracle_mod):
    q, k, v, do, cu = _inputs([9], H=1, d=4, seed=3)
    i0 = 4
    g = np.zeros_like(do)
    g[i0] = do[i0]
    dq, dk, dv = oracle.attention_fp64_backward(q, k, v, g, cu, True, 0.5)
    assert np.abs(dk[i0 + 1:]).max() == 0.0 and np.abs(dv[i0 + 1:]).max() == 0.0
    assert np.abs(dq[np.arange(9) != i0]).max() == 0.0
    assert np.abs(dk[:i0 + 1]).max() > 0.0 and np.abs(dv[:i0 + 1]).max() > 0.0


def test_backward_packed_equals_per_document(oracle_mod):
    q, k, v, do, cu = _inputs([6, 3, 8], H=2, d=8, seed=5)
    for causal in (False, True):
        grads = oracle.attention_fp64_backward(q, k, v, do, cu, causal, 0.3)
        for a, b in zip(cu[:-1], cu[1:]):
            single = oracle.attention_fp64_backward(q[a:b], k[a:b], v[a:b], do[a:b], None, causal, 0.3)
            for g, s in zip(grads, single):
                assert np.array_equal(g[a:b], s)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_with_stored_output(oracle_mod, causal):
    """D taken from a given output o. With the exact forward output it is the
    default backward (pinned above by finite differences). With o + delta, only
    D_i moves, by c_i = dO_i . delta_i, so dV is unchanged and, from
    dS = P o (dP - D): dQ moves by -scale c_i (P K)_i, which is attention with K
    in place of V, and dK by -scale P^T (c o Q), which is the dV that the
    upstream gradient c_i Q_i would get."""
    q, k, v, do, cu = _inputs([6, 1, 9], H=2, d=8, seed=21)
    scale = 0.45
    o, _ = oracle.attention_fp64(q, k, v, cu, causal, scale)
    ref = oracle.attention_fp64_backward(q, k, v, do, cu, causal, scale)
    same = oracle.attention_fp64_backward(q, k, v, do, cu, causal, scale, o=o)
    for a, b in zip(ref, same):
        assert np.allclose(a, b, rtol=1e-12, atol=1e-13)
    delta = np.random.default_rng(4).standard_normal(o.shape) * 1e-2
    dq, dk, dv = oracle.attention_fp64_backward(q, k, v, do, cu, causal, scale, o=o + delta)
    c = np.sum(do * delta, axis=2, keepdims=True)                      # [T, H, 1]
    pk, _ = oracle.attention_fp64(q, k, k, cu, causal, scale)          # (P K)_i
    assert np.allclose(dq - ref[0], -scale * c * pk, rtol=1e-10, atol=1e-13)
    _, _, ptcq = oracle.attention_fp64_backward(q, k, v, c * q, cu, causal, scale)
    assert np.allclose(dk - ref[1], -scale * ptcq, rtol=1e-10, atol=1e-13)
    assert np.array_equal(dv, ref[2])
