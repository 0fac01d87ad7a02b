"""CPU oracle for the fused low-precision attention forward pass.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package. The product
package never imports it, and the C code behind it (``attn_oracle.c``) shares
nothing with the CUDA library.

The oracle has three parts (see ``attn_oracle.h`` for the page passages):

* O-1 ``attention_fp64``: plain FP64 softmax attention, and
  ``attention_fp64_backward``: its gradients (dQ, dK, dV) for an upstream dO.
* O-2 ``quantize``: the bit-level rotate-and-quantise emulator (E4M3 token
  blocks, MXFP8 row/column blocks with E8M0 exponents).
* O-3 ``attention_emulate``: the running-softmax loop over the quantised
  operands, tiled by 128 keys as the kernel tiles it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_HDR = os.path.join(_HERE, "attn_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

E4M3_TOKBLOCK, MX_ROW32, MX_COL32, MX_TOKEN, NVFP4 = 0, 1, 2, 3, 4
MX_RULE_NOSAT, MX_RULE_OCP_FLOOR = 0, 1
QUANTIZE_P = 1
# the probabilities' exponential (emulation flags): 2^x, Schraudolph's, log-domain P (Mitchell)
EXP_HW, EXP_SCHRAUDOLPH, EXP_MITCHELL_P = 0, 1, 2
_EXP_FLAGS = {EXP_HW: 0, EXP_SCHRAUDOLPH: 2, EXP_MITCHELL_P: 4}
SCHRAUDOLPH_DELTA = 0.057984814725439975

_lock = threading.Lock()
_lib = None

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB_PATH) for p in (_SRC, _HDR))
    if stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _QT(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("layout", ctypes.c_int), ("block", ctypes.c_int),
                ("scales_f32", ctypes.c_void_p), ("scales_u8", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i32, u64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_double
            L.or_set_threads.argtypes = [i32]
            L.or_threads.restype = i32
            L.or_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.or_e4m3_decode.restype = dbl
            L.or_e4m3_encode.argtypes = [ctypes.c_float]
            L.or_e4m3_encode.restype = ctypes.c_uint8
            L.or_e2m1_decode.argtypes = [ctypes.c_uint8]
            L.or_e2m1_decode.restype = dbl
            L.or_e2m1_encode.argtypes = [ctypes.c_float]
            L.or_e2m1_encode.restype = ctypes.c_uint8
            L.or_e8m0_exponent.argtypes = [ctypes.c_float, i32]
            L.or_e8m0_exponent.restype = i32
            L.or_bf16_rne.argtypes = [ctypes.c_float]
            L.or_bf16_rne.restype = ctypes.c_uint16
            L.or_e4m3_encode_range.argtypes = [u64, u64, vp]
            L.or_signs.argtypes = [u64, i32, vp]
            L.or_fwht_f32.argtypes = [vp, i32]
            L.or_rotation_channel.argtypes = [i32, i32]
            L.or_rotation_channel.restype = i32
            L.or_splitmix64_next.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
            L.or_splitmix64_next.restype = u64
            L.or_num_blocks.argtypes = [vp, i32, i32, i32]
            L.or_num_blocks.restype = ctypes.c_long
            L.or_quantize.argtypes = [vp, i32, i32, i32, vp, i32, i32, i32, i32, u64, i32, vp, vp, vp]
            L.or_quantize.restype = i32
            L.or_attention_fp64.argtypes = [vp, vp, vp, i32, i32, i32, vp, i32, i32, dbl, vp, i32, vp, vp]
            L.or_attention_fp64_bwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, i32, i32, dbl, vp, vp, vp]
            L.or_attention_fp64_bwd_o.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp, i32, i32, dbl, vp, vp, vp]
            L.or_attention_emulate.argtypes = [ctypes.POINTER(_QT)] * 3 + [
                i32, i32, i32, vp, i32, i32, i32, i32, dbl, ctypes.c_float, i32, vp, i32, vp, vp, vp, vp, vp]
            L.or_attention_emulate.restype = i32
            L.or_attention_emulate_given_p.argtypes = [ctypes.POINTER(_QT)] * 3 + [
                i32, i32, i32, vp, i32, i32, i32, i32, dbl, ctypes.c_float, i32, vp, i32, vp, vp, vp, vp,
                ctypes.c_long, vp]
            L.or_attention_emulate_given_p.restype = i32
            L.or_exp2_schraudolph.argtypes = [dbl]
            L.or_exp2_schraudolph.restype = ctypes.c_float
            L.or_exp2_mitchell_code.argtypes = [dbl]
            L.or_exp2_mitchell_code.restype = ctypes.c_uint8
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _cu(cu_seqlens, T):
    if cu_seqlens is None:
        return None, 1
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    assert cu[0] == 0 and cu[-1] == T, "cu_seqlens must run from 0 to T"
    return cu, len(cu) - 1


def set_threads(n: int) -> int:
    return lib().or_set_threads(int(n))


def threads() -> int:
    return lib().or_threads()


# ---- number formats ------------------------------------------------------
def e4m3_decode_table() -> np.ndarray:
    L = lib()
    return np.array([L.or_e4m3_decode(i) for i in range(256)], dtype=np.float64)


def e2m1_decode_table() -> np.ndarray:
    L = lib()
    return np.array([L.or_e2m1_decode(i) for i in range(16)], dtype=np.float64)


def e2m1_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    L = lib()
    out = np.array([L.or_e2m1_encode(ctypes.c_float(v)) for v in x.ravel()], dtype=np.uint8)
    return out.reshape(x.shape)


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).ravel()
    out = np.empty(bits.size, dtype=np.uint8)
    L = lib()
    for i, b in enumerate(bits):  # scalar path: small arrays only
        out[i] = L.or_e4m3_encode(ctypes.c_float(np.uint32(b).view(np.float32)))
    return out.reshape(x.shape)


def e4m3_encode_range(start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint8)
    lib().or_e4m3_encode_range(start, count, out.ctypes.data)
    return out


def e8m0_exponent(amax: float, rule: int = MX_RULE_NOSAT) -> int:
    return lib().or_e8m0_exponent(float(amax), rule)


def bf16_rne(x: float) -> int:
    return lib().or_bf16_rne(float(x))


def splitmix64_stream(seed: int, n: int) -> list[int]:
    st = ctypes.c_uint64(seed)
    return [lib().or_splitmix64_next(ctypes.byref(st)) for _ in range(n)]


def signs(seed: int, d: int) -> np.ndarray:
    s = np.empty(d, dtype=np.float32)
    lib().or_signs(seed, d, s.ctypes.data)
    return s


def fwht(x) -> np.ndarray:
    y = np.array(x, dtype=np.float32, copy=True)
    flat = y.reshape(-1, y.shape[-1])
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        lib().or_fwht_f32(row.ctypes.data, row.size)
        flat[r] = row
    return flat.reshape(y.shape)


def rotation_channels(d: int) -> np.ndarray:
    """pi: the rotation stores the transform's output channel pi[p] at channel p."""
    return np.array([lib().or_rotation_channel(p, d) for p in range(d)], dtype=np.int64)


def rotate(x, seed: int) -> np.ndarray:
    """The quantiser's rotation of x [..., d] in fp32: sign flip, transform, stored order."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    return fwht(x * signs(seed, d))[..., rotation_channels(d)]


def num_blocks(cu_seqlens, T: int, block: int) -> int:
    cu, nd = _cu(cu_seqlens, T)
    return lib().or_num_blocks(_ptr(cu), nd, T, block)


# ---- O-2 -------------------------------------------------------------------
def quantize(x, cu_seqlens=None, layout=E4M3_TOKBLOCK, block=128, rotate=False, seed=0,
             mx_rule=MX_RULE_NOSAT):
    """Quantise x [T, H, d] (fp32 values). Returns (codes u8 [T,H,d], scales, status).

    scales: E4M3 token blocks -> fp32 [H, NB]; MX row32 -> u8 [T, H, d/32];
    MX col32 -> u8 [H, NG, d] (NG = document-local 32-token groups); MX token ->
    u8 [H, T] (one exponent per token and head over all d); NVFP4 -> the pair
    (fp32 [H, NB] per 128-token block, u8 [T, H, d/16] E4M3 scales), codes
    u8 [T, H, d/2] with two E2M1 codes per byte (even channel low).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, H, d = x.shape
    cu, nd = _cu(cu_seqlens, T)
    codes = np.zeros((T, H, d // 2 if layout == NVFP4 else d), dtype=np.uint8)
    sf = su = None
    if layout == E4M3_TOKBLOCK:
        sf = np.zeros((H, num_blocks(cu, T, block)), dtype=np.float32)
    elif layout == MX_ROW32:
        su = np.zeros((T, H, d // 32), dtype=np.uint8)
    elif layout == MX_COL32:
        su = np.zeros((H, num_blocks(cu, T, 32), d), dtype=np.uint8)
    elif layout == MX_TOKEN:
        su = np.zeros((H, T), dtype=np.uint8)
    elif layout == NVFP4:
        sf = np.zeros((H, num_blocks(cu, T, 128)), dtype=np.float32)
        su = np.zeros((T, H, d // 16), dtype=np.uint8)
    else:
        raise ValueError(layout)
    st = lib().or_quantize(x.ctypes.data, T, H, d, _ptr(cu), nd, layout, block, int(bool(rotate)),
                           seed & (2**64 - 1), mx_rule, codes.ctypes.data, _ptr(sf), _ptr(su))
    if layout == NVFP4:
        return codes, (sf, su), st
    return codes, (sf if sf is not None else su), st


class QTensor:
    """Quantised operand as the oracle produces it (logical scale layouts)."""

    def __init__(self, codes, scales, layout, block=128, rotated=False, seed=0):
        self.codes, self.scales, self.layout, self.block = codes, scales, layout, block
        self.rotated, self.seed = rotated, seed

    def _qt(self):
        if self.layout == NVFP4:
            sf, su = self.scales
        else:
            sf = self.scales if self.layout == E4M3_TOKBLOCK else None
            su = self.scales if self.layout != E4M3_TOKBLOCK else None
        return _QT(self.codes.ctypes.data, self.layout, self.block, _ptr(sf), _ptr(su))


def quantize_tensor(x, cu_seqlens=None, layout=E4M3_TOKBLOCK, block=128, rotate=False, seed=0,
                    mx_rule=MX_RULE_NOSAT) -> QTensor:
    codes, scales, st = quantize(x, cu_seqlens, layout, block, rotate, seed, mx_rule)
    if st == 1:
        raise ValueError("oracle quantiser rejected its arguments")
    if st != 0:
        raise FloatingPointError(f"oracle quantiser status {st}")
    return QTensor(codes, scales, layout, block, rotate, seed)


def dequantize(qt: QTensor, cu_seqlens=None) -> np.ndarray:
    """Decoded values code * scale in fp64 (rotation not undone)."""
    dec = e4m3_decode_table()
    T, H, d = qt.codes.shape
    if qt.layout == NVFP4:
        d = 2 * d
        e2 = e2m1_decode_table()
        lo, hi = e2[qt.codes & 15], e2[qt.codes >> 4]
        v = np.stack([lo, hi], axis=-1).reshape(T, H, d) * np.repeat(dec[qt.scales[1]], 16, axis=2)
        qt = QTensor(qt.codes, qt.scales[0], E4M3_TOKBLOCK, 128)
    else:
        v = dec[qt.codes]
    cu, nd = _cu(cu_seqlens, T)
    starts = np.zeros(T, dtype=np.int64)
    docs = np.zeros(T, dtype=np.int64)
    bounds = cu if cu is not None else np.array([0, T], dtype=np.int32)
    for i in range(len(bounds) - 1):
        docs[bounds[i]:bounds[i + 1]] = i
        starts[bounds[i]:bounds[i + 1]] = bounds[i]
    local = np.arange(T) - starts
    if qt.layout == E4M3_TOKBLOCK:
        b = qt.block
        nblk = [(int(bounds[i + 1] - bounds[i]) + b - 1) // b for i in range(len(bounds) - 1)]
        boff = np.concatenate([[0], np.cumsum(nblk)])[:-1]
        idx = boff[docs] + local // b                      # [T]
        sc = qt.scales[:, idx].T                           # [T, H]
        return v * sc[:, :, None].astype(np.float64)
    if qt.layout == MX_ROW32:
        X = qt.scales.astype(np.int64) - 127               # [T, H, d/32]
        return v * np.ldexp(1.0, np.repeat(X, 32, axis=2))
    if qt.layout == MX_TOKEN:
        X = qt.scales.T.astype(np.int64) - 127             # [T, H]
        return v * np.ldexp(1.0, X)[:, :, None]
    ng = [(int(bounds[i + 1] - bounds[i]) + 31) // 32 for i in range(len(bounds) - 1)]
    goff = np.concatenate([[0], np.cumsum(ng)])[:-1]
    gidx = goff[docs] + local // 32                        # [T]
    X = qt.scales[:, gidx, :].transpose(1, 0, 2).astype(np.int64) - 127   # [T, H, d]
    return v * np.ldexp(1.0, X)


# ---- O-1 -------------------------------------------------------------------
def attention_fp64(q, k, v, cu_seqlens=None, causal=False, softmax_scale=None, rows=None):
    """FP64 attention. Returns (o [R, H, d] fp64, lse [H, R] fp64)."""
    q, k, v = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v))
    T, H, d = q.shape
    cu, nd = _cu(cu_seqlens, T)
    scale = 1.0 / np.sqrt(d) if softmax_scale is None else float(softmax_scale)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    R = T if r is None else len(r)
    o = np.zeros((R, H, d), dtype=np.float64)
    lse = np.zeros((H, R), dtype=np.float64)
    lib().or_attention_fp64(q.ctypes.data, k.ctypes.data, v.ctypes.data, T, H, d, _ptr(cu), nd,
                            int(bool(causal)), scale, _ptr(r), R, o.ctypes.data, lse.ctypes.data)
    return o, lse


def attention_fp64_backward(q, k, v, dout, cu_seqlens=None, causal=False, softmax_scale=None, o=None):
    """Gradients of the FP64 attention for an upstream gradient dout.
    With `o` given ([T, H, d], the forward's stored output), D_i = dout_i . o_i
    comes from it. Returns (dq, dk, dv), each fp64 [T, H, d]."""
    q, k, v, dout = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v, dout))
    T, H, d = q.shape
    cu, nd = _cu(cu_seqlens, T)
    scale = 1.0 / np.sqrt(d) if softmax_scale is None else float(softmax_scale)
    dq, dk, dv = (np.zeros((T, H, d), dtype=np.float64) for _ in range(3))
    if o is None:
        lib().or_attention_fp64_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, T, H, d,
                                    _ptr(cu), nd, int(bool(causal)), scale, dq.ctypes.data, dk.ctypes.data,
                                    dv.ctypes.data)
    else:
        o = np.ascontiguousarray(o, dtype=np.float64)
        assert o.shape == q.shape
        lib().or_attention_fp64_bwd_o(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, o.ctypes.data,
                                      T, H, d, _ptr(cu), nd, int(bool(causal)), scale, dq.ctypes.data,
                                      dk.ctypes.data, dv.ctypes.data)
    return dq, dk, dv


# ---- O-3 -------------------------------------------------------------------
def exp2_schraudolph(x) -> np.ndarray:
    """Schraudolph's exponential of each x (float32 values; scalar path, small arrays)."""
    xs = np.asarray(x, dtype=np.float64)
    L = lib()
    return np.array([L.or_exp2_schraudolph(float(v)) for v in xs.ravel()], dtype=np.float32).reshape(xs.shape)


def exp2_mitchell_code(x) -> np.ndarray:
    """The log-domain E4M3 code of 2^x for each x (uint8; scalar path, small arrays)."""
    xs = np.asarray(x, dtype=np.float64)
    L = lib()
    return np.array([L.or_exp2_mitchell_code(float(v)) for v in xs.ravel()], dtype=np.uint8).reshape(xs.shape)


def attention_emulate(q: QTensor, k: QTensor, v: QTensor, cu_seqlens=None, causal=False,
                      exact=False, softmax_scale=None, rows=None, quantize_p=True, ties=False, rescale_tau=0.0,
                      exp_mode=EXP_HW, lse_ties=False):
    """Quantised-operand emulation. Returns (o fp32 [R,H,d], o_bf16 u16 [R,H,d], lse fp32 [H,R]),
    and with ties=True a fourth array [R,H,d]: the tie allowance (how far E4M3
    probability codes that sit within rounding of a code boundary can move each
    output element); with lse_ties=True as well a fifth [H,R], the same for lse
    (non-zero under the log-domain P only, whose row sum adds the codes' values).
    rescale_tau: a row's reference maximum moves only when a key tile's maximum
    exceeds it by more than this (log2 units; 0 = exact).
    exp_mode: EXP_HW (2^x), EXP_SCHRAUDOLPH or EXP_MITCHELL_P."""
    T, H, d = q.codes.shape
    if q.layout == NVFP4:
        d *= 2                                         # two E2M1 codes per byte
    if q.rotated != k.rotated or (q.rotated and q.seed != k.seed):
        raise ValueError("Q and K must carry the same rotation")
    cu, nd = _cu(cu_seqlens, T)
    scale = 1.0 / np.sqrt(d) if softmax_scale is None else float(softmax_scale)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    R = T if r is None else len(r)
    o = np.zeros((R, H, d), dtype=np.float32)
    ob = np.zeros((R, H, d), dtype=np.uint16)
    lse = np.zeros((H, R), dtype=np.float32)
    amb = np.zeros((R, H, d), dtype=np.float32) if ties else None
    lamb = np.zeros((H, R), dtype=np.float32) if (ties and lse_ties) else None
    qq, kk, vv = q._qt(), k._qt(), v._qt()
    st = lib().or_attention_emulate(ctypes.byref(qq), ctypes.byref(kk), ctypes.byref(vv), T, H, d,
                                    _ptr(cu), nd, int(bool(causal)), int(bool(exact)),
                                    int(bool(q.rotated)), scale, float(rescale_tau),
                                    (QUANTIZE_P if quantize_p else 0) | _EXP_FLAGS[exp_mode],
                                    _ptr(r), R, o.ctypes.data, ob.ctypes.data, lse.ctypes.data,
                                    None if amb is None else amb.ctypes.data,
                                    None if lamb is None else lamb.ctypes.data)
    if st != 0:
        raise ValueError(f"oracle emulation rejected its arguments (status {st})")
    if lamb is not None:
        return o, ob, lse, amb, lamb
    return (o, ob, lse, amb) if ties else (o, ob, lse)


def attention_emulate_given_p(q: QTensor, k: QTensor, v: QTensor, p_codes: np.ndarray, cu_seqlens=None,
                              causal=False, exact=False, softmax_scale=None, rows=None, rescale_tau=0.0,
                              exp_mode=EXP_HW):
    """The emulation with a device's E4M3 probability codes checked and used in
    place of its own. p_codes: uint8 [H, T, stride], the code row t of head h
    gave document-local key k at [h, t, k] (0 where the row sees no key).
    Returns (o fp32 [R,H,d], o_bf16 u16 [R,H,d], lse fp32 [H,R], counts) with
    counts = {same, tie_other, wrong, masked_nonzero}: keys whose device code is
    the emulation's own, keys whose device code is the other faithful code of a
    tie, keys with any other code, and unseen keys with a non-zero code."""
    T, H, d = q.codes.shape
    if q.layout == NVFP4:
        d *= 2                                         # two E2M1 codes per byte
    if q.rotated != k.rotated or (q.rotated and q.seed != k.seed):
        raise ValueError("Q and K must carry the same rotation")
    pc = np.ascontiguousarray(p_codes, dtype=np.uint8)
    if pc.ndim != 3 or pc.shape[0] != H or pc.shape[1] != T:
        raise ValueError("p_codes must be [H, T, stride]")
    cu, nd = _cu(cu_seqlens, T)
    scale = 1.0 / np.sqrt(d) if softmax_scale is None else float(softmax_scale)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    R = T if r is None else len(r)
    o = np.zeros((R, H, d), dtype=np.float32)
    ob = np.zeros((R, H, d), dtype=np.uint16)
    lse = np.zeros((H, R), dtype=np.float32)
    counts = np.zeros(4, dtype=np.int64)
    qq, kk, vv = q._qt(), k._qt(), v._qt()
    st = lib().or_attention_emulate_given_p(ctypes.byref(qq), ctypes.byref(kk), ctypes.byref(vv), T, H, d,
                                            _ptr(cu), nd, int(bool(causal)), int(bool(exact)),
                                            int(bool(q.rotated)), scale, float(rescale_tau), _EXP_FLAGS[exp_mode],
                                            _ptr(r), R, o.ctypes.data,
                                            ob.ctypes.data, lse.ctypes.data, pc.ctypes.data, pc.shape[2],
                                            counts.ctypes.data)
    if st != 0:
        raise ValueError(f"oracle emulation rejected its arguments (status {st})")
    names = ("same", "tie_other", "wrong", "masked_nonzero")
    return o, ob, lse, {n: int(c) for n, c in zip(names, counts)}


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)
