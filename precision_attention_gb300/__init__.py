"""Python binding of the GB300 fused low-precision attention library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libpa_gb300.so`` behind the C ABI of ``include/attn.h``. PyTorch
provides device memory and streams. There is no fallback: if the library is
missing or fails to load, every call raises.

The functions keep the C names:

    attn_quantize_sizes, attn_workspace_size, attn_fwd_workspace_size,
    attn_quantize, attn_quantize_qkv, attn_fp8_fwd, attn_fp8_fwd_ex,
    attn_bf16_fwd, attn_bwd_workspace_size, attn_bf16_bwd, attn_read_device_status,
    attn_status_string, attn_set_schedule, attn_device_sm_count
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa_gb300.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_DEVICE_TIMEOUT = 4
ATTN_ERR_NONFINITE = 5
ATTN_ERR_SEED_MISMATCH = 6
ATTN_ERR_BAD_SEQLENS = 7
ATTN_ERR_WORKSPACE = 8

ATTN_IN_F32, ATTN_IN_BF16 = 0, 1
ATTN_E4M3_TOKBLOCK, ATTN_MX_ROW32, ATTN_MX_COL32, ATTN_MX_TOKEN, ATTN_NVFP4 = 0, 1, 2, 3, 4
ATTN_MX_RULE_NOSAT, ATTN_MX_RULE_OCP_FLOOR = 0, 1
# include/attn.h: the FP8 forward at head_dim 128 moves a row's reference maximum
# only by more than this (log2 units); the other paths use the exact running max
ATTN_RESCALE_THRESHOLD = 0.75
# include/attn.h attn_exp_mode: the probabilities' exponential of the FP8 forward
ATTN_EXP_HW, ATTN_EXP_SCHRAUDOLPH, ATTN_EXP_MITCHELL_P = 0, 1, 2
# include/attn.h attn_schedule: the pair kernel's work order
ATTN_SCHED_STATIC, ATTN_SCHED_TICKET = 0, 1


def rescale_threshold(head_dim: int, fp8: bool = True) -> float:
    """The reference-maximum threshold the forward uses for this head_dim."""
    return ATTN_RESCALE_THRESHOLD if (fp8 and head_dim == 128) else 0.0

EXPORTS = ("attn_quantize_sizes", "attn_workspace_size", "attn_fwd_workspace_size", "attn_quantize",
           "attn_quantize_qkv", "attn_fp8_fwd",
           "attn_fp8_fwd_ex", "attn_bf16_fwd", "attn_read_device_status", "attn_status_string", "attn_device_sm_count", "attn_fp8_fwd_noalloc",
           "attn_set_wait_limit", "attn_set_schedule", "attn_bwd_workspace_size", "attn_bf16_bwd")


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} (status {status})")


class _Shape(ctypes.Structure):
    _fields_ = [("total_tokens", ctypes.c_int32), ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("num_docs", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p)]


class _QT(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("layout", ctypes.c_int32),
                ("block", ctypes.c_int32), ("mx_rule", ctypes.c_int32), ("rotated", ctypes.c_int32),
                ("hadamard_seed", ctypes.c_uint64)]


_lock = threading.Lock()
_lib = None
_pdump = None
PDUMP_LIB_PATH = os.path.join(_HERE, "libpa_gb300_pdump.so")


def _load(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    vp, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    S, Q = ctypes.POINTER(_Shape), ctypes.POINTER(_QT)
    L.attn_quantize_sizes.argtypes = [S, i32, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.attn_workspace_size.argtypes = [S, ctypes.POINTER(sz)]
    L.attn_fwd_workspace_size.argtypes = [S, i32, ctypes.POINTER(sz)]
    L.attn_quantize.argtypes = [vp, i32, i64, i64, S, i32, u64, Q, vp, sz, vp]
    L.attn_quantize_qkv.argtypes = [vp, vp, vp, i32, i64, i64, S, i32, u64, Q, Q, Q, vp, sz, vp]
    L.attn_fp8_fwd.argtypes = [Q, Q, Q, S, i32, i32, ctypes.c_float, vp, vp, vp, sz, vp]
    L.attn_fp8_fwd_ex.argtypes = [Q, Q, Q, S, i32, i32, ctypes.c_float, i32, vp, vp, vp, sz, vp]
    L.attn_bf16_fwd.argtypes = [vp, vp, vp, S, i32, ctypes.c_float, vp, vp, vp, sz, vp]
    L.attn_bwd_workspace_size.argtypes = [S, ctypes.POINTER(sz)]
    L.attn_bf16_bwd.argtypes = [vp, vp, vp, vp, vp, vp, S, i32, ctypes.c_float, vp, vp, vp, vp, sz, vp]
    L.attn_read_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    L.attn_fp8_fwd_noalloc.argtypes = [Q, Q, Q, S, i32, i32, ctypes.c_float, vp, vp, vp, vp]
    L.attn_fp8_fwd_noalloc.restype = ctypes.c_int32
    L.attn_status_string.argtypes = [i32]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_device_sm_count.argtypes = []
    L.attn_set_wait_limit.argtypes = [i64]
    L.attn_set_schedule.argtypes = [i32]
    for f in ("attn_quantize_sizes", "attn_workspace_size", "attn_fwd_workspace_size", "attn_quantize",
              "attn_quantize_qkv",              "attn_fp8_fwd", "attn_fp8_fwd_ex", "attn_bf16_fwd", "attn_read_device_status",
              "attn_device_sm_count", "attn_set_wait_limit", "attn_set_schedule", "attn_bwd_workspace_size",
              "attn_bf16_bwd"):
        getattr(L, f).restype = ctypes.c_int32
    if hasattr(L, "attn_pdump_set"):
        L.attn_pdump_set.argtypes = [vp, i64]
        L.attn_pdump_set.restype = ctypes.c_int32
    return L


def lib() -> ctypes.CDLL:
    """Load libpa_gb300.so (raises when it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with precision_attention_gb300.build.build()")
            _lib = _load(LIB_PATH)
    return _lib


def pdump_lib() -> ctypes.CDLL:
    """Load the test build libpa_gb300_pdump.so (include/attn_pdump.h): the same
    library whose FP8 kernels also report every probability code they hand to
    the P V product. For parity tests only."""
    global _pdump
    with _lock:
        if _pdump is None:
            if not os.path.exists(PDUMP_LIB_PATH):
                raise RuntimeError(f"{PDUMP_LIB_PATH} is missing: build it with build.build(pdump=True)")
            _pdump = _load(PDUMP_LIB_PATH)
    return _pdump


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def attn_device_sm_count() -> int:
    return int(lib().attn_device_sm_count())


def attn_set_schedule(schedule: int) -> None:
    """ATTN_SCHED_STATIC (default) or ATTN_SCHED_TICKET (items taken just in time) for
    later forward calls; process-wide."""
    _check(lib().attn_set_schedule(int(schedule)), "attn_set_schedule")


def attn_set_wait_limit(cycles: int) -> None:
    """Limit (SM cycles) of the attention kernels' bounded waits for later calls;
    cycles <= 0 restores the default. A short limit exercises the timeout path."""
    _check(lib().attn_set_wait_limit(int(cycles)), "attn_set_wait_limit")


def _check(st: int, where: str):
    if st != ATTN_OK:
        raise AttnError(st, where)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def make_shape(T: int, H: int, d: int, cu_seqlens: torch.Tensor | None) -> _Shape:
    nd = 1 if cu_seqlens is None else int(cu_seqlens.numel()) - 1
    ptr = None if cu_seqlens is None else cu_seqlens.data_ptr()
    return _Shape(T, H, d, nd, ptr)


def attn_quantize_sizes(T: int, H: int, d: int, num_docs: int, layout: int, block: int) -> tuple[int, int]:
    s = _Shape(T, H, d, num_docs, None if num_docs == 1 else 1)
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().attn_quantize_sizes(ctypes.byref(s), layout, block, ctypes.byref(cb), ctypes.byref(sb)),
           "attn_quantize_sizes")
    return cb.value, sb.value


def attn_workspace_size(T: int, H: int, d: int, num_docs: int) -> int:
    s = _Shape(T, H, d, num_docs, None if num_docs == 1 else 1)
    b = ctypes.c_size_t()
    _check(lib().attn_workspace_size(ctypes.byref(s), ctypes.byref(b)), "attn_workspace_size")
    return b.value


def attn_fwd_workspace_size(T: int, H: int, d: int, num_docs: int, causal: bool) -> int:
    s = _Shape(T, H, d, num_docs, None if num_docs == 1 else 1)
    b = ctypes.c_size_t()
    _check(lib().attn_fwd_workspace_size(ctypes.byref(s), int(causal), ctypes.byref(b)), "attn_fwd_workspace_size")
    return b.value


def attn_bwd_workspace_size(T: int, H: int, d: int, num_docs: int) -> int:
    s = _Shape(T, H, d, num_docs, None if num_docs == 1 else 1)
    b = ctypes.c_size_t()
    _check(lib().attn_bwd_workspace_size(ctypes.byref(s), ctypes.byref(b)), "attn_bwd_workspace_size")
    return b.value


def bwd_workspace(T: int, H: int, d: int, num_docs: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace buffer for attn_bf16_bwd."""
    return torch.zeros(attn_bwd_workspace_size(T, H, d, num_docs), dtype=torch.uint8, device=device)


def workspace(T: int, H: int, d: int, num_docs: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace buffer (torch allocates it; the library never does)."""
    n = attn_workspace_size(T, H, d, num_docs)
    return torch.zeros(n, dtype=torch.uint8, device=device)


@dataclass
class QTensor:
    codes: torch.Tensor        # uint8 [T, H, d]
    scales: torch.Tensor       # fp32 [H, nb_cap] or uint8 [H, nt_cap, 512]
    layout: int
    block: int
    mx_rule: int = ATTN_MX_RULE_NOSAT
    rotated: int = 0
    hadamard_seed: int = 0

    def dims(self):
        """(T, H, head_dim) of the operand (NVFP4 codes hold two channels per byte)."""
        T, H, w = self.codes.shape
        return T, H, 2 * w if self.layout == ATTN_NVFP4 else w

    def _c(self) -> _QT:
        return _QT(self.codes.data_ptr(), self.scales.data_ptr(), self.layout, self.block, self.mx_rule,
                   self.rotated, self.hadamard_seed)


def empty_qtensor(T: int, H: int, d: int, num_docs: int, layout: int, block: int,
                  mx_rule: int = ATTN_MX_RULE_NOSAT, device="cuda") -> QTensor:
    cb, sb = attn_quantize_sizes(T, H, d, num_docs, layout, block)
    if layout == ATTN_NVFP4:   # two E2M1 codes per byte; scales: one byte buffer (see nvfp4_scales)
        return QTensor(torch.empty((T, H, d // 2), dtype=torch.uint8, device=device),
                       torch.empty((sb,), dtype=torch.uint8, device=device), layout, block, mx_rule)
    codes = torch.empty((T, H, d), dtype=torch.uint8, device=device)
    if layout == ATTN_E4M3_TOKBLOCK:
        scales = torch.empty((H, sb // (4 * H)), dtype=torch.float32, device=device)
    elif layout == ATTN_MX_TOKEN:
        scales = torch.empty((H, sb // H), dtype=torch.uint8, device=device)
    else:
        scales = torch.empty((H, sb // (512 * H), 512), dtype=torch.uint8, device=device)
    return QTensor(codes, scales, layout, block, mx_rule)


def nvfp4_scales(qt: QTensor, num_docs: int):
    """Views of an ATTN_NVFP4 scales buffer (include/attn.h): the fp32 block scales
    [H, nt_cap] and the 1024-byte scale-factor tiles [H, nt_cap, 1024]."""
    T, H = qt.codes.shape[0], qt.codes.shape[1]
    ntcap = (T + 127) // 128 + num_docs
    off = (H * ntcap * 4 + 1023) // 1024 * 1024
    st = qt.scales[:H * ntcap * 4].view(torch.float32).view(H, ntcap)
    sf = qt.scales[off:off + H * ntcap * 1024].view(H, ntcap, 1024)
    return st, sf


def attn_quantize(x: torch.Tensor, cu_seqlens: torch.Tensor | None, layout: int, block: int = 128,
                  rotate: bool = False, hadamard_seed: int = 0, mx_rule: int = ATTN_MX_RULE_NOSAT,
                  ws: torch.Tensor | None = None, out: QTensor | None = None, stream=None) -> QTensor:
    """Rotate (optionally) and quantise x [T, H, d] (bf16 or fp32, channels contiguous)."""
    assert x.is_cuda and x.dim() == 3 and x.stride(2) == 1
    T, H, d = x.shape
    nd = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if ws is None:
        ws = workspace(T, H, d, nd, x.device)
    if out is None:
        out = empty_qtensor(T, H, d, nd, layout, block, mx_rule, x.device)
    dt = ATTN_IN_BF16 if x.dtype == torch.bfloat16 else ATTN_IN_F32
    assert x.dtype in (torch.bfloat16, torch.float32)
    shape = make_shape(T, H, d, cu_seqlens)
    c = out._c()
    _check(lib().attn_quantize(x.data_ptr(), dt, x.stride(0), x.stride(1), ctypes.byref(shape), int(bool(rotate)),
                               hadamard_seed & (2 ** 64 - 1), ctypes.byref(c), ws.data_ptr(), ws.numel(),
                               _stream(stream)), "attn_quantize")
    out.rotated, out.hadamard_seed = c.rotated, c.hadamard_seed
    return out


def attn_quantize_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor | None,
                      layout: int, block: int = 128, layout_v: int | None = None, block_v: int | None = None,
                      rotate: bool = False, hadamard_seed: int = 0, mx_rule: int = ATTN_MX_RULE_NOSAT,
                      ws: torch.Tensor | None = None, outs: tuple | None = None, stream=None):
    """Quantise Q, K (layout, block; rotated when `rotate`) and V (layout_v, block_v;
    by default the same as Q and K) in one launch. q, k, v: [T, H, d], one dtype and
    one stride pair. Returns (q8, k8, v8) as three attn_quantize calls would."""
    assert q.is_cuda and q.dim() == 3 and q.stride(2) == 1
    assert k.shape == q.shape and v.shape == q.shape and k.dtype == q.dtype and v.dtype == q.dtype
    assert k.stride() == q.stride() and v.stride() == q.stride()
    assert q.dtype in (torch.bfloat16, torch.float32)
    T, H, d = q.shape
    nd = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    layout_v = layout if layout_v is None else layout_v
    block_v = block if block_v is None else block_v
    if ws is None:
        ws = workspace(T, H, d, nd, q.device)
    if outs is None:
        outs = (empty_qtensor(T, H, d, nd, layout, block, mx_rule, q.device),
                empty_qtensor(T, H, d, nd, layout, block, mx_rule, q.device),
                empty_qtensor(T, H, d, nd, layout_v, block_v, mx_rule, q.device))
    dt = ATTN_IN_BF16 if q.dtype == torch.bfloat16 else ATTN_IN_F32
    shape = make_shape(T, H, d, cu_seqlens)
    cs = [o._c() for o in outs]
    _check(lib().attn_quantize_qkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), dt, q.stride(0), q.stride(1),
                                   ctypes.byref(shape), int(bool(rotate)), hadamard_seed & (2 ** 64 - 1),
                                   ctypes.byref(cs[0]), ctypes.byref(cs[1]), ctypes.byref(cs[2]), ws.data_ptr(),
                                   ws.numel(), _stream(stream)), "attn_quantize_qkv")
    for o, c in zip(outs, cs):
        o.rotated, o.hadamard_seed = c.rotated, c.hadamard_seed
    return tuple(outs)


def attn_fp8_fwd(q: QTensor, k: QTensor, v: QTensor, cu_seqlens: torch.Tensor | None, causal: bool = False,
                 causal_exact: bool = False, softmax_scale: float = 0.0, ws: torch.Tensor | None = None,
                 out: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """FP8 attention forward. Returns (o bf16 [T, H, d], lse fp32 [H, T])."""
    return attn_fp8_fwd_ex(q, k, v, cu_seqlens, causal, causal_exact, softmax_scale, ATTN_EXP_HW, ws, out, lse,
                           stream)


def attn_fp8_fwd_ex(q: QTensor, k: QTensor, v: QTensor, cu_seqlens: torch.Tensor | None, causal: bool = False,
                    causal_exact: bool = False, softmax_scale: float = 0.0, exp_mode: int = ATTN_EXP_HW,
                    ws: torch.Tensor | None = None, out: torch.Tensor | None = None,
                    lse: torch.Tensor | None = None, stream=None):
    """FP8 attention forward with a choice of the probabilities' exponential
    (ATTN_EXP_HW: attn_fp8_fwd itself; ATTN_EXP_SCHRAUDOLPH, ATTN_EXP_MITCHELL_P:
    the bit-level inference forms). Returns (o bf16 [T, H, d], lse fp32 [H, T])."""
    T, H, d = q.dims()
    nd = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = q.codes.device
    if ws is None:
        ws = workspace(T, H, d, nd, dev)
    if out is None:
        out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    shape = make_shape(T, H, d, cu_seqlens)
    cq, ck, cv = q._c(), k._c(), v._c()
    if exp_mode == ATTN_EXP_HW:
        _check(lib().attn_fp8_fwd(ctypes.byref(cq), ctypes.byref(ck), ctypes.byref(cv), ctypes.byref(shape),
                                  int(bool(causal)), int(bool(causal_exact)), float(softmax_scale), out.data_ptr(),
                                  lse.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)), "attn_fp8_fwd")
    else:
        _check(lib().attn_fp8_fwd_ex(ctypes.byref(cq), ctypes.byref(ck), ctypes.byref(cv), ctypes.byref(shape),
                                     int(bool(causal)), int(bool(causal_exact)), float(softmax_scale), int(exp_mode),
                                     out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)),
               "attn_fp8_fwd_ex")
    return out, lse


def attn_bf16_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor | None,
                  causal: bool = False, softmax_scale: float = 0.0, ws: torch.Tensor | None = None,
                  out: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """BF16 attention forward over contiguous bf16 [T, H, d] q, k, v."""
    assert q.dtype == k.dtype == v.dtype == torch.bfloat16
    assert q.is_contiguous() and k.is_contiguous() and v.is_contiguous()
    T, H, d = q.shape
    nd = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if ws is None:
        ws = workspace(T, H, d, nd, q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    shape = make_shape(T, H, d, cu_seqlens)
    _check(lib().attn_bf16_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(shape), int(bool(causal)),
                               float(softmax_scale), out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(),
                               _stream(stream)), "attn_bf16_fwd")
    return out, lse


def attn_bf16_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, dout: torch.Tensor,
                  lse: torch.Tensor, cu_seqlens: torch.Tensor | None, causal: bool = False,
                  softmax_scale: float = 0.0, ws: torch.Tensor | None = None, outs=None, stream=None):
    """BF16 attention backward: (dq, dk, dv) for the upstream gradient dout, from
    the forward's inputs, its bf16 output o and its lse (attn_bf16_fwd)."""
    ts = (q, k, v, o, dout)
    assert all(t.dtype == torch.bfloat16 and t.is_contiguous() for t in ts)
    assert lse.dtype == torch.float32 and lse.is_contiguous()
    T, H, d = q.shape
    nd = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if ws is None:
        ws = bwd_workspace(T, H, d, nd, q.device)
    if outs is None:
        outs = tuple(torch.empty_like(q) for _ in range(3))
    dq, dk, dv = outs
    shape = make_shape(T, H, d, cu_seqlens)
    _check(lib().attn_bf16_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                               lse.data_ptr(), ctypes.byref(shape), int(bool(causal)), float(softmax_scale),
                               dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), ws.numel(),
                               _stream(stream)), "attn_bf16_bwd")
    return dq, dk, dv


def attn_fp8_fwd_noalloc(q: QTensor, k: QTensor, v: QTensor, cu_seqlens: torch.Tensor | None,
                         causal: bool = False, causal_exact: bool = False, softmax_scale: float = 0.0,
                         out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                         status: torch.Tensor | None = None, stream=None):
    """attn_fp8_fwd without a workspace: scratch comes from the library's fixed
    16 MiB device array (for callers that cannot allocate; see include/attn.h).
    `status`, if given, is a 1-element int32 device tensor that receives the
    call's device status word. Returns (o, lse)."""
    T, H, d = q.dims()
    dev = q.codes.device
    if out is None:
        out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    shape = make_shape(T, H, d, cu_seqlens)
    cq, ck, cv = q._c(), k._c(), v._c()
    _check(lib().attn_fp8_fwd_noalloc(ctypes.byref(cq), ctypes.byref(ck), ctypes.byref(cv), ctypes.byref(shape),
                                      int(bool(causal)), int(bool(causal_exact)), float(softmax_scale),
                                      out.data_ptr(), lse.data_ptr(),
                                      None if status is None else status.data_ptr(), _stream(stream)),
           "attn_fp8_fwd_noalloc")
    return out, lse


def attn_fp8_fwd_pdump(q: QTensor, k: QTensor, v: QTensor, cu_seqlens: torch.Tensor | None, key_stride: int,
                       causal: bool = False, causal_exact: bool = False, softmax_scale: float = 0.0,
                       exp_mode: int = ATTN_EXP_HW):
    """attn_fp8_fwd through the test build, which also writes every E4M3
    probability code it hands to the P V MMA. Returns (o, lse, codes) with
    codes uint8 [H, T, key_stride]: codes[h, t, k] is what row t of head h gave
    document-local key k (0 where nothing was written)."""
    L = pdump_lib()
    T, H, d = q.dims()
    nd = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = q.codes.device
    ws = workspace(T, H, d, nd, dev)
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    codes = torch.zeros((H, T, key_stride), dtype=torch.uint8, device=dev)
    shape = make_shape(T, H, d, cu_seqlens)
    cq, ck, cv = q._c(), k._c(), v._c()
    _check(L.attn_pdump_set(codes.data_ptr(), key_stride), "attn_pdump_set")
    try:
        _check(L.attn_fp8_fwd_ex(ctypes.byref(cq), ctypes.byref(ck), ctypes.byref(cv), ctypes.byref(shape),
                                 int(bool(causal)), int(bool(causal_exact)), float(softmax_scale), int(exp_mode),
                                 out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), _stream(None)),
               "attn_fp8_fwd_ex (test build)")
        flags = ctypes.c_uint32()
        st = L.attn_read_device_status(ws.data_ptr(), _stream(None), ctypes.byref(flags))
        if st != ATTN_OK:
            raise AttnError(st, "attn_fp8_fwd (test build), device status")
    finally:
        L.attn_pdump_set(None, 0)
    return out, lse, codes


def attn_read_device_status(ws: torch.Tensor, stream=None) -> tuple[int, int]:
    """Synchronise, read and clear the workspace status word. Returns (status, raw flags)."""
    flags = ctypes.c_uint32()
    st = lib().attn_read_device_status(ws.data_ptr(), _stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)


def default_softmax_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
