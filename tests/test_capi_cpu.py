"""The C-ABI library loads on a machine without a GPU, exports every function
include/attn.h declares, and rejects bad arguments before touching the device.
"""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def pa():
    from precision_attention_gb300 import build
    build.build()
    import precision_attention_gb300 as pa
    pa.lib()
    return pa


def declared_functions():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(pa):
    decl = declared_functions()
    assert len(decl) >= 8
    lib = ctypes.CDLL(pa.LIB_PATH)
    for name in decl:
        assert hasattr(lib, name), name
    assert set(decl) == set(pa.EXPORTS)


def test_status_strings(pa):
    for s in range(9):
        assert pa.attn_status_string(s) and pa.attn_status_string(s) != "unknown status"
    assert pa.attn_status_string(99) == "unknown status"


def test_sizes(pa):
    T, H, d = 1000, 4, 128
    cb, sb = pa.attn_quantize_sizes(T, H, d, 1, pa.ATTN_E4M3_TOKBLOCK, 128)
    assert cb == T * H * d and sb == H * ((T + 127) // 128 + 1) * 4
    cb, sb = pa.attn_quantize_sizes(T, H, d, 3, pa.ATTN_MX_ROW32, 32)
    assert sb == H * ((T + 127) // 128 + 3) * 512
    cb, sb = pa.attn_quantize_sizes(T, H, 64, 1, pa.ATTN_E4M3_TOKBLOCK, 1)
    assert sb == H * (T + 1) * 4
    assert pa.attn_workspace_size(T, H, d, 3) % 256 == 0


def test_invalid_arguments_rejected_on_host(pa):
    L = pa.lib()
    shape = pa._Shape(100, 2, 96, 1, None)      # head_dim 96 unsupported
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.attn_quantize_sizes(ctypes.byref(shape), 0, 128, ctypes.byref(cb), ctypes.byref(sb)) == \
        pa.ATTN_ERR_UNSUPPORTED
    shape = pa._Shape(100, 2, 128, 1, None)
    assert L.attn_quantize_sizes(ctypes.byref(shape), 0, 100, ctypes.byref(cb), ctypes.byref(sb)) == \
        pa.ATTN_ERR_INVALID_ARG                  # block 100 not offered
    assert L.attn_quantize_sizes(ctypes.byref(pa._Shape(100, 2, 64, 1, None)), 1, 32, ctypes.byref(cb),
                                 ctypes.byref(sb)) == pa.ATTN_ERR_UNSUPPORTED   # MX needs d = 128
    assert L.attn_quantize_sizes(ctypes.byref(pa._Shape(100, 2, 128, 3, None)), 0, 128, ctypes.byref(cb),
                                 ctypes.byref(sb)) == pa.ATTN_ERR_INVALID_ARG   # 3 docs need cu_seqlens
    qt = pa._QT(None, None, 0, 128, 0, 0, 0)
    # null input / outputs: rejected before any CUDA call
    assert L.attn_quantize(None, 1, 256, 128, ctypes.byref(shape), 1, 1, ctypes.byref(qt), None, 0, None) == \
        pa.ATTN_ERR_INVALID_ARG
    assert L.attn_fp8_fwd(ctypes.byref(qt), ctypes.byref(qt), ctypes.byref(qt), ctypes.byref(shape), 0, 0, 0.0,
                          None, None, None, 0, None) == pa.ATTN_ERR_INVALID_ARG
    assert L.attn_bf16_fwd(None, None, None, ctypes.byref(shape), 0, 0.0, None, None, None, 0, None) == \
        pa.ATTN_ERR_INVALID_ARG
    assert L.attn_read_device_status(None, None, None) == pa.ATTN_ERR_WORKSPACE


def test_wait_limit_setting_is_host_only(pa):
    assert pa.lib().attn_set_wait_limit(1000) == pa.ATTN_OK
    assert pa.lib().attn_set_wait_limit(0) == pa.ATTN_OK     # back to the default


def test_schedule_setting_is_host_only(pa):
    L = pa.lib()
    assert L.attn_set_schedule(pa.ATTN_SCHED_TICKET) == pa.ATTN_OK
    assert L.attn_set_schedule(2) == pa.ATTN_ERR_INVALID_ARG
    assert L.attn_set_schedule(-1) == pa.ATTN_ERR_INVALID_ARG
    assert L.attn_set_schedule(pa.ATTN_SCHED_STATIC) == pa.ATTN_OK     # back to the default


def test_shape_rules_on_host(pa):
    """The shape checks every call starts with, through the two size queries (pure
    host functions: there cu_seqlens is only tested for presence, never read)."""
    L = pa.lib()
    cb, sb, wb = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    placeholder_cu = 1 << 20

    def sizes(shape, layout=0, block=128):
        return L.attn_quantize_sizes(ctypes.byref(shape), layout, block, ctypes.byref(cb), ctypes.byref(sb))

    def ws(shape):
        return L.attn_workspace_size(ctypes.byref(shape), ctypes.byref(wb))

    for T, H, nd, cu in [(0, 2, 1, None), (100, 0, 1, None), (100, 2, 0, None),   # empty shapes
                         (5, 2, 6, placeholder_cu)]:                              # more documents than tokens
        shape = pa._Shape(T, H, 128, nd, cu)
        assert sizes(shape) == pa.ATTN_ERR_INVALID_ARG and ws(shape) == pa.ATTN_ERR_INVALID_ARG
    assert sizes(pa._Shape(50000, 2, 128, 20000, placeholder_cu)) == pa.ATTN_OK   # no cap on the document count
    assert sizes(pa._Shape(1 << 26, 64, 128, 1, None)) == pa.ATTN_ERR_UNSUPPORTED          # T x H beyond int32
    assert sizes(pa._Shape(1024, 2, 128, 1024, placeholder_cu)) == pa.ATTN_OK              # one token per document
    assert sizes(pa._Shape(100, 2, 128, 1, None), layout=5, block=32) == pa.ATTN_ERR_INVALID_ARG   # no such layout
    assert sizes(pa._Shape(100, 2, 128, 1, None), layout=4, block=32) == pa.ATTN_ERR_INVALID_ARG   # NVFP4: block 128
    assert sizes(pa._Shape(100, 2, 64, 1, None), layout=4, block=128) == pa.ATTN_ERR_UNSUPPORTED   # NVFP4: d = 128
    cb4, sb4 = ctypes.c_size_t(), ctypes.c_size_t()
    shape4 = pa._Shape(1000, 2, 128, 3, placeholder_cu)
    assert L.attn_quantize_sizes(ctypes.byref(shape4), 4, 128, ctypes.byref(cb4), ctypes.byref(sb4)) == pa.ATTN_OK
    ntcap = (1000 + 127) // 128 + 3
    assert cb4.value == 1000 * 2 * 64                                      # two E2M1 codes per byte
    assert sb4.value == (2 * ntcap * 4 + 1023) // 1024 * 1024 + 2 * ntcap * 1024
    assert sizes(pa._Shape(100, 2, 64, 1, None), layout=3, block=1) == pa.ATTN_ERR_UNSUPPORTED     # MX: d = 128
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    shape = pa._Shape(100, 2, 128, 3, placeholder_cu)
    assert L.attn_quantize_sizes(ctypes.byref(shape), 3, 1, ctypes.byref(cb), ctypes.byref(sb)) == pa.ATTN_OK
    assert cb.value == 100 * 2 * 128 and sb.value == 2 * (100 + 3)         # one exponent byte per token and head
    assert sizes(pa._Shape(100, 2, 128, 1, None), layout=1, block=64) == pa.ATTN_OK   # block: E4M3 layout only
    shape = pa._Shape(100, 2, 128, 1, None)
    assert L.attn_quantize_sizes(ctypes.byref(shape), 0, 128, None, None) == pa.ATTN_ERR_INVALID_ARG
    assert L.attn_workspace_size(ctypes.byref(shape), None) == pa.ATTN_ERR_INVALID_ARG
    assert L.attn_workspace_size(None, ctypes.byref(wb)) == pa.ATTN_ERR_INVALID_ARG


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="uses placeholder device pointers; only run where no GPU could be reached")
def test_seed_mismatch_and_layout_rules_on_host(pa):
    """Q/K rotation mismatch and exact-mode rules are refused before launch.
    Placeholder aligned pointers pass the null checks and are never used."""
    L = pa.lib()
    fake = 1 << 20
    shape = pa._Shape(256, 2, 128, 1, None)
    q = pa._QT(fake, fake, 0, 128, 0, 1, 7)
    k = pa._QT(fake, fake, 0, 128, 0, 1, 8)
    v = pa._QT(fake, fake, 0, 128, 0, 0, 0)
    ws_small = 16
    # workspace too small is reported before the rotation check
    assert L.attn_fp8_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(shape), 0, 0, 0.0,
                          fake, fake, fake, ws_small, None) == pa.ATTN_ERR_WORKSPACE
    big = pa.attn_workspace_size(256, 2, 128, 1)
    assert L.attn_fp8_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(shape), 0, 0, 0.0,
                          fake, fake, fake, big, None) == pa.ATTN_ERR_SEED_MISMATCH
    k.hadamard_seed = 7
    # causal-exact needs causal and block 1 everywhere
    assert L.attn_fp8_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(shape), 0, 1, 0.0,
                          fake, fake, fake, big, None) == pa.ATTN_ERR_INVALID_ARG
    assert L.attn_fp8_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(shape), 1, 1, 0.0,
                          fake, fake, fake, big, None) == pa.ATTN_ERR_INVALID_ARG
    # MX Q/K with an E4M3 V is refused
    qm = pa._QT(fake, fake, 1, 32, 0, 1, 7)
    km = pa._QT(fake, fake, 1, 32, 0, 1, 7)
    assert L.attn_fp8_fwd(ctypes.byref(qm), ctypes.byref(km), ctypes.byref(v), ctypes.byref(shape), 0, 0, 0.0,
                          fake, fake, fake, big, None) == pa.ATTN_ERR_INVALID_ARG
    # MX causal-exact needs V with one exponent per token, and causal
    vcol = pa._QT(fake, fake, 2, 32, 0, 0, 0)
    vtok = pa._QT(fake, fake, 3, 1, 0, 0, 0)
    assert L.attn_fp8_fwd(ctypes.byref(qm), ctypes.byref(km), ctypes.byref(vcol), ctypes.byref(shape), 1, 1, 0.0,
                          fake, fake, fake, big, None) == pa.ATTN_ERR_INVALID_ARG
    assert L.attn_fp8_fwd(ctypes.byref(qm), ctypes.byref(km), ctypes.byref(vtok), ctypes.byref(shape), 0, 1, 0.0,
                          fake, fake, fake, big, None) == pa.ATTN_ERR_INVALID_ARG


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="uses placeholder device pointers; only run where no GPU could be reached")
def test_exp_mode_rules_on_host(pa):
    """attn_fp8_fwd_ex: an exp_mode outside the enum is an invalid argument; the
    bit-level modes are refused (unsupported) with causal-exact, per-column E4M3
    blocks, per-token MX V or head_dim 64 -- all before any device call."""
    L = pa.lib()
    fake = 1 << 20

    def call(q, k, v, shape, causal, exact, mode):
        ws = pa.attn_workspace_size(shape.total_tokens, shape.heads, shape.head_dim, 1)
        return L.attn_fp8_fwd_ex(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(shape), causal,
                                 exact, 0.0, mode, fake, fake, fake, ws, None)

    s128 = pa._Shape(256, 2, 128, 1, None)
    e = pa._QT(fake, fake, 0, 128, 0, 1, 7)
    ev = pa._QT(fake, fake, 0, 128, 0, 0, 0)
    assert call(e, e, ev, s128, 0, 0, 3) == pa.ATTN_ERR_INVALID_ARG
    assert call(e, e, ev, s128, 0, 0, -1) == pa.ATTN_ERR_INVALID_ARG
    e1 = pa._QT(fake, fake, 0, 1, 0, 1, 7)
    e1v = pa._QT(fake, fake, 0, 1, 0, 0, 0)
    assert call(e1, e1, e1v, s128, 1, 1, pa.ATTN_EXP_SCHRAUDOLPH) == pa.ATTN_ERR_UNSUPPORTED   # causal-exact
    e64 = pa._QT(fake, fake, 0, 64, 0, 1, 7)
    e64v = pa._QT(fake, fake, 0, 64, 0, 0, 0)
    assert call(e64, e64, e64v, s128, 0, 0, pa.ATTN_EXP_MITCHELL_P) == pa.ATTN_ERR_UNSUPPORTED  # blocks < tile
    s64 = pa._Shape(256, 2, 64, 1, None)
    assert call(e, e, ev, s64, 0, 0, pa.ATTN_EXP_SCHRAUDOLPH) == pa.ATTN_ERR_UNSUPPORTED        # head_dim 64
    m = pa._QT(fake, fake, 1, 32, 0, 1, 7)
    mtok = pa._QT(fake, fake, 3, 1, 0, 0, 0)
    assert call(m, m, mtok, s128, 1, 0, pa.ATTN_EXP_MITCHELL_P) == pa.ATTN_ERR_UNSUPPORTED      # per-token V
    # the other checks keep their order: a small workspace is still reported first
    assert L.attn_fp8_fwd_ex(ctypes.byref(e), ctypes.byref(e), ctypes.byref(ev), ctypes.byref(s128), 0, 0, 0.0,
                             pa.ATTN_EXP_SCHRAUDOLPH, fake, fake, fake, 16, None) == pa.ATTN_ERR_WORKSPACE


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="uses placeholder device pointers; only run where no GPU could be reached")
def test_nvfp4_forward_rules_on_host(pa):
    """The mixed NVFP4/FP8 forward: NVFP4 Q needs NVFP4 K and an E4M3 V in 128-token
    blocks (else invalid), head_dim 128 and no causal-exact mode (else unsupported)."""
    L = pa.lib()
    fake = 1 << 20
    shape = pa._Shape(256, 2, 128, 1, None)
    big = pa.attn_workspace_size(256, 2, 128, 1)

    def call(q, k, v, shp=shape, causal=0, exact=0):
        return L.attn_fp8_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(shp), causal, exact,
                              0.0, fake, fake, fake, big, None)

    nq = pa._QT(fake, fake, pa.ATTN_NVFP4, 128, 0, 1, 7)
    e = pa._QT(fake, fake, 0, 128, 0, 1, 7)
    ev = pa._QT(fake, fake, 0, 128, 0, 0, 0)
    ev64 = pa._QT(fake, fake, 0, 64, 0, 0, 0)
    mcol = pa._QT(fake, fake, pa.ATTN_MX_COL32, 32, 0, 0, 0)
    assert call(nq, e, ev) == pa.ATTN_ERR_INVALID_ARG            # K must be NVFP4 too
    assert call(nq, nq, ev64) == pa.ATTN_ERR_INVALID_ARG         # V blocks of 128 tokens
    assert call(nq, nq, mcol) == pa.ATTN_ERR_INVALID_ARG         # V in E4M3
    assert call(nq, nq, ev, causal=1, exact=1) == pa.ATTN_ERR_UNSUPPORTED
    nk8 = pa._QT(fake, fake, pa.ATTN_NVFP4, 128, 0, 1, 8)
    assert call(nq, nk8, ev) == pa.ATTN_ERR_SEED_MISMATCH


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="uses placeholder device pointers; only run where no GPU could be reached")
def test_quantize_qkv_layout_sets_on_host(pa):
    """attn_quantize_qkv takes only the operand sets the forward accepts (E4M3 with one
    block for all three; MX rows with MX columns or per-token V; NVFP4 with E4M3 V in
    128-token blocks): any other set is an invalid argument, refused before the
    workspace check, which every accepted set reaches (here a 16-byte workspace)."""
    L = pa.lib()
    fake = 1 << 20
    shape = pa._Shape(256, 2, 128, 1, None)

    def call(q, k, v, ws=16, dt=1, stride=256):
        return L.attn_quantize_qkv(fake, fake, fake, dt, stride, 128, ctypes.byref(shape), 1, 7, ctypes.byref(q),
                                   ctypes.byref(k), ctypes.byref(v), fake, ws, None)

    def qt(layout, block):
        return pa._QT(fake, fake, layout, block, 0, 0, 0)

    E, R, C, TOK, NV = (pa.ATTN_E4M3_TOKBLOCK, pa.ATTN_MX_ROW32, pa.ATTN_MX_COL32, pa.ATTN_MX_TOKEN,
                        pa.ATTN_NVFP4)
    accepted = [(qt(E, 128), qt(E, 128), qt(E, 128)), (qt(E, 1), qt(E, 1), qt(E, 1)),
                (qt(E, 64), qt(E, 64), qt(E, 64)), (qt(R, 32), qt(R, 32), qt(C, 32)),
                (qt(R, 32), qt(R, 32), qt(TOK, 1)), (qt(NV, 128), qt(NV, 128), qt(E, 128))]
    refused = [(qt(E, 128), qt(E, 64), qt(E, 128)), (qt(E, 128), qt(E, 128), qt(E, 64)),
               (qt(R, 32), qt(E, 128), qt(C, 32)), (qt(R, 32), qt(R, 32), qt(R, 32)),
               (qt(R, 32), qt(R, 32), qt(E, 128)), (qt(C, 32), qt(C, 32), qt(C, 32)),
               (qt(NV, 128), qt(NV, 128), qt(E, 64)), (qt(NV, 128), qt(E, 128), qt(E, 128)),
               (qt(E, 128), qt(E, 128), qt(NV, 128))]
    for q, k, v in accepted:
        assert call(q, k, v) == pa.ATTN_ERR_WORKSPACE, (q.layout, k.layout, v.layout, q.block, v.block)
    for q, k, v in refused:
        assert call(q, k, v) == pa.ATTN_ERR_INVALID_ARG, (q.layout, k.layout, v.layout, q.block, v.block)
    assert call(qt(E, 128), qt(E, 128), qt(E, 128), dt=2) == pa.ATTN_ERR_INVALID_ARG      # no such dtype
    assert call(qt(E, 128), qt(E, 128), qt(E, 128), stride=100) == pa.ATTN_ERR_INVALID_ARG  # 200-byte rows
    assert L.attn_quantize_qkv(fake, None, fake, 1, 256, 128, ctypes.byref(shape), 1, 7,
                               ctypes.byref(qt(E, 128)), ctypes.byref(qt(E, 128)), ctypes.byref(qt(E, 128)),
                               fake, 16, None) == pa.ATTN_ERR_INVALID_ARG                 # null K input
    assert L.attn_quantize_qkv(fake, fake, fake, 1, 256, 128, ctypes.byref(shape), 1, 7, ctypes.byref(qt(E, 128)),
                               None, ctypes.byref(qt(E, 128)), fake, 16, None) == pa.ATTN_ERR_INVALID_ARG


def test_test_build_exports_the_probability_dump_and_the_timed_library_does_not(pa):
    """libpa_gb300_pdump.so (include/attn_pdump.h) is the parity tests' build: it
    exports every call of include/attn.h plus attn_pdump_set; the library that
    is timed exports no such call."""
    from precision_attention_gb300 import build
    build.build(pdump=True)
    src = open(os.path.join(ROOT, "include", "attn_pdump.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    extra = sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))
    assert extra == ["attn_pdump_set"]
    test_lib = ctypes.CDLL(pa.PDUMP_LIB_PATH)
    for name in declared_functions() + extra:
        assert hasattr(test_lib, name), name
    assert not hasattr(ctypes.CDLL(pa.LIB_PATH), "attn_pdump_set")
    L = pa.pdump_lib()
    assert L.attn_pdump_set(None, 0) == pa.ATTN_OK
    assert L.attn_pdump_set(16, 100) == pa.ATTN_ERR_INVALID_ARG      # stride not a multiple of 128


def test_backward_arguments_rejected_on_host(pa):
    """attn_bf16_bwd: every synchronous check returns before any CUDA call."""
    L = pa.lib()
    T, H = 1000, 4
    fwd = pa.attn_workspace_size(T, H, 128, 3)
    bwd = pa.attn_bwd_workspace_size(T, H, 128, 3)
    # the forward's workspace plus lse log2(e) and D per (head, tile, row)
    assert bwd % 256 == 0 and bwd >= fwd + 2 * 4 * 128 * H * ((T + 127) // 128 + 3)
    fake = ctypes.c_void_p(1 << 20)                     # 16-byte aligned, never dereferenced
    odd = ctypes.c_void_p((1 << 20) + 2)
    ws = ctypes.c_void_p(1 << 24)
    cu = ctypes.c_void_p(1 << 21)

    def call(shape, ptrs=None, wsp=ws, nbytes=bwd, scale=0.0):
        p = ptrs or [fake] * 9
        return L.attn_bf16_bwd(p[0], p[1], p[2], p[3], p[4], p[5], ctypes.byref(shape), 1, scale,
                               p[6], p[7], p[8], wsp, nbytes, None)

    shape = pa._Shape(T, H, 128, 3, cu)
    for i in range(9):
        ptrs = [fake] * 9
        ptrs[i] = None
        assert call(shape, ptrs) == pa.ATTN_ERR_INVALID_ARG, i
        ptrs[i] = odd
        assert call(shape, ptrs) == pa.ATTN_ERR_INVALID_ARG, i
    assert call(shape, scale=float("nan")) == pa.ATTN_ERR_INVALID_ARG
    assert call(pa._Shape(T, H, 96, 3, cu)) == pa.ATTN_ERR_UNSUPPORTED       # d = 64 or 128 only
    assert call(shape, nbytes=bwd - 256) == pa.ATTN_ERR_WORKSPACE
    assert call(shape, nbytes=fwd) == pa.ATTN_ERR_WORKSPACE                  # the forward's is too small
    assert call(shape, wsp=ctypes.c_void_p((1 << 24) + 128)) == pa.ATTN_ERR_WORKSPACE
    assert call(pa._Shape(T, H, 128, 3, None)) == pa.ATTN_ERR_INVALID_ARG    # 3 documents need cu_seqlens
