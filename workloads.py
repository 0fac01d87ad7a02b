"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and shapes them; it holds none of the
attention or quantisation arithmetic. Both the oracle side (tests, CPU
baseline) and the CUDA side (tests, benchmark, smoke check) take their inputs
from here, so the two see the same values.

Workload recipes (numpy PCG64; seed = 1000 * workload_id + {Q: 0, K: 1, V: 2};
values drawn in fp32 and rounded to bf16 with round-to-nearest-even unless the
workload is fp32):

1 tiny       B1 H2 N256 d64, non-causal, fp32 N(0,1); E4M3 blocks of 64 tokens
2 fa3        B2 H32 N8192 d128, non-causal, N(0,1) with each entry an outlier
             N(0, sigma=10) with probability 0.001 (the 0.1%-outlier synthetic
             test of the FlashAttention-3 paper, as the "Fused attention kernel"
             page reports it); E4M3 blocks of 128 tokens
3 fa3_causal as 2, causal (default and causal-exact scaling)
4 outlier_ch B4 H16 N8448 d128, non-causal; Q, K: x_c = g_c * z + 3.0 with
             g_c = 20 on 4 channels drawn once from the seed (the same channels
             for Q and K), else 1; V N(0,1); MXFP8
5 packed     65536 tokens of packed documents with lengths
             floor(exp(U(ln 128, ln 16384))) drawn until the total reaches
             65536 (the last document takes the remainder), 32 heads, d128,
             causal, N(0,1) + 0.1% N(0,10) outliers; MXFP8, document-local
These stand in for the captured model activations the pages describe, which
are not available here.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

E4M3_TOKBLOCK, MX_ROW32, MX_COL32 = 0, 1, 2


@dataclass
class Workload:
    wid: int
    name: str
    batch: int
    heads: int
    seqlen: int
    head_dim: int
    causal: bool
    mx: bool
    block: int
    dist: str
    in_dtype: str = "bf16"
    packed_tokens: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def hadamard_seed(self) -> int:
        return 0x5EED0000 + self.wid


WORKLOADS = {
    1: Workload(1, "tiny_b1_h2_n256_d64", 1, 2, 256, 64, False, False, 64, "normal", "f32"),
    2: Workload(2, "fa3_b2_h32_n8192_d128", 2, 32, 8192, 128, False, False, 128, "outlier"),
    3: Workload(3, "fa3_causal_b2_h32_n8192_d128", 2, 32, 8192, 128, True, False, 128, "outlier"),
    4: Workload(4, "outlier_channels_b4_h16_n8448_d128_mxfp8", 4, 16, 8448, 128, False, True, 32,
                "outlier_channels"),
    5: Workload(5, "packed_docs_t65536_h32_d128_mxfp8_causal", 1, 32, 0, 128, True, True, 32,
                "outlier", packed_tokens=65536),
}


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), returned as fp32 values."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).reshape(x.shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bit patterns (uint16) of fp32 values that are already bf16-exact"""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def doc_lengths(total: int, lo: int, hi: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = []
    acc = 0
    while acc < total:
        L = int(np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi)))))
        L = min(L, total - acc)
        lens.append(L)
        acc += L
    return np.array(lens, dtype=np.int64)


def cu_from_lengths(lens) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def draw(shape, dist: str, seed: int, channels_seed: int | None = None) -> np.ndarray:
    """One seeded tensor [T, H, d] in fp32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if dist == "normal":
        return x
    if dist == "outlier":
        mask = rng.random(size=shape, dtype=np.float32) < 0.001
        n = int(mask.sum())
        x[mask] = rng.standard_normal(size=n, dtype=np.float32) * np.float32(10.0)
        return x
    if dist == "outlier_channels":
        d = shape[-1]
        crng = np.random.Generator(np.random.PCG64(channels_seed if channels_seed is not None else seed))
        ch = crng.choice(d, size=4, replace=False)
        g = np.ones(d, dtype=np.float32)
        g[ch] = 20.0
        return x * g + np.float32(3.0)
    raise ValueError(dist)


@dataclass
class Inputs:
    q: np.ndarray        # [T, H, d] fp32 values (bf16-exact unless fp32 workload)
    k: np.ndarray
    v: np.ndarray
    cu_seqlens: np.ndarray
    causal: bool
    wid: int
    in_dtype: str

    @property
    def T(self):
        return self.q.shape[0]


def make(wid: int, *, heads: int | None = None, seqlen: int | None = None, batch: int | None = None,
         lengths=None) -> Inputs:
    """Inputs for workload `wid`; heads / seqlen / batch / lengths override the
    shape for reduced-size parity cases (the distribution and seeds stay)."""
    w = WORKLOADS[wid]
    H = heads or w.heads
    d = w.head_dim
    if lengths is not None:
        lens = np.asarray(lengths, dtype=np.int64)
    elif w.packed_tokens and seqlen is None:
        lens = doc_lengths(w.packed_tokens, 128, 16384, seed=1000 * wid + 7)
    else:
        lens = np.full(batch or w.batch, seqlen or w.seqlen, dtype=np.int64)
    cu = cu_from_lengths(lens)
    T = int(cu[-1])
    vdist = "normal" if w.dist == "outlier_channels" else w.dist
    q = draw((T, H, d), w.dist, 1000 * wid + 0, channels_seed=1000 * wid + 9)
    k = draw((T, H, d), w.dist, 1000 * wid + 1, channels_seed=1000 * wid + 9)
    v = draw((T, H, d), vdist, 1000 * wid + 2)
    if w.in_dtype == "bf16":
        q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
    return Inputs(q, k, v, cu, w.causal, wid, w.in_dtype)


def attention_flops(cu_seqlens, heads: int, head_dim: int, causal: bool) -> float:
    """4 * H * d * L^2 per document, halved when causal (the causal discount of
    FLAMIA appendix E, Benchmarking Pitfalls)."""
    lens = np.diff(np.asarray(cu_seqlens, dtype=np.int64)).astype(np.float64)
    f = float(np.sum(4.0 * heads * head_dim * lens * lens))
    return f / 2.0 if causal else f
