// quant.cu -- fused rotate-and-quantise kernel (one launch per tensor).
//
// Sources: "Fused attention kernel", 8-bit forward pass (e4m3 codes, block
// quantisation, incoherent processing: random sign diagonal times Hadamard,
// applied to Q and K); FLAMIA section 2 (MX: 32-element blocks, one shared
// E8M0 scale) and section 4.3 (fused quantisation: one launch instead of many).
//
// Work unit: one 128-token tile of one document and one head. The kernel is
// persistent (two CTAs per SM) and double-buffers units in shared memory: a
// single TMA copy brings the next tile's 128 rows while the current one is
// rotated and encoded, so the HBM stream never waits for the arithmetic.
//
// Thread layout inside a unit: a row (token, head) of d channels is held by 8
// consecutive lanes, EPL = d / 8 channels each (lane sub-index sl holds
// channels sl*EPL .. sl*EPL+EPL-1); a warp holds 4 rows, the 8 warps 32 rows
// per pass, 4 passes per unit. The Hadamard transform runs its stages
// h = 1, 2, 4, ... in that order: in registers while h < EPL, then across the
// 8 lanes with shuffles (lane ^ 1, ^ 2, ^ 4). Every butterfly is
// (a, b) -> (a + b, a - b) in fp32 round-to-nearest, so the result does not
// depend on how elements are spread over lanes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "params.h"
#include "pdl.cuh"
#include "ptx.cuh"

namespace pa {

// SplitMix64 output j (0-based) of the stream started at `seed`: the state
// after j + 1 increments of the golden-ratio constant, then the mix.
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint32_t j) {
    uint64_t z = seed + 0x9E3779B97F4A7C15ULL * (uint64_t)(j + 1);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

template <int EPL>
__device__ __forceinline__ uint32_t sign_mask(const QuantParams& p, int sl) {
    uint32_t m = 0;
    if (p.rotate) {
#pragma unroll
        for (int i = 0; i < EPL; i++)
            if (splitmix64_at(p.seed, sl * EPL + i) >> 63) m |= 1u << i;
    }
    return m;
}

// EPL channels of one row from the shared-memory tile [128 rows][d] (bf16 or fp32)
template <int EPL, int ELT>
__device__ __forceinline__ void smem_row(const uint8_t* tile, int row, int sl, float (&v)[EPL]) {
    constexpr int D = EPL * 8;
    const uint4* src = reinterpret_cast<const uint4*>(tile + (row * D + sl * EPL) * ELT);
    if constexpr (ELT == 2) {
#pragma unroll
        for (int q = 0; q < EPL / 8; q++) {
            const uint4 u = src[q];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                v[q * 8 + 2 * k] = __uint_as_float(w[k] << 16);
                v[q * 8 + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < EPL / 4; q++) {
            const uint4 u = src[q];
            v[q * 4 + 0] = __uint_as_float(u.x);
            v[q * 4 + 1] = __uint_as_float(u.y);
            v[q * 4 + 2] = __uint_as_float(u.z);
            v[q * 4 + 3] = __uint_as_float(u.w);
        }
    }
}

// sign flip then the Walsh-Hadamard stages (see the file comment). Stage h = 1
// pairs neighbours held in one register pair; stages 2 .. EPL/2 run two
// butterflies per packed f32x2 add and fused multiply-add (fma(b, +-1, a) is
// a +- b rounded once, so every butterfly is the same IEEE operation as before).
//
// head_dim 64 (EPL 8): the three cross-lane stages compute o + s v with s = +-1
// from a full shuffle of the partner's values, leaving channel 8 l + r in lane l,
// register r.
//
// head_dim 128 (EPL 16): each cross-lane stage is a half exchange. Lane bit j
// (stage h = 16 << j) swaps places with register bit j + 1, whose stage (h = 2 << j)
// is done: a lane sends the value at register bit j + 1 = 1, keeps the one at 0,
// and the butterfly then runs in registers. For the kept and sent values to be the
// right ones, lanes with bit j set store stage 2 << j's outputs swapped ((a - b,
// a + b) into registers (r, r + 2^(j+1))), which is the same two operations with
// the sign operand exchanged. After the exchange a lane with bit j clear holds
// a = kept, b = received, one with bit j set a = received, b = kept: a + b is
// kept + received in both (IEEE addition commutes, signed zeros included), and
// a - b = fma(received, -s, s * kept) with s = +1 or -1, the product exact. Half
// as many shuffles as the full form; the values are bit-identical to the
// transform's, and lane l, register r ends holding Hadamard output channel
// (r & 1) | (l << 1) | ((r >> 1) << 4) (stored channel 16 l + r: the two 3-bit
// fields of the channel index at bits 1-3 and 4-6 swapped).
template <int EPL>
__device__ __forceinline__ void rotate_row(float (&v)[EPL], uint32_t smask, int lane) {
#pragma unroll
    for (int i = 0; i < EPL; i++) v[i] = __uint_as_float(__float_as_uint(v[i]) ^ (((smask >> i) & 1u) << 31));
#pragma unroll
    for (int i = 0; i < EPL; i += 2) {
        const float a = v[i], b = v[i + 1];
        v[i] = __fadd_rn(a, b);
        v[i + 1] = __fsub_rn(a, b);
    }
    if constexpr (EPL == 16) {
#pragma unroll
        for (int h = 2; h < 16; h <<= 1) {
            const float sg = (lane & (h >> 1)) ? -1.0f : 1.0f;   // lane bit j for h = 2 << j
            const float2 s2 = make_float2(sg, sg), n2 = make_float2(-sg, -sg);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                if (!(i & h)) {
                    const float2 a = make_float2(v[i], v[i + 1]), b = make_float2(v[i + h], v[i + h + 1]);
                    const float2 lo = __ffma2_rn(b, s2, a), hi = __ffma2_rn(b, n2, a);
                    v[i] = lo.x;
                    v[i + 1] = lo.y;
                    v[i + h] = hi.x;
                    v[i + h + 1] = hi.y;
                }
            }
        }
#pragma unroll
        for (int m = 1, K = 2; m < 8; m <<= 1, K <<= 1) {
            const float sg = (lane & m) ? -1.0f : 1.0f;
            const float2 s2 = make_float2(sg, sg), n2 = make_float2(-sg, -sg);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                if (!(i & K)) {
                    const float r0 = __shfl_xor_sync(0xFFFFFFFFu, v[i + K], m);
                    const float r1 = __shfl_xor_sync(0xFFFFFFFFu, v[i + K + 1], m);
                    const float2 keep = make_float2(v[i], v[i + 1]), recv = make_float2(r0, r1);
                    const float2 sum = __fadd2_rn(keep, recv);
                    const float2 dif = __ffma2_rn(recv, n2, __fmul2_rn(keep, s2));
                    v[i] = sum.x;
                    v[i + 1] = sum.y;
                    v[i + K] = dif.x;
                    v[i + K + 1] = dif.y;
                }
            }
        }
    } else {
        const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
        for (int h = 2; h < EPL; h <<= 1) {
#pragma unroll
            for (int i = 0; i < EPL; i += 2) {
                if (!(i & h)) {
                    const float2 a = make_float2(v[i], v[i + 1]), b = make_float2(v[i + h], v[i + h + 1]);
                    const float2 sum = __fadd2_rn(a, b), dif = __ffma2_rn(b, neg1, a);
                    v[i] = sum.x;
                    v[i + 1] = sum.y;
                    v[i + h] = dif.x;
                    v[i + h + 1] = dif.y;
                }
            }
        }
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) {
            const float sg = (lane & m) ? -1.0f : 1.0f;
            const float2 s2 = make_float2(sg, sg);
#pragma unroll
            for (int i = 0; i < EPL; i += 2) {
                const float o0 = __shfl_xor_sync(0xFFFFFFFFu, v[i], m);
                const float o1 = __shfl_xor_sync(0xFFFFFFFFu, v[i + 1], m);
                const float2 r = __ffma2_rn(make_float2(v[i], v[i + 1]), s2, make_float2(o0, o1));
                v[i] = r.x;
                v[i + 1] = r.y;
            }
        }
    }
}

// max of |a| over values, NaN-propagating (a NaN or infinity anywhere leaves a
// non-finite result, which the caller reports)
__device__ __forceinline__ float amax_nan(float m, float a) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(a)));
    return r;
}

// max(a, b), NaN-propagating (an infinity or NaN on either side survives)
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// max(m, |a|, |b|), NaN-propagating
__device__ __forceinline__ float amax_nan2(float m, float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(m), "f"(fabsf(a)), "f"(fabsf(b)));
    return r;
}

__device__ __forceinline__ bool finite_abs(float a) { return a <= 3.402823466e38f; }

// E8M0 exponent X of a block amax (NOSAT = smallest X with amax <= 448 * 2^X;
// OCP_FLOOR = floor(log2 amax) - 8), clamped to [-127, 127]
__device__ __forceinline__ int e8m0_exponent(float amax, int rule) {
    if (!(amax > 0.0f)) return -127;
    const uint32_t u = __float_as_uint(amax);
    const int ef = (int)((u >> 23) & 0xFF);
    if (ef == 0) return -127;                       // subnormal amax: X far below -127
    const int E = ef - 127;
    const uint32_t frac = u & 0x7FFFFFu;
    const int X = (rule == 1) ? E - 8 : (frac <= 0x600000u ? E - 8 : E - 7);   // 1.75 = 1 + 0x600000 / 2^23
    return X < -127 ? -127 : (X > 127 ? 127 : X);
}
__device__ __forceinline__ float pow2_neg(int X) {   // 2^-X for X in [-127, 126]
    return __uint_as_float((uint32_t)(127 - X) << 23);
}

// two fp32 -> two E2M1 codes in one byte (round to nearest even, beyond 6 saturates):
// `lo` in the low nibble
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}
// value of a non-negative E4M3 code (0x00..0x7E): exponent field e, mantissa m
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const uint32_t e = b >> 3, m = b & 7u;
    return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
}

template <int EPL>
__device__ __forceinline__ void store_codes(uint8_t* dst, const float (&y)[EPL], float mul) {
    uint32_t w[EPL / 4];
    const float2 m2 = make_float2(mul, mul);
#pragma unroll
    for (int i = 0; i < EPL / 4; i++) {
        const float2 a = __fmul2_rn(make_float2(y[4 * i], y[4 * i + 1]), m2);
        const float2 b = __fmul2_rn(make_float2(y[4 * i + 2], y[4 * i + 3]), m2);
        w[i] = pack_e4m3x4(a.x, a.y, b.x, b.y);
    }
    if constexpr (EPL == 16) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    }
}

// ---------------------------------------------------------------------------
// In-CTA document table: starts, prefix counts of 128-token tiles and of
// scale blocks. Returns false (after flagging the status word) when
// cu_seqlens is malformed.
struct DocTable {
    int32_t start[MAX_DOCS + 1];
    int32_t off_tile[MAX_DOCS + 1];   // exclusive prefix of ceil(L / 128); [nd] = total tiles
    int32_t off_blk[MAX_DOCS + 1];    // exclusive prefix of ceil(L / block)
};
// the table wherever it lives (shared memory, or the workspace for large batches)
struct DocTablePtrs {
    int32_t *start, *off_tile, *off_blk;
};

// Builds the table with the calling CTA (any number of documents, four per thread
// per round). On malformed cu_seqlens it flags the status word, leaves a table
// without tiles (off_tile[nd] = 0) and returns false.
__device__ bool build_doc_table(const QuantParams& p, DocTablePtrs tab, int* scratch) {
    int* bad = scratch;          // [1]
    int* wsum = scratch + 1;     // [2][32]: tile and block totals per warp (up to 32 warps)
    const int tid = threadIdx.x, nd = p.nd, nw = blockDim.x >> 5;
    const int lane = tid & 31, warp = tid >> 5;
    if (tid == 0) *bad = 0;
    __syncthreads();
    int carry_t = 0, carry_b = 0;
    for (int base = 0; base < nd; base += 4 * blockDim.x) {   // each thread: 4 consecutive documents
        int ct[4], cb[4], at = 0, ab = 0;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = base + tid * 4 + k;
            ct[k] = cb[k] = 0;
            if (i < nd) {
                const int st = p.cu ? p.cu[i] : 0, e = p.cu ? p.cu[i + 1] : p.T;
                tab.start[i] = st;
                if (e < st) *bad = 1;
                const int L = e > st ? e - st : 0;
                ct[k] = (L + 127) / 128;
                cb[k] = (L + p.block - 1) / p.block;
            }
            at += ct[k];
            ab += cb[k];
        }
        int it = at, ib = ab;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int xt = __shfl_up_sync(0xFFFFFFFFu, it, o);
            const int xb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
            if (lane >= o) { it += xt; ib += xb; }
        }
        if (lane == 31) { wsum[warp] = it; wsum[32 + warp] = ib; }
        __syncthreads();
        int bt = 0, bb = 0, tt = 0, tb = 0;
        for (int w = 0; w < nw; w++) {
            if (w < warp) { bt += wsum[w]; bb += wsum[32 + w]; }
            tt += wsum[w];
            tb += wsum[32 + w];
        }
        int rt = carry_t + bt + it - at, rb = carry_b + bb + ib - ab;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = base + tid * 4 + k;
            if (i < nd) { tab.off_tile[i] = rt; tab.off_blk[i] = rb; }
            rt += ct[k];
            rb += cb[k];
        }
        carry_t += tt;
        carry_b += tb;
        __syncthreads();   // wsum is reused by the next chunk
    }
    if (tid == 0) {
        const int c0 = p.cu ? p.cu[0] : 0, cn = p.cu ? p.cu[nd] : p.T;
        if (c0 != 0 || cn != p.T) *bad = 1;
        tab.start[nd] = cn;
        tab.off_tile[nd] = carry_t;
        tab.off_blk[nd] = carry_b;
    }
    __syncthreads();
    if (*bad) {
        if (tid == 0) {
            atomicOr(p.status, ST_BAD_SEQLENS);
            tab.off_tile[nd] = 0;
        }
        return false;
    }
    return true;
}

// The table of a batch with more documents than the quantiser's CTAs keep in
// shared memory, written once into the workspace ahead of the quantiser.
__global__ void __launch_bounds__(1024) doc_table_kernel(QuantParams p) {
    __shared__ int scratch[1 + 64];
    const DocTablePtrs tab{p.gtab, p.gtab + (p.nd + 1), p.gtab + 2 * (p.nd + 1)};
    build_doc_table(p, tab, scratch);
}

__device__ __forceinline__ int find_doc(const int32_t* off, int nd, int u) {
    int lo = 0, hi = nd - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

enum { QM_E4M3_BLOCK = 0, QM_E4M3_ROW = 1, QM_MX_ROW = 2, QM_MX_COL = 3, QM_MX_TOK = 4, QM_NVFP4 = 5 };

constexpr int QUANT_THREADS = 256;

// shared memory of the quantise kernel (dynamic; the two input stages first),
// every offset aligned for what it holds (TMA destinations 128 B, mbarriers 8 B)
// NST input stages: one tile in flight while the other is processed (a third stage
// of 32 KB, with two CTAs per SM, measured slower)
template <int EPL, int ELT>
struct QuantSmem {
    static constexpr int STAGE = 128 * EPL * 8 * ELT;   // 128 rows x d elements
    static constexpr int NST = 2;
    static constexpr int OFF_TAB = NST * STAGE;
    static constexpr int OFF_SCRATCH = (OFF_TAB + (int)sizeof(DocTable) + 127) / 128 * 128;   // 96 ints
    static constexpr int OFF_RED = OFF_SCRATCH + 96 * 4;                                     // float[2][8] + spare
    static constexpr int OFF_XS = OFF_RED + 4 * 8 * 128 * 4;                                 // int[4][128]
    static constexpr int OFF_BAR = OFF_XS + 4 * 128 * 4;                                     // uint64[NST]
    static constexpr int OFF_FLAG = OFF_BAR + NST * 8;                                       // int[2]
    static constexpr int BYTES = OFF_FLAG + 2 * 4 + 128;                                     // + base alignment
    static_assert(STAGE % 128 == 0 && OFF_SCRATCH % 128 == 0, "TMA destinations need 128-byte alignment");
    static_assert(OFF_XS % 16 == 0 && OFF_BAR % 8 == 0, "int4 reads and mbarriers need alignment");
};

// Layouts whose unit holds the whole tile in registers before its one barrier:
// the tile's stage is free after that barrier (quant_unit calls `release` there).
template <int QM, int HOLD>
constexpr bool quant_early_release() {
    return (QM == QM_E4M3_BLOCK && HOLD == 4) || QM == QM_NVFP4;
}

// One 128-token tile (unit g of head h) of one tensor, staged in shared memory at
// `tile`. rc counts the CTA's block reductions (red[] alternates between two
// eight-float slots, so one barrier per reduction suffices); `release()` is called
// by every thread once no thread reads the tile any more, in the layouts of
// quant_early_release().
template <int EPL, int ELT, int QM, int HOLD, class Rel>
__device__ __forceinline__ void quant_unit(const QuantParams& p, const DocTablePtrs& tab, const uint8_t* tile,
                                           float* red, int* xs, uint32_t smask, bool& nonfin, int g,
                                           int h, int doc, int s0, int L, int t0, int& rc, Rel& release) {
    constexpr int D = EPL * 8;
    const int H = p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, sl = lane & 7, rw = lane >> 3;
    (void)xs;
    (void)doc;
    if constexpr (QM == QM_E4M3_BLOCK) {
        constexpr int NBLK = 4 / HOLD;
#pragma unroll 1
        for (int blk = 0; blk < NBLK; blk++) {
            if (NBLK > 1 && t0 + blk * HOLD * 32 >= L) break;   // block past the document end (uniform)
            float y[HOLD][EPL];
            float amax = 0.0f;
#pragma unroll
            for (int hp = 0; hp < HOLD; hp++) {
                const int row = (blk * HOLD + hp) * 32 + warp * 4 + rw;
                smem_row<EPL, ELT>(tile, row, sl, y[hp]);
                if (t0 + row >= L) {
#pragma unroll
                    for (int i = 0; i < EPL; i++) y[hp][i] = 0.0f;
                }
                if (p.rotate) rotate_row<EPL>(y[hp], smask, lane);
#pragma unroll
                for (int i = 0; i < EPL; i += 2) amax = amax_nan2(amax, y[hp][i], y[hp][i + 1]);
            }
            const bool tbad = !finite_abs(amax);   // NaN or infinity in this thread's rows
            if (tbad) {
                nonfin = true;
                amax = 0.0f;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            float* rb = red + 8 * (rc++ & 1);
            if (lane == 0) rb[warp] = amax;
            const bool bad = __syncthreads_or(tbad) != 0;
            if constexpr (quant_early_release<QM, HOLD>()) release();
            amax = rb[0];
#pragma unroll
            for (int w = 1; w < 8; w++) amax = fmaxf(amax, rb[w]);
            // one IEEE division per thread: even lanes 448 / amax (the codes' multiplier),
            // odd lanes amax / 448 (the scale), the multiplier then shared from lane 0
            const bool odd = lane & 1;
            float dv = 0.0f;
            if (bad) dv = odd ? __int_as_float(0x7FC00000) : 0.0f;
            else if (amax > 0.0f) dv = __fdiv_rn(odd ? amax : 448.0f, odd ? 448.0f : amax);
            const float inv = __shfl_sync(0xFFFFFFFFu, dv, 0);
            if (tid == 1) {
                const int b = tab.off_blk[doc] + (t0 + blk * HOLD * 32) / (HOLD * 32);
                static_cast<float*>(p.scales)[(long long)h * p.scale_cap + b] = dv;
            }
#pragma unroll
            for (int hp = 0; hp < HOLD; hp++) {
                const int row = (blk * HOLD + hp) * 32 + warp * 4 + rw;
                if (t0 + row < L)
                    store_codes<EPL>(p.codes + ((long long)(s0 + t0 + row) * H + h) * D + sl * EPL, y[hp], inv);
            }
        }
    } else if constexpr (QM == QM_NVFP4) {
        // the 128-token tile is the fp32 block: amax over the tile gives s_t = amax / 2688
        // and inv = 448 / amax; each thread's 16 channels of a row are one group: its
        // E4M3 scale sf = E4M3(max |y inv|) and E2M1 codes of y inv (6 / sf), the scale
        // byte at its place in the MMA-ready tile (groups 4 kk .. 4 kk + 3 in tile kk)
        static_assert(EPL == 16, "NVFP4 groups are one thread's 16 channels");
        float y[4][EPL];
        float amax = 0.0f;
#pragma unroll
        for (int hp = 0; hp < 4; hp++) {
            const int row = hp * 32 + warp * 4 + rw;
            smem_row<EPL, ELT>(tile, row, sl, y[hp]);
            if (t0 + row >= L) {
#pragma unroll
                for (int i = 0; i < EPL; i++) y[hp][i] = 0.0f;
            }
            if (p.rotate) rotate_row<EPL>(y[hp], smask, lane);
#pragma unroll
            for (int i = 0; i < EPL; i += 2) amax = amax_nan2(amax, y[hp][i], y[hp][i + 1]);
        }
        const bool tbad = !finite_abs(amax);
        if (tbad) {
            nonfin = true;
            amax = 0.0f;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        float* rb = red + 8 * (rc++ & 1);
        if (lane == 0) rb[warp] = amax;
        const bool bad = __syncthreads_or(tbad) != 0;
        static_assert(quant_early_release<QM, HOLD>(), "the NVFP4 unit frees its stage itself");
        release();
        amax = rb[0];
#pragma unroll
        for (int w = 1; w < 8; w++) amax = fmaxf(amax, rb[w]);
        float inv = 0.0f, st_scale = 0.0f;
        if (bad) st_scale = __int_as_float(0x7FC00000);
        else if (amax > 0.0f) {
            inv = __fdiv_rn(448.0f, amax);
            st_scale = __fdiv_rn(amax, 2688.0f);
        }
        if (tid == 0) static_cast<float*>(p.scales)[(long long)h * p.scale_cap + g] = st_scale;
        uint8_t* sft = p.sf16 + ((long long)h * p.scale_cap + g) * 1024 + (sl >> 2) * 512;
#pragma unroll
        for (int hp = 0; hp < 4; hp++) {
            const int row = hp * 32 + warp * 4 + rw;
            // the group's largest |y inv| is fl(max |y| x inv): rounding is monotone
            float gy = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; i += 2) gy = amax_nan2(gy, y[hp][i], y[hp][i + 1]);
            const float gmax = __fmul_rn(gy, inv);
            const uint32_t sfb = cvt_e4m3x2(gmax, 0.0f) & 0xFFu;
            const float sfv = e4m3_value(sfb);
            const float r6 = red[16 + sfb];   // 6 / sf (table built at the kernel's start)
            uint32_t w[2] = {0u, 0u};
            if (sfv > 0.0f) {
                const float2 inv2 = make_float2(inv, inv), r62 = make_float2(r6, r6);
#pragma unroll
                for (int i = 0; i < EPL; i += 2) {
                    const float2 z = __fmul2_rn(make_float2(y[hp][i], y[hp][i + 1]), inv2);   // y x inv
                    const float2 c = __fmul2_rn(z, r62);                                      // then x 6 / sf
                    w[i >> 3] |= cvt_e2m1x2(c.x, c.y) << (4 * (i & 7));
                }
            }
            sft[(row % 32) * 16 + (row / 32) * 4 + (sl & 3)] = (uint8_t)sfb;   // this group's scale byte
            if (t0 + row < L)
                *reinterpret_cast<uint2*>(p.codes + ((long long)(s0 + t0 + row) * H + h) * (D / 2) + sl * 8) =
                    make_uint2(w[0], w[1]);
        }
    } else if constexpr (QM == QM_E4M3_ROW) {
        // The thread's four rows (one per pass) are held, so that the warp's 16 rows take
        // their two IEEE divisions in one step: lane l serves row (pass (l & 15) / 4,
        // group l & 3), lanes 0-15 forming 448 / amax and lanes 16-31 amax / 448 (one
        // division with lane-chosen operands), instead of all 8 lanes of a row
        // repeating both, pass after pass.
        float y[4][EPL];
        float am[4];   // each held row's maximum over its 8 lanes (NaN-propagating)
#pragma unroll
        for (int ps = 0; ps < 4; ps++) {
            const int row = ps * 32 + warp * 4 + rw;
            smem_row<EPL, ELT>(tile, row, sl, y[ps]);
            if (p.rotate) rotate_row<EPL>(y[ps], smask, lane);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; i += 2) amax = amax_nan2(amax, y[ps][i], y[ps][i + 1]);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) amax = max_nan(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            am[ps] = amax;
        }
        const int ri = lane & 15, pr = ri >> 2, gr = ri & 3;
        float a = 0.0f;
#pragma unroll
        for (int ps = 0; ps < 4; ps++) {
            const float t = __shfl_sync(0xFFFFFFFFu, am[ps], gr * 8);
            if (ps == pr) a = t;
        }
        const bool first = lane < 16;
        float dv = 0.0f;   // 448 / amax (the codes' multiplier) or amax / 448 (the scale)
        if (!finite_abs(a)) {
            if (!first) dv = __int_as_float(0x7FC00000);
        } else if (a > 0.0f) {
            dv = __fdiv_rn(first ? 448.0f : a, first ? a : 448.0f);
        }
        {   // block 1: the block index of a token is the token itself
            const int row = pr * 32 + warp * 4 + gr;
            if (!first && t0 + row < L) static_cast<float*>(p.scales)[(long long)h * p.scale_cap + s0 + t0 + row] = dv;
        }
#pragma unroll
        for (int ps = 0; ps < 4; ps++) {
            const float inv = __shfl_sync(0xFFFFFFFFu, dv, ps * 4 + rw);   // this thread's row, pass ps
            const int row = ps * 32 + warp * 4 + rw;
            if (t0 + row < L) {
                if (!finite_abs(am[ps])) nonfin = true;
                store_codes<EPL>(p.codes + ((long long)(s0 + t0 + row) * H + h) * D + sl * EPL, y[ps], inv);
            }
        }
    } else if constexpr (QM == QM_MX_TOK) {
        // one E8M0 exponent per (token, head) over all d channels (the causal-exact
        // MX mode's V): scale byte at the token's own column
#pragma unroll
        for (int ps = 0; ps < 4; ps++) {
            const int row = ps * 32 + warp * 4 + rw;
            const bool valid = t0 + row < L;
            float y[EPL];
            smem_row<EPL, ELT>(tile, row, sl, y);
            if (p.rotate) rotate_row<EPL>(y, smask, lane);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; i += 2) amax = amax_nan2(amax, y[i], y[i + 1]);
            // the row's maximum over its 8 lanes; a NaN or infinity in any lane survives
            // the NaN-propagating reduction and marks the row
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) amax = max_nan(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            const bool bad = !finite_abs(amax);
            if (bad) amax = 0.0f;
            if (valid) {
                if (bad) nonfin = true;
                const int X = e8m0_exponent(amax, p.mx_rule);
                if (sl == 0)
                    static_cast<uint8_t*>(p.scales)[(long long)h * p.scale_cap + s0 + t0 + row] = (uint8_t)(X + 127);
                store_codes<EPL>(p.codes + ((long long)(s0 + t0 + row) * H + h) * D + sl * EPL, y, pow2_neg(X));
            }
        }
    } else if constexpr (QM == QM_MX_ROW) {
        uint8_t* sct = static_cast<uint8_t*>(p.scales) + ((long long)h * p.scale_cap + g) * 512;
#pragma unroll
        for (int ps = 0; ps < 4; ps++) {
            const int r = ps * 32 + warp * 4 + rw;
            const bool valid = t0 + r < L;
            float y[EPL];
            smem_row<EPL, ELT>(tile, r, sl, y);
            if (p.rotate) rotate_row<EPL>(y, smask, lane);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; i += 2) amax = amax_nan2(amax, y[i], y[i + 1]);
            amax = max_nan(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));   // the 32-channel group's two lanes
            const bool bad = !finite_abs(amax);
            if (bad) amax = 0.0f;
            if (bad && valid) nonfin = true;
            const int X = valid ? e8m0_exponent(amax, p.mx_rule) : 0;
            // the group's scale byte, written by its first lane (group sl / 2 of the row)
            if ((sl & 1) == 0) sct[(r % 32) * 16 + (r / 32) * 4 + (sl >> 1)] = (uint8_t)(X + 127);
            if (valid)
                store_codes<EPL>(p.codes + ((long long)(s0 + t0 + r) * H + h) * D + sl * EPL, y, pow2_neg(X));
        }
    } else {   // QM_MX_COL
        // Column maxima straight from the staged tile: warp w takes group w / 2 and
        // channel pairs 32 (w % 2) .. + 31, one pair per lane, and scans the group's
        // 32 rows (one 32-bit bf16 pair or 64-bit fp32 pair per row: consecutive
        // words across the warp). No shuffles and one barrier. Each column's
        // multiplier 2^-X goes to shared memory as a float, four channels per
        // 16-byte slot ordered [group][slot of the lane's channels][lane of the
        // row], so that the row pass reads it conflict-free, one float4 per four
        // codes; the codes are then written row-parallel as in the other layouts.
        constexpr int NI = EPL / 4;                                  // float4 slots per lane and row
        float* xf = reinterpret_cast<float*>(xs);                    // [4][NI][8][4]
        auto xf_at = [&](int gi, int c) { return ((gi * NI + (c % EPL) / 4) * 8 + c / EPL) * 4 + (c & 3); };
        uint8_t* sct = static_cast<uint8_t*>(p.scales) + ((long long)h * p.scale_cap + g) * 512;
        {
            const int gi = warp >> 1, c = 2 * (32 * (warp & 1) + lane);   // first channel of the pair
            const int nrow = min(32, L - t0 - gi * 32);                     // rows inside the document
            float m0 = 0.0f, m1 = 0.0f;
            auto pair_at = [&](int r, float& v0, float& v1) {
                const int row = gi * 32 + r;
                if constexpr (ELT == 2) {
                    const uint32_t w2 = *reinterpret_cast<const uint32_t*>(tile + (row * D + c) * 2);
                    v0 = __uint_as_float(w2 << 16);
                    v1 = __uint_as_float(w2 & 0xFFFF0000u);
                } else {
                    const float2 f2 = *reinterpret_cast<const float2*>(tile + (row * D + c) * 4);
                    v0 = f2.x;
                    v1 = f2.y;
                }
            };
            int r = 0;
#pragma unroll 4
            for (; r + 1 < nrow; r += 2) {
                float a0, a1, b0, b1;
                pair_at(r, a0, a1);
                pair_at(r + 1, b0, b1);
                m0 = amax_nan2(m0, a0, b0);
                m1 = amax_nan2(m1, a1, b1);
            }
            if (r < nrow) {
                float a0, a1;
                pair_at(r, a0, a1);
                m0 = amax_nan(m0, a0);
                m1 = amax_nan(m1, a1);
            }
            if (!finite_abs(m0)) { nonfin = true; m0 = 0.0f; }
            if (!finite_abs(m1)) { nonfin = true; m1 = 0.0f; }
            const bool inside = nrow > 0;                    // groups past the document end: 127
            const int X0 = inside ? e8m0_exponent(m0, p.mx_rule) : 0;
            const int X1 = inside ? e8m0_exponent(m1, p.mx_rule) : 0;
            *reinterpret_cast<float2*>(xf + xf_at(gi, c)) = make_float2(pow2_neg(X0), pow2_neg(X1));
            sct[(c % 32) * 16 + (c / 32) * 4 + gi] = (uint8_t)(X0 + 127);
            sct[((c + 1) % 32) * 16 + ((c + 1) / 32) * 4 + gi] = (uint8_t)(X1 + 127);
        }
        __syncthreads();
#pragma unroll 1
        for (int gi = 0; gi < 4; gi++) {
            const int row = gi * 32 + warp * 4 + rw;
            if (t0 + row < L) {
                float y[EPL];
                smem_row<EPL, ELT>(tile, row, sl, y);
                uint32_t w4[EPL / 4];
#pragma unroll
                for (int i = 0; i < NI; i++) {
                    const float4 m4 = *reinterpret_cast<const float4*>(xf + ((gi * NI + i) * 8 + sl) * 4);
                    const float2 a = __fmul2_rn(make_float2(y[4 * i], y[4 * i + 1]), make_float2(m4.x, m4.y));
                    const float2 b = __fmul2_rn(make_float2(y[4 * i + 2], y[4 * i + 3]), make_float2(m4.z, m4.w));
                    w4[i] = pack_e4m3x4(a.x, a.y, b.x, b.y);
                }
                if constexpr (EPL == 16) {
                    *reinterpret_cast<uint4*>(p.codes + ((long long)(s0 + t0 + row) * H + h) * D + sl * EPL) =
                        make_uint4(w4[0], w4[1], w4[2], w4[3]);
                } else {
                    *reinterpret_cast<uint2*>(p.codes + ((long long)(s0 + t0 + row) * H + h) * D + sl * EPL) =
                        make_uint2(w4[0], w4[1]);
                }
            }
        }
    }}

// Units [ubeg, uend) of one tensor, stride gridDim.x, through the two-stage copy
// pipeline (stage k & 1); unit u is unit u - base of the tensor `p` describes.
// `issue` starts the copy of a later unit (of any tensor) into a freed stage.
// Returns false when a copy wait ran out.
template <int EPL, int ELT, int QM, int HOLD, class Issue>
__device__ __forceinline__ bool quant_range(const QuantParams& p, const DocTablePtrs& tab, uint8_t* sm,
                                            uint64_t* full, float* red, int* xs, volatile int* abort,
                                            uint32_t smask, bool& nonfin, int ubeg, int uend, int base, int n_units,
                                            int& k, int& rc, Issue& issue) {
    using S = QuantSmem<EPL, ELT>;
    const int H = p.H, nd = p.nd;
    constexpr int NST = S::NST;
    for (int u = ubeg; u < uend; u += gridDim.x, k++) {
        const int st = k % NST;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (k / NST) & 1, abort, 4000000000LL))) return false;
        const uint8_t* tile = sm + st * S::STAGE;
        const int uu = u - base;
        const int g = uu / H, h = uu % H;
        const int doc = find_doc(tab.off_tile, nd, g);
        const int s0 = tab.start[doc], L = tab.start[doc + 1] - s0;
        const int t0 = (g - tab.off_tile[doc]) * 128;      // first local token of the tile
        // the stage takes unit u + NST G once no thread reads it any more
        auto release = [&]() {
            if (threadIdx.x == 0 && u + NST * (int)gridDim.x < n_units) issue(u + NST * gridDim.x, st);
        };
        quant_unit<EPL, ELT, QM, HOLD>(p, tab, tile, red, xs, smask, nonfin, g, h, doc, s0, L, t0, rc, release);
        if constexpr (!quant_early_release<QM, HOLD>()) {
            __syncthreads();                                   // every read of this stage is done
            release();
        }
    }
    return true;
}

// One kernel for every layout. QM_E4M3_BLOCK: blocks of HOLD*32 tokens (32,
// 64 or 128), amax over the block's rows, scale = amax / 448, codes of
// y * (448 / amax). QM_E4M3_ROW: the same per (token, head). QM_MX_ROW: E8M0
// per (token, 32 channels). QM_MX_COL: E8M0 per (32 tokens, channel). MX scale
// bytes go to the unit's 512-byte tile at (r % 32) * 16 + (r / 32) * 4 + g;
// rows or groups past the document end get 127. QM_MX_TOK: E8M0 per (token,
// head) over all channels, one byte per token.
template <int EPL, int ELT, int QM, int HOLD, int QMV, int HOLDV, int NT>
__global__ void __launch_bounds__(QUANT_THREADS, 2)
    quant_tile_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                      const __grid_constant__ CUtensorMap tm2, const __grid_constant__ QuantParams p0,
                      const __grid_constant__ QuantParams p1, const __grid_constant__ QuantParams p2) {
    // NT = 1: one tensor (p0, layout QM); 3: Q, K (p0, p1, layout QM) and V (p2, layout
    // QMV) in one launch, the units of the three tensors one after another
    constexpr int ntens = NT;
    using S = QuantSmem<EPL, ELT>;
    // the forward's work-list kernel, if it comes next, touches nothing this one
    // reads or writes: it may run beside this kernel's last tiles
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    DocTable& stab = *reinterpret_cast<DocTable*>(sm + S::OFF_TAB);
    int* misc = reinterpret_cast<int*>(sm + S::OFF_SCRATCH);   // doc-table scratch, 65 ints
    float* red = reinterpret_cast<float*>(sm + S::OFF_RED);     // [2][8] used
    int* xs = reinterpret_cast<int*>(sm + S::OFF_XS);           // [4][128]
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S::OFF_BAR);   // [NST]
    constexpr int NST = S::NST;
    int* flag = reinterpret_cast<int*>(sm + S::OFF_FLAG);       // [1] abort ([0] spare)
    volatile int* abort = flag + 1;

    // the document table is the same for the three tensors (one shape)
    DocTablePtrs tab{stab.start, stab.off_tile, stab.off_blk};
    if (p0.gtab) {   // written by doc_table_kernel (a malformed batch has no tiles)
        tab = DocTablePtrs{p0.gtab, p0.gtab + (p0.nd + 1), p0.gtab + 2 * (p0.nd + 1)};
    } else if (!build_doc_table(p0, tab, misc)) {
        return;
    }
    const int H = p0.H, nd = p0.nd;
    const int n_units_t = tab.off_tile[nd] * H;   // units of one tensor
    const int n_units = n_units_t * ntens;
    const int tid = threadIdx.x, lane = tid & 31, sl = lane & 7;
    if (tid == 0) {
        for (int st = 0; st < NST; st++) mbar_init(&full[st], 1);
        flag[0] = 0;
        flag[1] = 0;
        fence_mbar_init();
    }
    if constexpr (QM == QM_NVFP4) {
        // 6 / sf for every non-negative E4M3 scale code (0 for the zero code), the IEEE
        // division each NVFP4 group would otherwise repeat, after the reduction slots
        if (tid < 128) {
            const float v = e4m3_value((uint32_t)tid);
            red[16 + tid] = v > 0.0f ? __fdiv_rn(6.0f, v) : 0.0f;
        }
    }
    __syncthreads();
    int issued[NST] = {};   // loads issued per stage (thread 0 only)
    auto issue = [&](int u, int st) {
        issued[st]++;
        const int t = u / n_units_t, uu = u % n_units_t;
        const int g = uu / H, h = uu % H;
        const int doc = find_doc(tab.off_tile, nd, g);
        const int t0 = tab.start[doc] + (g - tab.off_tile[doc]) * 128;
        mbar_arrive_expect_tx(&full[st], S::STAGE);
        tma_load_3d(sm + st * S::STAGE, t == 0 ? &tm0 : (t == 1 ? &tm1 : &tm2), &full[st], 0, h, t0);
    };
    if (tid == 0) {
        for (int st = 0; st < NST; st++)
            if (blockIdx.x + st * gridDim.x < n_units) issue(blockIdx.x + st * gridDim.x, st);
    }
    const uint32_t smask = sign_mask<EPL>(p0, sl);                      // Q and K: one rotation
    uint32_t smask_v = smask;
    if constexpr (NT == 3) smask_v = sign_mask<EPL>(p2, sl);
    bool nonfin = false;
    int k = 0, rc = 0;
    if constexpr (NT == 1) {
        quant_range<EPL, ELT, QM, HOLD>(p0, tab, sm, full, red, xs, abort, smask, nonfin, blockIdx.x, n_units,
                                        0, n_units, k, rc, issue);
    } else {
        // the three tensors one after another, each loop with its own parameters;
        // first(lo): this CTA's first unit at or after lo
        const int G = gridDim.x, b = blockIdx.x;
        auto first = [&](int lo) { return lo + ((b - lo % G) % G + G) % G; };
        const int n = n_units_t;
        if (quant_range<EPL, ELT, QM, HOLD>(p0, tab, sm, full, red, xs, abort, smask, nonfin, first(0), n, 0,
                                            n_units, k, rc, issue) &&
            quant_range<EPL, ELT, QM, HOLD>(p1, tab, sm, full, red, xs, abort, smask, nonfin, first(n), 2 * n,
                                            n, n_units, k, rc, issue))
            quant_range<EPL, ELT, QMV, HOLDV>(p2, tab, sm, full, red, xs, abort, smask_v, nonfin, first(2 * n),
                                              3 * n, 2 * n, n_units, k, rc, issue);
    }
    if (tid == 0) {
        // every issued copy must have landed before the CTA's shared memory goes away
        // (immediate on the normal path, where each issued unit was consumed)
        for (int st = 0; st < NST; st++)
            if (issued[st]) {
                const long long t0 = clock64();
                while (!mbar_try_wait(&full[st], (issued[st] - 1) & 1) && clock64() - t0 < 4000000000LL) {
                }
            }
    }
    if (nonfin) atomicOr(p0.status, ST_NONFINITE);
    if (*abort && tid == 0) atomicOr(p0.status, ST_TIMEOUT);
}

// ---------------------------------------------------------------------------
// maps[t] / ps[t] for the ntens tensors of the launch (1, or 3: Q, K with layout QM, V with QMV)
template <int EPL, int ELT, int QM, int HOLD, int NT, int QMV = QM, int HOLDV = HOLD>
static cudaError_t launch_q(const CUtensorMap* maps, const QuantParams* ps, int grid, cudaStream_t st) {
    using S = QuantSmem<EPL, ELT>;
    auto kern = quant_tile_kernel<EPL, ELT, QM, HOLD, QMV, HOLDV, NT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
    if (e != cudaSuccess) return e;
    const int t1 = NT == 3 ? 1 : 0, t2 = NT == 3 ? 2 : 0;
    kern<<<grid, QUANT_THREADS, S::BYTES, st>>>(maps[0], maps[t1], maps[t2], ps[0], ps[t1], ps[t2]);
    return cudaGetLastError();
}

// one tensor of any layout, or (layout_v >= 0) Q, K in `layout` and V in `layout_v`
template <int EPL, int ELT>
static cudaError_t launch_layout(const CUtensorMap* m, const QuantParams* ps, int layout, int layout_v, int grid,
                                 cudaStream_t st) {
    const int nt = layout_v >= 0 ? 3 : 1;
    if constexpr (EPL == 16) {   // MX and NVFP4 layouts: d = 128 only
        if (nt == 3) {
            if (layout == 1 && layout_v == 2) return launch_q<EPL, ELT, QM_MX_ROW, 1, 3, QM_MX_COL, 1>(m, ps, grid, st);
            if (layout == 1 && layout_v == 3) return launch_q<EPL, ELT, QM_MX_ROW, 1, 3, QM_MX_TOK, 1>(m, ps, grid, st);
            if (layout == 4 && layout_v == 0)
                return launch_q<EPL, ELT, QM_NVFP4, 4, 3, QM_E4M3_BLOCK, 4>(m, ps, grid, st);
        } else {
            if (layout == 1) return launch_q<EPL, ELT, QM_MX_ROW, 1, 1>(m, ps, grid, st);
            if (layout == 2) return launch_q<EPL, ELT, QM_MX_COL, 1, 1>(m, ps, grid, st);
            if (layout == 3) return launch_q<EPL, ELT, QM_MX_TOK, 1, 1>(m, ps, grid, st);
            if (layout == 4) return launch_q<EPL, ELT, QM_NVFP4, 4, 1>(m, ps, grid, st);
        }
    }
    if (layout != 0 || (nt == 3 && layout_v != 0)) return cudaErrorInvalidValue;
    switch (ps[0].block) {
        case 1: return nt == 3 ? launch_q<EPL, ELT, QM_E4M3_ROW, 1, 3>(m, ps, grid, st)
                               : launch_q<EPL, ELT, QM_E4M3_ROW, 1, 1>(m, ps, grid, st);
        case 32: return nt == 3 ? launch_q<EPL, ELT, QM_E4M3_BLOCK, 1, 3>(m, ps, grid, st)
                                : launch_q<EPL, ELT, QM_E4M3_BLOCK, 1, 1>(m, ps, grid, st);
        case 64: return nt == 3 ? launch_q<EPL, ELT, QM_E4M3_BLOCK, 2, 3>(m, ps, grid, st)
                                : launch_q<EPL, ELT, QM_E4M3_BLOCK, 2, 1>(m, ps, grid, st);
        default: return nt == 3 ? launch_q<EPL, ELT, QM_E4M3_BLOCK, 4, 3>(m, ps, grid, st)
                                : launch_q<EPL, ELT, QM_E4M3_BLOCK, 4, 1>(m, ps, grid, st);
    }
}

static bool input_map(CUtensorMap* m, const QuantParams& p) {
    const int elt = p.in_bf16 ? 2 : 4;
    return make_tensor_map_3d(m, p.x, p.in_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                              p.d, p.H, p.T, (uint64_t)p.hstride * elt, (uint64_t)p.tstride * elt, p.d, 128,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
}

// ps[0..ntens): one tensor, or Q, K, V (same shape, dtype and strides)
static cudaError_t launch_tensors(const QuantParams* ps, int ntens, int layout, int layout_v, cudaStream_t st) {
    const QuantParams& p = ps[0];
    if (p.gtab) {
        doc_table_kernel<<<1, 1024, 0, st>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    CUtensorMap m[3];
    for (int t = 0; t < ntens; t++)
        if (!input_map(&m[t], ps[t])) return cudaErrorInvalidValue;
    const long long units = (long long)ntens * p.H * (((long long)p.T + 127) / 128 + p.nd);
    const int sms = sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
    // two CTAs per SM except fp32 rows of 128 channels (128 KB of stages per CTA)
    const int per_sm = (p.d == 128 && !p.in_bf16) ? 1 : 2;
    const int grid = (int)(units < (long long)per_sm * sms ? units : (long long)per_sm * sms);
    if (p.d == 128) return p.in_bf16 ? launch_layout<16, 2>(m, ps, layout, layout_v, grid, st)
                                     : launch_layout<16, 4>(m, ps, layout, layout_v, grid, st);
    return p.in_bf16 ? launch_layout<8, 2>(m, ps, layout, layout_v, grid, st)
                     : launch_layout<8, 4>(m, ps, layout, layout_v, grid, st);
}

cudaError_t launch_quantize(const QuantParams& p, int layout, cudaStream_t st) {
    return launch_tensors(&p, 1, layout, -1, st);
}

cudaError_t launch_quantize_qkv(const QuantParams* ps, int layout_qk, int layout_v, cudaStream_t st) {
    return launch_tensors(ps, 3, layout_qk, layout_v, st);
}

}  // namespace pa
