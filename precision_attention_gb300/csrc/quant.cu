// quant.cu -- fused rotate-and-quantise kernels (one launch per tensor).
//
// Sources: "Fused attention kernel", 8-bit forward pass (e4m3 codes, block
// quantisation, incoherent processing: random sign diagonal times Hadamard,
// applied to Q and K); FLAMIA section 2 (MX: 32-element blocks, one shared
// E8M0 scale) and section 4.3 (fused quantisation: one launch instead of many).
//
// Thread layout (every kernel): a row = (token, head) of d channels is held by
// 8 consecutive lanes, EPL = d / 8 channels each (lane sub-index sl holds
// channels sl*EPL .. sl*EPL+EPL-1); a warp holds 4 rows. The Hadamard
// transform runs its stages h = 1, 2, 4, ... in that order: in registers while
// h < EPL, then across the 8 lanes with shuffles (lane ^ 1, ^ 2, ^ 4). Every
// butterfly is (a, b) -> (a + b, a - b) in fp32 with round-to-nearest, so the
// result does not depend on how elements are spread over lanes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "params.h"
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

template <int EPL>
__device__ __forceinline__ void load_row(const QuantParams& p, int t, int h, int sl, float (&v)[EPL]) {
    const long long off = (long long)t * p.tstride + (long long)h * p.hstride + sl * EPL;
    if (p.in_bf16) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.x) + off);
#pragma unroll
        for (int q = 0; q < EPL / 8; q++) {
            uint4 u = __ldg(src + q);
            uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                v[q * 8 + 2 * k] = __uint_as_float(w[k] << 16);
                v[q * 8 + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            }
        }
    } else {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + off);
#pragma unroll
        for (int q = 0; q < EPL / 4; q++) {
            float4 f = __ldg(src + q);
            v[q * 4 + 0] = f.x;
            v[q * 4 + 1] = f.y;
            v[q * 4 + 2] = f.z;
            v[q * 4 + 3] = f.w;
        }
    }
}

// sign flip then the Walsh-Hadamard stages (see the file comment)
template <int EPL>
__device__ __forceinline__ void rotate_row(float (&v)[EPL], uint32_t smask, int lane) {
#pragma unroll
    for (int i = 0; i < EPL; i++)
        if (smask & (1u << i)) v[i] = -v[i];
#pragma unroll
    for (int h = 1; h < EPL; h <<= 1) {
#pragma unroll
        for (int i = 0; i < EPL; i++) {
            if (!(i & h)) {
                const float a = v[i], b = v[i + h];
                v[i] = __fadd_rn(a, b);
                v[i + h] = __fsub_rn(a, b);
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < EPL; i++) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v[i], m);
            v[i] = upper ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);
        }
    }
}

__device__ __forceinline__ bool finite_abs(float a) { return a <= 3.402823466e38f; }

// E8M0 exponent X of a block amax (see the header: NOSAT = smallest X with
// amax <= 448 * 2^X; OCP_FLOOR = floor(log2 amax) - 8), clamped to [-127, 127]
__device__ __forceinline__ int e8m0_exponent(float amax, int rule) {
    if (!(amax > 0.0f)) return -127;
    const uint32_t u = __float_as_uint(amax);
    const int ef = (int)((u >> 23) & 0xFF);
    if (ef == 0) return -127;                       // subnormal amax: X far below -127
    const int E = ef - 127;
    const uint32_t frac = u & 0x7FFFFFu;
    int X = (rule == 1) ? E - 8 : (frac <= 0x600000u ? E - 8 : E - 7);   // 1.75 = 1 + 0x600000 / 2^23
    return X < -127 ? -127 : (X > 127 ? 127 : X);
}
__device__ __forceinline__ float pow2_neg(int X) {   // 2^-X for X in [-127, 126]
    return __uint_as_float((uint32_t)(127 - X) << 23);
}

template <int EPL>
__device__ __forceinline__ void store_codes(uint8_t* dst, const float (&y)[EPL], float mul) {
    uint32_t w[EPL / 4];
#pragma unroll
    for (int i = 0; i < EPL / 4; i++)
        w[i] = pack_e4m3x4(__fmul_rn(y[4 * i], mul), __fmul_rn(y[4 * i + 1], mul), __fmul_rn(y[4 * i + 2], mul),
                           __fmul_rn(y[4 * i + 3], mul));
    if constexpr (EPL == 16) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    }
}

// ---------------------------------------------------------------------------
// In-CTA document table: starts and prefix counts of `unit`-token pieces.
// Returns false (after flagging the status word) when cu_seqlens is malformed.
struct DocTable {
    int32_t start[MAX_DOCS + 1];
    int32_t off[MAX_DOCS + 1];   // exclusive prefix of ceil(L / unit); off[nd] = total
};

__device__ bool build_doc_table(const QuantParams& p, int unit, DocTable& tab) {
    __shared__ int bad;
    __shared__ int wsum[8];
    const int tid = threadIdx.x, nd = p.nd;
    if (tid == 0) bad = 0;
    __syncthreads();
    // each thread owns up to 4 consecutive documents
    int cnt[4], acc = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int i = tid * 4 + k;
        cnt[k] = 0;
        if (i < nd) {
            const int s = p.cu ? p.cu[i] : 0, e = p.cu ? p.cu[i + 1] : p.T;
            tab.start[i] = s;
            if (e < s) bad = 1;
            cnt[k] = (e - s + unit - 1) / unit;
            if (e < s) cnt[k] = 0;
        }
        acc += cnt[k];
    }
    if (tid == 0) {
        const int c0 = p.cu ? p.cu[0] : 0, cn = p.cu ? p.cu[nd] : p.T;
        if (c0 != 0 || cn != p.T) bad = 1;
        tab.start[nd] = cn;
    }
    // block-wide exclusive scan of acc
    const int lane = tid & 31, warp = tid >> 5;
    int inc = acc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; w++) base += wsum[w];
    int run = base + inc - acc;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int i = tid * 4 + k;
        if (i < nd) tab.off[i] = run;
        run += cnt[k];
    }
    if (tid == blockDim.x - 1) tab.off[nd] = run;
    __syncthreads();
    if (bad) {
        if (tid == 0) atomicOr(p.status, ST_BAD_SEQLENS);
        return false;
    }
    return true;
}

__device__ __forceinline__ int find_doc(const DocTable& tab, int nd, int u) {
    int lo = 0, hi = nd - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab.off[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------
// E4M3, blocks of BLOCK >= 32 tokens: one CTA (8 warps, 32 rows per pass) per
// (document-local block, head). scale = amax / 448, code = E4M3(y * (448 / amax)).
template <int EPL, int PASSES>
__global__ void __launch_bounds__(256) quant_e4m3_block_kernel(QuantParams p) {
    __shared__ DocTable tab;
    __shared__ float red[8];
    __shared__ int nonfin;
    if (!build_doc_table(p, p.block, tab)) return;
    const int H = p.H;
    const int ub = blockIdx.x / H, h = blockIdx.x % H;
    if (ub >= tab.off[p.nd]) return;
    const int doc = find_doc(tab, p.nd, ub);
    const int s = tab.start[doc], L = tab.start[doc + 1] - s;
    const int b0 = (ub - tab.off[doc]) * p.block;     // first local token of the block
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, sl = lane & 7, rw = lane >> 3;
    if (threadIdx.x == 0) nonfin = 0;
    const uint32_t smask = sign_mask<EPL>(p, sl);

    float y[PASSES][EPL];
    float amax = 0.0f;
    bool bad = false;
#pragma unroll
    for (int ps = 0; ps < PASSES; ps++) {
        const int lt = b0 + ps * 32 + warp * 4 + rw;   // local token
        const bool valid = (ps * 32 + warp * 4 + rw) < p.block && lt < L;
        if (valid) load_row<EPL>(p, s + lt, h, sl, y[ps]);
        else {
#pragma unroll
            for (int i = 0; i < EPL; i++) y[ps][i] = 0.0f;
        }
        if (p.rotate) rotate_row<EPL>(y[ps], smask, lane);   // whole warp takes part in the shuffles
#pragma unroll
        for (int i = 0; i < EPL; i++) {
            const float a = fabsf(y[ps][i]);
            if (!finite_abs(a)) bad = true;
            else amax = fmaxf(amax, a);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    __syncthreads();   // nonfin initialised
    if (bad) nonfin = 1;
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; w++) amax = fmaxf(amax, red[w]);
    float inv = 0.0f, scale = 0.0f;
    if (nonfin) {
        scale = __int_as_float(0x7FC00000);
        if (threadIdx.x == 0) atomicOr(p.status, ST_NONFINITE);
    } else if (amax > 0.0f) {
        inv = __fdiv_rn(448.0f, amax);
        scale = __fdiv_rn(amax, 448.0f);
    }
    if (threadIdx.x == 0) static_cast<float*>(p.scales)[(long long)h * p.scale_cap + ub] = scale;
#pragma unroll
    for (int ps = 0; ps < PASSES; ps++) {
        const int lt = b0 + ps * 32 + warp * 4 + rw;
        const bool valid = (ps * 32 + warp * 4 + rw) < p.block && lt < L;
        if (valid) store_codes<EPL>(p.codes + ((long long)(s + lt) * H + h) * p.d + sl * EPL, y[ps], inv);
    }
}

// E4M3 with one scale per (token, head) (block 1, the causal-exact layout):
// 4 rows per warp, amax over the row's 8 lanes. No document table is needed:
// the block index of token t is t itself.
template <int EPL>
__global__ void __launch_bounds__(256) quant_e4m3_row_kernel(QuantParams p) {
    const int lane = threadIdx.x & 31, sl = lane & 7;
    const long long row = (long long)blockIdx.x * 32 + (threadIdx.x >> 3);
    const long long nrows = (long long)p.T * p.H;
    const bool valid = row < nrows;
    const int t = valid ? (int)(row / p.H) : 0, h = valid ? (int)(row % p.H) : 0;
    const uint32_t smask = sign_mask<EPL>(p, sl);
    float y[EPL];
    if (valid) load_row<EPL>(p, t, h, sl, y);
    else {
#pragma unroll
        for (int i = 0; i < EPL; i++) y[i] = 0.0f;
    }
    if (p.rotate) rotate_row<EPL>(y, smask, lane);
    float amax = 0.0f;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const float a = fabsf(y[i]);
        if (!finite_abs(a)) bad = true;
        else amax = fmaxf(amax, a);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        bad = bad | (__shfl_xor_sync(0xFFFFFFFFu, (int)bad, o) != 0);
    }
    if (!valid) return;
    float inv = 0.0f, scale = 0.0f;
    if (bad) {
        scale = __int_as_float(0x7FC00000);
        if (sl == 0) atomicOr(p.status, ST_NONFINITE);
    } else if (amax > 0.0f) {
        inv = __fdiv_rn(448.0f, amax);
        scale = __fdiv_rn(amax, 448.0f);
    }
    if (sl == 0) static_cast<float*>(p.scales)[(long long)h * p.scale_cap + t] = scale;
    store_codes<EPL>(p.codes + ((long long)t * p.H + h) * p.d + sl * EPL, y, inv);
}

// MX row32 (Q, K; d = 128): one CTA per (document tile of 128 tokens, head),
// 4 passes of 32 rows. A pair of lanes holds one 32-channel group. The four
// group exponents of a row go to bytes (r%32)*16 + (r/32)*4 + g of the tile's
// 512-byte scale block; rows past the document end get 127 (2^0).
__global__ void __launch_bounds__(256) quant_mx_row_kernel(QuantParams p) {
    constexpr int EPL = 16;
    __shared__ DocTable tab;
    if (!build_doc_table(p, 128, tab)) return;
    const int H = p.H;
    const int g = blockIdx.x / H, h = blockIdx.x % H;
    if (g >= tab.off[p.nd]) return;
    const int doc = find_doc(tab, p.nd, g);
    const int s = tab.start[doc], L = tab.start[doc + 1] - s;
    const int t0 = (g - tab.off[doc]) * 128;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, sl = lane & 7, rw = lane >> 3;
    const uint32_t smask = sign_mask<EPL>(p, sl);
    uint8_t* tile = static_cast<uint8_t*>(p.scales) + ((long long)h * p.scale_cap + g) * 512;
#pragma unroll 1
    for (int ps = 0; ps < 4; ps++) {
        const int r = ps * 32 + warp * 4 + rw;
        const int lt = t0 + r;
        const bool valid = lt < L;
        float y[EPL];
        if (valid) load_row<EPL>(p, s + lt, h, sl, y);
        else {
#pragma unroll
            for (int i = 0; i < EPL; i++) y[i] = 0.0f;
        }
        if (p.rotate) rotate_row<EPL>(y, smask, lane);
        float amax = 0.0f;
        bool bad = false;
#pragma unroll
        for (int i = 0; i < EPL; i++) {
            const float a = fabsf(y[i]);
            if (!finite_abs(a)) bad = true;
            else amax = fmaxf(amax, a);
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        bad = bad | (__shfl_xor_sync(0xFFFFFFFFu, (int)bad, 1) != 0);
        if (bad && valid) atomicOr(p.status, ST_NONFINITE);
        const int X = valid ? e8m0_exponent(amax, p.mx_rule) : 0;
        // gather the 4 group bytes of the row into lane sl == 0
        uint32_t byte = (uint32_t)(X + 127);
        const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, byte, 2);
        const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, byte, 4);
        const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, byte, 6);
        if (sl == 0) {
            const uint32_t word = byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
            *reinterpret_cast<uint32_t*>(tile + (r % 32) * 16 + (r / 32) * 4) = word;
        }
        if (valid) store_codes<EPL>(p.codes + ((long long)(s + lt) * H + h) * p.d + sl * EPL, y, pow2_neg(X));
    }
}

// MX col32 (V; d = 128): one CTA per (32-token group of a document tile, head).
// Per channel amax over the group's tokens; exponent byte of channel c, group
// gi of tile g at (c%32)*16 + (c/32)*4 + gi. Groups past the document end get 127.
__global__ void __launch_bounds__(256) quant_mx_col_kernel(QuantParams p) {
    constexpr int EPL = 16;
    __shared__ DocTable tab;
    __shared__ float red[8][128];
    __shared__ int xs[128];
    __shared__ int nonfin;
    if (!build_doc_table(p, 128, tab)) return;
    const int H = p.H;
    const int h = blockIdx.x % H, gg = blockIdx.x / H;
    const int g = gg >> 2, gi = gg & 3;
    if (g >= tab.off[p.nd]) return;
    const int doc = find_doc(tab, p.nd, g);
    const int s = tab.start[doc], L = tab.start[doc + 1] - s;
    const int t0 = (g - tab.off[doc]) * 128 + gi * 32;
    uint8_t* tile = static_cast<uint8_t*>(p.scales) + ((long long)h * p.scale_cap + g) * 512;
    if (threadIdx.x == 0) nonfin = 0;
    if (t0 >= L) {   // group entirely past the document end
        if (threadIdx.x < 128) {
            const int c = threadIdx.x;
            tile[(c % 32) * 16 + (c / 32) * 4 + gi] = 127;
        }
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, sl = lane & 7, rw = lane >> 3;
    const int lt = t0 + warp * 4 + rw;
    const bool valid = lt < L;
    float y[EPL];
    if (valid) load_row<EPL>(p, s + lt, h, sl, y);
    else {
#pragma unroll
        for (int i = 0; i < EPL; i++) y[i] = 0.0f;
    }
    if (p.rotate) rotate_row<EPL>(y, sign_mask<EPL>(p, sl), lane);
    float a[EPL];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        a[i] = fabsf(y[i]);
        if (!finite_abs(a[i])) { bad = true; a[i] = 0.0f; }
        a[i] = fmaxf(a[i], __shfl_xor_sync(0xFFFFFFFFu, a[i], 8));
        a[i] = fmaxf(a[i], __shfl_xor_sync(0xFFFFFFFFu, a[i], 16));
    }
    __syncthreads();
    if (bad) nonfin = 1;
    if (rw == 0) {
#pragma unroll
        for (int i = 0; i < EPL; i++) red[warp][sl * EPL + i] = a[i];
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        const int c = threadIdx.x;
        float m = red[0][c];
#pragma unroll
        for (int w = 1; w < 8; w++) m = fmaxf(m, red[w][c]);
        const int X = e8m0_exponent(m, p.mx_rule);
        xs[c] = X;
        tile[(c % 32) * 16 + (c / 32) * 4 + gi] = (uint8_t)(X + 127);
    }
    __syncthreads();
    if (threadIdx.x == 0 && nonfin) atomicOr(p.status, ST_NONFINITE);
    if (!valid) return;
    uint32_t w[EPL / 4];
#pragma unroll
    for (int i = 0; i < EPL / 4; i++) {
        const int c = sl * EPL + 4 * i;
        w[i] = pack_e4m3x4(__fmul_rn(y[4 * i], pow2_neg(xs[c])), __fmul_rn(y[4 * i + 1], pow2_neg(xs[c + 1])),
                           __fmul_rn(y[4 * i + 2], pow2_neg(xs[c + 2])),
                           __fmul_rn(y[4 * i + 3], pow2_neg(xs[c + 3])));
    }
    *reinterpret_cast<uint4*>(p.codes + ((long long)(s + lt) * H + h) * p.d + sl * EPL) =
        make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------------------
// host launcher; returns a cudaError_t
cudaError_t launch_quantize(const QuantParams& p, int layout, cudaStream_t st) {
    const long long H = p.H;
    if (layout == 0) {
        if (p.block == 1) {
            const long long rows = (long long)p.T * H;
            const unsigned grid = (unsigned)((rows + 31) / 32);
            if (p.d == 128) quant_e4m3_row_kernel<16><<<grid, 256, 0, st>>>(p);
            else quant_e4m3_row_kernel<8><<<grid, 256, 0, st>>>(p);
        } else {
            const unsigned grid = (unsigned)(H * p.scale_cap);
            const int passes = p.block / 32;
            if (p.d == 128) {
                if (passes == 1) quant_e4m3_block_kernel<16, 1><<<grid, 256, 0, st>>>(p);
                else if (passes == 2) quant_e4m3_block_kernel<16, 2><<<grid, 256, 0, st>>>(p);
                else quant_e4m3_block_kernel<16, 4><<<grid, 256, 0, st>>>(p);
            } else {
                if (passes == 1) quant_e4m3_block_kernel<8, 1><<<grid, 256, 0, st>>>(p);
                else if (passes == 2) quant_e4m3_block_kernel<8, 2><<<grid, 256, 0, st>>>(p);
                else quant_e4m3_block_kernel<8, 4><<<grid, 256, 0, st>>>(p);
            }
        }
    } else if (layout == 1) {
        quant_mx_row_kernel<<<(unsigned)(H * p.scale_cap), 256, 0, st>>>(p);
    } else {
        quant_mx_col_kernel<<<(unsigned)(H * p.scale_cap * 4), 256, 0, st>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace pa
