// attn_bwd.cu -- attention backward (dQ, dK, dV) for BF16 operands, d = 128, on
// sm_103a (tcgen05 + TMEM + TMA).
//
// The gradients of softmax attention for an upstream gradient dO (FLAMIA
// section 1: the training call is the forward plus a backward over the same
// token blocks). With S = Q K^T, P = exp(scale S - lse) row by row (the
// forward's lse, so no probability is stored), the plain definition gives
//   dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D),  D = rowsum(dO o O),
//   dQ = scale dS K,   dK = scale dS^T Q.
// Causal masks and packed documents follow the forward: keys after the query
// and tokens of other documents get P = 0; every tile is document-local.
//
// Two launches after the work-list pass (the forward's one-query-tile list):
//   bwd_prep_kernel  D and lse log2(e) per row, stored per (head, 128-token
//                    tile) so the gradient kernel fetches a tile's 128 values
//                    with one bulk copy
//   attn_bwd_kernel  persistent; the work items alternate between two roles,
//                    both for one (document, head, 128-token tile):
//     dK/dV role   key tile j: K_j and V_j once, then each query tile i that
//                  sees it: S^T = K_j Q_i^T and dP^T = V_j dO_i^T into TMEM,
//                  P^T and dS^T in registers, written back into TMEM as bf16
//                  over S^T and dP^T, then dV += P^T dO_i and dK += dS^T Q_i
//                  with the A operand read from TMEM
//     dQ role      query tile i: Q_i and dO_i once, then each key tile j it
//                  sees: S = Q_i K_j^T, dP = dO_i V_j^T, dS into TMEM over dP,
//                  dQ += dS K_j
//   dQ is formed in its own role (S and dP computed a second time) rather than
//   accumulated across key tiles with atomics, so the gradients are
//   deterministic: one fixed summation order per output element.
// Warp roles: warp 0 TMA producer (the item's two row tiles, then the two
// stream tiles of each step, and in the dK/dV role the step's 128 lse and D
// values, into a 2-stage ring); warp 1 TMEM owner and MMA issuer; warps 2-9
// elementwise: two warps per 32-row TMEM lane quarter, each taking 64 of the
// 128 columns, and the epilogue.
// TMEM (512 columns): S [0,128), dP [128,256), dV or dQ [256,384), dK
// [384,512). P^T of column half hh goes to [64 hh, 64 hh + 32) and dS to
// [128 + 64 hh, ...): inside the columns that half itself loaded, so neither
// warp overwrites S or dP values its partner has yet to read.
// Every wait is bounded; on a timeout the CTA raises its flag, drains, frees
// TMEM and returns, and the host reads ATTN_ERR_DEVICE_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "pdl.cuh"

namespace pa {

namespace bwd {
constexpr int D = 128;
constexpr int TILE = 128 * D * 2;          // one bf16 tile of 128 rows: two 16 KB 128-byte-swizzled atoms
constexpr int NS = 2;                      // stream-tile stages
constexpr int OFF_R = 0;                   // row tiles R0, R1
constexpr int OFF_X = 2 * TILE;            // NS stages of the stream tiles X0, X1
constexpr int OFF_VEC = OFF_X + NS * 2 * TILE;   // NS x {lse log2(e) [128], D [128]}
constexpr int OFF_BAR = OFF_VEC + NS * 1024;
constexpr int SMEM = OFF_BAR + 512 + 1024;
constexpr int THREADS = 64 + 256;
constexpr uint32_t T_S = 0, T_DP = 128, T_O0 = 256, T_O1 = 384;
using C = Cfg<2, D, MODE_BF16>;
static_assert(C::TILE == TILE && C::ATOMS == 2, "bf16 d = 128 tiles are two 128-byte swizzle atoms");
static_assert(SMEM <= 227 * 1024, "backward shared memory exceeds the per-CTA limit");

struct Bars {
    uint64_t r_full, r_empty;
    uint64_t x_full[NS], x_empty[NS];
    uint64_t s_full;     // S and dP of the step are in TMEM
    uint64_t p_full;     // the step's P and dS are back in TMEM (256 arrivals)
    uint64_t o_done;     // the step's output MMAs completed
    uint64_t epi_done;   // the item's accumulators were read (256 arrivals)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 512, "backward barrier block exceeds its reserved space");

// One work item of the gradient kernel. Position `it` of the combined list holds
// work item it / 2 of the forward's list in one of the two roles; with an even
// grid, a CTA takes the two roles in turn from round to round, and every item
// appears once in each role.
struct Item {
    int kv;          // 1: dK/dV of key tile rt; 0: dQ of query tile rt
    int head, start, len, toff;
    int rt;          // the row tile (keys or queries), document-local
    int s0, n;       // stream tiles s0 .. s0 + n - 1
};
__device__ __forceinline__ Item decode(const BwdParams& p, int it) {
    Item x;
    x.kv = ((it & 1) ^ ((it / (int)gridDim.x) & 1)) == 0;
    const WorkItem w = p.items[it >> 1];
    const DocEntry d = p.docs[w.doc];
    const int nt = (d.len + 127) >> 7;
    x.head = w.head;
    x.start = d.start;
    x.len = d.len;
    x.toff = d.toff;
    x.n = w.ntiles;
    if (x.kv) {
        // causal: query tile qtile of the list sees qtile + 1 key tiles; key tile
        // nt - 1 - qtile is seen by as many query tiles (from itself to the last)
        x.rt = p.causal ? nt - 1 - w.qtile : w.qtile;
        x.s0 = p.causal ? x.rt : 0;
    } else {
        x.rt = w.qtile;
        x.s0 = 0;
    }
    return x;
}
}  // namespace bwd

// D = rowsum(dO o O) and lse log2(e) of every row, per (head, 128-token tile).
// Grid (tiles_cap, H); eight warps, one row per warp at a time.
__global__ void __launch_bounds__(256) bwd_prep_kernel(BwdParams p) {
    pdl_trigger();
    pdl_wait();   // the document table
    if (p.hdr->n_items <= 0) return;
    const int tg = blockIdx.x, h = blockIdx.y;
    int lo = 0, hi = p.nd - 1;   // the last document whose first tile is <= tg
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.docs[mid].toff <= tg) lo = mid; else hi = mid - 1;
    }
    const DocEntry d = p.docs[lo];
    const int lt = tg - d.toff;
    if (lt < 0 || lt >= (d.len + 127) / 128) return;   // past the last tile
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* vl = p.vec + ((long long)h * p.tiles_cap + tg) * 128;
    float* vd = vl + (long long)p.H * p.tiles_cap * 128;
    for (int r = warp; r < 128; r += 8) {
        const int loc = 128 * lt + r;
        float dsum = 0.0f, l2 = 0.0f;
        if (loc < d.len) {
            const long long base = ((long long)(d.start + loc) * p.H + h) * bwd::D + 4 * lane;
            const uint2 a = *reinterpret_cast<const uint2*>(p.o + base);
            const uint2 b = *reinterpret_cast<const uint2*>(p.dout + base);
            const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a.x));
            const float2 a1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a.y));
            const float2 b0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.x));
            const float2 b1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.y));
            dsum = a0.x * b0.x + a0.y * b0.y + a1.x * b1.x + a1.y * b1.y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xFFFFFFFFu, dsum, o);
            l2 = p.lse[(long long)h * p.T + d.start + loc] * 1.4426950408889634f;
        }
        if (lane == 0) {
            vl[r] = l2;
            vd[r] = dsum;
        }
    }
}

__global__ void __launch_bounds__(bwd::THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                    const BwdParams p) {
    using namespace bwd;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* B = reinterpret_cast<Bars*>(sm + OFF_BAR);
    volatile int* abort = &B->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long lim = p.wait_limit;

    if (threadIdx.x == 0) {
        mbar_init(&B->r_full, 1);
        mbar_init(&B->r_empty, 1);
        for (int i = 0; i < NS; i++) {
            mbar_init(&B->x_full[i], 1);
            mbar_init(&B->x_empty[i], 1);
        }
        mbar_init(&B->s_full, 1);
        mbar_init(&B->p_full, 256);
        mbar_init(&B->o_done, 1);
        mbar_init(&B->epi_done, 256);
        mbar_init(&B->drain, 1);
        B->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmq);
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        prefetch_tensormap(&tmdo);
    }
    if (warp == 1) {
        tmem_alloc(&B->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B->tmem_base;
    pdl_wait();   // the work list and the per-row vectors
    const int n_items = 2 * p.hdr->n_items;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        constexpr unsigned FULL = 0xFFFFFFFFu;
        int issued[NS];
        for (int i = 0; i < NS; i++) issued[i] = -1;
        int r_issued = -1;
        uint32_t g = 0;
        int qi = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, qi++) {
            const Item x = decode(p, it);
            const CUtensorMap* r0 = x.kv ? &tmk : &tmq;
            const CUtensorMap* r1 = x.kv ? &tmv : &tmdo;
            const CUtensorMap* x0 = x.kv ? &tmq : &tmk;
            const CUtensorMap* x1 = x.kv ? &tmdo : &tmv;
            if (!__all_sync(FULL, mbar_wait(&B->r_empty, (qi & 1) ^ 1, abort, lim))) break;
            r_issued = qi & 1;
            if (lane == 0) {
                mbar_arrive_expect_tx(&B->r_full, 2 * TILE);
                const int row = x.start + 128 * x.rt;
                for (int a = 0; a < 2; a++) {
                    tma_load_3d(sm + OFF_R + a * 16384, r0, &B->r_full, a * 64, x.head, row);
                    tma_load_3d(sm + OFF_R + TILE + a * 16384, r1, &B->r_full, a * 64, x.head, row);
                }
            }
            for (int t = 0; t < x.n; t++, g++) {
                const int st = g % NS;
                if (!__all_sync(FULL, mbar_wait(&B->x_empty[st], ((g / NS) & 1) ^ 1, abort, lim))) {
                    ok = false;
                    break;
                }
                issued[st] = (g / NS) & 1;
                if (lane == 0) {
                    const int tile = x.s0 + t;
                    const int row = x.start + 128 * tile;
                    uint8_t* xs = sm + OFF_X + st * 2 * TILE;
                    mbar_arrive_expect_tx(&B->x_full[st], 2 * TILE + (x.kv ? 1024 : 0));
                    for (int a = 0; a < 2; a++) {
                        tma_load_3d(xs + a * 16384, x0, &B->x_full[st], a * 64, x.head, row);
                        tma_load_3d(xs + TILE + a * 16384, x1, &B->x_full[st], a * 64, x.head, row);
                    }
                    if (x.kv) {   // the query tile's lse log2(e) and D
                        const float* vl = p.vec + ((long long)x.head * p.tiles_cap + x.toff + tile) * 128;
                        uint8_t* dst = sm + OFF_VEC + st * 1024;
                        bulk_load(dst, vl, 512, &B->x_full[st]);
                        bulk_load(dst + 512, vl + (long long)p.H * p.tiles_cap * 128, 512, &B->x_full[st]);
                    }
                }
            }
        }
        if (*abort && lane == 0) {   // let in-flight copies land before shared memory is released
            if (r_issued >= 0) wait_drain(&B->r_full, (uint32_t)r_issued, kDrainLimit);
            for (int s2 = 0; s2 < NS; s2++)
                if (issued[s2] >= 0) wait_drain(&B->x_full[s2], (uint32_t)issued[s2], kDrainLimit);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_s = idesc(1, 1, false, false, 128, 128);   // K-major A and B
            constexpr uint32_t id_o = idesc(1, 1, false, true, 128, 128);    // A from TMEM, MN-major B
            const uint32_t sR = smem_u32(sm + OFF_R), sX = smem_u32(sm + OFF_X);
            const uint64_t dr0 = desc_kmajor<2, D, MODE_BF16>(sR, 0);
            const uint64_t dr1 = desc_kmajor<2, D, MODE_BF16>(sR + TILE, 0);
            const uint64_t dx0 = desc_kmajor<2, D, MODE_BF16>(sX, 0);
            const uint64_t dx1 = desc_kmajor<2, D, MODE_BF16>(sX + TILE, 0);
            const uint64_t vx0 = desc_v<2, D, MODE_BF16>(sX, 0);          // the stream tiles as MN-major B
            const uint64_t vx1 = desc_v<2, D, MODE_BF16>(sX + TILE, 0);
            constexpr uint64_t STAGE16 = (uint64_t)(2 * TILE) >> 4;
            // TMEM column of K step kk of a P or dS operand (16 columns of keys or queries
            // per step; column halves at 0 and 64)
            auto acol = [](int kk) -> uint32_t { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); };
            uint32_t g = 0;
            int qi = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, qi++) {
                const Item x = decode(p, it);
                if (!mbar_wait(&B->r_full, qi & 1, abort, lim)) break;
                for (int t = 0; t < x.n; t++, g++) {
                    const int st = g % NS;
                    if (!mbar_wait(&B->x_full[st], (g / NS) & 1, abort, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t so = st * STAGE16;
#pragma unroll
                    for (int kk = 0; kk < 8; kk++)
                        mma_f16(tmem + T_S, dr0 + koff<2, D, MODE_BF16>(kk), dx0 + so + koff<2, D, MODE_BF16>(kk),
                                id_s, kk ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < 8; kk++)
                        mma_f16(tmem + T_DP, dr1 + koff<2, D, MODE_BF16>(kk), dx1 + so + koff<2, D, MODE_BF16>(kk),
                                id_s, kk ? 1u : 0u);
                    tc_commit(&B->s_full);
                    if (!mbar_wait(&B->p_full, g & 1, abort, lim)) {
                        ok = false;
                        break;
                    }
                    // the previous item's epilogue has read the accumulators
                    if (t == 0 && qi > 0 && !mbar_wait(&B->epi_done, (qi - 1) & 1, abort, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (x.kv) {
#pragma unroll
                        for (int kk = 0; kk < 8; kk++)   // dV += P^T dO
                            mma_f16_ta(tmem + T_O0, tmem + T_S + acol(kk), vx1 + so + voff<2, D, MODE_BF16>(kk), id_o,
                                       (t | kk) ? 1u : 0u);
#pragma unroll
                        for (int kk = 0; kk < 8; kk++)   // dK += dS^T Q
                            mma_f16_ta(tmem + T_O1, tmem + T_DP + acol(kk), vx0 + so + voff<2, D, MODE_BF16>(kk), id_o,
                                       (t | kk) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 8; kk++)   // dQ += dS K
                            mma_f16_ta(tmem + T_O0, tmem + T_DP + acol(kk), vx0 + so + voff<2, D, MODE_BF16>(kk), id_o,
                                       (t | kk) ? 1u : 0u);
                    }
                    tc_commit(&B->x_empty[st]);
                    if (t == x.n - 1) tc_commit(&B->r_empty);
                    tc_commit(&B->o_done);
                    // P and dS sit over S and dP: the next step's S waits for their readers
                    if (!mbar_wait(&B->o_done, g & 1, abort, lim)) {
                        ok = false;
                        break;
                    }
                }
            }
            // every MMA this thread issued has completed before TMEM is released
            tc_commit(&B->drain);
            wait_drain(&B->drain, 0, kDrainLimit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ elementwise + epilogue
        constexpr unsigned FULL = 0xFFFFFFFFu;
        const int hh = (warp - 2) >> 2;                      // column half
        const int quarter = warp & 3;                        // TMEM lane quarter
        const int r = quarter * 32 + lane;                   // row of the row tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float c = p.C;
        uint32_t g = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const Item x = decode(p, it);
            const int rpos = 128 * x.rt + r;                 // document-local position of this row
            // dQ role: this row's lse log2(e) and D
            float row_l2 = 0.0f, row_d = 0.0f;
            if (!x.kv) {
                const long long vi = ((long long)x.head * p.tiles_cap + x.toff + x.rt) * 128 + r;
                row_l2 = p.vec[vi];
                row_d = p.vec[vi + (long long)p.H * p.tiles_cap * 128];
            }
            for (int t = 0; t < x.n; t++, g++) {
                const int st = g % NS;
                if (!__all_sync(FULL, mbar_wait(&B->s_full, g & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                // the bulk-copied vectors: observe their barrier as well (its phase cannot
                // advance past this step before these threads arrive on p_full)
                if (x.kv && !__all_sync(FULL, mbar_wait(&B->x_full[st], (g / NS) & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int tile = x.s0 + t;
                const int cbase = 128 * tile + 64 * hh;       // document-local position of column 0 of this half
                // masked: the causal diagonal tile or a tile reaching past the document's end
                const bool need_mask = (p.causal && tile == x.rt) || (128 * tile + 128 > x.len);
                const float* vl = reinterpret_cast<const float*>(sm + OFF_VEC + st * 1024) + 64 * hh;
                const float* vd = vl + 128;
#pragma unroll
                for (int ch = 0; ch < 2; ch++) {
                    uint32_t us[32], ud[32];
                    tmem_ld32(tmem + lane_off + T_S + 64 * hh + 32 * ch, us);
                    tmem_ld32(tmem + lane_off + T_DP + 64 * hh + 32 * ch, ud);
                    tmem_wait_ld();
                    uint32_t pk[16], dk[16];
#pragma unroll
                    for (int u = 0; u < 32; u += 4) {
                        float l4[4], d4[4];
                        if (x.kv) {
                            const float4 a = *reinterpret_cast<const float4*>(vl + 32 * ch + u);
                            const float4 b = *reinterpret_cast<const float4*>(vd + 32 * ch + u);
                            l4[0] = a.x; l4[1] = a.y; l4[2] = a.z; l4[3] = a.w;
                            d4[0] = b.x; d4[1] = b.y; d4[2] = b.z; d4[3] = b.w;
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; e++) {
                                l4[e] = row_l2;
                                d4[e] = row_d;
                            }
                        }
                        float pe[4], ds[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            pe[e] = ex2(fmaf(__uint_as_float(us[u + e]), c, -l4[e]));
                            ds[e] = pe[e] * (__uint_as_float(ud[u + e]) - d4[e]);
                            if (need_mask) {
                                const int cpos = cbase + 32 * ch + u + e;
                                // dK/dV role: column = query, row = key; dQ role: the reverse
                                const bool vis = cpos < x.len &&
                                                 (!p.causal || (x.kv ? cpos >= rpos : cpos <= rpos));
                                pe[e] = vis ? pe[e] : 0.0f;
                                ds[e] = vis ? ds[e] : 0.0f;
                            }
                        }
                        pk[u / 2] = pack_bf16x2(pe[0], pe[1]);
                        pk[u / 2 + 1] = pack_bf16x2(pe[2], pe[3]);
                        dk[u / 2] = pack_bf16x2(ds[0], ds[1]);
                        dk[u / 2 + 1] = pack_bf16x2(ds[2], ds[3]);
                    }
                    if (x.kv) tmem_st16(tmem + lane_off + T_S + 64 * hh + 16 * ch, pk);
                    tmem_st16(tmem + lane_off + T_DP + 64 * hh + 16 * ch, dk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&B->p_full);
            }
            if (!ok) break;
            // epilogue: the accumulators of this half of the channels -> bf16 rows
            if (!__all_sync(FULL, mbar_wait(&B->o_done, (g - 1) & 1, abort, lim))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool store = rpos < x.len;
            const long long row = ((long long)(x.start + (store ? rpos : 0)) * p.H + x.head) * D + 64 * hh;
            for (int which = 0; which < (x.kv ? 2 : 1); which++) {
                // dK/dV role: dV (unscaled), then dK; dQ role: dQ
                const uint32_t col = (which ? T_O1 : T_O0) + 64 * hh;
                const float f = (x.kv && which == 0) ? 1.0f : p.scale;
                uint16_t* out = x.kv ? (which ? p.dk : p.dv) : p.dq;
                const float2 f2 = make_float2(f, f);
#pragma unroll
                for (int cc = 0; cc < 2; cc++) {
                    uint32_t u[32];
                    tmem_ld32(tmem + lane_off + col + 32 * cc, u);
                    tmem_wait_ld();
                    uint32_t pkd[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; i2++) {
                        const float2 v2 =
                            __fmul2_rn(make_float2(__uint_as_float(u[2 * i2]), __uint_as_float(u[2 * i2 + 1])), f2);
                        pkd[i2] = pack_bf16x2(v2.x, v2.y);
                    }
                    if (store) {
                        uint4* dst = reinterpret_cast<uint4*>(out + row + 32 * cc);
#pragma unroll
                        for (int i2 = 0; i2 < 4; i2++)
                            dst[i2] = make_uint4(pkd[4 * i2], pkd[4 * i2 + 1], pkd[4 * i2 + 2], pkd[4 * i2 + 3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&B->epi_done);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && *abort) atomicOr(&p.hdr->status, ST_TIMEOUT);
}

cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* dout, const BwdParams& p, int grid,
                       cudaStream_t st) {
    using namespace bwd;
    if (grid < 2 || (grid & 1)) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mdo;
    if (!make_map(&mq, q, 2, p.T, p.H, D, 64, true) || !make_map(&mk, k, 2, p.T, p.H, D, 64, true) ||
        !make_map(&mv, v, 2, p.T, p.H, D, 64, true) || !make_map(&mdo, dout, 2, p.T, p.H, D, 64, true))
        return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(bwd_prep_kernel, dim3((unsigned)p.tiles_cap, (unsigned)p.H), dim3(256), 0, st, p);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_bwd_kernel, dim3(grid), dim3(THREADS), SMEM, st, mq, mk, mv, mdo, p);
}

}  // namespace pa
