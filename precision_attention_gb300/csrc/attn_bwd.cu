// attn_bwd.cu -- attention backward (dQ, dK, dV) for BF16 operands, d = 64 or
// 128, on sm_103a (tcgen05 + TMEM + TMA).
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
// Three launches after the work-list pass (the forward's one-query-tile list),
// each a programmatic dependent of the one before:
//   bwd_prep_kernel  D and lse log2(e) per row, stored per (head, 128-token
//                    tile) so the gradient kernels fetch the values of a run
//                    of rows with one bulk copy
//   attn_bwd_kernel  persistent, in its dK/dV role (kv_only = 1; with
//                    kv_only = 0 its work items alternate between the two
//                    roles below), both for one (document, head, 128-token row
//                    tile), each a loop over 64-row stream tiles:
//     dK/dV role   key tile j: K_j and V_j once, then each 64-query tile i that
//                  sees it: S^T = K_j Q_i^T and dP^T = V_j dO_i^T into TMEM,
//                  P^T and dS^T in registers, stored as bf16 into shared
//                  memory, then dV += P^T dO_i and dK += dS^T Q_i
//     dQ role      query tile i: Q_i and dO_i once, then each 64-key tile j it
//                  sees: S = Q_i K_j^T, dP = dO_i V_j^T, dS into shared memory,
//                  dQ += dS K_j
//   dQ is formed in its own role (S and dP computed a second time) rather than
//   accumulated across key tiles with atomics, so the gradients are
//   deterministic: one fixed summation order per output element.
//   attn_bwd_dq_kernel  the dQ role with 128-key steps (below), the form the
//                    library launches after the dK/dV pass
// Warp roles: warp 0 TMA producer (the item's two row tiles, then the two
// stream tiles of each step, and in the dK/dV role the step's 64 lse and D
// values, into a 3-stage ring); warp 1 TMEM owner and MMA issuer; warps 2-9
// elementwise in two groups of four that take the steps in turn (one thread
// per row, all 64 columns), and together the epilogue.
// TMEM (512 columns): the item's two row tiles [0,128) as the A operand of S
// and dP (the elementwise warps copy them in from the TMA-loaded tiles once per
// item), so those MMAs read only their B slice from shared memory; S [128,192)
// and dP [192,256); dV or dQ [256,384), dK [384,512). Shared memory holds two
// P/dS buffers. The S/dP columns are free as soon as a group has loaded them,
// so the issuer keeps S and dP of the next step queued ahead of the output
// MMAs, and the tensor pipe runs S(g + 1), out(g), S(g + 2), out(g + 1), ...
// while the elementwise warps work on the step between.
// Every wait is bounded; on a timeout the CTA raises its flag, drains, frees
// TMEM and returns, and the host reads ATTN_ERR_DEVICE_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "attn_common.cuh"
#include "pdl.cuh"

namespace pa {

namespace bwd {
constexpr int SR = 64;                     // rows of a stream tile
constexpr int NS = 3;                      // stream-tile stages
constexpr int PT = 128 * SR * 2;           // a P or dS operand: 128 rows x 64 bf16, one 128-byte swizzle atom
constexpr int THREADS = 64 + 256;
// TMEM columns: the one S/dP buffer and the accumulators (the row tiles: Lay)
constexpr uint32_t T_R0 = 0, T_S = 128, T_DP = 192, T_O0 = 256, T_O1 = 384;

// shared-memory layout and shapes for head dimension D (64 or 128); a row of D
// bf16 channels is D / 64 atoms of the 128-byte swizzle
template <int D>
struct Lay {
    static constexpr int ATOMS = D / 64;
    static constexpr int TILE = 128 * D * 2;       // a row tile of 128 rows
    static constexpr int XTILE = SR * D * 2;       // a stream tile
    static constexpr int OFF_R = 0;                // row tiles R0, R1
    static constexpr int OFF_X = 2 * TILE;         // NS stages of the stream tiles X0, X1
    static constexpr int OFF_P = OFF_X + NS * 2 * XTILE;   // two buffers of {P, dS}
    static constexpr int OFF_VEC = OFF_P + 2 * 2 * PT;     // NS x {lse log2(e) [64], D [64]}
    static constexpr int OFF_BAR = OFF_VEC + NS * 512;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;
    static constexpr int KS = D / 16;              // K steps of S and dP (16 channels each)
    static constexpr int HD = D / 2;               // channels per warp half in the epilogue
    // the row tiles in TMEM as the A operand of S and dP: bf16 pairs, column c of a
    // row holding channels 2c, 2c + 1
    static constexpr uint32_t T_R1 = D / 2;
    static_assert(Cfg<2, D, MODE_BF16>::TILE == TILE && Cfg<2, D, MODE_BF16>::ATOMS == ATOMS,
                  "row tiles as the forward's bf16 tiles");
    static_assert(SMEM <= 227 * 1024, "backward shared memory exceeds the per-CTA limit");
};

struct Bars {
    uint64_t r_full, r_empty;   // the item's row tiles landed in shared memory / may be replaced
    uint64_t r_tmem;      // the item's row tiles copied into TMEM (256 arrivals)
    uint64_t x_full[NS], x_empty[NS];
    uint64_t s_full[2];   // S and dP of a step of group b are in TMEM
    uint64_t s_free[2];   // group b has loaded them (128 arrivals)
    uint64_t p_full[2];   // P and dS of the step are in shared-memory buffer b (128 arrivals)
    uint64_t o_done[2];   // the step's output MMAs, readers of P/dS buffer b, completed
    uint64_t epi_done;    // the item's accumulators were read (256 arrivals)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 512, "backward barrier block exceeds its reserved space");

// K-major B operand of S = R X^T: a 64-row stream tile, K step kk (32 bytes of channels)
__device__ __forceinline__ uint64_t desc_x_kmajor(uint32_t base, int kk) {
    return sdesc(base + (uint32_t)((kk >> 2) * (SR * 128) + (kk & 3) * 32), 16, 1024, SWZ_128B);
}
// MN-major B operand of the output products: the stream tile's rows are the K
// dimension (16 per step), its channels the N dimension (two atoms SR * 128 bytes apart)
__device__ __forceinline__ uint64_t desc_x_mn(uint32_t base, int kk) {
    return sdesc(base + (uint32_t)(kk * 16 * 128), SR * 128, 1024, SWZ_128B);
}
// K-major A operand of the output products: P or dS, 128 rows x 64 columns, K step kk
__device__ __forceinline__ uint64_t desc_p64(uint32_t base, int kk) {
    return sdesc(base + (uint32_t)(kk * 32), 16, 1024, SWZ_128B);
}

// One work item of the gradient kernel. Position `it` of the combined list holds
// work item it / 2 of the forward's list in one of the two roles; with an even
// grid, a CTA takes the two roles in turn from round to round, and every item
// appears once in each role.
struct Item {
    int kv;          // 1: dK/dV of key tile rt; 0: dQ of query tile rt
    int head, start, len, toff;
    int rt;          // the 128-row tile (keys or queries), document-local
    int s0, n;       // 64-row stream tiles s0 .. s0 + n - 1
};
__device__ __forceinline__ Item decode(const BwdParams& p, int it) {
    Item x;
    x.kv = p.kv_only || ((it & 1) ^ ((it / (int)gridDim.x) & 1)) == 0;
    const WorkItem w = p.items[p.kv_only ? it : it >> 1];
    const DocEntry d = p.docs[w.doc];
    const int nt = (d.len + 127) >> 7, n64 = (d.len + 63) >> 6;
    x.head = w.head;
    x.start = d.start;
    x.len = d.len;
    x.toff = d.toff;
    if (x.kv) {
        // causal: query tile qtile of the list sees qtile + 1 key tiles; key tile
        // nt - 1 - qtile is seen by as many query tiles (from itself to the last)
        x.rt = p.causal ? nt - 1 - w.qtile : w.qtile;
        x.s0 = p.causal ? 2 * x.rt : 0;
        x.n = n64 - x.s0;
    } else {
        x.rt = w.qtile;
        x.s0 = 0;
        x.n = p.causal ? min(2 * x.rt + 2, n64) : n64;
    }
    return x;
}
}  // namespace bwd

// D = rowsum(dO o O) and lse log2(e) of every row, per (head, 128-token tile).
// Grid (tiles_cap, H); eight warps, one row per warp at a time.
template <int D>
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
            const long long base = ((long long)(d.start + loc) * p.H + h) * D + (D / 32) * lane;
            if constexpr (D == 128) {
                const uint2 a = *reinterpret_cast<const uint2*>(p.o + base);
                const uint2 b = *reinterpret_cast<const uint2*>(p.dout + base);
                const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a.x));
                const float2 a1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a.y));
                const float2 b0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.x));
                const float2 b1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.y));
                dsum = a0.x * b0.x + a0.y * b0.y + a1.x * b1.x + a1.y * b1.y;
            } else {
                const uint32_t a = *reinterpret_cast<const uint32_t*>(p.o + base);
                const uint32_t b = *reinterpret_cast<const uint32_t*>(p.dout + base);
                const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a));
                const float2 b0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b));
                dsum = a0.x * b0.x + a0.y * b0.y;
            }
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

template <int D>
__global__ void __launch_bounds__(bwd::THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                    const __grid_constant__ CUtensorMap sxq, const __grid_constant__ CUtensorMap sxk,
                    const __grid_constant__ CUtensorMap sxv, const __grid_constant__ CUtensorMap sxdo,
                    const BwdParams p) {
    // tm*: 128-row boxes (the row tiles); sx*: 64-row boxes (the stream tiles)
    using namespace bwd;
    using L = Lay<D>;
    constexpr int TILE = L::TILE, XTILE = L::XTILE, ATOMS = L::ATOMS;
    constexpr int OFF_R = L::OFF_R, OFF_X = L::OFF_X, OFF_P = L::OFF_P, OFF_VEC = L::OFF_VEC, OFF_BAR = L::OFF_BAR;
    constexpr uint32_t T_R1 = L::T_R1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* B = reinterpret_cast<Bars*>(sm + OFF_BAR);
    volatile int* abort = &B->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long lim = p.wait_limit;

    if (threadIdx.x == 0) {
        mbar_init(&B->r_full, 1);
        mbar_init(&B->r_tmem, 256);
        mbar_init(&B->r_empty, 1);
        for (int i = 0; i < NS; i++) {
            mbar_init(&B->x_full[i], 1);
            mbar_init(&B->x_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&B->s_full[i], 1);
            mbar_init(&B->s_free[i], 128);
            mbar_init(&B->p_full[i], 128);
            mbar_init(&B->o_done[i], 1);
        }
        mbar_init(&B->epi_done, 256);
        mbar_init(&B->drain, 1);
        B->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmq);
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        prefetch_tensormap(&tmdo);
        prefetch_tensormap(&sxq);
        prefetch_tensormap(&sxk);
        prefetch_tensormap(&sxv);
        prefetch_tensormap(&sxdo);
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
    const int n_items = (p.kv_only ? 1 : 2) * p.hdr->n_items;

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
            const CUtensorMap* x0 = x.kv ? &sxq : &sxk;
            const CUtensorMap* x1 = x.kv ? &sxdo : &sxv;
            if (!__all_sync(FULL, mbar_wait(&B->r_empty, (qi & 1) ^ 1, abort, lim))) break;
            r_issued = qi & 1;
            if (lane == 0) {
                mbar_arrive_expect_tx(&B->r_full, 2 * TILE);
                const int row = x.start + 128 * x.rt;
                for (int a = 0; a < ATOMS; a++) {
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
                    const int s64 = x.s0 + t;
                    const int row = x.start + SR * s64;
                    uint8_t* xs = sm + OFF_X + st * 2 * XTILE;
                    mbar_arrive_expect_tx(&B->x_full[st], 2 * XTILE + (x.kv ? 512 : 0));
                    for (int a = 0; a < ATOMS; a++) {
                        tma_load_3d(xs + a * (SR * 128), x0, &B->x_full[st], a * 64, x.head, row);
                        tma_load_3d(xs + XTILE + a * (SR * 128), x1, &B->x_full[st], a * 64, x.head, row);
                    }
                    if (x.kv) {   // the 64 queries' lse log2(e) and D
                        const float* vl = p.vec + ((long long)x.head * p.tiles_cap + x.toff + (s64 >> 1)) * 128 +
                                          64 * (s64 & 1);
                        uint8_t* dst = sm + OFF_VEC + st * 512;
                        bulk_load(dst, vl, 256, &B->x_full[st]);
                        bulk_load(dst + 256, vl + (long long)p.H * p.tiles_cap * 128, 256, &B->x_full[st]);
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
        // The whole warp runs the loop, so the descriptors are computed in converged
        // code from values every lane shares; lane 0 alone executes the MMAs and
        // their commits.
        {
            constexpr unsigned FULL = 0xFFFFFFFFu;
            const bool leader = lane == 0;
            constexpr uint32_t id_s = idesc(1, 1, false, false, 128, SR);    // A from TMEM, K-major B, N = 64
            constexpr uint32_t id_o = idesc(1, 1, false, true, 128, D);      // K-major A, MN-major B
            const uint32_t sX = smem_u32(sm + OFF_X);
            // Descriptors are built once: every operand sits at a fixed shared-memory
            // address, so a stage, buffer or K step only adds a constant to the
            // start-address field (addresses stay below 256 KB, the field never carries).
            const uint32_t sP0 = smem_u32(sm + OFF_P);
            const uint64_t dxk = desc_x_kmajor(sX, 0), dxm = desc_x_mn(sX, 0), dpa = desc_p64(sP0, 0);
            constexpr uint64_t XST16 = (uint64_t)(2 * XTILE) >> 4, X1_16 = (uint64_t)XTILE >> 4;
            constexpr uint64_t PB16 = (uint64_t)(2 * PT) >> 4, DS16 = (uint64_t)PT >> 4;
            constexpr uint64_t KP16 = 32 >> 4, KX16 = (16 * 128) >> 4;   // out K step: 16 columns of P, 16 rows of X
            auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
                return __all_sync(FULL, mbar_wait(bar, parity, abort, lim));
            };
            // step gs: S and dP of its stream stage into TMEM buffer gs & 1
            // (A, the row tiles, from TMEM: each MMA reads only its 2 KB B slice from
            // shared memory, so the N = 64 products run at the tensor rate)
            auto issue_s = [&](uint32_t gs) {
                const uint64_t x0 = dxk + (gs % NS) * XST16, x1 = x0 + X1_16;
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < L::KS; kk++) {
                        const uint64_t xo = (uint64_t)((kk >> 2) * (SR * 128) + (kk & 3) * 32) >> 4;
                        mma_f16_ta(tmem + T_S, tmem + T_R0 + 8 * kk, x0 + xo, id_s, kk ? 1u : 0u);
                    }
#pragma unroll
                    for (int kk = 0; kk < L::KS; kk++) {
                        const uint64_t xo = (uint64_t)((kk >> 2) * (SR * 128) + (kk & 3) * 32) >> 4;
                        mma_f16_ta(tmem + T_DP, tmem + T_R1 + 8 * kk, x1 + xo, id_s, kk ? 1u : 0u);
                    }
                    tc_commit(&B->s_full[gs & 1]);
                }
                __syncwarp();
            };
            uint32_t g = 0;     // steps whose output MMAs are issued
            uint32_t gs = 0;    // steps whose S and dP are issued
            int qi = 0;
            bool ok = true;
            // S and dP of step gs, once its stream tiles have landed and the elementwise
            // warps have loaded step gs - 1 out of the S/dP columns
            auto try_issue_s = [&]() -> bool {
                if (!wait_all(&B->x_full[gs % NS], (gs / NS) & 1)) return false;
                if (gs >= 1 && !wait_all(&B->s_free[(gs - 1) & 1], ((gs - 1) >> 1) & 1)) return false;
                tc_fence_after();
                issue_s(gs);
                gs++;
                return true;
            };
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, qi++) {
                const Item x = decode(p, it);
                if (!wait_all(&B->r_tmem, qi & 1)) break;   // the row tiles, in TMEM
                const uint32_t g_end = g + x.n;   // this item's steps: g .. g_end - 1
                for (int t = 0; t < x.n && ok; t++, g++) {
                    // S and dP one step ahead of the output MMAs, within the item: the pipe
                    // runs S(g + 1), out(g), S(g + 2), out(g + 1), ... (S(g + 2) waits for the
                    // stream stage that out(g - 1) frees, so it is issued after out(g))
                    while (ok && gs < g_end && gs <= g + 1) ok = try_issue_s();
                    if (!ok) break;
                    if (!wait_all(&B->p_full[g & 1], (g >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    // the previous item's epilogue has read the accumulators
                    if (t == 0 && qi > 0 && !wait_all(&B->epi_done, (qi - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t x0 = dxm + (g % NS) * XST16, x1 = x0 + X1_16;
                    const uint64_t pb = dpa + (g & 1) * PB16, db = pb + DS16;
                    const uint32_t acc0 = t ? 1u : 0u;
                    if (leader) {
                        if (x.kv) {
#pragma unroll
                            for (int kk = 0; kk < 4; kk++)   // dV += P^T dO
                                mma_f16(tmem + T_O0, pb + kk * KP16, x1 + kk * KX16, id_o, kk ? 1u : acc0);
#pragma unroll
                            for (int kk = 0; kk < 4; kk++)   // dK += dS^T Q
                                mma_f16(tmem + T_O1, db + kk * KP16, x0 + kk * KX16, id_o, kk ? 1u : acc0);
                        } else {
#pragma unroll
                            for (int kk = 0; kk < 4; kk++)   // dQ += dS K
                                mma_f16(tmem + T_O0, db + kk * KP16, x0 + kk * KX16, id_o, kk ? 1u : acc0);
                        }
                        tc_commit(&B->x_empty[g % NS]);
                        tc_commit(&B->o_done[g & 1]);
                        if (t == x.n - 1) tc_commit(&B->r_empty);
                    }
                    __syncwarp();
                }
            }
            // every MMA lane 0 issued has completed before TMEM is released
            if (leader) {
                tc_commit(&B->drain);
                wait_drain(&B->drain, 0, kDrainLimit);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ elementwise + epilogue
        // Two groups of four warps take the steps in turn (group gr: the steps g with
        // g % 2 == gr, TMEM and P/dS buffer gr), so one group's chain (S from TMEM, P and
        // dS, stores) overlaps the other's; within a group, warp w covers TMEM lane
        // quarter w % 4 and one thread a row, all 64 columns.
        constexpr unsigned FULL = 0xFFFFFFFFu;
        const int gr = (warp - 2) >> 2;                      // step group
        const int quarter = warp & 3;                        // TMEM lane quarter
        const int r = quarter * 32 + lane;                   // row of the row tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float2 c2 = make_float2(p.C, p.C);
        uint32_t g = 0;
        int qi = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, qi++) {
            const Item x = decode(p, it);
            const int rpos = 128 * x.rt + r;                 // document-local position of this row
            // dQ role: this row's lse log2(e) and D
            float row_l2 = 0.0f, row_d = 0.0f;
            if (!x.kv) {
                const long long vi = ((long long)x.head * p.tiles_cap + x.toff + x.rt) * 128 + r;
                row_l2 = p.vec[vi];
                row_d = p.vec[vi + (long long)p.H * p.tiles_cap * 128];
            }
            // the item's row tiles into TMEM (group 0: R0, group 1: R1; a thread its row).
            // Every MMA of the previous item has completed: its epilogue waited for them.
            if (ok && !__all_sync(FULL, mbar_wait(&B->r_full, qi & 1, abort, lim))) ok = false;
            if (ok) {
                const uint8_t* rt = sm + OFF_R + gr * TILE + r * 128;
#pragma unroll
                for (int a = 0; a < ATOMS; a++) {
                    uint32_t w[32];
#pragma unroll
                    for (int c8 = 0; c8 < 8; c8++) {
                        const uint4 v4 = *reinterpret_cast<const uint4*>(rt + a * 16384 + ((c8 ^ (r & 7)) << 4));
                        w[4 * c8] = v4.x;
                        w[4 * c8 + 1] = v4.y;
                        w[4 * c8 + 2] = v4.z;
                        w[4 * c8 + 3] = v4.w;
                    }
                    tmem_st32(tmem + lane_off + (gr ? T_R1 : T_R0) + 32 * a, w);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&B->r_tmem);
            }
            for (int t = 0; t < x.n && ok; t++, g++) {
                const int st = g % NS, b = g & 1;
                if (b != gr) continue;
                if (!__all_sync(FULL, mbar_wait(&B->s_full[b], (g >> 1) & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                // the bulk-copied vectors: observe their barrier as well (its phase cannot
                // advance past this step before this group arrives on p_full)
                if (x.kv && !__all_sync(FULL, mbar_wait(&B->x_full[st], (g / NS) & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int s64 = x.s0 + t;
                const int cbase = SR * s64;                   // document-local position of column 0
                // masked: a stream tile inside the causal diagonal tile, or one reaching
                // past the document's end
                const bool need_mask = (p.causal && (s64 >> 1) == x.rt) || (SR * s64 + SR > x.len);
                const float* vl = reinterpret_cast<const float*>(sm + OFF_VEC + st * 512);
                const float* vd = vl + 64;
                const uint32_t tb = tmem + lane_off + T_S;
                // S and dP of all 64 columns first: the S/dP columns go back to the issuer
                // before any arithmetic, so S and dP of step g + 1 can start at once
                uint32_t us[64], ud[64];
                {
                    uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&us[0]);
                    uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&us[32]);
                    uint32_t (&d0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ud[0]);
                    uint32_t (&d1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ud[32]);
                    tmem_ld32(tb, s0);
                    tmem_ld32(tb + 32, s1);
                    tmem_ld32(tb + 64, d0);
                    tmem_ld32(tb + 96, d1);
                }
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&B->s_free[b]);   // the S/dP columns may take step g + 1
                // the P/dS buffer was last read by the output MMAs of step g - 2
                if (g >= 2 && !__all_sync(FULL, mbar_wait(&B->o_done[b], ((g - 2) >> 1) & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                uint8_t* pbuf = sm + OFF_P + b * 2 * PT;
                // P = 2^(S c - lse log2 e), dS = P (dP - D), in pairs, 8 columns (one 16-byte
                // chunk of each row) at a time, stored as they are formed into the 128-byte
                // swizzled K-major rows; one branch-free unrolled loop per (role, masked) case
                auto compute = [&](auto kv_c, auto mask_c) {
                    constexpr bool KV = decltype(kv_c)::value, MASK = decltype(mask_c)::value;
#pragma unroll
                    for (int cc = 0; cc < 8; cc++) {
                        uint32_t pw[4], dw[4];
#pragma unroll
                        for (int v = 0; v < 8; v += 4) {
                            const int col = 8 * cc + v;
                            float2 l01, l23, d01, d23;
                            if constexpr (KV) {
                                const float4 a = *reinterpret_cast<const float4*>(vl + col);
                                const float4 bb = *reinterpret_cast<const float4*>(vd + col);
                                l01 = make_float2(-a.x, -a.y);
                                l23 = make_float2(-a.z, -a.w);
                                d01 = make_float2(-bb.x, -bb.y);
                                d23 = make_float2(-bb.z, -bb.w);
                            } else {
                                l01 = l23 = make_float2(-row_l2, -row_l2);
                                d01 = d23 = make_float2(-row_d, -row_d);
                            }
                            const float2 x01 = __ffma2_rn(
                                make_float2(__uint_as_float(us[col]), __uint_as_float(us[col + 1])), c2, l01);
                            const float2 x23 = __ffma2_rn(
                                make_float2(__uint_as_float(us[col + 2]), __uint_as_float(us[col + 3])), c2, l23);
                            float2 p01 = make_float2(ex2(x01.x), ex2(x01.y));
                            float2 p23 = make_float2(ex2(x23.x), ex2(x23.y));
                            const float2 g01 = __fadd2_rn(
                                make_float2(__uint_as_float(ud[col]), __uint_as_float(ud[col + 1])), d01);
                            const float2 g23 = __fadd2_rn(
                                make_float2(__uint_as_float(ud[col + 2]), __uint_as_float(ud[col + 3])), d23);
                            float2 s01 = __fmul2_rn(p01, g01);
                            float2 s23 = __fmul2_rn(p23, g23);
                            if constexpr (MASK) {
                                float* pp[4] = {&p01.x, &p01.y, &p23.x, &p23.y};
                                float* ss[4] = {&s01.x, &s01.y, &s23.x, &s23.y};
#pragma unroll
                                for (int e = 0; e < 4; e++) {
                                    const int cpos = cbase + col + e;
                                    // dK/dV role: column = query, row = key; dQ role: the reverse
                                    const bool vis =
                                        cpos < x.len && (!p.causal || (KV ? cpos >= rpos : cpos <= rpos));
                                    *pp[e] = vis ? *pp[e] : 0.0f;
                                    *ss[e] = vis ? *ss[e] : 0.0f;
                                }
                            }
                            pw[v / 2] = pack_bf16x2(p01.x, p01.y);
                            pw[v / 2 + 1] = pack_bf16x2(p23.x, p23.y);
                            dw[v / 2] = pack_bf16x2(s01.x, s01.y);
                            dw[v / 2 + 1] = pack_bf16x2(s23.x, s23.y);
                        }
                        const int off = r * 128 + ((cc ^ (r & 7)) << 4);
                        if constexpr (KV)
                            *reinterpret_cast<uint4*>(pbuf + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                        *reinterpret_cast<uint4*>(pbuf + PT + off) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
                    }
                };
                if (x.kv) {
                    if (need_mask) compute(std::true_type{}, std::true_type{});
                    else compute(std::true_type{}, std::false_type{});
                } else {
                    if (need_mask) compute(std::false_type{}, std::true_type{});
                    else compute(std::false_type{}, std::false_type{});
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&B->p_full[b]);
            }
            // epilogue: the group that ran the item's last step waits for its output MMAs
            // (it has waited on every earlier phase of that barrier), then both groups
            // store: warp w the rows of lane quarter w % 4, channel half hh. Every
            // elementwise thread reaches this barrier once per item, stopped or not, and
            // all take the same exit decision from it.
            if (ok && ((g - 1) & 1) == (uint32_t)gr &&
                !__all_sync(FULL, mbar_wait(&B->o_done[gr], ((g - 1) >> 1) & 1, abort, lim)))
                ok = false;
            if (named_bar_or(1, 256, !ok || *abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int hh = gr;
            const bool store = rpos < x.len;
            const long long row = ((long long)(x.start + (store ? rpos : 0)) * p.H + x.head) * D + L::HD * hh;
            for (int which = 0; which < (x.kv ? 2 : 1); which++) {
                // dK/dV role: dV (unscaled), then dK; dQ role: dQ
                const uint32_t col = (which ? T_O1 : T_O0) + L::HD * hh;
                const float f = (x.kv && which == 0) ? 1.0f : p.scale;
                uint16_t* out = x.kv ? (which ? p.dk : p.dv) : p.dq;
                const float2 f2 = make_float2(f, f);
#pragma unroll
                for (int cc = 0; cc < L::HD / 32; cc++) {
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

// ---------------------------------------------------------------------------
// dQ in its own kernel, 128 keys per step. With only one accumulator (dQ), TMEM
// holds the item's Q and dO tiles as the A operand [0, D), S [128,256) and dP
// [256,384) at N = 128, and dQ [384, 384 + D): S and dP take half the MMA
// instructions per FLOP of the 64-row steps above, which the issuing thread is
// bound by. Warp 0 streams the K and V tiles of each key tile (2 stages), warp 1
// issues (S and dP of the next step ahead of dQ += dS K of this one), warps 2-9
// form dS for 64 of the 128 keys each (two warps per TMEM lane quarter) into one
// of two shared-memory dS buffers, and together the epilogue.
namespace bwdq {
constexpr int NS = 2;
constexpr int DST = 128 * 128 * 2;   // dS: 128 query rows x 128 keys, two 128-byte swizzle atoms
template <int D>
struct Lay {
    static constexpr int ATOMS = D / 64;
    static constexpr int XT = 128 * D * 2;               // a 128-row K or V tile
    static constexpr int OFF_X = 0;                      // NS stages of {K, V}
    static constexpr int OFF_DS = OFF_X + NS * 2 * XT;   // two dS buffers
    static constexpr int OFF_BAR = OFF_DS + 2 * DST;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;
    static constexpr int KS = D / 16;                    // K steps of S and dP
    static constexpr int HD = D / 2;                     // dQ channels per warp half
    static constexpr uint32_t T_Q = 0, T_DO = D / 2, T_S = 128, T_DP = 256, T_DQ = 384;
    static_assert(SMEM <= 227 * 1024, "dQ kernel shared memory exceeds the per-CTA limit");
};
struct Bars {
    uint64_t r_tmem;                 // Q and dO of the item in TMEM (256 arrivals)
    uint64_t x_full[NS], x_empty[NS];
    uint64_t s_full;                 // S and dP of a step in TMEM
    uint64_t s_free;                 // loaded by the elementwise warps (256 arrivals)
    uint64_t p_full[2];              // dS of the step in shared-memory buffer b (256 arrivals)
    uint64_t o_done[2];              // the step's dQ MMAs, readers of dS buffer b, completed
    uint64_t epi_done;               // the item's dQ was read (256 arrivals)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 512, "dQ kernel barrier block exceeds its reserved space");
}  // namespace bwdq

template <int D>
__global__ void __launch_bounds__(bwd::THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const BwdParams p) {
    using namespace bwdq;
    using L = Lay<D>;
    constexpr unsigned FULL = 0xFFFFFFFFu;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* B = reinterpret_cast<Bars*>(sm + L::OFF_BAR);
    volatile int* abort = &B->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long lim = p.wait_limit;
    if (threadIdx.x == 0) {
        mbar_init(&B->r_tmem, 256);
        for (int i = 0; i < NS; i++) {
            mbar_init(&B->x_full[i], 1);
            mbar_init(&B->x_empty[i], 1);
        }
        mbar_init(&B->s_full, 1);
        mbar_init(&B->s_free, 256);
        for (int i = 0; i < 2; i++) {
            mbar_init(&B->p_full[i], 256);
            mbar_init(&B->o_done[i], 1);
        }
        mbar_init(&B->epi_done, 256);
        mbar_init(&B->drain, 1);
        B->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
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
    const int n_items = p.hdr->n_items;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int issued[NS];
        for (int i = 0; i < NS; i++) issued[i] = -1;
        uint32_t g = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const WorkItem w = p.items[it];
            const DocEntry d = p.docs[w.doc];
            for (int t = 0; t < w.ntiles; t++, g++) {
                const int st = g % NS;
                if (!__all_sync(FULL, mbar_wait(&B->x_empty[st], ((g / NS) & 1) ^ 1, abort, lim))) {
                    ok = false;
                    break;
                }
                issued[st] = (g / NS) & 1;
                if (lane == 0) {
                    uint8_t* xs = sm + L::OFF_X + st * 2 * L::XT;
                    mbar_arrive_expect_tx(&B->x_full[st], 2 * L::XT);
                    for (int a = 0; a < L::ATOMS; a++) {
                        tma_load_3d(xs + a * 16384, &tmk, &B->x_full[st], a * 64, w.head, d.start + 128 * t);
                        tma_load_3d(xs + L::XT + a * 16384, &tmv, &B->x_full[st], a * 64, w.head, d.start + 128 * t);
                    }
                }
            }
        }
        if (*abort && lane == 0)
            for (int s2 = 0; s2 < NS; s2++)
                if (issued[s2] >= 0) wait_drain(&B->x_full[s2], (uint32_t)issued[s2], kDrainLimit);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (warp-wide loop)
        const bool leader = lane == 0;
        constexpr uint32_t id_s = idesc(1, 1, false, false, 128, 128);   // A from TMEM, K-major B, N = 128
        constexpr uint32_t id_o = idesc(1, 1, false, true, 128, D);      // K-major A (dS), MN-major B (K)
        const uint32_t sX = smem_u32(sm + L::OFF_X), sD = smem_u32(sm + L::OFF_DS);
        const uint64_t dk0 = desc_kmajor<2, D, MODE_BF16>(sX, 0);        // K (and V) as the K-major B of S, dP
        const uint64_t dkm = desc_v<2, D, MODE_BF16>(sX, 0);             // K as the MN-major B of dQ
        const uint64_t dsa = desc_p<2>(sD, 0);                            // dS as the K-major A of dQ
        constexpr uint64_t XST16 = (uint64_t)(2 * L::XT) >> 4, V16 = (uint64_t)L::XT >> 4, DS16 = (uint64_t)DST >> 4;
        auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(FULL, mbar_wait(bar, parity, abort, lim));
        };
        uint32_t g = 0, gs = 0;
        int qi = 0;
        bool ok = true;
        auto try_issue_s = [&]() -> bool {
            if (!wait_all(&B->x_full[gs % NS], (gs / NS) & 1)) return false;
            if (gs >= 1 && !wait_all(&B->s_free, (gs - 1) & 1)) return false;   // S, dP of gs - 1 loaded
            tc_fence_after();
            const uint64_t bk = dk0 + (gs % NS) * XST16, bv = bk + V16;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < L::KS; kk++)
                    mma_f16_ta(tmem + L::T_S, tmem + L::T_Q + 8 * kk, bk + koff<2, D, MODE_BF16>(kk), id_s, kk ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < L::KS; kk++)
                    mma_f16_ta(tmem + L::T_DP, tmem + L::T_DO + 8 * kk, bv + koff<2, D, MODE_BF16>(kk), id_s,
                               kk ? 1u : 0u);
                tc_commit(&B->s_full);
            }
            __syncwarp();
            gs++;
            return true;
        };
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, qi++) {
            const WorkItem w = p.items[it];
            if (!wait_all(&B->r_tmem, qi & 1)) break;
            const uint32_t g_end = g + w.ntiles;
            for (int t = 0; t < w.ntiles && ok; t++, g++) {
                while (ok && gs < g_end && gs <= g + 1) ok = try_issue_s();
                if (!ok) break;
                if (!wait_all(&B->p_full[g & 1], (g >> 1) & 1)) {
                    ok = false;
                    break;
                }
                if (t == 0 && qi > 0 && !wait_all(&B->epi_done, (qi - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t a0 = dsa + (g & 1) * DS16, bk = dkm + (g % NS) * XST16;
                const uint32_t acc0 = t ? 1u : 0u;
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < 8; kk++)   // dQ += dS K, 16 keys per step
                        mma_f16(tmem + L::T_DQ, a0 + poff(kk), bk + voff<2, D, MODE_BF16>(kk), id_o, kk ? 1u : acc0);
                    tc_commit(&B->x_empty[g % NS]);
                    tc_commit(&B->o_done[g & 1]);
                }
                __syncwarp();
            }
        }
        if (leader) {
            tc_commit(&B->drain);
            wait_drain(&B->drain, 0, kDrainLimit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ elementwise + epilogue
        const int hh = (warp - 2) >> 2;                  // key half (64 of the 128 keys)
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;               // query row of the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float2 c2 = make_float2(p.C, p.C);
        uint32_t g = 0;
        int qi = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, qi++) {
            const WorkItem w = p.items[it];
            const DocEntry d = p.docs[w.doc];
            const int rt = w.qtile, len = d.len;
            const int rpos = 128 * rt + r;
            const long long vi = ((long long)w.head * p.tiles_cap + d.toff + rt) * 128 + r;
            const float row_l2 = p.vec[vi];
            const float row_d = p.vec[vi + (long long)p.H * p.tiles_cap * 128];
            // Q (half 0) or dO (half 1) of this row into TMEM; rows past the document's end
            // are zero. Every MMA of the previous item has completed (its epilogue waited).
            {
                const uint16_t* src = hh ? p.dout : p.q;
                const bool in_doc = rpos < len;
                const uint4* row4 =
                    reinterpret_cast<const uint4*>(src + ((long long)(d.start + (in_doc ? rpos : 0)) * p.H + w.head) * D);
#pragma unroll
                for (int a = 0; a < L::ATOMS; a++) {
                    uint32_t wv[32];
#pragma unroll
                    for (int c8 = 0; c8 < 8; c8++) {
                        const uint4 v4 = in_doc ? __ldg(row4 + 8 * a + c8) : make_uint4(0, 0, 0, 0);
                        wv[4 * c8] = v4.x;
                        wv[4 * c8 + 1] = v4.y;
                        wv[4 * c8 + 2] = v4.z;
                        wv[4 * c8 + 3] = v4.w;
                    }
                    tmem_st32(tmem + lane_off + (hh ? L::T_DO : L::T_Q) + 32 * a, wv);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&B->r_tmem);
            }
            for (int t = 0; t < w.ntiles && ok; t++, g++) {
                const int b = g & 1;
                if (!__all_sync(FULL, mbar_wait(&B->s_full, g & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t us[64], ud[64];
                {
                    uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&us[0]);
                    uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&us[32]);
                    uint32_t (&d0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ud[0]);
                    uint32_t (&d1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&ud[32]);
                    tmem_ld32(tmem + lane_off + L::T_S + 64 * hh, s0);
                    tmem_ld32(tmem + lane_off + L::T_S + 64 * hh + 32, s1);
                    tmem_ld32(tmem + lane_off + L::T_DP + 64 * hh, d0);
                    tmem_ld32(tmem + lane_off + L::T_DP + 64 * hh + 32, d1);
                }
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&B->s_free);
                if (g >= 2 && !__all_sync(FULL, mbar_wait(&B->o_done[b], ((g - 2) >> 1) & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                const int kbase = 128 * t + 64 * hh;            // document-local key of column 0 of this half
                const bool need_mask = (p.causal && t == rt) || (128 * t + 128 > len);
                uint8_t* dsb = sm + L::OFF_DS + b * DST + hh * 16384;
                // dS = 2^(S c - lse log2 e) (dP - D), 8 keys (one 16-byte chunk) at a time
                auto compute = [&](auto mask_c) {
                    constexpr bool MASK = decltype(mask_c)::value;
                    const float2 l2 = make_float2(-row_l2, -row_l2), dd = make_float2(-row_d, -row_d);
#pragma unroll
                    for (int cc = 0; cc < 8; cc++) {
                        uint32_t dw[4];
#pragma unroll
                        for (int v = 0; v < 8; v += 2) {
                            const int col = 8 * cc + v;
                            const float2 x2 = __ffma2_rn(
                                make_float2(__uint_as_float(us[col]), __uint_as_float(us[col + 1])), c2, l2);
                            float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
                            const float2 g2 = __fadd2_rn(
                                make_float2(__uint_as_float(ud[col]), __uint_as_float(ud[col + 1])), dd);
                            float2 s2 = __fmul2_rn(p2, g2);
                            if constexpr (MASK) {
                                const int k0 = kbase + col;
                                const bool v0 = k0 < len && (!p.causal || k0 <= rpos);
                                const bool v1 = k0 + 1 < len && (!p.causal || k0 + 1 <= rpos);
                                s2.x = v0 ? s2.x : 0.0f;
                                s2.y = v1 ? s2.y : 0.0f;
                            }
                            dw[v / 2] = pack_bf16x2(s2.x, s2.y);
                        }
                        *reinterpret_cast<uint4*>(dsb + r * 128 + ((cc ^ (r & 7)) << 4)) =
                            make_uint4(dw[0], dw[1], dw[2], dw[3]);
                    }
                };
                if (need_mask) compute(std::true_type{});
                else compute(std::false_type{});
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&B->p_full[b]);
            }
            // epilogue: every thread has waited on each earlier phase of the last step's
            // o_done barrier; the barrier below gives all threads one exit decision
            if (ok && !__all_sync(FULL, mbar_wait(&B->o_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort, lim)))
                ok = false;
            if (named_bar_or(1, 256, !ok || *abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool store = rpos < len;
            const long long row = ((long long)(d.start + (store ? rpos : 0)) * p.H + w.head) * D + L::HD * hh;
            const float2 f2 = make_float2(p.scale, p.scale);
#pragma unroll
            for (int cc = 0; cc < L::HD / 32; cc++) {
                uint32_t u[32];
                tmem_ld32(tmem + lane_off + L::T_DQ + L::HD * hh + 32 * cc, u);
                tmem_wait_ld();
                uint32_t pkd[16];
#pragma unroll
                for (int i2 = 0; i2 < 16; i2++) {
                    const float2 v2 =
                        __fmul2_rn(make_float2(__uint_as_float(u[2 * i2]), __uint_as_float(u[2 * i2 + 1])), f2);
                    pkd[i2] = pack_bf16x2(v2.x, v2.y);
                }
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(p.dq + row + 32 * cc);
#pragma unroll
                    for (int i2 = 0; i2 < 4; i2++)
                        dst[i2] = make_uint4(pkd[4 * i2], pkd[4 * i2 + 1], pkd[4 * i2 + 2], pkd[4 * i2 + 3]);
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

template <int D>
static cudaError_t launch_bwd_t(const void* q, const void* k, const void* v, const void* dout, const BwdParams& p,
                                int grid, cudaStream_t st) {
    using namespace bwd;
    using L = Lay<D>;
    CUtensorMap m[8];   // q, k, v, dO with 128-row boxes (the row tiles), then with 64-row boxes
    const void* base[4] = {q, k, v, dout};
    for (int i = 0; i < 8; i++)
        if (!make_tensor_map_3d(&m[i], base[i & 3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, p.H, p.T, (uint64_t)D * 2,
                                (uint64_t)p.H * D * 2, 64, i < 4 ? 128 : SR, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(bwd_prep_kernel<D>, dim3((unsigned)p.tiles_cap, (unsigned)p.H), dim3(256), 0, st, p);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    BwdParams pk = p;
    pk.kv_only = 1;   // dK, dV here; dQ in the kernel after it
    e = launch_pdl(attn_bwd_kernel<D>, dim3(grid), dim3(THREADS), L::SMEM, st, m[0], m[1], m[2], m[3], m[4], m[5],
                   m[6], m[7], pk);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bwdq::Lay<D>::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_bwd_dq_kernel<D>, dim3(grid), dim3(THREADS), bwdq::Lay<D>::SMEM, st, m[1], m[2], p);
}

cudaError_t launch_bwd(int D, const void* q, const void* k, const void* v, const void* dout, const BwdParams& p,
                       int grid, cudaStream_t st) {
    if (grid < 2 || (grid & 1)) return cudaErrorInvalidValue;
    if (D == 128) return launch_bwd_t<128>(q, k, v, dout, p, grid, st);
    if (D == 64) return launch_bwd_t<64>(q, k, v, dout, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace pa
