// attn_fwd.cu -- fused attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// The loop is the running softmax of "Fused attention kernel", Implementation
// sketch: per key block S = Q K^T, new row max, rescale exp(m_old - m_new) of
// the old row sum and output, P V accumulation, one normalisation at the end,
// lse = m + log l; every key block is scored. The 8-bit operands and their
// scales come from the quantiser (8-bit forward pass: e4m3, block scales,
// rotated Q and K; FLAMIA section 2: block-scaled MMA consuming 32-element
// E8M0 scales). Score scales are folded into one multiplier per tile (FLAMIA
// section 4.3, "folding score scales"). Causal tiles above the diagonal are
// skipped and the diagonal tile is masked; packed documents are addressed in
// place through the document table (FLAMIA 4.1).
//
// One CTA per SM, persistent over work items (query tile of 128 rows of one
// document and head). Warp roles:
//   warp 0      TMA producer: Q tile once per item, K and V tiles of each key
//               block into an NS-stage ring (plus the MX scale tiles)
//   warp 1      TMEM owner and MMA issuer: S_j = Q K_j^T into one of two TMEM
//               S buffers, then O += P_{j-1} V_{j-1}
//   warps 2-5   softmax: one thread per query row; S row from TMEM, scale,
//               mask, running max/sum, exp2, P row to shared memory (E4M3 or
//               BF16), O rescale in TMEM, final normalisation and stores
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256 + d), MX scale
// factors from column 384.
// Every mbarrier wait is bounded; on a timeout the CTA raises a flag, stops,
// drains its TMA copies, frees TMEM and returns, and the host reads
// ATTN_ERR_DEVICE_TIMEOUT from the status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include "params.h"
#include "ptx.cuh"

namespace pa {

enum { MODE_BF16 = 0, MODE_E4M3_TILE = 1, MODE_E4M3_COL = 2, MODE_MX = 3 };

template <int ELT, int D, int MODE>
struct Cfg {
    static constexpr int RB = D * ELT;                  // bytes per Q/K/V row
    static constexpr bool SW128 = RB >= 128;
    static constexpr int ATOMS = SW128 ? RB / 128 : 1;  // 128-byte column blocks per row
    static constexpr int BOX_ELEMS = SW128 ? 128 / ELT : D;
    static constexpr int TILE = 128 * RB;
    static constexpr int PBYTES = 128 * 128 * ELT;
    static constexpr int NS = ELT == 2 ? 2 : 4;
    static constexpr int KSTEPS_S = RB / 32;            // 32 bytes of K per MMA
    static constexpr int KSTEPS_PV = 128 * ELT / 32;
    static constexpr int KPER = 32 / ELT;               // keys per P V MMA
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_P = OFF_Q + TILE;
    static constexpr int OFF_KV = OFF_P + PBYTES;
    static constexpr int OFF_SF = OFF_KV + NS * 2 * TILE;
    static constexpr int SF_BYTES = MODE == MODE_MX ? 512 * (2 + 2 * NS) : 0;
    static constexpr int OFF_BAR = OFF_SF + SF_BYTES;
    // at least 116 KB so that one CTA (which allocates all 512 TMEM columns) fits per SM
    static constexpr int SMEM = (OFF_BAR + 512 + 1024) > 116 * 1024 ? (OFF_BAR + 512 + 1024) : 116 * 1024;
    // TMEM columns
    static constexpr uint32_t T_O = 256, T_SFQ = 384, T_SFP = 388, T_SFK = 392, T_SFV = 400;
};

struct Bars {
    uint64_t q_full, q_empty, p_full, o_done;
    uint64_t s_full[2], s_empty[2];
    uint64_t k_full[4], v_full[4], kv_empty[4];
    float tile_scale[4][2];   // E4M3 tile mode: K and V block scale of the tile in each stage
    uint32_t tmem_base;
    int abort;
};

template <int ELT, int D, int MODE>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int kk) {
    using C = Cfg<ELT, D, MODE>;
    if constexpr (C::SW128) {
        const uint32_t off = (uint32_t)(kk * 32);
        return sdesc(base + (off / 128) * (128 * 128) + (off % 128), 16, 1024, SWZ_128B);
    } else {
        return sdesc(base + (uint32_t)kk * 32, 16, 512, SWZ_64B);
    }
}
// P: 128 rows x 128 keys, K-major, row = 128 * ELT bytes (always 128-byte swizzle)
template <int ELT>
__device__ __forceinline__ uint64_t desc_p(uint32_t base, int kk) {
    const uint32_t off = (uint32_t)(kk * 32);
    return sdesc(base + (off / 128) * (128 * 128) + (off % 128), 16, 1024, SWZ_128B);
}
// V as the MN-major B operand of P V: rows are keys, channels contiguous
template <int ELT, int D, int MODE>
__device__ __forceinline__ uint64_t desc_v(uint32_t base, int kk) {
    using C = Cfg<ELT, D, MODE>;
    if constexpr (C::SW128) {
        return sdesc(base + (uint32_t)(kk * C::KPER * 128), 128 * 128, 1024, SWZ_128B);
    } else {
        return sdesc(base + (uint32_t)(kk * C::KPER * 64), 128 * 64, 512, SWZ_64B);
    }
}
__device__ __forceinline__ uint64_t desc_sf(uint32_t base) { return sdesc(base, 0, 128, SWZ_NONE); }

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
}

template <int ELT, int D, int MODE>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const FwdParams p) {
    using C = Cfg<ELT, D, MODE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* B = reinterpret_cast<Bars*>(sm + C::OFF_BAR);
    volatile int* abort = &B->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long lim = p.wait_limit;

    if (threadIdx.x == 0) {
        mbar_init(&B->q_full, 1);
        mbar_init(&B->q_empty, 1);
        mbar_init(&B->p_full, 128);
        mbar_init(&B->o_done, 1);
        for (int i = 0; i < 2; i++) {
            mbar_init(&B->s_full[i], 1);
            mbar_init(&B->s_empty[i], 128);
        }
        for (int i = 0; i < C::NS; i++) {
            mbar_init(&B->k_full[i], 1);
            mbar_init(&B->v_full[i], 1);
            mbar_init(&B->kv_empty[i], 1);
        }
        B->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmq);
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    if constexpr (MODE == MODE_MX) {
        if (warp == 2) {   // P's block scales: all 2^0 (biased 127)
            reinterpret_cast<uint4*>(sm + C::OFF_SF + 512)[lane] = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            fence_proxy_async_smem();
        }
    }
    if (warp == 1) {
        tmem_alloc(&B->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B->tmem_base;
    const int n_items = p.hdr->n_items;

    const uint32_t sQ = smem_u32(sm + C::OFF_Q);
    const uint32_t sP = smem_u32(sm + C::OFF_P);
    const uint32_t sKV = smem_u32(sm + C::OFF_KV);
    const uint32_t sSF = smem_u32(sm + C::OFF_SF);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued[4] = {-1, -1, -1, -1};   // parity of the last load per stage
            int q_issued = -1;
            uint32_t g = 0;
            int qi = 0;
            for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x, qi++) {
                const WorkItem w = p.items[it];
                const DocEntry d = p.docs[w.doc];
                if (!mbar_wait(&B->q_empty, (qi & 1) ^ 1, abort, lim)) break;
                const uint32_t qbytes = C::TILE + (MODE == MODE_MX ? 512 : 0);
                mbar_arrive_expect_tx(&B->q_full, qbytes);
                q_issued = qi & 1;
                for (int a = 0; a < C::ATOMS; a++)
                    tma_load_3d(sm + C::OFF_Q + a * 16384, &tmq, &B->q_full, a * C::BOX_ELEMS, w.head,
                                d.start + 128 * w.qtile);
                if constexpr (MODE == MODE_MX)
                    bulk_load(sm + C::OFF_SF, p.mq + ((long long)w.head * p.ntcap + d.toff + w.qtile) * 512, 512,
                              &B->q_full);
                for (int j = 0; j < w.ntiles; j++, g++) {
                    const int st = g % C::NS;
                    if (!mbar_wait(&B->kv_empty[st], ((g / C::NS) & 1) ^ 1, abort, lim)) break;
                    const int k0 = d.start + 128 * j;
                    uint8_t* kt = sm + C::OFF_KV + st * 2 * C::TILE;
                    uint8_t* vt = kt + C::TILE;
                    issued[st] = (g / C::NS) & 1;
                    if constexpr (MODE == MODE_E4M3_TILE) {
                        // read by the softmax warps after they observe k_full's phase
                        B->tile_scale[st][0] = p.sk[w.head * p.capk + d.boff_k + (128 * j) / p.bk];
                        B->tile_scale[st][1] = p.sv[w.head * p.capv + d.boff_v + (128 * j) / p.bv];
                    }
                    mbar_arrive_expect_tx(&B->k_full[st], qbytes);
                    for (int a = 0; a < C::ATOMS; a++)
                        tma_load_3d(kt + a * 16384, &tmk, &B->k_full[st], a * C::BOX_ELEMS, w.head, k0);
                    if constexpr (MODE == MODE_MX)
                        bulk_load(sm + C::OFF_SF + 1024 + st * 512,
                                  p.mk + ((long long)w.head * p.ntcap + d.toff + j) * 512, 512, &B->k_full[st]);
                    mbar_arrive_expect_tx(&B->v_full[st], qbytes);
                    for (int a = 0; a < C::ATOMS; a++)
                        tma_load_3d(vt + a * 16384, &tmv, &B->v_full[st], a * C::BOX_ELEMS, w.head, k0);
                    if constexpr (MODE == MODE_MX)
                        bulk_load(sm + C::OFF_SF + 1024 + C::NS * 512 + st * 512,
                                  p.mv + ((long long)w.head * p.ntcap + d.toff + j) * 512, 512, &B->v_full[st]);
                }
            }
            if (*abort) {   // let in-flight copies land before shared memory is released
                if (q_issued >= 0) wait_drain(&B->q_full, (uint32_t)q_issued, lim);
                for (int s = 0; s < C::NS; s++)
                    if (issued[s] >= 0) {
                        wait_drain(&B->k_full[s], (uint32_t)issued[s], lim);
                        wait_drain(&B->v_full[s], (uint32_t)issued[s], lim);
                    }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t id_s, id_pv;
            if constexpr (ELT == 2) {
                id_s = idesc(1, 1, false, false, 128, 128);
                id_pv = idesc(1, 1, false, true, 128, D);
            } else {
                id_s = idesc(0, 0, false, false, 128, 128);
                id_pv = idesc(0, 0, false, true, 128, D);
            }
            if constexpr (MODE == MODE_MX) tc_cp_sf(tmem + C::T_SFP, desc_sf(sSF + 512));
            uint32_t g = 0, pvc = 0;
            int qi = 0;
            auto issue_pv = [&](uint32_t gx, bool first) -> bool {
                const int st = gx % C::NS;
                if (!mbar_wait(&B->p_full, pvc & 1, abort, lim)) return false;
                pvc++;
                if (!mbar_wait(&B->v_full[st], (gx / C::NS) & 1, abort, lim)) return false;
                tc_fence_after();
                const uint32_t vbase = sKV + st * 2 * C::TILE + C::TILE;
                if constexpr (MODE == MODE_MX) {
                    const uint32_t sfv = tmem + C::T_SFV + (gx & 1) * 4;
                    tc_cp_sf(sfv, desc_sf(sSF + 1024 + C::NS * 512 + st * 512));
#pragma unroll
                    for (int kk = 0; kk < C::KSTEPS_PV; kk++)
                        mma_mxf8(tmem + C::T_O, desc_p<ELT>(sP, kk), desc_v<ELT, D, MODE>(vbase, kk),
                                 idesc_mx(0, 0, false, true, 128, D, kk, kk), tmem + C::T_SFP, sfv,
                                 (first && kk == 0) ? 0u : 1u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < C::KSTEPS_PV; kk++) {
                        if constexpr (ELT == 2)
                            mma_f16(tmem + C::T_O, desc_p<ELT>(sP, kk), desc_v<ELT, D, MODE>(vbase, kk), id_pv,
                                    (first && kk == 0) ? 0u : 1u);
                        else
                            mma_f8(tmem + C::T_O, desc_p<ELT>(sP, kk), desc_v<ELT, D, MODE>(vbase, kk), id_pv,
                                   (first && kk == 0) ? 0u : 1u);
                    }
                }
                tc_commit(&B->o_done);
                tc_commit(&B->kv_empty[st]);
                return true;
            };
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, qi++) {
                const WorkItem w = p.items[it];
                if (!mbar_wait(&B->q_full, qi & 1, abort, lim)) break;
                tc_fence_after();
                if constexpr (MODE == MODE_MX) tc_cp_sf(tmem + C::T_SFQ, desc_sf(sSF));
                const int nt = w.ntiles;
                for (int j = 0; j < nt && ok; j++) {
                    const uint32_t gj = g + j;
                    const int st = gj % C::NS, b = gj & 1;
                    if (!mbar_wait(&B->k_full[st], (gj / C::NS) & 1, abort, lim)) { ok = false; break; }
                    if (!mbar_wait(&B->s_empty[b], ((gj >> 1) & 1) ^ 1, abort, lim)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t kbase = sKV + st * 2 * C::TILE;
                    const uint32_t dS = tmem + b * 128;
                    if constexpr (MODE == MODE_MX) {
                        const uint32_t sfk = tmem + C::T_SFK + (gj & 1) * 4;
                        tc_cp_sf(sfk, desc_sf(sSF + 1024 + st * 512));
#pragma unroll
                        for (int kk = 0; kk < C::KSTEPS_S; kk++)
                            mma_mxf8(dS, desc_kmajor<ELT, D, MODE>(sQ, kk), desc_kmajor<ELT, D, MODE>(kbase, kk),
                                     idesc_mx(0, 0, false, false, 128, 128, kk, kk), tmem + C::T_SFQ, sfk,
                                     kk ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < C::KSTEPS_S; kk++) {
                            if constexpr (ELT == 2)
                                mma_f16(dS, desc_kmajor<ELT, D, MODE>(sQ, kk), desc_kmajor<ELT, D, MODE>(kbase, kk),
                                        id_s, kk ? 1u : 0u);
                            else
                                mma_f8(dS, desc_kmajor<ELT, D, MODE>(sQ, kk), desc_kmajor<ELT, D, MODE>(kbase, kk),
                                       id_s, kk ? 1u : 0u);
                        }
                    }
                    tc_commit(&B->s_full[b]);
                    if (j == nt - 1) tc_commit(&B->q_empty);
                    if (j > 0 && !issue_pv(gj - 1, j == 1)) ok = false;
                }
                if (ok && !issue_pv(g + nt - 1, nt == 1)) ok = false;
                g += nt;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;                       // query row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t g = 0, pvw = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const WorkItem w = p.items[it];
            const DocEntry d = p.docs[w.doc];
            const int h = w.head, L = d.len, nt = w.ntiles;
            const int rloc = 128 * w.qtile + r;                  // row position in the document
            const int rcl = rloc < L ? rloc : L - 1;
            float qs = 1.0f, ref = 1.0f;
            if constexpr (MODE == MODE_E4M3_TILE) qs = p.sq[h * p.capq + d.boff_q + (128 * w.qtile) / p.bq];
            if constexpr (MODE == MODE_E4M3_COL) qs = p.sq[h * p.capq + d.boff_q + rcl / p.bq];
            if constexpr (MODE == MODE_E4M3_TILE || MODE == MODE_E4M3_COL)
                ref = p.exact ? p.vref[(long long)h * p.T + d.start + rcl] : p.vref[(long long)h * p.nd + w.doc];
            float m = -INFINITY, l = 0.0f;
            for (int j = 0; j < nt; j++) {
                const uint32_t gj = g + j;
                const int b = gj & 1;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&B->s_full[b], (gj >> 1) & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float s[128];
                {
                    uint32_t u0[32], u1[32], u2[32], u3[32];
                    const uint32_t ta = tmem + lane_off + b * 128;
                    tmem_ld32(ta, u0);
                    tmem_ld32(ta + 32, u1);
                    tmem_ld32(ta + 64, u2);
                    tmem_ld32(ta + 96, u3);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        s[i] = __uint_as_float(u0[i]);
                        s[32 + i] = __uint_as_float(u1[i]);
                        s[64 + i] = __uint_as_float(u2[i]);
                        s[96 + i] = __uint_as_float(u3[i]);
                    }
                }
                tc_fence_before();
                mbar_arrive(&B->s_empty[b]);
                const int k0 = 128 * j;                           // first key position of the tile
                // score multiplier
                float c = p.C;
                float rj = 1.0f;
                if constexpr (MODE == MODE_E4M3_TILE) {
                    const int st = gj % C::NS;
                    // acquire the producer's stores: its arrive on k_full[st] released them, and
                    // the stage cannot be refilled before this tile's P is handed over
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&B->k_full[st], (gj / C::NS) & 1, abort, lim))) {
                        ok = false;
                        break;
                    }
                    const float ks = B->tile_scale[st][0];
                    const float sv = B->tile_scale[st][1];
                    c = qs * ks * p.C;
                    rj = (sv > 0.0f && ref > 0.0f) ? __fdiv_rn(sv, ref) : 1.0f;
                }
                if constexpr (MODE == MODE_E4M3_COL) {
                    const float qc = qs * p.C;
#pragma unroll 8
                    for (int t = 0; t < 128; t++) {
                        const int kl = (k0 + t) < L ? k0 + t : L - 1;
                        s[t] = s[t] * (p.sk[h * p.capk + d.boff_k + kl / p.bk] * qc);
                    }
                    c = 1.0f;
                }
                const bool diag = p.causal && j == w.qtile;
                const bool tail = !p.causal && (k0 + 128 > L);
                if (diag || tail) {
                    const int lim_k = diag ? (rloc - k0) : (L - 1 - k0);   // last visible key offset
#pragma unroll
                    for (int t = 0; t < 128; t++)
                        if (t > lim_k) s[t] = -INFINITY;
                }
                // a zero block scale would turn masked -inf into NaN: the smallest normal
                // multiplier keeps -inf and leaves finite scores at about zero instead
                c = fmaxf(c, 1.17549435e-38f);
                // row max: eight chains of 3-input max
                float mx8[8];
#pragma unroll
                for (int k8 = 0; k8 < 8; k8++) {
                    float a = s[16 * k8];
#pragma unroll
                    for (int i = 1; i < 15; i += 2) a = fmax3(a, s[16 * k8 + i], s[16 * k8 + i + 1]);
                    mx8[k8] = fmaxf(a, s[16 * k8 + 15]);
                }
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]));
                const float mt = mx * c;
                const float m_new = fmaxf(m, mt);
                const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
                const float alpha = (m == -INFINITY) ? 0.0f : ex2(m - m_new);
                float bias = 8.0f - m_use;
                if constexpr (MODE == MODE_E4M3_TILE) bias += __log2f(rj);
                uint32_t pk[ELT == 1 ? 32 : 64];
                float rowsum;
                if constexpr (MODE != MODE_E4M3_COL) {
                    // p = 2^(s * c + bias): pairs through the packed FMA, exp2 on MUFU,
                    // row sum in four packed accumulators
                    const float2 c2 = make_float2(c, c), b2 = make_float2(bias, bias);
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f)};
#pragma unroll
                    for (int t = 0; t < 128; t += 8) {
                        float e[8];
#pragma unroll
                        for (int u = 0; u < 8; u += 2) {
                            const float2 x = __ffma2_rn(make_float2(s[t + u], s[t + u + 1]), c2, b2);
                            e[u] = ex2(x.x);
                            e[u + 1] = ex2(x.y);
                            acc[u >> 1] = __fadd2_rn(acc[u >> 1], make_float2(e[u], e[u + 1]));
                        }
                        if constexpr (ELT == 1) {
                            pk[t / 4] = pack_e4m3x4(e[0], e[1], e[2], e[3]);
                            pk[t / 4 + 1] = pack_e4m3x4(e[4], e[5], e[6], e[7]);
                        } else {
#pragma unroll
                            for (int u = 0; u < 4; u++) pk[t / 2 + u] = pack_bf16x2(e[2 * u], e[2 * u + 1]);
                        }
                    }
                    const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
                    const float2 a = __fadd2_rn(a01, a23);
                    rowsum = a.x + a.y;
                } else {
                    float rs8[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int t = 0; t < 128; t += 4) {
                        float e[4];
#pragma unroll
                        for (int u = 0; u < 4; u++) {
                            e[u] = ex2(fmaf(s[t + u], c, bias));
                            rs8[(t + u) & 7] += e[u];
                            const int kl = (k0 + t + u) < L ? k0 + t + u : L - 1;
                            const float sv = p.sv[h * p.capv + d.boff_v + kl / p.bv];
                            const float rt = (sv > 0.0f && ref > 0.0f) ? __fdiv_rn(sv, ref) : 1.0f;
                            e[u] = e[u] * rt;
                        }
                        pk[t / 4] = pack_e4m3x4(e[0], e[1], e[2], e[3]);
                    }
                    rowsum = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
                }
                float ltile = rowsum;
                if constexpr (MODE == MODE_E4M3_TILE) ltile = rowsum * __fdiv_rn(1.0f, rj);
                l = alpha * l + ltile;
                m = m_new;
                if (j > 0) {
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&B->o_done, pvw & 1, abort, lim))) {
                        ok = false;
                        break;
                    }
                    pvw++;
                    tc_fence_after();
                    if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
                        uint32_t u[32];
#pragma unroll
                        for (int cc = 0; cc < D / 32; cc++) {
                            const uint32_t ta = tmem + lane_off + C::T_O + cc * 32;
                            tmem_ld32(ta, u);
                            tmem_wait_ld();
                            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const float2 v2 = __fmul2_rn(make_float2(__uint_as_float(u[i]), __uint_as_float(u[i + 1])), a2);
                                u[i] = __float_as_uint(v2.x);
                                u[i + 1] = __float_as_uint(v2.y);
                            }
                            tmem_st32(ta, u);
                        }
                        tmem_wait_st();
                    }
                }
                // P row -> shared memory, 128-byte swizzled K-major rows
#pragma unroll
                for (int ch = 0; ch < 8 * ELT; ch++) {
                    const int atom = ch >> 3, cc = ch & 7;
                    uint8_t* dst = sm + C::OFF_P + atom * 16384 + r * 128 + ((cc ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&B->p_full);
            }
            if (!ok) break;
            // epilogue: O / l -> bf16, lse
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&B->o_done, pvw & 1, abort, lim))) {
                ok = false;
                break;
            }
            pvw++;
            tc_fence_after();
            const float fin = (l > 0.0f) ? __fdiv_rn(ref, l) : 0.0f;
            const bool store = rloc < L;
            uint16_t* orow = p.o + ((long long)(d.start + rcl) * p.H + h) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; cc++) {
                uint32_t u[32];
                tmem_ld32(tmem + lane_off + C::T_O + cc * 32, u);
                tmem_wait_ld();
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; i++)
                    packed[i] = pack_bf16x2(__uint_as_float(u[2 * i]) * fin, __uint_as_float(u[2 * i + 1]) * fin);
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                }
            }
            if (store)
                p.lse[(long long)h * p.T + d.start + rloc] =
                    (l > 0.0f) ? 0.69314718055994531f * (m + __log2f(l) - 8.0f) : -INFINITY;
            tc_fence_before();
            g += nt;
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
// host side
// [T][H][D] tensor, box = (box_elems channels, 1 head, 128 tokens)
static bool make_map(CUtensorMap* m, const void* base, int elt, int T, int H, int D, int box_elems, bool sw128) {
    return make_tensor_map_3d(m, base, elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              D, H, T, (uint64_t)D * elt, (uint64_t)H * D * elt, box_elems, 128,
                              sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int ELT, int D, int MODE>
static cudaError_t launch_t(const void* q, const void* k, const void* v, const FwdParams& p, int grid,
                            cudaStream_t st) {
    using C = Cfg<ELT, D, MODE>;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, ELT, p.T, p.H, D, C::BOX_ELEMS, C::SW128) ||
        !make_map(&mk, k, ELT, p.T, p.H, D, C::BOX_ELEMS, C::SW128) ||
        !make_map(&mv, v, ELT, p.T, p.H, D, C::BOX_ELEMS, C::SW128))
        return cudaErrorInvalidValue;
    auto kern = attn_fwd_kernel<ELT, D, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, 192, C::SMEM, st>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

// mode: 0 bf16, 1 E4M3 tile scales, 2 E4M3 per-column scales, 3 MX
cudaError_t launch_attn(int mode, int D, const void* q, const void* k, const void* v, const FwdParams& p, int grid,
                        cudaStream_t st) {
    if (mode == MODE_BF16) return D == 128 ? launch_t<2, 128, MODE_BF16>(q, k, v, p, grid, st)
                                           : launch_t<2, 64, MODE_BF16>(q, k, v, p, grid, st);
    if (mode == MODE_E4M3_TILE) return D == 128 ? launch_t<1, 128, MODE_E4M3_TILE>(q, k, v, p, grid, st)
                                                : launch_t<1, 64, MODE_E4M3_TILE>(q, k, v, p, grid, st);
    if (mode == MODE_E4M3_COL) return D == 128 ? launch_t<1, 128, MODE_E4M3_COL>(q, k, v, p, grid, st)
                                               : launch_t<1, 64, MODE_E4M3_COL>(q, k, v, p, grid, st);
    if (mode == MODE_MX && D == 128) return launch_t<1, 128, MODE_MX>(q, k, v, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace pa
