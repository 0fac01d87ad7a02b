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
// Two kernels. attn_pair_kernel (below) runs the FP8 modes at d = 128 (E4M3
// token-block scales and MXFP8) with two query tiles per CTA. attn_fwd_kernel
// runs the BF16 comparator path and the E4M3 modes at d = 64, one query tile
// (128 rows of one document and head) per work item, one CTA per SM,
// persistent over the work items. Its warp roles:
//   warp 0      TMA producer: Q tile once per item, K and V tiles of each key
//               block into an NS-stage ring
//   warp 1      TMEM owner and MMA issuer: S_j = Q K_j^T into one of two TMEM
//               S buffers, then O += P_{j-1} V_{j-1}
//   warps 2-9   softmax: two warps per 32-row TMEM lane quarter, each holding
//               half of the S columns of its rows; S from TMEM, scale, mask,
//               running max (combined through shared memory) and sum, exp2, P to
//               shared memory (E4M3 or BF16), O rescale in TMEM, final
//               normalisation and stores
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256 + d).
// Every mbarrier wait is bounded; on a timeout the CTA raises a flag, stops,
// drains its TMA copies, frees TMEM and returns, and the host reads
// ATTN_ERR_DEVICE_TIMEOUT from the status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "pdl.cuh"

namespace pa {

struct Bars {
    uint64_t q_full, q_empty;
    uint64_t p_full[2];       // P of tile g handed over -> p_full[g % PBUF]
    uint64_t pv_done[2];      // P V of tile g completes -> pv_done[g % PBUF]
    uint64_t s_full[2], s_empty[2];
    uint64_t k_full[8], v_full[8], k_empty[8], v_empty[8];   // K slots free after S, V slots after P V
    // E4M3 tile mode: score multiplier, log2(r), 1/r of key tile g in slot g % 8. The
    // producer runs at most NS + 1 tiles ahead of the softmax reading them (it needs
    // the K slot that S of tile g - NS frees), so eight slots never collide.
    float tile_scale[8][4];
    uint64_t sc_full[8];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    // the two warps sharing a row quarter exchange row maxima and row sums through
    // shared memory; ep_max[half][quarter] = 1 + last tile whose maxima are written,
    // ep_sum[half][quarter] = 1 + last item whose row sums are written
    int ep_max[2][4];
    int ep_sum[2][4];
};

template <int ELT, int D, int MODE>
__global__ void __launch_bounds__(Cfg<ELT, D, MODE>::THREADS, 1)
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
        mbar_init(&B->p_full[0], 32 * C::SOFTMAX_WARPS);
        mbar_init(&B->p_full[1], 32 * C::SOFTMAX_WARPS);
        for (int i = 0; i < 8; i++) {
            (&B->ep_max[0][0])[i] = 0;
            (&B->ep_sum[0][0])[i] = 0;
        }
        mbar_init(&B->pv_done[0], 1);
        mbar_init(&B->pv_done[1], 1);
        for (int i = 0; i < 2; i++) {
            mbar_init(&B->s_full[i], 1);
            mbar_init(&B->s_empty[i], 32 * C::SOFTMAX_WARPS);
        }
        for (int i = 0; i < 8; i++) mbar_init(&B->sc_full[i], 1);
        mbar_init(&B->drain, 1);
        for (int i = 0; i < C::NS; i++) {
            mbar_init(&B->k_full[i], 1);
            mbar_init(&B->v_full[i], 1);
            mbar_init(&B->k_empty[i], 1);
            mbar_init(&B->v_empty[i], 1);
        }
        B->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmq);
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
    pdl_wait();   // the work list, the scales and the codes of the kernels before this one
    const int n_items = p.hdr->n_items;

    const uint32_t sQ = smem_u32(sm + C::OFF_Q);
    const uint32_t sP = smem_u32(sm + C::OFF_P);
    const uint32_t sKV = smem_u32(sm + C::OFF_KV);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp runs the loop: lane 0 issues the copies; in E4M3 tile mode the
        // lanes first load the block scales of the next 32 key tiles in parallel (one
        // tile each), so no tile waits on a dependent global load.
        constexpr unsigned FULL = 0xFFFFFFFFu;
        int issued[8] = {-1, -1, -1, -1, -1, -1, -1, -1};   // parity of the last load per stage
        int q_issued = -1;
        uint32_t g = 0;
        int qi = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, qi++) {
            const WorkItem w = p.items[it];
            const DocEntry d = p.docs[w.doc];
            float qs = 1.0f, ref = 1.0f;
            if constexpr (MODE == MODE_E4M3_TILE) {
                qs = p.sq[w.head * p.capq + d.boff_q + (128 * w.qtile) / p.bq];
                ref = p.vref[(long long)w.head * p.nd + w.doc];
            }
            if (!__all_sync(FULL, mbar_wait(&B->q_empty, (qi & 1) ^ 1, abort, lim))) break;
            const uint32_t qbytes = C::TILE;
            q_issued = qi & 1;
            if (lane == 0) {
                mbar_arrive_expect_tx(&B->q_full, qbytes);
                for (int a = 0; a < C::ATOMS; a++)
                    tma_load_3d(sm + C::OFF_Q + a * 16384, &tmq, &B->q_full, a * C::BOX_ELEMS, w.head,
                                d.start + 128 * w.qtile);
            }
            float t_c = 0.0f, t_lr = 0.0f, t_ir = 1.0f;   // this lane's tile of the current group of 32
            const float inv_ref = ref > 0.0f ? __fdiv_rn(1.0f, ref) : 0.0f;
            for (int j = 0; j < w.ntiles; j++, g++) {
                if constexpr (MODE == MODE_E4M3_TILE) {
                    if ((j & 31) == 0 && j + lane < w.ntiles) {
                        // the tile's folded score multiplier and V ratio r = s_v x (1 / ref)
                        const int jt = j + lane;
                        const float ks = p.sk[w.head * p.capk + d.boff_k + (128 * jt) / p.bk];
                        const float sv = p.sv[w.head * p.capv + d.boff_v + (128 * jt) / p.bv];
                        const float rj = (sv > 0.0f && ref > 0.0f) ? __fmul_rn(sv, inv_ref) : 1.0f;
                        t_c = qs * ks * p.C;
                        t_lr = __log2f(rj);
                        t_ir = __fdiv_rn(1.0f, rj);
                    }
                }
                const int st = g % C::NS;
                if (!__all_sync(FULL, mbar_wait(&B->k_empty[st], ((g / C::NS) & 1) ^ 1, abort, lim))) {
                    ok = false;
                    break;
                }
                issued[st] = (g / C::NS) & 1;
                if constexpr (MODE == MODE_E4M3_TILE) {
                    const float c = __shfl_sync(FULL, t_c, j & 31);
                    const float lr = __shfl_sync(FULL, t_lr, j & 31);
                    const float ir = __shfl_sync(FULL, t_ir, j & 31);
                    if (lane == 0) {   // released to the softmax warps through sc_full
                        B->tile_scale[g & 7][0] = c;
                        B->tile_scale[g & 7][1] = lr;
                        B->tile_scale[g & 7][2] = ir;
                        mbar_arrive(&B->sc_full[g & 7]);
                    }
                }
                if (lane == 0) {
                    const int k0 = d.start + 128 * j;
                    uint8_t* kt = sm + C::OFF_KV + st * 2 * C::TILE;
                    mbar_arrive_expect_tx(&B->k_full[st], qbytes);
                    for (int a = 0; a < C::ATOMS; a++)
                        tma_load_3d(kt + a * 16384, &tmk, &B->k_full[st], a * C::BOX_ELEMS, w.head, k0);
                }
                if (!__all_sync(FULL, mbar_wait(&B->v_empty[st], ((g / C::NS) & 1) ^ 1, abort, lim))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    uint8_t* vt = sm + C::OFF_KV + st * 2 * C::TILE + C::TILE;
                    mbar_arrive_expect_tx(&B->v_full[st], qbytes);
                    for (int a = 0; a < C::ATOMS; a++)
                        tma_load_3d(vt + a * 16384, &tmv, &B->v_full[st], a * C::BOX_ELEMS, w.head,
                                    d.start + 128 * j);
                }
            }
        }
        if (*abort && lane == 0) {   // let in-flight copies land before shared memory is released
            if (q_issued >= 0) wait_drain(&B->q_full, (uint32_t)q_issued, kDrainLimit);
            for (int s2 = 0; s2 < C::NS; s2++)
                if (issued[s2] >= 0) {
                    wait_drain(&B->k_full[s2], (uint32_t)issued[s2], kDrainLimit);
                    wait_drain(&B->v_full[s2], (uint32_t)issued[s2], kDrainLimit);
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // One thread. Descriptors are built once: every operand tile sits at a fixed
        // shared-memory address, so a K step only adds a constant to the start-address
        // field (addresses stay below 256 KB, the field never carries).
        if (lane == 0) {
            constexpr uint32_t id_s = ELT == 2 ? idesc(1, 1, false, false, 128, 128) : idesc(0, 0, false, false, 128, 128);
            constexpr uint32_t id_pv = ELT == 2 ? idesc(1, 1, false, true, 128, D) : idesc(0, 0, false, true, 128, D);
            const uint64_t dq = desc_kmajor<ELT, D, MODE>(sQ, 0);
            const uint64_t dk0 = desc_kmajor<ELT, D, MODE>(sKV, 0);
            const uint64_t dv0 = desc_v<ELT, D, MODE>(sKV + C::TILE, 0);
            const uint64_t dp0 = desc_p<ELT>(sP, 0);
            constexpr uint64_t STAGE16 = (uint64_t)(2 * C::TILE) >> 4;   // descriptor step between stages
            constexpr uint64_t PBUF16 = (uint64_t)C::PBYTES >> 4;
            // Fixed order, S up to two key tiles ahead of P V (two S buffers), across
            // item boundaries:  S_0 S_1 | P V_0 S_2 | P V_1 S_3 | ...  as  S_{j+2} needs
            // only that the softmax has loaded S_j, which it does before P_j is ready.
            // Each step parks on the one barrier it needs (mbarrier.try_wait). Polling
            // several barriers instead costs a shared-memory instruction per test, and
            // those queue behind the softmax warps' MUFU and shared-memory traffic.
            int itS = blockIdx.x, jS = 0, qiS = 0;     // S stream cursor
            int itP = blockIdx.x, jP = 0;              // P V stream cursor
            uint32_t gS = 0, gP = 0;                   // global tile counters
            WorkItem wS = blockIdx.x < n_items ? p.items[blockIdx.x] : WorkItem{};
            WorkItem wP = wS;
            auto issue_s = [&]() -> bool {
                const int st = gS % C::NS, b = gS & 1;
                if (jS == 0 && !mbar_wait(&B->q_full, qiS & 1, abort, lim)) return false;
                if (!mbar_wait(&B->k_full[st], (gS / C::NS) & 1, abort, lim)) return false;
                if (!mbar_wait(&B->s_empty[b], ((gS >> 1) & 1) ^ 1, abort, lim)) return false;
                tc_fence_after();
                const uint64_t dk = dk0 + st * STAGE16;
                const uint32_t dS = tmem + b * 128;
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS_S; kk++) {
                    if constexpr (ELT == 2)
                        mma_f16(dS, dq + koff<ELT, D, MODE>(kk), dk + koff<ELT, D, MODE>(kk), id_s, kk ? 1u : 0u);
                    else
                        mma_f8(dS, dq + koff<ELT, D, MODE>(kk), dk + koff<ELT, D, MODE>(kk), id_s, kk ? 1u : 0u);
                }
                tc_commit(&B->s_full[b]);
                tc_commit(&B->k_empty[st]);
                gS++;
                if (++jS == wS.ntiles) {           // last S of the item: Q may be replaced
                    tc_commit(&B->q_empty);
                    jS = 0;
                    qiS++;
                    itS += gridDim.x;
                    if (itS < n_items) wS = p.items[itS];
                }
                return true;
            };
            auto issue_pv = [&]() -> bool {
                const int st = gP % C::NS;
                if (!mbar_wait(&B->v_full[st], (gP / C::NS) & 1, abort, lim)) return false;
                if (!mbar_wait(&B->p_full[gP % C::PBUF], (gP / C::PBUF) & 1, abort, lim)) return false;
                tc_fence_after();
                const uint64_t dv = dv0 + st * STAGE16;
                const uint64_t dp = dp0 + (gP % C::PBUF) * PBUF16;
                const bool first = jP == 0;
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS_PV; kk++) {
                    if constexpr (ELT == 2)
                        mma_f16(tmem + C::T_O, dp + poff(kk), dv + voff<ELT, D, MODE>(kk), id_pv,
                                (first && kk == 0) ? 0u : 1u);
                    else
                        mma_f8(tmem + C::T_O, dp + poff(kk), dv + voff<ELT, D, MODE>(kk), id_pv,
                               (first && kk == 0) ? 0u : 1u);
                }
                tc_commit(&B->pv_done[gP % C::PBUF]);
                tc_commit(&B->v_empty[st]);
                gP++;
                if (++jP == wP.ntiles) {
                    jP = 0;
                    itP += gridDim.x;
                    if (itP < n_items) wP = p.items[itP];
                }
                return true;
            };
            bool ok = true;
            while (ok && itP < n_items) {
                while (ok && itS < n_items && gS < gP + 2) ok = issue_s();
                if (ok) ok = issue_pv();
            }
            // every MMA this thread issued has completed before TMEM is released
            tc_commit(&B->drain);
            wait_drain(&B->drain, 0, kDrainLimit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        // warps 2..9: the two warps with the same TMEM lane quarter share the
        // 32 rows of that quarter, each taking one half of the S columns
        // (and of the O columns); they combine row maxima through shared memory
        // and a 64-thread named barrier.
        const int hh = (warp - 2) >> 2;                           // column half
        const int quarter = warp & 3;                             // TMEM lane quarter
        const int r = quarter * 32 + lane;                        // query row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        int items_done = 0;
        // publish this warp's values (already stored) as epoch `e` and wait, bounded and
        // abort-aware, until the partner warp has published the same epoch
        auto pair_exchange = [&](int* mine, int* theirs, int e) -> bool {
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                *reinterpret_cast<volatile int*>(mine) = e;
            }
            bool got = true;
            if (lane == 0) {
                const volatile int* t = reinterpret_cast<const volatile int*>(theirs);
                if (*t < e) {
                    const long long t0 = clock64();
                    while (*t < e) {
                        if (*abort || clock64() - t0 > lim) {
                            *abort = 1;
                            got = false;
                            break;
                        }
                    }
                }
                __threadfence_block();
            }
            return __shfl_sync(0xFFFFFFFFu, (int)got, 0) != 0;
        };
        float* xch = reinterpret_cast<float*>(sm + C::OFF_XCH);   // [parity][half][row]
        float* xl = reinterpret_cast<float*>(sm + C::OFF_XL);     // [half][row]
        uint32_t g = 0;
        bool ok = true;
        // P V of global tile gx has completed (its barrier cannot move further before
        // this thread hands over a later P)
        auto wait_pv = [&](uint32_t gx) -> bool {
            return __all_sync(0xFFFFFFFFu, mbar_wait(&B->pv_done[gx % C::PBUF], (gx / C::PBUF) & 1, abort, lim));
        };
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const WorkItem w = p.items[it];
            const DocEntry d = p.docs[w.doc];
            const int h = w.head, L = d.len, nt = w.ntiles;
            const int rloc = 128 * w.qtile + r;                   // row position in the document
            const int rcl = rloc < L ? rloc : L - 1;
            float qs = 1.0f, ref = 1.0f;
            if constexpr (MODE == MODE_E4M3_COL) {
                qs = p.sq[h * p.capq + d.boff_q + rcl / p.bq];
                ref = p.exact ? p.vref[(long long)h * p.T + d.start + rcl] : p.vref[(long long)h * p.nd + w.doc];
            }
            if constexpr (MODE == MODE_E4M3_TILE) ref = p.vref[(long long)h * p.nd + w.doc];
            const float inv_ref = ref > 0.0f ? __fdiv_rn(1.0f, ref) : 0.0f;   // V ratios: s_v x (1 / ref)
            float m = -INFINITY, l = 0.0f;
            for (int j = 0; j < nt; j++) {
                const uint32_t gj = g + j;
                const int b = gj & 1;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&B->s_full[b], (gj >> 1) & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float s[C::HC];
                {
                    uint32_t u0[32], u1[32];
                    const uint32_t ta = tmem + lane_off + b * 128 + hh * C::HC;
                    tmem_ld32(ta, u0);
                    tmem_ld32(ta + 32, u1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        s[i] = __uint_as_float(u0[i]);
                        s[32 + i] = __uint_as_float(u1[i]);
                    }
                }
                const int k0 = 128 * j + hh * C::HC;                // first key position of this thread's columns
                float c = p.C, lr = 0.0f, invr = 1.0f;
                if constexpr (MODE == MODE_E4M3_TILE) {
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&B->sc_full[gj & 7], (gj >> 3) & 1, abort, lim))) {
                        ok = false;
                        break;
                    }
                    c = B->tile_scale[gj & 7][0];
                    lr = B->tile_scale[gj & 7][1];
                    invr = B->tile_scale[gj & 7][2];
                }
                tc_fence_before();
                mbar_arrive(&B->s_empty[b]);
                if constexpr (MODE == MODE_E4M3_COL) {
                    const float qc = qs * p.C;
#pragma unroll 8
                    for (int t = 0; t < C::HC; t++) {
                        const int kl = (k0 + t) < L ? k0 + t : L - 1;
                        s[t] = s[t] * (p.sk[h * p.capk + d.boff_k + kl / p.bk] * qc);
                    }
                    c = 1.0f;
                }
                const bool diag = p.causal && j == w.qtile;
                const bool tail = !p.causal && (128 * j + 128 > L);
                if (diag || tail) {
                    const int lim_k = diag ? (rloc - k0) : (L - 1 - k0);   // last visible column offset
#pragma unroll
                    for (int t = 0; t < C::HC; t++)
                        if (t > lim_k) s[t] = -INFINITY;
                }
                // a zero block scale would turn masked -inf into NaN: the smallest normal
                // multiplier keeps -inf and leaves finite scores at about zero instead
                c = fmaxf(c, 1.17549435e-38f);
                // row max of this half: four chains of 3-input max, then the partner's half
                float mx4[4];
#pragma unroll
                for (int k4 = 0; k4 < 4; k4++) {
                    float a = s[16 * k4];
#pragma unroll
                    for (int i2 = 1; i2 < 15; i2 += 2) a = fmax3(a, s[16 * k4 + i2], s[16 * k4 + i2 + 1]);
                    mx4[k4] = fmaxf(a, s[16 * k4 + 15]);
                }
                const float pmax = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
                xch[((gj & 1) * 2 + hh) * 128 + r] = pmax;
                if (!pair_exchange(&B->ep_max[hh][quarter], &B->ep_max[hh ^ 1][quarter], (int)gj + 1)) {
                    ok = false;
                    break;
                }
                const float mx = fmaxf(pmax, xch[((gj & 1) * 2 + (hh ^ 1)) * 128 + r]);
                // running max (log2 units) and the rescale factor of the old state
                const float mt = mx * c;
                const float m_new = fmaxf(m, mt);
                const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
                const float alpha = (m == -INFINITY) ? 0.0f : (m_new > m ? ex2(m - m_new) : 1.0f);
                const float bias = 8.0f - m_use + lr;
                uint32_t pk[ELT == 1 ? 16 : 32];
                float rowsum;
                if constexpr (MODE != MODE_E4M3_COL) {
                    // p = 2^(s * c + bias): pairs through the packed FMA, exp2 on MUFU,
                    // row sum in four packed accumulators
                    const float2 c2 = make_float2(c, c), b2 = make_float2(bias, bias);
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f)};
#pragma unroll
                    for (int t = 0; t < C::HC; t += 8) {
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
                    float rs4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int t = 0; t < C::HC; t += 4) {
                        float e[4];
#pragma unroll
                        for (int u = 0; u < 4; u++) {
                            e[u] = ex2(fmaf(s[t + u], c, bias));
                            rs4[u] += e[u];
                            const int kl = (k0 + t + u) < L ? k0 + t + u : L - 1;
                            const float sv = p.sv[h * p.capv + d.boff_v + kl / p.bv];
                            const float rt = (sv > 0.0f && ref > 0.0f) ? __fmul_rn(sv, inv_ref) : 1.0f;
                            e[u] = e[u] * rt;
                        }
                        pk[t / 4] = pack_e4m3x4(e[0], e[1], e[2], e[3]);
                    }
                    rowsum = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
                }
#ifdef PA_PDUMP
                if constexpr (ELT == 1) {
                    if (p.pdump && rloc < L && k0 + C::HC <= p.pdump_stride) {
                        uint4* dst =
                            reinterpret_cast<uint4*>(p.pdump + ((long long)h * p.T + d.start + rloc) * p.pdump_stride + k0);
#pragma unroll
                        for (int i = 0; i < C::HC / 16; i++)
                            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
#endif
                l = alpha * l + rowsum * invr;
                m = m_new;
                // O rescale (when any row of the warp moved its max): after P V of the
                // previous tile, before this tile's P is handed over
                if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
                    if (!wait_pv(gj - 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    {
                        uint32_t u[32];
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                        for (int cc = 0; cc < C::HD / 32; cc++) {
                            const uint32_t ta = tmem + lane_off + C::T_O + hh * C::HD + cc * 32;
                            tmem_ld32(ta, u);
                            tmem_wait_ld();
#pragma unroll
                            for (int i2 = 0; i2 < 32; i2 += 2) {
                                const float2 v2 =
                                    __fmul2_rn(make_float2(__uint_as_float(u[i2]), __uint_as_float(u[i2 + 1])), a2);
                                u[i2] = __float_as_uint(v2.x);
                                u[i2 + 1] = __float_as_uint(v2.y);
                            }
                            tmem_st32(ta, u);
                        }
                        tmem_wait_st();
                    }
                }
                // the P buffer of this tile was last read by P V of tile gj - PBUF
                if (gj >= (uint32_t)C::PBUF && !wait_pv(gj - C::PBUF)) {
                    ok = false;
                    break;
                }
                // this half of the P row -> shared memory (128-byte swizzled K-major rows)
                uint8_t* pbuf = sm + C::OFF_P + (gj % C::PBUF) * C::PBYTES;
#pragma unroll
                for (int ch = 0; ch < 4 * ELT; ch++) {
                    const int gch = hh * 4 * ELT + ch;                 // 16-byte chunk within the row
                    const int atom = gch >> 3, cc = gch & 7;
                    uint8_t* dst = pbuf + atom * 16384 + r * 128 + ((cc ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&B->p_full[gj % C::PBUF]);
            }
            if (!ok) break;
            // epilogue: row sum of both halves, O / l -> bf16 (this half of the columns), lse
            xl[hh * 128 + r] = l;
            if (!pair_exchange(&B->ep_sum[hh][quarter], &B->ep_sum[hh ^ 1][quarter], ++items_done)) {
                ok = false;
                break;
            }
            const float lt = l + xl[(hh ^ 1) * 128 + r];
            if (!wait_pv(g + nt - 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float fin = (lt > 0.0f) ? __fdiv_rn(ref, lt) : 0.0f;
            const bool store = rloc < L;
            uint16_t* orow = p.o + ((long long)(d.start + rcl) * p.H + h) * D + hh * C::HD;
            const float2 f2 = make_float2(fin, fin);
#pragma unroll
            for (int cc = 0; cc < C::HD / 32; cc++) {
                uint32_t u[32];
                tmem_ld32(tmem + lane_off + C::T_O + hh * C::HD + cc * 32, u);
                tmem_wait_ld();
                uint32_t packed[16];
#pragma unroll
                for (int i2 = 0; i2 < 16; i2++) {
                    const float2 v2 =
                        __fmul2_rn(make_float2(__uint_as_float(u[2 * i2]), __uint_as_float(u[2 * i2 + 1])), f2);
                    packed[i2] = pack_bf16x2(v2.x, v2.y);
                }
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                    for (int i2 = 0; i2 < 4; i2++)
                        dst[i2] = make_uint4(packed[4 * i2], packed[4 * i2 + 1], packed[4 * i2 + 2], packed[4 * i2 + 3]);
                }
            }
            if (store && hh == 0)
                p.lse[(long long)h * p.T + d.start + rloc] =
                    (lt > 0.0f) ? 0.69314718055994531f * (m + __log2f(lt) - 8.0f) : -INFINITY;
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
// Two query tiles per CTA (E4M3 and MXFP8 codes, d = 128).
//
// The same loop as attn_fwd_kernel, with the CTA's work item widened to the
// query tiles 2p and 2p + 1 of a (document, head): both share every K and V
// tile, and their two dependency chains (S -> softmax -> P -> P V) interleave
// on the tensor pipe and on the SM sub-partitions, so one tile's softmax runs
// while the other tile's MMAs execute.
//   warp 0      producer: both Q tiles once per item, K and V tiles (and MX
//               scale tiles) into a 4-stage ring (3 for MX)
//   warp 1      TMEM owner; its lane 0 issues the MMAs of query tile 0 and
//   warp 10     lane 0 those of query tile 1, each in a fixed order with S one
//               key tile ahead: S_q(j+1) = Q_q K_{j+1}^T, then P_q V_j
//   warps 2-5   softmax of query tile 0, warps 6-9 of query tile 1: one thread
//               per row, all 128 columns
// TMEM: one S buffer [0,128) that the two query tiles take in turns (S_0(j), then
// S_1(j) once group 0 has loaded S_0(j), then S_0(j+1) once group 1 has loaded
// S_1(j)), O0 [256,384), O1 [384,512); P, the A operand of P V, in TMEM: E4M3 two
// buffers per query tile at 128 + 32 (2q + b), so the softmax of tile j writes P
// while P V of tile j - 1 may still read the other one; MX one buffer per query
// tile at 176 + 32q, beside the block-scaled MMAs' scale factors at [128,176).
// A K slot is released by S_1j's completion (S_1j is issued after S_0j completed), a V
// slot after both P V of tile j.
template <int MODE>
struct PairCfgT {
    // MX: Q K^T block-scaled (scale factors of Q and K in TMEM); MXPV: P V block-scaled
    // as well (V's 32-token exponents). MODE_MX_EXACT keeps the first and folds V's
    // per-token exponent into P instead (as the E4M3 per-column mode folds V scales).
    static constexpr bool MX = MODE == MODE_MX || MODE == MODE_MX_EXACT;
    static constexpr bool MXPV = MODE == MODE_MX;
    // NV: Q K^T on NVFP4 operands (E2M1, E4M3 scales per 16 channels in TMEM, fp32
    // 128-token block scales folded into the score multiplier as in the E4M3 tile
    // mode), P V on E4M3 as there
    static constexpr bool NV = MODE == MODE_NVFP4;
    static constexpr bool SFT = MX || NV;             // scale factors in TMEM
    // P lives in TMEM, the A operand of P V read from there: two buffers per query
    // tile, one when TMEM also holds scale factors
    static constexpr int PBUF = SFT ? 1 : 2;
    static constexpr int TILE = 128 * 128;           // bytes of a 128 x 128 E4M3 tile (one ring slot)
    static constexpr int QKB = NV ? TILE / 2 : TILE;  // bytes of a Q or K tile (NVFP4: 64-byte rows)
    static constexpr int QD = NV ? 64 : 128;          // Q / K row bytes (descriptor geometry)
    static constexpr int NS = MX ? 3 : 4;             // K/V ring depth
    static constexpr int OFF_Q = 0;                   // Q0, Q1
    static constexpr int OFF_KV = 2 * TILE;           // stage s: K at +2s TILE, V at +(2s + 1) TILE
    // MX scale tiles, 512 bytes each: Q0, Q1, P (all 2^0), K per stage, V per stage
    static constexpr int OFF_SF = OFF_KV + NS * 2 * TILE;
    // NV: 1024 bytes (two K = 64 steps) each: Q0, Q1, K per stage
    static constexpr int SF_BYTES = MX ? 512 * (3 + 2 * NS) : NV ? 1024 * (2 + NS) : 0;
    // per-key scales of key tile g, staged per stage: float [NS][2][128]. E4M3 per-column
    // mode (blocks shorter than a tile, causal-exact): K and V scales; MX exact mode: V's
    // 2^X only (K's exponents are inside the block-scaled MMA)
    static constexpr bool COLS = MODE == MODE_E4M3_COL || MODE == MODE_MX_EXACT;
    static constexpr bool KCOLS = MODE == MODE_E4M3_COL;
    static constexpr int OFF_KSC = OFF_SF + SF_BYTES;
    static constexpr int KSC_BYTES = COLS ? NS * 1024 : 0;
    // Q tiles of the next item (double buffer: item k uses buffer k % 2, so the next
    // item's Q lands while this one runs), and their scale tiles (NVFP4): E4M3 per-column
    // scales 4.5% faster, NVFP4 1.4%, E4M3 tile scales 0.5%. Not in the MX layouts, where
    // the second buffer gained nothing
    static constexpr bool QDB = !MX;
    static constexpr int OFF_Q2 = OFF_KSC + KSC_BYTES;
    static constexpr int OFF_SFQ2 = OFF_Q2 + (QDB ? 2 * TILE : 0);
    static constexpr int SFQ2_BYTES = (QDB && NV) ? 2048 : 0;
    static constexpr int OFF_BAR = OFF_SFQ2 + SFQ2_BYTES;
    static constexpr int SMEM = OFF_BAR + 1024 + 1024;
    static constexpr int THREADS = 352;
    // Q buffer of the k-th item and the parity of its use; shared-memory offsets of Q
    // buffer b and of its scale tiles
    static constexpr int q_buf(int k) { return QDB ? (k & 1) : 0; }
    static constexpr uint32_t q_par(int k) { return QDB ? ((k >> 1) & 1) : (k & 1); }
    static constexpr int q_off(int b) { return b ? OFF_Q2 : OFF_Q; }
    static constexpr int sfq_off(int b) { return b ? OFF_SFQ2 : OFF_SF; }
    static constexpr uint32_t T_O = 256;              // O_q at T_O + 128 q
    // S_q at 128 q; MX: one S buffer at 0 shared by both query tiles, and the scale
    // factors in the columns that frees: Q_q at T_SFQ + 4q, P at T_SFP + 4q, K and V
    // of key tile g at T_SFK / T_SFV + 8q + 4 (g % 2)
    static constexpr bool SHARED_S = true;
    static constexpr uint32_t T_S1 = SHARED_S ? 0 : 128;
    static constexpr uint32_t T_SFQ = 128, T_SFP = 136, T_SFK = 144, T_SFV = 160;
    static constexpr uint32_t T_P = SFT ? 176 : 128;  // P of query tile q, buffer b at T_P + 32 (PBUF q + b)
    // NV: Q_q's scale factors at T_NQ + 8q, K of key tile g (issuer q) at T_NK + 16q + 8 (g % 2)
    static constexpr uint32_t T_NQ = 128, T_NK = 144;
};
static_assert(PairCfgT<MODE_E4M3_TILE>::SMEM <= 227 * 1024, "pair kernel shared memory exceeds the per-CTA limit");
static_assert(PairCfgT<MODE_MX>::SMEM <= 227 * 1024, "pair kernel shared memory exceeds the per-CTA limit");
static_assert(PairCfgT<MODE_MX_EXACT>::SMEM <= 227 * 1024, "pair kernel shared memory exceeds the per-CTA limit");
static_assert(PairCfgT<MODE_NVFP4>::SMEM <= 227 * 1024, "pair kernel shared memory exceeds the per-CTA limit");
static_assert(PairCfgT<MODE_E4M3_TILE>::NS <= 8 && PairCfgT<MODE_MX>::NS <= 8, "K/V ring deeper than its barriers");

struct PairBars {
    uint64_t q_full, q_empty;           // Q buffer 0 (buffer 1: q_full1, q_empty1 below)
    uint64_t s_full[2], s_empty[2];     // per query tile
    uint64_t p_full[2][2], pv_done[2][2];   // per query tile and P buffer
    uint64_t k_full[8], v_full[8], k_empty[8], v_empty[8];
    uint64_t drain[2];
    uint64_t ksc_full[8], ksc_empty[8];   // per-column mode: key scales of a stage written / read
    uint64_t q_full1, q_empty1;           // Q buffer 1 (the double buffer of the non-MX modes)
    uint64_t ring_full[8], ring_empty[8];   // just-in-time schedule: item k in slot k % 8
    int ring[8];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(PairBars) <= 1024, "pair kernel barrier block exceeds its reserved space");

template <int MODE, int EXPM, bool DYN>
__global__ void __launch_bounds__(PairCfgT<MODE>::THREADS, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const FwdParams p) {
    using PC = PairCfgT<MODE>;
    using C = Cfg<1, 128, MODE>;   // descriptor helpers of the 128-byte-row E4M3 tiles
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PairBars* B = reinterpret_cast<PairBars*>(sm + PC::OFF_BAR);
    volatile int* abort = &B->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long lim = p.wait_limit;
    constexpr unsigned FULL = 0xFFFFFFFFu;

    if (threadIdx.x == 0) {
        mbar_init(&B->q_full, 1);
        mbar_init(&B->q_empty, 1);   // S_1 of the item's last key tile (after S_0's)
        mbar_init(&B->q_full1, 1);
        mbar_init(&B->q_empty1, 1);
        for (int q = 0; q < 2; q++) {
            mbar_init(&B->s_full[q], 1);
            mbar_init(&B->s_empty[q], 128);
            for (int b = 0; b < 2; b++) {
                mbar_init(&B->p_full[q][b], 128);
                mbar_init(&B->pv_done[q][b], 1);
            }
        }
        for (int i = 0; i < PC::NS; i++) {
            mbar_init(&B->k_full[i], 1);
            mbar_init(&B->v_full[i], 1);
            mbar_init(&B->k_empty[i], 1);   // S_1 of the key tile (after S_0's)
            mbar_init(&B->v_empty[i], 2);
        }
        mbar_init(&B->drain[0], 1);
        mbar_init(&B->drain[1], 1);
        for (int i = 0; i < PC::NS; i++) {
            mbar_init(&B->ksc_full[i], 32);    // every producer lane, after its stores
            mbar_init(&B->ksc_empty[i], 256);  // every softmax thread of both query tiles
        }
        for (int i = 0; i < 8; i++) {
            mbar_init(&B->ring_full[i], 1);    // the producer, after writing the slot
            mbar_init(&B->ring_empty[i], 12);  // 8 softmax warps + 2 issuers x (S, P cursor)
        }
        B->abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmq);
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    if constexpr (PC::MX) {
        if (warp == 2) {   // P's block scales: all 2^0 (biased 127)
            reinterpret_cast<uint4*>(sm + PC::OFF_SF + 1024)[lane] =
                make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
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
    pdl_wait();   // the work list, the scales and the codes of the kernels before this one
    const int n_items = p.hdr->n_items;
    const uint32_t sQ = smem_u32(sm + PC::OFF_Q);
    const uint32_t sKV = smem_u32(sm + PC::OFF_KV);
    const uint32_t sSF = smem_u32(sm + PC::OFF_SF);
    (void)sSF;
    // Work item of this CTA in round k. Causal: the CTAs take rounds of gridDim.x
    // items of the longest-first list in alternating directions, so that long and
    // short items even out across CTAs. Otherwise (equal items, head-major) the same
    // direction every round, which keeps each round's heads on the same SMs and
    // their K/V in the nearer L2 partition. Every role walks the same sequence.
    const bool snake = p.causal != 0;
    auto item_of = [&](int k) -> int {
        const int g = (int)gridDim.x, b = (int)blockIdx.x;
        return k * g + ((snake && (k & 1)) ? g - 1 - b : b);
    };
    // Just-in-time schedule (DYN): the producer takes item k by ticket when it starts
    // the item's loads (CTA b's first item is b; then an atomic counter the work-list
    // pass set to the grid size) and hands it through slot k % 8 of a ring to the
    // issuers' S and P cursors and the softmax warps, in the same order. An index past
    // the list ends every role.
    constexpr int kEnd = 0x7FFFFFFF;
    auto seq_producer = [&](int k) -> int {   // warp 0, all lanes
        if constexpr (!DYN) return item_of(k);
        int it = kEnd;
        if (lane == 0) {
            const int sl = k & 7;
            if (mbar_wait(&B->ring_empty[sl], ((k >> 3) & 1) ^ 1, abort, lim)) {
                const int t = k == 0 ? (int)blockIdx.x : atomicAdd(&p.hdr->ticket, 1);
                it = t < n_items ? t : kEnd;
                B->ring[sl] = it;
                mbar_arrive(&B->ring_full[sl]);   // releases the slot's write to the readers
            }
        }
        return __shfl_sync(FULL, it, 0);
    };
    auto seq_issuer = [&](int k, int cursors) -> int {   // one issuing thread; cursors freeing the slot
        if constexpr (!DYN) return item_of(k);
        const int sl = k & 7;
        if (!mbar_wait(&B->ring_full[sl], (k >> 3) & 1, abort, lim)) return kEnd;
        const int it = *reinterpret_cast<volatile int*>(&B->ring[sl]);
        for (int c = 0; c < cursors; c++) mbar_arrive(&B->ring_empty[sl]);
        return it;
    };
    auto seq_softmax = [&](int k) -> int {   // a softmax warp, all lanes
        if constexpr (!DYN) return item_of(k);
        const int sl = k & 7;
        if (!__all_sync(FULL, mbar_wait(&B->ring_full[sl], (k >> 3) & 1, abort, lim))) return kEnd;
        const int it = *reinterpret_cast<volatile int*>(&B->ring[sl]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->ring_empty[sl]);
        return it;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int issued[8] = {-1, -1, -1, -1, -1, -1, -1, -1};   // parity of the last load per stage
        int q_issued[2] = {-1, -1};   // parity of the last load per Q buffer
        uint32_t g = 0;
        int qi = 0;
        bool ok = true;
        for (int k = 0, it = seq_producer(0); it < n_items && ok; it = seq_producer(++k), qi++) {
            const WorkItem w = p.items[it];
            const DocEntry d = p.docs[w.doc];
            const int qb = PC::q_buf(qi);   // Q buffer of this item
            if (!__all_sync(FULL, mbar_wait((qb ? &B->q_empty1 : &B->q_empty), PC::q_par(qi) ^ 1, abort, lim))) break;
            q_issued[qb] = PC::q_par(qi);
            // MX: the second query tile's scale tile exists only inside the document
            const bool q1_in = 2 * w.qtile + 1 < (d.len + 127) / 128;
            const uint32_t qbytes =
                2 * PC::QKB + (PC::MX ? (q1_in ? 1024 : 512) : PC::NV ? (q1_in ? 2048 : 1024) : 0);
            if (lane == 0) {
                uint64_t* qf = (qb ? &B->q_full1 : &B->q_full);
                uint8_t* qdst = sm + PC::q_off(qb);
                uint8_t* sfdst = sm + PC::sfq_off(qb);
                mbar_arrive_expect_tx(qf, qbytes);
                tma_load_3d(qdst, &tmq, qf, 0, w.head, d.start + 256 * w.qtile);
                tma_load_3d(qdst + PC::TILE, &tmq, qf, 0, w.head, d.start + 256 * w.qtile + 128);
                if constexpr (PC::MX) {
                    const long long t0 = (long long)w.head * p.ntcap + d.toff + 2 * w.qtile;
                    bulk_load(sfdst, p.mq + t0 * 512, 512, qf);
                    if (q1_in) bulk_load(sfdst + 512, p.mq + (t0 + 1) * 512, 512, qf);
                } else if constexpr (PC::NV) {
                    const long long t0 = (long long)w.head * p.ntcap + d.toff + 2 * w.qtile;
                    bulk_load(sfdst, p.mq + t0 * 1024, 1024, qf);
                    if (q1_in) bulk_load(sfdst + 1024, p.mq + (t0 + 1) * 1024, 1024, qf);
                }
            }
            for (int j = 0; j < w.ntiles; j++, g++) {
                const int st = g % PC::NS;
                if (!__all_sync(FULL, mbar_wait(&B->k_empty[st], ((g / PC::NS) & 1) ^ 1, abort, lim))) {
                    ok = false;
                    break;
                }
                issued[st] = (g / PC::NS) & 1;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&B->k_full[st], PC::QKB + (PC::MX ? 512 : PC::NV ? 1024 : 0));
                    tma_load_3d(sm + PC::OFF_KV + st * 2 * PC::TILE, &tmk, &B->k_full[st], 0, w.head,
                                d.start + 128 * j);
                    if constexpr (PC::MX)
                        bulk_load(sm + PC::OFF_SF + 1536 + st * 512,
                                  p.mk + ((long long)w.head * p.ntcap + d.toff + j) * 512, 512, &B->k_full[st]);
                    if constexpr (PC::NV)
                        bulk_load(sm + PC::OFF_SF + 2048 + st * 1024,
                                  p.mk + ((long long)w.head * p.ntcap + d.toff + j) * 1024, 1024, &B->k_full[st]);
                }
                if (!__all_sync(FULL, mbar_wait(&B->v_empty[st], ((g / PC::NS) & 1) ^ 1, abort, lim))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&B->v_full[st], PC::TILE + (PC::MXPV ? 512 : 0));
                    tma_load_3d(sm + PC::OFF_KV + st * 2 * PC::TILE + PC::TILE, &tmv, &B->v_full[st], 0, w.head,
                                d.start + 128 * j);
                    if constexpr (PC::MXPV)
                        bulk_load(sm + PC::OFF_SF + 1536 + PC::NS * 512 + st * 512,
                                  p.mv + ((long long)w.head * p.ntcap + d.toff + j) * 512, 512, &B->v_full[st]);
                }
                if constexpr (PC::COLS) {
                    // each key's K and V scale of this tile (keys past the document end
                    // repeat the last one; they are masked anyway), four keys per lane
                    if (!__all_sync(FULL, mbar_wait(&B->ksc_empty[st], ((g / PC::NS) & 1) ^ 1, abort, lim))) {
                        ok = false;
                        break;
                    }
                    float* ksc = reinterpret_cast<float*>(sm + PC::OFF_KSC + st * 1024);
                    float kv[4], vv[4];
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        const int kl = min(128 * j + 4 * lane + u, d.len - 1);
                        if constexpr (PC::KCOLS) {
                            kv[u] = p.sk[w.head * p.capk + d.boff_k + kl / p.bk];
                            vv[u] = p.sv[w.head * p.capv + d.boff_v + kl / p.bv];
                        } else {   // V exponent byte -> 2^X (0 for X = -127: the token's V codes are 0)
                            const uint32_t b = p.mv[w.head * p.capv + d.boff_v + kl];
                            kv[u] = 1.0f;
                            vv[u] = b ? __uint_as_float(b << 23) : 0.0f;
                        }
                    }
                    *reinterpret_cast<float4*>(ksc + 4 * lane) = make_float4(kv[0], kv[1], kv[2], kv[3]);
                    *reinterpret_cast<float4*>(ksc + 128 + 4 * lane) = make_float4(vv[0], vv[1], vv[2], vv[3]);
                    mbar_arrive(&B->ksc_full[st]);
                }
            }
        }
        if (*abort && lane == 0) {   // let in-flight copies land before shared memory is released
            for (int b = 0; b < 2; b++)
                if (q_issued[b] >= 0) wait_drain(b ? &B->q_full1 : &B->q_full, (uint32_t)q_issued[b], kDrainLimit);
            for (int s2 = 0; s2 < PC::NS; s2++)
                if (issued[s2] >= 0) {
                    wait_drain(&B->k_full[s2], (uint32_t)issued[s2], kDrainLimit);
                    wait_drain(&B->v_full[s2], (uint32_t)issued[s2], kDrainLimit);
                }
        }
        __syncwarp();
    } else if (warp == 1 || warp == PC::THREADS / 32 - 1) {
        // ------------------------------------------------------------ MMA issuers
        // One thread per query tile (warp 1: tile 0, the last warp: tile 1), so that
        // neither chain S_q -> softmax_q -> P_q V waits behind the other's. Each issues
        // in a fixed order with S one key tile ahead of P V (across item boundaries):
        //   S_0 | S_1 P V_0 | S_2 P V_1 | ...
        // and parks on the one barrier it needs (mbarrier.try_wait). A V slot is released
        // once both issuers have committed their P V that read it, a K slot (and the Q
        // tiles) by issuer 1's S commit.
        if (lane == 0) {
            const int q = warp == 1 ? 0 : 1;
            constexpr uint32_t id_s = idesc(0, 0, false, false, 128, 128);
            constexpr uint32_t id_pv = idesc(0, 0, false, true, 128, 128);
            constexpr uint64_t TILE16 = (uint64_t)PC::TILE >> 4;
            constexpr uint64_t STAGE16 = (uint64_t)(2 * PC::TILE) >> 4;
            // this query tile's Q in each of the two Q buffers (item k uses buffer k % 2)
            const uint64_t dqb[2] = {desc_kmajor<1, PC::QD, MODE>(smem_u32(sm + PC::q_off(0)), 0) + q * TILE16,
                                     desc_kmajor<1, PC::QD, MODE>(smem_u32(sm + PC::q_off(1)), 0) + q * TILE16};
            const uint32_t sfqb[2] = {smem_u32(sm + PC::sfq_off(0)), smem_u32(sm + PC::sfq_off(1))};
            const uint64_t dk0 = desc_kmajor<1, PC::QD, MODE>(sKV, 0);
            const uint64_t dv0 = desc_v<1, 128, MODE>(sKV + PC::TILE, 0);
            const uint32_t tS = tmem + q * PC::T_S1, tO = tmem + PC::T_O + q * 128;
            // MX: this query tile's Q, P, K and V scale-factor columns
            const uint32_t sfq = tmem + PC::T_SFQ + 4 * q, sfp = tmem + PC::T_SFP + 4 * q;
            const uint32_t sfk0 = tmem + PC::T_SFK + 8 * q, sfv0 = tmem + PC::T_SFV + 8 * q;
            if constexpr (PC::MXPV) tc_cp_sf(sfp, desc_sf(sSF + 1024));
            int kS = 0, itS = seq_issuer(0, 2), jS = 0, qiS = 0;   // the P cursor starts on the same item
            uint32_t gS = 0;
            WorkItem wS = itS < n_items ? p.items[itS] : WorkItem{};
            int kP = 0, itP = itS, jP = 0;
            uint32_t gP = 0;
            WorkItem wP = wS;
            // NVFP4: the K scale factors of key tile gS are already in their TMEM slot,
            // copied right after the previous S (off the hand-over between S buffers) when
            // the tile had landed by then
            bool sf_pre = false;
            auto copy_k_sf = [&](uint32_t gx) {
                const int sx = gx % PC::NS;
                if constexpr (PC::NV) {
                    const uint32_t nk = tmem + PC::T_NK + 16 * q + 8 * (gx & 1);
                    tc_cp_sf(nk, desc_sf(sSF + 2048 + sx * 1024));
                    tc_cp_sf(nk + 4, desc_sf(sSF + 2048 + sx * 1024 + 512));
                } else if constexpr (PC::MX) {
                    tc_cp_sf(sfk0 + 4 * (gx & 1), desc_sf(sSF + 1536 + sx * 512));
                }
            };
            auto issue_s = [&]() -> bool {   // S_q of key tile gS
                const int st = gS % PC::NS;
                if (jS == 0 && !mbar_wait(PC::q_buf(qiS) ? &B->q_full1 : &B->q_full, PC::q_par(qiS), abort, lim)) return false;
                if (!mbar_wait(&B->k_full[st], (gS / PC::NS) & 1, abort, lim)) return false;
                const uint64_t dq = dqb[PC::q_buf(qiS)];
                const uint32_t sfqs = sfqb[PC::q_buf(qiS)];   // this item's Q scale tiles (MX, NVFP4)
                (void)sfqs;
                if constexpr (PC::SHARED_S) {
                    // one S buffer, written S_0(g), S_1(g), S_0(g + 1), ...: S_0(g) once the
                    // other group has loaded S_1(g - 1), S_1(g) once this one has loaded S_0(g)
                    if (q == 0 ? (gS >= 1 && !mbar_wait(&B->s_empty[1], (gS - 1) & 1, abort, lim))
                               : !mbar_wait(&B->s_empty[0], gS & 1, abort, lim))
                        return false;
                } else {
                    if (!mbar_wait(&B->s_empty[q], (gS & 1) ^ 1, abort, lim)) return false;
                }
                tc_fence_after();
                const uint64_t dk = dk0 + st * STAGE16;
                if constexpr (PC::NV) {
                    // E4M3 scale factors of Q_q (once per item) and of this key tile, two
                    // 512-byte tiles each (K = 64 per MMA), then two block-scaled MMAs
                    const uint32_t nq = tmem + PC::T_NQ + 8 * q, nk = tmem + PC::T_NK + 16 * q + 8 * (gS & 1);
                    if (jS == 0) {
                        tc_cp_sf(nq, desc_sf(sfqs + 1024 * q));
                        tc_cp_sf(nq + 4, desc_sf(sfqs + 1024 * q + 512));
                    }
                    if (!sf_pre) copy_k_sf(gS);
#pragma unroll
                    for (int kk = 0; kk < 2; kk++)
                        mma_nvf4(tS, dq + koff<1, 64, MODE>(kk), dk + koff<1, 64, MODE>(kk), idesc_nvf4(128, 128),
                                 nq + 4 * kk, nk + 4 * kk, kk ? 1u : 0u);
                } else if constexpr (PC::MX) {
                    if (jS == 0) tc_cp_sf(sfq, desc_sf(sfqs + 512 * q));
                    const uint32_t sfk = sfk0 + 4 * (gS & 1);
                    copy_k_sf(gS);
#pragma unroll
                    for (int kk = 0; kk < C::KSTEPS_S; kk++)
                        mma_mxf8(tS, dq + koff<1, 128, MODE>(kk), dk + koff<1, 128, MODE>(kk),
                                 idesc_mx(0, 0, false, false, 128, 128, kk, kk), sfq, sfk, kk ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < C::KSTEPS_S; kk++)
                        mma_f8(tS, dq + koff<1, 128, MODE>(kk), dk + koff<1, 128, MODE>(kk), id_s, kk ? 1u : 0u);
                }
                tc_commit(&B->s_full[q]);
                // S_1(g) is issued only once S_0(g) has completed (its row loads freed the
                // buffer), so S_1's completion alone releases the K slot and, after an
                // item's last key tile, the Q tiles
                if (q == 1) tc_commit(&B->k_empty[st]);
                gS++;
                if (++jS == wS.ntiles) {   // last S of the item: Q may be replaced
                    if (q == 1) tc_commit(PC::q_buf(qiS) ? &B->q_empty1 : &B->q_empty);
                    jS = 0;
                    qiS++;
                    itS = seq_issuer(++kS, 1);
                    if (itS < n_items) wS = p.items[itS];
                }
                sf_pre = false;
                if constexpr (PC::NV) {
                    // the next key tile's scale factors into the other slot, if it has landed
                    // (tcgen05 copies and MMAs of this thread run in issue order, so the S two
                    // tiles back has read that slot before the copy writes it). NVFP4 only: its
                    // two copies per tile moved off the hand-over save 2.5% there, while moving
                    // the MX layouts' single copy measured 1.2% slower
                    if (itS < n_items && mbar_test(&B->k_full[gS % PC::NS], (gS / PC::NS) & 1)) {
                        tc_fence_after();
                        copy_k_sf(gS);
                        sf_pre = true;
                    }
                }
                return true;
            };
            auto issue_pv = [&]() -> bool {   // P_q V of key tile gP
                const int st = gP % PC::NS;
                if (!mbar_wait(&B->v_full[st], (gP / PC::NS) & 1, abort, lim)) return false;
                if (!mbar_wait(&B->p_full[q][gP & 1], (gP >> 1) & 1, abort, lim)) return false;
                tc_fence_after();
                const uint64_t dv = dv0 + st * STAGE16;
                const uint32_t tp = tmem + PC::T_P + 32 * (PC::PBUF * q + gP % PC::PBUF);   // P, A from TMEM
                const bool first = jP == 0;
                if constexpr (PC::MXPV) {
                    const uint32_t sfv = sfv0 + 4 * (gP & 1);
                    tc_cp_sf(sfv, desc_sf(sSF + 1536 + PC::NS * 512 + st * 512));
#pragma unroll
                    for (int kk = 0; kk < C::KSTEPS_PV; kk++)
                        mma_mxf8_ta(tO, tp + 8 * kk, dv + voff<1, 128, MODE>(kk),
                                    idesc_mx(0, 0, false, true, 128, 128, kk, kk), sfp, sfv, (first && kk == 0) ? 0u : 1u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < C::KSTEPS_PV; kk++)
                        mma_f8_ta(tO, tp + 8 * kk, dv + voff<1, 128, MODE>(kk), id_pv, (first && kk == 0) ? 0u : 1u);
                }
                tc_commit(&B->pv_done[q][gP & 1]);
                tc_commit(&B->v_empty[st]);
                gP++;
                if (++jP == wP.ntiles) {
                    jP = 0;
                    itP = seq_issuer(++kP, 1);
                    if (itP < n_items) wP = p.items[itP];
                }
                return true;
            };
            bool ok = itS >= n_items || issue_s();
            while (ok && itP < n_items) {
                if (itS < n_items && !issue_s()) break;
                ok = issue_pv();
            }
            // every MMA this thread issued has completed before TMEM is released
            tc_commit(&B->drain[q]);
            wait_drain(&B->drain[q], 0, kDrainLimit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int q = (warp - 2) >> 2;                            // query tile of this group
        const int quarter = warp & 3;                             // TMEM lane quarter
        const int r = quarter * 32 + lane;                        // row within the query tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + q * PC::T_S1;
        const uint32_t tO = tmem + lane_off + PC::T_O + q * 128;
        uint32_t g = 0;
        bool ok = true;
        auto wait_pv = [&](uint32_t gx) -> bool {
            return __all_sync(FULL, mbar_wait(&B->pv_done[q][gx & 1], (gx >> 1) & 1, abort, lim));
        };
        for (int k = 0, it = seq_softmax(0); it < n_items && ok; it = seq_softmax(++k)) {
            const WorkItem w = p.items[it];
            const DocEntry d = p.docs[w.doc];
            const int h = w.head, L = d.len, nt = w.ntiles;
            const int ntd = (L + 127) / 128;
            const int qt = 2 * w.qtile + q;                       // query tile within the document
            const int qtc = qt < ntd ? qt : ntd - 1;
            const int rloc = 128 * qt + r;                        // row position in the document
            const int rcl = rloc < L ? rloc : L - 1;
            float qs = 1.0f, ref = 1.0f;   // MX: the scales are inside the MMAs
            if constexpr (MODE == MODE_E4M3_TILE || MODE == MODE_NVFP4) {
                qs = p.sq[h * p.capq + d.boff_q + (128 * qtc) / p.bq];
                ref = p.vref[(long long)h * p.nd + w.doc];
            } else if constexpr (MODE == MODE_E4M3_COL) {
                qs = p.sq[h * p.capq + d.boff_q + rcl / p.bq];
                ref = p.exact ? p.vref[(long long)h * p.T + d.start + rcl] : p.vref[(long long)h * p.nd + w.doc];
            } else if constexpr (MODE == MODE_MX_EXACT) {   // V's reference exponent, as 2^X
                ref = p.exact ? p.vref[(long long)h * p.T + d.start + rcl] : p.vref[(long long)h * p.nd + w.doc];
            }
            const float inv_ref = ref > 0.0f ? __fdiv_rn(1.0f, ref) : 0.0f;   // V ratios: s_v x (1 / ref)
            float m = -INFINITY, l = 0.0f;
            // E4M3 tile mode: the key tiles' multipliers {K scale x C, log2 r, 1 / r}, one
            // tile ahead of use (written by the V-reference pass before this launch)
            const float4* tsc = p.tsc + (long long)h * p.tsc_cap + d.toff;
            float4 tnext = make_float4(0.0f, 0.0f, 1.0f, 0.0f);
            if constexpr (MODE == MODE_E4M3_TILE || MODE == MODE_NVFP4) tnext = tsc[0];
            for (int j = 0; j < nt; j++) {
                const uint32_t gj = g + j;
                float c = p.C, lr = 0.0f, invr = 1.0f;
                if constexpr (MODE == MODE_E4M3_TILE || MODE == MODE_NVFP4) {
                    c = qs * tnext.x;
                    lr = tnext.y;
                    invr = tnext.z;
                    if (j + 1 < nt) tnext = tsc[j + 1];
                }
                if (!__all_sync(FULL, mbar_wait(&B->s_full[q], gj & 1, abort, lim))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float s[128];
                {
                    uint32_t u[128];
                    tmem_ld128(tS, u);   // the whole row in one load
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 128; i++) s[i] = __uint_as_float(u[i]);
                }
                tc_fence_before();
                mbar_arrive(&B->s_empty[q]);
                const int k0 = 128 * j;                              // first key position of the tile
                const float* ksc = reinterpret_cast<const float*>(sm + PC::OFF_KSC + (gj % PC::NS) * 1024);
                if constexpr (PC::COLS) {
                    if (!__all_sync(FULL, mbar_wait(&B->ksc_full[gj % PC::NS], (gj / PC::NS) & 1, abort, lim))) {
                        ok = false;
                        break;
                    }
                    if constexpr (PC::KCOLS) {
                        // each key's K scale here; the row's factor q_scale x C enters with
                        // the exponent's FFMA (and the row maximum) below
#pragma unroll
                        for (int t = 0; t < 128; t += 4) {
                            const float4 k4 = *reinterpret_cast<const float4*>(ksc + t);
                            const float2 a = __fmul2_rn(make_float2(s[t], s[t + 1]), make_float2(k4.x, k4.y));
                            const float2 b = __fmul2_rn(make_float2(s[t + 2], s[t + 3]), make_float2(k4.z, k4.w));
                            s[t] = a.x;
                            s[t + 1] = a.y;
                            s[t + 2] = b.x;
                            s[t + 3] = b.y;
                        }
                    }
                    c = qs * p.C;
                }
                // causal: key tiles past the query tile are fully masked (the pair's
                // first tile visits one key tile more than it needs), the diagonal
                // tile keeps keys <= the row; otherwise keys past the document end
                const bool mask = p.causal ? (j >= qt) : (k0 + 128 > L);
                if (mask) {
                    const int lim_k = p.causal ? (rloc - k0) : (L - 1 - k0);   // last visible column
#pragma unroll
                    for (int t = 0; t < 128; t++)
                        if (t > lim_k) s[t] = -INFINITY;
                }
                c = fmaxf(c, 1.17549435e-38f);   // keeps masked -inf when a block scale is 0
                float mx8[8];
#pragma unroll
                for (int k8 = 0; k8 < 8; k8++) {
                    float a = s[16 * k8];
#pragma unroll
                    for (int i2 = 1; i2 < 15; i2 += 2) a = fmax3(a, s[16 * k8 + i2], s[16 * k8 + i2 + 1]);
                    mx8[k8] = fmaxf(a, s[16 * k8 + 15]);
                }
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]));
                // reference max (log2 units) and the rescale factor of the old state: the
                // reference moves to the running max only when that exceeds it by more than
                // ATTN_RESCALE_THRESHOLD, so that most key tiles leave O as it is; then
                // 2^(s' - m + 8) <= 2^8.75 < 448 keeps every probability code finite
                const float mt = mx * c;
                const float m_cand = fmaxf(m, mt);
                const float m_new = (m == -INFINITY || m_cand > m + ATTN_RESCALE_THRESHOLD) ? m_cand : m;
                const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
                const float alpha = (m == -INFINITY) ? 0.0f : (m_new > m ? ex2(m - m_new) : 1.0f);
                const float bias = 8.0f - m_use + lr;
                uint32_t pk[32];
                float rowsum;
                if constexpr (!PC::COLS && EXPM == ATTN_EXP_HW) {
                    const float2 c2 = make_float2(c, c), b2 = make_float2(bias, bias);
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f)};
#pragma unroll
                    for (int t = 0; t < 128; t += 8) {
                        float e[8];
#pragma unroll
                        for (int u = 0; u < 8; u += 2) {
                            const float2 xx = __ffma2_rn(make_float2(s[t + u], s[t + u + 1]), c2, b2);
                            e[u] = ex2(xx.x);
                            e[u + 1] = ex2(xx.y);
                            acc[u >> 1] = __fadd2_rn(acc[u >> 1], make_float2(e[u], e[u + 1]));
                        }
                        pk[t / 4] = pack_e4m3x4(e[0], e[1], e[2], e[3]);
                        pk[t / 4 + 1] = pack_e4m3x4(e[4], e[5], e[6], e[7]);
                    }
                    const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
                    rowsum = a.x + a.y;
                } else if constexpr (!PC::COLS && EXPM == ATTN_EXP_SCHRAUDOLPH) {
                    // Schraudolph: p = the fp32 value with bits 2^23 (u + 127), u = x - delta.
                    // y = sat((u + 126) / 256) in [0, 1) (-inf and u < -126 give 0), then
                    // n = round(2^22 y) = round(2^14 (u + 126)) lands in the low mantissa bits of
                    // y 2^22 + 1.5 2^23; shifted left by 9 that word is 2^31 + 2^9 n, so adding
                    // 2^31 + 2^23 leaves p's bits 2^9 n + 2^23 (n < 2^22: no carry anywhere)
                    constexpr float kOff = (float)(126.0 - ATTN_SCHRAUDOLPH_DELTA);
                    const float c1 = c * 0.00390625f, b1 = (bias + kOff) * 0.00390625f;
                    const float2 r2 = make_float2(4194304.0f, 4194304.0f), k2 = make_float2(12582912.0f, 12582912.0f);
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f)};
#pragma unroll
                    for (int t = 0; t < 128; t += 8) {
                        float e[8];
#pragma unroll
                        for (int u = 0; u < 8; u += 2) {
                            const float2 yy = make_float2(fma_sat(s[t + u], c1, b1), fma_sat(s[t + u + 1], c1, b1));
                            const float2 tt = __ffma2_rn(yy, r2, k2);
                            e[u] = __uint_as_float((__float_as_uint(tt.x) << 9) + 0x80800000u);
                            e[u + 1] = __uint_as_float((__float_as_uint(tt.y) << 9) + 0x80800000u);
                            acc[u >> 1] = __fadd2_rn(acc[u >> 1], make_float2(e[u], e[u + 1]));
                        }
                        pk[t / 4] = pack_e4m3x4(e[0], e[1], e[2], e[3]);
                        pk[t / 4 + 1] = pack_e4m3x4(e[4], e[5], e[6], e[7]);
                    }
                    const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
                    rowsum = a.x + a.y;
                } else if constexpr (!PC::COLS && EXPM == ATTN_EXP_MITCHELL_P) {
                    // log-domain P: code = round(8 u + 56) in [0, 126]. y = sat((8 u + 56) / 128),
                    // then the code lands in the low byte of y 128 + 1.5 2^23 (x <= 8.75 keeps
                    // 128 y <= 126). Word << 20 = code << 20: the fp32 whose value is 2^-120 times
                    // the code's E4M3 value (normal and subnormal codes alike); the row sum adds
                    // those and takes the 2^120 back once.
                    constexpr float kOff = (float)(0.4375 - ATTN_SCHRAUDOLPH_DELTA / 16.0);
                    const float c1 = c * 0.0625f, b1 = fmaf(bias, 0.0625f, kOff);
                    const float2 r2 = make_float2(128.0f, 128.0f), k2 = make_float2(12582912.0f, 12582912.0f);
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f)};
#pragma unroll
                    for (int t = 0; t < 128; t += 8) {
                        uint32_t w[8];
#pragma unroll
                        for (int u = 0; u < 8; u += 2) {
                            const float2 yy = make_float2(fma_sat(s[t + u], c1, b1), fma_sat(s[t + u + 1], c1, b1));
                            const float2 tt = __ffma2_rn(yy, r2, k2);
                            w[u] = __float_as_uint(tt.x);
                            w[u + 1] = __float_as_uint(tt.y);
                            acc[u >> 1] = __fadd2_rn(acc[u >> 1],
                                                     make_float2(__uint_as_float(w[u] << 20), __uint_as_float(w[u + 1] << 20)));
                        }
                        pk[t / 4] = __byte_perm(__byte_perm(w[0], w[1], 0x0040), __byte_perm(w[2], w[3], 0x0040), 0x5410);
                        pk[t / 4 + 1] = __byte_perm(__byte_perm(w[4], w[5], 0x0040), __byte_perm(w[6], w[7], 0x0040), 0x5410);
                    }
                    const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
                    rowsum = (a.x + a.y) * 1.329227995784916e36f;   // 2^120
                } else {
                    // p = 2^(s' + bias), row sum of the unquantised p, then each key's V
                    // ratio r = s_v x (1 / ref) folded in. A key whose V scale is 0 has
                    // all-zero V codes, so its ratio (0 here) changes no output.
                    const float2 c2 = make_float2(c, c), b2 = make_float2(bias, bias);
                    const float2 ir2 = make_float2(inv_ref, inv_ref);
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f)};
#pragma unroll
                    for (int t = 0; t < 128; t += 8) {
                        const float4 va = *reinterpret_cast<const float4*>(ksc + 128 + t);
                        const float4 vb = *reinterpret_cast<const float4*>(ksc + 128 + t + 4);
                        const float sv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
                        float e[8];
#pragma unroll
                        for (int u = 0; u < 8; u += 2) {
                            const float2 xx = __ffma2_rn(make_float2(s[t + u], s[t + u + 1]), c2, b2);
                            const float2 ee = make_float2(ex2(xx.x), ex2(xx.y));
                            acc[u >> 1] = __fadd2_rn(acc[u >> 1], ee);
                            const float2 pr = __fmul2_rn(ee, __fmul2_rn(make_float2(sv[u], sv[u + 1]), ir2));
                            e[u] = pr.x;
                            e[u + 1] = pr.y;
                        }
                        pk[t / 4] = pack_e4m3x4(e[0], e[1], e[2], e[3]);
                        pk[t / 4 + 1] = pack_e4m3x4(e[4], e[5], e[6], e[7]);
                    }
                    const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
                    rowsum = a.x + a.y;
                    tc_fence_before();
                    mbar_arrive(&B->ksc_empty[gj % PC::NS]);
                }
#ifdef PA_PDUMP
                if (p.pdump && rloc < L && k0 + 128 <= p.pdump_stride) {
                    uint4* dst = reinterpret_cast<uint4*>(p.pdump + ((long long)h * p.T + d.start + rloc) * p.pdump_stride + k0);
#pragma unroll
                    for (int i = 0; i < 8; i++) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
#endif
                l = alpha * l + rowsum * invr;
                m = m_new;
                // P buffer gj & 1 was last read by P V of tile gj - 2. A rescale of O needs
                // P V of tile gj - 1 complete (and with it every earlier one); without a
                // rescale, P V of tile gj may queue right behind it on the tensor pipe.
                const bool rescale = j > 0 && __any_sync(FULL, alpha != 1.0f);
                if (rescale ? !wait_pv(gj - 1) : (gj >= (uint32_t)PC::PBUF && !wait_pv(gj - PC::PBUF))) {
                    ok = false;
                    break;
                }
                // the P row -> TMEM: word c holds keys 4c .. 4c + 3, as the MMA reads A
                tmem_st32(tmem + lane_off + PC::T_P + 32 * (PC::PBUF * q + gj % PC::PBUF), pk);
                tmem_wait_st();
                if (rescale) {
                    tc_fence_after();
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int cc = 0; cc < 4; cc += 2) {   // two 32-column loads per round trip
                        uint32_t u[32], w[32];
                        tmem_ld32(tO + cc * 32, u);
                        tmem_ld32(tO + cc * 32 + 32, w);
                        tmem_wait_ld();
#pragma unroll
                        for (int i2 = 0; i2 < 32; i2 += 2) {
                            const float2 v2 =
                                __fmul2_rn(make_float2(__uint_as_float(u[i2]), __uint_as_float(u[i2 + 1])), a2);
                            u[i2] = __float_as_uint(v2.x);
                            u[i2 + 1] = __float_as_uint(v2.y);
                            const float2 w2 =
                                __fmul2_rn(make_float2(__uint_as_float(w[i2]), __uint_as_float(w[i2 + 1])), a2);
                            w[i2] = __float_as_uint(w2.x);
                            w[i2 + 1] = __float_as_uint(w2.y);
                        }
                        tmem_st32(tO + cc * 32, u);
                        tmem_st32(tO + cc * 32 + 32, w);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(&B->p_full[q][gj & 1]);
            }
            if (!ok) break;
            // epilogue: O / l -> bf16, lse
            if (!wait_pv(g + nt - 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float fin = (l > 0.0f) ? __fdiv_rn(ref, l) : 0.0f;
            const bool store = rloc < L;
            uint16_t* orow = p.o + ((long long)(d.start + rcl) * p.H + h) * 128;
            const float2 f2 = make_float2(fin, fin);
#pragma unroll
            for (int cc = 0; cc < 4; cc++) {
                uint32_t u[32];
                tmem_ld32(tO + cc * 32, u);
                tmem_wait_ld();
                uint32_t packed[16];
#pragma unroll
                for (int i2 = 0; i2 < 16; i2++) {
                    const float2 v2 =
                        __fmul2_rn(make_float2(__uint_as_float(u[2 * i2]), __uint_as_float(u[2 * i2 + 1])), f2);
                    packed[i2] = pack_bf16x2(v2.x, v2.y);
                }
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                    for (int i2 = 0; i2 < 4; i2++)
                        dst[i2] = make_uint4(packed[4 * i2], packed[4 * i2 + 1], packed[4 * i2 + 2], packed[4 * i2 + 3]);
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
    return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM, st, mq, mk, mv, p);
}

// DYN: the just-in-time (ticket) work order, instantiated with the hardware exp2 only
template <int MODE, int EXPM = ATTN_EXP_HW, bool DYN = false>
static cudaError_t launch_pair(const void* q, const void* k, const void* v, const FwdParams& p, int grid,
                               cudaStream_t st) {
    if constexpr (EXPM == ATTN_EXP_HW && !DYN) {
        if (p.dyn) return launch_pair<MODE, EXPM, true>(q, k, v, p, grid, st);
    }
    using PC = PairCfgT<MODE>;
    CUtensorMap mq, mk, mv;
    // Q, K rows: 128 E4M3 bytes (128-byte swizzle), or 64 NVFP4 bytes (64-byte swizzle)
    if (!make_map(&mq, q, 1, p.T, p.H, PC::QD, PC::QD, !PC::NV) || !make_map(&mk, k, 1, p.T, p.H, PC::QD, PC::QD, !PC::NV) ||
        !make_map(&mv, v, 1, p.T, p.H, 128, 128, true))
        return cudaErrorInvalidValue;
    auto kern = attn_pair_kernel<MODE, EXPM, DYN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PC::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(PC::THREADS), PC::SMEM, st, mq, mk, mv, p);
}

// mode: 0 bf16, 1 E4M3 tile scales, 2 E4M3 per-column scales, 3 MX, 4 MX with per-token V (causal-exact)
cudaError_t launch_attn(int mode, int expm, int D, const void* q, const void* k, const void* v, const FwdParams& p,
                        int grid, cudaStream_t st) {
    if (expm != ATTN_EXP_HW) {
        if (D != 128) return cudaErrorInvalidValue;
        if (mode == MODE_E4M3_TILE)
            return expm == ATTN_EXP_SCHRAUDOLPH ? launch_pair<MODE_E4M3_TILE, ATTN_EXP_SCHRAUDOLPH>(q, k, v, p, grid, st)
                                                : launch_pair<MODE_E4M3_TILE, ATTN_EXP_MITCHELL_P>(q, k, v, p, grid, st);
        if (mode == MODE_MX)
            return expm == ATTN_EXP_SCHRAUDOLPH ? launch_pair<MODE_MX, ATTN_EXP_SCHRAUDOLPH>(q, k, v, p, grid, st)
                                                : launch_pair<MODE_MX, ATTN_EXP_MITCHELL_P>(q, k, v, p, grid, st);
        if (mode == MODE_NVFP4)
            return expm == ATTN_EXP_SCHRAUDOLPH ? launch_pair<MODE_NVFP4, ATTN_EXP_SCHRAUDOLPH>(q, k, v, p, grid, st)
                                                : launch_pair<MODE_NVFP4, ATTN_EXP_MITCHELL_P>(q, k, v, p, grid, st);
        return cudaErrorInvalidValue;
    }
    if (mode == MODE_BF16) return D == 128 ? launch_t<2, 128, MODE_BF16>(q, k, v, p, grid, st)
                                           : launch_t<2, 64, MODE_BF16>(q, k, v, p, grid, st);
    // E4M3 and MX at d = 128: two query tiles per CTA (the work list is built in pair mode)
    if (mode == MODE_E4M3_TILE) return D == 128 ? launch_pair<MODE_E4M3_TILE>(q, k, v, p, grid, st)
                                                : launch_t<1, 64, MODE_E4M3_TILE>(q, k, v, p, grid, st);
    if (mode == MODE_E4M3_COL) return D == 128 ? launch_pair<MODE_E4M3_COL>(q, k, v, p, grid, st)
                                               : launch_t<1, 64, MODE_E4M3_COL>(q, k, v, p, grid, st);
    if (mode == MODE_MX && D == 128) return launch_pair<MODE_MX>(q, k, v, p, grid, st);
    if (mode == MODE_MX_EXACT && D == 128) return launch_pair<MODE_MX_EXACT>(q, k, v, p, grid, st);
    if (mode == MODE_NVFP4 && D == 128) return launch_pair<MODE_NVFP4>(q, k, v, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace pa
