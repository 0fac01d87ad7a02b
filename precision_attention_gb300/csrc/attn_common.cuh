// attn_common.cuh -- pieces shared by the attention kernels: kernel modes, the
// tile configuration of the one-tile kernel (whose descriptor helpers the pair
// kernels reuse), shared-memory matrix descriptors of the Q/K/V/P tiles and
// the bounded drain wait.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "params.h"
#include "ptx.cuh"

namespace pa {

enum { MODE_BF16 = 0, MODE_E4M3_TILE = 1, MODE_E4M3_COL = 2, MODE_MX = 3, MODE_MX_EXACT = 4, MODE_NVFP4 = 5 };

template <int ELT, int D, int MODE>
struct Cfg {
    static constexpr int RB = D * ELT;                  // bytes per Q/K/V row
    static constexpr bool SW128 = RB >= 128;
    static constexpr int ATOMS = SW128 ? RB / 128 : 1;  // 128-byte column blocks per row
    static constexpr int BOX_ELEMS = SW128 ? 128 / ELT : D;
    static constexpr int TILE = 128 * RB;
    static constexpr int PBYTES = 128 * 128 * ELT;
    static constexpr int PBUF = ELT == 1 ? 2 : 1;       // P buffers (BF16: one, for shared-memory room)
    static constexpr int NS = ELT == 2 ? 2 : 5;         // K/V ring depth
    static constexpr int KSTEPS_S = RB / 32;            // 32 bytes of K per MMA
    static constexpr int KSTEPS_PV = 128 * ELT / 32;
    static constexpr int KPER = 32 / ELT;               // keys per P V MMA
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_P = OFF_Q + TILE;
    static constexpr int OFF_KV = OFF_P + PBUF * PBYTES;
    static constexpr int OFF_XCH = OFF_KV + NS * 2 * TILE;  // float [2 parities][2 halves][128 rows] row maxima
    static constexpr int OFF_XL = OFF_XCH + 2 * 2 * 128 * 4; // float [2 halves][128 rows] row sums
    static constexpr int OFF_BAR = OFF_XL + 2 * 128 * 4;
    // at least 116 KB so that one CTA (which allocates all 512 TMEM columns) fits per SM
    static constexpr int SMEM = (OFF_BAR + 512 + 1024) > 116 * 1024 ? (OFF_BAR + 512 + 1024) : 116 * 1024;
    static constexpr int SOFTMAX_WARPS = 8;                  // two warps (column halves) per row quarter
    static constexpr int THREADS = 64 + 32 * SOFTMAX_WARPS;
    static constexpr int HC = 64;                            // S columns per softmax thread
    static constexpr int HD = D / 2;                         // O columns per softmax thread
    // TMEM columns
    static constexpr uint32_t T_O = 256;
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

// start-address increments (16-byte units) of K step kk for each operand
template <int ELT, int D, int MODE>
__device__ __forceinline__ constexpr uint64_t koff(int kk) {
    using C = Cfg<ELT, D, MODE>;
    return C::SW128 ? (uint64_t)(((kk * 32) / 128) * (128 * 128) + (kk * 32) % 128) >> 4 : (uint64_t)(kk * 32) >> 4;
}
__device__ __forceinline__ constexpr uint64_t poff(int kk) {
    return (uint64_t)(((kk * 32) / 128) * (128 * 128) + (kk * 32) % 128) >> 4;
}
template <int ELT, int D, int MODE>
__device__ __forceinline__ constexpr uint64_t voff(int kk) {
    using C = Cfg<ELT, D, MODE>;
    return C::SW128 ? (uint64_t)(kk * C::KPER * 128) >> 4 : (uint64_t)(kk * C::KPER * 64) >> 4;
}

// Limit of the end-of-kernel drains (copies and MMAs already in flight when a wait
// gave up): those complete by themselves, so the drains keep this long limit
// whatever the (possibly short) limit of the ordinary waits.
constexpr long long kDrainLimit = 4000000000LL;

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
}

// host: tensor map of a [T][H][D] tensor, box = (box_elems channels, 1 head, 128 tokens)
inline bool make_map(CUtensorMap* m, const void* base, int elt, int T, int H, int D, int box_elems, bool sw128) {
    return make_tensor_map_3d(m, base, elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              D, H, T, (uint64_t)D * elt, (uint64_t)H * D * elt, box_elems, 128,
                              sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace pa
