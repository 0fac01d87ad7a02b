// params.h -- launch parameter blocks shared by the host launchers and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace pa {

struct QuantParams {
    const void* x;
    int in_bf16;
    long long tstride, hstride;   // elements
    int T, H, d, nd;
    const int32_t* cu;            // may be null (one document)
    uint8_t* codes;               // [T][H][d]
    void* scales;
    long long scale_cap;          // nb_cap (E4M3) or nt_cap (MX)
    int block;
    int rotate;
    unsigned long long seed;
    int mx_rule;
    uint32_t* status;
    uint8_t* sf16;                // NVFP4: the 1024-byte scale-factor tiles [H][scale_cap]
    int32_t* gtab;                // device document table [3][nd + 1] (start, tile prefix, block
                                  // prefix) written by doc_table_kernel, or null: each CTA builds
                                  // its own in shared memory (nd <= MAX_DOCS)
};

struct SchedParams {
    const int32_t* cu;     // may be null
    int nd, T, H, causal;
    int bq, bk, bv;        // E4M3 scale blocks (1 when unused)
    WsHeader* hdr;
    DocEntry* docs;
    WorkItem* items;
    long long items_cap;
    int qpair;             // 1: an item covers the query tiles 2p and 2p + 1 of a document
    int ticket0;           // first ticket of the forward's just-in-time schedule (its grid size)
};

struct VrefParams {
    const float* sv;          // V scales (E4M3 layouts), or
    const uint8_t* sv_e8;     // V exponents X + 127 per token (MX token layout): scale 2^X, 0 for X = -127
    long long sv_cap;
    const DocEntry* docs;
    const WsHeader* hdr;
    float* vref;
    int H, nd, T, exact, bv;
    // per (head, 128-token key tile) multipliers, written when tiles != 0:
    // {K scale x C, log2 r, 1 / r, 0} with r = V scale x (1 / ref)
    int tiles, bk;
    const float* sk;
    long long sk_cap;
    float C;
    float4* tsc;
    long long tsc_cap;
};

struct FwdParams {
    const DocEntry* docs;
    const WorkItem* items;
    WsHeader* hdr;
    uint16_t* o;          // bf16 [T][H][D]
    float* lse;           // [H][T]
    int T, H, nd;
    int causal, exact;
    float C;              // softmax_scale * log2(e) (/ d when Q and K are rotated)
    const float *sq, *sk, *sv;
    long long capq, capk, capv;
    int bq, bk, bv;
    const float* vref;
    const uint8_t *mq, *mk, *mv;
    long long ntcap;
    const float4* tsc;    // per (head, key tile) multipliers (E4M3 tile mode), see VrefParams
    long long tsc_cap;
    long long wait_limit;
    int dyn;              // 1: items taken just in time by ticket (pair kernel), else static rounds
    // test build only (PA_PDUMP): every E4M3 probability code handed to the P V MMA,
    // byte [(h * T + t) * pdump_stride + k] for row t, document-local key k
    uint8_t* pdump;
    long long pdump_stride;
};

// The backward (BF16 operands, d = 64 or 128). Per-row vectors are kept per (head,
// 128-token tile) so that one tile's 128 values are one aligned 512-byte copy:
// vec[0][h][tile][r] = lse log2(e), vec[1][h][tile][r] = rowsum(dO o O), tile =
// DocEntry::toff + local tile, rows past the document's end 0.
struct BwdParams {
    const DocEntry* docs;
    const WorkItem* items;
    WsHeader* hdr;
    const uint16_t* q;       // bf16 [T][H][D] (the dQ kernel's row tiles)
    const uint16_t* o;       // bf16 [T][H][D] (prep)
    const uint16_t* dout;    // bf16 [T][H][D] (prep)
    const float* lse;        // [H][T] natural log (prep)
    float* vec;              // [2][H][tiles_cap][128]
    long long tiles_cap;
    uint16_t *dq, *dk, *dv;  // bf16 [T][H][D]
    int T, H, nd, causal;
    float C;                 // softmax_scale * log2(e)
    float scale;             // softmax_scale
    long long wait_limit;
    int kv_only;             // 1: the gradient kernel takes only the dK/dV role (dQ has its own kernel)
};

// host: a 3-D tiled tensor map over [d2][d1][d0] (d0 contiguous), box (box0, 1, box2)
bool make_tensor_map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t d0, uint64_t d1,
                        uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box2,
                        CUtensorMapSwizzle swizzle);
// host: multiprocessor count of the current device (cached per device)
int sm_count();

cudaError_t launch_quantize(const QuantParams& p, int layout, cudaStream_t st);
// Q, K (ps[0], ps[1], layout_qk) and V (ps[2], layout_v) in one launch: same shape, dtype and strides
cudaError_t launch_quantize_qkv(const QuantParams* ps, int layout_qk, int layout_v, cudaStream_t st);
cudaError_t launch_sched(const SchedParams& p, cudaStream_t st);
cudaError_t launch_vref(const VrefParams& p, cudaStream_t st);
// mode: 0 bf16, 1 E4M3 with one scale per tile, 2 E4M3 per-column scales, 3 MXFP8,
// 4 MXFP8 Q and K with one V exponent per token (the causal-exact MX mode); expm: the
// probabilities' exponential (attn_exp_mode; the bit-level ones with modes 1 and 3 at D = 128)
// the backward after its work list: the per-row vectors, then the gradient kernel
// (q, k, v, dout: bf16 [T][H][D], D = 64 or 128; grid: CTAs of the persistent
// gradient kernel, even)
cudaError_t launch_bwd(int D, const void* q, const void* k, const void* v, const void* dout, const BwdParams& p,
                       int grid, cudaStream_t st);
cudaError_t launch_attn(int mode, int expm, int D, const void* q, const void* k, const void* v, const FwdParams& p,
                        int grid, cudaStream_t st);

}  // namespace pa
