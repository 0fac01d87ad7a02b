// capi.cu -- the extern "C" boundary declared in include/attn.h: argument
// validation, workspace layout and the kernel launches. No allocation, no
// stream synchronisation (except attn_read_device_status, by definition).
#include <atomic>
#include <cmath>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/attn.h"
#ifdef PA_PDUMP
#include "../../include/attn_pdump.h"
#endif
#include "params.h"

using namespace pa;

namespace {

constexpr long long kWaitLimit = 4000000000LL;   // SM cycles (about 2 s) before a wait gives up
std::atomic<long long> g_wait_limit{kWaitLimit};   // attn_set_wait_limit
std::atomic<int> g_schedule{ATTN_SCHED_STATIC};     // attn_set_schedule
#ifdef PA_PDUMP
uint8_t* g_pdump = nullptr;                        // attn_pdump_set (test build)
long long g_pdump_stride = 0;
#endif

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status check_shape(const attn_shape* s) {
    if (!s) return ATTN_ERR_INVALID_ARG;
    if (s->total_tokens < 1 || s->heads < 1 || s->num_docs < 1) return ATTN_ERR_INVALID_ARG;
    if (s->head_dim != 64 && s->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if (!s->cu_seqlens && s->num_docs != 1) return ATTN_ERR_INVALID_ARG;
    if (s->num_docs > s->total_tokens) return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(s->total_tokens) * s->heads > (1LL << 31) - 1) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

long long blocks_cap(const attn_shape* s, int block) {
    return (static_cast<long long>(s->total_tokens) + block - 1) / block + s->num_docs;
}
long long tiles_cap(const attn_shape* s) { return blocks_cap(s, 128); }

attn_status check_ws(const attn_shape* s, void* ws, size_t bytes) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return ATTN_ERR_WORKSPACE;
    if (bytes < ws_layout(s->total_tokens, s->heads, s->num_docs).total) return ATTN_ERR_WORKSPACE;
    return ATTN_OK;
}

bool valid_block(int layout, int block) {
    if (layout == ATTN_E4M3_TOKBLOCK) return block == 1 || block == 32 || block == 64 || block == 128;
    if (layout == ATTN_NVFP4) return block == 128;
    return layout == ATTN_MX_ROW32 || layout == ATTN_MX_COL32 || layout == ATTN_MX_TOKEN;
}

attn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace

namespace pa {

// Every synchronous check of attn_fp8_fwd, in its order; the workspace is checked
// only when check_workspace is set (the no-allocation entry point has none).
// *mode receives the kernel mode (1 E4M3 one scale per tile, 2 E4M3 per-column
// scales, 3 MX, 4 MX with per-token V, 5 NVFP4 Q K^T with E4M3 V).
attn_status fp8_fwd_check(const attn_qtensor* q, const attn_qtensor* k, const attn_qtensor* v,
                          const attn_shape* shape, int causal, int causal_exact, float softmax_scale, const void* o,
                          const float* lse, bool check_workspace, void* workspace, size_t workspace_bytes,
                          int* mode) {
    attn_status st = check_shape(shape);
    if (st != ATTN_OK) return st;
    if (!q || !k || !v || !o || !lse || !mode) return ATTN_ERR_INVALID_ARG;
    if (!q->codes || !k->codes || !v->codes || !q->scales || !k->scales || !v->scales) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q->codes) || !aligned16(k->codes) || !aligned16(v->codes) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(q->scales) || !aligned16(k->scales) || !aligned16(v->scales))
        return ATTN_ERR_INVALID_ARG;
    if (!(softmax_scale <= 0.0f || std::isfinite(softmax_scale))) return ATTN_ERR_INVALID_ARG;
    if (check_workspace && (st = check_ws(shape, workspace, workspace_bytes)) != ATTN_OK) return st;
    const bool mx = q->layout == ATTN_MX_ROW32;
    const bool nv = q->layout == ATTN_NVFP4;
    if (nv) {
        // mixed NVFP4/FP8: NVFP4 Q and K, E4M3 V with one scale per 128-token block
        if (k->layout != ATTN_NVFP4 || v->layout != ATTN_E4M3_TOKBLOCK) return ATTN_ERR_INVALID_ARG;
        if (q->block != 128 || k->block != 128 || v->block != 128) return ATTN_ERR_INVALID_ARG;
        if (shape->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
        if (causal_exact) return ATTN_ERR_UNSUPPORTED;   // the 128-token block scales span later tokens
    } else if (mx) {
        if (k->layout != ATTN_MX_ROW32 || (v->layout != ATTN_MX_COL32 && v->layout != ATTN_MX_TOKEN))
            return ATTN_ERR_INVALID_ARG;
        if (shape->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
        // causal-exact MX: V needs one exponent per token (its 32-token column blocks
        // would let a later token change an earlier row's scale)
        if (causal_exact && (!causal || v->layout != ATTN_MX_TOKEN)) return ATTN_ERR_INVALID_ARG;
    } else {
        if (q->layout != ATTN_E4M3_TOKBLOCK || k->layout != ATTN_E4M3_TOKBLOCK || v->layout != ATTN_E4M3_TOKBLOCK)
            return ATTN_ERR_INVALID_ARG;
        if (!valid_block(0, q->block) || !valid_block(0, k->block) || !valid_block(0, v->block))
            return ATTN_ERR_INVALID_ARG;
    }
    if (v->rotated) return ATTN_ERR_INVALID_ARG;
    if (q->rotated != k->rotated || (q->rotated && q->hadamard_seed != k->hadamard_seed))
        return ATTN_ERR_SEED_MISMATCH;
    if (!mx && causal_exact && (!causal || q->block != 1 || k->block != 1 || v->block != 1))
        return ATTN_ERR_INVALID_ARG;
    *mode = v->layout == ATTN_MX_TOKEN ? 4 : 3;
    if (!mx) *mode = (q->block == 128 && k->block == 128 && v->block == 128 && !causal_exact) ? 1 : 2;
    if (nv) *mode = 5;
    return ATTN_OK;
}

}  // namespace pa

extern "C" {

const char* attn_status_string(int32_t s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case ATTN_ERR_NONFINITE: return "non-finite input in a quantisation block";
        case ATTN_ERR_SEED_MISMATCH: return "Q and K rotations differ";
        case ATTN_ERR_BAD_SEQLENS: return "malformed cu_seqlens";
        case ATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown status";
    }
}

attn_status attn_quantize_sizes(const attn_shape* shape, int32_t layout, int32_t block, size_t* codes_bytes,
                                size_t* scales_bytes) {
    attn_status st = check_shape(shape);
    if (st != ATTN_OK) return st;
    if (!codes_bytes || !scales_bytes) return ATTN_ERR_INVALID_ARG;
    if (layout < 0 || layout > 4 || !valid_block(layout, block)) return ATTN_ERR_INVALID_ARG;
    if (layout != ATTN_E4M3_TOKBLOCK && shape->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    const long long T = shape->total_tokens, H = shape->heads, d = shape->head_dim;
    *codes_bytes = static_cast<size_t>(T * H * (layout == ATTN_NVFP4 ? d / 2 : d));
    if (layout == ATTN_NVFP4)
        *scales_bytes = nvfp4_sf_offset(H, tiles_cap(shape)) + static_cast<size_t>(H * tiles_cap(shape)) * 1024;
    else if (layout == ATTN_E4M3_TOKBLOCK)
        *scales_bytes = static_cast<size_t>(H * blocks_cap(shape, block)) * sizeof(float);
    else if (layout == ATTN_MX_TOKEN)
        *scales_bytes = static_cast<size_t>(H * blocks_cap(shape, 1));
    else
        *scales_bytes = static_cast<size_t>(H * tiles_cap(shape)) * 512;
    return ATTN_OK;
}

attn_status attn_workspace_size(const attn_shape* shape, size_t* bytes) {
    attn_status st = check_shape(shape);
    if (st != ATTN_OK) return st;
    if (!bytes) return ATTN_ERR_INVALID_ARG;
    *bytes = ws_layout(shape->total_tokens, shape->heads, shape->num_docs).total;
    return ATTN_OK;
}

attn_status attn_fwd_workspace_size(const attn_shape* shape, int32_t causal, size_t* bytes) {
    (void)causal;   // the work list holds one entry per query-tile unit either way
    return attn_workspace_size(shape, bytes);
}

// Checks one output operand and its input against the shape and fills its kernel parameters.
static attn_status quant_params(const void* x, int32_t in_dtype, int64_t token_stride, int64_t head_stride,
                                const attn_shape* shape, int32_t rotate, uint64_t hadamard_seed,
                                const attn_qtensor* out, void* workspace, QuantParams* pp) {
    if (!x || !out || !out->codes || !out->scales) return ATTN_ERR_INVALID_ARG;
    if (in_dtype != ATTN_IN_F32 && in_dtype != ATTN_IN_BF16) return ATTN_ERR_INVALID_ARG;
    if (!valid_block(out->layout, out->block) || out->layout < 0 || out->layout > 4) return ATTN_ERR_INVALID_ARG;
    if (out->layout != ATTN_E4M3_TOKBLOCK && shape->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if (out->mx_rule != ATTN_MX_RULE_NOSAT && out->mx_rule != ATTN_MX_RULE_OCP_FLOOR) return ATTN_ERR_INVALID_ARG;
    const int elt = in_dtype == ATTN_IN_BF16 ? 2 : 4;
    if (!aligned16(x) || !aligned16(out->codes) || !aligned16(out->scales)) return ATTN_ERR_INVALID_ARG;
    if (token_stride < 1 || head_stride < 1 || (token_stride * elt) % 16 || (head_stride * elt) % 16)
        return ATTN_ERR_INVALID_ARG;
    QuantParams& p = *pp;
    std::memset(&p, 0, sizeof(p));
    p.x = x;
    p.in_bf16 = in_dtype == ATTN_IN_BF16;
    p.tstride = token_stride;
    p.hstride = head_stride;
    p.T = shape->total_tokens;
    p.H = shape->heads;
    p.d = shape->head_dim;
    p.nd = shape->num_docs;
    p.cu = shape->cu_seqlens;
    p.codes = static_cast<uint8_t*>(out->codes);
    p.scales = out->scales;
    // MX layouts have fixed blocks (32 channels or tokens; one token): the caller's
    // `block` field does not reach the kernel's block arithmetic for them
    p.block = out->layout == ATTN_E4M3_TOKBLOCK ? out->block
              : out->layout == ATTN_NVFP4        ? 128
              : (out->layout == ATTN_MX_TOKEN ? 1 : 32);
    p.scale_cap = out->layout == ATTN_E4M3_TOKBLOCK ? blocks_cap(shape, out->block)
                  : out->layout == ATTN_MX_TOKEN     ? blocks_cap(shape, 1)
                                                     : tiles_cap(shape);
    p.sf16 = out->layout == ATTN_NVFP4
                 ? static_cast<uint8_t*>(out->scales) + nvfp4_sf_offset(shape->heads, tiles_cap(shape))
                 : nullptr;
    p.rotate = rotate != 0;
    p.seed = hadamard_seed;
    p.mx_rule = out->mx_rule;
    p.status = &static_cast<WsHeader*>(workspace)->status;
    p.gtab = shape->num_docs > MAX_DOCS
                 ? reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
                                              ws_layout(shape->total_tokens, shape->heads, shape->num_docs).qtab_off)
                 : nullptr;
    return ATTN_OK;
}

static void mark_rotation(attn_qtensor* out, int32_t rotate, uint64_t hadamard_seed) {
    out->rotated = rotate != 0;
    out->hadamard_seed = rotate ? hadamard_seed : 0;
}

attn_status attn_quantize(const void* x, int32_t in_dtype, int64_t token_stride, int64_t head_stride,
                          const attn_shape* shape, int32_t rotate, uint64_t hadamard_seed, attn_qtensor* out,
                          void* workspace, size_t workspace_bytes, void* stream) {
    attn_status st = check_shape(shape);
    if (st != ATTN_OK) return st;
    QuantParams p;
    if ((st = quant_params(x, in_dtype, token_stride, head_stride, shape, rotate, hadamard_seed, out, workspace, &p)) !=
        ATTN_OK)
        return st;
    if ((st = check_ws(shape, workspace, workspace_bytes)) != ATTN_OK) return st;
    st = cuda_status(launch_quantize(p, out->layout, static_cast<cudaStream_t>(stream)));
    if (st == ATTN_OK) mark_rotation(out, rotate, hadamard_seed);
    return st;
}

attn_status attn_quantize_qkv(const void* q, const void* k, const void* v, int32_t in_dtype, int64_t token_stride,
                              int64_t head_stride, const attn_shape* shape, int32_t rotate, uint64_t hadamard_seed,
                              attn_qtensor* q_out, attn_qtensor* k_out, attn_qtensor* v_out, void* workspace,
                              size_t workspace_bytes, void* stream) {
    attn_status st = check_shape(shape);
    if (st != ATTN_OK) return st;
    if (!q_out || !k_out || !v_out) return ATTN_ERR_INVALID_ARG;
    QuantParams ps[3];
    const void* xs[3] = {q, k, v};
    attn_qtensor* outs[3] = {q_out, k_out, v_out};
    for (int t = 0; t < 3; t++)
        if ((st = quant_params(xs[t], in_dtype, token_stride, head_stride, shape, t < 2 ? rotate : 0, hadamard_seed,
                               outs[t], workspace, &ps[t])) != ATTN_OK)
            return st;
    // the pairs one launch serves: Q and K alike, V in the layout the forward takes with them
    const int lq = q_out->layout, lv = v_out->layout;
    bool ok = k_out->layout == lq;
    if (lq == ATTN_E4M3_TOKBLOCK)
        ok = ok && lv == ATTN_E4M3_TOKBLOCK && k_out->block == q_out->block && v_out->block == q_out->block;
    else if (lq == ATTN_MX_ROW32)
        ok = ok && (lv == ATTN_MX_COL32 || lv == ATTN_MX_TOKEN);
    else if (lq == ATTN_NVFP4)
        ok = ok && lv == ATTN_E4M3_TOKBLOCK && v_out->block == 128;
    else
        ok = false;
    if (!ok) return ATTN_ERR_INVALID_ARG;
    if ((st = check_ws(shape, workspace, workspace_bytes)) != ATTN_OK) return st;
    st = cuda_status(launch_quantize_qkv(ps, lq, lv, static_cast<cudaStream_t>(stream)));
    if (st == ATTN_OK) {
        mark_rotation(q_out, rotate, hadamard_seed);
        mark_rotation(k_out, rotate, hadamard_seed);
        mark_rotation(v_out, 0, 0);
    }
    return st;
}

static attn_status forward(int mode, int expm, const void* q, const void* k, const void* v, const attn_qtensor* qq,
                           const attn_qtensor* qk, const attn_qtensor* qv, const attn_shape* shape, int causal,
                           int exact, float softmax_scale, int rotated, void* o, float* lse, void* workspace,
                           cudaStream_t stream) {
    const int T = shape->total_tokens, H = shape->heads, d = shape->head_dim, nd = shape->num_docs;
    const WsLayout L = ws_layout(T, H, nd);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    DocEntry* docs = reinterpret_cast<DocEntry*>(ws + L.docs_off);
    WorkItem* items = reinterpret_cast<WorkItem*>(ws + L.items_off);
    float* vref = reinterpret_cast<float*>(ws + L.vref_off);
    float4* tsc = reinterpret_cast<float4*>(ws + L.tsc_off);
    const bool e4m3 = mode == 1 || mode == 2 || mode == 5;   // fp32 block scales (NVFP4: Q, K's 128-token ones)

    SchedParams sp;
    sp.cu = shape->cu_seqlens;
    sp.nd = nd;
    sp.T = T;
    sp.H = H;
    sp.causal = causal;
    sp.bq = e4m3 ? qq->block : 1;
    sp.bk = e4m3 ? qk->block : 1;
    sp.bv = e4m3 ? qv->block : 1;
    sp.hdr = hdr;
    sp.docs = docs;
    sp.items = items;
    sp.items_cap = L.items_cap;
    sp.qpair = mode >= 1 && d == 128;   // FP8, d = 128: two query tiles per item
    const int grid = attn_device_sm_count();
    if (grid < 1) return ATTN_ERR_CUDA;
    sp.ticket0 = grid;
    cudaError_t e = launch_sched(sp, stream);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;

    FwdParams fp;
    std::memset(&fp, 0, sizeof(fp));
    fp.docs = docs;
    fp.items = items;
    fp.hdr = hdr;
    fp.o = static_cast<uint16_t*>(o);
    fp.lse = lse;
    fp.T = T;
    fp.H = H;
    fp.nd = nd;
    fp.causal = causal;
    fp.exact = exact;
    const double sc = softmax_scale > 0.0f ? static_cast<double>(softmax_scale) : 1.0 / std::sqrt((double)d);
    fp.C = static_cast<float>(sc * 1.4426950408889634 / (rotated ? static_cast<double>(d) : 1.0));
    fp.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
    fp.dyn = g_schedule.load(std::memory_order_relaxed) == ATTN_SCHED_TICKET;
#ifdef PA_PDUMP
    fp.pdump = g_pdump;
    fp.pdump_stride = g_pdump_stride;
#endif
    fp.bq = fp.bk = fp.bv = 1;
    if (e4m3) {
        fp.sq = static_cast<const float*>(qq->scales);
        fp.sk = static_cast<const float*>(qk->scales);
        fp.sv = static_cast<const float*>(qv->scales);
        fp.capq = blocks_cap(shape, qq->block);
        fp.capk = blocks_cap(shape, qk->block);
        fp.capv = blocks_cap(shape, qv->block);
        fp.bq = qq->block;
        fp.bk = qk->block;
        fp.bv = qv->block;
        fp.vref = vref;
        VrefParams vp;
        std::memset(&vp, 0, sizeof(vp));
        vp.sv = fp.sv;
        vp.sv_cap = fp.capv;
        vp.docs = docs;
        vp.hdr = hdr;
        vp.vref = vref;
        vp.H = H;
        vp.nd = nd;
        vp.T = T;
        vp.exact = exact;
        vp.bv = qv->block;
        vp.tiles = ((mode == 1 || mode == 5) && !exact) ? 1 : 0;
        vp.bk = qk->block;
        vp.sk = fp.sk;
        vp.sk_cap = fp.capk;
        vp.C = fp.C;
        vp.tsc = tsc;
        vp.tsc_cap = L.tsc_cap;
        fp.tsc = tsc;
        fp.tsc_cap = L.tsc_cap;
        if (mode == 5) {   // NVFP4: the 16-channel scale tiles after the fp32 block scales
            const size_t off = nvfp4_sf_offset(H, tiles_cap(shape));
            fp.mq = static_cast<const uint8_t*>(qq->scales) + off;
            fp.mk = static_cast<const uint8_t*>(qk->scales) + off;
            fp.ntcap = tiles_cap(shape);
        }
        if ((e = launch_vref(vp, stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    } else if (mode == 3 || mode == 4) {
        fp.mq = static_cast<const uint8_t*>(qq->scales);
        fp.mk = static_cast<const uint8_t*>(qk->scales);
        fp.mv = static_cast<const uint8_t*>(qv->scales);
        fp.ntcap = tiles_cap(shape);
        if (mode == 4) {
            // V exponents per token: the V references (running maxima in the exact mode)
            fp.capv = blocks_cap(shape, 1);
            fp.bv = 1;
            fp.vref = vref;
            VrefParams vp;
            std::memset(&vp, 0, sizeof(vp));
            vp.sv_e8 = fp.mv;
            vp.sv_cap = fp.capv;
            vp.docs = docs;
            vp.hdr = hdr;
            vp.vref = vref;
            vp.H = H;
            vp.nd = nd;
            vp.T = T;
            vp.exact = exact;
            vp.bv = 1;
            if ((e = launch_vref(vp, stream)) != cudaSuccess) return ATTN_ERR_CUDA;
        }
    }
    e = launch_attn(mode, expm, d, q, k, v, fp, grid, stream);
    return e == cudaSuccess ? ATTN_OK : (e == cudaErrorInvalidValue ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_CUDA);
}

attn_status attn_fp8_fwd(const attn_qtensor* q, const attn_qtensor* k, const attn_qtensor* v,
                         const attn_shape* shape, int32_t causal, int32_t causal_exact, float softmax_scale,
                         void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    int mode = 0;
    attn_status st = pa::fp8_fwd_check(q, k, v, shape, causal, causal_exact, softmax_scale, o, lse, true, workspace,
                                       workspace_bytes, &mode);
    if (st != ATTN_OK) return st;
    return forward(mode, ATTN_EXP_HW, q->codes, k->codes, v->codes, q, k, v, shape, causal != 0, causal_exact != 0,
                   softmax_scale, q->rotated, o, lse, workspace, static_cast<cudaStream_t>(stream));
}

attn_status attn_fp8_fwd_ex(const attn_qtensor* q, const attn_qtensor* k, const attn_qtensor* v,
                            const attn_shape* shape, int32_t causal, int32_t causal_exact, float softmax_scale,
                            int32_t exp_mode, void* o, float* lse, void* workspace, size_t workspace_bytes,
                            void* stream) {
    int mode = 0;
    attn_status st = pa::fp8_fwd_check(q, k, v, shape, causal, causal_exact, softmax_scale, o, lse, true, workspace,
                                       workspace_bytes, &mode);
    if (st != ATTN_OK) return st;
    if (exp_mode < ATTN_EXP_HW || exp_mode > ATTN_EXP_MITCHELL_P) return ATTN_ERR_INVALID_ARG;
    // the bit-level exponentials: the pair kernel's E4M3 tile and MX paths (inference)
    if (exp_mode != ATTN_EXP_HW && (shape->head_dim != 128 || (mode != 1 && mode != 3 && mode != 5)))
        return ATTN_ERR_UNSUPPORTED;
    return forward(mode, exp_mode, q->codes, k->codes, v->codes, q, k, v, shape, causal != 0, causal_exact != 0,
                   softmax_scale, q->rotated, o, lse, workspace, static_cast<cudaStream_t>(stream));
}

attn_status attn_bf16_fwd(const void* q, const void* k, const void* v, const attn_shape* shape, int32_t causal,
                          float softmax_scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                          void* stream) {
    attn_status st = check_shape(shape);
    if (st != ATTN_OK) return st;
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_INVALID_ARG;
    if (!(softmax_scale <= 0.0f || std::isfinite(softmax_scale))) return ATTN_ERR_INVALID_ARG;
    if ((st = check_ws(shape, workspace, workspace_bytes)) != ATTN_OK) return st;
    return forward(0, ATTN_EXP_HW, q, k, v, nullptr, nullptr, nullptr, shape, causal != 0, 0, softmax_scale, 0, o, lse,
                   workspace, static_cast<cudaStream_t>(stream));
}

static size_t bwd_vec_off(const attn_shape* s) { return ws_layout(s->total_tokens, s->heads, s->num_docs).total; }

attn_status attn_bwd_workspace_size(const attn_shape* shape, size_t* bytes) {
    attn_status st = check_shape(shape);
    if (st != ATTN_OK) return st;
    if (!bytes) return ATTN_ERR_INVALID_ARG;
    *bytes = align_up(bwd_vec_off(shape) + 2 * sizeof(float) * 128 * static_cast<size_t>(shape->heads) *
                                               static_cast<size_t>(tiles_cap(shape)),
                      256);
    return ATTN_OK;
}

attn_status attn_bf16_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, const attn_shape* shape, int32_t causal, float softmax_scale, void* dq,
                          void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
    attn_status st = check_shape(shape);
    if (st != ATTN_OK) return st;
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return ATTN_ERR_INVALID_ARG;
    if (!(softmax_scale <= 0.0f || std::isfinite(softmax_scale))) return ATTN_ERR_INVALID_ARG;
    size_t need = 0;
    attn_bwd_workspace_size(shape, &need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return ATTN_ERR_WORKSPACE;
    const int T = shape->total_tokens, H = shape->heads, nd = shape->num_docs;
    const WsLayout L = ws_layout(T, H, nd);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int grid = attn_device_sm_count();
    if (grid < 2) return ATTN_ERR_CUDA;
    grid &= ~1;   // even: each CTA alternates between the two roles (see attn_bwd.cu)

    SchedParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.cu = shape->cu_seqlens;
    sp.nd = nd;
    sp.T = T;
    sp.H = H;
    sp.causal = causal != 0;
    sp.bq = sp.bk = sp.bv = 1;
    sp.hdr = reinterpret_cast<WsHeader*>(ws);
    sp.docs = reinterpret_cast<DocEntry*>(ws + L.docs_off);
    sp.items = reinterpret_cast<WorkItem*>(ws + L.items_off);
    sp.items_cap = L.items_cap;
    sp.qpair = 0;
    sp.ticket0 = grid;
    if (launch_sched(sp, s) != cudaSuccess) return ATTN_ERR_CUDA;

    BwdParams bp;
    std::memset(&bp, 0, sizeof(bp));
    bp.docs = sp.docs;
    bp.items = sp.items;
    bp.hdr = sp.hdr;
    bp.q = static_cast<const uint16_t*>(q);
    bp.o = static_cast<const uint16_t*>(o);
    bp.dout = static_cast<const uint16_t*>(dout);
    bp.lse = lse;
    bp.vec = reinterpret_cast<float*>(ws + bwd_vec_off(shape));
    bp.tiles_cap = tiles_cap(shape);
    bp.dq = static_cast<uint16_t*>(dq);
    bp.dk = static_cast<uint16_t*>(dk);
    bp.dv = static_cast<uint16_t*>(dv);
    bp.T = T;
    bp.H = H;
    bp.nd = nd;
    bp.causal = causal != 0;
    const double sc =
        softmax_scale > 0.0f ? static_cast<double>(softmax_scale) : 1.0 / std::sqrt(static_cast<double>(shape->head_dim));
    bp.scale = static_cast<float>(sc);
    bp.C = static_cast<float>(sc * 1.4426950408889634);
    bp.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
    const cudaError_t e = launch_bwd(shape->head_dim, q, k, v, dout, bp, grid, s);
    return e == cudaSuccess ? ATTN_OK : (e == cudaErrorInvalidValue ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_CUDA);
}

#ifdef PA_PDUMP
attn_status attn_pdump_set(void* buf, int64_t key_stride) {
    if (buf && (key_stride < 128 || key_stride % 128 || (reinterpret_cast<uintptr_t>(buf) & 15u)))
        return ATTN_ERR_INVALID_ARG;
    g_pdump = static_cast<uint8_t*>(buf);
    g_pdump_stride = buf ? key_stride : 0;
    return ATTN_OK;
}
#endif

attn_status attn_set_schedule(int32_t schedule) {
    if (schedule != ATTN_SCHED_STATIC && schedule != ATTN_SCHED_TICKET) return ATTN_ERR_INVALID_ARG;
    g_schedule.store(schedule, std::memory_order_relaxed);
    return ATTN_OK;
}

attn_status attn_set_wait_limit(int64_t cycles) {
    g_wait_limit.store(cycles > 0 ? static_cast<long long>(cycles) : kWaitLimit, std::memory_order_relaxed);
    return ATTN_OK;
}

attn_status attn_read_device_status(void* workspace, void* stream, uint32_t* flags_out) {
    if (!workspace) return ATTN_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
    uint32_t w = 0;
    if (cudaMemcpy(&w, workspace, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemset(workspace, 0, sizeof(w)) != cudaSuccess) return ATTN_ERR_CUDA;
    if (flags_out) *flags_out = w;
    if (w & ST_TIMEOUT) return ATTN_ERR_DEVICE_TIMEOUT;
    if (w & ST_BAD_SEQLENS) return ATTN_ERR_BAD_SEQLENS;
    if (w & ST_NONFINITE) return ATTN_ERR_NONFINITE;
    return ATTN_OK;
}

int32_t attn_device_sm_count(void) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

}  // extern "C"
